// CPU oracle, in C++, for the Mixtral-style MoE expert layer (forward and
// backward).
//
// TEST INFRASTRUCTURE ONLY. This file exists to check the CUDA path. Only the
// test suite and the smoke check load the library built from it
// (oracle/libmoe_oracle.so, through oracle/cpp_oracle.py); the product path
// never calls it and has no CPU fallback. It shares no code with the CUDA
// library, nor with the numpy oracle next to it: the two oracles are written
// independently and are checked against each other and against the pins.
//
// It is written as the per-expert loop that the sources describe, in double
// precision, with plain loops and no blocking or fusion: for every expert,
// take the (token, slot) pairs routed to it, run the expert's SwiGLU MLP on
// those tokens, scale by the routing weight and add the result back into the
// token rows.
//
// Sources (short tags in the comments below):
//
// [EMT]     "Efficient MoE Training for Biological Foundation Models"
//           (NVIDIA Developer Blog tutorial): §Challenge 1 (the per-expert
//           loop over an expert mask, routing weights and an index_add of the
//           expert outputs; GroupedLinear over split sizes with 2 x the
//           intermediate size as FC1 width), §Challenge 2 (MXFP8: one scale
//           per block of 32 consecutive values), §Challenge 3 (gate_up ->
//           ScaledSwiGLU -> down; the SwiGLU output is multiplied by the
//           routing probabilities).
// [MOEBIO]  "How MoE Architecture Cuts Costs and Boosts Efficiency: Efficient
//           Training of Biological Foundation Models", the Router paragraph
//           (Top-K routing keeps the K highest-scoring experts).
// [OCPMX]   OCP Microscaling Formats (MX) v1.0: a block of 32 elements shares
//           an E8M0 scale 2^(floor(log2 max|V|) - emax_elem); elements round
//           to nearest, ties to even, and saturate. E4M3: emax_elem 8, largest
//           normal 448, smallest normal 2^-6, 3 mantissa bits. E2M1: emax_elem
//           2, values 0, 0.5, 1, 1.5, 2, 3, 4, 6.
// [MXFP4-HOPPER] the hgpu.org abstract on MXFP4 training of MoE models:
//           activations kept in MXFP4 while the GEMMs run in FP8, FP8 -> FP4
//           directly, and a scale-aware row-wise -> column-wise FP4 copy.
//
// Readings where the sources are silent (the same readings as the numpy
// oracle; each is listed in the design notes):
//
// * top-k ties go to the lower expert index; +0 and -0 tie (logits are
//   finite);
// * routing weights are the softmax over the k selected logits;
// * SwiGLU is silu(gate) * up, gate = FC1 columns [0, F), up = [F, 2F);
// * within one expert the routed rows are ordered by token, then slot;
// * the router receives a gradient through the k selected softmax weights;
// * an all-zero MX block gets scale byte 0 (exponent clamped to -127) and
//   zero elements that keep their sign; a block holding Inf or NaN gets scale
//   byte 0xFF and E4M3 element bytes 0x7F (E2M1 element codes 0);
// * in the MXFP8 modes every GEMM consumes operands whose 32-blocks run along
//   its reduction index: x, H, dOut and dY1 along their columns for the
//   forward and dgrad products, W1 along H and W2 along F in the forward, W1
//   along 2F and W2 along H in the dgrads, and the wgrad operands (x, H,
//   dOut, dY1) along tokens inside an expert group, whose rows are padded
//   with zeros to a multiple of 32; intermediate activations (H, dY1) are
//   rounded to float32 before they are quantised; the elementwise backward is
//   straight-through;
// * the SwiGLU backward reads gate and up through their bf16 copies (the
//   forward saves them in bf16) unless save_bf16 is 0; the forward SwiGLU
//   reads the GEMM result unrounded;
// * with MXFP4-carried activations the wgrad operands x and H are the chain
//   row-wise MXFP8 -> row-wise MXFP4 (same blocks) -> column-wise MXFP4
//   (blocks of 32 group rows, scales recomputed from the decoded values);
//   the last step to column-wise MXFP8 is lossless, so those are the values.
//
// Matrices are row-major: x [T, H], logits [T, E], W1 [E, H, 2F], W2 [E, F, H].

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// ------------------------------------------------------------------ matrices

struct Mat {
  long r = 0, c = 0;
  std::vector<double> v;
  Mat() = default;
  Mat(long rows, long cols) : r(rows), c(cols), v((size_t)(rows * cols), 0.0) {}
  double& at(long i, long j) { return v[(size_t)(i * c + j)]; }
  double at(long i, long j) const { return v[(size_t)(i * c + j)]; }
};

// C = A B, each C[i][j] summed over the shared index in ascending order.
Mat matmul(const Mat& A, const Mat& B) {
  Mat C(A.r, B.c);
  for (long i = 0; i < A.r; ++i)
    for (long q = 0; q < A.c; ++q) {
      const double a = A.at(i, q);
      for (long j = 0; j < B.c; ++j) C.at(i, j) += a * B.at(q, j);
    }
  return C;
}

Mat transpose(const Mat& A) {
  Mat T(A.c, A.r);
  for (long i = 0; i < A.r; ++i)
    for (long j = 0; j < A.c; ++j) T.at(j, i) = A.at(i, j);
  return T;
}

Mat cols(const Mat& A, long c0, long n) {
  Mat B(A.r, n);
  for (long i = 0; i < A.r; ++i)
    for (long j = 0; j < n; ++j) B.at(i, j) = A.at(i, c0 + j);
  return B;
}

Mat slice_expert(const double* base, long e, long rows, long cols_) {
  Mat M(rows, cols_);
  std::memcpy(M.v.data(), base + (size_t)(e * rows * cols_), sizeof(double) * rows * cols_);
  return M;
}

// ---------------------------------------------------------- rounding helpers

double to_f32(double a) { return (double)(float)a; }

// float32 -> bfloat16, round to nearest even on the 16 dropped bits [the
// bfloat16 format: float32's sign and exponent, 7 fraction bits].
double to_bf16(double a) {
  float f = (float)a;
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if (std::isnan(f)) {
    u |= 0x00400000u;
  } else {
    const uint32_t lsb = (u >> 16) & 1u;
    u = (u + 0x7FFFu + lsb) & 0xFFFF0000u;
  }
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// ------------------------------------------------------------- MX formats

struct Fmt {
  int emax;        // exponent of the largest binade [OCPMX]
  int min_normal;  // exponent of the smallest normal value
  int mant_bits;
  double max;      // largest magnitude
};
const Fmt kE4M3 = {8, -6, 3, 448.0};
const Fmt kE2M1 = {2, 0, 1, 6.0};
constexpr int kBlock = 32;

// Round a >= 0 to the format's grid, ties to even, saturating. In the binade
// [2^b, 2^(b+1)) the spacing is 2^(b - mant_bits); below the smallest normal
// the spacing of the smallest binade applies (subnormals). Division by a
// power of two is exact, so rounding the quotient to the nearest integer,
// ties to even, is exact round-to-nearest-even.
double grid_round(double a, const Fmt& f) {
  if (a == 0.0) return 0.0;
  int ex;
  std::frexp(a, &ex);  // a = m 2^ex, m in [0.5, 1): floor(log2 a) = ex - 1
  int b = ex - 1;
  if (b < f.min_normal) b = f.min_normal;
  const double q = std::ldexp(1.0, b - f.mant_bits);
  const double r = std::nearbyint(a / q) * q;  // default mode: to nearest, ties to even
  return r < f.max ? r : f.max;
}

// Shared exponent of a finite block: floor(log2 amax) - emax, clamped to
// [-127, 127]; -127 for an all-zero block.
int block_exponent(double amax, const Fmt& f) {
  if (amax == 0.0) return -127;
  int ex;
  std::frexp(amax, &ex);
  int e = ex - 1 - f.emax;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Element bits of a grid magnitude r (E4M3: exponent bias 7; E2M1: bias 1).
uint8_t encode_magnitude(double r, const Fmt& f) {
  if (r == 0.0) return 0;
  const int bias = f.min_normal < 0 ? 1 - f.min_normal : 1;  // E4M3 7, E2M1 1
  int ex;
  std::frexp(r, &ex);
  const int b = ex - 1;
  if (b < f.min_normal)  // subnormal: a multiple of the smallest spacing
    return (uint8_t)std::lrint(std::ldexp(r, f.mant_bits - f.min_normal));
  const long mant = std::lrint((std::ldexp(r, -b) - 1.0) * (1 << f.mant_bits));
  return (uint8_t)(((b + bias) << f.mant_bits) | mant);
}

// One block of 32 values (v[i * stride]): its scale byte and element codes
// (sign bit above the magnitude bits), and/or the values it carries
// sign(v) RNE(|v| 2^-e) 2^e (NaN for a block holding Inf or NaN).
void mx_block(const double* v, long stride, const Fmt& f, uint8_t* codes, long code_stride,
              uint8_t* scale, double* out, long out_stride) {
  double amax = 0.0;
  bool finite = true;
  for (int i = 0; i < kBlock; ++i) {
    const double a = std::fabs(v[i * stride]);
    if (!std::isfinite(a)) finite = false;
    else if (a > amax) amax = a;
  }
  const int sign_shift = f.mant_bits == 3 ? 7 : 3;
  if (!finite) {
    if (scale) *scale = 0xFF;
    for (int i = 0; i < kBlock; ++i) {
      if (codes) codes[i * code_stride] = f.mant_bits == 3 ? 0x7F : 0;
      if (out) out[i * out_stride] = NAN;
    }
    return;
  }
  const int e = block_exponent(amax, f);
  if (scale) *scale = (uint8_t)(e + 127);
  for (int i = 0; i < kBlock; ++i) {
    const double x = v[i * stride];
    const double r = grid_round(std::ldexp(std::fabs(x), -e), f);
    if (codes)
      codes[i * code_stride] =
          (uint8_t)(encode_magnitude(r, f) | ((std::signbit(x) ? 1 : 0) << sign_shift));
    if (out) out[i * out_stride] = std::copysign(std::ldexp(r, e), x);
  }
}

// The values an MX operand carries, blocks of 32 along `axis` (the axis
// length must be a multiple of 32).
Mat qdq(const Mat& a, int axis, const Fmt& f) {
  Mat o(a.r, a.c);
  if (axis == 1) {
    for (long i = 0; i < a.r; ++i)
      for (long b = 0; b < a.c / kBlock; ++b)
        mx_block(&a.v[(size_t)(i * a.c + b * kBlock)], 1, f, nullptr, 0, nullptr,
                 &o.v[(size_t)(i * a.c + b * kBlock)], 1);
  } else {
    for (long b = 0; b < a.r / kBlock; ++b)
      for (long j = 0; j < a.c; ++j)
        mx_block(&a.v[(size_t)(b * kBlock * a.c + j)], a.c, f, nullptr, 0, nullptr,
                 &o.v[(size_t)(b * kBlock * a.c + j)], a.c);
  }
  return o;
}

Mat pad_rows(const Mat& a) {
  Mat p((a.r + kBlock - 1) / kBlock * kBlock, a.c);
  std::copy(a.v.begin(), a.v.end(), p.v.begin());
  return p;
}

Mat first_rows(const Mat& a, long n) {
  Mat o(n, a.c);
  std::copy(a.v.begin(), a.v.begin() + n * a.c, o.v.begin());
  return o;
}

// Column-wise MXFP8 of one expert group's rows: blocks of 32 group rows, the
// group padded with zero rows.
Mat qdq_cols_in_group(const Mat& a) { return first_rows(qdq(pad_rows(a), 0, kE4M3), a.r); }

// The MXFP4-activation chain of a wgrad operand [MXFP4-HOPPER].
Mat act4_cols_in_group(const Mat& a) {
  Mat p = pad_rows(a);
  Mat row8 = qdq(p, 1, kE4M3);
  Mat row4 = qdq(row8, 1, kE2M1);
  Mat col4 = qdq(row4, 0, kE2M1);
  return first_rows(col4, a.r);
}

Mat map(const Mat& a, double (*fn)(double)) {
  Mat o(a.r, a.c);
  for (size_t i = 0; i < a.v.size(); ++i) o.v[i] = fn(a.v[i]);
  return o;
}

// ------------------------------------------------------------- routing

// [MOEBIO Router; EMT §Challenge 1 routing weights]: the k best experts of
// one token (strictly greater wins, so ties keep the lower index), and the
// softmax over their logits.
void route_token(const double* lg, int E, int k, int32_t* idx, double* w) {
  std::vector<char> taken((size_t)E, 0);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e)
      if (!taken[(size_t)e] && (best < 0 || lg[e] > lg[best])) best = e;
    taken[(size_t)best] = 1;
    idx[j] = best;
  }
  double sum = 0.0;
  for (int j = 0; j < k; ++j) {
    w[j] = std::exp(lg[idx[j]] - lg[idx[0]]);
    sum += w[j];
  }
  for (int j = 0; j < k; ++j) w[j] /= sum;
}

double sigmoid(double z) { return 1.0 / (1.0 + std::exp(-z)); }
double silu(double z) { return z * sigmoid(z); }
double dsilu(double z) {
  const double s = sigmoid(z);
  return s * (1.0 + z * (1.0 - s));
}

enum Mode { kBF16 = 0, kMXFP8 = 1, kMXFP8Act4 = 2 };

struct ExpertOut {
  Mat y2, dxp, dW1, dW2;
  std::vector<double> dp;
};

// One expert on its n routed rows [EMT §Challenge 1 and §Challenge 3]:
// forward [g | u] = x W1, h = silu(g) u p, y2 = h W2; backward
// dH = dY2 W2^T, dA = dH p, dp = sum_f dH silu(g) u, dg = dA u silu'(g),
// du = dA silu(g), dY1 = [dg | du], dW2 = H^T dY2, dX = dY1 W1^T,
// dW1 = X^T dY1, with the MXFP8 operand values where the mode says so.
ExpertOut expert(const Mat& xe, const std::vector<double>& p, const Mat& W1e, const Mat& W2e,
                 const Mat& dy2, Mode mode, bool save_bf16) {
  const long n = xe.r, F = W2e.r;
  const bool mx = mode != kBF16;
  // forward
  const Mat xin = mx ? qdq(xe, 1, kE4M3) : xe;
  const Mat w1f = mx ? qdq(W1e, 0, kE4M3) : W1e;  // blocks along H
  const Mat y1 = matmul(xin, w1f);
  Mat g = cols(y1, 0, F), u = cols(y1, F, F), h(n, F);
  for (long i = 0; i < n; ++i)
    for (long f = 0; f < F; ++f) h.at(i, f) = silu(g.at(i, f)) * u.at(i, f) * p[(size_t)i];
  const Mat h32 = map(h, to_f32);
  const Mat hin = mx ? qdq(h32, 1, kE4M3) : h;
  const Mat w2f = mx ? qdq(W2e, 0, kE4M3) : W2e;  // blocks along F
  ExpertOut o;
  o.y2 = matmul(hin, w2f);
  // backward
  if (save_bf16) {
    g = map(g, to_bf16);
    u = map(u, to_bf16);
  }
  const Mat dy2_row = mx ? qdq(dy2, 1, kE4M3) : dy2;
  const Mat w2d = mx ? qdq(W2e, 1, kE4M3) : W2e;  // blocks along H
  const Mat dh = matmul(dy2_row, transpose(w2d));
  Mat dy1(n, 2 * F);
  o.dp.assign((size_t)n, 0.0);
  for (long i = 0; i < n; ++i)
    for (long f = 0; f < F; ++f) {
      const double gv = g.at(i, f), uv = u.at(i, f), d = dh.at(i, f);
      const double dA = d * p[(size_t)i];
      o.dp[(size_t)i] += d * (silu(gv) * uv);
      dy1.at(i, f) = dA * uv * dsilu(gv);
      dy1.at(i, F + f) = dA * silu(gv);
    }
  Mat dy1_row = dy1, dy1_col = dy1, h_col = h, dy2_col = dy2, x_col = xe;
  if (mx) {
    const Mat dy1_32 = map(dy1, to_f32);
    dy1_row = qdq(dy1_32, 1, kE4M3);
    dy1_col = qdq_cols_in_group(dy1_32);
    dy2_col = qdq_cols_in_group(dy2);
    if (mode == kMXFP8Act4) {
      h_col = act4_cols_in_group(h32);
      x_col = act4_cols_in_group(xe);
    } else {
      h_col = qdq_cols_in_group(h32);
      x_col = qdq_cols_in_group(xe);
    }
  }
  const Mat w1d = mx ? qdq(W1e, 1, kE4M3) : W1e;  // blocks along 2F
  o.dW2 = matmul(transpose(h_col), dy2_col);
  o.dxp = matmul(dy1_row, transpose(w1d));
  o.dW1 = matmul(transpose(x_col), dy1_col);
  return o;
}

}  // namespace

extern "C" {

// Top-k routing of T tokens over E experts: idx [T, k] (best first), w [T, k].
// Returns 0, or -1 for bad sizes.
int moe_oracle_route(const double* logits, int T, int E, int k, int32_t* idx, double* w) {
  if (T < 0 || E < 1 || k < 1 || k > E) return -1;
  for (int t = 0; t < T; ++t)
    route_token(logits + (size_t)t * E, E, k, idx + (size_t)t * k, w + (size_t)t * k);
  return 0;
}

// dlogits [T, E] from dp = dL/dw [T, k]: dl[t, idx_j] = w_j (dp_j - sum_i w_i dp_i),
// zero for experts that were not selected.
int moe_oracle_route_backward(const double* dp, const double* w, const int32_t* idx, int T,
                              int E, int k, double* dlogits) {
  if (T < 0 || E < 1 || k < 1 || k > E) return -1;
  for (int t = 0; t < T; ++t) {
    double s = 0.0;
    for (int j = 0; j < k; ++j) s += w[(size_t)t * k + j] * dp[(size_t)t * k + j];
    double* row = dlogits + (size_t)t * E;
    for (int e = 0; e < E; ++e) row[e] = 0.0;
    for (int j = 0; j < k; ++j)
      row[idx[(size_t)t * k + j]] = w[(size_t)t * k + j] * (dp[(size_t)t * k + j] - s);
  }
  return 0;
}

// Expert-sort plan of the T*k routed rows [EMT §Challenge 1 split sizes]:
// counts [E]; offsets [E+1] = exclusive prefix sum of counts rounded up to
// `align`; dest [T*k] = permuted row of flat index t*k+j (a group keeps flat
// order); src [src_cap] = flat index held by each permuted row, -1 for
// padding rows and rows past offsets[E]. Returns 0, or -1 for bad arguments.
int moe_oracle_permute_plan(const int32_t* idx, int T, int k, int E, int align, int32_t* counts,
                            int32_t* offsets, int32_t* dest, int32_t* src, long long src_cap) {
  if (T < 0 || k < 1 || E < 1 || align < 1) return -1;
  const long n = (long)T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (long f = 0; f < n; ++f) {
    if (idx[f] < 0 || idx[f] >= E) return -1;
    ++counts[idx[f]];
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e)
    offsets[e + 1] = offsets[e] + (counts[e] + align - 1) / align * align;
  if (offsets[E] > src_cap) return -1;
  std::vector<int32_t> next(offsets, offsets + E);
  for (long long r = 0; r < src_cap; ++r) src[r] = -1;
  for (long f = 0; f < n; ++f) {
    dest[f] = next[(size_t)idx[f]]++;
    src[dest[f]] = (int32_t)f;
  }
  return 0;
}

// xp [rows, H] = zeros, then xp[dest[t*k+j]] = x[t].
int moe_oracle_permute(const double* x, const int32_t* dest, int T, int H, int k, long long rows,
                       double* xp) {
  for (long long i = 0; i < rows * H; ++i) xp[i] = 0.0;
  for (long f = 0; f < (long)T * k; ++f) {
    if (dest[f] < 0 || dest[f] >= rows) return -1;
    std::memcpy(xp + (size_t)dest[f] * H, x + (size_t)(f / k) * H, sizeof(double) * H);
  }
  return 0;
}

// out[t] = sum over j of w[t, j] y[dest[t*k+j]] (w = 1 where w is null),
// slots added in ascending j.
int moe_oracle_unpermute(const double* y, const int32_t* dest, const double* w, int T, int H,
                         int k, double* out) {
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h) {
      double s = 0.0;
      for (int j = 0; j < k; ++j) {
        const double wj = w ? w[(size_t)t * k + j] : 1.0;
        s += wj * y[(size_t)dest[(size_t)t * k + j] * H + h];
      }
      out[(size_t)t * H + h] = s;
    }
  return 0;
}

// MX quantisation of a [rows, cols] matrix with 32-blocks along `axis`
// (0: down the rows, 1: along the columns): codes [rows, cols] (E4M3 bytes
// for fmt 8; E2M1 codes 0..15, one per byte, for fmt 4) and scales (E8M0
// bytes: [rows, cols/32] for axis 1, [rows/32, cols] for axis 0).
int moe_oracle_mx_quantize(const double* a, long long rows, long long cols, int axis, int fmt,
                           uint8_t* codes, uint8_t* scales) {
  const Fmt& f = fmt == 4 ? kE2M1 : kE4M3;
  if ((fmt != 4 && fmt != 8) || (axis != 0 && axis != 1)) return -1;
  if (axis == 1) {
    if (cols % kBlock) return -1;
    for (long long i = 0; i < rows; ++i)
      for (long long b = 0; b < cols / kBlock; ++b)
        mx_block(a + i * cols + b * kBlock, 1, f, codes + i * cols + b * kBlock, 1,
                 scales + i * (cols / kBlock) + b, nullptr, 0);
  } else {
    if (rows % kBlock) return -1;
    for (long long b = 0; b < rows / kBlock; ++b)
      for (long long j = 0; j < cols; ++j)
        mx_block(a + b * kBlock * cols + j, cols, f, codes + b * kBlock * cols + j, cols,
                 scales + b * cols + j, nullptr, 0);
  }
  return 0;
}

// Router projection [MOEBIO Router: a score for every expert per token]:
// logits [T, E] = x [T, H] Wr [H, E], then top-k routing (idx, w [T, k]), and
// the load-balancing statistics [MOEBIO "Engineering Challenges of Efficient
// Training": an auxiliary loss against uneven expert load] in aux [1 + 2E]:
// aux[0] = L = E sum_e f_e P_e, aux[1 + e] = f_e = the fraction of the T*k
// routed pairs that go to expert e, aux[1 + E + e] = P_e = the mean over
// tokens of the softmax probability of expert e over all E logits.
int moe_oracle_router_forward(const double* x, const double* Wr, int T, int H, int E, int k,
                              double* logits, int32_t* idx, double* w, double* aux) {
  if (T < 1 || H < 1 || E < 1 || k < 1 || k > E) return -1;
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      for (int h = 0; h < H; ++h) s += x[(size_t)t * H + h] * Wr[(size_t)h * E + e];
      logits[(size_t)t * E + e] = s;
    }
  moe_oracle_route(logits, T, E, k, idx, w);
  double* f = aux + 1;
  double* P = aux + 1 + E;
  for (int e = 0; e < E; ++e) f[e] = P[e] = 0.0;
  for (long i = 0; i < (long)T * k; ++i) f[idx[i]] += 1.0;
  for (int e = 0; e < E; ++e) f[e] /= (double)T * k;
  std::vector<double> s((size_t)E);
  for (int t = 0; t < T; ++t) {
    const double* l = logits + (size_t)t * E;
    double m = l[0], z = 0.0;
    for (int e = 1; e < E; ++e) m = l[e] > m ? l[e] : m;
    for (int e = 0; e < E; ++e) z += (s[(size_t)e] = std::exp(l[e] - m));
    for (int e = 0; e < E; ++e) P[e] += s[(size_t)e] / z / T;
  }
  aux[0] = 0.0;
  for (int e = 0; e < E; ++e) aux[0] += f[e] * P[e];
  aux[0] *= E;
  return 0;
}

// Router backward: dlogits = dlogits_route + coeff * dL/dlogits, where
// dL/dl[t, e] = (E / T) s[t, e] (f_e - sum_i f_i s[t, i]) with the routed
// fractions f held fixed (the selection has no gradient) and s the softmax
// over all E logits; then dx = dlogits Wr^T and dWr = x^T dlogits.
int moe_oracle_router_backward(const double* x, const double* Wr, const double* logits,
                               const double* f, const double* dlogits_route, double coeff, int T,
                               int H, int E, double* dlogits, double* dx, double* dWr) {
  if (T < 1 || H < 1 || E < 1) return -1;
  std::vector<double> s((size_t)E);
  for (int t = 0; t < T; ++t) {
    const double* l = logits + (size_t)t * E;
    double m = l[0], z = 0.0, c = 0.0;
    for (int e = 1; e < E; ++e) m = l[e] > m ? l[e] : m;
    for (int e = 0; e < E; ++e) z += (s[(size_t)e] = std::exp(l[e] - m));
    for (int e = 0; e < E; ++e) {
      s[(size_t)e] /= z;
      c += f[e] * s[(size_t)e];
    }
    for (int e = 0; e < E; ++e)
      dlogits[(size_t)t * E + e] = dlogits_route[(size_t)t * E + e] +
                                   coeff * ((double)E / T) * s[(size_t)e] * (f[e] - c);
  }
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int e = 0; e < E; ++e) acc += dlogits[(size_t)t * E + e] * Wr[(size_t)h * E + e];
      dx[(size_t)t * H + h] = acc;
    }
  // dWr[h, e] summed over tokens in ascending order
  for (long i = 0; i < (long)H * E; ++i) dWr[i] = 0.0;
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h)
      for (int e = 0; e < E; ++e)
        dWr[(size_t)h * E + e] += x[(size_t)t * H + h] * dlogits[(size_t)t * E + e];
  return 0;
}

// The whole layer, forward and backward, as the per-expert loop of
// [EMT §Challenge 1], for the loss L = sum(out * dout).
// mode: 0 BF16 (exact products), 1 MXFP8, 2 MXFP8 with MXFP4-carried
// activations; save_bf16: the SwiGLU backward reads gate/up in bf16.
// Outputs: out, dX [T, H]; dW1 [E, H, 2F]; dW2 [E, F, H]; dlogits [T, E];
// dp [T, k]; idx, w [T, k]. Returns 0, or -1 for bad sizes (the MXFP8 modes
// need H and F to be multiples of 32).
int moe_oracle_layer(const double* x, const double* logits, const double* W1, const double* W2,
                     const double* dout, int T, int H, int F, int E, int k, int mode,
                     int save_bf16, double* out, double* dX, double* dW1, double* dW2,
                     double* dlogits, double* dp, int32_t* idx, double* w) {
  if (T < 0 || H < 1 || F < 1 || E < 1 || k < 1 || k > E || mode < 0 || mode > 2) return -1;
  if (mode != kBF16 && (H % kBlock || F % kBlock)) return -1;
  moe_oracle_route(logits, T, E, k, idx, w);
  for (long i = 0; i < (long)T * H; ++i) out[i] = dX[i] = 0.0;
  for (long e = 0; e < E; ++e) {
    std::vector<long> tok, slot;
    for (long t = 0; t < T; ++t)
      for (long j = 0; j < k; ++j)
        if (idx[t * k + j] == e) {
          tok.push_back(t);
          slot.push_back(j);
        }
    const long n = (long)tok.size();
    Mat xe(n, H), dy2(n, H);
    std::vector<double> p((size_t)n);
    for (long i = 0; i < n; ++i) {
      std::memcpy(&xe.v[(size_t)(i * H)], x + (size_t)tok[(size_t)i] * H, sizeof(double) * H);
      std::memcpy(&dy2.v[(size_t)(i * H)], dout + (size_t)tok[(size_t)i] * H,
                  sizeof(double) * H);
      p[(size_t)i] = w[tok[(size_t)i] * k + slot[(size_t)i]];
    }
    const ExpertOut o = expert(xe, p, slice_expert(W1, e, H, 2L * F), slice_expert(W2, e, F, H),
                               dy2, (Mode)mode, save_bf16 != 0);
    for (long i = 0; i < n; ++i) {
      const long t = tok[(size_t)i];
      for (long c = 0; c < H; ++c) {
        out[t * H + c] += o.y2.at(i, c);
        dX[t * H + c] += o.dxp.at(i, c);
      }
      dp[t * k + slot[(size_t)i]] = o.dp[(size_t)i];
    }
    std::memcpy(dW1 + (size_t)(e * H * 2L * F), o.dW1.v.data(), sizeof(double) * H * 2L * F);
    std::memcpy(dW2 + (size_t)(e * F * H), o.dW2.v.data(), sizeof(double) * F * H);
  }
  return moe_oracle_route_backward(dp, w, idx, T, E, k, dlogits);
}

}  // extern "C"
