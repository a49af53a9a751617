// The router in front of the expert layer: the projection of the hidden
// states to per-expert logits, and the auxiliary load-balancing loss.
//
// "How MoE Architecture Cuts Costs and Boosts Efficiency: Efficient Training
// of Biological Foundation Models": the Router paragraph (a score for every
// expert per token, of which the top K are kept) and "Engineering Challenges
// of Efficient Training" (an auxiliary load-balancing loss added to the
// training objective penalises uneven expert load).
//
//   logits[t, e] = sum_h x[t, h] * Wr[h, e]          (x, Wr bf16; fp32 accumulation)
//   s[t, :]      = softmax over all E of logits[t, :]
//   f_e          = (# routed (t, j) with idx[t, j] = e) / (T * k)
//   P_e          = (1 / T) * sum_t s[t, e]
//   L_aux        = E * sum_e f_e * P_e
//   dL_aux / dlogits[t, e] = (E / T) * s[t, e] * (f_e - sum_i f_i * s[t, i])
// (f is piecewise constant: the top-k selection carries no gradient.)
//
// All kernels are memory-bound. The three contractions run on warp-level
// bf16 MMAs (see "tensor-core tiles" below), the statistics in SIMT code;
// every reduction is done in a fixed order (per-warp or per-block partials,
// then one ordered pass), so results do not depend on scheduling.
#include "common.cuh"

namespace moe {
namespace router {

constexpr int kMaxE = 256;

// ------------------------------------------------------------ tensor-core tiles
// The three contractions (x Wr, dl Wr^T, x^T dl) are memory-bound with N = E
// small, so they use warp-level bf16 MMAs (m16n8k16, fp32 accumulation): the
// arithmetic then costs next to nothing and each kernel streams its operands
// once. Products of two bf16 are exact in fp32. The fp32 logit gradient dl
// enters as two bf16 terms, hi = bf16(dl) and lo = bf16(dl - hi), which carry
// about 16 significant bits; the dropped remainder is below 2^-16 |dl|.
//
// Operand registers follow the m16n8k16 fragment layout (lane = 4 g + c):
//   A (16 x 16, row-major): a0 = A[g][2c..2c+1], a1 = A[g+8][2c..], a2 = A[g][2c+8..], a3 = A[g+8][2c+8..]
//   B (16 x 8, k-major):    b0 = B[2c..2c+1][g], b1 = B[2c+8..2c+9][g]
//   C (16 x 8):             c0, c1 = C[g][2c..2c+1], c2, c3 = C[g+8][2c..2c+1]
// A sum over k does not depend on the order of its terms, and the rows of A
// and the columns of B may be given any labels, so each kernel assigns
// hidden columns and tokens to k, m and n so that every lane loads 16
// contiguous bytes; the assignment is stated at each kernel.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// (v0, v1) -> hi = bf16 pair, lo = bf16 pair of the remainders.
__device__ __forceinline__ void split_bf16(float v0, float v1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = pack_bf16(v0 - __low2float(h), v1 - __high2float(h));
}

__device__ __forceinline__ uint4 ld_v4(const __nv_bfloat16* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// 16-byte cp.async into shared memory (a shared-window address), zero-filled
// when !valid. Each lane later reads back only what it copied itself, so a
// per-thread cp.async.wait_group is the only synchronisation needed.
__device__ __forceinline__ void cp16s(uint32_t d, const void* gmem, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d),
               "l"(reinterpret_cast<uint64_t>(gmem)), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ------------------------------------------------------------ projection
// WrT[e][h] = Wr[h][e] for e < E, 0 for E <= e < 8 * ceil(E / 8).
__global__ void router_wt_kernel(const __nv_bfloat16* __restrict__ wr, int H, int E, int Ep,
                                 __nv_bfloat16* __restrict__ wt) {
  const long long n = (long long)Ep * H;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int e = (int)(i / H);
    const long long h = i - (long long)e * H;
    wt[i] = e < E ? wr[h * E + e] : __float2bfloat16_rn(0.f);
  }
}

// logits[t, e] = sum_h x[t, h] Wr[h, e]. CTA: one tile of 16 tokens and NTG
// n-tiles (blockIdx.y picks the group); warp w takes the 128-column chunks
// w, w + 8, ... of H, and the 8 warp sums are added in warp order through
// shared memory.
// Labels: in chunk h0, lane (g, c) loads x[t0 + g] and x[t0 + g + 8] at
// columns h0 + 32 q + 8 c + (0..7), q = 0..3 (16 bf16 pairs p = 4 q + i), and
// WrT[e] at the same columns; MMA j takes pairs 2 j (k = 2c, 2c+1) and 2 j + 1
// (k = 2c + 8, 2c + 9) of both.
constexpr int kLWarps = 8;
constexpr int kLChunk = 128;

// NTG = n-tiles (8 experts each) per CTA; blockIdx.y picks the group.
template <int NTG>
__global__ void __launch_bounds__(kLWarps * 32, NTG <= 2 ? 4 : 2)
    router_logits_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ wt,
                         int T, int H, int E, float* __restrict__ logits) {
  constexpr int EW = 8 * NTG;  // experts per CTA
  __shared__ float red[kLWarps][16][EW + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const long long t0 = (long long)blockIdx.x * 16;
  const int nt0 = blockIdx.y * NTG;
  const int ntn = min(NTG, (E + 7) / 8 - nt0);
  const long long ta = t0 + g, tb = t0 + g + 8;
  const bool va = ta < T, vb = tb < T;
  float acc[NTG][4];
#pragma unroll
  for (int n = 0; n < NTG; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
  const int nch = (H + kLChunk - 1) / kLChunk;
  for (int ch = warp; ch < nch; ch += kLWarps) {
    const int h0 = ch * kLChunk;
    uint32_t xa[16], xb[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int h = h0 + 32 * q + 8 * c;
      uint4 ua = make_uint4(0, 0, 0, 0), ub = ua;
      if (h < H) {
        if (va) ua = ld_v4(x + ta * H + h);
        if (vb) ub = ld_v4(x + tb * H + h);
      }
      xa[4 * q] = ua.x, xa[4 * q + 1] = ua.y, xa[4 * q + 2] = ua.z, xa[4 * q + 3] = ua.w;
      xb[4 * q] = ub.x, xb[4 * q + 1] = ub.y, xb[4 * q + 2] = ub.z, xb[4 * q + 3] = ub.w;
    }
#pragma unroll
    for (int n = 0; n < NTG; ++n) {
      if (n < ntn) {
        const __nv_bfloat16* wrow = wt + (long long)(8 * (nt0 + n) + g) * H;
        uint32_t wf[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int h = h0 + 32 * q + 8 * c;
          const uint4 u = h < H ? ld_v4(wrow + h) : make_uint4(0, 0, 0, 0);
          wf[4 * q] = u.x, wf[4 * q + 1] = u.y, wf[4 * q + 2] = u.z, wf[4 * q + 3] = u.w;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          mma_bf16(acc[n], xa[2 * j], xb[2 * j], xa[2 * j + 1], xb[2 * j + 1], wf[2 * j],
                   wf[2 * j + 1]);
      }
    }
  }
#pragma unroll
  for (int n = 0; n < NTG; ++n) {
    if (n < ntn) {
      red[warp][g][8 * n + 2 * c] = acc[n][0];
      red[warp][g][8 * n + 2 * c + 1] = acc[n][1];
      red[warp][g + 8][8 * n + 2 * c] = acc[n][2];
      red[warp][g + 8][8 * n + 2 * c + 1] = acc[n][3];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 16 * EW; i += kLWarps * 32) {
    const int r = i / EW, el = i % EW, e = 8 * nt0 + el;
    if (el < 8 * ntn && e < E && t0 + r < T) {
      float s = red[0][r][el];
#pragma unroll
      for (int w = 1; w < kLWarps; ++w) s += red[w][r][el];
      logits[(t0 + r) * E + e] = s;
    }
  }
}

// ------------------------------------------------------------ aux statistics
// One warp per token: softmax over E (lane l holds e = l + 32 s), summed per
// expert into this warp's row of shared memory (tokens in increasing order);
// the CTA then adds its 8 warp rows in order and writes one partial row.
constexpr int kAThreads = 256;
constexpr int kATokens = 32;  // tokens per CTA

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// softmax of one token's logits across the warp; p[s] for e = lane + 32 s.
__device__ __forceinline__ void warp_softmax(const float* row, int E, int lane,
                                             float (&p)[kMaxE / 32]) {
  float m = -INFINITY;
#pragma unroll
  for (int s = 0; s < kMaxE / 32; ++s) {
    const int e = lane + 32 * s;
    p[s] = e < E ? row[e] : -INFINITY;
    m = fmaxf(m, p[s]);
  }
  m = warp_max(m);
  float z = 0.f;
#pragma unroll
  for (int s = 0; s < kMaxE / 32; ++s) {
    const int e = lane + 32 * s;
    p[s] = e < E ? expf(p[s] - m) : 0.f;
    z += p[s];
  }
  const float inv = 1.f / warp_sum(z);
#pragma unroll
  for (int s = 0; s < kMaxE / 32; ++s) p[s] *= inv;
}

__global__ void __launch_bounds__(kAThreads)
    router_aux_partial_kernel(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                              int T, int E, int k, float* __restrict__ part_s,
                              int32_t* __restrict__ part_c) {
  __shared__ float s_acc[kAThreads / 32][kMaxE];
  __shared__ int32_t c_acc[kAThreads / 32][kMaxE];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = lane; e < kMaxE; e += 32) {
    s_acc[warp][e] = 0.f;
    c_acc[warp][e] = 0;
  }
  __syncwarp();
  const long long t0 = (long long)blockIdx.x * kATokens;
  for (int i = warp; i < kATokens; i += kAThreads / 32) {
    const long long t = t0 + i;
    if (t >= T) break;
    float p[kMaxE / 32];
    warp_softmax(logits + t * E, E, lane, p);
#pragma unroll
    for (int s = 0; s < kMaxE / 32; ++s) {
      const int e = lane + 32 * s;
      if (e < E) s_acc[warp][e] += p[s];
    }
    if (lane < k) {
      const int e = idx[t * k + lane];
      if (e >= 0 && e < E) atomicAdd(&c_acc[warp][e], 1);  // integer: order-free
    }
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kAThreads) {
    float s = 0.f;
    int32_t c = 0;
    for (int w = 0; w < kAThreads / 32; ++w) {
      s += s_acc[w][e];
      c += c_acc[w][e];
    }
    part_s[(long long)blockIdx.x * E + e] = s;
    part_c[(long long)blockIdx.x * E + e] = c;
  }
}

// One block of 8 warps: for each expert, lane l adds the partial rows
// l, l + 32, ... in order and the warp combines the 32 lane sums with a fixed
// butterfly, so the result does not depend on scheduling; then the loss.
// aux = [loss, f_0..f_{E-1}, P_0..P_{E-1}].
__global__ void __launch_bounds__(256)
    router_aux_final_kernel(const float* __restrict__ part_s, const int32_t* __restrict__ part_c,
                            int nblocks, int T, int E, int k, float* __restrict__ aux) {
  __shared__ float prod[kMaxE];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = warp; e < E; e += 8) {
    float s = 0.f;
    long long c = 0;
#pragma unroll 4
    for (int b = lane; b < nblocks; b += 32) {
      s += part_s[(long long)b * E + e];
      c += part_c[(long long)b * E + e];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s += __shfl_xor_sync(0xffffffffu, s, o);
      c += __shfl_xor_sync(0xffffffffu, c, o);
    }
    const float f = (float)((double)c / ((double)T * k));
    const float P = s / (float)T;
    if (lane == 0) {
      aux[1 + e] = f;
      aux[1 + E + e] = P;
      prod[e] = f * P;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float sum = 0.f;
    for (int i = 0; i < E; ++i) sum += prod[i];
    aux[0] = (float)E * sum;
  }
}

// ------------------------------------------------------------ backward
// dl[t, e] = dl_route[t, e] + coeff * (E / T) * s[t, e] * (f_e - sum_i f_i s[t, i]).
__global__ void __launch_bounds__(256)
    router_aux_backward_kernel(const float* __restrict__ logits, const float* __restrict__ aux,
                               const float* __restrict__ dl_route, float coeff, int T, int E,
                               float* __restrict__ dl) {
  const int lane = threadIdx.x & 31;
  const float* f = aux + 1;
  for (long long t = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); t < T;
       t += (long long)gridDim.x * 8) {
    float p[kMaxE / 32];
    warp_softmax(logits + t * E, E, lane, p);
    float c = 0.f;
#pragma unroll
    for (int s = 0; s < kMaxE / 32; ++s) {
      const int e = lane + 32 * s;
      if (e < E) c = fmaf(f[e], p[s], c);
    }
    c = warp_sum(c);
    const float scale = coeff * (float)E / (float)T;
#pragma unroll
    for (int s = 0; s < kMaxE / 32; ++s) {
      const int e = lane + 32 * s;
      if (e < E) {
        const float g = scale * p[s] * (f[e] - c);
        dl[t * E + e] = (dl_route ? dl_route[t * E + e] : 0.f) + g;
      }
    }
  }
}

// dx[t, h] = dx_in[t, h] + sum_e dl[t, e] Wr[h, e]: C = A B with A = dl (16
// tokens x 16 experts per k step, hi and lo terms), B[e][h] = Wr[h, e] and
// the accumulator started from dx_in. Warp: one block of 32 columns hb (four
// n-tiles), token tiles [tile0, tile1). Labels: column n = 2c + (0, 1) of
// n-tile j is hidden column hb + 8c + 2j + (0, 1), so that lane (g, c) holds
// the 8 contiguous columns hb + 8c + (0..7) of rows t0 + g and t0 + g + 8
// (16-byte loads of dx_in and stores of dx); B column g of n-tile j is then
// hb + 8 (g >> 1) + 2j + (g & 1).
__device__ __forceinline__ float dl_at(const float* dl, long long t, int e, long long T, int E) {
  return (t < T && e < E) ? __ldg(dl + t * E + e) : 0.f;
}
__device__ __forceinline__ uint32_t wr_pair(const __nv_bfloat16* wr, int h, int e, int E) {
  const unsigned short* w = reinterpret_cast<const unsigned short*>(wr) + (long long)h * E;
  const uint32_t lo = e < E ? w[e] : 0u, hi = e + 1 < E ? w[e + 1] : 0u;
  return lo | (hi << 16);
}

constexpr int kDXStages = 4;  // dx_in tiles in flight per warp (cp.async ring)

__global__ void __launch_bounds__(256, 3)
    router_dx_kernel(const float* __restrict__ dl, const __nv_bfloat16* __restrict__ wr,
                     const __nv_bfloat16* __restrict__ dx_in, int T, int H, int E,
                     int tiles_per_cta, __nv_bfloat16* __restrict__ dx_out) {
  __shared__ uint4 ring[8][kDXStages][2][32];  // [warp][slot][row g / g + 8][lane]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int hb = (blockIdx.x * 8 + warp) * 32;
  if (hb >= H) return;
  const long long tile0 = (long long)blockIdx.y * tiles_per_cta;
  const long long tile1 = min((tile0 + tiles_per_cta), ((long long)T + 15) / 16);
  const int ks_n = (E + 15) / 16;
  // B fragments of the first k step stay in registers (all of them when E <= 16)
  uint32_t b0[4], b1[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int h = hb + 8 * (g >> 1) + 2 * j + (g & 1);
    b0[j] = wr_pair(wr, h, 2 * c, E);
    b1[j] = wr_pair(wr, h, 2 * c + 8, E);
  }
  // dx_in rows g and g + 8 of a tile, copied by this lane into ring slot s
  // Cursors (one pointer step per tile): xi at dx_in row 16 tile + g and
  // column hb + 8c of the next tile to copy; dli at dl row 16 tile + g,
  // expert 2c, of the next tile to load.
  const long long row0 = tile0 * 16 + g;
  const __nv_bfloat16* xi = dx_in ? dx_in + row0 * H + hb + 8 * c : nullptr;
  const float* dli = dl + row0 * E + 2 * c;
  const long long xstep = 16LL * H;
  const uint32_t ring_lane = static_cast<uint32_t>(__cvta_generic_to_shared(&ring[warp][0][0][lane]));
  const bool e0 = 2 * c < E, e1 = 2 * c + 1 < E, e8 = 2 * c + 8 < E, e9 = 2 * c + 9 < E;
  long long ti = tile0, tl = tile0;  // tile of the next copy / dl load
  auto issue = [&](int s) {
    if (xi && ti < tile1) {
      const long long ta = ti * 16 + g;
      const uint32_t d = ring_lane + s * (2 * 32 * 16);
      cp16s(d, ta < T ? xi : dx_in, ta < T);
      cp16s(d + 512, ta + 8 < T ? xi + 8 * H : dx_in, ta + 8 < T);
      xi += xstep;
    }
    ++ti;
    cp_commit();
  };
  // the first k step's dl values of the next tile (rows g, g + 8; experts
  // 2c, 2c+1, 2c+8, 2c+9)
  auto load_dl = [&](float (&v)[8]) {
    const long long ta = tl * 16 + g;
    const bool ra = tl < tile1 && ta < T, rb = tl < tile1 && ta + 8 < T;
    const float* q = dli;
    v[0] = ra && e0 ? __ldg(q) : 0.f;
    v[1] = ra && e1 ? __ldg(q + 1) : 0.f;
    v[2] = rb && e0 ? __ldg(q + 8 * E) : 0.f;
    v[3] = rb && e1 ? __ldg(q + 8 * E + 1) : 0.f;
    v[4] = ra && e8 ? __ldg(q + 8) : 0.f;
    v[5] = ra && e9 ? __ldg(q + 9) : 0.f;
    v[6] = rb && e8 ? __ldg(q + 8 * E + 8) : 0.f;
    v[7] = rb && e9 ? __ldg(q + 8 * E + 9) : 0.f;
    dli += 16 * E;
    ++tl;
  };
#pragma unroll
  for (int s = 0; s < kDXStages - 1; ++s) issue(s);
  float dv[8];
  load_dl(dv);
  int slot = 0;
  for (long long tile = tile0; tile < tile1; ++tile) {
    issue((slot + kDXStages - 1) % kDXStages);
    float dn[8];
    load_dl(dn);  // next tile's, one step ahead
    cp_wait<kDXStages - 1>();
    const long long ta = tile * 16 + g, tb = ta + 8;
    float acc[4][4];
    {
      uint4 ua = make_uint4(0, 0, 0, 0), ub = ua;
      if (dx_in) {
        ua = ring[warp][slot][0][lane];
        ub = ring[warp][slot][1][lane];
      }
      const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[j][0] = __uint_as_float(wa[j] << 16);
        acc[j][1] = __uint_as_float(wa[j] & 0xFFFF0000u);
        acc[j][2] = __uint_as_float(wb[j] << 16);
        acc[j][3] = __uint_as_float(wb[j] & 0xFFFF0000u);
      }
    }
    for (int ks = 0; ks < ks_n; ++ks) {
      const int e0 = 16 * ks;
      float v[8];
      if (ks == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = dv[i];
      } else {
        v[0] = dl_at(dl, ta, e0 + 2 * c, T, E), v[1] = dl_at(dl, ta, e0 + 2 * c + 1, T, E);
        v[2] = dl_at(dl, tb, e0 + 2 * c, T, E), v[3] = dl_at(dl, tb, e0 + 2 * c + 1, T, E);
        v[4] = dl_at(dl, ta, e0 + 2 * c + 8, T, E), v[5] = dl_at(dl, ta, e0 + 2 * c + 9, T, E);
        v[6] = dl_at(dl, tb, e0 + 2 * c + 8, T, E), v[7] = dl_at(dl, tb, e0 + 2 * c + 9, T, E);
      }
      uint32_t ah[4], al[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) split_bf16(v[2 * i], v[2 * i + 1], ah[i], al[i]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t c0 = b0[j], c1 = b1[j];
        if (ks > 0) {
          const int h = hb + 8 * (g >> 1) + 2 * j + (g & 1);
          c0 = wr_pair(wr, h, e0 + 2 * c, E);
          c1 = wr_pair(wr, h, e0 + 2 * c + 8, E);
        }
        mma_bf16(acc[j], ah[0], ah[1], ah[2], ah[3], c0, c1);
        mma_bf16(acc[j], al[0], al[1], al[2], al[3], c0, c1);
      }
    }
    if (ta < T) {
      uint4 o;
      o.x = pack_bf16(acc[0][0], acc[0][1]);
      o.y = pack_bf16(acc[1][0], acc[1][1]);
      o.z = pack_bf16(acc[2][0], acc[2][1]);
      o.w = pack_bf16(acc[3][0], acc[3][1]);
      *reinterpret_cast<uint4*>(dx_out + ta * H + hb + 8 * c) = o;
    }
    if (tb < T) {
      uint4 o;
      o.x = pack_bf16(acc[0][2], acc[0][3]);
      o.y = pack_bf16(acc[1][2], acc[1][3]);
      o.z = pack_bf16(acc[2][2], acc[2][3]);
      o.w = pack_bf16(acc[3][2], acc[3][3]);
      *reinterpret_cast<uint4*>(dx_out + tb * H + hb + 8 * c) = o;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) dv[i] = dn[i];
    slot = (slot + 1) % kDXStages;
  }
  cp_wait<0>();
}

// Partial dWr over a token slice: part[z, h, e] = sum_{t in slice z} x[t, h] dl[t, e]:
// C = A B with A[h][t] = x[t, h] (M = hidden columns, K = tokens) and B = dl
// (hi and lo terms). CTA: 256 columns and NTG n-tiles (blockIdx.z picks the
// group) over token slice blockIdx.y; warp w owns the 64 columns
// hb = 256 blockIdx.x + 64 (w & 3) (four m-tiles) in half w >> 2 of the slice,
// in k steps of 16, and the two halves are added in order through shared
// memory. (A CTA thus reads 512 contiguous bytes of each x row.) Labels:
// lane (g, c) loads the 8 columns hb + 8g + (0..7) of tokens t0 + 2c,
// t0 + 2c + 1 (and + 8, + 9) and pairs them token-wise; m-tile u row g is
// column hb + 8g + 2u, row g + 8 is hb + 8g + 2u + 1.
constexpr int kWK = 16;
constexpr int kWSliceUnit = 2 * kWK;  // token slices are multiples of 2 halves x 16

constexpr int kWStages = 4;  // k steps of x in flight per warp (cp.async ring)

// shared memory: the x ring [8 warps][kWStages][4 rows][32 lanes] x 16 B, reused
// after the main loop for the warp sums [8 warps][64 columns][8 NTG + 1]
template <int NTG>
constexpr size_t dw_smem_bytes() {
  const size_t ring = (size_t)8 * kWStages * 4 * 32 * 16;
  const size_t red = (size_t)8 * 64 * (8 * NTG + 1) * 4;
  return ring > red ? ring : red;
}

template <int NTG>
__global__ void __launch_bounds__(256, NTG == 1 ? 3 : 2)
    router_dw_partial_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ dl,
                             int T, int H, int E, int slice, float* __restrict__ part) {
  constexpr int EW = 8 * NTG, LD = EW + 1;
  extern __shared__ __align__(16) float dsm[];
  uint4* ring = reinterpret_cast<uint4*>(dsm) + (size_t)(threadIdx.x >> 5) * kWStages * 4 * 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int hb = blockIdx.x * 256 + 64 * (warp & 3);
  const int nt0 = blockIdx.z * NTG;
  const int ntn = min(NTG, (E + 7) / 8 - nt0);
  const long long sb = (long long)blockIdx.y * slice;
  const long long wb = sb + (long long)(warp >> 2) * (slice / 2);
  const long long te = min((long long)T, wb + slice / 2);
  // warps past H (when H % 256 != 0) still take part in the block barriers
  const int nsteps = (hb < H && te > wb) ? (int)((te - wb + kWK - 1) / kWK) : 0;
  // rows t0 + 2c + {0, 1, 8, 9} of k step i, columns hb + 8g .. + 7
  // Cursors (one pointer step per k step): xi at row wb + 2c of the next k
  // step to copy, dli at dl row wb + 2c, expert 8 nt0 + g, of the next k step
  // to load; token tl (relative to wb) is valid while tl < span.
  const int span = nsteps > 0 ? (int)(te - wb) : 0;
  const long long xstep = (long long)kWK * H;
  const __nv_bfloat16* xi = x + (nsteps > 0 ? (wb + 2 * c) * H + hb + 8 * g : 0);
  const float* dli = dl + (nsteps > 0 ? (wb + 2 * c) * E : 0) + 8 * nt0 + g;
  const uint32_t ring_lane = static_cast<uint32_t>(__cvta_generic_to_shared(ring + lane));
  int ii = 0, il = 0;  // k step of the next copy / dl load
  auto issue = [&](int s) {
    const int tl = ii * kWK + 2 * c;
    if (ii < nsteps) {
      const uint32_t d = ring_lane + s * (4 * 32 * 16);
      cp16s(d, tl < span ? xi : x, tl < span);
      cp16s(d + 512, tl + 1 < span ? xi + H : x, tl + 1 < span);
      cp16s(d + 1024, tl + 8 < span ? xi + 8 * H : x, tl + 8 < span);
      cp16s(d + 1536, tl + 9 < span ? xi + 9 * H : x, tl + 9 < span);
      xi += xstep;
    }
    ++ii;
    cp_commit();
  };
  // dl values of the next k step: tokens 2c + {0, 1, 8, 9}, experts 8 (nt0 + n) + g
  auto load_dl = [&](float (&v)[NTG][4]) {
    const int tl = il * kWK + 2 * c;
    const bool on = il < nsteps;
#pragma unroll
    for (int n = 0; n < NTG; ++n) {
      const bool en = on && n < ntn && 8 * (nt0 + n) + g < E;
      const float* q = dli + 8 * n;
      v[n][0] = en && tl < span ? __ldg(q) : 0.f;
      v[n][1] = en && tl + 1 < span ? __ldg(q + E) : 0.f;
      v[n][2] = en && tl + 8 < span ? __ldg(q + 8 * E) : 0.f;
      v[n][3] = en && tl + 9 < span ? __ldg(q + 9 * E) : 0.f;
    }
    if (on) dli += kWK * E;
    ++il;
  };
  float acc[4][NTG][4];
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int n = 0; n < NTG; ++n) acc[u][n][0] = acc[u][n][1] = acc[u][n][2] = acc[u][n][3] = 0.f;
#pragma unroll
  for (int s = 0; s < kWStages - 1; ++s) issue(s);
  // dl values of the next D k steps in registers (dq[d]: step i + d); D = 3
  // for one n-tile, 1 where the accumulators leave no room
  constexpr int D = NTG == 1 ? 3 : 1;
  float dq[D][NTG][4];
#pragma unroll
  for (int d = 0; d < D; ++d) load_dl(dq[d]);
  int slot = 0;
  for (int i = 0; i < nsteps; ++i) {
    issue((slot + kWStages - 1) % kWStages);
    float dn[NTG][4];
    load_dl(dn);
    cp_wait<kWStages - 1>();
    uint32_t P[8], Q[8];
    {
      const uint4* rs = ring + slot * 128 + lane;
      const uint4 r0 = rs[0], r1 = rs[32], r2 = rs[64], r3 = rs[96];
      const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w}, w1[4] = {r1.x, r1.y, r1.z, r1.w};
      const uint32_t w2[4] = {r2.x, r2.y, r2.z, r2.w}, w3[4] = {r3.x, r3.y, r3.z, r3.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        P[2 * q] = __byte_perm(w0[q], w1[q], 0x5410);
        P[2 * q + 1] = __byte_perm(w0[q], w1[q], 0x7632);
        Q[2 * q] = __byte_perm(w2[q], w3[q], 0x5410);
        Q[2 * q + 1] = __byte_perm(w2[q], w3[q], 0x7632);
      }
    }
#pragma unroll
    for (int n = 0; n < NTG; ++n) {
      uint32_t bh0, bl0, bh1, bl1;
      split_bf16(dq[0][n][0], dq[0][n][1], bh0, bl0);
      split_bf16(dq[0][n][2], dq[0][n][3], bh1, bl1);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        mma_bf16(acc[u][n], P[2 * u], P[2 * u + 1], Q[2 * u], Q[2 * u + 1], bh0, bh1);
        mma_bf16(acc[u][n], P[2 * u], P[2 * u + 1], Q[2 * u], Q[2 * u + 1], bl0, bl1);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int d = 0; d + 1 < D; ++d) dq[d][n][q] = dq[d + 1][n][q];
        dq[D - 1][n][q] = dn[n][q];
      }
    }
    slot = (slot + 1) % kWStages;
  }
  cp_wait<0>();
  __syncthreads();  // the ring is reused for the warp sums
  float* red = dsm + warp * 64 * LD;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int hl = 8 * g + 2 * u;
#pragma unroll
    for (int n = 0; n < NTG; ++n) {
      const int el = 8 * n + 2 * c;
      red[hl * LD + el] = acc[u][n][0];
      red[hl * LD + el + 1] = acc[u][n][1];
      red[(hl + 1) * LD + el] = acc[u][n][2];
      red[(hl + 1) * LD + el + 1] = acc[u][n][3];
    }
  }
  __syncthreads();
  float* out = part + (long long)blockIdx.y * H * E;
  for (int i = threadIdx.x; i < 256 * EW; i += 256) {
    const int hc = i / EW, el = i % EW, e = 8 * nt0 + el;  // hc: column within the CTA
    const int h = blockIdx.x * 256 + hc;
    if (el < 8 * ntn && e < E && h < H) {
      // half 0 (warp hc / 64), then half 1 (warp 4 + hc / 64)
      const float v = dsm[((hc >> 6) * 64 + (hc & 63)) * LD + el] +
                      dsm[((4 + (hc >> 6)) * 64 + (hc & 63)) * LD + el];
      out[(long long)h * E + e] = v;
    }
  }
}

// dWr[h, e] = sum over slices z (in order) of part[z, h, e], rounded to bf16.
__global__ void router_dw_final_kernel(const float* __restrict__ part, int slices, long long HE,
                                       __nv_bfloat16* __restrict__ dwr) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < HE;
       i += (long long)gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int z = 0; z < slices; ++z) s += part[z * HE + i];
    dwr[i] = __float2bfloat16_rn(s);
  }
}

// ------------------------------------------------------------ host helpers
constexpr int kHAlign = 64;  // H granule (16-byte rows of 8 bf16, 64-column warp blocks)

inline long long aux_blocks(int T) { return ((long long)T + kATokens - 1) / kATokens; }
inline int padded_experts(int E) { return (E + 7) / 8 * 8; }

// n-tiles (8 experts each) per CTA of the projection and of the dWr partials.
inline int logits_ntg(int E) {
  const int nt = (E + 7) / 8;
  return nt >= 5 ? 8 : nt >= 3 ? 4 : nt;
}
inline int dw_ntg(int E) {
  const int nt = (E + 7) / 8;
  return nt >= 2 ? 2 : 1;  // four n-tiles' accumulators would not fit two CTAs per SM
}
// Token slices of the dWr reduction: one wave of CTAs (three per SM for one
// n-tile, two otherwise: the register budget), each slice a multiple of
// 8 warps x 16 tokens.
inline int dw_slices(int T, int H, int E) {
  const int ntg = dw_ntg(E);
  const long long ctas = (long long)((H + 255) / 256) * (((E + 7) / 8 + ntg - 1) / ntg);
  long long z = 148LL * (ntg == 1 ? 3 : 2) / ctas;
  const long long max_z = ((long long)T + kWSliceUnit - 1) / kWSliceUnit;
  if (z > max_z) z = max_z;
  if (z < 1) z = 1;
  return (int)z;
}
inline long long dw_slice_len(int T, int slices) {
  return (((long long)T + slices - 1) / slices + kWSliceUnit - 1) / kWSliceUnit * kWSliceUnit;
}

inline size_t up256(size_t b) { return (b + 255) / 256 * 256; }

}  // namespace router
}  // namespace moe

using namespace moe;
namespace RT = moe::router;

namespace {
bool router_shape_ok(int T, int H, int E, int k) {
  return T >= 1 && H >= RT::kHAlign && H % RT::kHAlign == 0 && E >= 1 && E <= RT::kMaxE &&
         k >= 1 && k <= 8 && k <= E && (long long)T * E < (1LL << 31) &&
         (long long)T * H < (1LL << 40);
}

size_t wt_bytes(int H, int E) { return RT::up256((size_t)RT::padded_experts(E) * H * 2); }

template <int NTG>
int launch_dw(dim3 grid, cudaStream_t st, const __nv_bfloat16* x, const float* dl, int T, int H,
              int E, int slice, float* part) {
  constexpr size_t smem = RT::dw_smem_bytes<NTG>();
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(RT::router_dw_partial_kernel<NTG>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr = true;
  }
  RT::router_dw_partial_kernel<NTG><<<grid, 256, smem, st>>>(x, dl, T, H, E, slice, part);
  return MOE_OK;
}
}  // namespace

extern "C" size_t moe_router_workspace_size(int T, int H, int E) {
  if (T < 1 || H < RT::kHAlign || H % RT::kHAlign || E < 1 || E > RT::kMaxE) return 0;
  // forward: WrT, then the aux partial sums
  const size_t fwd = wt_bytes(H, E) + RT::up256((size_t)RT::aux_blocks(T) * E * 4) * 2;
  // backward: partial dWr of every token slice
  const size_t bwd = RT::up256((size_t)RT::dw_slices(T, H, E) * H * E * 4);
  return fwd > bwd ? fwd : bwd;
}

extern "C" int moe_router_forward(const void* x, const void* w_r, int T, int H, int E, int k,
                                  float* logits, int32_t* idx, float* w, float* aux,
                                  void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (!router_shape_ok(T, H, E, k) || !x || !w_r || !logits || !idx || !w || !aux ||
      !workspace || !aligned16(x) || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      workspace_bytes < moe_router_workspace_size(T, H, E))
    return MOE_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* wt = reinterpret_cast<__nv_bfloat16*>(ws);
  const int Ep = RT::padded_experts(E);
  {
    long long blocks = ((long long)Ep * H + 255) / 256;
    if (blocks > 148 * 8) blocks = 148 * 8;
    RT::router_wt_kernel<<<(unsigned)blocks, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(w_r), H, E, Ep, wt);
  }
  const int ntg = RT::logits_ntg(E);
  dim3 grid((unsigned)(((long long)T + 15) / 16), (unsigned)((Ep / 8 + ntg - 1) / ntg));
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  switch (ntg) {
    case 1: RT::router_logits_kernel<1><<<grid, RT::kLWarps * 32, 0, st>>>(xb, wt, T, H, E, logits); break;
    case 2: RT::router_logits_kernel<2><<<grid, RT::kLWarps * 32, 0, st>>>(xb, wt, T, H, E, logits); break;
    case 4: RT::router_logits_kernel<4><<<grid, RT::kLWarps * 32, 0, st>>>(xb, wt, T, H, E, logits); break;
    default: RT::router_logits_kernel<8><<<grid, RT::kLWarps * 32, 0, st>>>(xb, wt, T, H, E, logits); break;
  }
  int r = launch_status();
  if (r != MOE_OK) return r;
  r = moe_route(logits, T, E, k, idx, w, stream);
  if (r != MOE_OK) return r;
  const long long nb = RT::aux_blocks(T);
  float* part_s = reinterpret_cast<float*>(ws + wt_bytes(H, E));
  int32_t* part_c = reinterpret_cast<int32_t*>(ws + wt_bytes(H, E) +
                                               RT::up256((size_t)nb * E * 4));
  RT::router_aux_partial_kernel<<<(unsigned)nb, RT::kAThreads, 0, st>>>(logits, idx, T, E, k,
                                                                        part_s, part_c);
  RT::router_aux_final_kernel<<<1, 256, 0, st>>>(part_s, part_c, (int)nb, T, E, k, aux);
  return launch_status();
}

extern "C" int moe_router_backward(const void* x, const void* w_r, const float* logits,
                                   const float* aux, const float* dlogits_route, float aux_coeff,
                                   int T, int H, int E, float* dlogits, const void* dx_in,
                                   void* dx_out, void* dw_r, void* workspace,
                                   size_t workspace_bytes, moe_stream_t stream) {
  if (!router_shape_ok(T, H, E, 1) || !x || !w_r || !logits || !aux || !dlogits || !dx_out ||
      !dw_r || !workspace || !aligned16(x) || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      workspace_bytes < moe_router_workspace_size(T, H, E) || !aligned16(dx_out) ||
      (dx_in && !aligned16(dx_in)))
    return MOE_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  long long blocks = ((long long)T + 7) / 8;
  if (blocks > 148 * 16) blocks = 148 * 16;
  RT::router_aux_backward_kernel<<<(unsigned)blocks, 256, 0, st>>>(logits, aux, dlogits_route,
                                                                   aux_coeff, T, E, dlogits);
  {
    // dx: CTAs of 8 column blocks (256 columns) x a run of token tiles, one
    // wave of three CTAs per SM
    const long long col_ctas = (H + 255) / 256;
    const long long tiles = ((long long)T + 15) / 16;
    long long tok_ctas = 148 * 3 / col_ctas;
    if (tok_ctas < 1) tok_ctas = 1;
    if (tok_ctas > tiles) tok_ctas = tiles;
    const long long per = (tiles + tok_ctas - 1) / tok_ctas;
    dim3 gdx((unsigned)col_ctas, (unsigned)((tiles + per - 1) / per));
    RT::router_dx_kernel<<<gdx, 256, 0, st>>>(dlogits, static_cast<const __nv_bfloat16*>(w_r),
                                              static_cast<const __nv_bfloat16*>(dx_in), T, H, E,
                                              (int)per, static_cast<__nv_bfloat16*>(dx_out));
  }
  const int slices = RT::dw_slices(T, H, E);
  const long long slice = RT::dw_slice_len(T, slices);
  const int used = (int)(((long long)T + slice - 1) / slice);  // slices that hold tokens
  float* part = static_cast<float*>(workspace);
  const int ntg = RT::dw_ntg(E);
  dim3 gdw((unsigned)((H + 255) / 256), (unsigned)used, (unsigned)(((E + 7) / 8 + ntg - 1) / ntg));
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  int rc = MOE_OK;
  if (ntg == 1)
    rc = launch_dw<1>(gdw, st, xb, dlogits, T, H, E, (int)slice, part);
  else
    rc = launch_dw<2>(gdw, st, xb, dlogits, T, H, E, (int)slice, part);
  if (rc != MOE_OK) return rc;
  const long long HE = (long long)H * E;
  long long fb = (HE + 255) / 256;
  if (fb > 148 * 8) fb = 148 * 8;
  RT::router_dw_final_kernel<<<(unsigned)fb, 256, 0, st>>>(part, used, HE,
                                                          static_cast<__nv_bfloat16*>(dw_r));
  return launch_status();
}
