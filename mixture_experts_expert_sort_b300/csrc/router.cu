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
// All kernels are memory-bound SIMT code; every reduction over tokens is done
// in a fixed order (per-block partials, then one ordered pass), so results do
// not depend on scheduling.
#include "common.cuh"

namespace moe {
namespace router {

constexpr int kMaxE = 256;

// ------------------------------------------------------------ projection
// Experts are handled in groups of 8 (E padded up to G = groups * 8, groups a
// power of two). CTA: 256 threads = groups x (256 / groups) tokens; thread
// (g = tid / tpc, token tid % tpc) owns 8 logits. One H slice per blockIdx.y,
// walked in chunks of 64: x (tpc x 64) and Wr (64 x G, zero-padded) are staged
// in shared memory as fp32, and each h costs 1 + 2 shared loads for 8 FMAs.
// Each slice writes partial logits; a second pass adds the slices in order.
constexpr int kPH = 64;   // hidden chunk
constexpr int kPThreads = 256;

inline __host__ __device__ int expert_groups(int E) {
  int g = 1;
  while (g * 8 < E) g *= 2;
  return g;
}

__global__ void __launch_bounds__(kPThreads)
    router_logits_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ wr,
                         int T, int H, int E, int h_slice, float* __restrict__ part) {
  extern __shared__ float rsm[];
  const int groups = expert_groups(E), G = groups * 8, tpc = kPThreads / groups;
  float* xs = rsm;                      // [tpc][kPH + 1]
  float* ws = rsm + tpc * (kPH + 1);    // [kPH][G]
  const int tid = threadIdx.x;
  const int g = tid / tpc, tl = tid % tpc;
  const long long t0 = (long long)blockIdx.x * tpc;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const int hb = blockIdx.y * h_slice, he = min(H, hb + h_slice);
  for (int h0 = hb; h0 < he; h0 += kPH) {
    // x chunk: tpc rows x 8 vectors of 8 bf16
    for (int i = tid; i < tpc * 8; i += kPThreads) {
      const int r = i >> 3, v = i & 7;
      const long long t = t0 + r;
      float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (t < T) {
        const uint4 u = *reinterpret_cast<const uint4*>(x + t * H + h0 + 8 * v);
        const __nv_bfloat162* hp = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 pq = __bfloat1622float2(hp[q]);
          f[2 * q] = pq.x;
          f[2 * q + 1] = pq.y;
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) xs[r * (kPH + 1) + 8 * v + j] = f[j];
    }
    for (int i = tid; i < kPH * G; i += kPThreads) {
      const int hh = i / G, e = i % G;
      ws[i] = e < E ? __bfloat162float(wr[(long long)(h0 + hh) * E + e]) : 0.f;
    }
    __syncthreads();
    const float* xr = xs + tl * (kPH + 1);
    const float4* wg = reinterpret_cast<const float4*>(ws + 8 * g);
#pragma unroll 8
    for (int hh = 0; hh < kPH; ++hh) {
      const float xv = xr[hh];
      const float4 a = wg[hh * (G / 4)], b = wg[hh * (G / 4) + 1];
      acc[0] = fmaf(xv, a.x, acc[0]);
      acc[1] = fmaf(xv, a.y, acc[1]);
      acc[2] = fmaf(xv, a.z, acc[2]);
      acc[3] = fmaf(xv, a.w, acc[3]);
      acc[4] = fmaf(xv, b.x, acc[4]);
      acc[5] = fmaf(xv, b.y, acc[5]);
      acc[6] = fmaf(xv, b.z, acc[6]);
      acc[7] = fmaf(xv, b.w, acc[7]);
    }
    __syncthreads();
  }
  const long long t = t0 + tl;
  if (t < T) {
    float* out = part + (long long)blockIdx.y * T * E + t * E;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (8 * g + i < E) out[8 * g + i] = acc[i];
  }
}

// logits = sum over the H slices, in slice order.
__global__ void router_logits_sum_kernel(const float* __restrict__ part, int slices, long long TE,
                                         float* __restrict__ logits) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < TE;
       i += (long long)gridDim.x * blockDim.x) {
    float s = part[i];
    for (int z = 1; z < slices; ++z) s += part[z * TE + i];
    logits[i] = s;
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
  for (int e = warp; e < kMaxE; e += 8) {
    float s = 0.f;
    long long c = 0;
    if (e < E)
      for (int b = lane; b < nblocks; b += 32) {
        s += part_s[(long long)b * E + e];
        c += part_c[(long long)b * E + e];
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s += __shfl_xor_sync(0xffffffffu, s, o);
      c += __shfl_xor_sync(0xffffffffu, c, o);
    }
    float f = 0.f, P = 0.f;
    if (e < E) {
      f = (float)((double)c / ((double)T * k));
      P = s / (float)T;
      if (lane == 0) {
        aux[1 + e] = f;
        aux[1 + E + e] = P;
      }
    }
    if (lane == 0) prod[e] = f * P;
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

// dx[t, h] = dx_in[t, h] + sum_e dl[t, e] * Wr[h, e]. CTA: one block of hb
// columns (Wr for them staged transposed in shared memory as bf16, Wt[e][h],
// so a lane's 16-byte reads are contiguous) and a chunk of tokens; one warp
// per token, each lane producing 16-byte output vectors (8 columns).
constexpr int kDXSmem = 96 * 1024;  // bytes of staged Wt per CTA

inline __host__ __device__ int dx_cols(int H, int E) {
  int hb = kDXSmem / (2 * E) / 256 * 256;  // multiple of 256 columns
  if (hb < 256) hb = 256;
  return hb < H ? hb : H;
}

__global__ void __launch_bounds__(256)
    router_dx_kernel(const float* __restrict__ dl, const __nv_bfloat16* __restrict__ wr,
                     const __nv_bfloat16* __restrict__ dx_in, int T, int H, int E,
                     int tokens_per_cta, __nv_bfloat16* __restrict__ dx_out) {
  extern __shared__ __align__(16) __nv_bfloat16 wt[];  // [E][hb]
  const int hb = dx_cols(H, E);
  const int h0 = blockIdx.x * hb;
  const int ncol = min(hb, H - h0);
  if (E % 8 == 0) {
    // 16-byte reads of Wr rows (8 experts), scattered into the 8 rows of Wt
    for (int i = threadIdx.x; i < ncol * (E / 8); i += blockDim.x) {
      const int hh = i / (E / 8), e0 = 8 * (i % (E / 8));
      const uint4 u = *reinterpret_cast<const uint4*>(wr + (long long)(h0 + hh) * E + e0);
      const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
      for (int j = 0; j < 8; ++j) wt[(e0 + j) * hb + hh] = b[j];
    }
  } else {
    for (int i = threadIdx.x; i < E * ncol; i += blockDim.x) {
      const int hh = i / E, e = i % E;  // read Wr rows contiguously
      wt[e * hb + hh] = wr[(long long)(h0 + hh) * E + e];
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long tb = (long long)blockIdx.y * tokens_per_cta;
  const long long te = min((long long)T, tb + tokens_per_cta);
  for (long long t = tb + warp; t < te; t += 8) {
    const float* dlr = dl + t * E;
    for (int v = lane; 8 * v < ncol; v += 32) {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int e = 0; e < E; ++e) {
        const float d = __ldg(dlr + e);
        const uint4 u = *reinterpret_cast<const uint4*>(wt + e * hb + 8 * v);
        const __nv_bfloat162* hp = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 w2 = __bfloat1622float2(hp[q]);
          acc[2 * q] = fmaf(d, w2.x, acc[2 * q]);
          acc[2 * q + 1] = fmaf(d, w2.y, acc[2 * q + 1]);
        }
      }
      const long long off = t * H + h0 + 8 * v;
      if (dx_in) {
        const uint4 u = *reinterpret_cast<const uint4*>(dx_in + off);
        const __nv_bfloat162* hp = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __bfloat1622float2(hp[q]);
          acc[2 * q] += f.x;
          acc[2 * q + 1] += f.y;
        }
      }
      uint4 o;
      __nv_bfloat162* op = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int q = 0; q < 4; ++q) op[q] = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
      *reinterpret_cast<uint4*>(dx_out + off) = o;
    }
  }
}

// Partial dWr over a token slice: part[z, h, e] = sum_{t in slice z} x[t, h] dl[t, e].
// CTA: 256 threads = groups x hc columns (hc = 256 / groups); thread (g, h)
// owns 8 experts of one column. Tokens in chunks of 32 staged in shared
// memory (x as fp32 [32][hc + 1], dl as [32][G]).
constexpr int kWT = 32;

__global__ void __launch_bounds__(256)
    router_dw_partial_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ dl,
                             int T, int H, int E, int slice, float* __restrict__ part) {
  extern __shared__ float wsm[];
  const int groups = expert_groups(E), G = groups * 8, hc = 256 / groups;
  float* xs = wsm;                   // [kWT][hc + 1]
  float* ds = wsm + kWT * (hc + 1);  // [kWT][G]
  const int tid = threadIdx.x;
  const int g = tid / hc, hl = tid % hc;
  const int h0 = blockIdx.x * hc;
  const long long tb = (long long)blockIdx.y * slice;
  const long long te = min((long long)T, tb + slice);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (long long c0 = tb; c0 < te; c0 += kWT) {
    // x: 32 rows x hc columns, 16-byte vectors of 8 bf16
    for (int i = tid; i < kWT * (hc / 8); i += 256) {
      const int r = i / (hc / 8), v = i % (hc / 8);
      const long long t = c0 + r;
      float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (t < te && h0 + 8 * v < H) {
        const uint4 u = *reinterpret_cast<const uint4*>(x + t * H + h0 + 8 * v);
        const __nv_bfloat162* hp = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 pq = __bfloat1622float2(hp[q]);
          f[2 * q] = pq.x;
          f[2 * q + 1] = pq.y;
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) xs[r * (hc + 1) + 8 * v + j] = f[j];
    }
    for (int i = tid; i < kWT * G; i += 256) {
      const int r = i / G, e = i % G;
      const long long t = c0 + r;
      ds[i] = (t < te && e < E) ? dl[t * E + e] : 0.f;
    }
    __syncthreads();
    const float4* dg = reinterpret_cast<const float4*>(ds + 8 * g);
#pragma unroll 8
    for (int r = 0; r < kWT; ++r) {
      const float xv = xs[r * (hc + 1) + hl];
      const float4 a = dg[r * (G / 4)], b = dg[r * (G / 4) + 1];
      acc[0] = fmaf(xv, a.x, acc[0]);
      acc[1] = fmaf(xv, a.y, acc[1]);
      acc[2] = fmaf(xv, a.z, acc[2]);
      acc[3] = fmaf(xv, a.w, acc[3]);
      acc[4] = fmaf(xv, b.x, acc[4]);
      acc[5] = fmaf(xv, b.y, acc[5]);
      acc[6] = fmaf(xv, b.z, acc[6]);
      acc[7] = fmaf(xv, b.w, acc[7]);
    }
    __syncthreads();
  }
  const int h = h0 + hl;
  if (h < H) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (8 * g + i < E) part[((long long)blockIdx.y * H + h) * E + 8 * g + i] = acc[i];
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
inline long long aux_blocks(int T) { return ((long long)T + kATokens - 1) / kATokens; }

// H slices of the projection (multiples of kPH): enough CTAs to keep about
// eight per SM busy.
inline long long logit_token_blocks(int T, int E) {
  const int tpc = kPThreads / expert_groups(E);
  return ((long long)T + tpc - 1) / tpc;
}
inline int logit_slices(int T, int H, int E) {
  const long long tok_blocks = logit_token_blocks(T, E);
  long long z = (148 * 8 + tok_blocks - 1) / tok_blocks;
  const long long max_z = H / kPH;
  if (z > max_z) z = max_z;
  if (z < 1) z = 1;
  return (int)z;
}
inline int logit_slice_len(int H, int slices) {
  return (H / kPH + slices - 1) / slices * kPH;
}

// Token slices of the dWr reduction: enough CTAs to keep about eight per SM busy.
inline int dw_cols(int E) { return 256 / expert_groups(E); }
inline int dw_slices(int T, int H, int E) {
  const long long cols = (H + dw_cols(E) - 1) / dw_cols(E);
  long long z = (148 * 8 + cols - 1) / cols;
  const long long max_z = ((long long)T + kWT - 1) / kWT;
  if (z > max_z) z = max_z;
  if (z < 1) z = 1;
  return (int)z;
}

inline size_t up256(size_t b) { return (b + 255) / 256 * 256; }

}  // namespace router
}  // namespace moe

using namespace moe;
namespace RT = moe::router;

namespace {
bool router_shape_ok(int T, int H, int E, int k) {
  return T >= 1 && H >= RT::kPH && H % RT::kPH == 0 && E >= 1 && E <= RT::kMaxE && k >= 1 &&
         k <= 8 && k <= E && (long long)T * E < (1LL << 31);
}

int launch_logits(const void* x, const void* wr, int T, int H, int E, float* part,
                  float* logits, cudaStream_t st) {
  auto kern = RT::router_logits_kernel;
  const int groups = RT::expert_groups(E), tpc = RT::kPThreads / groups;
  const size_t smem = (size_t)(tpc * (RT::kPH + 1) + RT::kPH * groups * 8) * sizeof(float);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  const int slices = RT::logit_slices(T, H, E);
  const int slice_len = RT::logit_slice_len(H, slices);
  const int used = (H + slice_len - 1) / slice_len;  // slices that hold any h
  dim3 grid((unsigned)RT::logit_token_blocks(T, E), (unsigned)used);
  kern<<<grid, RT::kPThreads, smem, st>>>(static_cast<const __nv_bfloat16*>(x),
                                          static_cast<const __nv_bfloat16*>(wr), T, H, E,
                                          slice_len, part);
  const long long TE = (long long)T * E;
  long long blocks = (TE + 255) / 256;
  if (blocks > 148 * 8) blocks = 148 * 8;
  RT::router_logits_sum_kernel<<<(unsigned)blocks, 256, 0, st>>>(part, used, TE, logits);
  return launch_status();
}

int launch_dw(const void* x, const float* dl, int T, int H, int E, int slices, float* part,
              cudaStream_t st) {
  auto kern = RT::router_dw_partial_kernel;
  const int groups = RT::expert_groups(E), hc = RT::dw_cols(E);
  const size_t smem = (size_t)(RT::kWT * (hc + 1) + RT::kWT * groups * 8) * sizeof(float);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  const long long slice = (((long long)T + slices - 1) / slices + RT::kWT - 1) / RT::kWT * RT::kWT;
  dim3 grid((unsigned)((H + hc - 1) / hc), (unsigned)slices);
  kern<<<grid, 256, smem, st>>>(static_cast<const __nv_bfloat16*>(x), dl, T, H, E, (int)slice,
                                part);
  return launch_status();
}
}  // namespace

extern "C" size_t moe_router_workspace_size(int T, int H, int E) {
  if (T < 1 || H < RT::kPH || H % RT::kPH || E < 1 || E > RT::kMaxE) return 0;
  // forward: partial logits of every H slice, then the aux partial sums
  const size_t lg = RT::up256((size_t)RT::logit_slices(T, H, E) * T * E * 4);
  const size_t aux = RT::up256((size_t)RT::aux_blocks(T) * E * 4) * 2;
  // backward: partial dWr of every token slice
  const size_t dw = RT::up256((size_t)RT::dw_slices(T, H, E) * H * E * 4);
  return (lg > aux ? lg : aux) > dw ? (lg > aux ? lg : aux) : dw;
}

extern "C" int moe_router_forward(const void* x, const void* w_r, int T, int H, int E, int k,
                                  float* logits, int32_t* idx, float* w, float* aux,
                                  void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (!router_shape_ok(T, H, E, k) || !x || !w_r || !logits || !idx || !w || !aux ||
      !workspace || !aligned16(x) || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      workspace_bytes < moe_router_workspace_size(T, H, E))
    return MOE_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  float* part = static_cast<float*>(workspace);  // partial logits, consumed before the aux pass
  int r = launch_logits(x, w_r, T, H, E, part, logits, st);
  if (r != MOE_OK) return r;
  r = moe_route(logits, T, E, k, idx, w, stream);
  if (r != MOE_OK) return r;
  const long long nb = RT::aux_blocks(T);
  float* part_s = static_cast<float*>(workspace);
  int32_t* part_c = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) +
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
  if (!router_shape_ok(T, H, E, 1) || !x || !w_r || !aligned16(w_r) || !logits || !aux ||
      !dlogits || !dx_out ||
      !dw_r || !workspace || !aligned16(x) || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      workspace_bytes < moe_router_workspace_size(T, H, E) ||
      !aligned16(dx_out) || (dx_in && !aligned16(dx_in)))
    return MOE_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  long long blocks = ((long long)T + 7) / 8;
  if (blocks > 148 * 16) blocks = 148 * 16;
  RT::router_aux_backward_kernel<<<(unsigned)blocks, 256, 0, st>>>(logits, aux, dlogits_route,
                                                                   aux_coeff, T, E, dlogits);
  {
    const int hb = RT::dx_cols(H, E);
    const long long col_blocks = (H + hb - 1) / hb;
    long long tok_blocks = (148 * 2 + col_blocks - 1) / col_blocks;  // ~2 CTAs per SM
    if (tok_blocks > (T + 7) / 8) tok_blocks = (T + 7) / 8;
    if (tok_blocks < 1) tok_blocks = 1;
    const int tpc = (int)(((long long)T + tok_blocks - 1) / tok_blocks);
    const size_t smem = (size_t)E * hb * 2;
    if (cudaFuncSetAttribute(RT::router_dx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    dim3 gdx((unsigned)col_blocks, (unsigned)(((long long)T + tpc - 1) / tpc));
    RT::router_dx_kernel<<<gdx, 256, smem, st>>>(dlogits, static_cast<const __nv_bfloat16*>(w_r),
                                                  static_cast<const __nv_bfloat16*>(dx_in), T, H,
                                                  E, tpc, static_cast<__nv_bfloat16*>(dx_out));
  }
  const int slices = RT::dw_slices(T, H, E);
  float* part = static_cast<float*>(workspace);
  const int r = launch_dw(x, dlogits, T, H, E, slices, part, st);
  if (r != MOE_OK) return r;
  const long long HE = (long long)H * E;
  long long fb = (HE + 255) / 256;
  if (fb > 148 * 8) fb = 148 * 8;
  RT::router_dw_final_kernel<<<(unsigned)fb, 256, 0, st>>>(part, slices, HE,
                                                          static_cast<__nv_bfloat16*>(dw_r));
  return launch_status();
}
