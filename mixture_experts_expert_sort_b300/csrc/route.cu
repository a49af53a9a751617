// Top-k routing with renormalised softmax weights, and its backward.
//
// "How MoE Architecture Cuts Costs and Boosts Efficiency: Efficient Training
// of Biological Foundation Models", Router paragraph: keep the K highest
// scoring experts. "Efficient MoE Training for Biological Foundation Models",
// §Challenge 1: the routing weights that scale each expert's output.
//
// One warp per token. Lane l holds logits e = l, l+32, ...; k rounds of a
// warp arg-max (largest value, then lowest index) select the experts in
// descending order. HBM-bound: reads T*E*4 bytes, writes T*k*8.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kMaxE = 256;
constexpr int kMaxPerLane = kMaxE / 32;
constexpr int kMaxK = 8;

// (value, index) ordering: a beats b if a.v > b.v, or equal and a.i < b.i.
// Comparisons use float ==, so +0 and -0 tie and go to the lower index.
__device__ __forceinline__ bool beats(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E,
                                                    int k, int32_t* __restrict__ idx,
                                                    float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int warps_per_block = blockDim.x >> 5;
  for (long long t = (long long)blockIdx.x * warps_per_block + (threadIdx.x >> 5); t < T;
       t += (long long)gridDim.x * warps_per_block) {
    float v[kMaxPerLane];
    const float* row = logits + t * E;
#pragma unroll
    for (int s = 0; s < kMaxPerLane; ++s) {
      int e = lane + 32 * s;
      v[s] = (e < E) ? row[e] : 0.f;
    }
    unsigned taken = 0;  // bit s set: v[s] already selected (or out of range)
#pragma unroll
    for (int s = 0; s < kMaxPerLane; ++s)
      if (lane + 32 * s >= E) taken |= 1u << s;
    float sel_v[kMaxK];
    int sel_i[kMaxK];
    for (int j = 0; j < k; ++j) {
      float bv = 0.f;
      int bi = 0x7fffffff;
#pragma unroll
      for (int s = 0; s < kMaxPerLane; ++s) {
        if (!(taken >> s & 1u)) {
          int e = lane + 32 * s;
          if (bi == 0x7fffffff || beats(v[s], e, bv, bi)) {
            bv = v[s];
            bi = e;
          }
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (oi != 0x7fffffff && (bi == 0x7fffffff || beats(ov, oi, bv, bi))) {
          bv = ov;
          bi = oi;
        }
      }
      sel_v[j] = bv;
      sel_i[j] = bi;
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    }
    if (lane == 0) {
      float z[kMaxK];
      float sum = 0.f;
      for (int j = 0; j < k; ++j) {
        z[j] = expf(sel_v[j] - sel_v[0]);
        sum += z[j];
      }
      float inv = 1.f / sum;
      for (int j = 0; j < k; ++j) {
        idx[t * k + j] = sel_i[j];
        w[t * k + j] = z[j] * inv;
      }
    }
  }
}

// dp partials -> g_j (fixed order) -> softmax-over-top-k backward.
__global__ void route_backward_kernel(const float* __restrict__ dp, long long ld_dp, int n_part,
                                      const int32_t* __restrict__ dest,
                                      const float* __restrict__ w,
                                      const int32_t* __restrict__ idx, int T, int E, int k,
                                      float* __restrict__ dlogits) {
  long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  float g[kMaxK];
  float s = 0.f;
  for (int j = 0; j < k; ++j) {
    long long i = t * k + j;
    long long row = dest ? (long long)dest[i] : i;
    const float* p = dp + row * ld_dp;
    float acc = 0.f;
    for (int c = 0; c < n_part; ++c) acc += p[c];
    g[j] = acc;
    s += w[i] * acc;
  }
  float* out = dlogits + t * E;
  for (int e = 0; e < E; ++e) out[e] = 0.f;
  for (int j = 0; j < k; ++j) {
    int e = idx[t * k + j];
    if (e < 0 || e >= E) {
      raise_device_error(MOE_DEVERR_BAD_INDEX);
      continue;
    }
    out[e] = w[t * k + j] * (g[j] - s);
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_route(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                         moe_stream_t stream) {
  if (T < 0 || E < 1 || E > kMaxE || k < 1 || k > E || k > kMaxK) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  if (!logits || !idx || !w) return MOE_ERR_ARG;
  const int threads = 256, warps = threads / 32;
  long long blocks = ((long long)T + warps - 1) / warps;
  if (blocks > 148 * 16) blocks = 148 * 16;
  route_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(logits, T, E, k, idx, w);
  return launch_status();
}

extern "C" int moe_route_backward(const float* dp, long long ld_dp, int n_part,
                                  const int32_t* dest, const float* w, const int32_t* idx, int T,
                                  int E, int k, float* dlogits, moe_stream_t stream) {
  if (T < 0 || E < 1 || k < 1 || k > E || k > kMaxK || n_part < 1 || ld_dp < n_part)
    return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  if (!dp || !w || !idx || !dlogits) return MOE_ERR_ARG;
  const int threads = 128;
  long long blocks = ((long long)T + threads - 1) / threads;
  route_backward_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
      dp, ld_dp, n_part, dest, w, idx, T, E, k, dlogits);
  return launch_status();
}

extern "C" const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_ARG: return "MOE_ERR_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: shape or device not supported";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA runtime call failed";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE: the device error word was set";
    default: return "unknown moe_status";
  }
}

extern "C" int moe_device_error(moe_stream_t stream, unsigned* flags) {
  if (!flags) return MOE_ERR_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return MOE_ERR_CUDA;
  *flags = v;
  return v ? MOE_ERR_DEVICE : MOE_OK;
}
