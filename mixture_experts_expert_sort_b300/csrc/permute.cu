// Expert sort (stable counting sort of routed rows by expert), permute and
// unpermute.
//
// "Efficient MoE Training for Biological Foundation Models", §Challenge 1:
// each expert's token list (the expert_mask / torch.where step of the
// per-expert loop), the per-expert token counts (split_sizes) that grouped
// execution takes, the gather that makes each expert's tokens contiguous,
// and the index_add that combines the expert outputs.
//
// The plan is three small launches over chunks of 1024 routed rows, one warp
// per chunk: (1) per-chunk expert histograms, (2) a column scan over chunks
// plus the padded exclusive scan over experts, (3) a stable scatter in which
// each warp walks its chunk 32 rows at a time and ranks equal experts with
// __match_any_sync. Ranks therefore follow the flat row index t*k + j, which
// is the order the oracle's stable sort produces, so dest/src are bit-exact.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kPlanChunk = 1024;
constexpr int kPlanWarps = 8;
constexpr int kPlanMaxE = 1024;

__global__ void __launch_bounds__(kPlanWarps * 32)
    plan_hist_kernel(const int32_t* __restrict__ idx, long long Tk, int E,
                     int32_t* __restrict__ chunk_counts, long long n_chunks,
                     int32_t* __restrict__ src, long long src_rows) {
  extern __shared__ int32_t s_cnt[];  // [kPlanWarps][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Fill src with -1 (the scatter launch that follows overwrites real rows).
  for (long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x; r < src_rows;
       r += (long long)gridDim.x * blockDim.x)
    src[r] = -1;
  int32_t* cnt = s_cnt + warp * E;
  long long chunk = (long long)blockIdx.x * kPlanWarps + warp;
  if (chunk >= n_chunks) return;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  long long beg = chunk * kPlanChunk, end = beg + kPlanChunk;
  if (end > Tk) end = Tk;
  for (long long i = beg + lane; i < end; i += 32) {
    int e = idx[i];
    if (e >= 0 && e < E)
      atomicAdd(&cnt[e], 1);
    else
      raise_device_error(MOE_DEVERR_BAD_INDEX);
  }
  __syncwarp();
  for (int e = lane; e < E; e += 32) chunk_counts[chunk * E + e] = cnt[e];
}

// One block: chunk_counts -> per-chunk base ranks (in place), counts, offsets.
__global__ void __launch_bounds__(1024)
    plan_scan_kernel(int32_t* __restrict__ chunk_counts, long long n_chunks, int E, int align,
                     int32_t* __restrict__ counts, int32_t* __restrict__ offsets) {
  __shared__ int32_t s_pad[kPlanMaxE];
  __shared__ int32_t s_warp[32];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (long long c = 0; c < n_chunks; ++c) {
      int v = chunk_counts[c * E + e];
      chunk_counts[c * E + e] = run;
      run += v;
    }
    counts[e] = run;
    s_pad[e] = (run + align - 1) / align * align;
  }
  __syncthreads();
  // Exclusive scan of s_pad over E <= 1024 entries: one element per thread.
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  int v = (t < E) ? s_pad[t] : 0;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int wv = (lane < (int)(blockDim.x >> 5)) ? s_warp[lane] : 0;
    int wi = wv;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    s_warp[lane] = wi - wv;  // exclusive prefix of warp totals
  }
  __syncthreads();
  int excl = s_warp[warp] + incl - v;
  if (t < E) offsets[t] = excl;
  if (t == E - 1) offsets[E] = excl + v;
}

__global__ void __launch_bounds__(kPlanWarps * 32)
    plan_scatter_kernel(const int32_t* __restrict__ idx, long long Tk, int E,
                        const int32_t* __restrict__ chunk_base, long long n_chunks,
                        const int32_t* __restrict__ offsets, int32_t* __restrict__ dest,
                        int32_t* __restrict__ src, long long src_rows) {
  extern __shared__ int32_t s_cnt[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* cnt = s_cnt + warp * E;
  long long chunk = (long long)blockIdx.x * kPlanWarps + warp;
  if (chunk >= n_chunks) return;
  for (int e = lane; e < E; e += 32) cnt[e] = offsets[e] + chunk_base[chunk * E + e];
  __syncwarp();
  long long beg = chunk * kPlanChunk, end = beg + kPlanChunk;
  if (end > Tk) end = Tk;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (long long base = beg; base < end; base += 32) {
    long long i = base + lane;
    int e = (i < end) ? idx[i] : -1;
    bool valid = (i < end) && e >= 0 && e < E;
    int key = valid ? e : -1;
    unsigned peers = __match_any_sync(0xffffffffu, key);
    int rank = __popc(peers & lt_mask);
    int d = -1;
    if (valid) d = cnt[e] + rank;
    __syncwarp();
    if (valid && rank == 0) cnt[e] += __popc(peers);
    __syncwarp();
    if (i < end) {
      if (valid && d >= src_rows) {
        raise_device_error(MOE_DEVERR_CAPACITY);
        d = -1;
      }
      dest[i] = d;
      if (d >= 0) src[d] = (int32_t)i;
    }
  }
}

// xp[dest[t*k+j]] = x[t]; padding rows zero. One warp per token, four
// independent 16-byte loads in flight per lane before the k scattered
// stores. The last blocks zero the padding rows: kPadWarps warps per expert,
// each taking every kPadWarps-th padding row of its expert. With xp NULL
// only the per-row routing weights p_rows are written.
constexpr int kPadWarps = 32;

__global__ void __launch_bounds__(256)
    permute_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ dest,
                   const int32_t* __restrict__ offsets, const int32_t* __restrict__ counts,
                   const float* __restrict__ w, int T, int HV, int E, int k, uint4* __restrict__ xp,
                   float* __restrict__ p_rows, int tok_blocks) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((int)blockIdx.x >= tok_blocks) {
    const int gw = (blockIdx.x - tok_blocks) * 8 + warp;
    const int e = gw / kPadWarps, part = gw % kPadWarps;
    if (e >= E) return;
    const long long r0 = (long long)offsets[e] + counts[e], r1 = offsets[e + 1];
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (long long r = r0 + part; r < r1; r += kPadWarps) {
      if (xp)
        for (int v = lane; v < HV; v += 32) xp[r * HV + v] = z;
      if (p_rows && lane == 0) p_rows[r] = 0.f;
    }
    return;
  }
  for (long long t = (long long)blockIdx.x * 8 + warp; t < T; t += (long long)tok_blocks * 8) {
    int d[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) d[j] = (j < k) ? dest[t * k + j] : -1;
    if (p_rows && lane < k && d[lane] >= 0) p_rows[d[lane]] = w[t * k + lane];
    if (!xp) continue;
    const uint4* xr = x + t * HV;
    int v = lane;
    for (; v + 96 < HV; v += 128) {
      uint4 val[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) val[u] = __ldcs(xr + v + 32 * u);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (d[j] >= 0) {
#pragma unroll
          for (int u = 0; u < 4; ++u) xp[(long long)d[j] * HV + v + 32 * u] = val[u];
        }
    }
    for (; v < HV; v += 32) {
      const uint4 val = __ldcs(xr + v);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (d[j] >= 0) xp[(long long)d[j] * HV + v] = val;
    }
  }
}

__device__ __forceinline__ void acc_bf16x8(float* acc, const uint4& v, float s) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float2 f = __bfloat1622float2(h[q]);
    acc[2 * q] = fmaf(s, f.x, acc[2 * q]);
    acc[2 * q + 1] = fmaf(s, f.y, acc[2 * q + 1]);
  }
}

// out[t] = sum_j w[t,j] * y[dest[t*k+j]], fp32 in slot order, one rounding.
// One warp per token; each lane issues the K row loads of two 16-byte
// vectors before it sums them. K is a template parameter so that the load
// buffers hold exactly K rows (occupancy: 2K vectors of registers per lane).
template <int K>
__global__ void __launch_bounds__(256)
    unpermute_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ dest,
                     const float* __restrict__ w, int T, int HV, uint4* __restrict__ out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (long long t = (long long)blockIdx.x * 8 + warp; t < T; t += (long long)gridDim.x * 8) {
    int d[K];
    float s[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      d[j] = dest[t * K + j];
      s[j] = w ? w[t * K + j] : 1.f;
    }
    for (int v0 = lane; v0 < HV; v0 += 64) {
      const bool two = v0 + 32 < HV;
      uint4 in[2][K];
#pragma unroll
      for (int j = 0; j < K; ++j) {
        const bool ok = d[j] >= 0;
        in[0][j] = ok ? __ldcs(y + (long long)d[j] * HV + v0) : make_uint4(0, 0, 0, 0);
        in[1][j] = (ok && two) ? __ldcs(y + (long long)d[j] * HV + v0 + 32) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (h == 1 && !two) break;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < K; ++j)
          if (d[j] >= 0) acc_bf16x8(acc, in[h][j], s[j]);
        uint4 o;
        __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
        for (int q = 0; q < 4; ++q) oh[q] = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
        __stcs(out + t * HV + v0 + 32 * h, o);
      }
    }
  }
}

template <int K>
void launch_unpermute(const uint4* y, const int32_t* dest, const float* w, int T, int HV,
                      uint4* out, unsigned blocks, cudaStream_t st) {
  unpermute_kernel<K><<<blocks, 256, 0, st>>>(y, dest, w, T, HV, out);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" long long moe_rows_padded_max(int T, int E, int k, int align) {
  if (T < 0 || E < 1 || k < 1 || align < 1) return -1;
  return (long long)T * k + (long long)E * (align - 1);
}

extern "C" size_t moe_permute_plan_workspace_size(int T, int E, int k) {
  if (T < 0 || E < 1 || k < 1) return 0;
  long long Tk = (long long)T * k;
  long long n_chunks = (Tk + kPlanChunk - 1) / kPlanChunk;
  if (n_chunks < 1) n_chunks = 1;
  size_t bytes = (size_t)n_chunks * (size_t)E * sizeof(int32_t);
  return (bytes + 255) / 256 * 256;
}

namespace moe {
// Shared by the workspace-taking entry point and any variant that supplies
// its own scratch: enqueues the three plan launches on `chunk_counts`.
static int permute_plan_launch(const int32_t* idx, int T, int E, int k, int align,
                               int32_t* counts, int32_t* offsets, int32_t* dest, int32_t* src,
                               long long src_rows, int32_t* chunk_counts, cudaStream_t st) {
  long long Tk = (long long)T * k;
  long long n_chunks = (Tk + kPlanChunk - 1) / kPlanChunk;
  size_t smem = (size_t)kPlanWarps * E * sizeof(int32_t);
  long long hist_blocks = (n_chunks + kPlanWarps - 1) / kPlanWarps;
  long long fill_blocks = (src_rows + 255) / 256;
  if (fill_blocks > 148 * 8) fill_blocks = 148 * 8;
  long long blocks1 = hist_blocks > fill_blocks ? hist_blocks : fill_blocks;
  if (blocks1 < 1) blocks1 = 1;
  plan_hist_kernel<<<(unsigned)blocks1, kPlanWarps * 32, smem, st>>>(idx, Tk, E, chunk_counts,
                                                                    n_chunks, src, src_rows);
  plan_scan_kernel<<<1, 1024, 0, st>>>(chunk_counts, n_chunks, E, align, counts, offsets);
  if (hist_blocks > 0)
    plan_scatter_kernel<<<(unsigned)hist_blocks, kPlanWarps * 32, smem, st>>>(
        idx, Tk, E, chunk_counts, n_chunks, offsets, dest, src, src_rows);
  return launch_status();
}

static int permute_plan_check(const int32_t* idx, int T, int E, int k, int align,
                              const int32_t* counts, const int32_t* offsets, const int32_t* dest,
                              const int32_t* src, long long src_rows) {
  if (T < 0 || E < 1 || E > kPlanMaxE || k < 1 || k > E || align < 1 || align > 4096)
    return MOE_ERR_ARG;
  long long Tk = (long long)T * k;
  if (Tk + (long long)E * (align - 1) >= (1LL << 31)) return MOE_ERR_ARG;
  if (src_rows < moe_rows_padded_max(T, E, k, align)) return MOE_ERR_ARG;
  if (!counts || !offsets || !src) return MOE_ERR_ARG;
  if (T > 0 && (!idx || !dest)) return MOE_ERR_ARG;
  return MOE_OK;
}
}  // namespace moe

extern "C" int moe_permute_plan(const int32_t* idx, int T, int E, int k, int align,
                                int32_t* counts, int32_t* offsets, int32_t* dest, int32_t* src,
                                long long src_rows, void* workspace, size_t workspace_bytes,
                                moe_stream_t stream) {
  int st = permute_plan_check(idx, T, E, k, align, counts, offsets, dest, src, src_rows);
  if (st != MOE_OK) return st;
  if (!workspace || workspace_bytes < moe_permute_plan_workspace_size(T, E, k) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MOE_ERR_ARG;
  return permute_plan_launch(idx, T, E, k, align, counts, offsets, dest, src, src_rows,
                             static_cast<int32_t*>(workspace), (cudaStream_t)stream);
}

extern "C" int moe_permute(const void* x, const int32_t* dest, const int32_t* offsets,
                           const int32_t* counts, const float* w, int T, int H, int E, int k,
                           void* xp, float* p_rows, moe_stream_t stream) {
  if (T < 0 || H < 8 || H % 8 || E < 1 || k < 1 || k > 8 || k > E) return MOE_ERR_ARG;
  if (!offsets || !counts || (T > 0 && !dest)) return MOE_ERR_ARG;
  if ((w == nullptr) != (p_rows == nullptr)) return MOE_ERR_ARG;
  if (!xp && !p_rows) return MOE_ERR_ARG;  // nothing to write
  if (xp && ((T > 0 && !x) || (x && !aligned16(x)) || !aligned16(xp))) return MOE_ERR_ARG;
  int HV = H / 8;
  long long tb = ((long long)T + 7) / 8;
  if (tb > 148 * 16) tb = 148 * 16;
  int pad_blocks = (E * kPadWarps + 7) / 8;
  permute_kernel<<<(unsigned)(tb + pad_blocks), 256, 0, (cudaStream_t)stream>>>(
      static_cast<const uint4*>(x), dest, offsets, counts, w, T, HV, E, k,
      static_cast<uint4*>(xp), p_rows, (int)tb);
  return launch_status();
}

extern "C" int moe_unpermute(const void* y, const int32_t* dest, const float* w, int T, int H,
                             int k, void* out, moe_stream_t stream) {
  if (T < 0 || H < 8 || H % 8 || k < 1 || k > 8) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  if (!y || !dest || !out || !aligned16(y) || !aligned16(out)) return MOE_ERR_ARG;
  long long blocks = ((long long)T + 7) / 8;
  if (blocks > 148 * 16) blocks = 148 * 16;
  const uint4* yv = static_cast<const uint4*>(y);
  uint4* ov = static_cast<uint4*>(out);
  const unsigned nb = (unsigned)blocks;
  cudaStream_t st = (cudaStream_t)stream;
  switch (k) {
    case 1: launch_unpermute<1>(yv, dest, w, T, H / 8, ov, nb, st); break;
    case 2: launch_unpermute<2>(yv, dest, w, T, H / 8, ov, nb, st); break;
    case 3: launch_unpermute<3>(yv, dest, w, T, H / 8, ov, nb, st); break;
    case 4: launch_unpermute<4>(yv, dest, w, T, H / 8, ov, nb, st); break;
    case 5: launch_unpermute<5>(yv, dest, w, T, H / 8, ov, nb, st); break;
    case 6: launch_unpermute<6>(yv, dest, w, T, H / 8, ov, nb, st); break;
    case 7: launch_unpermute<7>(yv, dest, w, T, H / 8, ov, nb, st); break;
    default: launch_unpermute<8>(yv, dest, w, T, H / 8, ov, nb, st); break;
  }
  return launch_status();
}
