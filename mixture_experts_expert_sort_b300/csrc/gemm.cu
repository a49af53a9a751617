// Persistent grouped GEMM on the 5th-generation tensor cores (tcgen05), fed
// by TMA, with fused epilogues.
//
// "Efficient MoE Training for Biological Foundation Models", §Challenge 1
// (GroupedLinear: one grouped operation over all local experts, each with
// its own weights and its own number of tokens, the split sizes) and
// §Challenge 3 (the GroupedLinear -> ScaledSwiGLU -> GroupedLinear sequence
// fused, with the SwiGLU and the routing-probability scaling applied to the
// FC1 result before it is written, plus a matching fused backward).
//
// Structure of one CTA (one per SM, persistent over output tiles):
//   warp 0      TMA producer: stages A and B tiles (128B swizzle) into a ring
//               of shared-memory stages, signalling `full` mbarriers.
//   warp 1      allocates TMEM; one elected thread issues tcgen05.mma for
//               each stage and commits to the stage's `empty` mbarrier, and
//               to the accumulator's `tfull` mbarrier at the end of a tile.
//   warps 2..5  epilogue: tcgen05.ld the fp32 accumulator (each warp owns a
//               32-lane quarter of TMEM = 32 rows of the tile), apply the
//               epilogue, store to global memory, release the accumulator.
// Two accumulators of BN fp32 columns each let the epilogue of one tile run
// under the main loop of the next.
//
// Tiles are 128 x BN x 64 (BF16). Expert groups are visited in order; within
// a group (FPROP) the m-tiles of one n-tile are adjacent, so a weight tile is
// read from HBM once and the group's activations stay in L2. In WGRAD the
// tiles along the smaller of M and N run fastest, so the smaller operand of
// the expert stays in L2 and the larger one is read once.
//
// Two problem shapes ("modes"):
//   FPROP: rows [o_e, o_{e+1}) of A times expert e's B (forward and dgrad).
//   WGRAD: C_e = A_e^T * B_e with the reduction over expert e's rows.
// Every wait is bounded: after kWaitLimitNs the kernel records
// MOE_DEVERR_TIMEOUT, stops issuing work, lets its copies land, frees TMEM
// and returns.
#include "common.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace moe {
namespace gemm {

enum Mode { FPROP = 0, WGRAD = 1 };
enum Epi { EPI_STORE = 0, EPI_SWIGLU_FWD = 1, EPI_SWIGLU_BWD = 2 };

constexpr int BM = 128;
// BF16 K per stage: 64 elements = 128 bytes = one 128-byte swizzle row.
// (32-element stages with 64-byte rows allow a deeper ring but double the
// TMA row requests of K-major operands, which measured slower.)
constexpr int BK = 64;
constexpr int kKRowBytes = BK * 2;            // one K-major row of a stage
constexpr int kKAtomBytes = 8 * kKRowBytes;   // 8-row swizzle atom (K-major)
constexpr int kThreads = 192;
constexpr int kMaxGroups = 256;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

struct Params {
  const int32_t* offsets;  // [E+1] group row offsets
  int E;
  int M, N, K;  // FPROP: N, K fixed (M per group); WGRAD: M, N fixed (K per group)
  int F;        // SwiGLU epilogues: FFN width (gate | up split of FC1 columns)
  int b_kmajor; // FPROP: 1 if expert B is stored [N, K], 0 if [K, N]
  __nv_bfloat16* C;          // EPI_STORE output, EPI_SWIGLU_BWD dY1 [rows, 2F]
  long long ldc;
  long long c_group_stride;  // WGRAD: elements between experts' outputs
  const float* p_rows;       // per-row routing weight (SwiGLU epilogues)
  __nv_bfloat16* GU;         // FWD: out [rows, 2F] (gate | up); BWD: in
  __nv_bfloat16* Hout;       // FWD: out [rows, F]
  float* dp_part;            // BWD: [rows, n_part] partial dL/dp per n-tile
  int n_part;
  // Row gather of one operand (template parameter G): permuted row r is row
  // g_src[r] / g_div of the source (g_rows rows, read through a tensor map
  // with one-row boxes), or zeros where g_src[r] < 0 or r >= g_n. A source
  // row past g_rows is read as zeros and reported as MOE_DEVERR_BAD_INDEX.
  long long g_rows;
  const int32_t* g_src;
  int g_div;
  long long g_n;
  long long l2_elems;  // L2 share of the resident tile band, in elements
};

// CG = 2: a CTA pair shares each tile (M = 256), each CTA staging its own 128
// rows of A and half of the B columns, so a stage is 32 KB instead of 48.
// FUSED: the SwiGLU epilogues move their bf16 tiles by TMA through a per-warp
// buffer (32 x 32 boxes, 2 KB each: FC1 stages g, u and h; the FC2 dgrad
// receives gate and up and stages dg and du).
constexpr int kEpiBufBytes = 8192;
// The plain epilogue stores its bf16 tile through TMA too, as 32 x 32 boxes
// from two per-warp buffers of 2 KB (one box being written while the other is
// read). Per-lane stores of 32 different rows cost the L1 one pass per row,
// time that the main loop's shared-memory operand reads then wait for.
constexpr int kStoreBufBytes = 4096;

// GATHER: the producer keeps the source row of each gathered operand row of
// a tile (FPROP, 128) or stage (WGRAD, 64) in shared memory.
template <int BN, int CG = 1, bool FUSED = false, bool GATHER = false>
struct Smem {
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = (BN / CG) * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (CG == 2 || BN != 256) ? 6 : 4;
  static constexpr int kEpiOffset = kStages * kStageBytes;  // 1024-byte aligned
  static constexpr int kGatherOffset = kEpiOffset + 4 * (FUSED ? kEpiBufBytes : kStoreBufBytes);
  static constexpr int kBarOffset = kGatherOffset + (GATHER ? BM * 4 : 0);
  // full[S], empty[S], tfull[2], tempty[2], drain, gate/up loads[4]
  static constexpr int kNumBars = 2 * kStages + 5 + (FUSED ? 4 : 0);
  static constexpr int kMiscOffset = kBarOffset + kNumBars * 8;
  // misc: tmem base (4), abort flag (4), tile prefix [kMaxGroups + 1] ints
  static constexpr int kPrefixOffset = kMiscOffset + 16;
  static constexpr int kBytes = kPrefixOffset + (kMaxGroups + 1) * 4;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 B
  static_assert(kAlloc <= 232448, "shared memory budget");
};

struct TileInfo {
  int e, mt, nt;
  long long row0;  // FPROP: first row of the group; WGRAD: first reduction row
  int rows;        // rows in the group
  int k_iters;
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      raise_device_error(MOE_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// Wait for in-flight asynchronous work at kernel exit: bounded by time only.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
      raise_device_error(MOE_DEVERR_TIMEOUT);
      return;
    }
  }
}

template <int MODE, int BN, int CG>
__device__ __forceinline__ void decode_tile(const Params& p, const int* prefix, int t, int& e_hint,
                                            TileInfo& ti) {
  constexpr int kTileM = BM * CG;
  int e = e_hint;
  while (prefix[e + 1] <= t) ++e;
  e_hint = e;
  const int local = t - prefix[e];
  const long long o0 = p.offsets[e], o1 = p.offsets[e + 1];
  ti.e = e;
  ti.row0 = o0;
  ti.rows = (int)(o1 - o0);
  const int K = MODE == FPROP ? p.K : ti.rows;
  const int mtiles = MODE == FPROP ? (ti.rows + kTileM - 1) / kTileM : p.M / kTileM;
  // an expert's whole grid: m-tiles fastest, except for a weight gradient
  // whose A (M columns) is the larger operand
  const bool prefer_m = MODE == FPROP || p.M <= p.N;
  // bands of at least two waves of tiles
  const int min_band = 2 * (int)(CG == 2 ? gridDim.x >> 1 : gridDim.x);
  band_order(local, mtiles, p.N / BN, kTileM, BN, p.l2_elems / max(K, 1), prefer_m, min_band,
             ti.mt, ti.nt);
  ti.k_iters = K / BK;
}

// Global column of B-tile half h (each half is BN/2 columns wide).
template <int EPI, int BN>
__device__ __forceinline__ int b_half_col(const Params& p, int nt, int h) {
  if (EPI == EPI_SWIGLU_FWD) return h * p.F + nt * (BN / 2);
  return nt * BN + h * (BN / 2);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void store32_bf16(__nv_bfloat16* dst, const float* v) {
  uint4* o = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    o[q] = make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                      pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
}

__device__ __forceinline__ void load32_bf16(const __nv_bfloat16* src, float* v) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u = s[q];
    v[8 * q + 0] = bf16_lo(u.x);
    v[8 * q + 1] = bf16_hi(u.x);
    v[8 * q + 2] = bf16_lo(u.y);
    v[8 * q + 3] = bf16_hi(u.y);
    v[8 * q + 4] = bf16_lo(u.z);
    v[8 * q + 5] = bf16_hi(u.z);
    v[8 * q + 6] = bf16_lo(u.w);
    v[8 * q + 7] = bf16_hi(u.w);
  }
}

// Logistic function from the hardware exponential and the hardware
// approximate reciprocal (relative error ~2^-22; 1/inf = 0 gives 0 for very
// negative z).
__device__ __forceinline__ float sigmoidf_fast(float z) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + __expf(-z)));
  return r;
}

// Lane `lane`'s 32 values as bf16 into row `lane` of a 32 x 32 box (64-byte
// rows) at `box`, in the 64-byte swizzle of a TMA copy with
// CU_TENSOR_MAP_SWIZZLE_64B: 16-byte chunk i of row r sits at i ^ ((r >> 1) & 3).
__device__ __forceinline__ void stage_bf16_row(uint8_t* box, int lane, const float* v) {
  uint4* d = reinterpret_cast<uint4*>(box + lane * 64);
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    d[q ^ sw] = make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                           pack_bf16(v[8 * q + 4], v[8 * q + 5]),
                           pack_bf16(v[8 * q + 6], v[8 * q + 7]));
}

// Row `lane` of such a box as 32 floats.
__device__ __forceinline__ void read_bf16_row(const uint8_t* box, int lane, float* v) {
  const uint4* s = reinterpret_cast<const uint4*>(box + lane * 64);
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = s[q ^ sw];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * q + 2 * j] = bf16_lo(w[j]);
      v[8 * q + 2 * j + 1] = bf16_hi(w[j]);
    }
  }
}

// TMA load of the saved gate and up boxes (32 rows x 32 columns, 64-byte
// swizzle) of gate/up column `col` and row `rb` to dst, completing on bar.
__device__ __forceinline__ void load_gate_up(const CUtensorMap* tm, uint32_t dst, int col, int F,
                                             int rb, uint32_t bar) {
  ptx::mbar_arrive_expect_tx(bar, 4096);
  ptx::tma_load_2d(dst, tm, col, rb, bar);
  ptx::tma_load_2d(dst + 2048, tm, F + col, rb, bar);
}

// tmC, tmD: the fused epilogues' bf16 tiles, written (or read) as 32 x 32
// boxes by TMA: FC1 + SwiGLU stores [g | u] (tmC) and H (tmD); FC2 dgrad +
// SwiGLU backward reads the saved [g | u] (tmC) and stores dY1 (tmD). A warp
// whose 32 rows straddle the end of a group uses per-lane loads and stores.
// G: which operand is read through a row gather (tmA or tmB is then a map of
// the un-permuted source with one-row boxes): 0 none, 1 A, 2 B (WGRAD only).
template <int MODE, int EPI, int BN, int A_MN, int B_MN, int CG, int G>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmC,
                             const __grid_constant__ CUtensorMap tmD, const Params p) {
  constexpr bool kFused = EPI != EPI_STORE;
  using L = Smem<BN, CG, kFused, G != 0>;
  constexpr bool kPair = CG == 2;
  // Rows of A (and columns of B) this CTA stages per stage, and the tile's M.
  constexpr int kTileM = BM * CG;
  constexpr int kBCols = BN / CG;  // this CTA's share of the tile's B columns
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t bar0 = sbase + L::kBarOffset;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (L::kStages + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * L::kStages + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * L::kStages + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * L::kStages + 4);
  auto gu_bar_of = [&](int w) { return bar0 + 8u * (2 * L::kStages + 5 + w); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::kMiscOffset);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::kMiscOffset + 4);
  int* s_prefix = reinterpret_cast<int*>(smem + L::kPrefixOffset);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = p.N / BN;
  // CTA pairs: rank 0 (the leader) issues the MMAs; tiles are dealt out per pair.
  const uint32_t rank = kPair ? ptx::cluster_ctarank() : 0u;
  const int unit = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int n_units = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull_bar(b), 1);
      // single CTA: every epilogue thread arrives; pair: one arrival per
      // epilogue warp of both CTAs, on the leader's barrier
      ptx::mbar_init(tempty_bar(b), kPair ? 8 : 128);
    }
    ptx::mbar_init(drain_bar, 1);
    if (kFused)
      for (int w = 0; w < 4; ++w) ptx::mbar_init(gu_bar_of(w), 1);
    ptx::fence_mbar_init();
    *s_abort = 0;
    // Tile prefix over groups.
    int acc = 0;
    bool bad = false;
    s_prefix[0] = 0;
    for (int e = 0; e < p.E; ++e) {
      int rows = p.offsets[e + 1] - p.offsets[e];
      int mt;
      if (MODE == FPROP) {
        mt = (rows + kTileM - 1) / kTileM;
      } else {
        mt = p.M / kTileM;
        if (rows % BK) bad = true;
      }
      acc += mt * n_tiles;
      s_prefix[e + 1] = acc;
    }
    if (bad) raise_device_error(MOE_DEVERR_LAYOUT);
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
    ptx::tma_prefetch_desc(&tmC);
    if (kFused) ptx::tma_prefetch_desc(&tmD);
  }
  if (warp == 1) {
    if (kPair) {
      ptx::tmem_alloc_cg2(ptx::smem_u32(s_tmem), 2 * BN);
      ptx::tmem_relinquish_cg2();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(s_tmem), 2 * BN);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  // A pair's barriers must be initialised in both CTAs before either CTA's
  // copies, commits or arrivals can reach them.
  if (kPair)
    ptx::cluster_sync();
  else
    __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int total_tiles = s_prefix[p.E];

  if (warp == 0 && G != 0) {
    // ------------------------------------------------- producer, row gather
    // The whole warp looks up the source row of every gathered operand row
    // (the tile's 128 A rows once per tile in FPROP, the stage's 64 reduction
    // rows in WGRAD, prefetched a stage ahead) into shared memory; lane 0
    // arms the stage and issues the other operand's box loads, and each lane
    // issues a tile::gather4 of four 128-byte rows. Every such TMA request
    // moves 512 bytes, so the gathered stream runs at the TMA unit's request
    // rate rather than at the bandwidth a 16 KB box load reaches.
    int* s_grow = reinterpret_cast<int*>(smem + L::kGatherOffset);
    // source row of a src entry; rows past the source (g_rows) are the
    // tensor map's zero fill, and a src entry past it is also reported
    auto src_row = [&](int sv) -> int {
      if (sv < 0) return (int)p.g_rows;
      const int r = sv / p.g_div;
      if (r >= p.g_rows) {
        raise_device_error(MOE_DEVERR_BAD_INDEX);
        return (int)p.g_rows;
      }
      return r;
    };
    auto raw_src = [&](long long r) -> int { return r < p.g_n ? p.g_src[r] : -1; };
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed_phase[L::kStages];
    bool armed[L::kStages];
    for (int s = 0; s < L::kStages; ++s) armed[s] = false;
    int e_hint = 0;
    bool ok = true;
    for (int t = unit; t < total_tiles && ok; t += n_units) {
      TileInfo ti;
      decode_tile<MODE, BN, CG>(p, s_prefix, t, e_hint, ti);
      int nx0 = 0, nx1 = 0;  // WGRAD: src entries of the next stage's rows
      if (MODE == FPROP) {
        const long long r0 = ti.row0 + (long long)ti.mt * kTileM + (long long)rank * BM;
        __syncwarp();  // the previous tile's copies are issued
        for (int i = lane; i < BM; i += 32) s_grow[i] = src_row(raw_src(r0 + i));
        __syncwarp();
      } else {
        nx0 = raw_src(ti.row0 + lane);
        nx1 = raw_src(ti.row0 + 32 + lane);
      }
      for (int kb = 0; kb < ti.k_iters; ++kb) {
        if (lane == 0) ok = wait_bar(empty_bar(stage), phase ^ 1u, s_abort);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        const int k0 = kb * BK;
        if (MODE == WGRAD) {
          __syncwarp();  // the previous stage's copies are issued
          s_grow[lane] = src_row(nx0);
          s_grow[lane + 32] = src_row(nx1);
          if (kb + 1 < ti.k_iters) {  // prefetch the next stage's entries
            nx0 = raw_src(ti.row0 + k0 + BK + lane);
            nx1 = raw_src(ti.row0 + k0 + BK + 32 + lane);
          }
        }
        const uint32_t a_dst = sbase + stage * L::kStageBytes;
        const uint32_t b_dst = a_dst + L::kABytes;
        const uint32_t fb = kPair ? ptx::mapa_shared(full_bar(stage), 0) : full_bar(stage);
        if (lane == 0 && rank == 0) {
          ptx::mbar_arrive_expect_tx(full_bar(stage), CG * L::kStageBytes);
          armed[stage] = true;
          armed_phase[stage] = phase;
        }
        __syncwarp();  // the stage is armed (and s_grow written) before any copy
        auto load = [&](uint32_t dst, const CUtensorMap* tm, int c0, int c1) {
          if (kPair)
            ptx::tma_load_2d_cg2(dst, tm, c0, c1, fb);
          else
            ptx::tma_load_2d(dst, tm, c0, c1, fb);
        };
        // n_rows gathered rows (s_grow[0 .. n_rows)) of columns c0 .. c0+63
        // to dst, one tile::gather4 of four rows per lane
        auto gather = [&](uint32_t dst, const CUtensorMap* tm, int c0, int n_rows) {
          for (int i = lane; i < n_rows / 4; i += 32) {
            const int* rr = s_grow + 4 * i;
            if (kPair)
              ptx::tma_gather4_cg2(dst + i * 512, tm, c0, rr[0], rr[1], rr[2], rr[3], fb);
            else
              ptx::tma_gather4(dst + i * 512, tm, c0, rr[0], rr[1], rr[2], rr[3], fb);
          }
        };
        if (MODE == FPROP) {
          gather(a_dst, &tmA, k0, BM);  // A: this CTA's 128 rows, K-major
          if (lane == 0) {
            if (B_MN) {
#pragma unroll
              for (int c = 0; c < kBCols / 64; ++c) {
                const int cc = (int)rank * (kBCols / 64) + c;
                const int h = cc / (BN / 128), off = (cc % (BN / 128)) * 64;
                const int n = b_half_col<EPI, BN>(p, ti.nt, h) + off;
                load(b_dst + c * (BK * 128), &tmB, n, ti.e * p.K + k0);
              }
            } else {
#pragma unroll
              for (int h = 0; h < 2 / CG; ++h) {
                const int n = b_half_col<EPI, BN>(p, ti.nt, kPair ? (int)rank : h);
                load(b_dst + h * (BN / 2) * kKRowBytes, &tmB, k0, ti.e * p.N + n);
              }
            }
          }
        } else {
          // WGRAD: the gathered operand's 64 reduction rows are s_grow[0 .. 64)
          const int r = (int)(ti.row0 + k0);
#pragma unroll
          for (int c = 0; c < BM / 64; ++c) {
            const int m = ti.mt * kTileM + (int)rank * BM + c * 64;
            if (G == 1)
              gather(a_dst + c * (BK * 128), &tmA, m, BK);
            else if (lane == 0)
              load(a_dst + c * (BK * 128), &tmA, m, r);
          }
#pragma unroll
          for (int c = 0; c < kBCols / 64; ++c) {
            const int n = ti.nt * BN + (int)rank * kBCols + c * 64;
            if (G == 2)
              gather(b_dst + c * (BK * 128), &tmB, n, BK);
            else if (lane == 0)
              load(b_dst + c * (BK * 128), &tmB, n, r);
          }
        }
        if (++stage == L::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // Let every armed copy land before the CTA can exit (bounded).
    if (lane == 0)
      for (int s = 0; s < L::kStages; ++s)
        if (armed[s]) drain_wait(full_bar(s), armed_phase[s]);
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (ptx::elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed_phase[L::kStages];
      bool armed[L::kStages];
      for (int s = 0; s < L::kStages; ++s) armed[s] = false;
      int e_hint = 0;
      bool ok = true;
      for (int t = unit; t < total_tiles && ok; t += n_units) {
        TileInfo ti;
        decode_tile<MODE, BN, CG>(p, s_prefix, t, e_hint, ti);
        for (int kb = 0; kb < ti.k_iters; ++kb) {
          if (!wait_bar(empty_bar(stage), phase ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          const uint32_t a_dst = sbase + stage * L::kStageBytes;
          const uint32_t b_dst = a_dst + L::kABytes;
          // Completion of both CTAs' copies of a pair is counted on the leader's barrier.
          const uint32_t fb = kPair ? ptx::mapa_shared(full_bar(stage), 0) : full_bar(stage);
          if (rank == 0) {
            ptx::mbar_arrive_expect_tx(full_bar(stage), CG * L::kStageBytes);
            armed[stage] = true;
            armed_phase[stage] = phase;
          }
          auto load = [&](uint32_t dst, const CUtensorMap* tm, int c0, int c1) {
            if (kPair)
              ptx::tma_load_2d_cg2(dst, tm, c0, c1, fb);
            else
              ptx::tma_load_2d(dst, tm, c0, c1, fb);
          };
          const int k0 = kb * BK;
          if (MODE == FPROP) {
            // A: this CTA's 128 rows of the tile, K-major, one box of 128 rows x BK.
            load(a_dst, &tmA, k0, (int)(ti.row0 + (long long)ti.mt * kTileM + rank * BM));
            if (B_MN) {
              // B_e stored [K, N]: this CTA's kBCols columns as chunks of [BK K rows][64 N].
#pragma unroll
              for (int c = 0; c < kBCols / 64; ++c) {
                const int cc = (int)rank * (kBCols / 64) + c;  // chunk of the whole tile
                const int h = cc / (BN / 128), off = (cc % (BN / 128)) * 64;
                const int n = b_half_col<EPI, BN>(p, ti.nt, h) + off;
                load(b_dst + c * (BK * 128), &tmB, n, ti.e * p.K + k0);
              }
            } else {
              // B_e stored [N, K]: boxes of BN/2 rows x BK (one per CTA of a pair).
#pragma unroll
              for (int h = 0; h < 2 / CG; ++h) {
                const int n = b_half_col<EPI, BN>(p, ti.nt, kPair ? (int)rank : h);
                load(b_dst + h * (BN / 2) * kKRowBytes, &tmB, k0, ti.e * p.N + n);
              }
            }
          } else {
            // WGRAD: A = X [rows, M] and B = Y [rows, N], both MN-major.
            const int r = (int)(ti.row0 + k0);
#pragma unroll
            for (int c = 0; c < BM / 64; ++c)
              load(a_dst + c * (BK * 128), &tmA, ti.mt * kTileM + (int)rank * BM + c * 64, r);
#pragma unroll
            for (int c = 0; c < kBCols / 64; ++c)
              load(b_dst + c * (BK * 128), &tmB, ti.nt * BN + (int)rank * kBCols + c * 64, r);
          }
          if (++stage == L::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Let every armed copy land before the CTA can exit (bounded). The
      // leader's barriers count both CTAs' copies of a pair.
      for (int s = 0; s < L::kStages; ++s)
        if (armed[s]) drain_wait(full_bar(s), armed_phase[s]);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (rank == 0 && ptx::elect_one()) {
      constexpr uint32_t idesc = ptx::idesc_bf16(kTileM, BN, MODE == WGRAD ? 1 : A_MN, B_MN);
      constexpr uint16_t kBoth = 3;  // commit to the barrier of both CTAs of a pair
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int e_hint = 0;
      bool ok = true;
      for (int t = unit; t < total_tiles && ok; t += n_units) {
        TileInfo ti;
        decode_tile<MODE, BN, CG>(p, s_prefix, t, e_hint, ti);
        if (!wait_bar(tempty_bar(acc), acc_phase ^ 1u, s_abort)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < ti.k_iters; ++kb) {
          if (!wait_bar(full_bar(stage), phase, s_abort)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = sbase + stage * L::kStageBytes;
          const uint32_t b_addr = a_addr + L::kABytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            uint64_t da, db;
            if (MODE == WGRAD || A_MN)
              da = ptx::smem_desc(a_addr + kk * 2048, BK * 128, 1024, ptx::kSwizzle128B);
            else
              da = ptx::smem_desc(a_addr + kk * 32, 16, kKAtomBytes, ptx::kSwizzle128B);
            if (B_MN)
              db = ptx::smem_desc(b_addr + kk * 2048, BK * 128, 1024, ptx::kSwizzle128B);
            else
              db = ptx::smem_desc(b_addr + kk * 32, 16, kKAtomBytes, ptx::kSwizzle128B);
            if (kPair)
              ptx::mma_bf16_cg2(d_tmem, da, db, idesc, (kb | kk) ? 1u : 0u);
            else
              ptx::mma_bf16(d_tmem, da, db, idesc, (kb | kk) ? 1u : 0u);
          }
          if (kPair)
            ptx::mma_commit_cg2(empty_bar(stage), kBoth);
          else
            ptx::mma_commit(empty_bar(stage));
          if (++stage == L::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (ti.k_iters > 0) {
          if (kPair)
            ptx::mma_commit_cg2(tfull_bar(acc), kBoth);
          else
            ptx::mma_commit(tfull_bar(acc));
        } else {
          ptx::mbar_arrive(tfull_bar(acc));
          if (kPair) ptx::mbar_arrive_remote(ptx::mapa_shared(tfull_bar(acc), 1));
        }
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // All MMAs issued by this thread complete before TMEM is released.
      if (kPair)
        ptx::mma_commit_cg2(drain_bar, 1);
      else
        ptx::mma_commit(drain_bar);
      drain_wait(drain_bar, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;  // row of this CTA's part of the tile
    // The accumulator-free arrival goes to the leader's barrier (one per warp
    // for a pair).
    int acc = 0;
    uint32_t acc_phase = 0;
    int e_hint = 0;
    // this warp's boxes (fused: the SwiGLU tiles; plain: two store boxes)
    uint8_t* ebuf = smem + L::kEpiOffset + (warp - 2) * (kFused ? kEpiBufBytes : kStoreBufBytes);
    const uint32_t ebuf_s = ptx::smem_u32(ebuf);
    const uint32_t gu_bar = gu_bar_of(warp - 2);
    uint32_t gu_phase = 0;
    bool gu_pending = false;  // a gate/up load of this warp is in flight
    for (int t = unit; t < total_tiles; t += n_units) {
      TileInfo ti;
      decode_tile<MODE, BN, CG>(p, s_prefix, t, e_hint, ti);
      // First row of this warp's 32 within the group, and whether the group
      // holds all 32 (TMA boxes) or none of them.
      const int wrow0 = ti.mt * kTileM + (int)rank * BM + q * 32;
      const bool warp_full = wrow0 + 32 <= ti.rows;
      const long long rb = ti.row0 + wrow0;
      if (EPI == EPI_SWIGLU_BWD && MODE == FPROP && warp_full) {
        // The saved gate/up of the first chunk does not depend on the
        // accumulator: fetch it while the tile's MMAs run.
        if (lane == 0) {
          ptx::fence_proxy_async_smem();  // after the previous tile's reads of the boxes
          load_gate_up(&tmC, ebuf_s, ti.nt * BN, p.F, (int)rb, gu_bar);
        }
        gu_pending = true;
      }
      if (!wait_bar(tfull_bar(acc), acc_phase, s_abort)) break;
      ptx::tc_fence_after();
      const uint32_t tm = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      const bool has_acc = ti.k_iters > 0;
      const int mrow = ti.mt * kTileM + (int)rank * BM + r;  // row of the group's tile rows
      // Plain epilogue through TMA: chunk c's 32 x 32 box of this warp's rows
      // (C row crow0) goes out from buffer c & 1.
      auto store_box = [&](int c, const float* f, long long crow0) {
        uint8_t* box = ebuf + (c & 1) * 2048;
        if (lane == 0) ptx::bulk_wait_read_1();  // the box written two chunks ago was read
        __syncwarp();
        stage_bf16_row(box, lane, f);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_2d(&tmC, ti.nt * BN + c * 32, (int)crow0, ptx::smem_u32(box));
          ptx::bulk_commit_group();
        }
      };
      if (MODE == WGRAD) {
        // C viewed as [E * M, N]: this warp's rows start at e * M + its first row
        const long long crow0 = (long long)ti.e * p.M + (mrow - lane);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          float f[32];
          if (has_acc) {
            ptx::tmem_ld_32x32b_x32(tm + c * 32, v);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = 0.f;
          }
          store_box(c, f, crow0);
        }
      } else {
        const int lrow = mrow;
        const bool row_ok = lrow < ti.rows;
        const long long grow = ti.row0 + lrow;
        if (EPI == EPI_STORE) {
          // A warp whose rows straddle the end of a ragged group stores per lane.
          __nv_bfloat16* crow = p.C + grow * p.ldc + (long long)ti.nt * BN;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32];
            float f[32];
            ptx::tmem_ld_32x32b_x32(tm + c * 32, v);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
            if (warp_full)
              store_box(c, f, rb);
            else if (row_ok)
              store32_bf16(crow + c * 32, f);
          }
        } else if (EPI == EPI_SWIGLU_FWD && warp_full) {
          // [g | u] and H leave as 32 x 32 boxes through this warp's buffer
          const float pr = p.p_rows[grow];
          const int n0 = ti.nt * (BN / 2);
          const long long F = p.F;
#pragma unroll 1
          for (int c = 0; c < BN / 64; ++c) {
            uint32_t vg[32], vu[32];
            ptx::tmem_ld_32x32b_x32(tm + c * 32, vg);
            ptx::tmem_ld_32x32b_x32(tm + BN / 2 + c * 32, vu);
            if (lane == 0) ptx::bulk_wait_read_all();  // the previous boxes were read
            __syncwarp();
            ptx::tmem_ld_wait();
            float g[32], u[32], h[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              g[i] = __uint_as_float(vg[i]);
              u[i] = __uint_as_float(vu[i]);
              h[i] = g[i] * sigmoidf_fast(g[i]) * u[i] * pr;
            }
            stage_bf16_row(ebuf, lane, g);
            stage_bf16_row(ebuf + 2048, lane, u);
            stage_bf16_row(ebuf + 4096, lane, h);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int col = n0 + c * 32;
              ptx::tma_store_2d(&tmC, col, (int)rb, ebuf_s);
              ptx::tma_store_2d(&tmC, (int)(F + col), (int)rb, ebuf_s + 2048);
              ptx::tma_store_2d(&tmD, col, (int)rb, ebuf_s + 4096);
              ptx::bulk_commit_group();
            }
          }
        } else if (EPI == EPI_SWIGLU_FWD) {
          const float pr = row_ok ? p.p_rows[grow] : 0.f;
          const int n0 = ti.nt * (BN / 2);
          const long long F = p.F;
#pragma unroll 1
          for (int c = 0; c < BN / 64; ++c) {
            uint32_t vg[32], vu[32];
            ptx::tmem_ld_32x32b_x32(tm + c * 32, vg);
            ptx::tmem_ld_32x32b_x32(tm + BN / 2 + c * 32, vu);
            ptx::tmem_ld_wait();
            float g[32], u[32], h[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              g[i] = __uint_as_float(vg[i]);
              u[i] = __uint_as_float(vu[i]);
              h[i] = g[i] * sigmoidf_fast(g[i]) * u[i] * pr;
            }
            if (row_ok) {
              const long long col = n0 + c * 32;
              store32_bf16(p.GU + grow * 2 * F + col, g);
              store32_bf16(p.GU + grow * 2 * F + F + col, u);
              store32_bf16(p.Hout + grow * F + col, h);
            }
          }
        } else if (warp_full) {  // EPI_SWIGLU_BWD through TMA boxes
          const float pr = p.p_rows[grow];
          const int n0 = ti.nt * BN;
          const long long F = p.F;
          float dp = 0.f;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tm + c * 32, v);  // dH, read while gate/up are waited for
            if (!wait_bar(gu_bar, gu_phase, s_abort)) {
              ptx::tmem_ld_wait();
              break;
            }
            gu_phase ^= 1u;
            gu_pending = false;
            float g[32], u[32];
            read_bf16_row(ebuf, lane, g);
            read_bf16_row(ebuf + 2048, lane, u);
            __syncwarp();  // the warp is done reading the boxes
            if (c + 1 < BN / 32) {
              if (lane == 0) {
                ptx::fence_proxy_async_smem();
                load_gate_up(&tmC, ebuf_s, n0 + (c + 1) * 32, (int)F, (int)rb, gu_bar);
              }
              gu_pending = true;
            }
            ptx::tmem_ld_wait();
            float dg[32], du[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float dh = __uint_as_float(v[i]);
              const float s = sigmoidf_fast(g[i]);
              const float silu = g[i] * s;
              dp = fmaf(dh, silu * u[i], dp);
              const float da = dh * pr;
              dg[i] = da * u[i] * s * (1.f + g[i] * (1.f - s));
              du[i] = da * silu;
            }
            if (lane == 0) ptx::bulk_wait_read_all();  // the previous dY1 boxes were read
            __syncwarp();
            stage_bf16_row(ebuf + 4096, lane, dg);
            stage_bf16_row(ebuf + 6144, lane, du);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int col = n0 + c * 32;
              ptx::tma_store_2d(&tmD, col, (int)rb, ebuf_s + 4096);
              ptx::tma_store_2d(&tmD, (int)(F + col), (int)rb, ebuf_s + 6144);
              ptx::bulk_commit_group();
            }
          }
          p.dp_part[grow * p.n_part + ti.nt] = dp;
        } else {  // EPI_SWIGLU_BWD, per lane: accumulator holds dH for F-columns [nt*BN, +BN)
          const float pr = row_ok ? p.p_rows[grow] : 0.f;
          const int n0 = ti.nt * BN;
          const long long F = p.F;
          float dp = 0.f;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tm + c * 32, v);
            ptx::tmem_ld_wait();
            if (row_ok) {
              const long long col = n0 + c * 32;
              float g[32], u[32], dg[32], du[32];
              load32_bf16(p.GU + grow * 2 * F + col, g);
              load32_bf16(p.GU + grow * 2 * F + F + col, u);
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const float dh = __uint_as_float(v[i]);
                const float s = sigmoidf_fast(g[i]);
                const float silu = g[i] * s;
                dp = fmaf(dh, silu * u[i], dp);
                const float da = dh * pr;
                dg[i] = da * u[i] * s * (1.f + g[i] * (1.f - s));
                du[i] = da * silu;
              }
              store32_bf16(p.C + grow * p.ldc + col, dg);
              store32_bf16(p.C + grow * p.ldc + F + col, du);
            }
          }
          if (row_ok) p.dp_part[grow * p.n_part + ti.nt] = dp;
        }
      }
      ptx::tc_fence_before();
      if (kPair) {
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            ptx::mbar_arrive_relaxed(tempty_bar(acc));
          else
            ptx::mbar_arrive_remote_relaxed(ptx::mapa_shared(tempty_bar(acc), 0));
        }
      } else {
        ptx::mbar_arrive_relaxed(tempty_bar(acc));
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // Bulk stores must be complete, and a gate/up load left in flight by an
    // abort must have landed, before this CTA's shared memory goes away.
    if (lane == 0) {
      ptx::bulk_wait_all();
      if (kFused && gu_pending) drain_wait(gu_bar, gu_phase);
    }
  }
  ptx::tc_fence_before();
  __syncwarp();
  // A pair leaves together: the leader's MMAs write the peer's tensor memory
  // and the peer's copies and arrivals reach the leader's barriers.
  if (kPair)
    ptx::cluster_sync();
  else
    __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    if (kPair)
      ptx::tmem_dealloc_cg2(tmem_base, 2 * BN);
    else
      ptx::tmem_dealloc(tmem_base, 2 * BN);
  }
}

// ------------------------------------------------------------------ host side

using moe::make_tmap;

// K-major BF16 operands: 128-byte rows, 128-byte swizzle (matches kSwizzle128B).
constexpr CUtensorMapSwizzle kKSwz = CU_TENSOR_MAP_SWIZZLE_128B;

static int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

// tiles_bound: an upper bound on the tiles of the launch (for CG = 2, on the
// 256-row tiles that CTA pairs take).
template <int MODE, int EPI, int BN, int A_MN, int B_MN, int CG = 1, int G = 0>
static int launch(const CUtensorMap& ta, const CUtensorMap& tb, const Params& p_in,
                  long long tiles_bound, cudaStream_t st, const CUtensorMap* tc = nullptr,
                  const CUtensorMap* td = nullptr) {
  Params p = p_in;
  p.l2_elems = kL2BandBytes / 2;
  auto kern = grouped_gemm_bf16_kernel<MODE, EPI, BN, A_MN, B_MN, CG, G>;
  const int smem = Smem<BN, CG, EPI != EPI_STORE, G != 0>::kAlloc;
  const CUtensorMap& mc = tc ? *tc : tb;  // plain epilogue: C; fused: see the kernel
  const CUtensorMap& md = td ? *td : tb;
  static bool attr_set = false;
  static int max_units = 0;  // co-resident CTAs (CG = 1) or CTA pairs (CG = 2)
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    max_units = num_sms();
    if (CG == 2) {
      cudaLaunchConfig_t q = {};
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = 2;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      q.gridDim = dim3(2 * (num_sms() / 2));
      q.blockDim = dim3(kThreads);
      q.dynamicSmemBytes = smem;
      q.attrs = qa;
      q.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess || n < 1) return MOE_ERR_CUDA;
      max_units = n;
    }
    attr_set = true;
  }
  long long units = tiles_bound < max_units ? tiles_bound : max_units;
  if (units < 1) units = 1;
  if (CG == 1) {
    kern<<<(unsigned)units, kThreads, smem, st>>>(ta, tb, mc, md, p);
    return launch_status();
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(2 * units));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, ta, tb, mc, md, p) != cudaSuccess) return MOE_ERR_CUDA;
  return launch_status();
}

}  // namespace gemm
}  // namespace moe

using namespace moe;
using namespace moe::gemm;

namespace {
constexpr CUtensorMapDataType kBF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;

bool gemm_common_ok(const void* A, const void* B, const void* C, const int32_t* offsets, int E) {
  return A && B && C && offsets && E >= 1 && E <= kMaxGroups && aligned16(A) && aligned16(B) &&
         aligned16(C);
}

// A row gather, when given, must name its map and a source of 1 .. 2^31-1 rows.
bool gather_ok(const moe_row_gather* g) {
  return !g || (g->src && g->src_div >= 1 && g->src_rows >= 1 && g->src_rows < (1LL << 31));
}

// The gathered operand [src_rows, cols] at base: permuted row r < rows is its
// row src[r] / src_div (zeros where src[r] < 0), read through a map of
// one-row boxes of 64 columns (128 bytes, 128-byte swizzle), four rows per
// tile::gather4.
bool set_gather(Params& p, CUtensorMap* m, const void* base, long long cols,
                const moe_row_gather* g, long long rows) {
  p.g_rows = g->src_rows;
  p.g_src = g->src;
  p.g_div = g->src_div;
  p.g_n = rows;
  return make_tmap(m, base, kBF16, 2, g->src_rows, cols, cols, 1, 64, kKSwz);
}
}  // namespace

extern "C" int moe_grouped_gemm_bf16(int mode, const void* A, const void* B, int b_layout,
                                     const int32_t* offsets, int E, long long rows, int M, int N,
                                     int K, void* C, const moe_row_gather* ga,
                                     const moe_row_gather* gb, moe_stream_t stream) {
  if (!gemm_common_ok(A, B, C, offsets, E) || rows < 0 || rows >= (1LL << 31)) return MOE_ERR_ARG;
  if (!gather_ok(ga) || !gather_ok(gb) || (ga && gb) || (mode == MOE_GEMM_FPROP && gb))
    return MOE_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  Params p{};
  p.offsets = offsets;
  p.E = E;
  p.M = M;
  p.N = N;
  p.K = K;
  p.C = static_cast<__nv_bfloat16*>(C);
  CUtensorMap ta, tb;
  if (mode == MOE_GEMM_FPROP) {
    if (N < 128 || N % 128 || K < BK || K % BK || (b_layout != 0 && b_layout != 1))
      return MOE_ERR_ARG;
    if (rows == 0) return MOE_OK;
    p.ldc = N;
    p.b_kmajor = b_layout;
    const bool bn256 = (N % 256) == 0;
    if (b_layout == 0) {
      if (!make_tmap(&tb, B, kBF16, 2, (long long)E * K, N, N, BK, 64)) return MOE_ERR_CUDA;
    } else {
      if (!make_tmap(&tb, B, kBF16, 2, (long long)E * N, K, K, bn256 ? 128 : 64, BK, kKSwz))
        return MOE_ERR_CUDA;
    }
    if (ga) {
      if (!set_gather(p, &ta, A, K, ga, rows)) return MOE_ERR_CUDA;
    } else if (!make_tmap(&ta, A, kBF16, 2, rows, K, K, BM, BK, kKSwz)) {
      return MOE_ERR_CUDA;
    }
    long long bound = (rows / BM + E) * (long long)(N / 128);
    // C [rows, N], stored by TMA in 32 x 32 boxes
    CUtensorMap tc;
    if (!make_tmap(&tc, C, kBF16, 2, rows, N, N, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
      return MOE_ERR_CUDA;
    if (ga) {
      if (bn256)
        return b_layout ? launch<FPROP, EPI_STORE, 256, 0, 0, 2, 1>(ta, tb, p, bound, st, &tc)
                        : launch<FPROP, EPI_STORE, 256, 0, 1, 2, 1>(ta, tb, p, bound, st, &tc);
      return b_layout ? launch<FPROP, EPI_STORE, 128, 0, 0, 1, 1>(ta, tb, p, bound, st, &tc)
                      : launch<FPROP, EPI_STORE, 128, 0, 1, 1, 1>(ta, tb, p, bound, st, &tc);
    }
    if (bn256)
      return b_layout ? launch<FPROP, EPI_STORE, 256, 0, 0, 2>(ta, tb, p, bound, st, &tc)
                      : launch<FPROP, EPI_STORE, 256, 0, 1, 2>(ta, tb, p, bound, st, &tc);
    return b_layout ? launch<FPROP, EPI_STORE, 128, 0, 0>(ta, tb, p, bound, st, &tc)
                    : launch<FPROP, EPI_STORE, 128, 0, 1>(ta, tb, p, bound, st, &tc);
  }
  if (mode == MOE_GEMM_WGRAD) {
    if (M < BM || M % BM || N < 128 || N % 128) return MOE_ERR_ARG;
    p.ldc = N;
    p.c_group_stride = (long long)M * N;
    const bool bn256 = (N % 256) == 0;
    if (rows > 0) {
      if (ga ? !set_gather(p, &ta, A, M, ga, rows)
             : !make_tmap(&ta, A, kBF16, 2, rows, M, M, BK, 64))
        return MOE_ERR_CUDA;
      if (gb ? !set_gather(p, &tb, B, N, gb, rows)
             : !make_tmap(&tb, B, kBF16, 2, rows, N, N, BK, 64))
        return MOE_ERR_CUDA;
    } else {
      // No rows at all: every expert's gradient is zero; maps are never read.
      if (!make_tmap(&ta, C, kBF16, 2, M, N, N, BK, 64)) return MOE_ERR_CUDA;
      tb = ta;
    }
    long long bound = (long long)E * (M / BM) * (N / 128);
    const int g = rows > 0 ? (ga ? 1 : gb ? 2 : 0) : 0;
    // C viewed as [E * M, N], stored by TMA in 32 x 32 boxes
    CUtensorMap tc;
    if (!make_tmap(&tc, C, kBF16, 2, (long long)E * M, N, N, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
      return MOE_ERR_CUDA;
    if (bn256 && M % 256 == 0)
      return g == 1   ? launch<WGRAD, EPI_STORE, 256, 1, 1, 2, 1>(ta, tb, p, bound, st, &tc)
             : g == 2 ? launch<WGRAD, EPI_STORE, 256, 1, 1, 2, 2>(ta, tb, p, bound, st, &tc)
                      : launch<WGRAD, EPI_STORE, 256, 1, 1, 2>(ta, tb, p, bound, st, &tc);
    if (bn256)
      return g == 1   ? launch<WGRAD, EPI_STORE, 256, 1, 1, 1, 1>(ta, tb, p, bound, st, &tc)
             : g == 2 ? launch<WGRAD, EPI_STORE, 256, 1, 1, 1, 2>(ta, tb, p, bound, st, &tc)
                      : launch<WGRAD, EPI_STORE, 256, 1, 1>(ta, tb, p, bound, st, &tc);
    return g == 1   ? launch<WGRAD, EPI_STORE, 128, 1, 1, 1, 1>(ta, tb, p, bound, st, &tc)
           : g == 2 ? launch<WGRAD, EPI_STORE, 128, 1, 1, 1, 2>(ta, tb, p, bound, st, &tc)
                    : launch<WGRAD, EPI_STORE, 128, 1, 1>(ta, tb, p, bound, st, &tc);
  }
  return MOE_ERR_ARG;
}

extern "C" int moe_fc1_swiglu_bf16(const void* xp, const void* w1, const int32_t* offsets,
                                   const float* p_rows, int E, long long rows, int H, int F,
                                   void* gu, void* h, const moe_row_gather* gx,
                                   moe_stream_t stream) {
  if (!gemm_common_ok(xp, w1, gu, offsets, E) || !h || !aligned16(h) || !p_rows || !gather_ok(gx))
    return MOE_ERR_ARG;
  if (H < BK || H % BK || F < 64 || F % 64 || rows < 0 || rows >= (1LL << 31)) return MOE_ERR_ARG;
  if (rows == 0) return MOE_OK;
  Params p{};
  p.offsets = offsets;
  p.E = E;
  p.N = 2 * F;
  p.K = H;
  p.F = F;
  p.p_rows = p_rows;
  p.GU = static_cast<__nv_bfloat16*>(gu);
  p.Hout = static_cast<__nv_bfloat16*>(h);
  CUtensorMap ta, tb, tc, td;
  if (!make_tmap(&tb, w1, kBF16, 2, (long long)E * H, 2 * F, 2 * F, BK, 64)) return MOE_ERR_CUDA;
  if (gx) {
    if (!set_gather(p, &ta, xp, H, gx, rows)) return MOE_ERR_CUDA;
  } else if (!make_tmap(&ta, xp, kBF16, 2, rows, H, H, BM, BK, kKSwz)) {
    return MOE_ERR_CUDA;
  }
  // [g | u] and H stored in 32 x 32 boxes
  if (!make_tmap(&tc, gu, kBF16, 2, rows, 2LL * F, 2LL * F, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_tmap(&td, h, kBF16, 2, rows, F, F, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return MOE_ERR_CUDA;
  long long bound_base = rows / BM + E;
  cudaStream_t st = (cudaStream_t)stream;
  if (F % 128 == 0)
    return gx ? launch<FPROP, EPI_SWIGLU_FWD, 256, 0, 1, 2, 1>(ta, tb, p, bound_base * (F / 128),
                                                               st, &tc, &td)
              : launch<FPROP, EPI_SWIGLU_FWD, 256, 0, 1, 2>(ta, tb, p, bound_base * (F / 128), st,
                                                            &tc, &td);
  return gx ? launch<FPROP, EPI_SWIGLU_FWD, 128, 0, 1, 1, 1>(ta, tb, p, bound_base * (F / 64), st,
                                                             &tc, &td)
            : launch<FPROP, EPI_SWIGLU_FWD, 128, 0, 1>(ta, tb, p, bound_base * (F / 64), st, &tc,
                                                       &td);
}

extern "C" int moe_swiglu_bwd_parts(int F) {
  if (F < 128 || F % 128) return 0;
  return (F % 256 == 0) ? F / 256 : F / 128;
}

extern "C" int moe_fc2_dgrad_swiglu_bwd_bf16(const void* dy2, const void* w2,
                                             const int32_t* offsets, const float* p_rows,
                                             const void* gu, int E, long long rows, int H, int F,
                                             void* dy1, float* dp_part, const moe_row_gather* gdy,
                                             moe_stream_t stream) {
  if (!gemm_common_ok(dy2, w2, dy1, offsets, E) || !gu || !aligned16(gu) || !p_rows || !dp_part ||
      !gather_ok(gdy))
    return MOE_ERR_ARG;
  if (H < BK || H % BK || F < 128 || F % 128 || rows < 0 || rows >= (1LL << 31)) return MOE_ERR_ARG;
  if (rows == 0) return MOE_OK;
  Params p{};
  p.offsets = offsets;
  p.E = E;
  p.N = F;
  p.K = H;
  p.F = F;
  p.p_rows = p_rows;
  p.GU = const_cast<__nv_bfloat16*>(static_cast<const __nv_bfloat16*>(gu));
  p.C = static_cast<__nv_bfloat16*>(dy1);
  p.ldc = 2LL * F;
  p.dp_part = dp_part;
  p.n_part = moe_swiglu_bwd_parts(F);
  const bool bn256 = (F % 256) == 0;
  CUtensorMap ta, tb, tc, td;
  // dH = dY2 * W2_e^T: B_e = W2_e stored [F, H] = [N, K], K-major.
  if (!make_tmap(&tb, w2, kBF16, 2, (long long)E * F, H, H, bn256 ? 128 : 64, BK, kKSwz))
    return MOE_ERR_CUDA;
  if (gdy) {
    if (!set_gather(p, &ta, dy2, H, gdy, rows)) return MOE_ERR_CUDA;
  } else if (!make_tmap(&ta, dy2, kBF16, 2, rows, H, H, BM, BK, kKSwz)) {
    return MOE_ERR_CUDA;
  }
  // saved [g | u] read, dY1 stored, in 32 x 32 boxes
  if (!make_tmap(&tc, gu, kBF16, 2, rows, 2LL * F, 2LL * F, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_tmap(&td, dy1, kBF16, 2, rows, 2LL * F, 2LL * F, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return MOE_ERR_CUDA;
  long long bound = (rows / BM + E) * (long long)(F / 128);
  cudaStream_t st = (cudaStream_t)stream;
  if (gdy)
    return bn256 ? launch<FPROP, EPI_SWIGLU_BWD, 256, 0, 0, 2, 1>(ta, tb, p, bound, st, &tc, &td)
                 : launch<FPROP, EPI_SWIGLU_BWD, 128, 0, 0, 1, 1>(ta, tb, p, bound, st, &tc, &td);
  return bn256 ? launch<FPROP, EPI_SWIGLU_BWD, 256, 0, 0, 2>(ta, tb, p, bound, st, &tc, &td)
               : launch<FPROP, EPI_SWIGLU_BWD, 128, 0, 0>(ta, tb, p, bound, st, &tc, &td);
}
