// Block-scaled MXFP8 grouped GEMM on tcgen05 (kind::mxf8f6f4, E4M3 x E4M3
// with one E8M0 scale per 32 K-values), with fused quantising epilogues.
//
// "Efficient MoE Training for Biological Foundation Models", §Challenge 2
// (MXFP8: a scale per block of 32 consecutive values; MXFP8 GEMMs run on
// Blackwell's block-scaled tensor-core instructions) and §Challenge 3 (the
// fused grouped MLP: SwiGLU, routing-probability scaling and quantisation
// folded into the grouped GEMMs, forward and backward).
//
// Same warp roles as the BF16 kernel. Differences:
//  * Both operands are K-major E4M3 (column-wise MXFP8 copies are stored
//    transposed, so wgrad operands are K-major too). A stage is 128 K-bytes:
//    A 128x128 B, B 256x128 B (two 128-row boxes), plus the stage's scale
//    tiles (512 B for A, 2 x 512 B for B) fetched with bulk copies.
//  * The MMA thread moves each stage's scales from shared memory into tensor
//    memory with tcgen05.cp (32x128b, replicated to the four lane quarters)
//    and issues four K=32 MMAs; scale byte kb of each 32-bit TMEM word is
//    selected by the instruction descriptor's scale ids.
//  * Tensor memory: two full fp32 accumulators (N = 256 columns each) would
//    fill all 512 columns and leave none for scales. Tiles alternate between
//    columns [0, 256) and [192, 448), which share [192, 256). The epilogue
//    first copies the shared 64 columns to registers and releases them, so
//    the next tile's MMAs start while the epilogue still works on the rest.
//    Columns [448, 512) hold the scale factors of the shared-memory stages.
//  * Quantising epilogues: each warp owns 32 rows of the tile, one per lane.
//    Row-wise blocks (32 columns of one row) are quantised by their lane.
//    Column-wise blocks (one column over the warp's 32 rows) are transposed
//    through a per-warp shared-memory buffer, after which each lane holds one
//    column and quantises it like a row, storing its 32 contiguous bytes.
#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace gemm_mx {

using gemm::FPROP;
using gemm::WGRAD;
using gemm::EPI_STORE;
using gemm::EPI_SWIGLU_FWD;
using gemm::EPI_SWIGLU_BWD;

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;  // bytes of E4M3 = elements per stage
constexpr int kMaxGroups = gemm::kMaxGroups;

constexpr int kABytes = BM * BK;
constexpr int kBBytes = BN * BK;
constexpr int kSfaBytes = 512;
constexpr int kSfbBytes = 1024;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSfStageBytes = kSfaBytes + kSfbBytes;
constexpr int kTxBytes = kStageBytes + kSfStageBytes;
// Per-warp transpose buffer of the column-wise quantiser: 32 rows x 36 words
// (rows 16-byte aligned for vector writes; column reads hit 32 banks).
constexpr int kXposeStride = 36;
constexpr int kXposeWords = 32 * kXposeStride;
constexpr int kGuRowBytes = 144;

// Shared-memory layout and warp counts of one kernel flavour. The plain
// (store / wgrad) kernels use a 4-stage ring and 4 epilogue warps; the fused
// quantising epilogues carry much more work per tile, so they run 8
// epilogue warps (two per TMEM lane quarter, each taking every other
// 32-column chunk) and keep a 3-stage ring to make room for the warps'
// transpose buffers.
template <bool FUSED>
struct Cfg {
  static constexpr int kStages = FUSED ? 3 : 4;
  static constexpr int kEpiWarps = FUSED ? 8 : 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  // A/B stages stay 1024-byte aligned (128B-swizzle atoms); the scale tiles
  // of all stages follow in a region of their own.
  static constexpr int kSfOffset = kStages * kStageBytes;
  static constexpr int kXposeOffset = kSfOffset + kStages * kSfStageBytes;
  // Per-warp staging of gate/up: the backward epilogue reads the saved values
  // through it (cp.async; 32 rows x (64 B gate + 64 B up), rows padded to
  // 144 B); the forward epilogue writes its gate and up boxes (2 x 2 KB)
  // there for TMA stores. 128-byte aligned.
  static constexpr int kGuOffset = kXposeOffset + (FUSED ? kEpiWarps * kXposeWords * 4 : 0);
  static constexpr int kBarOffset = kGuOffset + (FUSED ? kEpiWarps * 32 * kGuRowBytes : 0);
  // full[S], empty[S], tfull[2], region_empty[3], drain
  static constexpr int kNumBars = 2 * kStages + 6;
  static constexpr int kMiscOffset = kBarOffset + kNumBars * 8;
  static constexpr int kPrefixOffset = kMiscOffset + 16;
  static constexpr int kSmemBytes = kPrefixOffset + (kMaxGroups + 1) * 4;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
};

// Tensor-memory columns.
constexpr int kAcc1Col = 192;     // accumulator of odd tiles: [192, 448)
constexpr int kSfTmemCol = 448;   // scale factors: [448, 512)
constexpr int kSfColsPerStage = 12;  // 4 (A) + 8 (B)
static_assert(kSfTmemCol + 4 * kSfColsPerStage <= 512, "TMEM budget");
static_assert(kAcc1Col + BN <= kSfTmemCol, "TMEM budget");

struct MxParams {
  const int32_t* offsets;
  int E;
  int M, N, K;  // FPROP: N, K (M per group); WGRAD: M, N (K per group)
  int F;
  const uint8_t* sfa;
  long long sfa_ktiles;  // 128-wide K tiles per 128-row scale tile row of A
  const uint8_t* sfb;
  long long sfb_ktiles;
  long long b_rows;        // rows of the B operand tensor
  long long b_row_stride;  // FPROP: B rows per expert (row-wise weight copies)
  long long b_k_stride;    // FPROP: K per expert (column-wise weight copies)
  __nv_bfloat16* C;
  long long ldc;
  long long c_group_stride;
  const float* p_rows;
  __nv_bfloat16* GU;
  uint8_t* q_row;  // row-wise MXFP8 output [rows, q_row_ld]
  uint8_t* s_row;
  long long q_row_ld;
  uint8_t* q_col;  // column-wise MXFP8 output [cols, q_col_ld] (transposed)
  uint8_t* s_col;
  long long q_col_ld;
  float* dp_part;
  int n_part;
};

struct TileInfo {
  int e, mt, nt;
  long long row0;
  int rows;
  int k_iters;
};

template <int MODE>
__device__ __forceinline__ void decode_tile(const MxParams& p, const int* prefix, int t,
                                            int& e_hint, TileInfo& ti) {
  int e = e_hint;
  while (prefix[e + 1] <= t) ++e;
  e_hint = e;
  const int local = t - prefix[e];
  const long long o0 = p.offsets[e], o1 = p.offsets[e + 1];
  ti.e = e;
  ti.row0 = o0;
  ti.rows = (int)(o1 - o0);
  if (MODE == FPROP) {
    const int mtiles = (ti.rows + BM - 1) / BM;
    ti.mt = local % mtiles;
    ti.nt = local / mtiles;
    ti.k_iters = p.K / BK;
  } else {
    const int mtiles = p.M / BM;
    ti.mt = local % mtiles;
    ti.nt = local / mtiles;
    ti.k_iters = ti.rows / BK;
  }
}

// First B row of tile half h (each half is 128 rows of B = 128 output columns).
template <int EPI>
__device__ __forceinline__ int b_half_row(const MxParams& p, int nt, int h) {
  if (EPI == EPI_SWIGLU_FWD) return h * p.F + nt * (BN / 2);
  return nt * BN + h * (BN / 2);
}

// ---------------------------------------------------------------- epilogue helpers

// Row-wise MXFP8 of 32 consecutive values held by one thread: 32 code bytes
// to dst (16-byte aligned) and the scale byte to *sdst.
__device__ __forceinline__ void quant_row32(const float* v, uint8_t* dst, uint8_t* sdst) {
  // Non-negative floats order like their bit patterns; Inf and NaN are the largest.
  uint32_t mbits = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) mbits = max(mbits, __float_as_uint(v[i]) & 0x7FFFFFFFu);
  const uint32_t sb = mbits < 0x7F800000u ? mx_scale_byte(__uint_as_float(mbits)) : 0xFFu;
  uint32_t w[8];
  if (sb == 0xFFu) {
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = 0x7F7F7F7Fu;
  } else {
    const float inv = mx_inv_scale(sb);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i] = (uint32_t)cvt_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv) |
             ((uint32_t)cvt_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv) << 16);
  }
  uint4* o = reinterpret_cast<uint4*>(dst);
  o[0] = make_uint4(w[0], w[1], w[2], w[3]);
  o[1] = make_uint4(w[4], w[5], w[6], w[7]);
  *sdst = (uint8_t)sb;
}

// Column-wise MXFP8 of a 32 x 32 block held one row per lane (v[i] is row
// `lane`, column i): every column is one block. The block is transposed
// through this warp's buffer `xs` (32 rows of kXposeStride words), after
// which lane c holds column c and quantises it like a row: its 32 codes go to
// q + (f0 + c) * ld + rb and its scale byte to the tiled layout of an operand
// with ld columns. Called by all 32 lanes of the warp.
__device__ __forceinline__ void quant_col_block32(const float* v, uint8_t* q, uint8_t* sq,
                                                  long long ld, long long f0, long long rb,
                                                  float* xs, int lane) {
  __syncwarp();
  float4* row = reinterpret_cast<float4*>(xs + lane * kXposeStride);
#pragma unroll
  for (int i = 0; i < 8; ++i) row[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  __syncwarp();
  float c[32];
#pragma unroll
  for (int r = 0; r < 32; ++r) c[r] = xs[r * kXposeStride + lane];
  quant_row32(c, q + (f0 + lane) * ld + rb, sq + mx_scale_offset(f0 + lane, rb >> 5, ld));
}

// Tile-local accumulator chunk c (32 columns) of this warp's 32 rows: from
// the registers sh when the chunk lies in the shared TMEM region (already
// drained: local chunks 6, 7 of even tiles, 0, 1 of odd tiles), else from
// TMEM. NSH = 2: the warp drained both shared chunks (sh[0..63]); NSH = 1:
// it takes only chunks of parity h and drained the one of them that is
// shared (sh[0..31]). c is a run-time value; sh is read at constant indices.
template <int NSH>
__device__ __forceinline__ void acc_chunk(int c, bool odd, int h, const float* sh,
                                          uint32_t tl_tile, float* f) {
  const int s = odd ? c : c - 6;
  if (NSH == 2 ? s == 0 : s == h) {
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = sh[i];
  } else if (NSH == 2 && s == 1) {
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = sh[NSH == 2 ? 32 + i : i];
  } else {
    uint32_t v[32];
    ptx::tmem_ld_32x32b_x32(tl_tile + c * 32, v);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
  }
}

// Asynchronous copy of this lane's row of a 32-column gate/up chunk
// (2 x 64 bytes of bf16) into its staging row in shared memory.
__device__ __forceinline__ void stage_gu_chunk(const MxParams& p, long long grow, long long col,
                                               uint32_t dst) {
  const __nv_bfloat16* g = p.GU + grow * 2 * p.F + col;
  const __nv_bfloat16* u = g + p.F;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    ptx::cp_async_16(dst + 16 * i, g + 8 * i);
    ptx::cp_async_16(dst + 64 + 16 * i, u + 8 * i);
  }
  ptx::cp_async_commit();
}

// Element i (a compile-time index after unrolling) of 32 packed bf16 values.
__device__ __forceinline__ float bf16_at(const uint4* s, int i) {
  const uint4 v = s[i >> 3];
  const int w = (i >> 1) & 3;
  const uint32_t word = w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
  return (i & 1) ? gemm::bf16_hi(word) : gemm::bf16_lo(word);
}

__device__ __forceinline__ void unpack_bf16x32(const uint4* s, float* v) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t w[4] = {s[q].x, s[q].y, s[q].z, s[q].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * q + 2 * j] = gemm::bf16_lo(w[j]);
      v[8 * q + 2 * j + 1] = gemm::bf16_hi(w[j]);
    }
  }
}

// The epilogue of one tile for this warp's 32 rows (lane = row). Fused
// epilogues split the tile's 32-column chunks between two warps per lane
// quarter by parity h; the plain ones take every chunk (h = 0, NSH = 2).
template <int MODE, int EPI>
__device__ __forceinline__ void epilogue_tile(const MxParams& p, const TileInfo& ti, bool odd,
                                              int h, const float* sh, uint32_t tl_tile, int q,
                                              int lane, float* xs, uint8_t* gu_stage,
                                              const CUtensorMap* tm_gu) {
  const long long lrow = (long long)ti.mt * BM + q * 32 + lane;
  const bool has_acc = ti.k_iters > 0;
  if (MODE == WGRAD) {
    __nv_bfloat16* crow = p.C + (long long)ti.e * p.c_group_stride + lrow * p.ldc +
                          (long long)ti.nt * BN;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      float f[32];
      if (has_acc) {
        acc_chunk<2>(c, odd, 0, sh, tl_tile, f);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = 0.f;
      }
      gemm::store32_bf16(crow + c * 32, f);
    }
    return;
  }
  const bool row_ok = lrow < ti.rows;
  const long long grow = ti.row0 + lrow;
  const long long rb = ti.row0 + (long long)ti.mt * BM + q * 32;  // first row of the warp
  if (EPI == EPI_STORE) {
    const int ncol = p.N - ti.nt * BN;
    __nv_bfloat16* crow = p.C + grow * p.ldc + (long long)ti.nt * BN;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      float f[32];
      acc_chunk<2>(c, odd, 0, sh, tl_tile, f);
      if (row_ok && c * 32 < ncol) gemm::store32_bf16(crow + c * 32, f);
    }
  } else if (EPI == EPI_SWIGLU_FWD) {
    // Tile-local chunks 0..3 are gate, 4..7 are up, for F-columns n0 .. n0+127;
    // this warp takes h-columns chunks c = h, h + 2.
    const float pr = row_ok ? p.p_rows[grow] : 0.f;
    const long long F = p.F;
#pragma unroll 1
    for (int c = h; c < 4; c += 2) {
      float g[32], u[32];
      acc_chunk<1>(c, odd, h, sh, tl_tile, g);
      acc_chunk<1>(c + 4, odd, h, sh, tl_tile, u);
      const long long col = (long long)ti.nt * (BN / 2) + c * 32;
      // [g | u] in bf16: the warp's 32 x 32 gate and up boxes are staged in
      // shared memory (row `lane` = 64 bytes each) and written by TMA.
      if (lane == 0) ptx::bulk_wait_read_all();  // previous boxes have been read
      __syncwarp();
      gemm::store32_bf16(reinterpret_cast<__nv_bfloat16*>(gu_stage + lane * 64), g);
      gemm::store32_bf16(reinterpret_cast<__nv_bfloat16*>(gu_stage + 2048 + lane * 64), u);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const uint32_t sa = ptx::smem_u32(gu_stage);
        ptx::tma_store_2d(tm_gu, (int)col, (int)rb, sa);
        ptx::tma_store_2d(tm_gu, (int)(F + col), (int)rb, sa + 2048);
        ptx::bulk_commit_group();
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) g[i] = g[i] * gemm::sigmoidf_fast(g[i]) * u[i] * pr;  // h
      if (row_ok)
        quant_row32(g, p.q_row + grow * p.q_row_ld + col,
                    p.s_row + mx_scale_offset(grow, col >> 5, p.q_row_ld));
      quant_col_block32(g, p.q_col, p.s_col, p.q_col_ld, col, rb, xs, lane);
    }
  } else {  // EPI_SWIGLU_BWD: accumulator = dH for F-columns nt*256 + [0, 256)
    const float pr = row_ok ? p.p_rows[grow] : 0.f;
    const long long F = p.F;
    const int ncol = p.N - ti.nt * BN;
    float dp = 0.f;
    // Saved gate/up of this warp's next chunk, staged into shared memory
    // while the current chunk is quantised (rows are whole 128-row groups,
    // so every lane's row is valid).
    const uint32_t gu_row = ptx::smem_u32(gu_stage) + lane * kGuRowBytes;
    const uint4* gu_mine = reinterpret_cast<const uint4*>(gu_stage + lane * kGuRowBytes);
    if (h * 32 < ncol) stage_gu_chunk(p, grow, (long long)ti.nt * BN + h * 32, gu_row);
#pragma unroll 1
    for (int c = h; c < 8 && c * 32 < ncol; c += 2) {  // N tail: uniform across the warp
      const long long col = (long long)ti.nt * BN + c * 32;
      float dg[32], du[32];
      acc_chunk<1>(c, odd, h, sh, tl_tile, dg);  // dH for now
      ptx::cp_async_wait_all();
      uint4 gc[4], uc[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        gc[i] = gu_mine[i];
        uc[i] = gu_mine[4 + i];
      }
      if (c + 2 < 8 && (c + 2) * 32 < ncol) stage_gu_chunk(p, grow, col + 64, gu_row);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float g = bf16_at(gc, i), u = bf16_at(uc, i);
        const float sg = gemm::sigmoidf_fast(g);
        const float silu = g * sg;
        dp = fmaf(dg[i], silu * u, dp);
        const float da = dg[i] * pr;  // dA = dH * p
        dg[i] = da * u * sg * (1.f + g * (1.f - sg));
        du[i] = da * silu;
      }
      // dg into columns [0, F), du into [F, 2F), both directions.
      if (row_ok) {
        quant_row32(dg, p.q_row + grow * p.q_row_ld + col,
                    p.s_row + mx_scale_offset(grow, col >> 5, p.q_row_ld));
        quant_row32(du, p.q_row + grow * p.q_row_ld + F + col,
                    p.s_row + mx_scale_offset(grow, (F + col) >> 5, p.q_row_ld));
      }
      quant_col_block32(dg, p.q_col, p.s_col, p.q_col_ld, col, rb, xs, lane);
      quant_col_block32(du, p.q_col, p.s_col, p.q_col_ld, F + col, rb, xs, lane);
    }
    // This warp's partial of dL/dp over its chunks; the two warps of a lane
    // quarter write the two halves of the tile's partial (n_part = 2 per tile).
    if (row_ok) p.dp_part[grow * p.n_part + 2 * ti.nt + h] = dp;
  }
}

template <int MODE, int EPI>
__global__ void __launch_bounds__(Cfg<EPI != EPI_STORE>::kThreads, 1)
    grouped_gemm_mxf8_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmC, const MxParams p) {
  using L = Cfg<EPI != EPI_STORE>;
  constexpr int kStages = L::kStages;
  constexpr int kSfOffset = L::kSfOffset;
  constexpr int kBarOffset = L::kBarOffset;
  constexpr int kMiscOffset = L::kMiscOffset;
  constexpr int kPrefixOffset = L::kPrefixOffset;
  constexpr int kEpiThreads = 32 * L::kEpiWarps;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t bar0 = sbase + kBarOffset;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  // TMEM regions: 0 = [0, 192) (even tiles only), 1 = [192, 256) (shared),
  // 2 = [256, 448) (odd tiles only).
  auto region_bar = [&](int r) { return bar0 + 8u * (2 * kStages + 2 + r); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 5);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kMiscOffset);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kMiscOffset + 4);
  int* s_prefix = reinterpret_cast<int*>(smem + kPrefixOffset);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = (p.N + BN - 1) / BN;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) ptx::mbar_init(tfull_bar(b), 1);
    for (int r = 0; r < 3; ++r) ptx::mbar_init(region_bar(r), kEpiThreads);
    ptx::mbar_init(drain_bar, 1);
    ptx::fence_mbar_init();
    *s_abort = 0;
    int acc = 0;
    bool bad = false;
    s_prefix[0] = 0;
    for (int e = 0; e < p.E; ++e) {
      int rows = p.offsets[e + 1] - p.offsets[e];
      if (rows % BM) bad = true;
      int mt = (MODE == FPROP) ? (rows + BM - 1) / BM : p.M / BM;
      acc += mt * n_tiles;
      s_prefix[e + 1] = acc;
    }
    if (bad) {
      // Tiles would straddle groups (and the output buffers): do no work.
      raise_device_error(MOE_DEVERR_LAYOUT);
      for (int e = 0; e < p.E; ++e) s_prefix[e + 1] = 0;
    }
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(s_tmem), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int total_tiles = s_prefix[p.E];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (ptx::elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed_phase[kStages];
      bool armed[kStages];
      for (int s = 0; s < kStages; ++s) armed[s] = false;
      int e_hint = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        TileInfo ti;
        decode_tile<MODE>(p, s_prefix, t, e_hint, ti);
        const long long a_row = (MODE == FPROP) ? ti.row0 + (long long)ti.mt * BM
                                                : (long long)ti.mt * BM;
        for (int kb = 0; kb < ti.k_iters; ++kb) {
          if (!gemm::wait_bar(empty_bar(stage), phase ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          const uint32_t a_dst = sbase + stage * kStageBytes;
          const uint32_t b_dst = a_dst + kABytes;
          const uint32_t sfa_dst = sbase + kSfOffset + stage * kSfStageBytes;
          const uint32_t sfb_dst = sfa_dst + kSfaBytes;
          ptx::mbar_arrive_expect_tx(full_bar(stage), kTxBytes);
          armed[stage] = true;
          armed_phase[stage] = phase;
          const long long a_k = (MODE == FPROP) ? (long long)kb * BK : ti.row0 + (long long)kb * BK;
          ptx::tma_load_2d(a_dst, &tmA, (int)a_k, (int)a_row, full_bar(stage));
          ptx::bulk_load(sfa_dst, p.sfa + ((a_row / 128) * p.sfa_ktiles + a_k / 128) * 512,
                         kSfaBytes, full_bar(stage));
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            long long b_row, b_k;
            if (MODE == FPROP) {
              b_row = ti.e * p.b_row_stride + b_half_row<EPI>(p, ti.nt, h);
              b_k = ti.e * p.b_k_stride + (long long)kb * BK;
            } else {
              b_row = (long long)ti.nt * BN + h * (BN / 2);
              b_k = a_k;
            }
            ptx::tma_load_2d(b_dst + h * (BN / 2) * BK, &tmB, (int)b_k, (int)b_row,
                             full_bar(stage));
            // A half past the last row of B (the N tail of the last expert) reads
            // zeros through TMA; its scales are never used, so fetch the last tile.
            const long long sb_row = b_row < p.b_rows ? b_row : p.b_rows - 128;
            ptx::bulk_load(sfb_dst + h * 512,
                           p.sfb + ((sb_row / 128) * p.sfb_ktiles + b_k / 128) * 512, 512,
                           full_bar(stage));
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < kStages; ++s)
        if (armed[s]) gemm::drain_wait(full_bar(s), armed_phase[s]);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (ptx::elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      int e_hint = 0;
      bool ok = true;
      uint32_t uses[3] = {0, 0, 0};  // completed uses of each TMEM region
      int j = 0;                      // tiles processed by this CTA
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x, ++j) {
        TileInfo ti;
        decode_tile<MODE>(p, s_prefix, t, e_hint, ti);
        const int own = (j & 1) ? 2 : 0;
        // Wait until both regions of this tile were drained by the epilogue.
        if (!gemm::wait_bar(region_bar(1), (uses[1] & 1u) ^ 1u, s_abort)) break;
        if (!gemm::wait_bar(region_bar(own), (uses[own] & 1u) ^ 1u, s_abort)) break;
        uses[1]++;
        uses[own]++;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + ((j & 1) ? (uint32_t)kAcc1Col : 0u);
        for (int kb = 0; kb < ti.k_iters; ++kb) {
          if (!gemm::wait_bar(full_bar(stage), phase, s_abort)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = sbase + stage * kStageBytes;
          const uint32_t b_addr = a_addr + kABytes;
          const uint32_t sfa_addr = sbase + kSfOffset + stage * kSfStageBytes;
          const uint32_t sfb_addr = sfa_addr + kSfaBytes;
          const uint32_t sf_col = kSfTmemCol + stage * kSfColsPerStage;
          // scales: smem (32 rows x 16 B per 128-row tile) -> TMEM, 4 columns each
          ptx::tmem_cp_32x128b_warpx4(tmem_base + sf_col,
                                      ptx::smem_desc(sfa_addr, 128, 128, ptx::kSwizzleNone));
          ptx::tmem_cp_32x128b_warpx4(tmem_base + sf_col + 4,
                                      ptx::smem_desc(sfb_addr, 128, 128, ptx::kSwizzleNone));
          ptx::tmem_cp_32x128b_warpx4(tmem_base + sf_col + 8,
                                      ptx::smem_desc(sfb_addr + 512, 128, 128,
                                                     ptx::kSwizzleNone));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t da = ptx::smem_desc(a_addr + kk * 32, 16, 1024, ptx::kSwizzle128B);
            const uint64_t db = ptx::smem_desc(b_addr + kk * 32, 16, 1024, ptx::kSwizzle128B);
            ptx::mma_mxf8(d_tmem, da, db, ptx::idesc_mxf8(BM, BN, kk, kk), tmem_base + sf_col,
                          tmem_base + sf_col + 4, (kb | kk) ? 1u : 0u);
          }
          ptx::mma_commit(empty_bar(stage));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (ti.k_iters > 0)
          ptx::mma_commit(tfull_bar(j & 1));
        else
          ptx::mbar_arrive(tfull_bar(j & 1));
      }
      ptx::mma_commit(drain_bar);
      gemm::drain_wait(drain_bar, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;   // chunk parity (fused: two warps per quarter)
    constexpr int NSH = L::kEpiWarps == 8 ? 1 : 2;  // shared chunks drained per warp
    float* xs = reinterpret_cast<float*>(smem + L::kXposeOffset) + (warp - 2) * kXposeWords;
    uint8_t* gu_stage = smem + L::kGuOffset + (warp - 2) * 32 * kGuRowBytes;
    const uint32_t tl_lanes = tmem_base + ((uint32_t)(q * 32) << 16);
    int e_hint = 0;
    int j = 0;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++j) {
      TileInfo ti;
      decode_tile<MODE>(p, s_prefix, t, e_hint, ti);
      if (!gemm::wait_bar(tfull_bar(j & 1), (uint32_t)((j >> 1) & 1), s_abort)) break;
      ptx::tc_fence_after();
      const bool odd = (j & 1) != 0;
      // Drain this warp's part of the shared region [192, 256) (TMEM columns
      // 192 + 32h for the fused kernels, all 64 for the plain ones) and hand
      // the region back to the MMA thread.
      float sh[32 * NSH];
      if (ti.k_iters > 0) {
#pragma unroll
        for (int c = 0; c < NSH; ++c) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(tl_lanes + kAcc1Col + (NSH == 1 ? 32 * h : 32 * c), v);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) sh[c * 32 + i] = __uint_as_float(v[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32 * NSH; ++i) sh[i] = 0.f;
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(region_bar(1));
      epilogue_tile<MODE, EPI>(p, ti, odd, h, sh, tl_lanes + (odd ? (uint32_t)kAcc1Col : 0u), q,
                               lane, xs, gu_stage, &tmC);
      ptx::tc_fence_before();
      ptx::mbar_arrive(region_bar(odd ? 2 : 0));
    }
    // Bulk stores must be complete before this CTA's shared memory goes away.
    if (EPI == EPI_SWIGLU_FWD && lane == 0) ptx::bulk_wait_all();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 512);
  }
}

template <int MODE, int EPI>
static int launch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                  const MxParams& p, long long tiles_bound, cudaStream_t st) {
  using L = Cfg<EPI != EPI_STORE>;
  auto kern = grouped_gemm_mxf8_kernel<MODE, EPI>;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemAlloc) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    attr_set = true;
  }
  long long grid = tiles_bound < gemm::num_sms() ? tiles_bound : gemm::num_sms();
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, L::kThreads, L::kSmemAlloc, st>>>(ta, tb, tc, p);
  return launch_status();
}

static bool u8_map(CUtensorMap* m, const void* base, long long rows, long long cols) {
  // K-major E4M3 operand [rows, cols], box 128 rows x 128 bytes, 128B swizzle.
  return gemm::make_tmap(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, rows, cols, cols, 128, 128);
}

}  // namespace gemm_mx
}  // namespace moe

using namespace moe;
namespace MX = moe::gemm_mx;

namespace {
bool mx_ptrs_ok(const void* a, const void* sa, const void* b, const void* sb, const void* c) {
  return a && sa && b && sb && c && aligned16(a) && aligned16(sa) && aligned16(b) &&
         aligned16(sb) && aligned16(c);
}
}  // namespace

extern "C" int moe_grouped_gemm_mxfp8(int mode, const uint8_t* a, const uint8_t* sa,
                                      long long a_rows, long long a_cols, const uint8_t* b,
                                      const uint8_t* sb, long long b_rows, long long b_cols,
                                      long long b_row_stride, long long b_k_stride,
                                      const int32_t* offsets, int E, int M, int N, int K, void* C,
                                      moe_stream_t stream) {
  if (!mx_ptrs_ok(a, sa, b, sb, C) || !offsets || E < 1 || E > MX::kMaxGroups) return MOE_ERR_ARG;
  if (a_rows <= 0 || a_cols <= 0 || b_rows <= 0 || b_cols <= 0 || a_rows % 128 || a_cols % 128 ||
      b_rows % 128 || b_cols % 128 || a_rows >= (1LL << 31) || a_cols >= (1LL << 31) ||
      b_rows >= (1LL << 31) || b_cols >= (1LL << 31))
    return MOE_ERR_ARG;
  // the mode's own shape rules, all checked before any CUDA call
  if (mode == MOE_GEMM_FPROP) {
    if (N < 128 || N % 128 || K < MX::BK || K % MX::BK || b_row_stride < 0 || b_k_stride < 0)
      return MOE_ERR_ARG;
    // every B row and K index that any expert touches must lie inside B
    if ((E - 1) * b_row_stride + ((N + MX::BN - 1) / MX::BN) * MX::BN > b_rows + MX::BN / 2 ||
        (E - 1) * b_k_stride + K > b_cols || K > a_cols)
      return MOE_ERR_ARG;
  } else if (mode == MOE_GEMM_WGRAD) {
    if (M < MX::BM || M % MX::BM || N < MX::BN || N % MX::BN || M > a_rows || N > b_rows ||
        a_cols != b_cols)
      return MOE_ERR_ARG;
  } else {
    return MOE_ERR_ARG;
  }
  MX::MxParams p{};
  p.offsets = offsets;
  p.E = E;
  p.M = M;
  p.N = N;
  p.K = K;
  p.sfa = sa;
  p.sfa_ktiles = a_cols / 128;
  p.sfb = sb;
  p.sfb_ktiles = b_cols / 128;
  p.b_rows = b_rows;
  p.C = static_cast<__nv_bfloat16*>(C);
  p.ldc = N;
  CUtensorMap ta, tb;
  if (!MX::u8_map(&ta, a, a_rows, a_cols) || !MX::u8_map(&tb, b, b_rows, b_cols)) return MOE_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  if (mode == MOE_GEMM_FPROP) {
    p.b_row_stride = b_row_stride;
    p.b_k_stride = b_k_stride;
    long long bound = (a_rows / MX::BM + E) * (long long)((N + MX::BN - 1) / MX::BN);
    return MX::launch<FPROP, EPI_STORE>(ta, tb, tb, p, bound, st);
  }
  p.c_group_stride = (long long)M * N;
  long long bound = (long long)E * (M / MX::BM) * (N / MX::BN);
  return MX::launch<WGRAD, EPI_STORE>(ta, tb, tb, p, bound, st);
}

extern "C" int moe_fc1_swiglu_mxfp8(const uint8_t* xq, const uint8_t* sx, long long rows, int H,
                                    const uint8_t* w1t, const uint8_t* sw1t,
                                    const int32_t* offsets, const float* p_rows, int E, int F,
                                    void* gu, uint8_t* hq_row, uint8_t* sh_row, uint8_t* hq_col,
                                    uint8_t* sh_col, moe_stream_t stream) {
  if (!mx_ptrs_ok(xq, sx, w1t, sw1t, gu) || !offsets || !p_rows || !hq_row || !sh_row ||
      !hq_col || !sh_col || !aligned16(hq_row) || E < 1 || E > MX::kMaxGroups)
    return MOE_ERR_ARG;
  if (rows <= 0 || rows % 128 || rows >= (1LL << 31) || H < 128 || H % 128 || F < 128 || F % 128)
    return MOE_ERR_ARG;
  MX::MxParams p{};
  p.offsets = offsets;
  p.E = E;
  p.N = 2 * F;
  p.K = H;
  p.F = F;
  p.sfa = sx;
  p.sfa_ktiles = H / 128;
  p.sfb = sw1t;
  p.sfb_ktiles = (long long)E * H / 128;
  p.b_rows = 2LL * F;
  p.b_row_stride = 0;
  p.b_k_stride = H;
  p.p_rows = p_rows;
  p.GU = static_cast<__nv_bfloat16*>(gu);
  p.q_row = hq_row;
  p.s_row = sh_row;
  p.q_row_ld = F;
  p.q_col = hq_col;
  p.s_col = sh_col;
  p.q_col_ld = rows;
  CUtensorMap ta, tb, tc;
  if (!MX::u8_map(&ta, xq, rows, H) || !MX::u8_map(&tb, w1t, 2LL * F, (long long)E * H))
    return MOE_ERR_CUDA;
  // [g | u] output, written by TMA in 32 x 32 boxes
  if (!gemm::make_tmap(&tc, gu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, 2LL * F, 2LL * F, 32,
                       32, CU_TENSOR_MAP_SWIZZLE_NONE))
    return MOE_ERR_CUDA;
  long long bound = (rows / MX::BM + E) * (long long)(F / 128);
  return MX::launch<FPROP, EPI_SWIGLU_FWD>(ta, tb, tc, p, bound, (cudaStream_t)stream);
}

extern "C" int moe_fc2_dgrad_swiglu_bwd_mxfp8(const uint8_t* dy2q, const uint8_t* sdy2,
                                              long long rows, int H, const uint8_t* w2q,
                                              const uint8_t* sw2, const int32_t* offsets,
                                              const float* p_rows, const void* gu, int E, int F,
                                              uint8_t* dy1q_row, uint8_t* sdy1_row,
                                              uint8_t* dy1q_col, uint8_t* sdy1_col,
                                              float* dp_part, moe_stream_t stream) {
  if (!mx_ptrs_ok(dy2q, sdy2, w2q, sw2, gu) || !offsets || !p_rows || !dy1q_row || !sdy1_row ||
      !dy1q_col || !sdy1_col || !dp_part || !aligned16(dy1q_row) || E < 1 || E > MX::kMaxGroups)
    return MOE_ERR_ARG;
  if (rows <= 0 || rows % 128 || rows >= (1LL << 31) || H < 128 || H % 128 || F < 128 || F % 128)
    return MOE_ERR_ARG;
  MX::MxParams p{};
  p.offsets = offsets;
  p.E = E;
  p.N = F;
  p.K = H;
  p.F = F;
  p.sfa = sdy2;
  p.sfa_ktiles = H / 128;
  p.sfb = sw2;
  p.sfb_ktiles = H / 128;
  p.b_rows = (long long)E * F;
  p.b_row_stride = F;
  p.b_k_stride = 0;
  p.p_rows = p_rows;
  p.GU = const_cast<__nv_bfloat16*>(static_cast<const __nv_bfloat16*>(gu));
  p.q_row = dy1q_row;
  p.s_row = sdy1_row;
  p.q_row_ld = 2LL * F;
  p.q_col = dy1q_col;
  p.s_col = sdy1_col;
  p.q_col_ld = rows;
  p.dp_part = dp_part;
  p.n_part = 2 * ((F + MX::BN - 1) / MX::BN);  // two epilogue warps per row and tile
  CUtensorMap ta, tb;
  if (!MX::u8_map(&ta, dy2q, rows, H) || !MX::u8_map(&tb, w2q, (long long)E * F, H)) return MOE_ERR_CUDA;
  long long bound = (rows / MX::BM + E) * (long long)((F + MX::BN - 1) / MX::BN);
  return MX::launch<FPROP, EPI_SWIGLU_BWD>(ta, tb, tb, p, bound, (cudaStream_t)stream);
}
