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
//    column and quantises it like a row.
//  * Epilogue memory traffic goes through TMA. A warp-wide store or load in
//    which every lane touches a different row costs the L1 one pass per
//    cache line (32 per instruction), which starved these epilogues. So the
//    code bytes of every 32 x 32 block are staged in the warp's buffer and
//    written by TMA tensor stores, and the backward reads the saved gate/up
//    values through TMA loads (one mbarrier per epilogue warp, prefetched a
//    chunk ahead). Only the scale bytes (four cache lines per warp store)
//    are stored directly.
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
constexpr int kSfaBytes = 512;
constexpr int kSfbBytes = 1024;  // both 128-row halves of the tile's B scales
constexpr int kSfStageBytes = kSfaBytes + kSfbBytes;
// Per-warp transpose buffer of the column-wise quantiser: 32 rows x 36 words
// (rows 16-byte aligned for vector writes; column reads hit 32 banks).
constexpr int kXposeStride = 36;
constexpr int kXposeWords = 32 * kXposeStride;
// Per-warp buffer: the transposes use its first 4608 bytes; afterwards it
// stages the warp's 32 x 32-byte code boxes (1 KB each, 32-byte swizzle) for
// TMA stores. 1024-byte aligned so that every box is swizzle-aligned.
constexpr int kWarpBufBytes = 5120;
// Per-warp gate/up staging: two 32 x 32 bf16 boxes (64-byte rows, 64-byte
// swizzle): the backward's TMA loads, the forward's TMA stores.
constexpr int kGuBytes = 4096;
// The plain epilogue stores its bf16 tile through TMA as 32 x 32 boxes from
// two per-warp buffers of 2 KB (one being written while the other is read):
// per-lane stores of 32 different rows cost the L1 one pass per row, and the
// main loop's shared-memory operand reads wait for them.
constexpr int kStoreBufBytes = 4096;

__host__ __device__ constexpr int round1024(int x) { return (x + 1023) / 1024 * 1024; }

// Shared-memory layout and warp counts of one kernel flavour. The plain
// (store / wgrad) kernels use a 4-stage ring and 4 epilogue warps; the fused
// quantising epilogues carry much more work per tile, so they run 8
// epilogue warps (two per TMEM lane quarter, each taking every other
// 32-column chunk) and keep a 3-stage ring to make room for the warps'
// transpose buffers.
//
// CG = 2: a CTA pair shares each tile (M = 256 rows, the leader issuing the
// MMAs): each CTA stages its own 128 rows of A and half of the tile's B rows
// (32 KB per stage instead of 48), plus the scales of its A rows and of all
// the tile's B rows (each SM's tensor core reads the scales of every column
// of B it multiplies from its own tensor memory). The stage bytes freed go to
// a deeper ring.
//
// The ring's depth sets how much of the operand round trip (a stage's TMA
// load after the stage is freed) the tensor work in flight covers: copies of
// the plain pair kernel took 1.15, 1.19 and 1.36 ms with 5, 4 and 3 stages on
// one Mixtral-shape GEMM. The FC1 epilogue therefore stages its gate/up boxes
// in its transpose buffer instead of a buffer of their own, which leaves room
// for a fifth stage; the FC2-dgrad epilogue loads the next chunk's gate/up
// boxes while it transposes, so it keeps both buffers and four stages.
template <int EPI, int CG = 1>
struct Cfg {
  static constexpr bool FUSED = EPI != EPI_STORE;
  static constexpr bool kGuBuf = EPI == EPI_SWIGLU_BWD;  // gate/up boxes need their own buffer
  static constexpr int kStages =
      FUSED ? (CG == 2 ? (kGuBuf ? 4 : 5) : 3) : (CG == 2 ? 5 : 4);
  static constexpr int kBBytes = (BN / CG) * BK;  // this CTA's B rows per stage
  static constexpr int kStageBytes = kABytes + kBBytes;
  // bytes of one stage counted on the leader's full barrier (both CTAs of a pair)
  static constexpr int kTxBytes = CG * (kStageBytes + kSfStageBytes);
  static constexpr int kEpiWarps = FUSED ? 8 : 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  // A/B stages stay 1024-byte aligned (128B-swizzle atoms); the scale tiles
  // of all stages follow in a region of their own.
  static constexpr int kSfOffset = kStages * kStageBytes;
  static constexpr int kXposeOffset = round1024(kSfOffset + kStages * kSfStageBytes);
  static constexpr int kGuOffset =
      kXposeOffset + kEpiWarps * (FUSED ? kWarpBufBytes : kStoreBufBytes);
  static constexpr int kBarOffset = kGuOffset + (kGuBuf ? kEpiWarps * kGuBytes : 0);
  // full[S], empty[S], tfull[2], region_empty[3], drain, gate/up loads[epilogue warps]
  static constexpr int kNumBars = 2 * kStages + 6 + (FUSED ? kEpiWarps : 0);
  static constexpr int kMiscOffset = kBarOffset + kNumBars * 8;
  static constexpr int kPrefixOffset = kMiscOffset + 16;
  // tile prefix [kMaxGroups + 1] ints, then the group offsets [kMaxGroups + 1]
  static constexpr int kSmemBytes = kPrefixOffset + 2 * (kMaxGroups + 1) * 4;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
  static_assert(448 + kStages * 12 <= 512, "TMEM budget: scale columns of every stage");
};

// Tensor-memory columns.
constexpr int kAcc1Col = 192;     // accumulator of odd tiles: [192, 448)
constexpr int kSfTmemCol = 448;   // scale factors: [448, 512)
constexpr int kSfColsPerStage = 12;  // 4 (A) + 8 (B)
static_assert(kSfTmemCol + 5 * kSfColsPerStage <= 512, "TMEM budget");
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
  long long l2_elems;  // L2 share of the resident tile band, in elements (bytes)
};

struct TileInfo {
  int e, mt, nt;
  long long row0;
  int rows;
  int k_iters;
};

template <int MODE, int CG>
__device__ __forceinline__ void decode_tile(const MxParams& p, const int* prefix, int t,
                                            int& e_hint, TileInfo& ti) {
  constexpr int kTileM = BM * CG;
  int e = e_hint;
  while (prefix[e + 1] <= t) ++e;
  e_hint = e;
  const int local = t - prefix[e];
  // group offsets, copied to shared memory after the tile prefix at start-up
  const int* offs = prefix + kMaxGroups + 1;
  const long long o0 = offs[e], o1 = offs[e + 1];
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
  band_order(local, mtiles, (p.N + BN - 1) / BN, kTileM, BN, p.l2_elems / max(K, 1), prefer_m, min_band,
             ti.mt, ti.nt);
  ti.k_iters = K / BK;
}

// First B row of tile half h (each half is 128 rows of B = 128 output columns).
template <int EPI>
__device__ __forceinline__ int b_half_row(const MxParams& p, int nt, int h) {
  if (EPI == EPI_SWIGLU_FWD) return h * p.F + nt * (BN / 2);
  return nt * BN + h * (BN / 2);
}

// ---------------------------------------------------------------- epilogue helpers

// max(|a|, |b|, |c|), NaN when any input is NaN (one three-input instruction).
__device__ __forceinline__ float absmax3(float a, float b, float c) {
  float d;
  asm("max.NaN.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// MXFP8 of 32 consecutive values held by one thread: their 32 E4M3 codes in
// w[0..7] (value 4i + j in byte j of w[i]); returns the E8M0 scale byte.
__device__ __forceinline__ uint32_t quant32(const float* v, uint32_t* w) {
  // amax as a tree of three-input maxima (depth 4); Inf and NaN give scale 0xFF.
  float t[11];
#pragma unroll
  for (int k = 0; k < 10; ++k) t[k] = absmax3(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
  t[10] = absmax3(v[30], v[31], v[31]);
  const float u0 = absmax3(t[0], t[1], t[2]), u1 = absmax3(t[3], t[4], t[5]);
  const float u2 = absmax3(t[6], t[7], t[8]), u3 = absmax3(t[9], t[10], t[10]);
  const uint32_t mbits = __float_as_uint(absmax3(u0, u1, absmax3(u2, u3, u3))) & 0x7FFFFFFFu;
  const uint32_t sb = mbits < 0x7F800000u ? mx_scale_byte(__uint_as_float(mbits)) : 0xFFu;
  if (sb == 0xFFu) {
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = 0x7F7F7F7Fu;
  } else {
    const float inv = mx_inv_scale(sb);
    const uint64_t inv2 = ptx::f2_pack(inv, inv);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float a0, a1, a2, a3;  // v * 2^-e, two at a time
      ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(v[4 * i], v[4 * i + 1]), inv2), a0, a1);
      ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(v[4 * i + 2], v[4 * i + 3]), inv2), a2, a3);
      w[i] = (uint32_t)cvt_e4m3x2(a0, a1) | ((uint32_t)cvt_e4m3x2(a2, a3) << 16);
    }
  }
  return sb;
}

// Column-wise MXFP8 of a 32 x 32 block held one row per lane (v[i] is row
// `lane`, column i): every column is one block. The block is transposed
// through this warp's buffer `xs` (32 rows of kXposeStride words), after
// which lane c holds column c and quantises it: its 32 codes go to w[0..7]
// and its scale byte to the tiled layout of an operand with ld columns (row
// f0 + c, 32-row block rb / 32). Called by all 32 lanes.
__device__ __forceinline__ void quant_col32(const float* v, uint32_t* w, uint8_t* sq, long long ld,
                                            long long f0, long long rb, float* xs, int lane) {
  __syncwarp();
  float4* row = reinterpret_cast<float4*>(xs + lane * kXposeStride);
#pragma unroll
  for (int i = 0; i < 8; ++i) row[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  __syncwarp();
  float c[32];
#pragma unroll
  for (int r = 0; r < 32; ++r) c[r] = xs[r * kXposeStride + lane];
  sq[mx_scale_offset(f0 + lane, rb >> 5, ld)] = (uint8_t)quant32(c, w);
}

// Lane `lane`'s 32 code bytes into row `lane` of a 32 x 32-byte box at `box`
// (1 KB, 256-byte aligned), in the 32-byte swizzle a TMA store with
// CU_TENSOR_MAP_SWIZZLE_32B reads: 16-byte chunk i of row r sits at chunk
// i ^ ((r >> 2) & 1). Row r and r + 4 then fall in different bank halves.
__device__ __forceinline__ void stage_codes(uint8_t* box, int lane, const uint32_t* w) {
  uint4* d = reinterpret_cast<uint4*>(box + lane * 32);
  const int sw = (lane >> 2) & 1;
  d[sw] = make_uint4(w[0], w[1], w[2], w[3]);
  d[sw ^ 1] = make_uint4(w[4], w[5], w[6], w[7]);
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

// TMA load of the gate and up boxes (32 rows x 32 columns of bf16, 64-byte
// swizzle) of gate/up column `col` and row `rb` into this warp's staging
// buffer, completing on `bar`. Issued by one lane.
__device__ __forceinline__ void load_gu(const CUtensorMap* tm_gu, uint32_t dst, int col, int F,
                                        int rb, uint32_t bar) {
  ptx::mbar_arrive_expect_tx(bar, kGuBytes);
  ptx::tma_load_2d(dst, tm_gu, col, rb, bar);
  ptx::tma_load_2d(dst + 2048, tm_gu, F + col, rb, bar);
}

// Accumulator chunk c (tile-local, 32 columns) of this warp's 32 rows: a copy
// of `regs` when given (the chunk drained from the shared TMEM region), else
// read from TMEM. The read is only issued here; acc_ready() waits for it, so
// work that does not need the values can go in between.
__device__ __forceinline__ void load_acc(int c, const float* regs, uint32_t tl_tile, uint32_t* v) {
  if (regs) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(regs[i]);
  } else {
    ptx::tmem_ld_32x32b_x32(tl_tile + c * 32, v);
  }
}
__device__ __forceinline__ void acc_ready() { ptx::tmem_ld_wait(); }

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

// FC1 + SwiGLU epilogue of one gate/up chunk pair c (h-columns
// nt*128 + c*32 + [0, 32)) for this warp's 32 rows: [g | u] to bf16 through
// TMA stores, then H = silu(g) u p quantised row- and column-wise, its code
// boxes written by TMA. g_regs / u_regs: the drained shared-region chunk, if
// this pair holds it.
__device__ __forceinline__ void fwd_pair(const MxParams& p, const TileInfo& ti, int c,
                                         const float* g_regs, const float* u_regs, float pr,
                                         bool row_ok, long long grow, long long rb,
                                         uint32_t tl_tile, int lane, float* xs,
                                         uint8_t* gu_stage, const CUtensorMap* tm_gu,
                                         const CUtensorMap* tm_qr, const CUtensorMap* tm_qc) {
  const long long F = p.F;
  uint8_t* xb = reinterpret_cast<uint8_t*>(xs);
  uint32_t gv[32], uv[32];
  load_acc(c, g_regs, tl_tile, gv);
  load_acc(c + 4, u_regs, tl_tile, uv);
  const long long col = (long long)ti.nt * (BN / 2) + c * 32;
  // [g | u] in bf16: the warp's 32 x 32 gate and up boxes are staged in shared
  // memory (row `lane` = 64 bytes each) and written by TMA. The wait also
  // frees this warp's code boxes of its previous chunk.
  if (lane == 0) ptx::bulk_wait_read_all();
  __syncwarp();
  acc_ready();
  float g[32], u[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    g[i] = __uint_as_float(gv[i]);
    u[i] = __uint_as_float(uv[i]);
  }
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
  for (int i = 0; i < 32; i += 2) {  // h = silu(g) u p, two columns at a time
    const uint64_t g2 = ptx::f2_pack(g[i], g[i + 1]);
    const uint64_t s2 = ptx::f2_pack(gemm::sigmoidf_fast(g[i]), gemm::sigmoidf_fast(g[i + 1]));
    const uint64_t h2 = ptx::f2_mul(ptx::f2_mul(ptx::f2_mul(g2, s2), ptx::f2_pack(u[i], u[i + 1])),
                                    ptx::f2_pack(pr, pr));
    ptx::f2_unpack(h2, g[i], g[i + 1]);
  }
  // H: the column-wise block through the transpose (unless the caller wants
  // no column-wise copy), then the row-wise block.
  const bool cols = p.q_col != nullptr;
  uint32_t wc[8], wr[8];
  // the gate/up boxes sit in the same buffer: their TMA stores must have read them
  if (lane == 0) ptx::bulk_wait_read_all();
  __syncwarp();
  if (cols) quant_col32(g, wc, p.s_col, p.q_col_ld, col, rb, xs, lane);
  const uint32_t sb = quant32(g, wr);
  if (row_ok) p.s_row[mx_scale_offset(grow, col >> 5, p.q_row_ld)] = (uint8_t)sb;
  __syncwarp();  // every lane has read its column out of the buffer
  stage_codes(xb, lane, wr);
  if (cols) stage_codes(xb + 1024, lane, wc);
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    const uint32_t xb_s = ptx::smem_u32(xb);
    ptx::tma_store_2d(tm_qr, (int)col, (int)rb, xb_s);
    if (cols) ptx::tma_store_2d(tm_qc, (int)rb, (int)col, xb_s + 1024);
    ptx::bulk_commit_group();
  }
}

// The FC2-dgrad epilogue's chunks for a warp of parity h: tile-local chunks
// h, h + 2, h + 4, h + 6 that lie inside the tile's ncol columns, the one in
// the shared TMEM region (h of odd tiles, 6 + h of even ones) first. Four
// bits per chunk in bits 0..15, the count in bits 16 and up.
__host__ __device__ __forceinline__ uint32_t bwd_chunk_order(bool odd, int h, int ncol) {
  const int cs = odd ? h : 6 + h;
  uint32_t ord = 0;
  int n = 0;
  if (cs * 32 < ncol) ord |= (uint32_t)cs << (4 * n++);
  for (int c = h; c < 8; c += 2)
    if (c != cs && c * 32 < ncol) ord |= (uint32_t)c << (4 * n++);
  return ord | ((uint32_t)n << 16);
}

// Column block of gate/up chunk c (tile-local) of tile ti.
__device__ __forceinline__ int bwd_col(const TileInfo& ti, int c) { return ti.nt * BN + c * 32; }

// FC2-dgrad + SwiGLU-backward epilogue of the i-th chunk of `ord` for this
// warp's 32 rows. dH comes from `regs` (the drained shared-region chunk) or
// TMEM; the saved gate/up from this warp's TMA boxes (waited on here; the
// next chunk's boxes are requested as soon as these are read); dY1 = [dg | du]
// is quantised row- and column-wise and its four code boxes written by TMA;
// this chunk's part of dL/dp is added to dp. Returns false on an abort.
__device__ __forceinline__ bool bwd_chunk(const MxParams& p, const TileInfo& ti, uint32_t ord,
                                          int i, const float* regs, float pr, bool row_ok,
                                          long long grow, long long rb, uint32_t tl_tile,
                                          int lane, float* xs, uint8_t* gu_stage,
                                          const CUtensorMap* tm_gu, const CUtensorMap* tm_qr,
                                          const CUtensorMap* tm_qc, uint32_t gu_bar,
                                          uint32_t& gu_phase, bool& gu_pending,
                                          volatile int* s_abort, uint64_t& dp2) {
  const long long F = p.F;
  const int n = (int)(ord >> 16);
  const int c = (int)((ord >> (4 * i)) & 15);
  const long long col = bwd_col(ti, c);
  uint8_t* xb = reinterpret_cast<uint8_t*>(xs);
  uint32_t dhv[32];
  load_acc(c, regs, tl_tile, dhv);  // dH (awaited here: holding it across the gate/up wait spills)
  acc_ready();
  if (!gemm::wait_bar(gu_bar, gu_phase, s_abort)) return false;
  gu_phase ^= 1u;
  gu_pending = false;
  // Lane r reads row r of the boxes, whose 16-byte chunk j sits at
  // j ^ ((r >> 1) & 3) under the 64-byte swizzle.
  const int sw = (lane >> 1) & 3;
  const uint4* g_row = reinterpret_cast<const uint4*>(gu_stage + lane * 64);
  const uint4* u_row = reinterpret_cast<const uint4*>(gu_stage + 2048 + lane * 64);
  uint4 gc[4], uc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    gc[j] = g_row[j ^ sw];
    uc[j] = u_row[j ^ sw];
  }
  __syncwarp();  // the warp is done reading the boxes
  if (i + 1 < n) {
    if (lane == 0) {
      ptx::fence_proxy_async_smem();
      load_gu(tm_gu, ptx::smem_u32(gu_stage), bwd_col(ti, (int)((ord >> (4 * (i + 1))) & 15)),
              (int)F, (int)rb, gu_bar);
    }
    gu_pending = true;
  }
  float dg[32], du[32];
  // Two columns at a time in packed fp32 pairs (dp2 keeps the even- and
  // odd-column partial sums of dL/dp apart).
  const uint64_t pr2 = ptx::f2_pack(pr, pr);
  const uint64_t one2 = ptx::f2_pack(1.f, 1.f), neg_one2 = ptx::f2_pack(-1.f, -1.f);
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const float g0 = bf16_at(gc, j), g1 = bf16_at(gc, j + 1);
    const uint64_t g2 = ptx::f2_pack(g0, g1);
    const uint64_t u2 = ptx::f2_pack(bf16_at(uc, j), bf16_at(uc, j + 1));
    const uint64_t dh2 = ptx::f2_pack(__uint_as_float(dhv[j]), __uint_as_float(dhv[j + 1]));
    const uint64_t s2 = ptx::f2_pack(gemm::sigmoidf_fast(g0), gemm::sigmoidf_fast(g1));
    const uint64_t silu2 = ptx::f2_mul(g2, s2);
    const uint64_t dh_silu2 = ptx::f2_mul(dh2, silu2);
    dp2 = ptx::f2_fma(dh_silu2, u2, dp2);                    // dL/dp += dH silu(g) u
    ptx::f2_unpack(ptx::f2_mul(dh_silu2, pr2), du[j], du[j + 1]);  // dA silu(g), dA = dH p
    // silu'(g) = s (1 + g (1 - s)) = s + silu (1 - s)
    const uint64_t dsilu2 = ptx::f2_fma(silu2, ptx::f2_fma(s2, neg_one2, one2), s2);
    ptx::f2_unpack(ptx::f2_mul(ptx::f2_mul(ptx::f2_mul(dh2, pr2), u2), dsilu2), dg[j], dg[j + 1]);
  }
  // dg into columns [0, F), du into [F, 2F), both directions: the column-wise
  // blocks through the transpose, then the row-wise ones; the four code boxes
  // go out by TMA.
  if (lane == 0) ptx::bulk_wait_read_all();  // the previous chunk's boxes were read
  __syncwarp();
  uint32_t cg[8], cu[8], rg[8], ru[8];
  quant_col32(dg, cg, p.s_col, p.q_col_ld, col, rb, xs, lane);
  quant_col32(du, cu, p.s_col, p.q_col_ld, F + col, rb, xs, lane);
  const uint32_t sbg = quant32(dg, rg), sbu = quant32(du, ru);
  if (row_ok) {
    p.s_row[mx_scale_offset(grow, col >> 5, p.q_row_ld)] = (uint8_t)sbg;
    p.s_row[mx_scale_offset(grow, (F + col) >> 5, p.q_row_ld)] = (uint8_t)sbu;
  }
  __syncwarp();  // every lane has read its column out of the buffer
  stage_codes(xb, lane, rg);
  stage_codes(xb + 1024, lane, ru);
  stage_codes(xb + 2048, lane, cg);
  stage_codes(xb + 3072, lane, cu);
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    const uint32_t xb_s = ptx::smem_u32(xb);
    ptx::tma_store_2d(tm_qr, (int)col, (int)rb, xb_s);
    ptx::tma_store_2d(tm_qr, (int)(F + col), (int)rb, xb_s + 1024);
    ptx::tma_store_2d(tm_qc, (int)rb, (int)col, xb_s + 2048);
    ptx::tma_store_2d(tm_qc, (int)rb, (int)(F + col), xb_s + 3072);
    ptx::bulk_commit_group();
  }
  return true;
}

// The epilogue of one tile for this warp's 32 rows (lane = row). Fused
// epilogues split the tile's 32-column chunks between two warps per lane
// quarter by parity h; the plain ones take every chunk (h = 0, NSH = 2).
template <int MODE, int EPI>
__device__ __forceinline__ void epilogue_tile(const MxParams& p, const TileInfo& ti, bool odd,
                                              int h, const float* sh, uint32_t tl_tile, int q,
                                              int lane, float* xs, uint8_t* gu_stage,
                                              const CUtensorMap* tm_gu, const CUtensorMap* tm_qr,
                                              const CUtensorMap* tm_qc, uint32_t gu_bar,
                                              uint32_t& gu_phase, bool& gu_pending,
                                              volatile int* s_abort, int rbase) {
  // rbase: first row of this CTA's 128 rows within the group (FPROP) or of M
  // (WGRAD)
  const long long lrow = (long long)rbase + q * 32 + lane;
  const bool has_acc = ti.k_iters > 0;
  // Plain epilogues: chunk c's 32 x 32 box of this warp's rows (C row crow0 of
  // the map tm_gu, which is the output's map here) leaves from buffer c & 1.
  uint8_t* sbuf = reinterpret_cast<uint8_t*>(xs);
  auto store_box = [&](int c, const float* f, long long crow0) {
    uint8_t* box = sbuf + (c & 1) * 2048;
    if (lane == 0) ptx::bulk_wait_read_1();  // the box written two chunks ago was read
    __syncwarp();
    gemm::stage_bf16_row(box, lane, f);
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      ptx::tma_store_2d(tm_gu, ti.nt * BN + c * 32, (int)crow0, ptx::smem_u32(box));
      ptx::bulk_commit_group();
    }
  };
  if (MODE == WGRAD) {
    // C viewed as [E * M, N]: this warp's rows start at e * M + its first row
    const long long crow0 = (long long)ti.e * p.M + (lrow - lane);
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      float f[32];
      if (has_acc) {
        acc_chunk<2>(c, odd, 0, sh, tl_tile, f);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = 0.f;
      }
      store_box(c, f, crow0);
    }
    return;
  }
  const bool row_ok = lrow < ti.rows;
  const long long grow = ti.row0 + lrow;
  const long long rb = ti.row0 + (long long)rbase + q * 32;  // first row of the warp
  if (EPI == EPI_STORE) {
    // Groups hold whole 128-row blocks here, so a live warp's 32 rows all lie in
    // its group; the box store clips the N tail and rows past the end of C.
    const int ncol = p.N - ti.nt * BN;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      float f[32];
      acc_chunk<2>(c, odd, 0, sh, tl_tile, f);
      if (c * 32 < ncol) store_box(c, f, rb);
    }
  } else if (EPI == EPI_SWIGLU_FWD) {
    // Tile-local chunks 0..3 are gate, 4..7 are up, for F-columns n0 .. n0+127;
    // this warp takes the h-column chunks c = h, h + 2. The pair holding its
    // drained shared-region chunk (local chunk h of odd tiles, 6 + h of even
    // ones) goes first, outside the loop, so those registers are free after it.
    const float pr = row_ok ? p.p_rows[grow] : 0.f;
    const int c0 = odd ? h : 2 + h;
    fwd_pair(p, ti, c0, odd ? sh : nullptr, odd ? nullptr : sh, pr, row_ok, grow, rb, tl_tile,
             lane, xs, gu_stage, tm_gu, tm_qr, tm_qc);
    fwd_pair(p, ti, c0 ^ 2, nullptr, nullptr, pr, row_ok, grow, rb, tl_tile, lane, xs, gu_stage,
             tm_gu, tm_qr, tm_qc);
  } else {  // EPI_SWIGLU_BWD: accumulator = dH for F-columns nt*256 + [0, 256)
    const float pr = row_ok ? p.p_rows[grow] : 0.f;
    const int ncol = p.N - ti.nt * BN;
    uint64_t dp2 = ptx::f2_pack(0.f, 0.f);
    // This warp's chunks (parity h, inside the N tail), four bits each, the
    // one in the shared TMEM region first: it is processed from the drained
    // registers outside the loop, which frees them for the rest.
    const uint32_t ord = bwd_chunk_order(odd, h, ncol);
    const int n = (int)(ord >> 16);
    const bool first_shared = n > 0 && (int)(ord & 15) == (odd ? h : 6 + h);
    if (n > 0 && !bwd_chunk(p, ti, ord, 0, first_shared ? sh : nullptr, pr, row_ok, grow, rb,
                            tl_tile, lane, xs, gu_stage, tm_gu, tm_qr, tm_qc, gu_bar, gu_phase,
                            gu_pending, s_abort, dp2))
      return;
#pragma unroll 1
    for (int i = 1; i < n; ++i)
      if (!bwd_chunk(p, ti, ord, i, nullptr, pr, row_ok, grow, rb, tl_tile, lane, xs, gu_stage,
                     tm_gu, tm_qr, tm_qc, gu_bar, gu_phase, gu_pending, s_abort, dp2))
        return;
    float dp_even, dp_odd;
    ptx::f2_unpack(dp2, dp_even, dp_odd);
    const float dp = dp_even + dp_odd;
    // This warp's partial of dL/dp over its chunks; the two warps of a lane
    // quarter write the two halves of the tile's partial (n_part = 2 per tile).
    if (row_ok) p.dp_part[grow * p.n_part + 2 * ti.nt + h] = dp;
  }
}

template <int MODE, int EPI, int CG>
__global__ void __launch_bounds__(Cfg<EPI, CG>::kThreads, 1)
    grouped_gemm_mxf8_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmSFA,
                             const __grid_constant__ CUtensorMap tmSFB,
                             const __grid_constant__ CUtensorMap tmC,
                             const __grid_constant__ CUtensorMap tmQr,
                             const __grid_constant__ CUtensorMap tmQc, const MxParams p) {
  using L = Cfg<EPI, CG>;
  constexpr bool kPair = CG == 2;
  constexpr int kTileM = BM * CG;
  constexpr int kStageBytes = L::kStageBytes;
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
  // gate/up loads of epilogue warp w (fused kernels)
  auto gu_bar_of = [&](int w) { return bar0 + 8u * (2 * kStages + 6 + w); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kMiscOffset);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kMiscOffset + 4);
  int* s_prefix = reinterpret_cast<int*>(smem + kPrefixOffset);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = (p.N + BN - 1) / BN;
  // CTA pairs: rank 0 (the leader) issues the MMAs; tiles are dealt out per pair.
  const uint32_t rank = kPair ? ptx::cluster_ctarank() : 0u;
  const int unit = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int n_units = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) ptx::mbar_init(tfull_bar(b), 1);
    // single CTA: every epilogue thread releases a region; pair: one arrival
    // per epilogue warp of both CTAs, on the leader's barrier
    for (int r = 0; r < 3; ++r) ptx::mbar_init(region_bar(r), kPair ? 2 * L::kEpiWarps : kEpiThreads);
    ptx::mbar_init(drain_bar, 1);
    if (EPI != EPI_STORE)
      for (int w = 0; w < L::kEpiWarps; ++w) ptx::mbar_init(gu_bar_of(w), 1);
    ptx::fence_mbar_init();
    *s_abort = 0;
    int acc = 0;
    bool bad = false;
    s_prefix[0] = 0;
    int* s_offs = s_prefix + kMaxGroups + 1;
    for (int e = 0; e <= p.E; ++e) s_offs[e] = p.offsets[e];
    for (int e = 0; e < p.E; ++e) {
      int rows = s_offs[e + 1] - s_offs[e];
      if (rows % BM) bad = true;
      int mt = (MODE == FPROP) ? (rows + kTileM - 1) / kTileM : p.M / kTileM;
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
    ptx::tma_prefetch_desc(&tmSFA);
    ptx::tma_prefetch_desc(&tmSFB);
    ptx::tma_prefetch_desc(&tmC);
    if (EPI != EPI_STORE) {
      ptx::tma_prefetch_desc(&tmQr);
      ptx::tma_prefetch_desc(&tmQc);
    }
  }
  if (warp == 1) {
    if (kPair) {
      ptx::tmem_alloc_cg2(ptx::smem_u32(s_tmem), 512);
      ptx::tmem_relinquish_cg2();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(s_tmem), 512);
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
      for (int t = unit; t < total_tiles && ok; t += n_units) {
        TileInfo ti;
        decode_tile<MODE, CG>(p, s_prefix, t, e_hint, ti);
        // this CTA's 128 rows of A
        const long long a_row = (MODE == FPROP ? ti.row0 : 0LL) + (long long)ti.mt * kTileM +
                                (long long)rank * BM;
        for (int kb = 0; kb < ti.k_iters; ++kb) {
          if (!gemm::wait_bar(empty_bar(stage), phase ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          const uint32_t a_dst = sbase + stage * kStageBytes;
          const uint32_t b_dst = a_dst + kABytes;
          const uint32_t sfa_dst = sbase + kSfOffset + stage * kSfStageBytes;
          const uint32_t sfb_dst = sfa_dst + kSfaBytes;
          // Completion of both CTAs' copies of a pair is counted on the leader's barrier.
          const uint32_t fb = kPair ? ptx::mapa_shared(full_bar(stage), 0) : full_bar(stage);
          if (rank == 0) {
            ptx::mbar_arrive_expect_tx(full_bar(stage), L::kTxBytes);
            armed[stage] = true;
            armed_phase[stage] = phase;
          }
          auto load = [&](uint32_t dst, const CUtensorMap* tm, long long c0, long long c1) {
            if (kPair)
              ptx::tma_load_2d_cg2(dst, tm, (int)c0, (int)c1, fb);
            else
              ptx::tma_load_2d(dst, tm, (int)c0, (int)c1, fb);
          };
          const long long a_k = (MODE == FPROP) ? (long long)kb * BK : ti.row0 + (long long)kb * BK;
          load(a_dst, &tmA, a_k, a_row);
          // a 512-byte scale tile is one row of 128 words of the scale map
          load(sfa_dst, &tmSFA, (a_k / 128) * 128, a_row / 128);
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
            // B rows: both halves (one CTA), or this CTA's half (pair). A half
            // past the last row of B (the N tail of the last expert) reads
            // zeros, data and scales alike.
            if (!kPair || h == (int)rank) load(b_dst + (kPair ? 0 : h * (BN / 2) * BK), &tmB, b_k, b_row);
            // B scales: both halves in every CTA
            load(sfb_dst + h * 512, &tmSFB, (b_k / 128) * 128, b_row / 128);
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
    if (rank == 0 && ptx::elect_one()) {
      constexpr uint16_t kBoth = 3;  // commit to the barrier of both CTAs of a pair
      int stage = 0;
      uint32_t phase = 0;
      int e_hint = 0;
      bool ok = true;
      uint32_t uses[3] = {0, 0, 0};  // completed uses of each TMEM region
      int j = 0;                      // tiles processed by this CTA
      for (int t = unit; t < total_tiles && ok; t += n_units, ++j) {
        TileInfo ti;
        decode_tile<MODE, CG>(p, s_prefix, t, e_hint, ti);
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
          // (in each CTA of a pair, from its own shared memory)
          const uint64_t sd[3] = {ptx::smem_desc(sfa_addr, 128, 128, ptx::kSwizzleNone),
                                  ptx::smem_desc(sfb_addr, 128, 128, ptx::kSwizzleNone),
                                  ptx::smem_desc(sfb_addr + 512, 128, 128, ptx::kSwizzleNone)};
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            if (kPair)
              ptx::tmem_cp_32x128b_warpx4_cg2(tmem_base + sf_col + 4 * c, sd[c]);
            else
              ptx::tmem_cp_32x128b_warpx4(tmem_base + sf_col + 4 * c, sd[c]);
          }
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t da = ptx::smem_desc(a_addr + kk * 32, 16, 1024, ptx::kSwizzle128B);
            const uint64_t db = ptx::smem_desc(b_addr + kk * 32, 16, 1024, ptx::kSwizzle128B);
            if (kPair)
              ptx::mma_mxf8_cg2(d_tmem, da, db, ptx::idesc_mxf8(kTileM, BN, kk, kk),
                                tmem_base + sf_col, tmem_base + sf_col + 4, (kb | kk) ? 1u : 0u);
            else
              ptx::mma_mxf8(d_tmem, da, db, ptx::idesc_mxf8(BM, BN, kk, kk), tmem_base + sf_col,
                            tmem_base + sf_col + 4, (kb | kk) ? 1u : 0u);
          }
          if (kPair)
            ptx::mma_commit_cg2(empty_bar(stage), kBoth);
          else
            ptx::mma_commit(empty_bar(stage));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (ti.k_iters > 0) {
          if (kPair)
            ptx::mma_commit_cg2(tfull_bar(j & 1), kBoth);
          else
            ptx::mma_commit(tfull_bar(j & 1));
        } else {
          ptx::mbar_arrive(tfull_bar(j & 1));
          if (kPair) ptx::mbar_arrive_remote(ptx::mapa_shared(tfull_bar(j & 1), 1));
        }
      }
      if (kPair)
        ptx::mma_commit_cg2(drain_bar, 1);
      else
        ptx::mma_commit(drain_bar);
      gemm::drain_wait(drain_bar, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;   // chunk parity (fused: two warps per quarter)
    constexpr int NSH = L::kEpiWarps == 8 ? 1 : 2;  // shared chunks drained per warp
    // fused: the transpose and code boxes; plain: the two store boxes
    float* xs = reinterpret_cast<float*>(
        smem + L::kXposeOffset +
        (warp - 2) * (EPI != EPI_STORE ? kWarpBufBytes : kStoreBufBytes));
    // FC2 dgrad: the gate/up loads' own buffer; FC1: the transpose buffer
    // (its gate/up boxes are stored before the transpose reuses it)
    uint8_t* gu_stage = L::kGuBuf ? smem + L::kGuOffset + (warp - 2) * kGuBytes
                                  : reinterpret_cast<uint8_t*>(xs);
    const uint32_t gu_bar = gu_bar_of(warp - 2);
    uint32_t gu_phase = 0;
    bool gu_pending = false;  // a gate/up load of this warp is in flight
    const uint32_t tl_lanes = tmem_base + ((uint32_t)(q * 32) << 16);
    int e_hint = 0;
    int j = 0;
    // Release of a TMEM region: every thread (one CTA), or one arrival per warp
    // on the leader's barrier (pair).
    auto release = [&](int r) {
      ptx::tc_fence_before();
      if (kPair) {
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            ptx::mbar_arrive_relaxed(region_bar(r));
          else
            ptx::mbar_arrive_remote_relaxed(ptx::mapa_shared(region_bar(r), 0));
        }
      } else {
        ptx::mbar_arrive_relaxed(region_bar(r));
      }
    };
    for (int t = unit; t < total_tiles; t += n_units, ++j) {
      TileInfo ti;
      decode_tile<MODE, CG>(p, s_prefix, t, e_hint, ti);
      // This CTA's rows of the tile; in a pair the second CTA's half of the
      // last tile of a group can lie past the group (groups are padded to 128
      // rows): its accumulator is then not stored.
      const int rbase = ti.mt * kTileM + (int)rank * BM;
      const bool live = MODE == WGRAD || rbase < ti.rows;
      if (EPI == EPI_SWIGLU_BWD && live) {
        // The saved gate/up of this warp's first chunk does not depend on the
        // accumulator: fetch it while the tile's MMAs run.
        const uint32_t ord = bwd_chunk_order((j & 1) != 0, h, p.N - ti.nt * BN);
        if ((ord >> 16) > 0) {
          if (lane == 0) {
            ptx::fence_proxy_async_smem();  // after the previous tile's reads of the boxes
            load_gu(&tmC, ptx::smem_u32(gu_stage), bwd_col(ti, (int)(ord & 15)), p.F,
                    (int)(ti.row0 + (long long)rbase + q * 32), gu_bar);
          }
          gu_pending = true;
        }
      }
      if (!gemm::wait_bar(tfull_bar(j & 1), (uint32_t)((j >> 1) & 1), s_abort)) break;
      ptx::tc_fence_after();
      const bool odd = (j & 1) != 0;
      // Drain this warp's part of the shared region [192, 256) (TMEM columns
      // 192 + 32h for the fused kernels, all 64 for the plain ones) and hand
      // the region back to the MMA thread.
      float sh[32 * NSH];
      if (ti.k_iters > 0 && live) {
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
      release(1);
      if (live)
        epilogue_tile<MODE, EPI>(p, ti, odd, h, sh, tl_lanes + (odd ? (uint32_t)kAcc1Col : 0u),
                                 q, lane, xs, gu_stage, &tmC, &tmQr, &tmQc, gu_bar, gu_phase,
                                 gu_pending, s_abort, rbase);
      release(odd ? 2 : 0);
    }
    // Bulk stores must be complete, and a gate/up load left in flight by an
    // abort must have landed, before this CTA's shared memory goes away.
    if (lane == 0) {
      ptx::bulk_wait_all();
      if (EPI != EPI_STORE && gu_pending) gemm::drain_wait(gu_bar, gu_phase);
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
      ptx::tmem_dealloc_cg2(tmem_base, 512);
    else
      ptx::tmem_dealloc(tmem_base, 512);
  }
}

// Tensor maps of one launch: A and B data, their scale tiles, and the fused
// epilogues' gate/up and code maps (the plain kernels pass any map there).
struct Maps {
  CUtensorMap a, b, sfa, sfb, c, qr, qc;
};

// tiles_bound: an upper bound on the launch's 128-row tiles.
template <int MODE, int EPI, int CG = 1>
static int launch(const Maps& m, const MxParams& p_in, long long tiles_bound, cudaStream_t st) {
  MxParams p = p_in;
  p.l2_elems = kL2BandBytes;  // one-byte elements
  using L = Cfg<EPI, CG>;
  auto kern = grouped_gemm_mxf8_kernel<MODE, EPI, CG>;
  static bool attr_set = false;
  static int max_units = 0;  // co-resident CTAs (CG = 1) or CTA pairs (CG = 2)
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemAlloc) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    max_units = gemm::num_sms();
    if (CG == 2) {
      cudaLaunchConfig_t q = {};
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = 2;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      q.gridDim = dim3(2 * (gemm::num_sms() / 2));
      q.blockDim = dim3(L::kThreads);
      q.dynamicSmemBytes = L::kSmemAlloc;
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
    kern<<<(unsigned)units, L::kThreads, L::kSmemAlloc, st>>>(m.a, m.b, m.sfa, m.sfb, m.c, m.qr,
                                                              m.qc, p);
    return launch_status();
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(2 * units));
  cfg.blockDim = dim3(L::kThreads);
  cfg.dynamicSmemBytes = L::kSmemAlloc;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, m.a, m.b, m.sfa, m.sfb, m.c, m.qr, m.qc, p) != cudaSuccess)
    return MOE_ERR_CUDA;
  return launch_status();
}

// The tiled scales of an MXFP8 operand with mn rows and kdim columns as a 2-D
// tensor of 512-byte tiles: one row of (kdim/128) * 128 words per 128 rows of
// the operand, loaded a tile (128 words) at a time.
static bool scale_map(CUtensorMap* m, const void* base, long long mn, long long kdim) {
  return gemm::make_tmap(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, mn / 128, (kdim / 128) * 128,
                         (kdim / 128) * 128, 1, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
}

static bool u8_map(CUtensorMap* m, const void* base, long long rows, long long cols) {
  // K-major E4M3 operand [rows, cols], box 128 rows x 128 bytes, 128B swizzle.
  return gemm::make_tmap(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, rows, cols, cols, 128, 128);
}

// Quantised epilogue output [rows, cols] (E4M3 codes), written in 32 x 32-byte
// boxes staged with the 32-byte swizzle.
static bool code_map(CUtensorMap* m, const void* base, long long rows, long long cols) {
  return gemm::make_tmap(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, rows, cols, cols, 32, 32,
                         CU_TENSOR_MAP_SWIZZLE_32B);
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
  MX::Maps m;
  if (!MX::u8_map(&m.a, a, a_rows, a_cols) || !MX::u8_map(&m.b, b, b_rows, b_cols) ||
      !MX::scale_map(&m.sfa, sa, a_rows, a_cols) || !MX::scale_map(&m.sfb, sb, b_rows, b_cols))
    return MOE_ERR_CUDA;
  // the output, stored by TMA in 32 x 32 boxes: FPROP C [a_rows, N], WGRAD C
  // viewed as [E * M, N]
  if (!gemm::make_tmap(&m.c, C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                       mode == MOE_GEMM_FPROP ? a_rows : (long long)E * M, N, N, 32, 32,
                       CU_TENSOR_MAP_SWIZZLE_64B))
    return MOE_ERR_CUDA;
  m.qr = m.qc = m.b;  // not used by the plain epilogue
  cudaStream_t st = (cudaStream_t)stream;
  if (mode == MOE_GEMM_FPROP) {
    p.b_row_stride = b_row_stride;
    p.b_k_stride = b_k_stride;
    long long bound = (a_rows / MX::BM + E) * (long long)((N + MX::BN - 1) / MX::BN);
    return MX::launch<FPROP, EPI_STORE, 2>(m, p, bound, st);
  }
  p.c_group_stride = (long long)M * N;
  long long bound = (long long)E * (M / MX::BM) * (N / MX::BN);
  if (M % 256 == 0) return MX::launch<WGRAD, EPI_STORE, 2>(m, p, bound, st);
  return MX::launch<WGRAD, EPI_STORE>(m, p, bound, st);
}

extern "C" int moe_fc1_swiglu_mxfp8(const uint8_t* xq, const uint8_t* sx, long long rows, int H,
                                    const uint8_t* w1t, const uint8_t* sw1t,
                                    const int32_t* offsets, const float* p_rows, int E, int F,
                                    void* gu, uint8_t* hq_row, uint8_t* sh_row, uint8_t* hq_col,
                                    uint8_t* sh_col, moe_stream_t stream) {
  // The column-wise copy of H is optional (both pointers NULL: not written).
  if (!mx_ptrs_ok(xq, sx, w1t, sw1t, gu) || !offsets || !p_rows || !hq_row || !sh_row ||
      (hq_col == nullptr) != (sh_col == nullptr) || !aligned16(hq_row) || !aligned16(hq_col) ||
      E < 1 || E > MX::kMaxGroups)
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
  MX::Maps m;
  if (!MX::u8_map(&m.a, xq, rows, H) || !MX::u8_map(&m.b, w1t, 2LL * F, (long long)E * H) ||
      !MX::scale_map(&m.sfa, sx, rows, H) ||
      !MX::scale_map(&m.sfb, sw1t, 2LL * F, (long long)E * H))
    return MOE_ERR_CUDA;
  // [g | u] output, written by TMA in 32 x 32 boxes
  if (!gemm::make_tmap(&m.c, gu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, 2LL * F, 2LL * F, 32,
                       32, CU_TENSOR_MAP_SWIZZLE_NONE))
    return MOE_ERR_CUDA;
  // H codes: row-wise [rows, F], column-wise [F, rows] (the row-wise map
  // stands in when there is no column-wise copy; it is then never used)
  if (!MX::code_map(&m.qr, hq_row, rows, F) ||
      !MX::code_map(&m.qc, hq_col ? hq_col : hq_row, hq_col ? F : rows, hq_col ? rows : F))
    return MOE_ERR_CUDA;
  long long bound = (rows / MX::BM + E) * (long long)(F / 128);
  return MX::launch<FPROP, EPI_SWIGLU_FWD, 2>(m, p, bound, (cudaStream_t)stream);
}

extern "C" int moe_fc2_dgrad_swiglu_bwd_mxfp8(const uint8_t* dy2q, const uint8_t* sdy2,
                                              long long rows, int H, const uint8_t* w2q,
                                              const uint8_t* sw2, const int32_t* offsets,
                                              const float* p_rows, const void* gu, int E, int F,
                                              uint8_t* dy1q_row, uint8_t* sdy1_row,
                                              uint8_t* dy1q_col, uint8_t* sdy1_col,
                                              float* dp_part, moe_stream_t stream) {
  if (!mx_ptrs_ok(dy2q, sdy2, w2q, sw2, gu) || !offsets || !p_rows || !dy1q_row || !sdy1_row ||
      !dy1q_col || !sdy1_col || !dp_part || !aligned16(dy1q_row) || !aligned16(dy1q_col) ||
      E < 1 || E > MX::kMaxGroups)
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
  MX::Maps m;
  if (!MX::u8_map(&m.a, dy2q, rows, H) || !MX::u8_map(&m.b, w2q, (long long)E * F, H) ||
      !MX::scale_map(&m.sfa, sdy2, rows, H) || !MX::scale_map(&m.sfb, sw2, (long long)E * F, H))
    return MOE_ERR_CUDA;
  // saved [g | u], read by TMA in 32 x 32 boxes with the 64-byte swizzle
  if (!gemm::make_tmap(&m.c, gu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, 2LL * F, 2LL * F, 32,
                       32, CU_TENSOR_MAP_SWIZZLE_64B))
    return MOE_ERR_CUDA;
  // dY1 codes: row-wise [rows, 2F], column-wise [2F, rows]
  if (!MX::code_map(&m.qr, dy1q_row, rows, 2LL * F) ||
      !MX::code_map(&m.qc, dy1q_col, 2LL * F, rows))
    return MOE_ERR_CUDA;
  long long bound = (rows / MX::BM + E) * (long long)((F + MX::BN - 1) / MX::BN);
  // CTA pairs: each SM stages half of the B tile, which leaves more of the
  // shared-memory bandwidth to the epilogue's transposes and staging.
  return MX::launch<FPROP, EPI_SWIGLU_BWD, 2>(m, p, bound, (cudaStream_t)stream);
}
