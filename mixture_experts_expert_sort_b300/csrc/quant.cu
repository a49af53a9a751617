// MXFP8 quantisation, row-wise and column-wise in one pass, with an optional
// row gather that fuses the expert permute into it.
//
// "Efficient MoE Training for Biological Foundation Models", §Challenge 2
// (a scale for each block of 32 consecutive values) and §Challenge 3 (BF16
// master values quantised before each low-precision GEMM); the rule is the
// OCP Microscaling (MX) v1.0 one for E4M3 elements and E8M0 scales.
//
// A CTA of 256 threads works on tiles of 32 rows x 256 columns held in a
// ring of shared-memory tiles filled by cp.async: a row pass (one 32-value
// block per thread) and a column pass (one word column = two columns per
// thread). HBM-bound: 2 bytes read and 1 + 1/32 bytes written per element
// and direction.
#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kQRows = 32;
constexpr int kQCols = 256;      // tile width; a last tile of 128 columns is allowed
constexpr int kQThreads = 256;

// Per half, max(|a|, |b|) of two packed bf16 pairs (NaN when either is NaN);
// the sign bits of the result are not meaningful.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Per half, the largest |value| of n packed bf16 pairs, as a tree (sign bits
// cleared: non-negative bf16 order like their bit patterns, and Inf/NaN are
// the largest).
template <int N>
__device__ __forceinline__ uint32_t absmax_pairs(const uint32_t* w) {
  uint32_t t[N / 2];
#pragma unroll
  for (int i = 0; i < N / 2; ++i) t[i] = absmax_bf16x2(w[2 * i], w[2 * i + 1]);
#pragma unroll
  for (int n = N / 4; n >= 1; n /= 2)
#pragma unroll
    for (int i = 0; i < n; ++i) t[i] = absmax_bf16x2(t[2 * i], t[2 * i + 1]);
  return t[0] & 0x7FFF7FFFu;
}

// Largest |value| of 32 bf16 (16 packed words) as bf16 bits.
__device__ __forceinline__ uint32_t amax_bf16x32(const uint32_t* w) {
  const uint32_t m = absmax_pairs<16>(w);
  return max(m >> 16, m & 0xFFFFu);
}

__device__ __forceinline__ uint32_t scale_of_bf16_amax(uint32_t abits) {
  return abits >= 0x7F80u ? 0xFFu : mx_scale_byte(__uint_as_float(abits << 16));
}

// E4M3 codes of the four bf16 values in words a, b (low half first), each
// scaled by the power of two in both halves of inv2 (exact), as one word.
__device__ __forceinline__ uint32_t codes4(uint32_t a, uint32_t b, uint64_t inv2) {
  float a0, a1, b0, b1;
  ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(a << 16),
                                          __uint_as_float(a & 0xFFFF0000u)), inv2), a0, a1);
  ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(b << 16),
                                          __uint_as_float(b & 0xFFFF0000u)), inv2), b0, b1);
  return (uint32_t)cvt_e4m3x2(a0, a1) | ((uint32_t)cvt_e4m3x2(b0, b1) << 16);
}

// E4M3 codes of 32 bf16 values (packed pairs in w) with scale byte sb.
// half: 0 = each word's low element only, 1 = high only, 2 = both (32 values
// from 16 words). Writes 8 words of codes.
__device__ __forceinline__ void codes_of(const uint32_t* w, uint32_t sb, uint32_t* out) {
  if (sb == 0xFFu) {
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = 0x7F7F7F7Fu;
    return;
  }
  const float inv = mx_inv_scale(sb);
  const uint64_t inv2 = ptx::f2_pack(inv, inv);
#pragma unroll
  for (int i = 0; i < 8; ++i) out[i] = codes4(w[2 * i], w[2 * i + 1], inv2);
}

// Shared-memory tile: 32 rows x 256 bf16 (512 bytes per row); 16-byte chunk
// j of row r sits at chunk j ^ ((j >> 3) & 7) ^ (4 * ((r >> 4) & 1)), which
// makes the row pass's 16-byte accesses (8 lanes = 8 blocks of one row per
// phase) and the column pass's 4-byte reads (16 adjacent words from rows r
// and r + 16 per warp) conflict-free.
__device__ __forceinline__ int qchunk(int j, int row) {
  return j ^ ((j >> 3) & 7) ^ (((row >> 4) & 1) << 2);
}

// E4M3 codes of 16 bf16 values (8 packed words) with scale byte sb: 4 words.
__device__ __forceinline__ void codes_of16(const uint32_t* w, uint32_t sb, uint32_t* out) {
  if (sb == 0xFFu) {
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = 0x7F7F7F7Fu;
    return;
  }
  const float inv = mx_inv_scale(sb);
  const uint64_t inv2 = ptx::f2_pack(inv, inv);
#pragma unroll
  for (int i = 0; i < 4; ++i) out[i] = codes4(w[2 * i], w[2 * i + 1], inv2);
}

constexpr int kQStages = 4;  // tiles in the shared-memory ring
constexpr int kQTileWords = kQRows * 128;
constexpr int kQSmemBytes = kQStages * kQTileWords * 4;

__device__ __forceinline__ void cp_async_16z(uint32_t dst, const void* src, bool valid) {
  // zero-fills the 16 bytes when !valid (source size 0)
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(valid ? 16 : 0)
               : "memory");
}

// The tiles of 32 rows x 256 columns are dealt out in work items: an item is
// a run of `chunk` consecutive row tiles of one 256-column strip, and items
// are numbered with the strip fastest, so the CTAs in flight cover all the
// strips of a few row ranges (complete lines of the row-wise output) and each
// CTA writes runs of chunk x 32 bytes of every column of its strip (the
// column-wise output). CTA i takes items i, i + gridDim.x, ...; inside an item
// the next tile is one row tile down, so only the first tile of an item needs
// an integer division.
// A ring of kQStages tiles in shared memory: each thread copies its own 64
// bytes (row rr, 32-column block b) of the tile kQStages-1 steps ahead with
// cp.async straight into the swizzled layout, so three tiles are in flight
// per CTA without holding registers. Row pass: thread (rr, b) quantises its
// block row-wise. Column pass: thread c owns the word column c (columns 2c
// and 2c+1) and quantises both 32-row column blocks. Amax is taken on packed
// bf16 halves with an integer max.
struct QCursor {
  int item;    // work item (n_items or more: past the end)
  int rt, ct;  // row tile and column strip of the tile
  int rt_end;  // end of the item's row tiles
};

__global__ void __launch_bounds__(kQThreads)
    mxfp8_quant_kernel(const __nv_bfloat16* __restrict__ in, long long rows, int cols,
                       long long ld, const int32_t* __restrict__ src, int src_div, int dirs,
                       uint8_t* __restrict__ q_row, uint8_t* __restrict__ s_row,
                       uint8_t* __restrict__ q_col, uint8_t* __restrict__ s_col, int chunk) {
  extern __shared__ __align__(16) uint32_t qsm[];  // [kQStages][32 rows x 128 words]
  const int tid = threadIdx.x;
  const int rr = tid >> 3, b = tid & 7;  // row pass: row rr, 32-column block b
  // Tile counts fit in 32 bits (checked on the host).
  const int row_tiles = (int)(rows / kQRows);
  const int col_tiles = (cols + kQCols - 1) / kQCols;
  const int n_items = ((row_tiles + chunk - 1) / chunk) * col_tiles;
  const int step = gridDim.x;

  auto start = [&](QCursor& c, int item) {
    c.item = item;
    if (item < n_items) {
      const int ch = item / col_tiles;
      c.ct = item - ch * col_tiles;
      c.rt = ch * chunk;
      c.rt_end = min(c.rt + chunk, row_tiles);
    }
  };
  auto advance = [&](QCursor& c) {
    if (++c.rt >= c.rt_end) start(c, c.item + step);
  };
  // Input row of this thread for the cursor's tile (-1: a zero row).
  auto src_row = [&](const QCursor& c) -> long long {
    const long long r = (long long)c.rt * kQRows + rr;
    if (!src) return r;
    const int sv = src[r];
    return sv < 0 ? -1 : (long long)(sv / src_div);
  };
  // Copy this thread's 64 bytes of the cursor's tile (input row in_row) into ring slot s.
  auto issue = [&](const QCursor& c, long long in_row, int s) {
    const int col = c.ct * kQCols + 32 * b;
    const bool ok = in_row >= 0 && col < cols;
    const __nv_bfloat16* g = ok ? in + in_row * ld + col : in;
    const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(qsm + s * kQTileWords + rr * 128));
#pragma unroll
    for (int q = 0; q < 4; ++q) cp_async_16z(base + 16 * qchunk(4 * b + q, rr), g + 8 * q, ok);
  };

  // Prologue: the first kQStages-1 tiles of this CTA, and the row index of the next.
  QCursor cur, ahead;
  start(cur, blockIdx.x);
  ahead = cur;
#pragma unroll
  for (int s = 0; s < kQStages - 1; ++s) {
    if (ahead.item < n_items) {
      issue(ahead, src_row(ahead), s);
      advance(ahead);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  long long row_ahead = ahead.item < n_items ? src_row(ahead) : 0;

  int slot = 0;
  while (cur.item < n_items) {
    // Issue the tile kQStages-1 steps ahead into the slot freed last iteration.
    if (ahead.item < n_items) {
      issue(ahead, row_ahead, (slot + kQStages - 1) % kQStages);
      advance(ahead);
      if (ahead.item < n_items) row_ahead = src_row(ahead);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group %0;" ::"n"(kQStages - 1) : "memory");
    __syncthreads();  // tile `cur` is complete in slot `slot` for all threads
    const uint32_t* tile = qsm + slot * kQTileWords;
    const long long r0 = (long long)cur.rt * kQRows;
    const int c0 = cur.ct * kQCols;
    const int ncol = min(kQCols, cols - c0);  // 256, or 128 for a last half tile
    if ((dirs & MOE_QUANT_ROWWISE) && 32 * b < ncol) {
      uint32_t w[16];
      const uint4* row = reinterpret_cast<const uint4*>(tile + rr * 128);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = row[qchunk(4 * b + q, rr)];
        w[4 * q] = u.x;
        w[4 * q + 1] = u.y;
        w[4 * q + 2] = u.z;
        w[4 * q + 3] = u.w;
      }
      const long long r = r0 + rr;
      const uint32_t sb = scale_of_bf16_amax(amax_bf16x32(w));
      uint32_t o[8];
      codes_of(w, sb, o);
      uint4* dst = reinterpret_cast<uint4*>(q_row + r * cols + c0 + 32 * b);
      dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
      s_row[mx_scale_offset(r, (c0 >> 5) + b, cols)] = (uint8_t)sb;
    }
    if (dirs & MOE_QUANT_COLWISE) {
      // Lane pair (2c, 2c+1) owns word column c (columns 2c and 2c+1); each
      // lane of the pair takes 16 of the 32 rows and the pair combines its
      // maxima with one shuffle.
      const int c = tid >> 1, half = tid & 1;
      if (2 * c < ncol) {
        uint32_t col[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = 16 * half + i;
          col[i] = tile[r * 128 + 4 * qchunk(c >> 2, r) + (c & 3)];
        }
        uint32_t m = absmax_pairs<16>(col);
        m = __vmaxu2(m, __shfl_xor_sync(0xffffffffu, m, 1));
        const uint32_t sb0 = scale_of_bf16_amax(m & 0xFFFFu), sb1 = scale_of_bf16_amax(m >> 16);
        uint32_t lo[8], hi[8], o[4];
        // repack: column 2c = low halves, column 2c+1 = high halves
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          lo[i] = (col[2 * i] & 0xFFFFu) | (col[2 * i + 1] << 16);
          hi[i] = (col[2 * i] >> 16) | (col[2 * i + 1] & 0xFFFF0000u);
        }
        const long long rb = r0 + 16 * half;
        codes_of16(lo, sb0, o);
        *reinterpret_cast<uint4*>(q_col + (long long)(c0 + 2 * c) * rows + rb) =
            make_uint4(o[0], o[1], o[2], o[3]);
        codes_of16(hi, sb1, o);
        *reinterpret_cast<uint4*>(q_col + (long long)(c0 + 2 * c + 1) * rows + rb) =
            make_uint4(o[0], o[1], o[2], o[3]);
        if (half == 0) s_col[mx_scale_offset(c0 + 2 * c, r0 >> 5, rows)] = (uint8_t)sb0;
        else s_col[mx_scale_offset(c0 + 2 * c + 1, r0 >> 5, rows)] = (uint8_t)sb1;
      }
    }
    __syncthreads();  // slot is reused by the copies issued next iteration
    slot = (slot + 1) % kQStages;
    advance(cur);
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Tiled scales -> row-major [mn, kdim/32]. The four scales of row r and
// 32-column blocks 4j .. 4j+3 are one aligned 32-bit word in both layouts, so
// each thread moves one word: tiled word (tile (r/128, j), lane r % 32,
// quarter (r % 128) / 32) to row-major word r * (kdim/128) + j. Consecutive
// threads take consecutive output words (coalesced stores; the loads of a
// warp fall in one or two 512-byte tiles).
__global__ void __launch_bounds__(256)
    mx_scales_canonical_kernel(const uint32_t* __restrict__ tiled, long long mn, int kt,
                               uint32_t* __restrict__ canon) {
  const long long words = mn * kt;
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < words; i += gridDim.x * 256LL) {
    const long long r = i / kt;
    const int j = (int)(i - r * kt);
    const int rr = (int)(r & 127);
    canon[i] = tiled[((r >> 7) * kt + j) * 128 + (rr & 31) * 4 + (rr >> 5)];
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int mxfp8_scales_to_canonical(const uint8_t* tiled, long long mn, int kdim,
                                         uint8_t* canon, moe_stream_t stream) {
  if (mn < 0 || mn % 128 || kdim <= 0 || kdim % 128 || mn >= (1LL << 40)) return MOE_ERR_ARG;
  if (mn == 0) return MOE_OK;
  if (!tiled || !canon || (reinterpret_cast<uintptr_t>(tiled) & 3u) ||
      (reinterpret_cast<uintptr_t>(canon) & 3u))
    return MOE_ERR_ARG;
  const long long bytes = mn * (kdim / 32);
  const uintptr_t a = reinterpret_cast<uintptr_t>(tiled), c = reinterpret_cast<uintptr_t>(canon);
  if (a < c + (uintptr_t)bytes && c < a + (uintptr_t)bytes) return MOE_ERR_ARG;  // overlap
  const long long words = bytes / 4;
  long long blocks = (words + 255) / 256;
  if (blocks > 148 * 8) blocks = 148 * 8;
  mx_scales_canonical_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(
      reinterpret_cast<const uint32_t*>(tiled), mn, kdim / 128, reinterpret_cast<uint32_t*>(canon));
  return launch_status();
}

extern "C" int mxfp8_quantize(const void* in, long long rows, int cols, long long ld,
                              const int32_t* src, int src_div, int dirs, uint8_t* q_row,
                              uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                              moe_stream_t stream) {
  if (rows < 0 || rows % 128 || cols <= 0 || cols % 128 || ld < cols || ld % 8) return MOE_ERR_ARG;
  if (dirs < 1 || dirs > 3 || (src && src_div < 1)) return MOE_ERR_ARG;
  if (rows == 0) return MOE_OK;
  if (!in || !aligned16(in)) return MOE_ERR_ARG;
  if ((dirs & MOE_QUANT_ROWWISE) && (!q_row || !s_row || !aligned16(q_row))) return MOE_ERR_ARG;
  if ((dirs & MOE_QUANT_COLWISE) && (!q_col || !s_col || !aligned16(q_col))) return MOE_ERR_ARG;
  const long long row_tiles = rows / kQRows, col_tiles = (cols + kQCols - 1) / kQCols;
  const long long tiles = row_tiles * col_tiles;
  if (tiles >= (1LL << 31) - 148LL * 3 * 4) return MOE_ERR_UNSUPPORTED;
  const long long ctas = 148 * 3;  // 3 CTAs (192 KB of ring) per SM
  // Row tiles per work item: up to 8 (a 256-byte run of each column-wise
  // output row), and about 32 items per CTA or more, so that the CTAs left
  // with one item more than the others idle the rest for 3% of the time at most.
  long long chunk = tiles / (32 * ctas);
  chunk = chunk < 1 ? 1 : chunk > 8 ? 8 : chunk;
  const long long items = ((row_tiles + chunk - 1) / chunk) * col_tiles;
  long long blocks = items < ctas ? items : ctas;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(mxfp8_quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kQSmemBytes) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr_set = true;
  }
  mxfp8_quant_kernel<<<(unsigned)blocks, kQThreads, kQSmemBytes, (cudaStream_t)stream>>>(
      static_cast<const __nv_bfloat16*>(in), rows, cols, ld, src, src_div, dirs, q_row, s_row,
      q_col, s_col, (int)chunk);
  return launch_status();
}
