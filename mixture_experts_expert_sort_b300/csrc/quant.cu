// MXFP8 quantisation, row-wise and column-wise in one pass, with an optional
// row gather that fuses the expert permute into it.
//
// "Efficient MoE Training for Biological Foundation Models", §Challenge 2
// (a scale for each block of 32 consecutive values) and §Challenge 3 (BF16
// master values quantised before each low-precision GEMM); the rule is the
// OCP Microscaling (MX) v1.0 one for E4M3 elements and E8M0 scales.
//
// A CTA of 128 threads works on tiles of 32 rows x 128 columns. Thread
// (r, b) loads its row's 32-value block straight from global memory (the
// warp reads 8 rows x 256 contiguous bytes), quantises it row-wise in
// registers and parks the values in shared memory; after one barrier thread c
// walks column c down the 32 rows for the column-wise block. The next tile's
// loads are issued before the current tile is processed. HBM-bound: 2 bytes
// read and 1 + 1/32 bytes written per element and direction.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kQRows = 32;
constexpr int kQCols = 128;
constexpr int kQThreads = 128;
constexpr int kQBand = 32;  // row tiles per band of the tile order

__device__ __forceinline__ void quant32(const float* v, uint32_t sbyte, uint4& lo, uint4& hi) {
  uint32_t wds[8];
  if (sbyte == 0xFFu) {
#pragma unroll
    for (int i = 0; i < 8; ++i) wds[i] = 0x7F7F7F7Fu;
  } else {
    float inv = mx_inv_scale(sbyte);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t a = cvt_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv);
      uint32_t b = cvt_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv);
      wds[i] = a | (b << 16);
    }
  }
  lo = make_uint4(wds[0], wds[1], wds[2], wds[3]);
  hi = make_uint4(wds[4], wds[5], wds[6], wds[7]);
}

__device__ __forceinline__ float block_amax(const float* v) {
  float m = 0.f;
  bool finite = true;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float a = fabsf(v[i]);
    finite = finite && (a <= 3.402823466e38f);  // false for Inf and NaN
    m = fmaxf(m, a);
  }
  return finite ? m : __uint_as_float(0x7F800000u);
}

// Staging tile for the column-wise pass: 32 rows of 132 floats. The row
// pass writes 16-byte vectors with the 32-column block b rotated by 8b words
// (conflict-free for 8 lanes per phase); the column pass reads one column
// per thread, 32 banks per warp.
constexpr int kQStride = 132;

__device__ __forceinline__ int qtile_col(int b, int j) { return 32 * b + ((j + 8 * b) & 31); }

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* v) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int z = 0; z < 4; ++z) {
    float2 f = __bfloat1622float2(h[z]);
    v[2 * z] = f.x;
    v[2 * z + 1] = f.y;
  }
}

// One CTA works through tiles of 32 rows x 128 columns (grid-stride). Each
// thread loads the next tile's 64 bytes of its row while it quantises the
// current one, and the gather index is fetched two tiles ahead, so loads
// stay in flight across the whole loop.
__global__ void __launch_bounds__(kQThreads)
    mxfp8_quant_kernel(const __nv_bfloat16* __restrict__ in, long long rows, int cols,
                       long long ld, const int32_t* __restrict__ src, int src_div, int dirs,
                       uint8_t* __restrict__ q_row, uint8_t* __restrict__ s_row,
                       uint8_t* __restrict__ q_col, uint8_t* __restrict__ s_col) {
  __shared__ __align__(16) float tile[kQRows * kQStride];
  const int tid = threadIdx.x;
  const int rr = tid >> 2, b = tid & 3;  // row-pass role: row rr, 32-column block b
  const long long row_tiles = rows / kQRows;
  const int col_tiles = cols / kQCols;
  const long long n_tiles = row_tiles * col_tiles;
  const long long step = gridDim.x;

  // Tile order: bands of kQBand row tiles (1024 rows); inside a band the
  // tiles run down the rows first, then across the columns. The CTAs in
  // flight then cover a few thousand columns of about a thousand rows, which
  // keeps the row reads, the row-wise writes and the column-wise writes
  // (rows of the transposed output) in long contiguous runs.
  auto tile_r0 = [&](long long t) -> long long {
    const long long band = t / (kQBand * (long long)col_tiles);
    const long long local = t - band * kQBand * (long long)col_tiles;
    const long long rows_in = min((long long)kQBand, row_tiles - band * kQBand);
    return (band * kQBand + local % rows_in) * kQRows;
  };
  auto tile_c0 = [&](long long t) -> int {
    const long long band = t / (kQBand * (long long)col_tiles);
    const long long local = t - band * kQBand * (long long)col_tiles;
    const long long rows_in = min((long long)kQBand, row_tiles - band * kQBand);
    return (int)(local / rows_in) * kQCols;
  };
  // Input row of this thread for tile t (-1: a zero row).
  auto src_row = [&](long long t) -> long long {
    const long long r = tile_r0(t) + rr;
    if (!src) return r;
    const int sv = src[r];
    return sv < 0 ? -1 : (long long)(sv / src_div);
  };
  auto load = [&](long long t, long long in_row, uint4* raw) {
    const int c0 = tile_c0(t);
    if (in_row < 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) raw[q] = make_uint4(0, 0, 0, 0);
    } else {
      const uint4* p = reinterpret_cast<const uint4*>(in + in_row * ld + c0 + 32 * b);
#pragma unroll
      for (int q = 0; q < 4; ++q) raw[q] = __ldcs(p + q);
    }
  };

  long long t = blockIdx.x;
  uint4 raw[4];
  long long row_next2 = 0;
  if (t < n_tiles) {
    load(t, src_row(t), raw);
    if (t + step < n_tiles) row_next2 = src_row(t + step);
  }
  for (; t < n_tiles; t += step) {
    const long long r0 = tile_r0(t);
    const int c0 = tile_c0(t);
    float v[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) bf16x8_to_f32(raw[q], v + 8 * q);
    // Next tile's data (row index fetched one iteration ago) and the row index
    // of the tile after it.
    if (t + step < n_tiles) {
      const long long row_next = row_next2;
      if (t + 2 * step < n_tiles) row_next2 = src_row(t + 2 * step);
      load(t + step, row_next, raw);
    }
    const long long r = r0 + rr;
    if (dirs & MOE_QUANT_ROWWISE) {
      uint32_t sb = mx_scale_byte(block_amax(v));
      uint4 lo, hi;
      quant32(v, sb, lo, hi);
      uint4* o = reinterpret_cast<uint4*>(q_row + r * cols + c0 + 32 * b);
      o[0] = lo;
      o[1] = hi;
      s_row[mx_scale_offset(r, (c0 >> 5) + b, cols)] = (uint8_t)sb;
    }
    if (dirs & MOE_QUANT_COLWISE) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        *reinterpret_cast<float4*>(&tile[rr * kQStride + qtile_col(b, 4 * k)]) =
            make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
      __syncthreads();
      const int c = tid, cb = c >> 5, cj = c & 31;
      float w[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) w[i] = tile[i * kQStride + qtile_col(cb, cj)];
      uint32_t sb = mx_scale_byte(block_amax(w));
      uint4 lo, hi;
      quant32(w, sb, lo, hi);
      uint4* o = reinterpret_cast<uint4*>(q_col + (long long)(c0 + c) * rows + r0);
      o[0] = lo;
      o[1] = hi;
      s_col[mx_scale_offset(c0 + c, r0 >> 5, rows)] = (uint8_t)sb;
      __syncthreads();
    }
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

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
  long long tiles = (rows / kQRows) * (cols / kQCols);
  long long blocks = tiles < 148 * 12 ? tiles : 148 * 12;
  mxfp8_quant_kernel<<<(unsigned)blocks, kQThreads, 0, (cudaStream_t)stream>>>(
      static_cast<const __nv_bfloat16*>(in), rows, cols, ld, src, src_div, dirs, q_row, s_row,
      q_col, s_col);
  return launch_status();
}
