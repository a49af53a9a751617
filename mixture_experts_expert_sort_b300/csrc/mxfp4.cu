// MXFP4 activation compression: direct FP8 <-> FP4 conversion and the
// scale-aware FP4 row-wise -> column-wise conversion.
//
// The hgpu.org abstract on MXFP4 training of MoE models on Hopper keeps
// activations in MXFP4 while the GEMMs run in FP8: FP8 values go to FP4 and
// back without a BF16 round trip, and the column-wise FP4 copy (the operand
// of a weight-gradient GEMM) is derived from the row-wise one with new block
// scales. Formats per OCP Microscaling v1.0: 32-element blocks with an E8M0
// scale 2^(floor(log2 amax) - emax_elem); E2M1 elements (emax 2, magnitudes
// 0, 0.5, 1, 1.5, 2, 3, 4, 6) and E4M3 elements (emax 8) round to nearest
// even and saturate.
//
// Every conversion decodes exactly (E4M3, E2M1 and the scales are all exact
// in fp32 and half) and applies the output format's rule, so it equals
// quantising the decoded values. Their bytes make them memory-bound work;
// in practice the row-wise conversions run at 50-60% of the copy bandwidth and
// the row -> column one is limited by integer issue (about 16 instructions
// per element).
#include "common.cuh"

namespace moe {
namespace {

// E8M0 byte of an MXFP4 block maximum: e = clamp(floor(log2 amax) - 2, -127, 127)
// from the float exponent field (a zero or subnormal amax gives e <= -129).
__device__ __forceinline__ uint32_t mx4_scale_byte(float amax) {
  const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFF);
  if (ef == 0xFF) return 0xFFu;
  const int e = ef - 127 - 2;
  return (uint32_t)((e < -127 ? -127 : e) + 127);
}

// 2^(s - 127) and 2^(127 - s) for a finite scale byte s, exactly (2^-127 is
// the float subnormal 0x00400000).
__device__ __forceinline__ float e8m0_value(uint32_t s) {
  return s == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(s << 23);
}
__device__ __forceinline__ float e8m0_inverse(uint32_t s) {
  const int f = 254 - (int)s;
  return f > 0 ? __uint_as_float((uint32_t)f << 23) : __uint_as_float(0x00400000u);
}

// Magnitude of E2M1 code m (0..7) with the sign of bit 3: 0, .5, 1, 1.5, 2, 3, 4, 6.
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const uint32_t m = c & 7u;
  const uint32_t mag = m >= 2 ? (((m >> 1) + 126u) << 23) | ((m & 1u) << 22)
                              : (m ? 0x3F000000u : 0u);
  return __uint_as_float(mag | ((c & 8u) << 28));
}

// Two floats -> one byte of two E2M1 codes (round to nearest even, saturate
// to +-6), hardware conversion; `lo` goes to the low nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Four E4M3 bytes -> four floats, exactly (via half).
__device__ __forceinline__ void e4m3x4_to_float(uint32_t w, float* f) {
  uint32_t h01, h23;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"((uint16_t)(w & 0xFFFFu)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"((uint16_t)(w >> 16)));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h01));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h23));
  f[0] = a.x, f[1] = a.y, f[2] = b.x, f[3] = b.y;
}

// True when any of the four E4M3 bytes is a NaN code (0x7F / 0xFF).
__device__ __forceinline__ bool e4m3x4_has_nan(uint32_t w) {
  return __vcmpeq4(w & 0x7F7F7F7Fu, 0x7F7F7F7Fu) != 0;
}

// ---------------------------------------------- FP4 -> FP8 in integer arithmetic
// For an MXFP4 block with scale byte s4 whose largest magnitude code is
// m_max > 0, the largest value is E2M1(m_max) 2^(s4-127) with
// floor(log2) = fl + s4 - 127, fl = (m_max >> 1) - 1; the MXFP8 rule gives
// s8 = max(fl + s4 - 8, 0) (the exponent clamps at -127, never at 127), and
// every element E2M1(m) 2^(s4-127) is E2M1(m) 2^k 2^(s8-127) with
// k = s4 - s8 in [0, 9], an E4M3 value: byte 0 for m = 0, (k + 6) << 3 for
// m = 1 (0.5 2^k), and (((m >> 1) + k + 6) << 3) | ((m & 1) << 2) for m >= 2.
// These eight bytes form a table (two registers) that one prmt reads for
// four codes at once; a second prmt supplies the sign bytes.
struct Fp8Table {
  uint32_t lo, hi;
};
__device__ __forceinline__ uint32_t mx4_max_mag(const uint32_t* w, int n) {
  uint32_t m = 0;
  for (int i = 0; i < n; ++i) m = __vmaxu4(m, __vmaxu4(w[i] & 0x07070707u, (w[i] >> 4) & 0x07070707u));
  m = __vmaxu4(m, m >> 16);  // byte-wise: bytes 0, 1 now hold the maxima of pairs
  return __vmaxu4(m, m >> 8) & 0xFFu;
}
// s8 byte and the byte table for a finite block (s4 < 0xFF)
__device__ __forceinline__ uint32_t fp8_table(uint32_t mmax, uint32_t s4, Fp8Table& t) {
  if (mmax == 0) {
    t.lo = t.hi = 0;
    return 0;
  }
  const int fl = (int)(mmax >> 1) - 1;
  const int s8 = max(fl + (int)s4 - 8, 0);
  const uint32_t base = (uint32_t)((int)s4 - s8 + 6) << 3;  // (k + 6) << 3
  t.lo = base * 0x01010100u + 0x0C080000u;                    // 0, base, base+8, base+12
  t.hi = base * 0x01010101u + 0x1C181410u;                    // base+16 .. base+28
  return (uint32_t)s8;
}
// Eight E2M1 codes (one word) -> eight E4M3 bytes (two words).
__device__ __forceinline__ void fp8_from_codes8(uint32_t w, const Fp8Table& t, uint32_t& b0,
                                                uint32_t& b1) {
  b0 = __byte_perm(t.lo, t.hi, w & 0x7777u) | __byte_perm(0u, 0x80808080u, (w & 0x8888u) >> 1);
  const uint32_t u = w >> 16;
  b1 = __byte_perm(t.lo, t.hi, u & 0x7777u) | __byte_perm(0u, 0x80808080u, (u & 0x8888u) >> 1);
}

// ------------------------------------------------------------ row-wise conversions
// One thread per 32-element block of a row; consecutive threads take
// consecutive blocks, so a warp reads 1 KB (FP8) or 512 B (FP4) contiguously.

__global__ void __launch_bounds__(256)
    mxfp4_from_mxfp8_kernel(const uint8_t* __restrict__ q8, const uint8_t* __restrict__ s8,
                            long long rows, int cols, uint8_t* __restrict__ q4,
                            uint8_t* __restrict__ s4) {
  const int kbs = cols / 32;
  const long long n = rows * kbs;
  const long long stride = (long long)gridDim.x * blockDim.x;
  // the next block's bytes are loaded while this one is converted
  uint4 na = make_uint4(0, 0, 0, 0), nb = na;
  uint32_t ns = 0;
  auto load = [&](long long i) {
    const long long r = i / kbs;
    const int kb = (int)(i - r * kbs);
    const uint4* src = reinterpret_cast<const uint4*>(q8 + r * cols + 32 * kb);
    na = __ldcs(src), nb = __ldcs(src + 1);
    ns = s8[mx_scale_offset(r, kb, cols)];
  };
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) load(i);
  for (; i < n; i += stride) {
    const long long r = i / kbs;
    const int kb = (int)(i - r * kbs);
    const uint4 a = na, b = nb;
    const uint32_t sin = ns;
    if (i + stride < n) load(i + stride);
    const long long so = mx_scale_offset(r, kb, cols);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    bool nan = sin == 0xFFu;
#pragma unroll
    for (int q = 0; q < 8; ++q) nan |= e4m3x4_has_nan(w[q]);
    uint4 out = make_uint4(0, 0, 0, 0);
    uint32_t sout = 0xFFu;
    if (!nan) {
      // largest magnitude code (E4M3 magnitudes order like their 7-bit codes)
      uint32_t m = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) m = __vmaxu4(m, w[q] & 0x7F7F7F7Fu);
      m = __vmaxu4(m, m >> 16);
      m = __vmaxu4(m, m >> 8) & 0xFFu;
      // floor(log2) of E4M3(m): exponent field - 7, or floor(log2 mant) - 9 when subnormal
      const int ef = (int)(m >> 3);
      const int flc = ef ? ef - 7 : 31 - __clz((int)(m & 7u)) - 9;
      int e4 = m ? flc + (int)sin - 127 - 2 : -127;
      e4 = max(-127, min(127, e4));
      sout = (uint32_t)(e4 + 127);
      // element = E4M3 value * 2^(s8 - 127 - e4): one exact power of two
      // (an all-zero block has nothing to scale; its exponent field could overflow)
      const float mul = m ? __uint_as_float((uint32_t)((int)sin - e4) << 23) : 1.0f;
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float f0[4], f1[4];
        e4m3x4_to_float(w[2 * q], f0);
        e4m3x4_to_float(w[2 * q + 1], f1);
        o[q] = cvt_e2m1x2(f0[0] * mul, f0[1] * mul) | (cvt_e2m1x2(f0[2] * mul, f0[3] * mul) << 8) |
               (cvt_e2m1x2(f1[0] * mul, f1[1] * mul) << 16) |
               (cvt_e2m1x2(f1[2] * mul, f1[3] * mul) << 24);
      }
      out = make_uint4(o[0], o[1], o[2], o[3]);
    }
    __stcs(reinterpret_cast<uint4*>(q4 + r * (cols / 2) + 16 * kb), out);
    s4[so] = (uint8_t)sout;
  }
}

__global__ void __launch_bounds__(256)
    mxfp8_from_mxfp4_kernel(const uint8_t* __restrict__ q4, const uint8_t* __restrict__ s4,
                            long long rows, int cols, uint8_t* __restrict__ q8,
                            uint8_t* __restrict__ s8) {
  const int kbs = cols / 32;
  const long long n = rows * kbs;
  const long long stride = (long long)gridDim.x * blockDim.x;
  // the next block's bytes are loaded while this one is converted
  uint4 na = make_uint4(0, 0, 0, 0);
  uint32_t ns = 0;
  auto load = [&](long long i) {
    const long long r = i / kbs;
    const int kb = (int)(i - r * kbs);
    na = __ldcs(reinterpret_cast<const uint4*>(q4 + r * (cols / 2) + 16 * kb));
    ns = s4[mx_scale_offset(r, kb, cols)];
  };
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) load(i);
  for (; i < n; i += stride) {
    const long long r = i / kbs;
    const int kb = (int)(i - r * kbs);
    const uint4 a = na;
    const uint32_t sin = ns;
    if (i + stride < n) load(i + stride);
    const long long so = mx_scale_offset(r, kb, cols);
    uint4 o0 = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu), o1 = o0;
    uint32_t sout = 0xFFu;
    if (sin != 0xFFu) {
      const uint32_t w[4] = {a.x, a.y, a.z, a.w};
      Fp8Table t;
      sout = fp8_table(mx4_max_mag(w, 4), sin, t);
      fp8_from_codes8(w[0], t, o0.x, o0.y);
      fp8_from_codes8(w[1], t, o0.z, o0.w);
      fp8_from_codes8(w[2], t, o1.x, o1.y);
      fp8_from_codes8(w[3], t, o1.z, o1.w);
    }
    uint4* dst = reinterpret_cast<uint4*>(q8 + r * cols + 32 * kb);
    __stcs(dst, o0);
    __stcs(dst + 1, o1);
    s8[so] = (uint8_t)sout;
  }
}

// ------------------------------------------------------------ row -> column
// CTA: tiles of 128 rows x 128 columns (grid-stride) through a ring of
// kRCStages tiles in shared memory, filled by cp.async: the packed codes
// (128 rows x 64 bytes, two 16-byte chunks per thread) and the 512-byte
// scale tile holding exactly the tile's row-block scales. Each tile's scales
// are turned into floats once (NaN for 0xFF); each thread then takes one
// byte column (columns 2b and 2b + 1) of one 32-row block, decodes the two
// codes of every byte through a 16-entry table, quantises both columns as
// column blocks and writes 16 (FP4) or 32 (FP8) bytes of the transposed
// output for each; the four row blocks of a column write adjacent bytes.
// About 16 instructions per element, mostly integer (nibble extraction, block
// maxima, E2M1 packing): the ALU pipe, not DRAM, sets the speed.
constexpr int kRCRows = 128, kRCCols = 128, kRCStages = 3;
constexpr int kRCDataBytes = kRCRows * (kRCCols / 2);
constexpr int kRCTileBytes = kRCDataBytes + 512;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d),
               "l"(reinterpret_cast<uint64_t>(gmem))
               : "memory");
}

// 32 values (all finite) -> 16 bytes of E2M1 codes; returns the scale byte.
__device__ __forceinline__ uint32_t encode_e2m1_col(const float* v, float amax, uint4& out) {
  const uint32_t s = mx4_scale_byte(amax);
  const float inv = e8m0_inverse(s);
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t b0 = cvt_e2m1x2(v[8 * q] * inv, v[8 * q + 1] * inv);
    const uint32_t b1 = cvt_e2m1x2(v[8 * q + 2] * inv, v[8 * q + 3] * inv);
    const uint32_t b2 = cvt_e2m1x2(v[8 * q + 4] * inv, v[8 * q + 5] * inv);
    const uint32_t b3 = cvt_e2m1x2(v[8 * q + 6] * inv, v[8 * q + 7] * inv);
    w[q] = __byte_perm(b0 | (b1 << 8), b2 | (b3 << 8), 0x5410);
  }
  out = make_uint4(w[0], w[1], w[2], w[3]);
  return s;
}

template <bool TO_FP8>
__device__ __forceinline__ void store_col_block(const float* v, float amax, bool nan,
                                                uint8_t* __restrict__ qc, uint8_t* __restrict__ sc,
                                                long long rows, long long col, long long rb) {
  const long long so = mx_scale_offset(col, rb >> 5, rows);
  uint4 o4 = make_uint4(0, 0, 0, 0);
  uint32_t s4out = 0xFFu;
  if (!nan) s4out = encode_e2m1_col(v, amax, o4);
  if (!TO_FP8) {
    __stcs(reinterpret_cast<uint4*>(qc + col * (rows / 2) + (rb >> 1)), o4);
    sc[so] = (uint8_t)s4out;
  } else {
    uint4 o0 = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu), o1 = o0;
    uint32_t s8out = 0xFFu;
    if (!nan) {  // the FP4 column block to MXFP8 (lossless)
      const uint32_t w[4] = {o4.x, o4.y, o4.z, o4.w};
      Fp8Table tb;
      s8out = fp8_table(mx4_max_mag(w, 4), s4out, tb);
      fp8_from_codes8(w[0], tb, o0.x, o0.y);
      fp8_from_codes8(w[1], tb, o0.z, o0.w);
      fp8_from_codes8(w[2], tb, o1.x, o1.y);
      fp8_from_codes8(w[3], tb, o1.z, o1.w);
    }
    uint4* dst = reinterpret_cast<uint4*>(qc + col * rows + rb);
    __stcs(dst, o0);
    __stcs(dst + 1, o1);
    sc[so] = (uint8_t)s8out;
  }
}

template <bool TO_FP8>
__global__ void __launch_bounds__(256, 2)
    mxfp4_row_to_col_kernel(const uint8_t* __restrict__ q4, const uint8_t* __restrict__ s4,
                            long long rows, int cols, uint8_t* __restrict__ qc,
                            uint8_t* __restrict__ sc) {
  __shared__ __align__(16) uint8_t ring[kRCStages][kRCTileBytes];
  __shared__ float sf[kRCRows][4];  // row-block scales of the current tile as floats
  __shared__ float tab[16];         // E2M1 code -> value
  const int tid = threadIdx.x;
  if (tid < 16) tab[tid] = e2m1_value((uint32_t)tid);
  const int col_tiles = cols / kRCCols;
  const long long n_tiles = (rows / kRCRows) * col_tiles;
  const long long step = gridDim.x;
  auto issue = [&](long long t, int slot) {
    if (t < n_tiles) {
      const long long rt = t / col_tiles;
      const int ct = (int)(t - rt * col_tiles);
      const uint8_t* src = q4 + rt * kRCRows * (cols / 2) + ct * (kRCCols / 2);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int chunk = tid + 256 * j;  // row chunk >> 2, 16-byte piece chunk & 3
        cp_async16(&ring[slot][chunk * 16], src + (long long)(chunk >> 2) * (cols / 2) + 16 * (chunk & 3));
      }
      if (tid < 32)  // the scale tile (row tile rt, k tile ct)
        cp_async16(&ring[slot][kRCDataBytes + tid * 16], s4 + (rt * col_tiles + ct) * 512 + tid * 16);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
#pragma unroll
  for (int i = 0; i < kRCStages - 1; ++i) issue(blockIdx.x + i * step, i);
  int slot = 0;
  const int bc = tid & 63, h = tid >> 6;  // byte column (columns 2bc, 2bc+1), row block
  for (long long t = blockIdx.x; t < n_tiles; t += step) {
    issue(t + (kRCStages - 1) * step, (slot + kRCStages - 1) % kRCStages);
    asm volatile("cp.async.wait_group %0;" ::"n"(kRCStages - 1) : "memory");
    __syncthreads();  // tile t landed (and tab is written)
    {
      // scale of (row 32a + b, block c) is byte 16b + 4a + c of the scale tile
      const uint8_t* st = ring[slot] + kRCDataBytes;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int e = tid + 256 * j;  // e = 16 b + 4 a + c
        const uint32_t sv = st[e];
        sf[32 * ((e >> 2) & 3) + (e >> 4)][e & 3] =
            sv == 0xFFu ? __uint_as_float(0x7FC00000u) : e8m0_value(sv);
      }
    }
    __syncthreads();
    const uint8_t* data = ring[slot] + (32 * h) * (kRCCols / 2) + bc;
    const int blk = bc >> 4;  // 32-column block of columns 2bc, 2bc+1
    float v0[32], v1[32];
    float m0 = 0.f, m1 = 0.f;
    bool nan = false;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint32_t byte = data[i * (kRCCols / 2)];
      const float s = sf[32 * h + i][blk];
      nan |= s != s;
      v0[i] = tab[byte & 15u] * s;
      v1[i] = tab[byte >> 4] * s;
      m0 = fmaxf(m0, fabsf(v0[i]));
      m1 = fmaxf(m1, fabsf(v1[i]));
    }
    __syncthreads();  // the slot and sf are rewritten next iteration
    const long long rt = t / col_tiles;
    const long long col = (t - rt * col_tiles) * kRCCols + 2 * bc;
    const long long rb = rt * kRCRows + 32 * h;  // first row of these column blocks
    store_col_block<TO_FP8>(v0, m0, nan, qc, sc, rows, col, rb);
    store_col_block<TO_FP8>(v1, m1, nan, qc, sc, rows, col + 1, rb);
    slot = (slot + 1) % kRCStages;
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

int check_mx4_args(const void* a, const void* sa, long long rows, int cols, const void* b,
                   const void* sb) {
  if (rows <= 0 || rows % 128 || cols <= 0 || cols % 128) return MOE_ERR_ARG;
  if (!a || !sa || !b || !sb || !aligned16(a) || !aligned16(b)) return MOE_ERR_ARG;
  if (rows * (long long)cols >= (1LL << 40)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

unsigned row_blocks_grid(long long rows, int cols) {
  const long long n = rows * (cols / 32);
  long long g = (n + 255) / 256;
  return (unsigned)(g < 148 * 8 ? g : 148 * 8);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int mxfp4_from_mxfp8(const uint8_t* q8, const uint8_t* s8, long long rows, int cols,
                                uint8_t* q4, uint8_t* s4, moe_stream_t stream) {
  const int rc = check_mx4_args(q8, s8, rows, cols, q4, s4);
  if (rc != MOE_OK) return rc;
  mxfp4_from_mxfp8_kernel<<<row_blocks_grid(rows, cols), 256, 0, (cudaStream_t)stream>>>(
      q8, s8, rows, cols, q4, s4);
  return launch_status();
}

extern "C" int mxfp8_from_mxfp4(const uint8_t* q4, const uint8_t* s4, long long rows, int cols,
                                uint8_t* q8, uint8_t* s8, moe_stream_t stream) {
  const int rc = check_mx4_args(q4, s4, rows, cols, q8, s8);
  if (rc != MOE_OK) return rc;
  mxfp8_from_mxfp4_kernel<<<row_blocks_grid(rows, cols), 256, 0, (cudaStream_t)stream>>>(
      q4, s4, rows, cols, q8, s8);
  return launch_status();
}

namespace {
template <bool TO_FP8>
int launch_row_to_col(const uint8_t* q4, const uint8_t* s4, long long rows, int cols,
                      uint8_t* qc, uint8_t* sc, moe_stream_t stream) {
  const int rc = check_mx4_args(q4, s4, rows, cols, qc, sc);
  if (rc != MOE_OK) return rc;
  const long long tiles = (rows / kRCRows) * (cols / kRCCols);
  const unsigned grid = (unsigned)(tiles < 148 * 2 ? tiles : 148 * 2);  // one wave, 2 CTAs per SM
  mxfp4_row_to_col_kernel<TO_FP8><<<grid, 256, 0, (cudaStream_t)stream>>>(q4, s4, rows, cols, qc,
                                                                          sc);
  return launch_status();
}
}  // namespace

extern "C" int mxfp4_rowwise_to_colwise(const uint8_t* q4, const uint8_t* s4, long long rows,
                                        int cols, uint8_t* q4c, uint8_t* s4c,
                                        moe_stream_t stream) {
  return launch_row_to_col<false>(q4, s4, rows, cols, q4c, s4c, stream);
}

extern "C" int mxfp8_colwise_from_mxfp4_rowwise(const uint8_t* q4, const uint8_t* s4,
                                                long long rows, int cols, uint8_t* q8c,
                                                uint8_t* s8c, moe_stream_t stream) {
  return launch_row_to_col<true>(q4, s4, rows, cols, q8c, s8c, stream);
}
