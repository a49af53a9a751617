// Shared device/host helpers for libmoe (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Device error word: kernels OR MOE_DEVERR_* flags into it instead of trapping.
// libmoe is one translation unit (libmoe.cu), so the definition lives here.
__device__ unsigned int g_device_error = 0;

__device__ __forceinline__ void raise_device_error(unsigned flag) {
  atomicOr(&g_device_error, flag);
}

inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMxBlock = 32;

// ---------------------------------------------------------------- MXFP8 rule
// OCP MX v1.0 with E4M3 elements (emax 8): scale exponent
// e = clamp(floor(log2 amax) - 8, -127, 127), read from the float32 exponent
// field (a zero or subnormal amax clamps to -127). Returns the E8M0 byte, or
// 0xFF for a non-finite amax.
__device__ __forceinline__ uint32_t mx_scale_byte(float amax) {
  uint32_t bits = __float_as_uint(amax);
  int ef = (int)((bits >> 23) & 0xFF);
  if (ef == 0xFF) return 0xFFu;
  int e = ef - 127 - 8;
  e = e < -127 ? -127 : e;
  return (uint32_t)(e + 127);
}

// 2^-e as float for a scale byte s = e + 127 (s in [0, 254]); exact.
__device__ __forceinline__ float mx_inv_scale(uint32_t s) {
  int e = (int)s - 127;
  return __uint_as_float((uint32_t)(127 - e) << 23);
}

// Two floats -> two E4M3 bytes (round to nearest even, saturate to +-448),
// hardware conversion. Low byte holds `a`.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(r) : "f"(a), "f"(b));
  return r;
}

// ------------------------------------------------------------ tile order
// Order of the tiles of one expert's mtiles x ntiles output grid in a grouped
// GEMM. Where neither operand of the expert fits in its L2 share, the tiles
// run in bands of g m-tiles (or g n-tiles): the band's rows of one operand stay
// in L2 while the other operand streams through once per band, and inside a
// band the banded index runs fastest, so the tiles in flight together share
// each k-slice of the streamed operand. The direction that streams fewer bytes
// wins. Where an operand fits, or where a band would hold fewer than
// `min_band_tiles` tiles (so that one wave of tiles spans several bands),
// the whole expert is one band along m (prefer_m) or along n.
// `band_rows` is the L2 share of the resident band in operand rows of K
// elements; tile_m / tile_n are the operand rows one tile reads of A / B.
__host__ __device__ __forceinline__ int band_size(long long band_rows, int tile, int tiles) {
  const long long g = band_rows / tile;
  return g < 1 ? 1 : g > tiles ? tiles : (int)g;
}

__host__ __device__ __forceinline__ void band_order(int local, int mtiles, int ntiles, int tile_m,
                                                    int tile_n, long long band_rows, bool prefer_m,
                                                    int min_band_tiles, int& mt, int& nt) {
  const int gm = band_size(band_rows, tile_m, mtiles);
  const int gn = band_size(band_rows, tile_n, ntiles);
  bool band_m = prefer_m;
  int g = prefer_m ? mtiles : ntiles;
  if (gm < mtiles || gn < ntiles) {
    if (gm == mtiles) {
      band_m = true;
      g = mtiles;
    } else if (gn == ntiles) {
      band_m = false;
      g = ntiles;
    } else {
      // operand rows read from DRAM: the streamed operand once per band, the
      // banded one once
      const long long cost_m =
          (long long)((mtiles + gm - 1) / gm) * ntiles * tile_n + (long long)mtiles * tile_m;
      const long long cost_n =
          (long long)((ntiles + gn - 1) / gn) * mtiles * tile_m + (long long)ntiles * tile_n;
      band_m = cost_m <= cost_n;
      g = band_m ? gm : gn;
    }
    if ((long long)g * (band_m ? ntiles : mtiles) < min_band_tiles) {
      band_m = prefer_m;
      g = prefer_m ? mtiles : ntiles;
    }
  }
  if (band_m) {
    const int per = g * ntiles, b = local / per, r = local - b * per, m0 = b * g;
    const int gs = g < mtiles - m0 ? g : mtiles - m0;
    mt = m0 + r % gs;
    nt = r / gs;
  } else {
    const int per = g * mtiles, b = local / per, r = local - b * per, n0 = b * g;
    const int gs = g < ntiles - n0 ? g : ntiles - n0;
    nt = n0 + r % gs;
    mt = r / gs;
  }
}

// L2 share given to the resident band of a grouped GEMM (bytes). The 126 MB
// L2 also holds the streamed operand's k-slices in flight and the output
// tiles on their way to memory.
#ifndef MOE_L2_BAND_MB
#define MOE_L2_BAND_MB 32
#endif
constexpr long long kL2BandBytes = (long long)MOE_L2_BAND_MB << 20;

// Byte offset of the scale for (row r, 32-column block kb) in the tiled
// scale layout of an operand with K columns (see mxfp8_quantize in moe.h).
__device__ __forceinline__ long long mx_scale_offset(long long r, long long kb, long long K) {
  long long tile = (r >> 7) * (K >> 7) + (kb >> 2);
  int rr = (int)(r & 127);
  return tile * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (int)(kb & 3);
}

}  // namespace moe
