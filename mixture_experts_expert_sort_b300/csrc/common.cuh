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

// Byte offset of the scale for (row r, 32-column block kb) in the tiled
// scale layout of an operand with K columns (see mxfp8_quantize in moe.h).
__device__ __forceinline__ long long mx_scale_offset(long long r, long long kb, long long K) {
  long long tile = (r >> 7) * (K >> 7) + (kb >> 2);
  int rr = (int)(r & 127);
  return tile * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (int)(kb & 3);
}

}  // namespace moe
