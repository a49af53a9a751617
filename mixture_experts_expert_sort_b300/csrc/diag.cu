// Self-test of the library's failure detection: the bounded wait that every
// pipelined kernel uses (gemm::wait_bar) runs out on an mbarrier that nothing
// arrives at, records MOE_DEVERR_TIMEOUT in the device error word and
// returns, so the context stays usable and the host reads the status.
#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(64) selftest_wait_timeout_kernel() {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = ptx::smem_u32(&bar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);  // one arrival expected; none ever comes
    ptx::fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  // one lane of each warp waits, as the producer and MMA warps do; the first
  // to reach the limit sets the abort flag and the other leaves on it
  if ((threadIdx.x & 31) == 0)
    gemm::wait_bar(b, 0u, reinterpret_cast<volatile int*>(&abort_flag));
  __syncthreads();
}

}  // namespace
}  // namespace moe

extern "C" int moe_selftest_wait_timeout(moe_stream_t stream) {
  moe::selftest_wait_timeout_kernel<<<1, 64, 0, (cudaStream_t)stream>>>();
  return moe::launch_status();
}

// Host-side check of the grouped GEMMs' tile order: the (m-tile, n-tile) that
// the kernels' band_order gives each local tile index of one expert's grid.
extern "C" int moe_selftest_tile_order(int mtiles, int ntiles, int tile_m, int tile_n,
                                       long long band_rows, int prefer_m, int min_band_tiles,
                                       int32_t* mt, int32_t* nt) {
  if (mtiles < 1 || ntiles < 1 || tile_m < 1 || tile_n < 1 || band_rows < 0 || !mt || !nt ||
      (long long)mtiles * ntiles >= (1LL << 31))
    return MOE_ERR_ARG;
  for (int t = 0; t < mtiles * ntiles; ++t) {
    int m, n;
    moe::band_order(t, mtiles, ntiles, tile_m, tile_n, band_rows, prefer_m != 0, min_band_tiles,
                    m, n);
    mt[t] = m;
    nt[t] = n;
  }
  return MOE_OK;
}
