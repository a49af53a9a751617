// moe_permute_plan_static: the expert-sort plan without any caller workspace.
//
// Some callers cannot allocate device memory at the point where they plan a
// batch: engines that hand a plugin no workspace and forbid allocation after
// start-up, or latency-critical loops where cudaMalloc's implicit device
// synchronisation is not acceptable. For them this entry point keeps the
// plan's scratch (the per-chunk expert histograms) in a fixed array that is
// part of the library's device image. It launches the same three kernels as
// moe_permute_plan and gives bit-identical results.
//
// The array lives for as long as the library is loaded, on every GPU that
// loads it (1 MiB each; every device has its own copy). All calls on one
// device share that device's copy: the plan overwrites every scratch word it
// reads during the same call, so no clearing is needed between calls, but
// calls on the same device that run at the same time on the GPU (different
// streams or host threads) race and must be serialised by the caller. Calls
// on different devices use different copies and do not race.
//
// The device address of the array is looked up by the first call on each
// device and kept. A cudaDeviceReset destroys the module image it points
// into, so after a reset this entry point must not be called again in the
// same process.
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr long long kPlanStaticScratchInts = MOE_PLAN_STATIC_SCRATCH_INTS;

static __device__ __align__(256) int32_t g_plan_static_scratch[kPlanStaticScratchInts];

constexpr int kMaxDevices = 64;
static std::mutex g_plan_static_mu;
static int32_t* g_plan_static_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device. In host code
// the array's name is only a host-side stand-in, so the address must be
// looked up once per device, with that device current.
static int plan_static_scratch(int32_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_plan_static_mu);
  if (!g_plan_static_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_plan_static_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_plan_static_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_plan_static_ptr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_permute_plan_static(const int32_t* idx, int T, int E, int k, int align,
                                       int32_t* counts, int32_t* offsets, int32_t* dest,
                                       int32_t* src, long long src_rows, moe_stream_t stream) {
  int st = permute_plan_check(idx, T, E, k, align, counts, offsets, dest, src, src_rows);
  if (st != MOE_OK) return st;
  const long long Tk = (long long)T * k;
  const long long n_chunks = (Tk + kPlanChunk - 1) / kPlanChunk;
  if (n_chunks * (long long)E > kPlanStaticScratchInts) return MOE_ERR_UNSUPPORTED;
  int32_t* scratch = nullptr;
  st = plan_static_scratch(&scratch);
  if (st != MOE_OK) return st;
  return permute_plan_launch(idx, T, E, k, align, counts, offsets, dest, src, src_rows, scratch,
                             (cudaStream_t)stream);
}
