// moe_permute_static_scratch: step 2 (the expert-sorted permutation and the
// optional gather) for callers that cannot hand the library any device memory
// and must not have it allocate any.
//
// Who needs it: code that owns no workspace at the point where it routes, for
// example a hook inside a serving engine that reserved all of HBM for its own
// pool up front, or a latency-critical path where cudaMalloc/cudaFree (which
// can synchronise the whole device) are not allowed. moe_permute takes its
// per-segment histograms from the caller's workspace; this entry point takes
// them from a fixed array of device memory that is part of the library image
// itself (MOE_PERMUTE_STATIC_SCRATCH_BYTES, loaded once per device and held
// until the process exits), so nothing is allocated per call.
//
// The kernels are the ones moe_permute launches, on the same arguments; only
// where the histograms live differs, so the results are identical.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kMaxScratchDevices = 64;

// Histogram scratch, shared by every call on a device. The count kernel writes
// every entry that the scan and scatter kernels read, so nothing in it has to
// start at zero.
static __device__ __align__(256) uint8_t g_permute_scratch[MOE_PERMUTE_STATIC_SCRATCH_BYTES];

// Per-device set-up state. A successful lookup is kept for the life of the
// process; so is the verdict that a device is not a compute capability 10.3
// part, which cannot change. A lookup that failed for any other reason (for
// example a first call made inside a stream capture, or an earlier error) is
// not kept: the next call on that device tries again.
struct ScratchSlot {
  std::mutex mu;
  void* ptr = nullptr;
  bool unsupported = false;
};

ScratchSlot g_slot[kMaxScratchDevices];

// With the device current: check it is a compute capability 10.3 part and look
// up the device address of the scratch array (this may load the library's
// module onto the device).
moe_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return MOE_ERR_CUDA;
  ScratchSlot& slot = g_slot[dev];
  std::lock_guard<std::mutex> lock(slot.mu);
  if (slot.ptr != nullptr) {
    *out = slot.ptr;
    return MOE_OK;
  }
  if (slot.unsupported) return MOE_ERR_UNSUPPORTED_DEVICE;
  // an error the caller left pending stays as it was; only this lookup's own failure is cleared
  const cudaError_t pending = cudaPeekAtLastError();
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    if (pending == cudaSuccess) (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  if (major != 10 || minor != 3) {
    slot.unsupported = true;
    return MOE_ERR_UNSUPPORTED_DEVICE;
  }
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_permute_scratch);
  if (e != cudaSuccess || ptr == nullptr) {
    if (pending == cudaSuccess) (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  slot.ptr = ptr;
  *out = ptr;
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

extern "C" {

moe_status_t moe_permute_static_scratch(const int32_t* topk_ids, int32_t T, int32_t E, int32_t k,
                                        int32_t* expert_offsets, int32_t* sorted_token_ids, int32_t* inv_perm,
                                        const uint16_t* x, int32_t H, uint16_t* x_perm, int32_t* status,
                                        uint32_t flags, void* stream) {
  using namespace moe;
  CallRange range_("moe_permute_static_scratch");
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > 1024 || k < 1 || k > E) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (check_T(T, k) != MOE_OK) return MOE_ERR_UNSUPPORTED_SHAPE;   // the same row limit as moe_permute
  const int64_t Tk = static_cast<int64_t>(T) * k;
  if (T == 0) return MOE_OK;
  if (topk_ids == nullptr || expert_offsets == nullptr || sorted_token_ids == nullptr || inv_perm == nullptr)
    return MOE_ERR_INVALID_ARG;
  const bool gather = x != nullptr && x_perm != nullptr;
  if ((x != nullptr) != (x_perm != nullptr)) return MOE_ERR_INVALID_ARG;
  if (gather && (H < 8 || H % 8 || !aligned16(x) || !aligned16(x_perm))) return MOE_ERR_INVALID_ARG;
  // the histograms: one row of E counts per segment of assignments
  const size_t need = static_cast<size_t>(permute_blocks(Tk)) * static_cast<size_t>(E) * sizeof(int32_t);
  if (need > MOE_PERMUTE_STATIC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const moe_status_t st = scratch_for_current_device(&scratch);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_permute(topk_ids, T, E, k, expert_offsets, sorted_token_ids, inv_perm,
                                 static_cast<int32_t*>(scratch), status, s);
  if (e == cudaSuccess && gather)
    e = launch_gather(x, sorted_token_ids, expert_offsets, E, static_cast<int>(Tk), H,
                      (flags & MOE_FLAG_ROWS_MMA_ORDER) != 0, x_perm, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
