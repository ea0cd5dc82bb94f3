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

struct ScratchSlot {
  void* ptr = nullptr;
  moe_status_t setup = MOE_ERR_CUDA;
};

ScratchSlot g_slot[kMaxScratchDevices];
std::once_flag g_slot_once[kMaxScratchDevices];

// Once per device, with that device current: check it is a compute capability
// 10.3 part and look up the device address of the scratch array. The lookup
// loads this library's module on the device if it is not loaded yet.
moe_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return MOE_ERR_CUDA;
  std::call_once(g_slot_once[dev], [dev] {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      g_slot[dev].setup = MOE_ERR_CUDA;
      return;
    }
    if (major != 10 || minor != 3) {
      g_slot[dev].setup = MOE_ERR_UNSUPPORTED_DEVICE;
      return;
    }
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_permute_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      (void)cudaGetLastError();  // leave no sticky error behind for the caller's next call
      g_slot[dev].setup = MOE_ERR_CUDA;
      return;
    }
    g_slot[dev].ptr = ptr;
    g_slot[dev].setup = MOE_OK;
  });
  *out = g_slot[dev].ptr;
  return g_slot[dev].setup;
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
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > 1024 || k < 1 || k > E) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int64_t Tk = static_cast<int64_t>(T) * k;
  if (Tk > (int64_t(1) << 24)) return MOE_ERR_UNSUPPORTED_SHAPE;
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
