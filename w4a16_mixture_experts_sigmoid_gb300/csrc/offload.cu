// The routed-expert bank in host memory ("Kimi-K2.6" catalog page, the
// paragraph on running with expert offload: 8 of 384 experts per token, so a
// token's expert traffic is a small slice of the checkpoint and the bank can
// sit in system RAM). Each layer call copies the experts that received rows
// from the host bank, which the GPU reads over the host link (NVLink-C2C on a
// Grace-Blackwell node), into a device bank of the same layout; the grouped
// GEMMs then read that device bank as usual. Experts with no rows are not
// copied, so a decode step moves only the touched experts' bytes.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kStageThreads = 512;
constexpr int64_t kChunk = int64_t(1) << 20;   // bytes of one tensor slice a block copies

struct StageTensor {
  const uint4* src;   // device-accessible address of the host bank tensor
  uint4* dst;         // device bank tensor, same layout
  int64_t per_expert; // bytes per expert (a multiple of 16)
  int64_t chunks;     // ceil(per_expert / kChunk)
};

struct StageArgs {
  StageTensor t[4];
  int64_t chunk_base[5];   // prefix of chunks over the tensors (per expert)
  const int32_t* offsets;  // [E+1]
  int E;
};

// grid.x = E * chunks per expert (all four tensors). A block whose expert has no rows returns at
// once; the others copy one slice of one tensor of their expert with 16-byte loads and stores.
// The successor (the gate/up GEMM, one CTA per SM holding the whole register file) is released
// only as the copy's blocks finish, so that its CTAs, which wait for the whole copy anyway, do not
// hold SMs that the copy's remaining blocks could use.
__global__ void __launch_bounds__(kStageThreads) stage_kernel(const __grid_constant__ StageArgs a) {
  griddep_wait();
  const int64_t per = a.chunk_base[4];
  const int e = static_cast<int>(blockIdx.x / per);
  if (e >= a.E) {
    griddep_launch();
    return;
  }
  if (__ldg(a.offsets + e + 1) - __ldg(a.offsets + e) <= 0) {
    griddep_launch();
    return;
  }
  int64_t c = blockIdx.x - static_cast<int64_t>(e) * per;
  int ti = 0;
  while (ti < 3 && c >= a.chunk_base[ti + 1]) ++ti;
  c -= a.chunk_base[ti];
  const StageTensor& t = a.t[ti];
  const int64_t lo = c * kChunk, hi = min(t.per_expert, lo + kChunk);
  const int64_t base = static_cast<int64_t>(e) * t.per_expert;
  const uint4* src = t.src + (base + lo) / 16;
  uint4* dst = t.dst + (base + lo) / 16;
  const int64_t n = (hi - lo) / 16;
  // four loads in flight per thread before the stores
  int64_t i = threadIdx.x;
  for (; i + 3 * kStageThreads < n; i += 4 * kStageThreads) {
    const uint4 v0 = src[i], v1 = src[i + kStageThreads], v2 = src[i + 2 * kStageThreads],
                v3 = src[i + 3 * kStageThreads];
    dst[i] = v0;
    dst[i + kStageThreads] = v1;
    dst[i + 2 * kStageThreads] = v2;
    dst[i + 3 * kStageThreads] = v3;
  }
  for (; i < n; i += kStageThreads) dst[i] = src[i];
  griddep_launch();
}

}  // namespace

cudaError_t launch_stage_experts(const void* const host_dev[4], void* const dev[4], const int64_t bytes[4],
                                 const int32_t* offsets, int E, cudaStream_t s) {
  StageArgs a;
  a.offsets = offsets;
  a.E = E;
  a.chunk_base[0] = 0;
  for (int i = 0; i < 4; ++i) {
    a.t[i].src = static_cast<const uint4*>(host_dev[i]);
    a.t[i].dst = static_cast<uint4*>(dev[i]);
    a.t[i].per_expert = bytes[i];
    a.t[i].chunks = (bytes[i] + kChunk - 1) / kChunk;
    a.chunk_base[i + 1] = a.chunk_base[i] + a.t[i].chunks;
  }
  const int64_t blocks = static_cast<int64_t>(E) * a.chunk_base[4];
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  (void)launch_pdl(stage_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kStageThreads), 0, s, a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
