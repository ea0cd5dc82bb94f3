// Host-side launchers of the kernels (one translation unit each), called by
// the C-ABI layer in moe_abi.cu. Every launcher validates nothing: the ABI
// layer checks arguments first. Each returns the launch's cudaError_t.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include "moe_w4a16.h"

namespace moe {

// Largest number of token-expert assignments (T * top_k) any entry point accepts.
constexpr int64_t kMaxRows = int64_t(1) << 24;

// The assignment-count rule shared by every entry point: MOE_OK, MOE_ERR_INVALID_ARG for T < 0,
// or MOE_ERR_UNSUPPORTED_SHAPE beyond kMaxRows.
inline moe_status_t check_T(int32_t T, int32_t k) {
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * k > kMaxRows) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

// An NVTX range named after a C-ABI entry point, open for the call's host-side
// life (argument checks and launches), so profilers attribute each kernel to
// the call that launched it. Costs one pointer test when no tool is attached.
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

// counts kernels launched by this library (moe_launch_count)
void count_launches(uint64_t n);

// defined fp32 sigmoid + top-k routing
cudaError_t launch_sigmoid(const float* logits, int64_t n, float* scores, cudaStream_t s);
cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t s);

// expert-sorted permutation (count, scan, scatter) and row gather
int permute_blocks(int64_t Tk);  // number of segments of the count/scatter kernels
cudaError_t launch_permute(const int32_t* ids, int T, int E, int k, int32_t* offsets, int32_t* sorted_ids,
                           int32_t* inv_perm, int32_t* hist, int* status, cudaStream_t s);
// x_perm[row] = x[sorted_ids[row]], in natural or MMA K order (see gemm_tc.cu)
cudaError_t launch_gather(const uint16_t* x, const int32_t* sorted_ids, const int32_t* offsets, int E, int R,
                          int H, bool mma_order, uint16_t* x_perm, cudaStream_t s);
// dst = src rows (natural order) rewritten in MMA K order
cudaError_t launch_to_mma_order(const uint16_t* src, uint16_t* dst, int64_t rows, int K, cudaStream_t s);

// combine; y and addend are bf16 rows, or fp32 rows when y_f32 (the residual is always bf16)
cudaError_t launch_combine(const void* y, const int32_t* inv, const float* w, int T, int k, int H,
                           const void* addend, const uint16_t* residual, bool y_f32, uint16_t* out, cudaStream_t s);
// out[t] = bf16(x[t] / sqrt(mean(x[t]^2) + eps)), fp32 arithmetic
cudaError_t launch_rmsnorm(const uint16_t* x, int T, int H, float eps, uint16_t* out, cudaStream_t s);

// grouped GEMM problem description shared by both GEMM implementations
struct GemmProblem {
  int op;                  // MOE_GEMM_GATEUP_SILU or MOE_GEMM_DOWN
  bool bf16_weights;       // dense bf16 weights (shared expert) instead of int4
  const void* w;           // int32 [E][rows][K/8] or bf16 [rows][K]
  const uint16_t* scales;  // bf16 [E][rows][K/32] (int4 only)
  const uint16_t* a;       // bf16 [R][K], expert-sorted rows
  const int32_t* offsets;  // [E+1], or null with uniform_rows >= 0
  uint16_t* out;           // bf16 [R][out_cols]
  float* out_f32 = nullptr;  // down only: when set, the rows are written here in fp32 instead of `out`
  int* status;
  int E;
  int K;
  int rows_per_expert;     // 2I (gate/up) or H (down)
  int out_cols;            // I (gate/up) or H (down)
  int R;                   // rows of a and out
  int uniform_rows;        // >= 0: a single group of that many rows
  int min_rows = 1;        // only experts with min_rows <= rows <= max_rows are computed
  int max_rows = 1 << 30;
  int ksplit = 1;          // K slices (divides the K stages); > 1 needs `partial`
  float* partial = nullptr;  // fp32 [ksplit][R][2][out_cols] (gate/up) or [ksplit][R][out_cols]
  bool a_mma_order;        // rows of a are stored in MMA K order
  bool out_mma_order;      // gate/up: write h in MMA K order
  int wfmt = 0;            // WFMT_INT4: int4 + bf16 scale per 32; WFMT_FP4: E2M1 + E4M3 scale per 16
  // The weights (and offsets) were complete before the calls queued ahead of this launch began:
  // the kernel may then stream weights while its predecessor in the stream finishes. Otherwise
  // (weights written by the previous kernel, or by a caller's kernel we cannot see) it waits first.
  bool weights_ready = false;
  const float* gscale = nullptr;   // WFMT_FP4: fp32 scale of each expert's matrix, [E]
};

// weight formats of the routed experts
enum WeightFormat { WFMT_INT4 = 0, WFMT_FP4 = 1 };

cudaError_t launch_gemm_simt(const GemmProblem& p, cudaStream_t s);

enum ASource { A_TMEM_DQ = 0, A_SMEM_DQ = 1, A_SMEM_BF16 = 2 };
// returns cudaErrorNotSupported if no kernel exists for (asrc, tokens_per_tile)
cudaError_t launch_gemm_tc(const GemmProblem& p, int asrc, int tokens_per_tile, int num_sms, cudaStream_t s);

// the same GEMM on CTA pairs (int4 weights, A in tensor memory, rows in MMA K order): one
// cta_group::2 MMA covers 256 weight rows over two SMs; nt in {16, 32, 64, 128}
cudaError_t launch_gemm_pair(const GemmProblem& p, int tokens_per_tile, int num_sms, cudaStream_t s);

// copy every expert with rows (offsets) of the four bank tensors from the host bank (device-accessible
// addresses of page-locked host memory) into the device bank of the same layout; bytes: per expert
cudaError_t launch_stage_experts(const void* const host_dev[4], void* const dev[4], const int64_t bytes[4],
                                 const int32_t* offsets, int E, cudaStream_t s);

cudaError_t launch_expire_wait(int* status, int64_t timeout_ns, cudaStream_t s);

}  // namespace moe
