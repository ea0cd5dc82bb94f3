// CUDA-core baseline of the grouped expert GEMMs (steps 3 and 4), selected by
// MOE_FLAG_GEMM_SIMT. One warp computes one output unit (a gate/up row pair,
// or one down row) for up to 8 expert-sorted token rows at a time: it walks
// the row's int32 words, dequantises each nibble to fp32 exactly (q * scale),
// and accumulates dot products in fp32. No tensor cores, no shared-memory
// staging: the reference point the tensor-core kernel is measured against.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kTok = 8;

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// 8 consecutive weights of row `row`, word c (int4) or elements 8c..8c+7 (bf16)
template <bool BF16W>
__device__ __forceinline__ void load_w8(const GemmProblem& p, int64_t row, int c, float (&wv)[8]) {
  if (BF16W) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.w) + row * p.K) + c);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      wv[2 * i] = __uint_as_float(u[i] << 16);
      wv[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
  } else {
    const uint32_t word = static_cast<uint32_t>(__ldg(static_cast<const int32_t*>(p.w) + row * (p.K / 8) + c));
    const float s = bf16f(__ldg(p.scales + row * (p.K / 32) + c / 4));
#pragma unroll
    for (int j = 0; j < 8; ++j) wv[j] = static_cast<float>(static_cast<int>((word >> (4 * j)) & 15u) - 8) * s;
  }
}

template <int OP, bool BF16W>
__global__ void __launch_bounds__(kWarps * 32) gemm_simt_kernel(GemmProblem p) {
  griddep_wait();    // the predecessor in the stream has finished and its writes are visible
  griddep_launch();  // the successor may start its own prologue
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x * kWarps + warp;
  const int e = blockIdx.y;
  const int units = (OP == MOE_GEMM_GATEUP_SILU) ? p.out_cols : p.rows_per_expert;
  if (unit >= units) return;
  int r0, r1;
  if (p.uniform_rows >= 0) { r0 = 0; r1 = p.uniform_rows; }
  else { r0 = p.offsets[e]; r1 = p.offsets[e + 1]; }
  const int64_t wbase = static_cast<int64_t>(e) * p.rows_per_expert;
  const int64_t row_a = wbase + unit;                          // gate row, or the down row
  const int64_t row_b = wbase + p.out_cols + unit;             // up row (gate/up only)
  const int words = p.K / 8;
  for (int t0 = r0; t0 < r1; t0 += kTok) {
    const int nt = min(kTok, r1 - t0);
    float acc_a[kTok], acc_b[kTok];
#pragma unroll
    for (int t = 0; t < kTok; ++t) { acc_a[t] = 0.f; acc_b[t] = 0.f; }
    for (int c = lane; c < words; c += 32) {
      float wa[8], wb[8];
      load_w8<BF16W>(p, row_a, c, wa);
      if (OP == MOE_GEMM_GATEUP_SILU) load_w8<BF16W>(p, row_b, c, wb);
#pragma unroll
      for (int t = 0; t < kTok; ++t) {
        if (t < nt) {
          const uint4 xv = __ldg(reinterpret_cast<const uint4*>(p.a + static_cast<int64_t>(t0 + t) * p.K) + c);
          const uint32_t u[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float x0 = __uint_as_float(u[i] << 16), x1 = __uint_as_float(u[i] & 0xFFFF0000u);
            // the pair holds inputs (2i, 2i+1) in natural order, (i, i+4) in MMA K order
            const int k0 = p.a_mma_order ? i : 2 * i;
            const int k1 = p.a_mma_order ? i + 4 : 2 * i + 1;
            acc_a[t] = fmaf(wa[k0], x0, acc_a[t]);
            acc_a[t] = fmaf(wa[k1], x1, acc_a[t]);
            if (OP == MOE_GEMM_GATEUP_SILU) {
              acc_b[t] = fmaf(wb[k0], x0, acc_b[t]);
              acc_b[t] = fmaf(wb[k1], x1, acc_b[t]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kTok; ++t) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        acc_a[t] += __shfl_xor_sync(0xFFFFFFFFu, acc_a[t], off);
        if (OP == MOE_GEMM_GATEUP_SILU) acc_b[t] += __shfl_xor_sync(0xFFFFFFFFu, acc_b[t], off);
      }
    }
    if (lane == 0) {
      for (int t = 0; t < nt; ++t) {
        float v;
        if (OP == MOE_GEMM_GATEUP_SILU) {
          const float g = acc_a[t];
          v = g / (1.0f + __expf(-g)) * acc_b[t];
        } else {
          v = acc_a[t];
        }
        int col = unit;
        if (OP == MOE_GEMM_GATEUP_SILU && p.out_mma_order) col = (unit & ~7) | ((unit & 3) << 1) | ((unit >> 2) & 1);
        const int64_t o = static_cast<int64_t>(t0 + t) * p.out_cols + col;
        if (OP == MOE_GEMM_DOWN && p.out_f32 != nullptr) p.out_f32[o] = v;
        else p.out[o] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
      }
    }
  }
}

}  // namespace

cudaError_t launch_gemm_simt(const GemmProblem& p, cudaStream_t s) {
  const int units = (p.op == MOE_GEMM_GATEUP_SILU) ? p.out_cols : p.rows_per_expert;
  const int groups = p.uniform_rows >= 0 ? 1 : p.E;
  dim3 grid((units + kWarps - 1) / kWarps, groups);
  if (p.op == MOE_GEMM_GATEUP_SILU) {
    if (p.bf16_weights) (void)launch_pdl(gemm_simt_kernel<MOE_GEMM_GATEUP_SILU, true>, dim3(grid), dim3(kWarps * 32), 0, s, p);
    else (void)launch_pdl(gemm_simt_kernel<MOE_GEMM_GATEUP_SILU, false>, dim3(grid), dim3(kWarps * 32), 0, s, p);
  } else {
    if (p.bf16_weights) (void)launch_pdl(gemm_simt_kernel<MOE_GEMM_DOWN, true>, dim3(grid), dim3(kWarps * 32), 0, s, p);
    else (void)launch_pdl(gemm_simt_kernel<MOE_GEMM_DOWN, false>, dim3(grid), dim3(kWarps * 32), 0, s, p);
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
