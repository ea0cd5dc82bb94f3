// Step 5: the top-k weighted combine back to token order,
//   out[t] = bf16( sum_j w[t,j] * y[inv[t*k+j]]  (+ addend[t])  (+ residual[t]) ),
// y and addend in bf16 or fp32 (the layer passes fp32: one bf16 rounding fewer),
// fp32 accumulation in rank order j, then the shared expert's output, then the
// residual stream of a layer stack, one rounding to bf16 at the end.
// The pages' MoE sums the selected experts' outputs per token ("feat(pytorch):
// support Kimi K2.6", MoE routing); where the weights enter is not spelled out,
// and multiplying after the down projection is the reading used here.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// Eight consecutive values of a row: bf16 (one 16-byte load) or fp32 (two).
template <bool F32>
__device__ __forceinline__ void load8(const void* base, int64_t idx8, float (&f)[8]) {
  if (F32) {
    const float4* q = reinterpret_cast<const float4*>(base) + 2 * idx8;
    const float4 a = __ldg(q), b = __ldg(q + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  } else {
    unpack8(__ldg(reinterpret_cast<const uint4*>(base) + idx8), f);
  }
}

// grid: (ceil(H/8 / blockDim), T); each thread owns 8 consecutive columns of one token.
template <bool F32>
__global__ void __launch_bounds__(128) combine_kernel(const void* __restrict__ y, const int32_t* __restrict__ inv,
                                                      const float* __restrict__ w, int T, int k, int H8,
                                                      const void* __restrict__ addend,
                                                      const uint4* __restrict__ residual, uint4* __restrict__ out) {
  griddep_wait();    // the predecessor in the stream has finished and its writes are visible
  griddep_launch();  // the successor may start its own prologue
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= H8) return;
  for (int t = blockIdx.y; t < T; t += gridDim.y) {
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  // eight assignments at a time: their rows and weights are loaded before any is added, so the
  // loads overlap; the sum still runs in rank order j
  for (int j0 = 0; j0 < k; j0 += 8) {
    int pj[8];
    float wj[8];
    float yv[8][8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u;
      pj[u] = (j < k) ? __ldg(inv + (int64_t)t * k + j) : -1;
      wj[u] = (j < k) ? __ldg(w + (int64_t)t * k + j) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (pj[u] >= 0) load8<F32>(y, (int64_t)pj[u] * H8 + c, yv[u]);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (pj[u] < 0) continue;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[u], yv[u][i], acc[i]);
    }
  }
  if (addend != nullptr) {
    float f[8];
    load8<F32>(addend, (int64_t)t * H8 + c, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += f[i];
  }
  if (residual != nullptr) {
    float f[8];
    unpack8(__ldg(residual + (int64_t)t * H8 + c), f);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += f[i];
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  out[(int64_t)t * H8 + c] = o;
  }
}

}  // namespace

cudaError_t launch_combine(const void* y, const int32_t* inv, const float* w, int T, int k, int H,
                           const void* addend, const uint16_t* residual, bool y_f32, uint16_t* out, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int H8 = H / 8;
  dim3 grid((H8 + 127) / 128, T < 65535 ? T : 65535);
  if (y_f32)
    (void)launch_pdl(combine_kernel<true>, dim3(grid), dim3(128), 0, s, y, inv, w, T, k, H8, addend, reinterpret_cast<const uint4*>(residual),
                                              reinterpret_cast<uint4*>(out));
  else
    (void)launch_pdl(combine_kernel<false>, dim3(grid), dim3(128), 0, s, y, inv, w, T, k, H8, addend, reinterpret_cast<const uint4*>(residual),
                                               reinterpret_cast<uint4*>(out));
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
