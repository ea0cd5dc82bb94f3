// The pre-norm of a stack of MoE layers: x_{l+1} = x_l + MoE_l(RMSNorm(x_l)).
// The pages give the model's layer count and its 60 MoE layers ("Kimi-K2.6",
// GEOMETRY) but not how consecutive layers are joined; a plain residual
// x + MoE(x) grows without bound through a few layers of this width, and the
// reading used here is the usual pre-norm residual with a parameter-free
// RMSNorm (no learned gain: the gains belong to trained weights).
//
//   out[t, :] = bf16( x[t, :] / sqrt( mean_i x[t, i]^2 + eps ) )
//
// in fp32: squares summed per thread in column order, then across the block;
// one IEEE square root and one IEEE division per element. The residual add
// itself happens in the combine kernel (fp32, one rounding with the layer's
// output).
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kNormThreads = 256;

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

// grid-stride over rows; each block reduces one row at a time
__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const uint4* __restrict__ x, int T, int H8, float eps,
                                                               uint4* __restrict__ out) {
  griddep_wait();    // the predecessor in the stream has finished and its writes are visible
  griddep_launch();  // the successor may start its own prologue
  __shared__ float part[kNormThreads / 32];
  __shared__ float rms_s;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const uint4* row = x + static_cast<int64_t>(t) * H8;
    float ss = 0.0f;
    for (int c = threadIdx.x; c < H8; c += kNormThreads) {
      float f[8];
      unpack8(__ldg(row + c), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = __fadd_rn(ss, __fmul_rn(f[i], f[i]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, off));
    if (lane == 0) part[warp] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
      float tot = 0.0f;
      for (int w = 0; w < kNormThreads / 32; ++w) tot = __fadd_rn(tot, part[w]);
      const float ms = __fdiv_rn(tot, static_cast<float>(H8 * 8));
      rms_s = __fsqrt_rn(__fadd_rn(ms, eps));
    }
    __syncthreads();
    const float r = rms_s;
    for (int c = threadIdx.x; c < H8; c += kNormThreads) {
      float f[8];
      unpack8(__ldg(row + c), f);
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(__fdiv_rn(f[2 * i], r), __fdiv_rn(f[2 * i + 1], r));
        o[i] = *reinterpret_cast<const uint32_t*>(&p);
      }
      out[static_cast<int64_t>(t) * H8 + c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    __syncthreads();   // part / rms_s are reused by the next row
  }
}

}  // namespace

cudaError_t launch_rmsnorm(const uint16_t* x, int T, int H, float eps, uint16_t* out, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int blocks = T < 4096 ? T : 4096;
  (void)launch_pdl(rmsnorm_kernel, dim3(blocks), dim3(kNormThreads), 0, s, reinterpret_cast<const uint4*>(x), T, H / 8, eps,
                                                 reinterpret_cast<uint4*>(out));
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
