// Step 1: the router. score = sigmoid of the fp32 logit, top-k with the lowest
// expert index winning ties, the k scores renormalised to sum to one.
//
// The pages name MoE routing ("feat(pytorch): support Kimi K2.6", Motivation)
// and its size ("Kimi-K2.6" catalog page: 8 of 384 routed experts per token)
// but not the function; the sigmoid / tie / renormalisation reading is the one
// documented in moe_w4a16.h. For the result to be bit-identical everywhere the
// sigmoid is not expf-based: it is a fixed sequence of IEEE fp32 operations
// (Cody & Waite range reduction of exp, degree-7 Taylor polynomial), each one
// written with an explicit round-to-nearest intrinsic so that nothing is fused
// into an FMA. This translation unit is compiled without fast-math, so
// subnormals are kept.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// fp32 constants, by bit pattern:
//   log2(e) rounded to fp32; ln 2 split into the multiple of 2^-14 nearest to
//   it (hi, 14 significant bits) and the fp32 rounding of the remainder (lo);
//   Taylor coefficients 1/m! rounded to fp32, m = 2..7.
__device__ __forceinline__ float k_log2e() { return __int_as_float(0x3FB8AA3B); }
__device__ __forceinline__ float k_ln2_hi() { return __int_as_float(0x3F317400); }
__device__ __forceinline__ float k_ln2_lo() { return __int_as_float(0xB7F40417); }

__device__ __forceinline__ float exp_defined(float t) {
  if (t != t) return t;
  if (t > 88.0f) return __int_as_float(0x7F800000);
  if (t < -87.0f) return 0.0f;
  const float n = rintf(__fmul_rn(t, k_log2e()));  // round half to even
  const float r = __fsub_rn(__fsub_rn(t, __fmul_rn(n, k_ln2_hi())), __fmul_rn(n, k_ln2_lo()));
  float p = __int_as_float(0x39500D01);                      // 1/5040
  p = __fadd_rn(__fmul_rn(p, r), __int_as_float(0x3AB60B61));  // 1/720
  p = __fadd_rn(__fmul_rn(p, r), __int_as_float(0x3C088889));  // 1/120
  p = __fadd_rn(__fmul_rn(p, r), __int_as_float(0x3D2AAAAB));  // 1/24
  p = __fadd_rn(__fmul_rn(p, r), __int_as_float(0x3E2AAAAB));  // 1/6
  p = __fadd_rn(__fmul_rn(p, r), 0.5f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  const float two_n = __int_as_float((static_cast<int>(n) + 127) << 23);  // n in [-126, 127]
  return __fmul_rn(p, two_n);
}

__device__ __forceinline__ float sigmoid_defined(float x) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, exp_defined(-x)));
}

// ranking key: NaN below every score (scores lie in [0, 1])
__device__ __forceinline__ float rank_key(float s) { return (s != s) ? -1.0f : s; }

__device__ __forceinline__ bool better(float ka, int ea, float kb, int eb) {
  return ka > kb || (ka == kb && ea < eb);
}

__global__ void sigmoid_kernel(const float* __restrict__ x, int64_t n, float* __restrict__ y) {
  griddep_wait();    // the predecessor in the stream has finished and its writes are visible
  griddep_launch();  // the successor may start its own prologue
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    y[i] = sigmoid_defined(x[i]);
}

constexpr int kRouteWarps = 4;

// One warp per token, k <= 32. Lane L owns experts L, L+32, ... (SLOTS of them, E <= 32 * SLOTS): all of
// its logits are loaded first, so the loads overlap, then turned into scores in registers. Each
// of the k rounds takes the best remaining score of every lane and a warp arg-max (lowest index
// on ties); the winning lane marks its slot taken and broadcasts the raw score, which lane j keeps
// for round j. The weights divide by the rank-order sum, accumulated one score at a time.
template <int SLOTS>
__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel_reg(const float* __restrict__ logits, int T, int E,
                                                                      int k, int32_t* __restrict__ ids,
                                                                      float* __restrict__ wout) {
  griddep_wait();    // the predecessor in the stream has finished and its writes are visible
  griddep_launch();  // the successor may start its own prologue
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouteWarps + warp;
  if (t >= T) return;
  const float* lrow = logits + (int64_t)t * E;
  float sc[SLOTS];
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    const int e = lane + 32 * i;
    sc[i] = (e < E) ? __ldg(lrow + e) : 0.0f;
  }
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) sc[i] = sigmoid_defined(sc[i]);
  uint32_t taken = 0;  // bit i: expert lane + 32 i selected
  float my_sel = 0.0f; // lane j < k: the score chosen in round j
  for (int j = 0; j < k; ++j) {
    float bk = -2.0f;
    int be = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < SLOTS; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !(taken & (1u << i))) {
        const float kv = rank_key(sc[i]);
        if (better(kv, e, bk, be)) { bk = kv; be = e; }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ok = __shfl_xor_sync(0xFFFFFFFFu, bk, off);
      const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, off);
      if (better(ok, oe, bk, be)) { bk = ok; be = oe; }
    }
    float sv = 0.0f;
#pragma unroll
    for (int i = 0; i < SLOTS; ++i)
      if (lane + 32 * i == be) sv = sc[i];
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    sv = __shfl_sync(0xFFFFFFFFu, sv, be & 31);
    if (lane == (j & 31)) my_sel = sv;
    if (lane == 0) ids[(int64_t)t * k + j] = be;
  }
  float S = __shfl_sync(0xFFFFFFFFu, my_sel, 0);
  for (int j = 1; j < k; ++j) S = __fadd_rn(S, __shfl_sync(0xFFFFFFFFu, my_sel, j));
  if (lane < k) {
    const float wj = (S == 0.0f) ? __fdiv_rn(1.0f, static_cast<float>(k)) : __fdiv_rn(my_sel, S);
    wout[(int64_t)t * k + lane] = wj;
  }
}

// Any k: scores in shared memory (the general path, used when k > 32).
// One warp per token. Scores live in shared memory; lane L owns experts
// L, L+32, ... and keeps a bit per owned expert once it is selected.
__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel_smem(const float* __restrict__ logits, int T, int E,
                                                                  int k, int32_t* __restrict__ ids,
                                                                  float* __restrict__ wout) {
  griddep_wait();    // the predecessor in the stream has finished and its writes are visible
  griddep_launch();  // the successor may start its own prologue
  extern __shared__ float sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* score = sm + warp * (E + k);
  float* sel = score + E;
  const int t = blockIdx.x * kRouteWarps + warp;
  if (t >= T) return;
  const float* lrow = logits + (int64_t)t * E;
  for (int e = lane; e < E; e += 32) score[e] = sigmoid_defined(lrow[e]);
  __syncwarp();
  uint32_t taken = 0;  // bit i: expert lane + 32 i selected
  for (int j = 0; j < k; ++j) {
    float bk = -2.0f;
    int be = 0x7FFFFFFF;
    for (int i = 0, e = lane; e < E; ++i, e += 32) {
      if (taken & (1u << i)) continue;
      const float kv = rank_key(score[e]);
      if (better(kv, e, bk, be)) { bk = kv; be = e; }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ok = __shfl_xor_sync(0xFFFFFFFFu, bk, off);
      const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, off);
      if (better(ok, oe, bk, be)) { bk = ok; be = oe; }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == 0) {
      ids[(int64_t)t * k + j] = be;
      sel[j] = score[be];
    }
  }
  __syncwarp();
  if (lane == 0) {
    float S = sel[0];
    for (int j = 1; j < k; ++j) S = __fadd_rn(S, sel[j]);
    if (S == 0.0f) {
      const float u = __fdiv_rn(1.0f, static_cast<float>(k));
      for (int j = 0; j < k; ++j) wout[(int64_t)t * k + j] = u;
    } else {
      for (int j = 0; j < k; ++j) wout[(int64_t)t * k + j] = __fdiv_rn(sel[j], S);
    }
  }
}

}  // namespace

cudaError_t launch_sigmoid(const float* logits, int64_t n, float* scores, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  (void)launch_pdl(sigmoid_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, logits, n, scores);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((T + kRouteWarps - 1) / kRouteWarps);
  const int slots = (E + 31) / 32;
  if (k <= 32 && slots <= 32) {
    if (slots <= 4) (void)launch_pdl(route_kernel_reg<4>, dim3(blocks), dim3(kRouteWarps * 32), 0, s, logits, T, E, k, ids, w);
    else if (slots <= 8) (void)launch_pdl(route_kernel_reg<8>, dim3(blocks), dim3(kRouteWarps * 32), 0, s, logits, T, E, k, ids, w);
    else if (slots <= 12) (void)launch_pdl(route_kernel_reg<12>, dim3(blocks), dim3(kRouteWarps * 32), 0, s, logits, T, E, k, ids, w);
    else if (slots <= 16) (void)launch_pdl(route_kernel_reg<16>, dim3(blocks), dim3(kRouteWarps * 32), 0, s, logits, T, E, k, ids, w);
    else (void)launch_pdl(route_kernel_reg<32>, dim3(blocks), dim3(kRouteWarps * 32), 0, s, logits, T, E, k, ids, w);
  } else {
    const size_t smem = sizeof(float) * kRouteWarps * (E + k);
    (void)launch_pdl(route_kernel_smem, dim3(blocks), dim3(kRouteWarps * 32), smem, s, logits, T, E, k, ids, w);
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
