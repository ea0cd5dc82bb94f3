// Step 2: the expert-sorted permutation of the T*k (token, expert) assignments
// and the gather of activation rows into that order.
//
// Assignment i = t*k + j. Row order = stable sort of the assignments by
// expert id: every result is a pure function of topk_ids, independent of
// scheduling (the only atomics are order-free counts).
//
//   count   (one block per segment of kSeg assignments): per-segment histogram.
//   scan    (one block): per-expert prefix over segments, then offsets[E+1].
//   scatter (one block per segment): per-warp histograms and bases, then each
//           warp walks its slice (an eighth of the segment) 32 assignments at a
//           time in order, ranking equal ids with __match_any_sync.
// When the assignments fit one segment (small batches) one block does all three
// in the same order, without the launches between them; the results are the
// same.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kSeg = 4096;        // assignments per segment
constexpr int kScatterWarps = 8;  // warps per scatter block, each owns kSeg / 8 assignments

__global__ void __launch_bounds__(256) count_kernel(const int32_t* __restrict__ ids, int64_t Tk, int E,
                                                    int32_t* __restrict__ hist, int* status) {
  griddep_wait();    // the predecessor in the stream has finished and its writes are visible
  griddep_launch();  // the successor may start its own prologue
  extern __shared__ int32_t h[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const int64_t lo = (int64_t)blockIdx.x * kSeg;
  const int64_t hi = min(Tk, lo + kSeg);
  bool bad = false;
  for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) {
    const int e = ids[i];
    if (e >= 0 && e < E) atomicAdd(&h[e], 1);
    else bad = true;
  }
  if (bad) record_status(status, MOE_ERR_DEVICE_BOUNDS);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(int64_t)blockIdx.x * E + e] = h[e];
}

// hist[b][e] <- number of assignments to e in segments < b (exclusive over b);
// offsets <- exclusive scan of per-expert totals.
__global__ void __launch_bounds__(1024) scan_kernel(int32_t* __restrict__ hist, int nblk, int E,
                                                    int32_t* __restrict__ offsets) {
  griddep_wait();    // the predecessor in the stream has finished and its writes are visible
  griddep_launch();  // the successor may start its own prologue
  __shared__ int32_t warp_sum[32];
  const int e = threadIdx.x;
  int32_t run = 0;
  if (e < E) {
    for (int b = 0; b < nblk; ++b) {
      const int32_t c = hist[(int64_t)b * E + e];
      hist[(int64_t)b * E + e] = run;
      run += c;
    }
  }
  // block-wide exclusive scan of run over e (E <= 1024 = blockDim)
  const int lane = e & 31, warp = e >> 5;
  int32_t v = (e < E) ? run : 0;
  int32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t ws = warp_sum[lane];
    int32_t wi = ws;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t o = __shfl_up_sync(0xFFFFFFFFu, wi, off);
      if (lane >= off) wi += o;
    }
    warp_sum[lane] = wi - ws;  // exclusive prefix of warps
  }
  __syncthreads();
  const int32_t excl = warp_sum[warp] + incl - v;
  if (e < E) offsets[e] = excl;
  if (e == E - 1) offsets[E] = excl + v;
}

// Walks warp `warp`'s slice [lo, hi) of the assignments 32 at a time in order and places each
// valid one at its expert's running base in `mybase` (this warp's row of bases), ranking equal ids
// within the 32 with __match_any_sync; an out-of-range id gets inv = -1.
__device__ __forceinline__ void scatter_slice(const int32_t* __restrict__ ids, int64_t lo, int64_t hi, int k, int E,
                                              int32_t* mybase, int32_t* __restrict__ sorted_ids,
                                              int32_t* __restrict__ inv) {
  const int lane = threadIdx.x & 31;
  for (int64_t i0 = lo; i0 < hi; i0 += 32) {
    const int64_t i = i0 + lane;
    int e = (i < hi) ? ids[i] : -1;
    const bool ok = (e >= 0 && e < E);
    if (!ok) e = -1;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    int32_t pos = 0;
    if (ok) pos = mybase[e] + rank;
    __syncwarp();
    if (ok && rank == 0) mybase[e] += __popc(peers);
    __syncwarp();
    if (ok) {
      sorted_ids[pos] = static_cast<int32_t>(i / k);
      inv[i] = pos;
    } else if (i < hi) {
      inv[i] = -1;
    }
  }
}

__global__ void __launch_bounds__(kScatterWarps * 32) scatter_kernel(const int32_t* __restrict__ ids, int64_t Tk,
                                                                     int k, int E,
                                                                     const int32_t* __restrict__ hist,
                                                                     const int32_t* __restrict__ offsets,
                                                                     int32_t* __restrict__ sorted_ids,
                                                                     int32_t* __restrict__ inv) {
  griddep_wait();    // the predecessor in the stream has finished and its writes are visible
  griddep_launch();  // the successor may start its own prologue
  extern __shared__ int32_t wb[];  // [kScatterWarps][E]: per-warp counts, then per-warp bases
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kScatterWarps * E; i += blockDim.x) wb[i] = 0;
  __syncthreads();
  // warp w owns the w-th of eight contiguous slices of this block's segment (a multiple of 32
  // assignments each, 512 for a full segment), so short batches keep every warp busy
  const int64_t seg_lo = (int64_t)blockIdx.x * kSeg;
  const int64_t seg_n = min((int64_t)kSeg, Tk - seg_lo);
  const int64_t slice = ((seg_n + kScatterWarps - 1) / kScatterWarps + 31) / 32 * 32;
  const int64_t lo = min(seg_lo + seg_n, seg_lo + (int64_t)warp * slice);
  const int64_t hi = min(seg_lo + seg_n, lo + slice);
  for (int64_t i = lo + lane; i < hi; i += 32) {
    const int e = ids[i];
    if (e >= 0 && e < E) atomicAdd(&wb[warp * E + e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t base = offsets[e] + hist[(int64_t)blockIdx.x * E + e];
    for (int w = 0; w < kScatterWarps; ++w) {
      const int32_t c = wb[w * E + e];
      wb[w * E + e] = base;
      base += c;
    }
  }
  __syncthreads();
  scatter_slice(ids, lo, hi, k, E, wb + warp * E, sorted_ids, inv);
}

// count, scan and scatter in one block, for 1 <= Tk <= kSeg. The warps' slices, the per-warp bases
// and the walk are the scatter kernel's for segment 0 (whose bases over earlier segments are 0), so
// every output equals the three-kernel path's.
__global__ void __launch_bounds__(kScatterWarps * 32) permute_one_block_kernel(const int32_t* __restrict__ ids, int Tk,
                                                                               int k, int E,
                                                                               int32_t* __restrict__ offsets,
                                                                               int32_t* __restrict__ sorted_ids,
                                                                               int32_t* __restrict__ inv,
                                                                               int* status) {
  griddep_wait();    // the predecessor in the stream has finished and its writes are visible
  griddep_launch();  // the successor may start its own prologue
  extern __shared__ int32_t wb[];  // [kScatterWarps][E]: per-warp counts, then per-warp bases
  __shared__ int32_t warp_sum[kScatterWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kScatterWarps * E; i += blockDim.x) wb[i] = 0;
  __syncthreads();
  const int slice = ((Tk + kScatterWarps - 1) / kScatterWarps + 31) / 32 * 32;
  const int lo = min(Tk, warp * slice);
  const int hi = min(Tk, lo + slice);
  bool bad = false;
  for (int i = lo + lane; i < hi; i += 32) {
    const int e = ids[i];
    if (e >= 0 && e < E) atomicAdd(&wb[warp * E + e], 1);
    else bad = true;
  }
  if (bad) record_status(status, MOE_ERR_DEVICE_BOUNDS);
  __syncthreads();
  // thread t owns experts [t*per, t*per + per): their totals, a block-wide exclusive scan of the
  // totals, then offsets and each warp's base for those experts
  const int per = (E + blockDim.x - 1) / blockDim.x;
  const int e0 = threadIdx.x * per, e1 = min(E, e0 + per);
  int32_t mine = 0;
  for (int e = e0; e < e1; ++e)
    for (int w = 0; w < kScatterWarps; ++w) mine += wb[w * E + e];
  int32_t incl = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  int32_t before = 0;
  for (int w = 0; w < warp; ++w) before += warp_sum[w];
  int32_t base = before + incl - mine;
  for (int e = e0; e < e1; ++e) {
    offsets[e] = base;
    for (int w = 0; w < kScatterWarps; ++w) {
      const int32_t c = wb[w * E + e];
      wb[w * E + e] = base;
      base += c;
    }
  }
  if (threadIdx.x == blockDim.x - 1) offsets[E] = before + incl;
  __syncthreads();
  scatter_slice(ids, lo, hi, k, E, wb + warp * E, sorted_ids, inv);
}

// Eight bf16 inputs (one 16-byte chunk) from natural order to the tensor-core
// GEMM's K order [0,4,1,5,2,6,3,7] (see gemm_tc.cu).
__device__ __forceinline__ uint4 to_mma_order8(const uint4 v) {
  return make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632), __byte_perm(v.y, v.w, 0x5410),
                    __byte_perm(v.y, v.w, 0x7632));
}

// x_perm[row] = x[sorted_ids[row]] for rows < offsets[E]; 16-byte copies.
template <bool MMA_ORDER>
__global__ void __launch_bounds__(256) gather_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ sorted_ids,
                                                     const int32_t* __restrict__ offsets, int E, int R, int H8,
                                                     uint4* __restrict__ xp) {
  griddep_wait();    // the predecessor in the stream has finished and its writes are visible
  griddep_launch();  // the successor may start its own prologue
  const int valid = offsets[E];
  for (int row = blockIdx.x; row < R && row < valid; row += gridDim.x) {
    const uint4* src = x + (int64_t)sorted_ids[row] * H8;
    uint4* dst = xp + (int64_t)row * H8;
    for (int c = threadIdx.x; c < H8; c += blockDim.x) {
      const uint4 v = __ldg(src + c);
      dst[c] = MMA_ORDER ? to_mma_order8(v) : v;
    }
  }
}

__global__ void __launch_bounds__(256) to_mma_order_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                           int64_t n8) {
  griddep_wait();    // the predecessor in the stream has finished and its writes are visible
  griddep_launch();  // the successor may start its own prologue
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = to_mma_order8(__ldg(src + i));
}

}  // namespace

int permute_blocks(int64_t Tk) { return static_cast<int>((Tk + kSeg - 1) / kSeg); }

cudaError_t launch_permute(const int32_t* ids, int T, int E, int k, int32_t* offsets, int32_t* sorted_ids,
                           int32_t* inv_perm, int32_t* hist, int* status, cudaStream_t s) {
  const int64_t Tk = (int64_t)T * k;
  const int nblk = permute_blocks(Tk);
  if (nblk == 1) {
    (void)launch_pdl(permute_one_block_kernel, dim3(1), dim3(kScatterWarps * 32), sizeof(int32_t) * kScatterWarps * E, s,
                     ids, static_cast<int>(Tk), k, E, offsets, sorted_ids, inv_perm, status);
    count_launches(1);
    return cudaGetLastError();
  }
  (void)launch_pdl(count_kernel, dim3(nblk), dim3(256), sizeof(int32_t) * E, s, ids, Tk, E, hist, status);
  (void)launch_pdl(scan_kernel, dim3(1), dim3(1024), 0, s, hist, nblk, E, offsets);
  (void)launch_pdl(scatter_kernel, dim3(nblk), dim3(kScatterWarps * 32), sizeof(int32_t) * kScatterWarps * E, s, ids, Tk, k, E, hist, offsets,
                                                                                     sorted_ids, inv_perm);
  count_launches(3);
  return cudaGetLastError();
}

cudaError_t launch_gather(const uint16_t* x, const int32_t* sorted_ids, const int32_t* offsets, int E, int R, int H,
                          bool mma_order, uint16_t* x_perm, cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
  const int blocks = R < 4096 ? R : 4096;
  if (mma_order)
    (void)launch_pdl(gather_kernel<true>, dim3(blocks), dim3(256), 0, s, reinterpret_cast<const uint4*>(x), sorted_ids, offsets, E, R, H / 8,
                                               reinterpret_cast<uint4*>(x_perm));
  else
    (void)launch_pdl(gather_kernel<false>, dim3(blocks), dim3(256), 0, s, reinterpret_cast<const uint4*>(x), sorted_ids, offsets, E, R, H / 8,
                                                reinterpret_cast<uint4*>(x_perm));
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_to_mma_order(const uint16_t* src, uint16_t* dst, int64_t rows, int K, cudaStream_t s) {
  const int64_t n8 = rows * (K / 8);
  if (n8 <= 0) return cudaSuccess;
  int64_t blocks = (n8 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  (void)launch_pdl(to_mma_order_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, reinterpret_cast<const uint4*>(src),
                                                                    reinterpret_cast<uint4*>(dst), n8);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
