// The C ABI of the library (declared in include/moe_w4a16.h): argument and
// shape validation before any launch, the workspace layout, the per-device
// property cache, and the launch sequence of moe_forward. Everything that
// computes runs in the kernels of the other translation units.
#include "common.cuh"
#include "internal.h"

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

namespace moe {

static std::atomic<uint64_t> g_launches{0};
void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

}  // namespace moe

namespace {

using namespace moe;

constexpr int kMaxDevices = 64;
constexpr int kMaxDim = 32768;                  // H, I, shared_I
constexpr int kSplitMaxT = 256;                 // the shared expert and the router split K for T up to this
constexpr int kMaxSplit = 32;                   // K slices at most
constexpr int kSplitRows = 2048;                // K slices x T at most (bounds the fp32 partial sums)
constexpr double kBf16StageBytes = 128.0 * 256 * 2;   // weight bytes of one K stage of a bf16 tile

struct DevInfo {
  int sms = 0;
  bool supported = false;
};

DevInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];

moe_status_t current_device(DevInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::call_once(g_dev_once[dev], [dev] {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    g_dev[dev].sms = sms;
    g_dev[dev].supported = (major == 10 && minor == 3);
  });
  *out = g_dev[dev];
  return out->supported ? MOE_OK : MOE_ERR_UNSUPPORTED_DEVICE;
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

moe_status_t check_dims(const moe_dims_t& d, int fmt = WFMT_INT4) {
  if (d.E < 1 || d.E > 1024 || d.top_k < 1 || d.top_k > d.E) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d.group != (fmt == WFMT_FP4 ? 16 : 32)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d.H < 32 || d.H % 32 || d.H > kMaxDim || d.I < 32 || d.I % 32 || d.I > kMaxDim) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

moe_status_t check_weights(const moe_weights_t* w, bool need_shared) {
  if (w == nullptr || w->w13_packed == nullptr || w->w13_scale == nullptr || w->w2_packed == nullptr ||
      w->w2_scale == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(w->w13_packed) || !aligned16(w->w13_scale) || !aligned16(w->w2_packed) || !aligned16(w->w2_scale))
    return MOE_ERR_INVALID_ARG;
  const bool has_shared = w->shared_wgu != nullptr || w->shared_wd != nullptr || w->shared_I != 0;
  if (has_shared || need_shared) {
    if (w->shared_wgu == nullptr || w->shared_wd == nullptr || !aligned16(w->shared_wgu) || !aligned16(w->shared_wd))
      return MOE_ERR_INVALID_ARG;
    if (w->shared_I < 64 || w->shared_I % 64 || w->shared_I > kMaxDim) return MOE_ERR_UNSUPPORTED_SHAPE;
  }
  return MOE_OK;
}

moe_status_t check_weights_fp4(const moe_weights_fp4_t* w) {
  if (w == nullptr || w->w13_packed == nullptr || w->w13_scale == nullptr || w->w13_gscale == nullptr ||
      w->w2_packed == nullptr || w->w2_scale == nullptr || w->w2_gscale == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(w->w13_packed) || !aligned16(w->w13_scale) || !aligned16(w->w2_packed) || !aligned16(w->w2_scale))
    return MOE_ERR_INVALID_ARG;
  const bool has_shared = w->shared_wgu != nullptr || w->shared_wd != nullptr || w->shared_I != 0;
  if (has_shared) {
    if (w->shared_wgu == nullptr || w->shared_wd == nullptr || !aligned16(w->shared_wgu) || !aligned16(w->shared_wd))
      return MOE_ERR_INVALID_ARG;
    if (w->shared_I < 64 || w->shared_I % 64 || w->shared_I > kMaxDim) return MOE_ERR_UNSUPPORTED_SHAPE;
  }
  return MOE_OK;
}

// One layer's weights as the kernels take them, in either routed-expert format.
struct LayerW {
  int fmt;
  const int32_t* w13;
  const void* s13;
  const float* g13;
  const int32_t* w2;
  const void* s2;
  const float* g2;
  const uint16_t* sh_gu;
  const uint16_t* sh_d;
  int32_t shared_I;
};

LayerW layer_w(const moe_weights_t* w) {
  return {WFMT_INT4, w->w13_packed, w->w13_scale, nullptr, w->w2_packed, w->w2_scale, nullptr,
          w->shared_wgu, w->shared_wd, w->shared_I};
}
LayerW layer_w(const moe_weights_fp4_t* w) {
  return {WFMT_FP4, w->w13_packed, w->w13_scale, w->w13_gscale, w->w2_packed, w->w2_scale, w->w2_gscale,
          w->shared_wgu, w->shared_wd, w->shared_I};
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// The most K slices a T-token bf16 launch may take; the partial-sum buffers are sized for it.
int max_split(int32_t T) {
  if (T > kSplitMaxT) return 1;
  return std::max(1, std::min(kMaxSplit, kSplitRows / std::max(T, 1)));
}

// fp32 partial sums of a K-split bf16 GEMM with T output rows of `cols` columns
size_t split_part_bytes(int32_t T, int64_t cols) {
  return T <= kSplitMaxT ? static_cast<size_t>(max_split(T)) * T * cols * 4 : 0;
}

// Workspace layout of moe_forward (byte offsets, each 256-aligned). With the router projection
// (moe_forward_project) the logits and the router GEMM's K-slice sums follow.
struct Layout {
  size_t ids, w, offsets, sorted, inv, hist, xperm, h, y, hs, ys, part, part_bytes, logits, rpart, rpart_bytes, end;
};

Layout layout(const moe_dims_t& d, int32_t T, int32_t shared_I, bool project = false) {
  Layout L;
  const size_t Tk = static_cast<size_t>(T) * d.top_k;
  size_t off = 256;  // status word
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L.ids = take(Tk * 4);
  L.w = take(Tk * 4);
  L.offsets = take(static_cast<size_t>(d.E + 1) * 4);
  L.sorted = take(Tk * 4);
  L.inv = take(Tk * 4);
  L.hist = take(static_cast<size_t>(permute_blocks(static_cast<int64_t>(Tk))) * d.E * 4);
  L.xperm = take(Tk * d.H * 2);
  L.h = take(Tk * d.I * 2);
  L.y = take(Tk * d.H * 4);   // fp32 rows: the down GEMM's output is not rounded before the combine
  L.hs = take(static_cast<size_t>(T) * shared_I * 2);
  L.ys = take(shared_I > 0 ? static_cast<size_t>(T) * d.H * 4 : 0);
  // fp32 partial sums of the shared expert's K slices (small batches only)
  L.part_bytes = shared_I > 0 && T <= kSplitMaxT
                     ? static_cast<size_t>(max_split(T)) * T * std::max(2 * shared_I, d.H) * 4 : 0;
  L.part = take(L.part_bytes);
  L.logits = take(project ? static_cast<size_t>(T) * d.E * 4 : 0);
  L.rpart_bytes = project ? split_part_bytes(T, d.E) : 0;
  L.rpart = take(L.rpart_bytes);
  L.end = off;
  return L;
}

// K slices for a bf16 launch of `tiles` tiles over a K loop of `stages` stages, at T tokens, whose
// slices each write `slice_bytes` of fp32 partial sums (read back once by the finishing kernel);
// 1 when the tiles already cover the SMs. A slice count divides the stages and is at most
// max_split(T). Where some count gives every SM a tile, the counts that do are weighed by an
// estimate of the launch's time, in bytes at the whole GPU's rate: the busiest SM's stages x a
// stage's weight bytes x the SMs (every SM streams at about the same rate), plus the partial sums
// written and read; the least wins, ties going to fewer slices. Otherwise the most slices allowed.
int pick_ksplit(int64_t tiles, int stages, int sms, int32_t T, double slice_bytes) {
  if (tiles >= sms) return 1;
  const int most = std::min(max_split(T), stages);
  int first = 0, last = 1;   // the fewest slices that cover the SMs; the most allowed
  for (int d = 2; d <= most; ++d) {
    if (stages % d) continue;
    last = d;
    if (first == 0 && tiles * d >= sms) first = d;
  }
  if (first == 0) return last;
  int best = first;
  double best_cost = 0.0;
  for (int d = first; d <= most; ++d) {
    if (stages % d) continue;
    const int64_t per_sm = (tiles * d + sms - 1) / sms;
    const double cost = static_cast<double>(per_sm * (stages / d)) * kBf16StageBytes * sms + 2.0 * d * slice_bytes;
    if (d == first || cost < best_cost) {
      best = d;
      best_cost = cost;
    }
  }
  return best;
}

int auto_tokens_per_tile(int64_t rows, int groups) {
  const double m = static_cast<double>(rows) / (groups > 0 ? groups : 1);
  if (m <= 8.0) return 16;
  if (m <= 18.0) return 32;
  if (m <= 40.0) return 64;
  return 128;
}

// One grouped GEMM. rows_mma_order: a (and, for gate/up, out) are stored in
// the tensor-core K order. The tensor-core kernel needs its token rows in that
// order; natural-order rows are first rewritten into `scratch` (R * K * 2 bytes).
// out is bf16, or fp32 for the down projection with MOE_FLAG_OUT_F32.
moe_status_t run_grouped_gemm(int32_t op, const moe_dims_t& d, const LayerW& w, const uint16_t* a,
                              int32_t T, const int32_t* offsets, void* out, int* status, uint32_t flags,
                              bool rows_mma_order, uint16_t* scratch, int sms, cudaStream_t s,
                              bool weights_ready = false) {
  GemmProblem p;
  p.weights_ready = weights_ready;
  p.op = op;
  p.bf16_weights = false;
  p.a = a;
  p.offsets = offsets;
  const bool f32 = op == MOE_GEMM_DOWN && (flags & MOE_FLAG_OUT_F32);
  p.out = f32 ? nullptr : static_cast<uint16_t*>(out);
  p.out_f32 = f32 ? static_cast<float*>(out) : nullptr;
  p.status = status;
  p.E = d.E;
  p.R = T * d.top_k;
  p.uniform_rows = -1;
  p.a_mma_order = rows_mma_order;
  p.out_mma_order = rows_mma_order;
  p.wfmt = w.fmt;
  if (op == MOE_GEMM_GATEUP_SILU) {
    p.w = w.w13;
    p.scales = static_cast<const uint16_t*>(w.s13);
    p.gscale = w.g13;
    p.K = d.H;
    p.rows_per_expert = 2 * d.I;
    p.out_cols = d.I;
  } else {
    p.w = w.w2;
    p.scales = static_cast<const uint16_t*>(w.s2);
    p.gscale = w.g2;
    p.K = d.I;
    p.rows_per_expert = d.H;
    p.out_cols = d.H;
  }
  if (flags & MOE_FLAG_GEMM_SIMT) {
    if (w.fmt != WFMT_INT4) return MOE_ERR_UNSUPPORTED_SHAPE;   // the CUDA-core baseline reads int4 only
    return cuda_status(launch_gemm_simt(p, s));
  }
  const int asrc = (flags & MOE_FLAG_A_SMEM) ? A_SMEM_DQ : A_TMEM_DQ;
  int nt = static_cast<int>((flags >> 8) & 0xFFu);
  const bool auto_nt = nt == 0;
  if (nt == 0) {
    nt = auto_tokens_per_tile(p.R, d.E);
    if (asrc == A_SMEM_DQ && nt > 32) nt = 32;
  }
  if (!p.a_mma_order) {
    if (scratch == nullptr) return MOE_ERR_WORKSPACE_TOO_SMALL;
    const cudaError_t ec = launch_to_mma_order(a, scratch, p.R, p.K, s);
    if (ec != cudaSuccess) return MOE_ERR_CUDA;
    p.a = scratch;
    p.a_mma_order = true;
  }
  // CTA pairs: one pair MMA covers 256 weight rows over two SMs (A in tensor memory only), and
  // each CTA loads half of the token rows, so a 128-token tile's B ring has five stages instead
  // of two. On by request, and by default for the launches of prefill-shaped batches where it
  // measured faster than one CTA per tile (prefill_t4096_zipf): both down launches (1.64 against
  // 1.76 ms together) and the gate/up launch with 128-token tiles (1.50 against 1.58 ms, cold
  // serialised launches); the gate/up launch with 32-token tiles was 5% slower on pairs (0.96
  // against 0.92 ms), and at decode sizes one CTA per tile is as fast or faster.
  const bool pair_req = (flags & MOE_FLAG_GEMM_PAIR) != 0;
  auto launch = [&](const GemmProblem& q, int tiles_nt, bool pair_default) {
    const bool pair = (pair_req || (pair_default && !(flags & MOE_FLAG_A_SMEM))) && asrc == A_TMEM_DQ;
    return pair ? launch_gemm_pair(q, tiles_nt, sms, s) : launch_gemm_tc(q, asrc, tiles_nt, sms, s);
  };
  cudaError_t e;
  if (auto_nt && nt == 128) {
    // Many rows per expert on average, but skewed routing leaves a long tail of experts with a
    // few rows, for which a 128-token tile is mostly padding: experts with up to 32 rows go to a
    // launch with 32-token tiles, the rest to one with 128-token tiles. Each launch keeps only
    // its experts, found from the offsets on the device.
    GemmProblem small = p;
    small.max_rows = 32;
    e = launch(small, 32, op == MOE_GEMM_DOWN);
    if (e == cudaSuccess) {
      GemmProblem big = p;
      big.min_rows = 33;
      e = launch(big, 128, true);
    }
  } else {
    e = launch(p, nt, false);
  }
  if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(e);
}

// The dense shared expert. Its weights make only 2*Is/128 gate/up and H/128 down tiles, fewer
// than the SMs when a small batch fills one token tile; then each GEMM splits its K loop into
// slices (fp32 partial sums in `part`, finished by a second kernel) so that every SM streams
// weights. part may be null (no split). out is bf16, or fp32 with MOE_FLAG_OUT_F32.
moe_status_t run_shared(const moe_dims_t& d, const LayerW& w, const uint16_t* x, int32_t T, uint16_t* hs,
                        void* out, int* status, uint32_t flags, int sms, float* part, cudaStream_t s,
                        bool weights_ready = false) {
  const int Is = w.shared_I;
  GemmProblem p;
  p.weights_ready = weights_ready;
  p.bf16_weights = true;
  p.scales = nullptr;
  p.offsets = nullptr;
  p.status = status;
  p.E = 1;
  p.R = T;
  p.uniform_rows = T;
  p.a_mma_order = false;
  p.out_mma_order = false;
  // gate/up: [T][H] -> hs [T][Is]
  p.op = MOE_GEMM_GATEUP_SILU;
  p.w = w.sh_gu;
  p.a = x;
  p.out = hs;
  p.K = d.H;
  p.rows_per_expert = 2 * Is;
  p.out_cols = Is;
  const int nt = T <= 16 ? 16 : (T <= 32 ? 32 : 64);
  const bool split = part != nullptr && T <= kSplitMaxT && !(flags & MOE_FLAG_GEMM_SIMT);
  const int64_t chunks = (T + nt - 1) / nt;
  if (split) {
    p.ksplit = pick_ksplit(chunks * (Is / 64), (d.H + 255) / 256, sms, T, static_cast<double>(T) * 2 * Is * 4);
    p.partial = part;
  }
  cudaError_t e = (flags & MOE_FLAG_GEMM_SIMT) ? launch_gemm_simt(p, s) : launch_gemm_tc(p, A_SMEM_BF16, nt, sms, s);
  if (e != cudaSuccess) return e == cudaErrorNotSupported ? MOE_ERR_UNSUPPORTED_SHAPE : MOE_ERR_CUDA;
  // down: hs [T][Is] -> out [T][H]
  p.op = MOE_GEMM_DOWN;
  p.w = w.sh_d;
  p.a = hs;
  const bool f32 = (flags & MOE_FLAG_OUT_F32) != 0;
  p.out = f32 ? nullptr : static_cast<uint16_t*>(out);
  p.out_f32 = f32 ? static_cast<float*>(out) : nullptr;
  p.K = Is;
  p.rows_per_expert = d.H;
  p.out_cols = d.H;
  if (split) p.ksplit = pick_ksplit(chunks * ((d.H + 127) / 128), (Is + 255) / 256, sms, T, static_cast<double>(T) * d.H * 4);
  e = (flags & MOE_FLAG_GEMM_SIMT) ? launch_gemm_simt(p, s) : launch_gemm_tc(p, A_SMEM_BF16, nt, sms, s);
  if (e != cudaSuccess) return e == cudaErrorNotSupported ? MOE_ERR_UNSUPPORTED_SHAPE : MOE_ERR_CUDA;
  return MOE_OK;
}

// The router's logit projection, logits fp32 [T][E] = x [T][H] * Wg^T (Wg bf16 [E][H]), on the
// bf16 tensor-core kernel: the gate's E rows are the weight rows, the tokens the narrow operand,
// fp32 rows out. Small batches split K as the shared expert does (part may be null: no split).
moe_status_t run_router(const uint16_t* x, const uint16_t* wg, int32_t T, int32_t E, int32_t H, float* logits,
                        int* status, uint32_t flags, int sms, float* part, cudaStream_t s) {
  GemmProblem p;   // weights_ready stays false: the gate matrix is the caller's, the first read of the call
  p.op = MOE_GEMM_DOWN;
  p.bf16_weights = true;
  p.w = wg;
  p.scales = nullptr;
  p.a = x;
  p.offsets = nullptr;
  p.out = nullptr;
  p.out_f32 = logits;
  p.status = status;
  p.E = 1;
  p.K = H;
  p.rows_per_expert = E;
  p.out_cols = E;
  p.R = T;
  p.uniform_rows = T;
  p.a_mma_order = false;
  p.out_mma_order = false;
  const int nt = T <= 16 ? 16 : (T <= 32 ? 32 : 64);
  if (part != nullptr && T <= kSplitMaxT && !(flags & MOE_FLAG_GEMM_SIMT)) {
    const int64_t chunks = (T + nt - 1) / nt;
    p.ksplit = pick_ksplit(chunks * ((E + 127) / 128), (H + 255) / 256, sms, T, static_cast<double>(T) * E * 4);
    p.partial = part;
  }
  const cudaError_t e =
      (flags & MOE_FLAG_GEMM_SIMT) ? launch_gemm_simt(p, s) : launch_gemm_tc(p, A_SMEM_BF16, nt, sms, s);
  if (e != cudaSuccess) return e == cudaErrorNotSupported ? MOE_ERR_UNSUPPORTED_SHAPE : MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t check_router(const uint16_t* x, const uint16_t* wg, int32_t T, int32_t E, int32_t H) {
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > 1024 || H < 32 || H % 32 || H > kMaxDim) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T > 0 && (x == nullptr || wg == nullptr || !aligned16(x) || !aligned16(wg))) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// A host bank staged into the device bank before the GEMMs (moe_forward_offload).
struct Staging {
  const void* src[4];   // device-accessible addresses of the host bank's w13, s13, w2, s2
  void* dst[4];         // the device bank's
  int64_t bytes[4];     // per expert
};

int64_t bank_bytes_per_expert(const moe_dims_t& d, int i) {
  const int64_t H = d.H, I = d.I;
  switch (i) {
    case 0: return 2 * I * (H / 8) * 4;
    case 1: return 2 * I * (H / 32) * 2;
    case 2: return H * (I / 8) * 4;
    default: return H * (I / 32) * 2;
  }
}

// Device-accessible addresses of a host bank: each tensor must be page-locked host memory mapped
// into the device's address space (cudaHostAlloc / pinned memory on a unified-addressing system).
// An error the caller left pending stays as it was.
moe_status_t host_bank(const moe_dims_t& d, const moe_weights_t* hw, const moe_weights_t* dw, Staging* st) {
  const void* h[4] = {hw->w13_packed, hw->w13_scale, hw->w2_packed, hw->w2_scale};
  void* dv[4] = {const_cast<int32_t*>(dw->w13_packed), const_cast<uint16_t*>(dw->w13_scale),
                 const_cast<int32_t*>(dw->w2_packed), const_cast<uint16_t*>(dw->w2_scale)};
  const cudaError_t pending = cudaPeekAtLastError();
  for (int i = 0; i < 4; ++i) {
    void* p = nullptr;
    if (cudaHostGetDevicePointer(&p, const_cast<void*>(h[i]), 0) != cudaSuccess || p == nullptr ||
        !aligned16(p)) {
      if (pending == cudaSuccess) (void)cudaGetLastError();
      return MOE_ERR_INVALID_ARG;
    }
    st->src[i] = p;
    st->dst[i] = dv[i];
    st->bytes[i] = bank_bytes_per_expert(d, i);
  }
  return MOE_OK;
}

// One layer. residual (nullable, [T][H]) is added to the output in the combine's fp32 sum.
moe_status_t forward_device(const moe_dims_t& d, const LayerW& w, const uint16_t* x, const float* logits,
                            int32_t T, const uint16_t* residual, uint16_t* out, uint8_t* ws, uint32_t flags, int sms,
                            cudaStream_t s, const Staging* stage = nullptr) {
  const Layout L = layout(d, T, w.shared_I);
  int* status = reinterpret_cast<int*>(ws);
  int32_t* ids = reinterpret_cast<int32_t*>(ws + L.ids);
  float* tw = reinterpret_cast<float*>(ws + L.w);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  int32_t* sorted = reinterpret_cast<int32_t*>(ws + L.sorted);
  int32_t* inv = reinterpret_cast<int32_t*>(ws + L.inv);
  int32_t* hist = reinterpret_cast<int32_t*>(ws + L.hist);
  uint16_t* xperm = reinterpret_cast<uint16_t*>(ws + L.xperm);
  uint16_t* h = reinterpret_cast<uint16_t*>(ws + L.h);
  float* y = reinterpret_cast<float*>(ws + L.y);
  const int R = T * d.top_k;
  // the tensor-core GEMMs exchange activation rows in their K order; the CUDA-core path in natural order
  const bool mma_order = (flags & MOE_FLAG_GEMM_SIMT) == 0;
  cudaError_t e = launch_route(logits, T, d.E, d.top_k, ids, tw, s);
  if (e == cudaSuccess) e = launch_permute(ids, T, d.E, d.top_k, offsets, sorted, inv, hist, status, s);
  if (e == cudaSuccess) e = launch_gather(x, sorted, offsets, d.E, R, d.H, mma_order, xperm, s);
  if (e == cudaSuccess && stage != nullptr)   // the touched experts, host bank -> device bank
    e = launch_stage_experts(stage->src, stage->dst, stage->bytes, offsets, d.E, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  // A GEMM with weights_ready reads the bank and the offsets without waiting for its predecessor.
  // The offsets are complete by then because the gather kernel sits between the permutation and
  // the GEMM: it waits for the permutation to finish before it lets the GEMM launch. (A kernel that
  // wrote the offsets and then let the GEMM launch directly would race with it.) A bank staged by
  // this call is the predecessor's own output, so those GEMMs wait.
  const bool ready = stage == nullptr;
  moe_status_t st = run_grouped_gemm(MOE_GEMM_GATEUP_SILU, d, w, xperm, T, offsets, h, status, flags, mma_order,
                                     nullptr, sms, s, ready);
  if (st != MOE_OK) return st;
  // y (and the shared expert's output) stay fp32 until the combine's one bf16 rounding
  st = run_grouped_gemm(MOE_GEMM_DOWN, d, w, h, T, offsets, y, status, flags | MOE_FLAG_OUT_F32, mma_order, nullptr,
                        sms, s, ready);
  if (st != MOE_OK) return st;
  const float* addend = nullptr;
  if (w.sh_gu != nullptr) {
    uint16_t* hs = reinterpret_cast<uint16_t*>(ws + L.hs);
    float* ys = reinterpret_cast<float*>(ws + L.ys);
    float* part = L.part_bytes > 0 ? reinterpret_cast<float*>(ws + L.part) : nullptr;
    st = run_shared(d, w, x, T, hs, ys, status, flags | MOE_FLAG_OUT_F32, sms, part, s, true);
    if (st != MOE_OK) return st;
    addend = ys;
  }
  return cuda_status(launch_combine(y, inv, tw, T, d.top_k, d.H, addend, residual, true, out, s));
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE_BOUNDS: return "expert id out of range";
    case MOE_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
  }
  return "unknown status";
}

size_t moe_workspace_size(moe_dims_t d, int32_t T, int32_t shared_I, uint32_t flags) {
  if ((check_dims(d) != MOE_OK && check_dims(d, WFMT_FP4) != MOE_OK) || check_T(T, d.top_k) != MOE_OK || shared_I < 0)
    return 0;
  return layout(d, T, shared_I, (flags & MOE_FLAG_ROUTER_PROJECT) != 0).end;
}

size_t moe_router_workspace_size(int32_t T, int32_t E, int32_t H) {
  if (T < 0 || E < 1 || E > 1024 || H < 32 || H % 32 || H > kMaxDim) return 0;
  return 256 + align256(split_part_bytes(T, E));
}

size_t moe_host_staging_size(moe_dims_t d, int32_t T) {
  if (check_dims(d) != MOE_OK || check_T(T, d.top_k) != MOE_OK) return 0;
  return align256(static_cast<size_t>(T) * d.H * 2) * 2 + align256(static_cast<size_t>(T) * d.E * 4);
}

moe_status_t moe_route(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* topk_ids, float* topk_w,
                       void* stream) {
  CallRange range_("moe_route");
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > 1024 || k < 1 || k > E) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return MOE_OK;
  if (logits == nullptr || topk_ids == nullptr || topk_w == nullptr) return MOE_ERR_INVALID_ARG;
  DevInfo di;
  moe_status_t st = current_device(&di);
  if (st != MOE_OK) return st;
  return cuda_status(launch_route(logits, T, E, k, topk_ids, topk_w, as_stream(stream)));
}

moe_status_t moe_router_logits(const uint16_t* x, const uint16_t* w_gate, int32_t T, int32_t E, int32_t H,
                               float* logits, void* ws, size_t ws_bytes, uint32_t flags, void* stream) {
  CallRange range_("moe_router_logits");
  moe_status_t st = check_router(x, w_gate, T, E, H);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (logits == nullptr || ws == nullptr || !aligned16(logits) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_router_workspace_size(T, E, H)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  DevInfo di;
  if ((st = current_device(&di)) != MOE_OK) return st;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  float* part = split_part_bytes(T, E) > 0 ? reinterpret_cast<float*>(w8 + 256) : nullptr;
  return run_router(x, w_gate, T, E, H, logits, reinterpret_cast<int*>(w8), flags, di.sms, part, as_stream(stream));
}

moe_status_t moe_route_project(const uint16_t* x, const uint16_t* w_gate, int32_t T, int32_t E, int32_t H, int32_t k,
                               float* logits, int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes,
                               uint32_t flags, void* stream) {
  CallRange range_("moe_route_project");
  if (k < 1 || k > E) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T > 0 && (topk_ids == nullptr || topk_w == nullptr)) return MOE_ERR_INVALID_ARG;
  moe_status_t st = moe_router_logits(x, w_gate, T, E, H, logits, ws, ws_bytes, flags, stream);
  if (st != MOE_OK || T == 0) return st;
  return cuda_status(launch_route(logits, T, E, k, topk_ids, topk_w, as_stream(stream)));
}

moe_status_t moe_sigmoid_scores(const float* logits, int64_t n, float* scores, void* stream) {
  CallRange range_("moe_sigmoid_scores");
  if (n < 0) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (logits == nullptr || scores == nullptr) return MOE_ERR_INVALID_ARG;
  DevInfo di;
  moe_status_t st = current_device(&di);
  if (st != MOE_OK) return st;
  return cuda_status(launch_sigmoid(logits, n, scores, as_stream(stream)));
}

moe_status_t moe_permute(const int32_t* topk_ids, int32_t T, int32_t E, int32_t k, int32_t* expert_offsets,
                         int32_t* sorted_token_ids, int32_t* inv_perm, const uint16_t* x, int32_t H,
                         uint16_t* x_perm, void* ws, size_t ws_bytes, uint32_t flags, void* stream) {
  CallRange range_("moe_permute");
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > 1024 || k < 1 || k > E) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (check_T(T, k) != MOE_OK) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return MOE_OK;
  if (topk_ids == nullptr || expert_offsets == nullptr || sorted_token_ids == nullptr || inv_perm == nullptr ||
      ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  const bool gather = x != nullptr && x_perm != nullptr;
  if ((x != nullptr) != (x_perm != nullptr)) return MOE_ERR_INVALID_ARG;
  if (gather && (H < 8 || H % 8 || !aligned16(x) || !aligned16(x_perm))) return MOE_ERR_INVALID_ARG;
  const int64_t Tk = static_cast<int64_t>(T) * k;
  const size_t need = 256 + static_cast<size_t>(permute_blocks(Tk)) * E * 4;
  if (ws_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
  DevInfo di;
  moe_status_t st = current_device(&di);
  if (st != MOE_OK) return st;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  cudaStream_t s = as_stream(stream);
  cudaError_t e = launch_permute(topk_ids, T, E, k, expert_offsets, sorted_token_ids, inv_perm,
                                 reinterpret_cast<int32_t*>(w8 + 256), reinterpret_cast<int*>(w8), s);
  if (e == cudaSuccess && gather)
    e = launch_gather(x, sorted_token_ids, expert_offsets, E, static_cast<int>(Tk), H,
                      (flags & MOE_FLAG_ROWS_MMA_ORDER) != 0, x_perm, s);
  return cuda_status(e);
}

moe_status_t moe_w4a16_grouped_gemm(int32_t op, moe_dims_t d, const moe_weights_t* w, const uint16_t* a_rows,
                                    int32_t T, const int32_t* expert_offsets, uint16_t* out_rows, void* ws,
                                    size_t ws_bytes, uint32_t flags, void* stream) {
  CallRange range_("moe_w4a16_grouped_gemm");
  if (op != MOE_GEMM_GATEUP_SILU && op != MOE_GEMM_DOWN) return MOE_ERR_INVALID_ARG;
  if (op == MOE_GEMM_GATEUP_SILU && (flags & MOE_FLAG_OUT_F32)) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_dims(d);
  if (st != MOE_OK) return st;
  if ((st = check_T(T, d.top_k)) != MOE_OK) return st;
  if ((st = check_weights(w, false)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (a_rows == nullptr || expert_offsets == nullptr || out_rows == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(a_rows) || !aligned16(out_rows) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  const bool rows_mma = (flags & MOE_FLAG_ROWS_MMA_ORDER) != 0;
  const size_t K = (op == MOE_GEMM_GATEUP_SILU) ? d.H : d.I;
  const bool convert = !rows_mma && !(flags & MOE_FLAG_GEMM_SIMT);
  const size_t need = 256 + (convert ? align256(static_cast<size_t>(T) * d.top_k * K * 2) : 0);
  if (ws_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
  DevInfo di;
  if ((st = current_device(&di)) != MOE_OK) return st;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  return run_grouped_gemm(op, d, layer_w(w), a_rows, T, expert_offsets, static_cast<void*>(out_rows), reinterpret_cast<int*>(w8),
                          flags, rows_mma,
                          convert ? reinterpret_cast<uint16_t*>(w8 + 256) : nullptr, di.sms, as_stream(stream));
}

moe_status_t moe_shared_expert(moe_dims_t d, const moe_weights_t* w, const uint16_t* x, int32_t T, uint16_t* out,
                               void* ws, size_t ws_bytes, uint32_t flags, void* stream) {
  CallRange range_("moe_shared_expert");
  moe_status_t st = check_dims(d);
  if (st != MOE_OK) return st;
  if ((st = check_T(T, d.top_k)) != MOE_OK) return st;
  if (w == nullptr) return MOE_ERR_INVALID_ARG;
  if (w->shared_wgu == nullptr || w->shared_wd == nullptr || !aligned16(w->shared_wgu) || !aligned16(w->shared_wd))
    return MOE_ERR_INVALID_ARG;
  if (w->shared_I < 64 || w->shared_I % 64 || w->shared_I > kMaxDim) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return MOE_OK;
  if (x == nullptr || out == nullptr || ws == nullptr || !aligned16(x) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  const Layout L = layout(d, T, w->shared_I);
  if (ws_bytes < L.end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  DevInfo di;
  if ((st = current_device(&di)) != MOE_OK) return st;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  float* part = L.part_bytes > 0 ? reinterpret_cast<float*>(w8 + L.part) : nullptr;
  return run_shared(d, layer_w(w), x, T, reinterpret_cast<uint16_t*>(w8 + L.hs), out, reinterpret_cast<int*>(w8), flags,
                    di.sms, part, as_stream(stream));
}

moe_status_t moe_combine(const uint16_t* y_rows, const int32_t* inv_perm, const float* topk_w, int32_t T, int32_t k,
                         int32_t H, const uint16_t* addend, uint16_t* out, void* stream) {
  CallRange range_("moe_combine");
  if (T < 0 || k < 1 || H < 8 || H % 8) return MOE_ERR_INVALID_ARG;
  if (check_T(T, k) != MOE_OK) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return MOE_OK;
  if (y_rows == nullptr || inv_perm == nullptr || topk_w == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_rows) || !aligned16(out) || (addend != nullptr && !aligned16(addend))) return MOE_ERR_INVALID_ARG;
  DevInfo di;
  moe_status_t st = current_device(&di);
  if (st != MOE_OK) return st;
  return cuda_status(launch_combine(y_rows, inv_perm, topk_w, T, k, H, addend, nullptr, false, out, as_stream(stream)));
}

moe_status_t moe_combine_f32(const float* y_rows, const int32_t* inv_perm, const float* topk_w, int32_t T, int32_t k,
                             int32_t H, const float* addend, uint16_t* out, void* stream) {
  CallRange range_("moe_combine_f32");
  if (T < 0 || k < 1 || H < 8 || H % 8) return MOE_ERR_INVALID_ARG;
  if (check_T(T, k) != MOE_OK) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return MOE_OK;
  if (y_rows == nullptr || inv_perm == nullptr || topk_w == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_rows) || !aligned16(out) || (addend != nullptr && !aligned16(addend))) return MOE_ERR_INVALID_ARG;
  DevInfo di;
  moe_status_t st = current_device(&di);
  if (st != MOE_OK) return st;
  return cuda_status(launch_combine(y_rows, inv_perm, topk_w, T, k, H, addend, nullptr, true, out, as_stream(stream)));
}

moe_status_t moe_forward(moe_dims_t d, const moe_weights_t* w, const uint16_t* x, const float* logits, int32_t T,
                         uint16_t* out, void* ws, size_t ws_bytes, uint32_t flags, void* stream) {
  CallRange range_("moe_forward");
  moe_status_t st = check_dims(d);
  if (st != MOE_OK) return st;
  if ((st = check_T(T, d.top_k)) != MOE_OK) return st;
  if ((st = check_weights(w, false)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (x == nullptr || logits == nullptr || out == nullptr || ws == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < layout(d, T, w->shared_I).end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  DevInfo di;
  if ((st = current_device(&di)) != MOE_OK) return st;
  return forward_device(d, layer_w(w), x, logits, T, nullptr, out, static_cast<uint8_t*>(ws), flags, di.sms,
                        as_stream(stream));
}

moe_status_t moe_fp4_grouped_gemm(int32_t op, moe_dims_t d, const moe_weights_fp4_t* w, const uint16_t* a_rows,
                                  int32_t T, const int32_t* expert_offsets, uint16_t* out_rows, void* ws,
                                  size_t ws_bytes, uint32_t flags, void* stream) {
  CallRange range_("moe_fp4_grouped_gemm");
  if (op != MOE_GEMM_GATEUP_SILU && op != MOE_GEMM_DOWN) return MOE_ERR_INVALID_ARG;
  if (op == MOE_GEMM_GATEUP_SILU && (flags & MOE_FLAG_OUT_F32)) return MOE_ERR_INVALID_ARG;
  if (flags & (MOE_FLAG_GEMM_SIMT | MOE_FLAG_A_SMEM)) return MOE_ERR_UNSUPPORTED_SHAPE;
  moe_status_t st = check_dims(d, WFMT_FP4);
  if (st != MOE_OK) return st;
  if ((st = check_T(T, d.top_k)) != MOE_OK) return st;
  if ((st = check_weights_fp4(w)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (a_rows == nullptr || expert_offsets == nullptr || out_rows == nullptr || ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(a_rows) || !aligned16(out_rows) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  const bool rows_mma = (flags & MOE_FLAG_ROWS_MMA_ORDER) != 0;
  const size_t K = (op == MOE_GEMM_GATEUP_SILU) ? d.H : d.I;
  const size_t need = 256 + (rows_mma ? 0 : align256(static_cast<size_t>(T) * d.top_k * K * 2));
  if (ws_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
  DevInfo di;
  if ((st = current_device(&di)) != MOE_OK) return st;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  return run_grouped_gemm(op, d, layer_w(w), a_rows, T, expert_offsets, static_cast<void*>(out_rows),
                          reinterpret_cast<int*>(w8), flags, rows_mma,
                          rows_mma ? nullptr : reinterpret_cast<uint16_t*>(w8 + 256), di.sms, as_stream(stream));
}

moe_status_t moe_forward_fp4(moe_dims_t d, const moe_weights_fp4_t* w, const uint16_t* x, const float* logits,
                             int32_t T, uint16_t* out, void* ws, size_t ws_bytes, uint32_t flags, void* stream) {
  CallRange range_("moe_forward_fp4");
  if (flags & (MOE_FLAG_GEMM_SIMT | MOE_FLAG_A_SMEM)) return MOE_ERR_UNSUPPORTED_SHAPE;
  moe_status_t st = check_dims(d, WFMT_FP4);
  if (st != MOE_OK) return st;
  if ((st = check_T(T, d.top_k)) != MOE_OK) return st;
  if ((st = check_weights_fp4(w)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (x == nullptr || logits == nullptr || out == nullptr || ws == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < layout(d, T, w->shared_I).end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  DevInfo di;
  if ((st = current_device(&di)) != MOE_OK) return st;
  return forward_device(d, layer_w(w), x, logits, T, nullptr, out, static_cast<uint8_t*>(ws), flags, di.sms,
                        as_stream(stream));
}

moe_status_t moe_stage_experts(moe_dims_t d, const moe_weights_t* host_w, const int32_t* expert_offsets,
                               const moe_weights_t* dev_w, void* stream) {
  CallRange range_("moe_stage_experts");
  moe_status_t st = check_dims(d);
  if (st != MOE_OK) return st;
  if ((st = check_weights(host_w, false)) != MOE_OK) return st;
  if ((st = check_weights(dev_w, false)) != MOE_OK) return st;
  if (expert_offsets == nullptr) return MOE_ERR_INVALID_ARG;
  DevInfo di;
  if ((st = current_device(&di)) != MOE_OK) return st;
  Staging sg;
  if ((st = host_bank(d, host_w, dev_w, &sg)) != MOE_OK) return st;
  return cuda_status(launch_stage_experts(sg.src, sg.dst, sg.bytes, expert_offsets, d.E, as_stream(stream)));
}

moe_status_t moe_forward_offload(moe_dims_t d, const moe_weights_t* host_w, const moe_weights_t* dev_w,
                                 const uint16_t* x, const float* logits, int32_t T, uint16_t* out, void* ws,
                                 size_t ws_bytes, uint32_t flags, void* stream) {
  CallRange range_("moe_forward_offload");
  moe_status_t st = check_dims(d);
  if (st != MOE_OK) return st;
  if ((st = check_T(T, d.top_k)) != MOE_OK) return st;
  if ((st = check_weights(host_w, false)) != MOE_OK) return st;
  if ((st = check_weights(dev_w, false)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (x == nullptr || logits == nullptr || out == nullptr || ws == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < layout(d, T, dev_w->shared_I).end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  DevInfo di;
  if ((st = current_device(&di)) != MOE_OK) return st;
  Staging sg;
  if ((st = host_bank(d, host_w, dev_w, &sg)) != MOE_OK) return st;
  return forward_device(d, layer_w(dev_w), x, logits, T, nullptr, out, static_cast<uint8_t*>(ws), flags, di.sms,
                        as_stream(stream), &sg);
}

moe_status_t moe_forward_project(moe_dims_t d, const moe_weights_t* w, const uint16_t* w_gate, const uint16_t* x,
                                 int32_t T, uint16_t* out, void* ws, size_t ws_bytes, uint32_t flags, void* stream) {
  CallRange range_("moe_forward_project");
  moe_status_t st = check_dims(d);
  if (st != MOE_OK) return st;
  if ((st = check_T(T, d.top_k)) != MOE_OK) return st;
  if ((st = check_weights(w, false)) != MOE_OK) return st;
  if ((st = check_router(x, w_gate, T, d.E, d.H)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (out == nullptr || ws == nullptr || !aligned16(out) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  const Layout L = layout(d, T, w->shared_I, true);
  if (ws_bytes < L.end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  DevInfo di;
  if ((st = current_device(&di)) != MOE_OK) return st;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  float* logits = reinterpret_cast<float*>(w8 + L.logits);
  float* part = L.rpart_bytes > 0 ? reinterpret_cast<float*>(w8 + L.rpart) : nullptr;
  cudaStream_t s = as_stream(stream);
  st = run_router(x, w_gate, T, d.E, d.H, logits, reinterpret_cast<int*>(w8), flags, di.sms, part, s);
  if (st != MOE_OK) return st;
  return forward_device(d, layer_w(w), x, logits, T, nullptr, out, w8, flags, di.sms, s);
}

moe_status_t moe_forward_host(moe_dims_t d, const moe_weights_t* w, const uint16_t* x_host, const float* logits_host,
                              int32_t T, uint16_t* out_host, void* ws, size_t ws_bytes, uint32_t flags,
                              void* stream) {
  CallRange range_("moe_forward_host");
  moe_status_t st = check_dims(d);
  if (st != MOE_OK) return st;
  if ((st = check_T(T, d.top_k)) != MOE_OK) return st;
  if ((st = check_weights(w, false)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (x_host == nullptr || logits_host == nullptr || out_host == nullptr || ws == nullptr || !aligned16(ws))
    return MOE_ERR_INVALID_ARG;
  const size_t base = layout(d, T, w->shared_I).end;
  if (ws_bytes < base + moe_host_staging_size(d, T)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  DevInfo di;
  if ((st = current_device(&di)) != MOE_OK) return st;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  const size_t xb = static_cast<size_t>(T) * d.H * 2, lb = static_cast<size_t>(T) * d.E * 4;
  uint16_t* dx = reinterpret_cast<uint16_t*>(w8 + base);
  float* dl = reinterpret_cast<float*>(w8 + base + align256(xb));
  uint16_t* dout = reinterpret_cast<uint16_t*>(w8 + base + align256(xb) + align256(lb));
  cudaStream_t s = as_stream(stream);
  if (cudaMemcpyAsync(dx, x_host, xb, cudaMemcpyHostToDevice, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpyAsync(dl, logits_host, lb, cudaMemcpyHostToDevice, s) != cudaSuccess) return MOE_ERR_CUDA;
  st = forward_device(d, layer_w(w), dx, dl, T, nullptr, dout, w8, flags, di.sms, s);
  if (st != MOE_OK) return st;
  return cuda_status(cudaMemcpyAsync(out_host, dout, xb, cudaMemcpyDeviceToHost, s));
}

moe_status_t moe_check_status(void* ws, void* stream) {
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (v != 0 && cudaMemset(ws, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status_t>(v);
}

moe_status_t moe_rmsnorm(const uint16_t* x, int32_t T, int32_t H, float eps, uint16_t* out, void* stream) {
  CallRange range_("moe_rmsnorm");
  if (T < 0 || H < 8 || H % 8 || H > kMaxDim || !(eps >= 0.0f)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (x == nullptr || out == nullptr || !aligned16(x) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  DevInfo di;
  moe_status_t st = current_device(&di);
  if (st != MOE_OK) return st;
  return cuda_status(launch_rmsnorm(x, T, H, eps, out, as_stream(stream)));
}

size_t moe_stack_workspace_size(moe_dims_t d, int32_t T, int32_t shared_I, uint32_t flags) {
  const size_t base = moe_workspace_size(d, T, shared_I, flags);
  if (base == 0) return 0;
  return base + 3 * align256(static_cast<size_t>(T) * d.H * 2);
}

moe_status_t moe_stack_forward(moe_dims_t d, const moe_weights_t* layers, int32_t L, const float* const* logits,
                               const uint16_t* x, int32_t T, float eps, uint16_t* out, void* ws, size_t ws_bytes,
                               uint32_t flags, void* stream) {
  CallRange range_("moe_stack_forward");
  moe_status_t st = check_dims(d);
  if (st != MOE_OK) return st;
  if ((st = check_T(T, d.top_k)) != MOE_OK) return st;
  if (L < 1 || layers == nullptr || logits == nullptr || !(eps >= 0.0f)) return MOE_ERR_INVALID_ARG;
  int32_t shared_I = 0;
  for (int32_t l = 0; l < L; ++l) {
    if ((st = check_weights(&layers[l], false)) != MOE_OK) return st;
    if (l > 0 && layers[l].shared_I != shared_I) return MOE_ERR_INVALID_ARG;   // one workspace layout for all
    shared_I = layers[l].shared_I;
  }
  if (T == 0) return MOE_OK;
  if (x == nullptr || out == nullptr || ws == nullptr || !aligned16(x) || !aligned16(out) || !aligned16(ws))
    return MOE_ERR_INVALID_ARG;
  for (int32_t l = 0; l < L; ++l)
    if (logits[l] == nullptr) return MOE_ERR_INVALID_ARG;
  const size_t base = layout(d, T, shared_I).end;
  const size_t xb = align256(static_cast<size_t>(T) * d.H * 2);
  if (ws_bytes < base + 3 * xb) return MOE_ERR_WORKSPACE_TOO_SMALL;
  DevInfo di;
  if ((st = current_device(&di)) != MOE_OK) return st;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  uint16_t* xn = reinterpret_cast<uint16_t*>(w8 + base);
  uint16_t* ping[2] = {reinterpret_cast<uint16_t*>(w8 + base + xb), reinterpret_cast<uint16_t*>(w8 + base + 2 * xb)};
  cudaStream_t s = as_stream(stream);
  const uint16_t* cur = x;
  for (int32_t l = 0; l < L; ++l) {
    uint16_t* next = (l == L - 1) ? out : ping[l & 1];
    if (launch_rmsnorm(cur, T, d.H, eps, xn, s) != cudaSuccess) return MOE_ERR_CUDA;
    st = forward_device(d, layer_w(&layers[l]), xn, logits[l], T, cur, next, w8, flags, di.sms, s);
    if (st != MOE_OK) return st;
    cur = next;
  }
  return MOE_OK;
}

uint64_t moe_launch_count(void) { return moe::g_launches.load(std::memory_order_relaxed); }

moe_status_t moe_debug_expire_wait(void* ws, int64_t timeout_ns, void* stream) {
  CallRange range_("moe_debug_expire_wait");
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  if (timeout_ns < 1000000) timeout_ns = 1000000;
  if (timeout_ns > 2000000000) timeout_ns = 2000000000;
  DevInfo di;
  moe_status_t st = current_device(&di);
  if (st != MOE_OK) return st;
  return cuda_status(launch_expire_wait(static_cast<int*>(ws), timeout_ns, as_stream(stream)));
}

}  // extern "C"
