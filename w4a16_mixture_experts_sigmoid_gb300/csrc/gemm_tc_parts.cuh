// Pieces shared by the two tensor-core grouped-GEMM kernels (one CTA per tile in
// gemm_tc.cu; a CTA pair per tile in gemm_pair.cu): the kernel parameters, the
// tile decode of the persistent schedule, the int4 -> bf16 dequantisation, the
// barrier arithmetic of the A buffers, and the host-side tensor-map encoding.
// Included by those two translation units only.
#pragma once

#include "common.cuh"
#include "internal.h"

#include <mutex>

namespace moe {
namespace tc {

constexpr int BM = 128;            // weight rows per tile (MMA M)
constexpr int BK = 256;            // K per pipeline stage
constexpr int KSUB = 64;           // K per 128-byte swizzle row
constexpr int NSUB = BK / KSUB;    // swizzle sub-tiles per stage
constexpr int kThreads = 512;      // 16 warps, 128 registers a thread
constexpr int kFirstDqWarp = 2;
constexpr int kFirstEpiWarp = 10;
constexpr int kBProducerWarp = 14;
constexpr int kSecondMmaWarp = 15;
constexpr int kMaxE = 1024;
constexpr int kSmemLimit = 232448;  // dynamic shared memory per CTA on sm_100-class parts
constexpr int kAlignSlack = 1024;
constexpr int kAuxBytes = 7168;

struct TcParams {
  CUtensorMap tm_w;  // int4 words [rows_total][K/8] (box 32 x 64) or bf16 weights [rows_total][K] (box 64 x 16)
  CUtensorMap tm_s;  // bf16 scales [rows_total][K/32] (box 8 x 64), when scale_tma
  CUtensorMap tm_b;  // bf16 token rows [R][K] (box 64 x NT)
  const uint16_t* scales;  // int4: bf16 [rows][K/32]; fp4: E4M3 bytes [rows][K/16] (read through a byte pointer)
  const float* gscale;     // fp4: per-expert fp32 scale, applied to the fp32 sums in the epilogue
  const int32_t* offsets;
  uint16_t* out;
  float* out_f32;          // down: fp32 rows instead of bf16 `out`, when set
  int* status;
  int E, K, rows_per_expert, out_cols, uniform_rows, scale_tma, rows_total, R, out_mma_order;
  int min_rows, max_rows;  // experts outside [min_rows, max_rows] rows are left to another launch
  int weights_ready;       // 0: the tile table and the weight stream wait for the predecessor grid
  int ksplit;              // K slices per tile (1: whole K); > 1 (bf16 weights only) writes fp32 partial sums
  float* partial;          // [ksplit][R][2][I] (gate/up) or [ksplit][R][H] (down), when ksplit > 1
  unsigned long long timeout_ns;
};

// Shared memory holds two rings. The weight ring (int4 words + scales, or
// dense bf16 weights) is released by the dequant warps as soon as they have
// the stage in registers, so HBM streaming never waits on the tensor pipe; the
// token-row ring (operand B) is released by the MMA commit. With dense bf16
// weights the MMA reads both, and the two rings advance in lock step.
struct TileInfo {
  int wt;      // weight tile (128 rows; for gate/up 64 gate + 64 up rows)
  int e;       // expert
  int row0;    // first token row of the chunk
  int nvalid;  // token rows of the chunk that belong to the expert
  int split;   // K slice: stages [split * nk, (split + 1) * nk) of the whole K loop
};

__device__ __forceinline__ TileInfo decode_tile(int i, int n_act, const int16_t* act_e, const int* tpre,
                                                const TcParams& p, int nt, int ksplit) {
  int lo = 0, hi = n_act - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tpre[mid] <= i) lo = mid;
    else hi = mid - 1;
  }
  TileInfo t;
  t.e = act_e[lo];
  int start, cnt;
  if (p.uniform_rows >= 0) { start = 0; cnt = p.uniform_rows; }
  else { start = p.offsets[t.e]; cnt = p.offsets[t.e + 1] - start; }
  const int nch = (cnt + nt - 1) / nt;
  int rem = i - tpre[lo];
  t.split = 0;
  if (ksplit > 1) {
    t.split = rem % ksplit;
    rem /= ksplit;
  }
  t.wt = rem / nch;
  const int c = rem - t.wt * nch;
  t.row0 = start + c * nt;
  t.nvalid = min(nt, cnt - c * nt);
  return t;
}

// Bounded wait by every lane of a warp, with a warp-uniform verdict: lanes that
// saw the phase complete and lanes that timed out or saw the abort flag agree
// on one outcome, so no .sync.aligned instruction runs with part of the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const TcParams& p, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, p.timeout_ns, abort_flag, p.status);
  return __all_sync(0xFFFFFFFFu, ok);
}

// MMA issue in one of two forms, chosen per kernel at compile time. WARP: the whole issuer warp
// runs the loop in lockstep (warp_wait) and one elected lane issues each MMA and commit (the
// *_elect forms); with 128-token tiles this made the gate/up GEMM 2% and the pair down GEMM 7%
// faster at prefill. Otherwise lane 0 alone runs the loop, which measured 4% faster for the
// 16- to 64-token tiles of decode.
template <bool WARP>
__device__ __forceinline__ bool iss_wait(uint64_t* bar, uint32_t parity, const TcParams& p, volatile int* abort_flag) {
  if (WARP) return warp_wait(bar, parity, p, abort_flag);
  return mbar_wait(bar, parity, p.timeout_ns, abort_flag, p.status);
}

template <bool WARP>
__device__ __forceinline__ void iss_mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if (WARP) mma_ts_elect(d, a, b, idesc, acc);
  else mma_ts(d, a, b, idesc, acc);
}

template <bool WARP>
__device__ __forceinline__ void iss_mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if (WARP) mma_ss_elect(d, a, b, idesc, acc);
  else mma_ss(d, a, b, idesc, acc);
}

template <bool WARP>
__device__ __forceinline__ void iss_commit(uint64_t* bar) {
  if (WARP) mma_commit_elect(bar);
  else mma_commit(bar);
}

// The same with cluster-scope acquire (barriers that the peer CTA of a pair arrives on).
__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity, const TcParams& p,
                                                  volatile int* abort_flag) {
  const bool ok = mbar_wait_cluster(bar, parity, p.timeout_ns, abort_flag, p.status);
  return __all_sync(0xFFFFFFFFu, ok);
}

template <bool WARP>
__device__ __forceinline__ bool iss_wait_cluster(uint64_t* bar, uint32_t parity, const TcParams& p,
                                                 volatile int* abort_flag) {
  if (WARP) return warp_wait_cluster(bar, parity, p, abort_flag);
  return mbar_wait_cluster(bar, parity, p.timeout_ns, abort_flag, p.status);
}

template <bool WARP>
__device__ __forceinline__ void iss_mma_ts_pair(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if (WARP) mma_ts_pair_elect(d, a, b, idesc, acc);
  else mma_ts_pair(d, a, b, idesc, acc);
}

template <bool WARP>
__device__ __forceinline__ void iss_commit_pair(uint64_t* bar, uint16_t mask) {
  if (WARP) mma_commit_pair_elect(bar, mask);
  else mma_commit_pair(bar, mask);
}

// One 16-byte chunk = four int32 words = 32 inputs of one scale group ->
// 16 bf16x2 registers in MMA K order: register 4i+m holds bf16(q*s) of inputs
// 8i+m (low half) and 8i+m+4 (high half) of the chunk, q = nibble - 8. Two
// exact forms; both round the exact product q*s once to nearest even, so they
// agree bit for bit (up to the sign of a zero product):
// * FAST, for 2^-126 <= |s| < 2^-5 (exponent field 1..121, which holds for
//   every practical int4 group scale): bits 0..7 of a bf16 read as a linear
//   field, b * 2^-133 for every b < 256 (the subnormals and the first normal
//   binade), so a nibble n masked in place at bits 0..3 of a half is
//   n * 2^-133 and at bits 4..7 is n * 2^-129. One packed fma with
//   S = s * 2^133 or s * 2^129 (133 or 129 added to s's exponent field, still
//   a normal bf16) and C = -8 s (exact) gives n*s - 8s = q*s, computed exactly
//   and rounded once. Nibbles m and m+1 of a word need no shift between them:
//   one shift by 8 per word, an AND and an fma a pair.
// * otherwise (any scale): one lop3 makes the bf16 pattern 0x43<nibble> =
//   128 + n exactly, one packed subtract of 136 gives q exactly, one packed
//   multiply rounds q*s once: a lop3, a subtract and a multiply a pair.
// The form is chosen once per stage for a whole warp (int4_stage_fast): a
// branch per chunk cost the kernels ~18% in instruction scheduling.
// Written as PTX: the packed bf16 operations through the cuda_bf16 intrinsics
// take more issue slots. s2: the group's bf16 scale in both halves.
template <bool FAST>
__device__ __forceinline__ void dequant_group(const uint4& wv, uint32_t s2, uint32_t* out16) {
  const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
  if (FAST) {
    const uint32_t S0 = s2 + 0x42804280u;   // exponent field + 133 in both halves (no carry: <= 254)
    const uint32_t S1 = s2 + 0x40804080u;   // exponent field + 129
    uint32_t C2;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(C2) : "r"(s2), "r"(0xC100C100u));   // 0xC100 = bf16 -8
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        // nibbles m (low half) and m + 4 (high half): m even at bits 0..3 of each half of the word
        // (m = 2 after a shift by 8), m odd at bits 4..7
        const uint32_t src = (m < 2) ? w4[i] : (w4[i] >> 8);
        const uint32_t t = src & ((m & 1) ? 0x00F000F0u : 0x000F000Fu);
        asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(out16[4 * i + m]) : "r"(t), "r"((m & 1) ? S1 : S0), "r"(C2));
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        uint32_t pr, q;
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(pr) : "r"(w4[i] >> (4 * m)), "r"(0x000F000Fu), "r"(0x43004300u));
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(q) : "r"(pr), "r"(0x43084308u));   // 0x4308 = bf16 136
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(out16[4 * i + m]) : "r"(q), "r"(s2));
      }
    }
  }
}

// True when every one of a stage row's eight bf16 scales (sw4: four words of two) has its
// exponent field in 1..121, the FAST form's range. Per half h: m = h & 0x7F80 is the exponent
// field times 128; m + 0x4300 reaches bit 15 exactly when the field is >= 122, and m + 0x7F80
// exactly when it is >= 1 (neither sum carries into the next half).
__device__ __forceinline__ bool int4_row_fast(const uint32_t (&sw4)[4]) {
  uint32_t bad = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t m = sw4[j] & 0x7F807F80u;
    bad |= (m + 0x43004300u) | ~(m + 0x7F807F80u);
  }
  return (bad & 0x80008000u) == 0;
}

// The 4-bit float format: one 16-byte chunk of E2M1 codes = four words = 32 inputs, two blocks of
// 16 with their own scale, -> 16 bf16x2 registers in MMA K order (register 4i+m: inputs 8i+m and
// 8i+m+4, as dequant_group). A code's magnitude bits (two exponent bits, one mantissa bit) moved to
// bf16 bits 6..8 and its sign to bit 15 read as the code's value times 2^-126 (the codes +-0.5 as
// bf16 subnormals); one packed multiply by the block's scale times 2^118 (fp4_block_scale) gives
// the weight times 2^-8, exactly: E2M1 values have two significant bits and E4M3 scales four, and
// every such product times 2^-8 is a normal bf16 (2^-18 .. 10.5). The epilogue multiplies the fp32
// sums by the matrix scale times 2^8, which gives the same fp32 products as unscaled weights would.
// Per pair: a shift or two, a select (lop3) of the magnitude and sign bits, an AND, a multiply.
__device__ __forceinline__ void dequant_group_fp4(const uint4& wv, uint32_t S_blk0, uint32_t S_blk1,
                                                  uint32_t* out16) {
  const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t S = (i < 2) ? S_blk0 : S_blk1;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      // magnitude bits 4m..4m+2 of each half to 6..8, sign bit 4m+3 to 15
      const uint32_t a = (m <= 1) ? (w4[i] << (6 - 4 * m)) : (w4[i] >> (4 * m - 6));
      const uint32_t b = w4[i] << (12 - 4 * m);
      uint32_t sel;
      asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(sel) : "r"(a), "r"(b), "r"(0x01C001C0u));   // a where c, else b
      const uint32_t bits = sel & 0x81C081C0u;
      asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(out16[4 * i + m]) : "r"(bits), "r"(S));
    }
  }
}

// E4M3 scale byte -> its value times 2^118 as bf16 in both halves of a register. The byte's
// exponent and mantissa bits moved to bf16 bits 4..10 and its sign to bit 15 read as the scale
// times 2^-120 (subnormal scales too); packed multiplies by 2^127 and 2^111 are exact (the largest
// scale, 448, becomes 1.75 * 2^126).
__device__ __forceinline__ uint32_t fp4_block_scale(uint32_t b) {
  const uint32_t h = ((b & 0x7Fu) << 4) | ((b & 0x80u) << 8);
  uint32_t v, S;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(v) : "r"(__byte_perm(h, 0, 0x1010)), "r"(0x7F007F00u));   // bf16 2^127
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(S) : "r"(v), "r"(0x77007700u));                            // bf16 2^111
  return S;
}

// The factor the fp4 epilogue applies to the fp32 sums: the matrix scale times 2^8 (see above).
__device__ __forceinline__ float fp4_sum_scale(float gscale) { return gscale * 256.0f; }

// Dequantise chunk c (0..7) of a stage row in the weight format FMT; sw4: the row's 16 scale bytes of
// the stage (int4: eight bf16 scales, one per chunk; fp4: sixteen E4M3 scales, two per chunk).
template <int FMT, bool FAST = false>
__device__ __forceinline__ void dequant_chunk(const uint4& wv, const uint32_t (&sw4)[4], int c, uint32_t* out16) {
  if (FMT == WFMT_FP4) {
    const uint32_t pair = (sw4[c >> 1] >> ((c & 1) * 16)) & 0xFFFFu;   // scale bytes 2c, 2c + 1
    dequant_group_fp4(wv, fp4_block_scale(pair & 0xFFu), fp4_block_scale(pair >> 8), out16);
  } else {
    // chunk c's scale is half c % 2 of word c / 2: one byte permute copies it into both halves
    // (4% faster down GEMMs and 5% faster gate/up at 32-token tiles than a shift or mask and a multiply)
    dequant_group<FAST>(wv, __byte_perm(sw4[c >> 1], 0, (c & 1) ? 0x3232 : 0x1010), out16);
  }
}

// A buffer b is reused every NB stages and the stages alternate between two dequant groups, so
// its barriers are kept per (g % 2, b); the stages sharing one are P = lcm(2, NB) apart and g / P
// counts the earlier ones. Buffer b is handed from stage g to stage g + NB: stage g waits for as
// many releases of its (group, buffer) pair as there are stages g' <= g in its class mod P with
// g' >= NB.
__device__ __forceinline__ int a_releases_needed(int g, int nb, int period) {
  return g / period + (g % period >= nb ? 1 : 0);
}

// position of input j inside its block of 8 when a row is stored in MMA order
__device__ __forceinline__ int mma_order_pos(int j) { return (j & ~7) | ((j & 3) << 1) | ((j >> 2) & 1); }

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeFn get_encode() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
  });
  return fn;
}

inline bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t dim0, uint64_t dim1,
                 uint64_t row_bytes, uint32_t box0, uint32_t box1, CUtensorMapSwizzle sw) {
  EncodeFn enc = get_encode();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// x coordinate, in elements of the scale tensor map, of stage ks's scales: a stage's 16 bytes of a row are
// eight bf16 (int4) or sixteen E4M3 bytes (fp4). A TMA load must start on a 16-byte boundary, which this
// keeps for every stage.
template <int FMT>
__host__ __device__ constexpr int scale_x_per_stage() { return FMT == WFMT_FP4 ? 16 : 8; }

// Tensor map of a stage's scales: 64 rows x 16 bytes (int4: eight bf16 per row of the stage's 256
// inputs; fp4: sixteen E4M3 bytes). K must be a multiple of 256 (16-byte row stride).
inline bool make_scale_map(CUtensorMap* m, int wfmt, const void* scales, int K, int64_t rows_total) {
  if (wfmt == WFMT_FP4)
    return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, scales, K / 16, rows_total, K / 16, 16, 64,
                       CU_TENSOR_MAP_SWIZZLE_NONE);
  return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, K / 32, rows_total, K / 16, 8, 64,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace tc
}  // namespace moe
