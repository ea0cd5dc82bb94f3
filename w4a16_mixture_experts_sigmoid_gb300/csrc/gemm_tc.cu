// Steps 3 and 4 on the 5th-generation tensor cores: the grouped W4A16 expert
// GEMMs over expert-sorted token rows, for sm_103a.
//
// Weight format ("Kimi-K2.6" catalog page, QUANT/PARAMS: int4 in int32
// containers, symmetric, group 32): W[n, k] = q * s with q = nibble - 8,
// nibble of input k = bits 4(k%8).. of word k/8 of row n, s the bf16 scale of
// group k/32. Expert shapes (GEOMETRY): W13 = [gate; up] is [2I][H], W2 is [H][I].
//
// Orientation ("swap AB"): the MMA's M = 128 weight rows, its N = NT token
// rows of one expert, K = the reduction dimension. A tile is one 128-row slab
// of one expert's weights; a decode step touches ~1-3 tokens per expert, so
// tokens are the narrow operand. On this part an M=128, K=16 MMA costs the
// same ~45 cycles for every N <= 64 (it is bound by reading the 128x16 A tile),
// so the MMA count, not N, sets the tensor-core floor of a decode step.
//
// K order inside the MMA: each int32 word's eight nibbles are turned into four
// bf16 pairs with one AND/OR each, pair m holding inputs m and m+4 of the
// word. The MMA therefore sees the K order [0,4,1,5,2,6,3,7] inside every
// block of 8 inputs. A dot product does not depend on the order of its terms,
// so the token rows (operand B) are stored in the same order ("MMA order"):
// the gather writes x rows that way and the gate/up epilogue writes h that
// way, at no extra cost.
//
// One persistent CTA per SM, 16 warps:
//   warp 0      builds the tile list, then is the weight producer: TMA of int4
//               words + bf16 scales (or dense bf16 weights) into the weight ring.
//   warp 14     token-row producer: TMA of the token rows into their ring; a
//               warp of its own so that the weight stream never waits on it.
//   warps 1, 15 MMA issuers (lane 0 each, or with 128-token tiles the whole
//               warp with one elected lane issuing; warp 1 also owns the
//               tensor-memory allocation). A thread can issue one M=128 MMA
//               about every 50 cycles whatever N <= 64 is, while the tensor
//               core accepts MMAs from several threads at once; so each of
//               the two dequant groups has its own issuer and its own fp32
//               accumulators, and the epilogue adds the two. (With 128 tokens
//               per tile one issuer keeps up with the math, and tensor memory
//               holds one set.)
//   warps 2-9   dequantise, in two groups of four that take alternate stages:
//               each thread owns one weight row (= one TMEM lane) of its
//               group's stage and turns its 256 nibbles into bf16(q*s) in the
//               MMA's A operand: tensor memory (default) or swizzled shared
//               memory (MOE_FLAG_A_SMEM).
//   warps 10-13 epilogue: TMEM -> registers -> SiLU(gate)*up (gate/up) or the
//               plain row (down) -> bf16 rows in global memory. Accumulators
//               are double-buffered, so the epilogue of one tile overlaps the
//               MMAs of the next.
// Dense bf16 weights (the shared expert) skip the dequantiser: TMA loads the
// weight tile straight into the swizzled layout (natural K order).
//
// Gate/up pairing: within each 32-lane quarter q of the 128 lanes, lanes
// 0-15 hold gate rows j0+16q+0..15 and lanes 16-31 the up rows with the same
// j, so the epilogue pairs them with one shuffle.
//
// Every wait is bounded (mbar_wait): an expired wait records
// MOE_ERR_DEVICE_TIMEOUT in the status word, every role leaves its loop, the
// producer lets its copies in flight land, the MMA issuer lets its MMAs
// finish, and the CTA frees its tensor memory before returning.
#include "gemm_tc_parts.cuh"

#include <atomic>
#include <cstring>
#include <mutex>
#include <type_traits>

namespace moe {
namespace {

using namespace tc;

template <int ASRC, int NT>
struct Cfg {
  static constexpr bool kDq = ASRC != A_SMEM_BF16;
  static constexpr int kAStage = kDq ? BM * 128 : NSUB * BM * 128;
  static constexpr int kSStage = kDq ? BM * 16 : 0;
  static constexpr int kWStage = kAStage + kSStage;
  static constexpr int kBStage = NSUB * NT * 128;
  static constexpr int kNBuf = (ASRC == A_TMEM_DQ) ? (NT <= 32 ? 3 : 2) : (ASRC == A_SMEM_DQ ? 2 : 1);
  static constexpr int kABuf = (ASRC == A_SMEM_DQ) ? NSUB * BM * 128 : 0;
  static constexpr int kAvail = kSmemLimit - kAlignSlack - kAuxBytes - (ASRC == A_SMEM_DQ ? kNBuf * kABuf : 0);
  static constexpr int kBFit = (kAvail - 3 * kWStage) / kBStage;
  static constexpr int kBStagesDq = (kNBuf + 3 < kBFit ? kNBuf + 3 : kBFit);
  static constexpr int kWStagesDq = (kAvail - kBStagesDq * kBStage) / kWStage;
  static constexpr int kLock = kAvail / (kWStage + kBStage);
  static constexpr int kWStages = kDq ? (kWStagesDq > 12 ? 12 : kWStagesDq) : (kLock > 8 ? 8 : kLock);
  static constexpr int kBStages = kDq ? kBStagesDq : kWStages;
  // try_wait.parity cannot tell phase k from phase k+2, so a barrier may be waited on only by a
  // consumer that cannot run two phases ahead of it. Stages alternate between two consumers
  // (dequant groups, MMA issuers) by g % 2, so every "full" barrier and every A-buffer barrier
  // is kept per (g % 2, slot): the stages that share one are lcm(2, ring) apart and are all
  // taken by one consumer in order.
  static constexpr int kWPeriod = (kWStages % 2 == 0) ? kWStages : 2 * kWStages;
  static constexpr int kBPeriod = (kBStages % 2 == 0) ? kBStages : 2 * kBStages;
  static constexpr int kAPeriod = (kNBuf % 2 == 0) ? kNBuf : 2 * kNBuf;
  // A token-row slot is free once the MMAs of the stage that used it are done, which the same
  // stage's A-buffer release already says. When kAPeriod >= kBStages the token-row producer waits
  // for that release instead of a commit of its own (one commit per stage fewer for the issuers):
  // the release's barrier cannot move on twice before the producer's next load, which it needs.
  static constexpr bool kBViaA = kDq && kAPeriod >= kBStages;
  static constexpr int kMmaGroups = NT <= 64 ? 2 : 1;   // MMA issuers, each with its own accumulators
  static constexpr int kAccCol = (ASRC == A_TMEM_DQ) ? kNBuf * 128 : 0;
  static constexpr int kColsNeeded = kAccCol + 2 * kMmaGroups * NT;   // double-buffered per issuer
  static constexpr int kTmemCols = kColsNeeded <= 32 ? 32 : kColsNeeded <= 64 ? 64 : kColsNeeded <= 128 ? 128
                                   : kColsNeeded <= 256 ? 256 : 512;
  static constexpr int kSmemBytes =
      kAlignSlack + kWStages * kWStage + kBStages * kBStage + kNBuf * kABuf + kAuxBytes;
  static_assert(kWStages >= 2 && kBStages >= 2, "each ring needs at least two stages");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory overflow");
  static_assert(8 * (3 * kWStages + 3 * kBStages + 4 * kNBuf + 5) + 16 + 2 * kMaxE + 4 * (kMaxE + 1) <= kAuxBytes,
                "barriers and tile table overflow the aux area");
  static_assert(kColsNeeded <= 512, "tensor memory overflow");
  static_assert(kWStage % 1024 == 0 && kBStage % 1024 == 0, "stages must keep 1024-byte alignment");
};

// YF32 (down only): the rows are written in fp32 to p.out_f32 instead of bf16 to p.out. A compile-time
// choice: a run-time branch on the output type in the epilogue made the down kernel ~25% slower at
// 32- and 128-token tiles, whichever type it wrote.
template <int OP, int ASRC, int NT, int FMT = WFMT_INT4, bool YF32 = false>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
  using C = Cfg<ASRC, NT>;
  constexpr int SW = C::kWStages;
  constexpr int SB = C::kBStages;
  constexpr int NB = C::kNBuf;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* bring = smem + SW * C::kWStage;
  uint8_t* abuf = bring + SB * C::kBStage;
  uint8_t* aux = abuf + NB * C::kABuf;
  uint64_t* wfull = reinterpret_cast<uint64_t*>(aux);   // [2][SW]: (stage parity, slot)
  uint64_t* wempty = wfull + 2 * SW;
  uint64_t* bfull = wempty + SW;                         // [2][SB]
  uint64_t* bempty = bfull + 2 * SB;
  uint64_t* afull = bempty + SB;      // [2][NB]: (dequant group, A buffer)
  uint64_t* aempty = afull + 2 * NB;  // [2][NB]
  uint64_t* accfull = aempty + 2 * NB;   // [2]
  uint64_t* accempty = accfull + 2;  // [2]
  uint64_t* drain = accempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* n_act_s = reinterpret_cast<int*>(tmem_slot + 2);
  int16_t* act_e = reinterpret_cast<int16_t*>(tmem_slot + 4);
  int* tpre = reinterpret_cast<int*>(act_e + kMaxE);

  // The successor in the stream may launch now: its CTAs take SMs as this grid's CTAs leave. The
  // token-row producer always waits for the predecessor grid to finish (griddep_wait below). With
  // weights_ready the tile table and the weight stream need not: the launcher guarantees that the
  // weights and the expert offsets were complete before the kernels queued ahead of this one began
  // (within one layer the offsets come from the permutation, finished before the predecessor could
  // start); otherwise warp 0 waits too.
  griddep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_wt = (OP == MOE_GEMM_GATEUP_SILU) ? (p.out_cols + 63) / 64 : (p.rows_per_expert + BM - 1) / BM;
  // K slices exist only for the dense bf16 weights (the shared expert); the int4 kernels are
  // compiled without them: the slice arithmetic and the partial-sum epilogue cost the routed
  // GEMMs 1-4% when present.
  const int ksplit = (ASRC == A_SMEM_BF16) ? p.ksplit : 1;
  const int nk = ((p.K + BK - 1) / BK) / ksplit;   // stages per tile (its K slice)

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2 * SW; ++s) mbar_init(&wfull[s], 32);
    for (int s = 0; s < SW; ++s) mbar_init(&wempty[s], C::kDq ? 4 : 1);
    for (int s = 0; s < 2 * SB; ++s) mbar_init(&bfull[s], 1);
    for (int s = 0; s < SB; ++s) mbar_init(&bempty[s], 1);
    for (int b = 0; b < 2 * NB; ++b) { mbar_init(&afull[b], 4); mbar_init(&aempty[b], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&accfull[a], C::kMmaGroups); mbar_init(&accempty[a], 4); }
    mbar_init(drain, C::kMmaGroups);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  if (warp == 0) {
    if (!p.weights_ready) griddep_wait();
    // compact list of experts with rows, and the prefix of their tile counts
    if (p.uniform_rows >= 0) {
      if (lane == 0) {
        const int chunks = (p.uniform_rows + NT - 1) / NT;
        *n_act_s = p.uniform_rows > 0 ? 1 : 0;
        act_e[0] = 0;
        tpre[0] = 0;
        tpre[1] = n_wt * chunks * ksplit;
      }
    } else {
      // every expert's row count is loaded before the scan, so the loads overlap
      int cnts[kMaxE / 32];
#pragma unroll
      for (int c = 0; c < kMaxE / 32; ++c) {
        const int e = 32 * c + lane;
        cnts[c] = (e < p.E) ? __ldg(p.offsets + e + 1) - __ldg(p.offsets + e) : 0;
      }
      int base_a = 0, base_t = 0;
#pragma unroll
      for (int c = 0; c < kMaxE / 32; ++c) {
        const int e0 = 32 * c;
        if (e0 >= p.E) break;
        const int e = e0 + lane;
        const int cnt = cnts[c];
        const bool f = cnt >= p.min_rows && cnt <= p.max_rows && cnt > 0;
        const int ntl = f ? n_wt * ((cnt + NT - 1) / NT) * ksplit : 0;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, f);
        int incl = ntl;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
          if (lane >= off) incl += o;
        }
        if (f) {
          const int pos = base_a + __popc(m & ((1u << lane) - 1u));
          act_e[pos] = static_cast<int16_t>(e);
          tpre[pos] = base_t + incl - ntl;
        }
        base_a += __popc(m);
        base_t += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      if (lane == 0) {
        *n_act_s = base_a;
        tpre[base_a] = base_t;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_act = *n_act_s;
  const int total = tpre[n_act];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = l2_policy_evict_first();
    constexpr int kScaleX = scale_x_per_stage<FMT>();   // one stage of scales, in map elements (16 bytes)
    const uint32_t txw = C::kAStage + ((C::kDq && p.scale_tma) ? BM * 16 : 0);
    const int kg = p.K / 32;
    int g = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < total && ok; i += gridDim.x) {
      const TileInfo ti = decode_tile(i, n_act, act_e, tpre, p, NT, ksplit);
      const int ebase = ti.e * p.rows_per_expert;
      int grow_lo, grow_hi;
      if (OP == MOE_GEMM_GATEUP_SILU) { grow_lo = ebase + ti.wt * 64; grow_hi = ebase + p.out_cols + ti.wt * 64; }
      else { grow_lo = ebase + ti.wt * BM; grow_hi = grow_lo + 64; }
      const int kb = ti.split * nk;   // first stage of this tile's K slice
      for (int ks = 0; ks < nk; ++ks, ++g) {
        const int sw = g % SW;
        uint64_t* wf = &wfull[(g & 1) * SW + sw];
        if (!warp_wait(&wempty[sw], ((g / SW) & 1) ^ 1, p, abort_flag)) { ok = false; break; }
        uint8_t* sa = smem + sw * C::kWStage;
        uint8_t* ss = sa + C::kAStage;
        if (C::kDq && !p.scale_tma && FMT == WFMT_INT4) {
          // scales by plain loads (row stride not 16-byte aligned): lane owns rows lane + 32 r
          uint16_t* sc = reinterpret_cast<uint16_t*>(ss);
          for (int r = lane; r < BM; r += 32) {
            const int grow = (r < 64) ? grow_lo + r : grow_hi + (r - 64);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int gi = (kb + ks) * 8 + q;
              uint16_t v = 0;
              if (gi < kg && grow < p.rows_total) v = p.scales[static_cast<int64_t>(grow) * kg + gi];
              sc[r * 8 + q] = v;
            }
          }
        } else if (C::kDq && !p.scale_tma) {
          // E4M3 scale bytes, one per 16 inputs: 16 a row per stage
          const uint8_t* src = reinterpret_cast<const uint8_t*>(p.scales);
          const int kb16 = p.K / 16;
          for (int r = lane; r < BM; r += 32) {
            const int grow = (r < 64) ? grow_lo + r : grow_hi + (r - 64);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const int gi = (kb + ks) * 16 + q;
              uint8_t v = 0;
              if (gi < kb16 && grow < p.rows_total) v = src[static_cast<int64_t>(grow) * kb16 + gi];
              ss[r * 16 + q] = v;
            }
          }
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(wf, txw);
          if (!C::kDq) {
#pragma unroll
            for (int sub = 0; sub < NSUB; ++sub) {
#pragma unroll
              for (int rb = 0; rb < 8; ++rb) {
                int grow;
                if (OP == MOE_GEMM_GATEUP_SILU) grow = (rb & 1) * p.out_cols + ti.wt * 64 + 16 * (rb >> 1);
                else grow = ti.wt * BM + 16 * rb;
                tma_load_2d(sa + sub * (BM * 128) + rb * 2048, &p.tm_w, wf, (kb + ks) * BK + sub * KSUB, grow,
                            pol_w);
              }
            }
          } else {
            tma_load_2d(sa, &p.tm_w, wf, (kb + ks) * (BK / 8), grow_lo, pol_w);
            tma_load_2d(sa + 64 * 128, &p.tm_w, wf, (kb + ks) * (BK / 8), grow_hi, pol_w);
            if (p.scale_tma) {
              tma_load_2d(ss, &p.tm_s, wf, (kb + ks) * kScaleX, grow_lo, pol_w);
              tma_load_2d(ss + 64 * 16, &p.tm_s, wf, (kb + ks) * kScaleX, grow_hi, pol_w);
            }
          }
        } else {
          mbar_arrive(wf);
        }
      }
    }
    // let every copy issued into this CTA's shared memory land before exit
    if (lane == 0) {
      for (int d = 0; d < SW && d < g; ++d) {
        const int gg = g - 1 - d;
        mbar_wait(&wfull[(gg & 1) * SW + gg % SW], (gg / C::kWPeriod) & 1, p.timeout_ns, nullptr, p.status);
      }
    }
    __syncwarp();
  } else if (warp == kBProducerWarp) {
    // ------------------------------------------------------------ token-row producer (one lane)
    if (lane == 0) {
      griddep_wait();   // the token rows are the predecessor's output
      const uint64_t pol_b = l2_policy_evict_last();
      constexpr uint32_t txb = NSUB * NT * 128;
      int g = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < total && ok; i += gridDim.x) {
        const TileInfo ti = decode_tile(i, n_act, act_e, tpre, p, NT, ksplit);
        for (int ks = 0; ks < nk; ++ks, ++g) {
          const int sbi = g % SB;
          if (C::kBViaA) {
            if (g >= SB) {
              const int gn = g - SB + NB;   // the next user of the A buffer of stage g - SB
              const int need = a_releases_needed(gn, NB, C::kAPeriod);
              if (!mbar_wait(&aempty[(gn & 1) * NB + gn % NB], (need - 1) & 1, p.timeout_ns, abort_flag, p.status)) {
                ok = false;
                break;
              }
            }
          } else if (!mbar_wait(&bempty[sbi], ((g / SB) & 1) ^ 1, p.timeout_ns, abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t* sb = bring + sbi * C::kBStage;
          uint64_t* bf = &bfull[(g & 1) * SB + sbi];
          mbar_arrive_expect_tx(bf, txb);
#pragma unroll
          for (int sub = 0; sub < NSUB; ++sub)
            tma_load_2d(sb + sub * (NT * 128), &p.tm_b, bf, (ti.split * nk + ks) * BK + sub * KSUB, ti.row0, pol_b);
        }
      }
      for (int d = 0; d < SB && d < g; ++d) {
        const int gg = g - 1 - d;
        mbar_wait(&bfull[(gg & 1) * SB + gg % SB], (gg / C::kBPeriod) & 1, p.timeout_ns, nullptr, p.status);
      }
    }
    __syncwarp();
  } else if (warp == 1 || (C::kMmaGroups == 2 && warp == kSecondMmaWarp)) {
    // ------------------------------------------------------------ MMA issuers
    // With 128-token tiles the whole warp runs the loop and one elected lane issues (iss_wait)
    constexpr bool W = NT >= 128;
    if (W || lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, NT);
      const int mg = (warp == 1) ? 0 : 1;  // with two issuers, issuer mg takes the stages g with g % 2 == mg
      int g = 0, it = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < total && ok; i += gridDim.x, ++it) {
        const int ab = it & 1;
        if (!iss_wait<W>(&accempty[ab], ((it >> 1) & 1) ^ 1, p, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + C::kAccCol + (mg * 2 + ab) * NT;
        bool first = true;
        for (int ks = 0; ks < nk; ++ks, ++g) {
          if (C::kMmaGroups == 2 && (g & 1) != mg) continue;
          const int sw = g % SW, sbi = g % SB;
          const int b = g % NB;
          if (!iss_wait<W>(&bfull[(g & 1) * SB + sbi], (g / C::kBPeriod) & 1, p, abort_flag)) {
            ok = false;
            break;
          }
          if (C::kDq) {
            if (!iss_wait<W>(&afull[(g & 1) * NB + b], (g / C::kAPeriod) & 1, p, abort_flag)) {
              ok = false;
              break;
            }
          } else {
            if (!iss_wait<W>(&wfull[(g & 1) * SW + sw], (g / C::kWPeriod) & 1, p, abort_flag)) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + sw * C::kWStage);
          const uint32_t sb = smem_u32(bring + sbi * C::kBStage);
          const uint64_t bdesc0 = sw128_kmajor_desc(sb);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const int sub = kk >> 2;
            const uint32_t koff = (kk & 3) * 32;
            // K step kk: the stage's descriptor plus a constant (the start-address field counts
            // 16-byte units and cannot carry out: shared memory is below 2^18 bytes)
            const uint64_t bdesc = bdesc0 + ((sub * (NT * 128) + koff) >> 4);
            const uint32_t acc = (!first || kk > 0) ? 1u : 0u;
            if (ASRC == A_TMEM_DQ) {
              iss_mma_ts<W>(d_tmem, tmem + b * 128 + kk * 8, bdesc, idesc, acc);
            } else if (ASRC == A_SMEM_DQ) {
              const uint64_t adesc = sw128_kmajor_desc(smem_u32(abuf + b * C::kABuf) + sub * (BM * 128) + koff);
              iss_mma_ss<W>(d_tmem, adesc, bdesc, idesc, acc);
            } else {
              const uint64_t adesc = sw128_kmajor_desc(sa + sub * (BM * 128) + koff);
              iss_mma_ss<W>(d_tmem, adesc, bdesc, idesc, acc);
            }
          }
          first = false;
          if (!C::kBViaA) iss_commit<W>(&bempty[sbi]);
          if (C::kDq) iss_commit<W>(&aempty[((g + NB) & 1) * NB + b]);   // to the group of the next user
          else iss_commit<W>(&wempty[sw]);
        }
        if (!ok) break;
        iss_commit<W>(&accfull[ab]);   // an issuer with no stage in this tile arrives at once
      }
      // let every MMA issued by this thread finish before tensor memory is freed
      iss_commit<W>(drain);
      iss_wait<W>(drain, 0, p, nullptr);
    }
    __syncwarp();
  } else if (warp >= kFirstDqWarp && warp < kFirstEpiWarp) {
    // ------------------------------------------------------------ dequantise
    if (ASRC != A_SMEM_BF16) {
      const int grp = (warp - kFirstDqWarp) >> 2;  // takes the stages g with g % 2 == grp
      const int q = warp & 3;                      // TMEM lane quarter this warp may access (warp id mod 4)
      const int l = 32 * q + lane;
      const int r_sm = (OP == MOE_GEMM_GATEUP_SILU) ? (lane < 16 ? 16 * q + lane : 64 + 16 * q + (lane - 16)) : l;
      const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
      // Gate/up addresses chunk c of its stage row as (stage + row_x) ^ (c << 4): the row's 128-byte
      // slot is 128-aligned, so the XOR applies the row's swizzle phase in one instruction (gate/up
      // 2.5% faster at decode; the same loads in the down kernel made it slower, so down keeps the
      // pointer form).
      const uint32_t row_x = static_cast<uint32_t>(r_sm) * 128u + (static_cast<uint32_t>(r_sm & 7) << 4);
      int g = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < total && ok; i += gridDim.x) {
        for (int ks = 0; ks < nk; ++ks, ++g) {
          if ((g & 1) != grp) continue;
          const int sw = g % SW;
          const int b = g % NB;
          const int a_need = a_releases_needed(g, NB, C::kAPeriod);
          if (!warp_wait(&wfull[(g & 1) * SW + sw], (g / C::kWPeriod) & 1, p, abort_flag)) { ok = false; break; }
          // the stage row comes into registers in two halves of four 16-byte chunks; once the
          // second half is loaded the stage goes back to the producer
          const uint8_t* arow = smem + sw * C::kWStage + r_sm * 128;
          const uint4 sv = *reinterpret_cast<const uint4*>(smem + sw * C::kWStage + C::kAStage + r_sm * 16);
          const uint32_t sw4[4] = {sv.x, sv.y, sv.z, sv.w};
          uint4 wv[4];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            wv[c] = (OP == MOE_GEMM_GATEUP_SILU) ? ld_shared_v4((smem_u32(smem + sw * C::kWStage) + row_x) ^ (c << 4))
                                                 : *reinterpret_cast<const uint4*>(arow + ((c ^ (r_sm & 7)) << 4));
          // The conversion's form (dequant_group) is chosen once per stage for the whole warp: the
          // exact fma form when every scale of the warp's rows allows it, else the general one.
          const bool fast = (FMT == WFMT_INT4) && __all_sync(0xFFFFFFFFu, int4_row_fast(sw4));
          auto convert = [&](auto fast_tag) -> bool {
            constexpr bool kFast = decltype(fast_tag)::value;
            // The first half row's conversion needs no A buffer, so for gate/up it runs before the
            // wait for one (gate/up 3% faster at decode; the same for down made it 2% slower).
            constexpr int kPreChunks = (OP == MOE_GEMM_GATEUP_SILU) ? 4 : 0;
            uint32_t pre[kPreChunks > 0 ? kPreChunks : 1][16];
#pragma unroll
            for (int c = 0; c < kPreChunks; ++c) dequant_chunk<FMT, kFast>(wv[c], sw4, c, pre[c]);
            if (a_need > 0 && !warp_wait(&aempty[grp * NB + b], (a_need - 1) & 1, p, abort_flag)) return false;
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              if (half == 1) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                  wv[c] = (OP == MOE_GEMM_GATEUP_SILU)
                              ? ld_shared_v4((smem_u32(smem + sw * C::kWStage) + row_x) ^ ((c + 4) << 4))
                              : *reinterpret_cast<const uint4*>(arow + (((c + 4) ^ (r_sm & 7)) << 4));
                __syncwarp();
                if (lane == 0) mbar_arrive(&wempty[sw]);
              }
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
                const int c = half * 4 + cc;
                uint32_t dqc[16];
                if (c >= kPreChunks) dequant_chunk<FMT, kFast>(wv[cc], sw4, c, dqc);
                const uint32_t* dq = (c < kPreChunks) ? pre[c < kPreChunks ? c : 0] : dqc;
                if (ASRC == A_TMEM_DQ) {
                  tmem_st8(lane_base + b * 128 + c * 16, dq);
                  tmem_st8(lane_base + b * 128 + c * 16 + 8, dq + 8);
                } else {
                  uint8_t* ab = abuf + b * C::kABuf + (c >> 1) * (BM * 128) + l * 128;
#pragma unroll
                  for (int m = 0; m < 4; ++m)
                    *reinterpret_cast<uint4*>(ab + ((((c & 1) * 4 + m) ^ (l & 7)) << 4)) =
                        make_uint4(dq[4 * m], dq[4 * m + 1], dq[4 * m + 2], dq[4 * m + 3]);
                }
              }
            }
            if (ASRC == A_TMEM_DQ) tmem_wait_st();
            else fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&afull[grp * NB + b]);
            return true;
          };
          if (!(fast ? convert(std::true_type{}) : convert(std::false_type{}))) { ok = false; break; }
        }
      }
    }
  } else if (warp >= kFirstEpiWarp && warp < kFirstEpiWarp + 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int l = 32 * q + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
    int it = 0;
    for (int i = blockIdx.x; i < total; i += gridDim.x, ++it) {
      const TileInfo ti = decode_tile(i, n_act, act_e, tpre, p, NT, ksplit);
      const int ab = it & 1;
      if (!warp_wait(&accfull[ab], (it >> 1) & 1, p, abort_flag)) break;
      tc_fence_after();
      // which issuers accumulated into this tile: with one stage per tile only the one whose parity it has
      const int g0 = it * nk;
      const bool use0 = C::kMmaGroups == 1 || nk >= 2 || (g0 & 1) == 0;
      const bool use1 = C::kMmaGroups == 2 && (nk >= 2 || (g0 & 1) == 1);
#pragma unroll
      for (int cb = 0; cb < NT; cb += 16) {
        uint32_t v[16];
        __syncwarp();
        if (use0) {
          tmem_ld16(lane_base + C::kAccCol + ab * NT + cb, v);
          tmem_wait_ld();
        }
        if (use1) {
          uint32_t v1[16];
          tmem_ld16(lane_base + C::kAccCol + (2 + ab) * NT + cb, v1);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 16; ++c)
            v[c] = use0 ? __float_as_uint(__uint_as_float(v[c]) + __uint_as_float(v1[c])) : v1[c];
        }
        if (FMT == WFMT_FP4) {
          const float gs = fp4_sum_scale(__ldg(p.gscale + ti.e));   // the expert's fp32 matrix scale, x 2^8
#pragma unroll
          for (int c = 0; c < 16; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * gs);
        }
        if (ASRC == A_SMEM_BF16 && ksplit > 1) {
          // one K slice: its raw fp32 sums go to the partial buffer, each lane its own weight row
          // (gate/up: lanes 0-15 the gate rows, 16-31 the up rows of the same outputs)
          if (OP == MOE_GEMM_GATEUP_SILU) {
            const int j = ti.wt * 64 + 16 * q + (lane & 15);
            if (j < p.out_cols) {
#pragma unroll
              for (int c = 0; c < 16; ++c) {
                const int row = ti.row0 + cb + c;
                if (cb + c < ti.nvalid && row < p.R)
                  p.partial[(static_cast<int64_t>(ti.split * p.R + row) * 2 + (lane >> 4)) * p.out_cols + j] =
                      __uint_as_float(v[c]);
              }
            }
          } else {
            const int n = ti.wt * BM + l;
            if (n < p.out_cols) {
#pragma unroll
              for (int c = 0; c < 16; ++c) {
                const int row = ti.row0 + cb + c;
                if (cb + c < ti.nvalid && row < p.R)
                  p.partial[static_cast<int64_t>(ti.split * p.R + row) * p.out_cols + n] = __uint_as_float(v[c]);
              }
            }
          }
        } else if (OP == MOE_GEMM_GATEUP_SILU) {
          float u[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) u[c] = __shfl_down_sync(0xFFFFFFFFu, __uint_as_float(v[c]), 16);
          const int j = ti.wt * 64 + 16 * q + lane;
          if (lane < 16 && j < p.out_cols) {
            const int col = p.out_mma_order ? mma_order_pos(j) : j;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int row = ti.row0 + cb + c;
              if (cb + c < ti.nvalid && row < p.R) {
                const float gt = __uint_as_float(v[c]);
                const float h = __fdividef(gt, 1.0f + __expf(-gt)) * u[c];  // SiLU(g) * u, rounded to bf16 below
                p.out[static_cast<int64_t>(row) * p.out_cols + col] = __bfloat16_as_ushort(__float2bfloat16_rn(h));
              }
            }
          }
        } else {
          const int n = ti.wt * BM + l;
          if (n < p.out_cols) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int row = ti.row0 + cb + c;
              if (cb + c < ti.nvalid && row < p.R) {
                const int64_t o = static_cast<int64_t>(row) * p.out_cols + n;
                if (YF32) p.out_f32[o] = __uint_as_float(v[c]);
                else p.out[o] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[c])));
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accempty[ab]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

template <int OP, int ASRC, int NT, int FMT, bool YF32>
cudaError_t run_y(const TcParams& prm, int grid, cudaStream_t s) {
  using C = Cfg<ASRC, NT>;
  // the shared-memory opt-in is per device: remember it per device ordinal
  static std::atomic<uint64_t> opted_in{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit == 0 || !(opted_in.load() & bit)) {
    e = cudaFuncSetAttribute(tc_gemm_kernel<OP, ASRC, NT, FMT, YF32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    opted_in.fetch_or(bit);
  }
  (void)launch_pdl(tc_gemm_kernel<OP, ASRC, NT, FMT, YF32>, dim3(grid), dim3(kThreads), C::kSmemBytes, s, prm);
  count_launches(1);
  return cudaGetLastError();
}

// the down kernels come in both output types; gate/up writes bf16 h only
template <int OP, int ASRC, int NT, int FMT = WFMT_INT4>
cudaError_t run(const TcParams& prm, int grid, cudaStream_t s) {
  if (OP == MOE_GEMM_DOWN && prm.out_f32 != nullptr) return run_y<OP, ASRC, NT, FMT, OP == MOE_GEMM_DOWN>(prm, grid, s);
  return run_y<OP, ASRC, NT, FMT, false>(prm, grid, s);
}

// After a launch with K slices: out[r][c] = bf16 of the finished sums, the slices added in order
// (gate/up: SiLU(gate) * up, as the epilogue computes it; down: the plain sum).
template <int OP>
__global__ void __launch_bounds__(256) splitk_finish_kernel(const float* __restrict__ part, int S, int R, int cols,
                                                            int out_mma_order, uint16_t* __restrict__ out,
                                                            float* __restrict__ out_f32) {
  griddep_wait();    // the predecessor in the stream has finished and its writes are visible
  griddep_launch();  // the successor may start its own prologue
  const int64_t n = static_cast<int64_t>(R) * cols;
  for (int64_t i = blockIdx.x * 256LL + threadIdx.x; i < n; i += static_cast<int64_t>(gridDim.x) * 256) {
    const int64_t row = i / cols;
    const int col = static_cast<int>(i - row * cols);
    float a = 0.0f, b = 0.0f;
    for (int sl = 0; sl < S; ++sl) {
      if (OP == MOE_GEMM_GATEUP_SILU) {
        a += part[((static_cast<int64_t>(sl) * R + row) * 2) * cols + col];
        b += part[((static_cast<int64_t>(sl) * R + row) * 2 + 1) * cols + col];
      } else {
        a += part[(static_cast<int64_t>(sl) * R + row) * cols + col];
      }
    }
    const float v = (OP == MOE_GEMM_GATEUP_SILU) ? __fdividef(a, 1.0f + __expf(-a)) * b : a;
    const int oc = (OP == MOE_GEMM_GATEUP_SILU && out_mma_order) ? mma_order_pos(col) : col;
    if (out_f32 != nullptr) out_f32[row * cols + oc] = v;
    else out[row * cols + oc] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
}

template <int OP>
cudaError_t dispatch(const TcParams& prm, int asrc, int nt, int grid, int wfmt, cudaStream_t s) {
  if (wfmt == WFMT_FP4) {
    if (asrc != A_TMEM_DQ) return cudaErrorNotSupported;
    switch (nt) {
      case 16: return run<OP, A_TMEM_DQ, 16, WFMT_FP4>(prm, grid, s);
      case 32: return run<OP, A_TMEM_DQ, 32, WFMT_FP4>(prm, grid, s);
      case 64: return run<OP, A_TMEM_DQ, 64, WFMT_FP4>(prm, grid, s);
      case 128: return run<OP, A_TMEM_DQ, 128, WFMT_FP4>(prm, grid, s);
    }
    return cudaErrorNotSupported;
  }
  switch (asrc) {
    case A_TMEM_DQ:
      switch (nt) {
        case 16: return run<OP, A_TMEM_DQ, 16>(prm, grid, s);
        case 32: return run<OP, A_TMEM_DQ, 32>(prm, grid, s);
        case 64: return run<OP, A_TMEM_DQ, 64>(prm, grid, s);
        case 128: return run<OP, A_TMEM_DQ, 128>(prm, grid, s);
      }
      break;
    case A_SMEM_DQ:
      switch (nt) {
        case 16: return run<OP, A_SMEM_DQ, 16>(prm, grid, s);
        case 32: return run<OP, A_SMEM_DQ, 32>(prm, grid, s);
      }
      break;
    case A_SMEM_BF16:
      switch (nt) {
        case 16: return run<OP, A_SMEM_BF16, 16>(prm, grid, s);
        case 32: return run<OP, A_SMEM_BF16, 32>(prm, grid, s);
        case 64: return run<OP, A_SMEM_BF16, 64>(prm, grid, s);
      }
      break;
  }
  return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_gemm_tc(const GemmProblem& p, int asrc, int nt, int num_sms, cudaStream_t s) {
  if (p.R <= 0) return cudaSuccess;
  if (p.bf16_weights != (asrc == A_SMEM_BF16)) return cudaErrorNotSupported;
  // int4 weights are dequantised in MMA K order: the token rows must be stored that way too
  if (!p.bf16_weights && !p.a_mma_order) return cudaErrorNotSupported;
  if (!p.bf16_weights && p.E > kMaxE) return cudaErrorNotSupported;
  TcParams prm;
  memset(&prm, 0, sizeof(prm));
  const int groups = p.uniform_rows >= 0 ? 1 : p.E;
  const int64_t rows_total = static_cast<int64_t>(groups) * p.rows_per_expert;
  bool ok;
  if (p.bf16_weights) {
    ok = make_map_2d(&prm.tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.w, p.K, rows_total, 2ull * p.K, KSUB, 16,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    ok = make_map_2d(&prm.tm_w, CU_TENSOR_MAP_DATA_TYPE_INT32, p.w, p.K / 8, rows_total, p.K / 2, BK / 8, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B);
    prm.scale_tma = (p.K % 256 == 0) ? 1 : 0;
    if (ok && prm.scale_tma)
      ok = make_scale_map(&prm.tm_s, p.wfmt, p.scales, p.K, rows_total);
  }
  if (ok)
    ok = make_map_2d(&prm.tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.a, p.K, p.R, 2ull * p.K, KSUB, nt,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  prm.scales = p.scales;
  prm.gscale = p.gscale;
  prm.offsets = p.offsets;
  prm.out = p.out;
  prm.out_f32 = (p.op == MOE_GEMM_DOWN) ? p.out_f32 : nullptr;
  if (p.wfmt == WFMT_FP4 && (p.bf16_weights || p.gscale == nullptr)) return cudaErrorInvalidValue;
  prm.status = p.status;
  prm.E = p.E;
  prm.K = p.K;
  prm.rows_per_expert = p.rows_per_expert;
  prm.out_cols = p.out_cols;
  prm.uniform_rows = p.uniform_rows;
  prm.min_rows = p.min_rows;
  prm.max_rows = p.max_rows;
  prm.weights_ready = p.weights_ready ? 1 : 0;
  prm.ksplit = p.ksplit;
  prm.partial = p.partial;
  if (p.ksplit < 1 || ((p.K + BK - 1) / BK) % p.ksplit != 0 || (p.ksplit > 1 && p.partial == nullptr) ||
      (p.ksplit > 1 && !p.bf16_weights))
    return cudaErrorInvalidValue;
  prm.rows_total = static_cast<int>(rows_total);
  prm.R = p.R;
  prm.out_mma_order = p.out_mma_order ? 1 : 0;
  prm.timeout_ns = 2000000000ull;
  // upper bound on tiles: every expert with rows contributes ceil(rows/nt) <= rows/nt + 1 chunks
  const int n_wt = (p.op == MOE_GEMM_GATEUP_SILU) ? (p.out_cols + 63) / 64 : (p.rows_per_expert + BM - 1) / BM;
  const int64_t chunks = static_cast<int64_t>(p.R) / nt + (groups < p.R ? groups : p.R);
  const int64_t tiles = chunks * n_wt * p.ksplit;
  const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
  cudaError_t e = (p.op == MOE_GEMM_GATEUP_SILU) ? dispatch<MOE_GEMM_GATEUP_SILU>(prm, asrc, nt, grid, p.wfmt, s)
                                                 : dispatch<MOE_GEMM_DOWN>(prm, asrc, nt, grid, p.wfmt, s);
  if (e != cudaSuccess || p.ksplit == 1) return e;
  const int64_t n = static_cast<int64_t>(p.R) * p.out_cols;
  const int fb = static_cast<int>((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  if (p.op == MOE_GEMM_GATEUP_SILU)
    (void)launch_pdl(splitk_finish_kernel<MOE_GEMM_GATEUP_SILU>, dim3(fb), dim3(256), 0, s, p.partial, p.ksplit, p.R, p.out_cols,
                                                                  p.out_mma_order ? 1 : 0, p.out, nullptr);
  else
    (void)launch_pdl(splitk_finish_kernel<MOE_GEMM_DOWN>, dim3(fb), dim3(256), 0, s, p.partial, p.ksplit, p.R, p.out_cols, 0, p.out,
                                                           p.out_f32);
  count_launches(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// self-test of the bounded waits: nothing ever arrives on this barrier
// ---------------------------------------------------------------------------
namespace {
__global__ void expire_wait_kernel(int* status, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0, timeout_ns, &abort_flag, status);
}
}  // namespace

cudaError_t launch_expire_wait(int* status, int64_t timeout_ns, cudaStream_t s) {
  expire_wait_kernel<<<1, 32, 0, s>>>(status, static_cast<unsigned long long>(timeout_ns));
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
