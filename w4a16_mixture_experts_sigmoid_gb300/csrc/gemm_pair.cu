// Steps 3 and 4 on CTA pairs: the grouped W4A16 expert GEMMs with one tcgen05
// MMA (cta_group::2, M = 256) covering the weight rows of two SMs.
//
// Same computation, weight format and K order as the one-CTA kernel in
// gemm_tc.cu ("Kimi-K2.6" catalog page, QUANT/PARAMS and GEOMETRY): a tile is
// now 256 weight rows of one expert (gate/up: 128 gate + 128 up rows) against
// NT token rows, run by a cluster of two CTAs on two SMs:
//   - each CTA streams and dequantises its own 128 weight rows into its own
//     tensor memory (rows 0-127 of the pair's A operand in CTA 0, 128-255 in
//     CTA 1), exactly as the one-CTA kernel does;
//   - each CTA loads half of the tile's token rows (NT/2) into its own shared
//     memory; the pair MMA reads both halves;
//   - one thread of CTA 0 issues the MMAs for both SMs, so each SM sees half as
//     many MMA issues per weight byte (an M=256 pair MMA costs about the same
//     issue time as an M=128 one);
//   - each CTA's accumulator rows sit in its own tensor memory, and each CTA
//     runs the epilogue of its rows.
// Cross-CTA hand-offs: CTA 1's token-row copies complete on CTA 0's "B full"
// barrier (cp.async.bulk.tensor with cta_group::2); CTA 1's dequant and
// epilogue warps arrive remotely on CTA 0's "A full" and "accumulator empty"
// barriers; the MMA commits arrive on both CTAs' barriers (multicast).
//
// Every wait is bounded as in the one-CTA kernel; the pair meets at a cluster
// barrier before it frees its tensor memory.
#include "gemm_tc_parts.cuh"

#include <atomic>
#include <cstring>
#include <type_traits>

namespace moe {
namespace {

using namespace tc;

template <int NT>
struct PairCfg {
  static constexpr int kHalf = NT / 2;                 // token rows loaded by each CTA
  static constexpr int kAStage = BM * 128;             // 128 rows x 256 inputs of int4
  static constexpr int kSStage = BM * 16;              // their bf16 scales
  static constexpr int kWStage = kAStage + kSStage;
  static constexpr int kBStage = NSUB * kHalf * 128;   // this CTA's half of the token rows, bf16
  static constexpr int kNBuf = NT <= 32 ? 3 : 2;       // A buffers in tensor memory (128 columns each)
  static constexpr int kAvail = kSmemLimit - kAlignSlack - kAuxBytes;
  static constexpr int kBFit = (kAvail - 3 * kWStage) / kBStage;
  static constexpr int kBStages = (kNBuf + 3 < kBFit ? kNBuf + 3 : kBFit);
  static constexpr int kWStagesFit = (kAvail - kBStages * kBStage) / kWStage;
  static constexpr int kWStages = kWStagesFit > 12 ? 12 : kWStagesFit;
  static constexpr int kWPeriod = (kWStages % 2 == 0) ? kWStages : 2 * kWStages;
  static constexpr int kBPeriod = (kBStages % 2 == 0) ? kBStages : 2 * kBStages;
  static constexpr int kAPeriod = (kNBuf % 2 == 0) ? kNBuf : 2 * kNBuf;
  static constexpr bool kBViaA = kAPeriod >= kBStages;
  static constexpr int kMmaGroups = NT <= 64 ? 2 : 1;
  static constexpr int kAccCol = kNBuf * 128;
  static constexpr int kColsNeeded = kAccCol + 2 * kMmaGroups * NT;
  static constexpr int kTmemCols = kColsNeeded <= 32 ? 32 : kColsNeeded <= 64 ? 64 : kColsNeeded <= 128 ? 128
                                   : kColsNeeded <= 256 ? 256 : 512;
  static constexpr int kSmemBytes = kAlignSlack + kWStages * kWStage + kBStages * kBStage + kAuxBytes;
  static_assert(NT >= 16 && NT % 16 == 0, "pair MMAs need N a multiple of 16");
  static_assert(kWStages >= 2 && kBStages >= 2, "each ring needs at least two stages");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory overflow");
  static_assert(8 * (3 * kWStages + 3 * kBStages + 4 * kNBuf + 5) + 16 + 2 * kMaxE + 4 * (kMaxE + 1) <= kAuxBytes,
                "barriers and tile table overflow the aux area");
  static_assert(kColsNeeded <= 512, "tensor memory overflow");
  static_assert(kWStage % 1024 == 0 && kBStage % 1024 == 0, "stages must keep 1024-byte alignment");
};

// YF32 (down only): fp32 rows to p.out_f32 instead of bf16 to p.out, chosen at compile time (a run-time
// branch in the epilogue costs the down kernels ~25%)
template <int OP, int NT, int FMT, bool YF32>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_pair_kernel(const __grid_constant__ TcParams p) {
  using C = PairCfg<NT>;
  constexpr int SW = C::kWStages;
  constexpr int SB = C::kBStages;
  constexpr int NB = C::kNBuf;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* bring = smem + SW * C::kWStage;
  uint8_t* aux = bring + SB * C::kBStage;
  uint64_t* wfull = reinterpret_cast<uint64_t*>(aux);   // [2][SW]: (stage parity, slot)
  uint64_t* wempty = wfull + 2 * SW;
  uint64_t* bfull = wempty + SW;                         // [2][SB], CTA 0's are the ones used
  uint64_t* bempty = bfull + 2 * SB;
  uint64_t* afull = bempty + SB;      // [2][NB]: (dequant group, A buffer), CTA 0's are the ones used
  uint64_t* aempty = afull + 2 * NB;  // [2][NB]
  uint64_t* accfull = aempty + 2 * NB;   // [2]
  uint64_t* accempty = accfull + 2;      // [2], CTA 0's are the ones used
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
  const uint32_t rank = cluster_ctarank();   // 0: issues the pair's MMAs; 1: its partner
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  // weight tiles of 256 rows: gate/up 128 gate + 128 up rows, split 64 + 64 per CTA; down 128 rows per CTA
  const int n_wt = (OP == MOE_GEMM_GATEUP_SILU) ? (p.out_cols + 127) / 128 : (p.rows_per_expert + 255) / 256;
  const int nk = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2 * SW; ++s) mbar_init(&wfull[s], 32);
    for (int s = 0; s < SW; ++s) mbar_init(&wempty[s], 4);
    for (int s = 0; s < 2 * SB; ++s) mbar_init(&bfull[s], 1);
    for (int s = 0; s < SB; ++s) mbar_init(&bempty[s], 1);
    for (int b = 0; b < 2 * NB; ++b) { mbar_init(&afull[b], 8); mbar_init(&aempty[b], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&accfull[a], C::kMmaGroups); mbar_init(&accempty[a], 8); }
    mbar_init(drain, C::kMmaGroups);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, C::kTmemCols);
  if (warp == 0) {
    if (!p.weights_ready) griddep_wait();
    // compact list of experts with rows, and the prefix of their tile counts (both CTAs build the
    // same list from the same offsets)
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
      const int ntl = f ? n_wt * ((cnt + NT - 1) / NT) : 0;
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
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers are initialised before either arrives on the other's
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_act = *n_act_s;
  const int total = tpre[n_act];

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer (this CTA's rows)
    const uint64_t pol_w = l2_policy_evict_first();
    constexpr int kScaleX = scale_x_per_stage<FMT>();   // one stage of scales, in map elements (16 bytes)
    const uint32_t txw = C::kAStage + (p.scale_tma ? BM * 16 : 0);
    const int kg = p.K / 32;
    int g = 0;
    bool ok = true;
    for (int i = pair; i < total && ok; i += n_pairs) {
      const TileInfo ti = decode_tile(i, n_act, act_e, tpre, p, NT, 1);
      const int wt = 2 * ti.wt + static_cast<int>(rank);   // this CTA's 128-row slice of the pair tile
      const int ebase = ti.e * p.rows_per_expert;
      int grow_lo, grow_hi;
      if (OP == MOE_GEMM_GATEUP_SILU) { grow_lo = ebase + wt * 64; grow_hi = ebase + p.out_cols + wt * 64; }
      else { grow_lo = ebase + wt * BM; grow_hi = grow_lo + 64; }
      for (int ks = 0; ks < nk; ++ks, ++g) {
        const int sw = g % SW;
        uint64_t* wf = &wfull[(g & 1) * SW + sw];
        if (!warp_wait(&wempty[sw], ((g / SW) & 1) ^ 1, p, abort_flag)) { ok = false; break; }
        uint8_t* sa = smem + sw * C::kWStage;
        uint8_t* ss = sa + C::kAStage;
        if (!p.scale_tma && FMT == WFMT_INT4) {
          uint16_t* sc = reinterpret_cast<uint16_t*>(ss);
          for (int r = lane; r < BM; r += 32) {
            const int grow = (r < 64) ? grow_lo + r : grow_hi + (r - 64);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int gi = ks * 8 + q;
              uint16_t v = 0;
              if (gi < kg && grow < p.rows_total) v = p.scales[static_cast<int64_t>(grow) * kg + gi];
              sc[r * 8 + q] = v;
            }
          }
        } else if (!p.scale_tma) {
          const uint8_t* src = reinterpret_cast<const uint8_t*>(p.scales);
          const int kb16 = p.K / 16;
          for (int r = lane; r < BM; r += 32) {
            const int grow = (r < 64) ? grow_lo + r : grow_hi + (r - 64);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const int gi = ks * 16 + q;
              uint8_t v = 0;
              if (gi < kb16 && grow < p.rows_total) v = src[static_cast<int64_t>(grow) * kb16 + gi];
              ss[r * 16 + q] = v;
            }
          }
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(wf, txw);
          tma_load_2d(sa, &p.tm_w, wf, ks * (BK / 8), grow_lo, pol_w);
          tma_load_2d(sa + 64 * 128, &p.tm_w, wf, ks * (BK / 8), grow_hi, pol_w);
          if (p.scale_tma) {
            tma_load_2d(ss, &p.tm_s, wf, ks * kScaleX, grow_lo, pol_w);
            tma_load_2d(ss + 64 * 16, &p.tm_s, wf, ks * kScaleX, grow_hi, pol_w);
          }
        } else {
          mbar_arrive(wf);
        }
      }
    }
    if (lane == 0) {
      for (int d = 0; d < SW && d < g; ++d) {
        const int gg = g - 1 - d;
        mbar_wait(&wfull[(gg & 1) * SW + gg % SW], (gg / C::kWPeriod) & 1, p.timeout_ns, nullptr, p.status);
      }
    }
    __syncwarp();
  } else if (warp == kBProducerWarp) {
    // ------------------------------------------------------------ token-row producer (this CTA's half)
    if (lane == 0) {
      griddep_wait();   // the token rows are the predecessor's output
      const uint64_t pol_b = l2_policy_evict_last();
      constexpr uint32_t txb = NSUB * NT * 128;   // both halves land on CTA 0's barrier
      int g = 0;
      bool ok = true;
      for (int i = pair; i < total && ok; i += n_pairs) {
        const TileInfo ti = decode_tile(i, n_act, act_e, tpre, p, NT, 1);
        const int row = ti.row0 + static_cast<int>(rank) * C::kHalf;
        for (int ks = 0; ks < nk; ++ks, ++g) {
          const int sbi = g % SB;
          if (C::kBViaA) {
            if (g >= SB) {
              const int gn = g - SB + NB;
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
          const uint32_t bf_leader = mapa_shared(smem_u32(bf), 0);
          if (rank == 0) mbar_arrive_expect_tx(bf, txb);
#pragma unroll
          for (int sub = 0; sub < NSUB; ++sub)
            tma_load_2d_pair(sb + sub * (C::kHalf * 128), &p.tm_b, bf_leader, ks * BK + sub * KSUB, row, pol_b);
        }
      }
      if (rank == 0) {
        // both halves of every stage issued land before this CTA's exit; CTA 1 waits at the final
        // cluster barrier, after this
        for (int d = 0; d < SB && d < g; ++d) {
          const int gg = g - 1 - d;
          mbar_wait_cluster(&bfull[(gg & 1) * SB + gg % SB], (gg / C::kBPeriod) & 1, p.timeout_ns, nullptr, p.status);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1 || (C::kMmaGroups == 2 && warp == kSecondMmaWarp)) {
    // ------------------------------------------------------------ MMA issuers (CTA 0 only)
    // with 128-token tiles the whole warp runs the loop and one elected lane issues (iss_wait)
    constexpr bool W = NT >= 128;
    if (rank == 0 && (W || lane == 0)) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, NT);
      const int mg = (warp == 1) ? 0 : 1;
      int g = 0, it = 0;
      bool ok = true;
      for (int i = pair; i < total && ok; i += n_pairs, ++it) {
        const int ab = it & 1;
        if (!iss_wait_cluster<W>(&accempty[ab], ((it >> 1) & 1) ^ 1, p, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + C::kAccCol + (mg * 2 + ab) * NT;
        bool first = true;
        for (int ks = 0; ks < nk; ++ks, ++g) {
          if (C::kMmaGroups == 2 && (g & 1) != mg) continue;
          const int sbi = g % SB;
          const int b = g % NB;
          if (!iss_wait_cluster<W>(&bfull[(g & 1) * SB + sbi], (g / C::kBPeriod) & 1, p, abort_flag)) {
            ok = false;
            break;
          }
          if (!iss_wait_cluster<W>(&afull[(g & 1) * NB + b], (g / C::kAPeriod) & 1, p, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bdesc0 = sw128_kmajor_desc(smem_u32(bring + sbi * C::kBStage));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // K step kk: swizzle sub-tile kk / 4, 32-byte column kk % 4 (the start-address field
            // counts 16-byte units and cannot carry out: shared memory is below 2^18 bytes)
            const uint32_t off = (kk >> 2) * (C::kHalf * 128) + (kk & 3) * 32;
            const uint32_t acc = (!first || kk > 0) ? 1u : 0u;
            iss_mma_ts_pair<W>(d_tmem, tmem + b * 128 + kk * 8, bdesc0 + (off >> 4), idesc, acc);
          }
          first = false;
          if (!C::kBViaA) iss_commit_pair<W>(&bempty[sbi], 3);
          iss_commit_pair<W>(&aempty[((g + NB) & 1) * NB + b], 3);
        }
        if (!ok) break;
        iss_commit_pair<W>(&accfull[ab], 3);
      }
      iss_commit_pair<W>(drain, 3);
      iss_wait<W>(drain, 0, p, nullptr);
    }
    __syncwarp();
  } else if (warp >= kFirstDqWarp && warp < kFirstEpiWarp) {
    // ------------------------------------------------------------ dequantise (this CTA's rows)
    const int grp = (warp - kFirstDqWarp) >> 2;
    const int q = warp & 3;
    const int r_sm = (OP == MOE_GEMM_GATEUP_SILU) ? (lane < 16 ? 16 * q + lane : 64 + 16 * q + (lane - 16)) : 32 * q + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
    int g = 0;
    bool ok = true;
    for (int i = pair; i < total && ok; i += n_pairs) {
      for (int ks = 0; ks < nk; ++ks, ++g) {
        if ((g & 1) != grp) continue;
        const int sw = g % SW;
        const int b = g % NB;
        const int a_need = a_releases_needed(g, NB, C::kAPeriod);
        if (!warp_wait(&wfull[(g & 1) * SW + sw], (g / C::kWPeriod) & 1, p, abort_flag)) { ok = false; break; }
        const uint8_t* arow = smem + sw * C::kWStage + r_sm * 128;
        const uint4 sv = *reinterpret_cast<const uint4*>(smem + sw * C::kWStage + C::kAStage + r_sm * 16);
        const uint32_t sw4[4] = {sv.x, sv.y, sv.z, sv.w};
        uint4 wv[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) wv[c] = *reinterpret_cast<const uint4*>(arow + ((c ^ (r_sm & 7)) << 4));
        // the conversion's form, once per stage for the whole warp (as in the single-CTA kernel)
        const bool fast = (FMT == WFMT_INT4) && __all_sync(0xFFFFFFFFu, int4_row_fast(sw4));
        auto convert = [&](auto fast_tag) -> bool {
          constexpr bool kFast = decltype(fast_tag)::value;
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
              for (int c = 0; c < 4; ++c) wv[c] = *reinterpret_cast<const uint4*>(arow + (((c + 4) ^ (r_sm & 7)) << 4));
              __syncwarp();
              if (lane == 0) mbar_arrive(&wempty[sw]);
            }
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              const int c = half * 4 + cc;
              uint32_t dqc[16];
              if (c >= kPreChunks) dequant_chunk<FMT, kFast>(wv[cc], sw4, c, dqc);
              const uint32_t* dq = (c < kPreChunks) ? pre[c < kPreChunks ? c : 0] : dqc;
              tmem_st8(lane_base + b * 128 + c * 16, dq);
              tmem_st8(lane_base + b * 128 + c * 16 + 8, dq + 8);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            uint64_t* af = &afull[grp * NB + b];
            if (rank == 0) mbar_arrive(af);
            else mbar_arrive_remote(mapa_shared(smem_u32(af), 0));
          }
          return true;
        };
        if (!(fast ? convert(std::true_type{}) : convert(std::false_type{}))) { ok = false; break; }
      }
    }
  } else if (warp >= kFirstEpiWarp && warp < kFirstEpiWarp + 4) {
    // ------------------------------------------------------------ epilogue (this CTA's rows)
    const int q = warp & 3;
    const int l = 32 * q + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
    int it = 0;
    for (int i = pair; i < total; i += n_pairs, ++it) {
      const TileInfo ti = decode_tile(i, n_act, act_e, tpre, p, NT, 1);
      const int wt = 2 * ti.wt + static_cast<int>(rank);
      const int ab = it & 1;
      if (!warp_wait(&accfull[ab], (it >> 1) & 1, p, abort_flag)) break;
      tc_fence_after();
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
          const float gs = fp4_sum_scale(__ldg(p.gscale + ti.e));
#pragma unroll
          for (int c = 0; c < 16; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * gs);
        }
        if (OP == MOE_GEMM_GATEUP_SILU) {
          float u[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) u[c] = __shfl_down_sync(0xFFFFFFFFu, __uint_as_float(v[c]), 16);
          const int j = wt * 64 + 16 * q + lane;
          if (lane < 16 && j < p.out_cols) {
            const int col = p.out_mma_order ? mma_order_pos(j) : j;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int row = ti.row0 + cb + c;
              if (cb + c < ti.nvalid && row < p.R) {
                const float gt = __uint_as_float(v[c]);
                const float h = __fdividef(gt, 1.0f + __expf(-gt)) * u[c];
                p.out[static_cast<int64_t>(row) * p.out_cols + col] = __bfloat16_as_ushort(__float2bfloat16_rn(h));
              }
            }
          }
        } else {
          const int n = wt * BM + l;
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
      if (lane == 0) {
        if (rank == 0) mbar_arrive(&accempty[ab]);
        else mbar_arrive_remote(mapa_shared(smem_u32(&accempty[ab]), 0));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // CTA 0's MMAs have drained before either CTA frees its tensor memory
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, C::kTmemCols);
}

// Clusters of two that can be resident at once, per device ordinal and kernel.
template <int OP, int NT, int FMT, bool YF32>
int max_pairs(cudaStream_t s, int num_sms) {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int v = cached[dev].load();
  if (v > 0) return v;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (num_sms / 2));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = PairCfg<NT>::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_pair_kernel<OP, NT, FMT, YF32>, &cfg) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    n = num_sms / 2;
  }
  cached[dev].store(n);
  return n;
}

template <int OP, int NT, int FMT, bool YF32>
cudaError_t run_pair_y(const TcParams& prm, int64_t pair_tiles, int num_sms, cudaStream_t s) {
  using C = PairCfg<NT>;
  static std::atomic<uint64_t> opted_in{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit == 0 || !(opted_in.load() & bit)) {
    e = cudaFuncSetAttribute(tc_gemm_pair_kernel<OP, NT, FMT, YF32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    opted_in.fetch_or(bit);
  }
  const int cap = max_pairs<OP, NT, FMT, YF32>(s, num_sms);
  const int pairs = static_cast<int>(pair_tiles < cap ? pair_tiles : cap);
  if (pairs <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see griddep_launch in the kernel
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, tc_gemm_pair_kernel<OP, NT, FMT, YF32>, prm);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int OP, int NT, int FMT>
cudaError_t run_pair(const TcParams& prm, int64_t pair_tiles, int num_sms, cudaStream_t s) {
  if (OP == MOE_GEMM_DOWN && prm.out_f32 != nullptr)
    return run_pair_y<OP, NT, FMT, OP == MOE_GEMM_DOWN>(prm, pair_tiles, num_sms, s);
  return run_pair_y<OP, NT, FMT, false>(prm, pair_tiles, num_sms, s);
}

template <int OP, int FMT>
cudaError_t dispatch_pair(const TcParams& prm, int nt, int64_t pair_tiles, int num_sms, cudaStream_t s) {
  switch (nt) {
    case 16: return run_pair<OP, 16, FMT>(prm, pair_tiles, num_sms, s);
    case 32: return run_pair<OP, 32, FMT>(prm, pair_tiles, num_sms, s);
    case 64: return run_pair<OP, 64, FMT>(prm, pair_tiles, num_sms, s);
    case 128: return run_pair<OP, 128, FMT>(prm, pair_tiles, num_sms, s);
  }
  return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_gemm_pair(const GemmProblem& p, int nt, int num_sms, cudaStream_t s) {
  if (p.R <= 0) return cudaSuccess;
  if (p.bf16_weights || !p.a_mma_order || p.ksplit != 1) return cudaErrorNotSupported;
  if (p.E > kMaxE || num_sms < 2) return cudaErrorNotSupported;
  if (p.wfmt == WFMT_FP4 && p.gscale == nullptr) return cudaErrorInvalidValue;
  TcParams prm;
  memset(&prm, 0, sizeof(prm));
  const int groups = p.uniform_rows >= 0 ? 1 : p.E;
  const int64_t rows_total = static_cast<int64_t>(groups) * p.rows_per_expert;
  bool ok = make_map_2d(&prm.tm_w, CU_TENSOR_MAP_DATA_TYPE_INT32, p.w, p.K / 8, rows_total, p.K / 2, BK / 8, 64,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  prm.scale_tma = (p.K % 256 == 0) ? 1 : 0;
  if (ok && prm.scale_tma) ok = make_scale_map(&prm.tm_s, p.wfmt, p.scales, p.K, rows_total);
  // each CTA loads half of a tile's token rows
  if (ok)
    ok = make_map_2d(&prm.tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.a, p.K, p.R, 2ull * p.K, KSUB, nt / 2,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  prm.scales = p.scales;
  prm.gscale = p.gscale;
  prm.offsets = p.offsets;
  prm.out = p.out;
  prm.out_f32 = (p.op == MOE_GEMM_DOWN) ? p.out_f32 : nullptr;
  prm.status = p.status;
  prm.E = p.E;
  prm.K = p.K;
  prm.rows_per_expert = p.rows_per_expert;
  prm.out_cols = p.out_cols;
  prm.uniform_rows = p.uniform_rows;
  prm.min_rows = p.min_rows;
  prm.max_rows = p.max_rows;
  prm.weights_ready = p.weights_ready ? 1 : 0;
  prm.ksplit = 1;
  prm.partial = nullptr;
  prm.rows_total = static_cast<int>(rows_total);
  prm.R = p.R;
  prm.out_mma_order = p.out_mma_order ? 1 : 0;
  prm.timeout_ns = 2000000000ull;
  const int n_wt = (p.op == MOE_GEMM_GATEUP_SILU) ? (p.out_cols + 127) / 128 : (p.rows_per_expert + 255) / 256;
  const int64_t chunks = static_cast<int64_t>(p.R) / nt + (groups < p.R ? groups : p.R);
  const int64_t pair_tiles = chunks * n_wt;
  if (p.wfmt == WFMT_FP4)
    return (p.op == MOE_GEMM_GATEUP_SILU)
               ? dispatch_pair<MOE_GEMM_GATEUP_SILU, WFMT_FP4>(prm, nt, pair_tiles, num_sms, s)
               : dispatch_pair<MOE_GEMM_DOWN, WFMT_FP4>(prm, nt, pair_tiles, num_sms, s);
  return (p.op == MOE_GEMM_GATEUP_SILU) ? dispatch_pair<MOE_GEMM_GATEUP_SILU, WFMT_INT4>(prm, nt, pair_tiles, num_sms, s)
                                        : dispatch_pair<MOE_GEMM_DOWN, WFMT_INT4>(prm, nt, pair_tiles, num_sms, s);
}

}  // namespace moe
