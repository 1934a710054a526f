// Persistent tcgen05 GEMM engine on CTA pairs (cta_group::2) for sm_103a.
//
// A cluster of two CTAs (two SMs) computes one 256 x 256 tile: CTA r of the pair loads A
// rows [128r, 128r+128) and B columns [128r, 128r+128) of the tile's 64-deep K slices
// into its own shared memory, the leader CTA (r = 0) issues tcgen05.mma.cta_group::2
// (M = 256, N = 256), and each CTA's TMEM receives its 128 rows x 256 fp32 columns.
// Each SM thus streams half of B per MMA (the pair shares the B slice) and keeps two
// 256-column accumulators, so one tile's epilogue overlaps the next tile's MMAs.
//
// Pair signalling (no data multicast; each CTA loads its own operands):
//   full[s]    leader only: its producer's arrive.expect_tx of both halves' bytes; both
//              CTAs' TMA loads of stage s complete_tx on it (cp.async.bulk.tensor with
//              .cta_group::2 and the leader's barrier address from mapa).
//   empty[s]   both: the leader's MMA warp commits once per stage with the multicast form
//              of tcgen05.commit, arriving on the barrier at the same offset in both CTAs.
//   tfull[a]   both: likewise, one commit per tile.
//   tempty[a]  leader only: 4 local + 4 peer epilogue warps arrive (peer remotely).
// Every wait is bounded as in the single-CTA engine.
#pragma once
#include "tl_engine.cuh"

namespace tl {

struct Geo2 {
  static constexpr int kStages = 6;
  static constexpr int kABytes = 128 * kBK * 2;        // 16 KB: this CTA's 128 rows of A
  static constexpr int kBBytes = 128 * kBK * 2;        // 16 KB: this CTA's 128 columns of B
  static constexpr int kStageBytes = kABytes + kBBytes;  // 32 KB
  static constexpr int kAccStride = 256;
  static constexpr int kAccBufs = 2;
  static_assert(kStages * kStageBytes == kRingBytes, "stage ring");
};

// Waits on barriers completed from the peer CTA (remote TMA transactions, remote
// tcgen05.commit, remote arrivals) use the CTA-scope try_wait of mbar_wait: the barrier's
// own completion orders what it guards (the transaction count for TMA data, the commit for
// MMA completion, tcgen05.wait::ld before the arrival for TMEM reads), as in CUTLASS's two-SM
// kernels.  Measured against cluster-scope acquire on the GEMM+RS pair kernel: 2311.6 vs
// 2333.4 us under ncu.

// One 64-deep K slice of the pair tile: 4 x tcgen05.mma.cta_group::2 (256 x 256 x 16).
__device__ __forceinline__ void mma_stage_pair(uint32_t d, uint32_t a0, uint32_t b0, int kb) {
  constexpr uint32_t idesc = umma_idesc_bf16(256, kBN, true);
#pragma unroll
  for (int k = 0; k < kBK / 16; ++k) {
    const uint64_t ad = umma_desc_sw128(a0 + k * 32, 16, 1024);
    const uint64_t bd = umma_desc_sw128(b0 + k * 2048, TL_B_LBO, TL_B_SBO);
    umma_bf16_pair(d, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
  }
}

template <class Op, bool Trace>
__device__ __forceinline__ void pair_producer(const typename Op::Params& p, const Smem& sm, int lane, int gi,
                                              int gn, uint32_t rank) {
  const Common& c = p.common;
  const int ntiles = Op::num_tiles(p);
  uint32_t stage = 0, phase = 0;
  uint32_t filled = 0, fill_parity = 0;
  bool ok = true;
  constexpr bool tr = Trace;
  for (int t = gi; t < ntiles && ok; t += gn) {
    Job j = Op::job(p, t);
    j.rank = static_cast<int>(rank);
    const uint64_t tt0 = tr ? globaltimer() : 0;
    uint64_t stall = 0;
    for (int kb = 0; kb < j.kblocks; ++kb) {
      const uint64_t w0 = tr ? globaltimer() : 0;
      Op::wait_deps(p, j, kb, lane);
      if (tr && lane == 0) {
        const uint64_t w1 = globaltimer();
        if (w1 - w0 > kTraceMinWaitNs) trace_span(c, kTrProdWait, t, w0, w1);
      }
      if (lane == 0) {
        const uint64_t e0 = tr ? globaltimer() : 0;
        ok = rank == 0 ? mbar_wait(&sm.empty[stage], phase ^ 1u, c, kSiteEmpty)
                       : mbar_wait(&sm.empty[stage], phase ^ 1u, c, kSiteEmpty);
        if (tr) stall += globaltimer() - e0;
        if (ok) {
          // the leader's full[stage] counts both CTAs' bytes; the loads below complete on it
          if (rank == 0) mbar_arrive_expect_tx(&sm.full[stage], 2 * Op::kTxBytes);
          Op::load(p, j, kb, sm.a(stage), sm.b(stage), &sm.full[stage]);
          filled |= 1u << stage;
          fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      if (++stage == Geo2::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (tr && lane == 0) {
      trace_span(c, kTrProdTile, t, tt0, globaltimer());
      trace_span(c, kTrProdStall, t, tt0, tt0 + stall);
    }
  }
  // Drain (leader): its full[s] completes when both CTAs' loads of that fill have landed.
  if (lane == 0 && rank == 0) {
    for (int s = 0; s < Geo2::kStages; ++s)
      if (filled & (1u << s)) mbar_wait(&sm.full[s], (fill_parity >> s) & 1u, c, kSiteDrain);
  }
  __syncwarp();
}

// Leader: issue the pair MMAs and commit their completion to both CTAs' barriers.  The
// peer's MMA warp has nothing to do.
template <class Op, bool Trace>
__device__ __forceinline__ void pair_mma(const typename Op::Params& p, const Smem& sm, int lane, uint32_t tmem_base,
                                         int gi, int gn, uint32_t rank) {
  if (rank != 0) return;
  const Common& c = p.common;
  const int ntiles = Op::num_tiles(p);
  uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
  bool ok = true;
  constexpr bool tr = Trace;
  for (int t = gi; t < ntiles && ok; t += gn) {
    const Job j = Op::job(p, t);
    if (lane == 0) {
      const uint64_t a0t = tr ? globaltimer() : 0;
      ok = mbar_wait(&sm.tempty[acc], acc_phase ^ 1u, c, kSiteTmemEmpty);
      tc_fence_after();
      const uint64_t tt0 = tr ? globaltimer() : 0;
      if (tr && tt0 - a0t > kTraceMinWaitNs) trace_span(c, kTrMmaAccWait, t, a0t, tt0);
      uint64_t starve = 0;
      const uint32_t d = tmem_base + acc * Geo2::kAccStride;
      for (int kb = 0; kb < j.kblocks && ok; ++kb) {
        const uint64_t f0 = tr ? globaltimer() : 0;
        ok = mbar_wait(&sm.full[stage], phase, c, kSiteFull);
        if (tr) starve += globaltimer() - f0;
        if (!ok) break;
        tc_fence_after();
        mma_stage_pair(d, smem_u32(sm.a(stage)), smem_u32(sm.b(stage)), kb);
        umma_commit_pair_both(&sm.empty[stage]);
        if (++stage == Geo2::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        umma_commit_pair_both(&sm.tfull[acc]);
      }
      if (tr) {
        trace_span(c, kTrMmaTile, t, tt0, globaltimer());
        trace_span(c, kTrMmaStarve, t, tt0, tt0 + starve);
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (++acc == Geo2::kAccBufs) {
      acc = 0;
      acc_phase ^= 1u;
    }
  }
  // Drain: every pair MMA issued has completed before TMEM is freed.
  if (lane == 0) {
    umma_commit_pair(sm.drain);
    mbar_wait(sm.drain, 0, c, kSiteDrain);
  }
  __syncwarp();
}

template <class Op, bool Trace>
__device__ __forceinline__ void pair_epilogue(const typename Op::Params& p, const Smem& sm, int warp, int lane,
                                              uint32_t tmem_base, int gi, int gn, uint32_t rank) {
  constexpr int E = Op::kEpiWarps;
  static_assert(E == 4, "pair epilogue uses one warp per TMEM lane quadrant");
  const Common& c = p.common;
  const int ntiles = Op::num_tiles(p);
  const int q = warp & 3;
  const int ew = warp - 2;
  EpiStage es;
  es.nbuf = 2;
  es.buf[0] = sm.epi + (ew * 2) * kEpiBufBytes;
  es.buf[1] = sm.epi + (ew * 2 + 1) * kEpiBufBytes;
  es.idx = 0;
  Op::template epilogue_prologue<Trace>(p, ew, lane);
  const uint32_t tempty_leader0 = mapa_shared(smem_u32(&sm.tempty[0]), 0);
  uint32_t acc = 0, acc_phase = 0;
  bool ok = true;
  constexpr bool tr = Trace;
  for (int t = gi; t < ntiles && ok; t += gn) {
    Job j = Op::job(p, t);
    j.rank = static_cast<int>(rank);
    const uint64_t w0 = tr ? globaltimer() : 0;
    ok = rank == 0 ? mbar_wait(&sm.tfull[acc], acc_phase, c, kSiteTmemFull)
                   : mbar_wait(&sm.tfull[acc], acc_phase, c, kSiteTmemFull);
    if (!ok) break;
    tc_fence_after();
    if (tr && lane == 0) {
      const uint64_t tt0 = globaltimer();
      if (tt0 - w0 > kTraceMinWaitNs) trace_span(c, kTrEpiWait, t, w0, tt0);
      trace_open(c, kTrEpiTile, t, tt0);
    }
    // This CTA's 128 rows are rows [128 rank, 128 rank + 128) of the pair tile; the ops'
    // epilogues address row half h at taddr + 256 h, so offset the base by -256 rank.
    const uint32_t taddr = tmem_base + acc * Geo2::kAccStride + (static_cast<uint32_t>(q * 32) << 16) - rank * 256u;
    Op::epilogue(p, j, taddr, q, lane, es, static_cast<int>(rank), static_cast<int>(rank) + 1);
    if (Op::publishes(p, j)) {
      if (lane == 0) {
        bulk_wait<0>();
        fence_proxy_async_global();
        __threadfence();
        const uint32_t old = atomicAdd(&sm.epi_cnt[acc], 1u);
        if ((old & (E - 1u)) == E - 1u) {
          __threadfence();
          Op::publish(p, j);
        }
      }
      __syncwarp();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (rank == 0)
        mbar_arrive(&sm.tempty[acc]);
      else
        mbar_arrive_cluster(tempty_leader0 + acc * 8u);
    }
    if (tr && lane == 0) trace_close(c, globaltimer());
    if (++acc == Geo2::kAccBufs) {
      acc = 0;
      acc_phase ^= 1u;
    }
  }
  if (lane == 0) bulk_wait<0>();
  __syncwarp();
}

template <class Op, bool Trace>
__global__ void __launch_bounds__(op_max_threads<Op>(), 1)
    persistent_kernel_pair(const __grid_constant__ typename Op::Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Smem sm;
  sm.stages = base;
  sm.stage_bytes = Geo2::kStageBytes;
  sm.a_bytes = Geo2::kABytes;
  sm.epi = base + kRingBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm.epi + kEpiBytes);
  sm.full = bars;
  sm.empty = bars + Geo2::kStages;
  sm.tfull = bars + 2 * Geo2::kStages;
  sm.tempty = bars + 2 * Geo2::kStages + 2;
  sm.drain = bars + 2 * Geo2::kStages + 4;
  sm.tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * Geo2::kStages + 5);
  sm.epi_cnt = sm.tmem_slot + 2;
  static_assert((2 * Geo2::kStages + 5) * 8 + 16 <= kBarBytes - 4 * kTraceWarps, "barrier area");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int gi = static_cast<int>(blockIdx.x >> 1);
  const int gn = static_cast<int>(gridDim.x >> 1);
  if constexpr (Trace) trace_begin();
  if (threadIdx.x == 0) {
    for (int s = 0; s < Geo2::kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.tfull[b], 1);
      mbar_init(&sm.tempty[b], 2 * Op::kEpiWarps);
    }
    mbar_init(sm.drain, 1);
    sm.epi_cnt[0] = 0;
    sm.epi_cnt[1] = 0;
    fence_mbar_init();
    Op::prefetch(p);
  }
  if (warp == 1) {
    tmem_alloc_pair(sm.tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers and TMEM are ready before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;

  if (warp == 0) {
    pair_producer<Op, Trace>(p, sm, lane, gi, gn, rank);
  } else if (warp == 1) {
    pair_mma<Op, Trace>(p, sm, lane, tmem_base, gi, gn, rank);
  } else if (warp < 2 + Op::kEpiWarps) {
    pair_epilogue<Op, Trace>(p, sm, warp, lane, tmem_base, gi, gn, rank);
  } else {
    Op::template mover<Trace>(p, warp - 2 - Op::kEpiWarps, lane);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the leader's MMAs are drained and both epilogues are done with TMEM
  if constexpr (Trace) trace_end(p.common);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace tl
