// Persistent, warp-specialised tcgen05 GEMM engine for sm_103a.
//
// One CTA per SM walks the global tile sequence t = blockIdx.x, blockIdx.x + grid, ...
// Warp roles:
//   warp 0      TMA producer.  Before a tile's loads it performs the consumer side
//               of the tile-centric signal primitives (consumer_tile_wait /
//               peer_tile_wait of "TileLink ...", §3.2 Table 3): the whole warp polls the
//               tile's ready signals with acquire loads, then fences the async proxy,
//               then lane 0 issues the TMA loads of the 4-stage A/B ring.
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators) and issues
//               tcgen05.mma from one lane; tcgen05.commit frees smem stages and hands
//               finished accumulators to the epilogue.
//   warps 2..   epilogue (4 warps, or 8 = one warpgroup per 128-row half of a 256-row
//               tile): tcgen05.ld -> registers -> per-op math -> swizzled smem
//               staging -> TMA store / TMA bulk reduction; then the producer side of the
//               signal primitives (producer_tile_notify) for tiles others wait on.
//   warps 6..   shard mover (tile_pull_data of §3.2.2, pull mode): copies shard chunks
//               between the emulated ranks' buffers and releases one signal per chunk.
// The communication tile (mover chunk) and the compute tile (128x256) are chosen
// independently, as in the decoupled design space of §3.1.
//
// Every wait is bounded by the context's timeout (on %globaltimer).  A signal wait that
// runs out records TL_ERR_TIMEOUT in the status word and the producer continues, so the
// pipeline drains normally; an mbarrier wait that runs out (an internal fault) records
// the error and the role stops after draining its own copies in flight.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "tl_ptx.cuh"
#include "tl_sched.h"

namespace tl {

constexpr int kMaxStages = 4;
constexpr int kBStageBytes = kBN * kBK * 2;  // 32 KB of B per stage
constexpr int kEpiBufBytes = 32 * 128;       // 32 rows x 128 B
constexpr int kEpiBytes = 4 * 2 * kEpiBufBytes;  // 4 warps x 2 buffers
constexpr int kBarBytes = 256;
constexpr int kRingBytes = 196608;  // the A/B stage ring: 4 x 48 KB (BM = 128) or 3 x 64 KB (BM = 256)
constexpr int kSmemBytes = 1024 + kRingBytes + kEpiBytes + kBarBytes;
constexpr int kTmemCols = 512;

// Tile geometry.  BM = 128: one 128x256 accumulator per tile, 4 stages of 48 KB, two
// TMEM accumulators so the epilogue of one tile overlaps the next tile's MMAs.
// BM = 256: two 128x256 accumulators per tile (rows 0-127 and 128-255) fed by the same
// B slice, 3 stages of 64 KB, one TMEM buffer.  The 256-row tile reads each B slice from
// shared memory once per two MMAs, cutting shared-memory traffic per MMA from ~24 KB to
// ~20 KB (operand reads + TMA fill), which is what bounds the 128-row tile.
template <int BM>
struct Geo {
  static_assert(BM == 128 || BM == 256, "tile rows");
  static constexpr int kStages = BM == 256 ? 3 : 4;
  static constexpr int kABytes = BM * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBStageBytes;
  static constexpr int kAccBufs = BM == 256 ? 1 : 2;
  static constexpr int kAccStride = BM == 256 ? 512 : 256;  // TMEM columns per accumulator buffer
  static_assert(kStages * kStageBytes == kRingBytes, "stage ring");
};
constexpr int kMaxMoverWarps = 4;

// Status codes written to the device status word (host maps them to TL_ERR_*).
constexpr unsigned kStatusTimeout = 4;
// Places a wait can run out (recorded in DevStatus::where).
enum WaitSite : unsigned {
  kSiteSignal = 1, kSiteEmpty = 2, kSiteFull = 3, kSiteTmemEmpty = 4, kSiteTmemFull = 5,
  kSitePeer = 6, kSiteDrain = 7, kSiteCombine = 8
};

struct DevStatus {
  unsigned int code;
  unsigned int where;
  unsigned int abort;
  unsigned int pad;
  unsigned long long info;
};

// One trace span: a warp role's activity [t0, t0 + dur) in %globaltimer nanoseconds.
struct TraceRec {
  unsigned long long t0;
  unsigned int dur;
  unsigned int tag;  // kind << 24 | (tile or chunk index & 0xffffff)
};

struct Common {
  DevStatus* status;
  unsigned long long epoch;       // this call's signal value (never 0)
  unsigned long long timeout_ns;  // bound of every wait
  int mover_warps;
  int trace_cap;                  // spans per warp the trace buffer holds
  int trace_ctas;                 // CTAs the trace buffer holds
  unsigned int* trace_hdr;        // trace buffer (null: tracing off): header, counts, spans
  TraceRec* trace;
};

// ------------------------------------------------------------------ trace spans
// Span kinds (the trace buffer's tag field carries kind << 24 | index).
enum TraceKind : unsigned {
  kTrProdTile = 1,     // producer: the tile's first wait .. its last load issued
  kTrProdWait = 2,     // producer: one dependency-signal wait
  kTrProdStall = 3,    // producer: total wait for free ring stages in the tile (t0 = tile start)
  kTrMmaTile = 4,      // MMA: accumulator acquired .. the tile's last commit issued
  kTrMmaStarve = 5,    // MMA: total wait for filled stages in the tile (t0 = tile start)
  kTrMmaAccWait = 6,   // MMA: wait for a free accumulator
  kTrEpiTile = 7,      // epilogue: accumulator full .. accumulator released
  kTrEpiWait = 8,      // epilogue: wait for a full accumulator
  kTrMoverChunk = 9,   // mover: one chunk copied and signalled
  kTrSideTile = 10,    // side partition: one unit of work from the start of its wait (e.g. one y tile)
  kTrSideWait = 11,    // side partition: its signal wait
};
constexpr int kTraceWarps = 16;           // warps per CTA with a span list
constexpr unsigned kTraceMinWaitNs = 200;  // shorter waits are not recorded
constexpr unsigned kTraceMagic = 0x544c5452u;
constexpr int kTraceHdrWords = 8;

// Per-warp span counters: 16 words at a fixed place in the barrier area of dynamic
// shared memory, which neither engine's barriers nor any side role use.
__device__ __forceinline__ uint32_t* trace_slots() {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  return reinterpret_cast<uint32_t*>(base + kRingBytes + kEpiBytes + kBarBytes - 4 * kTraceWarps);
}

__device__ __forceinline__ bool tracing(const Common& c) { return c.trace_hdr != nullptr; }

// Record one span of the calling warp (call from one lane).
__device__ __forceinline__ void trace_span(const Common& c, unsigned kind, int index, uint64_t t0, uint64_t t1) {
  if (!tracing(c) || static_cast<int>(blockIdx.x) >= c.trace_ctas) return;
  const int w = static_cast<int>(threadIdx.x >> 5);
  if (w >= kTraceWarps) return;
  uint32_t* cnt = trace_slots() + w;
  const uint32_t i = *cnt;
  *cnt = i + 1;
  if (i < static_cast<uint32_t>(c.trace_cap)) {
    TraceRec r;
    r.t0 = t0;
    const uint64_t d = t1 > t0 ? t1 - t0 : 0;
    r.dur = d > 0xffffffffull ? 0xffffffffu : static_cast<unsigned>(d);
    r.tag = (kind << 24) | (static_cast<unsigned>(index) & 0xffffffu);
    c.trace[(static_cast<size_t>(blockIdx.x) * kTraceWarps + w) * c.trace_cap + i] = r;
  }
}

// Open a span of the calling warp at t0 (call from one lane); trace_close sets its duration.
// Nothing stays live in registers in between, which keeps the epilogue's register budget.
__device__ __forceinline__ void trace_open(const Common& c, unsigned kind, int index, uint64_t t0) {
  trace_span(c, kind, index, t0, t0);
}
__device__ __forceinline__ void trace_close(const Common& c, uint64_t t1) {
  if (!tracing(c) || static_cast<int>(blockIdx.x) >= c.trace_ctas) return;
  const int w = static_cast<int>(threadIdx.x >> 5);
  if (w >= kTraceWarps) return;
  const uint32_t i = trace_slots()[w] - 1;
  if (i < static_cast<uint32_t>(c.trace_cap)) {
    TraceRec* r = c.trace + (static_cast<size_t>(blockIdx.x) * kTraceWarps + w) * c.trace_cap + i;
    const uint64_t d = t1 > r->t0 ? t1 - r->t0 : 0;
    r->dur = d > 0xffffffffull ? 0xffffffffu : static_cast<unsigned>(d);
  }
}

// Kernel start (all threads, before the CTA's first barrier): zero the span counters.
__device__ __forceinline__ void trace_begin() {
  if (threadIdx.x < kTraceWarps) trace_slots()[threadIdx.x] = 0;
}

// Kernel end (all threads, after the CTA's last barrier): publish the span counts, and
// from CTA 0 the header {magic, version 1, grid, warps per CTA, spans per warp, CTAs held}.
__device__ __forceinline__ void trace_end(const Common& c) {
  if (!tracing(c) || static_cast<int>(blockIdx.x) >= c.trace_ctas) return;
  if (threadIdx.x < kTraceWarps)
    c.trace_hdr[kTraceHdrWords + blockIdx.x * kTraceWarps + threadIdx.x] = trace_slots()[threadIdx.x];
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    c.trace_hdr[0] = kTraceMagic;
    c.trace_hdr[1] = 1u;
    c.trace_hdr[2] = gridDim.x;
    c.trace_hdr[3] = kTraceWarps;
    c.trace_hdr[4] = static_cast<unsigned>(c.trace_cap);
    c.trace_hdr[5] = static_cast<unsigned>(c.trace_ctas);
  }
}

__device__ __forceinline__ void report_timeout(DevStatus* st, unsigned where, unsigned long long info) {
  if (atomicCAS(&st->code, 0u, kStatusTimeout) == 0u) {
    st->where = where;
    st->info = info;
  }
  atomicExch(&st->abort, 1u);
}

__device__ __forceinline__ bool aborted(const DevStatus* st) {
  return ld_relaxed_gpu_u32(&st->abort) != 0u;
}

// Bounded mbarrier wait.  Returns false (and records the site) when it runs out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const Common& c, unsigned site) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer();
  uint32_t n = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++n & 63u) == 0u && globaltimer() - t0 > 4ull * c.timeout_ns) {
      report_timeout(c.status, site, 0);
      return false;
    }
  }
  return true;
}

// Warp-collective signal wait: every lane polls its share of `count` signals at
// flags[i] until each equals `want` (acquire), then the async proxy is fenced so the
// TMA loads that follow observe the data the signals publish.  Returns false on
// timeout (or if another wait already aborted the call); the caller proceeds anyway.
__device__ __forceinline__ bool warp_wait_signals(const uint64_t* flags, int count, uint64_t want,
                                                  const Common& c, int lane, unsigned site,
                                                  unsigned long long info) {
  bool ok = true;
  uint64_t t0 = 0;
  uint32_t n = 0;
  for (;;) {
    bool mine = true;
    for (int i = lane; i < count; i += 32) mine &= (ld_acquire_gpu(flags + i) == want);
    if (__all_sync(0xffffffffu, mine)) break;
    if ((++n & 15u) == 0u) {
      uint64_t now = globaltimer();
      if (t0 == 0) t0 = now;
      const bool expired = (now - t0 > c.timeout_ns) || aborted(c.status);
      if (__any_sync(0xffffffffu, expired)) {
        if (lane == 0) report_timeout(c.status, site, info);
        ok = false;
        break;
      }
    }
  }
  fence_proxy_async_global();
  return ok;
}

// Single-signal wait by every lane of a warp (used by epilogue warps for peer signals).
__device__ __forceinline__ bool warp_wait_one(const uint64_t* flag, uint64_t want, const Common& c, int lane,
                                              unsigned site, unsigned long long info) {
  return warp_wait_signals(flag, 1, want, c, lane, site, info);
}

// Generic tile description produced by an op's scheduler.
struct Job {
  int kind;     // op-specific
  int a_sel;    // which A tensor map
  int a_row;    // A row coordinate
  int b_sel;    // which B tensor map
  int b_col;    // B column coordinate
  int b_z;      // third B coordinate (expert), 0 if unused
  int kblocks;  // K / 64, rounded up
  int x0, x1, x2, x3;  // op-specific (ranks, owners, blocks)
  int rank = 0;        // CTA of a pair (pair engine): which 128-row / 128-column half it owns
};

// Defaults for the optional hooks of an op (an op derives from OpBase<its Params>).
template <class P>
struct OpBase {
  // Whether this CTA belongs to the GEMM partition; (gi, gn) = its index / partition size.
  static __device__ bool gemm_partition(const P&, int&, int&) { return true; }
  // Work of CTAs outside the GEMM partition (all threads of the CTA).  The hooks that run
  // outside the GEMM roles take the kernel's Trace flag (true: they may record spans).
  template <bool Trace>
  static __device__ void side_role(const P&, int, int, uint8_t*) {}
  static __device__ void producer_init(const P&) {}
  static __device__ void prefetch(const P&) {}
  static __device__ bool publishes(const P&, const Job&) { return false; }
  static __device__ void publish(const P&, const Job&) {}
  template <bool Trace>
  static __device__ void mover(const P&, int, int) {}
  // Work the epilogue warps may do before their first tile (they idle until then).
  template <bool Trace>
  static __device__ void epilogue_prologue(const P&, int, int) {}
  // Work of a GEMM-partition CTA after its last tile (all threads; the shared memory and the
  // tensor memory are free by then).
  template <bool Trace>
  static __device__ void after_gemm(const P&, int, int, uint8_t*) {}
  static constexpr int kEpiWarps = 4;   // epilogue warps (4, or 8 = one warpgroup per 128-row half)
  static constexpr int kMaxMovers = 4;  // mover warps the launch bounds allow
  // Dependent launch: the kernel is launched with programmatic stream serialization, so its
  // CTAs may start (barrier set-up, TMEM allocation) while the kernel that writes its tables
  // still runs; every role waits for that kernel (grid_dep_wait) before its first read.
  static constexpr bool kDependentLaunch = false;
};

// Threads per CTA the launch bounds of an op's kernel allow.
template <class Op>
constexpr int op_max_threads() {
  return (2 + Op::kEpiWarps + Op::kMaxMovers) * 32;
}

struct Smem {
  uint8_t* stages;
  int stage_bytes;
  int a_bytes;
  uint8_t* epi;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tfull;
  uint64_t* tempty;
  uint64_t* drain;
  uint32_t* tmem_slot;
  uint32_t* epi_cnt;  // [2] publish-round counters, one per TMEM accumulator
  __device__ uint8_t* a(int s) const { return stages + s * stage_bytes; }
  __device__ uint8_t* b(int s) const { return stages + s * stage_bytes + a_bytes; }
};

// Write one 32-row x 128-byte chunk (lane = row) into a staging buffer laid out in the
// TMA 128-byte swizzle: 16-byte piece j of row r lives at piece (j ^ (r & 7)).
__device__ __forceinline__ void stage_row128(uint8_t* buf, int lane, const uint32_t (&w)[32]) {
  const uint32_t base = smem_u32(buf) + lane * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t piece = static_cast<uint32_t>(j ^ (lane & 7));
    st_shared_v4(base + piece * 16, w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  }
}

// Epilogue staging state of one warp: one or two 4 KB chunk buffers (32 rows x 128 B).
// With two, filling one overlaps the TMA engine reading the other; with 8 epilogue warps
// the 32 KB staging area leaves one buffer per warp.
struct EpiStage {
  uint8_t* buf[2];
  int idx;
  int nbuf;
  // Get a free buffer: the bulk group that last read it has finished reading smem.
  __device__ __forceinline__ uint8_t* acquire(int lane) {
    if (lane == 0) {
      if (nbuf == 2)
        bulk_wait_read<1>();
      else
        bulk_wait_read<0>();
    }
    __syncwarp();
    return buf[idx];
  }
  __device__ __forceinline__ void flip() {
    if (nbuf == 2) idx ^= 1;
  }
};

template <class Op, bool Trace>
__device__ __forceinline__ void role_producer(const typename Op::Params& p, const Smem& sm, int lane, int gi,
                                              int gn) {
  const Common& c = p.common;
  const int ntiles = Op::num_tiles(p);
  constexpr int kStages = Geo<Op::kBM>::kStages;
  uint32_t stage = 0, phase = 0;
  uint32_t filled = 0, fill_parity = 0;  // per-stage: fill issued / parity of that fill
  bool ok = true;
  constexpr bool tr = Trace;
  Op::producer_init(p);
  for (int t = gi; t < ntiles && ok; t += gn) {
    const Job j = Op::job(p, t);
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
        ok = mbar_wait(&sm.empty[stage], phase ^ 1u, c, kSiteEmpty);
        if (tr) stall += globaltimer() - e0;
        if (ok) {
          mbar_arrive_expect_tx(&sm.full[stage], Op::kTxBytes);
          Op::load(p, j, kb, sm.a(stage), sm.b(stage), &sm.full[stage]);
          filled |= 1u << stage;
          fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      if (++stage == kStages) { stage = 0; phase ^= 1u; }
    }
    if (tr && lane == 0) {
      trace_span(c, kTrProdTile, t, tt0, globaltimer());
      trace_span(c, kTrProdStall, t, tt0, tt0 + stall);
    }
  }
  // Drain: every TMA fill this warp issued must have landed before the CTA exits.
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s)
      if (filled & (1u << s)) mbar_wait(&sm.full[s], (fill_parity >> s) & 1u, c, kSiteDrain);
  }
  __syncwarp();
}

template <class Op, bool Trace>
__device__ __forceinline__ void role_mma(const typename Op::Params& p, const Smem& sm, int lane,
                                         uint32_t tmem_base, int gi, int gn) {
  using G = Geo<Op::kBM>;
  constexpr int kStages = G::kStages;
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
      const uint32_t d = tmem_base + acc * G::kAccStride;
      for (int kb = 0; kb < j.kblocks && ok; ++kb) {
        const uint64_t f0 = tr ? globaltimer() : 0;
        ok = mbar_wait(&sm.full[stage], phase, c, kSiteFull);
        if (tr) starve += globaltimer() - f0;
        if (!ok) break;
        tc_fence_after();
        const uint32_t a0 = smem_u32(sm.a(stage));
        const uint32_t b0 = smem_u32(sm.b(stage));
        Op::mma_stage(j, d, a0, b0, kb);
        umma_commit(&sm.empty[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      if (ok) umma_commit(&sm.tfull[acc]);
      if (tr) {
        trace_span(c, kTrMmaTile, t, tt0, globaltimer());
        trace_span(c, kTrMmaStarve, t, tt0, tt0 + starve);
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (++acc == G::kAccBufs) {
      acc = 0;
      acc_phase ^= 1u;
    }
  }
  // Drain: all MMAs this thread issued complete before TMEM is freed.
  if (lane == 0) {
    umma_commit(sm.drain);
    mbar_wait(sm.drain, 0, c, kSiteDrain);
  }
  __syncwarp();
}

template <class Op, bool Trace>
__device__ __forceinline__ void role_epilogue(const typename Op::Params& p, const Smem& sm, int warp,
                                              int lane, uint32_t tmem_base, int gi, int gn) {
  using G = Geo<Op::kBM>;
  const Common& c = p.common;
  const int ntiles = Op::num_tiles(p);
  constexpr int E = Op::kEpiWarps;
  const int q = warp & 3;   // TMEM lane quadrant this warp may access
  const int ew = warp - 2;  // epilogue warp index 0..E-1
  EpiStage es;
  es.nbuf = 8 / E;
  es.buf[0] = sm.epi + (ew * es.nbuf) * kEpiBufBytes;
  es.buf[1] = sm.epi + (ew * es.nbuf + es.nbuf - 1) * kEpiBufBytes;
  es.idx = 0;
  Op::template epilogue_prologue<Trace>(p, ew, lane);
  // With 8 warps, warps ew and ew+4 share a lane quadrant and take one 128-row half each.
  const int h0 = E == 8 ? ew / 4 : 0;
  const int h1 = E == 8 ? h0 + 1 : Op::kBM / 128;
  uint32_t acc = 0, acc_phase = 0;
  bool ok = true;
  constexpr bool tr = Trace;
  for (int t = gi; t < ntiles && ok; t += gn) {
    const Job j = Op::job(p, t);
    const uint64_t w0 = tr ? globaltimer() : 0;
    ok = mbar_wait(&sm.tfull[acc], acc_phase, c, kSiteTmemFull);
    if (!ok) break;
    tc_fence_after();
    if (tr && lane == 0) {
      const uint64_t tt0 = globaltimer();
      if (tt0 - w0 > kTraceMinWaitNs) trace_span(c, kTrEpiWait, t, w0, tt0);
      trace_open(c, kTrEpiTile, t, tt0);
    }
    const uint32_t taddr = tmem_base + acc * G::kAccStride + (static_cast<uint32_t>(q * 32) << 16);
    Op::epilogue(p, j, taddr, q, lane, es, h0, h1);
    if (Op::publishes(p, j)) {
      // producer_tile_notify: the last of the four warps to see its own stores of this
      // tile complete publishes the tile's signal (release).  Each warp arrives here
      // before it frees the accumulator, so arrivals of consecutive rounds on one TMEM
      // buffer never interleave and a plain modulo-4 counter identifies the last one.
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
    if (lane == 0) mbar_arrive(&sm.tempty[acc]);
    if (tr && lane == 0) trace_close(c, globaltimer());
    if (++acc == G::kAccBufs) {
      acc = 0;
      acc_phase ^= 1u;
    }
  }
  if (lane == 0) bulk_wait<0>();
  __syncwarp();
}

// Trace: the instantiation that records spans (launched while the context has a trace
// buffer); the other one carries no trace code at all.
template <class Op, bool Trace>
__global__ void __launch_bounds__(op_max_threads<Op>(), 1)
    persistent_kernel(const __grid_constant__ typename Op::Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using G = Geo<Op::kBM>;
  Smem sm;
  sm.stages = base;
  sm.stage_bytes = G::kStageBytes;
  sm.a_bytes = G::kABytes;
  sm.epi = base + kRingBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm.epi + kEpiBytes);
  sm.full = bars;
  sm.empty = bars + kMaxStages;
  sm.tfull = bars + 2 * kMaxStages;
  sm.tempty = bars + 2 * kMaxStages + 2;
  sm.drain = bars + 2 * kMaxStages + 4;
  sm.tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kMaxStages + 5);
  sm.epi_cnt = sm.tmem_slot + 2;
  static_assert((2 * kMaxStages + 5) * 8 + 16 <= kBarBytes - 4 * kTraceWarps, "barrier area");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if constexpr (Trace) {
    trace_begin();
    __syncthreads();
  }
  // CTAs outside the GEMM partition (e.g. a combine partition) run the op's side role.
  int gi = blockIdx.x, gn = gridDim.x;
  if (!Op::gemm_partition(p, gi, gn)) {
    if constexpr (Op::kDependentLaunch) grid_dep_wait();
    Op::template side_role<Trace>(p, warp, lane, smem_raw);
    if constexpr (Trace) {
      __syncthreads();
      trace_end(p.common);
    }
    return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < G::kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.tfull[b], 1);
      mbar_init(&sm.tempty[b], Op::kEpiWarps);
    }
    mbar_init(sm.drain, 1);
    sm.epi_cnt[0] = 0;
    sm.epi_cnt[1] = 0;
    fence_mbar_init();
    Op::prefetch(p);
  }
  if (warp == 1) {
    tmem_alloc(sm.tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;
  if constexpr (Op::kDependentLaunch) grid_dep_wait();

  if (warp == 0) {
    role_producer<Op, Trace>(p, sm, lane, gi, gn);
  } else if (warp == 1) {
    role_mma<Op, Trace>(p, sm, lane, tmem_base, gi, gn);
  } else if (warp < 2 + Op::kEpiWarps) {
    role_epilogue<Op, Trace>(p, sm, warp, lane, tmem_base, gi, gn);
  } else {
    Op::template mover<Trace>(p, warp - 2 - Op::kEpiWarps, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  Op::template after_gemm<Trace>(p, warp, lane, smem_raw);
  if constexpr (Trace) {
    __syncthreads();
    trace_end(p.common);
  }
}

// ------------------------------------------------------------------ shared epilogue pieces

// Load 64 accumulator columns [col, col+64) of this warp's 32 rows.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, int col, float (&v)[64]) {
  float a[32], b[32];
  tmem_ld32(taddr + col, a);
  tmem_ld32(taddr + col + 32, b);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = a[i];
    v[32 + i] = b[i];
  }
}

__device__ __forceinline__ void pack64_bf16(const float (&v)[64], uint32_t (&w)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
}

// Stage 64 bf16 columns of 32 rows and TMA-store them at (x, y) of `map` (box {64, 32}).
__device__ __forceinline__ void store_bf16_chunk(const CUtensorMap* map, EpiStage& es, int lane,
                                                 const float (&v)[64], int x, int y) {
  uint32_t w[32];
  pack64_bf16(v, w);
  uint8_t* buf = es.acquire(lane);
  stage_row128(buf, lane, w);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, buf, x, y);
    bulk_commit();
  }
  es.flip();
}

// Stage 32 fp32 columns of 32 rows and TMA-store (reduce = false) or TMA-add (reduce = true)
// them at (x, y) of `map` (box {32, 32}).
__device__ __forceinline__ void store_f32_chunk(const CUtensorMap* map, EpiStage& es, int lane,
                                                const float (&v)[32], int x, int y, bool reduce) {
  uint32_t w[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i]);
  uint8_t* buf = es.acquire(lane);
  stage_row128(buf, lane, w);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (reduce)
      tma_reduce_add_2d(map, buf, x, y);
    else
      tma_store_2d(map, buf, x, y);
    bulk_commit();
  }
  es.flip();
}

// Operand layouts in shared memory (both written by TMA with the 128-byte swizzle):
//   A (K-major): 128-row groups of 128 B rows; 8-row core groups 1024 B apart (SBO); a K
//     step of 16 elements advances the start address by 32 B inside the swizzle atom.
//   B (MN-major, B is K x N row-major): BN/64 column groups of [64 k-rows x 128 B]
//     (8 KB each) -> LBO = 8192 B between 64-column groups, SBO = 1024 B between
//     8-row K groups; a K step of 16 rows advances the start by 2048 B.
#ifndef TL_B_LBO
#define TL_B_LBO 8192
#endif
#ifndef TL_B_SBO
#define TL_B_SBO 1024
#endif

// The standard single-accumulator MMA stage: 4 x (128x256x16) into d.
__device__ __forceinline__ void mma_stage_256(uint32_t d, uint32_t a0, uint32_t b0, int kb) {
  constexpr uint32_t idesc = umma_idesc_bf16(kBM, kBN, true);
#pragma unroll
  for (int k = 0; k < kBK / 16; ++k) {
    const uint64_t ad = umma_desc_sw128(a0 + k * 32, 16, 1024);
    const uint64_t bd = umma_desc_sw128(b0 + k * 2048, TL_B_LBO, TL_B_SBO);
    umma_bf16(d, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
  }
}

// The 256-row MMA stage: per K step of 16, rows 0-127 of A into d and rows 128-255 into
// d + 256, both against the same B slice (4 x 2 x (128x256x16)).
__device__ __forceinline__ void mma_stage_256x256(uint32_t d, uint32_t a0, uint32_t b0, int kb) {
  constexpr uint32_t idesc = umma_idesc_bf16(kBM, kBN, true);
#pragma unroll
  for (int k = 0; k < kBK / 16; ++k) {
    const uint64_t ad0 = umma_desc_sw128(a0 + k * 32, 16, 1024);
    const uint64_t ad1 = umma_desc_sw128(a0 + 128 * 128 + k * 32, 16, 1024);
    const uint64_t bd = umma_desc_sw128(b0 + k * 2048, TL_B_LBO, TL_B_SBO);
    const uint32_t accum = (kb > 0 || k > 0) ? 1u : 0u;
    umma_bf16(d, ad0, bd, idesc, accum);
    umma_bf16(d + 256, ad1, bd, idesc, accum);
  }
}

// MMA stage for a tile of BM rows.
template <int BM>
__device__ __forceinline__ void mma_stage_bm(uint32_t d, uint32_t a0, uint32_t b0, int kb) {
  if constexpr (BM == 256)
    mma_stage_256x256(d, a0, b0, kb);
  else
    mma_stage_256(d, a0, b0, kb);
}

// Mover copy of `bytes` (multiple of 16) from src to dst by `nthreads` threads.
__device__ __forceinline__ void copy_chunk(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t nvec,
                                           int tid, int nthreads) {
  constexpr int U = 8;
  size_t i = tid;
  for (; i + (U - 1) * nthreads < nvec; i += U * nthreads) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) r[u] = __ldg(src + i + u * nthreads);
#pragma unroll
    for (int u = 0; u < U; ++u) dst[i + u * nthreads] = r[u];
  }
  for (; i < nvec; i += nthreads) dst[i] = __ldg(src + i);
}

}  // namespace tl
