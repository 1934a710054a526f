// Sequence-parallel self-attention with the KV AllGather overlapped ("TileLink: Generating
// Efficient Compute-Communication Overlapping Kernels using Tile-Centric Primitives", §5
// Figure 6 text and §7.2 self-attention: the KV cache sequence S is split into W shards,
// one per rank, gathered while the attention of the rank's queries runs over the shards as
// they arrive; "Triton-distributed ...", §3.7 swizzle: the local shard first).
//
// Persistent clusters of two CTAs (one per SM) walk (head, 256-query tile) work items; CTA r
// of a pair owns queries [128 r, 128 r + 128) of the tile.  When the items do not fill the
// last wave evenly (nwork mod pairs = rem, 0 < 2 rem <= pairs) the last rem items are split
// into two halves of their key blocks, one per pair: a wave of halves replaces a partial wave
// of whole items.  A half writes its unnormalised O, running max and sum to the workspace;
// whichever half of an item finishes second (an epoch-tagged exchange on a counter) combines
// both in a fixed order, (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / (l_0 2^(m_0 - m) + l_1 2^(m_1 - m)),
// so the result does not depend on which finished first (the flash-decoding split of the keys).
// Each item is non-causal flash attention over all W shards in blocks of 256 keys, on tcgen05
// pair MMAs (cta_group::2):
//   S(J) = Q K_J^T     M = 256 queries, N = 256 keys, K = 128 head dims: CTA r's A is its
//                      128 query rows, its B half the keys [128 r, 128 r + 128) of the block
//                      (K-major); TMEM columns [0, 256) of each CTA receive its rows' scores;
//   O += P(J) V_J      M = 256, N = 128 head dims, K = 256 keys, A from TMEM: the softmax
//                      writes P (bf16, two per 32-bit column) to columns [256, 384); CTA r's
//                      B half is head dims [64 r, 64 r + 64) of V (MN-major); O is columns
//                      [384, 512).
// S and P have separate columns, so S(J + 1) is computed while the softmax of block J runs,
// and P(J) V_J while the softmax of block J + 1 runs: the MMA thread issues S(J + 1) as soon
// as every softmax warp has read S(J), then P(J) V_J once P(J) is written.
// Warps of each CTA:
//   warp 0     TMA producer: its Q rows (two buffers, so the next item's Q is loaded early),
//              per key block its K half (2 boxes) and V half (4 boxes of 64 keys x its 64
//              head dims) through 2-stage rings; every load completes on the pair leader's
//              barrier; the first block of a remote shard slice waits on the slice's block
//              signals (one warp-wide poll).
//   warp 1     TMEM allocation (both CTAs) and, in the leader, the pair MMAs (one thread).
//   warps 2-9  softmax, two warpgroups: warpgroup g takes keys [128 g, 128 g + 128) of every
//              block, one row per thread, in base 2 (the 1/sqrt(d) scale folded into one
//              multiply-add per score).  A thread reads its 128 scores from TMEM once and
//              announces "S read" at once; it keeps 64 of them in fp32 and 64 as f16 offsets
//              from its block max (the register budget).  The two warps of a TMEM lane quadrant (one per group,
//              the same 32 rows) exchange their block maxima through shared memory, so both
//              use one running max m per row and one O; each keeps the sum l_g of its own
//              keys.  m moves only when the block's max exceeds it by more than 2^8
//              (kRescaleLog2): until then P <= 256 and O, l_g keep the stale max, which cancels
//              in the final division; a move rescales O in TMEM (group g its head dims
//              [64 g, 64 g + 64)) once P(J - 1) V_{J-1} has completed.  At the end of an
//              item the partners exchange l_g and group g writes head dims [64 g, 64 g + 64)
//              of O / (l_0 + l_1) as bf16.
//   warps 10-11 movers: remote K/V blocks (up to 32 KB each) into the shard-major gathered
//              buffers, one release signal per 128-key block, in the order the items need
//              them (groups of heads one wave covers, shard by shard, the local shard last).
// The softmax warps of both CTAs arrive on the leader's barriers for "S read", "P written"
// and "O read by the epilogue" (relaxed cluster-scope arrivals: a release at cluster scope
// costs a full memory barrier per arrival); the leader's MMA commits arrive on both CTAs'
// barriers (one multicast commit).  The pipeline counters run on across items.  Every wait
// is bounded.
// Shard lengths need not be multiples of 256 (the Ragged instantiation): a shard's last key
// block and the last query tile may be partial.  TMA zero-fills the absent rows, the softmax
// gives the absent keys no weight, and the absent query rows are not stored.
#include "tl_host.h"

namespace tl {

namespace attn {
constexpr int kD = 128;          // head dim
constexpr int kBQ = 128;         // queries per CTA (a pair's tile is 256)
constexpr int kBKV = 256;        // keys per block
constexpr int kSigBlk = 128;     // keys per mover block (one signal each)
constexpr int kBox = 16384;      // one 64-column SW128 box of 128 rows
constexpr int kBox64 = 8192;     // one 64-column SW128 box of 64 rows
constexpr int kQBytes = 2 * kBox;      // this CTA's 128 queries x 128 dims
constexpr int kKBytes = 2 * kBox;      // this CTA's 128 keys of a block x 128 dims
constexpr int kVBytes = 4 * kBox64;    // 256 keys x this CTA's 64 dims: 4 boxes of 64 keys
constexpr int kQStages = 2;
constexpr int kStages = 2;
constexpr int kRedBytes = 2 * 2 * kBQ * 4;  // [exchange parity][group][row] floats
constexpr int kBarBytes = 256;
constexpr int kSmem = 1024 + kQStages * kQBytes + kStages * (kKBytes + kVBytes) + kRedBytes + kBarBytes;
constexpr uint32_t kColP = 256;  // TMEM columns of P (bf16 pairs; group g at + 64 g)
constexpr int kMaxTail = 40;     // split items the workspace holds partial results for
constexpr size_t kPartO = static_cast<size_t>(kBQ) * kD * 4;  // one CTA's fp32 O of a half
constexpr size_t kPartML = static_cast<size_t>(kBQ) * 2 * 4;  // one CTA's (m, l) of a half
constexpr uint32_t kColO = 384;  // TMEM columns of O
// Of a thread's 128 scores, those kept in fp32 (the rest as f16 offsets).  64 measured best
// (attn_16k 389 us); keeping more in fp32 raises register pressure past the 168-register cap:
// 96 gave 397 us, 80 gave 442 us and 112 gave 841 us.
constexpr int kKeepF32 = 64;
static_assert(kKeepF32 % 2 == 0 && kKeepF32 <= 128, "fp32 / f16 split");
constexpr float kRescaleLog2 = 8.0f;  // move the running max once it grows by more than this
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSoftWarps = 8;
constexpr int kMovers = 2;
constexpr int kThreads = (2 + kSoftWarps + kMovers) * 32;
static_assert(kSmem <= 232448, "shared memory");
}  // namespace attn

struct AttnParams {
  CUtensorMap q;      // {d, Lq, H}, box {64, 128, 1}
  CUtensorMap k_loc;  // local K shard {d, Lr, H}, box {64, 128, 1}
  CUtensorMap k_gat;  // gathered K, shard-major [W][H][Lr][d] as {d, Lr, W H}, box {64, 128, 1}
  CUtensorMap v_loc;  // local V shard {d, Lr, H}, box {64, 64, 1}
  CUtensorMap v_gat;  // gathered V, shard-major, box {64, 64, 1}
  Common common;
  const uint8_t* kshard[8];
  const uint8_t* vshard[8];
  uint8_t* kg;
  uint8_t* vg;
  __nv_bfloat16* out;  // [H, Lq, d]
  uint64_t* flags;     // [W][H][ceil(Lr / 128)]: K and V block gathered
  float* part_o;       // [tail item][half][CTA of the pair][128 rows][128 dims] fp32
  float* part_ml;      // [tail item][half][CTA of the pair][128 rows][m, l] fp32
  unsigned long long* tail_ctr;  // [tail item][CTA of the pair]: epoch of the first half done
  int W, rank, Lq, Lr, heads;
  int nfull, ntail;    // whole items [0, nfull); items [nfull, nfull + ntail) split in halves
  float scale;  // 1 / sqrt(d)
};

// A 3-D TMA box into this CTA's shared memory, completing on the pair leader's mbarrier
// (given by its shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int x, int y,
                                                 int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// D[tmem of both CTAs] (+)= A[tmem of both CTAs, M split] * B[smem of both CTAs, N split].
__device__ __forceinline__ void umma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// S = Q K^T on the pair: M = 256, N = 256, K = 128 (8 steps of 16 head dims).  Each step's
// descriptors are the first step's plus a constant: the start-address field (address >> 4,
// bits 0-13) cannot carry out, shared-memory addresses being below 2^18 bytes.
__device__ __forceinline__ void attn_mma_s(uint32_t d, uint32_t q0, uint32_t k0) {
  constexpr uint32_t idesc = umma_idesc_bf16(256, 256, false);
  const uint64_t a0 = umma_desc_sw128(q0, 16, 1024), b0 = umma_desc_sw128(k0, 16, 1024);
#pragma unroll
  for (int kb = 0; kb < 2; ++kb)
#pragma unroll
    for (int k = 0; k < 4; ++k)
      umma_bf16_pair(d, a0 + ((kb * attn::kBox + k * 32) >> 4), b0 + ((kb * attn::kBox + k * 32) >> 4), idesc,
                     (kb | k) ? 1u : 0u);
}

// O (+)= P V on the pair: M = 256, N = 128, K = 256 keys (16 steps).  P is in TMEM at columns
// [p, p + 128) (16 keys per 8 columns); this CTA's V half is 64 head dims wide, its 64-key
// boxes 8 KB apart.
__device__ __forceinline__ void attn_mma_pv(uint32_t d, uint32_t p, uint32_t v0, bool acc) {
  constexpr uint32_t idesc = umma_idesc_bf16(256, 128, true);
  const uint64_t b0 = umma_desc_sw128(v0, 8192, 1024);
#pragma unroll
  for (int kb = 0; kb < 4; ++kb)
#pragma unroll
    for (int k = 0; k < 4; ++k)
      umma_ts_pair(d, p + (kb * 4 + k) * 8, b0 + ((kb * attn::kBox64 + k * 2048) >> 4), idesc,
                   (acc || kb || k) ? 1u : 0u);
}

// Store 32 consecutive 32-bit columns of this warp's 32 TMEM lanes (no wait).
__device__ __forceinline__ void tmem_st32_raw(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// Paired fp32 arithmetic (two lanes of one 64-bit register pair per instruction) and the
// three-input maximum: the softmax issues about a third fewer instructions per score.
__device__ __forceinline__ unsigned long long f2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long fadd2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two fp32 values as an f16x2 pair (round to nearest; lo in the low half) and back.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ void unpack_f16x2(uint32_t v, float& lo, float& hi) {
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi) : "r"(v));
}

// Relaxed arrival on an mbarrier given by its shared::cluster address: no memory ordering is
// implied (a release at cluster scope costs a full memory barrier on every call).  Used where
// what the arrival announces is already complete in this thread: its TMEM reads
// (tcgen05.wait::ld) or writes (tcgen05.wait::st), then tcgen05.fence::before_thread_sync.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Arrive once on the mbarrier at `bar`'s offset in both CTAs of the pair when every pair MMA
// issued so far has completed (one multicast commit).
__device__ __forceinline__ void commit_both(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               ::"r"(smem_u32(bar)), "h"(static_cast<uint16_t>(3))
               : "memory");
}

// A pair's work units, in order: the whole items pair, pair + P, ... below nfull, then (for
// pair < 2 ntail) half pair mod 2 of the split item nfull + pair / 2.  half = -1 for a whole
// item; key blocks [jb, je) of the item's block order.
struct AttnUnit {
  int it, jb, je, half;
};
__device__ __forceinline__ int attn_whole_units(int pair, int npairs, int nfull) {
  return pair < nfull ? (nfull - pair + npairs - 1) / npairs : 0;
}
__device__ __forceinline__ AttnUnit attn_unit(int k, int pair, int npairs, int nfull, int nblk) {
  AttnUnit u;
  if (k < attn_whole_units(pair, npairs, nfull)) {
    u.it = pair + k * npairs;
    u.jb = 0;
    u.je = nblk;
    u.half = -1;
  } else {
    u.it = nfull + pair / 2;
    u.half = pair & 1;
    u.jb = u.half ? nblk / 2 : 0;
    u.je = u.half ? nblk : nblk / 2;
  }
  return u;
}

// Ragged: some shard length l_r is not a multiple of 256 (a partial last key block of every
// shard and a partial last query tile); the common case is compiled without those checks.
template <bool Ragged>
__global__ void __launch_bounds__(attn::kThreads, 1) attn_kernel(const __grid_constant__ AttnParams p) {
  using namespace attn;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = base;                        // [kQStages]
  uint8_t* sk = sq + kQStages * kQBytes;     // [kStages]
  uint8_t* sv = sk + kStages * kKBytes;      // [kStages]
  float* red = reinterpret_cast<float*>(sv + kStages * kVBytes);  // [parity][group][row]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sv + kStages * kVBytes + kRedBytes);
  // counted on the leader (the peer's copies are unused): loads of both CTAs, arrivals of
  // both CTAs' softmax warps
  uint64_t* qfull = bars;        // [2]
  uint64_t* kfull = bars + 2;    // [2]
  uint64_t* vfull = bars + 4;    // [2]
  uint64_t* sfree = bars + 6;    // all 16 softmax warps of the pair have read S(J)
  uint64_t* pready = bars + 7;   // all 16 wrote P(J) (and rescaled O)
  uint64_t* ofree = bars + 8;    // all 16 have read O at the end of an item
  // in both CTAs, arrived on by the leader's MMA commits
  uint64_t* qempty = bars + 9;   // [2] the item's last S MMA has read Q
  uint64_t* kempty = bars + 11;  // [2]
  uint64_t* vempty = bars + 13;  // [2]
  uint64_t* sfull = bars + 15;   // S(J) is in TMEM
  uint64_t* pfree = bars + 16;   // P(J) V_J complete (P free, O stable)
  uint64_t* drain = bars + 17;
  // this CTA's partner warps (the two softmax warps of one TMEM lane quadrant), per exchange
  uint64_t* xq = bars + 18;      // [4]
  // this CTA's softmax warps, once per split item: all 8 wrote their partial results; the
  // counter exchange is done and its outcome is in tail_second
  uint64_t* tail_w = bars + 22;
  uint64_t* tail_r = bars + 23;
  volatile uint32_t* tail_second = reinterpret_cast<volatile uint32_t*>(bars + 24);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 25);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const bool leader = crank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const Common& c = p.common;
  const int bps = (p.Lr + kBKV - 1) / kBKV;       // 256-key blocks per shard (the last may be partial)
  const int sbs = (p.Lr + kSigBlk - 1) / kSigBlk;  // 128-key signal blocks per shard
  const int nblk = p.W * bps;                      // key blocks per item
  const int nqt = (p.Lq + 2 * kBQ - 1) / (2 * kBQ);  // 256-query tiles (the last may be partial)
  const int nunits = attn_whole_units(pair, npairs, p.nfull) + (pair < 2 * p.ntail ? 1 : 0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&qfull[s], 1);
      mbar_init(&qempty[s], 1);
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
    }
    mbar_init(sfree, 2 * kSoftWarps);
    mbar_init(pready, 2 * kSoftWarps);
    mbar_init(ofree, 2 * kSoftWarps);
    mbar_init(sfull, 1);
    mbar_init(pfree, 1);
    mbar_init(drain, 1);
    for (int q = 0; q < 4; ++q) mbar_init(&xq[q], 2);
    mbar_init(tail_w, kSoftWarps);
    mbar_init(tail_r, 1);
    fence_mbar_init();
    tma_prefetch_map(&p.q);
    tma_prefetch_map(&p.k_loc);
    tma_prefetch_map(&p.v_loc);
    tma_prefetch_map(&p.k_gat);
    tma_prefetch_map(&p.v_gat);
  }
  if (warp == 1) {
    tmem_alloc_pair(tslot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers and TMEM are ready before any remote arrival or MMA
  tc_fence_after();
  const uint32_t tmem = *tslot;
  auto lead = [](uint64_t* bar) { return mapa_shared(smem_u32(bar), 0); };

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    bool ok = true;
    uint32_t filled = 0, par = 0;  // leader's drain: K stages bits 0-1, V 2-3, Q 4-5
    int J = 0;
    for (int kq = 0; kq < nunits && ok; ++kq) {
      const AttnUnit u = attn_unit(kq, pair, npairs, p.nfull, nblk);
      const int h = u.it / nqt, qt = u.it - h * nqt;
      const int qs = kq & 1;
      const uint32_t qph = (kq >> 1) & 1;
      if (lane == 0) {
        ok = mbar_wait(&qempty[qs], qph ^ 1u, c, kSiteEmpty);
        if (ok) {
          if (leader) mbar_arrive_expect_tx(&qfull[qs], 2 * kQBytes);
          const int y = qt * 2 * kBQ + static_cast<int>(crank) * kBQ;
          tma_load_3d_pair(sq + qs * kQBytes, &p.q, lead(&qfull[qs]), 0, y, h);
          tma_load_3d_pair(sq + qs * kQBytes + kBox, &p.q, lead(&qfull[qs]), 64, y, h);
          filled |= 16u << qs;
          par = (par & ~(16u << qs)) | (qph << (qs + 4));
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      for (int j = u.jb; j < u.je && ok; ++j, ++J) {
        const int step = j / bps, blk = j - step * bps;
        const int r = (p.rank + step) % p.W;
        const bool local = step == 0;
        if (!local && (blk == 0 || j == u.jb)) {
          // consumer_tile_wait on the shard's slice of this head: all its blocks gathered
          ok = warp_wait_signals(p.flags + (static_cast<size_t>(r) * p.heads + h) * sbs, sbs, c.epoch, c, lane,
                                 kSiteSignal, (7ull << 60) | (static_cast<unsigned long long>(r) << 32) | h);
          if (!ok) break;
        }
        const int s = J & 1;
        const uint32_t ph = (J >> 1) & 1;
        const int y = blk * kBKV;
        const int z = local ? h : r * p.heads + h;  // the gathered buffers hold shard r at z = r H + h
        const CUtensorMap* km = local ? &p.k_loc : &p.k_gat;
        const CUtensorMap* vm = local ? &p.v_loc : &p.v_gat;
        if (lane == 0) {
          ok = mbar_wait(&kempty[s], ph ^ 1u, c, kSiteEmpty);
          if (ok) {
            if (leader) mbar_arrive_expect_tx(&kfull[s], 2 * kKBytes);
            const int yk = y + static_cast<int>(crank) * kBQ;  // this CTA's 128 keys of the block
            tma_load_3d_pair(sk + s * kKBytes, km, lead(&kfull[s]), 0, yk, z);
            tma_load_3d_pair(sk + s * kKBytes + kBox, km, lead(&kfull[s]), 64, yk, z);
            filled |= 1u << s;
            par = (par & ~(1u << s)) | (ph << s);
          }
          if (ok) ok = mbar_wait(&vempty[s], ph ^ 1u, c, kSiteEmpty);
          if (ok) {
            if (leader) mbar_arrive_expect_tx(&vfull[s], 2 * kVBytes);
            const int xv = static_cast<int>(crank) * 64;  // this CTA's 64 head dims
#pragma unroll
            for (int kb = 0; kb < 4; ++kb)
              tma_load_3d_pair(sv + s * kVBytes + kb * kBox64, vm, lead(&vfull[s]), xv, y + kb * 64, z);
            filled |= 4u << s;
            par = (par & ~(4u << s)) | (ph << (s + 2));
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      }
    }
    if (lane == 0 && leader) {  // drain: every fill of both CTAs has landed before the pair exits
      for (int s = 0; s < 2; ++s) {
        if (filled & (16u << s)) mbar_wait(&qfull[s], (par >> (s + 4)) & 1u, c, kSiteDrain);
        if (filled & (1u << s)) mbar_wait(&kfull[s], (par >> s) & 1u, c, kSiteDrain);
        if (filled & (4u << s)) mbar_wait(&vfull[s], (par >> (s + 2)) & 1u, c, kSiteDrain);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    // Per block J: S(J + 1) (the next item's first block when J ends an item) once the
    // softmax has read S(J), then P(J) V_J once P(J) is written.
    if (leader && lane == 0) {
      const int nwhole = attn_whole_units(pair, npairs, p.nfull);
      // key blocks of unit k
      auto nb_of = [&](int k) { return k < nwhole ? nblk : ((pair & 1) ? nblk - nblk / 2 : nblk / 2); };
      int total = nwhole * nblk + (nunits > nwhole ? nb_of(nwhole) : 0);
      const uint32_t sk0 = smem_u32(sk), sv0 = smem_u32(sv), sq0 = smem_u32(sq);
      // S of block Jn (position jn in item kqn), and its commits
      auto issue_s = [&](int Jn, int jn, int kqn) -> bool {
        const int s = Jn & 1;
        if (jn == 0 && !mbar_wait(&qfull[kqn & 1], (kqn >> 1) & 1, c, kSiteFull)) return false;
        if (!mbar_wait(&kfull[s], (Jn >> 1) & 1, c, kSiteFull)) return false;
        tc_fence_after();
        attn_mma_s(tmem, sq0 + (kqn & 1) * kQBytes, sk0 + s * kKBytes);
        commit_both(sfull);
        commit_both(&kempty[s]);
        if (jn == nb_of(kqn) - 1) commit_both(&qempty[kqn & 1]);
        return true;
      };
      bool ok = true;
      if (total > 0) ok = issue_s(0, 0, 0);
      int j = 0, kq = 0;
      for (int J = 0; J < total && ok; ++J) {
        const int s = J & 1;
        const int jn = j + 1 == nb_of(kq) ? 0 : j + 1, kqn = jn == 0 ? kq + 1 : kq;
        if (J + 1 < total) {  // S(J + 1) overwrites S(J): every softmax warp has read it
          ok = mbar_wait(sfree, J & 1, c, kSiteTmemEmpty) && issue_s(J + 1, jn, kqn);
          if (!ok) break;
        }
        ok = mbar_wait(&vfull[s], (J >> 1) & 1, c, kSiteFull);
        // the previous item's epilogue has read O before this item's first P V overwrites it
        if (ok && j == 0 && kq > 0) ok = mbar_wait(ofree, (kq - 1) & 1, c, kSiteTmemEmpty);
        if (ok) ok = mbar_wait(pready, J & 1, c, kSiteFull);
        if (!ok) break;
        tc_fence_after();
        attn_mma_pv(tmem + kColO, tmem + kColP, sv0 + s * kVBytes, j > 0);
        commit_both(pfree);
        commit_both(&vempty[s]);
        j = jn;
        kq = kqn;
      }
      umma_commit_pair(drain);
      mbar_wait(drain, 0, c, kSiteDrain);
    }
    __syncwarp();
  } else if (warp < 2 + kSoftWarps) {
    // ------------------------------------------------------------ softmax (one row per thread)
    const int g = (warp - 2) >> 2;          // warpgroup: keys [128 g, 128 g + 128) of a block
    const int qd = warp & 3;                // TMEM lane quadrant of this warp (and its partner's)
    const int row = qd * 32 + lane;         // query row inside the CTA's 128
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    const uint32_t tog = tmem + kColO + g * 64;  // this group's half of O (head dims [64 g, 64 g + 64))
    const float sl2 = p.scale * kLog2e;     // raw score -> base-2 exponent
    bool ok = true;
    int J0 = 0;
    uint32_t nx = 0;  // exchanges with the partner warp so far
    // Exchange one float per row with the partner warp (same rows, other key group) through
    // red, double-buffered by exchange parity: exchange n + 2 rewrites a buffer only after the
    // partner has arrived for exchange n + 1, i.e. after it read exchange n.  Bounded waits.
    auto post = [&](float mine) {
      red[(nx & 1) * 2 * kBQ + g * kBQ + row] = mine;
      __syncwarp();
      if (lane == 0) mbar_arrive(&xq[qd]);
    };
    auto collect = [&](float& other) -> bool {
      if (!mbar_wait(&xq[qd], nx & 1, c, kSiteTmemFull)) return false;
      other = red[(nx & 1) * 2 * kBQ + (1 - g) * kBQ + row];
      ++nx;
      return true;
    };
    auto exchange = [&](float mine, float& other) -> bool {
      post(mine);
      return collect(other);
    };
    bool pfree_seen = true;  // P(J - 1) V_{J-1} known complete
    int ntail_done = 0;  // split items this CTA took part in
    for (int kq = 0; kq < nunits && ok; ++kq) {
      int nb, blk;  // the unit's key blocks; the block index inside the current shard
      {
        const AttnUnit u = attn_unit(kq, pair, npairs, p.nfull, nblk);
        nb = u.je - u.jb;
        blk = u.jb % bps - 1;
      }
      float m2 = -INFINITY, l = 0.f;  // running max (base-2 units, common to both groups), this group's sum
      for (int j = 0; j < nb && ok; ++j) {
        const int J = J0 + j;
        if (++blk == bps) blk = 0;
        // The wait results are warp-uniform, as the warp-collective TMEM accesses below need:
        // the converged warp runs each try_wait and timer read as one instruction.
        ok = mbar_wait(sfull, J & 1, c, kSiteTmemFull);
        if (!ok) break;
        tc_fence_after();
        // Keys past the end of a shard (its partial last block, zero-filled by TMA) get no
        // weight: their scores become -inf.
        const int valid = Ragged ? p.Lr - blk * kBKV - g * 128 : 128;
        // One read of this group's 128 scores.  The block max needs them all; then the first
        // 64 stay in fp32 and the second 64 are kept as f16 pairs of y' = s sl2 - lm (lm this
        // group's block max, base 2): y' <= 0, and for the weights that matter (y' within
        // about 2^4 of 0) f16's 11-bit significand is finer than P's bf16 rounding.  S(J) is
        // then read, and S(J + 1) can be computed while the exponentials run.
        float x0[kKeepF32];
        uint32_t h1[(128 - kKeepF32) / 2];
        float lm;  // this group's block max (base 2)
        float r1;  // the reference the f16 offsets are taken from
        {
          uint32_t rr[4][32];
#pragma unroll
          for (int cb = 0; cb < 4; ++cb) tmem_ld32_issue(tmem + g * 128 + cb * 32 + lane_off, rr[cb]);
          tmem_ld_wait(rr[0]);
          tmem_ld_after(rr[1]);
          tmem_ld_after(rr[2]);
          tmem_ld_after(rr[3]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_relaxed(lead(sfree));
          float x[128];
#pragma unroll
          for (int i = 0; i < 128; ++i) x[i] = __uint_as_float(rr[i >> 5][i & 31]);
          if constexpr (Ragged) {
            if (valid < 128) {
#pragma unroll
              for (int i = 0; i < 128; ++i) x[i] = i < valid ? x[i] : -INFINITY;
            }
          }
          // x[8, 120) sixteen at a time onto x[0, 8), then x[120, 128)
          float mx[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mx[k] = x[k];
#pragma unroll
          for (int i = 8; i < 120; i += 16)
#pragma unroll
            for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], x[i + k], x[i + 8 + k]);
#pragma unroll
          for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], x[120 + k]);
          lm = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) *
               sl2;  // the scale is positive: max commutes with it
          // The offsets are taken from the running max before this block, unless this group's
          // block max exceeds it by more than 2^8 (an item's first block included), then from
          // the block max: y' <= 2^8 either way, and unless the max moves they are the
          // exponents themselves.  (Ragged: an item's first block with no valid key in this
          // group has r1 = -inf and y' = -inf.)
          r1 = lm > m2 + kRescaleLog2 ? lm : m2;
          const float nlm = (Ragged && r1 == -INFINITY) ? 0.f : -r1;
#pragma unroll
          for (int i = 0; i < kKeepF32; ++i) x0[i] = x[i];
          const unsigned long long sl2x2 = f2(sl2, sl2), nlm2 = f2(nlm, nlm);
#pragma unroll
          for (int i = 0; i < (128 - kKeepF32) / 2; ++i) {
            float y0, y1;
            f2_split(ffma2(f2(x[kKeepF32 + 2 * i], x[kKeepF32 + 1 + 2 * i]), sl2x2, nlm2), y0, y1);
            h1[i] = pack_f16x2(y0, y1);
          }
        }
        post(lm);
        float bm2;
        {
          float other;
          ok = collect(other);
          if (!ok) break;
          bm2 = fmaxf(lm, other);  // the block's max over all 256 keys: the same in both partners
        }
        pfree_seen = J == 0;
        if (j == 0) {
          m2 = bm2;  // the item's first P V overwrites O
        } else if (__any_sync(0xffffffffu, bm2 > m2 + kRescaleLog2)) {
          // both partners take this branch (same rows, same values); O is stable once
          // P(J - 1) V_{J-1} has completed, and P(J) V_J waits for this thread's P
          const float mn = fmaxf(m2, bm2);
          const float corr = ex2_approx(m2 - mn);  // 0 while the row has seen only absent keys
          ok = mbar_wait(pfree, (J - 1) & 1, c, kSiteTmemFull);
          if (!ok) break;
          pfree_seen = true;
          tc_fence_after();
#pragma unroll 1
          for (int cb = 0; cb < 2; ++cb) {
            float o[32];
            tmem_ld32(tog + cb * 32 + lane_off, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= corr;
            tmem_st32(tog + cb * 32 + lane_off, o);
          }
          l *= corr;
          m2 = mn;
        }
        // P and its sum: the first 64 from the scores, the second 64 from y' + (lm - m2) (<= 2^8:
        // lm <= the block max <= m2 + 2^8).
        // (Ragged: a row whose keys so far are all absent has m2 = -inf; its P is 0.)
        const float nm = (Ragged && m2 == -INFINITY) ? 0.f : -m2;
        const float d1 = (Ragged && (r1 == -INFINITY || m2 == -INFINITY)) ? 0.f : r1 - m2;
        unsigned long long sum2[4];  // 8 partial sums, two per register pair
        uint32_t pk[64];
#pragma unroll
        for (int i = 0; i < 4; ++i) sum2[i] = 0ull;
        {
          const unsigned long long sl2x2 = f2(sl2, sl2), nm2 = f2(nm, nm);
#pragma unroll
          for (int i = 0; i < kKeepF32 / 2; ++i) {
            float y0, y1;
            f2_split(ffma2(f2(x0[2 * i], x0[2 * i + 1]), sl2x2, nm2), y0, y1);
            const float e0 = ex2_approx(y0), e1 = ex2_approx(y1);
            sum2[i & 3] = fadd2(sum2[i & 3], f2(e0, e1));
            pk[i] = pack_bf16x2(e0, e1);
          }
        }
        {
          if (__any_sync(0xffffffffu, d1 != 0.f)) {  // the max moved (or an item's first block)
            const unsigned long long d2 = f2(d1, d1);
#pragma unroll
            for (int i = 0; i < (128 - kKeepF32) / 2; ++i) {
              float y0, y1;
              unpack_f16x2(h1[i], y0, y1);
              f2_split(fadd2(f2(y0, y1), d2), y0, y1);
              const float e0 = ex2_approx(y0), e1 = ex2_approx(y1);
              sum2[i & 3] = fadd2(sum2[i & 3], f2(e0, e1));
              pk[kKeepF32 / 2 + i] = pack_bf16x2(e0, e1);
            }
          } else {
#pragma unroll
            for (int i = 0; i < (128 - kKeepF32) / 2; ++i) {
              float y0, y1;
              unpack_f16x2(h1[i], y0, y1);
              const float e0 = ex2_approx(y0), e1 = ex2_approx(y1);
              sum2[i & 3] = fadd2(sum2[i & 3], f2(e0, e1));
              pk[kKeepF32 / 2 + i] = pack_bf16x2(e0, e1);
            }
          }
        }
        {
          const unsigned long long s2 = fadd2(fadd2(sum2[0], sum2[1]), fadd2(sum2[2], sum2[3]));
          float a, b;
          f2_split(s2, a, b);
          l += a + b;
        }
        // P(J - 1) has been read by P(J - 1) V_{J-1} before P(J) replaces it
        if (!pfree_seen) {
          ok = mbar_wait(pfree, (J - 1) & 1, c, kSiteTmemEmpty);
          if (!ok) break;
          tc_fence_after();
        }
        // P (bf16, keys 2i and 2i + 1 of this group in column i)
        tmem_st32_raw(tmem + kColP + g * 64 + lane_off, pk);
        tmem_st32_raw(tmem + kColP + g * 64 + 32 + lane_off, pk + 32);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(lead(pready));
      }
      // The unit's last P V has completed.  A whole item writes O / (l_0 + l_1); this group
      // writes head dims [64 g, 64 g + 64).
      const int Jl = J0 + nb - 1;
      J0 += nb;
      if (ok) ok = mbar_wait(pfree, Jl & 1, c, kSiteTmemFull);
      tc_fence_after();
      float ol = 0.f;
      if (ok) ok = exchange(l, ol);
      const AttnUnit u = attn_unit(kq, pair, npairs, p.nfull, nblk);
      const int h = u.it / nqt, qt = u.it - h * nqt;
      // Every lane takes part in the (warp-collective) TMEM loads; rows past the end of the
      // queries (a partial last tile) are only not stored.
      const int qrow = qt * 2 * kBQ + static_cast<int>(crank) * kBQ + row;
      const bool live = !Ragged || qrow < p.Lq;
      uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(h) * p.Lq + qrow) * kD + g * 64);
      if (ok && u.half < 0) {
        const float inv = 1.0f / (l + ol);
#pragma unroll 1
        for (int cb = 0; cb < 2; ++cb) {
          float o[32];
          tmem_ld32(tog + cb * 32 + lane_off, o);
          if (live) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[cb * 4 + v] = make_uint4(pack_bf16x2(o[8 * v] * inv, o[8 * v + 1] * inv),
                                           pack_bf16x2(o[8 * v + 2] * inv, o[8 * v + 3] * inv),
                                           pack_bf16x2(o[8 * v + 4] * inv, o[8 * v + 5] * inv),
                                           pack_bf16x2(o[8 * v + 6] * inv, o[8 * v + 7] * inv));
          }
        }
      } else if (ok) {
        // A half: write this CTA's partial results, then exchange the epoch into the item's
        // counter; the half that finds this call's epoch there already combines.
        const int t = u.it - p.nfull;
        const size_t slot = (static_cast<size_t>(t) * 2 + u.half) * 2 + crank;
        const size_t other = (static_cast<size_t>(t) * 2 + (1 - u.half)) * 2 + crank;
        float* po = p.part_o + slot * (kPartO / 4) + static_cast<size_t>(row) * kD + g * 64;
#pragma unroll 1
        for (int cb = 0; cb < 2; ++cb) {
          float o[32];
          tmem_ld32(tog + cb * 32 + lane_off, o);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            reinterpret_cast<float4*>(po + cb * 32)[v] = make_float4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
        }
        const float lt = l + ol;
        if (g == 0) reinterpret_cast<float2*>(p.part_ml + slot * (kPartML / 4))[row] = make_float2(m2, lt);
        __threadfence();
        __syncwarp();
        if (lane == 0) mbar_arrive(tail_w);
        if (warp == 2 && lane == 0) {
          ok = mbar_wait(tail_w, ntail_done & 1, c, kSiteTmemFull);
          if (ok) {
            __threadfence();
            const unsigned long long prev = atomicExch(p.tail_ctr + static_cast<size_t>(t) * 2 + crank, c.epoch);
            *tail_second = prev == c.epoch ? 1u : 0u;
          }
          mbar_arrive(tail_r);
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (ok) ok = mbar_wait(tail_r, ntail_done & 1, c, kSiteTmemFull);
        ++ntail_done;
        if (ok && *tail_second) {
          __threadfence();
          const float* qo = p.part_o + other * (kPartO / 4) + static_cast<size_t>(row) * kD + g * 64;
          const float2 mlo = __ldcg(reinterpret_cast<const float2*>(p.part_ml + other * (kPartML / 4)) + row);
          // half 0's values first, whichever half this is
          const float ma = u.half == 0 ? m2 : mlo.x, la = u.half == 0 ? lt : mlo.y;
          const float mb = u.half == 0 ? mlo.x : m2, lb = u.half == 0 ? mlo.y : lt;
          const float m = fmaxf(ma, mb);
          const float ca = ex2_approx(ma - m), cbb = ex2_approx(mb - m);
          const float inv = 1.0f / (la * ca + lb * cbb);
          const float wa = ca * inv, wb = cbb * inv;
#pragma unroll 1
          for (int cb = 0; cb < 2; ++cb) {
            // this half's O is still in TMEM (the next unit's first P V waits for ofree)
            float o[32], q[32];
            tmem_ld32(tog + cb * 32 + lane_off, o);
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              const float4 t4 = __ldcg(reinterpret_cast<const float4*>(qo + cb * 32) + v);
              q[4 * v] = t4.x;
              q[4 * v + 1] = t4.y;
              q[4 * v + 2] = t4.z;
              q[4 * v + 3] = t4.w;
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = u.half == 0 ? o[i] * wa + q[i] * wb : q[i] * wa + o[i] * wb;
            if (live) {
#pragma unroll
              for (int v = 0; v < 4; ++v)
                dst[cb * 4 + v] = make_uint4(pack_bf16x2(o[8 * v], o[8 * v + 1]), pack_bf16x2(o[8 * v + 2], o[8 * v + 3]),
                                             pack_bf16x2(o[8 * v + 4], o[8 * v + 5]),
                                             pack_bf16x2(o[8 * v + 6], o[8 * v + 7]));
            }
          }
        }
      }
      if (ok) {
        // O read: the next unit's first P V may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(lead(ofree));
      }
      tc_fence_before();
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ movers
    // The gather in the order the work items need it: heads in groups of hg, the heads that
    // one wave of items (npairs consecutive items) covers; for each group the shard steps
    // rank + 1, rank + 2, ... (the local shard last), each over the group's heads and their
    // 128-key blocks.  K and V of a block, then its signal.  Each lane keeps 16 vectors of
    // 16 bytes in flight.
    const int mw = warp - 2 - kSoftWarps;
    const int nw = static_cast<int>(gridDim.x) * kMovers;
    const int hg = (npairs + nqt - 1) / nqt < p.heads ? (npairs + nqt - 1) / nqt : p.heads;
    const int per_grp = p.W * hg * sbs;
    const int total = p.W * p.heads * sbs;
    for (int gb = blockIdx.x * kMovers + mw; gb < total; gb += nw) {
      const int grp = gb / per_grp;
      int rem = gb - grp * per_grp;
      const int gs = p.heads - grp * hg < hg ? p.heads - grp * hg : hg;  // heads in this group
      const int i = rem / (gs * sbs);
      rem -= i * gs * sbs;
      const int hh = grp * hg + rem / sbs, b = rem % sbs;
      const int r = (p.rank + 1 + i) % p.W;
      const int rows = min(kSigBlk, p.Lr - b * kSigBlk);  // the last block may be partial
      const size_t row_bytes = static_cast<size_t>(kD) * 2;
      const size_t src = (static_cast<size_t>(hh) * p.Lr + static_cast<size_t>(b) * kSigBlk) * row_bytes;
      const size_t dst = ((static_cast<size_t>(r) * p.heads + hh) * p.Lr + static_cast<size_t>(b) * kSigBlk) * row_bytes;
      const int nvec = (Ragged ? rows : kSigBlk) * static_cast<int>(row_bytes / 16);
#pragma unroll 1
      for (int t = 0; t < 2; ++t) {  // K, then V
        const uint4* s4 = reinterpret_cast<const uint4*>((t ? p.vshard[r] : p.kshard[r]) + src);
        uint4* d4 = reinterpret_cast<uint4*>((t ? p.vg : p.kg) + dst);
        for (int v0 = lane; v0 < nvec; v0 += 16 * 32) {
          uint4 buf[16];
#pragma unroll
          for (int u = 0; u < 16; ++u)
            if (v0 + u * 32 < nvec) buf[u] = __ldg(s4 + v0 + u * 32);
#pragma unroll
          for (int u = 0; u < 16; ++u)
            if (v0 + u * 32 < nvec) d4[v0 + u * 32] = buf[u];
        }
      }
      __threadfence();
      __syncwarp();
      if (lane == 0) st_release_gpu(p.flags + (static_cast<size_t>(r) * p.heads + hh) * sbs + b, c.epoch);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the leader's MMAs are drained and both CTAs are done with TMEM and remote barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace tl

using namespace tl;

// ============================================================================ C ABI
static size_t attn_al256(size_t x) { return (x + 255) & ~size_t(255); }

static bool attn_shape_ok(int W, int heads, int l_r, int d) {
  return W >= 1 && W <= 8 && heads >= 0 && l_r >= 0 && d == attn::kD &&
         static_cast<long long>(W) * l_r < (1LL << 30);
}

// Split items the workspace holds partial results for: at most one per two pairs of any grid
// up to 2 kMaxTail pairs, and no more than there are items.
static size_t attn_max_tail(int heads, int l_r) {
  const size_t nwork = static_cast<size_t>(heads) * ((l_r + 2 * attn::kBQ - 1) / (2 * attn::kBQ));
  return nwork < static_cast<size_t>(attn::kMaxTail) ? nwork : static_cast<size_t>(attn::kMaxTail);
}

// Workspace: gathered K, gathered V, block signals, split-item partials (O, then m and l),
// split-item counters; each region 256-byte aligned.
struct AttnLayout {
  size_t kv, v_off, flags_off, part_o_off, part_ml_off, ctr_off, total;
};
static AttnLayout attn_layout(int W, int heads, int l_r, int d) {
  AttnLayout L;
  L.kv = static_cast<size_t>(heads) * W * l_r * d * 2;
  const size_t flags = static_cast<size_t>(W) * heads * ((l_r + attn::kSigBlk - 1) / attn::kSigBlk) * 8;
  const size_t tail = attn_max_tail(heads, l_r);
  L.v_off = attn_al256(L.kv);
  L.flags_off = L.v_off + attn_al256(L.kv);
  L.part_o_off = L.flags_off + attn_al256(flags);
  L.part_ml_off = L.part_o_off + attn_al256(tail * 4 * attn::kPartO);
  L.ctr_off = L.part_ml_off + attn_al256(tail * 4 * attn::kPartML);
  L.total = L.ctr_off + attn_al256(tail * 2 * 8);
  return L;
}

extern "C" size_t tl_ag_attention_workspace_bytes(int W, int heads, int l_r, int d) {
  if (!attn_shape_ok(W, heads, l_r, d)) return 0;
  return attn_layout(W, heads, l_r, d).total;
}

extern "C" int tl_ag_attention(tl_ctx* ctx, int W, int rank, const void* q, const void* const* k_shards,
                               const void* const* v_shards, void* out, void* workspace, size_t workspace_bytes,
                               int heads, int l_r, int d, tl_stream_t stream) {
  if (!ctx || !attn_shape_ok(W, heads, l_r, d) || rank < 0 || rank >= W) return TL_ERR_INVALID;
  if (heads == 0 || l_r == 0) return TL_OK;
  if (!q || !k_shards || !v_shards || !out || !workspace) return TL_ERR_INVALID;
  if (!aligned16(q) || !aligned16(out) || !aligned16(workspace)) return TL_ERR_INVALID;
  for (int r = 0; r < W; ++r)
    if (!k_shards[r] || !v_shards[r] || !aligned16(k_shards[r]) || !aligned16(v_shards[r])) return TL_ERR_INVALID;
  if (workspace_bytes < tl_ag_attention_workspace_bytes(W, heads, l_r, d)) return TL_ERR_WORKSPACE;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return TL_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const AttnLayout lay = attn_layout(W, heads, l_r, d);

  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.kg = ws;
  p.vg = ws + lay.v_off;
  p.flags = reinterpret_cast<uint64_t*>(ws + lay.flags_off);
  p.part_o = reinterpret_cast<float*>(ws + lay.part_o_off);
  p.part_ml = reinterpret_cast<float*>(ws + lay.part_ml_off);
  p.tail_ctr = reinterpret_cast<unsigned long long*>(ws + lay.ctr_off);
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t WH = static_cast<uint64_t>(W) * heads;
  if (!tmap_3d(&p.q, BF, 2, q, d, l_r, heads, 64, 128, 1) ||
      !tmap_3d(&p.k_loc, BF, 2, k_shards[rank], d, l_r, heads, 64, 128, 1) ||
      !tmap_3d(&p.k_gat, BF, 2, p.kg, d, l_r, WH, 64, 128, 1) ||
      !tmap_3d(&p.v_loc, BF, 2, v_shards[rank], d, l_r, heads, 64, 64, 1) ||
      !tmap_3d(&p.v_gat, BF, 2, p.vg, d, l_r, WH, 64, 64, 1))
    return TL_ERR_CUDA;
  p.common = make_common(ctx);
  p.common.trace_hdr = nullptr;  // the attention kernel records no trace spans
  p.common.trace = nullptr;
  for (int r = 0; r < W; ++r) {
    p.kshard[r] = static_cast<const uint8_t*>(k_shards[r]);
    p.vshard[r] = static_cast<const uint8_t*>(v_shards[r]);
  }
  p.out = static_cast<__nv_bfloat16*>(out);
  p.W = W;
  p.rank = rank;
  p.Lq = l_r;
  p.Lr = l_r;
  p.heads = heads;
  p.scale = 1.0f / sqrtf(static_cast<float>(d));

  // Clusters of two CTAs, one CTA per SM, no more clusters than can be resident at once: a
  // CTA waiting on a block's signal is co-resident with the mover warps that will set it.
  auto kern = l_r % attn::kBKV == 0 ? attn_kernel<false> : attn_kernel<true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, attn::kSmem) != cudaSuccess) {
    (void)cudaGetLastError();
    return TL_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(attn::kThreads, 1, 1);
  cfg.dynamicSmemBytes = attn::kSmem;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int max_clusters[2] = {-1, -1};  // per instantiation
  const int ki = l_r % attn::kBKV == 0 ? 0 : 1;
  if (max_clusters[ki] < 0) {
    cfg.gridDim = dim3(ctx->sms & ~1, 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      return TL_ERR_UNSUPPORTED;
    }
    max_clusters[ki] = n;
  }
  int nclusters = ctx->ctas / 2;
  if (nclusters > max_clusters[ki]) nclusters = max_clusters[ki];
  if (nclusters < 1) return TL_ERR_UNSUPPORTED;
  cfg.gridDim = dim3(2 * nclusters, 1, 1);
  // Split the last items into halves when they would fill less than half of the last wave
  // (and the workspace holds their partials); a half needs at least one key block.
  {
    const int nqt = (l_r + 2 * attn::kBQ - 1) / (2 * attn::kBQ);
    const int nwork = heads * nqt, nblk = W * ((l_r + attn::kBKV - 1) / attn::kBKV);
    const int rem = nwork % nclusters;
    const bool split = rem > 0 && 2 * rem <= nclusters && nblk >= 2 &&
                       static_cast<size_t>(rem) <= attn_max_tail(heads, l_r);
    p.ntail = split ? rem : 0;
    p.nfull = nwork - p.ntail;
  }
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return TL_ERR_CUDA;
  }
  return TL_OK;
}
