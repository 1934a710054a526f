// Sequence-parallel self-attention with the KV AllGather overlapped ("TileLink: Generating
// Efficient Compute-Communication Overlapping Kernels using Tile-Centric Primitives", §5
// Figure 6 text and §7.2 self-attention: the KV cache sequence S is split into W shards,
// one per rank, gathered while the attention of the rank's queries runs over the shards as
// they arrive; "Triton-distributed ...", §3.7 swizzle: the local shard first).
//
// Persistent clusters of two CTAs (one per SM) walk (head, 256-query tile) work items; CTA r
// of a pair owns queries [128 r, 128 r + 128) of the tile.  Each item is non-causal flash
// attention over all W shards in blocks of 256 keys, on tcgen05 pair MMAs (cta_group::2):
//   S_J = Q K_J^T      M = 256 queries, N = 256 keys, K = 128 head dims: CTA r's A is its
//                      128 query rows, its B half the keys [128 r, 128 r + 128) of the block
//                      (K-major), and its TMEM gets its rows' 256 scores;
//   O_g += P_g V_g     for each half g of the block's keys: M = 256 queries, N = 128 head
//                      dims, K = 128 keys: CTA r's A is its rows of P_g, its B half the head
//                      dims [64 r, 64 r + 64) of V (MN-major).  The two halves keep separate
//                      accumulators O_0, O_1 (and separate running max and sum), combined
//                      once per item: a flash-decoding style split of the keys inside the block.
// Warps of each CTA:
//   warp 0     TMA producer: its Q rows, then per key block its K half (2 boxes) and V half
//              (4 boxes) through 2-stage rings; every load completes on the pair leader's
//              barrier; the first block of a remote shard slice waits on the slice's block
//              signals (one warp-wide poll).
//   warp 1     TMEM allocation (both CTAs) and, in the leader, the pair MMAs (one thread).
//   warps 2-9  softmax, two warpgroups: warpgroup g takes keys [128 g, 128 g + 128) of every
//              block for all 128 rows (one row per thread), with its own running max m_g and
//              sum l_g in base 2 (the 1/sqrt(d) scale folded into one multiply-add per score);
//              P_g (bf16) goes into its half of the shared-memory P buffer in the MMA's
//              K-major 128-byte-swizzled layout.  The running max of a row moves only when
//              the block's max exceeds it by more than 2^8 (kRescaleLog2): until then P <= 256
//              and O_g, l_g keep the stale max, which cancels in the final division; a move
//              rescales O_g in TMEM after the previous P_g V_g has completed.  At the end of
//              an item the groups exchange m_g, l_g and each writes 64 head dims of
//              (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / (l_0 2^(m_0 - m) + l_1 2^(m_1 - m)) as bf16.
//   warps 10-11 movers: remote K/V blocks (up to 32 KB each) into the shard-major gathered
//              buffers, one release signal per 128-key block, in the order the items need
//              them (groups of heads one wave covers, shard by shard, the local shard last).
// The softmax warps of both CTAs arrive on the leader's barriers for "S read" and "P_g
// written" (relaxed cluster-scope arrivals: a release at cluster scope costs a full memory
// barrier per arrival); the leader's MMA commits arrive on both CTAs' barriers (one
// multicast commit).  TMEM columns (each CTA, its 128 rows): S [0, 256),
// O_0 [256, 384), O_1 [384, 512).  The pipeline counters run on across items.  Every wait
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
constexpr int kQBytes = 2 * kBox;   // this CTA's 128 queries x 128 dims
constexpr int kKBytes = 2 * kBox;   // this CTA's 128 keys of a block x 128 dims
constexpr int kVBytes = 4 * 8192;   // 256 keys x this CTA's 64 dims: 4 boxes of 64 keys
constexpr int kPBytes = 4 * kBox;   // 128 rows x 256 keys: 4 boxes of 64 keys
constexpr int kStages = 2;
constexpr int kRedBytes = 2 * kBQ * 4;  // one float per row and softmax warpgroup
constexpr int kBarBytes = 192;
constexpr int kSmem = 1024 + kQBytes + kStages * (kKBytes + kVBytes) + kPBytes + kRedBytes + kBarBytes;
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
  int W, rank, Lq, Lr, heads;
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

// S_J = Q K_J^T on the pair: M = 256, N = 256, K = 128 (8 steps of 16 head dims).
__device__ __forceinline__ void attn_mma_s(uint32_t d, uint32_t q0, uint32_t k0) {
  constexpr uint32_t idesc = umma_idesc_bf16(256, 256, false);
#pragma unroll
  for (int kb = 0; kb < 2; ++kb)
#pragma unroll
    for (int k = 0; k < 4; ++k)
      umma_bf16_pair(d, umma_desc_sw128(q0 + kb * attn::kBox + k * 32, 16, 1024),
                     umma_desc_sw128(k0 + kb * attn::kBox + k * 32, 16, 1024), idesc, (kb | k) ? 1u : 0u);
}

// O_g (+)= P_g V_g on the pair: M = 256, N = 128, K = 128 keys (8 steps); each CTA's V half
// is 64 head dims wide (one 64-column group), its 64-key boxes 8 KB apart.
__device__ __forceinline__ void attn_mma_pv(uint32_t d, uint32_t p0, uint32_t v0, bool acc) {
  constexpr uint32_t idesc = umma_idesc_bf16(256, 128, true);
#pragma unroll
  for (int kb = 0; kb < 2; ++kb)
#pragma unroll
    for (int k = 0; k < 4; ++k)
      umma_bf16_pair(d, umma_desc_sw128(p0 + kb * attn::kBox + k * 32, 16, 1024),
                     umma_desc_sw128(v0 + kb * 8192 + k * 2048, 8192, 1024), idesc, (acc || kb || k) ? 1u : 0u);
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

// Relaxed arrival on an mbarrier given by its shared::cluster address: no memory ordering is
// implied (a release at cluster scope costs a full memory barrier on every call).  Used where
// what the arrival announces is already complete in this thread: its TMEM reads
// (tcgen05.wait::ld, then tcgen05.fence::before_thread_sync) or its P stores, made visible to
// the tensor core by fence.proxy.async before the arrival.
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

// Ragged: some shard length l_r is not a multiple of 256 (a partial last key block of every
// shard and a partial last query tile); the common case is compiled without those checks.
template <bool Ragged>
__global__ void __launch_bounds__(attn::kThreads, 1) attn_kernel(const __grid_constant__ AttnParams p) {
  using namespace attn;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = base;
  uint8_t* sk = sq + kQBytes;
  uint8_t* sv = sk + kStages * kKBytes;
  uint8_t* sp = sv + kStages * kVBytes;
  float* red = reinterpret_cast<float*>(sp + kPBytes);  // [group][row]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sp + kPBytes + kRedBytes);
  // counted on the leader (the peer's copies are unused): loads of both CTAs, arrivals of
  // both CTAs' softmax warps
  uint64_t* qfull = bars;
  uint64_t* kfull = bars + 1;    // [2]
  uint64_t* vfull = bars + 3;    // [2]
  uint64_t* sfree = bars + 5;    // every softmax warp of the pair has read its S half
  uint64_t* pready = bars + 6;   // [2] group g: its 8 warps of the pair wrote P_g, O_g rescaled
  // in both CTAs, arrived on by the leader's MMA commits
  uint64_t* qempty = bars + 8;   // the item's last S MMA has read Q
  uint64_t* kempty = bars + 9;   // [2]
  uint64_t* vempty = bars + 11;  // [2]
  uint64_t* sfull = bars + 13;   // S_J is in TMEM
  uint64_t* pfree = bars + 14;   // [2] group g: P_g V_g of the block complete (P_g free, O_g stable)
  uint64_t* drain = bars + 16;
  // this CTA's softmax warps, once per item
  uint64_t* xw = bars + 17;      // all 8 wrote their m_g, l_g to red
  uint64_t* xr = bars + 18;      // all 8 read the other group's
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 19);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const bool leader = crank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const Common& c = p.common;
  const int bps = (p.Lr + kBKV - 1) / kBKV;       // 256-key blocks per shard (the last may be partial)
  const int sbs = (p.Lr + kSigBlk - 1) / kSigBlk;  // 128-key signal blocks per shard
  const int nblk = p.W * bps;                      // key blocks per item
  const int nqt = (p.Lq + 2 * kBQ - 1) / (2 * kBQ);  // 256-query tiles (the last may be partial)
  const int nwork = p.heads * nqt;
  if (threadIdx.x == 0) {
    mbar_init(qfull, 1);
    mbar_init(qempty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
    }
    mbar_init(sfull, 1);
    mbar_init(sfree, 2 * kSoftWarps);  // counted on the leader: the softmax warps of both CTAs
    for (int g = 0; g < 2; ++g) {
      mbar_init(&pready[g], kSoftWarps);  // the 4 warps of group g in each CTA
      mbar_init(&pfree[g], 1);
    }
    mbar_init(drain, 1);
    mbar_init(xw, kSoftWarps);
    mbar_init(xr, kSoftWarps);
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
    uint32_t filled = 0, par = 0;  // leader's drain: K stages (bits 0-1), V stages (bits 2-3)
    int J = 0, kq = 0;
    for (int it = pair; it < nwork && ok; it += npairs, ++kq) {
      const int h = it / nqt, qt = it - h * nqt;
      if (lane == 0) {
        ok = mbar_wait(qempty, (kq & 1) ^ 1u, c, kSiteEmpty);
        if (ok) {
          if (leader) mbar_arrive_expect_tx(qfull, 2 * kQBytes);
          const int y = qt * 2 * kBQ + static_cast<int>(crank) * kBQ;
          tma_load_3d_pair(sq, &p.q, lead(qfull), 0, y, h);
          tma_load_3d_pair(sq + kBox, &p.q, lead(qfull), 64, y, h);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      for (int j = 0; j < nblk && ok; ++j, ++J) {
        const int step = j / bps, blk = j - step * bps;
        const int r = (p.rank + step) % p.W;
        const bool local = step == 0;
        if (!local && blk == 0) {
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
              tma_load_3d_pair(sv + s * kVBytes + kb * 8192, vm, lead(&vfull[s]), xv, y + kb * 64, z);
            filled |= 4u << s;
            par = (par & ~(4u << s)) | (ph << (s + 2));
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      }
    }
    if (lane == 0 && leader) {  // drain: every fill of both CTAs has landed before the pair exits
      if (kq > 0) mbar_wait(qfull, (kq - 1) & 1, c, kSiteDrain);
      for (int s = 0; s < kStages; ++s) {
        if (filled & (1u << s)) mbar_wait(&kfull[s], (par >> s) & 1u, c, kSiteDrain);
        if (filled & (4u << s)) mbar_wait(&vfull[s], (par >> (s + 2)) & 1u, c, kSiteDrain);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (leader && lane == 0) {
      bool ok = true;
      const uint32_t q0 = smem_u32(sq), p0 = smem_u32(sp);
      const uint32_t ts = tmem, to = tmem + 256;  // S; O_0 (O_1 at + 128)
      int J0 = 0, kq = 0;
      for (int it = pair; it < nwork && ok; it += npairs, ++kq, J0 += nblk) {
        ok = mbar_wait(qfull, kq & 1, c, kSiteFull);
        tc_fence_after();
        for (int j = 0; j <= nblk && ok; ++j) {
          if (j < nblk) {  // S of block J0 + j (S has one TMEM buffer: its last reader is done)
            const int J = J0 + j, s = J & 1;
            const uint32_t ph = (J >> 1) & 1;
            ok = (J == 0 || mbar_wait(sfree, (J - 1) & 1, c, kSiteTmemEmpty)) && mbar_wait(&kfull[s], ph, c, kSiteFull);
            if (!ok) break;
            tc_fence_after();
            attn_mma_s(ts, q0, smem_u32(sk + s * kKBytes));
            commit_both(&kempty[s]);
            commit_both(sfull);
            if (j == nblk - 1) commit_both(qempty);
          }
          if (j >= 1) {  // O_g += P_g V_g of block J0 + j - 1, g = 0, 1
            const int I = J0 + j - 1, s = I & 1;
            const uint32_t ph = (I >> 1) & 1;
            ok = mbar_wait(&vfull[s], ph, c, kSiteFull);
            if (!ok) break;
#pragma unroll 1
            for (int g = 0; g < 2 && ok; ++g) {
              ok = mbar_wait(&pready[g], I & 1, c, kSiteFull);
              if (!ok) break;
              tc_fence_after();
              attn_mma_pv(to + g * 128, p0 + g * 2 * kBox, smem_u32(sv + s * kVBytes) + g * 2 * 8192, j > 1);
              commit_both(&pfree[g]);
            }
            if (!ok) break;
            commit_both(&vempty[s]);
          }
        }
      }
      umma_commit_pair(drain);
      mbar_wait(drain, 0, c, kSiteDrain);
    }
    __syncwarp();
  } else if (warp < 2 + kSoftWarps) {
    // ------------------------------------------------------------ softmax (one row per thread)
    const int g = (warp - 2) >> 2;          // warpgroup: keys [128 g, 128 g + 128) of a block
    const int qd = warp & 3;                // TMEM lane quadrant of this warp
    const int row = qd * 32 + lane;         // query row inside the CTA's 128
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    const uint32_t tog = tmem + 256 + g * 128;  // O_g
    const float sl2 = p.scale * kLog2e;     // raw score -> base-2 exponent
    bool ok = true;
    int J0 = 0;
    uint32_t nx = 0;  // exchanges so far
    // Exchange one float per row with the other warpgroup through red (bounded waits: a
    // timeout elsewhere never leaves a warp blocked here).
    auto exchange = [&](float mine, float& other) -> bool {
      if (nx > 0 && !mbar_wait(xr, (nx - 1) & 1, c, kSiteTmemFull)) return false;  // red is free again
      red[g * kBQ + row] = mine;
      __syncwarp();
      if (lane == 0) mbar_arrive(xw);
      if (!mbar_wait(xw, nx & 1, c, kSiteTmemFull)) return false;
      other = red[(1 - g) * kBQ + row];
      __syncwarp();
      if (lane == 0) mbar_arrive(xr);
      ++nx;
      return true;
    };
    for (int it = pair; it < nwork && ok; it += npairs, J0 += nblk) {
      const int h = it / nqt, qt = it - h * nqt;
      float m2 = -INFINITY, l = 0.f;  // this group's running max (base-2 units) and sum
      int blk = -1;                   // block index inside the current shard
      for (int j = 0; j < nblk && ok; ++j) {
        const int J = J0 + j;
        if (++blk == bps) blk = 0;
        // The wait results are warp-uniform, as the warp-collective TMEM accesses below need:
        // the converged warp runs each try_wait and timer read as one instruction.
        ok = mbar_wait(sfull, J & 1, c, kSiteTmemFull);
        if (!ok) break;
        tc_fence_after();
        float x[128];
        {
          uint32_t rr[4][32];
#pragma unroll
          for (int cb = 0; cb < 4; ++cb) tmem_ld32_issue(tmem + g * 128 + cb * 32 + lane_off, rr[cb]);
          tmem_ld_wait(rr[0]);
          tmem_ld_after(rr[1]);
          tmem_ld_after(rr[2]);
          tmem_ld_after(rr[3]);
#pragma unroll
          for (int i = 0; i < 128; ++i) x[i] = __uint_as_float(rr[i >> 5][i & 31]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(lead(sfree));
        if constexpr (Ragged) {
          // keys past the end of a shard (its partial last block, zero-filled by TMA) get no
          // weight: their scores become -inf before the maximum
          const int valid = p.Lr - blk * kBKV - g * 128;
          if (valid < 128) {
#pragma unroll
            for (int i = 0; i < 128; ++i) x[i] = i < valid ? x[i] : -INFINITY;
          }
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = x[i];
#pragma unroll
        for (int i = 8; i < 128; i += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], x[i + k], x[i + 8 + k]);
        const float bm2 = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) *
                          sl2;  // the scale is positive: max commutes with it
        if (j == 0) {
          m2 = bm2;  // the item's first P_g V_g overwrites O_g
        } else if (__any_sync(0xffffffffu, bm2 > m2 + kRescaleLog2)) {
          const float mn = fmaxf(m2, bm2);
          const float corr = ex2_approx(m2 - mn);  // 0 while the group has seen only absent keys
          // O_g is stable once P_g V_g of the previous block has completed
          ok = mbar_wait(&pfree[g], (J - 1) & 1, c, kSiteTmemFull);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb) {
            float o[32];
            tmem_ld32(tog + cb * 32 + lane_off, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= corr;
            tmem_st32(tog + cb * 32 + lane_off, o);
          }
          l *= corr;
          m2 = mn;
        }
        // (Ragged: a group whose keys so far are all absent has m2 = -inf; its P is 0.)
        const float nm = (Ragged && m2 == -INFINITY) ? 0.f : -m2;
        unsigned long long sum2[4];  // 8 partial sums, two per register pair
        uint32_t pk[64];
#pragma unroll
        for (int i = 0; i < 4; ++i) sum2[i] = 0ull;
        const unsigned long long sl2x2 = f2(sl2, sl2), nm2 = f2(nm, nm);
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          float y0, y1;
          f2_split(ffma2(f2(x[2 * i], x[2 * i + 1]), sl2x2, nm2), y0, y1);
          const float e0 = ex2_approx(y0), e1 = ex2_approx(y1);
          sum2[i & 3] = fadd2(sum2[i & 3], f2(e0, e1));
          pk[i] = pack_bf16x2(e0, e1);
        }
        {
          const unsigned long long s2 = fadd2(fadd2(sum2[0], sum2[1]), fadd2(sum2[2], sum2[3]));
          float a, b;
          f2_split(s2, a, b);
          l += a + b;
        }
        // P_g's half of the buffer was last read by P_g V_g of block J - 1
        if (J > 0) ok = mbar_wait(&pfree[g], (J - 1) & 1, c, kSiteTmemEmpty);
        if (!ok) break;
        // P_g (bf16) as the K-major, 128-byte-swizzled A operand: keys [64 b, 64 b + 64) of
        // this row are 128 bytes of box b; 16-byte piece u sits at piece u ^ (row & 7).
        const uint32_t prow = smem_u32(sp) + row * 128;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint32_t* v = pk + kb * 32 + u * 4;
            st_shared_v4(prow + (2 * g + kb) * kBox + ((u ^ (row & 7)) << 4), v[0], v[1], v[2], v[3]);
          }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(lead(&pready[g]));
      }
      // Both halves' last P V of the item have completed: combine
      //   O = (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / (l_0 2^(m_0 - m) + l_1 2^(m_1 - m)),
      // m = max(m_0, m_1); this group writes head dims [64 g, 64 g + 64).
      const int Jl = J0 + nblk - 1;
      if (ok) ok = mbar_wait(&pfree[0], Jl & 1, c, kSiteTmemFull) && mbar_wait(&pfree[1], Jl & 1, c, kSiteTmemFull);
      tc_fence_after();
      float om = 0.f, ol = 0.f;
      if (ok) ok = exchange(m2, om) && exchange(l, ol);
      if (ok) {
        const float m = fmaxf(m2, om);
        const float a_mine = ex2_approx(m2 - m), a_other = ex2_approx(om - m);
        const float inv = 1.0f / (l * a_mine + ol * a_other);
        const float c0 = (g == 0 ? a_mine : a_other) * inv, c1 = (g == 0 ? a_other : a_mine) * inv;
        // Every lane takes part in the (warp-collective) TMEM loads; rows past the end of
        // the queries (a partial last tile) are only not stored.
        const int qrow = qt * 2 * kBQ + static_cast<int>(crank) * kBQ + row;
        const bool live = !Ragged || qrow < p.Lq;
        uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(h) * p.Lq + qrow) * kD + g * 64);
#pragma unroll 1
        for (int cb = 0; cb < 2; ++cb) {
          float o0[32], o1[32];
          tmem_ld32(tmem + 256 + g * 64 + cb * 32 + lane_off, o0);
          tmem_ld32(tmem + 384 + g * 64 + cb * 32 + lane_off, o1);
#pragma unroll
          for (int i = 0; i < 32; ++i) o0[i] = o0[i] * c0 + o1[i] * c1;
          if (live) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              dst[cb * 4 + u] = make_uint4(pack_bf16x2(o0[8 * u], o0[8 * u + 1]), pack_bf16x2(o0[8 * u + 2], o0[8 * u + 3]),
                                           pack_bf16x2(o0[8 * u + 4], o0[8 * u + 5]),
                                           pack_bf16x2(o0[8 * u + 6], o0[8 * u + 7]));
          }
        }
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

extern "C" size_t tl_ag_attention_workspace_bytes(int W, int heads, int l_r, int d) {
  if (!attn_shape_ok(W, heads, l_r, d)) return 0;
  const size_t kv = static_cast<size_t>(heads) * W * l_r * d * 2;
  const size_t flags = static_cast<size_t>(W) * heads * ((l_r + attn::kSigBlk - 1) / attn::kSigBlk) * 8;
  return 2 * attn_al256(kv) + attn_al256(flags);
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
  const size_t kv = static_cast<size_t>(heads) * W * l_r * d * 2;

  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.kg = ws;
  p.vg = ws + attn_al256(kv);
  p.flags = reinterpret_cast<uint64_t*>(ws + 2 * attn_al256(kv));
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
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return TL_ERR_CUDA;
  }
  return TL_OK;
}
