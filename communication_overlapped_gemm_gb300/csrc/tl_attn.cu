// Sequence-parallel self-attention with the KV AllGather overlapped ("TileLink: Generating
// Efficient Compute-Communication Overlapping Kernels using Tile-Centric Primitives", §5
// Figure 6 text and §7.2 self-attention: the KV cache sequence S is split into W shards,
// one per rank, gathered while the attention of the rank's queries runs over the shards as
// they arrive; "Triton-distributed ...", §3.7 swizzle: the local shard first).
//
// One persistent cooperative CTA per SM walks (head, 128-query tile) work items; each item
// is non-causal flash attention over all W shards on tcgen05, head dim 128:
//   warp 0    TMA producer: the item's Q, then per 128-key block K (2 boxes) and V (4 boxes)
//             through 2-stage rings; the first block of a remote shard slice waits on the
//             slice's block signals (one warp-wide poll).
//   warp 1    TMEM allocation and the MMAs: S_j = Q K_j^T into one of two S buffers, then
//             O += P_{j-1} V_{j-1} once the softmax warps have published P_{j-1}.
//   warps 2-5 softmax, one query row per thread: S row from TMEM, running max and sum in
//             base 2 (the 1/sqrt(d) scale folded into one multiply-add per score), P (bf16)
//             into one of two shared-memory buffers in the MMA's K-major 128-byte-swizzled
//             layout.  The running max of a row moves only when the block's max exceeds it
//             by more than 2^8 (kRescaleLog2): until then P <= 256 and O, l keep the stale
//             max, which cancels in O / l.  A move rescales the warp's O rows in TMEM after
//             the previous P V has completed; writing P waits only for the P V two blocks
//             back.  Finally O / l as bf16.
//   warps 6-7 movers: remote K/V blocks (up to 32 KB each) into the shard-major gathered
//             buffers, one release signal per block, the local shard last.
// The pipeline counters run on across items.  TMEM columns: S0 [0, 128), S1 [128, 256),
// O [256, 384).  Every wait is bounded.
// Shard lengths need not be multiples of 128 (the Ragged instantiation): a shard's last key
// block and the last query tile may be partial.  TMA zero-fills the absent rows, the softmax
// gives the absent keys no weight, and the absent query rows are not stored.
#include "tl_host.h"

namespace tl {

namespace attn {
constexpr int kD = 128;        // head dim
constexpr int kBQ = 128;       // queries per work item
constexpr int kBKV = 128;      // keys per block
constexpr int kBlk = 16384;    // one 64-column SW128 box of 128 rows
constexpr int kQBytes = 2 * kBlk;
constexpr int kKBytes = 2 * kBlk;   // K block: 2 boxes of 64 head-dim columns
constexpr int kVBytes = 2 * kBlk;   // V block: 4 boxes of 64 keys x 64 head-dim columns
constexpr int kPBytes = 2 * kBlk;
constexpr int kStages = 2;
constexpr int kSmem = 1024 + kQBytes + kStages * (kKBytes + kVBytes) + 2 * kPBytes + 256;
constexpr float kRescaleLog2 = 8.0f;  // move the running max once it grows by more than this
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMovers = 2;
constexpr int kThreads = (6 + kMovers) * 32;
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
  uint64_t* flags;     // [W][H][Lr / 128]: K and V block gathered
  int W, rank, Lq, Lr, heads;
  float scale;  // 1 / sqrt(d)
};

// S_j = Q K_j^T: M = 128 queries, N = 128 keys, K = 128 head dims (K is a K-major B operand).
__device__ __forceinline__ void attn_mma_s(uint32_t d, uint32_t q0, uint32_t k0) {
  constexpr uint32_t idesc = umma_idesc_bf16(128, 128, false);
#pragma unroll
  for (int kb = 0; kb < 2; ++kb)
#pragma unroll
    for (int k = 0; k < 4; ++k)
      umma_bf16(d, umma_desc_sw128(q0 + kb * attn::kBlk + k * 32, 16, 1024),
                umma_desc_sw128(k0 + kb * attn::kBlk + k * 32, 16, 1024), idesc, (kb | k) ? 1u : 0u);
}

// O (+)= P_j V_j: M = 128 queries, N = 128 head dims, K = 128 keys (V is an MN-major B operand,
// its two 64-column groups 8 KB apart inside a 64-key box pair).
__device__ __forceinline__ void attn_mma_pv(uint32_t d, uint32_t p0, uint32_t v0, bool acc) {
  constexpr uint32_t idesc = umma_idesc_bf16(128, 128, true);
#pragma unroll
  for (int kb = 0; kb < 2; ++kb)
#pragma unroll
    for (int k = 0; k < 4; ++k)
      umma_bf16(d, umma_desc_sw128(p0 + kb * attn::kBlk + k * 32, 16, 1024),
                umma_desc_sw128(v0 + kb * attn::kBlk + k * 2048, 8192, 1024), idesc,
                (acc || kb || k) ? 1u : 0u);
}

// Ragged: some shard length l_r is not a multiple of 128 (a partial last key block of every
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
  uint64_t* bars = reinterpret_cast<uint64_t*>(sp + 2 * kPBytes);
  uint64_t* qfull = bars;
  uint64_t* kfull = bars + 1;   // [2]
  uint64_t* kempty = bars + 3;  // [2]
  uint64_t* vfull = bars + 5;   // [2]
  uint64_t* vempty = bars + 7;  // [2]
  uint64_t* sfull = bars + 9;   // [2] S of block J in TMEM buffer J % 2
  uint64_t* sfree = bars + 11;  // [2] softmax has read the S buffer
  uint64_t* pready = bars + 13; // [2] P of block J in buffer J % 2 written, O rescaled
  uint64_t* pfree = bars + 15;  // [2] P V of block J (P buffer J % 2) complete
  uint64_t* drain = bars + 17;
  uint64_t* qempty = bars + 18; // the item's last S MMA has read Q
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 19);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Common& c = p.common;
  const int bps = (p.Lr + kBKV - 1) / kBKV;  // key blocks per shard (the last may be partial)
  const int nblk = p.W * bps;                 // key blocks per item
  const int nqt = (p.Lq + kBQ - 1) / kBQ;     // query tiles (the last may be partial)
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
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sfree[s], 4);
      mbar_init(&pready[s], 4);
      mbar_init(&pfree[s], 1);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
    tma_prefetch_map(&p.q);
    tma_prefetch_map(&p.k_loc);
    tma_prefetch_map(&p.v_loc);
    tma_prefetch_map(&p.k_gat);
    tma_prefetch_map(&p.v_gat);
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    uint32_t filled = 0, par = 0;  // K stages (bits 0-1) and V stages (bits 2-3) in flight
    int J = 0, kq = 0;
    for (int it = blockIdx.x; it < nwork && ok; it += gridDim.x, ++kq) {
      const int h = it / nqt, qt = it - h * nqt;
      if (lane == 0) {
        ok = mbar_wait(qempty, (kq & 1) ^ 1u, c, kSiteEmpty);
        if (ok) {
          mbar_arrive_expect_tx(qfull, kQBytes);
          tma_load_3d(sq, &p.q, qfull, 0, qt * kBQ, h);
          tma_load_3d(sq + kBlk, &p.q, qfull, 64, qt * kBQ, h);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      for (int j = 0; j < nblk && ok; ++j, ++J) {
        const int step = j / bps, blk = j - step * bps;
        const int r = (p.rank + step) % p.W;
        const bool local = step == 0;
        if (!local && blk == 0) {
          // consumer_tile_wait on the shard's slice of this head: all its blocks gathered
          ok = warp_wait_signals(p.flags + (static_cast<size_t>(r) * p.heads + h) * bps, bps, c.epoch, c, lane,
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
            mbar_arrive_expect_tx(&kfull[s], kKBytes);
            tma_load_3d(sk + s * kKBytes, km, &kfull[s], 0, y, z);
            tma_load_3d(sk + s * kKBytes + kBlk, km, &kfull[s], 64, y, z);
            filled |= 1u << s;
            par = (par & ~(1u << s)) | (ph << s);
          }
          if (ok) ok = mbar_wait(&vempty[s], ph ^ 1u, c, kSiteEmpty);
          if (ok) {
            mbar_arrive_expect_tx(&vfull[s], kVBytes);
#pragma unroll
            for (int kb = 0; kb < 2; ++kb)
#pragma unroll
              for (int g = 0; g < 2; ++g)
                tma_load_3d(sv + s * kVBytes + kb * kBlk + g * 8192, vm, &vfull[s], g * 64, y + kb * 64, z);
            filled |= 4u << s;
            par = (par & ~(4u << s)) | (ph << (s + 2));
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      }
    }
    if (lane == 0) {  // drain: every fill issued has landed before the CTA exits
      if (kq > 0) mbar_wait(qfull, (kq - 1) & 1, c, kSiteDrain);
      for (int s = 0; s < kStages; ++s) {
        if (filled & (1u << s)) mbar_wait(&kfull[s], (par >> s) & 1u, c, kSiteDrain);
        if (filled & (4u << s)) mbar_wait(&vfull[s], (par >> (s + 2)) & 1u, c, kSiteDrain);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      const uint32_t q0 = smem_u32(sq), p0 = smem_u32(sp);
      const uint32_t to = tmem + 256;
      int J0 = 0, kq = 0;
      for (int it = blockIdx.x; it < nwork && ok; it += gridDim.x, ++kq, J0 += nblk) {
        ok = mbar_wait(qfull, kq & 1, c, kSiteFull);
        tc_fence_after();
        for (int j = 0; j <= nblk && ok; ++j) {
          if (j < nblk) {  // S of block J0 + j
            const int J = J0 + j, s = J & 1;
            const uint32_t ph = (J >> 1) & 1;
            ok = mbar_wait(&sfree[s], ph ^ 1u, c, kSiteTmemEmpty) && mbar_wait(&kfull[s], ph, c, kSiteFull);
            if (!ok) break;
            tc_fence_after();
            attn_mma_s(tmem + s * 128, q0, smem_u32(sk + s * kKBytes));
            umma_commit(&kempty[s]);
            umma_commit(&sfull[s]);
            if (j == nblk - 1) umma_commit(qempty);
          }
          if (j >= 1) {  // O += P V of block J0 + j - 1
            const int I = J0 + j - 1, s = I & 1;
            const uint32_t ph = (I >> 1) & 1;
            ok = mbar_wait(&pready[s], ph, c, kSiteFull) && mbar_wait(&vfull[s], ph, c, kSiteFull);
            if (!ok) break;
            tc_fence_after();
            attn_mma_pv(to, p0 + s * kPBytes, smem_u32(sv + s * kVBytes), j > 1);
            umma_commit(&vempty[s]);
            umma_commit(&pfree[s]);
          }
        }
      }
      umma_commit(drain);
      mbar_wait(drain, 0, c, kSiteDrain);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------ softmax (one row per thread)
    const int qd = warp & 3;               // TMEM lane quadrant of this warp
    const int row = qd * 32 + lane;        // query row inside the tile
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    const float sl2 = p.scale * kLog2e;  // raw score -> base-2 exponent
    bool ok = true;
    int J0 = 0;
    for (int it = blockIdx.x; it < nwork && ok; it += gridDim.x, J0 += nblk) {
      const int h = it / nqt, qt = it - h * nqt;
      float m2 = -INFINITY, l = 0.f;  // running max (base-2 units) and sum of the row
      int blk = -1;                   // block index inside the current shard
      for (int j = 0; j < nblk && ok; ++j) {
        const int J = J0 + j, s = J & 1;
        if (++blk == bps) blk = 0;
        const uint32_t ph = (J >> 1) & 1;
        // The wait results are warp-uniform, as the warp-collective TMEM accesses below need:
        // the converged warp runs each try_wait and timer read as one instruction.
        ok = mbar_wait(&sfull[s], ph, c, kSiteTmemFull);
        if (!ok) break;
        tc_fence_after();
        float x[128];
        {
          uint32_t r[4][32];
#pragma unroll
          for (int cb = 0; cb < 4; ++cb) tmem_ld32_issue(tmem + s * 128 + cb * 32 + lane_off, r[cb]);
          tmem_ld_wait(r[0]);
          tmem_ld_after(r[1]);
          tmem_ld_after(r[2]);
          tmem_ld_after(r[3]);
#pragma unroll
          for (int i = 0; i < 128; ++i) x[i] = __uint_as_float(r[i >> 5][i & 31]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfree[s]);
        if constexpr (Ragged) {
          // keys past the end of a shard (its partial last block, zero-filled by TMA) get no
          // weight: their scores become -inf before the maximum
          const int valid = p.Lr - blk * kBKV;
          if (valid < kBKV) {
#pragma unroll
            for (int i = 0; i < 128; ++i) x[i] = i < valid ? x[i] : -INFINITY;
          }
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = x[i];
#pragma unroll
        for (int i = 8; i < 128; ++i) mx[i & 7] = fmaxf(mx[i & 7], x[i]);
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
          for (int i = 0; i < w; ++i) mx[i] = fmaxf(mx[i], mx[i + w]);
        const float bm2 = mx[0] * sl2;  // the scale is positive: max commutes with it
        if (j == 0) {
          m2 = bm2;  // the item's first P V overwrites O
        } else if (__any_sync(0xffffffffu, bm2 > m2 + kRescaleLog2)) {
          const float mn = fmaxf(m2, bm2);
          const float corr = ex2_approx(m2 - mn);
          // O is stable once the P V of the previous block has completed
          ok = mbar_wait(&pfree[(J - 1) & 1], ((J - 1) >> 1) & 1, c, kSiteTmemFull);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb) {
            float o[32];
            tmem_ld32(tmem + 256 + cb * 32 + lane_off, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= corr;
            tmem_st32(tmem + 256 + cb * 32 + lane_off, o);
          }
          l *= corr;
          m2 = mn;
        }
        const float nm = -m2;
        float sum[8];
        uint32_t pk[64];
#pragma unroll
        for (int i = 0; i < 8; ++i) sum[i] = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const float e0 = ex2_approx(fmaf(x[2 * i], sl2, nm));
          const float e1 = ex2_approx(fmaf(x[2 * i + 1], sl2, nm));
          sum[(2 * i) & 7] += e0;
          sum[(2 * i + 1) & 7] += e1;
          pk[i] = pack_bf16x2(e0, e1);
        }
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
          for (int i = 0; i < w; ++i) sum[i] += sum[i + w];
        l += sum[0];
        // P buffer s was last read by the P V of block J - 2
        ok = mbar_wait(&pfree[s], ph ^ 1u, c, kSiteTmemEmpty);
        if (!ok) break;
        // P (bf16) as the K-major, 128-byte-swizzled A operand: keys [64 kb, 64 kb + 64) of
        // this row are 128 bytes of box kb; 16-byte piece u sits at piece u ^ (row & 7).
        const uint32_t prow = smem_u32(sp) + s * kPBytes + row * 128;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint32_t* v = pk + kb * 32 + u * 4;
            st_shared_v4(prow + kb * kBlk + ((u ^ (row & 7)) << 4), v[0], v[1], v[2], v[3]);
          }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pready[s]);
      }
      const int Jl = J0 + nblk - 1;  // the item's last P V
      if (ok) ok = mbar_wait(&pfree[Jl & 1], (Jl >> 1) & 1, c, kSiteTmemFull);
      tc_fence_after();
      if (ok) {
        // Every lane takes part in the (warp-collective) TMEM loads; rows past the end of
        // the queries (a partial last tile) are only not stored.
        const bool live = !Ragged || qt * kBQ + row < p.Lq;
        const float inv = 1.0f / l;
        uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(h) * p.Lq + qt * kBQ + row) * kD);
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
          float o[32];
          tmem_ld32(tmem + 256 + cb * 32 + lane_off, o);
          if (live) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              dst[cb * 4 + u] = make_uint4(pack_bf16x2(o[8 * u] * inv, o[8 * u + 1] * inv),
                                           pack_bf16x2(o[8 * u + 2] * inv, o[8 * u + 3] * inv),
                                           pack_bf16x2(o[8 * u + 4] * inv, o[8 * u + 5] * inv),
                                           pack_bf16x2(o[8 * u + 6] * inv, o[8 * u + 7] * inv));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ movers
    // Block g of the gather: shard step i = g / (H bps) taken from rank + 1 on (the local
    // shard last), head and key block inside it; K and V of the block, then its signal.
    const int nw = static_cast<int>(gridDim.x) * kMovers;
    const int per_step = p.heads * bps;
    const int total = p.W * per_step;
    for (int g = blockIdx.x * kMovers + (warp - 6); g < total; g += nw) {
      const int i = g / per_step, rem = g - i * per_step;
      const int hh = rem / bps, b = rem - hh * bps;
      const int r = (p.rank + 1 + i) % p.W;
      const size_t rows = static_cast<size_t>(min(kBKV, p.Lr - b * kBKV));  // the last block may be partial
      const size_t row_bytes = static_cast<size_t>(kD) * 2;
      const size_t src = (static_cast<size_t>(hh) * p.Lr + static_cast<size_t>(b) * kBKV) * row_bytes;
      const size_t dst = ((static_cast<size_t>(r) * p.heads + hh) * p.Lr + static_cast<size_t>(b) * kBKV) * row_bytes;
      constexpr size_t kFullVec = static_cast<size_t>(kBKV) * kD * 2 / 16;  // a full block in 16-byte vectors
      if (!Ragged || rows == static_cast<size_t>(kBKV)) {  // full blocks: a compile-time trip count
        copy_chunk(reinterpret_cast<const uint4*>(p.kshard[r] + src), reinterpret_cast<uint4*>(p.kg + dst), kFullVec,
                   lane, 32);
        copy_chunk(reinterpret_cast<const uint4*>(p.vshard[r] + src), reinterpret_cast<uint4*>(p.vg + dst), kFullVec,
                   lane, 32);
      } else {
        copy_chunk(reinterpret_cast<const uint4*>(p.kshard[r] + src), reinterpret_cast<uint4*>(p.kg + dst),
                   rows * row_bytes / 16, lane, 32);
        copy_chunk(reinterpret_cast<const uint4*>(p.vshard[r] + src), reinterpret_cast<uint4*>(p.vg + dst),
                   rows * row_bytes / 16, lane, 32);
      }
      __threadfence();
      __syncwarp();
      if (lane == 0) st_release_gpu(p.flags + (static_cast<size_t>(r) * p.heads + hh) * bps + b, c.epoch);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
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
  const size_t flags = static_cast<size_t>(W) * heads * ((l_r + attn::kBKV - 1) / attn::kBKV) * 8;
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

  // One cooperative CTA per SM: a CTA waiting on a block's signal is co-resident with the
  // mover warps that will set it.
  auto kern = l_r % attn::kBKV == 0 ? attn_kernel<false> : attn_kernel<true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, attn::kSmem) != cudaSuccess) {
    (void)cudaGetLastError();
    return TL_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctx->ctas, 1, 1);
  cfg.blockDim = dim3(attn::kThreads, 1, 1);
  cfg.dynamicSmemBytes = attn::kSmem;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    (void)cudaGetLastError();
    return TL_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return TL_ERR_CUDA;
  }
  return TL_OK;
}
