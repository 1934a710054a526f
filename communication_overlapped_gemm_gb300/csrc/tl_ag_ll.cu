// AllGather + GEMM with the low-latency push gather ("Triton-distributed ...", §3.2
// Algorithm 1, push-mode AllGather, and the low-latency AllGather it describes before
// Algorithm 4: the ready flag travels inside every word of the message, so no separate signal,
// and no fence before it, is needed).  For small problems, where a call is dominated by the
// latency of the remote shard's copy, signal and poll rather than by bandwidth.
//
//   C [(W*m_per_rank) x n] = [A_0; A_1; ...; A_{W-1}] . B        (as tl_ag_gemm)
//
// LL slabs: shard r's element pair (row, 2c..2c+1) travels as one 8-byte word
//   w = (signal << 32) | bf16x2(A_r[row][2c], A_r[row][2c+1])
// at word (r * m_per_rank + row) * k/2 + c of the workspace's LL region, where signal is the
// low 32 bits of the call's epoch (never 0).  An aligned 8-byte access is single-copy atomic,
// so a reader that sees this call's signal in a word also sees that word's data.
//
// One kernel, one CTA per SM at most (a cooperative launch: every CTA that polls is
// co-resident with the CTAs that write):
//   CTAs [0, ntiles)      one 128 x 256 output tile each:
//     warp 0      TMA: B's k-blocks (and A's, for the self rank's rows, read in place);
//     warp 1      TMEM allocation and the MMAs (one elected thread), into 256 TMEM columns;
//     warps 2-23  for a remote row block, read the tile's LL words of up to 4 k-blocks at a
//                 time (one round of the stage ring, every load in flight together), poll the
//                 ones that do not carry this call's signal yet, and write the bf16 pairs into
//                 the stages' A buffers in the MMA's 128-byte-swizzled K-major layout;
//                 then warps 4-7 drain the accumulator (bf16 C, clipped at n and the rows).
//   CTAs [ntiles, grid)   the owners of the remote shards: push every 16-byte piece of each
//                 remote shard as two 16-byte stores of LL words (each word single-copy
//                 atomic, the pair a vector of two).
// Every wait is bounded; on a timeout the call reports TL_ERR_TIMEOUT and all roles still
// finish their protocol (TMA fills drained, MMAs completed) before the CTA exits.
#include "tl_host.h"

namespace tl {

namespace agll {
constexpr int kTileM = 128;
constexpr int kTileN = 256;
constexpr int kStages = 4;
constexpr int kABytes = kTileM * kBK * 2;      // 16 KB: 128 rows x 64 k, SW128 K-major
constexpr int kBBytes = kBK * kTileN * 2;      // 32 KB: 4 boxes of 64 k-rows x 64 n-columns
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kWarps = 24;
constexpr int kThreads = kWarps * 32;
constexpr int kUnpackWarps = kWarps - 2;       // warps 2..23
constexpr int kUnpackThreads = kUnpackWarps * 32;
constexpr int kPieces = kTileM * kBK / 8;      // 16-byte pieces of A per k-block (1024)
// The unpack warps fill all kStages stages of a round at once (their loads in flight together):
constexpr int kPiecesPerThread = (kStages * kPieces + kUnpackThreads - 1) / kUnpackThreads;  // 6
constexpr int kSmem = 1024 + kStages * kStageBytes + 256;
constexpr int kPushUnroll = 4;                 // 16-byte source pieces in flight per pusher
}  // namespace agll

struct AgLLParams {
  CUtensorMap a_local;  // shard `rank`: {k, m_per_rank}, box {64, 128}
  CUtensorMap b;        // {n, k}, box {64, 64}
  Common common;
  const uint8_t* shard[8];
  unsigned long long* ll;  // [W][m_per_rank][k/2]
  __nv_bfloat16* c;        // [W*m_per_rank][n]
  int W, rank, mpr, n, k, mps, nbn, kblocks, ntiles, npush;
};

__device__ __forceinline__ unsigned long long ll_word(uint32_t data, uint32_t sig) {
  return (static_cast<unsigned long long>(sig) << 32) | data;
}

__device__ __forceinline__ void st_volatile_v2_u64(unsigned long long* p, unsigned long long a,
                                                   unsigned long long b) {
  asm volatile("st.volatile.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}

__device__ __forceinline__ void ld_volatile_v2_u64(const unsigned long long* p, unsigned long long& a,
                                                   unsigned long long& b) {
  asm volatile("ld.volatile.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

// The owners of the remote shards: every 16-byte piece e of shard r (row-major, k/8 pieces
// per row) becomes the four LL words 4e .. 4e+3 of shard r's slab.
__device__ __forceinline__ void ll_push(const AgLLParams& p, int pb) {
  using namespace agll;
  const uint32_t sig = static_cast<uint32_t>(p.common.epoch);
  const long long per_shard = static_cast<long long>(p.mpr) * (p.k / 8);
  const long long total = (p.W - 1) * per_shard;
  const long long nthreads = static_cast<long long>(p.npush) * blockDim.x;
  for (long long v0 = static_cast<long long>(pb) * blockDim.x + threadIdx.x; v0 < total;
       v0 += kPushUnroll * nthreads) {
    uint4 d[kPushUnroll];
    int rr[kPushUnroll];
    long long ee[kPushUnroll];
#pragma unroll
    for (int u = 0; u < kPushUnroll; ++u) {
      const long long v = v0 + u * nthreads;
      rr[u] = -1;
      if (v < total) {
        const int i = static_cast<int>(v / per_shard);  // the (i+1)-th shard after the self rank
        ee[u] = v - i * per_shard;
        rr[u] = (p.rank + 1 + i) % p.W;
        d[u] = __ldg(reinterpret_cast<const uint4*>(p.shard[rr[u]]) + ee[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kPushUnroll; ++u) {
      if (rr[u] < 0) continue;
      unsigned long long* dst = p.ll + (static_cast<size_t>(rr[u]) * per_shard + ee[u]) * 4;
      st_volatile_v2_u64(dst, ll_word(d[u].x, sig), ll_word(d[u].y, sig));
      st_volatile_v2_u64(dst + 2, ll_word(d[u].z, sig), ll_word(d[u].w, sig));
    }
  }
}

__global__ void __launch_bounds__(agll::kThreads, 1) ag_ll_kernel(const __grid_constant__ AgLLParams p) {
  using namespace agll;
  if (static_cast<int>(blockIdx.x) >= p.ntiles) {
    ll_push(p, blockIdx.x - p.ntiles);
    return;
  }
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kStages * kStageBytes);
  uint64_t* fullb = bars;                // [kStages] TMA bytes of the stage landed
  uint64_t* fulla = bars + kStages;      // [kStages] every unpack warp wrote its A pieces
  uint64_t* empty = bars + 2 * kStages;  // [kStages] the MMAs of the stage completed
  uint64_t* tfull = bars + 3 * kStages;  // the accumulator is complete
  uint64_t* drain = tfull + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Common& c = p.common;
  const int t = blockIdx.x;
  const int rb = t / p.nbn, cb = t - rb * p.nbn;
  const int src = rb / p.mps;                  // the shard (rank) this row block comes from
  const int row0 = (rb - src * p.mps) * kTileM;  // first row inside that shard
  const bool local = src == p.rank;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&fullb[s], 1);
      mbar_init(&fulla[s], kUnpackWarps);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
    tma_prefetch_map(&p.a_local);
    tma_prefetch_map(&p.b);
  }
  if (warp == 1) {
    tmem_alloc(tslot, kTileN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA
    if (lane == 0) {
      bool ok = true;
      uint32_t filled = 0, par = 0;
      for (int kb = 0; kb < p.kblocks && ok; ++kb) {
        const int s = kb % kStages;
        const uint32_t ph = (kb / kStages) & 1;
        ok = mbar_wait(&empty[s], ph ^ 1u, c, kSiteEmpty);
        if (!ok) break;
        uint8_t* sa = base + s * kStageBytes;
        uint8_t* sb = sa + kABytes;
        mbar_arrive_expect_tx(&fullb[s], local ? kABytes + kBBytes : kBBytes);
        if (local) tma_load_2d(sa, &p.a_local, &fullb[s], kb * kBK, row0);
#pragma unroll
        for (int g = 0; g < kTileN / 64; ++g) tma_load_2d(sb + g * 8192, &p.b, &fullb[s], cb * kTileN + g * 64, kb * kBK);
        filled |= 1u << s;
        par = (par & ~(1u << s)) | (ph << s);
      }
      for (int s = 0; s < kStages; ++s)  // drain: every fill issued has landed
        if (filled & (1u << s)) mbar_wait(&fullb[s], (par >> s) & 1u, c, kSiteDrain);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA
    if (lane == 0) {
      bool ok = true;
      for (int kb = 0; kb < p.kblocks && ok; ++kb) {
        const int s = kb % kStages;
        const uint32_t ph = (kb / kStages) & 1;
        ok = mbar_wait(&fullb[s], ph, c, kSiteFull) && (local || mbar_wait(&fulla[s], ph, c, kSiteFull));
        if (!ok) break;
        tc_fence_after();
        const uint32_t a0 = smem_u32(base + s * kStageBytes);
        mma_stage_256(tmem, a0, a0 + kABytes, kb);
        umma_commit(&empty[s]);
      }
      if (ok) umma_commit(tfull);
      umma_commit(drain);  // every MMA issued has completed before TMEM is freed
      mbar_wait(drain, 0, c, kSiteDrain);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ unpack, then epilogue
    const int ut = threadIdx.x - 64;  // 0 .. kUnpackThreads-1
    bool ok = true;
    if (!local) {
      const uint32_t sig = static_cast<uint32_t>(c.epoch);
      const size_t words_per_row = static_cast<size_t>(p.k) / 2;
      const unsigned long long* slab = p.ll + (static_cast<size_t>(src) * p.mpr + row0) * words_per_row;
      for (int kb0 = 0; kb0 < p.kblocks && ok; kb0 += kStages) {
        // one round: k-blocks kb0 .. kb0 + nkb - 1 in stages 0 .. nkb - 1
        const int nkb = p.kblocks - kb0 < kStages ? p.kblocks - kb0 : kStages;
        const uint32_t ph = (kb0 / kStages) & 1;
        for (int j = 0; j < nkb && ok; ++j) ok = mbar_wait(&empty[j], ph ^ 1u, c, kSiteEmpty);
        if (!ok) break;  // the MMA thread stopped: nothing will consume these stages
        // piece q = ut + i * kUnpackThreads of the round: stage q / kPieces, row (q % kPieces) / 8,
        // 16-byte piece q % 8 of that row's 64 columns
        unsigned long long w[kPiecesPerThread][4];
        bool have[kPiecesPerThread];
#pragma unroll
        for (int i = 0; i < kPiecesPerThread; ++i) {
          const int q = ut + i * kUnpackThreads;
          const int col = (kb0 + q / kPieces) * kBK + (q & 7) * 8;
          have[i] = q < nkb * kPieces && col < p.k;
          if (have[i]) {
            const unsigned long long* src4 = slab + static_cast<size_t>((q % kPieces) >> 3) * words_per_row + col / 2;
            ld_volatile_v2_u64(src4, w[i][0], w[i][1]);
            ld_volatile_v2_u64(src4 + 2, w[i][2], w[i][3]);
          }
        }
        // poll the words that do not carry this call's signal yet
        uint64_t t0 = 0;
        uint32_t n = 0;
        for (;;) {
          bool ready = true;
#pragma unroll
          for (int i = 0; i < kPiecesPerThread; ++i) {
            if (!have[i]) continue;
            if (static_cast<uint32_t>(w[i][0] >> 32) == sig && static_cast<uint32_t>(w[i][1] >> 32) == sig &&
                static_cast<uint32_t>(w[i][2] >> 32) == sig && static_cast<uint32_t>(w[i][3] >> 32) == sig)
              continue;
            ready = false;
            const int q = ut + i * kUnpackThreads;
            const int col = (kb0 + q / kPieces) * kBK + (q & 7) * 8;
            const unsigned long long* src4 = slab + static_cast<size_t>((q % kPieces) >> 3) * words_per_row + col / 2;
            ld_volatile_v2_u64(src4, w[i][0], w[i][1]);
            ld_volatile_v2_u64(src4 + 2, w[i][2], w[i][3]);
          }
          if (ready) break;
          if ((++n & 15u) == 0u) {
            const uint64_t now = globaltimer();
            if (t0 == 0) t0 = now;
            if (now - t0 > c.timeout_ns || aborted(c.status)) {
              report_timeout(c.status, kSiteSignal, (9ull << 60) | (static_cast<unsigned long long>(src) << 32) | rb);
              ok = false;
              break;
            }
          }
        }
        // A (K-major, 128-byte swizzle): row r's 16-byte piece j sits at r * 128 + (j ^ (r & 7)) * 16
#pragma unroll
        for (int i = 0; i < kPiecesPerThread; ++i) {
          const int q = ut + i * kUnpackThreads;
          if (q >= nkb * kPieces) continue;
          const int r = (q % kPieces) >> 3, j = q & 7;
          const uint32_t addr = smem_u32(base + (q / kPieces) * kStageBytes) + r * 128 + ((j ^ (r & 7)) << 4);
          if (have[i])
            st_shared_v4(addr, static_cast<uint32_t>(w[i][0]), static_cast<uint32_t>(w[i][1]),
                         static_cast<uint32_t>(w[i][2]), static_cast<uint32_t>(w[i][3]));
          else
            st_shared_v4(addr, 0u, 0u, 0u, 0u);  // columns past k
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
          for (int j = 0; j < nkb; ++j) mbar_arrive(&fulla[j]);
      }
    }
    if (warp >= 4 && warp < 8) {
      // epilogue: TMEM lane quadrant q = warp - 4 holds rows 32q .. 32q+31 of the tile
      const int qd = warp - 4;
      const bool acc_ok = __all_sync(0xffffffffu, mbar_wait(tfull, 0, c, kSiteTmemFull));
      tc_fence_after();
      if (acc_ok) {
        const int row = rb * kTileM + qd * 32 + lane;  // row of C (the row block is whole: m_per_rank % 128 == 0)
        __nv_bfloat16* crow = p.c + static_cast<size_t>(row) * p.n;
#pragma unroll 1
        for (int cc = 0; cc < kTileN / 32; ++cc) {
          float v[32];
          tmem_ld32(tmem + cc * 32 + (static_cast<uint32_t>(qd * 32) << 16), v);
          const int col0 = cb * kTileN + cc * 32;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (col0 + u * 8 + 8 > p.n) break;  // n % 8 == 0: 16-byte pieces are whole or absent
            *reinterpret_cast<uint4*>(crow + col0 + u * 8) =
                make_uint4(pack_bf16x2(v[8 * u], v[8 * u + 1]), pack_bf16x2(v[8 * u + 2], v[8 * u + 3]),
                           pack_bf16x2(v[8 * u + 4], v[8 * u + 5]), pack_bf16x2(v[8 * u + 6], v[8 * u + 7]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTileN);
  }
}

int ag_ll_tiles(int W, int m_per_rank, int n) {
  return W * (m_per_rank / agll::kTileM) * ((n + agll::kTileN - 1) / agll::kTileN);
}

int ag_ll_capable(const tl_ctx* ctx, int W, int m_per_rank, int n, int k) {
  if (W < 2 || m_per_rank % agll::kTileM != 0 || n % 8 != 0 || k % 8 != 0) return 0;
  if (ag_layout(W, m_per_rank, k).ll_bytes == 0) return 0;
  return ag_ll_tiles(W, m_per_rank, n) + 1 <= ctx->ctas ? 1 : 0;
}

int ag_ll_launch(tl_ctx* ctx, int W, int rank, const void* const* a_shards, const void* b, void* c, uint8_t* ws,
                 int m_per_rank, int n, int k, cudaStream_t stream) {
  using namespace agll;
  if (!ag_ll_capable(ctx, W, m_per_rank, n, k)) return TL_ERR_UNSUPPORTED;
  const AgLayout L = ag_layout(W, m_per_rank, k);
  AgLLParams p;
  std::memset(&p, 0, sizeof(p));
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!tmap_2d(&p.a_local, BF, 2, a_shards[rank], k, m_per_rank, 64, kTileM) || !tmap_2d(&p.b, BF, 2, b, n, k, 64, 64))
    return TL_ERR_CUDA;
  p.common = make_common(ctx);
  p.common.trace_hdr = nullptr;  // no trace spans in this kernel
  p.common.trace = nullptr;
  for (int r = 0; r < W; ++r) p.shard[r] = static_cast<const uint8_t*>(a_shards[r]);
  p.ll = reinterpret_cast<unsigned long long*>(ws + L.ll_off);
  p.c = static_cast<__nv_bfloat16*>(c);
  p.W = W;
  p.rank = rank;
  p.mpr = m_per_rank;
  p.n = n;
  p.k = k;
  p.mps = m_per_rank / kTileM;
  p.nbn = (n + kTileN - 1) / kTileN;
  p.kblocks = (k + kBK - 1) / kBK;
  p.ntiles = ag_ll_tiles(W, m_per_rank, n);
  // pushers: one 16-byte piece per thread where the CTAs left allow it
  const long long pieces = static_cast<long long>(W - 1) * m_per_rank * (k / 8);
  long long want = (pieces + kThreads - 1) / kThreads;
  if (want < 1) want = 1;
  if (want > ctx->ctas - p.ntiles) want = ctx->ctas - p.ntiles;
  p.npush = static_cast<int>(want);

  if (cudaFuncSetAttribute(ag_ll_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess) {
    (void)cudaGetLastError();
    return TL_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.ntiles + p.npush, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, ag_ll_kernel, p);
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

}  // namespace tl

extern "C" int tl_ag_gemm_ll_capable(const tl_ctx* ctx, int W, int m_per_rank, int n, int k) {
  if (!ctx || W < 1 || W > 8 || m_per_rank < 0 || n < 0 || k < 0) return 0;
  return tl::ag_ll_capable(ctx, W, m_per_rank, n, k);
}
