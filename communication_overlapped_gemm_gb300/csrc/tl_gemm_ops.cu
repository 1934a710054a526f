// AllGather+GEMM, GEMM+ReduceScatter and the CTA-chained 2-layer MLP on the
// persistent tcgen05 engine, plus their C-ABI entry points.
#include <cuda_bf16.h>

#include "tl_engine2.cuh"
#include "tl_host.h"

namespace tl {

// ============================================================================ shared op pieces

// A 2-D TMA tile load: plain (single CTA) or, in a CTA pair, completing on the leader's
// barrier at the same shared offset as `bar`.
template <bool Pair>
__device__ __forceinline__ void load_tile(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y) {
  if constexpr (Pair)
    tma_load_2d_pair(dst, m, mapa_shared(smem_u32(bar), 0), x, y);
  else
    tma_load_2d(dst, m, bar, x, y);
}

// Wait for the `chunks` mover signals of one slab.
__device__ __forceinline__ void wait_slab(const uint64_t* flags, int chunks, const Common& c, int lane,
                                          unsigned long long info) {
  warp_wait_signals(flags, chunks, c.epoch, c, lane, kSiteSignal, info);
}

// Pull one chunk of a shard into the gathered buffer and release its signal
// (tile_pull_data + producer notify of "TileLink ...", §3.2; pull-mode AllGather of
// "Triton-distributed ...", §3.2 Algorithm 2, with the chunk as the communication tile).
// `bar` is the named barrier of the `nthreads` threads that copy together.
__device__ __forceinline__ void mover_chunk(const uint8_t* src, uint8_t* dst, size_t bytes, uint64_t* flag,
                                            bool signal, const Common& c, int tid, int nthreads, int bar = 2) {
  copy_chunk(reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), bytes / 16, tid, nthreads);
  __threadfence();
  named_bar_sync(bar, nthreads);
  if (tid == 0 && signal) st_release_gpu(flag, c.epoch);
}

// Exact-form GELU, 0.5 x (1 + erf(x / sqrt 2)), with erf from Abramowitz & Stegun,
// "Handbook of Mathematical Functions", formula 7.1.26 (|error| <= 1.5e-7 for x >= 0, odd
// extension for x < 0), evaluated with the fast exp and divide intrinsics: far below the
// bf16 rounding of H and cheaper than the IEEE erff in the layer-1 epilogue.
__device__ __forceinline__ float gelu_erf(float x) {
  const float z = fabsf(x) * 0.70710678118654752f;
  const float t = __fdividef(1.0f, 1.0f + 0.3275911f * z);
  const float poly = t * (0.254829592f + t * (-0.284496736f + t * (1.421413741f + t * (-1.453152027f + t * 1.061405429f))));
  const float e = 1.0f - poly * __expf(-z * z);
  return 0.5f * x * (1.0f + copysignf(e, x));
}

// One step of a GEMM+RS summation chain, on a BM x 256 partial tile held in TMEM (rows
// 128h..128h+127 of the tile are TMEM columns [256h, 256h+256)).  The chain of an output tile
// has W steps, pos = 0..W-1; step pos > 0 first waits for step pos-1's signal on the tile
// (peer_tile_wait).  Then:
//   - a non-final step writes its fp32 result to st_map at rows st_row..: a TMA store, or
//     with `reduce` a TMA bulk reduce-add (the owner-slot chain's middle steps);
//   - with `prev`, the step first adds the running partial at prev (row-major, stride n,
//     the tile's first row) in registers (a ring hop, or the slot chain's final step);
//   - the final step writes bf16 rows of `out_map` at orow.
// The fp32 order of every output element is therefore fixed by the chain order.
template <int BM>
__device__ __forceinline__ void rs_epilogue(const CUtensorMap* st_map, int st_row, bool reduce, const float* prev,
                                            const CUtensorMap* out_map, int orow, const uint64_t* flag, int pos,
                                            int W, int n0, int n, const Common& c, uint32_t taddr, int q, int lane,
                                            EpiStage& es, int h0, int h1, unsigned long long info) {
  const bool last = pos == W - 1;
  if (pos > 0) warp_wait_one(flag, (c.epoch << 4) | static_cast<unsigned long long>(pos), c, lane, kSitePeer, info);
#pragma unroll 1
  for (int h = h0; h < h1; ++h) {
    const uint32_t th = taddr + h * 256;
    const int r = h * 128 + q * 32;  // this warp's first row inside the tile
    const float* src_row = prev ? prev + static_cast<size_t>(r + lane) * n : nullptr;
    if (!last) {
#pragma unroll 1
      for (int ch = 0; ch < kBN / 32; ++ch) {
        const int x = n0 + ch * 32;
        if (x >= n) break;
        float v[32];
        tmem_ld32(th + ch * 32, v);
        if (prev) {
          const float* src = src_row + x;
          if (x + 32 <= n) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 s4 = __ldcg(reinterpret_cast<const float4*>(src) + i);
              v[4 * i] += s4.x;
              v[4 * i + 1] += s4.y;
              v[4 * i + 2] += s4.z;
              v[4 * i + 3] += s4.w;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (x + i < n) v[i] += __ldcg(src + i);
          }
        }
        store_f32_chunk(st_map, es, lane, v, x, st_row + r, reduce);
      }
    } else {
#pragma unroll 1
      for (int ch = 0; ch < kBN / 64; ++ch) {
        const int x = n0 + ch * 64;
        if (x >= n) break;
        float v[64];
        tmem_ld64(th, ch * 64, v);
        if (prev) {
          const float* src = src_row + x;
          if (x + 64 <= n) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float4 s4 = __ldcg(reinterpret_cast<const float4*>(src) + i);
              v[4 * i] += s4.x;
              v[4 * i + 1] += s4.y;
              v[4 * i + 2] += s4.z;
              v[4 * i + 3] += s4.w;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 64; ++i)
              if (x + i < n) v[i] += __ldcg(src + i);
          }
        }
        store_bf16_chunk(out_map, es, lane, v, x, orow + r);
      }
    }
  }
}

// ============================================================================ AllGather + GEMM
struct AgParams {
  CUtensorMap a_local;  // shard `rank` read in place: {k, m_per_rank}, box {64, BM}
  CUtensorMap a_gath;   // gathered buffer T: {k, W*m_per_rank}, box {64, BM}
  CUtensorMap b;        // {n, k}, box {64, 64}
  CUtensorMap c;        // {n, W*m_per_rank}, box {64, 32}
  Common common;
  const uint8_t* shard[8];
  uint8_t* gath;
  uint64_t* flags;  // [W][spr][chunks]
  long long shard_bytes, slab_bytes;
  int W, rank, m_per_rank, mps, spr, n, k, nbk, kblocks, swizzle, chunks, skip_chunk;
  int boost;      // chunks [0, boost) are split with the epilogue warps (see ag_mover)
  int copy_self;  // 1: the self rank's shard is copied too (last); 0: only the W-1 remote shards
  int quarters;   // K parts of a slab (1..4); a slab's chunks are cpq row pieces of each part
  int cpq;        // chunks per K part (chunks = quarters * cpq)
  int qcols;      // columns per K part (a multiple of 64; the last part may be shorter or empty)
  int kb_q;       // 64-column k-blocks per K part (qcols / 64)
  int head;       // shards at the head of the mover order, copied K part first together
};

// Offsets (bytes) of the 16-byte vectors v = tid + u * nthreads, u = 0..7, of a block of rows
// with `vr` vectors per row and a row stride of `stride` bytes, stepped from (row, col)
// without a division per vector (the movers share the SM's issue slots with the GEMM roles).
struct RowWalk {
  int row, col, drow, dcol, vr;
  size_t stride;
  __device__ __forceinline__ RowWalk(int v0, int nthreads, int vr_, size_t stride_) : vr(vr_), stride(stride_) {
    row = v0 / vr;
    col = v0 - row * vr;
    drow = nthreads / vr;
    dcol = nthreads - drow * vr;
  }
  __device__ __forceinline__ size_t offset() const { return static_cast<size_t>(row) * stride + col * 16; }
  __device__ __forceinline__ void step() {
    row += drow;
    col += dcol;
    if (col >= vr) {
      col -= vr;
      ++row;
    }
  }
};

// Copy `rows` rows of `row_bytes` bytes (a multiple of 16) from src to each of the `ndst`
// destinations, all with a row stride of `stride` bytes, by `nthreads` threads: 16-byte
// vectors, 8 loads in flight, each vector loaded once and stored ndst times (the push of one
// source chunk to every peer).  Whole rows (row_bytes == stride) are one contiguous block.
__device__ __forceinline__ void copy_rows_multi(const uint8_t* __restrict__ src, uint8_t* const (&dst)[8], int ndst,
                                                size_t stride, int rows, int row_bytes, int tid, int nthreads) {
  int vr = row_bytes / 16;
  int nr = rows;
  if (static_cast<size_t>(row_bytes) == stride) {  // contiguous: one row of rows * vr vectors
    vr *= rows;
    nr = 1;
  }
  const int nvec = nr * vr;
  if (nvec == 0) return;
  constexpr int U = 8;
  RowWalk w(tid, nthreads, vr, stride);
  for (int i = tid; i < nvec; i += U * nthreads) {
    uint4 r[U];
    size_t off[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      off[u] = w.offset();
      w.step();
      if (i + u * nthreads < nvec) r[u] = __ldg(reinterpret_cast<const uint4*>(src + off[u]));
    }
#pragma unroll 1
    for (int d = 0; d < ndst; ++d) {
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (i + u * nthreads < nvec) *reinterpret_cast<uint4*>(dst[d] + off[u]) = r[u];
    }
  }
}

// A contiguous block of nvec 16-byte vectors, 8 loads in flight per thread.
__device__ __forceinline__ void copy_contig(const uint4* __restrict__ s4, uint4* __restrict__ d4, int nvec, int tid,
                                            int nthreads) {
  constexpr int U = 8;
  for (int i = tid; i < nvec; i += U * nthreads) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i + u * nthreads < nvec) r[u] = __ldg(s4 + i + u * nthreads);
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i + u * nthreads < nvec) d4[i + u * nthreads] = r[u];
  }
}

// One destination: the same vectors, with the store offsets walked again rather than kept
// in registers.
__device__ __forceinline__ void copy_rows(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, size_t stride,
                                          int rows, int row_bytes, int tid, int nthreads) {
  constexpr int U = 8;
  if (static_cast<size_t>(row_bytes) == stride) {
    copy_contig(reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), rows * (row_bytes / 16), tid,
                nthreads);
    return;
  }
  const int vr = row_bytes / 16;
  const int nvec = rows * vr;
  RowWalk wl(tid, nthreads, vr, stride);
  RowWalk wst = wl;
  for (int i = tid; i < nvec; i += U * nthreads) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (i + u * nthreads < nvec) r[u] = __ldg(reinterpret_cast<const uint4*>(src + wl.offset()));
      wl.step();
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (i + u * nthreads < nvec) *reinterpret_cast<uint4*>(dst + wst.offset()) = r[u];
      wst.step();
    }
  }
}

// Position of chunk g of one gather (see ag_copy): shard i of the mover's order, K part q,
// slab, row piece.  The first `head` shards go K part first together, the others one by one,
// each K part first as well.
struct ChunkPos {
  int i, q, slab, piece;
};
__device__ __forceinline__ ChunkPos chunk_pos(int g, int head, int spr, int chunks, int cpq) {
  const int per_shard = spr * chunks;
  const int head_chunks = head * per_shard;
  const bool in_head = g < head_chunks;
  const int grp0 = in_head ? 0 : head + (g - head_chunks) / per_shard;  // first shard of the group
  const int gsz = in_head ? head : 1;
  int rem = in_head ? g : (g - head_chunks) % per_shard;
  ChunkPos c;
  c.q = rem / (gsz * spr * cpq);
  rem -= c.q * gsz * spr * cpq;
  c.i = grp0 + rem / (spr * cpq);
  rem -= (c.i - grp0) * spr * cpq;
  c.slab = rem / cpq;
  c.piece = rem - c.slab * cpq;
  return c;
}

// The shard mover: pull the remote shards (and, with copy_self, the self rank's own, last)
// into the gathered buffer, one release signal per chunk.  A 128-row slab is cut along K into
// `quarters` parts of qcols columns, and each part into cpq pieces of 128/cpq rows: a chunk
// is one piece of one part.  Order: the first `head` shards of the mover's order (those the
// first wave of tiles reads) go K part first, part 0 of all their slabs, then part 1, ..., so
// those tiles start once part 0 of their rows has landed and later parts arrive ahead of
// their k-blocks (a tile waits for part q before its k-block q * kb_q); the later shards
// follow one after another, each K part first as well.  Chunk g belongs to CTA g mod grid.
// With `boost`, the epilogue warps, idle until their first tile, join the mover warps on the
// head: the two groups copy each head chunk together (named barrier 4 over both), so part 0
// lands first and in the least time; the mover warps then copy the rest alone.
template <bool Trace>
__device__ __forceinline__ void ag_chunk(const AgParams& p, int g, int tid, int nthreads, int bar) {
  const ChunkPos cp = chunk_pos(g, p.head, p.spr, p.chunks, p.cpq);
  const int r = ag_mover_rank(p.W, p.rank, p.swizzle, cp.i);
  const int c0 = cp.q * p.qcols;
  const int cols = c0 >= p.k ? 0 : (p.k - c0 < p.qcols ? p.k - c0 : p.qcols);
  const int piece_rows = tl::kBM / p.cpq;
  const size_t row_stride = static_cast<size_t>(p.k) * 2;
  const size_t off = (static_cast<size_t>(cp.slab) * tl::kBM + static_cast<size_t>(cp.piece) * piece_rows) * row_stride +
                     static_cast<size_t>(c0) * 2;
  const uint64_t t0 = Trace ? globaltimer() : 0;
  copy_rows(p.shard[r] + off, p.gath + static_cast<size_t>(r) * p.shard_bytes + off, row_stride, piece_rows, cols * 2,
            tid, nthreads);
  __threadfence();
  named_bar_sync(bar, nthreads);
  if (tid == 0 && g != p.skip_chunk)
    st_release_gpu(p.flags + (static_cast<size_t>(r) * p.spr + cp.slab) * p.chunks + cp.q * p.cpq + cp.piece,
                   p.common.epoch);
  if (Trace && tid == 0) trace_span(p.common, kTrMoverChunk, g, t0, globaltimer());
}

// group 0: the mover warps (tid < movers * 32); group 1: the epilogue warps (boost only).
template <bool Trace>
__device__ __forceinline__ void ag_copy(const AgParams& p, int tid, int nthreads, int group, int epi_threads) {
  const int total = (p.W - 1 + p.copy_self) * p.spr * p.chunks;
  int g = blockIdx.x;
  if (p.boost > 0) {
    const int both = nthreads + epi_threads;  // mover + epilogue threads of this CTA
    const int t = group == 0 ? tid : nthreads + tid;
    for (; g < p.boost; g += gridDim.x) ag_chunk<Trace>(p, g, t, both, 4);
    if (group == 1) return;
  }
  for (; g < total; g += gridDim.x) ag_chunk<Trace>(p, g, tid, nthreads, 2);
}

template <bool Trace>
__device__ __forceinline__ void ag_mover(const AgParams& p, int mw, int lane, int epi_threads) {
  ag_copy<Trace>(p, mw * 32 + lane, p.common.mover_warps * 32, 0, epi_threads);
}

// Pair = true: 256-row tiles on a CTA pair (tl_engine2.cuh); this CTA owns rows and B
// columns [128 rank, 128 rank + 128) of the tile.
template <int BM, bool Pair = false>
struct AgOp : OpBase<AgParams> {
  using Params = AgParams;
  static constexpr int kBM = BM;
  // bf16 epilogue; the single-CTA 256-row tile has one accumulator, so its epilogue stalls the
  // next tile's MMAs: 8 warps (one warpgroup per 128-row half) drain it twice as fast.
  static constexpr int kEpiWarps = (BM == 256 && !Pair) ? 8 : 4;
  static constexpr int kMaxMovers = 4;
  static constexpr uint32_t kTxBytes = Pair ? Geo2::kStageBytes : Geo<BM>::kStageBytes;
  static __device__ int num_tiles(const Params& p) { return ag_num_tiles(p.W, p.mps, p.nbk); }
  static __device__ Job job(const Params& p, int t) {
    const AgTile a = ag_tile(t, p.W, p.rank, p.mps, p.nbk, p.swizzle);
    Job j;
    j.kind = 0;
    j.a_sel = a.src == p.rank ? 0 : 1;
    j.a_row = (a.src == p.rank ? 0 : a.src * p.m_per_rank) + a.mb * BM;
    j.b_sel = 0;
    j.b_col = a.nb * kBN;
    j.b_z = 0;
    j.kblocks = p.kblocks;
    j.x0 = a.src;
    j.x1 = a.mb;
    j.x2 = a.src * p.m_per_rank + a.mb * BM;  // row of C
    j.x3 = 0;
    return j;
  }
  static __device__ void prefetch(const Params& p) {
    tma_prefetch_map(&p.a_local);
    tma_prefetch_map(&p.a_gath);
    tma_prefetch_map(&p.b);
    tma_prefetch_map(&p.c);
  }
  // consumer_tile_wait: the k-blocks of K part q of a remote row block are read only after
  // the part's chunks of its BM/128 slabs (this CTA's slab, on a pair) have been released.
  static __device__ void wait_deps(const Params& p, const Job& j, int kb, int lane) {
    // K part q of a gathered row block before its first k-block (at most 4 parts; no division
    // here: the producer warp's per-k-block work is on the pipeline's critical path)
    if (j.a_sel == 0 || (kb != 0 && kb != p.kb_q && kb != 2 * p.kb_q && kb != 3 * p.kb_q)) return;
    const int q = kb == 0 ? 0 : kb == p.kb_q ? 1 : kb == 2 * p.kb_q ? 2 : 3;
    constexpr int kSlabs = Pair ? 1 : BM / 128;  // 128-row slabs this CTA reads
    const int slab0 = j.x1 * (BM / 128) + (Pair ? j.rank : 0);
#pragma unroll
    for (int sl = 0; sl < kSlabs; ++sl) {
      const uint64_t* f = p.flags + (static_cast<size_t>(j.x0) * p.spr + slab0 + sl) * p.chunks + q * p.cpq;
      wait_slab(f, p.cpq, p.common, lane, (static_cast<unsigned long long>(j.x0) << 32) | (j.x1 << 4) | q);
    }
  }
  static __device__ void load(const Params& p, const Job& j, int kb, uint8_t* sa, uint8_t* sb, uint64_t* bar) {
    const int r0 = Pair ? 128 * j.rank : 0;
    load_tile<Pair>(sa, j.a_sel ? &p.a_gath : &p.a_local, bar, kb * kBK, j.a_row + r0);
#pragma unroll
    for (int g = 0; g < (Pair ? 2 : kBN / 64); ++g)
      load_tile<Pair>(sb + g * 8192, &p.b, bar, j.b_col + r0 + g * 64, kb * kBK);
  }
  static __device__ void mma_stage(const Job&, uint32_t d, uint32_t a0, uint32_t b0, int kb) {
    mma_stage_bm<BM>(d, a0, b0, kb);
  }
  static __device__ void epilogue(const Params& p, const Job& j, uint32_t taddr, int q, int lane, EpiStage& es,
                                 int h0, int h1) {
#pragma unroll 1
    for (int h = h0; h < h1; ++h) {
#pragma unroll 1
      for (int ch = 0; ch < kBN / 64; ++ch) {
        const int x = j.b_col + ch * 64;
        if (x >= p.n) break;
        float v[64];
        tmem_ld64(taddr + h * 256, ch * 64, v);
        store_bf16_chunk(&p.c, es, lane, v, x, j.x2 + h * 128 + q * 32);
      }
    }
  }
  template <bool Trace>
  static __device__ void mover(const Params& p, int mw, int lane) {
    ag_mover<Trace>(p, mw, lane, kEpiWarps * 32);
  }
  template <bool Trace>
  static __device__ void epilogue_prologue(const Params& p, int ew, int lane) {
    if (p.boost > 0) ag_copy<Trace>(p, ew * 32 + lane, p.common.mover_warps * 32, 1, kEpiWarps * 32);
  }
};

// ============================================================================ GEMM + ReduceScatter
struct RsParams {
  CUtensorMap a[8];    // A_p: {k_r, m}, box {64, BM}
  CUtensorMap b[8];    // B_p: {n, k_r}, box {64, 64}
  CUtensorMap out[8];  // out_o: {n, m/W}, box {64, 32}
  CUtensorMap acc;     // owner-slot chain: the fp32 slot {n, m}; ring: the W receive buffers
                       // {n, W*m} (rank q's at rows q*m ..); box {32, 32}
  Common common;
  const float* acc_ptr;
  uint64_t* flags;  // [m/128][nbk] (a tile uses the signal of its first 128-row block)
  int W, m, mo, mbo, n, nbk, kblocks, swizzle, ring;
};

template <int BM, bool Pair = false>
struct RsOp : OpBase<RsParams> {
  using Params = RsParams;
  static constexpr int kBM = BM;
  // fp32 reduction epilogue of a whole tile: 8 warps when the single-CTA 256-row tile has
  // one TMEM accumulator; the pair keeps two, so 4 suffice.
  static constexpr int kEpiWarps = (BM == 256 && !Pair) ? 8 : 4;
  static constexpr int kMaxMovers = 0;
  static constexpr uint32_t kTxBytes = Pair ? Geo2::kStageBytes : Geo<BM>::kStageBytes;
  static __device__ int num_tiles(const Params& p) { return rs_num_tiles(p.W, p.mbo, p.nbk); }
  static __device__ Job job(const Params& p, int t) {
    const RsTile r = p.ring ? rs_ring_tile(t, p.W, p.mbo, p.nbk, BM) : rs_tile(t, p.W, p.mbo, p.nbk, BM, p.swizzle);
    Job j;
    j.kind = r.s;  // position in the tile's summation chain
    j.a_sel = r.p;
    j.a_row = r.o * p.mo + r.mb * BM;
    j.b_sel = r.p;
    j.b_col = r.nb * kBN;
    j.b_z = 0;
    j.kblocks = p.kblocks;
    j.x0 = r.p;
    j.x1 = r.o;
    j.x2 = r.mb;
    j.x3 = r.nb;
    return j;
  }
  static __device__ void prefetch(const Params& p) { tma_prefetch_map(&p.acc); }
  static __device__ void wait_deps(const Params&, const Job&, int, int) {}
  static __device__ void load(const Params& p, const Job& j, int kb, uint8_t* sa, uint8_t* sb, uint64_t* bar) {
    const int r0 = Pair ? 128 * j.rank : 0;
    load_tile<Pair>(sa, &p.a[j.a_sel], bar, kb * kBK, j.a_row + r0);
#pragma unroll
    for (int g = 0; g < (Pair ? 2 : kBN / 64); ++g)
      load_tile<Pair>(sb + g * 8192, &p.b[j.b_sel], bar, j.b_col + r0 + g * 64, kb * kBK);
  }
  static __device__ void mma_stage(const Job&, uint32_t d, uint32_t a0, uint32_t b0, int kb) {
    mma_stage_bm<BM>(d, a0, b0, kb);
  }
  // signal of the first 128-row block this CTA writes (each CTA of a pair owns one block)
  static __device__ int tile_id(const Params& p, const Job& j) {
    return (j.a_row / 128 + (Pair ? j.rank : 0)) * p.nbk + j.x3;
  }
  // Owner-slot chain: step p stores (p = 0) or TMA-adds (0 < p < W-1) its partial into the
  // owner's slot, the last producer adds the slot in registers and writes bf16.  Ring: hop s
  // (producer q) adds the running partial in its own receive buffer (s > 0) and stores the sum
  // into rank q+1's receive buffer, the owner (last hop) writes bf16.
  static __device__ void epilogue(const Params& p, const Job& j, uint32_t taddr, int q, int lane, EpiStage& es,
                                 int h0, int h1) {
    const int pos = j.kind, grow = j.a_row;
    const unsigned long long info = static_cast<unsigned long long>(grow) << 20 | static_cast<unsigned>(j.b_col);
    const uint64_t* flag = p.flags + tile_id(p, j);
    if (p.ring) {
      const int next = (j.x0 + 1) % p.W;
      const float* prev = pos > 0 ? p.acc_ptr + (static_cast<size_t>(j.x0) * p.m + grow) * p.n : nullptr;
      rs_epilogue<BM>(&p.acc, next * p.m + grow, false, prev, &p.out[j.x1], j.x2 * BM, flag, pos, p.W, j.b_col, p.n,
                      p.common, taddr, q, lane, es, h0, h1, info);
    } else {
      const float* prev = (pos > 0 && pos == p.W - 1) ? p.acc_ptr + static_cast<size_t>(grow) * p.n : nullptr;
      rs_epilogue<BM>(&p.acc, grow, pos > 0, prev, &p.out[j.x1], j.x2 * BM, flag, pos, p.W, j.b_col, p.n, p.common,
                      taddr, q, lane, es, h0, h1, info);
    }
  }
  // peer_tile_notify: step pos of this tile's chain is complete.
  static __device__ bool publishes(const Params& p, const Job& j) { return j.kind != p.W - 1; }
  static __device__ void publish(const Params& p, const Job& j) {
    st_release_gpu(p.flags + tile_id(p, j), (p.common.epoch << 4) | static_cast<unsigned long long>(j.kind + 1));
  }
};

// ============================================================================ 2-layer MLP chain
struct Mlp2Params {
  CUtensorMap x_local[8];  // X_r in place: {h, Tr}, box {64, BM}
  CUtensorMap w1[8];       // {f, h}, box {64, 64}
  CUtensorMap w2[8];       // {h, f}, box {64, 64}
  CUtensorMap out[8];      // {h, Tr}, box {64, 32}
  CUtensorMap x_gath;      // per-rank gathered X: {h, W*T}, box {64, BM}
  CUtensorMap h_st;        // H: {f, W*T}, box {64, 32}
  CUtensorMap h_ld;        // H: {f, W*T}, box {64, BM}
  CUtensorMap acc;         // fp32 slot {h, T}, box {32, 32}
  Common common;
  const uint8_t* x[8];
  uint8_t* xg;
  const float* acc_ptr;
  uint64_t* ag_flags;  // [W gathering rank][W src][spr][chunks]
  uint64_t* h_flags;   // [W][T/128][nb1]
  uint64_t* rs_flags;  // [T/128][nb2]
  long long shard_bytes, slab_bytes;
  int W, T, Tr, h, f, mps, spr, nb1, kb1, nb2, kb2, swizzle, chunks, skip_chunk;
  int push;  // 1: each shard is read once and pushed to the W-1 other ranks' copies; 0: pull
};

template <int BM, bool Pair = false>
struct Mlp2Op : OpBase<Mlp2Params> {
  using Params = Mlp2Params;
  static constexpr int kBM = BM;
  static constexpr int kSub = BM / 128;             // 128-row blocks per tile
  static constexpr int kOwn = Pair ? 1 : BM / 128;  // 128-row blocks this CTA reads / writes
  static constexpr int kEpiWarps = (BM == 256 && !Pair) ? 8 : 4;  // erf-GELU and fp32 reduction epilogues
  static constexpr int kMaxMovers = (BM == 256 && !Pair) ? 2 : 4;
  static constexpr uint32_t kTxBytes = Pair ? Geo2::kStageBytes : Geo<BM>::kStageBytes;
  static __device__ int per_rank(const Params& p) { return p.W * p.mps * (p.nb1 + p.nb2); }
  static __device__ int num_tiles(const Params& p) { return p.W * per_rank(p); }
  // kind 1: layer-1 tile of rank x0 on shard x1, row block x2, column block x3
  // kind 2: layer-2 tile of producer x0 for owner x1, row block x2, column block x3
  static __device__ Job job(const Params& p, int t) {
    const int pr = per_rank(p);
    const int r = t / pr;
    const int u = t - r * pr;
    const int n1 = p.W * p.mps * p.nb1;
    Job j;
    j.b_z = 0;
    if (u < n1) {
      const AgTile a = ag_tile(u, p.W, r, p.mps, p.nb1, p.swizzle);
      j.kind = 1;
      j.a_sel = a.src == r ? 0 : 1;
      j.a_row = a.src == r ? a.mb * BM : r * p.T + a.src * p.Tr + a.mb * BM;
      j.b_sel = r;
      j.b_col = a.nb * kBN;
      j.kblocks = p.kb1;
      j.x0 = r;
      j.x1 = a.src;
      j.x2 = a.mb;
      j.x3 = a.nb;
    } else {
      // this rank is the producer; it walks owners (r + 1 + step) mod W
      const int per_owner = p.mps * p.nb2;
      const int v = u - n1;
      const int step = v / per_owner;
      const int w = v - step * per_owner;
      j.kind = 2;
      j.x0 = r;
      j.x1 = rs_owner(p.W, r, step, p.swizzle);
      j.x2 = w / p.nb2;
      j.x3 = w - j.x2 * p.nb2;
      j.a_sel = 0;
      j.a_row = r * p.T + j.x1 * p.Tr + j.x2 * BM;
      j.b_sel = r;
      j.b_col = j.x3 * kBN;
      j.kblocks = p.kb2;
    }
    return j;
  }
  static __device__ void prefetch(const Params& p) {
    tma_prefetch_map(&p.x_gath);
    tma_prefetch_map(&p.h_st);
    tma_prefetch_map(&p.h_ld);
    tma_prefetch_map(&p.acc);
  }
  // first 128-row block (of T) this CTA covers
  static __device__ int row_block(const Params& p, const Job& j) {
    return (j.x1 * p.Tr) / 128 + j.x2 * kSub + (Pair ? j.rank : 0);
  }
  // Once per tile, before its first k-block: the gathered slabs a layer-1 tile reads, or the
  // layer-1 tiles of the row block a layer-2 tile reads.  (The chain's gather is not cut
  // along K: per-part waits measured slower here, as most layer-1 tiles read remote rows.)
  static __device__ void wait_deps(const Params& p, const Job& j, int kb, int lane) {
    if (kb != 0) return;
    if (j.kind == 1) {
      if (j.a_sel == 0) return;
      const uint64_t* f = p.ag_flags +
                          ((static_cast<size_t>(j.x0) * p.W + j.x1) * p.spr + j.x2 * kSub + (Pair ? j.rank : 0)) *
                              p.chunks;
      wait_slab(f, kOwn * p.chunks, p.common, lane, (static_cast<unsigned long long>(j.x1) << 32) | j.x2);
    } else {
      // CTA-level chain: the layer-1 tiles that produce this row block of H_r are done.
      const int rb = row_block(p, j);
      const uint64_t* f = p.h_flags + (static_cast<size_t>(j.x0) * (p.T / 128) + rb) * p.nb1;
      warp_wait_signals(f, kOwn * p.nb1, p.common.epoch, p.common, lane, kSiteSignal,
                        (2ull << 60) | (static_cast<unsigned long long>(j.x0) << 32) | rb);
    }
  }
  static __device__ void load(const Params& p, const Job& j, int kb, uint8_t* sa, uint8_t* sb, uint64_t* bar) {
    const int r0 = Pair ? 128 * j.rank : 0;
    if (j.kind == 1) {
      load_tile<Pair>(sa, j.a_sel ? &p.x_gath : &p.x_local[j.x0], bar, kb * kBK, j.a_row + r0);
#pragma unroll
      for (int g = 0; g < (Pair ? 2 : kBN / 64); ++g)
        load_tile<Pair>(sb + g * 8192, &p.w1[j.b_sel], bar, j.b_col + r0 + g * 64, kb * kBK);
    } else {
      load_tile<Pair>(sa, &p.h_ld, bar, kb * kBK, j.a_row + r0);
#pragma unroll
      for (int g = 0; g < (Pair ? 2 : kBN / 64); ++g)
        load_tile<Pair>(sb + g * 8192, &p.w2[j.b_sel], bar, j.b_col + r0 + g * 64, kb * kBK);
    }
  }
  static __device__ void mma_stage(const Job&, uint32_t d, uint32_t a0, uint32_t b0, int kb) {
    mma_stage_bm<BM>(d, a0, b0, kb);
  }
  static __device__ int h_row(const Params& p, const Job& j) { return j.x0 * p.T + j.x1 * p.Tr + j.x2 * BM; }
  static __device__ int rs_tile_id(const Params& p, const Job& j) { return row_block(p, j) * p.nb2 + j.x3; }
  static __device__ void epilogue(const Params& p, const Job& j, uint32_t taddr, int q, int lane, EpiStage& es,
                                 int h0, int h1) {
    if (j.kind == 1) {
#pragma unroll 1
      for (int hh = h0; hh < h1; ++hh) {
        const int row = h_row(p, j) + hh * 128 + q * 32;
#pragma unroll 1
        for (int ch = 0; ch < kBN / 64; ++ch) {
          const int x = j.b_col + ch * 64;
          if (x >= p.f) break;
          float v[64];
          tmem_ld64(taddr + hh * 256, ch * 64, v);
#pragma unroll
          for (int i = 0; i < 64; ++i) v[i] = gelu_erf(v[i]);
          store_bf16_chunk(&p.h_st, es, lane, v, x, row);
        }
      }
    } else {
      const int grow = j.x1 * p.Tr + j.x2 * BM, pos = j.x0;
      const float* prev = (pos > 0 && pos == p.W - 1) ? p.acc_ptr + static_cast<size_t>(grow) * p.h : nullptr;
      rs_epilogue<BM>(&p.acc, grow, pos > 0, prev, &p.out[j.x1], j.x2 * BM, p.rs_flags + rs_tile_id(p, j), pos, p.W,
                      j.b_col, p.h, p.common, taddr, q, lane, es, h0, h1,
                      static_cast<unsigned long long>(grow) << 20 | static_cast<unsigned>(j.b_col));
    }
  }
  static __device__ bool publishes(const Params& p, const Job& j) { return j.kind == 1 || j.x0 != p.W - 1; }
  static __device__ void publish(const Params& p, const Job& j) {
    if (j.kind == 1) {
      const int rb = row_block(p, j);
#pragma unroll
      for (int s = 0; s < kOwn; ++s)
        st_release_gpu(p.h_flags + (static_cast<size_t>(j.x0) * (p.T / 128) + rb + s) * p.nb1 + j.x3, p.common.epoch);
    } else {
      st_release_gpu(p.rs_flags + rs_tile_id(p, j), (p.common.epoch << 4) | static_cast<unsigned long long>(j.x0 + 1));
    }
  }
  // Every emulated rank r needs the other ranks' X shards in its own copy of X (rows r*T ..);
  // a rank's own shard is read in place by its layer-1 tiles, so its slot of the copy is not
  // written.  Chunks are row pieces of 128-row slabs, a shard's slabs in order.
  //   pull ("Triton-distributed ...", §3.2 Algorithm 2): rank r, in turn (rank 0's first),
  //     copies shards (r+1) mod W, (r+2) mod W, ... into its copy;
  //   push (§3.2 Algorithm 1): each shard, in the order 1, 2, ..., W-1, 0, is read once and
  //     written into the W-1 other ranks' copies, each with its own release signal.
  template <bool Trace>
  static __device__ void mover(const Params& p, int mw, int lane) {
    const int nthreads = p.common.mover_warps * 32;
    const int tid = mw * 32 + lane;
    const int per_shard = p.spr * p.chunks;
    const int piece_rows = tl::kBM / p.chunks;  // slabs are 128 rows (not this op's tile rows)
    const size_t row_stride = static_cast<size_t>(p.h) * 2;
    const int total = p.W < 2 ? 0 : (p.push ? p.W * per_shard : p.W * (p.W - 1) * per_shard);
    for (int g = blockIdx.x; g < total; g += gridDim.x) {
      int r = -1, gg = g;  // r: the one gathering rank (pull); all others (push)
      if (!p.push) {
        r = g / ((p.W - 1) * per_shard);
        gg = g - r * (p.W - 1) * per_shard;
      }
      const ChunkPos cp = chunk_pos(gg, 0, p.spr, p.chunks, p.chunks);
      const int src = ag_mover_rank(p.W, p.push ? 0 : r, p.swizzle, cp.i);
      const size_t off = (static_cast<size_t>(cp.slab) * tl::kBM + static_cast<size_t>(cp.piece) * piece_rows) *
                         row_stride;
      uint8_t* dst[8];
      int nd = 0;
      for (int d = 0; d < p.W; ++d)
        if (d != src && (p.push || d == r))
          dst[nd++] = p.xg + (static_cast<size_t>(d) * p.T + static_cast<size_t>(src) * p.Tr) * p.h * 2 + off;
      copy_rows_multi(p.x[src] + off, dst, nd, row_stride, piece_rows, p.h * 2, tid, nthreads);
      __threadfence();
      named_bar_sync(2, nthreads);
      if (tid < p.W && tid != src && (p.push || tid == r) && g != p.skip_chunk)
        st_release_gpu(p.ag_flags + ((static_cast<size_t>(tid) * p.W + src) * p.spr + cp.slab) * p.chunks + cp.piece,
                       p.common.epoch);
    }
  }
};

// ============================================================================ AllGather alone
// The pull-mode AllGather as its own kernel (the communication task of "Triton-
// distributed ...", §3.2 Algorithm 2, without a consumer): the fused AllGather+GEMM's chunk
// order and signals with whole-row chunks (no K parts: nothing waits on them here), every
// shard including the self rank's (last), on several CTAs of copy warps per SM.  With whole
// rows a chunk is one contiguous block: chunk g of the gather is block g mod (spr * chunks)
// of shard i = g / (spr * chunks) in the mover's order.
constexpr int kAllgatherWarps = 16;  // copy warps per CTA of the standalone AllGather
#ifndef TL_AG_ALONE_CTAS_PER_SM
#define TL_AG_ALONE_CTAS_PER_SM 4
#endif
__global__ void __launch_bounds__(kAllgatherWarps * 32, 2) allgather_kernel(const __grid_constant__ AgParams p) {
  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int per_shard = p.spr * p.chunks;
  const int total = p.W * per_shard;
  const size_t piece_bytes = static_cast<size_t>(tl::kBM / p.chunks) * p.k * 2;
  for (int g = blockIdx.x; g < total; g += gridDim.x) {
    const int i = g / per_shard, rem = g - i * per_shard;
    const int r = ag_mover_rank(p.W, p.rank, p.swizzle, i);
    const size_t off = static_cast<size_t>(rem) * piece_bytes;
    copy_contig(reinterpret_cast<const uint4*>(p.shard[r] + off),
                reinterpret_cast<uint4*>(p.gath + static_cast<size_t>(r) * p.shard_bytes + off),
                static_cast<int>(piece_bytes / 16), tid, nthreads);
    __threadfence();
    __syncthreads();
    if (tid == 0 && g != p.skip_chunk) st_release_gpu(p.flags + static_cast<size_t>(r) * per_shard + rem, p.common.epoch);
  }
}

// The same AllGather moved by the TMA unit instead of the SMs' load/store path (the
// copy-engine mover of the pages' AG, "TileLink ...", §7.2, in its GB300 form: each SM's own
// bulk-copy engine): one thread per CTA streams its chunks through kTmaStages shared-memory
// stages of kTmaStage bytes, a bulk load (completing on the stage's mbarrier) then a bulk
// store, and releases a chunk's signal once every store of it has completed.  Same chunk
// order and signals as allgather_kernel.
constexpr int kTmaStages = 6;
constexpr int kTmaStage = 32768;
constexpr int kTmaSmem = kTmaStages * kTmaStage + kTmaStages * 8 + 128;

__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void bulk_store_1d(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}

__global__ void __launch_bounds__(32, 1) allgather_tma_kernel(const __grid_constant__ AgParams p) {
  extern __shared__ __align__(128) uint8_t tsm[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(tsm + kTmaStages * kTmaStage);
  if (threadIdx.x != 0) return;
  for (int s = 0; s < kTmaStages; ++s) mbar_init(&bars[s], 1);
  fence_mbar_init();
  const Common& c = p.common;
  const int per_shard = p.spr * p.chunks;
  const int total = p.W * per_shard;
  const size_t piece_bytes = static_cast<size_t>(tl::kBM / p.chunks) * p.k * 2;
  const int subs = static_cast<int>((piece_bytes + kTmaStage - 1) / kTmaStage);  // stage-sized parts per chunk
  const int mine = total > static_cast<int>(blockIdx.x) ? (total - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int njobs = mine * subs;  // this CTA's bulk copies: chunk blockIdx.x + t * grid, part sp
  // job j -> its chunk's shard slot offset, the part's offset and size
  auto where = [&](int j, const uint8_t*& src, uint8_t*& dst, uint32_t& bytes, uint64_t*& flag) {
    const int t = j / subs, sp = j - t * subs;
    const int g = blockIdx.x + t * gridDim.x;
    const int i = g / per_shard, rem = g - i * per_shard;
    const int r = ag_mover_rank(p.W, p.rank, p.swizzle, i);
    const size_t o = static_cast<size_t>(rem) * piece_bytes + static_cast<size_t>(sp) * kTmaStage;
    const size_t left = piece_bytes - static_cast<size_t>(sp) * kTmaStage;
    src = p.shard[r] + o;
    dst = p.gath + static_cast<size_t>(r) * p.shard_bytes + o;
    bytes = static_cast<uint32_t>(left < kTmaStage ? left : kTmaStage);
    flag = (sp == subs - 1 && g != p.skip_chunk) ? p.flags + static_cast<size_t>(r) * per_shard + rem : nullptr;
  };
  auto load = [&](int j) {
    const uint8_t* src;
    uint8_t* dst;
    uint32_t bytes;
    uint64_t* flag;
    where(j, src, dst, bytes, flag);
    const int s = j % kTmaStages;
    mbar_arrive_expect_tx(&bars[s], bytes);
    bulk_load_1d(tsm + s * kTmaStage, src, bytes, &bars[s]);
  };
  // signals of chunks whose last store is issued but not yet known complete, oldest first
  constexpr int kPend = kTmaStages + 1;
  uint64_t* pend_flag[kPend] = {};
  int pend_last[kPend] = {};
  int npend = 0;
  auto retire = [&](int upto) {  // release the chunks whose last store is job <= upto
    int k = 0;
    while (k < npend && pend_last[k] <= upto) ++k;
    if (k == 0) return;
    fence_proxy_async_global();
    for (int i = 0; i < k; ++i) st_release_gpu(pend_flag[i], c.epoch);
    for (int i = k; i < npend; ++i) {
      pend_flag[i - k] = pend_flag[i];
      pend_last[i - k] = pend_last[i];
    }
    npend -= k;
  };
  // loads run kTmaStages - 1 jobs ahead of the stores
  int issued = 0, landed = 0;  // loads issued; loads waited for
  for (int j = 0; j < njobs && j < kTmaStages - 1; ++j, ++issued) load(j);
  bool ok = true;
  for (int j = 0; j < njobs && ok; ++j) {
    const int s = j % kTmaStages;
    ok = mbar_wait(&bars[s], (j / kTmaStages) & 1, c, kSiteFull);
    if (!ok) break;
    ++landed;
    const uint8_t* src;
    uint8_t* dst;
    uint32_t bytes;
    uint64_t* flag;
    where(j, src, dst, bytes, flag);
    bulk_store_1d(dst, tsm + s * kTmaStage, bytes);
    bulk_commit();
    if (flag) {
      if (npend == kPend) {  // more chunks in flight than slots: drain the oldest first
        bulk_wait<0>();
        retire(j);
      }
      pend_flag[npend] = flag;
      pend_last[npend] = j;
      ++npend;
    }
    const int jn = j + kTmaStages - 1;  // the next load goes into the stage store j - 1 read
    if (jn < njobs) {
      bulk_wait_read<1>();
      load(jn);
      ++issued;
    }
    if ((j % kTmaStages) == kTmaStages - 1) {  // every kTmaStages jobs: release what has landed
      bulk_wait<kTmaStages - 1>();
      retire(j - (kTmaStages - 1));
    }
  }
  // a wait that ran out leaves loads in flight: let them land (bounded) before the CTA exits
  for (int j = landed; j < issued; ++j) mbar_wait(&bars[j % kTmaStages], (j / kTmaStages) & 1, c, kSiteDrain);
  bulk_wait<0>();  // every store has completed (and nothing reads shared memory any more)
  if (ok) retire(njobs);
}

// ============================================================================ ReduceScatter alone
// The push-mode ReduceScatter of "Triton-distributed ...", §3.3 Algorithm 3, as its own
// kernel: each owner o receives rows [o*m/W, (o+1)*m/W) of the W ranks' fp32 partials and
// sums them, R = T[0] + T[1] + ... + T[W-1], in that order (the order of tl_gemm_rs's
// chain), rounded to bf16 once.  Every thread takes 4 columns of one row per pass (a 16-byte
// vector from each partial, W loads in flight, then an 8-byte bf16 store); two 512-thread
// blocks per SM; the partials are read once, with the streaming (evict-first) hint.
struct RsAloneParams {
  const float4* part[8];
  uint2* out[8];
  long long units;  // m * n / 4
  int W, mo, n4;
};

__global__ void __launch_bounds__(512, 2) reduce_scatter_kernel(const __grid_constant__ RsAloneParams p) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; u < p.units; u += stride) {
    float4 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < p.W) v[q] = __ldcs(p.part[q] + u);
    float4 acc = v[0];
#pragma unroll
    for (int q = 1; q < 8; ++q) {
      if (q < p.W) {
        acc.x += v[q].x;
        acc.y += v[q].y;
        acc.z += v[q].z;
        acc.w += v[q].w;
      }
    }
    const long long row = u / p.n4;
    const int c4 = static_cast<int>(u - row * p.n4);
    const int o = static_cast<int>(row / p.mo);
    const long long orow = row - static_cast<long long>(o) * p.mo;
    p.out[o][orow * p.n4 + c4] = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
  }
}

}  // namespace tl

using namespace tl;

// ============================================================================ C ABI
static bool ag_shape_ok(int W, int mpr, int n, int k) {
  return W >= 1 && W <= 8 && mpr >= 0 && n >= 0 && k >= 0 && mpr % kBM == 0 && n % 8 == 0 && k % 8 == 0;
}

// Tile rows used for a row extent: 256 when every block of the extent is a 256 multiple.
static int pick_bm(int rows) { return rows % 256 == 0 ? 256 : 128; }

// The mover's K parts of a slab (see ag_copy): up to `want` (cfg.mover_kparts: 1, 2 or 4)
// parts of whole 64-column k-blocks, at least 16 k-blocks each (a wait per part costs a
// signal round trip), cpq = chunks / parts row pieces each.
struct KParts {
  int quarters, cpq, kb_q, qcols;
};
static KParts k_parts(int chunks, int k, int want) {
  KParts r;
  if (want <= 0) want = 1;
  const int kblocks = ceil_div(k, kBK);
  r.quarters = 1;
  while (r.quarters < want && r.quarters * 2 <= chunks && kblocks >= 16 * r.quarters * 2) r.quarters *= 2;
  r.cpq = chunks / r.quarters;
  const int kbq = ceil_div(kblocks, r.quarters);
  r.kb_q = kbq > 0 ? kbq : 1;
  r.qcols = r.kb_q * kBK;
  return r;
}
static void ag_parts(AgParams& p, int k, int want) {
  const KParts kp = k_parts(p.chunks, k, want);
  p.k = k;
  p.quarters = kp.quarters;
  p.cpq = kp.cpq;
  p.kb_q = kp.kb_q;
  p.qcols = kp.qcols;
}

namespace tl {
AgLayout ag_layout(int W, int m_per_rank, int k) {
  AgLayout L;
  L.gath_bytes = static_cast<size_t>(W) * m_per_rank * k * 2;
  L.flags_off = align256(L.gath_bytes);
  L.flags_bytes = static_cast<size_t>(W) * (m_per_rank / kBM) * 32 * 8;
  L.ll_off = L.flags_off + align256(L.flags_bytes);
  const long long elems = static_cast<long long>(W) * m_per_rank * k;
  L.ll_bytes = elems <= kLLMaxElems ? static_cast<size_t>(elems) * 4 : 0;
  L.total = L.ll_off + align256(L.ll_bytes);
  return L;
}

int ag_gemm_check(const tl_ctx* ctx, int W, int rank, const void* const* a_shards, const void* b, const void* c,
                  int m_per_rank, int n, int k) {
  if (!ctx || !ag_shape_ok(W, m_per_rank, n, k) || rank < 0 || rank >= W) return TL_ERR_INVALID;
  if (m_per_rank == 0 || n == 0 || k == 0) return TL_OK;
  if (!a_shards || !b || !c) return TL_ERR_INVALID;
  for (int r = 0; r < W; ++r)
    if (!a_shards[r] || !aligned16(a_shards[r])) return TL_ERR_INVALID;
  if (!aligned16(b) || !aligned16(c)) return TL_ERR_INVALID;
  return TL_OK;
}
}  // namespace tl

extern "C" size_t tl_ag_gemm_workspace_bytes(int W, int m_per_rank, int n, int k) {
  if (!ag_shape_ok(W, m_per_rank, n, k)) return 0;
  return ag_layout(W, m_per_rank, k).total;
}

extern "C" int tl_ag_gemm(tl_ctx* ctx, int W, int rank, const void* const* a_shards, const void* b, void* c,
                          void* workspace, size_t workspace_bytes, int m_per_rank, int n, int k,
                          tl_stream_t stream) {
  const int chk = ag_gemm_check(ctx, W, rank, a_shards, b, c, m_per_rank, n, k);
  if (chk != TL_OK) return chk;
  if (m_per_rank == 0 || n == 0 || k == 0) return TL_OK;
  if (!workspace || !aligned16(workspace)) return TL_ERR_INVALID;
  const AgLayout L = ag_layout(W, m_per_rank, k);
  if (workspace_bytes < L.total) return TL_ERR_WORKSPACE;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return TL_ERR_CUDA;
  if (ctx->cfg.ag_ll && W > 1)
    return ag_ll_launch(ctx, W, rank, a_shards, b, c, static_cast<uint8_t*>(workspace), m_per_rank, n, k,
                        reinterpret_cast<cudaStream_t>(stream));

  AgParams p;
  std::memset(&p, 0, sizeof(p));
  const int M = W * m_per_rank;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.gath = ws;
  p.flags = reinterpret_cast<uint64_t*>(ws + L.flags_off);
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int bm = pick_bm(m_per_rank);
  const bool pair = bm == 256 && ctx->cfg.pair_ctas == 1;
  const int abox = pair ? 128 : bm;  // a CTA of a pair loads 128 of the tile's 256 rows
  if (!tmap_2d(&p.a_local, BF, 2, a_shards[rank], k, m_per_rank, 64, abox) ||
      !tmap_2d(&p.a_gath, BF, 2, p.gath, k, M, 64, abox) || !tmap_2d(&p.b, BF, 2, b, n, k, 64, 64) ||
      !tmap_2d(&p.c, BF, 2, c, n, M, 64, 32))
    return TL_ERR_CUDA;
  p.common = make_common(ctx);
  for (int r = 0; r < W; ++r) p.shard[r] = static_cast<const uint8_t*>(a_shards[r]);
  p.W = W;
  p.rank = rank;
  p.m_per_rank = m_per_rank;
  p.mps = m_per_rank / bm;
  p.spr = m_per_rank / kBM;
  p.n = n;
  p.nbk = ceil_div(n, kBN);
  p.kblocks = ceil_div(k, kBK);
  p.swizzle = ctx->cfg.swizzle;
  p.chunks = ctx->cfg.chunks_per_slab;
  p.skip_chunk = ctx->cfg.debug_skip_chunk;
  p.shard_bytes = static_cast<long long>(m_per_rank) * k * 2;
  p.slab_bytes = static_cast<long long>(kBM) * k * 2;
  p.copy_self = 0;  // the GEMM reads the self shard in place; its slot of T is not written
  ag_parts(p, k, ctx->cfg.mover_kparts > 0 ? ctx->cfg.mover_kparts : 4);
  // The head: the next two shards, which the first wave of tiles reads; the epilogue warps
  // help copy it.
  p.head = W - 1 < 2 ? W - 1 : 2;
  p.boost = p.head * p.spr * p.chunks;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int movers = ctx->cfg.mover_warps;
  if (W == 1) {  // nothing to gather: the plain GEMM on shard 0 in place, no mover, no signals
    p.boost = 0;
    movers = 0;
  }
  int rc;
  if (pair)
    rc = launch_persistent_pair<AgOp<256, true>>(ctx, p, st, movers);
  else
    rc = bm == 256 ? launch_persistent<AgOp<256>>(ctx, p, st, movers) : launch_persistent<AgOp<128>>(ctx, p, st, movers);
  return rc;
}

static bool rs_shape_ok(int W, int m, int n, int kr) {
  return W >= 1 && W <= 8 && m >= 0 && n >= 0 && kr >= 0 && m % (kBM * W) == 0 && n % 8 == 0 && kr % 8 == 0;
}

// GEMM+RS workspace: the fp32 partial buffers (the owner slot, m x n; or, for the ring, W
// receive buffers of m x n), then one signal per 128-row block and 256-column block.
static size_t rs_acc_bytes(int W, int m, int n, bool ring) {
  return align256(static_cast<size_t>(ring ? W : 1) * m * n * 4);
}
static size_t rs_ws_bytes(int W, int m, int n, bool ring) {
  return rs_acc_bytes(W, m, n, ring) + align256(static_cast<size_t>(m / kBM) * ceil_div(n, kBN) * 8);
}

extern "C" size_t tl_gemm_rs_workspace_bytes(int W, int m, int n, int k_r) {
  if (!rs_shape_ok(W, m, n, k_r)) return 0;
  return rs_ws_bytes(W, m, n, false);
}

extern "C" size_t tl_gemm_rs_ring_workspace_bytes(int W, int m, int n, int k_r) {
  if (!rs_shape_ok(W, m, n, k_r)) return 0;
  return rs_ws_bytes(W, m, n, true);
}

extern "C" int tl_gemm_rs(tl_ctx* ctx, int W, const void* const* a, const void* const* b, void* const* out,
                          void* workspace, size_t workspace_bytes, int m, int n, int k_r, tl_stream_t stream) {
  if (!ctx || !rs_shape_ok(W, m, n, k_r)) return TL_ERR_INVALID;
  if (m == 0 || n == 0) return TL_OK;
  if (!a || !b || !out || !workspace || !aligned16(workspace)) return TL_ERR_INVALID;
  for (int r = 0; r < W; ++r)
    if (!a[r] || !b[r] || !out[r] || !aligned16(a[r]) || !aligned16(b[r]) || !aligned16(out[r]))
      return TL_ERR_INVALID;
  const bool ring = ctx->cfg.rs_ring != 0;
  if (workspace_bytes < rs_ws_bytes(W, m, n, ring)) return TL_ERR_WORKSPACE;
  if (k_r == 0) return TL_ERR_INVALID;  // an empty reduction has no tiles to chain; reject
  if (cudaSetDevice(ctx->device) != cudaSuccess) return TL_ERR_CUDA;

  RsParams p;
  std::memset(&p, 0, sizeof(p));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* acc = reinterpret_cast<float*>(ws);
  p.acc_ptr = acc;
  p.flags = reinterpret_cast<uint64_t*>(ws + rs_acc_bytes(W, m, n, ring));
  p.ring = ring ? 1 : 0;
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int mo = m / W;
  const int bm = pick_bm(mo);
  const bool pair = bm == 256 && ctx->cfg.pair_ctas != 0;
  for (int r = 0; r < W; ++r) {
    if (!tmap_2d(&p.a[r], BF, 2, a[r], k_r, m, 64, pair ? 128 : bm) || !tmap_2d(&p.b[r], BF, 2, b[r], n, k_r, 64, 64) ||
        !tmap_2d(&p.out[r], BF, 2, out[r], n, mo, 64, 32))
      return TL_ERR_CUDA;
  }
  if (!tmap_2d(&p.acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, acc, n, static_cast<uint64_t>(ring ? W : 1) * m, 32, 32))
    return TL_ERR_CUDA;
  p.common = make_common(ctx);
  p.W = W;
  p.m = m;
  p.mo = mo;
  p.mbo = mo / bm;
  p.n = n;
  p.nbk = ceil_div(n, kBN);
  p.kblocks = ceil_div(k_r, kBK);
  p.swizzle = ctx->cfg.swizzle;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (pair) return launch_persistent_pair<RsOp<256, true>>(ctx, p, st, 0);
  return bm == 256 ? launch_persistent<RsOp<256>>(ctx, p, st, 0) : launch_persistent<RsOp<128>>(ctx, p, st, 0);
}

static bool mlp2_shape_ok(int W, int T, int h, int f) {
  return W >= 1 && W <= 8 && T >= 0 && h >= 0 && f >= 0 && T % (kBM * W) == 0 && h % 8 == 0 && f % 8 == 0;
}

struct Mlp2Layout {
  size_t xg, hbuf, acc, agf, hf, rsf, total;
};
static Mlp2Layout mlp2_layout(int W, int T, int h, int f) {
  Mlp2Layout L;
  const size_t xg = static_cast<size_t>(W) * T * h * 2;
  const size_t hb = static_cast<size_t>(W) * T * f * 2;
  const size_t acc = static_cast<size_t>(T) * h * 4;
  const size_t agf = static_cast<size_t>(W) * W * (T / W / kBM) * 32 * 8;
  const size_t hf = static_cast<size_t>(W) * (T / kBM) * ceil_div(f, kBN) * 8;
  const size_t rsf = static_cast<size_t>(T / kBM) * ceil_div(h, kBN) * 8;
  L.xg = 0;
  L.hbuf = align256(xg);
  L.acc = L.hbuf + align256(hb);
  L.agf = L.acc + align256(acc);
  L.hf = L.agf + align256(agf);
  L.rsf = L.hf + align256(hf);
  L.total = L.rsf + align256(rsf);
  return L;
}

extern "C" size_t tl_mlp2_workspace_bytes(int W, int tokens, int hidden, int f_r) {
  if (!mlp2_shape_ok(W, tokens, hidden, f_r)) return 0;
  return mlp2_layout(W, tokens, hidden, f_r).total;
}

extern "C" int tl_mlp2(tl_ctx* ctx, int W, const void* const* x_shards, const void* const* w1,
                       const void* const* w2, void* const* out, void* workspace, size_t workspace_bytes, int tokens,
                       int hidden, int f_r, tl_stream_t stream) {
  if (!ctx || !mlp2_shape_ok(W, tokens, hidden, f_r)) return TL_ERR_INVALID;
  if (tokens == 0 || hidden == 0) return TL_OK;
  if (f_r == 0) return TL_ERR_INVALID;
  if (!x_shards || !w1 || !w2 || !out || !workspace || !aligned16(workspace)) return TL_ERR_INVALID;
  for (int r = 0; r < W; ++r)
    if (!x_shards[r] || !w1[r] || !w2[r] || !out[r] || !aligned16(x_shards[r]) || !aligned16(w1[r]) ||
        !aligned16(w2[r]) || !aligned16(out[r]))
      return TL_ERR_INVALID;
  if (workspace_bytes < tl_mlp2_workspace_bytes(W, tokens, hidden, f_r)) return TL_ERR_WORKSPACE;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return TL_ERR_CUDA;

  const Mlp2Layout L = mlp2_layout(W, tokens, hidden, f_r);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Mlp2Params p;
  std::memset(&p, 0, sizeof(p));
  const int Tr = tokens / W;
  p.xg = ws + L.xg;
  uint8_t* hb = ws + L.hbuf;
  float* acc = reinterpret_cast<float*>(ws + L.acc);
  p.acc_ptr = acc;
  p.ag_flags = reinterpret_cast<uint64_t*>(ws + L.agf);
  p.h_flags = reinterpret_cast<uint64_t*>(ws + L.hf);
  p.rs_flags = reinterpret_cast<uint64_t*>(ws + L.rsf);
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int bm = pick_bm(Tr);
  const bool pair = bm == 256 && ctx->cfg.pair_ctas != 0;
  const int abox = pair ? 128 : bm;
  for (int r = 0; r < W; ++r) {
    if (!tmap_2d(&p.x_local[r], BF, 2, x_shards[r], hidden, Tr, 64, abox) ||
        !tmap_2d(&p.w1[r], BF, 2, w1[r], f_r, hidden, 64, 64) ||
        !tmap_2d(&p.w2[r], BF, 2, w2[r], hidden, f_r, 64, 64) ||
        !tmap_2d(&p.out[r], BF, 2, out[r], hidden, Tr, 64, 32))
      return TL_ERR_CUDA;
    p.x[r] = static_cast<const uint8_t*>(x_shards[r]);
  }
  if (!tmap_2d(&p.x_gath, BF, 2, p.xg, hidden, static_cast<uint64_t>(W) * tokens, 64, abox) ||
      !tmap_2d(&p.h_st, BF, 2, hb, f_r, static_cast<uint64_t>(W) * tokens, 64, 32) ||
      !tmap_2d(&p.h_ld, BF, 2, hb, f_r, static_cast<uint64_t>(W) * tokens, 64, abox) ||
      !tmap_2d(&p.acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, acc, hidden, tokens, 32, 32))
    return TL_ERR_CUDA;
  p.common = make_common(ctx);
  p.W = W;
  p.T = tokens;
  p.Tr = Tr;
  p.h = hidden;
  p.f = f_r;
  p.mps = Tr / bm;
  p.spr = Tr / kBM;
  p.nb1 = ceil_div(f_r, kBN);
  p.kb1 = ceil_div(hidden, kBK);
  p.nb2 = ceil_div(hidden, kBN);
  p.kb2 = ceil_div(f_r, kBK);
  p.swizzle = ctx->cfg.swizzle;
  p.chunks = ctx->cfg.chunks_per_slab;
  p.skip_chunk = ctx->cfg.debug_skip_chunk;
  p.shard_bytes = static_cast<long long>(Tr) * hidden * 2;
  p.slab_bytes = static_cast<long long>(kBM) * hidden * 2;
  p.push = ctx->cfg.ag_push;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (pair) return launch_persistent_pair<Mlp2Op<256, true>>(ctx, p, st, ctx->cfg.mover_warps);
  return bm == 256 ? launch_persistent<Mlp2Op<256>>(ctx, p, st, ctx->cfg.mover_warps)
                   : launch_persistent<Mlp2Op<128>>(ctx, p, st, ctx->cfg.mover_warps);
}

extern "C" int tl_allgather(tl_ctx* ctx, int W, int rank, const void* const* a_shards, void* workspace,
                            size_t workspace_bytes, int m_per_rank, int k, tl_stream_t stream) {
  if (!ctx || !ag_shape_ok(W, m_per_rank, 8, k) || rank < 0 || rank >= W) return TL_ERR_INVALID;
  if (m_per_rank == 0 || k == 0) return TL_OK;
  if (!a_shards || !workspace || !aligned16(workspace)) return TL_ERR_INVALID;
  if (W == 1) return TL_OK;  // nothing to gather
  for (int r = 0; r < W; ++r)
    if (!a_shards[r] || !aligned16(a_shards[r])) return TL_ERR_INVALID;
  const AgLayout L = ag_layout(W, m_per_rank, k);
  if (workspace_bytes < L.total) return TL_ERR_WORKSPACE;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return TL_ERR_CUDA;
  AgParams p;
  std::memset(&p, 0, sizeof(p));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.gath = ws;
  p.flags = reinterpret_cast<uint64_t*>(ws + L.flags_off);
  p.common = make_common(ctx);
  // The standalone mover kernel has no dynamic shared memory for span counters: no trace.
  p.common.trace_hdr = nullptr;
  p.common.trace = nullptr;
  for (int r = 0; r < W; ++r) p.shard[r] = static_cast<const uint8_t*>(a_shards[r]);
  p.W = W;
  p.rank = rank;
  p.m_per_rank = m_per_rank;
  p.mps = m_per_rank / kBM;
  p.spr = m_per_rank / kBM;
  p.swizzle = ctx->cfg.swizzle;
  p.chunks = ctx->cfg.chunks_per_slab;
  p.skip_chunk = -1;
  p.copy_self = 1;
  ag_parts(p, k, 1);  // no consumer waits on K parts here: whole-row chunks copy fastest
  p.head = W < 2 ? W : 2;
  p.shard_bytes = static_cast<long long>(m_per_rank) * k * 2;
  p.slab_bytes = static_cast<long long>(kBM) * k * 2;
  // Alone, the copy has the whole GPU: TL_AG_ALONE_CTAS_PER_SM CTAs of kAllgatherWarps warps
  // per SM (two resident at a time), so one CTA's fence and barrier after a chunk overlap the
  // other CTA's loads.
  if (ctx->cfg.mover_tma) {
    if (cudaFuncSetAttribute(allgather_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTmaSmem) !=
        cudaSuccess) {
      (void)cudaGetLastError();
      return TL_ERR_CUDA;
    }
    allgather_tma_kernel<<<ctx->sms, 32, kTmaSmem, reinterpret_cast<cudaStream_t>(stream)>>>(p);
    return cudaGetLastError() == cudaSuccess ? TL_OK : TL_ERR_CUDA;
  }
  p.common.mover_warps = kAllgatherWarps;
  allgather_kernel<<<ctx->ctas * TL_AG_ALONE_CTAS_PER_SM, kAllgatherWarps * 32, 0,
                     reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? TL_OK : TL_ERR_CUDA;
}

extern "C" int tl_reduce_scatter(tl_ctx* ctx, int W, const float* const* partials, void* const* out, int m, int n,
                                 tl_stream_t stream) {
  if (!ctx || W < 1 || W > 8 || m < 0 || n < 0 || m % W != 0 || n % 4 != 0) return TL_ERR_INVALID;
  if (m == 0 || n == 0) return TL_OK;
  if (!partials || !out) return TL_ERR_INVALID;
  for (int r = 0; r < W; ++r)
    if (!partials[r] || !out[r] || !aligned16(partials[r]) || !aligned16(out[r])) return TL_ERR_INVALID;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return TL_ERR_CUDA;
  RsAloneParams p;
  std::memset(&p, 0, sizeof(p));
  for (int r = 0; r < W; ++r) {
    p.part[r] = reinterpret_cast<const float4*>(partials[r]);
    p.out[r] = static_cast<uint2*>(out[r]);
  }
  p.W = W;
  p.mo = m / W;
  p.n4 = n / 4;
  p.units = static_cast<long long>(m) * (n / 4);
  // Two 512-thread blocks per SM (the launch bounds), enough 16-byte loads in flight to
  // keep HBM busy; a grid-stride loop covers the rest.
  long long blocks = (p.units + 511) / 512;
  if (blocks > 2LL * ctx->sms) blocks = 2LL * ctx->sms;
  reduce_scatter_kernel<<<static_cast<unsigned>(blocks), 512, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? TL_OK : TL_ERR_CUDA;
}
