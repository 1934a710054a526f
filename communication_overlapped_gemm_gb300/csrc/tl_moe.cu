// MoE layer: routing, stable expert permutation (the dynamic tile-centric mapping
// tables), token gather, and one persistent launch in which a GEMM partition runs the
// grouped expert GEMMs while a dedicated combine partition scatter-adds finished
// output tiles back into token order as their ready signals arrive.
//
// "TileLink: Generating Efficient Compute-Communication Overlapping Kernels using
// Tile-Centric Primitives", §4.1 (dynamic mapping: lookup tables f_S_low/high, f_R
// filled at run time by the routing) and §7.2 (Gather + GroupGEMM; GroupGEMM + Scatter
// + TopK reduce as a producer/consumer chain); "Resource-aware Computation-
// Communication Overlap for multi-GPU ML Workloads", MoE abstract (a persistent
// producer covering all local experts; a persistent consumer on a small dedicated SM
// partition that handles output segments as tiles become ready).
#include <cuda_bf16.h>

#include "tl_host.h"

namespace tl {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopk = 8;

// ---------------------------------------------------------------------------- routing
// One warp per token: top-k of the fp32 logits (larger first, equal values to the
// lower expert index), softmax over all E logits in fp32 taken at the chosen experts,
// optionally divided by their sum over the chosen experts (renorm).  It lets the
// permutation kernel start at once (that kernel waits for this one before its first read).
__global__ void moe_route_kernel(const float* __restrict__ logits, int T, int E, int topk, int renorm,
                                 int* __restrict__ experts, float* __restrict__ gates) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  grid_dep_launch();
  if (t >= T) return;

  constexpr int kPer = kMaxExperts / 32;
  float v[kPer];
  const float* row = logits + static_cast<size_t>(t) * E;
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? row[e] : -INFINITY;
    mx = fmaxf(mx, v[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    if (lane + 32 * i < E) s += expf(v[i] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);

  uint32_t taken = 0;
  float g[kMaxTopk];
  float gsum = 0.f;
  for (int j = 0; j < topk; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !(taken & (1u << i)) && (v[i] > bv || (v[i] == bv && e < bi))) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    g[j < kMaxTopk ? j : 0] = expf(bv - mx) / s;
    gsum += g[j < kMaxTopk ? j : 0];
    if (lane == 0) experts[t * topk + j] = bi;
  }
  if (lane == 0)
    for (int j = 0; j < topk; ++j) gates[t * topk + j] = renorm ? g[j] / gsum : g[j];
}

// ---------------------------------------------------------------------------- permutation
// One block per expert e.  Every block histograms all assignments (so each knows all
// offsets without a grid-wide step), then ranks the assignments of its own expert in
// (t, j) order with a block-wide ballot scan.  Outputs:
//   perm[off_e + pos] = a                      (unpadded order: expert, t, j)
//   row_meta[row] = {token, gate bits} of the row's assignment ({-1, 0} on padding rows), so
//     the combine reads one 8-byte record per row instead of two dependent loads
//   tile_expert / tile_rows for each 128-row tile of the padded layout (the f_R / f_S tables)
// Launched as a dependent of the routing kernel: the zeroing CTAs run alongside it, the
// expert CTAs wait for it (grid_dep_wait) before they read the routing; the persistent
// kernel after it may start as soon as every CTA of this one is running.
__global__ void __launch_bounds__(1024) moe_permute_kernel(const int* __restrict__ experts, int n, int E, int topk,
                                                           const float* __restrict__ gates,
                                                           int* __restrict__ perm, int2* __restrict__ row_meta,
                                                           int* __restrict__ tile_expert, int* __restrict__ tile_rows,
                                                           int* __restrict__ num_mtiles, int* __restrict__ counts,
                                                           int* __restrict__ perm_out, int* __restrict__ counts_out,
                                                           float4* __restrict__ out, size_t out_vec,
                                                           int* __restrict__ combine_next) {
  __shared__ int hist[kMaxExperts];
  __shared__ int off[kMaxExperts + 1];
  __shared__ int poff[kMaxExperts + 1];
  __shared__ int warp_tot[32];
  __shared__ int warp_pre[32];
  const int e = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  grid_dep_launch();
  if (e >= E) {
    // CTAs past the experts zero the fp32 output the combine partition adds into, on the
    // SMs the per-expert CTAs leave idle.
    const size_t nz = gridDim.x - E;
    for (size_t i = (e - E) * static_cast<size_t>(blockDim.x) + tid; i < out_vec; i += nz * blockDim.x)
      out[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  for (int i = tid; i < E; i += blockDim.x) hist[i] = 0;
  grid_dep_wait();
  __syncthreads();
  for (int a = tid; a < n; a += blockDim.x) {
    const unsigned ex = static_cast<unsigned>(experts[a]);
    if (ex < static_cast<unsigned>(E)) atomicAdd(&hist[ex], 1);  // never index outside the table
  }
  __syncthreads();
  if (warp == 0) {  // exclusive prefix sums of the counts and the 128-padded counts (E <= 256)
    int c[kMaxExperts / 32], pc[kMaxExperts / 32];
    int sc = 0, sp = 0;
#pragma unroll
    for (int k = 0; k < kMaxExperts / 32; ++k) {  // lane holds experts [lane * per, lane * per + per)
      const int i = lane * (kMaxExperts / 32) + k;
      c[k] = i < E ? hist[i] : 0;
      pc[k] = (c[k] + kBM - 1) / kBM * kBM;
      sc += c[k];
      sp += pc[k];
    }
    int ic = sc, ip = sp;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int uc = __shfl_up_sync(0xffffffffu, ic, o), up = __shfl_up_sync(0xffffffffu, ip, o);
      if (lane >= o) {
        ic += uc;
        ip += up;
      }
    }
    int rc = ic - sc, rp = ip - sp;
#pragma unroll
    for (int k = 0; k < kMaxExperts / 32; ++k) {
      const int i = lane * (kMaxExperts / 32) + k;
      if (i < E) {
        off[i] = rc;
        poff[i] = rp;
      }
      rc += c[k];
      rp += pc[k];
    }
    if (lane == 31) {  // the totals
      off[E] = ic;
      poff[E] = ip;
    }
  }
  __syncthreads();
  // Stable ranks of this expert's assignments in one pass: warp w takes the contiguous
  // slice [w * seg, (w + 1) * seg) of the assignments, counts its matches, an exclusive scan
  // over the warps' counts gives each warp its first position, and each warp then writes its
  // matches in order (two block barriers in all).
  const int nw = blockDim.x >> 5;
  const int seg = ((n + nw - 1) / nw + 31) & ~31;
  const int s0 = warp * seg, s1 = min(n, s0 + seg);
  int mine_cnt = 0;
  for (int a0 = s0; a0 < s1; a0 += 32 * 8) {  // eight independent loads per lane in flight
    int ex[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int a = a0 + 32 * u + lane;
      ex[u] = a < s1 ? experts[a] : -1;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) mine_cnt += __popc(__ballot_sync(0xffffffffu, ex[u] == e));
  }
  if (lane == 0) warp_tot[warp] = mine_cnt;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < nw ? warp_tot[lane] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    warp_pre[lane] = incl - v;
  }
  __syncthreads();
  int running = warp_pre[warp];
  for (int a0 = s0; a0 < s1; a0 += 32 * 8) {
    int ex[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int a = a0 + 32 * u + lane;
      ex[u] = a < s1 ? experts[a] : -1;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int a = a0 + 32 * u + lane;
      const bool mine = ex[u] == e;
      const uint32_t ball = __ballot_sync(0xffffffffu, mine);
      if (mine) {
        const int pos = running + __popc(ball & ((1u << lane) - 1u));
        perm[off[e] + pos] = a;
        if (perm_out) perm_out[off[e] + pos] = a;
        row_meta[poff[e] + pos] = make_int2(a / topk, __float_as_int(gates[a]));
      }
      running += __popc(ball);
    }
  }
  const int cnt = hist[e];
  const int padded = poff[e + 1] - poff[e];
  for (int i = cnt + tid; i < padded; i += blockDim.x) {
    row_meta[poff[e] + i] = make_int2(-1, 0);
  }
  for (int i = tid; i < padded / kBM; i += blockDim.x) {
    const int tile = poff[e] / kBM + i;
    tile_expert[tile] = e;
    tile_rows[tile] = min(kBM, cnt - i * kBM);
  }
  if (tid == 0) {
    counts[e] = cnt;
    if (counts_out) counts_out[e] = cnt;
    if (e == 0) {
      *num_mtiles = poff[E] / kBM;
      *combine_next = 0;
    }
  }
}

// ---------------------------------------------------------------------------- grouped GEMMs + combine
struct MoeParams {
  CUtensorMap xp;    // gathered rows {H, R}, box {64, 128}
  CUtensorMap wg;    // {F, H, E}, box {64, 64, 1}
  CUtensorMap wu;    // {F, H, E}, box {64, 64, 1}
  CUtensorMap wd;    // {H, F, E}, box {64, 64, 1}
  CUtensorMap h_st;  // h {F, R}, box {64, 32}
  CUtensorMap h_ld;  // h {F, R}, box {64, 128}
  CUtensorMap y_st;  // y {H, R}, box {64, 32}
  CUtensorMap y_ld;  // y {H, R}, box {64, 128} (combine partition loads)
  Common common;
  const int* num_mtiles;
  const int* tile_expert;
  const int* tile_rows;
  const int2* row_meta;
  const __nv_bfloat16* x;  // tokens, gathered into xp by the mover warps
  __nv_bfloat16* xp_rows;  // the gathered rows (xp's memory)
  uint64_t* x_flags;       // [R/128][kGatherPieces]: piece of a row tile gathered
  const __nv_bfloat16* y;
  float* out;
  uint64_t* up_flags;  // [R/128][n_up]
  uint64_t* y_flags;   // [R/128][n_down]
  int* combine_next;   // the next y tile to combine (claimed at run time)
  int T, H, E, F, topk, n_up, n_down, kb_up, kb_down, combine_ctas, chunk, lag;
};

constexpr int kGatherRows = 4;                  // rows one mover warp gathers per signal
constexpr int kGatherPieces = kBM / kGatherRows;  // signals per 128-row tile

struct MoeSlot {
  int kind;  // 1 up-projection, 2 down-projection
  int i;     // row tile
  int nb;    // column block
};

// The tile order of the persistent kernel (see MoeOp) for m row tiles, n_up / n_down column
// blocks, chunks of G row tiles and a down chunk `lag` chunks behind its up chunk.  Host and
// device share it: the kernel's scheduler and tl_moe_tile_order / tl_moe_combine_order.
struct MoeOrder {
  int m, n_up, n_down, G, lag;
};
TL_HD int moe_rows_before(int c, int m, int G) { return c * G < m ? c * G : m; }
// Tiles before group g: the up tiles of chunks 0 .. min(g, nc) - 1 and the down tiles of
// chunks 0 .. g - lag - 1 (every chunk holds G row tiles but the last, which holds
// m - (nc - 1) G).
TL_HD int moe_group_start(const MoeOrder& o, int nc, int g) {
  const int cu = g < nc ? g : nc;
  int cd = g - o.lag < nc ? g - o.lag : nc;
  cd = cd > 0 ? cd : 0;
  return moe_rows_before(cu, o.m, o.G) * o.n_up + moe_rows_before(cd, o.m, o.G) * o.n_down;
}
TL_HD MoeSlot moe_slot(const MoeOrder& o, int t) {
  const int G = o.G;
  const int nc = (o.m + G - 1) / G;
  // the last group g with group_start(g) <= t (binary search over g in [0, nc + lag))
  int lo = 0, hi = nc + o.lag - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (moe_group_start(o, nc, mid) <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int g = lo;
  int w = t - moe_group_start(o, nc, g);
  if (g < nc) {
    const int gc = o.m - g * G < G ? o.m - g * G : G;
    if (w < gc * o.n_up) return MoeSlot{1, g * G + w % gc, w / gc};
    w -= gc * o.n_up;
  }
  const int c = g - o.lag;
  const int gc = o.m - c * G < G ? o.m - c * G : G;
  return MoeSlot{2, c * G + w % gc, w / gc};
}
// The v-th down-projection tile in production order (the order the combine claims them in).
TL_HD MoeSlot moe_down_slot(const MoeOrder& o, int v) {
  const int G = o.G;
  const int c = v / (G * o.n_down);
  const int gc = o.m - c * G < G ? o.m - c * G : G;
  const int w = v - c * G * o.n_down;
  return MoeSlot{2, c * G + w % gc, w / gc};
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

struct MoeOp : OpBase<MoeParams> {
  using Params = MoeParams;
  static constexpr int kBM = 128;
  // Two extra warps per CTA: the token gather (mover) in GEMM CTAs, combine workers in the
  // combine partition's CTAs.
  static constexpr int kMaxMovers = 2;
  static constexpr uint32_t kTxBytes = Geo<128>::kStageBytes;
  static constexpr bool kDependentLaunch = true;
  // The tile count and tile table come from the permutation kernel, which has completed
  // before any role of this kernel reads them (grid_dep_wait): read-only from then on, so
  // they go through the non-coherent cache (one L2 trip per SM, then L1 hits).
  static __device__ int mtiles(const Params& p) { return __ldg(p.num_mtiles); }
  static __device__ int num_tiles(const Params& p) { return mtiles(p) * (p.n_up + p.n_down); }
  static __device__ bool gemm_partition(const Params& p, int& gi, int& gn) {
    gn = gridDim.x - p.combine_ctas;
    gi = blockIdx.x;
    return static_cast<int>(blockIdx.x) < gn;
  }
  // Tile order.  Row tiles (128 padded rows, expert-major) are grouped in chunks of
  // p.chunk; U_c are chunk c's up-projection tiles and D_c its down-projection tiles.  The
  // sequence runs groups g = 0, 1, ...: group g is U_g (while g < chunks) followed by
  // D_{g - lag} (once g >= lag), so U_0 .. U_{lag-1} lead and D_{last-lag+1} .. D_last trail.
  // A down tile therefore comes after every up tile it waits on (no deadlock in a
  // co-resident grid), and `lag` chunks of up work separate a down chunk from the up tiles
  // it reads.  A small lag starts the down tiles (hence the combine's work) early; a lag of
  // at least the chunk count runs every up tile first, then every down tile, in chunk order.
  // Inside a chunk the row tile is the fastest index, so the row tiles of one expert, which
  // share its weight columns, run side by side.
  static __device__ __forceinline__ MoeOrder order(const Params& p, int m) {
    return MoeOrder{m, p.n_up, p.n_down, p.chunk, p.lag};
  }
  static __device__ MoeSlot slot(const Params& p, int m, int t) { return moe_slot(order(p, m), t); }
  static __device__ MoeSlot down_slot(const Params& p, int m, int v) { return moe_down_slot(order(p, m), v); }
  static __device__ Job job(const Params& p, int t) {
    const MoeSlot sl = slot(p, mtiles(p), t);
    Job j;
    j.kind = sl.kind;
    j.x0 = sl.i;
    j.x1 = sl.nb;
    if (sl.kind == 1) {
      j.b_col = sl.nb * 128;
      j.kblocks = p.kb_up;
    } else {
      j.b_col = sl.nb * kBN;
      j.kblocks = p.kb_down;
    }
    j.a_sel = 0;
    j.b_sel = 0;
    j.a_row = j.x0 * kBM;
    j.b_z = __ldg(p.tile_expert + j.x0);
    j.x2 = 0;
    j.x3 = 0;
    return j;
  }
  static __device__ void prefetch(const Params& p) {
    tma_prefetch_map(&p.xp);
    tma_prefetch_map(&p.wg);
    tma_prefetch_map(&p.wu);
    tma_prefetch_map(&p.wd);
    tma_prefetch_map(&p.h_ld);
  }
  // consumer_tile_wait: an up-projection tile reads its 128 gathered rows only after the
  // mover has released all of the row tile's pieces; a down-projection tile reads its row
  // tile of h only after all n_up up-projection tiles of that row tile have signalled.
  static __device__ void wait_deps(const Params& p, const Job& j, int kb, int lane) {
    if (kb != 0) return;
    if (j.kind == 1)
      warp_wait_signals(p.x_flags + static_cast<size_t>(j.x0) * kGatherPieces, kGatherPieces, p.common.epoch,
                        p.common, lane, kSiteSignal, (5ull << 60) | j.x0);
    else
      warp_wait_signals(p.up_flags + static_cast<size_t>(j.x0) * p.n_up, p.n_up, p.common.epoch, p.common, lane,
                        kSiteSignal, (3ull << 60) | j.x0);
  }
  // The token gather (the "Gather" before the grouped GEMM, overlapped with it): padded row
  // r of xp receives x[token of r] (zeros on padding rows).  Pieces of kGatherRows rows are
  // dealt to the GEMM CTAs' mover warps in row order, so the first chunks' rows come first;
  // each piece is published with its own release signal.
  template <bool Trace>
  static __device__ void mover(const Params& p, int mw, int lane) {
    const int nw = (static_cast<int>(gridDim.x) - p.combine_ctas) * p.common.mover_warps;
    const int total = mtiles(p) * kGatherPieces;
    const int vec_row = p.H / 8;  // 16-byte vectors per row
    for (int q = blockIdx.x * p.common.mover_warps + mw; q < total; q += nw) {
      const uint64_t t0 = Trace ? globaltimer() : 0;
#pragma unroll 1
      for (int r = q * kGatherRows; r < (q + 1) * kGatherRows; ++r) {
        const int tok = __ldg(&p.row_meta[r].x);
        uint4* dst = reinterpret_cast<uint4*>(p.xp_rows + static_cast<size_t>(r) * p.H);
        if (tok >= 0) {
          const uint4* src = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(tok) * p.H);
#pragma unroll 1
          for (int c0 = 0; c0 < vec_row; c0 += 8 * 32) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int c = c0 + u * 32 + lane;
              if (c < vec_row) v[u] = __ldg(src + c);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int c = c0 + u * 32 + lane;
              if (c < vec_row) dst[c] = v[u];
            }
          }
        } else {
          for (int c = lane; c < vec_row; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
        }
      }
      __threadfence();
      __syncwarp();
      if (lane == 0) {
        st_release_gpu(p.x_flags + q, p.common.epoch);
        if (Trace) trace_span(p.common, kTrMoverChunk, q, t0, globaltimer());
      }
    }
  }
  static __device__ void load(const Params& p, const Job& j, int kb, uint8_t* sa, uint8_t* sb, uint64_t* bar) {
    if (j.kind == 1) {
      tma_load_2d(sa, &p.xp, bar, kb * kBK, j.a_row);
      tma_load_3d(sb, &p.wg, bar, j.b_col, kb * kBK, j.b_z);
      tma_load_3d(sb + 8192, &p.wg, bar, j.b_col + 64, kb * kBK, j.b_z);
      tma_load_3d(sb + 16384, &p.wu, bar, j.b_col, kb * kBK, j.b_z);
      tma_load_3d(sb + 24576, &p.wu, bar, j.b_col + 64, kb * kBK, j.b_z);
    } else {
      tma_load_2d(sa, &p.h_ld, bar, kb * kBK, j.a_row);
#pragma unroll
      for (int g = 0; g < kBN / 64; ++g) tma_load_3d(sb + g * 8192, &p.wd, bar, j.b_col + g * 64, kb * kBK, j.b_z);
    }
  }
  // Up tiles load the gate and up weight columns as the four 64-column groups of one
  // 256-column B slice (gate 0-127, up 128-255), so both kinds are one 128x256 MMA per K
  // step: the gate accumulator in TMEM columns [0, 128), the up accumulator in [128, 256).
  // (Two 128-column MMAs per step ran at about half the tensor rate.)
  static __device__ void mma_stage(const Job&, uint32_t d, uint32_t a0, uint32_t b0, int kb) {
    mma_stage_256(d, a0, b0, kb);
  }
  static __device__ void epilogue(const Params& p, const Job& j, uint32_t taddr, int q, int lane, EpiStage& es,
                                 int, int) {
    const int row = j.a_row + q * 32;
    if (j.kind == 1) {
#pragma unroll 1
      for (int ch = 0; ch < 2; ++ch) {
        float g[64], u[64];
        tmem_ld64(taddr, ch * 64, g);
        tmem_ld64(taddr, 128 + ch * 64, u);
#pragma unroll
        // SiLU(g) * u with the fast exp and divide intrinsics (a few ulp in fp32, far below
        // the bf16 rounding of h): the IEEE expf and division made this epilogue as long as
        // the tile's MMAs.  Very negative g gives an infinite or > 2^126 divisor and 0.
        for (int i = 0; i < 64; ++i) g[i] = __fdividef(g[i], 1.0f + __expf(-g[i])) * u[i];
        store_bf16_chunk(&p.h_st, es, lane, g, j.b_col + ch * 64, row);
      }
    } else {
#pragma unroll 1
      for (int ch = 0; ch < kBN / 64; ++ch) {
        float v[64];
        tmem_ld64(taddr, ch * 64, v);
        store_bf16_chunk(&p.y_st, es, lane, v, j.b_col + ch * 64, row);
      }
    }
  }
  static __device__ bool publishes(const Params&, const Job&) { return true; }
  static __device__ void publish(const Params& p, const Job& j) {
    if (j.kind == 1)
      st_release_gpu(p.up_flags + static_cast<size_t>(j.x0) * p.n_up + j.x1, p.common.epoch);
    else
      st_release_gpu(p.y_flags + static_cast<size_t>(j.x0) * p.n_down + j.x1, p.common.epoch);
  }
  // Combine: y tiles are claimed in the order the GEMM partition produces them, from a
  // counter (combine_next); for each valid row a = (t, j): out[t, cols] += gate_a * y[a, cols]
  // (fp32 vector reductions; with a zeroed out and top-2, 0 + a + b == 0 + b + a, so the
  // result does not depend on which contribution lands first or which CTA adds it).  The
  // combine partition claims tiles from the start; each GEMM-partition CTA joins after its
  // last GEMM tile (after_gemm), so the tiles still waiting when the GEMM work ends are
  // spread over the whole grid instead of queueing on the partition.
  //
  // A CTA runs two independent halves (warps 0-3 and 4-7), each with its own 64 KB
  // shared-memory tile buffer: the half's first warp claims a tile, waits on its signal, one
  // lane TMA-loads the 128 x 256 y tile, and the half stages the 128 rows' (token, gate)
  // records.  Each warp then takes 32 rows: for every row, lane l scales columns
  // [4l, 4l+4) and [128+4l, 128+4l+4) by the gate and adds them into out[token] with two
  // fp32 vector reductions, so each warp instruction covers 512 contiguous bytes of the
  // output row.  While one half waits for its load the other reduces.
  template <bool Trace>
  static __device__ void combine(const Params& p, int warp, int lane, uint8_t* smem_raw) {
    uint8_t* base =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int kTileBytes = kBM * kBN * 2;  // 64 KB of bf16 y
    const int half = warp >> 2;
    if (half > 1) return;
    const int hw = warp & 3;  // warp inside the half
    uint8_t* buf = base + half * kTileBytes;
    int2* meta = reinterpret_cast<int2*>(base + 2 * kTileBytes) + half * kBM;
    uint8_t* ctl = base + 2 * kTileBytes + 2 * kBM * sizeof(int2);
    uint64_t* bar = reinterpret_cast<uint64_t*>(ctl) + half;
    int* claim = reinterpret_cast<int*>(ctl + 2 * sizeof(uint64_t)) + half;  // the half's claimed tile
    if (hw == 0 && lane == 0) {
      mbar_init(bar, 1);
      fence_mbar_init();
    }
    const int m = mtiles(p);
    const int total = m * p.n_down;
    // This lane's two 4-column groups: box g (64 columns each), byte offset inside the 128-B row.
    const int g0 = lane >> 4, g1 = 2 + (lane >> 4);
    const int piece = (lane & 15) >> 1, sub = (lane & 1) * 8;
    uint32_t phase = 0;
    for (;;) {
      if (hw == 0 && lane == 0) *claim = atomicAdd(p.combine_next, 1);
      named_bar_sync(1 + half, 128);
      const int v = *reinterpret_cast<volatile int*>(claim);
      if (v >= total) break;
      const MoeSlot sl = down_slot(p, m, v);
      if (hw == 0) {
        const uint64_t w0 = Trace ? globaltimer() : 0;
        warp_wait_one(p.y_flags + static_cast<size_t>(sl.i) * p.n_down + sl.nb, p.common.epoch, p.common, lane,
                      kSiteCombine, (4ull << 60) | v);
        if (Trace && lane == 0) {
          const uint64_t w1 = globaltimer();
          if (w1 - w0 > kTraceMinWaitNs) trace_span(p.common, kTrSideWait, v, w0, w1);
          trace_open(p.common, kTrSideTile, v, w0);
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar, kTileBytes);
#pragma unroll
          for (int g = 0; g < kBN / 64; ++g)
            tma_load_2d(buf + g * (kBM * 128), &p.y_ld, bar, sl.nb * kBN + g * 64, sl.i * kBM);
        }
      }
      const int tid = hw * 32 + lane;  // one row record per thread of the half
      meta[tid] = __ldcg(p.row_meta + sl.i * kBM + tid);
      mbar_wait(bar, phase, p.common, kSiteCombine);
      phase ^= 1u;
      named_bar_sync(1 + half, 128);
      const uint32_t b0 = smem_u32(buf);
#pragma unroll 4
      for (int r = hw * 32; r < hw * 32 + 32; ++r) {
        const int2 md = meta[r];
        if (md.x < 0) continue;
        // 128-byte swizzle of the TMA box: 16-byte piece j of row r sits at j ^ (r & 7)
        const uint32_t off = r * 128 + (((piece ^ (r & 7))) << 4) + sub;
        uint32_t a0, a1, c0, c1;
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(a0), "=r"(a1) : "r"(b0 + g0 * (kBM * 128) + off));
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(c0), "=r"(c1) : "r"(b0 + g1 * (kBM * 128) + off));
        const float gt = __int_as_float(md.y);
        const float2 fa = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&a0));
        const float2 fb = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&a1));
        const float2 fc = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&c0));
        const float2 fd = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&c1));
        float* o = p.out + static_cast<size_t>(md.x) * p.H + sl.nb * kBN + lane * 4;
        red_add_v4(o, gt * fa.x, gt * fa.y, gt * fb.x, gt * fb.y);
        red_add_v4(o + 128, gt * fc.x, gt * fc.y, gt * fd.x, gt * fd.y);
      }
      named_bar_sync(1 + half, 128);  // the tile buffer, records and claim are free again
      if (Trace && hw == 0 && lane == 0) trace_close(p.common, globaltimer());
    }
  }
  template <bool Trace>
  static __device__ void side_role(const Params& p, int warp, int lane, uint8_t* smem_raw) {
    combine<Trace>(p, warp, lane, smem_raw);
  }
  // The operand ring the tile buffers now reuse was last written by TMA and read by the
  // tensor cores (the async proxy): order those accesses before this thread's own.
  template <bool Trace>
  static __device__ void after_gemm(const Params& p, int warp, int lane, uint8_t* smem_raw) {
    fence_proxy_async_smem();
    combine<Trace>(p, warp, lane, smem_raw);
  }
};

}  // namespace tl

using namespace tl;

// ============================================================================ C ABI
static size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

struct MoeLayout {
  size_t experts, gates, perm, row_meta, tile_expert, tile_rows, num_mtiles, counts, xp, h, y, up_flags, y_flags,
      x_flags, combine_next, total;
  int rmax;
};

static MoeLayout moe_layout(int T, int H, int E, int F, int topk) {
  MoeLayout L;
  const size_t n = static_cast<size_t>(T) * topk;
  const long long r = static_cast<long long>(n) + 127LL * E;
  L.rmax = static_cast<int>((r + kBM - 1) / kBM * kBM);
  const size_t tiles = L.rmax / kBM;
  size_t o = 0;
  L.experts = o; o += al256(n * 4);
  L.gates = o; o += al256(n * 4);
  L.perm = o; o += al256(n * 4);
  L.row_meta = o; o += al256(static_cast<size_t>(L.rmax) * 8);
  L.tile_expert = o; o += al256(tiles * 4);
  L.tile_rows = o; o += al256(tiles * 4);
  L.num_mtiles = o; o += 256;
  L.counts = o; o += al256(static_cast<size_t>(E) * 4);
  L.xp = o; o += al256(static_cast<size_t>(L.rmax) * H * 2);
  L.h = o; o += al256(static_cast<size_t>(L.rmax) * F * 2);
  L.y = o; o += al256(static_cast<size_t>(L.rmax) * H * 2);
  L.up_flags = o; o += al256(tiles * (F / 128) * 8);
  L.y_flags = o; o += al256(tiles * (H / kBN) * 8);
  L.x_flags = o; o += al256(tiles * kGatherPieces * 8);
  L.combine_next = o; o += 256;
  L.total = o;
  return L;
}

// Row tiles per chunk of the tile order, and the lag of a down chunk behind its up chunk: at
// least the number of chunks, so every up tile runs before the first down tile.  With the
// GEMM CTAs joining the combine after their last tile, starting the down tiles (and the
// combine) early no longer pays: 252.9 us against 267.3 us with a lag of 6 chunks on the
// 4096-token, 64-expert layer.
constexpr int kMoeChunk = 2;
static int moe_lag(const MoeLayout& L) { return (L.rmax / kBM + kMoeChunk - 1) / kMoeChunk; }

static bool moe_shape_ok(int T, int H, int E, int F, int topk) {
  return T >= 1 && topk >= 1 && topk <= kMaxTopk && E >= topk && E <= kMaxExperts && H > 0 && F > 0 &&
         H % kBN == 0 && F % 128 == 0 && static_cast<long long>(T) * topk < (1LL << 30);
}

extern "C" size_t tl_moe_workspace_bytes(int T, int H, int E, int F, int topk) {
  if (!moe_shape_ok(T, H, E, F, topk)) return 0;
  return moe_layout(T, H, E, F, topk).total;
}

// The order tl_moe_combine's persistent kernel uses for a layer whose routing produced
// m_tiles padded row tiles (kind 1 = up, 2 = down, row tile, column block).
extern "C" int tl_moe_tile_order(int T, int H, int E, int F, int topk, int m_tiles, int* kind, int* row_tile,
                                 int* col_block, int cap) {
  if (!moe_shape_ok(T, H, E, F, topk)) return TL_ERR_INVALID;
  const MoeLayout L = moe_layout(T, H, E, F, topk);
  if (m_tiles < 0 || m_tiles > L.rmax / kBM) return TL_ERR_INVALID;
  const MoeOrder o{m_tiles, F / 128, H / kBN, kMoeChunk, moe_lag(L)};
  const int total = m_tiles * (o.n_up + o.n_down);
  if (!kind && !row_tile && !col_block) return total;
  if (!kind || !row_tile || !col_block || cap < total) return TL_ERR_INVALID;
  for (int t = 0; t < total; ++t) {
    const MoeSlot sl = moe_slot(o, t);
    kind[t] = sl.kind;
    row_tile[t] = sl.i;
    col_block[t] = sl.nb;
  }
  return total;
}

// The order the combine claims y tiles in (row tile, column block).
extern "C" int tl_moe_combine_order(int T, int H, int E, int F, int topk, int m_tiles, int* row_tile,
                                    int* col_block, int cap) {
  if (!moe_shape_ok(T, H, E, F, topk)) return TL_ERR_INVALID;
  const MoeLayout L = moe_layout(T, H, E, F, topk);
  if (m_tiles < 0 || m_tiles > L.rmax / kBM) return TL_ERR_INVALID;
  const MoeOrder o{m_tiles, F / 128, H / kBN, kMoeChunk, moe_lag(L)};
  const int total = m_tiles * o.n_down;
  if (!row_tile && !col_block) return total;
  if (!row_tile || !col_block || cap < total) return TL_ERR_INVALID;
  for (int v = 0; v < total; ++v) {
    const MoeSlot sl = moe_down_slot(o, v);
    row_tile[v] = sl.i;
    col_block[v] = sl.nb;
  }
  return total;
}

extern "C" int tl_moe_combine(tl_ctx* ctx, const void* x, const float* logits, int topk, const void* w_gate,
                              const void* w_up, const void* w_down, float* out, int* perm_out, int* counts_out,
                              void* workspace, size_t workspace_bytes, int T, int H, int E, int F,
                              tl_stream_t stream) {
  if (!ctx || !moe_shape_ok(T, H, E, F, topk)) return TL_ERR_INVALID;
  if (!x || !logits || !w_gate || !w_up || !w_down || !out || !workspace) return TL_ERR_INVALID;
  if (!aligned16(x) || !aligned16(logits) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
      !aligned16(out) || !aligned16(workspace) || (perm_out && !aligned16(perm_out)) ||
      (counts_out && !aligned16(counts_out)))
    return TL_ERR_INVALID;
  if (workspace_bytes < tl_moe_workspace_bytes(T, H, E, F, topk)) return TL_ERR_WORKSPACE;
  if (ctx->ctas <= ctx->cfg.combine_ctas) return TL_ERR_UNSUPPORTED;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return TL_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const MoeLayout L = moe_layout(T, H, E, F, topk);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* experts = reinterpret_cast<int*>(ws + L.experts);
  float* gates = reinterpret_cast<float*>(ws + L.gates);
  int* perm = reinterpret_cast<int*>(ws + L.perm);
  int2* row_meta = reinterpret_cast<int2*>(ws + L.row_meta);
  int* tile_expert = reinterpret_cast<int*>(ws + L.tile_expert);
  int* tile_rows = reinterpret_cast<int*>(ws + L.tile_rows);
  int* num_mtiles = reinterpret_cast<int*>(ws + L.num_mtiles);
  int* counts = reinterpret_cast<int*>(ws + L.counts);
  __nv_bfloat16* xp = reinterpret_cast<__nv_bfloat16*>(ws + L.xp);
  __nv_bfloat16* hb = reinterpret_cast<__nv_bfloat16*>(ws + L.h);
  __nv_bfloat16* yb = reinterpret_cast<__nv_bfloat16*>(ws + L.y);

  // The persistent kernel's parameters and tensor maps first, so that its launch follows the
  // routing and permutation launches without host work in between.
  MoeParams p;
  std::memset(&p, 0, sizeof(p));
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!tmap_2d(&p.xp, BF, 2, xp, H, L.rmax, 64, 128) || !tmap_3d(&p.wg, BF, 2, w_gate, F, H, E, 64, 64, 1) ||
      !tmap_3d(&p.wu, BF, 2, w_up, F, H, E, 64, 64, 1) || !tmap_3d(&p.wd, BF, 2, w_down, H, F, E, 64, 64, 1) ||
      !tmap_2d(&p.h_st, BF, 2, hb, F, L.rmax, 64, 32) || !tmap_2d(&p.h_ld, BF, 2, hb, F, L.rmax, 64, 128) ||
      !tmap_2d(&p.y_st, BF, 2, yb, H, L.rmax, 64, 32) || !tmap_2d(&p.y_ld, BF, 2, yb, H, L.rmax, 64, 128))
    return TL_ERR_CUDA;
  p.common = make_common(ctx);
  p.num_mtiles = num_mtiles;
  p.tile_expert = tile_expert;
  p.tile_rows = tile_rows;
  p.row_meta = row_meta;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.xp_rows = xp;
  p.x_flags = reinterpret_cast<uint64_t*>(ws + L.x_flags);
  p.y = yb;
  p.out = out;
  p.up_flags = reinterpret_cast<uint64_t*>(ws + L.up_flags);
  p.y_flags = reinterpret_cast<uint64_t*>(ws + L.y_flags);
  p.combine_next = reinterpret_cast<int*>(ws + L.combine_next);
  p.T = T;
  p.H = H;
  p.E = E;
  p.F = F;
  p.topk = topk;
  p.n_up = F / 128;
  p.n_down = H / kBN;
  p.kb_up = H / kBK;
  p.kb_down = F / kBK;
  p.combine_ctas = ctx->cfg.combine_ctas;
  p.chunk = kMoeChunk;
  p.lag = moe_lag(L);
  moe_route_kernel<<<(T + 7) / 8, 256, 0, st>>>(logits, T, E, topk, ctx->cfg.moe_renorm, experts, gates);
  if (cudaGetLastError() != cudaSuccess) return TL_ERR_CUDA;
  const int zero_ctas = ctx->sms > E ? ctx->sms - E : 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(E + zero_ctas, 1, 1);
  lc.blockDim = dim3(1024, 1, 1);
  lc.stream = st;
  cudaLaunchAttribute la[1];
  la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  la[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = la;
  lc.numAttrs = 1;
  if (cudaLaunchKernelEx(&lc, moe_permute_kernel, static_cast<const int*>(experts), T * topk, E, topk,
                         static_cast<const float*>(gates), perm, row_meta, tile_expert, tile_rows, num_mtiles, counts,
                         perm_out, counts_out, reinterpret_cast<float4*>(out),
                         static_cast<size_t>(T) * H / 4, p.combine_next) != cudaSuccess) {
    (void)cudaGetLastError();
    return TL_ERR_CUDA;
  }

  // Two extra warps per CTA: the token gather in the GEMM partition, combine workers in the
  // combine CTAs.
  return launch_persistent<MoeOp>(ctx, p, st, 2);
}
