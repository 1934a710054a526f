// Static tile-centric mappings (host and device).
//
// "TileLink: Generating Efficient Compute-Communication Overlapping Kernels using
// Tile-Centric Primitives", §4.1: a static mapping sends a tile id to a shape range,
// a source rank and a channel by affine arithmetic.  Here the tile id is the
// position of a tile in the persistent GEMM's global sequence, and the order is the
// rank swizzle of "Triton-distributed: Programming Overlapping Kernels on
// Distributed AI Systems with the Triton Compiler", §3.7:
//   AllGather+GEMM: step s computes with the shard of rank (rank + s) mod W, so each
//     rank starts on its local shard while the next one is being pulled (inside a step,
//     groups of row blocks: see ag_tile).
//   GEMM+ReduceScatter: inside each L2-sized band of the output, producer p starts at the
//     rows of owner (p + 1) mod W (see rs_tile).
// The same functions are compiled for the host (tl_*_tile_order, used by the tests)
// and for the device (the persistent kernels), so both agree by construction.
#pragma once

#if defined(__CUDACC__)
#define TL_HD __host__ __device__ __forceinline__
#else
#define TL_HD inline
#endif

namespace tl {

constexpr int kBM = 128;  // GEMM tile rows (one UMMA M)
constexpr int kBN = 256;  // GEMM tile columns (one UMMA N)
constexpr int kBK = 64;   // K per pipeline stage (one 128-byte swizzle atom of bf16)

TL_HD int ceil_div(int a, int b) { return (a + b - 1) / b; }

struct AgTile {
  int src;  // rank whose shard feeds this tile's rows
  int mb;   // row block inside that shard
  int nb;   // column block of C
};

// AllGather + GEMM: W steps of (mps row blocks x nbk column blocks).
TL_HD int ag_num_tiles(int W, int mps, int nbk) { return W * mps * nbk; }
TL_HD int ag_step_rank(int W, int rank, int swizzle, int s) { return swizzle ? (rank + s) % W : s; }
// Inside a step the tiles run in groups of TL_AG_GROUP row blocks, the row block fastest
// inside a group: a wave of CTAs then covers a block about 8 row blocks tall instead of a
// few full rows of tiles, so it needs fewer distinct A and B panels at once (measured: the
// 8192 x 8192 x 3584 plain GEMM 263-264 us against 268-270 us row-major).  0 = row-major.
#ifndef TL_AG_GROUP
#define TL_AG_GROUP 8
#endif
TL_HD AgTile ag_tile(int t, int W, int rank, int mps, int nbk, int swizzle) {
  const int per_step = mps * nbk;
  const int s = t / per_step;
  const int rem = t - s * per_step;
  AgTile r;
  r.src = ag_step_rank(W, rank, swizzle, s);
  if (TL_AG_GROUP > 0) {
    // groups of TL_AG_GROUP row blocks, the row block fastest inside a group
    const int gsz = TL_AG_GROUP * nbk;
    const int g = rem / gsz, r2 = rem - g * gsz;
    const int rows = mps - g * TL_AG_GROUP < TL_AG_GROUP ? mps - g * TL_AG_GROUP : TL_AG_GROUP;
    r.nb = r2 / rows;
    r.mb = g * TL_AG_GROUP + (r2 - r.nb * rows);
  } else {
    r.mb = rem / nbk;
    r.nb = rem - r.mb * nbk;
  }
  return r;
}

// Mover order: the copy of step s's shard is issued before step s+1's, the
// self rank's own shard (needed by nobody) last.  Returns the shard rank copied
// as the i-th shard, i = 0..W-1.
TL_HD int ag_mover_rank(int W, int rank, int swizzle, int i) {
  if (swizzle) return (rank + 1 + i) % W;  // i = W-1 -> rank itself
  // identity order: 0, 1, ... skipping `rank`, then `rank` last
  if (i == W - 1) return rank;
  return i < rank ? i : i + 1;
}

struct RsTile {
  int p;   // producer (emulated rank computing the partial)
  int o;   // owner of the output rows
  int mb;  // row block inside the owner's rows
  int nb;  // column block
  int s;   // position of this partial in the tile's summation chain (0 .. W-1)
};

// GEMM + ReduceScatter, banded.  The m x n output is cut into bands of kRsBandRows rows x
// kRsBandCols columns (the last band in each direction may be smaller), visited in
// row-major order.  Inside a band the producers run in the order p = 0..W-1, the fixed fp32
// summation order, and producer p's tiles of the band run with the column block slowest and
// the row block fastest.  So the W partial tiles of one output tile are produced one band
// pass apart, while the band's fp32 slot tiles (2048 x 4096 x 4 B = 32 MiB) stay in L2; a
// producer's pass reads its A rows of the band once and each B column slab once per band.
// (A producer-major order, every producer over the whole output in turn, streams the whole
// m x n fp32 slot through DRAM once per producer.)
// Rank swizzle ("Triton-distributed ...", §3.7: start from the next rank's chunk, the local
// chunk last): inside a band, producer p starts at the first row of owner (p + 1) mod W
// when that owner has rows in the band, and wraps around the band's rows from there.
#ifndef TL_RS_BAND_ROWS
#define TL_RS_BAND_ROWS 2048
#endif
#ifndef TL_RS_BAND_COLS
#define TL_RS_BAND_COLS 4096
#endif
constexpr int kRsBandRows = TL_RS_BAND_ROWS;
constexpr int kRsBandCols = TL_RS_BAND_COLS;
TL_HD int rs_num_tiles(int W, int mbo, int nbk) { return W * W * mbo * nbk; }
// Owner order of one producer's pass over all owners (the MLP chain's layer 2): (p + 1 + s) mod W.
TL_HD int rs_owner(int W, int p, int s, int swizzle) { return swizzle ? (p + 1 + s) % W : s; }
TL_HD int rs_band_mt(int bm) { return kRsBandRows / bm > 0 ? kRsBandRows / bm : 1; }
TL_HD int rs_band_nt() { return kRsBandCols / kBN > 0 ? kRsBandCols / kBN : 1; }
// mbo: row tiles per owner (tiles of bm rows); nbk: column tiles of the output.
TL_HD RsTile rs_tile(int t, int W, int mbo, int nbk, int bm, int swizzle) {
  const int mt = W * mbo;  // row tiles of the whole output
  const int bmt = rs_band_mt(bm), bnt = rs_band_nt();
  const int per_rowband = W * bmt * nbk;  // tiles of a full band row (all producers)
  const int br = t / per_rowband;
  int rem = t - br * per_rowband;
  const int r0 = br * bmt;
  const int R = mt - r0 < bmt ? mt - r0 : bmt;  // rows of this band
  const int bc = rem / (W * R * bnt);
  rem -= bc * W * R * bnt;
  const int c0 = bc * bnt;
  const int C = nbk - c0 < bnt ? nbk - c0 : bnt;  // columns of this band
  RsTile r;
  r.p = rem / (R * C);
  rem -= r.p * R * C;
  r.nb = c0 + rem / R;
  const int i = rem - (rem / R) * R;
  int start = 0;  // rotation of the band's rows for this producer
  if (swizzle) {
    const int os = (r.p + 1) % W;  // the owner this producer serves first
    const int rs = os * mbo;        // that owner's first row tile
    if (rs + mbo > r0 && rs < r0 + R) start = rs > r0 ? rs - r0 : 0;
  }
  int row = r0 + (i + start) % R;
  r.o = row / mbo;
  r.mb = row - r.o * mbo;
  r.s = r.p;
  return r;
}

// GEMM + ReduceScatter as a ring ("TileLink ...", §5, Figure 4 text: each rank reduces the
// partial it receives with its own and passes the result on, peer_tile_wait /
// peer_tile_notify between neighbours).  The partial of an output tile of owner o starts at
// rank o + 1 and travels o+1 -> o+2 -> ... -> o (mod W): hop s is computed by producer
// (o + 1 + s) mod W, and the owner, the last hop, writes bf16.  Order: owner by owner; each
// owner's rows in bands of kRsBandRows rows x kRsBandCols columns; inside a band the hops
// s = 0..W-1 in turn (every tile of a band at one hop shares one producer, so its B column
// slabs serve all the band's rows), and inside a hop the column block slowest, the row block
// fastest.  A hop waits only on the same tile's previous hop, earlier in the sequence.
TL_HD RsTile rs_ring_tile(int t, int W, int mbo, int nbk, int bm) {
  const int bmt = rs_band_mt(bm), bnt = rs_band_nt();
  const int per_owner = W * mbo * nbk;
  RsTile r;
  r.o = t / per_owner;
  int rem = t - r.o * per_owner;
  const int per_rowband = W * bmt * nbk;
  const int br = rem / per_rowband;
  rem -= br * per_rowband;
  const int r0 = br * bmt;
  const int R = mbo - r0 < bmt ? mbo - r0 : bmt;
  const int bc = rem / (W * R * bnt);
  rem -= bc * W * R * bnt;
  const int c0 = bc * bnt;
  const int C = nbk - c0 < bnt ? nbk - c0 : bnt;
  r.s = rem / (R * C);
  rem -= r.s * R * C;
  r.nb = c0 + rem / R;
  r.mb = r0 + rem - (rem / R) * R;
  r.p = (r.o + 1 + r.s) % W;
  return r;
}
}  // namespace tl
