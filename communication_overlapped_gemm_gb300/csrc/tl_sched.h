// Static tile-centric mappings (host and device).
//
// "TileLink: Generating Efficient Compute-Communication Overlapping Kernels using
// Tile-Centric Primitives", §4.1: a static mapping sends a tile id to a shape range,
// a source rank and a channel by affine arithmetic.  Here the tile id is the
// position of a tile in the persistent GEMM's global sequence, and the order is the
// rank swizzle of "Triton-distributed: Programming Overlapping Kernels on
// Distributed AI Systems with the Triton Compiler", §3.7:
//   AllGather+GEMM: step s computes with the shard of rank (rank + s) mod W, so each
//     rank starts on its local shard while the next one is being pulled.
//   GEMM+ReduceScatter: producer p walks owners (p + 1 + s) mod W, its own rows last,
//     so the chunk that must travel furthest is produced first.
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
TL_HD AgTile ag_tile(int t, int W, int rank, int mps, int nbk, int swizzle) {
  const int per_step = mps * nbk;
  const int s = t / per_step;
  const int rem = t - s * per_step;
  AgTile r;
  r.src = ag_step_rank(W, rank, swizzle, s);
  r.mb = rem / nbk;
  r.nb = rem - r.mb * nbk;
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
};

// GEMM + ReduceScatter: producers in order p = 0..W-1 (the fixed fp32 summation order).
// Producer p walks its W owners in the order (p + 1 + s) mod W, s = 0..W-1, taken in groups
// of kRsOwnerGroup consecutive owners.  Inside a group the column block is the slowest
// index and the owner's row block the fastest, so the tiles that run at the same time
// share a few column slabs of B_p and the group's rows of A_p: B_p is read once per owner
// group rather than once per wave of tiles.  Owners still come first in the rotated order,
// the producer's own rows in the last group.
constexpr int kRsOwnerGroup = 4;
TL_HD int rs_num_tiles(int W, int mbo, int nbk) { return W * W * mbo * nbk; }
TL_HD int rs_owner(int W, int p, int s, int swizzle) { return swizzle ? (p + 1 + s) % W : s; }
TL_HD RsTile rs_tile(int t, int W, int mbo, int nbk, int swizzle) {
  const int per_prod = W * mbo * nbk;
  RsTile r;
  r.p = t / per_prod;
  int rem = t - r.p * per_prod;
  const int full_group = kRsOwnerGroup * mbo * nbk;  // tiles of a group of kRsOwnerGroup owners
  const int g = rem / full_group;                     // every group but the last is full
  rem -= g * full_group;
  const int s0 = g * kRsOwnerGroup;
  const int gsz = W - s0 < kRsOwnerGroup ? W - s0 : kRsOwnerGroup;  // owners in this group
  r.nb = rem / (gsz * mbo);
  rem -= r.nb * gsz * mbo;
  const int s = s0 + rem / mbo;
  r.mb = rem - (s - s0) * mbo;
  r.o = rs_owner(W, r.p, s, swizzle);
  return r;
}

}  // namespace tl
