/*
 * tl.h - C ABI of the GB300 (sm_103a) tile-centric communication-overlapped GEMM library.
 *
 * The library computes, on ONE GPU, the four overlapped operators of the pages it is
 * built from, with the W tensor-parallel ranks emulated as W separate HBM buffers:
 *
 *   tl_ag_gemm      AllGather + GEMM:        C = [A_0; A_1; ...; A_{W-1}] . B
 *   tl_gemm_rs      GEMM + ReduceScatter:    out_o = rows_o( sum_p A_p . B_p )
 *   tl_mlp2         2-layer MLP chain:       out_o = rows_o( sum_r GELU(AG(X) . W1_r) . W2_r )
 *   tl_moe_combine  top-k MoE layer:         out_t = sum_j g_tj * (SiLU(x_t Wg_e) * (x_t Wu_e)) Wd_e
 *
 * "Communication" is the movement of shards between the ranks' buffers inside one HBM,
 * done by mover warps that publish per-chunk release flags; the persistent tcgen05 GEMM
 * waits on those flags (acquire) before its TMA loads, walking its tiles in a rank-swizzled
 * order that starts from the local shard.
 *
 * Sources (page titles; sections as printed on the pages):
 *   [TL] TileLink: Generating Efficient Compute-Communication Overlapping Kernels using
 *        Tile-Centric Primitives - §2.1 (tensor-parallel FFN), §3.1 (decoupled tile size /
 *        order / resource binding), §3.2 Table 3 (producer_tile_notify, consumer_tile_wait,
 *        peer_tile_notify/wait, tile_push_data, tile_pull_data), §4.1 (static and dynamic
 *        tile-centric mapping), §4.2 (release/acquire lowering), §6 (BlockChannel context).
 *   [TD] Triton-distributed: Programming Overlapping Kernels on Distributed AI Systems with
 *        the Triton Compiler - §2.1 (symmetric memory, signal exchange, async tasks),
 *        §3.2 Algorithm 2 (pull-mode AllGather), §3.3 Algorithm 3 (push-mode ReduceScatter),
 *        §3.7 (tile swizzle for AG+GEMM and GEMM+RS), §3.8 (signal reset, resource partition).
 *   [RA] Resource-aware Computation-Communication Overlap for multi-GPU ML Workloads -
 *        CTA-pipelining abstract (2-layer GEMM with CTA-level dependencies) and the MoE
 *        abstract (persistent expert producer, persistent combine consumer on a small
 *        dedicated SM partition, tile-level signalling).
 *
 * Conventions for every entry point
 *   - Matrices are row-major bf16 (IEEE bfloat16, passed as raw 16-bit storage), fp32 where
 *     stated.  Every device pointer must be 16-byte aligned.  Accumulation is fp32.
 *   - Ownership: the caller allocates every device buffer, including the workspace (size from
 *     the matching *_workspace_bytes function).  The library owns only the context (a small
 *     device status word).  No entry point allocates device memory.
 *   - A workspace must be zero-filled once before its first use (e.g. cudaMemset) and again
 *     after any call whose tl_ctx_check reported an error; between successful calls the
 *     library keeps it valid itself (its signals are epoch-valued, never reset).
 *   - Calls are asynchronous on `stream` and return once the work is enqueued.  Two calls that
 *     share a workspace must be ordered (same stream, or events).
 *   - Return values: TL_OK (0) or a negative TL_ERR_* code.  Argument errors are reported
 *     before anything is enqueued.  Device-side errors (a bounded wait that ran out) are read
 *     with tl_ctx_check after the stream has been synchronised.
 *   - Threading: a context is not thread-safe; use one per host thread.
 */
#ifndef TL_GB300_H
#define TL_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* == cudaStream_t / CUstream */
typedef struct CUstream_st* tl_stream_t;

/* ---------------------------------------------------------------- status codes */
#define TL_OK 0
#define TL_ERR_INVALID (-1)     /* null / misaligned pointer, unsupported shape, bad config      */
#define TL_ERR_UNSUPPORTED (-2) /* device is not sm_103 / co-residency of the persistent grid fails */
#define TL_ERR_CUDA (-3)        /* a CUDA runtime or driver call failed                          */
#define TL_ERR_TIMEOUT (-4)     /* (tl_ctx_check) a bounded device wait on a signal ran out        */
#define TL_ERR_WORKSPACE (-5)   /* workspace smaller than *_workspace_bytes                     */

/* ---------------------------------------------------------------- configuration
 * The BlockChannel-like launch context of [TL] §6: rank/world come per call; this struct
 * carries the decoupled design-space choices of [TL] §3.1 (communication tile size = mover
 * chunk, tile order = swizzle, resource binding = mover warps / combine partition) and the
 * bound on every device-side wait.
 */
typedef struct tl_config {
  int mover_warps;            /* warps per persistent CTA that move shards (1..4; default 4)          */
  int chunks_per_slab;        /* mover chunks, hence signals, per 128-row slab (1..32; default 32)     */
  int swizzle;                /* 0: identity tile order; 1: rank-swizzled ([TD] §3.7; default)          */
  int grid_ctas;              /* persistent CTAs; 0 = one per SM (default)                              */
  int combine_ctas;           /* MoE combine partition, CTAs = SMs ([RA]; default 8)                    */
  int debug_skip_chunk;       /* fault injection: this mover chunk is copied but never signalled (-1 off) */
  unsigned long long timeout_ns; /* bound of every device wait (default 2e9 ns)                       */
  int pair_ctas;              /* where shards / owner blocks are 256-row multiples, 256 x 256 tiles run
                                 on: 0 single CTAs; 1 CTA pairs (two SMs, tcgen05 cta_group::2) for
                                 every op; 2 (default) CTA pairs for tl_gemm_rs and tl_mlp2, whose
                                 heavier epilogues gain from the pair's double-buffered
                                 accumulators, single CTAs for tl_ag_gemm                           */
  int moe_renorm;             /* MoE gates: 0 (default) the softmax over all E logits taken at the
                                 chosen experts; 1 those values divided by their sum over the topk
                                 chosen experts (they then sum to 1 per token)                      */
  int rs_ring;                /* tl_gemm_rs reduction: 0 (default) the owner-slot chain; 1 a ring
                                 ([TL] §5, Figure 4 text), workspace from
                                 tl_gemm_rs_ring_workspace_bytes                                    */
  int ag_push;                /* tl_mlp2's AllGather, where every rank gathers: 0 (default) pull
                                 ([TD] §3.2 Algorithm 2, each rank reads every other shard); 1 push
                                 (Algorithm 1, each shard read once and written to the other ranks'
                                 copies).  tl_ag_gemm and tl_allgather gather into one rank, where
                                 both modes move the same bytes: they always pull              */
  int mover_kparts;           /* tl_ag_gemm's mover chunks along K ([TL] §3.1, the communication
                                 tile): 1 each chunk is whole rows of a 128-row slab; 2 or 4 each
                                 slab of the first two shards gathered is also cut into that many
                                 K parts (of at least 16 64-column k-blocks), copied part by
                                 part, and a tile waits for each part before its first k-block in
                                 it; 0 (default) 4.  tl_allgather and tl_mlp2 always copy whole
                                 rows (as measured on GB300, K parts only slow them)          */
  int ag_ll;                  /* tl_ag_gemm's gather protocol: 0 (default) pull with one signal
                                 per chunk; 1 low-latency push ([TD] §3.2 Algorithm 1 with the
                                 flag carried in every word): the remote shards' owners write
                                 8-byte words {bf16 x 2, call signal} into the workspace's LL
                                 slabs and each tile reads them straight into its operand
                                 buffer, with no separate signal or fence.  For small problems
                                 only (tl_ag_gemm_ll_capable); otherwise TL_ERR_UNSUPPORTED  */
  int mover_tma;              /* tl_allgather's copy engine: 0 (default) the SMs' load/store path
                                 (16-byte vectors, several CTAs of copy warps per SM); 1 the TMA
                                 unit of each SM (bulk copies through shared-memory stages, one
                                 issuing thread per SM): the pages' copy-engine mover ([TL]
                                 §7.2) in its GB300 form.  Same result and signals.          */
} tl_config;

typedef struct tl_ctx tl_ctx;

/* Fill *cfg with the defaults above.  Returns TL_OK, or TL_ERR_INVALID for cfg == NULL. */
int tl_config_default(tl_config* cfg);

/* Create a context on `device` (must be compute capability 10.3, i.e. sm_103).  cfg may be
 * NULL (defaults).  Allocates one small device status word.  On failure *out is NULL. */
int tl_ctx_create(tl_ctx** out, int device, const tl_config* cfg);

/* Destroy a context (NULL is ignored).  Synchronises the device first. */
void tl_ctx_destroy(tl_ctx* ctx);

/* Read and clear the device status word.  Call after synchronising the streams used with ctx.
 * Returns TL_OK, or TL_ERR_TIMEOUT if a bounded wait ran out (the results of that call are
 * undefined and its workspace must be zero-filled again), or TL_ERR_CUDA. */
int tl_ctx_check(tl_ctx* ctx);

/* Human-readable text for a status code (static storage). */
const char* tl_strerror(int code);

/* Library version, major*10000 + minor*100 + patch. */
int tl_version(void);

/* Number of SMs / persistent CTAs the context launches with. */
int tl_ctx_num_ctas(const tl_ctx* ctx);

/* ---------------------------------------------------------------- trace buffer
 * A per-CTA timeline of the persistent kernels.  Every warp role records spans into a
 * caller-owned device buffer.  A span is a %globaltimer start, a duration in ns, and a kind
 * plus a tile or chunk index.  The pages name no such facility.  It shows where a fused kernel
 * waits: a mover chunk landing, a tile waiting on its signal, the MMA warp starved of data.
 *
 * tl_trace_bytes(ctas, spans_per_warp): bytes a buffer needs to hold `ctas` CTAs.
 * tl_ctx_set_trace(ctx, buf, bytes, spans_per_warp): every later persistent-kernel launch on
 *   ctx records into buf.  buf is device memory, 16-byte aligned and caller-owned; it must stay
 *   valid while such launches run.  buf NULL turns tracing off.  Each launch overwrites the
 *   previous trace.  CTAs beyond what `bytes` holds are not recorded.  Spans beyond
 *   spans_per_warp are dropped, but the per-warp count still counts them.
 *   Returns TL_ERR_INVALID for a null ctx, a misaligned buf, a size below
 *   tl_trace_bytes(1, spans_per_warp), or spans_per_warp < 1.
 * Layout (little-endian), written by the kernels:
 *   uint32 header[8]: magic 0x544c5452, version 1, grid of the last launch, warps per CTA (16),
 *                     spans per warp, CTAs held, 0, 0
 *   uint32 count[CTAs held][16]: spans each warp recorded (may exceed spans per warp)
 *   span[CTAs held][16][spans per warp], 16 bytes each: uint64 t0_ns, uint32 dur_ns,
 *                     uint32 tag = kind << 24 | index
 * Kinds:
 *   1 producer tile; 2 producer signal wait; 3 producer ring-stall total (t0 = tile start);
 *   4 MMA tile; 5 MMA starve total (t0 = tile start); 6 MMA accumulator wait;
 *   7 epilogue tile; 8 epilogue accumulator wait;
 *   9 mover chunk; 10 side-partition unit (from the start of its wait); 11 side-partition wait.
 * Waits shorter than 200 ns are not recorded.
 * Warp w of a GEMM CTA: 0 producer, 1 MMA, 2.. epilogue, then the movers.  In a side partition
 * (the MoE combine CTAs) warps 0 and 4 record.  Only the persistent kernels trace.  While on,
 * tracing costs a few timer reads per tile and k-block.
 */
size_t tl_trace_bytes(int ctas, int spans_per_warp);
int tl_ctx_set_trace(tl_ctx* ctx, void* buf, size_t bytes, int spans_per_warp);

/* ---------------------------------------------------------------- AllGather + GEMM
 * [TL] §2.1, [TD] §3.2 Algorithm 2 (pull mode) and §3.7 (AG+GEMM swizzle).
 *
 *   C[(W*m_per_rank) x n] = A . B,  A = [A_0; ...; A_{W-1}] (rank order), B [k x n].
 *
 * a_shards: host array of W device pointers, shard r is bf16 [m_per_rank x k] (rank r's
 *           "local buffer").  b: bf16 [k x n].  c: bf16 [(W*m_per_rank) x n] (output).
 * workspace: device buffer of tl_ag_gemm_workspace_bytes(); its first W*m_per_rank*k*2
 *           bytes are the gathered A (the symmetric buffer T of Algorithm 2, rank order), the
 *           rest holds the per-chunk ready signals.
 * The emulated self rank `rank` (0 <= rank < W) reads its own shard in place; the mover pulls
 * the remote shards (rank+1) mod W, (rank+2) mod W, ... into their slots of T in that order,
 * and the GEMM visits row blocks of shard rank first, then (rank+1) mod W, ... waiting on each
 * slab's signals before its first load.  The self rank's slot of T is not written (nothing
 * reads it; tl_allgather fills all W slots).  The result does not depend on `rank` or the
 * swizzle.
 * W = 1 has nothing to gather: the call is the plain GEMM on shard 0, read in place, and the
 * gathered region of the workspace is not written.
 * Shapes: 1 <= W <= 8; m_per_rank % 128 == 0; n % 8 == 0; k % 8 == 0 (n, k need not be
 * tile multiples: ragged edges are zero-filled by TMA on load and clipped on store).
 * Any zero dimension is a no-op returning TL_OK.
 * Low-latency gather (cfg.ag_ll = 1, W > 1): instead of the mover and its chunk signals, the
 * owners of the remote shards push them as LL words {bf16 x 2, low 32 bits of the call's
 * signal} into the workspace's LL slabs, after the signal words, and every 128 x 256 output
 * tile reads the words of its rows straight into its operand buffer, polling only those that
 * do not carry this call's signal yet.  The gathered region is not written.  The result is
 * the same operation; for m_per_rank % 256 != 0 it is bit-identical to the pull path (the
 * same 128-row MMAs in the same k order).  Only problems with W * m_per_rank * k <= 2^20
 * (their workspace has the LL slabs) and at most (the context's CTAs - 1) output tiles can
 * take it (tl_ag_gemm_ll_capable); others return TL_ERR_UNSUPPORTED with nothing enqueued.
 * The LL slabs need no zeroing between calls on one context.
 */
size_t tl_ag_gemm_workspace_bytes(int W, int m_per_rank, int n, int k);
int tl_ag_gemm(tl_ctx* ctx, int W, int rank, const void* const* a_shards, const void* b, void* c,
               void* workspace, size_t workspace_bytes, int m_per_rank, int n, int k, tl_stream_t stream);
/* 1 if tl_ag_gemm on ctx with cfg.ag_ll = 1 runs the low-latency gather for this shape, else 0
 * (also 0 for a NULL ctx or a negative size; W = 1 has nothing to gather: 0). */
int tl_ag_gemm_ll_capable(const tl_ctx* ctx, int W, int m_per_rank, int n, int k);

/* ---------------------------------------------------------------- AllGather alone
 * [TD] §3.2 Algorithm 2 (pull-mode one-sided AllGather) as its own kernel: the shard mover of
 * tl_ag_gemm (same chunk order and signals, whole-row chunks) without the GEMM, run by four
 * CTAs of 16 warps per SM, two resident at a time (alone, the copy has the whole GPU).  Fills
 * the gathered buffer at the start of `workspace` (sized by tl_ag_gemm_workspace_bytes(W,
 * m_per_rank, 8, k)) with all of
 * [A_0; ...; A_{W-1}], the self rank's shard last, and releases every chunk signal.  Shapes
 * and errors as tl_ag_gemm; W = 1 is a no-op.  This is the "communication alone" leg of the
 * overlap measurement.
 */
int tl_allgather(tl_ctx* ctx, int W, int rank, const void* const* a_shards, void* workspace, size_t workspace_bytes,
                 int m_per_rank, int k, tl_stream_t stream);

/* ---------------------------------------------------------------- GEMM + ReduceScatter
 * [TD] §3.3 Algorithm 3 (each producer pushes its partial into the owner's slot, the owner
 * accumulates), [TL] §5 / Figure 4 text (producer tiles notify; peer tiles chain the partial
 * sums from rank to rank) and [TD] §3.7 (start at the next rank's chunk, own chunk last).
 *
 *   out_o [(m/W) x n] = rows [o*m/W, (o+1)*m/W) of  sum_{p=0}^{W-1} A_p . B_p
 *
 * a: W device pointers, A_p bf16 [m x k_r];  b: W device pointers, B_p bf16 [k_r x n];
 * out: W device pointers, out_o bf16 [(m/W) x n].
 * Owner-slot chain (cfg.rs_ring = 0, default).  workspace: tl_gemm_rs_workspace_bytes(): an
 * fp32 [m x n] accumulation slot (owner o owns rows o*m/W..) plus one signal per 128-row block
 * and 256-column block of the output.  The output is walked in bands of 2048 rows x 4096
 * columns; inside a band the producers run p = 0..W-1, producer p starting at the rows of
 * owner (p+1) mod W when the band holds some (swizzle = 1).  Producer 0 stores its partial
 * tile into the slot, producer p > 0 waits for producer p-1's signal on that tile
 * (peer_tile_wait) and adds its partial with a TMA bulk reduction, and producer W-1 adds its
 * partial to the slot in registers and writes bf16 out_o.  The fp32 summation order is fixed
 * (p = 0, 1, ..., W-1): results are bit-identical across runs, swizzle modes and grid sizes.
 * Ring (cfg.rs_ring = 1).  workspace: tl_gemm_rs_ring_workspace_bytes(): W fp32 [m x n]
 * receive buffers (rank q's at q*m*n*4 bytes), then the signals.  The partial of an output
 * tile of owner o starts at rank o+1 and travels o+1 -> o+2 -> ... -> o (mod W): each rank
 * waits for its predecessor's signal on the tile (peer_tile_wait), adds the partial in its
 * receive buffer to its own, stores the sum into the next rank's receive buffer and signals
 * it (peer_tile_notify); the owner, last, writes bf16 out_o.  The fp32 order of owner o's
 * rows is P_{o+1} + P_{o+2} + ... + P_o: fixed, so results are bit-identical run to run.
 * Shapes: 1 <= W <= 8; m % (128*W) == 0; n % 8 == 0; k_r % 8 == 0.
 */
size_t tl_gemm_rs_workspace_bytes(int W, int m, int n, int k_r);
size_t tl_gemm_rs_ring_workspace_bytes(int W, int m, int n, int k_r);
int tl_gemm_rs(tl_ctx* ctx, int W, const void* const* a, const void* const* b, void* const* out,
               void* workspace, size_t workspace_bytes, int m, int n, int k_r, tl_stream_t stream);

/* ---------------------------------------------------------------- ReduceScatter alone
 * [TD] §3.3 Algorithm 3 (push-mode ReduceScatter) as its own kernel, without a GEMM: the
 * communication half of tl_gemm_rs, and its "communication alone" leg in an overlap
 * measurement.
 *
 *   out_o [(m/W) x n] = rows [o*m/W, (o+1)*m/W) of  P_0 + P_1 + ... + P_{W-1}
 *
 * partials: host array of W device pointers, P_p fp32 [m x n] row-major (rank p's partial);
 * out: W device pointers, out_o bf16 [(m/W) x n].  The sum is taken in fp32 in the order
 * p = 0, 1, ..., W-1 (the order of tl_gemm_rs's chain) and rounded to bf16 once, so the
 * result is bit-identical run to run.  No workspace.  Partials are read once.
 * Shapes: 1 <= W <= 8; m % W == 0; n % 4 == 0.  m == 0 or n == 0 is a no-op.
 */
int tl_reduce_scatter(tl_ctx* ctx, int W, const float* const* partials, void* const* out, int m, int n,
                      tl_stream_t stream);

/* ---------------------------------------------------------------- 2-layer MLP chain
 * [TL] §2.1 (AG + GEMM -> activation -> GEMM + RS), [RA] CTA-pipelining (the second GEMM's
 * CTAs start as soon as the first GEMM's CTAs that produce their inputs are done).
 *
 *   X = [X_0; ...; X_{W-1}]  (tokens x hidden),   H_r = GELU(X . W1_r)  (exact erf GELU),
 *   out_o = rows_o( sum_r H_r . W2_r ).
 *
 * x_shards: W pointers, X_r bf16 [(tokens/W) x hidden]; w1: W pointers, bf16 [hidden x f_r];
 * w2: W pointers, bf16 [f_r x hidden]; out: W pointers, bf16 [(tokens/W) x hidden].
 * workspace: tl_mlp2_workspace_bytes(): per-rank gathered X (W x tokens x hidden bf16; rank
 * r's own shard is read in place, its slot of r's copy is not written) at offset 0, then, each at the next 256-byte boundary, the intermediate H (W x tokens x f_r bf16,
 * H_r at rows r*tokens.., readable after the call), the fp32 reduction slot (tokens x hidden)
 * and the signals.
 * One persistent launch runs, per emulated rank r: the mover (gather X into rank r's copy, by
 * pull or, with cfg.ag_push, push), layer-1 tiles (wait for each K quarter of their gathered
 * rows, GELU epilogue, notify per H tile) and layer-2 tiles (wait on the H tiles covering their
 * K range, then the owner-slot GEMM+RS chain; cfg.rs_ring does not apply here).
 * Shapes: 1 <= W <= 8; tokens % (128*W) == 0; hidden % 8 == 0; f_r % 8 == 0.
 */
size_t tl_mlp2_workspace_bytes(int W, int tokens, int hidden, int f_r);
int tl_mlp2(tl_ctx* ctx, int W, const void* const* x_shards, const void* const* w1, const void* const* w2,
            void* const* out, void* workspace, size_t workspace_bytes, int tokens, int hidden, int f_r,
            tl_stream_t stream);

/* ---------------------------------------------------------------- MoE layer with combine partition
 * [TL] §4.1 (dynamic mapping tables filled by the routing), §7.2 (Gather + GroupGEMM, then
 * GroupGEMM + Scatter + TopK reduce), [RA] MoE abstract (persistent expert producer; a
 * persistent combine consumer on `combine_ctas` dedicated SMs that handles output tiles as
 * their ready signals arrive; the GEMM partition's CTAs join it after their last GEMM tile,
 * each y tile claimed once at run time).
 *
 * x: bf16 [T x H]; logits: fp32 [T x E]; w_gate, w_up: bf16 [E x H x F]; w_down: bf16 [E x F x H].
 * out: fp32 [T x H] (written, not accumulated into).
 * perm_out (optional, may be NULL): int32 [T*topk]: perm_out[pos] = t*topk + j, assignments
 *   ordered by (expert, t, j).  counts_out (optional): int32 [E] assignments per expert.
 * Routing: experts = the topk largest logits (ties to the lower expert index), gates = softmax
 * over all E logits taken at those experts; with cfg.moe_renorm = 1 the topk gates of a token
 * are divided by their sum (the pages define no router: both readings are offered).
 *   y_(t,j) = (SiLU(x_t . Wg_e) * (x_t . Wu_e)) . Wd_e   (h kept in bf16, y in bf16)
 *   out_t   = sum_j gate_(t,j) * y_(t,j)                  (fp32)
 * workspace: tl_moe_workspace_bytes().
 * Three launches: the routing (a warp per token), the permutation and tile tables (a CTA per
 * expert, while the remaining CTAs zero `out`), then one persistent launch of one CTA per SM
 * whose GEMM partition runs the gather and the grouped GEMMs while the combine partition adds
 * finished y tiles into `out`.  The second and third are dependent launches (programmatic
 * stream serialization): each starts while the one before it runs and waits for it before
 * reading its results.  TL_ERR_UNSUPPORTED if the device cannot hold the persistent grid at
 * once.
 * Shapes: T >= 1; 1 <= topk <= 8; topk <= E <= 256; H % 256 == 0; F % 128 == 0.
 */
size_t tl_moe_workspace_bytes(int T, int H, int E, int F, int topk);
/* The tile order of tl_moe_combine's persistent kernel, for host-side checks ([TL] §4.1: the
 * tile-to-work mapping is filled at run time; here the closed form behind it).  m_tiles is
 * the number of 128-row padded row tiles the routing produced (sum over experts of
 * ceil(count_e / 128)); 0 <= m_tiles <= the bound the workspace is sized for.
 * tl_moe_tile_order: for t = 0..count-1, the tile's kind (1 = gate/up, 2 = down), row tile
 *   and column block (128 columns of F for kind 1, 256 columns of H for kind 2).
 * tl_moe_combine_order: for v = 0..count-1, the row tile and column block of the v-th y tile
 *   the combine claims.
 * Both return the number of tiles, or TL_ERR_INVALID (bad shape, m_tiles out of range, or
 * arrays shorter than `cap`).  Arrays may all be NULL to query the count.  Host only. */
int tl_moe_tile_order(int T, int H, int E, int F, int topk, int m_tiles, int* kind, int* row_tile, int* col_block,
                      int cap);
int tl_moe_combine_order(int T, int H, int E, int F, int topk, int m_tiles, int* row_tile, int* col_block, int cap);
int tl_moe_combine(tl_ctx* ctx, const void* x, const float* logits, int topk, const void* w_gate,
                   const void* w_up, const void* w_down, float* out, int* perm_out, int* counts_out,
                   void* workspace, size_t workspace_bytes, int T, int H, int E, int F, tl_stream_t stream);

/* ---------------------------------------------------------------- AllGather KV + self-attention
 * [TL] §5 (AllGather KV + self-attention: the KV cache sequence split into W equal shards)
 * and §7.2 (sequence-parallel self-attention; Table 4 Attn-1/Attn-2: head dim 128); [TD] §3.7
 * (the local shard first).  Non-causal (the pages give no mask):
 *   out[h] = softmax(q[h] K[h]^T / sqrt(d)) V[h],  K = [K_0 | K_1 | ... | K_{W-1}] along the
 *   sequence (rank order), V likewise.
 * q: bf16 [heads x l_r x d] (this rank's queries).  k_shards, v_shards: host arrays of W device
 * pointers, shard r bf16 [heads x l_r x d].  out: bf16 [heads x l_r x d].
 * workspace: tl_ag_attention_workspace_bytes(): the gathered K and V, shard-major
 * [W x heads x l_r x d] (shard r at r, filled completely, the local shard last), one signal
 * per (shard, head, 128-key block), and room for the partial results of split items (below).
 * One persistent launch of CTA pairs (clusters of 2, one CTA per SM): mover warps pull the
 * remote shards' K/V blocks into the gathered buffers and release each block's signal; the
 * attention of each (head, 256-query tile) reads its own shard in place first and a remote
 * shard's blocks once all of them are signalled.  The pages run this gather on the copy
 * engine from a second stream; that makes the kernel wait on work outside its own launch,
 * which nothing guarantees to run alongside it, so the gather runs inside the kernel, as for
 * tl_ag_gemm.  When the (head, tile) items leave the last wave of pairs less than half full,
 * those last items are each split into two halves of their keys that run on two pairs; the
 * half that finishes second combines both (in a fixed order: the result does not depend on
 * which finished first).
 * Shapes: 1 <= W <= 8; d == 128; any l_r (a shard's last 256-key block and the last 256-query
 * tile may be partial).  heads == 0 or l_r == 0 is a no-op.
 */
size_t tl_ag_attention_workspace_bytes(int W, int heads, int l_r, int d);
int tl_ag_attention(tl_ctx* ctx, int W, int rank, const void* q, const void* const* k_shards,
                    const void* const* v_shards, void* out, void* workspace, size_t workspace_bytes,
                    int heads, int l_r, int d, tl_stream_t stream);

/* ---------------------------------------------------------------- AllGather + GEMM without allocation
 * The pages have no counterpart of this entry point.  It exists for callers that cannot
 * allocate device memory when they call in: code being recorded into a CUDA graph by stream
 * capture (cudaMalloc cannot be recorded), plug-ins whose host framework owns the allocator
 * and gives out no scratch, and real-time paths that forbid allocation after start-up.
 *
 * Same operation, arguments, shapes and result as tl_ag_gemm, minus the workspace: the
 * gathered operand and the chunk signals live in a fixed device array of
 * TL_AG_GEMM_STATIC_SCRATCH_BYTES inside the library, which every GPU that loads the library
 * keeps until the process exits.  A problem whose tl_ag_gemm_workspace_bytes() exceeds that
 * size is rejected with TL_ERR_WORKSPACE before anything is enqueued.  The entry point
 * allocates nothing (no cudaMalloc, cudaFree or allocating library call).  Its first call on a
 * device looks up the array's device address with that device current; make that first call
 * before any stream capture begins.  The address is kept for the life of the process: after
 * cudaDeviceReset on that device (or anything else that destroys its primary context) the
 * entry point must not be called on that device again.  Every argument check (those of
 * tl_ag_gemm, then the size check) runs before anything is enqueued.  All calls share the one
 * array (each call clears the signals and overwrites the gathered operand), so calls whose GPU
 * work overlaps in time race and give undefined results: order them on one stream or with
 * events.
 */
#define TL_AG_GEMM_STATIC_SCRATCH_BYTES (16u << 20)
int tl_ag_gemm_static_scratch(tl_ctx* ctx, int W, int rank, const void* const* a_shards, const void* b, void* c,
                              int m_per_rank, int n, int k, tl_stream_t stream);

/* ---------------------------------------------------------------- host-side tile maps (no GPU)
 * The static tile-centric mappings the kernels use ([TL] §4.1), evaluated on the host by the
 * same code the device runs, for inspection and testing.
 *
 * Tiles are 256 x 256 when every shard (AG) or owner block (RS) is a multiple of 256 rows,
 * else 128 x 256; row blocks are reported in units of 128 rows (the first 128-row block a
 * tile covers), column blocks in units of 256 columns.
 * tl_ag_tile_order: for the AllGather + GEMM tile sequence t = 0..count-1 writes the source
 *   rank, the row block inside that rank's shard and the column block.  Returns the number of
 *   tiles, or TL_ERR_INVALID.  Arrays may be NULL to query the count; otherwise they must hold
 *   `cap` entries.
 * tl_rs_tile_order: the same for GEMM + ReduceScatter (owner-slot chain): producer, owner, row
 *   block within the owner's rows, column block.
 * tl_rs_ring_tile_order: the same for the ring (cfg.rs_ring = 1), plus each tile's hop (its
 *   position 0..W-1 on the ring of its owner's partial).
 */
int tl_ag_tile_order(int W, int rank, int m_per_rank, int n, int swizzle, int* src_rank, int* m_block,
                     int* n_block, int cap);
int tl_rs_tile_order(int W, int m, int n, int swizzle, int* producer, int* owner, int* m_block, int* n_block,
                     int cap);
int tl_rs_ring_tile_order(int W, int m, int n, int* producer, int* owner, int* m_block, int* n_block, int* hop,
                          int cap);

#ifdef __cplusplus
}
#endif
#endif /* TL_GB300_H */
