// Host-side internals shared by the op translation units: the context, TMA
// descriptor encoding (cuTensorMapEncodeTiled through the runtime's driver
// entry point) and the cooperative persistent launch.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/tl.h"
#include "tl_engine.cuh"
#include "tl_engine2.cuh"

struct tl_ctx {
  int device;
  int sms;
  int ctas;
  tl_config cfg;
  tl::DevStatus* status;      // device status word (the only memory the library owns)
  unsigned long long epoch;   // last signal value handed out
  void* trace_buf;            // caller-owned trace buffer (null: tracing off)
  int trace_cap;              // spans per warp
  int trace_ctas;             // CTAs the buffer holds
};

namespace tl {

bool tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner,
             uint64_t outer, uint32_t box_inner, uint32_t box_outer);
bool tmap_3d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t d0, uint64_t d1,
             uint64_t d2, uint32_t b0, uint32_t b1, uint32_t b2);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Next signal value of this context (never 0; < 2^59 so that (epoch << 4) | 15 fits in 64 bits).
// Values whose low 32 bits are 0 are skipped: the low-latency gather carries those 32 bits in
// every word, and a zero-filled workspace must never look written.
inline unsigned long long next_epoch(tl_ctx* ctx) {
  if ((++ctx->epoch & 0xffffffffull) == 0) ++ctx->epoch;
  return ctx->epoch;
}

inline Common make_common(tl_ctx* ctx) {
  Common c;
  c.status = ctx->status;
  c.epoch = next_epoch(ctx);
  c.timeout_ns = ctx->cfg.timeout_ns;
  c.mover_warps = ctx->cfg.mover_warps;  // clamped per op at launch (see launch_persistent)
  c.trace_cap = ctx->trace_cap;
  c.trace_ctas = ctx->trace_ctas;
  c.trace_hdr = static_cast<unsigned int*>(ctx->trace_buf);
  c.trace = ctx->trace_buf ? reinterpret_cast<TraceRec*>(static_cast<uint8_t*>(ctx->trace_buf) + 4 * kTraceHdrWords +
                                                         4 * kTraceWarps * static_cast<size_t>(ctx->trace_ctas))
                           : nullptr;
  return c;
}

int set_smem_attr(const void* kern);

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace of the AllGather (alone or fused with the GEMM): the gathered operand T
// (W x m_per_rank x k bf16, rank order) at offset 0, then the per-chunk signal words
// (W x m_per_rank/128 slabs x 32 chunks, 8 bytes each), then, for problems small enough for
// the low-latency gather (W * m_per_rank * k <= kLLMaxElems), the LL slabs: one 8-byte word
// {two bf16, call signal} per pair of elements of every shard (W x m_per_rank x k/2 words).
// Each region is 256-byte aligned.  tl_ag_gemm_workspace_bytes, tl_ag_gemm, tl_allgather and
// tl_ag_gemm_static_scratch all take their offsets from here.
constexpr long long kLLMaxElems = 1LL << 20;
struct AgLayout {
  size_t gath_bytes;   // the gathered operand
  size_t flags_off;    // first signal word
  size_t flags_bytes;  // all signal words
  size_t ll_off;       // first LL word
  size_t ll_bytes;     // all LL words (0: the problem is too large for the LL gather)
  size_t total;
};
AgLayout ag_layout(int W, int m_per_rank, int k);

// The argument checks of tl_ag_gemm that need no workspace (context, shape, rank, null and
// misaligned pointers): TL_OK or the code tl_ag_gemm returns for them.  An empty problem
// (a zero dimension) passes without looking at the pointers.
int ag_gemm_check(const tl_ctx* ctx, int W, int rank, const void* const* a_shards, const void* b, const void* c,
                  int m_per_rank, int n, int k);

// The low-latency push gather + GEMM (tl_ag_ll.cu): whether a problem can take it on this
// context (its workspace has LL slabs and its 128 x 256 tiles leave at least one CTA to push),
// and the launch (TL_ERR_UNSUPPORTED when it cannot).
int ag_ll_capable(const tl_ctx* ctx, int W, int m_per_rank, int n, int k);
int ag_ll_launch(tl_ctx* ctx, int W, int rank, const void* const* a_shards, const void* b, void* c, uint8_t* ws,
                 int m_per_rank, int n, int k, cudaStream_t stream);


// Launch of one persistent CTA per SM (or cfg.grid_ctas), so that every CTA that waits on a
// signal is co-resident with the CTAs that will set it: a cooperative launch, or for an op
// with kDependentLaunch a launch with programmatic stream serialization after a check that
// the device holds the whole grid at once (the two attributes are not combined; the kernel
// before it never waits on this one, so its CTAs only delay this grid's start).  While the
// context has a trace buffer the span-recording instantiation runs.
template <class Op>
int launch_persistent(tl_ctx* ctx, const typename Op::Params& p, cudaStream_t stream, int mover_warps) {
  auto kern = ctx->trace_buf ? persistent_kernel<Op, true> : persistent_kernel<Op, false>;
  int rc = set_smem_attr(reinterpret_cast<const void*>(kern));
  if (rc != TL_OK) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctx->ctas, 1, 1);
  if (mover_warps > Op::kMaxMovers) mover_warps = Op::kMaxMovers;
  cfg.blockDim = dim3((2 + Op::kEpiWarps + mover_warps) * 32, 1, 1);
  typename Op::Params q = p;  // the device movers size their loops by the launched warp count
  q.common.mover_warps = mover_warps;
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if constexpr (Op::kDependentLaunch) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, cfg.blockDim.x, kSmemBytes) != cudaSuccess) {
      (void)cudaGetLastError();
      return TL_ERR_CUDA;
    }
    if (per_sm * ctx->sms < ctx->ctas) return TL_ERR_UNSUPPORTED;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, q);
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

// Launch of the CTA-pair engine: clusters of 2 CTAs, as many as the device reports it can
// hold at once (at most one CTA per SM), so every CTA that waits on a signal is resident
// together with the CTAs that set it.  The cluster shape is the only launch attribute (the
// cooperative attribute is not combined with clusters); every wait stays bounded.
template <class Op>
int launch_persistent_pair(tl_ctx* ctx, const typename Op::Params& p, cudaStream_t stream, int mover_warps) {
  const int traced = ctx->trace_buf ? 1 : 0;
  auto kern = traced ? persistent_kernel_pair<Op, true> : persistent_kernel_pair<Op, false>;
  int rc = set_smem_attr(reinterpret_cast<const void*>(kern));
  if (rc != TL_OK) return rc;
  if (mover_warps > Op::kMaxMovers) mover_warps = Op::kMaxMovers;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3((2 + Op::kEpiWarps + mover_warps) * 32, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int max_clusters[2] = {-1, -1};  // per kernel instantiation
  if (max_clusters[traced] < 0) {
    cfg.gridDim = dim3(ctx->sms & ~1, 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      return TL_ERR_UNSUPPORTED;
    }
    max_clusters[traced] = n;
  }
  int nclusters = ctx->ctas / 2;
  if (nclusters > max_clusters[traced]) nclusters = max_clusters[traced];
  if (nclusters < 1) return TL_ERR_UNSUPPORTED;
  cfg.gridDim = dim3(2 * nclusters, 1, 1);
  typename Op::Params q = p;
  q.common.mover_warps = mover_warps;
  if (cudaLaunchKernelEx(&cfg, kern, q) != cudaSuccess) {
    (void)cudaGetLastError();
    return TL_ERR_CUDA;
  }
  return TL_OK;
}

}  // namespace tl
