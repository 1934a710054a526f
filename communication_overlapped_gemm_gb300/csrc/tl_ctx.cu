// Context, status word, TMA descriptor encoding and the host-side tile-map queries.
#include <cudaTypedefs.h>

#include <chrono>
#include <cstdio>
#include <mutex>
#include <random>

#include "tl_host.h"

// L2 promotion of every TMA tile access (CUtensorMapL2promotion: 0 none, 1 64 B, 2 128 B,
// 3 256 B sectors).
#ifndef TL_L2_PROMOTION
#define TL_L2_PROMOTION 3
#endif

namespace tl {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}
}  // namespace

static bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
                   const cuuint64_t* strides, const cuuint32_t* box) {
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const uint32_t inner_bytes = box[0] * (dt == CU_TENSOR_MAP_DATA_TYPE_FLOAT32 ? 4u : 2u);
  const CUtensorMapSwizzle sw = inner_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = g_encode(m, dt, rank, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, static_cast<CUtensorMapL2promotion>(TL_L2_PROMOTION),
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner,
             uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * static_cast<uint64_t>(esize)};
  cuuint32_t box[2] = {box_inner, box_outer};
  return encode(m, dt, 2, base, dims, strides, box);
}

bool tmap_3d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t d0, uint64_t d1,
             uint64_t d2, uint32_t b0, uint32_t b1, uint32_t b2) {
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * static_cast<uint64_t>(esize), d0 * d1 * static_cast<uint64_t>(esize)};
  cuuint32_t box[3] = {b0, b1, b2};
  return encode(m, dt, 3, base, dims, strides, box);
}

int set_smem_attr(const void* kern) {
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess) {
    (void)cudaGetLastError();
    return TL_ERR_CUDA;
  }
  return TL_OK;
}

}  // namespace tl

extern "C" {

int tl_version(void) { return 100; }

int tl_config_default(tl_config* cfg) {
  if (!cfg) return TL_ERR_INVALID;
  cfg->mover_warps = 4;
  cfg->chunks_per_slab = 32;
  cfg->swizzle = 1;
  cfg->grid_ctas = 0;
  cfg->combine_ctas = 8;
  cfg->debug_skip_chunk = -1;
  cfg->timeout_ns = 2000000000ull;
  cfg->pair_ctas = 2;
  cfg->moe_renorm = 0;
  cfg->rs_ring = 0;
  cfg->ag_push = 0;
  cfg->mover_kparts = 0;
  cfg->ag_ll = 0;
  cfg->mover_tma = 0;
  return TL_OK;
}

static bool pow2_le32(int c) { return c >= 1 && c <= 32 && (c & (c - 1)) == 0; }

int tl_ctx_create(tl_ctx** out, int device, const tl_config* cfg) {
  if (!out) return TL_ERR_INVALID;
  *out = nullptr;
  tl_config c;
  if (cfg)
    c = *cfg;
  else
    tl_config_default(&c);
  if (c.mover_warps < 1 || c.mover_warps > tl::kMaxMoverWarps || !pow2_le32(c.chunks_per_slab) ||
      (c.swizzle != 0 && c.swizzle != 1) || c.grid_ctas < 0 || c.combine_ctas < 1 || c.timeout_ns == 0 ||
      c.pair_ctas < 0 || c.pair_ctas > 2 || (c.moe_renorm != 0 && c.moe_renorm != 1) ||
      (c.rs_ring != 0 && c.rs_ring != 1) || (c.ag_push != 0 && c.ag_push != 1) ||
      (c.mover_kparts != 0 && c.mover_kparts != 1 && c.mover_kparts != 2 && c.mover_kparts != 4) ||
      (c.ag_ll != 0 && c.ag_ll != 1) || (c.mover_tma != 0 && c.mover_tma != 1))
    return TL_ERR_INVALID;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) {
    (void)cudaGetLastError();
    return TL_ERR_CUDA;
  }
  if (device < 0 || device >= ndev) return TL_ERR_INVALID;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return TL_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return TL_ERR_UNSUPPORTED;
  int prev = 0;
  cudaGetDevice(&prev);
  if (cudaSetDevice(device) != cudaSuccess) return TL_ERR_CUDA;
  tl_ctx* ctx = new tl_ctx();
  ctx->device = device;
  ctx->sms = prop.multiProcessorCount;
  ctx->ctas = c.grid_ctas > 0 ? (c.grid_ctas < ctx->sms ? c.grid_ctas : ctx->sms) : ctx->sms;
  if (c.combine_ctas >= ctx->ctas) c.combine_ctas = ctx->ctas > 1 ? ctx->ctas / 2 : 1;
  ctx->cfg = c;
  if (cudaMalloc(&ctx->status, sizeof(tl::DevStatus)) != cudaSuccess ||
      cudaMemset(ctx->status, 0, sizeof(tl::DevStatus)) != cudaSuccess) {
    (void)cudaGetLastError();
    delete ctx;
    cudaSetDevice(prev);
    return TL_ERR_CUDA;
  }
  cudaDeviceSynchronize();
  // Signal values start at a random point so that a workspace reused across contexts
  // never holds a value a new context would wait for.
  std::random_device rd;
  unsigned long long r = (static_cast<unsigned long long>(rd()) << 32) ^ rd() ^
                         static_cast<unsigned long long>(
                             std::chrono::high_resolution_clock::now().time_since_epoch().count());
  ctx->epoch = ((r & 0xFFFFFFFFFull) << 16) + 1;  // < 2^52
  cudaSetDevice(prev);
  *out = ctx;
  return TL_OK;
}

void tl_ctx_destroy(tl_ctx* ctx) {
  if (!ctx) return;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(ctx->device);
  cudaDeviceSynchronize();
  cudaFree(ctx->status);
  cudaSetDevice(prev);
  delete ctx;
}

int tl_ctx_check(tl_ctx* ctx) {
  if (!ctx) return TL_ERR_INVALID;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(ctx->device);
  tl::DevStatus st;
  int rc = TL_OK;
  if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpy(&st, ctx->status, sizeof(st), cudaMemcpyDeviceToHost) !=
                                                      cudaSuccess) {
    (void)cudaGetLastError();
    rc = TL_ERR_CUDA;
  } else if (st.code != 0) {
    rc = st.code == tl::kStatusTimeout ? TL_ERR_TIMEOUT : TL_ERR_CUDA;
    cudaMemset(ctx->status, 0, sizeof(tl::DevStatus));
    cudaDeviceSynchronize();
  }
  cudaSetDevice(prev);
  return rc;
}

int tl_ctx_num_ctas(const tl_ctx* ctx) { return ctx ? ctx->ctas : 0; }

// Trace buffer: header (8 words), per-warp counts (16 words per CTA), then the spans.  The
// header and counts take 32 + 64 * ctas bytes, a multiple of 16, so the spans stay aligned.
size_t tl_trace_bytes(int ctas, int spans_per_warp) {
  if (ctas < 1 || spans_per_warp < 1) return 0;
  return 4 * tl::kTraceHdrWords +
         static_cast<size_t>(ctas) * (4 * tl::kTraceWarps + sizeof(tl::TraceRec) * tl::kTraceWarps *
                                                                static_cast<size_t>(spans_per_warp));
}

int tl_ctx_set_trace(tl_ctx* ctx, void* buf, size_t bytes, int spans_per_warp) {
  if (!ctx) return TL_ERR_INVALID;
  if (!buf) {
    ctx->trace_buf = nullptr;
    ctx->trace_cap = 0;
    ctx->trace_ctas = 0;
    return TL_OK;
  }
  if (spans_per_warp < 1 || !tl::aligned16(buf) || bytes < tl_trace_bytes(1, spans_per_warp)) return TL_ERR_INVALID;
  const size_t per_cta = tl_trace_bytes(2, spans_per_warp) - tl_trace_bytes(1, spans_per_warp);
  const size_t held = (bytes - 4 * tl::kTraceHdrWords) / per_cta;
  ctx->trace_buf = buf;
  ctx->trace_cap = spans_per_warp;
  ctx->trace_ctas = held > 4096 ? 4096 : static_cast<int>(held);
  return TL_OK;
}

const char* tl_strerror(int code) {
  switch (code) {
    case TL_OK: return "ok";
    case TL_ERR_INVALID: return "invalid argument (null/misaligned pointer, unsupported shape or config)";
    case TL_ERR_UNSUPPORTED: return "unsupported device (needs sm_103) or persistent grid not co-resident";
    case TL_ERR_CUDA: return "CUDA runtime/driver error";
    case TL_ERR_TIMEOUT: return "a bounded device wait on a signal ran out";
    case TL_ERR_WORKSPACE: return "workspace smaller than required";
    default: return "unknown status";
  }
}

int tl_ag_tile_order(int W, int rank, int m_per_rank, int n, int swizzle, int* src_rank, int* m_block,
                     int* n_block, int cap) {
  if (W < 1 || W > 8 || rank < 0 || rank >= W || m_per_rank <= 0 || m_per_rank % tl::kBM || n <= 0 ||
      (swizzle != 0 && swizzle != 1))
    return TL_ERR_INVALID;
  const int bm = m_per_rank % 256 == 0 ? 256 : 128;  // the tile rows tl_ag_gemm uses
  const int mps = m_per_rank / bm, nbk = tl::ceil_div(n, tl::kBN);
  const int total = tl::ag_num_tiles(W, mps, nbk);
  if (!src_rank && !m_block && !n_block) return total;
  if (!src_rank || !m_block || !n_block || cap < total) return TL_ERR_INVALID;
  for (int t = 0; t < total; ++t) {
    tl::AgTile a = tl::ag_tile(t, W, rank, mps, nbk, swizzle);
    src_rank[t] = a.src;
    m_block[t] = a.mb * (bm / tl::kBM);
    n_block[t] = a.nb;
  }
  return total;
}

int tl_rs_tile_order(int W, int m, int n, int swizzle, int* producer, int* owner, int* m_block, int* n_block,
                     int cap) {
  if (W < 1 || W > 8 || m <= 0 || m % (tl::kBM * W) || n <= 0 || (swizzle != 0 && swizzle != 1))
    return TL_ERR_INVALID;
  const int bm = (m / W) % 256 == 0 ? 256 : 128;  // the tile rows tl_gemm_rs uses
  const int mbo = m / W / bm, nbk = tl::ceil_div(n, tl::kBN);
  const int total = tl::rs_num_tiles(W, mbo, nbk);
  if (!producer && !owner && !m_block && !n_block) return total;
  if (!producer || !owner || !m_block || !n_block || cap < total) return TL_ERR_INVALID;
  for (int t = 0; t < total; ++t) {
    tl::RsTile r = tl::rs_tile(t, W, mbo, nbk, bm, swizzle);
    producer[t] = r.p;
    owner[t] = r.o;
    m_block[t] = r.mb * (bm / tl::kBM);
    n_block[t] = r.nb;
  }
  return total;
}

int tl_rs_ring_tile_order(int W, int m, int n, int* producer, int* owner, int* m_block, int* n_block, int* hop,
                          int cap) {
  if (W < 1 || W > 8 || m <= 0 || m % (tl::kBM * W) || n <= 0) return TL_ERR_INVALID;
  const int bm = (m / W) % 256 == 0 ? 256 : 128;  // the tile rows tl_gemm_rs uses
  const int mbo = m / W / bm, nbk = tl::ceil_div(n, tl::kBN);
  const int total = tl::rs_num_tiles(W, mbo, nbk);
  if (!producer && !owner && !m_block && !n_block && !hop) return total;
  if (!producer || !owner || !m_block || !n_block || !hop || cap < total) return TL_ERR_INVALID;
  for (int t = 0; t < total; ++t) {
    tl::RsTile r = tl::rs_ring_tile(t, W, mbo, nbk, bm);
    producer[t] = r.p;
    owner[t] = r.o;
    m_block[t] = r.mb * (bm / tl::kBM);
    n_block[t] = r.nb;
    hop[t] = r.s;
  }
  return total;
}

}  // extern "C"
