// AllGather + GEMM for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device memory at the point where they call in:
// code being recorded into a CUDA graph by stream capture (cudaMalloc is not an
// operation a capture can record), plug-ins hosted by a framework that owns the
// allocator and hands out no scratch, and real-time paths that forbid allocation
// after start-up.  For them this file provides tl_ag_gemm_static_scratch: the same fused
// AllGather + GEMM as tl_ag_gemm, with its scratch (the gathered operand and the chunk
// signals) in a fixed array that is part of this library's device module.  The caller
// passes only inputs and outputs; nothing here calls cudaMalloc, cudaFree or any
// allocating routine.
//
// The array is kTlStaticScratchBytes (16 MiB) per GPU and stays allocated on every GPU
// that loads this module until the process exits.  Its device address is looked up once
// per device (cudaGetSymbolAddress with that device current) by the first call on that
// device, so that first call should happen before any stream capture begins.  The address
// is kept for the life of the process: after cudaDeviceReset (or anything else that
// destroys the device's primary context) it is stale, and this entry point must not be
// called on that device again.  Every call
// reuses the same array: the signal words are cleared at the start of each call and the
// gathered operand is fully overwritten, so nothing carries over; but two calls whose GPU
// work overlaps in time (unordered streams, several host threads) race on the array and
// give undefined results.
#include <mutex>

#include "tl_host.h"

namespace tl {

constexpr size_t kTlStaticScratchBytes = size_t(16) << 20;

// The scratch itself.  In host code this name only stands in for the symbol; it is never
// a device address.  Kernels get the address returned by cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_scratch[kTlStaticScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on `device` (which must be current), looked up once.
int scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return TL_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return TL_ERR_CUDA;
    }
    g_scratch_addr[device] = p;
  }
  *out = g_scratch_addr[device];
  return TL_OK;
}
}  // namespace

}  // namespace tl

// The fused AllGather + GEMM of tl_ag_gemm with the fixed array above as its workspace.
// Every argument check of tl_ag_gemm, and the size check against the array, runs before
// anything is enqueued, so a refused call leaves the array and the stream untouched.
extern "C" int tl_ag_gemm_static_scratch(tl_ctx* ctx, int W, int rank, const void* const* a_shards, const void* b,
                                         void* c, int m_per_rank, int n, int k, tl_stream_t stream) {
  const int chk = tl::ag_gemm_check(ctx, W, rank, a_shards, b, c, m_per_rank, n, k);
  if (chk != TL_OK) return chk;
  if (m_per_rank == 0 || n == 0 || k == 0) return TL_OK;  // empty problem: nothing to do, no scratch
  const tl::AgLayout L = tl::ag_layout(W, m_per_rank, k);
  if (L.total > tl::kTlStaticScratchBytes) return TL_ERR_WORKSPACE;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return TL_ERR_CUDA;
  void* scratch = nullptr;
  const int rc = tl::scratch_address(ctx->device, &scratch);
  if (rc != TL_OK) return rc;
  // Clear the signal words (and LL words) the previous call left, another context's included.
  if (cudaMemsetAsync(static_cast<unsigned char*>(scratch) + L.flags_off, 0, L.total - L.flags_off,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    (void)cudaGetLastError();
    return TL_ERR_CUDA;
  }
  return tl_ag_gemm(ctx, W, rank, a_shards, b, c, scratch, tl::kTlStaticScratchBytes, m_per_rank, n, k, stream);
}
