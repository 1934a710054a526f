// MoE layer (routing, permutation, grouped expert GEMMs, combine partition).
#include "tl_host.h"

extern "C" size_t tl_moe_workspace_bytes(int, int, int, int, int) { return 0; }

extern "C" int tl_moe_combine(tl_ctx*, const void*, const float*, int, const void*, const void*, const void*, float*,
                              int*, int*, void*, size_t, int, int, int, int, tl_stream_t) {
  return TL_ERR_UNSUPPORTED;
}
