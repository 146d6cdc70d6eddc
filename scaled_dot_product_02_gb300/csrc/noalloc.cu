// noalloc.cu -- sdpa_bwd_noalloc: the backward for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand the library a workspace: a plugin whose
// host application owns every device allocation and forbids others, a C
// program with no allocator of its own, or a latency-critical path that must
// not pay the device-wide synchronisation a cudaMalloc/cudaFree can cause.
// This entry point takes the backward's scratch (per-row statistics, the fp32
// dQ accumulator and, at head_dim 256/512, the P / dS score tiles of a chunk
// of keys) from a fixed array in the library's own device memory instead, so
// it needs no workspace argument and allocates nothing.
//
// The array below is created when the library's device code is loaded and
// every GPU that loads it holds SDPA_BWD_NOALLOC_MAX_BYTES until the process
// exits. All calls share it and it keeps the previous call's contents; the
// backward's kernels rewrite everything they read from it (the preprocess
// kernel rebuilds the statistics and zeroes the accumulator on every call,
// and each score tile is written before the GEMMs of its chunk read it), so
// nothing stale is used. Calls that overlap on the GPU (for example on two
// streams at once) race on the array and must be serialised by the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/sdpa.h"
#include "kernels.h"

static __device__ __align__(256) unsigned char g_bwd_scratch[SDPA_BWD_NOALLOC_MAX_BYTES];

namespace {

// Device address of g_bwd_scratch on the current device. In host code the
// symbol is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress (cached per device and context).
int scratch_address(void** out) {
  *out = sdpa::device_symbol_address(&g_bwd_scratch);
  return *out ? SDPA_OK : SDPA_ERR_CUDA;
}

}  // namespace

extern "C" SDPA_API int sdpa_bwd_noalloc(const sdpa_problem* p, const void* q, const void* k, const void* v,
                                         const void* o, const float* lse, const void* dout, void* dq, void* dk,
                                         void* dv, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                                         void* stream) {
  const int rc = sdpa_check_problem(p);
  if (rc != SDPA_OK) return rc;
  if (p->head_dim_v && p->head_dim_v != p->head_dim) return SDPA_ERR_UNSUPPORTED;  // forward-only pair
  if (sdpa_bwd_workspace_size(p) > (size_t)SDPA_BWD_NOALLOC_MAX_BYTES) return SDPA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const int arc = scratch_address(&scratch);
  if (arc != SDPA_OK) return arc;
  return sdpa_bwd(p, q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_kv, scratch,
                  (size_t)SDPA_BWD_NOALLOC_MAX_BYTES, stream);
}
