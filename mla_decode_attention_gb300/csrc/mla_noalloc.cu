// mla_decode_noalloc: dense paged decode whose schedule metadata and split
// workspace live in a fixed device array owned by this library, so the caller
// never has to allocate scratch memory.
//
// Who needs this: code that may run kernels but may not allocate device
// memory at that point, e.g. an inference engine's plugin "enqueue" hook that
// is handed only input/output pointers and a stream, or a latency-critical
// serving loop that must not hit cudaMalloc (which can synchronise the device
// and grow memory pools).  Such callers pass only inputs and outputs.
//
// Costs and limits: the array below is MLA_NOALLOC_SCRATCH_BYTES (40 MiB) and
// every GPU that loads this library holds it until the process exits.  All
// calls share it, so two calls that overlap on the GPU (different streams, or
// different host threads on the same device) race and corrupt each other's
// results; serialise them.  Nothing in it needs to start at zero: every call
// rewrites the metadata and every partial it later reads.
#include <cuda.h>

#include <cstdint>
#include <mutex>

#include "mla_decode.h"
#include "mla_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

// The array's device address depends on where the library's device code is
// loaded: once per CUDA context.  A context created after cudaDeviceReset,
// or a non-primary context made current by the caller, has its own copy at
// its own address, so the cache is keyed by the context current at the call.
constexpr int kMaxContexts = 64;
struct ScratchEntry {
  CUcontext ctx;
  void* ptr;
};
std::mutex g_scratch_mu;
ScratchEntry g_scratch[kMaxContexts] = {};
int g_scratch_n = 0;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of the scratch array in the current context.  The first
// call in a context looks it up with that context current (this can load the
// library's device code into it); later calls in that context reuse it.
int scratch_address(void** out) {
  CtxGetCurrentFn get = ctx_get_current();
  if (!get) return mla::record_error("cuCtxGetCurrent is not available", MLA_ERR_CUDA);
  CUcontext ctx = nullptr;
  void* p = nullptr;
  if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
    // no context yet: the symbol lookup makes the runtime set up the
    // device's primary context, which is then current
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return mla::record_cuda_error("cudaGetSymbolAddress(noalloc scratch)", e);
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr)
      return mla::record_error("no current CUDA context", MLA_ERR_CUDA);
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  for (int i = 0; i < g_scratch_n; ++i)
    if (g_scratch[i].ctx == ctx) {
      *out = g_scratch[i].ptr;
      return MLA_OK;
    }
  if (p == nullptr) {
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return mla::record_cuda_error("cudaGetSymbolAddress(noalloc scratch)", e);
  }
  if (g_scratch_n < kMaxContexts) {
    g_scratch[g_scratch_n++] = ScratchEntry{ctx, p};
  } else {  // a full cache keeps working: the oldest entry makes room
    for (int i = 1; i < kMaxContexts; ++i) g_scratch[i - 1] = g_scratch[i];
    g_scratch[kMaxContexts - 1] = ScratchEntry{ctx, p};
  }
  *out = p;
  return MLA_OK;
}

}  // namespace

extern "C" int mla_decode_noalloc(const void* q, const void* kv_cache, int kv_format,
                                  int64_t num_pages, const int32_t* block_table,
                                  int64_t block_table_stride, const int32_t* cache_seqlens,
                                  int batch, int s_q, int h_q, float softmax_scale, int causal,
                                  void* out, float* lse, uint32_t* err, cudaStream_t stream) {
  if (!q || !kv_cache || !block_table || !cache_seqlens || !out || !lse) return MLA_ERR_NULL;
  int device = 0;
  const cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return mla::record_cuda_error("cudaGetDevice", e);
  int parts = 0;
  int rc = mla_num_sm_parts(device, h_q, &parts);
  if (rc != MLA_OK) return rc;
  size_t meta_bytes = 0, ws_bytes = 0;
  rc = mla_metadata_size(batch, s_q, parts, &meta_bytes);
  if (rc != MLA_OK) return rc;
  rc = mla_workspace_size(batch, s_q, h_q, parts, &ws_bytes);
  if (rc != MLA_OK) return rc;
  const size_t meta_padded = (meta_bytes + 255) & ~static_cast<size_t>(255);
  if (meta_padded + ws_bytes > static_cast<size_t>(MLA_NOALLOC_SCRATCH_BYTES))
    return mla::record_error(
        "mla_decode_noalloc: metadata + split workspace for this shape exceed the fixed "
        "MLA_NOALLOC_SCRATCH_BYTES scratch; use mla_decode with caller-provided buffers",
        MLA_ERR_SHAPE);
  void* base = nullptr;
  rc = scratch_address(&base);
  if (rc != MLA_OK) return rc;
  unsigned char* scratch = static_cast<unsigned char*>(base);
  rc = mla_get_metadata(cache_seqlens, batch, s_q, causal, 0, parts, scratch, stream);
  if (rc != MLA_OK) return rc;
  return mla_decode(q, kv_cache, kv_format, num_pages, block_table, block_table_stride,
                    cache_seqlens, batch, s_q, h_q, softmax_scale, causal, scratch, parts,
                    scratch + meta_padded, out, lse, err, stream);
}
