// LSE combine of split-KV partials (DeepGEMM & FlashMLA article, section 7,
// split-KV merge formula).  Each split i stores o_i (already divided by its
// own sum l_i) and lse_i = m_i + ln l_i, so the merged result is
//   lse = ln sum_i exp(lse_i),   out = sum_i exp(lse_i - lse) o_i.
#include <cuda_bf16.h>

#include "mla_decode.h"
#include "mla_internal.h"
#include "mla_ptx.cuh"
#include "mla_schedule.cuh"

namespace mla {

namespace {

constexpr int kCombineThreads = 128;  // 4 output columns per thread
constexpr int kMaxSplitsCached = 64;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(
    const int32_t* __restrict__ meta, int h, int s_q, int num_parts, const float* __restrict__ ws_o,
    const float* __restrict__ ws_lse, __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  // The split kernel's writes are visible only after the primary grid is done.
  pdl_wait_primary();
  const int q = blockIdx.x, head = blockIdx.y;
  const int32_t* s = meta_seq(meta, num_parts, q);
  const int n_splits = s[kSNSplits];
  if (n_splits == 1) return;
  const int b = q / s_q, j = q % s_q;
  __nv_bfloat16* orow = out + (static_cast<int64_t>(q) * h + head) * kDv;
  float* lse_out = lse + (static_cast<int64_t>(b) * h + head) * s_q + j;
  const int d = threadIdx.x * 4;
  if (n_splits == 0) {  // no visible key: out = 0, lse = -inf
    const __nv_bfloat162 z = __floats2bfloat162_rn(0.f, 0.f);
    reinterpret_cast<__nv_bfloat162*>(orow + d)[0] = z;
    reinterpret_cast<__nv_bfloat162*>(orow + d)[1] = z;
    if (threadIdx.x == 0) *lse_out = -INFINITY;
    return;
  }
  const int off = s[kSSplitOff];
  __shared__ float w_sm[kMaxSplitsCached];
  __shared__ float lse_sm;
  if (threadIdx.x < 32) {
    float mx = -INFINITY;
    for (int i = threadIdx.x; i < n_splits; i += 32)
      mx = fmaxf(mx, ws_lse[static_cast<int64_t>(off + i) * h + head]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float ref = (mx == -INFINITY) ? 0.f : mx;
    float sum = 0.f;
    for (int i = threadIdx.x; i < n_splits; i += 32) {
      const float e = __expf(ws_lse[static_cast<int64_t>(off + i) * h + head] - ref);
      sum += e;
      if (i < kMaxSplitsCached) w_sm[i] = e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float total_lse = sum > 0.f ? ref + __logf(sum) : -INFINITY;
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    for (int i = threadIdx.x; i < n_splits && i < kMaxSplitsCached; i += 32) w_sm[i] *= inv;
    if (threadIdx.x == 0) lse_sm = total_lse;
  }
  __syncthreads();
  const float tl = lse_sm;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = 0; i < n_splits; ++i) {
    float w;
    if (i < kMaxSplitsCached) {
      w = w_sm[i];
    } else {
      const float li = ws_lse[static_cast<int64_t>(off + i) * h + head];
      w = tl == -INFINITY ? 0.f : __expf(li - tl);
    }
    const float4 o = *reinterpret_cast<const float4*>(ws_o + (static_cast<int64_t>(off + i) * h + head) * kDv + d);
    acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
  }
  reinterpret_cast<__nv_bfloat162*>(orow + d)[0] = __floats2bfloat162_rn(acc.x, acc.y);
  reinterpret_cast<__nv_bfloat162*>(orow + d)[1] = __floats2bfloat162_rn(acc.z, acc.w);
  if (threadIdx.x == 0) *lse_out = tl;
}

}  // namespace

int launch_combine(const void* metadata, int batch, int s_q, int h_q, int num_sm_parts,
                   const void* workspace, void* out, float* lse, cudaStream_t stream, bool pdl) {
  const int64_t rows = workspace_rows(batch, s_q, num_sm_parts) * h_q;
  const float* ws_o = static_cast<const float*>(workspace);
  const float* ws_lse = ws_o + rows * kDv;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(batch * s_q, h_q, 1);
  cfg.blockDim = dim3(kCombineThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, combine_kernel, static_cast<const int32_t*>(metadata),
                                           h_q, s_q, num_sm_parts, ws_o, ws_lse,
                                           static_cast<__nv_bfloat16*>(out), lse);
  return e == cudaSuccess ? MLA_OK : record_cuda_error("combine kernel launch", e);
}

}  // namespace mla

extern "C" int mla_combine(const void* metadata, int batch, int s_q, int h_q, int num_sm_parts,
                           const void* workspace, void* out, float* lse, cudaStream_t stream) {
  const int rc = mla::check_common(batch, s_q, h_q, num_sm_parts);
  if (rc != MLA_OK) return rc;
  if (!metadata || !workspace || !out || !lse) return MLA_ERR_NULL;
  if (!mla::aligned16(metadata) || !mla::aligned16(workspace) || !mla::aligned16(out))
    return MLA_ERR_ALIGN;
  return mla::launch_combine(metadata, batch, s_q, h_q, num_sm_parts, workspace, out, lse, stream,
                             false);
}
