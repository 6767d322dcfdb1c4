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

constexpr int kCombineWarps = 8;  // one output row (query token, head) per warp
constexpr int kCombineThreads = 32 * kCombineWarps;

// Lane l of a warp owns output columns [16 l, 16 l + 16): each split row is read
// as 2 KB contiguous per warp, and the bf16 row is written as 1 KB contiguous.
// At most 80 registers per thread (three CTAs, 24 warps per SM): no spills.
// attn_sink (optional, [h]): the merged row is scaled by e^lse / (e^lse + e^sink).
__global__ void __launch_bounds__(kCombineThreads, 3) combine_kernel(
    const int32_t* __restrict__ meta, int batch, int h, int s_q, int num_parts, const float* __restrict__ ws_o,
    const float* __restrict__ ws_lse, const int32_t* __restrict__ ws_ctrl, const float* __restrict__ attn_sink,
    __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  const int q = blockIdx.x;
  const int head = blockIdx.y * kCombineWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  pdl_wait_primary();
  // The split kernel recorded in the workspace which schedule it walked (-1
  // when it rejected the metadata) and whether that schedule left anything to
  // merge or fill; with nothing to do, no other word is read.
  const int32_t walked = ws_ctrl[0];
  if ((walked != 0 && walked != 1) || ws_ctrl[1] == 0) return;
  // Metadata for another shape: the split kernel computed nothing (and set
  // MLA_DEVERR_METADATA); write nothing either.  The topk and causal words
  // do not change the layout, so any matching batch / s_q / parts passes.
  if (meta[kHMagic] != kMetaMagic || meta[kHVersion] != kMetaVersion || meta[kHNSeq] != batch * s_q ||
      meta[kHParts] != num_parts || meta[kHSq] != s_q || meta[kHBatch] != batch)
    return;
  const bool use_b = walked == 1 && schedule_b(meta)[kHMagic] == kMetaMagic;
  const int32_t* sched = use_b ? schedule_b(meta) : meta;
  const int32_t* s = meta_seq(sched, num_parts, q);
  const int n_splits = s[kSNSplits];
  const int off = s[kSSplitOff];
  if (head >= h || n_splits == 1) return;  // single split: written by the split kernel
  const int b = q / s_q, j = q % s_q;
  __nv_bfloat16* orow = out + (static_cast<int64_t>(q) * h + head) * kDv + 16 * lane;
  float* lse_out = lse + (static_cast<int64_t>(b) * h + head) * s_q + j;
  if (n_splits == 0) {  // no visible key: out = 0, lse = -inf
    reinterpret_cast<uint4*>(orow)[0] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(orow)[1] = make_uint4(0u, 0u, 0u, 0u);
    if (lane == 0) *lse_out = -INFINITY;
    return;
  }
  const float4* src = reinterpret_cast<const float4*>(ws_o + (static_cast<int64_t>(off) * h + head) * kDv) + 4 * lane;
  const int64_t split_stride = static_cast<int64_t>(h) * kDv / 4;  // in float4
  // split 0's row is requested before the weights are known; split i + 1's
  // while split i is accumulated
  float4 cur[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) cur[c] = src[c];
  // merged lse = ref + ln sum_i exp(lse_i - ref), ref = max_i lse_i
  const float* lrow = ws_lse + static_cast<int64_t>(off) * h + head;
  float mx = -INFINITY;
  for (int i = lane; i < n_splits; i += 32) mx = fmaxf(mx, lrow[static_cast<int64_t>(i) * h]);
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, sh));
  const float ref = (mx == -INFINITY) ? 0.f : mx;
  float my_e = 0.f, sum = 0.f;
  for (int i = lane; i < n_splits; i += 32) {
    const float e = __expf(lrow[static_cast<int64_t>(i) * h] - ref);
    if (i < 32) my_e = e;
    sum += e;
  }
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
  const float total_lse = sum > 0.f ? ref + __logf(sum) : -INFINITY;
  float inv = sum > 0.f ? 1.f / sum : 0.f;
  if (attn_sink) inv *= attn_sink_factor(total_lse, attn_sink[head]);
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  for (int i = 0; i < n_splits; ++i) {
    float4 nxt[4];
    if (i + 1 < n_splits) {
#pragma unroll
      for (int c = 0; c < 4; ++c) nxt[c] = src[(i + 1) * split_stride + c];
    }
    const float w = (i < 32 ? __shfl_sync(0xffffffffu, my_e, i & 31) : __expf(lrow[static_cast<int64_t>(i) * h] - ref)) * inv;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      acc[4 * c] += w * cur[c].x; acc[4 * c + 1] += w * cur[c].y;
      acc[4 * c + 2] += w * cur[c].z; acc[4 * c + 3] += w * cur[c].w;
    }
    if (i + 1 < n_splits) {
#pragma unroll
      for (int c = 0; c < 4; ++c) cur[c] = nxt[c];
    }
  }
  uint32_t pk[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
  reinterpret_cast<uint4*>(orow)[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  reinterpret_cast<uint4*>(orow)[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  if (lane == 0) *lse_out = total_lse;
}

}  // namespace

int launch_combine(const void* metadata, int batch, int s_q, int h_q, int num_sm_parts,
                   const void* workspace, const float* attn_sink, void* out, float* lse,
                   cudaStream_t stream, bool pdl) {
  const int64_t rows = workspace_rows(batch, s_q, num_sm_parts) * h_q;
  const float* ws_o = static_cast<const float*>(workspace);
  const float* ws_lse = ws_o + rows * kDv;
  const int32_t* ws_ctrl = workspace_ctrl(workspace, rows);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(batch * s_q, (h_q + kCombineWarps - 1) / kCombineWarps, 1);
  cfg.blockDim = dim3(kCombineThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, combine_kernel, static_cast<const int32_t*>(metadata),
                                           batch, h_q, s_q, num_sm_parts, ws_o, ws_lse, ws_ctrl, attn_sink,
                                           static_cast<__nv_bfloat16*>(out), lse);
  return e == cudaSuccess ? MLA_OK : record_cuda_error("combine kernel launch", e);
}

}  // namespace mla

extern "C" int mla_combine(const void* metadata, int batch, int s_q, int h_q, int num_sm_parts,
                           const void* workspace, const float* attn_sink, void* out, float* lse,
                           cudaStream_t stream) {
  const int rc = mla::check_common(batch, s_q, h_q, num_sm_parts);
  if (rc != MLA_OK) return rc;
  if (!metadata || !workspace || !out || !lse) return MLA_ERR_NULL;
  if (!mla::aligned16(metadata) || !mla::aligned16(workspace) || !mla::aligned16(out))
    return MLA_ERR_ALIGN;
  return mla::launch_combine(metadata, batch, s_q, h_q, num_sm_parts, workspace, attn_sink, out, lse,
                             stream, false);
}
