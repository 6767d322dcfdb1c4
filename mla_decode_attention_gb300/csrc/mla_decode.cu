// Host entry points of the split-KV decode: argument checks, TMA tensor maps,
// the cluster launch of the split kernel and the PDL launch of the combine.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "mla_decode.h"
#include "mla_internal.h"
#include "mla_splitkv.cuh"
#include "mla_pair.cuh"

namespace mla {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 row-major tensor [rows, cols] (cols = 576, or 512 for V4.1
// queries) with row stride `stride_bytes`; boxes of [box_rows x 64 columns]
// with 128-byte swizzle.
bool make_rows_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t stride_bytes,
                   uint32_t box_rows, uint64_t cols = kDqk) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), rows};
  const cuuint64_t strides[1] = {stride_bytes};
  const cuuint32_t box[2] = {64u, box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The paged bf16 cache seen as a 4-D tensor [8-token groups][9 chunks][8
// rows][64 columns] (strides: row 1152 bytes, chunk 128 bytes, group 9216
// bytes); boxes of [8 groups][`chunks`][8 rows][64 columns] (one page's
// chunks, starting at the chunk given at load time) with 128-byte swizzle,
// landing as [group][chunk][row][128 bytes].
bool make_quad_map(CUtensorMap* m, const void* base, uint64_t num_pages, uint32_t chunks) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {64u, 8u, static_cast<cuuint64_t>(kDqk / 64), num_pages * (kPage / 8)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kDqk) * 2u, 128u, static_cast<cuuint64_t>(kDqk) * 2u * 8u};
  const cuuint32_t box[4] = {64u, 8u, chunks, static_cast<cuuint32_t>(kPage / 8)};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 tensor [rows, cols] whose rows start `stride_bytes` apart; boxes of
// [box_rows x 64 columns] with 128-byte swizzle.
bool make_strided_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                      uint64_t stride_bytes, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), rows};
  const cuuint64_t strides[1] = {stride_bytes};
  const cuuint32_t box[2] = {64u, box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte tensor [rows, cols] whose rows start `stride_bytes` apart; boxes of
// [box_rows x box_cols bytes], not swizzled.
bool make_byte_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                   uint64_t stride_bytes, uint32_t box_cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {stride_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <KvMode kMode>
int configure_kernel() {
  static int state = 0;  // 0 unset, 1 ok, -1 failed
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (state == 0) {
    const cudaError_t e = cudaFuncSetAttribute(
        mla_splitkv_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    state = e == cudaSuccess ? 1 : -1;
    if (e != cudaSuccess) return record_cuda_error("cudaFuncSetAttribute(split kernel)", e);
  }
  return state == 1 ? MLA_OK : record_error("split kernel configuration failed earlier", MLA_ERR_CUDA);
}

template <KvMode kMode>
int launch_split(const CUtensorMap& tm_q, const CUtensorMap& tm_kv, const SplitParams& prm,
                 cudaStream_t stream, const CUtensorMap* tm_codes = nullptr,
                 const CUtensorMap* tm_scales = nullptr) {
  int rc = configure_kernel<kMode>();
  if (rc != MLA_OK) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.num_parts * prm.n_hblk, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = prm.n_hblk;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // the FP8 code and scale maps are read only by the FP8 instantiation
  const cudaError_t e = cudaLaunchKernelEx(&cfg, mla_splitkv_kernel<kMode>, tm_q, tm_kv,
                                           tm_codes ? *tm_codes : tm_kv,
                                           tm_scales ? *tm_scales : tm_kv, prm);
  return e == cudaSuccess ? MLA_OK : record_cuda_error("split kernel launch", e);
}

// The query rows [n_seq * 128, 576] seen as [9 chunks][rows][64 columns]
// (chunk stride 128 bytes); boxes of [2 chunks x 128 rows x 64 columns] (a
// quarter of the latent part of one token's rows, 32 KB) with 128-byte swizzle.
bool make_q_latent_map(CUtensorMap* m, const void* q, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {64u, rows, static_cast<cuuint64_t>(kDqk / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kDqk) * 2u, 128u};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(pair::kRows), 2u};  // two chunks per box
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// tm_qa, tm_qb: the group-interleaved maps of the paged cache (chunks 0..3,
// 4..6 of a page); the sparse kernel does not read them.  The kernel loads the
// part's first query rows with the two query maps made here.
template <bool kSparse>
int launch_pair(const CUtensorMap& tm_kv, const CUtensorMap& tm_qa, const CUtensorMap& tm_qb,
                const SplitParams& prm, cudaStream_t stream) {
  CUtensorMap tm_ql, tm_qr;
  const uint64_t q_rows = static_cast<uint64_t>(prm.batch) * prm.s_q * pair::kRows;
  if (!make_q_latent_map(&tm_ql, prm.q, q_rows) || !make_rows_map(&tm_qr, prm.q, q_rows, kDqk * 2, pair::kRows))
    return record_error("cuTensorMapEncodeTiled failed for the query rows", MLA_ERR_CUDA);
  static int state = 0;  // 0 unset, 1 ok, -1 failed (per instantiation)
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (state == 0) {
      const cudaError_t e = cudaFuncSetAttribute(
          pair::mla_pair_kernel<kSparse>, cudaFuncAttributeMaxDynamicSharedMemorySize, pair::kSmemBytes);
      state = e == cudaSuccess ? 1 : -1;
      if (e != cudaSuccess) return record_cuda_error("cudaFuncSetAttribute(pair kernel)", e);
    }
    if (state != 1) return record_error("pair kernel configuration failed earlier", MLA_ERR_CUDA);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.num_parts * 2, 1, 1);
  cfg.blockDim = dim3(kSparse ? pair::kThreadsSparse : pair::kThreads, 1, 1);
  cfg.dynamicSmemBytes = pair::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // the kernel's prologue overlaps the previous kernel (e.g. the schedule);
  // it waits for that kernel's results before reading any input
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, pair::mla_pair_kernel<kSparse>, tm_kv, tm_qa, tm_qb, tm_ql, tm_qr, prm);
  return e == cudaSuccess ? MLA_OK : record_cuda_error("pair kernel launch", e);
}

}  // namespace

}  // namespace mla

using namespace mla;

extern "C" int mla_decode_splitkv(const void* q, const void* kv_cache, int kv_format,
                                  int64_t num_pages, const int32_t* block_table,
                                  int64_t block_table_stride, const int32_t* cache_seqlens,
                                  int batch, int s_q, int h_q, float softmax_scale, int causal,
                                  const void* metadata, int num_sm_parts, void* workspace,
                                  void* out, float* lse, uint32_t* err, cudaStream_t stream) {
  int rc = check_common(batch, s_q, h_q, num_sm_parts);
  if (rc != MLA_OK) return rc;
  if (!q || !kv_cache || !block_table || !cache_seqlens || !metadata || !workspace || !out || !lse)
    return MLA_ERR_NULL;
  if (kv_format != MLA_KV_BF16 && kv_format != MLA_KV_FP8_656 && kv_format != MLA_KV_FP8_528)
    return MLA_ERR_UNSUPPORTED;
  if (num_pages <= 0 || num_pages > (int64_t{1} << 25) || block_table_stride <= 0)
    return MLA_ERR_SHAPE;
  if (!(softmax_scale > 0.f) || !(softmax_scale < 1e30f)) return MLA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(metadata) || !aligned16(workspace) ||
      !aligned16(out))
    return MLA_ERR_ALIGN;

  const int n_seq = batch * s_q;
  const int n_hblk = head_blocks(h_q);
  const int rows = h_q < kRowsPerCta ? h_q : kRowsPerCta;
  // the V4.1 cache holds 512-wide keys (values are the whole key), others 576
  const bool v41 = kv_format == MLA_KV_FP8_528;
  const int d_qk = v41 ? kV41HeadDim : kDqk;
  CUtensorMap tm_q, tm_kv, tm_codes, tm_scales;
  if (!make_rows_map(&tm_q, q, static_cast<uint64_t>(n_seq) * h_q, d_qk * 2, rows, d_qk))
    return record_error("cuTensorMapEncodeTiled failed for q", MLA_ERR_CUDA);
  const bool fp8 = kv_format == MLA_KV_FP8_656;
  if (v41) {
    // the 512 e4m3 codes (boxes of 64 tokens x 64 codes) and the 16 e8m0
    // scales at byte 512 (boxes of 64 tokens x 16 bytes) of every 528-byte
    // token; no bf16 part (tm_kv is not read)
    const uint64_t tokens = static_cast<uint64_t>(num_pages) * kPage;
    if (!make_byte_map(&tm_codes, kv_cache, tokens, kV41HeadDim, kFp8V41TokenBytes, 64, kPage) ||
        !make_byte_map(&tm_scales, static_cast<const uint8_t*>(kv_cache) + kV41HeadDim, tokens, 16,
                       kFp8V41TokenBytes, 16, kPage))
      return record_error("cuTensorMapEncodeTiled failed for the V4.1 FP8 codes or scales", MLA_ERR_CUDA);
    tm_kv = tm_codes;
  } else if (!fp8) {
    if (!make_rows_map(&tm_kv, kv_cache, static_cast<uint64_t>(num_pages) * kPage, kDqk * 2, kPage))
      return record_error("cuTensorMapEncodeTiled failed for kv_cache", MLA_ERR_CUDA);
  } else {
    // the bf16 RoPE tail of every 656-byte token: 64 columns at byte 528,
    // row stride 656 bytes (both multiples of 16)
    const void* rope = static_cast<const uint8_t*>(kv_cache) + kFp8RopeOffset;
    if (!make_strided_map(&tm_kv, rope, static_cast<uint64_t>(num_pages) * kPage, 64,
                          kFp8TokenBytes, kPage))
      return record_error("cuTensorMapEncodeTiled failed for the FP8 RoPE columns", MLA_ERR_CUDA);
    // the 512 e4m3 codes (boxes of 64 tokens x 64 codes) and the 16 scale
    // bytes at byte 512 (boxes of 64 tokens x 16 bytes) of every token
    const uint64_t tokens = static_cast<uint64_t>(num_pages) * kPage;
    if (!make_byte_map(&tm_codes, kv_cache, tokens, kFp8ScaleOffset, kFp8TokenBytes, 64, kPage) ||
        !make_byte_map(&tm_scales, static_cast<const uint8_t*>(kv_cache) + kFp8ScaleOffset, tokens,
                       16, kFp8TokenBytes, 16, kPage))
      return record_error("cuTensorMapEncodeTiled failed for the FP8 codes or scales", MLA_ERR_CUDA);
  }

  SplitParams prm = {};
  prm.meta = static_cast<const int32_t*>(metadata);
  prm.block_table = block_table;
  prm.bt_stride = block_table_stride;
  prm.num_pages = num_pages;
  prm.cache_seqlens = cache_seqlens;
  prm.causal = causal ? 1 : 0;
  prm.batch = batch;
  prm.topk = 0;
  prm.kv_rows = static_cast<const __nv_bfloat16*>(kv_cache);
  prm.kv_fp8 = static_cast<const uint8_t*>(kv_cache);
  prm.q = static_cast<const __nv_bfloat16*>(q);
  const int64_t ws_rows = workspace_rows(batch, s_q, num_sm_parts) * h_q;
  prm.ws_o = static_cast<float*>(workspace);
  prm.ws_lse = prm.ws_o + ws_rows * kDv;
  prm.ws_ctrl = workspace_ctrl(workspace, ws_rows);
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.lse = lse;
  prm.err = err;
  prm.h = h_q;
  prm.d_qk = d_qk;
  prm.s_q = s_q;
  prm.num_parts = num_sm_parts;
  prm.n_hblk = n_hblk;
  prm.rows = rows;
  prm.scale_log2 = softmax_scale * 1.4426950408889634f;
  if (v41) return launch_split<KvMode::kPagedFp8V41>(tm_q, tm_kv, prm, stream, &tm_codes, &tm_scales);
  if (fp8) return launch_split<KvMode::kPagedFp8>(tm_q, tm_kv, prm, stream, &tm_codes, &tm_scales);
  // 128 query rows: the two-SM kernel (scores and softmax on one SM, P.V on the other)
  if (h_q == pair::kRows) {
    CUtensorMap tm_qa, tm_qb;
    if (!make_quad_map(&tm_qa, kv_cache, static_cast<uint64_t>(num_pages), 4) ||
        !make_quad_map(&tm_qb, kv_cache, static_cast<uint64_t>(num_pages), 3))
      return record_error("cuTensorMapEncodeTiled failed for the kv_cache page groups", MLA_ERR_CUDA);
    return launch_pair<false>(tm_kv, tm_qa, tm_qb, prm, stream);
  }
  return launch_split<KvMode::kPagedBf16>(tm_q, tm_kv, prm, stream);
}

extern "C" int mla_decode(const void* q, const void* kv_cache, int kv_format, int64_t num_pages,
                          const int32_t* block_table, int64_t block_table_stride,
                          const int32_t* cache_seqlens, int batch, int s_q, int h_q,
                          float softmax_scale, int causal, const void* metadata, int num_sm_parts,
                          void* workspace, void* out, float* lse, uint32_t* err,
                          cudaStream_t stream) {
  const int rc = mla_decode_splitkv(q, kv_cache, kv_format, num_pages, block_table,
                                    block_table_stride, cache_seqlens, batch, s_q, h_q,
                                    softmax_scale, causal, metadata, num_sm_parts, workspace, out,
                                    lse, err, stream);
  if (rc != MLA_OK) return rc;
  return launch_combine(metadata, batch, s_q, h_q, num_sm_parts, workspace, nullptr, out, lse, stream,
                        true);
}

extern "C" int mla_sparse_decode_splitkv(const void* q, const void* kv, int64_t s_kv,
                                         const int32_t* indices, int topk, int batch, int s_q,
                                         int h_q, float softmax_scale, const float* attn_sink,
                                         const void* metadata, int num_sm_parts, void* workspace, void* out,
                                         float* lse, uint32_t* err, cudaStream_t stream) {
  int rc = check_common(batch, s_q, h_q, num_sm_parts);
  if (rc != MLA_OK) return rc;
  if (!q || !kv || !indices || !metadata || !workspace || !out || !lse) return MLA_ERR_NULL;
  if (topk <= 0 || s_kv <= 0 || s_kv > (int64_t{1} << 31) - 1) return MLA_ERR_SHAPE;
  if (!(softmax_scale > 0.f) || !(softmax_scale < 1e30f)) return MLA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(metadata) || !aligned16(workspace) ||
      !aligned16(out))
    return MLA_ERR_ALIGN;

  const int n_seq = batch * s_q;
  const int rows = h_q < kRowsPerCta ? h_q : kRowsPerCta;
  CUtensorMap tm_q, tm_kv;
  if (!make_rows_map(&tm_q, q, static_cast<uint64_t>(n_seq) * h_q, kDqk * 2, rows))
    return record_error("cuTensorMapEncodeTiled failed for q", MLA_ERR_CUDA);
  // one-row boxes: each tile::gather4 fetches four arbitrary pool rows
  if (!make_rows_map(&tm_kv, kv, static_cast<uint64_t>(s_kv), kDqk * 2, 1))
    return record_error("cuTensorMapEncodeTiled failed for kv", MLA_ERR_CUDA);

  SplitParams prm = {};
  prm.meta = static_cast<const int32_t*>(metadata);
  prm.batch = batch;
  prm.causal = 0;
  prm.indices = indices;
  prm.attn_sink = attn_sink;
  prm.topk = topk;
  prm.s_kv = s_kv;
  prm.kv_rows = static_cast<const __nv_bfloat16*>(kv);
  prm.q = static_cast<const __nv_bfloat16*>(q);
  const int64_t ws_rows = workspace_rows(batch, s_q, num_sm_parts) * h_q;
  prm.ws_o = static_cast<float*>(workspace);
  prm.ws_lse = prm.ws_o + ws_rows * kDv;
  prm.ws_ctrl = workspace_ctrl(workspace, ws_rows);
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.lse = lse;
  prm.err = err;
  prm.h = h_q;
  prm.d_qk = kDqk;
  prm.s_q = s_q;
  prm.num_parts = num_sm_parts;
  prm.n_hblk = head_blocks(h_q);
  prm.rows = rows;
  prm.scale_log2 = softmax_scale * 1.4426950408889634f;
  // 128 query rows: the two-SM kernel with gathered keys
  return h_q == pair::kRows ? launch_pair<true>(tm_kv, tm_kv, tm_kv, prm, stream)
                            : launch_split<KvMode::kSparseBf16>(tm_q, tm_kv, prm, stream);
}

extern "C" int mla_sparse_decode(const void* q, const void* kv, int64_t s_kv,
                                 const int32_t* indices, int topk, int batch, int s_q, int h_q,
                                 float softmax_scale, const float* attn_sink, const void* metadata,
                                 int num_sm_parts, void* workspace, void* out, float* lse,
                                 uint32_t* err, cudaStream_t stream) {
  const int rc = mla_sparse_decode_splitkv(q, kv, s_kv, indices, topk, batch, s_q, h_q,
                                           softmax_scale, attn_sink, metadata, num_sm_parts,
                                           workspace, out, lse, err, stream);
  if (rc != MLA_OK) return rc;
  return launch_combine(metadata, batch, s_q, h_q, num_sm_parts, workspace, attn_sink, out, lse, stream,
                        true);
}

// DSA sparse prefill through the sparse decode path, each query token a
// request of one token (q [s_q, h_q, 576] is [s_q, 1, h_q, 576], indices
// [s_q, 1, topk] is [s_q, 1, topk], out [s_q, h_q, 512] is [s_q, 1, h_q, 512],
// lse [s_q, h_q] is [s_q, h_q, 1]).
extern "C" int mla_sparse_prefill(const void* q, const void* kv, int64_t s_kv, const int32_t* indices,
                                  int topk, int s_q, int h_q, float softmax_scale, const float* attn_sink,
                                  const void* metadata, int num_sm_parts, void* workspace, void* out,
                                  float* lse, uint32_t* err, cudaStream_t stream) {
  return mla_sparse_decode(q, kv, s_kv, indices, topk, s_q, 1, h_q, softmax_scale, attn_sink, metadata,
                           num_sm_parts, workspace, out, lse, err, stream);
}
