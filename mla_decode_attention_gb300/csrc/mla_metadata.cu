// Tile-schedule metadata (device kernel and host mirror) and small host
// entry points of the C ABI.
#include <algorithm>
#include <cstdio>
#include <vector>

#include "mla_decode.h"
#include "mla_internal.h"
#include "mla_ptx.cuh"
#include "mla_schedule.cuh"

namespace mla {

namespace {

constexpr int kSmemPrefixes = 8192;  // sequences whose cost prefixes the schedule keeps in smem
// Up to this many sequences the schedule builds the sequence records in shared
// memory and writes them out once at the end (no global read-after-write
// round trips between the phases).
constexpr int kSmemRecords = 256;
// one CTA of 128 threads up to this many sequences (fewer warps to meet at
// each barrier), else 1024
constexpr int kSmallMetaSeqs = 2048;
// schedule B's count of non-empty sequences rides in the low bits of the cost scan
constexpr int kCountBits = 25;  // n_seq <= 2^24

// Block-wide exclusive scan of one int64 per thread; returns the total.
template <int kMetaThreads>
__device__ int64_t block_exclusive_scan(int64_t v, int64_t* out_excl, int64_t* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t w = (lane < (kMetaThreads / 32)) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;  // inclusive
  }
  __syncthreads();
  const int64_t before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  const int64_t total = warp_sums[kMetaThreads / 32 - 1];
  __syncthreads();
  *out_excl = before;
  return total;
}

// One CTA builds the whole schedule.  Thread i owns the contiguous sequence
// chunk [i*chunk, (i+1)*chunk).
template <int kMetaThreads>
__global__ void __launch_bounds__(kMetaThreads) metadata_kernel(const int32_t* seqlens, int batch,
                                                                int s_q, int causal, int topk,
                                                                int num_parts, int32_t* meta) {
  __shared__ int64_t warp_sums[32];
  __shared__ int32_t s_prefix[kSmemPrefixes];
  __shared__ int32_t s_rec[kSmemRecords * kSeqWords];
  // a decode kernel launched next may start its prologue; it waits for this
  // grid to complete before it reads the schedule
  pdl_launch_dependents();
  const int n_seq = batch * s_q;
  // sequences are walked in group-major order k (schedule_groups)
  const int groups = schedule_groups(s_q, num_parts);
  const int n_g = n_seq / groups, parts_g = num_parts / groups;
  const int chunk = (n_seq + kMetaThreads - 1) / kMetaThreads;
  const int k0 = threadIdx.x * chunk;
  const int k1 = min(n_seq, k0 + chunk);

  __shared__ int32_t s_max_cost;
  __shared__ int64_t s_group_start[kMaxSq + 1];
  if (threadIdx.x == 0) s_max_cost = 0;
  __syncthreads();
  // the sequence records of schedule A: built in shared memory when they fit
  const bool rec_smem = n_seq <= kSmemRecords;
  int32_t* const recs = rec_smem ? s_rec : meta_seq(meta, num_parts, 0);
  auto rec = [&](int q) { return recs + kSeqWords * q; };

  // 1. tiles, keys and cost per sequence; chunk-local cost prefix.
  int64_t local = 0;
  int32_t local_max = 0, local_nonempty = 0;
  for (int k = k0; k < k1; ++k) {
    const int q = order_to_q(k, n_g, groups);
    const int32_t keys = seq_keys(seqlens, q / s_q, q % s_q, s_q, causal, topk);
    const int32_t nt = tiles_of(keys);
    int32_t* s = rec(q);
    s[kSTiles] = nt; s[kSKeys] = keys; s[5] = 0; s[6] = 0; s[7] = 0;
    s[kSCostPrefix] = static_cast<int32_t>(local);
    local += cost_of(nt);
    local_max = max(local_max, cost_of(nt));
    local_nonempty += nt > 0 ? 1 : 0;
  }
  atomicMax(&s_max_cost, local_max);
  int64_t packed_base;
  const int64_t packed_total = block_exclusive_scan<kMetaThreads>(
      (local << kCountBits) | local_nonempty, &packed_base, warp_sums);
  const int64_t base = packed_base >> kCountBits, total = packed_total >> kCountBits;
  const int64_t b_base = packed_base & ((int64_t{1} << kCountBits) - 1);
  const int64_t b_splits = packed_total & ((int64_t{1} << kCountBits) - 1);
  // where each group starts on the group-major cost line
  for (int k = k0; k < k1; ++k)
    if (k % n_g == 0)
      s_group_start[k / n_g] = base + rec(order_to_q(k, n_g, groups))[kSCostPrefix];
  if (threadIdx.x == 0) s_group_start[groups] = total;
  __syncthreads();
  // prefixes within each group's own cost line
  for (int k = k0; k < k1; ++k) {
    const int q = order_to_q(k, n_g, groups);
    int32_t* sq = rec(q);
    sq[kSCostPrefix] = static_cast<int32_t>(base + sq[kSCostPrefix] - s_group_start[k / n_g]);
    if (n_seq <= kSmemPrefixes) s_prefix[q] = sq[kSCostPrefix];
  }
  int64_t max_group_total = 0;
  for (int j = 0; j < groups; ++j) max_group_total = max(max_group_total, s_group_start[j + 1] - s_group_start[j]);
  __syncthreads();

  const int64_t per_part = max_group_total > 0 ? floordiv(max_group_total + parts_g - 1, parts_g) : 1;

  // 2. split counts per sequence (from the prefixes only).
  int64_t nsplit_local = 0;
  for (int k = k0; k < k1; ++k) {
    int32_t* s = rec(order_to_q(k, n_g, groups));
    const int32_t nt = s[kSTiles];
    const int32_t ns = nt > 0 ? 1 + inner_boundaries(s[kSCostPrefix], nt, per_part) : 0;
    s[kSNSplits] = ns;
    nsplit_local += ns;
  }
  int64_t split_base;
  const int64_t total_splits = block_exclusive_scan<kMetaThreads>(nsplit_local, &split_base, warp_sums);
  int64_t run = split_base;
  for (int k = k0; k < k1; ++k) {
    int32_t* s = rec(order_to_q(k, n_g, groups));
    s[kSSplitOff] = static_cast<int32_t>(run);
    run += s[kSNSplits];
  }
  __syncthreads();

  // 3. part ranges: part p is part p % parts_g of group p / parts_g
  // (the binary searches read the prefixes from shared memory when they fit)
  for (int p = threadIdx.x; p < num_parts; p += kMetaThreads) {
    const int j = p / parts_g;
    const int64_t total_j = s_group_start[j + 1] - s_group_start[j];
    if (n_seq <= kSmemPrefixes)
      fill_part(meta, GroupPrefix<ArrayPrefix>{ArrayPrefix{s_prefix}, j, groups}, n_g, total_j, per_part, p,
                p % parts_g, j, groups);
    else
      fill_part(meta, GroupPrefix<MetaPrefix>{MetaPrefix{meta, num_parts}, j, groups}, n_g, total_j, per_part,
                p, p % parts_g, j, groups);
  }

  // 4. schedule B (one whole sequence per part), when every sequence has a part.
  const bool has_b = n_seq <= num_parts;
  int32_t* mb = meta + meta_words(n_seq, num_parts);
  if (has_b) {
    int64_t run_b = b_base;
    for (int k = k0; k < k1; ++k) {
      const int q = order_to_q(k, n_g, groups);
      const int32_t* sa = rec(q);
      int32_t* sb = meta_seq(mb, num_parts, q);
      const int32_t nt = sa[kSTiles];
      sb[kSTiles] = nt; sb[kSSplitOff] = static_cast<int32_t>(run_b); sb[kSNSplits] = nt > 0 ? 1 : 0;
      sb[kSKeys] = sa[kSKeys]; sb[kSCostPrefix] = sa[kSCostPrefix]; sb[5] = 0; sb[6] = 0; sb[7] = 0;
      run_b += nt > 0 ? 1 : 0;
    }
    for (int p = threadIdx.x; p < num_parts; p += kMetaThreads) fill_whole_part(mb, num_parts, n_seq, p);
  }
  if (rec_smem) {  // schedule A's sequence records out to the metadata
    __syncthreads();
    int32_t* out = meta_seq(meta, num_parts, 0);
    for (int i = threadIdx.x; i < n_seq * kSeqWords; i += kMetaThreads) out[i] = s_rec[i];
  }

  if (threadIdx.x == 0) {
    const int32_t max_cost = s_max_cost;
    meta[kHMagic] = kMetaMagic; meta[kHVersion] = kMetaVersion; meta[kHNSeq] = n_seq;
    meta[kHParts] = num_parts; meta[kHTile] = kTileTokens; meta[kHSq] = s_q;
    meta[kHBatch] = batch; meta[kHCausal] = causal; meta[kHTopk] = topk;
    meta[kHTotalSplits] = static_cast<int32_t>(total_splits);
    meta[kHPerPart] = static_cast<int32_t>(per_part);
    meta[kHMaxCost] = max_cost;
    meta[kHHasB] = has_b ? 1 : 0;
    meta[kHGroups] = groups;
    for (int i = kHGroups + 1; i < kHeaderWords; ++i) meta[i] = 0;
    for (int i = 0; i < kHeaderWords; ++i) mb[i] = has_b ? meta[i] : 0;
    if (has_b) {
      mb[kHTotalSplits] = static_cast<int32_t>(b_splits);
      mb[kHPerPart] = max_cost;
      mb[kHHasB] = 0;
      mb[kHGroups] = 1;
    }
  }
}

// One thread waits on an mbarrier that nothing arrives on: the decode
// kernels' bounded wait gives up after its limit, flags MLA_DEVERR_TIMEOUT and
// returns, and the block exits normally.
__global__ void wait_timeout_kernel(uint32_t* err) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbarrier_init();
    (void)mbar_wait(smem_u32(&bar), 0, &abort_flag, err);
  }
}

}  // namespace

namespace {
thread_local char g_last_error[256] = "no error";
}

int record_cuda_error(const char* where, cudaError_t e) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(e),
                static_cast<int>(e));
  return MLA_ERR_CUDA;
}

int record_error(const char* what, int status) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s", what);
  return status;
}

int check_common(int batch, int s_q, int h_q, int num_sm_parts) {
  if (batch <= 0 || s_q <= 0 || s_q > kMaxSq || num_sm_parts <= 0) return MLA_ERR_SHAPE;
  if (!heads_supported(h_q)) return MLA_ERR_SHAPE;
  if (static_cast<int64_t>(batch) * s_q > (1 << 24)) return MLA_ERR_SHAPE;
  return MLA_OK;
}

}  // namespace mla

using namespace mla;

extern "C" const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_NULL: return "a required pointer is NULL";
    case MLA_ERR_SHAPE: return "unsupported or inconsistent size argument";
    case MLA_ERR_ALIGN: return "pointer or stride is not 16-byte aligned";
    case MLA_ERR_METADATA: return "metadata does not match this call";
    case MLA_ERR_CUDA: return "a CUDA runtime call failed";
    case MLA_ERR_UNSUPPORTED: return "device is not supported (needs sm_103 / sm_100 class)";
    default: return "unknown status";
  }
}

extern "C" const char* mla_last_error(void) { return g_last_error; }

extern "C" int mla_check_wait_timeout(uint32_t* err, cudaStream_t stream) {
  if (!err) return MLA_ERR_NULL;
  wait_timeout_kernel<<<1, 32, 0, stream>>>(err);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MLA_OK : record_cuda_error("wait-timeout check launch", e);
}

extern "C" int mla_num_sm_parts(int device, int h_q, int* num_sm_parts) {
  if (!num_sm_parts) return MLA_ERR_NULL;
  if (!heads_supported(h_q)) return MLA_ERR_SHAPE;
  int sms = 0;
  const cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) return record_cuda_error("cudaDeviceGetAttribute", e);
  *num_sm_parts = sms / head_blocks(h_q);
  return *num_sm_parts > 0 ? MLA_OK : MLA_ERR_UNSUPPORTED;
}

extern "C" int mla_metadata_size(int batch, int s_q, int num_sm_parts, size_t* bytes) {
  if (!bytes) return MLA_ERR_NULL;
  if (batch <= 0 || s_q <= 0 || s_q > kMaxSq || num_sm_parts <= 0) return MLA_ERR_SHAPE;
  *bytes = static_cast<size_t>(meta_total_words(batch * s_q, num_sm_parts)) * sizeof(int32_t);
  return MLA_OK;
}

extern "C" int mla_workspace_size(int batch, int s_q, int h_q, int num_sm_parts, size_t* bytes) {
  if (!bytes) return MLA_ERR_NULL;
  const int rc = check_common(batch, s_q, h_q, num_sm_parts);
  if (rc != MLA_OK) return rc;
  const int64_t rows = workspace_rows(batch, s_q, num_sm_parts) * h_q;
  *bytes = static_cast<size_t>(rows) * (kDv + 1) * sizeof(float) + kWorkspaceCtrlBytes;
  return MLA_OK;
}

static int check_meta_args(const int32_t* seqlens, int batch, int s_q, int topk, int num_sm_parts,
                           const void* meta) {
  if (!meta) return MLA_ERR_NULL;
  if (topk <= 0 && !seqlens) return MLA_ERR_NULL;
  if (batch <= 0 || s_q <= 0 || s_q > kMaxSq || num_sm_parts <= 0 || topk < 0)
    return MLA_ERR_SHAPE;
  if (static_cast<int64_t>(batch) * s_q > (1 << 24)) return MLA_ERR_SHAPE;
  if (!aligned16(meta)) return MLA_ERR_ALIGN;
  return MLA_OK;
}

extern "C" int mla_get_metadata(const int32_t* cache_seqlens, int batch, int s_q, int causal,
                                int topk, int num_sm_parts, void* metadata, cudaStream_t stream) {
  const int rc = check_meta_args(cache_seqlens, batch, s_q, topk, num_sm_parts, metadata);
  if (rc != MLA_OK) return rc;
  if (static_cast<int64_t>(batch) * s_q <= kSmallMetaSeqs)
    metadata_kernel<128><<<1, 128, 0, stream>>>(cache_seqlens, batch, s_q, causal ? 1 : 0, topk,
                                                num_sm_parts, static_cast<int32_t*>(metadata));
  else
    metadata_kernel<1024><<<1, 1024, 0, stream>>>(cache_seqlens, batch, s_q, causal ? 1 : 0, topk,
                                                  num_sm_parts, static_cast<int32_t*>(metadata));
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MLA_OK : record_cuda_error("metadata kernel launch", e);
}

extern "C" int mla_get_metadata_host(const int32_t* seqlens, int batch, int s_q, int causal,
                                     int topk, int num_sm_parts, void* metadata_host) {
  const int rc = check_meta_args(seqlens, batch, s_q, topk, num_sm_parts, metadata_host);
  if (rc != MLA_OK) return rc;
  int32_t* meta = static_cast<int32_t*>(metadata_host);
  const int n_seq = batch * s_q;
  const int groups = schedule_groups(s_q, num_sm_parts);
  const int n_g = n_seq / groups, parts_g = num_sm_parts / groups;
  // cost prefixes within each group, sequences in group-major order k
  std::vector<int64_t> group_total(groups, 0);
  int32_t max_cost = 0;
  for (int k = 0; k < n_seq; ++k) {
    const int q = order_to_q(k, n_g, groups), j = k / n_g;
    const int32_t keys = seq_keys(seqlens, q / s_q, q % s_q, s_q, causal ? 1 : 0, topk);
    const int32_t nt = tiles_of(keys);
    int32_t* s = meta_seq(meta, num_sm_parts, q);
    s[kSTiles] = nt; s[kSKeys] = keys; s[5] = 0; s[6] = 0; s[7] = 0;
    s[kSCostPrefix] = static_cast<int32_t>(group_total[j]);
    group_total[j] += cost_of(nt);
    if (cost_of(nt) > max_cost) max_cost = cost_of(nt);
  }
  int64_t max_group_total = 0;
  for (int j = 0; j < groups; ++j) max_group_total = std::max(max_group_total, group_total[j]);
  const int64_t per_part = max_group_total > 0 ? floordiv(max_group_total + parts_g - 1, parts_g) : 1;
  int64_t splits = 0;
  for (int k = 0; k < n_seq; ++k) {
    int32_t* s = meta_seq(meta, num_sm_parts, order_to_q(k, n_g, groups));
    const int32_t nt = s[kSTiles];
    s[kSNSplits] = nt > 0 ? 1 + inner_boundaries(s[kSCostPrefix], nt, per_part) : 0;
    s[kSSplitOff] = static_cast<int32_t>(splits);
    splits += s[kSNSplits];
  }
  for (int p = 0; p < num_sm_parts; ++p) {
    const int j = p / parts_g;
    fill_part(meta, GroupPrefix<MetaPrefix>{MetaPrefix{meta, num_sm_parts}, j, groups}, n_g, group_total[j],
              per_part, p, p % parts_g, j, groups);
  }
  meta[kHMagic] = kMetaMagic; meta[kHVersion] = kMetaVersion; meta[kHNSeq] = n_seq;
  meta[kHParts] = num_sm_parts; meta[kHTile] = kTileTokens; meta[kHSq] = s_q;
  meta[kHBatch] = batch; meta[kHCausal] = causal ? 1 : 0; meta[kHTopk] = topk;
  meta[kHTotalSplits] = static_cast<int32_t>(splits);
  meta[kHPerPart] = static_cast<int32_t>(per_part);
  meta[kHMaxCost] = max_cost;
  // schedule B (one whole sequence per part), when every sequence has a part
  const bool has_b = n_seq <= num_sm_parts;
  meta[kHHasB] = has_b ? 1 : 0;
  meta[kHGroups] = groups;
  for (int i = kHGroups + 1; i < kHeaderWords; ++i) meta[i] = 0;
  int32_t* mb = meta + meta_words(n_seq, num_sm_parts);
  for (int i = 0; i < kHeaderWords; ++i) mb[i] = has_b ? meta[i] : 0;
  if (has_b) {
    int64_t b_splits = 0;
    for (int k = 0; k < n_seq; ++k) {
      const int q = order_to_q(k, n_g, groups);
      const int32_t* sa = meta_seq(meta, num_sm_parts, q);
      int32_t* sb = meta_seq(mb, num_sm_parts, q);
      const int32_t nt = sa[kSTiles];
      sb[kSTiles] = nt; sb[kSSplitOff] = static_cast<int32_t>(b_splits); sb[kSNSplits] = nt > 0 ? 1 : 0;
      sb[kSKeys] = sa[kSKeys]; sb[kSCostPrefix] = sa[kSCostPrefix]; sb[5] = 0; sb[6] = 0; sb[7] = 0;
      b_splits += nt > 0 ? 1 : 0;
    }
    for (int p = 0; p < num_sm_parts; ++p) fill_whole_part(mb, num_sm_parts, n_seq, p);
    mb[kHTotalSplits] = static_cast<int32_t>(b_splits);
    mb[kHPerPart] = max_cost;
    mb[kHHasB] = 0;
    mb[kHGroups] = 1;
  }
  return MLA_OK;
}
