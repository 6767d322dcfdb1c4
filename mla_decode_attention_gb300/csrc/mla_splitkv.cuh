// Split-KV MLA decode kernel for sm_103a (tcgen05 MMA, TMEM accumulators,
// TMA-fed shared-memory ring, warp-specialised roles).
//
// One CTA owns 64 query rows (the heads of one block of one query token) and
// walks the (sequence, 128-key tile) range its schedule part assigns.  Per
// tile it computes, transposed so that key tokens sit on TMEM lanes:
//
//   S^T[128 tokens x 64 rows]  = K_tile[128 x 576] . Q^T          (QK^T, K = 576)
//   online softmax over tokens (column-wise, fp32, warp shuffles)
//   O^T[512 x 64 rows]        += V_tile^T[512 x 128] . P^T[128 x 64] (PV)
//
// with V_tile = the first 512 columns of the same shared-memory tile, so each
// 576-wide cached row is loaded once and feeds both products (FlashMLA deep
// dive, "Theoretical Analysis": K and V are the same latent row).  The TMEM
// accumulators hold O^T (4 x 64 columns) and S^T (64 columns); no output
// matrix lives in registers, which is why no seesaw schedule is needed here
// (the seesaw in the FlashMLA deep dive exists because WGMMA keeps O in
// registers).
//
// Roles (576 threads; 96 registers per thread: five warps share each of two
// SM sub-partitions):
//   warps 0..15    : four softmax warpgroups, query rows 16g .. 16g+15 each;
//                    FP8 cache: before each tile's scores they also convert
//                    the staged codes to bf16 in place (one 16-code unit per
//                    thread per chunk)
//   warp 16        : producer (lane 0; sparse: all lanes gather): TMA loads of
//                    Q (once per piece) and of each tile's 9 column chunks
//                    (two 64-token pages per chunk); FP8 cache: the raw codes
//                    and scales of the latent chunks (staged inside their
//                    slots) and the bf16 RoPE chunk, and with two head blocks
//                    the copy of every converted chunk into the peer CTA
//   warp 17        : TMEM allocation; lane 0 issues every MMA
//
// Shared memory (1024-byte aligned): 9 KV chunk slots of [128 tok x 64 col]
// bf16 (16 KB each, 128-byte swizzle), Q as 9 chunks of [64 rows x 64 col]
// (8 KB each).  Slot 8 (the RoPE columns) is dead after QK^T and holds P^T
// during PV.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstddef>

#include "mla_decode.h"
#include "mla_internal.h"
#include "mla_ptx.cuh"
#include "mla_schedule.cuh"

namespace mla {

constexpr int kRowsPerCta = 64;           // query rows per CTA = MMA N
constexpr int kChunks = 9;                // 576 / 64 columns
constexpr int kChunkBytes = kTileTokens * 64 * 2;   // 16 KB
constexpr int kQChunkBytes = kRowsPerCta * 64 * 2;  // 8 KB
constexpr int kSmemKv = 0;
constexpr int kSmemQ = kChunks * kChunkBytes;                 // 147456
constexpr int kSmemSmall = kSmemQ + kChunks * kQChunkBytes;   // 221184
constexpr int kNumBarriers = 3 * kChunks + 4;
constexpr int kSmallBytes = 8 * kNumBarriers + 16 + 5 * 4 * 4 * 4 * 16;
constexpr int kSmemBytes = kSmallBytes + kSmemSmall + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "dynamic shared memory per CTA");
constexpr int kSoftmaxGroups = 4;                  // warpgroups on the softmax
constexpr int kRowsPerGroup = kRowsPerCta / kSoftmaxGroups;  // 16 query rows each
constexpr int kSoftmaxWarp0 = 0;
constexpr int kProducerWarp = 4 * kSoftmaxGroups;
constexpr int kMmaWarp = kProducerWarp + 1;
constexpr int kThreads = 32 * (kMmaWarp + 1);
// A later tile moves the softmax reference only when a score exceeds it by
// more than this (log2 units): probabilities stay <= 2^8, exact in range.
constexpr float kRescaleLog2 = 8.f;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;     // O^T: 4 blocks of 64 columns
constexpr uint32_t kTmemS = 256;   // S^T: 64 columns
constexpr uint32_t kIdescQK = idesc_bf16(128, kRowsPerCta, false, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, kRowsPerCta, true, true);

enum class KvMode : int { kPagedBf16 = 0, kSparseBf16 = 1, kPagedFp8 = 2, kPagedFp8V41 = 3 };

// kPagedFp8: the 656-byte cache (fp32 scale per 128 latent codes, bf16 RoPE
// chunk); kPagedFp8V41: the 528-byte cache (FlashMLA README, "FP8 / FP4 KV
// Cache Format", V4.1): 512 e4m3 codes covering all 512 dimensions and 16
// e8m0 scales (one per 32 codes) at byte 512 of the token.  Keys and values
// are then 512 wide: QK^T runs over 8 chunks (no RoPE chunk) and P.V over
// the same 8 chunks.
__host__ __device__ constexpr bool is_fp8(KvMode m) {
  return m == KvMode::kPagedFp8 || m == KvMode::kPagedFp8V41;
}
__host__ __device__ constexpr int qk_chunks(KvMode m) { return m == KvMode::kPagedFp8V41 ? 8 : 9; }

// FP8 cache token: 512 e4m3 codes, 4 fp32 scales (one per 128 latent
// channels), 64 bf16 RoPE values (FlashMLA "Hopper FP8 sparse decode" note,
// "The FP8 KVCache Format").
constexpr int kFp8TokenBytes = 656;
constexpr int kFp8ScaleOffset = 512;
constexpr int kFp8RopeOffset = 528;
// V4.1 cache token (FlashMLA README, "FP8 / FP4 KV Cache Format"): 512 e4m3
// codes, then 16 e8m0 scales (one per 32 codes) at byte 512.
constexpr int kFp8V41TokenBytes = 528;
constexpr int kV41HeadDim = 512;
constexpr uint32_t kDequantBarrier = 5;  // FP8: all softmax warps (1..4: one softmax group each)
// staging of a latent chunk's raw FP8 data inside its own 16 KB bf16 slot
constexpr int kRawScaleOff = 4096;                  // [128 tokens][4 fp32 scales]
constexpr int kRawScaleBytes = kTileTokens * 16;
constexpr int kRawCodeOff = 8192;                   // [128 tokens][64 e4m3 codes]
constexpr int kRawCodeBytes = kTileTokens * 64;
static_assert(kRawScaleOff + kRawScaleBytes <= kRawCodeOff && kRawCodeOff + kRawCodeBytes <= kChunkBytes,
              "staging fits in the slot");

struct SplitParams {
  const int32_t* meta;     // schedule metadata (read-only)
  int32_t* ws_ctrl;        // workspace control words: [0] = the schedule walked (for the combine)
  const int32_t* block_table;
  int64_t bt_stride;       // dense: int32 entries per block-table row (page slots of a request)
  int64_t num_pages;       // dense: pages in the cache
  const int32_t* cache_seqlens;  // dense: [batch] lengths, checked against the metadata's key counts
  const int32_t* indices;  // sparse: [n_seq, topk]
  const float* attn_sink;  // sparse, optional: [h] sink logits (out scaled by e^lse / (e^lse + e^sink))
  int topk;
  int64_t s_kv;            // sparse: pool rows
  const __nv_bfloat16* kv_rows;  // dense: cache base (L2 prefetch); sparse: pool base
  const __nv_bfloat16* q;        // query rows, for L2 prefetch of the next piece
  const uint8_t* kv_fp8;         // FP8 cache base ([pages, 64, 656] bytes)
  float* ws_o;
  float* ws_lse;
  __nv_bfloat16* out;
  float* lse;
  uint32_t* err;
  int h;
  int d_qk;                // query / key width: 576, or 512 for the V4.1 cache
  int s_q;
  int batch;
  int causal;              // dense: causal flag of the call (checked against the metadata)
  int num_parts;
  int n_hblk;
  int rows;                // query rows loaded per CTA (min(h, 64))
  float scale_log2;        // softmax_scale * log2(e)
};

struct SmemSmall {
  // float arrays first: each row of 32 floats is read back as float4 vectors,
  // so every row must start on a 16-byte boundary.
  alignas(16) float red_max[kSoftmaxGroups][4][kRowsPerGroup];
  alignas(16) float red_sum[kSoftmaxGroups][4][kRowsPerGroup];
  alignas(16) float red_bsum[kSoftmaxGroups][4][kRowsPerGroup];
  alignas(16) float bcast[kSoftmaxGroups][4][kRowsPerGroup];
  alignas(16) float bcast2[kSoftmaxGroups][4][kRowsPerGroup];
  uint64_t full[kChunks];
  uint64_t empty[kChunks];
  uint64_t raw_full[kChunks - 1];  // FP8: raw codes and scales of a latent chunk landed
  uint64_t q_full, q_empty, s_full, p_full, o_done;
  uint32_t tmem_base;
  uint32_t abort;
};
static_assert(offsetof(SmemSmall, bcast) % 16 == 0 && offsetof(SmemSmall, bcast2) % 16 == 0,
              "broadcast rows are read as float4");
static_assert(offsetof(SmemSmall, full) % 8 == 0, "mbarriers are 8-byte objects");
static_assert(sizeof(SmemSmall) <= kSmallBytes, "small smem region");

// Reduce 32 per-thread values (one per query row of this warpgroup) over the
// warp's 32 lanes, leaving in lane l the reduction for row l.  Recursive
// halving: at each step a lane keeps the half of its vector that its lane bit
// selects and adds the partner's copy of that half.
template <bool kMax>
__device__ __forceinline__ float warp_reduce_scatter32(const float (&v)[32], int lane) {
  float a[16], b[8], c[4], d[2];
  bool hi = lane & 16;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float send = hi ? v[i] : v[i + 16];
    const float keep = hi ? v[i + 16] : v[i];
    const float r = __shfl_xor_sync(0xffffffffu, send, 16);
    a[i] = kMax ? fmaxf(keep, r) : keep + r;
  }
  hi = lane & 8;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float send = hi ? a[i] : a[i + 8];
    const float keep = hi ? a[i + 8] : a[i];
    const float r = __shfl_xor_sync(0xffffffffu, send, 8);
    b[i] = kMax ? fmaxf(keep, r) : keep + r;
  }
  hi = lane & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = hi ? b[i] : b[i + 4];
    const float keep = hi ? b[i + 4] : b[i];
    const float r = __shfl_xor_sync(0xffffffffu, send, 4);
    c[i] = kMax ? fmaxf(keep, r) : keep + r;
  }
  hi = lane & 2;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = hi ? c[i] : c[i + 2];
    const float keep = hi ? c[i + 2] : c[i];
    const float r = __shfl_xor_sync(0xffffffffu, send, 2);
    d[i] = kMax ? fmaxf(keep, r) : keep + r;
  }
  hi = lane & 1;
  const float send = hi ? d[0] : d[1];
  const float keep = hi ? d[1] : d[0];
  const float r = __shfl_xor_sync(0xffffffffu, send, 1);
  return kMax ? fmaxf(keep, r) : keep + r;
}

// Sum of 16 per-thread values (one per query row of the warpgroup) over the
// warp's 32 lanes; lanes l and l + 16 both end with the sum for row l & 15.
__device__ __forceinline__ float warp_sum_scatter16(const float (&v)[16], int lane) {
  float a[16], b[8], c[4], d[2];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = v[i] + __shfl_xor_sync(0xffffffffu, v[i], 16);
  bool hi = lane & 8;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float send = hi ? a[i] : a[i + 8];
    const float keep = hi ? a[i + 8] : a[i];
    b[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  hi = lane & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = hi ? b[i] : b[i + 4];
    const float keep = hi ? b[i + 4] : b[i];
    c[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  hi = lane & 2;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = hi ? c[i] : c[i + 2];
    const float keep = hi ? c[i + 2] : c[i];
    d[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  hi = lane & 1;
  const float send = hi ? d[0] : d[1];
  const float keep = hi ? d[1] : d[0];
  return keep + __shfl_xor_sync(0xffffffffu, send, 1);
}

__device__ __forceinline__ void load_bcast32(const float* src, float (&dst)[32]) {
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    const float4 t = *reinterpret_cast<const float4*>(src + i);
    dst[i] = t.x; dst[i + 1] = t.y; dst[i + 2] = t.z; dst[i + 3] = t.w;
  }
}

// Physical page of logical page `pg` of a sequence with `keys` keys whose
// block-table row is `bt_row`, or -1 when there is none: the entry is outside
// [0, num_pages), or the page slot lies past the row's bt_stride entries
// (more keys than the row can address).  Pages past the last one of the
// sequence (the second page of a tile's last 64-key half) map to the last.
__device__ __forceinline__ int32_t page_of(const SplitParams& p, const int32_t* bt_row, int32_t keys,
                                           int pg) {
  const int last = (keys - 1) / kPage;
  const int slot = pg < last ? pg : last;
  if (static_cast<int64_t>(slot) >= p.bt_stride) return -1;
  const int32_t blk = bt_row[slot];
  return (blk < 0 || static_cast<int64_t>(blk) >= p.num_pages) ? -1 : blk;
}

// Block-table row of sequence q (request q / s_q).
__device__ __forceinline__ const int32_t* bt_row_of(const SplitParams& p, int q) {
  return p.block_table + static_cast<int64_t>(q / p.s_q) * p.bt_stride;
}

// Dense: flags MLA_DEVERR_METADATA when the metadata's key count for sequence
// q differs from the one cache_seqlens and the causal flag give (metadata
// computed from other lengths).  The kernels keep walking the metadata's
// tiles; page_of keeps every block-table read inside its row.
__device__ __forceinline__ void check_seq_keys(const SplitParams& p, int q, int32_t keys) {
  if (!p.cache_seqlens) return;
  const int32_t want = seq_keys(p.cache_seqlens, q / p.s_q, q % p.s_q, p.s_q, p.causal, 0);
  if (want != keys && p.err) atomicOr(p.err, MLA_DEVERR_METADATA);
}

// Sparse: the first index among a query's n_slots index slots that names a
// pool row (warp-wide; every lane gets it), or 0 when there is none.
// Invalid slots are loaded from a row the query does name, so a masked slot
// (weight 0) never multiplies a row the caller did not ask for: 0 * NaN is
// NaN, and rows the query does not name may hold anything.
__device__ __forceinline__ int32_t first_valid_index(const int32_t* idx_row, int n_slots, int64_t s_kv,
                                                     int lane) {
  for (int base = 0; base < n_slots; base += 32) {
    const int slot = base + lane;
    const int32_t id = slot < n_slots ? idx_row[slot] : -1;
    const uint32_t m = __ballot_sync(0xffffffffu, id >= 0 && static_cast<int64_t>(id) < s_kv);
    if (m) return __shfl_sync(0xffffffffu, id, __ffs(m) - 1);
  }
  return 0;
}

// Sparse: the pool rows a warp loads for one 128-slot tile, lane L owning
// slots 4L .. 4L + 3 (id: the index list entries, -1 past the key count).
// Slots that name no row (-1, out of range) take the first row named in the
// tile, or, in a tile with none, the first row the query names (found by a
// scan of its list, `fallback`, computed once and cached in *fallback_cache,
// -2 = not yet known).  Out-of-range entries other than -1 set
// MLA_DEVERR_BAD_INDEX (when `flag`).
__device__ __forceinline__ void sparse_rows4(const SplitParams& p, const int32_t (&id)[4], int lane,
                                             const int32_t* idx_row, int n_slots, bool flag,
                                             int32_t* fallback_cache, int32_t (&y)[4]) {
  bool valid[4];
  int32_t first = -1;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    valid[i] = id[i] >= 0 && static_cast<int64_t>(id[i]) < p.s_kv;
    if (!valid[i] && id[i] != -1 && flag && p.err) atomicOr(p.err, MLA_DEVERR_BAD_INDEX);
    if (valid[i] && first < 0) first = id[i];
  }
  const uint32_t any = __ballot_sync(0xffffffffu, first >= 0);
  int32_t sub;
  if (any) {
    sub = __shfl_sync(0xffffffffu, first, __ffs(any) - 1);
  } else {
    if (*fallback_cache == -2) *fallback_cache = first_valid_index(idx_row, n_slots, p.s_kv, lane);
    sub = *fallback_cache;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) y[i] = valid[i] ? id[i] : sub;
}

// FP8 cache: 16 e4m3 codes of token dq_r (unit dq_u of a 64-code chunk) times
// their fp32 scale, rounded to bf16, into the chunk's 128-byte-swizzled row
// `row` (shared memory).  Kept out of line: inlined into the softmax loop it
// pushed that loop past the 96 registers a thread of this kernel may hold.
__device__ __noinline__ void convert_unit(uint32_t row, int dq_r, int dq_u, uint4 codes, float sc) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint32_t w0 = half ? codes.z : codes.x, w1 = half ? codes.w : codes.y;
    const float2 a0 = f16x2_to_f32x2(e4m3x2_to_f16x2(static_cast<uint16_t>(w0 & 0xFFFFu)));
    const float2 a1 = f16x2_to_f32x2(e4m3x2_to_f16x2(static_cast<uint16_t>(w0 >> 16)));
    const float2 a2 = f16x2_to_f32x2(e4m3x2_to_f16x2(static_cast<uint16_t>(w1 & 0xFFFFu)));
    const float2 a3 = f16x2_to_f32x2(e4m3x2_to_f16x2(static_cast<uint16_t>(w1 >> 16)));
    st_shared_v4(row + ((2 * dq_u + half) ^ (dq_r & 7)) * 16, pack_bf16x2(a0.x * sc, a0.y * sc),
                 pack_bf16x2(a1.x * sc, a1.y * sc), pack_bf16x2(a2.x * sc, a2.y * sc),
                 pack_bf16x2(a3.x * sc, a3.y * sc));
  }
}

template <KvMode kMode>
__global__ void __launch_bounds__(kThreads, 1)
    mla_splitkv_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_kv,
                       const __grid_constant__ CUtensorMap tm_codes,
                       const __grid_constant__ CUtensorMap tm_scales,
                       const __grid_constant__ SplitParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  SmemSmall* sm = reinterpret_cast<SmemSmall*>(smem + kSmemSmall);
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t kv_base = smem_base + kSmemKv;
  const uint32_t q_base = smem_base + kSmemQ;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int part = blockIdx.x / p.n_hblk;
  const int hb = blockIdx.x % p.n_hblk;
  // The metadata must describe this call; otherwise nothing is read or written.
  const bool meta_ok = meta_header_matches(p.meta, p.batch, p.s_q, p.num_parts, p.topk, p.causal);
  // Schedule B (whole sequences) only when nearly balanced: a tile of this
  // kernel takes ~3-6 us, so the ~26 us that splitting costs is ~4 tiles.
  constexpr int kSplitPenalty = 4;
  const int32_t* meta = meta_ok ? schedule_for(p.meta, kSplitPenalty) : p.meta;
  if (blockIdx.x == 0 && threadIdx.x == 32 * kSoftmaxWarp0) {  // a softmax thread: nothing to do yet
    // read by the combine after this grid: the schedule walked, or -1 when
    // the metadata was rejected (the combine then writes nothing), and
    // whether that schedule left anything to merge or fill
    p.ws_ctrl[1] = (meta_ok && (meta == p.meta || meta[kHTotalSplits] != meta[kHNSeq])) ? 1 : 0;
    p.ws_ctrl[0] = meta_ok ? (meta == p.meta ? 0 : 1) : -1;
    if (!meta_ok && p.err) atomicOr(p.err, MLA_DEVERR_METADATA);
  }

  // ---- setup: barriers, TMEM, zeroed padding rows of Q
  // FP8 with two head blocks: each CTA converts half of the latent chunks
  // (chunk c by head block c mod 2) and copies them into the peer's slots
  const bool share = is_fp8(kMode) && p.n_hblk == 2;
  constexpr int kQk = qk_chunks(kMode);  // key chunks of QK^T
  if (threadIdx.x == 0) {
    for (int c = 0; c < kChunks; ++c) {
      // FP8: a latent chunk is filled by this CTA's softmax warps (one
      // arrive each), or by one bulk copy from the peer (one local arm + bytes)
      const bool from_peer = share && c < kChunks - 1 && (c & 1) != hb;
      mbar_init(smem_u32(&sm->full[c]),
                (is_fp8(kMode) && c < kChunks - 1 && !from_peer) ? 4 * kSoftmaxGroups : 1);
      // a slot is free once the MMA threads of every CTA writing into it
      // have released it
      mbar_init(smem_u32(&sm->empty[c]), (share && c < kChunks - 1) ? 2 : 1);
    }
    for (int c = 0; c < kChunks - 1; ++c) mbar_init(smem_u32(&sm->raw_full[c]), 1);
    mbar_init(smem_u32(&sm->q_full), 1);
    mbar_init(smem_u32(&sm->q_empty), 1);
    mbar_init(smem_u32(&sm->s_full), 1);
    mbar_init(smem_u32(&sm->p_full), 4 * kSoftmaxGroups);  // one arrive per softmax warp
    mbar_init(smem_u32(&sm->o_done), 1);
    sm->abort = 0;
    fence_mbarrier_init();
    // the first tile's arm of every chunk the peer converts (the MMA thread
    // re-arms after each use)
    if (share)
      for (int c = hb ^ 1; c < kChunks - 1; c += 2) mbar_arrive_expect_tx(smem_u32(&sm->full[c]), kChunkBytes);
  }
  if (p.rows < kRowsPerCta) {
    // Rows [rows, 64) of every Q chunk are never written by TMA; zero them
    // once so the padded columns of S^T stay finite.
    const int pad_units = (kRowsPerCta - p.rows) * 8;
    for (int i = threadIdx.x; i < kChunks * pad_units; i += kThreads) {
      const int c = i / pad_units, k = i % pad_units;
      st_shared_v4(q_base + c * kQChunkBytes + p.rows * 128 + k * 16, 0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&sm->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kv);
    if (is_fp8(kMode)) {
      tma_prefetch_desc(&tm_codes);
      tma_prefetch_desc(&tm_scales);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (share) cluster_sync();  // peers' barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile uint32_t* abort_flag = &sm->abort;

  if (!meta_ok) {
    // nothing to do: every role is skipped, the teardown below still runs
  } else if (is_fp8(kMode) && warp == kProducerWarp) {
    // ===================================================== producer (FP8)
    // Lane 0 loads Q, the bf16 RoPE columns (chunk 8; 656-byte cache only) and, for every latent
    // chunk this CTA converts, the raw e4m3 codes and token scales by TMA into
    // that chunk's own slot (codes at +8 KB, scales at +4 KB), each as soon as
    // the slot is released; the softmax warps convert the slot in place.
    // With two head blocks, each converted slot then goes to the peer CTA's
    // slot by one bulk copy (the peer's MMA thread has armed its barrier).
    if (lane == 0) {
      const int own0 = share ? hb : 0, own_step = share ? 2 : 1;
      const int n_own = (kChunks - 1) / own_step;
      const int n_req = kMode == KvMode::kPagedFp8V41 ? n_own : n_own + 1;  // + the RoPE chunk
      PartCursor cur = walked_part_cursor(p.meta, meta, part);
      int q, t0, t1, split;
      uint32_t tile_ctr = 0, item_ctr = 0;
      bool ok = true;
      const uint64_t pol = l2_policy_evict_first();
      while (ok && next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
        ok = mbar_wait(smem_u32(&sm->q_empty), (item_ctr & 1) ^ 1, abort_flag, p.err);
        if (!ok) break;
        mbar_arrive_expect_tx(smem_u32(&sm->q_full), kQk * p.rows * 128);
        const int q_row = q * p.h + hb * kRowsPerCta;
        for (int c = 0; c < kQk; ++c)
          tma_load_2d(q_base + c * kQChunkBytes, &tm_q, c * 64, q_row, smem_u32(&sm->q_full),
                      l2_policy_evict_last());
        const int32_t keys = meta_seq(meta, p.num_parts, q)[kSKeys];
        const int32_t* bt_row = bt_row_of(p, q);
        check_seq_keys(p, q, keys);
        for (int t = t0; t < t1 && ok; ++t) {
          const uint32_t par = (tile_ctr & 1) ^ 1;
          int32_t blk[2];
          for (int h2 = 0; h2 < 2; ++h2) {
            blk[h2] = page_of(p, bt_row, keys, 2 * t + h2);
            if (blk[h2] < 0) {
              if (p.err) atomicOr(p.err, MLA_DEVERR_BAD_PAGE);
              blk[h2] = 0;  // read a valid page; the bad page's keys are wrong but finite
            }
          }
          // requests 0 .. n_own - 1: raw data of the owned latent chunks;
          // request n_own: the RoPE chunk (its slot also carries P until the
          // previous tile's P.V is done)
          int issued = 0;
          auto slot_of = [&](int i) { return i == n_own ? kChunks - 1 : own0 + own_step * i; };
          auto issue = [&](int i) {
            if (i == n_own) {
              const uint32_t bar = smem_u32(&sm->full[kChunks - 1]);
              mbar_arrive_expect_tx(bar, kChunkBytes);
              const uint32_t dst = kv_base + (kChunks - 1) * kChunkBytes;
              tma_load_2d(dst, &tm_kv, 0, blk[0] * kPage, bar, pol);
              tma_load_2d(dst + kChunkBytes / 2, &tm_kv, 0, blk[1] * kPage, bar, pol);
              return;
            }
            const int c = own0 + own_step * i;
            const uint32_t bar = smem_u32(&sm->raw_full[c]);
            const uint32_t slot = kv_base + c * kChunkBytes;
            mbar_arrive_expect_tx(bar, kRawCodeBytes + kRawScaleBytes);
            for (int h2 = 0; h2 < 2; ++h2) {
              tma_load_2d(slot + kRawCodeOff + h2 * (kRawCodeBytes / 2), &tm_codes, c * 64,
                          blk[h2] * kPage, bar, pol);
              tma_load_2d(slot + kRawScaleOff + h2 * (kRawScaleBytes / 2), &tm_scales, 0,
                          blk[h2] * kPage, bar);
            }
          };
          for (int k = 0; k < n_own && ok; ++k) {
            while (ok && issued <= k) {
              ok = mbar_wait(smem_u32(&sm->empty[slot_of(issued)]), par, abort_flag, p.err);
              if (ok) issue(issued++);
            }
            if (!share || !ok) continue;
            // chunk k converted: copy it to the peer; while waiting, make
            // every later request whose slot has been released
            const int c = own0 + own_step * k;
            const uint32_t fbar = smem_u32(&sm->full[c]);
            const uint64_t t_start = globaltimer_ns();
            while (ok && !mbar_try_wait_hint(fbar, tile_ctr & 1, 200)) {
              while (issued < n_req && mbar_test_wait(smem_u32(&sm->empty[slot_of(issued)]), par))
                issue(issued++);
              if (*abort_flag) {
                ok = false;
              } else if (globaltimer_ns() - t_start > kWaitTimeoutNs) {
                *abort_flag = 1u;
                if (p.err) atomicOr(p.err, MLA_DEVERR_TIMEOUT);
                ok = false;
              }
            }
            if (ok) {
              const uint32_t slot = kv_base + c * kChunkBytes;
              bulk_copy_to_peer(mapa_shared(slot, hb ^ 1), slot, kChunkBytes,
                                mapa_shared(fbar, hb ^ 1));
            }
          }
          while (ok && issued < n_req) {  // the RoPE chunk, if still due
            ok = mbar_wait(smem_u32(&sm->empty[slot_of(issued)]), par, abort_flag, p.err);
            if (ok) issue(issued++);
          }
          ++tile_ctr;
        }
        ++item_ctr;
      }
    }
  } else if (warp == kProducerWarp && kMode == KvMode::kSparseBf16) {
    // ===================================================== producer (gather)
    // Lane L gathers rows 4L..4L+3 of each 128-row tile with one tile::gather4
    // per column chunk; lane 0 owns the barriers.  Invalid slots (-1, out of
    // range, past topk) fetch pool row 0 and are masked by the softmax.
    PartCursor cur = walked_part_cursor(p.meta, meta, part);
    int q, t0, t1, split;
    uint32_t tile_ctr = 0, item_ctr = 0;
    int32_t issued[kChunks];  // tile counter of each slot's latest gather, -1 = none
    for (int c = 0; c < kChunks; ++c) issued[c] = -1;
    bool ok = true;
    while (ok && next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
      if (lane == 0) {
        ok = mbar_wait(smem_u32(&sm->q_empty), (item_ctr & 1) ^ 1, abort_flag, p.err);
        if (ok) {
          mbar_arrive_expect_tx(smem_u32(&sm->q_full), kChunks * p.rows * 128);
          const int q_row = q * p.h + hb * kRowsPerCta;
          for (int c = 0; c < kChunks; ++c)
            tma_load_2d(q_base + c * kQChunkBytes, &tm_q, c * 64, q_row, smem_u32(&sm->q_full),
                        l2_policy_evict_last());
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const int32_t* idx_row = p.indices + static_cast<int64_t>(q) * p.topk;
      const int32_t n_slots = meta_seq(meta, p.num_parts, q)[kSKeys];  // topk or topk_length
      int32_t fallback = -2;  // first row the query names, found when a tile names none
      for (int t = t0; t < t1 && ok; ++t) {
        int32_t id[4], rid[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int slot = t * kTileTokens + 4 * lane + i;
          id[i] = slot < n_slots ? idx_row[slot] : -1;
        }
        sparse_rows4(p, id, lane, idx_row, n_slots, true, &fallback, rid);
        const uint32_t par = (tile_ctr & 1) ^ 1;
        for (int c = 0; c < kChunks; ++c) {
          if (lane == 0) {
            ok = mbar_wait(smem_u32(&sm->empty[c]), par, abort_flag, p.err);
            if (ok) mbar_arrive_expect_tx(smem_u32(&sm->full[c]), kChunkBytes);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          tma_gather4(kv_base + c * kChunkBytes + 4 * lane * 128, &tm_kv, c * 64, rid[0], rid[1],
                      rid[2], rid[3], smem_u32(&sm->full[c]));
          issued[c] = static_cast<int32_t>(tile_ctr);
        }
        ++tile_ctr;
      }
      ++item_ctr;
    }
    if (!ok && lane == 0) {
      // Let gathers already in flight land before the CTA exits.
      for (int c = 0; c < kChunks; ++c) {
        if (issued[c] < 0) continue;
        const uint64_t t_start = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&sm->full[c]), static_cast<uint32_t>(issued[c]) & 1u) &&
               globaltimer_ns() - t_start < 1000000ull) {
        }
      }
    }
  } else if (warp == kProducerWarp) {
    // ===================================================== producer (TMA)
    if (lane == 0) {
      const uint64_t pol_kv = l2_policy_evict_first();
      const uint64_t pol_q = l2_policy_evict_last();
      PartCursor cur = walked_part_cursor(p.meta, meta, part);
      int q, t0, t1, split;
      uint32_t tile_ctr = 0, item_ctr = 0;
      int32_t issued[kChunks];  // tile counter of each slot's latest load, -1 = none
      for (int c = 0; c < kChunks; ++c) issued[c] = -1;
      bool ok = true;
      while (ok && next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
        // Q rows of this block: 9 boxes of [rows x 64 columns]
        ok = mbar_wait(smem_u32(&sm->q_empty), (item_ctr & 1) ^ 1, abort_flag, p.err);
        if (!ok) break;
        mbar_arrive_expect_tx(smem_u32(&sm->q_full), kChunks * p.rows * 128);
        const int q_row = q * p.h + hb * kRowsPerCta;
        for (int c = 0; c < kChunks; ++c)
          tma_load_2d(q_base + c * kQChunkBytes, &tm_q, c * 64, q_row, smem_u32(&sm->q_full), pol_q);
        {  // the next piece's query rows into L2
          PartCursor nc = cur;
          int nq, nt0, nt1, ns;
          if (next_piece(meta, p.num_parts, &nc, &nq, &nt0, &nt1, &ns))
            prefetch_l2(p.q + (static_cast<int64_t>(nq) * p.h + hb * kRowsPerCta) * p.d_qk,
                        p.rows * p.d_qk * 2);
        }
        const int32_t keys = meta_seq(meta, p.num_parts, q)[kSKeys];
        const int32_t* bt_row = bt_row_of(p, q);
        check_seq_keys(p, q, keys);
        for (int t = t0; t < t1 && ok; ++t) {
          int32_t y[2];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            int32_t blk = page_of(p, bt_row, keys, 2 * t + h2);
            if (blk < 0) {
              if (p.err) atomicOr(p.err, MLA_DEVERR_BAD_PAGE);
              blk = static_cast<int32_t>(p.num_pages);  // out of range: TMA fills zeros
            }
            y[h2] = blk * kPage;
          }
          const uint32_t par = (tile_ctr & 1) ^ 1;
          for (int c = 0; c < kChunks; ++c) {
            ok = mbar_wait(smem_u32(&sm->empty[c]), par, abort_flag, p.err);
            if (!ok) break;
            const uint32_t bar = smem_u32(&sm->full[c]);
            mbar_arrive_expect_tx(bar, kChunkBytes);
            const uint32_t dst = kv_base + c * kChunkBytes;
            tma_load_2d(dst, &tm_kv, c * 64, y[0], bar, pol_kv);
            tma_load_2d(dst + kChunkBytes / 2, &tm_kv, c * 64, y[1], bar, pol_kv);
            issued[c] = static_cast<int32_t>(tile_ctr);
          }
          ++tile_ctr;
        }
        ++item_ctr;
      }
      if (!ok) {
        // Let copies already in flight land before the CTA exits.
        for (int c = 0; c < kChunks; ++c) {
          if (issued[c] < 0) continue;
          const uint64_t t_start = globaltimer_ns();
          while (!mbar_try_wait(smem_u32(&sm->full[c]), static_cast<uint32_t>(issued[c]) & 1u) &&
                 globaltimer_ns() - t_start < 1000000ull) {
          }
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ===================================================== MMA issuer
    if (lane == 0) {
      PartCursor cur = walked_part_cursor(p.meta, meta, part);
      int q, t0, t1, split;
      uint32_t tile_ctr = 0, item_ctr = 0;
      bool ok = true;
      const uint32_t p_base = kv_base + 8 * kChunkBytes;
      while (ok && next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
        ok = mbar_wait(smem_u32(&sm->q_full), item_ctr & 1, abort_flag, p.err);
        if (!ok) break;
        for (int t = t0; t < t1 && ok; ++t) {
          const uint32_t par = tile_ctr & 1;
          // S^T = K_tile . Q^T: A = tile chunk (K-major), B = Q chunk (K-major)
          for (int c = 0; c < kQk; ++c) {
            // FP8 chunks converted by the peer complete on its bulk copy
            const bool from_peer = share && c < kChunks - 1 && (c & 1) != hb;
            ok = from_peer ? mbar_wait_cluster(smem_u32(&sm->full[c]), par, abort_flag, p.err)
                           : mbar_wait(smem_u32(&sm->full[c]), par, abort_flag, p.err);
            if (!ok) break;
            // next tile's arm: this phase is complete, so the arrive counts
            // toward the next one, before the peer can start its copy
            if (from_peer) mbar_arrive_expect_tx(smem_u32(&sm->full[c]), kChunkBytes);
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t a = sw128_desc(kv_base + c * kChunkBytes + 32 * k, 16, 1024);
              const uint64_t bq = sw128_desc(q_base + c * kQChunkBytes + 32 * k, 16, 1024);
              mma_bf16_ss(tmem + kTmemS, a, bq, kIdescQK, (c | k) != 0);
            }
          }
          if (!ok) break;
          if (t == t1 - 1) mma_commit(smem_u32(&sm->q_empty));
          mma_commit(smem_u32(&sm->s_full));
          // O^T += V^T . P^T: A = tile chunks 2m, 2m+1 read MN-major (the 64
          // latent columns of a chunk are contiguous), B = P^T in slot 8
          // (MN-major: the 64 rows of a token are contiguous)
          ok = mbar_wait(smem_u32(&sm->p_full), par, abort_flag, p.err);
          if (!ok) break;
          tc_fence_after();
          for (int m = 0; m < 4; ++m) {
#pragma unroll
            for (int s = 0; s < 8; ++s) {
              const uint64_t a = sw128_desc(kv_base + 2 * m * kChunkBytes + 2048 * s, kChunkBytes, 1024);
              const uint64_t bp = sw128_desc(p_base + 2048 * s, kChunkBytes, 1024);
              mma_bf16_ss(tmem + kTmemO + 64 * m, a, bp, kIdescPV, (t != t0 || s != 0) ? 1u : 0u);
            }
            if (share) {  // the slot is written by both CTAs' converters
              mma_commit_multicast(smem_u32(&sm->empty[2 * m]), 0x3);
              mma_commit_multicast(smem_u32(&sm->empty[2 * m + 1]), 0x3);
            } else {
              mma_commit(smem_u32(&sm->empty[2 * m]));
              mma_commit(smem_u32(&sm->empty[2 * m + 1]));
            }
          }
          mma_commit(smem_u32(&sm->empty[8]));
          if (t == t1 - 1) mma_commit(smem_u32(&sm->o_done));
          ++tile_ctr;
        }
        ++item_ctr;
      }
    }
  } else if (warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + 4 * kSoftmaxGroups) {
    // ===================================================== softmax / epilogue
    // Thread = one token row r of the tile (TMEM lane) x the 16 query rows of
    // its warpgroup (TMEM columns).  Probabilities are taken against a per-row
    // reference max m (log2 units).  The first tile of a piece sets m to the
    // exact column max.  A later tile keeps m unless one of its scores exceeds
    // the smallest reference by more than kRescaleLog2 (one warp max and one
    // barrier vote decide); then every row's m moves to its exact running max
    // and O^T and the sums are rescaled.  Two running sums per row: of the
    // fp32 probabilities (for the LSE) and of their bf16 roundings, i.e. the
    // weights the PV MMA multiplies (to normalise O), so a stale reference
    // leaves no coherent gain error on the output (flash-attention sparse-MLA
    // article: summing the bf16-rounded p brings the row gain to the noise
    // floor).  Each tile's 16 x 32 per-lane values are reduce-scattered over
    // the warp, so lane l keeps only the running sums of row l & 15 over the
    // warp's tokens; the four warps' sums meet in shared memory at the end.
    constexpr int R = kRowsPerGroup;
    const int g = (warp - kSoftmaxWarp0) >> 2;  // rows R*g .. R*g + R-1
    const int wq = warp & 3;                    // TMEM lane quarter
    const int r = wq * 32 + lane;               // token row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off + kTmemS + R * g;
    const uint32_t t_o = tmem + lane_off + kTmemO + R * g;
    const uint32_t p_slot = kv_base + 8 * kChunkBytes;
    const uint32_t bar_id = 1 + g;
    const int dq_r = (threadIdx.x - 32 * kSoftmaxWarp0) >> 2;  // FP8 conversion: token
    const int dq_u = threadIdx.x & 3;                           // and 16-code unit
    const float NEG_INF = -INFINITY;
    float* red_w = &sm->red_max[g][wq][0];
    float* bc_m = &sm->bcast[g][wq][0];
    float* bc_a = &sm->bcast2[g][wq][0];
    PartCursor cur = walked_part_cursor(p.meta, meta, part);
    int q, t0, t1, split;
    uint32_t tile_ctr = 0, item_ctr = 0;
    bool ok = true;
    while (ok && next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
      const int32_t* srec = meta_seq(meta, p.num_parts, q);
      const int32_t keys = srec[kSKeys];
      const int32_t* idx_row = (kMode == KvMode::kSparseBf16)
                                   ? p.indices + static_cast<int64_t>(q) * p.topk : nullptr;
      float m_true = NEG_INF;  // running max of row R*g + (lane & 15) (-inf: no key yet)
      float m_use = 0.f;       // reference the probabilities are taken against
      float m_low = NEG_INF;   // smallest m_true over the warpgroup's rows
      float lsum = 0.f;        // sum p of row R*g + (lane & 15) over this warp's tokens
      float bsum = 0.f;        // sum bf16(p) of the same row
      for (int t = t0; t < t1; ++t) {
        if constexpr (is_fp8(kMode)) {
          // ---- FP8: convert this tile's owned latent chunks in place.  Thread
          // = (token dq_r, 16-code unit dq_u); reads of the staging finish at
          // the named barrier before any bf16 write lands on it.  Every exit
          // is decided at a barrier, so all 16 warps leave together.
          const int own0 = share ? hb : 0, own_step = share ? 2 : 1;
#pragma unroll 1
          for (int c = own0; c < kChunks - 1; c += own_step) {
            if (lane == 0 && ok) ok = mbar_wait(smem_u32(&sm->raw_full[c]), tile_ctr & 1, abort_flag, p.err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            const uint32_t slot = kv_base + c * kChunkBytes;
            const uint4 codes = ld_shared_v4(slot + kRawCodeOff + dq_r * 64 + dq_u * 16);
            // the unit's scale: fp32 per 128 codes (656-byte cache), or e8m0
            // per 32 codes, 2^(byte - 127) (528-byte cache)
            const float sc = kMode == KvMode::kPagedFp8V41
                                 ? e8m0_to_f32(ld_shared_u8(slot + kRawScaleOff + dq_r * 16 + 2 * c + (dq_u >> 1)))
                                 : ld_shared_f32(slot + kRawScaleOff + dq_r * 16 + (c >> 1) * 4);
            ok = !named_barrier_or(kDequantBarrier, 128 * kSoftmaxGroups, !ok);
            if (!ok) break;
            convert_unit(slot + dq_r * 128, dq_r, dq_u, codes, sc);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm->full[c]));
          }
          if (!ok) break;
        }
        ok = mbar_wait(smem_u32(&sm->s_full), tile_ctr & 1, abort_flag, p.err);
        if constexpr (is_fp8(kMode))  // leave together (the barrier above)
          ok = !named_barrier_or(kDequantBarrier, 128 * kSoftmaxGroups, !ok);
        if (!ok) break;
        tc_fence_after();
        float x[R];
        tmem_ld16(t_s, x);
        tmem_wait_ld();
        const int tok = t * kTileTokens + r;
        bool valid = tok < keys;
        if (kMode == KvMode::kSparseBf16 && valid) {
          const int32_t id = idx_row[tok];
          valid = id >= 0 && static_cast<int64_t>(id) < p.s_kv;
        }
        // masked keys: -inf by selection, so a non-finite score of a masked
        // row cannot leak into the max or the sums
#pragma unroll
        for (int i = 0; i < R; ++i) x[i] = valid ? x[i] * p.scale_log2 : NEG_INF;
        bool full = true;
        if (t != t0) {
          float u = x[0];
#pragma unroll
          for (int i = 1; i < R; ++i) u = fmaxf(u, x[i]);
          u = warp_max_f32(u);
          full = named_barrier_or(bar_id, 128, u > m_low + kRescaleLog2);
        }
        if (full) {
          // exact column max of this tile over the 128 tokens
#pragma unroll
          for (int i = 0; i < R; i += 4) {
            const float w0 = warp_max_f32(x[i]), w1 = warp_max_f32(x[i + 1]);
            const float w2 = warp_max_f32(x[i + 2]), w3 = warp_max_f32(x[i + 3]);
            if (lane == 0) *reinterpret_cast<float4*>(red_w + i) = make_float4(w0, w1, w2, w3);
          }
          named_barrier_sync(bar_id, 128);
          const int row = lane & (R - 1);
          const float mt = fmaxf(fmaxf(sm->red_max[g][0][row], sm->red_max[g][1][row]),
                                 fmaxf(sm->red_max[g][2][row], sm->red_max[g][3][row]));
          const float m_new = fmaxf(m_true, mt);
          const float m_use_new = (m_new == NEG_INF) ? 0.f : m_new;
          const float alpha = (t == t0) ? 1.f : fast_exp2(m_use - m_use_new);
          m_true = m_new;
          m_use = m_use_new;
          m_low = warp_min_f32(m_true);
          if (lane < R) {
            bc_m[lane] = m_use;
            bc_a[lane] = alpha;
          }
          __syncwarp();
          if (t != t0 && __any_sync(0xffffffffu, alpha != 1.f)) {
            lsum *= alpha;  // this lane's row is row = lane & 15, whose factor is alpha
            bsum *= alpha;
            // PV of the previous tile completed before s_full of this tile
            // fired (one thread's tcgen05 operations complete in order)
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
              float o[R];
              tmem_ld16(t_o + 64 * m, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < R; i += 4) {
                const float4 a4 = *reinterpret_cast<const float4*>(bc_a + i);
                o[i] *= a4.x; o[i + 1] *= a4.y; o[i + 2] *= a4.z; o[i + 3] *= a4.w;
              }
              tmem_st16(t_o + 64 * m, o);
            }
            tmem_wait_st();
          }
        }
        // probabilities against the reference; P^T row r, rows R*g .. R*g+R-1
        // -> 16-byte units 2g, 2g+1 (swizzled)
        const uint32_t prow = p_slot + r * 128;
        float tp[R], tb[R];  // this tile's p and bf16(p) of the lane's token, per row
#pragma unroll
        for (int cu = 0; cu < 2; ++cu) {
          const float4 m0 = *reinterpret_cast<const float4*>(bc_m + 8 * cu);
          const float4 m1 = *reinterpret_cast<const float4*>(bc_m + 8 * cu + 4);
          float e[8];
          e[0] = fast_exp2(x[8 * cu + 0] - m0.x); e[1] = fast_exp2(x[8 * cu + 1] - m0.y);
          e[2] = fast_exp2(x[8 * cu + 2] - m0.z); e[3] = fast_exp2(x[8 * cu + 3] - m0.w);
          e[4] = fast_exp2(x[8 * cu + 4] - m1.x); e[5] = fast_exp2(x[8 * cu + 5] - m1.y);
          e[6] = fast_exp2(x[8 * cu + 6] - m1.z); e[7] = fast_exp2(x[8 * cu + 7] - m1.w);
          uint32_t pk[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            pk[k] = pack_bf16x2(e[2 * k], e[2 * k + 1]);
            tp[8 * cu + 2 * k] = e[2 * k];
            tp[8 * cu + 2 * k + 1] = e[2 * k + 1];
            tb[8 * cu + 2 * k] = __uint_as_float(pk[k] << 16);
            tb[8 * cu + 2 * k + 1] = __uint_as_float(pk[k] & 0xFFFF0000u);
          }
          const uint32_t unit = static_cast<uint32_t>((2 * g + cu) ^ (r & 7));
          st_shared_v4(prow + unit * 16, pk[0], pk[1], pk[2], pk[3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm->p_full));
        lsum += warp_sum_scatter16(tp, lane);  // row lane & 15, this warp's 32 tokens
        bsum += warp_sum_scatter16(tb, lane);
        ++tile_ctr;
      }
      if (!ok) break;
      // ---- epilogue: O^T / sum bf16(p) -> out (one split) or fp32 partial
      const int row = lane & (R - 1);
      if (lane < R) {
        sm->red_sum[g][wq][lane] = lsum;
        sm->red_bsum[g][wq][lane] = bsum;
      }
      named_barrier_sync(bar_id, 128);
      lsum = (sm->red_sum[g][0][row] + sm->red_sum[g][1][row]) +
             (sm->red_sum[g][2][row] + sm->red_sum[g][3][row]);
      bsum = (sm->red_bsum[g][0][row] + sm->red_bsum[g][1][row]) +
             (sm->red_bsum[g][2][row] + sm->red_bsum[g][3][row]);
      ok = mbar_wait(smem_u32(&sm->o_done), item_ctr & 1, abort_flag, p.err);
      if constexpr (is_fp8(kMode))  // the next piece starts at a shared barrier
        ok = !named_barrier_or(kDequantBarrier, 128 * kSoftmaxGroups, !ok);
      if (!ok) break;
      tc_fence_after();
      const bool has = lsum > 0.f && bsum > 0.f;
      const bool final_out = srec[kSNSplits] == 1;
      float inv_l = has ? 1.f / bsum : 0.f;
      const float lse_v = has ? (m_use + __log2f(lsum)) * 0.69314718055994531f : NEG_INF;
      // attention sink: applied here to a final row, by the combine to a split row
      if (p.attn_sink && final_out && hb * kRowsPerCta + R * g + row < p.h)
        inv_l *= attn_sink_factor(lse_v, p.attn_sink[hb * kRowsPerCta + R * g + row]);
      if (lane < R) bc_a[lane] = inv_l;
      __syncwarp();
      const volatile float* il = bc_a;  // 1 / sum of row i, read per store (broadcast)
      const int row0 = hb * kRowsPerCta + R * g;  // first head of this warpgroup
      const int split_row = srec[kSSplitOff] + split;
      const int b = q / p.s_q, j = q % p.s_q;
      // h is a multiple of 16, so a warpgroup's 16 rows are all heads or all padding
      if (row0 < p.h) {
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
          float o[R];  // O^T rows d of block m, columns = this warpgroup's 16 query rows
          tmem_ld16(t_o + 64 * m, o);
          tmem_wait_ld();
          const int d = 128 * m + 32 * wq + lane;
          // a row without keys (il = 0) is written as exact zeros: its O may
          // hold products of zero weights with rows nobody named
          if (final_out) {
            __nv_bfloat16* dst = p.out + (static_cast<int64_t>(q) * p.h + row0) * kDv + d;
#pragma unroll
            for (int i = 0; i < R; ++i) {
              const float f = il[i];
              dst[i * kDv] = __float2bfloat16_rn(f != 0.f ? o[i] * f : 0.f);
            }
          } else {
            float* dst = p.ws_o + (static_cast<int64_t>(split_row) * p.h + row0) * kDv + d;
#pragma unroll
            for (int i = 0; i < R; ++i) {
              const float f = il[i];
              dst[i * kDv] = f != 0.f ? o[i] * f : 0.f;
            }
          }
        }
      }
      if (wq == 0 && lane < R && row0 + lane < p.h) {
        if (final_out)
          p.lse[(static_cast<int64_t>(b) * p.h + row0 + lane) * p.s_q + j] = lse_v;
        else
          p.ws_lse[static_cast<int64_t>(split_row) * p.h + row0 + lane] = lse_v;
      }
      ++item_ctr;
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (share) cluster_sync();  // no peer still writes into this CTA's smem
  pdl_launch_dependents();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace mla
