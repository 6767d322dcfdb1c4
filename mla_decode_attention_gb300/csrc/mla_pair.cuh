// Paired-CTA MLA decode kernel for 128 query rows per query token (sm_103a).
//
// A cluster of two CTAs on two SMs shares one schedule part.  Per 128-key tile:
//
//   score CTA (rank 0):  S[128 rows x 128 tokens] = Q[128 x 576] . K_tile^T
//                        (tcgen05, A = Q resident in TMEM, B = K tile in smem,
//                        N = 128), then the online softmax with one thread per
//                        query row; P (bf16) and the per-row rescale factors go
//                        to the output CTA by a shared-memory bulk copy.
//   output CTA (rank 1): O[128 rows x 512] += P[128 x 128] . V_tile[128 x 512]
//                        (tcgen05, both operands in smem, N = 128 per d quarter),
//                        O in TMEM (all 512 columns); it writes the output rows.
//
// Both CTAs read the same cached rows (the score CTA all 576 columns, the
// output CTA the first 512: V is the latent part of the same row, FlashMLA
// deep dive, "Theoretical Analysis").  Splitting the two products over two SMs
// lets each issue MMAs of 128 x 128 x 16 (full tensor rate) and keeps keys
// loading while the previous tile is multiplied.  Score CTA TMEM: Q's 512
// latent columns (256 columns of bf16 pairs) and two S buffers, so QK of tile
// t + 1 runs while the softmax still reads tile t; Q's 64 RoPE columns sit in
// shared memory and enter QK through one smem-smem MMA chunk.  The softmax
// makes two passes over S in TMEM (row max, then probabilities), 32 columns
// at a time, so its code stays small.
//
// Paged cache: each group of K chunks (3g .. 3g + 2) and each half of V
// (chunks 0..3, 4..7) arrives as one 4-D box per page that lands as
// [8-token group][chunk][8 tokens][128 bytes]: a TMA box costs its SM a fixed
// time besides its bytes, so a [64 x 64] box per chunk and page moves about
// half as many bytes per SM-second.  In such a region chunk c of all 128
// tokens is a swizzled K-major operand whose 8-token groups lie 3 KB (V: 4 KB)
// apart, the second page's groups right after the first's, so QK stays one
// N = 128 product per chunk, and V read MN-major gives N = 256 products.
// Sparse keys are gathered four rows at a time into [128 tokens x 64 columns]
// chunks instead.
//
// Roles (paged cache: 256 threads per CTA, two warps per SM sub-partition, up
// to 224 registers each; gathered keys: 512 threads, 128 registers):
//   warp 0 lane 0        : paged: TMA issuer (K groups / V halves, one box per page)
//   warps 0, 2, 3, 8..13 : gathered: tile::gather4 issuers, one chunk of a tile
//                          each (score CTA: 9 chunks, output CTA: 8)
//   warp 1               : TMEM owner; lane 0 issues every MMA
//   warp 3               : paged score CTA: issues the P bulk copies (named
//                          barriers 1, 2 with warps 4..7 around the staging
//                          buffer); paged output CTA: hands P buffers back
//   warps 4..7           : row threads, thread r = query row r = TMEM lane r
//
// Waits are bounded (mbar_wait*); after an abort every role keeps walking its
// schedule without waiting, so the named barriers between warps 4..8 stay
// matched and every thread reaches the final cluster barrier.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstddef>

#include "mla_decode.h"
#include "mla_internal.h"
#include "mla_ptx.cuh"
#include "mla_schedule.cuh"
#include "mla_splitkv.cuh"

namespace mla {
namespace pair {

constexpr int kThreads = 256;                      // paged cache
// Gathered keys: one tile::gather4 costs its issuing warp ~84 clk (a warp's
// gathers go out one at a time), so the sparse kernel runs 16 warps (128
// registers each) and spreads the gathers of a tile over 9 warps in the score
// CTA (one chunk each) and 8 in the output CTA.
constexpr int kThreadsSparse = 512;
constexpr int kKIssuersSparse = 9;
constexpr int kVIssuersSparse = 8;
constexpr int kRows = 128;                         // query rows per cluster = TMEM lanes
constexpr int kChunk = kTileTokens * 64 * 2;       // 16 KB: [128 tokens x 64 columns] bf16
// score CTA
constexpr int kKGroups = 3;                        // K ring: 3 groups of 3 chunks
constexpr int kKGroupBytes = 3 * kChunk;           // 48 KB
constexpr int kQRope = kKGroups * kKGroupBytes;    // 147456: Q RoPE columns [128 x 64] bf16
constexpr int kStage = kQRope + kChunk;            // 163840: P staging
constexpr int kPBytes = kRows * kTileTokens * 2;   // 32768: P[128 rows x 128 tokens] bf16
constexpr int kSideAlpha = kPBytes;                // float alpha[128]
constexpr int kSideInvL = kPBytes + 512;           // float inv_l[128] (last tile of a piece)
constexpr int kSideFlags = kPBytes + 1024;         // uint32 per row warp: any alpha != 1
constexpr int kXferBytes = kPBytes + 1040;         // 33808 bytes per tile
// output CTA
constexpr int kVGroups = 4;                        // V ring: 128-wide d quarters
constexpr int kVGroupBytes = 2 * kChunk;           // 32 KB
constexpr int kPBuf0 = kVGroups * kVGroupBytes;    // 131072
constexpr int kPBufStride = 34816;                 // kXferBytes rounded up to 1 KB
constexpr int kBarOffset = kPBuf0 + 2 * kPBufStride;  // 200704 (score CTA ends at 197648)
constexpr int kEpi = kBarOffset + 1024;            // output CTA: 4 KB per row warp for the epilogue
// TMEM columns
constexpr uint32_t kQCol = 0;                      // score CTA: Q latent part, 256 columns
constexpr uint32_t kSCol = 256;                    // score CTA: S buffers at 256 and 384
constexpr uint32_t kIdescS = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescO = idesc_bf16(128, 128, false, true);
constexpr uint32_t kIdescO256 = idesc_bf16(128, 256, false, true);
// paged: one page's part of a K group ([8 groups][3 chunks][1 KB]) and of a V
// half ([8 groups][4 chunks][1 KB])
constexpr int kGroupPage = 3 * kPage * 128;        // 24 KB
constexpr int kHalfPage = 4 * kPage * 128;         // 32 KB
static_assert(2 * kGroupPage == kKGroupBytes && 4 * kHalfPage == kVGroups * kVGroupBytes, "paged regions");
constexpr uint32_t kRowThreads = 128;              // warps 4..7
// Softmax: one pass over S per tile after a piece's first; the row max is
// taken only when a tile's probabilities sum to more than this (2^kRescaleLog2).
constexpr float kMoveSum = 256.f;
static_assert(kMoveSum == 256.f && kRescaleLog2 == 8.f, "kMoveSum = 2^kRescaleLog2");
constexpr uint32_t kXferNamedThreads = 160;        // dense: warps 3..7

struct Bars {
  uint64_t kfull[kKGroups], kempty[kKGroups];      // score CTA K ring
  uint64_t vfull[kVGroups], vempty[kVGroups];      // output CTA V ring
  uint64_t s_full[2], s_free[2];                   // score CTA
  uint64_t q_tma;                                  // score CTA: a later piece's Q by TMA
  uint64_t q_box[4];                               // score CTA: the first piece's Q boxes in the K ring
  uint64_t q_stage_free, q_cp;                     // score CTA: later pieces' Q through the P staging buffer
  uint64_t p_free[2];                              // score CTA, arrived by the output CTA
  uint64_t p_full[2];                              // output CTA, completed by bulk copies
  uint64_t pv_done[2], o_full, o_free, o_drained, o_rescaled;  // output CTA
  uint64_t side_read[2];                           // output CTA: row threads read P's side data
  uint32_t tmem_base;
  uint32_t abort;
};
constexpr int kSmemBytes = kEpi + 4 * 4096 + 1024;
// The part's first query rows arrive by TMA: the latent columns as [8 chunks]
// [128 rows][128 B] in the (still empty) K ring, the RoPE columns in kQRope.
constexpr int kQLatentBytes = 8 * kRows * 128;     // 128 KB
constexpr int kQBoxBytes = 2 * kRows * 128;        // 32 KB: one query box, two chunks
static_assert(kQBoxBytes <= kXferBytes, "a query box fits the P staging buffer");
static_assert(kQLatentBytes <= kQRope, "Q staging in the K ring");
static_assert(kBarOffset % 16 == 0, "barrier block alignment");
static_assert(sizeof(Bars) <= 1024, "barrier block size");
static_assert(kStage + kXferBytes <= kBarOffset, "score CTA layout");
static_assert(kXferBytes <= kPBufStride && kXferBytes % 16 == 0, "P transfer size");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

// Sparse: the index list entries of key slots 128 t + 4 lane .. + 3 of
// sequence q (-1 past its n_slots = topk or topk_length); validated by the caller.
__device__ __forceinline__ void load_idx4(const SplitParams& p, int q, int t, int lane, int n_slots,
                                          int32_t (&id)[4]) {
  const int32_t* idx_row = p.indices + static_cast<int64_t>(q) * p.topk;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int slot = t * kTileTokens + 4 * lane + i;
    id[i] = slot < n_slots ? idx_row[slot] : -1;
  }
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Gather issuer index of a warp: warps 0, 2, 3, then 8, 9, ... (1 issues the
// MMAs, 4..7 are the row warps).
__device__ __forceinline__ int issuer_index(int warp) { return warp == 0 ? 0 : (warp < 4 ? warp - 1 : warp - 5); }

// One CTA per SM (shared memory); up to 224 registers per thread (8 warps, two
// per sub-partition), so each row thread's 128 scores stay in registers.
// kSparse: keys are pool rows named by p.indices (DSA top-k, -1 = none), read
// with tile::gather4 (the tensor map's box is one row); otherwise pages of the
// block table.  Paged: tm_qa, tm_qb view the cache as [8-token groups][9
// chunks][8 rows][64 columns] and load one page's [8][4][8][64] (V half) and
// [8][3][8][64] (K group) boxes; tm_kv is then unused.  tm_ql views the
// query rows as [9 chunks][rows][64 columns] with [2 x 128 x 64] boxes (a
// quarter of the latent part of one token's 128 rows), tm_qr as [rows][576]
// with [128 x 64] boxes (its RoPE part).
template <bool kSparse>
__global__ void __maxnreg__(kSparse ? 128 : 224)
    mla_pair_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_qa,
                    const __grid_constant__ CUtensorMap tm_qb, const __grid_constant__ CUtensorMap tm_ql,
                    const __grid_constant__ CUtensorMap tm_qr, const __grid_constant__ SplitParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOffset);
  const uint32_t base = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int part = blockIdx.x >> 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kKGroups; ++i) {
      mbar_init(smem_u32(&bars->kfull[i]), kSparse ? 3 : 1);  // sparse: three chunks per group
      // phase 0 completes when the first query rows staged in the slot are in
      // TMEM, phase t + 1 when tile t's products have read the slot's K group
      mbar_init(smem_u32(&bars->kempty[i]), 1);
    }
    for (int i = 0; i < kVGroups; ++i) {
      // sparse: two chunks per d quarter; paged: vfull[0], vfull[1] are the V halves
      mbar_init(smem_u32(&bars->vfull[i]), kSparse ? 2 : 1);
      mbar_init(smem_u32(&bars->vempty[i]), 1);
    }
    mbar_init(smem_u32(&bars->q_tma), 1);
    mbar_init(smem_u32(&bars->q_stage_free), 1);
    mbar_init(smem_u32(&bars->q_cp), 1);
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bars->q_box[i]), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars->s_full[b]), 1);
      mbar_init(smem_u32(&bars->s_free[b]), 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars->p_free[b]), 1);
      mbar_init(smem_u32(&bars->p_full[b]), 1);
      mbar_init(smem_u32(&bars->pv_done[b]), 1);
      mbar_init(smem_u32(&bars->side_read[b]), 4);
    }
    mbar_init(smem_u32(&bars->o_full), 1);
    mbar_init(smem_u32(&bars->o_free), 4);
    mbar_init(smem_u32(&bars->o_drained), 1);
    mbar_init(smem_u32(&bars->o_rescaled), 4);
    bars->abort = 0;
    fence_mbarrier_init();
    if (rank == 1) {  // both P buffers start empty and armed for their first copy
      mbar_arrive_expect_tx(smem_u32(&bars->p_full[0]), kXferBytes);
      mbar_arrive_expect_tx(smem_u32(&bars->p_full[1]), kXferBytes);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before any remote operation
  tc_fence_after();
  // Everything above overlaps the previous kernel of the stream (programmatic
  // dependent launch); its results (the schedule, the inputs) are read below.
  // The query rows of sequence `part` (the rows this part reads first when the
  // whole-sequence schedule is walked) start towards L2 before the wait: a
  // prefetch only warms L2, so rows a preceding kernel is still writing are
  // read for real after the wait all the same.
  if (rank == 0 && threadIdx.x == 32 * 2 && part < p.batch * p.s_q)
    prefetch_l2(p.q + static_cast<int64_t>(part) * kRows * kDqk, kRows * kDqk * 2);
  pdl_wait_primary();
  pdl_launch_dependents();  // the combine may launch now; it waits for this grid to finish
  // Schedule B (whole sequences) is walked when it is at most kSplitPenalty
  // tiles longer than A: on b=64, t=4096 (~2.3 us per dense tile) splitting
  // over 76 parts cost ~26 us in extra pieces and the combine for ~12 us of
  // better balance; a sparse tile takes about twice as long.
  constexpr int kSplitPenalty = kSparse ? 5 : 11;
  // The metadata must describe this call; otherwise nothing is read or written.
  const bool meta_ok = meta_header_matches(p.meta, p.batch, p.s_q, p.num_parts, p.topk, p.causal);
  const int32_t* meta = meta_ok ? schedule_for(p.meta, kSplitPenalty) : p.meta;
  if (blockIdx.x == 0 && threadIdx.x == blockDim.x - 1) {  // a thread with no work at the start
    // read by the combine after this grid: the schedule walked, or -1 when
    // the metadata was rejected (the combine then writes nothing), and
    // whether that schedule left anything to merge or fill
    p.ws_ctrl[1] = (meta_ok && (meta == p.meta || meta[kHTotalSplits] != meta[kHNSeq])) ? 1 : 0;
    p.ws_ctrl[0] = meta_ok ? (meta == p.meta ? 0 : 1) : -1;
    if (!meta_ok && p.err) atomicOr(p.err, MLA_DEVERR_METADATA);
  }
  const uint32_t tmem = bars->tmem_base;
  volatile uint32_t* abort_flag = &bars->abort;

  if (!meta_ok) {
    // nothing to do: every role is skipped, the teardown below still runs
  } else if (rank == 0) {
    // ================================================================ score CTA
    if (warp == 0 || warp == 2 || (kSparse && (warp == 3 || warp >= 8))) {
      // ---------------------------------------------------- K tile producers
      // Paged: lane 0 of warp 0 loads each group as one box per page.
      // Sparse: nine warps gather one chunk each; lane L gathers rows
      // 4L..4L+3 of the tile (invalid slots fetch pool row 0; the softmax
      // gives them zero weight); lane 0 owns the barriers.
      if (kSparse ? issuer_index(warp) < kKIssuersSparse : (warp == 0 && lane == 0)) {
        constexpr int kIssuers = kSparse ? kKIssuersSparse : 2;
        const int pw = issuer_index(warp);
        const uint64_t pol = l2_policy_evict_first();
        PartCursor cur = walked_part_cursor(p.meta, meta, part);
        int q, t0, t1, split;
        uint32_t tc = 0;
        int32_t issued[kKGroups];  // ring round of this issuer's last load per group slot
        for (int i = 0; i < kKGroups; ++i) issued[i] = -1;
        bool ok = true;
        bool first = true, q_issued = false;
        // The part's first query rows go through the K ring as four boxes,
        // each with its own barrier; the QK issuer moves each into TMEM as it
        // lands and releases a ring slot once the boxes in it are moved, so K
        // group g is requested while later boxes still arrive.
        auto issue_first_q = [&](int qq) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t bar = smem_u32(&bars->q_box[i]);
            mbar_arrive_expect_tx(bar, kQBoxBytes + (i == 0 ? kChunk : 0));
            if (i == 0) tma_load_2d(base + kQRope, &tm_qr, kDv, qq * kRows, bar, pol);
            tma_load_3d(base + i * kQBoxBytes, &tm_ql, 0, qq * kRows, 2 * i, bar, pol);
          }
          q_issued = true;
        };
        while (next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
          if (first) {
            first = false;
            if (pw == 0 && lane == 0) issue_first_q(q);
          }
          int32_t nid[4];  // sparse: the next tile's indices, requested one tile ahead
          const int32_t keys = meta_seq(meta, p.num_parts, q)[kSKeys];
          const int32_t* idx_row = p.indices + static_cast<int64_t>(q) * p.topk;
          const int32_t* bt_row = kSparse ? nullptr : bt_row_of(p, q);
          int32_t fallback = -2;  // sparse: first row the query names, found when a tile names none
          if constexpr (kSparse) load_idx4(p, q, t0, lane, keys, nid);
          else if (pw == 0) check_seq_keys(p, q, keys);
          for (int t = t0; t < t1; ++t, ++tc) {
            if (!ok) continue;
            int32_t y[4];
            if constexpr (kSparse) {
              int32_t id[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) id[i] = nid[i];
              if (t + 1 < t1) load_idx4(p, q, t + 1, lane, keys, nid);
              sparse_rows4(p, id, lane, idx_row, keys, pw == 0, &fallback, y);
            } else {
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {
                int32_t blk = page_of(p, bt_row, keys, 2 * t + h2);
                if (blk < 0) {
                  if (p.err && pw == 0) atomicOr(p.err, MLA_DEVERR_BAD_PAGE);
                  blk = static_cast<int32_t>(p.num_pages);  // out of range: TMA fills zeros
                }
                y[h2] = blk * kPage;
              }
            }
            if constexpr (!kSparse) {
              for (int g = 0; g < kKGroups && ok; ++g) {
                ok = mbar_wait(smem_u32(&bars->kempty[g]), tc & 1, abort_flag, p.err);
                if (!ok) break;
                const uint32_t bar = smem_u32(&bars->kfull[g]);
                mbar_arrive_expect_tx(bar, kKGroupBytes);
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2)  // the page's first 8-token group is y / 8
                  tma_load_4d(base + g * kKGroupBytes + h2 * kGroupPage, &tm_qb, 0, 0, 3 * g, y[h2] / 8, bar, pol);
                issued[g] = static_cast<int32_t>(tc);
              }
            }
            for (int c = pw; kSparse && c < kChunks && ok; c += kIssuers) {
              const int g = c / 3;
              const uint32_t slot = g, round = tc;  // one ring round per tile
              if (lane == 0) {
                ok = mbar_wait(smem_u32(&bars->kempty[slot]), round & 1, abort_flag, p.err);
                if (ok) mbar_arrive_expect_tx(smem_u32(&bars->kfull[slot]), kChunk);
              }
              if constexpr (kSparse) ok = __shfl_sync(0xffffffffu, ok, 0);
              if (!ok) break;
              const uint32_t bar = smem_u32(&bars->kfull[slot]);
              const uint32_t dst = base + slot * kKGroupBytes + (c - 3 * g) * kChunk;
              tma_gather4(dst + 4 * lane * 128, &tm_kv, c * 64, y[0], y[1], y[2], y[3], bar);
              issued[slot] = static_cast<int32_t>(round);
            }
          }
        }
        if (!ok && lane == 0) {  // let this issuer's copies in flight land before the CTA exits
          for (int i = 0; q_issued && i < 4; ++i) {
            const uint64_t t_start = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&bars->q_box[i]), 0) && globaltimer_ns() - t_start < 1000000ull) {
            }
          }
          for (int s = 0; s < kKGroups; ++s) {
            if (issued[s] < 0) continue;
            const uint64_t t_start = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&bars->kfull[s]), static_cast<uint32_t>(issued[s]) & 1u) &&
                   globaltimer_ns() - t_start < 1000000ull) {
            }
          }
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------- S = Q . K^T
      if (lane == 0) {
        PartCursor cur = walked_part_cursor(p.meta, meta, part);
        int q, t0, t1, split;
        uint32_t tc = 0, item = 0, qtma_n = 0, qcp_n = 0;  // completed phases of q_tma, q_cp
        bool ok = true, q_pending = false;  // q_pending: a query box is in flight
        const uint64_t qpol = l2_policy_evict_first();
        while (next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
          if (item > 0) {
            // a later piece's query rows: the RoPE part into kQRope and the
            // latent part two chunks at a time through the P staging buffer
            // (free once the previous piece's last P copy has read it, which
            // also means its QK products have completed), each pair moved into
            // TMEM by tcgen05.cp before the next one lands
            if (ok) ok = mbar_wait(smem_u32(&bars->q_stage_free), (item - 1) & 1, abort_flag, p.err);
            if (ok) tc_fence_after();
            for (int i = 0; i < 4 && ok; ++i) {
              const uint32_t bar = smem_u32(&bars->q_tma);
              mbar_arrive_expect_tx(bar, kQBoxBytes + (i == 0 ? kChunk : 0));
              if (i == 0) tma_load_2d(base + kQRope, &tm_qr, kDv, q * kRows, bar, qpol);
              tma_load_3d(base + kStage, &tm_ql, 0, q * kRows, 2 * i, bar, qpol);
              q_pending = true;
              ok = mbar_wait(bar, qtma_n & 1, abort_flag, p.err);
              if (!ok) break;
              q_pending = false;
              ++qtma_n;
              tc_fence_after();
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                const uint64_t qdesc = sw128_desc(base + kStage + c * (kRows * 128), 16, 1024);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  tmem_cp_128x256b(tmem + kQCol + 8 * (4 * (2 * i + c) + k), qdesc + static_cast<uint64_t>((32 * k) >> 4));
              }
              mma_commit(smem_u32(&bars->q_cp));
              ok = mbar_wait(smem_u32(&bars->q_cp), qcp_n & 1, abort_flag, p.err);  // the buffer takes the next pair
              ++qcp_n;
            }
          }
          if (item == 0) {
            // the first piece's latent Q, TMA-staged in the K ring as [8
            // chunks][128 rows][128 B] (128-byte swizzle, four two-chunk
            // boxes), goes into TMEM by tcgen05.cp, one K = 16 step (8
            // columns) per copy, box by box as they land; ring slot g (48 KB
            // at 48 g KB) is released once the boxes overlapping it are moved:
            // slot 0 after boxes 0, 1, slot 1 after box 2, slot 2 after box 3.
            // Its RoPE part is in kQRope (with box 0).
            static_assert(kKGroups == 3 && kKGroupBytes == 3 * kQBoxBytes / 2, "query boxes over the K ring slots");
#pragma unroll 1
            for (int i = 0; i < 4 && ok; ++i) {
              ok = mbar_wait(smem_u32(&bars->q_box[i]), 0, abort_flag, p.err);
              if (!ok) break;
              tc_fence_after();
#pragma unroll
              for (int c = 2 * i; c < 2 * i + 2; ++c) {
                const uint64_t qdesc = sw128_desc(base + c * (kRows * 128), 16, 1024);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  tmem_cp_128x256b(tmem + kQCol + 8 * (4 * c + k), qdesc + static_cast<uint64_t>((32 * k) >> 4));
              }
              if (i >= 1) mma_commit(smem_u32(&bars->kempty[i - 1]));  // the copies have read the slot
            }
          }
          const uint64_t rope_desc = sw128_desc(base + kQRope, 16, 1024);
          for (int t = t0; t < t1; ++t, ++tc) {
            if (!ok) continue;
            const uint32_t sb = tc & 1;
            ok = mbar_wait(smem_u32(&bars->s_free[sb]), ((tc >> 1) & 1) ^ 1, abort_flag, p.err);
            if (!ok) continue;
            tc_fence_after();
            const uint32_t d = tmem + kSCol + 128 * sb;
#pragma unroll
            for (int g = 0; g < 3; ++g) {
              const uint32_t slot = g;  // group g of every tile lives in slot g
              ok = mbar_wait(smem_u32(&bars->kfull[slot]), tc & 1, abort_flag, p.err);
              if (!ok) break;
              tc_fence_after();
              // paged: chunk 3g + cc at +1 KB cc, 8-token groups 3 KB apart;
              // sparse: [128 tokens x 128 B] chunks 16 KB apart
              const uint64_t bdesc = sw128_desc(base + slot * kKGroupBytes, 16, kSparse ? 1024 : 3072);
#pragma unroll
              for (int cc = 0; cc < 3; ++cc)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const uint64_t b = bdesc + static_cast<uint64_t>(((kSparse ? cc * kChunk : cc * 1024) + 32 * k) >> 4);
                  const uint32_t acc = (g | cc | k) != 0 ? 1u : 0u;
                  if (3 * g + cc < 8)  // latent columns: A = Q in TMEM
                    mma_bf16_ts(d, tmem + kQCol + 8 * (4 * (3 * g + cc) + k), b, kIdescS, acc);
                  else  // RoPE columns: A = Q RoPE part in smem
                    mma_bf16_ss(d, rope_desc + static_cast<uint64_t>((32 * k) >> 4), b, kIdescS, acc);
                }
              mma_commit(smem_u32(&bars->kempty[slot]));
            }
            if (!ok) continue;
            mma_commit(smem_u32(&bars->s_full[sb]));
          }
          ++item;
        }
        if (q_pending) {  // a query box still in flight: let it land before the CTA exits
          const uint64_t t_start = globaltimer_ns();
          while (!mbar_try_wait(smem_u32(&bars->q_tma), qtma_n & 1) && globaltimer_ns() - t_start < 1000000ull) {
          }
        }
      }
    } else if (warp >= 4 && warp < 8) {
      // ---------------------------------------------------- Q load, softmax, P
      // Thread r owns query row r: its scores are TMEM lane r, so the row max
      // and sums need no cross-thread exchange.  Probabilities are taken
      // against a per-row reference m (log2 units): the first tile of a piece
      // sets it to that tile's row max; a later tile moves it only when a
      // score exceeds it by more than kRescaleLog2, and then O and the sums
      // are rescaled by alpha = 2^(m_old - m_new).  Two running sums: of the
      // fp32 probabilities (for the LSE) and of their bf16 roundings, which
      // are the weights the PV product multiplies (to normalise O).
      const int r = threadIdx.x - 128;
      const uint32_t lane_off = static_cast<uint32_t>((warp - 4) * 32) << 16;
      const uint32_t stage = base + kStage;
      const uint32_t prow = stage + (r >> 3) * 1024 + (r & 7) * 128;
      const float sc = p.scale_log2;
      PartCursor cur = walked_part_cursor(p.meta, meta, part);
      int q, t0, t1, split;
      uint32_t tc = 0, item = 0;
      bool ok = true;
      while (next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
        const int32_t* srec = meta_seq(meta, p.num_parts, q);
        const int32_t keys = srec[kSKeys];
        // the piece's query rows come by TMA and tcgen05.cp (QK issuer); the
        // next piece's rows (147 KB, contiguous) start towards L2
        if (r == 0) {
          PartCursor nc = cur;
          int nq, nt0, nt1, nsplit;
          if (next_piece(meta, p.num_parts, &nc, &nq, &nt0, &nt1, &nsplit))
            prefetch_l2(p.q + static_cast<int64_t>(nq) * kRows * kDqk, kRows * kDqk * 2);
        }
        float m_use = 0.f, lsum = 0.f, bsum = 0.f;
        for (int t = t0; t < t1; ++t, ++tc) {
          const uint32_t sb = tc & 1;
          const uint32_t t_s = tmem + lane_off + kSCol + 128 * sb;
          // sparse: bit L of vm[k] = key slot t * 128 + 32 k + L names a pool row
          uint32_t vm[4] = {~0u, ~0u, ~0u, ~0u};
          int32_t sid[4];  // sparse: requested before the S wait, used after it
          if constexpr (kSparse) {
            const int32_t* idx_row = p.indices + static_cast<int64_t>(q) * p.topk;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int slot = t * kTileTokens + 32 * k + lane;
              sid[k] = slot < keys ? idx_row[slot] : -1;
            }
          }
          if (ok) ok = mbar_wait(smem_u32(&bars->s_full[sb]), (tc >> 1) & 1, abort_flag, p.err);
          ok = __all_sync(0xffffffffu, ok);
          if constexpr (kSparse) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              vm[k] = __ballot_sync(0xffffffffu, sid[k] >= 0 && static_cast<int64_t>(sid[k]) < p.s_kv);
          }
          const int n_valid = keys - t * kTileTokens;  // >= 1; < 128 only on the last tile
          const bool full = kSparse || n_valid >= kTileTokens;
          // Row max of the raw scores (the scale is positive) over the tile's
          // keys.  The first tile of a piece takes its reference from it.  A
          // later tile needs it only when its probabilities against the current
          // reference sum to more than 2^kRescaleLog2 (necessary for one of
          // them to exceed that bound), which is rare: then the warp finds the
          // max and, if the reference has to move, redoes the pass.
          auto row_max = [&]() {
            float u = -INFINITY;
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
              float v[32];
              tmem_ld32(t_s + 32 * i, v);
              tmem_wait_ld();
              if (!full) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 32 * i + j < n_valid ? v[j] : -INFINITY;
              }
              if constexpr (kSparse) {
                const uint32_t w = vm[0] * (i == 0) | vm[1] * (i == 1) | vm[2] * (i == 2) | vm[3] * (i == 3);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = (w >> j) & 1u ? v[j] : -INFINITY;
              }
#pragma unroll
              for (int j = 0; j < 32; j += 2) u = fmax3(u, v[j], v[j + 1]);
            }
            return u * sc;
          };
          float alpha = 1.f;
          if (ok && t == t0) {
            tc_fence_after();
            const float u = row_max();
            m_use = u == -INFINITY ? 0.f : u;
          }
          // p = 2^(s * scale - m) -> bf16 P row r in the staging buffer (two
          // 64-token chunks, 128-byte swizzle), and the two sums
          if constexpr (kSparse) {
            if (r == 0 && tc > 0) bulk_wait_read_all();  // the previous copy has read the staging
            named_barrier_sync(1, kRowThreads);
          } else {
            named_barrier_sync(1, kXferNamedThreads);  // warp 3's previous copy has read the staging
          }
          if (ok && t != t0) tc_fence_after();
          float ls = 0.f, bs = 0.f, ls2 = 0.f, bs2 = 0.f;
          for (bool again = ok; again;) {
            again = false;
            const float neg_m = -m_use;
            ls = 0.f; bs = 0.f; ls2 = 0.f; bs2 = 0.f;
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
              float v[32];
              tmem_ld32(t_s + 32 * i, v);
              tmem_wait_ld();
              if (!full) {  // keys past the end: s = -inf, p = 2^-inf = 0
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 32 * i + j < n_valid ? v[j] : -INFINITY;
              }
              if constexpr (kSparse) {  // slots without a pool row: p = 0
                const uint32_t w = vm[0] * (i == 0) | vm[1] * (i == 1) | vm[2] * (i == 2) | vm[3] * (i == 3);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = (w >> j) & 1u ? v[j] : -INFINITY;
              }
              // packed fp32x2 FMA/adds: one instruction per key pair
              uint32_t pk[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                float x0, x1;
                asm("{ .reg .b64 a, b, c, d; mov.b64 a, {%2, %3}; mov.b64 b, {%4, %4}; mov.b64 c, {%5, %5};"
                    " fma.rn.f32x2 d, a, b, c; mov.b64 {%0, %1}, d; }"
                    : "=f"(x0), "=f"(x1) : "f"(v[2 * j]), "f"(v[2 * j + 1]), "f"(sc), "f"(neg_m));
                const float e0 = fast_exp2(x0);
                const float e1 = fast_exp2(x1);
                pk[j] = pack_bf16x2(e0, e1);
                asm("{ .reg .b64 a, b, c; mov.b64 a, {%0, %1}; mov.b64 b, {%4, %5}; add.rn.f32x2 c, a, b; mov.b64 {%0, %1}, c;"
                    " mov.b64 a, {%2, %3}; mov.b64 b, {%6, %7}; add.rn.f32x2 c, a, b; mov.b64 {%2, %3}, c; }"
                    : "+f"(ls), "+f"(ls2), "+f"(bs), "+f"(bs2)
                    : "f"(e0), "f"(e1), "f"(__uint_as_float(pk[j] << 16)), "f"(__uint_as_float(pk[j] & 0xFFFF0000u)));
              }
              const uint32_t chunk = prow + (i >> 1) * 16384;
#pragma unroll
              for (int uu = 0; uu < 4; ++uu)
                st_shared_v4(chunk + ((((i & 1) * 4 + uu) ^ (r & 7)) << 4), pk[4 * uu], pk[4 * uu + 1],
                             pk[4 * uu + 2], pk[4 * uu + 3]);
            }
            bool move = false;
            if (__any_sync(0xffffffffu, t != t0 && !(ls + ls2 <= kMoveSum))) {
              const float u = row_max();
              if (u > m_use + kRescaleLog2) {  // move the reference; the warp redoes the pass
                const float a_new = fast_exp2(m_use - u);
                alpha *= a_new;
                m_use = u;
                lsum *= a_new;
                bsum *= a_new;
                move = true;
              }
            }
            again = __any_sync(0xffffffffu, move);
          }
          const uint32_t any = __any_sync(0xffffffffu, alpha != 1.f) ? 1u : 0u;
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->s_free[sb]));  // S buffer sb may be rewritten
          lsum += ls + ls2;
          bsum += bs + bs2;
          st_shared_f32(stage + kSideAlpha + 4 * r, alpha);
          if (t == t1 - 1) {
            float inv_l = bsum > 0.f ? 1.f / bsum : 0.f;
            // attention sink: applied with 1/l to a final row, by the combine to a split row
            if (kSparse && p.attn_sink && srec[kSNSplits] == 1) {
              const float lse_t = (lsum > 0.f && bsum > 0.f) ? (m_use + __log2f(lsum)) * 0.69314718055994531f
                                                             : -INFINITY;
              inv_l *= attn_sink_factor(lse_t, p.attn_sink[r]);
            }
            st_shared_f32(stage + kSideInvL + 4 * r, inv_l);
          }
          if (lane == 0) st_shared_u32(stage + kSideFlags + 4 * (warp - 4), any);
          fence_proxy_async_smem();
          if constexpr (!kSparse) named_barrier_arrive(2, kXferNamedThreads);  // staging full: warp 3 copies
          if constexpr (kSparse) named_barrier_sync(2, kRowThreads);  // staging full
          if (kSparse && r == 0 && ok) {  // one copy of tile tc into the peer's P buffer tc mod 2
            const uint32_t b = tc & 1;
            ok = mbar_wait_cluster(smem_u32(&bars->p_free[b]), ((tc >> 1) & 1) ^ 1, abort_flag, p.err);
            if (ok) {
              bulk_copy_to_peer(mapa_shared(base + kPBuf0 + b * kPBufStride, 1), base + kStage, kXferBytes,
                                mapa_shared(smem_u32(&bars->p_full[b]), 1));
              bulk_commit_group();
            }
          }
          if (kSparse && r == 0 && t == t1 - 1) {  // the staging buffer may take the next piece's query rows
            bulk_wait_read_all();
            mbar_arrive(smem_u32(&bars->q_stage_free));
          }
        }
        // LSE of row r for this piece
        const float lse_v = (lsum > 0.f && bsum > 0.f) ? (m_use + __log2f(lsum)) * 0.69314718055994531f
                                                       : -INFINITY;
        if (ok) {
          if (srec[kSNSplits] == 1) {
            const int b = q / p.s_q, j = q % p.s_q;
            p.lse[(static_cast<int64_t>(b) * kRows + r) * p.s_q + j] = lse_v;
          } else {
            p.ws_lse[static_cast<int64_t>(srec[kSSplitOff] + split) * kRows + r] = lse_v;
          }
        }
        ++item;
      }
      if (kSparse && r == 0) bulk_wait_all();  // the last copy has landed in the peer
    } else if (warp == 3 && !kSparse) {
      // ---------------------------------------------------- P transfers (dense)
      PartCursor cur = walked_part_cursor(p.meta, meta, part);
      int q, t0, t1, split;
      uint32_t tc = 0;
      bool ok = true;
      while (next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
        for (int t = t0; t < t1; ++t, ++tc) {
          if (lane == 0 && tc > 0) bulk_wait_read_all();
          __syncwarp();
          named_barrier_arrive(1, kXferNamedThreads);  // staging free
          named_barrier_sync(2, kXferNamedThreads);    // staging full
          if (lane == 0 && ok) {
            const uint32_t b = tc & 1;
            ok = mbar_wait_cluster(smem_u32(&bars->p_free[b]), ((tc >> 1) & 1) ^ 1, abort_flag, p.err);
            if (ok) {
              bulk_copy_to_peer(mapa_shared(base + kPBuf0 + b * kPBufStride, 1), base + kStage, kXferBytes,
                                mapa_shared(smem_u32(&bars->p_full[b]), 1));
              bulk_commit_group();
            }
          }
          if (lane == 0 && t == t1 - 1) {  // the staging buffer may take the next piece's query rows
            bulk_wait_read_all();
            mbar_arrive(smem_u32(&bars->q_stage_free));
          }
          __syncwarp();
        }
      }
      if (lane == 0) bulk_wait_all();
    }
  } else {
    // ================================================================ output CTA
    if (warp == 0 || warp == 2 || (kSparse && (warp == 3 || warp >= 8))) {
      // ---------------------------------------------------- V tile producers
      // Paged: lane 0 of warp 0 loads each V half (chunks 0..3, 4..7) as one
      // box per page.  Sparse: eight warps gather one chunk each; each issuer
      // loads into the same d quarter every tile, so it waits on that slot in
      // order.
      if (kSparse ? issuer_index(warp) < kVIssuersSparse : (warp == 0 && lane == 0)) {
        constexpr int kIssuers = kSparse ? kVIssuersSparse : 2;
        const int pw = issuer_index(warp);
        const uint64_t pol = l2_policy_evict_first();
        PartCursor cur = walked_part_cursor(p.meta, meta, part);
        int q, t0, t1, split;
        uint32_t tc = 0;
        int32_t issued[kVGroups];
        for (int i = 0; i < kVGroups; ++i) issued[i] = -1;
        bool ok = true;
        while (next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
          int32_t nid[4];  // sparse: the next tile's indices, requested one tile ahead
          const int32_t keys = meta_seq(meta, p.num_parts, q)[kSKeys];
          const int32_t* idx_row = p.indices + static_cast<int64_t>(q) * p.topk;
          const int32_t* bt_row = kSparse ? nullptr : bt_row_of(p, q);
          int32_t fallback = -2;
          if constexpr (kSparse) load_idx4(p, q, t0, lane, keys, nid);
          for (int t = t0; t < t1; ++t, ++tc) {
            if (!ok) continue;
            int32_t y[4];
            if constexpr (kSparse) {
              int32_t id[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) id[i] = nid[i];
              if (t + 1 < t1) load_idx4(p, q, t + 1, lane, keys, nid);
              sparse_rows4(p, id, lane, idx_row, keys, false, &fallback, y);
            } else {
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {
                int32_t blk = page_of(p, bt_row, keys, 2 * t + h2);
                if (blk < 0) blk = static_cast<int32_t>(p.num_pages);
                y[h2] = blk * kPage;
              }
            }
            if constexpr (!kSparse) {
              for (int hf = 0; hf < 2 && ok; ++hf) {
                ok = mbar_wait(smem_u32(&bars->vempty[hf]), (tc & 1) ^ 1, abort_flag, p.err);
                if (!ok) break;
                const uint32_t bar = smem_u32(&bars->vfull[hf]);
                mbar_arrive_expect_tx(bar, 2 * kHalfPage);
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2)
                  tma_load_4d(base + hf * 2 * kHalfPage + h2 * kHalfPage, &tm_qa, 0, 0, 4 * hf, y[h2] / 8, bar, pol);
                issued[hf] = static_cast<int32_t>(tc);
              }
            }
            for (int c = pw; kSparse && c < 8 && ok; c += kIssuers) {
              const uint32_t gv = 4 * tc + (c >> 1), slot = gv % kVGroups, round = gv / kVGroups;
              if (lane == 0) {
                ok = mbar_wait(smem_u32(&bars->vempty[slot]), (round & 1) ^ 1, abort_flag, p.err);
                if (ok) mbar_arrive_expect_tx(smem_u32(&bars->vfull[slot]), kChunk);
              }
              if constexpr (kSparse) ok = __shfl_sync(0xffffffffu, ok, 0);
              if (!ok) break;
              const uint32_t bar = smem_u32(&bars->vfull[slot]);
              const uint32_t dst = base + slot * kVGroupBytes + (c & 1) * kChunk;
              tma_gather4(dst + 4 * lane * 128, &tm_kv, c * 64, y[0], y[1], y[2], y[3], bar);
              issued[slot] = static_cast<int32_t>(round);
            }
          }
        }
        if (!ok && lane == 0) {
          for (int s = 0; s < kVGroups; ++s) {
            if (issued[s] < 0) continue;
            const uint64_t t_start = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&bars->vfull[s]), static_cast<uint32_t>(issued[s]) & 1u) &&
                   globaltimer_ns() - t_start < 1000000ull) {
            }
          }
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------- O += P . V
      if (lane == 0) {
        PartCursor cur = walked_part_cursor(p.meta, meta, part);
        int q, t0, t1, split;
        uint32_t tc = 0, item = 0, rc = 0;
        bool ok = true;
        while (next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
          for (int t = t0; t < t1; ++t, ++tc) {
            if (!ok) continue;
            const uint32_t b = tc & 1;
            const uint32_t pbuf = base + kPBuf0 + b * kPBufStride;
            ok = mbar_wait_cluster(smem_u32(&bars->p_full[b]), (tc >> 1) & 1, abort_flag, p.err);
            if (!ok) continue;
            if (t == t0) {
              ok = mbar_wait(smem_u32(&bars->o_free), (item & 1) ^ 1, abort_flag, p.err);
            } else {
              const uint4 f = ld_shared_v4(pbuf + kSideFlags);
              if ((f.x | f.y | f.z | f.w) != 0u) {
                mma_commit(smem_u32(&bars->o_drained));
                ok = mbar_wait(smem_u32(&bars->o_rescaled), rc & 1, abort_flag, p.err);
                ++rc;
              }
            }
            if (!ok) continue;
            tc_fence_after();
            const uint64_t pdesc = sw128_desc(pbuf, 16, 1024);
            if constexpr (!kSparse) {
              // paged: V half hf (N = 256: 64-column blocks 1 KB apart, 8-token
              // groups 4 KB apart) into O columns 256 hf ..
              for (int hf = 0; hf < 2 && ok; ++hf) {
                ok = mbar_wait(smem_u32(&bars->vfull[hf]), tc & 1, abort_flag, p.err);
                if (!ok) break;
                tc_fence_after();
                const uint64_t vdesc = sw128_desc(base + hf * 2 * kHalfPage, 1024, 4096);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                  mma_bf16_ss(tmem + 256 * hf,
                              pdesc + static_cast<uint64_t>(((s >> 2) * 16384 + (s & 3) * 32) >> 4),
                              vdesc + static_cast<uint64_t>((8192 * s) >> 4), kIdescO256,
                              (t != t0 || s != 0) ? 1u : 0u);
                mma_commit(smem_u32(&bars->vempty[hf]));
              }
            }
            for (int qd = 0; kSparse && qd < 4 && ok; ++qd) {
              const uint32_t gv = 4 * tc + qd, slot = gv % kVGroups;
              ok = mbar_wait(smem_u32(&bars->vfull[slot]), (gv / kVGroups) & 1, abort_flag, p.err);
              if (!ok) break;
              tc_fence_after();
              const uint64_t vdesc = sw128_desc(base + slot * kVGroupBytes, kChunk, 1024);
#pragma unroll
              for (int s = 0; s < 8; ++s)
                mma_bf16_ss(tmem + 128 * qd,
                            pdesc + static_cast<uint64_t>(((s >> 2) * 16384 + (s & 3) * 32) >> 4),
                            vdesc + static_cast<uint64_t>((2048 * s) >> 4), kIdescO,
                            (t != t0 || s != 0) ? 1u : 0u);
              mma_commit(smem_u32(&bars->vempty[slot]));
            }
            if (!ok) continue;
            mma_commit(smem_u32(&bars->pv_done[b]));
            if (t == t1 - 1) mma_commit(smem_u32(&bars->o_full));
          }
          ++item;
        }
      }
    } else if (warp >= 4 && warp < 8) {
      // ---------------------------------------------------- rescale, epilogue
      const int r = threadIdx.x - 128;
      const uint32_t t_o = tmem + (static_cast<uint32_t>((warp - 4) * 32) << 16);
      PartCursor cur = walked_part_cursor(p.meta, meta, part);
      int q, t0, t1, split;
      uint32_t tc = 0, item = 0, rc = 0;
      bool ok = true;
      while (next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
        const int32_t* srec = meta_seq(meta, p.num_parts, q);
        float inv_l = 0.f;
        for (int t = t0; t < t1; ++t, ++tc) {
          const uint32_t b = tc & 1;
          const uint32_t side = base + kPBuf0 + b * kPBufStride;
          if (ok) ok = mbar_wait_cluster(smem_u32(&bars->p_full[b]), (tc >> 1) & 1, abort_flag, p.err);
          ok = __all_sync(0xffffffffu, ok);
          float alpha = 1.f;
          uint32_t any = 0;
          if (ok) {
            alpha = ld_shared_f32(side + kSideAlpha + 4 * r);
            const uint4 f = ld_shared_v4(side + kSideFlags);
            any = f.x | f.y | f.z | f.w;
            if (t == t1 - 1) inv_l = ld_shared_f32(side + kSideInvL + 4 * r);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->side_read[b]));  // done with the side data
          if (kSparse && warp == 4 && lane == 0 && ok && tc >= 1) {
            // hand P buffer (tc - 1) mod 2 back: every row warp has read tile
            // tc - 1's side data and its PV has completed; armed for tile tc + 1
            const uint32_t pb = (tc - 1) & 1, ph = ((tc - 1) >> 1) & 1;
            ok = mbar_wait(smem_u32(&bars->side_read[pb]), ph, abort_flag, p.err);
            if (ok) ok = mbar_wait(smem_u32(&bars->pv_done[pb]), ph, abort_flag, p.err);
            if (ok) {
              mbar_arrive_expect_tx(smem_u32(&bars->p_full[pb]), kXferBytes);
              mbar_remote_arrive(mapa_shared(smem_u32(&bars->p_free[pb]), 0));
            }
          }
          if (ok && t != t0 && any != 0u) {
            ok = mbar_wait(smem_u32(&bars->o_drained), rc & 1, abort_flag, p.err);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
              tc_fence_after();
              if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                for (int blk = 0; blk < kDv / 32; ++blk) {
                  float v[32];
                  tmem_ld32(t_o + 32 * blk, v);
                  tmem_wait_ld();
#pragma unroll
                  for (int i = 0; i < 32; ++i) v[i] *= alpha;
                  tmem_st32(t_o + 32 * blk, v);
                }
                tmem_wait_st();
              }
              tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->o_rescaled));
            ++rc;
          }
        }
        // epilogue: O row r / sum of bf16(p) -> out (single split) or fp32 partial
        if (ok) ok = mbar_wait(smem_u32(&bars->o_full), item & 1, abort_flag, p.err);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          tc_fence_after();
          // Thread r holds row r of O; each 128-byte slice of the warp's 32 rows
          // goes through a swizzled 4 KB staging area so that every global
          // store instruction writes four whole 128-byte row segments.
          const bool final_out = srec[kSNSplits] == 1;
          const int64_t row0 = (final_out ? static_cast<int64_t>(q) : static_cast<int64_t>(srec[kSSplitOff] + split)) *
                                   kRows + 32 * (warp - 4);
          const uint32_t stg = base + kEpi + (warp - 4) * 4096;
          const int rr0 = lane >> 3, uu = lane & 7;
          if (final_out) {
#pragma unroll 1
            for (int blk = 0; blk < kDv / 64; ++blk) {  // 64 bf16 columns = 128 bytes per row
              uint32_t pk[32];
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {
                float v[32];
                tmem_ld32(t_o + 64 * blk + 32 * h2, v);
                tmem_wait_ld();
                // a row without keys (inv_l = 0) is written as exact zeros: its O
                // may hold products of zero weights with rows nobody named
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  pk[16 * h2 + i] = inv_l != 0.f ? pack_bf16x2(v[2 * i] * inv_l, v[2 * i + 1] * inv_l) : 0u;
              }
#pragma unroll
              for (int u = 0; u < 8; ++u)
                st_shared_v4(stg + lane * 128 + ((u ^ (lane & 7)) << 4), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2],
                             pk[4 * u + 3]);
              __syncwarp();
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int rr = 4 * j + rr0;
                const uint4 x = ld_shared_v4(stg + rr * 128 + ((uu ^ (rr & 7)) << 4));
                *reinterpret_cast<uint4*>(p.out + (row0 + rr) * kDv + 64 * blk + 8 * uu) = x;
              }
              __syncwarp();
            }
          } else {
#pragma unroll 1
            for (int blk = 0; blk < kDv / 32; ++blk) {  // 32 fp32 columns = 128 bytes per row
              float v[32];
              tmem_ld32(t_o + 32 * blk, v);
              tmem_wait_ld();
              if (inv_l == 0.f) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.f;
              }
#pragma unroll
              for (int u = 0; u < 8; ++u)
                st_shared_v4(stg + lane * 128 + ((u ^ (lane & 7)) << 4), __float_as_uint(v[4 * u] * inv_l),
                             __float_as_uint(v[4 * u + 1] * inv_l), __float_as_uint(v[4 * u + 2] * inv_l),
                             __float_as_uint(v[4 * u + 3] * inv_l));
              __syncwarp();
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int rr = 4 * j + rr0;
                const uint4 x = ld_shared_v4(stg + rr * 128 + ((uu ^ (rr & 7)) << 4));
                *reinterpret_cast<uint4*>(p.ws_o + (row0 + rr) * kDv + 32 * blk + 4 * uu) = x;
              }
              __syncwarp();
            }
          }
          tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->o_free));
        ++item;
      }
    } else if (warp == 3 && !kSparse) {
      // ---------------------------------------------------- P buffer hand-back
      PartCursor cur = walked_part_cursor(p.meta, meta, part);
      int q, t0, t1, split;
      uint32_t tc = 0;
      bool ok = true;
      while (next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
        for (int t = t0; t < t1; ++t, ++tc) {
          if (lane == 0 && ok) {
            const uint32_t b = tc & 1;
            ok = mbar_wait(smem_u32(&bars->side_read[b]), (tc >> 1) & 1, abort_flag, p.err);
            if (ok) ok = mbar_wait(smem_u32(&bars->pv_done[b]), (tc >> 1) & 1, abort_flag, p.err);
            if (ok) {
              mbar_arrive_expect_tx(smem_u32(&bars->p_full[b]), kXferBytes);  // armed for tile tc + 2
              mbar_remote_arrive(mapa_shared(smem_u32(&bars->p_free[b]), 0));
            }
          }
          __syncwarp();
        }
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no peer still copies into or arrives on this CTA's smem
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace pair
}  // namespace mla
