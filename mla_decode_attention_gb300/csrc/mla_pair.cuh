// Paired-CTA MLA decode kernel for 128 query rows per query token (sm_103a).
//
// A cluster of two CTAs on two SMs shares one schedule part.  Per 128-key tile:
//
//   score CTA (rank 0):  S[128 rows x 128 tokens] = Q[128 x 576] . K_tile^T
//                        (tcgen05; the 512 latent columns with A = Q in TMEM,
//                        the 64 RoPE columns with A = Q's RoPE part in shared
//                        memory), then the online softmax with one thread per
//                        query row; P (bf16) goes to its own TMEM and, with the
//                        per-row rescale factors, to the output CTA by one
//                        shared-memory bulk copy.  It also owns the last 64
//                        output columns: O[:, 448:512] += P . V_tile[:, 448:512]
//                        (A = P in TMEM, B = the tile's latent chunk 7).
//   output CTA (rank 1): copies P into its TMEM and computes
//                        O[:, 0:448] += P[128 x 128] . V_tile[128 x 448]
//                        (A = P in TMEM, B = V in shared memory; O in TMEM).
//
// Both CTAs read the same cached rows: the score CTA all 576 columns, the
// output CTA the first 448 (V is the latent part of the same row, FlashMLA
// deep dive, "Theoretical Analysis"; the second reader finds the rows in L2).
// Every PV product takes its A operand from TMEM: on this GPU a cluster whose
// CTAs keep issuing MMAs with A from TMEM in one CTA and A from shared memory
// in the other runs all of them at about half rate, while TMEM-A in both runs
// at full rate (a handful of shared-memory-A MMAs for the RoPE columns does
// not matter).  TMEM use:
//   score CTA:  [0, 256) Q latent part (bf16 pairs), [256, 384) S (fp32, one
//               buffer: the row threads load a tile's scores into registers
//               at once and free it), [384, 448) P (bf16 pairs), [448, 512)
//               O columns 448..511 (fp32)
//   output CTA: [0, 448) O columns 0..447 (fp32), [448, 512) P (bf16 pairs)
//
// Roles (384 threads, both CTAs; three warps per SM sub-partition, so each
// thread may hold 168 registers):
//   warps 0, 2 lane 0    : TMA issuers (dense; chunk c of a tile by issuer c mod
//                          2).  Sparse: warps 0, 2, 3, every lane gathers.
//   warp 1               : TMEM owner; lane 0 issues every MMA
//   warp 3 (dense)       : score CTA: the P bulk copies (named barriers 1, 2
//                          with warps 4..11 around the staging buffer);
//                          output CTA: hands consumed P buffers back
//   warps 4..11          : row threads: two per query row, thread (h, r) with
//                          r = 32 (warp mod 4) + lane = TMEM lane r and half
//                          h = 0 (warps 4..7) or 1 (warps 8..11).  Score CTA:
//                          tokens 64h .. 64h + 63 of each tile (Q loads, the
//                          softmax on those 64 scores, their P), output
//                          columns 448 + 32h .. +31 and, for h = 0, the LSE;
//                          output CTA: P tokens 64h .. +63 into TMEM, the
//                          rescale and epilogue of columns 224h .. 224h + 223.
//
// Waits are bounded (mbar_wait*); after an abort every role keeps walking its
// schedule without waiting, so the named barriers between warps 3..11 stay
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

constexpr int kThreads = 384;
constexpr int kRows = 128;                         // query rows per cluster = TMEM lanes
constexpr int kChunk = kTileTokens * 64 * 2;       // 16 KB: [128 tokens x 64 columns] bf16
// ---- score CTA shared memory
constexpr int kKGroups = 3;                        // K tile: groups {0,1,2}, {3,4,5}, {6,7,8}
constexpr int kKSlot2 = 6 * kChunk;                // group 2 slot: chunk 6, then chunk 8 (RoPE)
constexpr int kC7 = 8 * kChunk;                    // chunk 7 (columns 448..511), two buffers
constexpr int kQRope = 10 * kChunk;                // 163840: Q RoPE columns [128 x 64] bf16
constexpr int kStage = 11 * kChunk;                // 180224: P staging for the output CTA
constexpr int kPBytes = kRows * kTileTokens * 2;   // 32768: P[128 rows x 128 tokens] bf16
constexpr int kSideAlpha = kPBytes;                // float alpha[128]
constexpr int kSideInvL = kPBytes + 512;           // float inv_l[128] (last tile of a piece)
constexpr int kSideFlags = kPBytes + 1024;         // uint32 per row warp: any alpha != 1
constexpr int kXferBytes = kPBytes + 1040;         // 33808 bytes per tile
// ---- output CTA shared memory
constexpr int kVGroups = 4;                        // V quarters: chunks {0,1}, {2,3}, {4,5}, {6}
constexpr int kVGroupBytes = 2 * kChunk;           // 32 KB
constexpr int kPBuf0 = kVGroups * kVGroupBytes;    // 131072
constexpr int kPBufStride = 34816;                 // kXferBytes rounded up to 1 KB
constexpr int kEpi = kPBuf0 + 2 * kPBufStride;     // 200704: 2 KB per row warp for the epilogue
// score CTA: the two row threads of a query row exchange partial row maxima
// (per tile parity) and, at a piece's end, partial sums
constexpr int kRedMax = kStage + kXferBytes;       // 214032: float [2 parity][2 halves][128]
constexpr int kRedSum = kRedMax + 2048;            // float [2 sums][2 halves][128]
constexpr int kBarOffset = 219136;                 // after both layouts, same offset in both CTAs
// ---- output columns
constexpr int kDvOut = 448;                        // output CTA: columns 0..447
constexpr int kDvTail = kDv - kDvOut;              // score CTA: columns 448..511
// ---- TMEM columns
constexpr uint32_t kQCol = 0;                      // score CTA: Q latent part
constexpr uint32_t kSCol = 256;                    // score CTA: S
constexpr uint32_t kPColS = 384;                   // score CTA: P
constexpr uint32_t kOTailCol = 448;                // score CTA: O columns 448..511
constexpr uint32_t kOCol = 0;                      // output CTA: O columns 0..447
constexpr uint32_t kPColO = 448;                   // output CTA: P
constexpr uint32_t kIdescS = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescO128 = idesc_bf16(128, 128, false, true);
constexpr uint32_t kIdescO64 = idesc_bf16(128, 64, false, true);
constexpr uint32_t kRowThreads = 256;              // warps 4..11
constexpr uint32_t kXferNamedThreads = 288;        // dense: warps 3..11
constexpr uint32_t kRowExchange = 3;               // named barrier of the row-thread exchanges

struct Bars {
  // score CTA
  uint64_t kfull[kKGroups], kempty[kKGroups];      // K ring (group 2 includes chunk 7's buffer)
  uint64_t c7empty[2];                             // chunk-7 buffers, released by the P.V tail
  uint64_t q_full, q_free, s_full, s_free;
  uint64_t p_ready, p_tmem_free, o_tail_full;
  uint64_t p_free[2];                              // arrived by the output CTA
  // output CTA
  uint64_t vfull[kVGroups], vempty[kVGroups];      // V ring
  uint64_t p_full[2];                              // completed by the bulk copies
  uint64_t p_tmem_full, pv_done, o_full;
  uint64_t side_read[2];                           // row warps have read P buffer b
  uint32_t tmem_base;
  uint32_t abort;
};
constexpr int kSmemBytes = kBarOffset + 1024 + 1024;  // + barriers + alignment slack
static_assert(sizeof(Bars) <= 1024, "barrier block size");
static_assert(kRedSum + 2048 <= kBarOffset && kEpi + 8 * 2048 <= kBarOffset && kBarOffset % 1024 == 0,
              "CTA layouts");
static_assert(kXferBytes <= kPBufStride && kXferBytes % 16 == 0, "P transfer size");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

// Sparse: the index list entries of key slots 128 t + 4 lane .. + 3 of
// sequence q (-1 past its n_slots = topk or topk_length).
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

// Score CTA: the K tile's chunk c lands at this shared-memory offset for tile
// counter tc (chunk 7 alternates between two buffers).
__device__ __forceinline__ uint32_t k_chunk_offset(int c, uint32_t tc) {
  if (c < 6) return static_cast<uint32_t>(c * kChunk);
  if (c == 6) return kKSlot2;
  if (c == 7) return kC7 + (tc & 1) * kChunk;
  return kKSlot2 + kChunk;  // c == 8: RoPE columns
}

// One CTA per SM (shared memory); up to 168 registers per thread (12 warps,
// three per sub-partition), so a row thread's 64 scores stay in registers.
// kSparse: keys are pool rows named by p.indices (DSA top-k, -1 = none), read
// with tile::gather4 (the tensor map's box is one row); otherwise pages of the
// block table, read as [64 rows x 64 columns] boxes.
template <bool kSparse>
__global__ void __launch_bounds__(kThreads, 1)
    mla_pair_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ SplitParams p) {
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
      mbar_init(smem_u32(&bars->kfull[i]), 3);  // three chunks per group
      mbar_init(smem_u32(&bars->kempty[i]), 1);
    }
    for (int b = 0; b < 2; ++b) mbar_init(smem_u32(&bars->c7empty[b]), 1);
    mbar_init(smem_u32(&bars->q_full), 8);  // one arrive per row warp
    mbar_init(smem_u32(&bars->q_free), 1);
    mbar_init(smem_u32(&bars->s_full), 1);
    mbar_init(smem_u32(&bars->s_free), 8);
    mbar_init(smem_u32(&bars->p_ready), 8);
    mbar_init(smem_u32(&bars->p_tmem_free), 1);
    mbar_init(smem_u32(&bars->o_tail_full), 1);
    for (int i = 0; i < kVGroups; ++i) {
      mbar_init(smem_u32(&bars->vfull[i]), i < kVGroups - 1 ? 2 : 1);  // chunks per quarter
      mbar_init(smem_u32(&bars->vempty[i]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars->p_free[b]), 1);
      mbar_init(smem_u32(&bars->p_full[b]), 1);
      mbar_init(smem_u32(&bars->side_read[b]), 8);
    }
    mbar_init(smem_u32(&bars->p_tmem_full), 8);
    mbar_init(smem_u32(&bars->pv_done), 1);
    mbar_init(smem_u32(&bars->o_full), 1);
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
  pdl_wait_primary();
  pdl_launch_dependents();  // the combine may launch now; it waits for this grid to finish
  // Schedule B (whole sequences) is walked when it is at most kSplitPenalty
  // tiles longer than A: every extra piece costs a Q load and an epilogue and
  // every split row a combine read.
  constexpr int kSplitPenalty = kSparse ? 5 : 11;
  // The metadata must describe this call; otherwise nothing is read or written.
  const bool meta_ok = meta_header_matches(p.meta, p.batch, p.s_q, p.num_parts, p.topk, p.causal);
  const int32_t* meta = meta_ok ? schedule_for(p.meta, kSplitPenalty) : p.meta;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    // read by the combine after this grid: the schedule walked, or -1 when
    // the metadata was rejected (the combine then writes nothing)
    p.ws_ctrl[0] = meta_ok ? (meta == p.meta ? 0 : 1) : -1;
    if (!meta_ok && p.err) atomicOr(p.err, MLA_DEVERR_METADATA);
  }
  if (meta_ok && threadIdx.x == 0 && rank == 0) {  // the first piece's query rows start towards L2
    PartCursor c0 = part_cursor(meta, part);
    int q0, a0, b0, s0;
    if (next_piece(meta, p.num_parts, &c0, &q0, &a0, &b0, &s0))
      prefetch_l2(p.q + static_cast<int64_t>(q0) * kRows * kDqk, kRows * kDqk * 2);
  }
  const uint32_t tmem = bars->tmem_base;
  volatile uint32_t* abort_flag = &bars->abort;

  if (!meta_ok) {
    // nothing to do: every role is skipped, the teardown below still runs
  } else if (rank == 0) {
    // ================================================================ score CTA
    if (warp == 0 || warp == 2 || (kSparse && warp == 3)) {
      // ---------------------------------------------------- K tile producers
      // Dense: lane 0 of warps 0, 2 loads each chunk as two page boxes.
      // Sparse: warps 0, 2, 3 share the chunks (one gather4 costs its warp
      // ~80 clk to issue, so gathers need more issuing warps); lane L gathers
      // rows 4L..4L+3 of the tile for each chunk; lane 0 owns the barriers.
      // Chunks 0..6 and 8 reuse their group's slot once that group's QK is
      // done; chunk 7 alternates between two buffers, each free once the P.V
      // tail of the tile two back has read it.
      if (lane == 0 || kSparse) {
        constexpr int kIssuers = kSparse ? 3 : 2;
        const int pw = warp == 0 ? 0 : warp - 1;
        const uint64_t pol = l2_policy_evict_first();
        PartCursor cur = part_cursor(meta, part);
        int q, t0, t1, split;
        uint32_t tc = 0;
        int32_t issued[kKGroups];  // ring round of this issuer's last load per group
        for (int i = 0; i < kKGroups; ++i) issued[i] = -1;
        bool ok = true;
        while (next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
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
            for (int c = pw; c < kChunks && ok; c += kIssuers) {
              const int g = c / 3;
              if (lane == 0) {
                // every chunk waits for its group's previous round to be consumed,
                // so no arrival can land in a phase of kfull[g] before the
                // previous phase has completed (chunk 7's own buffers are fresh
                // for the first two tiles and would not hold it back); chunk 7
                // also waits for its buffer's last P.V tail
                ok = mbar_wait(smem_u32(&bars->kempty[g]), (tc & 1) ^ 1, abort_flag, p.err);
                if (ok && c == 7)
                  ok = mbar_wait(smem_u32(&bars->c7empty[tc & 1]), ((tc >> 1) & 1) ^ 1, abort_flag, p.err);
                if (ok) mbar_arrive_expect_tx(smem_u32(&bars->kfull[g]), kChunk);
              }
              if constexpr (kSparse) ok = __shfl_sync(0xffffffffu, ok, 0);
              if (!ok) break;
              const uint32_t bar = smem_u32(&bars->kfull[g]);
              const uint32_t dst = base + k_chunk_offset(c, tc);
              if constexpr (kSparse) {
                tma_gather4(dst + 4 * lane * 128, &tm_kv, c * 64, y[0], y[1], y[2], y[3], bar);
              } else {
                tma_load_2d(dst, &tm_kv, c * 64, y[0], bar, pol);
                tma_load_2d(dst + kChunk / 2, &tm_kv, c * 64, y[1], bar, pol);
              }
              issued[g] = static_cast<int32_t>(tc);
            }
          }
        }
        if (!ok && lane == 0) {  // let this issuer's copies in flight land before the CTA exits
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
      // ---------------------------------------------------- S = Q . K^T, O tail += P . V
      // Per tile: QK of tile tc (after the row threads have loaded S of tile
      // tc - 1), then the P.V tail of tile tc - 1 (its P is ready about when
      // QK of tile tc is issued).  The last tile's tail follows the piece.
      if (lane == 0) {
        PartCursor cur = part_cursor(meta, part);
        int q, t0, t1, split;
        uint32_t tc = 0, item = 0;
        bool ok = true;
        const uint64_t rope_desc = sw128_desc(base + kQRope, 16, 1024);
        // O[:, 448:512] (+)= P(u) . chunk 7 of tile u
        auto pv_tail = [&](uint32_t u, bool first) {
          ok = mbar_wait(smem_u32(&bars->p_ready), u & 1, abort_flag, p.err);
          if (!ok) return;
          tc_fence_after();
          const uint64_t vdesc = sw128_desc(base + kC7 + (u & 1) * kChunk, kChunk, 1024);
#pragma unroll
          for (int s = 0; s < 8; ++s)
            mma_bf16_ts(tmem + kOTailCol, tmem + kPColS + 8 * s, vdesc + static_cast<uint64_t>((2048 * s) >> 4),
                        kIdescO64, (!first || s != 0) ? 1u : 0u);
          mma_commit(smem_u32(&bars->c7empty[u & 1]));
          mma_commit(smem_u32(&bars->p_tmem_free));
        };
        while (next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
          if (ok) ok = mbar_wait(smem_u32(&bars->q_full), item & 1, abort_flag, p.err);
          for (int t = t0; t < t1; ++t, ++tc) {
            if (!ok) continue;
            ok = mbar_wait(smem_u32(&bars->s_free), (tc & 1) ^ 1, abort_flag, p.err);
            if (!ok) continue;
            tc_fence_after();
            const uint32_t d = tmem + kSCol;
#pragma unroll
            for (int g = 0; g < kKGroups; ++g) {
              ok = mbar_wait(smem_u32(&bars->kfull[g]), tc & 1, abort_flag, p.err);
              if (!ok) break;
              tc_fence_after();
#pragma unroll
              for (int cc = 0; cc < 3; ++cc) {
                const int c = 3 * g + cc;
                const uint64_t bdesc = sw128_desc(base + k_chunk_offset(c, tc), 16, 1024);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const uint64_t b = bdesc + static_cast<uint64_t>((32 * k) >> 4);
                  const uint32_t acc = (c | k) != 0 ? 1u : 0u;
                  if (c < 8)  // latent columns: A = Q in TMEM
                    mma_bf16_ts(d, tmem + kQCol + 8 * (4 * c + k), b, kIdescS, acc);
                  else  // RoPE columns: A = Q's RoPE part in shared memory
                    mma_bf16_ss(d, rope_desc + static_cast<uint64_t>((32 * k) >> 4), b, kIdescS, acc);
                }
              }
              mma_commit(smem_u32(&bars->kempty[g]));  // chunk 7's buffer is released by the tail
            }
            if (!ok) continue;
            mma_commit(smem_u32(&bars->s_full));
            if (t == t1 - 1) mma_commit(smem_u32(&bars->q_free));
            if (t > t0) pv_tail(tc - 1, t - 1 == t0);
          }
          if (ok && t1 > t0) {
            pv_tail(tc - 1, t1 - 1 == t0);
            if (ok) mma_commit(smem_u32(&bars->o_tail_full));
          }
          ++item;
        }
      }
    } else if (warp >= 4) {
      // ---------------------------------------------------- Q load, softmax, P, O tail
      // Thread (h, r) owns tokens 64h .. 64h + 63 of query row r: its scores
      // are TMEM lane r, columns 64h .., so the 64 scores of a tile are loaded
      // into registers at once, which frees S for the next tile's QK.
      // Probabilities are taken against a per-row reference m (log2 units):
      // the first tile of a piece sets it to that tile's row max; a later
      // tile moves it only when a score exceeds it by more than kRescaleLog2,
      // and then O and the sums are rescaled by alpha = 2^(m_old - m_new).
      // The two threads of a row meet (named barrier 3, partial maxima in
      // shared memory) on a piece's first tile, and on a later tile only when
      // some row of the CTA has to move its reference.  Two running sums per
      // thread: of the fp32 probabilities (for the LSE) and of their bf16
      // roundings, which are the weights the PV product multiplies (to
      // normalise O); the halves add theirs at the piece's end.
      const int h = warp >= 8 ? 1 : 0;
      const int r = 32 * (warp & 3) + lane;
      const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
      const uint32_t t_q = tmem + lane_off + kQCol;
      const uint32_t t_s = tmem + lane_off + kSCol + 64 * h;
      const uint32_t t_p = tmem + lane_off + kPColS + 32 * h;
      const uint32_t t_ot = tmem + lane_off + kOTailCol + 32 * h;
      const uint32_t stage = base + kStage;
      const uint32_t prow = stage + h * 16384 + (r >> 3) * 1024 + (r & 7) * 128;  // staging chunk h, row r
      const uint32_t qrope_row = base + kQRope + (r >> 3) * 1024 + (r & 7) * 128;
      float* red_max = reinterpret_cast<float*>(smem + kRedMax);  // [parity][half][row]
      float* red_sum = reinterpret_cast<float*>(smem + kRedSum);  // [lsum, bsum][half][row]
      const float sc = p.scale_log2;
      PartCursor cur = part_cursor(meta, part);
      int q, t0, t1, split;
      uint32_t tc = 0, item = 0;
      bool ok = true;
      while (next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
        const int32_t* srec = meta_seq(meta, p.num_parts, q);
        const int32_t keys = srec[kSKeys];
        // Q row r of token q: 512 latent columns -> TMEM (bf16 pairs, even k in
        // the low half), 64 RoPE columns -> smem (128-byte swizzled row r).
        // 72 16-byte units = nine blocks of 8 (blocks 0..7 latent, block 8
        // RoPE); half 0 loads blocks 0..3, half 1 blocks 4..8, two blocks (16
        // loads in flight) per round (sparse: one).
        if (ok) ok = mbar_wait(smem_u32(&bars->q_free), (item & 1) ^ 1, abort_flag, p.err);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          tc_fence_after();
          const uint4* qrow = reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(q) * kRows + r) * kDqk);
          const int n_blk = h == 0 ? 4 : 5;  // h = 0: blocks 0..3; h = 1: blocks 4..8
          constexpr int kStep = kSparse ? 1 : 2;  // sparse keeps index registers live: one block per round
#pragma unroll 1
          for (int k = 0; k < n_blk; k += kStep) {
            const int blk = 4 * h + k;
            const bool two = kStep == 2 && k + 1 < n_blk;
            uint4 v[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = ldg_nc_v4(qrow + 8 * blk + i);
            if (two) {
#pragma unroll
              for (int i = 0; i < 8; ++i) v[8 + i] = ldg_nc_v4(qrow + 8 * (blk + 1) + i);
            }
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
              if (bb == 1 && !two) break;
              if (blk + bb < kDv / 64) {
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  w[4 * i] = v[8 * bb + i].x; w[4 * i + 1] = v[8 * bb + i].y;
                  w[4 * i + 2] = v[8 * bb + i].z; w[4 * i + 3] = v[8 * bb + i].w;
                }
                tmem_st32u(t_q + 32 * (blk + bb), w);
              } else {  // block 8: the RoPE columns
#pragma unroll
                for (int u = 0; u < 8; ++u)
                  st_shared_v4(qrope_row + ((u ^ (r & 7)) << 4), v[8 * bb + u].x, v[8 * bb + u].y,
                               v[8 * bb + u].z, v[8 * bb + u].w);
              }
            }
          }
          if (h == 0 && r == 0) {  // the next piece's query rows (147 KB, contiguous) start towards L2
            PartCursor nc = cur;
            int nq, nt0, nt1, nsplit;
            if (next_piece(meta, p.num_parts, &nc, &nq, &nt0, &nt1, &nsplit))
              prefetch_l2(p.q + static_cast<int64_t>(nq) * kRows * kDqk, kRows * kDqk * 2);
          }
          tmem_wait_st();
          fence_proxy_async_smem();
          tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->q_full));
        float m_use = 0.f, lsum = 0.f, bsum = 0.f, inv_l = 0.f;
        for (int t = t0; t < t1; ++t, ++tc) {
          // sparse: bit L of vm[k] = key slot t * 128 + 64 h + 32 k + L names a pool row
          uint32_t vm[2] = {~0u, ~0u};
          int32_t sid[2];  // sparse: requested before the S wait, used after it
          if constexpr (kSparse) {
            const int32_t* idx_row = p.indices + static_cast<int64_t>(q) * p.topk;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int slot = t * kTileTokens + 64 * h + 32 * k + lane;
              sid[k] = slot < keys ? idx_row[slot] : -1;
            }
          }
          // this thread's 64 scores of the tile, into registers; S is then free
          float s[64];
          if (ok) ok = mbar_wait(smem_u32(&bars->s_full), tc & 1, abort_flag, p.err);
          ok = __all_sync(0xffffffffu, ok);
          if (ok) {
            tc_fence_after();
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              float v[32];
              tmem_ld32(t_s + 32 * i, v);
#pragma unroll
              for (int j = 0; j < 32; ++j) s[32 * i + j] = v[j];
            }
            tmem_wait_ld();
            tc_fence_before();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->s_free));
          if constexpr (kSparse) {
#pragma unroll
            for (int k = 0; k < 2; ++k)
              vm[k] = __ballot_sync(0xffffffffu, sid[k] >= 0 && static_cast<int64_t>(sid[k]) < p.s_kv);
          }
          // masked keys: -inf by selection (keys past the end, slots naming no row)
          const int n_valid = keys - t * kTileTokens - 64 * h;  // < 64 only on the last tile
          if (!kSparse && n_valid < 64) {
#pragma unroll
            for (int j = 0; j < 64; ++j) s[j] = j < n_valid ? s[j] : -INFINITY;
          }
          if constexpr (kSparse) {
#pragma unroll
            for (int j = 0; j < 64; ++j) s[j] = (vm[j >> 5] >> (j & 31)) & 1u ? s[j] : -INFINITY;
          }
          // Row max.  The first tile of a piece sets the reference to it; a
          // later tile moves the reference only when its max exceeds it by
          // more than kRescaleLog2 (O and the sums are then rescaled by alpha).
          float alpha = 1.f;
          {
            float u = -INFINITY;
#pragma unroll
            for (int j = 0; j < 64; j += 2) u = fmax3(u, s[j], s[j + 1]);
            u *= sc;
            // a later tile meets its partner only when some row must move
            const bool meet = t == t0 || named_barrier_or(kRowExchange, kRowThreads, u > m_use + kRescaleLog2);
            if (meet) {
              float* slot = red_max + (tc & 1) * 256;
              slot[128 * h + r] = u;
              named_barrier_sync(kRowExchange, kRowThreads);
              u = fmaxf(u, slot[128 * (h ^ 1) + r]);
              if (t == t0) {
                m_use = u == -INFINITY ? 0.f : u;
              } else if (u > m_use + kRescaleLog2) {
                alpha = fast_exp2(m_use - u);
                m_use = u;
                lsum *= alpha;
                bsum *= alpha;
              }
            }
          }
          // the staging buffer is free once the previous bulk copy has read it
          if constexpr (kSparse) {
            if (h == 0 && r == 0 && tc > 0) bulk_wait_read_all();
            named_barrier_sync(1, kRowThreads);
          } else {
            named_barrier_sync(1, kXferNamedThreads);  // warp 3's previous copy has read the staging
          }
          // P in TMEM is free once the previous tile's P.V tail has read it
          if (ok) ok = mbar_wait(smem_u32(&bars->p_tmem_free), (tc & 1) ^ 1, abort_flag, p.err);
          ok = __all_sync(0xffffffffu, ok);
          // p = 2^(s * scale - m) -> bf16: this thread's 64 P values into TMEM
          // and into staging chunk h (128-byte swizzle), and the two sums
          // (tcgen05.st is warp-wide, so the warp runs this together)
          float ls = 0.f, bs = 0.f, ls2 = 0.f, bs2 = 0.f;
          if (ok) {
            tc_fence_after();
            const float neg_m = -m_use;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              // packed fp32x2 FMA/adds: one instruction per key pair
              uint32_t pk[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                float x0, x1;
                asm("{ .reg .b64 a, b, c, d; mov.b64 a, {%2, %3}; mov.b64 b, {%4, %4}; mov.b64 c, {%5, %5};"
                    " fma.rn.f32x2 d, a, b, c; mov.b64 {%0, %1}, d; }"
                    : "=f"(x0), "=f"(x1) : "f"(s[32 * i + 2 * j]), "f"(s[32 * i + 2 * j + 1]), "f"(sc), "f"(neg_m));
                const float e0 = fast_exp2(x0);
                const float e1 = fast_exp2(x1);
                pk[j] = pack_bf16x2(e0, e1);
                asm("{ .reg .b64 a, b, c; mov.b64 a, {%0, %1}; mov.b64 b, {%4, %5}; add.rn.f32x2 c, a, b; mov.b64 {%0, %1}, c;"
                    " mov.b64 a, {%2, %3}; mov.b64 b, {%6, %7}; add.rn.f32x2 c, a, b; mov.b64 {%2, %3}, c; }"
                    : "+f"(ls), "+f"(ls2), "+f"(bs), "+f"(bs2)
                    : "f"(e0), "f"(e1), "f"(__uint_as_float(pk[j] << 16)), "f"(__uint_as_float(pk[j] & 0xFFFF0000u)));
              }
              tmem_st16u(t_p + 16 * i, pk);
#pragma unroll
              for (int uu = 0; uu < 4; ++uu)
                st_shared_v4(prow + (((4 * i + uu) ^ (r & 7)) << 4), pk[4 * uu], pk[4 * uu + 1], pk[4 * uu + 2],
                             pk[4 * uu + 3]);
            }
          }
          const uint32_t any = __any_sync(0xffffffffu, alpha != 1.f) ? 1u : 0u;
          if (ok) {
            tmem_wait_st();
            // this CTA's share of O follows the reference: rescaled after the
            // previous tile's tail (p_tmem_free) and before this tile's
            if (t != t0 && any != 0u) {
              float v[32];
              tmem_ld32(t_ot, v);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] *= alpha;
              tmem_st32(t_ot, v);
              tmem_wait_st();
            }
            tc_fence_before();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->p_ready));  // this warp's P of the tile is in TMEM
          lsum += ls + ls2;
          bsum += bs + bs2;
          const bool last = t == t1 - 1;
          if (last) {
            // the two halves of the row add their sums
            red_sum[128 * h + r] = lsum;
            red_sum[256 + 128 * h + r] = bsum;
            named_barrier_sync(kRowExchange, kRowThreads);
            lsum = h == 0 ? lsum + red_sum[128 + r] : red_sum[r] + lsum;
            bsum = h == 0 ? bsum + red_sum[256 + 128 + r] : red_sum[256 + r] + bsum;
            inv_l = bsum > 0.f ? 1.f / bsum : 0.f;
            // attention sink: applied with 1/l to a final row, by the combine to a split row
            if (kSparse && p.attn_sink && srec[kSNSplits] == 1) {
              const float lse_t = (lsum > 0.f && bsum > 0.f) ? (m_use + __log2f(lsum)) * 0.69314718055994531f
                                                             : -INFINITY;
              inv_l *= attn_sink_factor(lse_t, p.attn_sink[r]);
            }
          }
          if (h == 0) {
            st_shared_f32(stage + kSideAlpha + 4 * r, alpha);
            if (last) st_shared_f32(stage + kSideInvL + 4 * r, inv_l);
            if (lane == 0) st_shared_u32(stage + kSideFlags + 4 * (warp - 4), any);
          }
          fence_proxy_async_smem();
          if constexpr (!kSparse) named_barrier_arrive(2, kXferNamedThreads);  // staging full: warp 3 copies
          if constexpr (kSparse) named_barrier_sync(2, kRowThreads);  // staging full
          if (kSparse && h == 0 && r == 0 && ok) {  // one copy of tile tc into the peer's P buffer tc mod 2
            const uint32_t b = tc & 1;
            ok = mbar_wait_cluster(smem_u32(&bars->p_free[b]), ((tc >> 1) & 1) ^ 1, abort_flag, p.err);
            if (ok) {
              bulk_copy_to_peer(mapa_shared(base + kPBuf0 + b * kPBufStride, 1), base + kStage, kXferBytes,
                                mapa_shared(smem_u32(&bars->p_full[b]), 1));
              bulk_commit_group();
            }
          }
        }
        // LSE of row r for this piece, and output columns 448 + 32h .. +31
        const float lse_v = (lsum > 0.f && bsum > 0.f) ? (m_use + __log2f(lsum)) * 0.69314718055994531f
                                                       : -INFINITY;
        if (ok) ok = mbar_wait(smem_u32(&bars->o_tail_full), item & 1, abort_flag, p.err);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          tc_fence_after();
          const bool final_out = srec[kSNSplits] == 1;
          float v[32];
          tmem_ld32(t_ot, v);
          tmem_wait_ld();
          // a row without keys (inv_l = 0) is written as exact zeros: its O
          // may hold products of zero weights with rows nobody named
          const float f = inv_l;
          if (final_out) {
            const int b = q / p.s_q, j = q % p.s_q;
            uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(q) * kRows + r) * kDv + kDvOut + 32 * h);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float* x = &v[8 * u];
              dst[u] = f != 0.f ? make_uint4(pack_bf16x2(x[0] * f, x[1] * f), pack_bf16x2(x[2] * f, x[3] * f),
                                             pack_bf16x2(x[4] * f, x[5] * f), pack_bf16x2(x[6] * f, x[7] * f))
                                : make_uint4(0u, 0u, 0u, 0u);
            }
            if (h == 0) p.lse[(static_cast<int64_t>(b) * kRows + r) * p.s_q + j] = lse_v;
          } else {
            const int64_t row = static_cast<int64_t>(srec[kSSplitOff] + split) * kRows + r;
            float4* dst = reinterpret_cast<float4*>(p.ws_o + row * kDv + kDvOut + 32 * h);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float* x = &v[4 * u];
              dst[u] = f != 0.f ? make_float4(x[0] * f, x[1] * f, x[2] * f, x[3] * f)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (h == 0) p.ws_lse[row] = lse_v;
          }
          tc_fence_before();
        }
        ++item;
      }
      if (kSparse && h == 0 && r == 0) bulk_wait_all();  // the last copy has landed in the peer
    } else if (warp == 3 && !kSparse) {
      // ---------------------------------------------------- P transfers (dense)
      PartCursor cur = part_cursor(meta, part);
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
          __syncwarp();
        }
      }
      if (lane == 0) bulk_wait_all();
    }
  } else {
    // ================================================================ output CTA
    if (warp == 0 || warp == 2 || (kSparse && warp == 3)) {
      // ---------------------------------------------------- V tile producers
      // Columns 0..447 (chunks 0..6) of each tile, as four quarters: chunk c
      // into quarter c / 2.  Dense: lane 0 of warps 0, 2 (chunk c by c mod 2).
      // Sparse: warps 0, 2, 3 gather (chunk c by issuer c mod 3).
      if (lane == 0 || kSparse) {
        constexpr int kIssuers = kSparse ? 3 : 2;
        const int pw = warp == 0 ? 0 : warp - 1;
        const uint64_t pol = l2_policy_evict_first();
        PartCursor cur = part_cursor(meta, part);
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
            for (int c = pw; c < kDvOut / 64 && ok; c += kIssuers) {
              const int qd = c >> 1;
              if (lane == 0) {
                ok = mbar_wait(smem_u32(&bars->vempty[qd]), (tc & 1) ^ 1, abort_flag, p.err);
                if (ok) mbar_arrive_expect_tx(smem_u32(&bars->vfull[qd]), kChunk);
              }
              if constexpr (kSparse) ok = __shfl_sync(0xffffffffu, ok, 0);
              if (!ok) break;
              const uint32_t bar = smem_u32(&bars->vfull[qd]);
              const uint32_t dst = base + qd * kVGroupBytes + (c & 1) * kChunk;
              if constexpr (kSparse) {
                tma_gather4(dst + 4 * lane * 128, &tm_kv, c * 64, y[0], y[1], y[2], y[3], bar);
              } else {
                tma_load_2d(dst, &tm_kv, c * 64, y[0], bar, pol);
                tma_load_2d(dst + kChunk / 2, &tm_kv, c * 64, y[1], bar, pol);
              }
              issued[qd] = static_cast<int32_t>(tc);
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
      // ---------------------------------------------------- O[:, 0:448] += P . V
      if (lane == 0) {
        PartCursor cur = part_cursor(meta, part);
        int q, t0, t1, split;
        uint32_t tc = 0;
        bool ok = true;
        while (next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
          for (int t = t0; t < t1; ++t, ++tc) {
            if (!ok) continue;
            // P of this tile in TMEM (and O rescaled, and the previous piece's
            // epilogue done: the row threads do those first)
            ok = mbar_wait(smem_u32(&bars->p_tmem_full), tc & 1, abort_flag, p.err);
            if (!ok) continue;
            tc_fence_after();
            for (int qd = 0; qd < kVGroups && ok; ++qd) {
              ok = mbar_wait(smem_u32(&bars->vfull[qd]), tc & 1, abort_flag, p.err);
              if (!ok) break;
              tc_fence_after();
              const uint64_t vdesc = sw128_desc(base + qd * kVGroupBytes, kChunk, 1024);
              const uint32_t idesc = qd < kVGroups - 1 ? kIdescO128 : kIdescO64;
#pragma unroll
              for (int s = 0; s < 8; ++s)
                mma_bf16_ts(tmem + kOCol + 128 * qd, tmem + kPColO + 8 * s,
                            vdesc + static_cast<uint64_t>((2048 * s) >> 4), idesc, (t != t0 || s != 0) ? 1u : 0u);
              mma_commit(smem_u32(&bars->vempty[qd]));
            }
            if (!ok) continue;
            mma_commit(smem_u32(&bars->pv_done));
            if (t == t1 - 1) mma_commit(smem_u32(&bars->o_full));
          }
        }
      }
    } else if (warp >= 4) {
      // ---------------------------------------------------- P into TMEM, rescale, epilogue
      // Thread (h, r): row r (TMEM lane r), P tokens 64h .. 64h + 63 and O
      // columns 224h .. 224h + 223.
      const int h = warp >= 8 ? 1 : 0;
      const int r = 32 * (warp & 3) + lane;
      const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
      const uint32_t t_o = tmem + lane_off + kOCol + (kDvOut / 2) * h;
      const uint32_t t_p = tmem + lane_off + kPColO + 32 * h;
      PartCursor cur = part_cursor(meta, part);
      int q, t0, t1, split;
      uint32_t tc = 0, item = 0;
      bool ok = true;
      while (next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
        const int32_t* srec = meta_seq(meta, p.num_parts, q);
        float inv_l = 0.f;
        for (int t = t0; t < t1; ++t, ++tc) {
          const uint32_t b = tc & 1;
          const uint32_t side = base + kPBuf0 + b * kPBufStride;
          if (ok) ok = mbar_wait_cluster(smem_u32(&bars->p_full[b]), (tc >> 1) & 1, abort_flag, p.err);
          // the previous tile's P.V is done: O holds it, P in TMEM may be rewritten
          if (ok && tc > 0) ok = mbar_wait(smem_u32(&bars->pv_done), (tc - 1) & 1, abort_flag, p.err);
          ok = __all_sync(0xffffffffu, ok);
          if (ok) {
            tc_fence_after();
            const float alpha = ld_shared_f32(side + kSideAlpha + 4 * r);
            const uint4 f = ld_shared_v4(side + kSideFlags);
            if (t == t1 - 1) inv_l = ld_shared_f32(side + kSideInvL + 4 * r);
            if (t != t0 && (f.x | f.y | f.z | f.w) != 0u && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
              for (int blk = 0; blk < kDvOut / 64; ++blk) {
                float v[32];
                tmem_ld32(t_o + 32 * blk, v);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= alpha;
                tmem_st32(t_o + 32 * blk, v);
              }
            }
            // P row r, tokens 64h .. 64h + 63: chunk h of the buffer, 8 swizzled 16-byte units
            const uint32_t prow_o = side + h * 16384 + (r >> 3) * 1024 + (r & 7) * 128;
            uint32_t w[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint4 x = ld_shared_v4(prow_o + ((u ^ (r & 7)) << 4));
              w[4 * u] = x.x; w[4 * u + 1] = x.y; w[4 * u + 2] = x.z; w[4 * u + 3] = x.w;
            }
            tmem_st32u(t_p, w);
            tmem_wait_st();
            tc_fence_before();
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_u32(&bars->p_tmem_full));
            mbar_arrive(smem_u32(&bars->side_read[b]));  // done with P buffer b
          }
          if (kSparse && warp == 4 && lane == 0 && ok && tc >= 1) {
            // hand P buffer (tc - 1) mod 2 back: every row warp has read tile
            // tc - 1's buffer; armed for tile tc + 1
            const uint32_t pb = (tc - 1) & 1, ph = ((tc - 1) >> 1) & 1;
            ok = mbar_wait(smem_u32(&bars->side_read[pb]), ph, abort_flag, p.err);
            if (ok) {
              mbar_arrive_expect_tx(smem_u32(&bars->p_full[pb]), kXferBytes);
              mbar_remote_arrive(mapa_shared(smem_u32(&bars->p_free[pb]), 0));
            }
          }
        }
        // epilogue: O row r / sum of bf16(p) -> out (single split) or fp32 partial
        if (ok) ok = mbar_wait(smem_u32(&bars->o_full), item & 1, abort_flag, p.err);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          tc_fence_after();
          // Thread (h, r) holds row r of O's columns 224h ..; each 64-byte slice
          // of the warp's 32 rows goes through a swizzled 2 KB staging area so
          // that every global store instruction writes eight whole 64-byte row
          // segments.
          const bool final_out = srec[kSNSplits] == 1;
          const int64_t row0 = (final_out ? static_cast<int64_t>(q) : static_cast<int64_t>(srec[kSSplitOff] + split)) *
                                   kRows + 32 * (warp & 3);
          const uint32_t stg = base + kEpi + (warp - 4) * 2048;
          const int rr0 = lane >> 2, uu = lane & 3;
          const int col0 = (kDvOut / 2) * h;
          if (final_out) {
#pragma unroll 1
            for (int blk = 0; blk < kDvOut / 64; ++blk) {  // 32 bf16 columns = 64 bytes per row
              float v[32];
              tmem_ld32(t_o + 32 * blk, v);
              tmem_wait_ld();
              // a row without keys (inv_l = 0) is written as exact zeros: its O
              // may hold products of zero weights with rows nobody named
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) pk[i] = inv_l != 0.f ? pack_bf16x2(v[2 * i] * inv_l, v[2 * i + 1] * inv_l) : 0u;
#pragma unroll
              for (int u = 0; u < 4; ++u)
                st_shared_v4(stg + lane * 64 + ((u ^ (lane & 3)) << 4), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2],
                             pk[4 * u + 3]);
              __syncwarp();
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int rr = 8 * j + rr0;
                const uint4 x = ld_shared_v4(stg + rr * 64 + ((uu ^ (rr & 3)) << 4));
                *reinterpret_cast<uint4*>(p.out + (row0 + rr) * kDv + col0 + 32 * blk + 8 * uu) = x;
              }
              __syncwarp();
            }
          } else {
#pragma unroll 1
            for (int blk = 0; blk < kDvOut / 32; ++blk) {  // 16 fp32 columns = 64 bytes per row
              float v[16];
              tmem_ld16(t_o + 16 * blk, v);
              tmem_wait_ld();
              if (inv_l == 0.f) {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = 0.f;
              }
#pragma unroll
              for (int u = 0; u < 4; ++u)
                st_shared_v4(stg + lane * 64 + ((u ^ (lane & 3)) << 4), __float_as_uint(v[4 * u] * inv_l),
                             __float_as_uint(v[4 * u + 1] * inv_l), __float_as_uint(v[4 * u + 2] * inv_l),
                             __float_as_uint(v[4 * u + 3] * inv_l));
              __syncwarp();
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int rr = 8 * j + rr0;
                const uint4 x = ld_shared_v4(stg + rr * 64 + ((uu ^ (rr & 3)) << 4));
                *reinterpret_cast<uint4*>(p.ws_o + (row0 + rr) * kDv + col0 + 16 * blk + 4 * uu) = x;
              }
              __syncwarp();
            }
          }
          tc_fence_before();
        }
        ++item;
      }
    } else if (warp == 3 && !kSparse) {
      // ---------------------------------------------------- P buffer hand-back
      // A P buffer is free once the four row warps have copied it into TMEM
      // (P.V reads TMEM, not the buffer); armed for the tile two ahead.
      PartCursor cur = part_cursor(meta, part);
      int q, t0, t1, split;
      uint32_t tc = 0;
      bool ok = true;
      while (next_piece(meta, p.num_parts, &cur, &q, &t0, &t1, &split)) {
        for (int t = t0; t < t1; ++t, ++tc) {
          if (lane == 0 && ok) {
            const uint32_t b = tc & 1;
            ok = mbar_wait(smem_u32(&bars->side_read[b]), (tc >> 1) & 1, abort_flag, p.err);
            if (ok) {
              mbar_arrive_expect_tx(smem_u32(&bars->p_full[b]), kXferBytes);
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
