// Split-KV tile schedule shared by the metadata kernel, its host mirror and
// the decode kernels.  Pure integer arithmetic, compiled for host and device.
//
// Each (request b, new token j) is a sequence q = b * s_q + j whose keys are
// cut into 128-key tiles.  A sequence piece costs its tiles plus kFixedCost
// (the Q load and the epilogue).  The metadata holds two schedules (FlashMLA
// deep dive, "Tile Scheduler": balanced assignment of requests and blocks to
// SMs; DeepGEMM & FlashMLA article, section 7 "split-KV"):
//   A: the cost line cut into equal ranges, so a sequence may be split
//      between parts (its splits are merged by the combine).  With s_q > 1
//      new tokens per request (and num_parts a multiple of s_q), token j of
//      every request forms group j with its own cost line and num_parts / s_q
//      parts: part p of group 0 and part p of group j walk the same requests
//      in step, so one of them finds the other's cache rows still in L2;
//   B: (only when n_seq <= num_parts) part p walks the whole sequence p, so
//      nothing is split and the combine has nothing to merge.
// A decode kernel walks B when B's longest part costs at most its own split
// penalty more than A's balanced part: every extra piece pays a Q load and
// an epilogue, and every split row a combine read.  The metadata is read-only
// for the decode kernels; the schedule a call walked is recorded in that
// call's workspace (workspace_ctrl) for the combine.
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define MLA_HD __host__ __device__ __forceinline__
#else
#define MLA_HD inline
#endif

namespace mla {

constexpr int kTileTokens = 128;
constexpr int kFixedCost = 2;  // a piece switch (Q load, epilogue) costs about two tiles
constexpr int32_t kMetaMagic = 0x4D4C4131;  // "MLA1"
constexpr int32_t kMetaVersion = 4;

// header words (kHMaxCost: the largest single-sequence cost; kHHasB: 1 in
// schedule A's header when schedule B follows it, so a decode kernel makes its
// choice from the header's one cache line; kHGroups: the number of groups of
// schedule A, 1 or s_q)
enum : int {
  kHMagic = 0, kHVersion, kHNSeq, kHParts, kHTile, kHSq, kHBatch, kHCausal, kHTopk,
  kHTotalSplits, kHPerPart, kHMaxCost, kHHasB, kHGroups, kHeaderWords = 16
};
// q_begin, t_begin, q_end, t_end, split_begin, q_step, 0, 0: the part walks
// sequences q_begin, q_begin + q_step, ... (q_step = the number of groups)
constexpr int kPartWords = 8;
constexpr int kSeqWords = 8;   // n_tiles, split_offset, n_splits, keys, cost_prefix, 0, 0, 0
enum : int { kSTiles = 0, kSSplitOff, kSNSplits, kSKeys, kSCostPrefix };

MLA_HD int64_t meta_words(int n_seq, int num_parts) {
  return kHeaderWords + static_cast<int64_t>(kPartWords) * num_parts +
         static_cast<int64_t>(kSeqWords) * n_seq;
}
// Both schedules: A at word 0, B right after it.
MLA_HD int64_t meta_total_words(int n_seq, int num_parts) { return 2 * meta_words(n_seq, num_parts); }
MLA_HD int32_t* meta_part(int32_t* m, int p) { return m + kHeaderWords + kPartWords * p; }
MLA_HD const int32_t* meta_part(const int32_t* m, int p) {
  return m + kHeaderWords + kPartWords * p;
}
MLA_HD int32_t* meta_seq(int32_t* m, int num_parts, int q) {
  return m + kHeaderWords + kPartWords * num_parts + kSeqWords * q;
}
MLA_HD const int32_t* meta_seq(const int32_t* m, int num_parts, int q) {
  return m + kHeaderWords + kPartWords * num_parts + kSeqWords * q;
}

// Key count of sequence (b, j).  Sparse (topk > 0): topk, or, when lengths
// are given, the first topk_length[b * s_q + j] index slots (clamped to
// [0, topk]; FlashMLA sparse interface, "topk_length").
MLA_HD int32_t seq_keys(const int32_t* seqlens, int b, int j, int s_q, int causal, int topk) {
  if (topk > 0) {
    if (!seqlens) return topk;
    const int32_t n = seqlens[b * s_q + j];
    return n < 0 ? 0 : (n > topk ? topk : n);
  }
  int32_t L = seqlens[b];
  if (L < 0) L = 0;
  if (causal) {
    L = L - s_q + 1 + j;
    if (L < 0) L = 0;
  }
  return L;
}

MLA_HD int32_t tiles_of(int32_t keys) { return (keys + kTileTokens - 1) / kTileTokens; }
MLA_HD int32_t cost_of(int32_t n_tiles) { return n_tiles > 0 ? n_tiles + kFixedCost : 0; }

MLA_HD int64_t floordiv(int64_t a, int64_t b) {  // b > 0
  if (a >= 0 && a <= 0x7fffffff && b <= 0x7fffffff)  // the usual case: a 32-bit division
    return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
  return a >= 0 ? a / b : -((-a + b - 1) / b);
}

// Cost prefix of sequence q read from the metadata's sequence records, or from
// a copy of those prefixes (the device schedule keeps one in shared memory).
struct MetaPrefix {
  const int32_t* meta;
  int num_parts;
  MLA_HD int32_t operator()(int q) const { return meta_seq(meta, num_parts, q)[kSCostPrefix]; }
};
struct ArrayPrefix {
  const int32_t* a;
  MLA_HD int32_t operator()(int q) const { return a[q]; }
};

// Position (q, t) of cost offset x: q is the sequence whose cost range
// [prefix[q], prefix[q] + cost[q]) contains x; t is the tile at that offset
// (offsets inside the fixed cost map to tile 0).  x >= total maps to (n_seq, 0).
template <class Prefix>
MLA_HD void cost_position(const Prefix& prefix, int n_seq, int64_t total, int64_t x, int* q_out,
                          int* t_out) {
  if (x >= total) {
    *q_out = n_seq;
    *t_out = 0;
    return;
  }
  int lo = 0, hi = n_seq - 1;
  while (lo < hi) {  // largest q with prefix[q] <= x
    const int mid = (lo + hi + 1) >> 1;
    if (prefix(mid) <= x) lo = mid; else hi = mid - 1;
  }
  const int64_t local = x - prefix(lo);
  *q_out = lo;
  *t_out = static_cast<int>(local > kFixedCost ? local - kFixedCost : 0);
}

// Number of part boundaries p*per_part that fall strictly inside the tiles of
// a sequence with cost prefix `prefix` and `n_tiles` tiles (tile index >= 1).
MLA_HD int32_t inner_boundaries(int64_t prefix, int32_t n_tiles, int64_t per_part) {
  if (n_tiles <= 1) return 0;
  const int64_t lo = prefix + kFixedCost + 1;          // first offset with tile >= 1
  const int64_t hi = prefix + kFixedCost + n_tiles;    // one past the last offset
  return static_cast<int32_t>(floordiv(hi - 1, per_part) - floordiv(lo - 1, per_part));
}

// Groups of schedule A: s_q (one per new-token index j) when s_q > 1 and the
// parts divide evenly, else 1.  Group j's members are the sequences
// q = j + groups * m, m = 0 .. n_seq / groups - 1, in that order; the
// metadata builders walk all sequences in group-major order k = j * n_g + m.
MLA_HD int schedule_groups(int s_q, int num_parts) {
  return (s_q > 1 && num_parts % s_q == 0) ? s_q : 1;
}
MLA_HD int order_to_q(int k, int n_g, int groups) { return (k % n_g) * groups + k / n_g; }

// Cost prefix of member m of group j, from a per-sequence prefix functor.
template <class Prefix>
struct GroupPrefix {
  Prefix prefix;
  int j, groups;
  MLA_HD int32_t operator()(int m) const { return prefix(j + groups * m); }
};

// Fills the record of part p (the p_local-th part of group j, whose members
// have cost prefixes `prefix` within the group's cost line of length total).
template <class Prefix>
MLA_HD void fill_part(int32_t* meta, const Prefix& prefix, int n_members, int64_t total, int64_t per_part,
                      int p, int p_local, int j, int groups) {
  int mb, tb, me, te;
  const int64_t xb = static_cast<int64_t>(p_local) * per_part;
  int64_t xe = xb + per_part;
  if (xe > total) xe = total;
  cost_position(prefix, n_members, total, xb, &mb, &tb);
  cost_position(prefix, n_members, total, xe, &me, &te);
  int32_t split_begin = 0;
  if (mb < n_members && tb > 0)
    split_begin = static_cast<int32_t>(p_local - floordiv(prefix(mb) + kFixedCost, per_part));
  int32_t* r = meta_part(meta, p);
  r[0] = j + groups * mb; r[1] = tb; r[2] = j + groups * me; r[3] = te; r[4] = split_begin;
  r[5] = groups; r[6] = 0; r[7] = 0;
}

// Schedule B of a metadata buffer (its magic is 0 when it does not exist).
MLA_HD const int32_t* schedule_b(const int32_t* meta) {
  return meta + meta_words(meta[kHNSeq], meta[kHParts]);
}
MLA_HD int32_t* schedule_b(int32_t* meta) { return meta + meta_words(meta[kHNSeq], meta[kHParts]); }

// The schedule a decode kernel with split penalty `penalty` (tile units)
// walks: B when it exists and costs at most `penalty` more than A.
MLA_HD bool choose_whole_sequences(const int32_t* meta, int penalty) {
  return meta[kHHasB] == 1 &&
         static_cast<int64_t>(meta[kHMaxCost]) <= static_cast<int64_t>(meta[kHPerPart]) + penalty;
}
MLA_HD const int32_t* schedule_for(const int32_t* meta, int penalty) {
  return choose_whole_sequences(meta, penalty) ? schedule_b(meta) : meta;
}

// The work a part walks: pieces (q, [t0, t1), split index) in order.
struct PartCursor {
  int q, t, q_end, t_end, split, step;
};

// Schedule B's part p walks sequence p (none when p >= n_seq).
MLA_HD PartCursor whole_part_cursor(int n_seq, int p) {
  PartCursor c;
  c.q = p < n_seq ? p : n_seq; c.t = 0; c.q_end = p < n_seq ? p + 1 : n_seq; c.t_end = 0;
  c.split = 0; c.step = 1;
  return c;
}

// Schedule B's records.
MLA_HD void fill_whole_part(int32_t* meta_b, int num_parts, int n_seq, int p) {
  int32_t* r = meta_part(meta_b, p);
  const PartCursor c = whole_part_cursor(n_seq, p);
  r[0] = c.q; r[1] = c.t; r[2] = c.q_end; r[3] = c.t_end; r[4] = c.split;
  r[5] = c.step; r[6] = 0; r[7] = 0;
}

MLA_HD PartCursor part_cursor(const int32_t* meta, int p) {
  const int32_t* r = meta_part(meta, p);
  PartCursor c;
  c.q = r[0]; c.t = r[1]; c.q_end = r[2]; c.t_end = r[3]; c.split = r[4]; c.step = r[5];
  return c;
}

// The cursor of part p in `walked`, the schedule of metadata `meta_a` that a
// kernel walks: schedule B's is known from the header without a read.
MLA_HD PartCursor walked_part_cursor(const int32_t* meta_a, const int32_t* walked, int p) {
  return walked != meta_a ? whole_part_cursor(meta_a[kHNSeq], p) : part_cursor(walked, p);
}

// Advances to the next non-empty piece.  Returns false when the part is done.
MLA_HD bool next_piece(const int32_t* meta, int num_parts, PartCursor* c, int* q, int* t0,
                       int* t1, int* split) {
  while (c->q < c->q_end || (c->q == c->q_end && c->t < c->t_end)) {
    const int32_t n_tiles = meta_seq(meta, num_parts, c->q)[kSTiles];
    const int stop = (c->q == c->q_end) ? c->t_end : n_tiles;
    if (n_tiles > 0 && c->t < stop) {
      *q = c->q; *t0 = c->t; *t1 = stop; *split = c->split;
      c->q += c->step; c->t = 0; c->split = 0;
      return true;
    }
    c->q += c->step; c->t = 0; c->split = 0;
  }
  return false;
}

// True when the header of `meta` describes the call: the same magic and
// version, sequence count, part count, tile size, tokens per request and
// batch; for sparse calls (topk > 0) the same topk, for dense calls topk 0
// and the same causal flag.  A decode kernel that gets metadata built for
// another shape would index q, out and the page table with that shape's
// sequence numbers, so the kernels check this before touching any input.
MLA_HD bool meta_header_matches(const int32_t* meta, int batch, int s_q, int num_parts, int topk,
                                int causal) {
  if (meta[kHMagic] != kMetaMagic || meta[kHVersion] != kMetaVersion) return false;
  if (meta[kHNSeq] != batch * s_q || meta[kHParts] != num_parts || meta[kHTile] != kTileTokens)
    return false;
  if (meta[kHSq] != s_q || meta[kHBatch] != batch || meta[kHTopk] != topk) return false;
  return topk > 0 || meta[kHCausal] == (causal ? 1 : 0);
}

}  // namespace mla
