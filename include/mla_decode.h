/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) MLA decode library.
 *
 * The operation: Multi-head Latent Attention decode over an absorbed, paged
 * latent KV cache.  After weight absorption decode is MQA: h_q query heads
 * share ONE key head whose rows are 576 wide (512 latent + 64 RoPE), and V is
 * the first 512 columns of the same cached row (FlashMLA deep dive,
 * "Theoretical Analysis of the MLA Algorithm"; DeepGEMM & FlashMLA article,
 * section 6 "MLA", absorption).  For every query row (request b, new token j,
 * head h):
 *
 *     s_t  = softmax_scale * <q[b,j,h,:], K[t,:]>          (t in the key set)
 *     out  = sum_t exp(s_t - lse) * K[t, 0:512]            (bf16)
 *     lse  = ln sum_t exp(s_t)                              (fp32)
 *
 * computed as split-KV online softmax plus an LSE combine (DeepGEMM & FlashMLA
 * article, section 7 "split-KV" merge formula; FlashMLA deep dive, "tile
 * scheduler" and "programmatic dependent launch").  Calling convention
 * follows the FlashMLA README "Usage": schedule metadata once per shape, then
 * one decode call per step.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE memory owned by the caller.  The library
 *    never allocates, frees or synchronises; every launch goes on `stream`.
 *  - Return value: MLA_OK (0) or a negative MLA_ERR_* code.  Errors are
 *    detected on the host before any launch (nothing is launched then).
 *  - `err` (optional, may be NULL): a device uint32 word the kernels OR
 *    MLA_DEVERR_* bits into (bad page id, bad index, bounded-wait timeout,
 *    metadata that does not match the call).  The caller zeroes it and reads
 *    it back when it wants to.  Bad ids never fault: the row they name is
 *    masked out.
 *  - Metadata is read-only for every decode entry point.  Each decode kernel
 *    first compares the metadata header (magic, version, batch, s_q, number
 *    of parts, topk, causal) with its own arguments; on a mismatch it sets
 *    MLA_DEVERR_METADATA and returns without reading q, the cache or the
 *    page table and without writing out or lse (the combine then writes
 *    nothing either).
 *  - Row layouts (all contiguous, C order):
 *      q      [batch, s_q, h_q, 576] bf16
 *      out    [batch, s_q, h_q, 512] bf16
 *      lse    [batch, h_q, s_q]      fp32   (transposed w.r.t. out, as in the
 *                                            FlashMLA README "Return Values")
 *  - Supported shapes: d_qk = 576 (512 with the V4.1 cache, MLA_KV_FP8_528),
 *    d_v = 512, page block 64 tokens, h_q in {16, 32, 48, 64, 128},
 *    1 <= s_q <= 16.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status codes */
#define MLA_OK 0
#define MLA_ERR_NULL (-1)        /* a required pointer is NULL                 */
#define MLA_ERR_SHAPE (-2)       /* unsupported or inconsistent size argument  */
#define MLA_ERR_ALIGN (-3)       /* pointer or stride not 16-byte aligned      */
#define MLA_ERR_METADATA (-4)    /* metadata built for another shape/part count */
#define MLA_ERR_CUDA (-5)        /* a CUDA runtime call failed                 */
#define MLA_ERR_UNSUPPORTED (-6) /* device is not sm_103/sm_100 class          */

/* ------------------------------------------------ device error word (err) */
#define MLA_DEVERR_BAD_PAGE 1u   /* block_table entry outside [0, num_pages), *
                                  * or a length needing more page slots than *
                                  * block_table_stride                       */
#define MLA_DEVERR_BAD_INDEX 2u  /* sparse index < -1 or >= s_kv              */
#define MLA_DEVERR_TIMEOUT 4u    /* an internal wait ran out (kernel bailed)  */
#define MLA_DEVERR_METADATA 8u   /* metadata built for another shape (nothing *
                                  * was computed), or for other lengths      */

/* -------------------------------------------------------- KV cache formats */
#define MLA_KV_BF16 0    /* [num_pages, 64, 576] bf16, 1152 B per token        */
#define MLA_KV_FP8_656 1 /* [num_pages, 64, 656] bytes per token: 512 e4m3      *
                          * codes, 4 fp32 scales (one per 128 latent channels),  *
                          * 64 bf16 RoPE values (FlashMLA "Hopper FP8 sparse     *
                          * decode" note, "The FP8 KVCache Format")              */
#define MLA_KV_FP8_528 2 /* [num_pages, 64, 528] bytes per token, DeepSeek V4.1  *
                          * (head_dim 512): 512 e4m3 codes covering all 512      *
                          * dimensions (RoPE ones included), then 16 e8m0        *
                          * scales, one per 32 consecutive codes (FlashMLA       *
                          * README, "FP8 / FP4 KV Cache Format").  Keys are 512  *
                          * wide and the value is the whole key: q is            *
                          * [batch, s_q, h_q, 512] and out keeps 512 columns.    */

/* Human-readable name of a status code. Never NULL. */
const char* mla_status_string(int status);

/* Description of the last MLA_ERR_CUDA (or other recorded failure) raised on
 * the calling host thread: the failing call and the CUDA error text.  Never
 * NULL; the buffer is thread-local and overwritten by the next failure. */
const char* mla_last_error(void);

/*
 * Number of work parts the kernels spread over the device: one part per
 * group of ceil(h_q / 64) SMs (a part is one thread-block cluster; each
 * block of the cluster owns 64 query heads).  Writes *num_sm_parts.
 */
int mla_num_sm_parts(int device, int h_q, int* num_sm_parts);

/*
 * Size in bytes of the schedule metadata (both schedules, see
 * mla_get_metadata) for n_seq = batch * s_q query sequences and
 * num_sm_parts parts.
 */
int mla_metadata_size(int batch, int s_q, int num_sm_parts, size_t* bytes);

/*
 * Split-KV tile schedule (FlashMLA deep dive, "Tile Scheduler"; DeepGEMM &
 * FlashMLA article, section 7: computed once, reused by every layer and step
 * while shapes stay the same).  A device kernel on `stream` reads the
 * lengths and writes the int32 metadata; there is no host synchronisation.
 *
 * Each (request b, new token j) is one sequence whose key count is
 *   dense, causal:      max(0, cache_seqlens[b] - s_q + 1 + j)
 *   dense, non-causal:  cache_seqlens[b]
 *   sparse (topk > 0):  topk, or min(topk, max(0, cache_seqlens[b * s_q + j]))
 *                       when cache_seqlens is given (it is then topk_length,
 *                       one int32 per query token; may be NULL)
 * Sequences are cut into 128-key tiles.  The metadata holds two schedules
 * of W = 16 + 8 * parts + 8 * n_seq words each:
 *   A (words [0, W)): the tiles dealt out as contiguous ranges of balanced
 *     cost (tiles + 2 per sequence piece) to the parts; a sequence cut
 *     between parts becomes several splits that the combine step merges.
 *     With s_q > 1 and num_sm_parts a multiple of s_q, new token j of every
 *     request forms group j with its own cost line and num_sm_parts / s_q
 *     parts (parts [j * P/s_q, (j+1) * P/s_q)), so that the parts of the
 *     groups walk the same requests' keys at the same time;
 *   B (words [W, 2W)): present when n_seq <= num_sm_parts (else its magic is
 *     0 and the rest is not written): part p walks the whole sequence p, no
 *     sequence is split.
 * The decode kernels walk B when its largest part cost is at most a
 * kernel-specific split penalty (4 to 11 tiles) above A's balanced cost:
 * every extra piece costs a Q load and an epilogue, every split row a
 * combine read.  Layout of one schedule (int32):
 *   [0,16)                    header: magic 0x4D4C4131, version (4), n_seq,
 *                             num_sm_parts, tile_tokens (128), s_q, batch,
 *                             causal, topk, total_splits, cost_per_part,
 *                             largest sequence cost, has_b (1 in A's header
 *                             when B follows, else 0), groups, 0...
 *   [16, 16 + 8 * parts)      per part: q_begin, t_begin, q_end, t_end,
 *                             split_begin, q_step, 0, 0 (half-open range of
 *                             (sequence, tile) pairs, sequences q_begin,
 *                             q_begin + q_step, ..., q_step = groups)
 *   [.., + 8 * n_seq)         per sequence: n_tiles, split_offset, n_splits,
 *                             key count, cost prefix (within its group),
 *                             0, 0, 0
 * metadata: device buffer of mla_metadata_size() bytes, 16-byte aligned.
 */
int mla_get_metadata(const int32_t* cache_seqlens, int batch, int s_q, int causal, int topk,
                     int num_sm_parts, void* metadata, cudaStream_t stream);

/*
 * The same schedule computed on the host from host lengths into a host
 * buffer (identical bytes to mla_get_metadata).  For callers that already
 * hold the lengths on the host, and for testing the device schedule.
 */
int mla_get_metadata_host(const int32_t* cache_seqlens_host, int batch, int s_q, int causal,
                          int topk, int num_sm_parts, void* metadata_host);

/*
 * Size in bytes of the split workspace: fp32 partial outputs
 * [batch*s_q + num_sm_parts, h_q, 512], fp32 partial LSEs
 * [batch*s_q + num_sm_parts, h_q], then 64 bytes of control words (the
 * split kernel records there which of the metadata's two schedules it
 * walked and whether that schedule left rows to merge or fill; mla_combine
 * reads them).  One workspace serves one call at a time.
 */
int mla_workspace_size(int batch, int s_q, int h_q, int num_sm_parts, size_t* bytes);

/*
 * Dense paged decode (FlashMLA README "Usage": flash_mla_with_kvcache with
 * q, kvcache, block_table, cache_seqlens).  Runs the split-KV kernel and then
 * the combine kernel (programmatic dependent launch) on `stream`.
 *
 *  q            [batch, s_q, h_q, 576] bf16 ([.., 512] with MLA_KV_FP8_528)
 *  kv_cache     MLA_KV_BF16: [num_pages, 64, 576] bf16;
 *               MLA_KV_FP8_656: [num_pages, 64, 656] uint8;
 *               MLA_KV_FP8_528: [num_pages, 64, 528] uint8 (the value of a
 *               token is its whole 512-wide key)
 *  block_table  [batch, block_table_stride] int32; entry [b, p] = physical
 *               page of tokens 64p .. 64p+63 of request b.  Only the first
 *               ceil(cache_seqlens[b] / 64) entries of a row are read, and
 *               never more than block_table_stride of them: a length that
 *               needs more page slots than the row has sets
 *               MLA_DEVERR_BAD_PAGE, and the keys of the missing slots are
 *               masked out like those of a bad page id.
 *  cache_seqlens [batch] int32, cached tokens per request (new tokens
 *               included).  With causal != 0 and s_q > 1, new token j sees
 *               keys 0 .. cache_seqlens[b] - s_q + j.  The key counts come
 *               from the metadata; the kernel compares them with the ones
 *               cache_seqlens and causal give and sets MLA_DEVERR_METADATA
 *               on a difference (metadata computed from other lengths).
 *  Cache slots past a request's length inside its last page must hold
 *  finite values (they are masked, but multiply a zero weight).
 *  metadata     from mla_get_metadata(cache_seqlens, batch, s_q, causal, 0,
 *               num_sm_parts, ...) on the same lengths; read-only.
 *  workspace    mla_workspace_size() bytes, 16-byte aligned.
 *  out, lse     outputs as described at the top of this file.  A query row
 *               with no visible key gets out = 0, lse = -inf.
 */
int mla_decode(const void* q, const void* kv_cache, int kv_format, int64_t num_pages,
               const int32_t* block_table, int64_t block_table_stride,
               const int32_t* cache_seqlens, int batch, int s_q, int h_q, float softmax_scale,
               int causal, const void* metadata, int num_sm_parts, void* workspace, void* out,
               float* lse, uint32_t* err, cudaStream_t stream);

/*
 * The split-KV kernel of mla_decode alone (FlashMLA deep dive: the
 * splitkv_mla kernel, before combine).  Same arguments and layouts.  Query
 * rows whose keys fall in one split get their final out/lse here; rows cut
 * into several splits get fp32 partials in `workspace`, merged by a
 * following mla_combine on the same metadata and workspace.
 */
int mla_decode_splitkv(const void* q, const void* kv_cache, int kv_format, int64_t num_pages,
                       const int32_t* block_table, int64_t block_table_stride,
                       const int32_t* cache_seqlens, int batch, int s_q, int h_q,
                       float softmax_scale, int causal, const void* metadata, int num_sm_parts,
                       void* workspace, void* out, float* lse, uint32_t* err,
                       cudaStream_t stream);

/*
 * DSA top-k sparse decode (FlashMLA README, "indices Tensor"): each query
 * token attends only to the pool rows its index list names.
 *
 *  kv       [s_kv, 576] bf16 pool of latent rows (a paged cache viewed flat:
 *           row = page * 64 + offset)
 *  indices  [batch, s_q, topk] int32; -1 marks an invalid slot.  Any other
 *           value outside [0, s_kv) is also skipped and sets
 *           MLA_DEVERR_BAD_INDEX (FlashMLA itself does no bound check).
 *           Only rows a query token names are ever read for it: an invalid
 *           slot is loaded from a row the token does name (its weight is
 *           0), so the contents of unnamed pool rows (NaN included) never
 *           reach the output.  A token that names no row gets out = 0 and
 *           lse = -inf.
 *  attn_sink optional [h_q] fp32 device array (NULL = none; FlashMLA sparse
 *           interface, "attn_sink"): every output row of head h is scaled
 *           by exp(lse) / (exp(lse) + exp(attn_sink[h])); lse itself is
 *           returned unchanged.
 *  metadata from mla_get_metadata(topk_length, batch, s_q, 0, topk,
 *           num_sm_parts, ...).  topk_length (FlashMLA sparse interface,
 *           "topk_length") is NULL, or an int32 device array [batch * s_q]:
 *           query token (b, j) then attends only to its first
 *           topk_length[b * s_q + j] index slots (clamped to [0, topk]).
 *  Other arguments as for mla_decode.  Invariant to the order of indices up
 *  to floating-point rounding.
 */
int mla_sparse_decode(const void* q, const void* kv, int64_t s_kv, const int32_t* indices,
                      int topk, int batch, int s_q, int h_q, float softmax_scale,
                      const float* attn_sink, const void* metadata, int num_sm_parts, void* workspace,
                      void* out, float* lse, uint32_t* err, cudaStream_t stream);

/*
 * The split-KV kernel of mla_sparse_decode alone (the sparse counterpart of
 * mla_decode_splitkv).  Same arguments and layouts; rows whose keys were cut
 * into several splits need a following mla_combine on the same metadata and
 * workspace.
 */
int mla_sparse_decode_splitkv(const void* q, const void* kv, int64_t s_kv, const int32_t* indices,
                              int topk, int batch, int s_q, int h_q, float softmax_scale,
                              const float* attn_sink, const void* metadata, int num_sm_parts,
                              void* workspace, void* out, float* lse, uint32_t* err,
                              cudaStream_t stream);

/*
 * DSA sparse prefill (FlashMLA README, "DeepSeek Sparse Attention (DSA)
 * Prefill", flash_mla_sparse_fwd): s_q query tokens, each attending to the
 * pool rows its own index list names.  The same computation as
 * mla_sparse_decode with each query token as a request of one token
 * (batch = s_q, s_q = 1), and run by the same kernels; only the argument
 * shapes follow the prefill interface:
 *
 *  q        [s_q, h_q, 576] bf16
 *  kv       [s_kv, h_kv = 1, 576] bf16 pool (MLA: one latent row per token)
 *  indices  [s_q, h_kv = 1, topk] int32; -1 marks an invalid slot (other
 *           out-of-range values are skipped and flagged as for
 *           mla_sparse_decode)
 *  softmax_scale  the pages' sm_scale; d_v is 512, the only value they allow
 *  attn_sink optional [h_q] fp32 (NULL = none), as for mla_sparse_decode
 *  metadata from mla_get_metadata(topk_length, s_q, 1, 0, topk,
 *           num_sm_parts, ...); topk_length is NULL or an int32 device
 *           array [s_q]: token i attends only to its first topk_length[i]
 *           slots (clamped to [0, topk])
 *  workspace mla_workspace_size(s_q, 1, h_q, num_sm_parts) bytes
 *  out      [s_q, h_q, 512] bf16
 *  lse      [s_q, h_q] fp32 natural-log LSE (the pages' return-value text
 *           for this call is cut off; this is the decode call's
 *           [batch, h_q, seq_len_q] with one query token per batch entry)
 *
 * Errors, streams and ownership as for mla_sparse_decode.
 */
int mla_sparse_prefill(const void* q, const void* kv, int64_t s_kv, const int32_t* indices, int topk,
                       int s_q, int h_q, float softmax_scale, const float* attn_sink,
                       const void* metadata, int num_sm_parts, void* workspace, void* out,
                       float* lse, uint32_t* err, cudaStream_t stream);

/*
 * Failure-path check (no counterpart on the pages): launches one thread that
 * waits on a shared-memory barrier nothing ever completes, through the same
 * bounded wait every kernel of this library uses.  The wait gives up after
 * its limit (2 s), ORs MLA_DEVERR_TIMEOUT into *err (device memory) and the
 * kernel exits normally, so the context stays usable; no GPU fault, trap or
 * hang is involved.  Asynchronous on `stream`; returns MLA_ERR_NULL for a
 * NULL err, MLA_ERR_CUDA if the launch fails.
 */
int mla_check_wait_timeout(uint32_t* err, cudaStream_t stream);

/* Size of the device scratch array that mla_decode_noalloc uses (40 MiB). */
#define MLA_NOALLOC_SCRATCH_BYTES (40u * 1024u * 1024u)

/*
 * mla_decode without caller-provided scratch.  The source pages have no
 * counterpart to this entry point; it exists for callers that may launch
 * kernels but may not allocate device memory where they call it, such as an
 * inference engine's plugin enqueue hook that is handed only input/output
 * pointers and a stream, or a serving loop that must not hit cudaMalloc and
 * its implicit synchronisation.
 *
 * Arguments and layouts are those of mla_decode minus metadata, num_sm_parts
 * and workspace: the schedule and the split workspace go to a library-owned
 * device array of MLA_NOALLOC_SCRATCH_BYTES, and num_sm_parts is the
 * current device's default (mla_num_sm_parts).  Nothing is allocated and the
 * caller still passes every input and output.
 *
 *  - Limit: shapes whose metadata (rounded up to 256 bytes) plus workspace
 *    (mla_metadata_size + mla_workspace_size) exceed the array are rejected
 *    with MLA_ERR_SHAPE before any launch; mla_last_error() says why.  The
 *    b=64, s_q=1, h_q=128 decode fits; use mla_decode for larger batches.
 *  - The array exists once per device that loads this library and stays
 *    reserved until the process exits.
 *  - The first call in a CUDA context looks up the array's address in that
 *    context (the array is per context: a context created after
 *    cudaDeviceReset, or another context the caller made current, has its
 *    own copy) and caches it per context; make that first call before any
 *    stream capture.
 *  - Every call shares the array: calls that overlap on the GPU (other
 *    streams, other host threads on the same device) race and corrupt each
 *    other's results.  Nothing in it needs clearing between calls: every
 *    call rewrites the schedule and the control word before reading them.
 */
int mla_decode_noalloc(const void* q, const void* kv_cache, int kv_format, int64_t num_pages,
                       const int32_t* block_table, int64_t block_table_stride,
                       const int32_t* cache_seqlens, int batch, int s_q, int h_q,
                       float softmax_scale, int causal, void* out, float* lse, uint32_t* err,
                       cudaStream_t stream);

/*
 * LSE combine of split partials (DeepGEMM & FlashMLA article, section 7:
 * m = max m_i, l = sum l_i e^(m_i - m), o = sum o_i l_i e^(m_i - m) / l; here
 * with lse_i = m_i + ln l_i and o_i already divided by l_i).  mla_decode and
 * mla_sparse_decode launch it themselves; it is exported for callers that
 * run the split kernels through their own graph.  Writes out/lse for every
 * sequence with two or more splits, and zeros / -inf for empty sequences.
 * attn_sink: as for mla_sparse_decode (NULL for dense decode).
 */
int mla_combine(const void* metadata, int batch, int s_q, int h_q, int num_sm_parts,
                const void* workspace, const float* attn_sink, void* out, float* lse,
                cudaStream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* MLA_DECODE_H_ */
