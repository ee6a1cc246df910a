/*
 * pkv.h -- C ABI of a single-GPU paged decode-attention library (sm_103a).
 *
 * Decode-time attention over a block-paged KV cache: each sequence's tokens
 * live in fixed-size blocks of 16 token slots, found through a per-sequence
 * block table, and every decode step streams the sequence's whole visible
 * cache through the attention kernel once.
 *
 * Sources the operations follow (web pages on the paged KV cache):
 *   [MTPLX-1] "How the Paged KV Cache Works in MTPLX: Architecture and Implementation"
 *   [MTPLX-2] "How MTPLX Manages Memory Using Request-Sized Paged KV Cache"
 *   [MTPLX-3] "How MTPLX Manages Memory with KV Caching Strategies"
 *   [MLXCEL]  mlxcel manual, "KV Cache"
 *   [METAL]   metalworking, "The KV Cache"
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.   Every tensor argument is caller-owned DEVICE memory, contiguous and
 *           row-major in the shape documented beside it, and 16-byte aligned.
 *           The library allocates nothing on the device and keeps no state
 *           between calls; split-KV scratch is sized by
 *           pkv_split_workspace_bytes() and passed in by the caller.  The one
 *           exception is pkv_paged_attention_balanced_noalloc: its scratch is
 *           a static device array inside the library image that keeps the
 *           last call's contents (see its declaration for the rules).
 * Streams.  Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL
 *           is the legacy default stream).  The return value only reports the
 *           host-side argument checks and the launch itself.
 * Errors.   A call whose arguments fail the host checks returns
 *           PKV_ERR_INVALID_ARG or PKV_ERR_UNSUPPORTED and enqueues nothing;
 *           pkv_last_error() then describes the problem (per host thread).
 *           Problems only the device can see (a block id or slot out of
 *           range, a context longer than its table, a bounded wait that gave
 *           up) never trap: the affected token is skipped and a PKV_DEVERR_*
 *           bit is OR-ed into `*err_flags` when err_flags is non-NULL
 *           (caller-owned device uint32, zeroed by the caller).
 * Threads.  Stateless: calls may be made concurrently from several threads,
 *           except pkv_paged_attention_balanced_noalloc, whose calls share one
 *           array per device and must not overlap on the GPU.
 * Shapes.   block_size must be 16, head_dim 64 or 128, num_heads a multiple of
 *           num_kv_heads with a group size num_heads/num_kv_heads in
 *           {1, 2, 4, 8}.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t; no CUDA header is needed to use it. */
typedef struct CUstream_st *pkv_stream_t;

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* NULL/misaligned pointer, inconsistent sizes */
    PKV_ERR_UNSUPPORTED = 2,   /* valid request outside the compiled shapes */
    PKV_ERR_CUDA = 3           /* the kernel launch failed (see pkv_last_error) */
} pkv_status;

/* Bits OR-ed into *err_flags by the kernels. */
#define PKV_DEVERR_OOB_BLOCK 0x1u  /* a block_tables entry outside [0, num_blocks) */
#define PKV_DEVERR_OOB_SLOT 0x2u   /* a slot_mapping entry >= num_blocks * block_size */
#define PKV_DEVERR_CAPACITY 0x4u   /* a context longer than its table or partitions */
#define PKV_DEVERR_TIMEOUT 0x8u    /* a bounded pipeline wait gave up */
#define PKV_DEVERR_CASCADE 0x10u   /* a cascade member could not join its item (attended whole) */
#define PKV_DEVERR_PAGE_LIST 0x20u /* a sparse page-list entry was skipped (out of range or out of order) */

typedef enum pkv_dtype { PKV_F16 = 0, PKV_BF16 = 1, PKV_F32 = 2 } pkv_dtype;

typedef enum pkv_cache_kind {
    PKV_CACHE_F16 = 0,   /* K and V stored as fp16 */
    PKV_CACHE_BF16 = 1,  /* K and V stored as bf16 */
    PKV_CACHE_K8V4 = 2   /* K int8 symmetric, V 4-bit asymmetric (see below) */
} pkv_cache_kind;

/*
 * One layer's paged cache [MTPLX-1 §"4-D Tensor Structure": shape
 * [num_blocks, block_size, num_kv_heads, head_dim], 16 tokens per block].
 * Slot s is physical block s / 16, offset s % 16.
 *
 * PKV_CACHE_F16 / PKV_CACHE_BF16:
 *   k, v      [num_blocks, 16, num_kv_heads, head_dim]  fp16 or bf16
 *   k_scale, v_scale, v_zero unused (may be NULL)
 * PKV_CACHE_K8V4 [METAL §"The K/V asymmetry": K kept at 8 bits, V at 4;
 *   MTPLX-3 §"Quantization-Aware Allocation": per-block scale and zero
 *   tensors beside the codes], with G = head_dim / v_group (v_group = 32):
 *   k         int8  [num_blocks, 16, num_kv_heads, head_dim]   code in [-127, 127]
 *   v         uint8 [num_blocks, 16, num_kv_heads, head_dim/2] even dim in the low nibble
 *   k_scale   fp16  [num_blocks, num_kv_heads, 16]             one per (token, kv head)
 *   v_scale   fp16  [num_blocks, num_kv_heads, 16, G]          one per (token, kv head, group)
 *   v_zero    fp16  [num_blocks, num_kv_heads, 16, G]
 *   Dequantised values: k = code * k_scale;  v = code * v_scale + v_zero.
 */
typedef struct pkv_cache {
    int32_t kind;          /* pkv_cache_kind */
    int32_t num_blocks;
    int32_t block_size;    /* must be 16 */
    int32_t num_kv_heads;
    int32_t head_dim;      /* 64 or 128 */
    int32_t v_group;       /* K8V4: 32; ignored otherwise */
    void *k;
    void *v;
    void *k_scale;
    void *v_scale;
    void *v_zero;
} pkv_cache;

/*
 * The batch being decoded [MTPLX-2 §"Request-Sized Offset Tracking": each
 * request's stored-token count bounds what the kernel reads; METAL: fixed-size
 * blocks plus an indirection table].
 *   block_tables  int32 [num_seqs, max_blocks_per_seq]: logical block i of
 *                 sequence s is physical block block_tables[s][i]; entries past
 *                 ceil(context_lens[s] / 16) are never read.
 *   context_lens  int32 [num_seqs]: visible tokens of each sequence, counting the
 *                 q_len tokens being decoded (already written to the cache).
 *   q_len         query tokens per sequence: 1 for plain decode; > 1 for a
 *                 speculative verify block [MLXCEL §"Matrix-Absorbed MLA Decode",
 *                 §"Speculative Rewind"], where draft j of sequence s sees the
 *                 tokens [0, context_lens[s] - q_len + j + 1) (causal).
 *   sliding_window  0: every stored token is visible.  W > 0: only the last W
 *                 stored tokens, [max(0, context_lens[s] - W), context_lens[s]),
 *                 are visible (older ones are masked, their blocks not read)
 *                 [MTPLX-2 §"Sliding-Window Memory Control"]; the trim is of the
 *                 stored cache, so every draft row starts at the same token.
 *                 Negative: PKV_ERR_INVALID_ARG.  pkv_gather_kv_cache ignores it.
 */
typedef struct pkv_seqs {
    const int32_t *block_tables;
    const int32_t *context_lens;
    int32_t num_seqs;
    int32_t max_blocks_per_seq;
    int32_t q_len;
    int32_t sliding_window;
} pkv_seqs;

/*
 * Write new tokens' K and V into their cache slots [MLXCEL §"Attention Dispatch
 * and In-Place Decode Writes": the new row is written into the cache in place;
 * METAL names the reshape_and_cache kernel].
 *   k_new, v_new  [num_tokens, num_kv_heads, head_dim] in the cache's dtype
 *                 (PKV_CACHE_F16 or PKV_CACHE_BF16 caches only).
 *   slot_mapping  int64 [num_tokens]; a negative slot is padding and is skipped;
 *                 a slot >= num_blocks*16 is skipped and flags PKV_DEVERR_OOB_SLOT.
 * The copy is bit-exact.  num_tokens == 0 is a no-op.
 */
pkv_status pkv_reshape_and_cache(const pkv_cache *cache, const void *k_new, const void *v_new,
                                 const int64_t *slot_mapping, int32_t num_tokens,
                                 uint32_t *err_flags, pkv_stream_t stream);

/*
 * Quantise new tokens' K and V into a PKV_CACHE_K8V4 cache [METAL §"The K/V
 * asymmetry"; MTPLX-3 §"VllmMetalPagedKVCache": the quantised write path].
 *   k_new, v_new  [num_tokens, num_kv_heads, head_dim], src_dtype PKV_F16 or PKV_BF16.
 *   slot_mapping  as for pkv_reshape_and_cache.
 * The quantiser is a fixed fp32 operation sequence (IEEE division, round half
 * to even), so codes and scales are reproducible bit for bit:
 *   K: a = max|k|; s = fp16(a / 127); code = s == 0 ? 0 : clamp(rint(k / s), -127, 127)
 *   V (per group of 32 dims): s = fp16((max - min) / 15); z = fp16(min);
 *      code = s == 0 ? 0 : clamp(rint((v - z) / s), 0, 15)
 * Inputs must be finite with max|k| / 127, (max v - min v) / 15 and |min v|
 * representable in fp16; otherwise the codes are unspecified.
 */
pkv_status pkv_quantize_kv(const pkv_cache *cache, const void *k_new, const void *v_new,
                           pkv_dtype src_dtype, const int64_t *slot_mapping, int32_t num_tokens,
                           uint32_t *err_flags, pkv_stream_t stream);

/*
 * Single-pass paged decode attention [METAL: the pagedattention kernel, the GQA
 * stride trick kv_head = q_head / gqa_factor; MTPLX-2 §"Kernel Interface and
 * Memory Slicing": only the stored tokens are read].
 *   out  [num_seqs*q_len, num_heads, head_dim], out_dtype PKV_F16, PKV_BF16 or PKV_F32.
 *   q    [num_seqs*q_len, num_heads, head_dim], q_dtype PKV_F16 or PKV_BF16; for
 *        fp16/bf16 caches q_dtype must equal the cache dtype; K8V4 takes either.
 *   scale  multiplies q.k before the softmax (usually 1/sqrt(head_dim)).
 * out[r, h] = sum_t softmax_t(scale * q[r,h] . K[t, h/g]) V[t, h/g] over the
 * visible tokens of row r; a row with no visible token gets zeros.
 * Each (sequence, kv head) is handled whole by one CTA, which serves all g
 * query heads of the group, so each KV block is read from HBM once per step.
 * q_len > 1 (and the K8V4 cache) requires g * q_len <= 16.
 */
pkv_status pkv_paged_attention(void *out, pkv_dtype out_dtype, const void *q, pkv_dtype q_dtype,
                               int32_t num_heads, float scale, const pkv_cache *cache,
                               const pkv_seqs *seqs, uint32_t *err_flags, pkv_stream_t stream);

/*
 * Bytes of split-KV scratch for pkv_paged_attention_split: tmp_out
 * [num_rows, num_heads, max_partitions, head_dim] fp32 followed by max_logits
 * and exp_sums [num_rows, num_heads, max_partitions] fp32 each, each of the
 * three rounded up to 256 bytes.  Returns 0 for non-positive arguments.
 */
size_t pkv_split_workspace_bytes(int32_t num_rows, int32_t num_heads, int32_t head_dim,
                                 int32_t max_partitions);

/*
 * Split-KV paged attention, phase 1 [MLXCEL §"Paged Decode Storage and
 * Kernels": decode splits; METAL: split-KV decode kernels].  Partition p of a
 * sequence covers logical tokens [p*partition_size, (p+1)*partition_size);
 * for each row r, head h and partition p holding visible tokens it writes
 *   tmp_out[r,h,p,:]  = that partition's normalised attention output o_p,
 *   max_logits[r,h,p] = m_p, the largest scale*q.k in the partition,
 *   exp_sums[r,h,p]   = l_p = sum exp(scale*q.k - m_p),
 * and m_p = -inf, l_p = 0, o_p = 0 for a partition with no visible token of
 * that row.  Partitions at or past ceil(context_lens[s] / partition_size) are
 * not written.  partition_size must be a positive multiple of 16, and
 * max_partitions * partition_size must cover max_blocks_per_seq * 16
 * (a longer context flags PKV_DEVERR_CAPACITY).  Other arguments as for
 * pkv_paged_attention.
 */
pkv_status pkv_paged_attention_split(float *tmp_out, float *max_logits, float *exp_sums,
                                     int32_t partition_size, int32_t max_partitions,
                                     const void *q, pkv_dtype q_dtype, int32_t num_heads,
                                     float scale, const pkv_cache *cache, const pkv_seqs *seqs,
                                     uint32_t *err_flags, pkv_stream_t stream);

/*
 * Split-KV phase 2: log-sum-exp combination of the partitions written by
 * pkv_paged_attention_split, for partitions 0 .. ceil(context_lens[s] /
 * partition_size) - 1 of every row of sequence s:
 *   M = max_p m_p;  w_p = l_p * exp(m_p - M);  out = sum_p w_p o_p / sum_p w_p
 * (zeros when every l_p is 0).  The pages name the split but print no
 * combination rule; this is the identity that makes split attention equal
 * single-pass attention.
 *   out  [num_seqs*q_len, num_heads, head_dim] in out_dtype.
 */
pkv_status pkv_reduce(void *out, pkv_dtype out_dtype, const float *tmp_out,
                      const float *max_logits, const float *exp_sums, const pkv_seqs *seqs,
                      int32_t num_heads, int32_t head_dim, int32_t partition_size,
                      int32_t max_partitions, pkv_stream_t stream);

/*
 * Bytes of scratch for pkv_paged_attention_balanced: per-piece partial outputs
 * and max/sum pairs for up to 1024 CTAs plus one piece per (sequence, kv
 * head), and one int32 counter per (sequence, kv head).  Returns 0 for
 * non-positive arguments.
 */
size_t pkv_balanced_workspace_bytes(int32_t num_seqs, int32_t num_kv_heads, int32_t head_dim);

/*
 * Paged attention with split-KV partitions chosen for balance, in one launch
 * [mlxcel manual "KV Cache", §"Paged Decode Storage and Kernels": decode
 * splits; METAL: split-KV decode kernels].  Same result and arguments as
 * pkv_paged_attention; the difference is the schedule: one persistent CTA per
 * SM, and the batch's (sequence, kv head, 16-token block) list cut into equal
 * contiguous ranges, so a long sequence is spread over many SMs and a short one
 * shares an SM with its neighbours.  A (sequence, kv head) cut into pieces
 * leaves one partial per piece in `workspace`; the CTA that finishes its last
 * piece combines them with the log-sum-exp identity of pkv_reduce (an atomic
 * count decides who, nobody waits).
 *   workspace  device memory of pkv_balanced_workspace_bytes() bytes, 256-byte
 *              aligned, ZERO-FILLED before its first use; every call leaves its
 *              counters at zero again, so it can be reused without clearing by
 *              calls with the same num_seqs, num_kv_heads and head_dim (the
 *              counters' offset depends on them; clear it before a call with
 *              other sizes, and after a call that reported a device error).
 *              Calls that share one workspace must not overlap on the GPU.
 */
pkv_status pkv_paged_attention_balanced(void *out, pkv_dtype out_dtype, const void *q, pkv_dtype q_dtype,
                                        int32_t num_heads, float scale, const pkv_cache *cache,
                                        const pkv_seqs *seqs, void *workspace, size_t workspace_bytes,
                                        uint32_t *err_flags, pkv_stream_t stream);

/*
 * One decode step in one launch: the cache write of the step's new tokens
 * (pkv_reshape_and_cache, or pkv_quantize_kv for a K8V4 cache) and the balanced
 * attention of pkv_paged_attention_balanced, with the same results as those two
 * calls in that order.  This library's own arrangement of the write and the
 * read [MLXCEL §"Attention Dispatch and In-Place Decode Writes": the new row is
 * written into the cache buffer in place]; the pages print no fused call.
 *   k_new, v_new   [num_tokens, num_kv_heads, head_dim] of src_dtype (the cache
 *                  dtype for fp16/bf16 caches; PKV_F16 or PKV_BF16 for K8V4).
 *   slot_mapping   int64 [num_tokens]; < 0 skips the token.
 *   Token s*q_len + j (j < q_len) is draft j of sequence s.  When its slot is
 *   the slot of position context_lens[s] - q_len + j, the attention takes that
 *   row from k_new / v_new (quantised like the write, for K8V4) instead of
 *   waiting for the write; every other token is only written, and its slot must
 *   not be one this step's attention reads (else the read races the write).
 *   Other arguments, workspace and error reporting as for
 *   pkv_paged_attention_balanced and the write calls.
 */
pkv_status pkv_decode_step_balanced(void *out, pkv_dtype out_dtype, const void *q, pkv_dtype q_dtype,
                                    int32_t num_heads, float scale, const pkv_cache *cache, const pkv_seqs *seqs,
                                    const void *k_new, const void *v_new, pkv_dtype src_dtype,
                                    const int64_t *slot_mapping, int32_t num_tokens, void *workspace,
                                    size_t workspace_bytes, uint32_t *err_flags, pkv_stream_t stream);

/*
 * Cascade attention over shared whole-page prefixes [MLXCEL §"Paged Decode
 * Storage and Kernels": opt-in cascade attention for groups that share a
 * long whole-page prefix].  Same result as pkv_paged_attention (q_len 1, no
 * sliding window), computed so that an item's shared blocks are read once for
 * all its members.  Three launches on `stream`:
 *   set-up     one CTA checks the grouping and lists the work: the items, then
 *              every sequence from the end of its item's prefix (from 0 if it is
 *              in no item);
 *   attention  one balanced pass over that list (the schedule of
 *              pkv_paged_attention_balanced): an item's blocks are one tile
 *              stream for all its members, one query row each on tensor cores,
 *              giving each member a prefix partial; a sequence's own tokens give
 *              its other partial;
 *   reduce     the log-sum-exp combination of each row's two partials.
 *   members      int32 [num_items, item_width] device: the sequences of each
 *                item, < 0 pads.  The item's first member lends its block table.
 *   item_blocks  int32 [num_items] device: leading whole blocks the item shares.
 *                A member takes part only if its first item_blocks table entries
 *                equal the first member's, its context covers them and no other
 *                item holds it; otherwise PKV_DEVERR_CASCADE is flagged and the
 *                member is attended whole, so the output stays correct.
 *   item_width   1 .. 16 / (num_heads / num_kv_heads).
 *   workspace    pkv_cascade_workspace_bytes(...) bytes, 256-byte aligned; it
 *                needs no clearing.  Calls that share a workspace must not overlap.
 * q_len > 1 or a sliding window: PKV_ERR_UNSUPPORTED.
 */
size_t pkv_cascade_workspace_bytes(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t num_items, int32_t item_width);
pkv_status pkv_paged_attention_cascade(void *out, pkv_dtype out_dtype, const void *q, pkv_dtype q_dtype,
                                       int32_t num_heads, float scale, const pkv_cache *cache, const pkv_seqs *seqs,
                                       const int32_t *members, const int32_t *item_blocks, int32_t num_items,
                                       int32_t item_width, void *workspace, size_t workspace_bytes,
                                       uint32_t *err_flags, pkv_stream_t stream);

/*
 * Sparse page-indirection decode [MLXCEL §"Paged Decode Storage and Kernels":
 * sparse page-indirection decode, a KV-traffic deletion (METAL, "Long context
 * turns decode into a cache-streaming benchmark")].  Each sequence attends only
 * the stored tokens of the logical pages (16-token blocks) it lists; the other
 * pages are never read.  q_len 1, no sliding window.
 *   page_lists   int32 [num_seqs, max_pages] device: logical page indices in
 *                increasing order; entries past page_counts[s] are ignored; an
 *                entry outside [0, ceil(ctx / 16)) or not above the previous page
 *                taken is skipped and flags PKV_DEVERR_PAGE_LIST.
 *   page_counts  int32 [num_seqs] device.
 *   workspace    pkv_sparse_workspace_bytes(...) bytes, 256-byte aligned; needs
 *                no clearing.  Calls sharing a workspace must not overlap.
 * Two launches on `stream`: a set-up kernel compacts the listed pages' block ids
 * (one CTA per sequence), then the balanced attention streams the compacted
 * tables (it plans once the set-up has finished).  A sequence that lists no
 * page gets zeros.
 */
size_t pkv_sparse_workspace_bytes(int32_t num_seqs, int32_t num_kv_heads, int32_t head_dim, int32_t max_pages);
pkv_status pkv_paged_attention_sparse(void *out, pkv_dtype out_dtype, const void *q, pkv_dtype q_dtype,
                                      int32_t num_heads, float scale, const pkv_cache *cache, const pkv_seqs *seqs,
                                      const int32_t *page_lists, const int32_t *page_counts, int32_t max_pages,
                                      void *workspace, size_t workspace_bytes, uint32_t *err_flags,
                                      pkv_stream_t stream);

/*
 * Whether sparse page-indirection is worth using [MLXCEL §"Paged Decode Storage
 * and Kernels": a minimum sparsity gates it]: 1 if the listed pages leave out at
 * least min_sparsity of the pages of all sequences (HOST arrays: page_counts,
 * context_lens [num_seqs]), else 0.  Counts are clamped to each context's pages.
 */
int32_t pkv_sparse_worthwhile(const int32_t *page_counts, const int32_t *context_lens, int32_t num_seqs,
                              float min_sparsity);

/*
 * Host-side grouping for pkv_paged_attention_cascade [MLXCEL §"Paged Decode
 * Storage and Kernels": cascade groups gated by a minimum member count and a
 * minimum number of shared whole pages].  All pointers are HOST memory:
 *   block_tables  int32 [num_seqs, max_blocks_per_seq], context_lens int32 [num_seqs]
 *   members       out int32 [max_items, item_width], -1 pads
 *   item_blocks   out int32 [max_items]; *num_items = items written.
 * A sequence's whole pages are its first min(ctx / 16, max_blocks_per_seq)
 * blocks.  Sequences are sorted by their whole-page block ids; runs of
 * neighbours sharing >= min_shared_blocks leading blocks form groups of at least
 * max(min_members, 2), cut into near-equal items of <= item_width members (1..16),
 * each sharing the common prefix of its members.  Items past max_items are left
 * out (those sequences are attended whole).  No CUDA call; never fails on
 * valid pointers.
 */
pkv_status pkv_cascade_plan(const int32_t *block_tables, const int32_t *context_lens, int32_t num_seqs,
                            int32_t max_blocks_per_seq, int32_t min_members, int32_t min_shared_blocks,
                            int32_t item_width, int32_t max_items, int32_t *members, int32_t *item_blocks,
                            int32_t *num_items);

/* Bytes of device memory the library image reserves for
 * pkv_paged_attention_balanced_noalloc (32 MiB). */
#define PKV_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * pkv_paged_attention_balanced without a caller-provided workspace.  The pages
 * have no counterpart of this entry point: it exists for callers that cannot
 * allocate device memory themselves -- a plain C host program that links only
 * this library and owns no device allocator, or a serving loop that must not
 * allocate after start-up because its memory budget is fixed.  Its scratch is a
 * static array of PKV_NOALLOC_SCRATCH_BYTES inside the library's device image,
 * which every GPU that loads the library holds until the process exits.
 *   Limit: pkv_balanced_workspace_bytes(num_seqs, num_kv_heads, head_dim) must
 *   not exceed PKV_NOALLOC_SCRATCH_BYTES (about 3000 (sequence, kv head) pairs
 *   at head_dim 128, 6900 at head_dim 64); a larger batch returns
 *   PKV_ERR_INVALID_ARG with an explanation and launches nothing.
 *   Set-up: a call made while `stream` is not being captured looks up the
 *   array's device address in the current context (cudaGetSymbolAddress) and
 *   remembers it; a call made during stream capture uses the remembered
 *   address, so make the first call in each context (and the first after a
 *   cudaDeviceReset) before any capture, or it returns PKV_ERR_INVALID_ARG.
 *   Sharing: every call on a device uses the same array, which keeps the last
 *   call's contents; each call clears the part that must start at zero (one
 *   cudaMemsetAsync on `stream`, no allocation).  Calls that overlap on the GPU
 *   (other streams, other host threads) race on the array and give wrong
 *   results: serialise them.
 * Allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 * Arguments and result as for pkv_paged_attention_balanced.
 */
pkv_status pkv_paged_attention_balanced_noalloc(void *out, pkv_dtype out_dtype, const void *q, pkv_dtype q_dtype,
                                                int32_t num_heads, float scale, const pkv_cache *cache,
                                                const pkv_seqs *seqs, uint32_t *err_flags, pkv_stream_t stream);

/*
 * Copy every stored token of every sequence (all context_lens[s] of them; a
 * sliding window does not apply) back to contiguous storage [METAL names the
 * gather_kv_cache kernel].
 *   cu_seq_lens  int32 [num_seqs + 1] device: cu[0] = 0, cu[s+1] = cu[s] + context_lens[s].
 *   k_out, v_out [cu[num_seqs], num_kv_heads, head_dim] in the cache dtype
 *                (PKV_CACHE_F16 or PKV_CACHE_BF16 caches only).
 * Logical token t of sequence s goes to row cu[s] + t, bit-exact.  A token whose
 * block id is out of range is skipped (row left untouched) and flags
 * PKV_DEVERR_OOB_BLOCK.
 */
pkv_status pkv_gather_kv_cache(void *k_out, void *v_out, const int32_t *cu_seq_lens,
                               const pkv_cache *cache, const pkv_seqs *seqs, uint32_t *err_flags,
                               pkv_stream_t stream);

/*
 * Dequantising gather of a PKV_CACHE_K8V4 cache: every visible token of every
 * sequence to contiguous fp16 / bf16 rows, k = code * k_scale and
 * v = code * v_scale + v_zero [METAL §"The K/V asymmetry"; MTPLX-2
 * §"Quantization-Aware Memory Layout"], with the gather of pkv_gather_kv_cache.
 *   out_dtype    PKV_F16 or PKV_BF16.
 *   cu_seq_lens  int32 [num_seqs + 1] device, as for pkv_gather_kv_cache.
 *   k_out, v_out [cu[num_seqs], num_kv_heads, head_dim] of out_dtype, caller-owned,
 *                16-byte aligned.
 * Each value is formed in fp32 with one rounding (the K product is exact; V is
 * one fused multiply-add) and rounded to out_dtype to nearest even.  Errors as
 * for pkv_gather_kv_cache; a non-K8V4 cache is PKV_ERR_INVALID_ARG.
 */
pkv_status pkv_gather_kv_cache_dequant(void *k_out, void *v_out, pkv_dtype out_dtype, const int32_t *cu_seq_lens,
                                       const pkv_cache *cache, const pkv_seqs *seqs, uint32_t *err_flags,
                                       pkv_stream_t stream);

/* Static English text for a status code. */
const char *pkv_status_string(pkv_status status);

/* Description of the last non-OK status returned on this host thread ("" if none). */
const char *pkv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
