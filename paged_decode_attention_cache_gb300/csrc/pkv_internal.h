// pkv_internal.h -- parameter blocks and launchers shared between the C-ABI
// layer (api.cu) and the kernel translation units.  Host-side only types.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Kernel launch with programmatic stream serialisation: the kernel may start
// while the previous kernel of the stream is finishing, and waits on the device
// (griddepcontrol.wait) before it touches memory that kernel could write.
// PKV_PDL=0 in the environment launches without the attribute.
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Everything the attention kernels read besides the two tensor maps.
struct AttnParams {
    // outputs: exactly one of {out} or {tmp_out, max_logits, exp_sums} is set
    void* out;
    int32_t out_dtype;
    float* tmp_out;
    float* max_logits;
    float* exp_sums;
    int32_t partition_blocks;  // 16-token blocks per partition (whole table for single pass)
    int32_t max_partitions;    // partitions per row in tmp_out (1 for single pass)
    // queries
    const void* q;
    int32_t q_dtype;
    float scale_log2;  // scale * log2(e): scores are kept in base-2 units
    int32_t num_heads;
    int32_t num_kv_heads;
    int32_t q_len;
    // cache
    int32_t num_blocks;
    int32_t head_dim;
    const void* k_scale;  // K8V4 metadata
    const void* v_scale;
    const void* v_zero;
    // sequences
    const int32_t* block_tables;
    const int32_t* context_lens;
    int32_t num_seqs;
    int32_t max_blocks;
    int32_t window;     // sliding window in tokens, 0 = none
    uint32_t* err;
    // persistent scheduling
    int32_t mode;       // kModeSingle / kModeSplit / kModeBalanced
    int32_t stages;     // shared-memory ring depth (a multiple of the consumer warps)
    int32_t min_chunk;  // balanced: fewest 16-token blocks a CTA is given
    int32_t seg_cost;   // balanced: blocks' worth of time one more segment costs a CTA
    // fused decode step: the cache write of the step's new tokens in the same launch
    void* kc;                      // the cache's K / V code arrays (written by the fused step)
    void* vc;
    const void* k_new;             // [num_new, num_kv_heads, head_dim], src_dtype
    const void* v_new;
    const int64_t* slot_mapping;   // [num_new]
    int32_t num_new;               // 0: attention only
    int32_t src_dtype;
    // cascade attention [one pass over a list of num_items items, then the
    // sequences]: entry s of the list reads the block table of sequence
    // item_seq[s] from token seq_start[s] on, for query rows row_map[s * q_len + j]
    // (< 0: none); an item's partials go to partition part_offset + part
    const int32_t* row_map;
    const int32_t* item_seq;
    const int32_t* seq_start;
    int32_t num_items;
    int32_t part_offset;
    // 1: block_tables / context_lens come from the previous kernel (the sparse
    // set-up), so the kernel waits for it before planning
    int32_t wait_first;
    // timeline build only (PKV_TIMELINE): per-CTA %globaltimer stamps, see
    // attention_impl.cuh; null otherwise
    unsigned long long* timeline;
    float* part_o;      // balanced workspace: [slots, 16, head_dim] unnormalised partial outputs
    float* part_ml;     // [slots, 16, 2] (max, sum) in base-2 units
    int32_t* counters;  // [num_seqs * num_kv_heads] pieces finished per (sequence, kv head)
};

constexpr int kModeSingle = 0;
constexpr int kModeSplit = 1;
constexpr int kModeBalanced = 2;
constexpr int kMaxGrid = 1024;  // CTAs of a persistent launch (bounds the balanced workspace)
// Balanced schedule: a CTA gets at least kMinChunk blocks, and starting one more
// (sequence, kv head) segment is charged as kSegCost blocks (its merge and
// combine take about as long as streaming that many blocks).
constexpr int kBlockSize = 16;   // token slots per cache block
constexpr int kMinChunk = 8;
constexpr int kSegCost = 24;

// Persistent attention kernel (attention.cu): one CTA per SM at most, the
// (sequence, kv head, block) work list split into contiguous ranges.
bool attention_supported(int cache_kind, int head_dim, int gqa, int q_len);
// Tensor-core maths for K8/V4, for cascade passes and whenever a kv head serves
// at least kTcMinRows query rows (group size x q_len); the CUDA-core math for
// fp16/bf16 below that (group size 1 or 2 decode).
constexpr int kTcMinRows = 4;
bool attention_uses_tensor_cores(int cache_kind, int q_len, int gqa, bool cascade_pass = false);
// A pass of cascade attention: its own kernel instantiation (attention_cascade.cu)
inline bool is_cascade_pass(const AttnParams& p) { return p.seq_start != nullptr || p.row_map != nullptr; }
cudaError_t launch_attention(AttnParams p, int cache_kind, int gqa, const CUtensorMap& k_map,
                             const CUtensorMap& v_map, cudaStream_t stream);
// The fused decode step's kernels (attention_fused.cu); launch_attention calls
// it when p.num_new > 0.
cudaError_t launch_attention_cascade(AttnParams p, int cache_kind, int gqa, const CUtensorMap& km,
                                     const CUtensorMap& vm, cudaStream_t stream);
cudaError_t launch_attention_fused(AttnParams p, int cache_kind, int gqa, const CUtensorMap& km, const CUtensorMap& vm,
                                   cudaStream_t stream);
size_t balanced_workspace_bytes(int num_seqs, int num_kv_heads, int head_dim);

struct ReduceParams {
    void* out;
    int32_t out_dtype;
    const float* tmp_out;
    const float* max_logits;
    const float* exp_sums;
    const int32_t* context_lens;
    int32_t num_seqs;
    int32_t q_len;
    int32_t num_heads;
    int32_t head_dim;
    int32_t partition_size;
    int32_t max_partitions;
    int32_t window;     // sliding window in tokens, 0 = none
    // cascade (max_partitions 2): slot 0 of row s holds its own partial, slot 1
    // its item's when seq_start[s] > 0; null: not a cascade
    const int32_t* seq_start;
};
cudaError_t launch_reduce(const ReduceParams& p, cudaStream_t stream);

// Cascade set-up (one CTA): the pass's list -- items first, then the sequences
// -- with each entry's context, lending table, first token and query rows; a
// member joins its item only if its table holds the item's shared blocks, its
// context covers them and no other item holds it (else PKV_DEVERR_CASCADE).
struct CascadeParams {
    const int32_t* members;       // [num_items, width], < 0 padding
    const int32_t* item_blocks;   // [num_items] shared whole blocks
    const int32_t* block_tables;
    const int32_t* context_lens;
    int32_t num_items, width, num_seqs, max_blocks;
    int32_t* list_ctx;            // out [num_items + num_seqs]
    int32_t* list_seq;            // out [num_items + num_seqs]: the table each entry reads
    int32_t* list_start;          // out [num_items + num_seqs]: first visible token
    int32_t* list_rows;           // out [num_items + num_seqs, width]: query rows, -1 none
    int32_t* counters;            // the balanced pass's piece counters, cleared here
    int32_t num_counters;
    uint32_t* err;
};
cudaError_t launch_cascade_setup(const CascadeParams& p, cudaStream_t stream);

// Sparse page-indirection set-up (one CTA per sequence): the listed pages'
// block ids, compacted, and the compacted context (the tail page may be partial).
struct SparseParams {
    const int32_t* page_lists;    // [num_seqs, max_pages]
    const int32_t* page_counts;   // [num_seqs]
    const int32_t* block_tables;
    const int32_t* context_lens;
    int32_t num_seqs, max_pages, max_blocks;
    int32_t* table_out;           // out [num_seqs, max_pages]
    int32_t* ctx_out;             // out [num_seqs]
    int32_t* counters;            // the balanced pass's piece counters, cleared here
    int32_t num_counters;
    uint32_t* err;
};
cudaError_t launch_sparse_setup(const SparseParams& p, cudaStream_t stream);

struct CacheWriteParams {
    void* k_cache;
    void* v_cache;
    const void* k_new;
    const void* v_new;
    const int64_t* slot_mapping;
    int32_t num_tokens;
    int32_t num_blocks;
    int32_t num_kv_heads;
    int32_t head_dim;
    uint32_t* err;
    // K8V4 only
    void* k_scale;
    void* v_scale;
    void* v_zero;
    int32_t src_dtype;
};
cudaError_t launch_reshape_and_cache(const CacheWriteParams& p, int elem_bytes, cudaStream_t stream);
cudaError_t launch_quantize_kv(const CacheWriteParams& p, cudaStream_t stream);

struct GatherParams {
    void* k_out;
    void* v_out;
    const int32_t* cu_seq_lens;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    int32_t num_seqs;
    int32_t max_blocks;
    int32_t num_blocks;
    int32_t num_kv_heads;
    int32_t head_dim;
    uint32_t* err;
    // dequantising gather of a K8/V4 cache
    const void* k_scale;
    const void* v_scale;
    const void* v_zero;
    int32_t out_dtype;
};
cudaError_t launch_gather(const GatherParams& p, int elem_bytes, cudaStream_t stream);
cudaError_t launch_gather_dequant(const GatherParams& p, cudaStream_t stream);

}  // namespace pkv
