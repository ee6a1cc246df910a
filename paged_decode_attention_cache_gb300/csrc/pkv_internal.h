// pkv_internal.h -- parameter blocks and launchers shared between the C-ABI
// layer (api.cu) and the kernel translation units.  Host-side only types.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

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
    uint32_t* err;
};

// Returns cudaSuccess or the launch error.  The grid is
// (partitions, num_kv_heads, num_seqs); maps are K and V tile maps.
cudaError_t launch_decode_cc(const AttnParams& p, int cache_kind, int gqa, const CUtensorMap& k_map,
                             const CUtensorMap& v_map, int grid_parts, cudaStream_t stream);
cudaError_t launch_decode_tc(const AttnParams& p, int cache_kind, int gqa, const CUtensorMap& k_map,
                             const CUtensorMap& v_map, int grid_parts, cudaStream_t stream);
bool decode_cc_supported(int cache_kind, int head_dim, int gqa);
bool decode_tc_supported(int cache_kind, int head_dim, int gqa, int q_len);

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
};
cudaError_t launch_reduce(const ReduceParams& p, cudaStream_t stream);

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
};
cudaError_t launch_gather(const GatherParams& p, int elem_bytes, cudaStream_t stream);

}  // namespace pkv
