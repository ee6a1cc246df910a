// attention.cu -- host side of the attention kernels: which shapes run, the
// attention-only instantiation of the persistent kernel (attention_impl.cuh)
// and the balanced workspace size.  The fused decode step's instantiation is
// in attention_fused.cu, the cascade passes' in attention_cascade.cu.
#include "attention_impl.cuh"

namespace pkv {

bool attention_supported(int cache_kind, int head_dim, int gqa, int q_len) {
    const bool shape = (head_dim == 64 || head_dim == 128) && (gqa == 1 || gqa == 2 || gqa == 4 || gqa == 8);
    if (!shape || q_len < 1) return false;
    if (attention_uses_tensor_cores(cache_kind, q_len, gqa)) return gqa * q_len <= kMaxRows;
    return cache_kind == PKV_CACHE_F16 || cache_kind == PKV_CACHE_BF16;
}

// The CUDA-core math spends ~500 warp instructions per 16-token block at group
// size 4 and is latency-bound below the HBM rate (~36 GB/s per SM with 11
// consumer warps, slower with fewer); the MMA formulation needs ~150 and
// streams at ~42 GB/s per SM.  At group size 1 and 2 the CUDA-core math does
// proportionally less work and is a little faster (both measured).
bool attention_uses_tensor_cores(int cache_kind, int q_len, int gqa, bool cascade_pass) {
    return cascade_pass || cache_kind == PKV_CACHE_K8V4 || q_len > 1 || gqa * q_len >= kTcMinRows;
}

cudaError_t launch_attention(AttnParams p, int cache_kind, int gqa, const CUtensorMap& km, const CUtensorMap& vm,
                             cudaStream_t stream) {
    if (is_cascade_pass(p)) return launch_attention_cascade(p, cache_kind, gqa, km, vm, stream);
    if (p.num_new > 0) return launch_attention_fused(p, cache_kind, gqa, km, vm, stream);
    return launch_attention_impl<false, false>(p, cache_kind, gqa, km, vm, stream);
}

size_t balanced_workspace_bytes(int num_seqs, int num_kv_heads, int head_dim) {
    auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t pairs = size_t(num_seqs) * size_t(num_kv_heads);
    const size_t slots = size_t(kMaxGrid) + pairs;
    return a256(slots * kMaxRows * size_t(head_dim) * 4) + a256(slots * kMaxRows * 2 * 4) + a256(pairs * 4);
}

}  // namespace pkv
