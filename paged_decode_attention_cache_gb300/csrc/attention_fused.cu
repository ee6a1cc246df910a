// attention_fused.cu -- the fused decode step's instantiation of the attention
// kernel: the step's cache write (reshape_and_cache / quantize_kv) and the
// balanced attention in one launch.  Compiled apart from attention.cu so that
// the attention-only kernels keep their own register allocation.
#include "attention_impl.cuh"

namespace pkv {

cudaError_t launch_attention_fused(AttnParams p, int cache_kind, int gqa, const CUtensorMap& km, const CUtensorMap& vm,
                                   cudaStream_t stream) {
    return launch_attention_impl<true, false>(p, cache_kind, gqa, km, vm, stream);
}

}  // namespace pkv
