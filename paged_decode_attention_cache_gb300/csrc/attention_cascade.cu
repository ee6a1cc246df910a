// attention_cascade.cu -- the instantiation of the attention kernel for the
// pass of cascade attention [mlxcel manual "KV Cache", §"Paged Decode Storage
// and Kernels": cascade attention over shared whole-page prefixes]: one
// balanced pass over a list of items (a group's shared blocks, read through its
// lending member's table, one query row per member) followed by every sequence
// from its seq_start on; each entry's combined partial goes to its own slot of
// the rows it serves.  Compiled apart so that the other kernels carry none of it.
#include "attention_impl.cuh"

namespace pkv {

cudaError_t launch_attention_cascade(AttnParams p, int cache_kind, int gqa, const CUtensorMap& km,
                                     const CUtensorMap& vm, cudaStream_t stream) {
    return launch_attention_impl<false, true>(p, cache_kind, gqa, km, vm, stream);
}

}  // namespace pkv
