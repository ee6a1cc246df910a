// attention_cascade.cu -- the instantiation of the attention kernel for the two
// passes of cascade attention [mlxcel manual "KV Cache", §"Paged Decode Storage
// and Kernels": cascade attention over shared whole-page prefixes]: the suffix
// pass starts each sequence at its seq_start, the prefix pass reads an item's
// blocks through its lending member's table and maps the item's query rows to
// its members.  Compiled apart so that the other kernels carry none of it.
#include "attention_impl.cuh"

namespace pkv {

cudaError_t launch_attention_cascade(AttnParams p, int cache_kind, int gqa, const CUtensorMap& km,
                                     const CUtensorMap& vm, cudaStream_t stream) {
    return launch_attention_impl<false, true>(p, cache_kind, gqa, km, vm, stream);
}

}  // namespace pkv
