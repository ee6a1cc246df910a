// decode_tc.cu -- placeholder until the tensor-core kernel lands.
#include "pkv_internal.h"

namespace pkv {
bool decode_tc_supported(int, int, int, int) { return false; }
cudaError_t launch_decode_tc(const AttnParams&, int, int, const CUtensorMap&, const CUtensorMap&, int, cudaStream_t) {
    return cudaErrorNotSupported;
}
}  // namespace pkv
