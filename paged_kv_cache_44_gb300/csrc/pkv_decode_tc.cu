// placeholder until the tensor-core kernel lands
#include "pkv_internal.h"
namespace pkv {
bool decode_tc_supports(pkv_dtype, pkv_dtype, int, int) { return false; }  // stub
cudaError_t launch_decode_tc(const DecodeParams&, pkv_dtype, pkv_dtype, int, cudaStream_t) {
    return cudaErrorNotSupported;
}
}  // namespace pkv
