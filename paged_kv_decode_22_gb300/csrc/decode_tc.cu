// Tensor-core decode path (tcgen05 + TMA).  Not compiled in yet: every
// configuration takes the CUDA-core path.
#include "internal.h"

namespace pkd {

bool decode_tc_supported(int, int, int) { return false; }

cudaError_t launch_decode_tc(const DecodeArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace pkd
