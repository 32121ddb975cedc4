// Tensor-core (tcgen05) kernel for multi-token turns: not built yet; the CUDA-core kernel handles
// every sequence while tc_supported() is false.
#include "internal.h"

namespace pkv {

cudaError_t launch_tc(const FwdArgs &a, cudaStream_t s) {
    (void)a;
    (void)s;
    return cudaSuccess;
}

}  // namespace pkv
