// decode_persistent_d32.cu -- instantiations of the persistent decode kernel
// for head_dim 32, one per GQA group bound (2, 4, 8, 16).
#include "decode_persistent.cuh"

namespace ember {

PkKernel pk_kernel_d32(int G) {
    if (G <= 2) return k_decode_persist<32, 2>;
    if (G <= 4) return k_decode_persist<32, 4>;
    if (G <= 8) return k_decode_persist<32, 8>;
    return k_decode_persist<32, 16>;
}

}  // namespace ember
