// decode_persistent_d16.cu -- instantiations of the persistent decode kernel
// for head_dim 16, one per GQA group bound (2, 4, 8, 16).
#include "decode_persistent.cuh"

namespace ember {

PkKernel pk_kernel_d16(int G) {
    if (G <= 2) return k_decode_persist<16, 2>;
    if (G <= 4) return k_decode_persist<16, 4>;
    if (G <= 8) return k_decode_persist<16, 8>;
    return k_decode_persist<16, 16>;
}

}  // namespace ember
