// decode_persistent_d64.cu -- instantiations of the persistent decode kernel
// for head_dim 64, one per GQA group bound (2, 4, 8, 16).
#include "decode_persistent.cuh"

namespace ember {

PkKernel pk_kernel_d64(int G) {
    if (G <= 2) return k_decode_persist<64, 2>;
    if (G <= 4) return k_decode_persist<64, 4>;
    if (G <= 8) return k_decode_persist<64, 8>;
    return k_decode_persist<64, 16>;
}

}  // namespace ember
