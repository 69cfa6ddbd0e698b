// decode_persistent_d128.cu -- instantiations of the persistent decode kernel
// for head_dim 128, one per GQA group bound (2, 4, 8, 16).
#include "decode_persistent.cuh"

namespace ember {

PkKernel pk_kernel_d128(int G) {
    if (G <= 2) return k_decode_persist<128, 2>;
    if (G <= 4) return k_decode_persist<128, 4>;
    if (G <= 8) return k_decode_persist<128, 8>;
    return k_decode_persist<128, 16>;
}

}  // namespace ember
