// pa_decode_f16_g16.cu -- f16 instantiations of the decode and merge kernels,
// groups of 9..16 query heads per kv head.
#include "pa_decode_mma.cuh"

namespace pa {
bool decode_kernels_f16_g16(int head_dim, KernelSet *ks)
{
    return kernels_for_nt<__half, 2>(head_dim, ks);
}
}  // namespace pa
