// pa_decode_bf16_g16.cu -- bf16 instantiations of the decode and merge kernels,
// groups of 9..16 query heads per kv head.
#include "pa_decode_mma.cuh"

namespace pa {
bool decode_kernels_bf16_g16(int head_dim, KernelSet *ks)
{
    return kernels_for_nt<__nv_bfloat16, 2>(head_dim, ks);
}
}  // namespace pa
