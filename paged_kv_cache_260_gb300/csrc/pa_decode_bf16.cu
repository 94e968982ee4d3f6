// pa_decode_bf16.cu -- bf16 instantiations of the decode and merge kernels.
#include "pa_decode_mma.cuh"

namespace pa {
bool decode_kernels_bf16(int head_dim, int group, KernelSet *ks)
{
    return kernels_for<__nv_bfloat16>(head_dim, group, ks);
}
}  // namespace pa
