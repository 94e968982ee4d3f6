// pa_decode_f16.cu -- fp16 instantiations of the decode and merge kernels.
#include "pa_decode_mma.cuh"

namespace pa {
bool decode_kernels_f16(int head_dim, int group, KernelSet *ks)
{
    return kernels_for<__half>(head_dim, group, ks);
}
}  // namespace pa
