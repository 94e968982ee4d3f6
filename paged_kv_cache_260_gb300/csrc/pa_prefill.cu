// pa_prefill.cu -- instantiations of the tcgen05 chunked-prefill kernel.
#include "pa_prefill.cuh"

namespace pa {

template <typename T, int D>
static void prefill_entry(PrefillKernel *k)
{
    k->fn = reinterpret_cast<const void *>(&prefill_tc_kernel<T, D>);
    k->threads = PrefillShape<D>::THREADS;
    k->smem = PrefillShape<D>::SMEM;
    k->plan_fn = reinterpret_cast<const void *>(&prefill_plan_kernel);
}

bool prefill_kernel(int dtype, int head_dim, PrefillKernel *k)
{
    const bool bf = dtype == PA_DTYPE_BF16;
    if (head_dim == 64)
        bf ? prefill_entry<__nv_bfloat16, 64>(k) : prefill_entry<__half, 64>(k);
    else if (head_dim == 128)
        bf ? prefill_entry<__nv_bfloat16, 128>(k) : prefill_entry<__half, 128>(k);
    else
        return false;
    return true;
}

}  // namespace pa
