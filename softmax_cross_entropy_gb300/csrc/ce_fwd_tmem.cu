// Instantiations of the tensor-memory softcap kernel (see ce_fwd_tmem.cuh)
// for every logit type.
#include "ce_fwd_tmem.cuh"

namespace gbce {

const void* tmem_kernel(int dtype) {
    if (dtype == 0) return (const void*)&ce_fwd_tmem<float>;
    if (dtype == 1) return (const void*)&ce_fwd_tmem<__nv_bfloat16>;
    if (dtype == 2) return (const void*)&ce_fwd_tmem<__half>;
    return nullptr;
}

}  // namespace gbce
