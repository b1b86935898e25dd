// Instantiations of the register-resident forward kernel (see
// ce_fwd_reg.cuh) for class-weighted label smoothing with the class weights
// in shared memory: one CTA of 16 warps an SM, 8 vectors a thread, every
// logit type, with and without softcap.
#include "ce_fwd_reg.cuh"

namespace gbce {

namespace {
template <typename T>
const void* sw_of(bool softcap) {
    return softcap ? (const void*)&ce_fwd_reg<T, true, true, 8, false, 16, true>
                   : (const void*)&ce_fwd_reg<T, false, true, 8, false, 16, true>;
}
}  // namespace

const void* reg_kernel_sw(int dtype, bool softcap) {
    if (dtype == 0) return sw_of<float>(softcap);
    if (dtype == 1) return sw_of<__nv_bfloat16>(softcap);
    if (dtype == 2) return sw_of<__half>(softcap);
    return nullptr;
}

}  // namespace gbce
