// Instantiations of the register-resident forward kernel (see
// ce_fwd_reg.cuh) for f16 logits: 8 or 16 vectors a thread, with and without
// softcap, with and without class-weighted label smoothing. One translation
// unit per logit type so the variants compile in parallel.
#include "ce_fwd_reg.cuh"

namespace gbce {

const void* reg_kernel_f16(bool softcap, bool ws, int nvl) {
    if (nvl == 8) return reg_kernel_of<__half, 8>(softcap, ws);
    if (nvl == 16) return reg_kernel_of<__half, 16>(softcap, ws);
    return nullptr;
}

}  // namespace gbce
