// Instantiations of the staged forward kernel: bf16 logits with tanh softcap.
#include "ce_fwd_staged.cuh"

namespace gbce {

const void* staged_kernel_bf16_softcap(int cfg_index, bool wsmooth) {
#define GBCE_PICK(I, NT, NV)                                                     \
    if (cfg_index == I)                                                          \
        return wsmooth ? (const void*)&ce_fwd_staged<__nv_bfloat16, NT, NV, true, true> \
                       : (const void*)&ce_fwd_staged<__nv_bfloat16, NT, NV, true, false>;
    GBCE_PICK(0, 128, 4)
    GBCE_PICK(1, 256, 4)
    GBCE_PICK(2, 512, 4)
    GBCE_PICK(3, 512, 8)
#undef GBCE_PICK
    return nullptr;
}

}  // namespace gbce
