// Instantiations of the staged forward kernel: bf16 logits, with tanh softcap,
// with class-weighted label smoothing; one per CTA shape.
#include "ce_fwd_staged.cuh"

namespace gbce {

const void* staged_kernel_bf16_softcap_wsmooth(int cfg) {
    switch (cfg) {
    case 0: return (const void*)&ce_fwd_staged<__nv_bfloat16, 128, 4, true, true>;
    case 1: return (const void*)&ce_fwd_staged<__nv_bfloat16, 128, 8, true, true>;
    case 2: return (const void*)&ce_fwd_staged<__nv_bfloat16, 256, 4, true, true>;
    case 3: return (const void*)&ce_fwd_staged<__nv_bfloat16, 256, 8, true, true>;
    case 4: return (const void*)&ce_fwd_staged<__nv_bfloat16, 512, 4, true, true>;
    case 5: return (const void*)&ce_fwd_staged<__nv_bfloat16, 512, 8, true, true>;
    }
    return nullptr;
}

}  // namespace gbce
