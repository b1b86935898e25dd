// Instantiations of the staged forward kernel: bf16 logits, without softcap,
// without per-class smoothing weights; one per CTA shape.
#include "ce_fwd_staged.cuh"

namespace gbce {

const void* staged_kernel_bf16_nocap_plain(int cfg) {
    switch (cfg) {
    case 0: return (const void*)&ce_fwd_staged<__nv_bfloat16, 128, 4, false, false>;
    case 1: return (const void*)&ce_fwd_staged<__nv_bfloat16, 128, 8, false, false>;
    case 2: return (const void*)&ce_fwd_staged<__nv_bfloat16, 256, 4, false, false>;
    case 3: return (const void*)&ce_fwd_staged<__nv_bfloat16, 256, 8, false, false>;
    case 4: return (const void*)&ce_fwd_staged<__nv_bfloat16, 512, 4, false, false>;
    case 5: return (const void*)&ce_fwd_staged<__nv_bfloat16, 512, 8, false, false>;
    }
    return nullptr;
}

}  // namespace gbce
