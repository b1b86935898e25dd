// Instantiations of the staged forward kernel: f32 logits, without softcap,
// without per-class smoothing weights; one per CTA shape.
#include "ce_fwd_staged.cuh"

namespace gbce {

const void* staged_kernel_f32_nocap_plain(int cfg) {
    switch (cfg) {
    case 0: return (const void*)&ce_fwd_staged<float, 128, 4, false, false>;
    case 1: return (const void*)&ce_fwd_staged<float, 128, 8, false, false>;
    case 2: return (const void*)&ce_fwd_staged<float, 256, 4, false, false>;
    case 3: return (const void*)&ce_fwd_staged<float, 256, 8, false, false>;
    case 4: return (const void*)&ce_fwd_staged<float, 512, 4, false, false>;
    case 5: return (const void*)&ce_fwd_staged<float, 512, 8, false, false>;
    }
    return nullptr;
}

}  // namespace gbce
