// Instantiations of the staged forward kernel: f32 logits, without softcap,
// with class-weighted label smoothing; one per CTA shape.
#include "ce_fwd_staged.cuh"

namespace gbce {

const void* staged_kernel_f32_nocap_wsmooth(int cfg) {
    switch (cfg) {
    case 0: return (const void*)&ce_fwd_staged<float, 128, 4, false, true>;
    case 1: return (const void*)&ce_fwd_staged<float, 128, 8, false, true>;
    case 2: return (const void*)&ce_fwd_staged<float, 256, 4, false, true>;
    case 3: return (const void*)&ce_fwd_staged<float, 256, 8, false, true>;
    case 4: return (const void*)&ce_fwd_staged<float, 512, 4, false, true>;
    case 5: return (const void*)&ce_fwd_staged<float, 512, 8, false, true>;
    }
    return nullptr;
}

}  // namespace gbce
