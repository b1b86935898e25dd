// N-D forward kernels (class dimension 1) for f32 logits; one translation
// unit per logit type so the variants compile in parallel.
#include "ce_fwd_nd.cuh"
#include "ce_fwd_nd_split.cuh"

namespace gbce {

const void* nd_kernel_f32(bool vec, bool softcap, bool argmax) {
    return nd_kernel_of<float>(vec, softcap, argmax);
}

const void* nd_warp_f32(bool softcap, bool argmax) { return nd_warp_of<float>(softcap, argmax); }

NdSplitFns nd_split_f32(bool vec, bool softcap, bool argmax, bool smooth) {
    return nd_split_of<float>(vec, softcap, argmax, smooth);
}

}  // namespace gbce
