// N-D forward kernels (class dimension 1) for f16 logits; one translation
// unit per logit type so the variants compile in parallel.
#include "ce_fwd_nd.cuh"
#include "ce_fwd_nd_split.cuh"

namespace gbce {

const void* nd_kernel_f16(bool vec, bool softcap, bool argmax) {
    return nd_kernel_of<__half>(vec, softcap, argmax);
}

const void* nd_warp_f16(bool softcap, bool argmax) { return nd_warp_of<__half>(softcap, argmax); }

NdSplitFns nd_split_f16(bool vec, bool softcap, bool argmax, bool smooth) {
    return nd_split_of<__half>(vec, softcap, argmax, smooth);
}

}  // namespace gbce
