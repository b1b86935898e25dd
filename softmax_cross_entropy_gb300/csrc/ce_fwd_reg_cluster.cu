// Cluster variant of the register-resident forward kernel (a thread-block
// cluster of CTAs owns each row longer than one CTA holds), 16 vectors a
// thread, for the three logit types; in a file of its own so that it
// compiles in parallel with the single-CTA variants.
#include "ce_fwd_reg.cuh"

namespace gbce {

const void* reg_cluster_kernel(int dtype, bool softcap, bool ws) {
    if (dtype == 0) return reg_kernel_of<float, 16, true>(softcap, ws);
    if (dtype == 1) return reg_kernel_of<__nv_bfloat16, 16, true>(softcap, ws);
    if (dtype == 2) return reg_kernel_of<__half, 16, true>(softcap, ws);
    return nullptr;
}

}  // namespace gbce
