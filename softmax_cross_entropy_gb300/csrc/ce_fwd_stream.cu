// Instantiations of the streaming forward kernel without class-weighted
// label smoothing (see ce_fwd_stream.cuh).
#include "ce_fwd_stream.cuh"

namespace gbce {

const void* stream_kernel(int dtype, bool softcap, int vpt, int nw) {
    // two shapes: 8 consumer warps with 8 vectors a thread a slot (168
    // registers), or 16 warps with 4 (96 registers, a few bytes spilled);
    // both take 2048 vectors per slot
#define GBCE_STREAM(TT, SC)                                                         \
    (nw == 8 && vpt == 8                                                            \
         ? (const void*)&ce_fwd_stream<TT, SC, 8, 8, false>                         \
         : (nw == 16 && vpt == 4 ? (const void*)&ce_fwd_stream<TT, SC, 4, 16, false> \
                                 : nullptr))
    if (dtype == 0) return softcap ? GBCE_STREAM(float, true) : GBCE_STREAM(float, false);
    if (dtype == 1)
        return softcap ? GBCE_STREAM(__nv_bfloat16, true) : GBCE_STREAM(__nv_bfloat16, false);
#undef GBCE_STREAM
    if (dtype == 2) return stream_kernel_f16(softcap, vpt, nw);
    return nullptr;
}

// fp32 logits with the gradient to FwdArgs::gout in 16 bits, the same two
// shapes.
const void* stream_kernel_gout(bool softcap, int vpt, int nw) {
#define GBCE_STREAM_GO(SC)                                                                 \
    (nw == 8 && vpt == 8                                                                   \
         ? (const void*)&ce_fwd_stream<float, SC, 8, 8, false, false, true>                \
         : (nw == 16 && vpt == 4 ? (const void*)&ce_fwd_stream<float, SC, 4, 16, false, false, true> \
                                 : nullptr))
    return softcap ? GBCE_STREAM_GO(true) : GBCE_STREAM_GO(false);
#undef GBCE_STREAM_GO
}

}  // namespace gbce
