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

}  // namespace gbce
