// Instantiations of the streaming forward kernel for fp16 logits without
// class-weighted label smoothing (see ce_fwd_stream.cuh).
#include "ce_fwd_stream.cuh"

namespace gbce {

const void* stream_kernel_f16(bool softcap, int vpt, int nw) {
    if (nw == 8 && vpt == 8)
        return softcap ? (const void*)&ce_fwd_stream<__half, true, 8, 8, false>
                       : (const void*)&ce_fwd_stream<__half, false, 8, 8, false>;
    if (nw == 16 && vpt == 4)
        return softcap ? (const void*)&ce_fwd_stream<__half, true, 4, 16, false>
                       : (const void*)&ce_fwd_stream<__half, false, 4, 16, false>;
    return nullptr;
}

}  // namespace gbce
