// Instantiations of the streaming forward kernel with class weights and
// label smoothing: 8 consumer warps, 8 vectors a thread a slot, the weights
// in shared memory (see ce_fwd_stream.cuh).
#include "ce_fwd_stream.cuh"

namespace gbce {

const void* stream_kernel_ws(int dtype, bool softcap) {
    if (dtype == 0)
        return softcap ? (const void*)&ce_fwd_stream<float, true, 8, 8, true>
                       : (const void*)&ce_fwd_stream<float, false, 8, 8, true>;
    if (dtype == 1)
        return softcap ? (const void*)&ce_fwd_stream<__nv_bfloat16, true, 8, 8, true>
                       : (const void*)&ce_fwd_stream<__nv_bfloat16, false, 8, 8, true>;
    if (dtype == 2)
        return softcap ? (const void*)&ce_fwd_stream<__half, true, 8, 8, true>
                       : (const void*)&ce_fwd_stream<__half, false, 8, 8, true>;
    return nullptr;
}

}  // namespace gbce
