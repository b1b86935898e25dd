// The unfused (aten-shaped) form of softmax cross-entropy: _log_softmax,
// nll_loss_forward, nll_loss_backward and _log_softmax_backward_data, the
// ops a decomposed F.cross_entropy graph runs (tt-mlir pull request #9324,
// the table of decomposed aten ops on [1023, 128256] f32 logits and the
// #9339 description: max-shifted log-sum-exp, integer targets with
// ignore_index, mean/sum/none, zero gradients for an all-ignored batch).
// Class weights follow the aten operators' definitions.
//
// _log_softmax runs in the streaming kernel's log-softmax mode (TMA ring,
// one HBM read and one write per element); rows that are not 16-byte
// aligned take a general kernel. The other three are short kernels bound
// by HBM: a gather with a fixed-order reduction, a write-only scatter, and
// a two-pass row kernel whose second pass reads the incoming gradient
// again from L2.
#include <climits>

#include "ce_fwd_stream.cuh"

namespace gbce {
namespace {

template <typename T>
__device__ __forceinline__ float load_elem(const void* p, int64_t i) {
    return Vec<T>::load1(p, i);
}

// _log_softmax for any alignment: one CTA per row (grid-stride), the row's
// maximum, then sum exp(x - m), then the output, each pass over global
// memory (the later passes mostly from L2).
template <typename T>
__global__ void __launch_bounds__(kLsmGenericThreads) ce_lsm_generic(const __grid_constant__ LsmArgs a) {
    constexpr int NT = kLsmGenericThreads;
    __shared__ float sh[NT / 32];
    const int tid = threadIdx.x;
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        const int64_t base = r * a.C;
        float m = -INFINITY;
        for (int64_t j = tid; j < a.C; j += NT) m = fmaxf(m, load_elem<T>(a.x, base + j));
        __syncwarp();
        m = warp_max_f32(m);
        if ((tid & 31) == 0) sh[tid >> 5] = m;
        __syncthreads();
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) M = fmaxf(M, sh[w]);
        __syncthreads();
        float s = 0.f;
        for (int64_t j = tid; j < a.C; j += NT) s += ex2((load_elem<T>(a.x, base + j) - M) * kLog2e);
        const float S = block_sum_fixed<NT>(s, sh);
        __syncthreads();
        const float logS = logf(S);
        for (int64_t j = tid; j < a.C; j += NT)
            Vec<T>::store1(a.out, base + j, (load_elem<T>(a.x, base + j) - M) - logS);
    }
}

}  // namespace

const void* stream_kernel_lsm(int dtype) {
    if (dtype == 0) return (const void*)&ce_fwd_stream<float, false, 4, 16, false, true>;
    if (dtype == 1) return (const void*)&ce_fwd_stream<__nv_bfloat16, false, 4, 16, false, true>;
    if (dtype == 2) return (const void*)&ce_fwd_stream<__half, false, 4, 16, false, true>;
    return nullptr;
}

const void* lsm_generic_kernel(int dtype) {
    if (dtype == 0) return (const void*)&ce_lsm_generic<float>;
    if (dtype == 1) return (const void*)&ce_lsm_generic<__nv_bfloat16>;
    if (dtype == 2) return (const void*)&ce_lsm_generic<__half>;
    return nullptr;
}

}  // namespace gbce
