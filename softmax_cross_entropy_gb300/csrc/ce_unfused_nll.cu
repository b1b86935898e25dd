// The unfused (aten-shaped) ops other than _log_softmax: nll_loss_forward,
// nll_loss_backward and _log_softmax_backward_data (tt-mlir pull request
// #9324, the table of decomposed aten ops and the #9339 description; class
// weights as the aten operators define them: w[t] on the target term,
// total_weight = sum of w[t_i] over the rows that are not ignored).
#include "ce_kernels.cuh"

namespace gbce {
namespace {

template <typename T>
__device__ __forceinline__ int64_t nll_target(const T& a, int64_t r) {
    return a.tgt64 ? reinterpret_cast<const int64_t*>(a.target)[r]
                   : static_cast<int64_t>(reinterpret_cast<const int32_t*>(a.target)[r]);
}

// nll_loss_forward: l_i = -w[t_i] * logp[i, t_i] (0 for ignore_index).
// "none" writes l_i per row and total_weight 0; "sum"/"mean" add l_i and
// w[t_i] in double per CTA, then over the CTAs in a fixed order (grid_sum2);
// "mean" divides by total_weight (NaN when no row counts). A target outside
// [0, C) that is not ignore_index is recorded in the status word and the
// row is treated as ignored.
template <typename T>
__global__ void __launch_bounds__(kNllThreads) ce_nll_fwd(const __grid_constant__ NllFwdArgs a) {
    constexpr int NW = kNllThreads / 32;
    __shared__ double s_l[NW], s_w[NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    double L = 0.0, W = 0.0;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kNllThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kNllThreads + tid; i < a.rows; i += stride) {
        const int64_t t = nll_target(a, i);
        float l = 0.f;
        if (t != a.ignore_index) {
            if (t < 0 || t >= a.C) {
                atomicOr(&a.scratch->status, kDevErrTarget);
            } else {
                const float w = a.weight ? __ldg(a.weight + t) : 1.f;
                l = -w * Vec<T>::load1(a.logp, i * a.C + t);
                L += static_cast<double>(l);
                W += static_cast<double>(w);
            }
        }
        if (a.reduction == kRedNone) a.out[i] = l;
    }
    if (a.reduction == kRedNone) {
        if (blockIdx.x == 0 && tid == 0) a.total_weight[0] = 0.f;
        return;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        L += __shfl_xor_sync(0xffffffffu, L, o);
        W += __shfl_xor_sync(0xffffffffu, W, o);
    }
    if (lane == 0) {
        s_l[warp] = L;
        s_w[warp] = W;
    }
    __syncthreads();
    if (warp != 0) return;
    double u = 0.0, v = 0.0;
    if (lane == 0)
        for (int w = 0; w < NW; ++w) {
            u += s_l[w];
            v += s_w[w];
        }
    if (grid_sum2(a.scratch, u, v)) {
        a.out[0] = static_cast<float>(a.reduction == kRedMean ? u / v : u);
        a.total_weight[0] = static_cast<float>(v);
    }
}

// nll_loss_backward: every element of grad_input is written: zero, except
// grad_input[i, t_i] = -w[t_i] * g_i for counted rows, with g_i the row's
// grad_output ("none"), the scalar grad_output ("sum") or the scalar over
// total_weight ("mean"). One CTA per row (grid-stride), 16-byte stores; the
// thread whose vector holds the target writes it in that vector.
template <typename T>
__global__ void __launch_bounds__(kNllThreads) ce_nll_bwd(const __grid_constant__ NllBwdArgs a) {
    using VT = Vec<T>;
    constexpr int VE = VT::N;
    const float g_all = a.reduction == kRedNone ? 0.f
                        : a.reduction == kRedMean ? __ldg(a.grad_output) / __ldg(a.total_weight)
                                                  : __ldg(a.grad_output);
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        const int64_t t = nll_target(a, r);
        const bool counted = t != a.ignore_index && t >= 0 && t < a.C;
        if (t != a.ignore_index && !counted && threadIdx.x == 0)
            atomicOr(&a.scratch->status, kDevErrTarget);
        float val = 0.f;
        if (counted) {
            const float g = a.reduction == kRedNone ? __ldg(a.grad_output + r) : g_all;
            val = -(a.weight ? __ldg(a.weight + t) : 1.f) * g;
        }
        if (a.vec_ok) {
            uint4* row = reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.grad_input) + r * a.C);
            const int64_t nv = a.C / VE;
            const int64_t tv = counted ? t / VE : -1;
            for (int64_t v = threadIdx.x; v < nv; v += kNllThreads) {
                if (v == tv) {
                    float f[VE];
#pragma unroll
                    for (int j = 0; j < VE; ++j) f[j] = (j == t - tv * VE) ? val : 0.f;
                    row[v] = VT::pack(f);
                } else {
                    row[v] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
        } else {
            for (int64_t j = threadIdx.x; j < a.C; j += kNllThreads)
                VT::store1(a.grad_input, r * a.C + j, (counted && j == t) ? val : 0.f);
        }
    }
}

// _log_softmax_backward_data: dx = dy - exp(y) * sum_k dy_k per row. One
// CTA per row (grid-stride, one CTA per SM): pass 1 sums dy with an L2
// evict-last hint, so that pass 2, which reads dy and y (evict-first) and
// writes dx, finds dy in L2; the row sum is a fixed-order block reduction.
template <typename T>
__global__ void __launch_bounds__(kLsmBwdThreads) ce_lsm_bwd(const __grid_constant__ LsmBwdArgs a) {
    using VT = Vec<T>;
    constexpr int VE = VT::N;
    constexpr int NT = kLsmBwdThreads;
    __shared__ float sh[NT / 32];
    const int tid = threadIdx.x;
    const uint64_t keep = l2_evict_last_policy();
    const uint64_t once = l2_evict_first_policy();
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        const int64_t base = r * a.C;
        float s = 0.f;
        if (a.vec_ok) {
            const uint4* dy = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.dy) + base);
            const int64_t nv = a.C / VE;
#pragma unroll 4
            for (int64_t v = tid; v < nv; v += NT) {
                float f[VE];
                VT::unpack(ld_v4_hint(dy + v, keep), f);
#pragma unroll
                for (int j = 0; j < VE; ++j) s += f[j];
            }
        } else {
            for (int64_t j = tid; j < a.C; j += NT) s += VT::load1(a.dy, base + j);
        }
        const float S = block_sum_fixed<NT>(s, sh);
        __syncthreads();  // sh is reused by the next row
        if (a.vec_ok) {
            const uint4* dy = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.dy) + base);
            const uint4* y = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.y) + base);
            uint4* dx = reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.dx) + base);
            const int64_t nv = a.C / VE;
#pragma unroll 2
            for (int64_t v = tid; v < nv; v += NT) {
                float fd[VE], fy[VE];
                VT::unpack(ld_v4_hint(dy + v, once), fd);
                VT::unpack(ld_v4_hint(y + v, once), fy);
#pragma unroll
                for (int j = 0; j < VE; ++j) fd[j] = fmaf(-ex2(fy[j] * kLog2e), S, fd[j]);
                dx[v] = VT::pack(fd);
            }
        } else {
            for (int64_t j = tid; j < a.C; j += NT)
                VT::store1(a.dx, base + j,
                           fmaf(-ex2(VT::load1(a.y, base + j) * kLog2e), S, VT::load1(a.dy, base + j)));
        }
    }
}

}  // namespace

const void* nll_fwd_kernel(int dtype) {
    if (dtype == 0) return (const void*)&ce_nll_fwd<float>;
    if (dtype == 1) return (const void*)&ce_nll_fwd<__nv_bfloat16>;
    if (dtype == 2) return (const void*)&ce_nll_fwd<__half>;
    return nullptr;
}

const void* nll_bwd_kernel(int dtype) {
    if (dtype == 0) return (const void*)&ce_nll_bwd<float>;
    if (dtype == 1) return (const void*)&ce_nll_bwd<__nv_bfloat16>;
    if (dtype == 2) return (const void*)&ce_nll_bwd<__half>;
    return nullptr;
}

const void* lsm_bwd_kernel(int dtype) {
    if (dtype == 0) return (const void*)&ce_lsm_bwd<float>;
    if (dtype == 1) return (const void*)&ce_lsm_bwd<__nv_bfloat16>;
    if (dtype == 2) return (const void*)&ce_lsm_bwd<__half>;
    return nullptr;
}

}  // namespace gbce
