// General-path forward kernel and the backward kernel.
//
// The general forward handles what the staged kernel does not: rows whose
// byte length is not a multiple of 16 or that start unaligned, vocabularies
// larger than eight CTAs can stage, and the empty batch. One CTA owns a row
// at a time and makes three passes over it in global memory (max and
// argmax; exp-sum and smoothing sum; gradient), so the second and third
// reads come from L2 when the row fits. Same arithmetic and outputs as the
// staged kernel (Liger-Kernel cross-entropy kernel profile, §Forward Pass
// and §Key Patterns).
//
// Backward (same profile, §Backward Pass): the forward already stored the
// gradient, so backward multiplies it by grad_output, in place.
#include <climits>

#include "ce_kernels.cuh"

namespace gbce {

template <typename T, bool SOFTCAP>
__global__ void __launch_bounds__(kGenericThreads)
ce_fwd_generic(const __grid_constant__ FwdArgs a) {
    using VT = Vec<T>;
    constexpr int NT = kGenericThreads;
    constexpr int NW = NT / 32;
    __shared__ float red_m[NW];
    __shared__ int red_i[NW];
    __shared__ float red_s[NW];
    __shared__ float red_z[NW];
    __shared__ float red_p[NW];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const bool wsmooth = a.weight != nullptr && a.eps > 0.f;

    float D = 0.f;
    int n_valid = 0;
    if (a.reduction != kRedNone) denominators<NT>(a, red_p, D, n_valid);
    const float scale = a.reduction == kRedMean ? 1.f / D : 1.f;
    const float inv_V = 1.f / static_cast<float>(a.V);

    double accL = 0.0, accZ = 0.0;
    long long accC = 0;
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        const int64_t t = load_target(a, r);
        const bool counts = row_counts(a, t);
        const int64_t base = r * a.V;
        if (tid == 0 && t != a.ignore_index && !counts) atomicOr(&a.scratch->status, kDevErrTarget);
        if (!counts) {
            if (a.grad)
                for (int64_t j = tid; j < a.V; j += NT) VT::store1(a.x, base + j, 0.f);
            if (tid == 0) {
                if (a.reduction == kRedNone) {
                    a.loss[r] = 0.f;
                    if (a.want_z) a.zloss[r] = 0.f;
                    if (a.want_acc) a.acc[r] = 0.f;
                }
                if (a.want_pred) a.pred[r] = -1;
            }
            continue;
        }
        const float xt = tid == 0 ? VT::load1(a.x, base + t) : 0.f;
        const float wt = a.weight ? __ldg(a.weight + t) : 1.f;

        // pass 1: max and first argmax of the raw logits
        float tmax = -INFINITY;
        int tidx = INT_MAX;
        for (int64_t j = tid; j < a.V; j += NT) {
            const float v = VT::load1(a.x, base + j);
            if (v > tmax) {
                tmax = v;
                tidx = static_cast<int>(j);
            }
        }
        warp_argmax(tmax, tidx);
        if (lane == 0) {
            red_m[warp] = tmax;
            red_i[warp] = tidx;
        }
        __syncthreads();
        float mraw = red_m[0];
        int amax = red_i[0];
#pragma unroll
        for (int w = 1; w < NW; ++w) {
            if (red_m[w] > mraw || (red_m[w] == mraw && red_i[w] < amax)) {
                mraw = red_m[w];
                amax = red_i[w];
            }
        }
        // the row max of z (softcap is monotone); every difference below is
        // taken against it before scaling, which keeps them exact or nearly so
        const float M = SOFTCAP ? a.softcap * tanh_from_scaled(mraw * a.sc_k2) : mraw;
        const float shift = M == -INFINITY ? 0.f : M;

        // pass 2: S = sum exp(z - M), SZ = sum w (z - M), W = sum w
        float S = 0.f, SZ = 0.f, Wn = 0.f;
        for (int64_t j = tid; j < a.V; j += NT) {
            const float v = VT::load1(a.x, base + j);
            const float d = SOFTCAP ? fmaf(tanh_from_scaled(v * a.sc_k2), a.softcap, -shift)
                                    : v - shift;
            S += ex2(d * kLog2e);
            const float w = wsmooth ? __ldg(a.weight + j) : 1.f;
            SZ = fmaf(w, d, SZ);
            Wn += w;
        }
        S = warp_sum(S);
        SZ = warp_sum(SZ);
        Wn = warp_sum(Wn);
        if (lane == 0) {
            red_s[warp] = S;
            red_z[warp] = SZ;
            red_p[warp] = Wn;
        }
        __syncthreads();
        S = 0.f;
        SZ = 0.f;
        Wn = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            S += red_s[w];
            SZ += red_z[w];
            Wn += red_p[w];
        }
        const float logS = logf(S);

        if (tid == 0) {
            const float zt = SOFTCAP ? a.softcap * tanh_from_scaled(xt * a.sc_k2) : xt;
            float zl;
            const float l = row_loss(a, shift, logS, zt, wt,
                                     wsmooth ? Wn : static_cast<float>(a.V), SZ, zl);
            const bool correct = static_cast<int64_t>(amax) == t;
            if (a.reduction == kRedNone) {
                a.loss[r] = l;
                if (a.want_z) a.zloss[r] = zl;
                if (a.want_acc) a.acc[r] = correct ? 1.f : 0.f;
            } else {
                accL += static_cast<double>(l);
                accZ += static_cast<double>(zl);
                accC += correct ? 1 : 0;
            }
            if (a.want_pred) a.pred[r] = amax;
        }

        // pass 3: gradient in place (each thread rewrites only what it reads)
        if (a.grad) {
            const float lse = shift + logS;
            const float Wf = wsmooth ? Wn * inv_V : 1.f;
            const float Ac =
                scale * ((1.f - a.eps) * wt + a.eps * Wf + 2.f * a.lam * lse) / S;
            const float Bc = -scale * a.eps * inv_V;
            const float tfix = -scale * (1.f - a.eps) * wt;
            for (int64_t j = tid; j < a.V; j += NT) {
                const float v = VT::load1(a.x, base + j);
                float d, th = 0.f;
                if (SOFTCAP) {
                    th = tanh_from_scaled(v * a.sc_k2);
                    d = fmaf(th, a.softcap, -shift);
                } else {
                    d = v - shift;
                }
                float g = fmaf(Ac, ex2(d * kLog2e), wsmooth ? Bc * __ldg(a.weight + j) : Bc);
                if (j == t) g += tfix;
                if (SOFTCAP) g *= fmaf(-th, th, 1.f);
                VT::store1(a.x, base + j, g);
            }
        }
        // red_s, red_z, red_p are read above; the next row writes them only
        // after its first barrier, which every thread reaches after reading
    }
    // thread 0 holds the CTA's sums (it formed every row's loss)
    if (a.reduction != kRedNone) {
        __shared__ double red_l[NW], red_zz[NW];
        __shared__ long long red_cc[NW];
        __shared__ int s_flag;
        finish_scalars_cta(a, accL, accZ, accC, D, n_valid, &s_flag, red_l, red_zz, red_cc);
    }
}

template <typename T>
__global__ void __launch_bounds__(kBwdThreads) ce_bwd_scale(const __grid_constant__ BwdArgs a) {
    using VT = Vec<T>;
    constexpr int VE = VT::N;
    // launched as a programmatic dependent of the previous kernel on the
    // stream (the forward that stored the gradient): the launch overlaps
    // that kernel's end, and nothing is read before it has completed
    pdl_wait();
    if (!a.per_row && __ldg(a.g) == 1.f) return;  // multiplying by one changes nothing
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        const float g = a.per_row ? __ldg(a.g + r) : __ldg(a.g);
        if (g == 1.f) continue;
        if (a.vec_ok) {
            uint4* row = reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.x) + r * a.V);
            const int64_t nv = a.V / VE;
#pragma unroll 4
            for (int64_t v = threadIdx.x; v < nv; v += kBwdThreads) {
                float f[VE];
                VT::unpack(row[v], f);
#pragma unroll
                for (int j = 0; j < VE; ++j) f[j] *= g;
                row[v] = VT::pack(f);
            }
        } else {
            for (int64_t j = threadIdx.x; j < a.V; j += kBwdThreads)
                VT::store1(a.x, r * a.V + j, VT::load1(a.x, r * a.V + j) * g);
        }
    }
}

// Backward of the N-D form [N, C, inner]: dlogits *= grad_output, one value
// or one per position (n, s) for reduction "none". Each CTA walks the N * C
// lines of `inner` elements; a line's factors are grad_output[n * inner +
// s] for its n, so every position's factor multiplies its C classes.
template <typename T>
__global__ void __launch_bounds__(kBwdThreads) ce_bwd_nd_scale(const __grid_constant__ NdBwdArgs a) {
    using VT = Vec<T>;
    constexpr int VE = VT::N;
    pdl_wait();  // as in ce_bwd_scale
    if (!a.per_pos) {
        const float g = __ldg(a.g);
        if (g == 1.f) return;  // multiplying by one changes nothing
        const int64_t total = a.N * a.C * a.inner;
        const int64_t stride = static_cast<int64_t>(gridDim.x) * kBwdThreads;
        if (a.vec_ok) {
            uint4* v = reinterpret_cast<uint4*>(a.x);
#pragma unroll 4
            for (int64_t i = static_cast<int64_t>(blockIdx.x) * kBwdThreads + threadIdx.x;
                 i < total / VE; i += stride) {
                float f[VE];
                VT::unpack(v[i], f);
#pragma unroll
                for (int j = 0; j < VE; ++j) f[j] *= g;
                v[i] = VT::pack(f);
            }
        } else {
            for (int64_t i = static_cast<int64_t>(blockIdx.x) * kBwdThreads + threadIdx.x;
                 i < total; i += stride)
                VT::store1(a.x, i, VT::load1(a.x, i) * g);
        }
        return;
    }
    const int64_t lines = a.N * a.C;
    for (int64_t l = blockIdx.x; l < lines; l += gridDim.x) {
        const float* g = a.g + (l / a.C) * a.inner;
        T* line = reinterpret_cast<T*>(a.x) + l * a.inner;
        if (a.vec_ok) {
            uint4* v = reinterpret_cast<uint4*>(line);
            for (int64_t i = threadIdx.x; i < a.inner / VE; i += kBwdThreads) {
                float f[VE];
                VT::unpack(v[i], f);
#pragma unroll
                for (int j = 0; j < VE; ++j) f[j] *= __ldg(g + i * VE + j);
                v[i] = VT::pack(f);
            }
        } else {
            for (int64_t i = threadIdx.x; i < a.inner; i += kBwdThreads)
                VT::store1(line, i, VT::load1(line, i) * __ldg(g + i));
        }
    }
}

const void* nd_bwd_kernel(int dtype) {
    if (dtype == 0) return (const void*)&ce_bwd_nd_scale<float>;
    if (dtype == 1) return (const void*)&ce_bwd_nd_scale<__nv_bfloat16>;
    if (dtype == 2) return (const void*)&ce_bwd_nd_scale<__half>;
    return nullptr;
}

const void* reg_kernel_f32(bool softcap, bool ws, int nvl);
const void* reg_kernel_bf16(bool softcap, bool ws, int nvl);
const void* reg_kernel_f16(bool softcap, bool ws, int nvl);

const void* reg_kernel(int dtype, bool softcap, bool ws, int nvl) {
    if (dtype == 0) return reg_kernel_f32(softcap, ws, nvl);
    if (dtype == 1) return reg_kernel_bf16(softcap, ws, nvl);
    if (dtype == 2) return reg_kernel_f16(softcap, ws, nvl);
    return nullptr;
}

const void* nd_kernel_f32(bool vec, bool softcap, bool argmax);
const void* nd_kernel_bf16(bool vec, bool softcap, bool argmax);
const void* nd_kernel_f16(bool vec, bool softcap, bool argmax);

const void* nd_kernel(int dtype, bool vec, bool softcap, bool argmax) {
    if (dtype == 0) return nd_kernel_f32(vec, softcap, argmax);
    if (dtype == 1) return nd_kernel_bf16(vec, softcap, argmax);
    if (dtype == 2) return nd_kernel_f16(vec, softcap, argmax);
    return nullptr;
}

const void* nd_warp_f32(bool softcap, bool argmax);
const void* nd_warp_bf16(bool softcap, bool argmax);
const void* nd_warp_f16(bool softcap, bool argmax);

const void* nd_warp_kernel(int dtype, bool softcap, bool argmax) {
    if (dtype == 0) return nd_warp_f32(softcap, argmax);
    if (dtype == 1) return nd_warp_bf16(softcap, argmax);
    if (dtype == 2) return nd_warp_f16(softcap, argmax);
    return nullptr;
}

NdSplitFns nd_split_f32(bool vec, bool softcap, bool argmax, bool smooth);
NdSplitFns nd_split_bf16(bool vec, bool softcap, bool argmax, bool smooth);
NdSplitFns nd_split_f16(bool vec, bool softcap, bool argmax, bool smooth);

NdSplitFns nd_split_fns(int dtype, bool vec, bool softcap, bool argmax, bool smooth) {
    if (dtype == 0) return nd_split_f32(vec, softcap, argmax, smooth);
    if (dtype == 1) return nd_split_bf16(vec, softcap, argmax, smooth);
    if (dtype == 2) return nd_split_f16(vec, softcap, argmax, smooth);
    return NdSplitFns{nullptr, nullptr, nullptr, 0};
}

const void* generic_kernel(int dtype, bool softcap) {
    if (dtype == 0)
        return softcap ? (const void*)&ce_fwd_generic<float, true>
                       : (const void*)&ce_fwd_generic<float, false>;
    if (dtype == 1)
        return softcap ? (const void*)&ce_fwd_generic<__nv_bfloat16, true>
                       : (const void*)&ce_fwd_generic<__nv_bfloat16, false>;
    if (dtype == 2)
        return softcap ? (const void*)&ce_fwd_generic<__half, true>
                       : (const void*)&ce_fwd_generic<__half, false>;
    return nullptr;
}

const void* bwd_kernel(int dtype) {
    if (dtype == 0) return (const void*)&ce_bwd_scale<float>;
    if (dtype == 1) return (const void*)&ce_bwd_scale<__nv_bfloat16>;
    if (dtype == 2) return (const void*)&ce_bwd_scale<__half>;
    return nullptr;
}

}  // namespace gbce
