// Forward for N-D logits with the class dimension at axis 1, [N, C, d1..dk]
// (the tt-mlir pull request #9324 review comment: the reductions run over
// every non-class dimension; F.cross_entropy's N-D form). Each position
// (n, d1..dk) is one row of the 2-D definition, and its C logits sit
// `inner` = d1*...*dk elements apart, so a row is a strided column here.
//
// Layout of the work: a CTA owns a tile of 32 * VP consecutive positions
// (VP = 1, or the positions of one 16-byte vector when inner allows), the
// 32 lanes of every warp cover the tile's positions, and the warps split the
// classes (warp w takes classes w, w + 8, ...). Each load of a warp is thus
// one contiguous run of 32 * VP positions of one class: coalesced, whatever
// the class stride. Three phases per tile:
//   A  raw maximum and first argmax per position (the tile is copied to
//      shared memory on the way when it fits);
//   B  S = sum exp(z - M) and the smoothing sum sum w (z - M), from the
//      staged tile (or global memory);
//   C  the gradient, stored in place over the logits.
// The per-warp partials of phases A and B are merged per position in warp
// order, so every result is deterministic. Row definitions, loss terms and
// the gradient are those of the 2-D kernels (Liger-Kernel cross-entropy
// profile, §Forward Pass, §Backward Pass, §Key Patterns).
#pragma once

#include <climits>
#include <type_traits>

#include "ce_kernels.cuh"

namespace gbce {

// Loads and stores of VP consecutive positions of one class.
template <typename T, int VP>
struct NdIO {
    static constexpr bool kVec = VP > 1;
    static_assert(!kVec || VP == Vec<T>::N, "vector width must be 16 bytes");
    using Scalar = typename std::conditional<sizeof(T) == 4, uint32_t, uint16_t>::type;
    using Raw = typename std::conditional<kVec, uint4, Scalar>::type;

    __device__ __forceinline__ static Raw load(const void* base, int64_t i) {
        return *reinterpret_cast<const Raw*>(static_cast<const T*>(base) + i);
    }
    __device__ __forceinline__ static void store(void* base, int64_t i, const Raw& r) {
        *reinterpret_cast<Raw*>(static_cast<T*>(base) + i) = r;
    }
    __device__ __forceinline__ static void unpack(const Raw& r, float (&f)[VP]) {
        if constexpr (kVec) {
            Vec<T>::unpack(r, f);
        } else if constexpr (sizeof(T) == 4) {
            f[0] = __uint_as_float(r);
        } else if constexpr (std::is_same<T, __nv_bfloat16>::value) {
            f[0] = __uint_as_float(static_cast<uint32_t>(r) << 16);
        } else {
            f[0] = __half2float(__ushort_as_half(r));
        }
    }
    __device__ __forceinline__ static Raw pack(const float (&f)[VP]) {
        if constexpr (kVec) {
            return Vec<T>::pack(f);
        } else if constexpr (sizeof(T) == 4) {
            return __float_as_uint(f[0]);
        } else if constexpr (std::is_same<T, __nv_bfloat16>::value) {
            return __bfloat16_as_ushort(__float2bfloat16_rn(f[0]));
        } else {
            return __half_as_ushort(__float2half_rn(f[0]));
        }
    }
};

// Runs body(c, raw) over the classes c = first, first + step, ... < C, the
// loads of U classes issued before any of them is used.
template <int U, typename Raw, typename Load, typename Body>
__device__ __forceinline__ void nd_class_loop(int first, int step, int C, Load load, Body body) {
    int c = first;
#pragma unroll 1
    for (; c + (U - 1) * step < C; c += U * step) {
        Raw r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r[u] = load(c + u * step);
#pragma unroll
        for (int u = 0; u < U; ++u) body(c + u * step, r[u]);
    }
#pragma unroll 1
    for (; c < C; c += step) body(c, load(c));
}

template <typename T, int VP, bool SOFTCAP, bool ARGMAX>
__global__ void __launch_bounds__(kNdThreads)
ce_fwd_nd(const __grid_constant__ FwdArgs a) {
    using IO = NdIO<T, VP>;
    using Raw = typename IO::Raw;
    constexpr int NW = kNdWarps;
    constexpr int P = 32 * VP;               // positions per tile
    constexpr int U = VP > 1 ? 4 : 8;        // loads in flight per thread
    static_assert(P <= kNdThreads, "one merging thread per position");

    extern __shared__ __align__(16) unsigned char nd_smem[];
    float* red_a = reinterpret_cast<float*>(nd_smem);  // [NW][P]
    float* red_b = red_a + NW * P;                     // [NW][P]
    float* pos_shift = red_b + NW * P;                 // [P] M (0 when M = -inf)
    float* pos_ac = pos_shift + P;                     // [P] coefficient of exp(z - M)
    float* pos_tfix = pos_ac + P;                      // [P] correction at the target
    float* pos_bc = pos_tfix + P;                      // [P] smoothing constant
    int* pos_t = reinterpret_cast<int*>(pos_bc + P);   // [P] target, -1 if not counted
    int* pos_pred = pos_t + P;                         // [P] first argmax
    Raw* tile = reinterpret_cast<Raw*>(pos_pred + P);  // [C][32] when staged
    __shared__ double red_d[2 * NW];
    __shared__ long long red_n[NW];
    __shared__ int s_flag;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int wy = tid >> 5;
    const int C = static_cast<int>(a.V);
    const int64_t inner = a.inner;
    const int64_t rows = a.rows;
    const bool smooth = a.eps > 0.f;
    const bool wsmooth = smooth && a.weight != nullptr;
    const bool staged = a.nd_staged != 0;

    // D and the counted positions of the whole call come from the count
    // pre-pass (a.batch_counts); "none" needs neither
    float D = 0.f;
    int n_valid = 0;
    if (a.reduction != kRedNone) {
        D = static_cast<float>(a.batch_counts[0]);
        n_valid = static_cast<int>(a.batch_counts[1]);
    }
    // W = sum of the class weights, formed in the same order by every CTA
    float Wsum = static_cast<float>(C);
    if (wsmooth) {
        float s = 0.f;
        for (int c = tid; c < C; c += kNdThreads) s += __ldg(a.weight + c);
        Wsum = block_sum_fixed<kNdThreads>(s, red_a);
        __syncthreads();
    }
    const float inv_C = 1.f / static_cast<float>(C);
    const float scale = a.reduction == kRedMean ? 1.f / D : 1.f;
    const float Wf = wsmooth ? Wsum * inv_C : 1.f;

    double accL = 0.0, accZ = 0.0;
    long long accC = 0;
    const int64_t ntiles = (rows + P - 1) / P;
#pragma unroll 1
    for (int64_t ti = blockIdx.x; ti < ntiles; ti += gridDim.x) {
        const int64_t r0 = ti * P;
        const int64_t rl = r0 + static_cast<int64_t>(lane) * VP;  // this lane's first position
        const bool lane_ok = rl < rows;  // VP divides inner, hence rows
        int64_t lb = 0;                  // element offset of (rl, class 0)
        if (lane_ok) {
            const int64_t n = rl / inner;
            lb = n * C * inner + (rl - n * inner);
        }
        auto gload = [&](int c) -> Raw {
            return lane_ok ? IO::load(a.x, lb + static_cast<int64_t>(c) * inner) : Raw{};
        };
        auto sload = [&](int c) -> Raw { return tile[c * 32 + lane]; };

        // ---- phase A: raw maximum and first argmax of this warp's classes
        float xm[VP];
        int xi[VP];
#pragma unroll
        for (int v = 0; v < VP; ++v) {
            xm[v] = -INFINITY;
            xi[v] = INT_MAX;
        }
        nd_class_loop<U, Raw>(wy, NW, C, gload, [&](int c, const Raw& r) {
            if (staged) tile[c * 32 + lane] = r;
            float f[VP];
            IO::unpack(r, f);
#pragma unroll
            for (int v = 0; v < VP; ++v) {
                if (ARGMAX) {
                    if (f[v] > xm[v]) {  // classes arrive in increasing order
                        xm[v] = f[v];
                        xi[v] = c;
                    }
                } else {
                    xm[v] = fmaxf(xm[v], f[v]);
                }
            }
        });
#pragma unroll
        for (int v = 0; v < VP; ++v) {
            red_a[wy * P + lane * VP + v] = xm[v];
            reinterpret_cast<int*>(red_b)[wy * P + lane * VP + v] = xi[v];
        }
        __syncthreads();
        if (tid < P) {
            float m = red_a[tid];
            int mi = reinterpret_cast<int*>(red_b)[tid];
#pragma unroll
            for (int w = 1; w < NW; ++w) {
                const float o = red_a[w * P + tid];
                const int oi = reinterpret_cast<int*>(red_b)[w * P + tid];
                if (o > m || (o == m && oi < mi)) {
                    m = o;
                    mi = oi;
                }
            }
            // softcap is monotone: the largest z is the cap of the largest x
            const float M = SOFTCAP ? a.softcap * tanh_from_scaled(m * a.sc_k2) : m;
            pos_shift[tid] = M == -INFINITY ? 0.f : M;
            int tt = -1;
            const int64_t r = r0 + tid;
            if (r < rows) {
                const int64_t t = load_target(a, r);
                if (row_counts(a, t))
                    tt = static_cast<int>(t);
                else if (t != a.ignore_index)
                    atomicOr(&a.scratch->status, kDevErrTarget);
            }
            pos_t[tid] = tt;
            pos_pred[tid] = mi;
        }
        __syncthreads();

        // ---- phase B: S = sum exp(z - M), SZ = sum w (z - M)
        float sh[VP], S[VP], SZ[VP];
#pragma unroll
        for (int v = 0; v < VP; ++v) {
            sh[v] = pos_shift[lane * VP + v];
            S[v] = 0.f;
            SZ[v] = 0.f;
        }
        auto phase_b = [&](int c, const Raw& r) {
            float f[VP];
            IO::unpack(r, f);
            const float wc = wsmooth ? __ldg(a.weight + c) : 1.f;
#pragma unroll
            for (int v = 0; v < VP; ++v) {
                const float d = SOFTCAP ? fmaf(tanh_from_scaled(f[v] * a.sc_k2), a.softcap, -sh[v])
                                        : f[v] - sh[v];
                S[v] += ex2(d * kLog2e);
                if (smooth) SZ[v] = fmaf(wc, d, SZ[v]);
            }
        };
        if (staged)
            nd_class_loop<U, Raw>(wy, NW, C, sload, phase_b);
        else
            nd_class_loop<U, Raw>(wy, NW, C, gload, phase_b);
#pragma unroll
        for (int v = 0; v < VP; ++v) {
            red_a[wy * P + lane * VP + v] = S[v];
            red_b[wy * P + lane * VP + v] = SZ[v];
        }
        __syncthreads();
        if (tid < P) {
            float s = red_a[tid], sz = red_b[tid];
#pragma unroll
            for (int w = 1; w < NW; ++w) {
                s += red_a[w * P + tid];
                sz += red_b[w * P + tid];
            }
            const int64_t r = r0 + tid;
            const int tt = pos_t[tid];
            float ac = 0.f, tfix = 0.f, bc = 0.f;
            if (r < rows) {
                const bool counted = tt >= 0;
                const int mi = pos_pred[tid];
                if (counted) {
                    float xt;
                    if (staged) {  // element (tt, position tid) of the tile
                        using S1 = NdIO<T, 1>;
                        float f[1];
                        S1::unpack(reinterpret_cast<const typename S1::Raw*>(tile)[tt * P + tid], f);
                        xt = f[0];
                    } else {
                        const int64_t n = r / inner;
                        xt = Vec<T>::load1(a.x, n * C * inner + static_cast<int64_t>(tt) * inner +
                                                    (r - n * inner));
                    }
                    const float shift = pos_shift[tid];
                    const float zt = SOFTCAP ? a.softcap * tanh_from_scaled(xt * a.sc_k2) : xt;
                    const float wt = a.weight ? __ldg(a.weight + tt) : 1.f;
                    const float logS = logf(s);
                    float zl;
                    const float l = row_loss(a, shift, logS, zt, wt, wsmooth ? Wsum
                                                                             : static_cast<float>(C),
                                             sz, zl);
                    const bool correct = mi == tt;
                    if (a.reduction == kRedNone) {
                        a.loss[r] = l;
                        if (a.want_z) a.zloss[r] = zl;
                        if (a.want_acc) a.acc[r] = correct ? 1.f : 0.f;
                    } else {
                        accL += static_cast<double>(l);
                        accZ += static_cast<double>(zl);
                        accC += correct ? 1 : 0;
                    }
                    if (a.want_pred) a.pred[r] = mi;
                    const float lse = shift + logS;
                    ac = scale * ((1.f - a.eps) * wt + a.eps * Wf + 2.f * a.lam * lse) / s;
                    tfix = -scale * (1.f - a.eps) * wt;
                    bc = -scale * a.eps * inv_C;
                } else {
                    if (a.reduction == kRedNone) {
                        a.loss[r] = 0.f;
                        if (a.want_z) a.zloss[r] = 0.f;
                        if (a.want_acc) a.acc[r] = 0.f;
                    }
                    if (a.want_pred) a.pred[r] = -1;
                }
            }
            pos_ac[tid] = ac;
            pos_tfix[tid] = tfix;
            pos_bc[tid] = bc;
        }
        __syncthreads();

        // ---- phase C: the gradient, in place
        if (a.grad) {
            float ac[VP], tf[VP], bc[VP];
            int tv[VP];
#pragma unroll
            for (int v = 0; v < VP; ++v) {
                const int p = lane * VP + v;
                ac[v] = pos_ac[p];
                tf[v] = pos_tfix[p];
                bc[v] = pos_bc[p];
                tv[v] = pos_t[p];
            }
            auto phase_c = [&](int c, const Raw& r) {
                float f[VP];
                IO::unpack(r, f);
                const float wc = wsmooth ? __ldg(a.weight + c) : 1.f;
#pragma unroll
                for (int v = 0; v < VP; ++v) {
                    float d, th = 0.f;
                    if (SOFTCAP) {
                        th = tanh_from_scaled(f[v] * a.sc_k2);
                        d = fmaf(th, a.softcap, -sh[v]);
                    } else {
                        d = f[v] - sh[v];
                    }
                    float g = fmaf(ac[v], ex2(d * kLog2e), bc[v] * wc);
                    if (c == tv[v]) g += tf[v];
                    if (SOFTCAP) g *= fmaf(-th, th, 1.f);
                    // positions that do not count get exact zeros, whatever
                    // their logits hold
                    f[v] = tv[v] >= 0 ? g : 0.f;
                }
                if (lane_ok) IO::store(a.x, lb + static_cast<int64_t>(c) * inner, IO::pack(f));
            };
            if (staged)
                nd_class_loop<U, Raw>(wy, NW, C, sload, phase_c);
            else
                nd_class_loop<U, Raw>(wy, NW, C, gload, phase_c);
        }
        __syncthreads();  // the next tile overwrites the shared arrays
    }

    if (a.reduction != kRedNone) {
        // fixed-order CTA sum of the per-thread partials, then the last-CTA
        // epilogue over the grid
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            accL += __shfl_xor_sync(0xffffffffu, accL, o);
            accZ += __shfl_xor_sync(0xffffffffu, accZ, o);
            accC += __shfl_xor_sync(0xffffffffu, accC, o);
        }
        if (lane == 0) {
            red_d[wy] = accL;
            red_d[NW + wy] = accZ;
            red_n[wy] = accC;
        }
        __syncthreads();
        double L = 0.0, Z = 0.0;
        long long Cn = 0;
        if (tid == 0) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                L += red_d[w];
                Z += red_d[NW + w];
                Cn += red_n[w];
            }
        }
        __syncthreads();  // red_d is the epilogue's scratch next
        finish_scalars_cta(a, L, Z, Cn, D, n_valid, &s_flag, red_d, red_d + NW, red_n);
    }
}

// Kernel entry points of one logit type, by (vector loads, softcap, argmax).
template <typename T>
const void* nd_kernel_of(bool vec, bool softcap, bool argmax) {
    constexpr int VPV = Vec<T>::N;
    if (vec) {
        if (softcap)
            return argmax ? (const void*)&ce_fwd_nd<T, VPV, true, true>
                          : (const void*)&ce_fwd_nd<T, VPV, true, false>;
        return argmax ? (const void*)&ce_fwd_nd<T, VPV, false, true>
                      : (const void*)&ce_fwd_nd<T, VPV, false, false>;
    }
    if (softcap)
        return argmax ? (const void*)&ce_fwd_nd<T, 1, true, true>
                      : (const void*)&ce_fwd_nd<T, 1, true, false>;
    return argmax ? (const void*)&ce_fwd_nd<T, 1, false, true>
                  : (const void*)&ce_fwd_nd<T, 1, false, false>;
}

}  // namespace gbce
