// Fused softmax cross-entropy forward with the in-forward gradient: the
// streaming kernel.
//
// Method (Liger-Kernel cross-entropy kernel profile, §Forward Pass,
// §Backward Pass and §Key Patterns): per row a max-shifted log-sum-exp,
// the NLL with ignore_index, class weights on the target term, label
// smoothing and z-loss, the argmax, and the gradient of the reduced loss
// written in place over the logits.
//
// GB300 design:
//  * Warp specialisation. One producer warp keeps a ring of shared-memory
//    slots filled with 1-D bulk asynchronous copies (completion counted on
//    a `full` mbarrier per slot); 16 consumer warps compute, and each warp
//    hands a slot back through an `empty` mbarrier when it is done with it.
//  * Row groups. The consumer warps form ng groups; group g takes every
//    ng-th row of the CTA's rows, with its own ring slots, so several rows
//    are in flight per SM and one group's row-end merge overlaps the
//    others' streaming.
//  * Two passes per row. Pass 1 forms each thread's online-softmax
//    statistics (running max, sum of exp relative to it, first argmax,
//    smoothing sum); warps merge them with shuffles and the group with one
//    named barrier. Pass 2 recomputes exp from the logits (the SFU issues
//    about 30 ex2 per clock per SM, so the second exponential is cheap)
//    and stores the gradient with 16-byte coalesced stores. When a row
//    fits in the group's slots it stays there for both passes ("resident");
//    otherwise the producer streams it twice, the first time with an L2
//    evict-last hint so that the second read comes from L2, and HBM sees
//    one read and one write per element.
//  * Scalars. Per-row outputs come from the group leader; sums go through
//    per-CTA partials and the last-CTA fixed-order epilogue.
#pragma once

#include <climits>

#include "ce_kernels.cuh"

namespace gbce {

namespace {

constexpr uint32_t kStreamCopyChunk = 32768;

__device__ __forceinline__ int64_t imin64(int64_t x, int64_t y) { return x < y ? x : y; }

// exp2 arguments (z - m) * log2(e) for a pair. bf16 logits use one packed
// FFMA against the rounded m*log2(e) (that rounding is common to a thread's
// terms); fp32 logits subtract first.
template <typename T>
__device__ __forceinline__ float2 exp_arg2(float2 z, float m, float mL) {
    if (sizeof(T) == 2) return ffma2(z, make_float2(kLog2e, kLog2e), make_float2(-mL, -mL));
    return fmul2(fadd2(z, make_float2(-m, -m)), make_float2(kLog2e, kLog2e));
}

// Class weights of vector v (VE consecutive classes) from shared memory,
// where the 4-weight quarter h of vector v sits at float4 h * vrow + v, so
// that the lanes of a warp, which hold consecutive vectors, read
// consecutive 16-byte words.
template <int VE>
__device__ __forceinline__ void weights_of(const float4* w4, int v, int vrow, float (&w)[VE]) {
#pragma unroll
    for (int h = 0; h < VE / 4; ++h) {
        const float4 t = w4[h * vrow + v];
        w[4 * h] = t.x;
        w[4 * h + 1] = t.y;
        w[4 * h + 2] = t.z;
        w[4 * h + 3] = t.w;
    }
}

// Row statistics of one thread during pass 1 (see RowStats): the running
// reference m (the largest z seen; a finite sentinel before the first
// element), S = sum exp(z - m), the running sum of z for label smoothing, the
// element count, and the first vector holding the largest raw logit.
// add_chunk takes the thread's VPT vectors of one ring slot at once: one
// max and one rescale per slot, then VPT independent exp-sum chains of
// packed pairs.
template <typename T, bool SOFTCAP, int VPT, bool WS>
struct PassOne {
    using VT = Vec<T>;
    static constexpr int VE = VT::N;
    float m = -3.0e38f, mL = -3.0e38f * kLog2e, S = 0.f, sumz = 0.f, xmax = -INFINITY;
    int best = INT_MAX, nel = 0;  // best: first element index of the largest raw logit

    // q[k] is vector vidx0 + k * stride; unless FULL, it exists only when
    // vidx0 + k * stride < vend (the thread's vectors of the slot, in
    // increasing index order).
    //
    // With WS (class weights and label smoothing), sumz collects the
    // absolute sum of w * z over the thread's elements, the weights coming
    // from shared memory (w4, see weights_of); otherwise, when smooth, the
    // plain sum of z.
    template <bool FULL>
    __device__ __forceinline__ void add_chunk(const uint4 (&q)[VPT], int vidx0, int vend,
                                              int stride, const FwdArgs& a, bool smooth_rt,
                                              const float4* w4, int vrow, bool want_arg) {
        const bool smooth = WS || smooth_rt;
        typename VT::MaxAcc macc = VT::max_init();
        int nk = 0;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            if (FULL || vidx0 + k * stride < vend) {
                ++nk;
                macc = VT::max_fold(macc, q[k]);
            }
        }
        const float cm = VT::max_value(macc);
        if (!want_arg) {
            // no argmax asked for: only the largest raw logit (the softcap
            // of it is the row's largest z)
            xmax = fmaxf(xmax, cm);
        } else if (__any_sync(0xffffffffu, cm > xmax)) {
            const bool better = cm > xmax;
            // a new thread maximum (frequent at a row's start, rare later):
            // find the first vector and element that hold it
            if (better) {
                int ck = VPT - 1;
                uint4 qb = q[VPT - 1];
#pragma unroll
                for (int k = VPT - 1; k >= 0; --k) {
                    if ((FULL || vidx0 + k * stride < vend) && VT::vmax(q[k]) == cm) {
                        ck = k;
                        qb = q[k];
                    }
                }
                float fb[VE];
                VT::unpack(qb, fb);
                int j0 = VE - 1;
#pragma unroll
                for (int j = VE - 1; j >= 0; --j)
                    if (fb[j] == cm) j0 = j;
                xmax = cm;
                best = (vidx0 + ck * stride) * VE + j0;
            }
        }
        const float mz = SOFTCAP ? a.softcap * tanh_from_scaled(cm * a.sc_k2) : cm;
        const float mn = fmaxf(m, mz);
        S *= ex2((m - mn) * kLog2e);
        m = mn;
        mL = fmaxf(mn, -1.0e30f) * kLog2e;
        // softcap: the exp2 argument c1 r + c0 and z = s - 2 s r (softcap_r2)
        const float sc_c1 = -2.f * a.sc_slog2e;
        const float sc_c0 = fmaf(-mn, kLog2e, a.sc_slog2e);
        float2 sk[VPT], zk[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            sk[k] = make_float2(0.f, 0.f);
            zk[k] = make_float2(0.f, 0.f);
            if (FULL || vidx0 + k * stride < vend) {
                float f[VE], w[VE];
                VT::unpack(q[k], f);
                if (WS) weights_of<VE>(w4, vidx0 + k * stride, vrow, w);
#pragma unroll
                for (int j = 0; j < VE; j += 2) {
                    float2 z;
                    if constexpr (SOFTCAP) {
                        const float2 r = softcap_r2(f[j], f[j + 1], a.sc_k2);
                        const float2 ar = ffma2(r, make_float2(sc_c1, sc_c1),
                                                make_float2(sc_c0, sc_c0));
                        sk[k] = fadd2(sk[k], make_float2(ex2(ar.x), ex2(ar.y)));
                        if (WS || smooth)
                            z = ffma2(r, make_float2(-2.f * a.softcap, -2.f * a.softcap),
                                      make_float2(a.softcap, a.softcap));
                    } else {
                        z = make_float2(f[j], f[j + 1]);
                        const float2 ar = exp_arg2<T>(z, m, mL);
                        sk[k] = fadd2(sk[k], make_float2(ex2(ar.x), ex2(ar.y)));
                    }
                    if (WS)
                        zk[k] = ffma2(make_float2(w[j], w[j + 1]), z, zk[k]);
                    else if (smooth)
                        zk[k] = fadd2(zk[k], z);
                }
            }
        }
        float2 acc = sk[0], zacc = zk[0];
#pragma unroll
        for (int k = 1; k < VPT; ++k) {
            acc = fadd2(acc, sk[k]);
            if (smooth) zacc = fadd2(zacc, zk[k]);
        }
        S += acc.x + acc.y;
        if (smooth) sumz += zacc.x + zacc.y;
        nel += nk * VE;
    }

};

// Row statistics of a warp or group, all relative to M = softcap(X), the
// largest z: S = sum exp(z - M), SZ = sum (z - M) (label smoothing), n the
// element count, X the largest raw logit and I its first index.
struct RowSums {
    float M, S, SZ, n, X;
    int I;
};

template <bool SOFTCAP>
__device__ __forceinline__ float capped1(float x, const FwdArgs& a) {
    return SOFTCAP ? a.softcap * tanh_from_scaled(x * a.sc_k2) : x;
}

// Merge over the lanes of a warp, each lane holding (m, S, SZ, n, x, i)
// relative to its own m: the raw maximum X in one warp reduction and the
// first index holding it in another, one rescale per lane, then a
// butterfly of plain sums over `span` lanes (32, or the width of a block of
// lanes that all blocks repeat). Every lane ends with the same bits.
template <bool SOFTCAP>
__device__ __forceinline__ RowSums warp_merge(float m, float S, float SZ, float n, float x, int i,
                                              bool smooth, const FwdArgs& a, int span = 32) {
    __syncwarp();  // converged for the warp reductions
    const float X = warp_max_f32(x);
    const int I = warp_min_s32(x == X ? i : INT_MAX);
    const float M = capped1<SOFTCAP>(X, a);
    const bool live = S > 0.f && M != -INFINITY;
    float s = live ? S * ex2((m - M) * kLog2e) : 0.f;
    float sz = (smooth && live) ? fmaf(n, m - M, SZ) : 0.f;
    float nn = n;
#pragma unroll 1
    for (int o = span >> 1; o > 0; o >>= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, o);
        if (smooth) {
            sz += __shfl_xor_sync(0xffffffffu, sz, o);
            nn += __shfl_xor_sync(0xffffffffu, nn, o);
        }
    }
    return RowSums{M, s, sz, nn, X, I};
}

// Pass 2 for the thread's VPT vectors of one slot: gradient
// As * exp(z - M) + Bc (times dz/dx under softcap), packed and stored.
// With WS the constant term is Bc * w_k (class weights from shared memory;
// vg0 is the row vector index of the thread's first vector of the slot).
// spol: the L2 policy of the stores.
// Four fp32 gradient values as four bf16 or fp16 (gout of FwdArgs).
__device__ __forceinline__ uint2 pack4_16(const float (&g)[4], int bf16) {
    uint2 o;
    if (bf16) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(g[0], g[1]);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(g[2], g[3]);
        o.x = *reinterpret_cast<const uint32_t*>(&lo);
        o.y = *reinterpret_cast<const uint32_t*>(&hi);
    } else {
        const __half2 lo = __floats2half2_rn(g[0], g[1]);
        const __half2 hi = __floats2half2_rn(g[2], g[3]);
        o.x = *reinterpret_cast<const uint32_t*>(&lo);
        o.y = *reinterpret_cast<const uint32_t*>(&hi);
    }
    return o;
}

template <typename T, bool SOFTCAP, int VPT, bool FULL, bool WS>
__device__ __forceinline__ void grad_chunk(const uint4* ch, uint4* outv, int tg, int nv, int GT,
                                           float M, float ML, float As, float Bc,
                                           const FwdArgs& a, const float4* w4, int vrow,
                                           int vg0, uint64_t spol, uint2* gov) {
    using VT = Vec<T>;
    constexpr int VE = VT::N;
    // softcap (softcap_r2): exp2 argument c1 r + c0, constants times 4
    const float sc_c1 = -2.f * a.sc_slog2e;
    const float sc_c0 = fmaf(-M, kLog2e, a.sc_slog2e);
    const float As4 = 4.f * As, Bc4 = 4.f * Bc;
    uint4 q[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k)
        if (FULL || tg + k * GT < nv) q[k] = ch[tg + k * GT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        if (FULL || tg + k * GT < nv) {
            float f[VE], gr[VE], w[VE];
            VT::unpack(q[k], f);
            if (WS) weights_of<VE>(w4, vg0 + k * GT, vrow, w);
#pragma unroll
            for (int j = 0; j < VE; j += 2) {
                float2 g;
                if constexpr (SOFTCAP) {
                    // (As e + Bc) (1 - tanh^2) = (4 As e + 4 Bc) (r - r^2)
                    const float2 r = softcap_r2(f[j], f[j + 1], a.sc_k2);
                    const float2 ar = ffma2(r, make_float2(sc_c1, sc_c1), make_float2(sc_c0, sc_c0));
                    const float2 bc = WS ? fmul2(make_float2(Bc4, Bc4), make_float2(w[j], w[j + 1]))
                                         : make_float2(Bc4, Bc4);
                    g = ffma2(make_float2(As4, As4), make_float2(ex2(ar.x), ex2(ar.y)), bc);
                    g = fmul2(g, ffma2(make_float2(-r.x, -r.y), r, r));
                } else {
                    const float2 ar = exp_arg2<T>(make_float2(f[j], f[j + 1]), M, ML);
                    const float2 bc = WS ? fmul2(make_float2(Bc, Bc), make_float2(w[j], w[j + 1]))
                                         : make_float2(Bc, Bc);
                    g = ffma2(make_float2(As, As), make_float2(ex2(ar.x), ex2(ar.y)), bc);
                }
                gr[j] = g.x;
                gr[j + 1] = g.y;
            }
            if constexpr (VE == 4) {
                if (gov) {  // 16-bit gradient output beside fp32 logits
                    const float g4[4] = {gr[0], gr[1], gr[2], gr[3]};
                    gov[k * GT] = pack4_16(g4, a.gout_bf16);
                    continue;
                }
            }
            st_v4_hint(outv + k * GT, VT::pack(gr), spol);
        }
    }
}

// Log-softmax mode, pass 2 for the thread's VPT vectors of one slot:
// out = (z - M) - log S, packed and stored.
template <typename T, int VPT, bool FULL>
__device__ __forceinline__ void lsm_chunk(const uint4* ch, uint4* outv, int tg, int nv, int GT,
                                          float M, float logS) {
    using VT = Vec<T>;
    constexpr int VE = VT::N;
    uint4 q[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k)
        if (FULL || tg + k * GT < nv) q[k] = ch[tg + k * GT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        if (FULL || tg + k * GT < nv) {
            float f[VE];
            VT::unpack(q[k], f);
#pragma unroll
            for (int j = 0; j < VE; j += 2) {
                const float2 d = fadd2(fadd2(make_float2(f[j], f[j + 1]), make_float2(-M, -M)),
                                       make_float2(-logS, -logS));
                f[j] = d.x;
                f[j + 1] = d.y;
            }
            outv[k * GT] = VT::pack(f);
        }
    }
}

// Ring position of a group: slot within the group's slots and the phase bit
// of its current use, advanced without division.
struct RingPos {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next(int sg) {
        if (++slot == sg) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

}  // namespace

// NW consumer warps plus the producer warp; the register file is split
// across the SM's four sub-partitions, so 17 warps allow 96 registers a
// thread and 9 warps allow 168.
//
// WS: class weights with label smoothing. The weights then sit in shared
// memory after the ring (V floats, laid out for weights_of), loaded once per
// CTA, and each CTA forms their total W in the same fixed order.
//
// LSM: the log-softmax of every row (the unfused _log_softmax), written to
// a.out: no targets are read, no loss is formed, and pass 2 stores
// (x - M) - log S instead of the gradient.
// GO: fp32 logits whose gradient goes to a.gout in 16 bits (FwdArgs::gout);
// a variant of its own, so that the plain kernels carry none of it.
template <typename T, bool SOFTCAP, int VPT, int NW, bool WS, bool LSM = false, bool GO = false>
__global__ void __launch_bounds__(32 * (NW + 1), 1)
ce_fwd_stream(const __grid_constant__ FwdArgs a) {
    using VT = Vec<T>;
    constexpr int VE = VT::N;
    constexpr int NTC = 32 * NW;  // consumer threads

    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full_bar[kStreamMaxSlots];
    __shared__ __align__(8) uint64_t empty_bar[kStreamMaxSlots];
    __shared__ __align__(16) RowSums grec[kStreamMaxGroups][2][NW];
    __shared__ float red_p[NW];
    __shared__ double gpart_l[kStreamMaxGroups], gpart_z[kStreamMaxGroups];
    __shared__ int s_failed;
    __shared__ float s_D;
    __shared__ int s_nvalid;
    __shared__ uint32_t s_issued[kStreamMaxSlots];  // 0, or 2 + phase of the last use
    __shared__ int s_correct[kStreamMaxGroups];
    __shared__ double s_wsum[NW];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int ng = a.ng;
    const int G = NW / ng;  // warps per group
    const int GT = 32 * G;  // threads per group
    const int sg = a.sg;
    const int nchunk = a.nchunk;
    const int chunk_vec = a.chunk_vec;
    const uint32_t chunk_bytes = static_cast<uint32_t>(chunk_vec) * 16u;
    const int64_t vec_row = a.V / VE;
    const int64_t cid = blockIdx.x;
    const int64_t ncta = gridDim.x;
    // a second pass over the row (the gradient, or the log-softmax output);
    // without it (loss and metrics only) every row is streamed once
    const bool two_pass = LSM || a.grad;

    if (tid == 0) {
        for (int i = 0; i < ng * sg; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), static_cast<uint32_t>(G));
            s_issued[i] = 0;
        }
        for (int g = 0; g < kStreamMaxGroups; ++g) s_correct[g] = 0;
        s_failed = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NW) {
        // ------------------------------------------------------------ producer
        // The warp's lanes read the targets of the CTA's next 32 rows at once
        // (which rows count); lane 0 then issues the copies of those rows.
        const uint64_t pol_keep = l2_evict_last_policy();
        const uint64_t pol_once = l2_evict_first_policy();
        int pslot[kStreamMaxGroups];
        uint32_t pphase[kStreamMaxGroups];
#pragma unroll
        for (int k = 0; k < kStreamMaxGroups; ++k) {
            pslot[k] = 0;
            pphase[k] = 0;
        }
        int failed = 0;
        int g = 0;
        bool stall = a.test_stall && cid == 0;  // test hook (FwdArgs::test_stall)
        for (int64_t rb = cid; rb < a.rows && !failed; rb += 32 * ncta) {
            const int64_t rl = rb + lane * ncta;
            const bool lane_counts = rl < a.rows && (LSM || row_counts(a, load_target(a, rl)));
            const uint32_t counted = __ballot_sync(0xffffffffu, lane_counts);
            if (lane == 0) {
                for (int j = 0; j < 32 && !failed; ++j) {
                    const int64_t r = rb + j * ncta;
                    if (r >= a.rows) break;
                    const int gg = g;
                    g = (g + 1 == ng) ? 0 : g + 1;
                    if (!((counted >> j) & 1u)) continue;
                    const int passes = (a.resident || !two_pass) ? 1 : 2;
                    for (int p = 0; p < passes && !failed; ++p) {
                        for (int c = 0; c < nchunk; ++c) {
                            int ls = 0;
                            uint32_t ph = 0;
#pragma unroll
                            for (int k = 0; k < kStreamMaxGroups; ++k) {
                                if (k == gg) {
                                    ls = pslot[k];
                                    ph = pphase[k];
                                    if (++pslot[k] == sg) {
                                        pslot[k] = 0;
                                        pphase[k] ^= 1u;
                                    }
                                }
                            }
                            const int slot = gg * sg + ls;
                            if (!mbar_wait_bounded(smem_u32(&empty_bar[slot]), ph ^ 1u,
                                                   a.timeout_ns)) {
                                failed = 1;
                                break;
                            }
                            const int64_t v0 = static_cast<int64_t>(c) * chunk_vec;
                            const uint32_t bytes =
                                static_cast<uint32_t>(imin64(chunk_vec, vec_row - v0)) * 16u;
                            const uint32_t fb = smem_u32(&full_bar[slot]);
                            if (stall) {
                                stall = false;
                                continue;
                            }
                            mbar_arrive_expect_tx(fb, bytes);
                            const char* src = reinterpret_cast<const char*>(a.x) +
                                              (r * a.V + v0 * VE) * static_cast<int64_t>(sizeof(T));
                            const uint32_t dst =
                                smem_u32(ring + static_cast<size_t>(slot) * chunk_bytes);
                            const uint64_t pol = passes == 2 && p == 0 ? pol_keep : pol_once;
                            for (uint32_t off = 0; off < bytes; off += kStreamCopyChunk)
                                bulk_g2s(dst + off, src + off, min(kStreamCopyChunk, bytes - off),
                                         fb, pol);
                            s_issued[slot] = 2u + ph;  // nonzero: used; low bit: phase of the last use
                        }
                    }
                }
            }
            failed = __shfl_sync(0xffffffffu, failed, 0);
        }
        if (failed && lane == 0) {
            atomicOr(&a.scratch->status, kDevErrTimeout);
            s_failed = 1;
        }
    } else {
        // ------------------------------------------------------------ consumers
        const NamedSync all_consumers{15, NTC};
        float D = 0.f;
        int n_valid = 0;
        if (a.reduction != kRedNone) denominators<NTC>(a, red_p, D, n_valid, all_consumers);
        if (tid == 0) {
            s_D = D;
            s_nvalid = n_valid;
        }
        const float scale = a.reduction == kRedMean ? 1.f / D : 1.f;  // unused when D == 0
        const float inv_V = 1.f / static_cast<float>(a.V);
        const bool smooth = WS || a.eps != 0.f;
        const bool want_arg = a.want_pred || a.want_acc;
        const int vrow_w = static_cast<int>(vec_row);
        float4* w4 = reinterpret_cast<float4*>(ring + static_cast<size_t>(ng) * sg * chunk_bytes);
        float Wtot = static_cast<float>(a.V);
        if (WS) {
            // weights into shared memory; W = sum of the weights: a float sum
            // per thread over a fixed set of classes, then the threads' sums
            // added in double in thread order
            float* wsm = reinterpret_cast<float*>(w4);
            float wsum = 0.f;
            const int V = static_cast<int>(a.V);
            auto put = [&](int i, float w) {
                const int v = i / VE, e = i % VE;
                wsm[((e >> 2) * vrow_w + v) * 4 + (e & 3)] = w;
                wsum += w;
            };
            if ((reinterpret_cast<uintptr_t>(a.weight) & 15u) == 0) {
                const float4* src = reinterpret_cast<const float4*>(a.weight);
#pragma unroll 4
                for (int i4 = tid; i4 < V / 4; i4 += NTC) {
                    const float4 w = __ldg(src + i4);
                    put(4 * i4, w.x);
                    put(4 * i4 + 1, w.y);
                    put(4 * i4 + 2, w.z);
                    put(4 * i4 + 3, w.w);
                }
                for (int i = (V / 4) * 4 + tid; i < V; i += NTC) put(i, __ldg(a.weight + i));
            } else {
#pragma unroll 4
                for (int i = tid; i < V; i += NTC) put(i, __ldg(a.weight + i));
            }
            double ws = wsum;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
            if (lane == 0) s_wsum[warp] = ws;
            all_consumers();
            double wt_all = 0.0;
#pragma unroll
            for (int w = 0; w < NW; ++w) wt_all += s_wsum[w];
            Wtot = static_cast<float>(wt_all);
        }

        const int g = warp / G;
        const int wg = warp % G;
        const int tg = tid - g * GT;
        const NamedSync group_sync{1 + g, GT};
        const bool gleader = tid == g * GT;
        double accL = 0.0, accZ = 0.0;
        long long accC = 0;
        RingPos pos;
        bool failed = false;
        int rp = 0;
        const int vrow = static_cast<int>(vec_row);
        // Gradient stores go with an L2 evict-first hint: nothing reads them
        // in this kernel, and the rows that the second pass re-reads from L2
        // stay (measured: 1023 x 128256 fp32 213 -> 203 us, 4096 x 131072
        // bf16 -2.8%)
        const uint64_t spol = l2_evict_first_policy();
        // the thread of the group that handles vector v of a row (pass 1 and
        // pass 2 use the same assignment)
        // (GT is a power of two and every slot but a lone one spans a
        // multiple of GT vectors)
        auto owner_of = [&](int v) { return v & (GT - 1); };

        // the next row's target is read one row ahead
        const int64_t rstep = static_cast<int64_t>(ng) * ncta;
        const int64_t r_first = cid + static_cast<int64_t>(g) * ncta;
        int64_t t_next = (!LSM && r_first < a.rows) ? load_target(a, r_first) : 0;
        for (int64_t r = r_first; r < a.rows; r += rstep) {
            const int64_t t = t_next;
            if (!LSM && r + rstep < a.rows) t_next = load_target(a, r + rstep);
            const bool counts = LSM || row_counts(a, t);
            T* xrow = reinterpret_cast<T*>(a.x) + r * a.V;
            uint4* rowv = reinterpret_cast<uint4*>(xrow);
            // the 16-bit gradient's row (fp32 logits with gout only)
            uint2* gorow = (GO && sizeof(T) == 4)
                               ? reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.gout) + r * a.V)
                               : nullptr;
            if (!LSM && gleader && t != a.ignore_index && !counts)
                atomicOr(&a.scratch->status, kDevErrTarget);
            if (!counts) {
                // Ignored row: exact +0 gradient, zero per-row outputs, pred -1.
                if (a.grad)
                    for (int v = tg; v < vrow; v += GT) {
                        if (gorow)
                            gorow[v] = make_uint2(0u, 0u);
                        else
                            st_v4_hint(rowv + v, make_uint4(0u, 0u, 0u, 0u), spol);
                    }
                if (gleader) {
                    if (a.reduction == kRedNone) {
                        a.loss[r] = 0.f;
                        if (a.want_z) a.zloss[r] = 0.f;
                        if (a.want_acc) a.acc[r] = 0.f;
                    }
                    if (a.want_pred) a.pred[r] = -1;
                }
                continue;
            }
            const int tvec = static_cast<int>(t / VE);
            const bool t_owner = !LSM && tg == owner_of(tvec);
            float xt = 0.f;
            if (!LSM && (gleader || t_owner)) xt = VT::load1(xrow, t);  // before any store to this row
            const float wt = (!LSM && a.weight) ? __ldg(a.weight + t) : 1.f;

            // ---- pass 1: thread statistics over the row's slots
            PassOne<T, SOFTCAP, VPT, WS> st;
            const RingPos pos0 = pos;
            for (int c = 0, v0 = 0; c < nchunk; ++c, v0 += chunk_vec) {
                const int slot = g * sg + pos.slot;
                if (!failed && !mbar_wait_bounded(smem_u32(&full_bar[slot]), pos.phase,
                                                  a.timeout_ns)) {
                    failed = true;
                    atomicOr(&a.scratch->status, kDevErrTimeout);
                }
                const uint4* ch = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(slot) * chunk_bytes);
                const int nv = min(chunk_vec, vrow - v0);
                // this thread's vectors of the slot: tg, tg + GT, ... below nv
                uint4 q[VPT];
                if (nv == VPT * GT) {
#pragma unroll
                    for (int k = 0; k < VPT; ++k) q[k] = ch[tg + k * GT];
                    st.template add_chunk<true>(q, v0 + tg, v0 + nv, GT, a, smooth, w4,
                                                vrow_w, want_arg);
                } else {
#pragma unroll
                    for (int k = 0; k < VPT; ++k)
                        if (tg + k * GT < nv) q[k] = ch[tg + k * GT];
                    st.template add_chunk<false>(q, v0 + tg, v0 + nv, GT, a, smooth, w4,
                                                 vrow_w, want_arg);
                }
                if (!a.resident || !two_pass) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
                }
                pos.next(sg);
            }

            // ---- merge: warp, then one group barrier, then the group's warp records
            // (WS: sumz is absolute and merges unshifted, with n = 0)
            const RowSums wsum = warp_merge<SOFTCAP>(
                st.m, st.S,
                WS ? st.sumz : (smooth ? st.sumz - static_cast<float>(st.nel) * st.m : 0.f),
                WS ? 0.f : static_cast<float>(st.nel), st.xmax, st.best, smooth, a);
            if (lane == 0) grec[g][rp][wg] = wsum;
            group_sync();
            // every block of G lanes holds the G records once
            const RowSums rec = grec[g][rp][lane & (G - 1)];
            const RowSums tot = warp_merge<SOFTCAP>(rec.M, rec.S, rec.SZ, rec.n, rec.X, rec.I,
                                                    smooth, a, G);
            rp ^= 1;
            const float M = tot.M;
            const float logS = logf(tot.S);

            if (!LSM && gleader) {
                const float zt = SOFTCAP ? a.softcap * tanh_from_scaled(xt * a.sc_k2) : xt;
                float zl;
                const float l = row_loss(a, M, logS, zt, wt, Wtot,
                                         WS ? fmaf(-Wtot, M, tot.SZ) : tot.SZ, zl);
                const bool correct = tot.I < vrow * VE && static_cast<int64_t>(tot.I) == t;
                if (a.reduction == kRedNone) {
                    a.loss[r] = l;
                    if (a.want_z) a.zloss[r] = zl;
                    if (a.want_acc) a.acc[r] = correct ? 1.f : 0.f;
                } else {
                    accL += static_cast<double>(l);
                    accZ += static_cast<double>(zl);
                    accC += correct ? 1 : 0;
                }
                if (a.want_pred) a.pred[r] = tot.I < vrow * VE ? tot.I : -1;
            }

            // ---- pass 2: gradient in place
            //   scale * [ (1-eps) w_t (p - onehot) + (eps/V)(V p - 1) + 2 lam lse p ] * dz/dx
            // The one-hot term is added by the owner of the target's vector,
            // which rewrites that element after storing the vector.
            const float lse = M + logS;
            const float As =
                scale * ((1.f - a.eps) * wt + a.eps * (WS ? Wtot * inv_V : 1.f) + 2.f * a.lam * lse) /
                tot.S;
            const float Bc = -scale * a.eps * inv_V;
            const float ML = M * kLog2e;
            if (a.resident && two_pass) pos = pos0;
            for (int c = 0, v0 = 0; two_pass && c < nchunk; ++c, v0 += chunk_vec) {
                const int slot = g * sg + pos.slot;
                if (!a.resident && !failed &&
                    !mbar_wait_bounded(smem_u32(&full_bar[slot]), pos.phase, a.timeout_ns)) {
                    failed = true;
                    atomicOr(&a.scratch->status, kDevErrTimeout);
                }
                const uint4* ch = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(slot) * chunk_bytes);
                const int nv = min(chunk_vec, vrow - v0);
                if (LSM) {
                    uint4* ov = reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.out) + r * a.V) +
                                v0 + tg;
                    if (!failed) {
                        if (nv == VPT * GT)
                            lsm_chunk<T, VPT, true>(ch, ov, tg, nv, GT, M, logS);
                        else
                            lsm_chunk<T, VPT, false>(ch, ov, tg, nv, GT, M, logS);
                    }
                } else if (a.grad && !failed) {
                    uint2* gov = gorow ? gorow + v0 + tg : nullptr;
                    if (nv == VPT * GT)
                        grad_chunk<T, SOFTCAP, VPT, true, WS>(ch, rowv + v0 + tg, tg, nv, GT, M,
                                                              ML, As, Bc, a, w4, vrow_w, v0 + tg, spol,
                                                              gov);
                    else
                        grad_chunk<T, SOFTCAP, VPT, false, WS>(ch, rowv + v0 + tg, tg, nv, GT, M,
                                                               ML, As, Bc, a, w4, vrow_w, v0 + tg, spol,
                                                               gov);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
                pos.next(sg);
            }
            if (a.grad && !failed && t_owner) {
                float e, fac = 1.f;
                if (SOFTCAP) {
                    const float th = tanh_from_scaled(xt * a.sc_k2);
                    fac = fmaf(-th, th, 1.f);
                    e = ex2((a.softcap * th - M) * kLog2e);
                } else {
                    e = ex2((xt - M) * kLog2e);
                }
                const float gt = (fmaf(As, e, WS ? Bc * wt : Bc) - scale * (1.f - a.eps) * wt) * fac;
                if (gorow) {
                    uint16_t* go = reinterpret_cast<uint16_t*>(gorow);
                    if (a.gout_bf16)
                        go[t] = __bfloat16_as_ushort(__float2bfloat16_rn(gt));
                    else
                        go[t] = __half_as_ushort(__float2half_rn(gt));
                } else {
                    VT::store1(xrow, t, gt);
                }
            }
        }
        if (gleader) {
            gpart_l[g] = accL;
            gpart_z[g] = accZ;
            s_correct[g] = static_cast<int>(accC);
        }
        if (failed && lane == 0) s_failed = 1;
    }
    __syncthreads();

    if (s_failed && tid == NW * 32) {
        // drain copies that may still be in flight: wait (bounded) for the
        // last issued use of every slot
        for (int i = 0; i < ng * sg; ++i) {
            const uint32_t used = s_issued[i];
            if (used) (void)mbar_wait_bounded(smem_u32(&full_bar[i]), used & 1u, a.timeout_ns);
        }
    }
    if (a.reduction != kRedNone && tid < 32) {
        double L = 0.0, Z = 0.0;
        long long C = 0;
        for (int g = 0; g < ng; ++g) {
            L += gpart_l[g];
            Z += gpart_z[g];
            C += s_correct[g];
        }
        finish_scalars(a, cid, ncta, L, Z, C, s_D, s_nvalid);
    }
}

}  // namespace gbce
