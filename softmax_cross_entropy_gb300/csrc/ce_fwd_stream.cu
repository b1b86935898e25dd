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
#include <climits>

#include "ce_kernels.cuh"

namespace gbce {

namespace {

constexpr uint32_t kStreamCopyChunk = 32768;

__device__ __forceinline__ int64_t imin64(int64_t x, int64_t y) { return x < y ? x : y; }

// Row statistics of one thread during pass 1 (see RowStats): the running
// reference m (the largest z seen), S = sum exp(z - m), the running sum of
// z for label smoothing, the element count, and the first argmax of x.
template <typename T, bool SOFTCAP>
struct PassOne {
    using VT = Vec<T>;
    static constexpr int VE = VT::N;
    float m = -INFINITY, mL = 0.f, S = 0.f, sumz = 0.f, n = 0.f, xmax = -INFINITY;
    int idx = INT_MAX;

    // exp argument: bf16 logits use one FFMA (the rounding of m*log2e is
    // common to a thread's terms); fp32 logits subtract first.
    __device__ __forceinline__ float arg(float z) const {
        if (sizeof(T) == 2) return fmaf(z, kLog2e, -mL);
        return (z - m) * kLog2e;
    }

    __device__ __forceinline__ void add(const uint4& q, int col0, const FwdArgs& a,
                                        bool smooth) {
        float f[VE];
        VT::unpack(q, f);
        const float vm = VT::vmax(q);
        if (vm > xmax) {  // first occurrence of a new thread maximum
            xmax = vm;
            int j0 = VE - 1;
#pragma unroll
            for (int j = VE - 1; j >= 0; --j)
                if (f[j] == vm) j0 = j;
            idx = col0 + j0;
            const float mz = SOFTCAP ? a.softcap * tanh_from_scaled(vm * a.sc_k2) : vm;
            if (mz > m) {
                if (S > 0.f) S *= ex2((m - mz) * kLog2e);
                m = mz;
                mL = mz * kLog2e;
            }
        }
#pragma unroll
        for (int j = 0; j < VE; ++j) {
            float z;
            if (SOFTCAP) {
                z = a.softcap * tanh_from_scaled(f[j] * a.sc_k2);
            } else {
                z = f[j];
            }
            S += ex2(arg(z));
            if (smooth) sumz += z;
        }
        n += static_cast<float>(VE);
    }

    __device__ __forceinline__ RowStats stats(bool smooth) const {
        RowStats r = empty_stats();
        r.xmax = xmax;
        r.idx = idx;
        if (m != -INFINITY) {
            r.m = m;
            r.S = S;
            r.Wn = n;
            r.SZ = smooth ? sumz - n * m : 0.f;
        }
        return r;
    }
};

}  // namespace

template <typename T, bool SOFTCAP>
__global__ void __launch_bounds__(32 * (kStreamWarps + 1), 1)
ce_fwd_stream(const __grid_constant__ FwdArgs a) {
    using VT = Vec<T>;
    constexpr int VE = VT::N;
    constexpr int NW = kStreamWarps;
    constexpr int NTC = 32 * NW;  // consumer threads

    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full_bar[kStreamMaxSlots];
    __shared__ __align__(8) uint64_t empty_bar[kStreamMaxSlots];
    __shared__ __align__(16) RowStats grec[kStreamMaxGroups][2][NW];
    __shared__ float red_p[NW];
    __shared__ double gpart_l[kStreamMaxGroups], gpart_z[kStreamMaxGroups];
    __shared__ long long gpart_c[kStreamMaxGroups];
    __shared__ int s_failed;
    __shared__ float s_D;
    __shared__ int s_nvalid;
    __shared__ uint32_t s_issued[kStreamMaxSlots];  // last issued use of a slot, +1

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

    if (tid == 0) {
        for (int i = 0; i < ng * sg; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), static_cast<uint32_t>(G));
            s_issued[i] = 0;
        }
        s_failed = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_keep = l2_evict_last_policy();
            const uint64_t pol_once = l2_evict_first_policy();
            uint32_t seq[kStreamMaxGroups];
#pragma unroll
            for (int g = 0; g < kStreamMaxGroups; ++g) seq[g] = 0;
            bool failed = false;
            int g = 0;
            for (int64_t r = cid; r < a.rows && !failed; r += ncta) {
                const int gg = g;
                g = (g + 1 == ng) ? 0 : g + 1;
                if (!row_counts(a, load_target(a, r))) continue;
                const int passes = a.resident ? 1 : 2;
                for (int p = 0; p < passes && !failed; ++p) {
                    for (int c = 0; c < nchunk; ++c) {
                        uint32_t sq = 0;
#pragma unroll
                        for (int k = 0; k < kStreamMaxGroups; ++k)
                            if (k == gg) sq = seq[k]++;
                        const int slot = gg * sg + static_cast<int>(sq % sg);
                        const uint32_t ph = (sq / sg) & 1u;
                        if (!mbar_wait_bounded(smem_u32(&empty_bar[slot]), ph ^ 1u,
                                               a.timeout_ns)) {
                            failed = true;
                            break;
                        }
                        const int64_t v0 = static_cast<int64_t>(c) * chunk_vec;
                        const uint32_t bytes =
                            static_cast<uint32_t>(imin64(chunk_vec, vec_row - v0)) * 16u;
                        const uint32_t fb = smem_u32(&full_bar[slot]);
                        mbar_arrive_expect_tx(fb, bytes);
                        const char* src = reinterpret_cast<const char*>(a.x) +
                                          (r * a.V + v0 * VE) * static_cast<int64_t>(sizeof(T));
                        const uint32_t dst = smem_u32(ring + static_cast<size_t>(slot) * chunk_bytes);
                        const uint64_t pol = (!a.resident && p == 0) ? pol_keep : pol_once;
                        for (uint32_t off = 0; off < bytes; off += kStreamCopyChunk)
                            bulk_g2s(dst + off, src + off, min(kStreamCopyChunk, bytes - off), fb,
                                     pol);
                        s_issued[slot] = sq + 1;
                    }
                }
            }
            if (failed) {
                atomicOr(&a.scratch->status, kDevErrTimeout);
                s_failed = 1;
            }
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
        const bool smooth = a.eps != 0.f;

        const int g = warp / G;
        const int wg = warp % G;
        const int tg = tid - g * GT;
        const NamedSync group_sync{1 + g, GT};
        const bool gleader = tid == g * GT;
        double accL = 0.0, accZ = 0.0;
        long long accC = 0;
        uint32_t seq = 0;
        bool failed = false;
        int rp = 0;

        for (int64_t r = cid + static_cast<int64_t>(g) * ncta; r < a.rows;
             r += static_cast<int64_t>(ng) * ncta) {
            const int64_t t = load_target(a, r);
            const bool counts = row_counts(a, t);
            if (gleader && t != a.ignore_index && !counts)
                atomicOr(&a.scratch->status, kDevErrTarget);
            if (!counts) {
                // Ignored row: exact +0 gradient, zero per-row outputs, pred -1.
                if (a.grad) {
                    uint4* rowv = reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.x) + r * a.V);
                    for (int64_t v = tg; v < vec_row; v += GT) rowv[v] = make_uint4(0u, 0u, 0u, 0u);
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
            float xt = 0.f;
            if (gleader) xt = VT::load1(a.x, r * a.V + t);  // before any store to this row
            const float wt = a.weight ? __ldg(a.weight + t) : 1.f;

            // ---- pass 1: thread statistics over the row's slots
            PassOne<T, SOFTCAP> st;
            const uint32_t seq0 = seq;
            for (int c = 0; c < nchunk; ++c, ++seq) {
                const int slot = g * sg + static_cast<int>(seq % sg);
                if (!failed && !mbar_wait_bounded(smem_u32(&full_bar[slot]), (seq / sg) & 1u,
                                                  a.timeout_ns)) {
                    failed = true;
                    atomicOr(&a.scratch->status, kDevErrTimeout);
                }
                const uint4* ch = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(slot) * chunk_bytes);
                const int64_t v0 = static_cast<int64_t>(c) * chunk_vec;
                const int nv = static_cast<int>(imin64(chunk_vec, vec_row - v0));
                for (int v = tg; v < nv; v += GT)
                    st.add(ch[v], static_cast<int>((v0 + v) * VE), a, smooth);
                if (!a.resident) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
                }
            }

            // ---- merge: warp butterfly, one group barrier, lane-parallel group merge
            RowStats ws = st.stats(smooth);
            warp_stats_allreduce<32>(ws);
            if (lane == 0) grec[g][rp][wg] = ws;
            group_sync();
            RowStats tot = lane < G ? grec[g][rp][lane] : empty_stats();
            warp_stats_allreduce<32>(tot);
            rp ^= 1;
            const float M = tot.m;
            const float logS = logf(tot.S);

            if (gleader) {
                const float zt = SOFTCAP ? a.softcap * tanh_from_scaled(xt * a.sc_k2) : xt;
                float zl;
                const float l = row_loss(a, M, logS, zt, wt, static_cast<float>(a.V), tot.SZ, zl);
                const bool correct = static_cast<int64_t>(tot.idx) == t;
                if (a.reduction == kRedNone) {
                    a.loss[r] = l;
                    if (a.want_z) a.zloss[r] = zl;
                    if (a.want_acc) a.acc[r] = correct ? 1.f : 0.f;
                } else {
                    accL += static_cast<double>(l);
                    accZ += static_cast<double>(zl);
                    accC += correct ? 1 : 0;
                }
                if (a.want_pred) a.pred[r] = tot.idx;
            }

            // ---- pass 2: gradient in place
            //   scale * [ (1-eps) w_t (p - onehot) + (eps/V)(V p - 1) + 2 lam lse p ] * dz/dx
            const float lse = M + logS;
            const float As = scale * ((1.f - a.eps) * wt + a.eps + 2.f * a.lam * lse) / tot.S;
            const float Bc = -scale * a.eps * inv_V;
            const float tfix = -scale * (1.f - a.eps) * wt;
            const float ML = M * kLog2e;
            const int64_t tvec = t / VE;
            const int tj = static_cast<int>(t % VE);
            uint4* rowv = reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.x) + r * a.V);
            if (a.resident) seq = seq0;
            for (int c = 0; c < nchunk; ++c, ++seq) {
                const int slot = g * sg + static_cast<int>(seq % sg);
                if (!a.resident && !failed &&
                    !mbar_wait_bounded(smem_u32(&full_bar[slot]), (seq / sg) & 1u, a.timeout_ns)) {
                    failed = true;
                    atomicOr(&a.scratch->status, kDevErrTimeout);
                }
                const uint4* ch = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(slot) * chunk_bytes);
                const int64_t v0 = static_cast<int64_t>(c) * chunk_vec;
                const int nv = static_cast<int>(imin64(chunk_vec, vec_row - v0));
                if (a.grad && !failed) {
                    for (int v = tg; v < nv; v += GT) {
                        float f[VE], gr[VE], th[VE];
                        VT::unpack(ch[v], f);
#pragma unroll
                        for (int j = 0; j < VE; ++j) {
                            float z = f[j];
                            if (SOFTCAP) {
                                th[j] = tanh_from_scaled(f[j] * a.sc_k2);
                                z = a.softcap * th[j];
                            }
                            const float e = sizeof(T) == 2 ? ex2(fmaf(z, kLog2e, -ML))
                                                           : ex2((z - M) * kLog2e);
                            gr[j] = fmaf(As, e, Bc);
                        }
                        if (v0 + v == tvec) {
#pragma unroll
                            for (int j = 0; j < VE; ++j)
                                if (j == tj) gr[j] += tfix;
                        }
                        if (SOFTCAP) {
#pragma unroll
                            for (int j = 0; j < VE; ++j) gr[j] *= fmaf(-th[j], th[j], 1.f);
                        }
                        rowv[v0 + v] = VT::pack(gr);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
            }
        }
        if (gleader) {
            gpart_l[g] = accL;
            gpart_z[g] = accZ;
            gpart_c[g] = accC;
        }
        if (failed && lane == 0) s_failed = 1;
    }
    __syncthreads();

    if (s_failed && tid == NW * 32) {
        // drain copies that may still be in flight: wait (bounded) for the
        // last issued use of every slot
        for (int i = 0; i < ng * sg; ++i) {
            const uint32_t used = s_issued[i];
            if (used) (void)mbar_wait_bounded(smem_u32(&full_bar[i]), ((used - 1) / sg) & 1u,
                                              a.timeout_ns);
        }
    }
    if (a.reduction != kRedNone && tid == 0) {
        double L = 0.0, Z = 0.0;
        long long C = 0;
        for (int g = 0; g < ng; ++g) {
            L += gpart_l[g];
            Z += gpart_z[g];
            C += gpart_c[g];
        }
        finish_scalars(a, cid, ncta, L, Z, C, s_D, s_nvalid);
    }
}

const void* stream_kernel(int dtype, bool softcap) {
    if (dtype == 0)
        return softcap ? (const void*)&ce_fwd_stream<float, true>
                       : (const void*)&ce_fwd_stream<float, false>;
    if (dtype == 1)
        return softcap ? (const void*)&ce_fwd_stream<__nv_bfloat16, true>
                       : (const void*)&ce_fwd_stream<__nv_bfloat16, false>;
    return nullptr;
}

}  // namespace gbce
