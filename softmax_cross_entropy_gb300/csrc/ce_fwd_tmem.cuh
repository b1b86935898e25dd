// Fused softmax cross-entropy forward with the in-forward gradient for
// softcapped logits: the tensor-memory kernel.
//
// Method (Liger-Kernel cross-entropy kernel profile, §Forward Pass,
// §Backward Pass and §Key Patterns): per row z = s tanh(x / s), the
// log-sum-exp of z, the NLL with ignore_index, class weights on the target
// term, label smoothing and z-loss, the argmax of the raw logits, and the
// gradient of the reduced loss written in place over the logits.
//
// GB300 design. With a softcap every element costs two special-function
// operations for tanh (exp2 and a reciprocal) and one more for exp(z), and a
// kernel that streams a long row twice pays them twice. Here each element's
// tanh is formed once and kept on chip until the gradient needs it, in the
// SM's 256 KB of tensor memory (TMEM, otherwise the tensor cores'
// accumulator store) used as a scratchpad: 512 columns x 128 lanes of 32
// bits, one fp32 per element, so one SM keeps 65536 elements and a cluster
// of C CTAs (one an SM) keeps a row of up to C * 65536.
//  * Shift. z <= s, so exp(z - s) lies in (exp(-2s), 1] and needs no row
//    maximum: S' = sum exp(z - s) and lse = s + log S'. (The kernel is used
//    for s <= 40, where exp(-2s) stays a normal fp32.) With
//    r = 1 / (1 + exp(2x/s)): z - s = -2 s r and dz/dx = 4 r (1 - r).
//  * Pass 1. A producer warp streams the CTA's slice of each counted row
//    once from HBM through a ring of 32 KB shared-memory slots (1-D bulk
//    async copies, mbarrier completion); 16 consumer warps form r, exp2 of
//    -2 s r log2(e) and the sums S' and sum r, and store r to their own TMEM
//    lane and columns (tcgen05.st).
//  * Merge. Warps merge with shuffles, the CTA with one named barrier; the
//    cluster's CTAs exchange one record each through distributed shared
//    memory: every CTA stores its record into every CTA of the cluster and
//    arrives on their mbarrier, so the merge waits only for the records,
//    never on a cluster-wide barrier of all threads.
//  * Pass 2. r comes back from TMEM (tcgen05.ld): one exp2 an element,
//    gradient (As exp + Bc) 4 r (1 - r), packed and stored with 16-byte
//    stores. The ring meanwhile fills with the next row.
// Special-function operations: 4 an element instead of 6, HBM traffic one
// read and one write.
#pragma once

#include <climits>

#include "ce_kernels.cuh"

namespace gbce {

namespace {

constexpr int kTmNTC = 32 * kTmWarps;                 // consumer threads
constexpr int kTmChunkVec = kTmNTC * kTmVecPerThread;  // 16-byte vectors of one ring slot

// r of one 16-byte vector (VE values) to VE consecutive TMEM columns of this
// thread's lane; the whole warp executes it.
template <int VE>
__device__ __forceinline__ void tm_store(uint32_t taddr, const float (&v)[VE]) {
    if constexpr (VE == 8) {
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                taddr),
            "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
            "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
            "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
            : "memory");
    } else {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
                     "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
                     "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3]))
                     : "memory");
    }
}

template <int VE>
__device__ __forceinline__ void tm_load(uint32_t taddr, uint32_t (&v)[VE]) {
    if constexpr (VE == 8) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
              "=r"(v[7])
            : "r"(taddr)
            : "memory");
    } else {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                     : "r"(taddr)
                     : "memory");
    }
}

__device__ __forceinline__ void tm_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tm_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// A record of the cluster exchange stored into CTA `rank`'s shared memory.
__device__ __forceinline__ void st_dsmem_f4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// Arrival on an mbarrier of another CTA of the cluster; release at cluster
// scope orders this thread's earlier stores into that CTA before it.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                     cluster_addr)
                 : "memory");
}

// mbar_wait_bounded with acquire at cluster scope (the phase completes on
// arrivals of other CTAs, whose stores must be visible after it).
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint32_t bar, uint32_t parity,
                                                          uint64_t timeout_ns) {
    auto try_wait = [&](uint32_t suspend_ns) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "r"(suspend_ns)
            : "memory");
        return ok != 0;
    };
    if (try_wait(0u)) return true;
    const uint64_t t0 = global_timer_ns();
#pragma unroll 1
    while (!try_wait(20000u)) {
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
    return true;
}

struct TmRing {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next(int n) {
        if (++slot == n) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

}  // namespace

// The end of a CTA of the tensor-memory kernel: copies that may still be
// in flight after a timed-out wait land, the TMEM columns are freed, and no
// CTA leaves while another CTA of the cluster may still store into it.
__device__ __forceinline__ void tm_teardown(const FwdArgs& a, uint32_t tmem, const int& s_failed,
                                            const uint32_t* s_issued, uint64_t* full_bar, int sg,
                                            int tid, int warp) {
    __syncthreads();
    if (s_failed && tid == kTmWarps * 32) {
        for (int i = 0; i < sg; ++i) {
            const uint32_t used = s_issued[i];
            if (used) (void)mbar_wait_bounded(smem_u32(&full_bar[i]), used & 1u, a.timeout_ns);
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmCols)
                     : "memory");
    cluster_sync();
}

// The producer warp: its lanes read the targets of the cluster's next 32
// rows; lane 0 copies this CTA's slice of each counted row into the ring,
// slot by slot (1-D bulk async copies, completion on the slot's full
// barrier), after the consumers have released the slot.
template <typename T>
__device__ __forceinline__ void tm_produce(const FwdArgs& a, unsigned char* ring,
                                           uint64_t* full_bar, uint64_t* empty_bar,
                                           uint32_t* s_issued, int* s_failed, int sg, int nvec,
                                           int nchunk, int64_t v0c, int64_t clid, int64_t ncl,
                                           int lane) {
    constexpr int VE = Vec<T>::N;
    const uint64_t pol = l2_evict_first_policy();
    TmRing pos;
    int failed = 0;
    bool stall = a.test_stall && blockIdx.x == 0;  // test hook (FwdArgs::test_stall)
    for (int64_t rb = clid; rb < a.rows && !failed; rb += 32 * ncl) {
        const int64_t rl = rb + lane * ncl;
        const bool lane_counts = rl < a.rows && row_counts(a, load_target(a, rl));
        const uint32_t counted = __ballot_sync(0xffffffffu, lane_counts);
        if (lane == 0) {
            for (int j = 0; j < 32 && !failed; ++j) {
                const int64_t r = rb + j * ncl;
                if (r >= a.rows) break;
                if (!((counted >> j) & 1u)) continue;
                for (int c = 0; c < nchunk; ++c) {
                    const int slot = pos.slot;
                    if (!mbar_wait_bounded(smem_u32(&empty_bar[slot]), pos.phase ^ 1u,
                                           a.timeout_ns)) {
                        failed = 1;
                        break;
                    }
                    const uint32_t ph = pos.phase;
                    pos.next(sg);
                    if (stall) {
                        stall = false;
                        continue;
                    }
                    const int64_t cv0 = static_cast<int64_t>(c) * kTmChunkVec;
                    const uint32_t bytes =
                        static_cast<uint32_t>(min(static_cast<int64_t>(kTmChunkVec),
                                                  static_cast<int64_t>(nvec) - cv0)) *
                        16u;
                    const uint32_t fb = smem_u32(&full_bar[slot]);
                    mbar_arrive_expect_tx(fb, bytes);
                    const char* src = reinterpret_cast<const char*>(a.x) +
                                      (r * a.V + (v0c + cv0) * VE) *
                                          static_cast<int64_t>(sizeof(T));
                    const uint32_t dst = smem_u32(ring + static_cast<size_t>(slot) * kTmChunkVec * 16);
                    for (uint32_t off = 0; off < bytes; off += 32768u)
                        bulk_g2s(dst + off, src + off, min(32768u, bytes - off), fb, pol);
                    s_issued[slot] = 2u + ph;
                }
            }
        }
        failed = __shfl_sync(0xffffffffu, failed, 0);
    }
    if (failed && lane == 0) {
        atomicOr(&a.scratch->status, kDevErrTimeout);
        *s_failed = 1;
    }
}

// One CTA an SM: kTmWarps consumer warps and one producer warp. The grid is
// persistent: cluster k handles rows k, k + n_clusters, ...; CTA c of a
// cluster owns the row's vectors [c * a.tm_slice_vec, (c + 1) *
// a.tm_slice_vec), whose r values fit its TMEM (at most 128 columns a
// consumer thread).
template <typename T>
__global__ void __launch_bounds__(32 * (kTmWarps + 1), 1)
ce_fwd_tmem(const __grid_constant__ FwdArgs a) {
    using VT = Vec<T>;
    constexpr int VE = VT::N;

    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full_bar[kTmMaxSlots];
    __shared__ __align__(8) uint64_t empty_bar[kTmMaxSlots];
    __shared__ __align__(8) uint64_t xbar[2];          // cluster exchange, by counted-row parity
    __shared__ __align__(16) float4 xrec[2][kTmMaxCluster];  // the cluster's CTA records
    __shared__ __align__(16) float4 wrec[2][kTmWarps];       // this CTA's warp records
    __shared__ float red_p[kTmWarps];
    __shared__ uint32_t tmem_base_sh;
    __shared__ uint32_t s_issued[kTmMaxSlots];  // 0, or 2 + parity of the last copy
    __shared__ int s_failed;
    // thread 0's sums of the CTA's row losses, z-losses and correct rows, and
    // the batch denominators (in shared memory: no other thread needs
    // registers for them)
    __shared__ double s_accL, s_accZ;
    __shared__ long long s_accC;
    __shared__ float s_D;
    __shared__ int s_nvalid;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t crank = cluster_ctarank();
    const uint32_t csize = cluster_nctarank();
    const int64_t clid = cluster_id_x();
    const int64_t ncl = ncluster_x();
    const int sg = a.tm_slots;
    const int64_t vec_row = a.V / VE;
    const int64_t v0c = static_cast<int64_t>(crank) * a.tm_slice_vec;  // first vector of the slice
    const int nvec = static_cast<int>(
        max(static_cast<int64_t>(0), min(static_cast<int64_t>(a.tm_slice_vec), vec_row - v0c)));
    const int nchunk = (nvec + kTmChunkVec - 1) / kTmChunkVec;

    if (tid == 0) {
        for (int i = 0; i < sg; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), static_cast<uint32_t>(kTmWarps));
            s_issued[i] = 0;
        }
        mbar_init(smem_u32(&xbar[0]), csize);
        mbar_init(smem_u32(&xbar[1]), csize);
        s_failed = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                smem_u32(&tmem_base_sh)),
            "r"(kTmCols)
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    // every CTA's barriers are initialised before any other CTA arrives on them
    cluster_sync();
    const uint32_t tmem = tmem_base_sh;

    if (warp == kTmWarps) {
        tm_produce<T>(a, ring, full_bar, empty_bar, s_issued, &s_failed, sg, nvec, nchunk, v0c,
                      clid, ncl, lane);
    } else {
        // ------------------------------------------------------------ consumers
        const NamedSync all_consumers{15, kTmNTC};
        const NamedSync merge_sync{1, kTmNTC};
        float scale = 1.f;
        {
            float D = 0.f;
            int n_valid = 0;
            if (a.reduction != kRedNone) denominators<kTmNTC>(a, red_p, D, n_valid, all_consumers);
            if (a.reduction == kRedMean) scale = 1.f / D;  // unused when D == 0
            if (tid == 0) {
                s_D = D;
                s_nvalid = n_valid;
                s_accL = 0.0;
                s_accZ = 0.0;
                s_accC = 0;
            }
        }
        const float s = a.softcap;
        const float c1 = -2.f * a.sc_slog2e;  // exp2 argument of exp(z - s) = c1 r
        const float inv_V = 1.f / static_cast<float>(a.V);
        const bool want_arg = a.want_pred || a.want_acc;
        // this thread's TMEM lane (warp w reaches lanes 32 (w % 4) ...) and
        // its 128 columns of the CTA's kTmCols
        const uint32_t tbase =
            tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + static_cast<uint32_t>(warp >> 2) * 128u;
        const uint64_t spol = l2_evict_first_policy();
        TmRing pos;
        bool failed = false;
        int xi = 0;  // counted rows so far (exchange buffer and phase)
        for (int64_t r = clid; r < a.rows; r += ncl) {
            const int64_t t = load_target(a, r);
            const bool counts = row_counts(a, t);
            T* xrow = reinterpret_cast<T*>(a.x) + r * a.V;
            uint4* slice = reinterpret_cast<uint4*>(xrow) + v0c;
            if (!counts) {
                // ignored row: exact +0 gradient without reading it
                if (tid == 0 && crank == 0 && t != a.ignore_index)
                    atomicOr(&a.scratch->status, kDevErrTarget);
                if (a.grad)
                    for (int v = tid; v < nvec; v += kTmNTC)
                        st_v4_hint(slice + v, make_uint4(0u, 0u, 0u, 0u), spol);
                if (tid == 0 && crank == 0) {
                    if (a.reduction == kRedNone) {
                        a.loss[r] = 0.f;
                        if (a.want_z) a.zloss[r] = 0.f;
                        if (a.want_acc) a.acc[r] = 0.f;
                    }
                    if (a.want_pred) a.pred[r] = -1;
                }
                continue;
            }
            const int64_t tvec = t / VE - v0c;  // target's vector in this CTA's slice
            const bool t_here = tvec >= 0 && tvec < nvec;
            const bool t_owner = t_here && static_cast<int>(tvec % kTmNTC) == tid;
            float xt = 0.f;
            if (t_owner || (t_here && tid == 0)) xt = VT::load1(xrow, t);  // before any store
            const float wt = a.weight ? __ldg(a.weight + t) : 1.f;

            // ---- pass 1: r to TMEM, S' = sum exp(z - s), R = sum r, argmax
            float2 S2 = make_float2(0.f, 0.f), R2 = make_float2(0.f, 0.f);
            float xm = -INFINITY;
            int bi = INT_MAX;
            for (int c = 0; c < nchunk; ++c) {
                const int slot = pos.slot;
                if (!failed && !mbar_wait_bounded(smem_u32(&full_bar[slot]), pos.phase,
                                                  a.timeout_ns)) {
                    failed = true;
                    atomicOr(&a.scratch->status, kDevErrTimeout);
                }
                const uint4* ch = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(slot) * kTmChunkVec * 16);
                uint4 q[kTmVecPerThread];
#pragma unroll
                for (int k = 0; k < kTmVecPerThread; ++k) {
                    const int vl = c * kTmChunkVec + k * kTmNTC + tid;
                    q[k] = vl < nvec ? ch[k * kTmNTC + tid] : make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
                pos.next(sg);
#pragma unroll
                for (int k = 0; k < kTmVecPerThread; ++k) {
                    const int vl = c * kTmChunkVec + k * kTmNTC + tid;
                    const bool valid = vl < nvec;
                    float f[VE], rr[VE];
                    VT::unpack(q[k], f);
#pragma unroll
                    for (int j = 0; j < VE; j += 2) {
                        const float2 r2 = softcap_r2(f[j], f[j + 1], a.sc_k2);
                        rr[j] = r2.x;
                        rr[j + 1] = r2.y;
                        if (valid) {
                            const float2 ar = fmul2(r2, make_float2(c1, c1));
                            S2 = fadd2(S2, make_float2(ex2(ar.x), ex2(ar.y)));
                            R2 = fadd2(R2, r2);
                        }
                    }
                    if (want_arg && valid) {
                        const float vm = VT::vmax(q[k]);
                        if (vm > xm) {
                            int j0 = VE - 1;
#pragma unroll
                            for (int j = VE - 1; j >= 0; --j)
                                if (f[j] == vm) j0 = j;
                            xm = vm;
                            bi = static_cast<int>((v0c + vl) * VE) + j0;
                        }
                    }
                    tm_store<VE>(tbase + static_cast<uint32_t>((c * kTmVecPerThread + k) * VE), rr);
                }
            }
            tm_wait_st();

            // ---- merge: warp butterflies, one barrier, the CTA's 16 records
            float S = S2.x + S2.y, R = R2.x + R2.y;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                S += __shfl_xor_sync(0xffffffffu, S, o);
                R += __shfl_xor_sync(0xffffffffu, R, o);
            }
            float X = xm;
            int I = bi;
            if (want_arg) {
                X = warp_max_f32(xm);
                I = warp_min_s32(xm == X ? bi : INT_MAX);
            }
            const int p = xi & 1;
            if (lane == 0) wrec[p][warp] = make_float4(S, R, X, __int_as_float(I));
            merge_sync();
            {
                float Sc = 0.f, Rc = 0.f, Xc = -INFINITY;
                int Ic = INT_MAX;
#pragma unroll
                for (int w = 0; w < kTmWarps; ++w) {
                    const float4 q4 = wrec[p][w];
                    Sc += q4.x;
                    Rc += q4.y;
                    const int iw = __float_as_int(q4.w);
                    if (q4.z > Xc || (q4.z == Xc && iw < Ic)) {
                        Xc = q4.z;
                        Ic = iw;
                    }
                }
                S = Sc;
                R = Rc;
                X = Xc;
                I = Ic;
            }
            if (csize > 1) {
                // every CTA's record into every CTA of the cluster, then one
                // arrival on each of their exchange barriers
                if (tid == 0) {
                    const float4 mine = make_float4(S, R, X, __int_as_float(I));
                    const uint32_t rec = smem_u32(&xrec[p][crank]);
                    const uint32_t bar = smem_u32(&xbar[p]);
                    for (uint32_t q = 0; q < csize; ++q) st_dsmem_f4(map_to_rank(rec, q), mine);
                    for (uint32_t q = 0; q < csize; ++q) mbar_arrive_cluster(map_to_rank(bar, q));
                }
                if (!failed && !mbar_wait_cluster_bounded(smem_u32(&xbar[p]),
                                                          static_cast<uint32_t>(xi >> 1) & 1u,
                                                          a.timeout_ns)) {
                    failed = true;
                    atomicOr(&a.scratch->status, kDevErrTimeout);
                }
                float Sc = 0.f, Rc = 0.f, Xc = -INFINITY;
                int Ic = INT_MAX;
                for (uint32_t q = 0; q < csize; ++q) {
                    const float4 q4 = xrec[p][q];
                    Sc += q4.x;
                    Rc += q4.y;
                    const int iq = __float_as_int(q4.w);
                    if (q4.z > Xc || (q4.z == Xc && iq < Ic)) {
                        Xc = q4.z;
                        Ic = iq;
                    }
                }
                S = Sc;
                R = Rc;
                X = Xc;
                I = Ic;
            }
            ++xi;
            const float logS = logf(S);
            const float lse = s + logS;

            // ---- per-row outputs: the target's CTA (loss), rank 0 (pred)
            if (t_here && tid == 0) {
                const float zt = s * tanh_from_scaled(xt * a.sc_k2);
                float zl;
                // sum (z - s) = -2 s R
                const float l = row_loss(a, s, logS, zt, wt, static_cast<float>(a.V), -2.f * s * R, zl);
                const bool correct = static_cast<int64_t>(I) == t;
                if (a.reduction == kRedNone) {
                    a.loss[r] = l;
                    if (a.want_z) a.zloss[r] = zl;
                    if (a.want_acc) a.acc[r] = correct ? 1.f : 0.f;
                } else {
                    s_accL += static_cast<double>(l);
                    s_accZ += static_cast<double>(zl);
                    s_accC += correct ? 1 : 0;
                }
            }
            if (tid == 0 && crank == 0 && a.want_pred) a.pred[r] = I;

            // ---- pass 2: gradient in place from the r values in TMEM
            //   scale * [ (1-eps) w_t (p - onehot) + (eps/V)(V p - 1) + 2 lam lse p ] * dz/dx
            if (a.grad && !failed) {
                const float As = scale * ((1.f - a.eps) * wt + a.eps + 2.f * a.lam * lse) / S;
                const float Bc = -scale * a.eps * inv_V;
                const float2 As4 = make_float2(4.f * As, 4.f * As);
                const float2 Bc4 = make_float2(4.f * Bc, 4.f * Bc);
                // one vector's r values at a time (registers; two or four
                // at a time measured no faster, four spilled)
                for (int c = 0; c < nchunk; ++c) {
#pragma unroll
                    for (int k = 0; k < kTmVecPerThread; ++k) {
                        uint32_t rv[VE];
                        tm_load<VE>(tbase + static_cast<uint32_t>((c * kTmVecPerThread + k) * VE),
                                    rv);
                        tm_wait_ld();
                        const int vl = c * kTmChunkVec + k * kTmNTC + tid;
                        if (vl < nvec) {
                            float g[VE];
#pragma unroll
                            for (int j = 0; j < VE; j += 2) {
                                const float2 r2 =
                                    make_float2(__uint_as_float(rv[j]), __uint_as_float(rv[j + 1]));
                                const float2 ar = fmul2(r2, make_float2(c1, c1));
                                float2 gg = ffma2(As4, make_float2(ex2(ar.x), ex2(ar.y)), Bc4);
                                gg = fmul2(gg, ffma2(make_float2(-r2.x, -r2.y), r2, r2));
                                g[j] = gg.x;
                                g[j + 1] = gg.y;
                            }
                            st_v4_hint(slice + vl, VT::pack(g), spol);
                        }
                    }
                }
                if (t_owner) {
                    // the one-hot term, over the element just stored
                    const float th = tanh_from_scaled(xt * a.sc_k2);
                    const float e = ex2((s * th - s) * kLog2e);
                    const float gt =
                        (fmaf(As, e, Bc) - scale * (1.f - a.eps) * wt) * fmaf(-th, th, 1.f);
                    VT::store1(xrow, t, gt);
                }
            }
        }
        if (failed && lane == 0) s_failed = 1;
        // sums over the grid: thread 0 holds this CTA's partials
        if (a.reduction != kRedNone && tid < 32) {
            __syncwarp();  // thread 0's last shared-memory sums
            finish_scalars(a, blockIdx.x, gridDim.x, tid == 0 ? s_accL : 0.0,
                           tid == 0 ? s_accZ : 0.0, tid == 0 ? s_accC : 0, s_D, s_nvalid);
        }
    }
    tm_teardown(a, tmem, s_failed, s_issued, full_bar, sg, tid, warp);
}

}  // namespace gbce
