// Fused softmax cross-entropy forward with the in-forward gradient: the
// staged kernel (fast path).
//
// Method (Liger-Kernel cross-entropy kernel profile, §Forward Pass,
// §Backward Pass and §Key Patterns; tt-mlir pull request #9324 review
// comments on the mean reduction): per row, a max-shifted log-sum-exp of
// the (optionally softcapped) logits, the NLL with ignore_index, class
// weights, label smoothing and z-loss, the argmax, and the gradient of the
// reduced loss written in place over the logits.
//
// GB300 design (not the pages' one-program-per-row, two-pass loop):
//  * Row ownership. A thread-block cluster of C CTAs (C = 1 ... 16) owns a
//    row; CTA c owns a contiguous slice of slice_vec 16-byte vectors. The
//    grid is persistent: cluster k handles rows k, k + n_clusters, ...
//  * One HBM read per element. Thread 0 of every CTA keeps a ring of
//    `stages` shared-memory buffers filled by 1-D bulk asynchronous copies
//    (cp.async.bulk, completion counted on an mbarrier) for the next rows,
//    so loads of later rows overlap the compute and stores of this one.
//    Ignored rows are never loaded.
//  * Registers. Each thread copies its vectors of the staged slice into
//    registers; the buffer goes back to the copy engine after the row's one
//    block barrier. exp(z - m) (or tanh(x/s) under softcap) is kept per
//    element, so the gradient needs no second load and no second
//    exponential (one more under softcap).
//  * One barrier per row. Each thread forms online-softmax statistics of
//    its own elements (its max, sum of exp, smoothing sum, argmax); warps
//    merge them with shuffles; one __syncthreads publishes the warp
//    records; across the cluster one barrier.cluster makes the CTA records
//    readable through distributed shared memory, and every warp merges
//    them itself. Merges rescale sums to the larger max.
//  * One HBM write per element: the gradient is packed to the logit dtype
//    and stored with 16-byte coalesced stores over the row it came from.
//  * Scalars. Per-row outputs are written by the cluster's rank 0; sums
//    go through per-cluster partials and a last-CTA fixed-order epilogue.
#pragma once

#include <climits>
#include <type_traits>

#include "ce_kernels.cuh"

namespace gbce {

constexpr uint32_t kCopyChunk = 32768;  // bytes per bulk-copy instruction

template <typename T, int NT, int NV, bool SOFTCAP, bool WSMOOTH>
__global__ void __launch_bounds__(NT, (NT >= 512 ? 1 : 512 / NT))
ce_fwd_staged(const __grid_constant__ FwdArgs a) {
    using VT = Vec<T>;
    constexpr int VE = VT::N;  // elements per 16-byte vector
    constexpr int NW = NT / 32;

    extern __shared__ __align__(128) unsigned char dyn[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(16) RowStats red[2][NW];     // warp records, by row parity
    __shared__ __align__(16) float rec[2][8];         // this CTA's record, by exchange parity
    __shared__ float red_p[NW];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t crank = cluster_ctarank();
    const uint32_t csize = cluster_nctarank();
    const int64_t cid = cluster_id_x();
    const int64_t ncl = ncluster_x();
    const int stages = a.stages;

    const int64_t vec_row = a.V / VE;
    const int64_t vbeg = static_cast<int64_t>(crank) * a.slice_vec;
    const int nvec = static_cast<int>(
        max(static_cast<int64_t>(0), min(static_cast<int64_t>(a.slice_vec), vec_row - vbeg)));
    const uint32_t slice_bytes = static_cast<uint32_t>(a.slice_vec) * 16u;
    const uint32_t copy_bytes = static_cast<uint32_t>(nvec) * 16u;
    float* wsl = reinterpret_cast<float*>(dyn + static_cast<size_t>(stages) * slice_bytes);

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(smem_u32(&full_bar[s]), 1);
        fence_mbar_init();
    }
    __syncthreads();

    // ---- producer (thread 0): fill stage s with this CTA's slice of row r
    const uint64_t pol = l2_evict_first_policy();
    int64_t issued = 0;  // iterations whose stage fill was issued (thread 0)
    auto issue = [&](int64_t r, int s) {
        const uint32_t bar = smem_u32(&full_bar[s]);
        const int64_t t = load_target(a, r);
        if (copy_bytes != 0 && row_counts(a, t)) {
            mbar_arrive_expect_tx(bar, copy_bytes);
            const char* src = reinterpret_cast<const char*>(a.x) +
                              (r * a.V + vbeg * VE) * static_cast<int64_t>(sizeof(T));
            const uint32_t dst = smem_u32(dyn + static_cast<size_t>(s) * slice_bytes);
            for (uint32_t off = 0; off < copy_bytes; off += kCopyChunk)
                bulk_g2s(dst + off, src + off, min(kCopyChunk, copy_bytes - off), bar, pol);
        } else {
            mbar_arrive(bar);  // nothing to load: complete the phase at once
        }
        ++issued;
    };
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            const int64_t r = cid + s * ncl;
            if (r < a.rows) issue(r, s);
        }
    }

    // ---- prologue (overlaps the first copies): denominators, weight slice
    float D = 0.f;
    int n_valid = 0;
    if (a.reduction != kRedNone) denominators<NT>(a, red_p, D, n_valid);
    if (WSMOOTH) {
        // transposed [j][v] so that a warp reading element j of its vectors
        // touches consecutive words
        for (int i = tid; i < nvec * VE; i += NT)
            wsl[(i % VE) * a.slice_vec + i / VE] = __ldg(a.weight + vbeg * VE + i);
        __syncthreads();
    }
    const float scale = a.reduction == kRedMean ? 1.f / D : 1.f;  // unused when D == 0
    const float inv_V = 1.f / static_cast<float>(a.V);
    const bool smooth = a.eps != 0.f;

    const bool leader = crank == 0 && tid == 0;
    double accL = 0.0, accZ = 0.0;
    long long accC = 0;
    int xchg = 0;
    bool failed = false;
    int64_t fail_it = -1;

    int64_t it = 0;
    for (int64_t r = cid; r < a.rows; r += ncl, ++it) {
        const int s = static_cast<int>(it % stages);
        const uint32_t par = static_cast<uint32_t>((it / stages) & 1);
        const int64_t t = load_target(a, r);
        const bool counts = row_counts(a, t);
        if (leader && t != a.ignore_index && !counts) atomicOr(&a.scratch->status, kDevErrTarget);
        float xt = 0.f, wt = 0.f;
        if (counts) {
            wt = a.weight ? __ldg(a.weight + t) : 1.f;
            if (leader) xt = VT::load1(a.x, r * a.V + t);  // before any store to this row
        }
        bool ok = true;
        if (!failed) ok = mbar_wait_bounded(smem_u32(&full_bar[s]), par, a.timeout_ns);

        if (!counts) {
            // Ignored row: exact +0 gradient, zero per-row outputs, pred -1.
            const bool f = __syncthreads_or(!ok) != 0;
            if (f && !failed) fail_it = it;
            failed = failed || f;
            if (tid == 0 && !failed && r + stages * ncl < a.rows) issue(r + stages * ncl, s);
            if (a.grad && !failed) {
                uint4* rowv = reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.x) + r * a.V +
                                                       vbeg * VE);
                for (int v = tid; v < nvec; v += NT) rowv[v] = make_uint4(0u, 0u, 0u, 0u);
            }
            if (leader) {
                if (a.reduction == kRedNone) {
                    a.loss[r] = 0.f;
                    if (a.want_z) a.zloss[r] = 0.f;
                    if (a.want_acc) a.acc[r] = 0.f;
                }
                if (a.want_pred) a.pred[r] = -1;
            }
            continue;
        }

        // ---- 1. registers from the stage; the thread's max and first argmax
        const uint4* stg = reinterpret_cast<const uint4*>(dyn + static_cast<size_t>(s) * slice_bytes);
        uint4 xr[NV];
        float tmax = -INFINITY;
        int tk = -1;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = tid + k * NT;
            if (v < nvec) {
                xr[k] = stg[v];
                const float m = VT::vmax(xr[k]);
                if (m > tmax) {
                    tmax = m;
                    tk = k;
                }
            } else {
                xr[k] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        RowStats st = empty_stats();
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if (k == tk) {
                float f[VE];
                VT::unpack(xr[k], f);
                const int base = static_cast<int>((vbeg + tid + k * NT) * VE);
#pragma unroll
                for (int j = VE - 1; j >= 0; --j)
                    if (f[j] == tmax) st.idx = base + j;
            }
        }
        st.xmax = tmax;

        // ---- 2. exp(z - shift) once per element, relative to the thread's max
        const float shift = tk < 0 ? 0.f
                            : (SOFTCAP ? a.softcap * tanh_from_scaled(tmax * a.sc_k2) : tmax);
        float cc[NV][VE];
        float S = 0.f, SZ = 0.f, Wn = 0.f;
        auto exp_pass = [&](auto with_sums) {
            constexpr bool kSums = decltype(with_sums)::value;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int v = tid + k * NT;
                if (v < nvec) {
                    float f[VE];
                    VT::unpack(xr[k], f);
#pragma unroll
                    for (int j = 0; j < VE; ++j) {
                        float d;
                        if (SOFTCAP) {
                            const float th = tanh_from_scaled(f[j] * a.sc_k2);
                            d = fmaf(th, a.softcap, -shift);
                            cc[k][j] = th;
                        } else {
                            d = f[j] - shift;
                        }
                        const float e = ex2(d * kLog2e);
                        if (!SOFTCAP) cc[k][j] = e;
                        S += e;
                        if (kSums) {
                            if (WSMOOTH) {
                                const float w = wsl[j * a.slice_vec + v];
                                SZ = fmaf(w, d, SZ);
                                Wn += w;
                            } else {
                                SZ += d;
                            }
                        }
                    }
                    if (kSums && !WSMOOTH) Wn += static_cast<float>(VE);
                } else {
#pragma unroll
                    for (int j = 0; j < VE; ++j) cc[k][j] = 0.f;
                }
            }
        };
        if (smooth)
            exp_pass(std::true_type{});
        else
            exp_pass(std::false_type{});
        if (tk >= 0) {
            st.m = shift;
            st.S = S;
            st.SZ = SZ;
            st.Wn = Wn;
        }

        // ---- 3. merge: warp butterfly, one block barrier, CTA records
        warp_stats_allreduce<32>(st);
        const int rp = static_cast<int>(it & 1);
        if (lane == 0) red[rp][warp] = st;
        {
            const bool f = __syncthreads_or(!ok) != 0;
            if (f && !failed) fail_it = it;
            failed = failed || f;
        }
        // every thread holds its vectors: hand the stage back to the copy engine
        if (tid == 0 && !failed && r + stages * ncl < a.rows) issue(r + stages * ncl, s);
        RowStats tot = red[rp][0];
#pragma unroll
        for (int w = 1; w < NW; ++w) stats_merge(tot, red[rp][w]);

        // ---- 4. merge over the cluster through distributed shared memory
        if (csize > 1) {
            const int slot = xchg & 1;
            ++xchg;
            if (tid == 0) {
                rec[slot][0] = tot.m;
                rec[slot][1] = tot.S;
                rec[slot][2] = tot.SZ;
                rec[slot][3] = tot.Wn;
                rec[slot][4] = tot.xmax;
                rec[slot][5] = __int_as_float(tot.idx);
            }
            cluster_sync();
            RowStats cs = empty_stats();
            if (lane < static_cast<int>(csize)) {
                const uint32_t ra = map_to_rank(smem_u32(&rec[slot][0]), lane);
                const float4 q0 = ld_dsmem_f4(ra);
                const float4 q1 = ld_dsmem_f4(ra + 16);
                cs = RowStats{q0.x, q0.y, q0.z, q0.w, q1.x, __float_as_int(q1.y)};
            }
            warp_stats_allreduce<32>(cs);
            tot = cs;
        }
        const float M = tot.m;
        const float logS = logf(tot.S);
        const int am = tot.idx;

        // ---- 5. per-row outputs (rank 0 of the cluster)
        if (leader) {
            const float zt = SOFTCAP ? a.softcap * tanh_from_scaled(xt * a.sc_k2) : xt;
            float zl;
            const float l = row_loss(a, M, logS, zt, wt, WSMOOTH ? tot.Wn : static_cast<float>(a.V),
                                     tot.SZ, zl);
            const bool correct = static_cast<int64_t>(am) == t;
            if (a.reduction == kRedNone) {
                a.loss[r] = l;
                if (a.want_z) a.zloss[r] = zl;
                if (a.want_acc) a.acc[r] = correct ? 1.f : 0.f;
            } else {
                accL += static_cast<double>(l);
                accZ += static_cast<double>(zl);
                accC += correct ? 1 : 0;
            }
            if (a.want_pred) a.pred[r] = am;
        }

        // ---- 6. gradient in place:
        //   scale * [ (1-eps) w_t (p - onehot) + (eps/V)(W p - w) + 2 lam lse p ] * dz/dx
        if (a.grad && !failed) {
            const float lse = M + logS;
            const float Wn = WSMOOTH ? tot.Wn * inv_V : 1.f;
            const float A = scale * ((1.f - a.eps) * wt + a.eps * Wn + 2.f * a.lam * lse);
            const float c0 = ex2((shift - M) * kLog2e) / tot.S;  // p = e * c0
            const float Ac = A * c0;
            const float Bc = -scale * a.eps * inv_V;
            const float tfix = -scale * (1.f - a.eps) * wt;
            const int64_t tvec = t / VE - vbeg;
            const int tj = static_cast<int>(t % VE);
            uint4* rowv =
                reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.x) + r * a.V + vbeg * VE);
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int v = tid + k * NT;
                if (v < nvec) {
                    float g[VE];
#pragma unroll
                    for (int j = 0; j < VE; ++j) {
                        const float e = SOFTCAP ? ex2(fmaf(cc[k][j], a.softcap, -shift) * kLog2e)
                                                : cc[k][j];
                        const float b = WSMOOTH ? Bc * wsl[j * a.slice_vec + v] : Bc;
                        g[j] = fmaf(Ac, e, b);
                    }
                    if (v == tvec) {
#pragma unroll
                        for (int j = 0; j < VE; ++j)
                            if (j == tj) g[j] += tfix;
                    }
                    if (SOFTCAP) {
#pragma unroll
                        for (int j = 0; j < VE; ++j) g[j] *= fmaf(-cc[k][j], cc[k][j], 1.f);
                    }
                    rowv[v] = VT::pack(g);
                }
            }
        }
    }

    // No CTA may leave while a partner can still read its exchange record.
    if (csize > 1) cluster_sync();

    if (failed && tid == 0) {
        atomicOr(&a.scratch->status, kDevErrTimeout);
        // drain the fills issued after the failure point, each wait bounded
        for (int64_t j = fail_it; j < issued; ++j)
            (void)mbar_wait_bounded(smem_u32(&full_bar[j % stages]),
                                    static_cast<uint32_t>((j / stages) & 1), a.timeout_ns);
    }
    if (a.reduction != kRedNone && crank == 0 && tid < 32)
        finish_scalars(a, cid, ncl, accL, accZ, accC, D, n_valid);
}

}  // namespace gbce
