// Fused softmax cross-entropy forward with the in-forward gradient for rows
// of at most 64 KB: the register-resident kernel.
//
// Method (Liger-Kernel cross-entropy kernel profile, §Forward Pass,
// §Backward Pass, §Key Patterns): per row the max-shifted log-sum-exp, the
// NLL with ignore_index, class weights, label smoothing, z-loss, softcap,
// the argmax, and the gradient of the reduced loss written over the logits.
//
// GB300 design. A team of WPR warps owns one row at a time and each thread
// holds NVL (8 or 16) 16-byte vectors of it in registers, so a row of up to
// 512 B * NVL * WPR is read from HBM once and written once. Warp w of a
// team takes the row's vectors [w * 32 * NVL, (w + 1) * 32 * NVL): lane l
// holds vectors w * 32 * NVL + 32 k + l, so every access of a warp is 512
// contiguous bytes and the offsets between a thread's vectors are
// constants. A CTA holds several independent teams (one warp each for a
// 4096-element bf16 row), so an SM has a dozen or more rows in flight, and
// each team's leader copies the team's next row into a shared-memory buffer
// with a 1-D bulk async copy while the team computes the current one: the
// HBM latency of the next row hides behind this row's arithmetic, and the
// current row moves from the buffer into registers once. Per row:
//   1. raw maximum (packed 16-bit max for bf16/fp16), warp redux, one team
//      barrier for the row's maximum; the first argmax only when asked for;
//   2. S = sum exp(z - M) and the smoothing sum from the registers; a
//      second team barrier merges them;
//   3. the gradient As * exp(z - M) + Bc (times 1 - tanh^2 under softcap),
//      the exponential formed again from the registers (the SFU has room
//      for it, the register file has none for a copy of every e), stored
//      with 16-byte stores; the owner of the target's vector adds the
//      one-hot term and computes the row loss.
// Only row-level sums cross threads, in a fixed order, so results are
// deterministic. The mean denominator comes from the count kernel launched
// just before (its completion is awaited only where the first gradient
// needs it) or from the caller's batch counts.
#pragma once

#include <climits>

#include "ce_kernels.cuh"

namespace gbce {

// One fp32 from the shared memory of a CTA of the cluster (address from
// map_to_rank).
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Class weights of vector v (VE consecutive classes).
template <int VE>
__device__ __forceinline__ void reg_weights(const float* weight, int v, float (&w)[VE]) {
    const float4* wv = reinterpret_cast<const float4*>(weight + v * VE);
#pragma unroll
    for (int h = 0; h < VE / 4; ++h) {
        const float4 t4 = __ldg(wv + h);
        w[4 * h] = t4.x;
        w[4 * h + 1] = t4.y;
        w[4 * h + 2] = t4.z;
        w[4 * h + 3] = t4.w;
    }
}

// exp2 arguments (z - M) * log2(e): one packed FFMA against the rounded
// M * log2(e) for 16-bit logits, subtract first for fp32.
template <typename T>
__device__ __forceinline__ float2 reg_arg2(float2 z, float Ms, float ML) {
    if constexpr (sizeof(T) == 2)
        return ffma2(z, make_float2(kLog2e, kLog2e), make_float2(-ML, -ML));
    else
        return fmul2(fadd2(z, make_float2(-Ms, -Ms)), make_float2(kLog2e, kLog2e));
}

// Class weights of vector v from shared memory, where the 4-weight quarter
// h of vector v sits at float4 h * vrow + v: the lanes of a warp hold
// consecutive vectors and read consecutive 16-byte words.
template <int VE>
__device__ __forceinline__ void reg_weights_smem(const float4* w4, int v, int vrow,
                                                 float (&w)[VE]) {
#pragma unroll
    for (int h = 0; h < VE / 4; ++h) {
        const float4 t4 = w4[h * vrow + v];
        w[4 * h] = t4.x;
        w[4 * h + 1] = t4.y;
        w[4 * h + 2] = t4.z;
        w[4 * h + 3] = t4.w;
    }
}

// 8 vectors a thread: three CTAs of 8 warps an SM (85 registers a thread);
// 16 vectors: two (128 registers)
// CLU: the cluster variant (a.reg_cluster CTAs a row); otherwise one CTA
// holds whole rows and the cluster code folds away.
// MW: warps of a CTA. SW (class-weighted smoothing only): the V class
// weights sit in shared memory after the row buffers, loaded once per CTA,
// instead of being read from L1/L2 in both passes; one CTA of 16 warps an
// SM then holds one or two teams.
template <typename T, bool SOFTCAP, bool WS, int NVL, bool CLU, int MW = kRegMaxWarps,
          bool SW = false>
__global__ void __launch_bounds__(32 * MW, MW == 16 ? 1 : (NVL == 8 ? 3 : 2))
ce_fwd_reg(const __grid_constant__ FwdArgs a) {
    using VT = Vec<T>;
    constexpr int VE = VT::N;
    static_assert(!SW || (WS && !CLU), "shared-memory weights: class-weighted smoothing only");
    // a backward launched after this kernel (programmatic dependent launch)
    // may be scheduled now, which hides its launch; it waits for this grid's
    // completion before it reads anything (measured at 4096 x 4096 bf16:
    // the grad_output = 1 backward added 1.7 instead of about 2.5 us)
    pdl_launch_dependents();
    __shared__ float red_a[MW], red_b[MW], red_c[MW];
    __shared__ int red_i[MW];
    __shared__ double red_d[2][MW];
    __shared__ long long red_n[MW];
    __shared__ int s_flag;
    __shared__ __align__(8) uint64_t pf_bar[2 * MW];  // one per row buffer
    // each team leader's copy queue, kept in shared memory so that it takes
    // no registers in the other threads: the first of the team's rows not
    // yet looked at, the buffer the next copy goes to, and bit masks (bit k
    // for buffer k) of the unconsumed copies, of their completion parities
    // and of the parity the next copy into each buffer completes
    struct PfQueue {
        long long next;
        int k;
        uint32_t pend, pend_par, ph;
    };
    __shared__ PfQueue pfq[MW];
    __shared__ __align__(16) float cl_red[4];  // cluster mode: this CTA's max, S, SZ, argmax
    extern __shared__ __align__(128) unsigned char reg_smem[];  // teams x nbuf x reg_buf_stride

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int WPR = a.reg_wpr;           // warps of a team
    const int team = warp / WPR;
    const int wr = warp - team * WPR;    // warp within the team
    const int w0 = team * WPR;           // the team's first warp
    const int teams = (blockDim.x >> 5) / WPR;
    const int vrow = static_cast<int>(a.V / VE);
    // Rows longer than one CTA holds: a cluster of CL CTAs (one team of 8
    // warps each) owns a row, CTA c the slice of vectors [c * VPC, (c + 1) *
    // VPC); the row's maximum and sums merge across the cluster through
    // distributed shared memory.
    const int CL = CLU ? a.reg_cluster : 1;
    constexpr int VPC = MW * 32 * NVL;  // vectors of a CTA's slice (cluster mode)
    const int crank = CL > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int cta_vec0 = crank * VPC;              // first vector of this CTA's slice
    const int vbase = cta_vec0 + wr * 32 * NVL + lane;  // this thread's first vector
    const int vlim = vrow - vbase;           // its vector k exists when 32 k < vlim
    const bool smooth = WS || a.eps > 0.f;
    const bool want_arg = a.want_pred || a.want_acc;

    // barrier over the team's warps (named barrier 1 + team; a lone warp
    // needs only its own convergence)
    auto team_sync = [&]() {
        if (WPR == 1)
            __syncwarp();
        else
            asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(32 * WPR) : "memory");
    };
    // lane-level fixed-order sum of the team's per-warp values: the same
    // bits in every thread of the team
    auto team_sum = [&](const float* red) {
        float v = lane < WPR ? red[w0 + lane] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        return v;
    };

    // D = sum of w[t] over counted rows and the counted-row number come from
    // a.batch_counts ("sum" and "mean"): the caller's batch totals, or the
    // count kernel launched just before this one, which this launch
    // overlaps (programmatic dependent launch) until it first needs them.
    // (Every CTA reading the batch's targets itself was slower: they all hit
    // the same L2 lines at once.)
    float D = 0.f;
    int n_valid = 0;
    // "sum" without accuracy needs neither (and the host then launches no
    // count kernel)
    bool have_counts = a.reduction == kRedNone || (a.reduction == kRedSum && !a.want_acc);
    auto need_counts = [&]() {
        if (!have_counts) {
            pdl_wait();
            D = static_cast<float>(a.batch_counts[0]);
            n_valid = static_cast<int>(a.batch_counts[1]);
            have_counts = true;
        }
    };
    const float inv_V = 1.f / static_cast<float>(a.V);
    float Wtot = static_cast<float>(a.V);
    // SW: the weights' place in shared memory, after the teams' row buffers
    float4* w4s = reinterpret_cast<float4*>(
        reg_smem + static_cast<size_t>(teams) * a.reg_nbuf * a.reg_buf_stride);
    if (SW) {
        float* wsm = reinterpret_cast<float*>(w4s);
        for (int c = tid; c < a.V; c += blockDim.x) {
            const int v = c / VE, e = c % VE;
            wsm[((e >> 2) * vrow + v) * 4 + (e & 3)] = __ldg(a.weight + c);
        }
        // (visible to the CTA after the barriers of the sum below)
    }
    if (WS) {
        // W = sum of the class weights: every thread the same fixed order
        float s = 0.f;
        for (int c = tid; c < a.V; c += blockDim.x) s += __ldg(a.weight + c);
        s = warp_sum(s);
        if (lane == 0) red_a[warp] = s;
        __syncthreads();
        float v = lane < static_cast<int>(blockDim.x >> 5) ? red_a[lane] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        Wtot = v;
        __syncthreads();
    }
    const float Wf = WS ? Wtot * inv_V : 1.f;

    float accL = 0.f, accZ = 0.f;  // the rows whose target this thread owned
    int accC = 0;
    const int64_t nteams = CL > 1 ? static_cast<int64_t>(ncluster_x())
                                  : static_cast<int64_t>(gridDim.x) * teams;
    // Each team owns NB (a.reg_nbuf: 1 or 2) shared-memory buffers of one
    // row; its leader copies the team's next counted rows into them (1-D
    // bulk async copies, mbarrier completion), the counted rows taking the
    // buffers in turn, while the team computes the current row from
    // registers: the HBM latency of the next NB rows overlaps this row's
    // arithmetic.
    // bytes of the row this CTA's team copies (its slice in cluster mode)
    const uint32_t row_bytes =
        static_cast<uint32_t>(max(0, min(vrow - cta_vec0, CL > 1 ? VPC : vrow))) * 16u;
    const int NB = a.reg_nbuf;
    const uint32_t buf0 =
        smem_u32(reg_smem) + static_cast<uint32_t>(team * NB) * a.reg_buf_stride;
    const uint32_t bar0 = smem_u32(&pf_bar[team * NB]);
    const bool lead = wr == 0 && lane == 0;
    const uint64_t pol = l2_evict_first_policy();
    uint32_t cons_phase = 0;  // bit k: parity of buffer k's next completion
    int cons_k = 0;           // buffer of the team's next counted row
    bool failed = false;
    // test hook (FwdArgs::test_stall): the first copy of CTA 0's first team
    // is left out, so the team's wait for it runs out
    bool stall = a.test_stall && blockIdx.x == 0 && team == 0;
    int64_t r = CL > 1 ? static_cast<int64_t>(cluster_id_x())
                       : static_cast<int64_t>(blockIdx.x) * teams + team;
    PfQueue& Q = pfq[team];
    // leader only: copy the team's next counted row into buffer Q.k (its
    // previous row has been read by every thread of the team). hint_t is
    // the target of row hint_row, already in a register: the common case
    // (the next row of the team) then waits for no target load before its
    // copy is issued.
    auto prefetch_next = [&](int64_t hint_row, int64_t hint_t) {
        int64_t row = Q.next;
        while (row < a.rows &&
               !row_counts(a, row == hint_row ? hint_t : load_target(a, row)))
            row += nteams;
        if (row >= a.rows) {
            Q.next = row;
            return;
        }
        Q.next = row + nteams;
        const int k = Q.k;
        Q.k = (k + 1 == NB) ? 0 : k + 1;
        const uint32_t par = (Q.ph >> k) & 1u;
        Q.ph ^= 1u << k;
        if (stall) {
            stall = false;
            return;
        }
        const uint32_t bar = bar0 + 8u * static_cast<uint32_t>(k);
        const uint32_t buf = buf0 + static_cast<uint32_t>(k) * a.reg_buf_stride;
        const char* src = reinterpret_cast<const char*>(a.x) +
                          row * a.V * static_cast<int64_t>(sizeof(T)) +
                          static_cast<int64_t>(cta_vec0) * 16;
        mbar_arrive_expect_tx(bar, row_bytes);
        for (uint32_t off = 0; off < row_bytes; off += 32768u)
            bulk_g2s(buf + off, src + off, min(32768u, row_bytes - off), bar, pol);
        Q.pend |= 1u << k;
        Q.pend_par = (Q.pend_par & ~(1u << k)) | (par << k);
    };
    if (tid == 0) {
        for (int i = 0; i < teams * NB; ++i) mbar_init(smem_u32(&pf_bar[i]), 1);
        fence_mbar_init();
    }
    if (lead) Q = PfQueue{r, 0, 0u, 0u, 0u};
    __syncthreads();
    int64_t t_cur = r < a.rows ? load_target(a, r) : 0;                // row r
    int64_t t_nxt = r + nteams < a.rows ? load_target(a, r + nteams) : 0;  // row r + nteams
    // (a CTA whose slice is empty copies and waits for nothing)
    const bool has_slice = row_bytes > 0;
    if (lead && has_slice)
        for (int k = 0; k < NB; ++k) prefetch_next(r, t_cur);
#pragma unroll 1
    for (; r < a.rows; r += nteams) {
        const int64_t t = t_cur;
        const int64_t rn = r + nteams;
        t_cur = t_nxt;
        t_nxt = rn + nteams < a.rows ? load_target(a, rn + nteams) : 0;
        const bool counts = row_counts(a, t);
        T* xrow = reinterpret_cast<T*>(a.x) + r * a.V;
        uint4* rowv = reinterpret_cast<uint4*>(xrow);
        if (!counts) {
            // ignored row: exact +0 gradient without reading it (no buffer
            // holds it)
            if (lead && crank == 0 && t != a.ignore_index) atomicOr(&a.scratch->status, kDevErrTarget);
            if (a.grad) {
#pragma unroll
                for (int k = 0; k < NVL; ++k)
                    if (32 * k < vlim) st_v4_hint(rowv + vbase + 32 * k, make_uint4(0u, 0u, 0u, 0u), pol);
            }
            if (lead && crank == 0) {
                if (a.reduction == kRedNone) {
                    a.loss[r] = 0.f;
                    if (a.want_z) a.zloss[r] = 0.f;
                    if (a.want_acc) a.acc[r] = 0.f;
                }
                if (a.want_pred) a.pred[r] = -1;
            }
            continue;
        }
        // ---- the row into registers from its buffer: vector vbase + 32 k
        const int kb = cons_k;
        if (has_slice) {
            const uint32_t bar = bar0 + 8u * static_cast<uint32_t>(kb);
            if (!failed) {
                if (mbar_wait_bounded(bar, (cons_phase >> kb) & 1u, a.timeout_ns)) {
                    if (lead) Q.pend &= ~(1u << kb);
                } else {
                    failed = true;
                    if (lead) atomicOr(&a.scratch->status, kDevErrTimeout);
                }
            }
            cons_phase ^= 1u << kb;
            cons_k = (cons_k + 1 == NB) ? 0 : cons_k + 1;
        }
        uint4 q[NVL];
        const uint4* sb = reinterpret_cast<const uint4*>(
            reg_smem + static_cast<size_t>(team * NB + kb) * a.reg_buf_stride);
#pragma unroll
        for (int k = 0; k < NVL; ++k)
            q[k] = 32 * k < vlim ? sb[vbase - cta_vec0 + 32 * k] : make_uint4(0u, 0u, 0u, 0u);
        const int tvec = static_cast<int>(t / VE) - cta_vec0;  // in this CTA's slice
        const bool owner = tvec >= 0 && lane == (tvec & 31) && wr == tvec / (32 * NVL);
        // x_t from the buffer (before it takes the next row), not from HBM
        const float xt =
            owner ? VT::load1(sb, t - static_cast<int64_t>(cta_vec0) * VE) : 0.f;
        const float wt = a.weight ? __ldg(a.weight + t) : 1.f;

        // ---- 1. maximum of the raw logits
        typename VT::MaxAcc macc = VT::max_init();
#pragma unroll
        for (int k = 0; k < NVL; ++k)
            if (32 * k < vlim) macc = VT::max_fold(macc, q[k]);
        const float lm = VT::max_value(macc);
        __syncwarp();  // converged for the warp reductions
        const float wm = warp_max_f32(lm);
        float X = wm;
        if (WPR > 1) {
            if (lane == 0) red_a[warp] = wm;
            team_sync();
            X = warp_max_f32(lane < WPR ? red_a[w0 + lane] : -INFINITY);
        }
        // every thread of the team holds its vectors (the warp reduction
        // above, or the team barrier, follows every thread's buffer reads):
        // the buffer takes the team's next counted row
        if (lead && has_slice && !failed) prefetch_next(rn, t_cur);
        if (CL > 1) {
            // the row's maximum over the cluster: lane i reads CTA i's
            if (tid == 0) cl_red[0] = X;
            __syncwarp();
            cluster_sync();
            float o = -INFINITY;
            if (lane < CL) o = ld_dsmem_f32(map_to_rank(smem_u32(&cl_red[0]), lane));
            __syncwarp();
            X = warp_max_f32(o);
        }
        int cand = INT_MAX;
        if (want_arg) {
            // first element of this thread equal to the row maximum (the
            // thread's vectors come in increasing index order), by selects
#pragma unroll
            for (int k = NVL - 1; k >= 0; --k) {
                float f[VE];
                VT::unpack(q[k], f);
#pragma unroll
                for (int j = VE - 1; j >= 0; --j)
                    cand = (32 * k < vlim && f[j] == X) ? (vbase + 32 * k) * VE + j : cand;
            }
        }
        // softcap is monotone: the largest z is the cap of the largest x
        const float M = SOFTCAP ? a.softcap * tanh_from_scaled(X * a.sc_k2) : X;
        const float Ms = M == -INFINITY ? 0.f : M;
        const float ML = Ms * kLog2e;

        // ---- 2. S = sum exp(z - M), smoothing sum
        // (softcap: exp2 argument c1 r + c0 and z = s - 2 s r, softcap_r2)
        const float sc_c1 = -2.f * a.sc_slog2e;
        const float sc_c0 = fmaf(-Ms, kLog2e, a.sc_slog2e);
        float2 s2 = make_float2(0.f, 0.f), z2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < NVL; ++k) {
            if (32 * k < vlim) {
                float f[VE], w[VE];
                VT::unpack(q[k], f);
                if (WS) {
                    if (SW)
                        reg_weights_smem<VE>(w4s, vbase + 32 * k, vrow, w);
                    else
                        reg_weights<VE>(a.weight, vbase + 32 * k, w);
                }
#pragma unroll
                for (int j = 0; j < VE; j += 2) {
                    float2 z;
                    if constexpr (SOFTCAP) {
                        const float2 r = softcap_r2(f[j], f[j + 1], a.sc_k2);
                        const float2 ar = ffma2(r, make_float2(sc_c1, sc_c1),
                                                make_float2(sc_c0, sc_c0));
                        s2 = fadd2(s2, make_float2(ex2(ar.x), ex2(ar.y)));
                        if (smooth)
                            z = ffma2(r, make_float2(-2.f * a.softcap, -2.f * a.softcap),
                                      make_float2(a.softcap, a.softcap));
                    } else {
                        z = make_float2(f[j], f[j + 1]);
                        const float2 ar = reg_arg2<T>(z, Ms, ML);
                        s2 = fadd2(s2, make_float2(ex2(ar.x), ex2(ar.y)));
                    }
                    if (WS)
                        z2 = ffma2(make_float2(w[j], w[j + 1]), z, z2);
                    else if (smooth)
                        z2 = fadd2(z2, z);
                }
            }
        }
        __syncwarp();  // the ragged tail diverges
        float S = warp_sum(s2.x + s2.y);
        float ZS = smooth ? warp_sum(z2.x + z2.y) : 0.f;
        int I = cand;
        if (want_arg) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) I = min(I, __shfl_xor_sync(0xffffffffu, I, o));
        }
        if (WPR > 1) {
            if (lane == 0) {
                red_b[warp] = S;
                red_c[warp] = ZS;
                red_i[warp] = I;
            }
            team_sync();
            S = team_sum(red_b);
            if (smooth) ZS = team_sum(red_c);
            if (want_arg) {
                I = lane < WPR ? red_i[w0 + lane] : INT_MAX;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) I = min(I, __shfl_xor_sync(0xffffffffu, I, o));
            }
        }
        if (CL > 1) {
            // the row's sums over the cluster, added in rank order by a
            // fixed butterfly (the same bits in every thread)
            if (tid == 0) {
                cl_red[1] = S;
                cl_red[2] = ZS;
                cl_red[3] = __int_as_float(I);
            }
            __syncwarp();
            cluster_sync();
            float s_ = 0.f, z_ = 0.f;
            int i_ = INT_MAX;
            if (lane < CL) {
                const uint32_t rb = map_to_rank(smem_u32(&cl_red[0]), lane);
                s_ = ld_dsmem_f32(rb + 4);
                z_ = ld_dsmem_f32(rb + 8);
                i_ = __float_as_int(ld_dsmem_f32(rb + 12));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                s_ += __shfl_xor_sync(0xffffffffu, s_, o);
                z_ += __shfl_xor_sync(0xffffffffu, z_, o);
                i_ = min(i_, __shfl_xor_sync(0xffffffffu, i_, o));
            }
            S = s_;
            ZS = z_;
            I = i_;
        }
        const float logS = logf(S);
        const float lse = Ms + logS;
        // the element count of the smoothing sum is V; with weights, the sum
        // of w is W (sum (z - M) = sum z - V M, sum w (z - M) = sum wz - W M)
        const float SZ = smooth ? fmaf(-Wtot, Ms, ZS) : 0.f;

        // ---- row loss (the owner of the target's vector)
        if (owner) {
            const float zt = SOFTCAP ? a.softcap * tanh_from_scaled(xt * a.sc_k2) : xt;
            float zl;
            const float l = row_loss(a, Ms, logS, zt, wt, Wtot, SZ, zl);
            const bool correct = static_cast<int64_t>(I) == t;
            if (a.reduction == kRedNone) {
                a.loss[r] = l;
                if (a.want_z) a.zloss[r] = zl;
                if (a.want_acc) a.acc[r] = correct ? 1.f : 0.f;
            } else {
                accL += l;
                accZ += zl;
                accC += correct ? 1 : 0;
            }
            if (a.want_pred) a.pred[r] = I;
        }

        // ---- 3. gradient in place
        //   scale * [ (1-eps) w_t (p - onehot) + (eps/V)(W p - w) + 2 lam lse p ] * dz/dx
        if (a.grad) {
            need_counts();
            const float scale = a.reduction == kRedMean ? 1.f / D : 1.f;
            const float As = scale * ((1.f - a.eps) * wt + a.eps * Wf + 2.f * a.lam * lse) / S;
            const float Bc = -scale * a.eps * inv_V;
            const float As4 = 4.f * As, Bc4 = 4.f * Bc;  // softcap: times r - r^2
#pragma unroll
            for (int k = 0; k < NVL; ++k) {
                if (32 * k < vlim) {
                    float f[VE], g[VE], w[VE];
                    VT::unpack(q[k], f);
                    if (WS) {
                    if (SW)
                        reg_weights_smem<VE>(w4s, vbase + 32 * k, vrow, w);
                    else
                        reg_weights<VE>(a.weight, vbase + 32 * k, w);
                }
#pragma unroll
                    for (int j = 0; j < VE; j += 2) {
                        float2 gg;
                        if constexpr (SOFTCAP) {
                            // (As e + Bc) (1 - tanh^2) = (4 As e + 4 Bc) (r - r^2)
                            const float2 r = softcap_r2(f[j], f[j + 1], a.sc_k2);
                            const float2 ar = ffma2(r, make_float2(sc_c1, sc_c1),
                                                    make_float2(sc_c0, sc_c0));
                            const float2 bc = WS ? fmul2(make_float2(Bc4, Bc4), make_float2(w[j], w[j + 1]))
                                                 : make_float2(Bc4, Bc4);
                            gg = ffma2(make_float2(As4, As4), make_float2(ex2(ar.x), ex2(ar.y)), bc);
                            gg = fmul2(gg, ffma2(make_float2(-r.x, -r.y), r, r));
                        } else {
                            const float2 bc = WS ? fmul2(make_float2(Bc, Bc), make_float2(w[j], w[j + 1]))
                                                 : make_float2(Bc, Bc);
                            const float2 ar = reg_arg2<T>(make_float2(f[j], f[j + 1]), Ms, ML);
                            gg = ffma2(make_float2(As, As), make_float2(ex2(ar.x), ex2(ar.y)), bc);
                        }
                        g[j] = gg.x;
                        g[j + 1] = gg.y;
                    }
                    // (evict-first stores: measured 2% faster for short rows;
                    // the weighted-smoothing kernel keeps plain stores, which
                    // measured 1% faster there)
                    if constexpr (WS)
                        rowv[vbase + 32 * k] = VT::pack(g);
                    else
                        st_v4_hint(rowv + vbase + 32 * k, VT::pack(g), pol);
                }
            }
            if (owner) {
                // the one-hot term, over the element just stored
                float et, fac = 1.f;
                if (SOFTCAP) {
                    const float tt = tanh_from_scaled(xt * a.sc_k2);
                    fac = fmaf(-tt, tt, 1.f);
                    et = ex2((a.softcap * tt - Ms) * kLog2e);
                } else {
                    et = ex2((xt - Ms) * kLog2e);
                }
                const float gt =
                    (fmaf(As, et, WS ? Bc * wt : Bc) - scale * (1.f - a.eps) * wt) * fac;
                VT::store1(xrow, t, gt);
            }
        }
        // red_a is written again only after the next row's loads, by warps
        // that passed this row's second team barrier, which every warp of
        // the team reaches after reading red_a; red_b / red_c / red_i are
        // read before the next row's first team barrier
    }

    // copies still in flight (after a timeout) land before the CTA exits
    if (lead) {
        for (int k = 0; k < NB; ++k)
            if ((Q.pend >> k) & 1u)
                (void)mbar_wait_bounded(bar0 + 8u * static_cast<uint32_t>(k),
                                        (Q.pend_par >> k) & 1u, a.timeout_ns);
    }
    if (a.reduction != kRedNone) {
        need_counts();
        // fixed-order CTA sum of the per-thread partials: a thread holds the
        // rows whose target it owned, so the warp butterfly runs in fp32
        // (the fp64 pipe is narrow on this GPU) and the warps' sums in fp64
        float fl = accL, fz = accZ;
        int ic = accC;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            fl += __shfl_xor_sync(0xffffffffu, fl, o);
            fz += __shfl_xor_sync(0xffffffffu, fz, o);
            ic += __shfl_xor_sync(0xffffffffu, ic, o);
        }
        __syncthreads();  // the row loop's last reads of the shared arrays
        if (lane == 0) {
            red_d[0][warp] = fl;
            red_d[1][warp] = fz;
            red_n[warp] = ic;
        }
        __syncthreads();
        double L = 0.0, Z = 0.0;
        long long Cn = 0;
        if (tid == 0) {
            for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
                L += red_d[0][w];
                Z += red_d[1][w];
                Cn += red_n[w];
            }
        }
        __syncthreads();  // red_d is the epilogue's scratch next
        finish_scalars_cta(a, L, Z, Cn, D, n_valid, &s_flag, red_d[0], red_d[1], red_n);
    }
    // no CTA of a cluster leaves while another may still read its shared
    // memory
    if (CL > 1) {
        __syncwarp();
        cluster_sync();
    }
}

template <typename T, int NVL, bool CLU = false>
const void* reg_kernel_of(bool softcap, bool ws) {
    if (softcap)
        return ws ? (const void*)&ce_fwd_reg<T, true, true, NVL, CLU>
                  : (const void*)&ce_fwd_reg<T, true, false, NVL, CLU>;
    return ws ? (const void*)&ce_fwd_reg<T, false, true, NVL, CLU>
              : (const void*)&ce_fwd_reg<T, false, false, NVL, CLU>;
}

}  // namespace gbce
