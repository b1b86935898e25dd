// Forward for N-D logits [N, C, d1..dk] (class dimension 1) that reads every
// element from HBM once (the tt-mlir pull request #9324 review comment: the
// reductions run over every non-class dimension; row definitions, loss terms
// and gradient as in the 2-D kernels: Liger-Kernel cross-entropy profile,
// §Forward Pass, §Backward Pass, §Key Patterns).
//
// A position is one row of the 2-D definition; its C logits sit `inner`
// elements apart, so for one n the logits form a [C, inner] matrix whose
// rows are classes and whose columns are positions. A tile is P consecutive
// positions of one n (P x element size = 64 or 128 bytes a class row) and
// all C classes; a thread-block cluster of CL CTAs owns it, CTA k the class
// rows [k cc, (k + 1) cc) in its shared memory, loaded by a producer warp as
// 2-D TMA boxes of rb class rows (one mbarrier a block of rows). Sixteen
// consumer warps, each thread E positions (4 bytes of a class row) and every
// (512 / (P / E))-th row:
//  * pass A: maximum over the CTA's classes (and the first argmax when
//    predictions or accuracy are asked for), reduced over the row groups
//    in shared memory and over the cluster (each CTA stores its P records
//    into every CTA's shared memory and arrives once on its exchange
//    barrier; bounded waits; a one-CTA tile keeps its records);
//  * pass B: S = sum exp(x - M) and the smoothing sum; x at the target
//    read once from its row; the same two reductions;
//  * per-position outputs (rank 0 of the cluster) and the gradient's
//    coefficients; pass C: the gradient, stored to global memory from
//    registers, the one-hot term added where a block holds a target by
//    the thread that stored that row, each block of rows released to the
//    producer as the warps finish it, so the next tile's loads overlap the
//    rest of pass C.
// One HBM read and one write an element; the class slices stay on chip
// between the passes. Not for softcaps or class-weighted smoothing (the
// split kernels take those).
#include <cuda.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <string>

#include "ce_kernels.cuh"
#include "gbce.h"

namespace gbce {

ce_status tensor_map_rows_2d(CUtensorMap* map, int dtype, const void* p, int64_t outer,
                             int64_t inner, uint32_t box_inner, uint32_t box_outer);
ce_status record_cuda_failure(cudaError_t e, const char* what);
void record_message(const std::string& msg);

namespace {

constexpr int kNtConsumers = 512;               // sixteen consumer warps
constexpr int kNtThreads = kNtConsumers + 32;   // and the producer warp
constexpr int kNtMaxBlocks = 16;                // blocks of class rows a CTA
constexpr int kNtMaxCluster = 16;
constexpr int kNtBar = 1;                       // named barrier of the consumers

struct NdTileArgs {
    FwdArgs f;
    int64_t C, inner;
    int64_t tiles_per_n;  // ceil(inner / P)
    int64_t tiles;        // N * tiles_per_n
    int cc;               // classes a CTA (the cluster's last CTA may hold fewer)
    int rb;               // class rows a block (one TMA box)
    int nblk;             // blocks of a full slice
    uint32_t slice_bytes; // nblk * rb * row bytes
};

// Four bytes of a class row: E positions.
template <typename T>
struct NtIO;
template <>
struct NtIO<__nv_bfloat16> {
    static constexpr int E = 2;
    __device__ __forceinline__ static void unpack(uint32_t w, float (&f)[2]) {
        f[0] = __uint_as_float(w << 16);
        f[1] = __uint_as_float(w & 0xffff0000u);
    }
    __device__ __forceinline__ static uint32_t pack(const float (&f)[2]) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(f[0], f[1]);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
};
template <>
struct NtIO<__half> {
    static constexpr int E = 2;
    __device__ __forceinline__ static void unpack(uint32_t w, float (&f)[2]) {
        const __half2 h = *reinterpret_cast<const __half2*>(&w);
        const float2 v = __half22float2(h);
        f[0] = v.x;
        f[1] = v.y;
    }
    __device__ __forceinline__ static uint32_t pack(const float (&f)[2]) {
        const __half2 h = __floats2half2_rn(f[0], f[1]);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
};
template <>
struct NtIO<float> {
    static constexpr int E = 1;
    __device__ __forceinline__ static void unpack(uint32_t w, float (&f)[1]) {
        f[0] = __uint_as_float(w);
    }
    __device__ __forceinline__ static uint32_t pack(const float (&f)[1]) {
        return __float_as_uint(f[0]);
    }
};

__device__ __forceinline__ void nt_tma_load(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void nt_st_dsmem_f2(uint32_t addr, float2 v) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y)
                 : "memory");
}
__device__ __forceinline__ void nt_st_dsmem_f4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ void nt_fence_cluster() {
    asm volatile("fence.acq_rel.cluster;" ::: "memory");
}
__device__ __forceinline__ void nt_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                     cluster_addr)
                 : "memory");
}
__device__ __forceinline__ bool nt_wait_cluster(uint32_t bar, uint32_t parity,
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
__device__ __forceinline__ void nt_st_u32_hint(void* p, uint32_t v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.u32 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void nt_consumer_sync() {
    asm volatile("bar.sync %0, %1;" ::"r"(kNtBar), "r"(kNtConsumers) : "memory");
}

template <typename T, int TPR>
__global__ void __launch_bounds__(kNtThreads, 1)
ce_nd_tile(const __grid_constant__ CUtensorMap map, const __grid_constant__ NdTileArgs s) {
    using IO = NtIO<T>;
    constexpr int E = IO::E;
    constexpr int P = TPR * E;                  // positions a tile
    constexpr int RG = kNtConsumers / TPR;      // row groups
    constexpr uint32_t kRowBytes = P * sizeof(T);
    const FwdArgs& a = s.f;
    extern __shared__ unsigned char nt_raw[];
    __shared__ __align__(8) uint64_t full_bar[kNtMaxBlocks];
    __shared__ __align__(8) uint64_t empty_bar[kNtMaxBlocks];
    __shared__ __align__(8) uint64_t xbarA[2], xbarB[2];  // cluster exchanges, by tile parity
    __shared__ uint32_t s_issued[kNtMaxBlocks];           // 0, or 2 + parity of the last load
    __shared__ int s_failed;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t crank = cluster_ctarank();
    const uint32_t csize = cluster_nctarank();
    const int64_t clid = cluster_id_x();
    const int64_t ncl = ncluster_x();
    const int64_t C = s.C, inner = s.inner;
    const int c0 = static_cast<int>(crank) * s.cc;
    const int ncls = max(0, min(s.cc, static_cast<int>(C) - c0));  // classes this CTA holds
    const int nbu = (ncls + s.rb - 1) / s.rb;                       // blocks it uses
    // shared memory: the slice (128-byte aligned for the TMA), then the
    // exchange records [2][csize][P] (float2, then float4) and the row
    // groups' records [RG][P]
    const uint32_t raw0 = smem_u32(nt_raw);
    const uint32_t slice_s = (raw0 + 127u) & ~127u;
    unsigned char* slice = nt_raw + (slice_s - raw0);
    float2* xA = reinterpret_cast<float2*>(slice + s.slice_bytes);
    float4* xB = reinterpret_cast<float4*>(xA + 2 * csize * P);
    float4* red = xB + 2 * csize * P;

    if (tid == 0) {
        for (int j = 0; j < kNtMaxBlocks; ++j) {
            mbar_init(smem_u32(&full_bar[j]), 1);
            mbar_init(smem_u32(&empty_bar[j]), kNtConsumers / 32);
            s_issued[j] = 0;
        }
        for (int p = 0; p < 2; ++p) {
            mbar_init(smem_u32(&xbarA[p]), csize);
            mbar_init(smem_u32(&xbarB[p]), csize);
        }
        s_failed = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // a backward launched after this kernel may be scheduled now (it waits
    // for this grid before reading anything)
    pdl_launch_dependents();
    // every CTA's barriers are initialised before any other CTA arrives on them
    cluster_sync();

    if (warp == kNtConsumers / 32) {
        // ------------------------------------------------------------ producer
        // (the warp's lanes go round together; lane 0 waits and issues)
        int it = 0;
        int failed = 0;
        for (int64_t tile = clid; tile < s.tiles && !failed; tile += ncl, ++it) {
            const int64_t n = tile / s.tiles_per_n;
            const int x0 = static_cast<int>((tile - n * s.tiles_per_n) * P);
            const int64_t y0 = n * C + c0;
            for (int j = 0; j < nbu && !failed; ++j) {
                if (lane == 0) {
                    // the consumers have finished the previous tile's block j
                    if (!mbar_wait_bounded(smem_u32(&empty_bar[j]), (it & 1) ^ 1, a.timeout_ns)) {
                        failed = 1;
                    } else {
                        const uint32_t fb = smem_u32(&full_bar[j]);
                        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(s.rb) * kRowBytes);
                        nt_tma_load(slice_s + static_cast<uint32_t>(j * s.rb) * kRowBytes, &map,
                                    x0, static_cast<int>(y0 + static_cast<int64_t>(j) * s.rb), fb);
                        s_issued[j] = 2u + static_cast<uint32_t>(it & 1);
                    }
                }
                failed = __shfl_sync(0xffffffffu, failed, 0);
            }
        }
        if (failed && lane == 0) {
            atomicOr(&a.scratch->status, kDevErrTimeout);
            s_failed = 1;
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int tcol = tid % TPR;  // positions tcol * E .. of the tile
        const int rg = tid / TPR;    // row group: rows rg, rg + RG, ... of each block
        const uint64_t spol = l2_evict_first_policy();
        const bool smooth = a.eps > 0.f;
        const bool want_arg = a.want_pred || a.want_acc;
        const float inv_C = 1.f / static_cast<float>(C);
        const bool outputs = crank == 0 && rg == 0;  // per-position outputs: rank 0, row group 0
        bool failed = false;
        // D and the counted positions come from the count kernel launched just
        // before (programmatic dependent launch): read where first needed
        float D = 0.f;
        int n_valid = 0;
        bool have_counts = a.reduction == kRedNone;
        auto need_counts = [&]() {
            if (!have_counts) {
                pdl_wait();
                D = static_cast<float>(a.batch_counts[0]);
                n_valid = static_cast<int>(a.batch_counts[1]);
                have_counts = true;
            }
        };
        double accL = 0.0, accZ = 0.0;
        long long accC = 0;
        int it = 0;
#pragma unroll 1
        for (int64_t tile = clid; tile < s.tiles; tile += ncl, ++it) {
            const int par = it & 1;
            const int64_t n = tile / s.tiles_per_n;
            const int64_t sp0 = (tile - n * s.tiles_per_n) * P + tcol * E;  // first position in n
            const bool pos_ok = sp0 < inner;  // E divides inner: all E positions or none
            const int64_t r0 = n * inner + sp0;  // its row of the 2-D definition
            int tv[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                tv[e] = -1;
                if (pos_ok) {
                    const int64_t t = load_target(a, r0 + e);
                    if (row_counts(a, t))
                        tv[e] = static_cast<int>(t);
                    else if (outputs && t != a.ignore_index)
                        atomicOr(&a.scratch->status, kDevErrTarget);
                }
            }
            // ---- pass A: maximum and first argmax over this CTA's classes
            float m[E];
            int mi[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                m[e] = -INFINITY;
                mi[e] = INT_MAX;
            }
            for (int j = 0; j < nbu; ++j) {
                if (!failed &&
                    !mbar_wait_bounded(smem_u32(&full_bar[j]), static_cast<uint32_t>(par),
                                       a.timeout_ns)) {
                    failed = true;
                    atomicOr(&a.scratch->status, kDevErrTimeout);
                }
                const int rhi = min(ncls, (j + 1) * s.rb);
                if (want_arg) {
#pragma unroll 4
                    for (int r = j * s.rb + rg; r < rhi; r += RG) {
                        float f[E];
                        IO::unpack(*reinterpret_cast<const uint32_t*>(slice + r * kRowBytes + tcol * 4), f);
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            if (f[e] > m[e]) {  // rows in increasing order: the first maximum stays
                                m[e] = f[e];
                                mi[e] = c0 + r;
                            }
                        }
                    }
                } else {
#pragma unroll 8
                    for (int r = j * s.rb + rg; r < rhi; r += RG) {
                        float f[E];
                        IO::unpack(*reinterpret_cast<const uint32_t*>(slice + r * kRowBytes + tcol * 4), f);
#pragma unroll
                        for (int e = 0; e < E; ++e) m[e] = fmaxf(m[e], f[e]);
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < E; ++e)
                red[rg * P + tcol * E + e] = make_float4(m[e], __int_as_float(mi[e]), 0.f, 0.f);
            nt_consumer_sync();
            if (tid < P) {
                float M = -INFINITY;
                int I = INT_MAX;
                for (int g = 0; g < RG; ++g) {
                    const float4 q = red[g * P + tid];
                    const int iq = __float_as_int(q.y);
                    if (q.x > M || (q.x == M && iq < I)) {
                        M = q.x;
                        I = iq;
                    }
                }
                if (csize == 1) {
                    // one CTA a tile: the record stays in this CTA
                    xA[par * P + tid] = make_float2(M, __int_as_float(I));
                } else {
                    const uint32_t rec = smem_u32(&xA[(par * csize + crank) * P + tid]);
                    for (uint32_t q = 0; q < csize; ++q)
                        nt_st_dsmem_f2(map_to_rank(rec, q), make_float2(M, __int_as_float(I)));
                    nt_fence_cluster();
                }
            }
            nt_consumer_sync();
            if (csize > 1) {
                if (tid == 0)
                    for (uint32_t q = 0; q < csize; ++q)
                        nt_arrive_cluster(map_to_rank(smem_u32(&xbarA[par]), q));
                if (!failed && !nt_wait_cluster(smem_u32(&xbarA[par]),
                                                static_cast<uint32_t>(it >> 1) & 1u, a.timeout_ns)) {
                    failed = true;
                    atomicOr(&a.scratch->status, kDevErrTimeout);
                }
            }
            float sh[E];
            int xi[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                float M = -INFINITY;
                int I = INT_MAX;
                for (uint32_t q = 0; q < csize; ++q) {
                    const float2 v = xA[(par * csize + q) * P + tcol * E + e];
                    const int iq = __float_as_int(v.y);
                    if (v.x > M || (v.x == M && iq < I)) {
                        M = v.x;
                        I = iq;
                    }
                }
                sh[e] = M == -INFINITY ? 0.f : M;
                xi[e] = I == INT_MAX ? -1 : I;
            }
            // ---- pass B: S = sum exp(x - M), SZ = sum (x - M), x at the target
            float S[E], SZ[E], zt[E], fz[E];
#pragma unroll
            for (int e = 0; e < E; ++e) S[e] = SZ[e] = zt[e] = fz[e] = 0.f;
            for (int j = 0; j < nbu; ++j) {
                const int rhi = min(ncls, (j + 1) * s.rb);
#pragma unroll 8
                for (int r = j * s.rb + rg; r < rhi; r += RG) {
                    float f[E];
                    IO::unpack(*reinterpret_cast<const uint32_t*>(slice + r * kRowBytes + tcol * 4), f);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float d = f[e] - sh[e];
                        S[e] += ex2(d * kLog2e);
                        if (smooth) SZ[e] += d;
                    }
                }
            }
            // x at the target, read once by row group 0 when this CTA holds it
            if (rg == 0) {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int tr = tv[e] - c0;
                    if (tv[e] >= 0 && tr >= 0 && tr < ncls) {
                        float f[E];
                        IO::unpack(*reinterpret_cast<const uint32_t*>(slice + tr * kRowBytes + tcol * 4), f);
                        zt[e] = f[e];
                        fz[e] = 1.f;
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < E; ++e)
                red[rg * P + tcol * E + e] = make_float4(S[e], SZ[e], zt[e], fz[e]);
            nt_consumer_sync();
            if (tid < P) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int g = 0; g < RG; ++g) {
                    const float4 q = red[g * P + tid];
                    acc.x += q.x;
                    acc.y += q.y;
                    if (q.w != 0.f) {
                        acc.z = q.z;
                        acc.w = 1.f;
                    }
                }
                if (csize == 1) {
                    xB[par * P + tid] = acc;
                } else {
                    const uint32_t rec = smem_u32(&xB[(par * csize + crank) * P + tid]);
                    for (uint32_t q = 0; q < csize; ++q) nt_st_dsmem_f4(map_to_rank(rec, q), acc);
                    nt_fence_cluster();
                }
            }
            nt_consumer_sync();
            if (csize > 1) {
                if (tid == 0)
                    for (uint32_t q = 0; q < csize; ++q)
                        nt_arrive_cluster(map_to_rank(smem_u32(&xbarB[par]), q));
                if (!failed && !nt_wait_cluster(smem_u32(&xbarB[par]),
                                                static_cast<uint32_t>(it >> 1) & 1u, a.timeout_ns)) {
                    failed = true;
                    atomicOr(&a.scratch->status, kDevErrTimeout);
                }
            }
            // ---- per-position outputs and the gradient's coefficients
            need_counts();
            const float scale = a.reduction == kRedMean ? 1.f / D : 1.f;
            float ac[E], bc[E], tf[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                float St = 0.f, SZt = 0.f, zte = 0.f;
                for (uint32_t q = 0; q < csize; ++q) {
                    const float4 v = xB[(par * csize + q) * P + tcol * E + e];
                    St += v.x;
                    SZt += v.y;
                    if (v.w != 0.f) zte = v.z;
                }
                ac[e] = bc[e] = tf[e] = 0.f;
                if (!pos_ok) continue;
                const int64_t r = r0 + e;
                if (tv[e] >= 0) {
                    const float wt = a.weight ? __ldg(a.weight + tv[e]) : 1.f;
                    const float logS = logf(St);
                    if (outputs) {
                        float zl;
                        const float l =
                            row_loss(a, sh[e], logS, zte, wt, static_cast<float>(C), SZt, zl);
                        const bool correct = xi[e] == tv[e];
                        if (a.reduction == kRedNone) {
                            a.loss[r] = l;
                            if (a.want_z) a.zloss[r] = zl;
                            if (a.want_acc) a.acc[r] = correct ? 1.f : 0.f;
                        } else {
                            accL += static_cast<double>(l);
                            accZ += static_cast<double>(zl);
                            accC += correct ? 1 : 0;
                        }
                        if (a.want_pred) a.pred[r] = xi[e];
                    }
                    const float lse = sh[e] + logS;
                    ac[e] = scale * ((1.f - a.eps) * wt + a.eps + 2.f * a.lam * lse) / St;
                    bc[e] = -scale * a.eps * inv_C;
                    tf[e] = -scale * (1.f - a.eps) * wt;
                } else if (outputs) {
                    if (a.reduction == kRedNone) {
                        a.loss[r] = 0.f;
                        if (a.want_z) a.zloss[r] = 0.f;
                        if (a.want_acc) a.acc[r] = 0.f;
                    }
                    if (a.want_pred) a.pred[r] = -1;
                }
            }
            // ---- pass C: the gradient, block by block; each block goes back
            // to the producer once every consumer warp is done with it
            T* xg = reinterpret_cast<T*>(a.x) + n * C * inner + sp0;
            // the gradient of class row r for this thread's positions, with
            // the one-hot term at their targets (added apart, no contraction
            // into an FMA: with p_t = 1 the two cancel exactly)
            auto grad_row = [&](int r, bool onehot) {
                float f[E];
                IO::unpack(*reinterpret_cast<const uint32_t*>(slice + r * kRowBytes + tcol * 4), f);
                const int c = c0 + r;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    float g = fmaf(ac[e], ex2((f[e] - sh[e]) * kLog2e), bc[e]);
                    if (onehot && c == tv[e]) g = __fadd_rn(g, tf[e]);
                    f[e] = tv[e] >= 0 ? g : 0.f;  // exact zeros where a position does not count
                }
                nt_st_u32_hint(xg + static_cast<int64_t>(c) * inner, IO::pack(f), spol);
            };
            for (int j = 0; j < nbu; ++j) {
                if (a.grad && pos_ok) {
                    const int rlo = j * s.rb, rhi = min(ncls, rlo + s.rb);
#pragma unroll 8
                    for (int r = rlo + rg; r < rhi; r += RG) grad_row(r, false);
                    // the rows of this block holding a target of this
                    // thread's positions, stored again by the same thread
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const int tr = tv[e] - c0;
                        if (tv[e] >= 0 && tr >= rlo + rg && tr < rhi && (tr - rlo - rg) % RG == 0)
                            grad_row(tr, true);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&empty_bar[j]));
            }
        }
        if (failed && lane == 0) s_failed = 1;
        if (a.reduction != kRedNone) {
            need_counts();
            // thread tid < TPR of row group 0 holds its positions' partials
            // (rank 0 only): a fixed butterfly over warp 0, then the grid
            if (warp == 0) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    accL += __shfl_xor_sync(0xffffffffu, accL, o);
                    accZ += __shfl_xor_sync(0xffffffffu, accZ, o);
                    accC += __shfl_xor_sync(0xffffffffu, accC, o);
                }
                finish_scalars(a, blockIdx.x, gridDim.x, accL, accZ, accC, D, n_valid);
            }
        }
    }
    __syncthreads();
    if (s_failed && tid == kNtConsumers) {
        // loads that may still be in flight land before the CTA exits
        for (int j = 0; j < kNtMaxBlocks; ++j) {
            const uint32_t used = s_issued[j];
            if (used) (void)mbar_wait_bounded(smem_u32(&full_bar[j]), used & 1u, a.timeout_ns);
        }
    }
    // no CTA leaves while another CTA of the cluster may still store into it
    cluster_sync();
}

template <typename T>
const void* nd_tile_fn(int tpr) {
    return tpr == 32 ? (const void*)&ce_nd_tile<T, 32> : (const void*)&ce_nd_tile<T, 16>;
}

const void* nd_tile_kernel(int dtype, int tpr) {
    if (dtype == CE_F32) return nd_tile_fn<float>(tpr);
    if (dtype == CE_BF16) return nd_tile_fn<__nv_bfloat16>(tpr);
    if (dtype == CE_F16) return nd_tile_fn<__half>(tpr);
    return nullptr;
}

}  // namespace

// The single-read N-D forward for the call in `f` (rows = N * inner
// positions, V = C classes): plans the cluster (CTAs enough to hold a tile's
// classes in shared memory, at most max_cluster; 128-byte class rows when a
// cluster of at most 8 does, else, with narrow_rows, 64-byte ones and up to
// 16; of the sizes that fit, the one keeping the most SMs busy), encodes the
// class-row tensor map and launches. Returns CE_ERR_UNSUPPORTED (nothing
// launched) when the shape does not fit it; `after_count`: launched as a
// programmatic dependent of the count kernel just before.
ce_status nd_tile_launch(const FwdArgs& f, int dtype, int64_t N, int64_t C, int64_t inner,
                         int sm_count, int smem_optin, int max_cluster, bool narrow_rows,
                         bool after_count, cudaStream_t st) {
    const int64_t b = dtype == CE_F32 ? 4 : 2;
    const int E = static_cast<int>(4 / b);
    if (N * C > INT32_MAX || C > INT32_MAX / 2 || (inner * b) % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(f.x) % 16) != 0)
        return CE_ERR_UNSUPPORTED;
    for (int tpr : {32, 16}) {
        if (tpr == 16 && !narrow_rows) break;
        const void* fn = nd_tile_kernel(dtype, tpr);
        if (!fn) return CE_ERR_UNSUPPORTED;
        const int64_t P = static_cast<int64_t>(tpr) * E;
        const int64_t row_bytes = P * b;
        const int max_cl = std::min(max_cluster, tpr == 32 ? 8 : kNtMaxCluster);
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, fn);
        if (e != cudaSuccess) return record_cuda_failure(e, "N-D tile kernel attributes");
        const int64_t rg = kNtConsumers / tpr;
        // the exchange and row-group records a CTA, for the largest cluster
        const int64_t extra = 128 + 2 * max_cl * P * (8 + 16) + rg * P * 16;
        const int64_t budget = static_cast<int64_t>(smem_optin) - fa.sharedSizeBytes - extra;
        if (budget < row_bytes * 2) continue;
        const int64_t rows_max = std::min<int64_t>(budget / row_bytes, kNtMaxBlocks * 256);
        const int64_t cl_min = (C + rows_max - 1) / rows_max;
        if (cl_min > max_cl) continue;
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem_optin - fa.sharedSizeBytes));
        if (e == cudaSuccess && max_cl > 8)
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return record_cuda_failure(e, "N-D tile kernel attributes");
        // the cluster size that keeps the most SMs busy (clusters are placed
        // within a GPC, so some sizes leave SMs idle), the smaller on a tie
        struct Cand {
            int64_t cl = 0, cc = 0, rb = 0, nblk = 0, slice = 0, ncl = 0;
            size_t smem = 0;
        } best;
        for (int64_t cl0 = cl_min; cl0 <= max_cl; ++cl0) {
            const int64_t cc = (C + cl0 - 1) / cl0;
            const int64_t cl = (C + cc - 1) / cc;  // no empty CTA
            if (cl != cl0) continue;
            int64_t nblk = (cc + 255) / 256;
            int64_t rb = (cc + nblk - 1) / nblk;
            rb += rb & 1;  // blocks stay 128-byte aligned
            if (rb > 256) {
                ++nblk;
                rb = (cc + nblk - 1) / nblk;
                rb += rb & 1;
            }
            if (nblk > kNtMaxBlocks || rb > 256) continue;
            const int64_t slice = nblk * rb * row_bytes;
            const size_t smem = static_cast<size_t>(slice + 128 + 2 * cl * P * (8 + 16) + rg * P * 16);
            if (smem + fa.sharedSizeBytes > static_cast<size_t>(smem_optin)) continue;
            cudaLaunchConfig_t q = {};
            q.blockDim = dim3(kNtThreads);
            q.dynamicSmemBytes = smem;
            cudaLaunchAttribute ca;
            ca.id = cudaLaunchAttributeClusterDimension;
            ca.val.clusterDim.x = static_cast<unsigned>(cl);
            ca.val.clusterDim.y = 1;
            ca.val.clusterDim.z = 1;
            q.attrs = &ca;
            q.numAttrs = 1;
            q.gridDim = dim3(static_cast<unsigned>(cl * sm_count));
            int ncl = 0;
            if (cudaOccupancyMaxActiveClusters(&ncl, fn, &q) != cudaSuccess || ncl < 1) {
                cudaGetLastError();
                continue;
            }
            if (ncl * cl > best.ncl * best.cl) best = Cand{cl, cc, rb, nblk, slice, ncl, smem};
        }
        if (best.cl == 0) continue;
        NdTileArgs s = {};
        s.f = f;
        s.C = C;
        s.inner = inner;
        s.tiles_per_n = (inner + P - 1) / P;
        s.tiles = N * s.tiles_per_n;
        s.cc = static_cast<int>(best.cc);
        s.rb = static_cast<int>(best.rb);
        s.nblk = static_cast<int>(best.nblk);
        s.slice_bytes = static_cast<uint32_t>(best.slice);
        // a launch's CTAs stay within the scratch's partial-sum slots
        const int64_t units = std::max<int64_t>(
            1, std::min<int64_t>({s.tiles, best.ncl, kMaxUnits / best.cl,
                                  static_cast<int64_t>(sm_count) * 8 / best.cl}));
        CUtensorMap map;
        ce_status rc = tensor_map_rows_2d(&map, dtype, f.x, N * C, inner,
                                          static_cast<uint32_t>(P), static_cast<uint32_t>(best.rb));
        if (rc != CE_OK) return rc;
        cudaLaunchConfig_t lc = {};
        lc.blockDim = dim3(kNtThreads);
        lc.dynamicSmemBytes = best.smem;
        lc.stream = st;
        lc.gridDim = dim3(static_cast<unsigned>(units * best.cl));
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(best.cl);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        lc.attrs = attr;
        lc.numAttrs = 1;
        if (after_count) {
            attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[1].val.programmaticStreamSerializationAllowed = 1;
            lc.numAttrs = 2;
        }
        void* args[] = {&map, &s};
        e = cudaLaunchKernelExC(&lc, fn, args);
        if (e != cudaSuccess) return record_cuda_failure(e, "N-D tile kernel launch");
        if (std::getenv("GBCE_VERBOSE"))
            std::fprintf(stderr, "gbce nd tile: C=%lld inner=%lld P=%lld CL=%lld cc=%lld rb=%lld "
                                 "nblk=%lld clusters=%lld tiles=%lld\n",
                         static_cast<long long>(C), static_cast<long long>(inner),
                         static_cast<long long>(P), static_cast<long long>(best.cl),
                         static_cast<long long>(best.cc), static_cast<long long>(best.rb),
                         static_cast<long long>(best.nblk), static_cast<long long>(units),
                         static_cast<long long>(s.tiles));
        return CE_OK;
    }
    return CE_ERR_UNSUPPORTED;
}

}  // namespace gbce
