// Forward for N-D logits [N, C, d1..dk] (class dimension 1) when one tile
// of positions x all C classes does not fit on chip or there are too few
// tiles to fill the GPU: the classes of each tile are split into chunks
// that separate CTAs take (the tt-mlir pull request #9324 review comment:
// the reductions run over every non-class dimension; row definitions, loss
// terms and gradient as in the 2-D kernels: Liger-Kernel cross-entropy
// profile, §Forward Pass, §Backward Pass, §Key Patterns).
//
// A position is one row of the 2-D definition; its C logits sit `inner`
// elements apart. A tile is 32 * VP consecutive positions (VP = the
// positions of one 16-byte vector, or 1), a work item one (tile, chunk of
// classes). Three launches:
//   nd_stats  every item, once over its logits: online statistics per
//             position over the chunk's classes (running maximum m with
//             S = sum exp(z - m) and SZ = sum w (z - m) rescaled when m
//             grows, W = sum w, first raw argmax), merged over the CTA's
//             warps in warp order, one record per (position, chunk);
//   nd_merge  one warp per position merges its chunks' records (fixed lane
//             split and butterfly: the same bits every call), writes the
//             per-position outputs and the gradient's coefficients, and
//             adds the reduced scalars (last-CTA epilogue);
//   nd_grad   every item again, in reverse order (the last items' logits
//             are the likeliest to still be in L2): the gradient in place.
// Each element is read twice and written once.
#pragma once

#include <climits>
#include <type_traits>

#include "ce_fwd_nd.cuh"

namespace gbce {

constexpr int kNdSplitWarps = kNdSplitThreads / 32;

// exp2 argument of z - m (m the shift): the difference first, so the
// maximum's term is exp2(0) = 1 exactly (a position whose other classes
// are all -inf then has loss 0 exactly, as the definition gives).
template <typename T>
__device__ __forceinline__ float nd_arg(float z, float m, float /*mL*/) {
    return (z - m) * kLog2e;
}

// Statistics of one chunk of classes for the tile's positions: each warp
// takes every NW-th class of the chunk, U at a time (loads issued first);
// the running maximum is checked once per U classes and position.
// SMOOTH: the smoothing sums SZ and W are formed (label smoothing on).
// Vector positions (16 bytes a lane): each warp streams its classes
// through its own ring of kNdRing stages of U class rows in shared memory
// (cp.async, 16 bytes a lane, each lane reading back only what it copied),
// so the bytes in flight do not hold registers. The ring is reused for the
// merge over the warps at the end of each item.
constexpr int kNdRing = 4;
template <int VP>
constexpr size_t nd_stats_smem() {
    constexpr int U = VP > 1 ? 4 : 8;
    const size_t ring = VP > 1 ? static_cast<size_t>(kNdSplitWarps) * kNdRing * U * 32 * 16 : 0;
    const size_t red = static_cast<size_t>(kNdSplitWarps) * 32 * VP * sizeof(NdRec);
    return ring > red ? ring : red;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename T, int VP, bool SOFTCAP, bool ARGMAX, bool SMOOTH>
__global__ void __launch_bounds__(kNdSplitThreads, 2)
ce_nd_stats(const __grid_constant__ NdSplitArgs s) {
    using IO = NdIO<T, VP>;
    using Raw = typename IO::Raw;
    constexpr int NW = kNdSplitWarps;
    constexpr int P = 32 * VP;
    constexpr int U = VP > 1 ? 4 : 8;  // classes a step
    extern __shared__ __align__(16) unsigned char nd_dyn[];
    NdRec (*red)[P] = reinterpret_cast<NdRec (*)[P]>(nd_dyn);  // after the item's loop
    const FwdArgs& a = s.f;
    const int tid = threadIdx.x, lane = tid & 31, wy = tid >> 5;
    const int C = static_cast<int>(a.V);
    const int64_t inner = a.inner;
    const bool wsmooth = SMOOTH && a.weight != nullptr;
    const int64_t items = s.tiles * s.nch;
#pragma unroll 1
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int64_t tile = it / s.nch;
        const int ch = static_cast<int>(it - tile * s.nch);
        const int c0 = ch * s.cc, c1 = min(C, c0 + s.cc);
        const int64_t rl = tile * P + static_cast<int64_t>(lane) * VP;
        const bool lane_ok = rl < a.rows;  // VP divides inner, hence rows
        int64_t lb = 0;
        if (lane_ok) {
            const int64_t n = rl / inner;
            lb = n * C * inner + (rl - n * inner);
        }
        float m[VP], S[VP], SZ[VP], xm[VP];
        int xi[VP];
#pragma unroll
        for (int v = 0; v < VP; ++v) {
            m[v] = -INFINITY;
            S[v] = 0.f;
            SZ[v] = 0.f;
            xm[v] = -INFINITY;
            xi[v] = INT_MAX;
        }
        float Wn = 0.f;
        // n classes from c (step NW) whose raw values are in r
        auto step = [&](int c, int n, const Raw (&r)[U]) {
            float z[U][VP];
            float wc[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (u < n) {
                    IO::unpack(r[u], z[u]);
                    wc[u] = wsmooth ? __ldg(a.weight + c + u * NW) : 1.f;
                }
            }
            if (ARGMAX) {
                // classes in increasing order: a later equal value never wins
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (u < n) {
#pragma unroll
                        for (int v = 0; v < VP; ++v)
                            if (z[u][v] > xm[v]) {
                                xm[v] = z[u][v];
                                xi[v] = c + u * NW;
                            }
                    }
            }
            if (SOFTCAP) {
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (u < n) {
#pragma unroll
                        for (int v = 0; v < VP; ++v)
                            z[u][v] = a.softcap * tanh_from_scaled(z[u][v] * a.sc_k2);
                    }
            }
#pragma unroll
            for (int v = 0; v < VP; ++v) {
                float bm = z[0][v];
#pragma unroll
                for (int u = 1; u < U; ++u)
                    if (u < n) bm = fmaxf(bm, z[u][v]);
                if (bm > m[v]) {
                    // the running maximum grows: rescale what was summed
                    if (m[v] != -INFINITY) {
                        const float d = m[v] - bm;
                        S[v] *= ex2(d * kLog2e);
                        if (SMOOTH) SZ[v] = fmaf(Wn, d, SZ[v]);
                    }
                    m[v] = bm;
                }
                const float ms = m[v] == -INFINITY ? 0.f : m[v];
                const float mL = ms * kLog2e;
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (u < n) {
                        S[v] += ex2(nd_arg<T>(z[u][v], ms, mL));
                        if (SMOOTH) SZ[v] = fmaf(wc[u], z[u][v] - ms, SZ[v]);
                    }
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (u < n) Wn += wc[u];
        };
        auto load = [&](int c) -> Raw {
            return lane_ok ? IO::load(a.x, lb + static_cast<int64_t>(c) * inner) : Raw{};
        };
        if constexpr (VP > 1) {
            // this warp's classes c0 + wy + NW j, j < ncw, in blocks of U
            const int first = c0 + wy;
            const int ncw = first < c1 ? (c1 - first + NW - 1) / NW : 0;
            const int nb = (ncw + U - 1) / U;
            const uint32_t ring =
                smem_u32(nd_dyn) + static_cast<uint32_t>(wy * kNdRing * U * 32 + lane) * 16u;
            auto issue = [&](int blk) {
                if (blk < nb && lane_ok) {
                    const int n = min(U, ncw - blk * U);
                    const uint32_t slot = ring + static_cast<uint32_t>((blk % kNdRing) * U * 32) * 16u;
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (u < n)
                            cp_async16(slot + static_cast<uint32_t>(u * 32) * 16u,
                                       static_cast<const T*>(a.x) + lb +
                                           static_cast<int64_t>(first + (blk * U + u) * NW) * inner);
                }
                cp_async_commit();  // (possibly empty: the group count stays uniform)
            };
#pragma unroll
            for (int b = 0; b < kNdRing - 1; ++b) issue(b);
#pragma unroll 1
            for (int blk = 0; blk < nb; ++blk) {
                cp_async_wait<kNdRing - 2>();  // block blk has landed
                Raw r[U];
                const uint4* sl = reinterpret_cast<const uint4*>(nd_dyn) +
                                  (wy * kNdRing + blk % kNdRing) * U * 32 + lane;
#pragma unroll
                for (int u = 0; u < U; ++u) r[u] = sl[u * 32];
                issue(blk + kNdRing - 1);  // into the slot read one block ago
                step(first + blk * U * NW, min(U, ncw - blk * U), r);
            }
            cp_async_wait<0>();
            __syncthreads();  // every warp is done with its ring: red takes the space
        } else {
            int c = c0 + wy;
#pragma unroll 1
            for (; c + (U - 1) * NW < c1; c += U * NW) {
                Raw r[U];
#pragma unroll
                for (int u = 0; u < U; ++u) r[u] = load(c + u * NW);
                step(c, U, r);
            }
            if (c < c1) {  // the chunk's last classes of this warp: fewer than U
                Raw r[U];
                const int n = (c1 - c + NW - 1) / NW;
#pragma unroll
                for (int u = 0; u < U; ++u) r[u] = u < n ? load(c + u * NW) : Raw{};
                step(c, n, r);
            }
        }
#pragma unroll
        for (int v = 0; v < VP; ++v)
            red[wy][lane * VP + v] = NdRec{m[v], S[v], SZ[v], Wn, xm[v], xi[v]};
        __syncthreads();
        for (int p = tid; p < P; p += kNdSplitThreads) {
            const NdRec& r0 = red[0][p];
            RowStats acc{r0.m, r0.S, r0.SZ, r0.Wn, r0.xmax, r0.idx};
#pragma unroll
            for (int w = 1; w < NW; ++w) {
                const NdRec& r = red[w][p];
                stats_merge(acc, RowStats{r.m, r.S, r.SZ, r.Wn, r.xmax, r.idx});
            }
            s.rec[(tile * P + p) * s.nch + ch] =
                NdRec{acc.m, acc.S, acc.SZ, acc.Wn, acc.xmax, acc.idx};
        }
        __syncthreads();  // red is written again by the next item
    }
    // Launched as a programmatic dependent of the count kernel, it reads
    // nothing that kernel writes; this wait keeps it from completing before
    // the count kernel, so the merge launched after it sees the counts.
    pdl_wait();
}

// One warp a position: lane l merges chunks l, l + 32, ... in order, then a
// fixed butterfly combines the lanes (stats_merge does not depend on the
// order of its operands, so every lane ends with the same bits).
template <typename T, bool SOFTCAP>
__global__ void __launch_bounds__(kNdSplitThreads)
ce_nd_merge(const __grid_constant__ NdSplitArgs s) {
    const FwdArgs& a = s.f;
    constexpr int NW = kNdSplitWarps;
    __shared__ double red_d[2 * NW];
    __shared__ long long red_n[NW];
    __shared__ int s_flag;
    const int tid = threadIdx.x, lane = tid & 31, wy = tid >> 5;
    const int C = static_cast<int>(a.V);
    const int64_t inner = a.inner;
    const bool smooth = a.eps > 0.f;
    const bool wsmooth = smooth && a.weight != nullptr;
    float D = 0.f;
    int n_valid = 0;
    if (a.reduction != kRedNone) {
        D = static_cast<float>(a.batch_counts[0]);
        n_valid = static_cast<int>(a.batch_counts[1]);
    }
    float Wsum = static_cast<float>(C);
    if (wsmooth) {
        // W = sum of the class weights, the same order in every CTA
        __shared__ float red_w[kNdSplitThreads / 32];
        float w = 0.f;
        for (int c = tid; c < C; c += kNdSplitThreads) w += __ldg(a.weight + c);
        Wsum = block_sum_fixed<kNdSplitThreads>(w, red_w);
        __syncthreads();
    }
    const float inv_C = 1.f / static_cast<float>(C);
    const float scale = a.reduction == kRedMean ? 1.f / D : 1.f;
    const float Wf = wsmooth ? Wsum * inv_C : 1.f;
    double accL = 0.0, accZ = 0.0;
    long long accC = 0;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * NW;
#pragma unroll 1
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * NW + wy; r < a.rows; r += nwarps) {
        RowStats acc = empty_stats();
        for (int c = lane; c < s.nch; c += 32) {
            const NdRec q = s.rec[r * s.nch + c];
            stats_merge(acc, RowStats{q.m, q.S, q.SZ, q.Wn, q.xmax, q.idx});
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const RowStats b = shfl_xor_stats(acc, o);
            stats_merge(acc, b);
        }
        if (lane != 0) continue;
        const int64_t t = load_target(a, r);
        const bool counted = row_counts(a, t);
        if (!counted && t != a.ignore_index) atomicOr(&a.scratch->status, kDevErrTarget);
        NdCoef k{0.f, 0.f, 0.f, 0.f};
        const float shift = acc.m == -INFINITY ? 0.f : acc.m;
        k.shift = shift;
        if (counted) {
            const int64_t n = r / inner;
            const float xt = Vec<T>::load1(a.x, n * C * inner + t * inner + (r - n * inner));
            const float zt = SOFTCAP ? a.softcap * tanh_from_scaled(xt * a.sc_k2) : xt;
            const float wt = a.weight ? __ldg(a.weight + t) : 1.f;
            const float logS = logf(acc.S);
            // the chunk records' SZ are relative to their own maxima, merged
            // to the position's maximum; W of the smoothing term is the
            // weights' sum (or C)
            float zl;
            const float l = row_loss(a, shift, logS, zt, wt, wsmooth ? Wsum : static_cast<float>(C),
                                     acc.SZ, zl);
            const bool correct = acc.idx == static_cast<int>(t);
            if (a.reduction == kRedNone) {
                a.loss[r] = l;
                if (a.want_z) a.zloss[r] = zl;
                if (a.want_acc) a.acc[r] = correct ? 1.f : 0.f;
            } else {
                accL += static_cast<double>(l);
                accZ += static_cast<double>(zl);
                accC += correct ? 1 : 0;
            }
            if (a.want_pred) a.pred[r] = acc.idx;
            const float lse = shift + logS;
            k.ac = scale * ((1.f - a.eps) * wt + a.eps * Wf + 2.f * a.lam * lse) / acc.S;
            k.bc = -scale * a.eps * inv_C;
            // the target's element: the one-hot term added
            // the one-hot term added apart (no contraction into an FMA: with
            // p_t = 1 the two cancel exactly)
            const float et = ex2((zt - shift) * kLog2e);
            const float tfix = -scale * (1.f - a.eps) * wt;
            float gt = __fadd_rn(fmaf(k.ac, et, k.bc * (wsmooth ? wt : 1.f)), tfix);
            if (SOFTCAP) {
                const float th = tanh_from_scaled(xt * a.sc_k2);
                gt *= fmaf(-th, th, 1.f);
            }
            k.gt = gt;
        } else {
            if (a.reduction == kRedNone) {
                a.loss[r] = 0.f;
                if (a.want_z) a.zloss[r] = 0.f;
                if (a.want_acc) a.acc[r] = 0.f;
            }
            if (a.want_pred) a.pred[r] = -1;
        }
        s.coef[r] = k;
        s.tpos[r] = counted ? static_cast<int>(t) : -1;
    }
    if (a.reduction != kRedNone) {
        // lane 0 of each warp holds its positions' partials: warps in order
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

// The gradient of one chunk of classes for the tile's positions, classes
// split over the warps as in ce_nd_stats; the target's element is then
// overwritten with its whole gradient by the thread that wrote it.
template <typename T, int VP, bool SOFTCAP>
__global__ void __launch_bounds__(kNdSplitThreads)
ce_nd_grad(const __grid_constant__ NdSplitArgs s) {
    using IO = NdIO<T, VP>;
    using Raw = typename IO::Raw;
    constexpr int NW = kNdSplitWarps;
    constexpr int P = 32 * VP;
    constexpr int U = VP > 1 ? 8 : 16;  // loads in flight a thread
    const FwdArgs& a = s.f;
    const int tid = threadIdx.x, lane = tid & 31, wy = tid >> 5;
    const int C = static_cast<int>(a.V);
    const int64_t inner = a.inner;
    const bool wsmooth = a.eps > 0.f && a.weight != nullptr;
    const int64_t items = s.tiles * s.nch;
    // a backward launched after this kernel may be scheduled now (it waits
    // for this grid before reading anything)
    pdl_launch_dependents();
#pragma unroll 1
    for (int64_t i = blockIdx.x; i < items; i += gridDim.x) {
        const int64_t it = items - 1 - i;
        const int64_t tile = it / s.nch;
        const int ch = static_cast<int>(it - tile * s.nch);
        const int c0 = ch * s.cc, c1 = min(C, c0 + s.cc);
        const int64_t rl = tile * P + static_cast<int64_t>(lane) * VP;
        const bool lane_ok = rl < a.rows;
        int64_t lb = 0;
        float sh[VP], shL[VP], ac[VP], bc[VP], gt[VP];
        int tv[VP];
#pragma unroll
        for (int v = 0; v < VP; ++v) {
            sh[v] = shL[v] = ac[v] = bc[v] = gt[v] = 0.f;
            tv[v] = -1;
        }
        if (lane_ok) {
            const int64_t n = rl / inner;
            lb = n * C * inner + (rl - n * inner);
#pragma unroll
            for (int v = 0; v < VP; ++v) {
                const NdCoef k = s.coef[rl + v];
                sh[v] = k.shift;
                shL[v] = k.shift * kLog2e;
                ac[v] = k.ac;
                bc[v] = k.bc;
                gt[v] = k.gt;
                tv[v] = s.tpos[rl + v];
            }
        }
        auto body = [&](int c, const Raw& r) {
            float f[VP];
            IO::unpack(r, f);
            const float wc = wsmooth ? __ldg(a.weight + c) : 1.f;
#pragma unroll
            for (int v = 0; v < VP; ++v) {
                float g;
                if (SOFTCAP) {
                    const float th = tanh_from_scaled(f[v] * a.sc_k2);
                    const float z = th * a.softcap;
                    g = fmaf(ac[v], ex2(nd_arg<T>(z, sh[v], shL[v])), bc[v] * wc) *
                        fmaf(-th, th, 1.f);
                } else {
                    g = fmaf(ac[v], ex2(nd_arg<T>(f[v], sh[v], shL[v])), bc[v] * wc);
                }
                // positions that do not count get exact zeros
                f[v] = tv[v] >= 0 ? g : 0.f;
            }
            if (lane_ok) IO::store(a.x, lb + static_cast<int64_t>(c) * inner, IO::pack(f));
        };
        nd_class_loop<U, Raw>(c0 + wy, NW, c1, [&](int c) -> Raw {
            return lane_ok ? IO::load(a.x, lb + static_cast<int64_t>(c) * inner) : Raw{};
        }, body);
        if (lane_ok) {
#pragma unroll
            for (int v = 0; v < VP; ++v) {
                const int t = tv[v];
                if (t >= c0 && t < c1 && (t - c0) % NW == wy)
                    Vec<T>::store1(a.x, lb + static_cast<int64_t>(t) * inner + v, gt[v]);
            }
        }
    }
}

// Few classes (C <= 48) and vector positions: a warp owns a
// whole tile of 32 VP positions and all C classes. It copies the tile into
// its own C x 512 bytes of shared memory (cp.async, each lane its 16 bytes
// a class, read back only by that lane), then takes the maximum and first
// argmax, the sums and the gradient from there: no CTA barrier and no
// merge across warps, so the CTA's warps run their tiles independently
// and hide each other's HBM latency. One read and one write an element.
constexpr int kNdWarpMaxC = 48;  // 8 warps x 48 x 512 bytes: 192 KB a CTA
constexpr int kNdWarpThreads = 256;
template <typename T, bool SOFTCAP, bool ARGMAX>
__global__ void __launch_bounds__(kNdWarpThreads)
ce_nd_warp(const __grid_constant__ FwdArgs a) {
    constexpr int VP = Vec<T>::N;
    constexpr int P = 32 * VP;
    constexpr int NW = kNdWarpThreads / 32;
    using IO = NdIO<T, VP>;
    extern __shared__ __align__(16) unsigned char nd_dyn[];
    __shared__ double red_d[2 * NW];
    __shared__ long long red_n[NW];
    __shared__ int s_flag;
    const int tid = threadIdx.x, lane = tid & 31, wy = tid >> 5;
    const int C = static_cast<int>(a.V);
    const int64_t inner = a.inner;
    const bool smooth = a.eps > 0.f;
    const bool wsmooth = smooth && a.weight != nullptr;
    // this lane's 16-byte slot of class c: tile + (c * 32 + lane) * 16
    const uint32_t tile = smem_u32(nd_dyn) + static_cast<uint32_t>(wy * C * 32 + lane) * 16u;
    const uint4* tl = reinterpret_cast<const uint4*>(nd_dyn) + wy * C * 32 + lane;
    // a backward launched after this kernel may be scheduled now (it waits
    // for this grid before reading anything)
    pdl_launch_dependents();
    // D and the counted positions come from the count kernel launched just
    // before, which this launch overlaps (programmatic dependent launch): read
    // where first needed, after the first tile's statistics
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
    float Wsum = static_cast<float>(C);
    if (wsmooth) {
        // W = sum of the class weights, the same order in every thread
        float w = 0.f;
        for (int c = 0; c < C; ++c) w += __ldg(a.weight + c);
        Wsum = w;
    }
    const float inv_C = 1.f / static_cast<float>(C);
    const float Wf = wsmooth ? Wsum * inv_C : 1.f;
    double accL = 0.0, accZ = 0.0;
    long long accC = 0;
    const int64_t ntiles = (a.rows + P - 1) / P;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * NW;
#pragma unroll 1
    for (int64_t ti = static_cast<int64_t>(blockIdx.x) * NW + wy; ti < ntiles; ti += nwarps) {
        const int64_t rl = ti * P + static_cast<int64_t>(lane) * VP;
        const bool lane_ok = rl < a.rows;  // VP divides inner, hence rows
        int64_t lb = 0;
        if (lane_ok) {
            const int64_t n = rl / inner;
            lb = n * C * inner + (rl - n * inner);
            for (int c = 0; c < C; ++c)
                cp_async16(tile + static_cast<uint32_t>(c * 32) * 16u,
                           static_cast<const T*>(a.x) + lb + static_cast<int64_t>(c) * inner);
        }
        cp_async_commit();
        int tv[VP];
#pragma unroll
        for (int v = 0; v < VP; ++v) {
            int t = -1;
            if (lane_ok) {
                const int64_t tt = load_target(a, rl + v);
                if (row_counts(a, tt))
                    t = static_cast<int>(tt);
                else if (tt != a.ignore_index)
                    atomicOr(&a.scratch->status, kDevErrTarget);
            }
            tv[v] = t;
        }
        cp_async_wait<0>();
        // ---- maximum of z and first argmax of x
        float m[VP], xm[VP];
        int xi[VP];
#pragma unroll
        for (int v = 0; v < VP; ++v) {
            m[v] = -INFINITY;
            xm[v] = -INFINITY;
            xi[v] = -1;
        }
#pragma unroll 1
        for (int c = 0; c < C; ++c) {
            float f[VP];
            IO::unpack(tl[c * 32], f);
#pragma unroll
            for (int v = 0; v < VP; ++v) {
                if (ARGMAX && f[v] > xm[v]) {  // classes in increasing order
                    xm[v] = f[v];
                    xi[v] = c;
                }
                const float z = SOFTCAP ? a.softcap * tanh_from_scaled(f[v] * a.sc_k2) : f[v];
                m[v] = fmaxf(m[v], z);
            }
        }
        // ---- S = sum exp(z - M), SZ = sum w (z - M), z at the target
        float S[VP], SZ[VP], zt[VP], sh[VP], shL[VP];
#pragma unroll
        for (int v = 0; v < VP; ++v) {
            sh[v] = m[v] == -INFINITY ? 0.f : m[v];
            shL[v] = sh[v] * kLog2e;
            S[v] = 0.f;
            SZ[v] = 0.f;
            zt[v] = 0.f;
        }
#pragma unroll 1
        for (int c = 0; c < C; ++c) {
            float f[VP];
            IO::unpack(tl[c * 32], f);
            const float wc = wsmooth ? __ldg(a.weight + c) : 1.f;
#pragma unroll
            for (int v = 0; v < VP; ++v) {
                const float z = SOFTCAP ? a.softcap * tanh_from_scaled(f[v] * a.sc_k2) : f[v];
                S[v] += ex2(nd_arg<T>(z, sh[v], shL[v]));
                if (smooth) SZ[v] = fmaf(wc, z - sh[v], SZ[v]);
                if (c == tv[v]) zt[v] = z;
            }
        }
        // ---- per-position outputs and the gradient's coefficients
        need_counts();
        const float scale = a.reduction == kRedMean ? 1.f / D : 1.f;
        float ac[VP], bc[VP], tf[VP];
#pragma unroll
        for (int v = 0; v < VP; ++v) {
            ac[v] = bc[v] = tf[v] = 0.f;
            if (!lane_ok) continue;
            const int64_t r = rl + v;
            if (tv[v] >= 0) {
                const float wt = a.weight ? __ldg(a.weight + tv[v]) : 1.f;
                const float logS = logf(S[v]);
                float zl;
                const float l = row_loss(a, sh[v], logS, zt[v], wt, Wsum, SZ[v], zl);
                const bool correct = xi[v] == tv[v];
                if (a.reduction == kRedNone) {
                    a.loss[r] = l;
                    if (a.want_z) a.zloss[r] = zl;
                    if (a.want_acc) a.acc[r] = correct ? 1.f : 0.f;
                } else {
                    accL += static_cast<double>(l);
                    accZ += static_cast<double>(zl);
                    accC += correct ? 1 : 0;
                }
                if (a.want_pred) a.pred[r] = xi[v];
                const float lse = sh[v] + logS;
                ac[v] = scale * ((1.f - a.eps) * wt + a.eps * Wf + 2.f * a.lam * lse) / S[v];
                bc[v] = -scale * a.eps * inv_C;
                tf[v] = -scale * (1.f - a.eps) * wt;
            } else {
                if (a.reduction == kRedNone) {
                    a.loss[r] = 0.f;
                    if (a.want_z) a.zloss[r] = 0.f;
                    if (a.want_acc) a.acc[r] = 0.f;
                }
                if (a.want_pred) a.pred[r] = -1;
            }
        }
        // ---- the gradient in place
        if (a.grad && lane_ok) {
#pragma unroll 1
            for (int c = 0; c < C; ++c) {
                float f[VP];
                IO::unpack(tl[c * 32], f);
                const float wc = wsmooth ? __ldg(a.weight + c) : 1.f;
#pragma unroll
                for (int v = 0; v < VP; ++v) {
                    float g, th = 0.f, z;
                    if (SOFTCAP) {
                        th = tanh_from_scaled(f[v] * a.sc_k2);
                        z = th * a.softcap;
                    } else {
                        z = f[v];
                    }
                    g = fmaf(ac[v], ex2(nd_arg<T>(z, sh[v], shL[v])), bc[v] * wc);
                    if (c == tv[v]) g += tf[v];
                    if (SOFTCAP) g *= fmaf(-th, th, 1.f);
                    f[v] = tv[v] >= 0 ? g : 0.f;  // exact zeros where a position does not count
                }
                IO::store(a.x, lb + static_cast<int64_t>(c) * inner, IO::pack(f));
            }
        }
        __syncwarp();  // every lane done with the tile before the next copies
    }
    if (a.reduction != kRedNone) {
        need_counts();
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

template <typename T>
const void* nd_warp_of(bool softcap, bool argmax) {
    if (softcap)
        return argmax ? (const void*)&ce_nd_warp<T, true, true> : (const void*)&ce_nd_warp<T, true, false>;
    return argmax ? (const void*)&ce_nd_warp<T, false, true> : (const void*)&ce_nd_warp<T, false, false>;
}

// Entry points of one logit type by (vector positions, softcap, argmax).
template <typename T>
NdSplitFns nd_split_of(bool vec, bool softcap, bool argmax, bool smooth) {
    constexpr int VPV = Vec<T>::N;
    NdSplitFns f{};
#define GBCE_ND_SPLIT(VP, SC)                                                                 \
    f.stats = argmax ? (smooth ? (const void*)&ce_nd_stats<T, VP, SC, true, true>              \
                               : (const void*)&ce_nd_stats<T, VP, SC, true, false>)            \
                     : (smooth ? (const void*)&ce_nd_stats<T, VP, SC, false, true>             \
                               : (const void*)&ce_nd_stats<T, VP, SC, false, false>);          \
    f.merge = (const void*)&ce_nd_merge<T, SC>;                                               \
    f.grad = (const void*)&ce_nd_grad<T, VP, SC>;                                             \
    f.stats_smem = nd_stats_smem<VP>();
    if (vec) {
        if (softcap) {
            GBCE_ND_SPLIT(VPV, true)
        } else {
            GBCE_ND_SPLIT(VPV, false)
        }
    } else {
        if (softcap) {
            GBCE_ND_SPLIT(1, true)
        } else {
            GBCE_ND_SPLIT(1, false)
        }
    }
#undef GBCE_ND_SPLIT
    return f;
}

}  // namespace gbce
