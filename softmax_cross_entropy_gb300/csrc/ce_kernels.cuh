// Kernel-side contract shared by the forward kernels and the host
// dispatcher: the argument block, the scratch layout, and the prologue /
// epilogue steps every forward variant runs.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ce_device.cuh"

namespace gbce {

enum : int { kRedNone = 0, kRedSum = 1, kRedMean = 2 };
enum : unsigned { kDevErrTarget = 1u, kDevErrTimeout = 2u };

// Per-cluster partial sums of the scalar outputs.
struct alignas(32) Partial {
    double loss;
    double zloss;
    long long n_correct;
    long long pad;
};

// Library-owned scratch: a self-resetting ticket for the last-CTA epilogue,
// a sticky error word, and one Partial per cluster.
struct Scratch {
    unsigned ticket;
    unsigned status;
    unsigned pad[62];
    Partial partials[1];  // really kMaxPartials
};
constexpr int kMaxPartials = 4096;
constexpr size_t kScratchBytes = sizeof(Scratch) + (kMaxPartials - 1) * sizeof(Partial);

struct FwdArgs {
    void* x;  // [rows, V] logits, overwritten with dlogits when grad != 0
    int64_t rows;
    int64_t V;
    const void* target;  // [rows] int32 or int64
    int tgt64;
    const float* weight;  // [V] or nullptr
    int64_t ignore_index;
    float eps;           // label smoothing
    float lam;           // lse_square_scale
    float softcap;       // s (> 0) when the kernel is the softcap variant
    float sc_k2;         // 2 * log2(e) / s
    float sc_slog2e;     // s * log2(e)
    int reduction;
    int grad, want_z, want_acc, want_pred;
    float* loss;
    float* zloss;
    float* acc;
    int64_t* pred;
    // layout of the staged kernel
    int slice_vec;  // 16-byte vectors of one row owned by one CTA
    int stages;     // depth of the shared-memory ring
    uint64_t timeout_ns;
    Scratch* scratch;
};

__device__ __forceinline__ int64_t load_target(const FwdArgs& a, int64_t r) {
    return a.tgt64 ? reinterpret_cast<const int64_t*>(a.target)[r]
                   : static_cast<int64_t>(reinterpret_cast<const int32_t*>(a.target)[r]);
}

// A row takes part in the loss when its target is neither ignore_index nor
// out of range (an out-of-range target is reported and treated as ignored).
__device__ __forceinline__ bool row_counts(const FwdArgs& a, int64_t t) {
    return t != a.ignore_index && t >= 0 && t < a.V;
}

// Block-wide fixed-order reduction helpers. `sh` must hold NT/32 entries
// and must not be reused until a later __syncthreads.
template <int NT>
__device__ __forceinline__ float block_sum_fixed(float v, float* sh) {
    constexpr int NW = NT / 32;
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) r += sh[w];
    return r;
}

// Prologue: the mean denominator D = sum of w[t_i] over counted rows, the
// counted-row number, and (for weighted label smoothing) W = sum_j w_j.
// Every CTA computes them in the same fixed order, so all CTAs hold
// bit-identical values without any inter-CTA communication.
template <int NT>
__device__ __forceinline__ void denominators(const FwdArgs& a, bool need_W, float* sh,
                                             float& D, int& n_valid, float& W) {
    float d = 0.f;
    int n = 0;
    for (int64_t i = threadIdx.x; i < a.rows; i += NT) {
        const int64_t t = load_target(a, i);
        if (row_counts(a, t)) {
            d += a.weight ? __ldg(a.weight + t) : 1.f;
            ++n;
        }
    }
    D = block_sum_fixed<NT>(d, sh);
    __syncthreads();
    {
        // integer count through the same fixed tree (exact)
        int v = n;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if ((threadIdx.x & 31) == 0) reinterpret_cast<int*>(sh)[threadIdx.x >> 5] = v;
        __syncthreads();
        int r = 0;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) r += reinterpret_cast<int*>(sh)[w];
        n_valid = r;
        __syncthreads();
    }
    if (!a.weight) D = static_cast<float>(n_valid);
    W = static_cast<float>(a.V);
    if (need_W) {
        float s = 0.f;
        for (int64_t j = threadIdx.x; j < a.V; j += NT) s += __ldg(a.weight + j);
        W = block_sum_fixed<NT>(s, sh);
        __syncthreads();
    }
}

// Per-row loss from the row's scalars:
//   (1-eps) w_t (lse - z_t) + (eps/V) (W lse - sum_j w_j z_j) + lam lse^2
__device__ __forceinline__ float row_loss(const FwdArgs& a, float lse, float zt, float wt,
                                          float W, float swz, float& zl) {
    zl = a.lam * lse * lse;
    const float ce = wt * (lse - zt);
    const float sm = (W * lse - swz) / static_cast<float>(a.V);
    return (1.f - a.eps) * ce + a.eps * sm + zl;
}

// Epilogue for "sum" and "mean": each participating CTA publishes its
// partials; the last one to arrive (atomic ticket) adds them in index order
// and writes the scalar outputs, then resets the ticket for the next call.
// Called by one thread per participating CTA.
__device__ __forceinline__ void finish_scalars(const FwdArgs& a, int64_t slot, int64_t nslots,
                                               double l, double z, long long nc, float D,
                                               int n_valid) {
    Scratch* s = a.scratch;
    s->partials[slot].loss = l;
    s->partials[slot].zloss = z;
    s->partials[slot].n_correct = nc;
    __threadfence();
    const unsigned prev = atomicAdd(&s->ticket, 1u);
    if (prev != static_cast<unsigned>(nslots - 1)) return;
    __threadfence();
    double L = 0.0, Z = 0.0;
    long long C = 0;
    for (int64_t c = 0; c < nslots; ++c) {
        const volatile Partial* p = &s->partials[c];
        L += p->loss;
        Z += p->zloss;
        C += p->n_correct;
    }
    if (a.reduction == kRedMean) {
        // no counted row: 0/0 = NaN, as the mean of an empty set
        L = L / static_cast<double>(D);
        Z = Z / static_cast<double>(D);
    }
    a.loss[0] = static_cast<float>(L);
    if (a.want_z) a.zloss[0] = static_cast<float>(Z);
    if (a.want_acc) a.acc[0] = static_cast<float>(static_cast<double>(C) / n_valid);
    s->ticket = 0u;
}

// ---------------------------------------------------------------- variants

// Staged-kernel shapes: threads per CTA and 16-byte vectors each thread
// keeps in registers. A CTA holds at most nt * nv vectors of one row.
struct StagedCfg {
    int nt;
    int nv;
};
constexpr int kNumStagedCfgs = 4;
constexpr StagedCfg kStagedCfgs[kNumStagedCfgs] = {{128, 4}, {256, 4}, {512, 4}, {512, 8}};
constexpr int kMaxStages = 8;
constexpr int kGenericThreads = 256;
constexpr int kBwdThreads = 256;

struct BwdArgs {
    const float* g;  // one value, or one per row
    int per_row;
    void* x;         // [rows, V]
    int64_t rows;
    int64_t V;
    int vec_ok;      // rows are 16-byte aligned and V * sizeof(T) % 16 == 0
};

// Kernel entry points by variant, for cudaLaunchKernelExC and the occupancy
// API (nullptr for an unknown variant). Forward kernels take one FwdArgs,
// the backward kernel one BwdArgs, both by value.
const void* staged_kernel_bf16_plain(int cfg_index, bool wsmooth);
const void* staged_kernel_bf16_softcap(int cfg_index, bool wsmooth);
const void* staged_kernel_f32_plain(int cfg_index, bool wsmooth);
const void* staged_kernel_f32_softcap(int cfg_index, bool wsmooth);
const void* generic_kernel(int dtype, bool softcap);
const void* bwd_kernel(int dtype);

}  // namespace gbce
