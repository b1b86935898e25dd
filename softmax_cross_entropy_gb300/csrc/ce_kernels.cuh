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
// a sticky error word, the batch counts {D, counted rows} a count pre-pass
// leaves for the N-D forward, and one Partial per cluster.
struct Scratch {
    unsigned ticket;
    unsigned status;
    unsigned pad0[2];  // pad0[0]: abort flag of the tensor-core GEMM launch
    double counts[2];
    unsigned pad[56];
    Partial partials[1];  // really kMaxPartials
};
static_assert(sizeof(Partial) == 32, "partial-sum slot layout");
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
    // layout of the streaming kernel
    int ng;         // row groups per CTA
    int sg;         // ring slots per group
    int chunk_vec;  // 16-byte vectors per ring slot
    int nchunk;     // slots one row occupies
    int resident;   // 1: a row stays in its slots for both passes
    uint64_t timeout_ns;
    Scratch* scratch;
    void* out;  // log-softmax mode: [rows, V] output (may equal x)
    // fp32 logits, streaming kernel: the gradient goes to gout [rows, V] as
    // bf16 (gout_bf16 = 1) or fp16, rounded once, and the logits stay as
    // they were (the fused linear cross-entropy's G); nullptr: in place
    void* gout;
    int gout_bf16;
    // {D, n_valid} of the whole batch when this call is one shard of it
    // (the mean scale and the accuracy use them instead of this call's own
    // counts), or nullptr
    const double* batch_counts;
    // N-D layout [N, C, inner] (class dimension 1): rows = N * inner
    // positions, V = C classes; element (position r, class c) sits at
    // (r / inner) * C * inner + c * inner + r % inner
    int64_t inner;
    int nd_staged;  // 1: the N-D kernel keeps its tile in shared memory
    int reg_wpr;    // register-resident kernel: warps a row team has
    uint32_t reg_buf_stride;  // register-resident kernel: bytes of a team's row buffer
    int reg_nbuf;             // register-resident kernel: row buffers a team (1 or 2)
    int tm_slice_vec;         // tensor-memory kernel: 16-byte vectors of a CTA's slice of a row
    int tm_slots;             // tensor-memory kernel: ring slots
    int reg_cluster;  // register-resident kernel: CTAs of the cluster that owns a row (0, 1: one CTA)
    // test hook: CTA 0 does not issue its first bulk copy, so the wait for
    // it runs out (status CE_ERR_TIMEOUT, outputs invalid, nothing faults)
    int test_stall;
};

// Arguments of one forward call as the C ABI receives them (host side).
struct FwdCall {
    void* logits;
    int dtype;
    int64_t rows, V;
    const void* target;
    const float* weight;
    int64_t ignore_index;
    float label_smoothing, lse_square_scale, softcap;
    int reduction;
    uint32_t flags;
    float* loss;
    float* z_loss;
    float* acc;
    int64_t* pred;
    const double* batch_counts;
    void* gout = nullptr;  // FwdArgs::gout (internal callers only)
    int gout_dtype = 0;    // CE_BF16 or CE_F16 with gout
};

// Arguments of the unfused (aten-shaped) kernels.
struct NllFwdArgs {  // nll_loss_forward
    const void* logp;  // [rows, C]
    const void* target;
    int tgt64;
    const float* weight;  // [C] or nullptr
    int64_t rows, C, ignore_index;
    int reduction;
    float* out;           // [rows] ("none") or [1]
    float* total_weight;  // [1]
    Scratch* scratch;
};

struct NllBwdArgs {  // nll_loss_backward
    const float* grad_output;  // [rows] ("none") or [1]
    const float* total_weight;  // [1], read for "mean"
    void* grad_input;           // [rows, C], written
    const void* target;
    int tgt64;
    const float* weight;
    int64_t rows, C, ignore_index;
    int reduction;
    int vec_ok;  // 16-byte rows
    Scratch* scratch;
};

struct LsmBwdArgs {  // _log_softmax_backward_data
    const void* dy;  // [rows, C] incoming gradient
    const void* y;   // [rows, C] log-softmax output
    void* dx;        // [rows, C] (may equal dy)
    int64_t rows, C;
    int vec_ok;
};

struct LsmArgs {  // _log_softmax, general kernel (any alignment)
    const void* x;
    void* out;
    int64_t rows, C;
};

// Arguments of the shard-count kernel (ce_count).
struct CountArgs {
    const void* target;
    int tgt64;
    const float* weight;
    int64_t rows, V, ignore_index;
    double* counts;  // out: {sum of w[t] over counted rows, counted rows}
    Scratch* scratch;
};

// Programmatic dependent launch: a kernel that produces what the next
// launch on its stream needs lets that launch start early
// (pdl_launch_dependents), and the next launch waits for the producer's
// completion and memory (pdl_wait) only where it reads the result. Without
// the launch attribute on the dependent launch both are no-ops.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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

// Prologue: the mean denominator D = sum of w[t_i] over counted rows and the
// counted-row number. Every CTA computes them in the same fixed order, so
// all CTAs hold bit-identical values without inter-CTA communication.
struct CtaSync {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// Barrier over the first `n` threads of the CTA (named barrier `id`).
struct NamedSync {
    int id, n;
    __device__ __forceinline__ void operator()() const {
        asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
    }
};

template <int NT, typename Sync = CtaSync>
__device__ __forceinline__ void denominators(const FwdArgs& a, float* sh, float& D, int& n_valid,
                                             Sync sync = Sync()) {
    if (a.batch_counts) {  // one shard of a batch whose counts are given
        D = static_cast<float>(a.batch_counts[0]);
        n_valid = static_cast<int>(a.batch_counts[1]);
        return;
    }
    float d = 0.f;
    int n = 0;
#pragma unroll 8
    for (int64_t i = threadIdx.x; i < a.rows; i += NT) {
        const int64_t t = load_target(a, i);
        if (row_counts(a, t)) {
            d += a.weight ? __ldg(a.weight + t) : 1.f;
            ++n;
        }
    }
    d = warp_sum(d);
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = d;
    sync();
    float dd = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) dd += sh[w];
    D = dd;
    sync();
    int v = n;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) reinterpret_cast<int*>(sh)[threadIdx.x >> 5] = v;
    sync();
    int r = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) r += reinterpret_cast<int*>(sh)[w];
    n_valid = r;
    sync();
    if (!a.weight) D = static_cast<float>(n_valid);  // exact count
}

// Online softmax statistics of a set of elements of one row, relative to a
// reference m (the largest z of the set): S = sum exp(z - m),
// SZ = sum w (z - m), Wn = sum w (the element count without weights), and
// the first argmax (xmax, idx) of the raw logits. An empty set has
// m = -inf. Sets are merged with the usual rescaling.
struct RowStats {
    float m, S, SZ, Wn, xmax;
    int idx;
};

__device__ __forceinline__ RowStats empty_stats() {
    return RowStats{-INFINITY, 0.f, 0.f, 0.f, -INFINITY, 0x7fffffff};
}

// a <- a (+) b. The result does not depend on the order of a and b, bit
// for bit (every product and sum is rounded explicitly, per side), so the
// lanes of a butterfly reduction and the CTAs of a cluster agree exactly.
__device__ __forceinline__ void stats_merge(RowStats& a, const RowStats& b) {
    if (b.xmax > a.xmax || (b.xmax == a.xmax && b.idx < a.idx)) {
        a.xmax = b.xmax;
        a.idx = b.idx;
    }
    if (b.m == -INFINITY) return;
    if (a.m == -INFINITY) {
        a.m = b.m;
        a.S = b.S;
        a.SZ = b.SZ;
        a.Wn = b.Wn;
        return;
    }
    const float M = fmaxf(a.m, b.m);
    const float da = __fsub_rn(a.m, M);
    const float db = __fsub_rn(b.m, M);
    a.S = __fadd_rn(__fmul_rn(a.S, ex2(__fmul_rn(da, kLog2e))),
                    __fmul_rn(b.S, ex2(__fmul_rn(db, kLog2e))));
    a.SZ = __fadd_rn(__fmaf_rn(a.Wn, da, a.SZ), __fmaf_rn(b.Wn, db, b.SZ));
    a.Wn = __fadd_rn(a.Wn, b.Wn);
    a.m = M;
}

__device__ __forceinline__ RowStats shfl_xor_stats(const RowStats& v, int o) {
    RowStats r;
    r.m = __shfl_xor_sync(0xffffffffu, v.m, o);
    r.S = __shfl_xor_sync(0xffffffffu, v.S, o);
    r.SZ = __shfl_xor_sync(0xffffffffu, v.SZ, o);
    r.Wn = __shfl_xor_sync(0xffffffffu, v.Wn, o);
    r.xmax = __shfl_xor_sync(0xffffffffu, v.xmax, o);
    r.idx = __shfl_xor_sync(0xffffffffu, v.idx, o);
    return r;
}

// Butterfly all-reduce over the low `width` lanes groups (width a power of
// two); every lane ends with the same bits.
template <int WIDTH>
__device__ __forceinline__ void warp_stats_allreduce(RowStats& v) {
#pragma unroll
    for (int o = WIDTH / 2; o > 0; o >>= 1) {
        const RowStats b = shfl_xor_stats(v, o);
        stats_merge(v, b);
    }
}

// Per-row loss from the row's merged statistics (M = max z, S = sum
// exp(z - M), SZ = sum w (z - M), W = sum w):
//   (1-eps) w_t (lse - z_t) + (eps/V) sum_j w_j (lse - z_j) + lam lse^2
// with lse - z_t = (M - z_t) + log S and
// sum_j w_j (lse - z_j) = W log S - SZ, which keeps every difference small.
__device__ __forceinline__ float row_loss(const FwdArgs& a, float M, float logS, float zt,
                                          float wt, float W, float SZ, float& zl) {
    const float lse = M + logS;
    zl = a.lam * lse * lse;
    const float ce = wt * ((M - zt) + logS);
    const float sm = (W * logS - SZ) / static_cast<float>(a.V);
    return (1.f - a.eps) * ce + a.eps * sm + zl;
}

// Epilogue for "sum" and "mean" for launches of a few hundred CTAs at most
// (it keeps the hot loop's register allocation of the streaming and staged
// kernels free of spills, which the two-level form below does not): each
// participating CTA publishes its
// partials; the last one to arrive (atomic ticket) adds them and writes the
// scalar outputs, then resets the ticket for the next call. Called by all 32
// lanes of one warp of each participating CTA; lane 0 holds the CTA's
// partials. In the last CTA, lane k adds the slots k, k + 32, ... in order
// and a fixed butterfly combines the lanes, so the result does not depend on
// which CTA finishes last (one dependent L2 read per slot in a single thread
// would cost tens of microseconds at a thousand slots).
__device__ __forceinline__ void finish_scalars(const FwdArgs& a, int64_t slot, int64_t nslots,
                                               double l, double z, long long nc, float D,
                                               int n_valid) {
    Scratch* s = a.scratch;
    const int lane = threadIdx.x & 31;
    int last = 0;
    if (lane == 0) {
        s->partials[slot].loss = l;
        s->partials[slot].zloss = z;
        s->partials[slot].n_correct = nc;
        __threadfence();
        last = atomicAdd(&s->ticket, 1u) == static_cast<unsigned>(nslots - 1);
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __threadfence();
    double L = 0.0, Z = 0.0;
    long long C = 0;
    for (int64_t c = lane; c < nslots; c += 32) {
        L += __ldcg(&s->partials[c].loss);
        Z += __ldcg(&s->partials[c].zloss);
        C += __ldcg(&s->partials[c].n_correct);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        L += __shfl_xor_sync(0xffffffffu, L, o);
        Z += __shfl_xor_sync(0xffffffffu, Z, o);
        C += __shfl_xor_sync(0xffffffffu, C, o);
    }
    if (lane != 0) return;
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

// Epilogue for "sum" and "mean" for launches of many CTAs, called by every
// thread of every CTA (thread 0 holding the CTA's partials; `flag` a shared
// int). Thread 0 publishes the partials to the CTA's slot and takes a ticket
// with a release atomic; in the last CTA to arrive, thread t adds slots t,
// t + nt, ... in order and a fixed warp butterfly and warp order combine the
// threads, so the result does not depend on which CTA finishes last, and no
// thread adds more than a few slots one after another.
__device__ __forceinline__ void finish_scalars_cta(const FwdArgs& a, double l, double z,
                                                   long long nc, float D, int n_valid,
                                                   int* flag, double* red_l, double* red_z,
                                                   long long* red_c) {
    Scratch* s = a.scratch;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nw = static_cast<int>(blockDim.x >> 5);
    if (tid == 0) {
        Partial* p = &s->partials[blockIdx.x];
        p->loss = l;
        p->zloss = z;
        p->n_correct = nc;
        unsigned t;
        // release: the slot is visible before the ticket moves; acquire: the
        // last CTA sees every slot
        asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;"
                     : "=r"(t)
                     : "l"(&s->ticket)
                     : "memory");
        *flag = t == gridDim.x - 1;
    }
    __syncthreads();
    if (!*flag) return;
    double L = 0.0, Z = 0.0;
    long long C = 0;
    for (unsigned c = tid; c < gridDim.x; c += blockDim.x) {
        L += __ldcg(&s->partials[c].loss);
        Z += __ldcg(&s->partials[c].zloss);
        C += __ldcg(&s->partials[c].n_correct);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        L += __shfl_xor_sync(0xffffffffu, L, o);
        Z += __shfl_xor_sync(0xffffffffu, Z, o);
        C += __shfl_xor_sync(0xffffffffu, C, o);
    }
    if (lane == 0) {
        red_l[warp] = L;
        red_z[warp] = Z;
        red_c[warp] = C;
    }
    __syncthreads();
    if (tid != 0) return;
    L = 0.0;
    Z = 0.0;
    C = 0;
    for (int w = 0; w < nw; ++w) {
        L += red_l[w];
        Z += red_z[w];
        C += red_c[w];
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

// Partial-sum records a launch of `units` CTAs (or clusters) needs in the
// scratch: one per CTA (or cluster).
__host__ __device__ constexpr int64_t records_for(int64_t units) { return units; }
// The most CTAs (or clusters) a launch with the library scratch may have.
constexpr int64_t kMaxUnits = kMaxPartials;

// Adds two doubles over the CTAs of a grid in a fixed order (as
// finish_scalars does): called by the 32 lanes of one warp of every CTA,
// lane 0 holding its CTA's (u, v). Returns true in lane 0 of the last CTA
// to arrive, with the grid's totals in u and v, and resets the ticket.
__device__ __forceinline__ bool grid_sum2(Scratch* s, double& u, double& v) {
    const int lane = threadIdx.x & 31;
    int last = 0;
    if (lane == 0) {
        s->partials[blockIdx.x].loss = u;
        s->partials[blockIdx.x].zloss = v;
        __threadfence();
        last = atomicAdd(&s->ticket, 1u) == gridDim.x - 1;
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) return false;
    __threadfence();
    double U = 0.0, W = 0.0;
    for (unsigned c = lane; c < gridDim.x; c += 32) {
        U += __ldcg(&s->partials[c].loss);
        W += __ldcg(&s->partials[c].zloss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        U += __shfl_xor_sync(0xffffffffu, U, o);
        W += __shfl_xor_sync(0xffffffffu, W, o);
    }
    if (lane != 0) return false;
    u = U;
    v = W;
    s->ticket = 0u;
    return true;
}

// ---------------------------------------------------------------- variants

// Staged-kernel shapes: threads per CTA and 16-byte vectors each thread
// keeps in registers. A CTA holds at most nt * nv vectors of one row; with
// at most 128 registers a thread, 512 / nt CTAs fit on an SM by registers.
struct StagedCfg {
    int nt;
    int nv;
};
constexpr int kNumStagedCfgs = 6;
constexpr StagedCfg kStagedCfgs[kNumStagedCfgs] = {{128, 4}, {128, 8}, {256, 4},
                                                   {256, 8}, {512, 4}, {512, 8}};
constexpr int kMaxCluster = 16;
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
const void* staged_kernel_bf16_nocap_plain(int cfg);
const void* staged_kernel_bf16_nocap_wsmooth(int cfg);
const void* staged_kernel_bf16_softcap_plain(int cfg);
const void* staged_kernel_bf16_softcap_wsmooth(int cfg);
const void* staged_kernel_f32_nocap_plain(int cfg);
const void* staged_kernel_f32_nocap_wsmooth(int cfg);
const void* staged_kernel_f32_softcap_plain(int cfg);
const void* staged_kernel_f32_softcap_wsmooth(int cfg);
const void* stream_kernel(int dtype, bool softcap, int vpt, int nw);
const void* stream_kernel_f16(bool softcap, int vpt, int nw);
// fp32 logits, gradient to FwdArgs::gout (16-bit), the same shapes
const void* stream_kernel_gout(bool softcap, int vpt, int nw);
// class weights with label smoothing: 8 consumer warps, 8 vectors a thread
const void* stream_kernel_ws(int dtype, bool softcap);
constexpr int kStreamMaxSlots = 48;   // ring slots (all groups) of the streaming kernel
constexpr int kStreamMaxGroups = 8;
const void* generic_kernel(int dtype, bool softcap);
// register-resident kernel for rows of at most 64 KB: a team of WPR warps
// owns a row, nvl (8 or 16) 16-byte vectors a thread; a CTA has one or more
// teams, at most kRegMaxWarps warps
const void* reg_kernel(int dtype, bool softcap, bool ws, int nvl);
// Its class-weighted smoothing variant with the weights in shared memory:
// 16 warps a CTA, 8 vectors a thread.
const void* reg_kernel_sw(int dtype, bool softcap);
// The softcap kernel that keeps tanh's intermediate in tensor memory
// (ce_fwd_tmem.cuh): kTmWarps consumer warps and a producer warp, one CTA
// an SM with all of the SM's TMEM (kTmCols columns), clusters of up to
// kTmMaxCluster CTAs a row.
const void* tmem_kernel(int dtype);
constexpr int kTmWarps = 16;
constexpr int kTmCols = 32 * kTmWarps;  // TMEM columns a CTA allocates
constexpr int kTmVecPerThread = 4;  // 16-byte vectors a consumer thread takes from a slot
constexpr int kTmMaxSlots = 8;
constexpr int kTmMaxCluster = 8;
constexpr int kRegSwWarps = 16;
// The register-resident kernel's cluster variant (16 vectors a thread).
const void* reg_cluster_kernel(int dtype, bool softcap, bool ws);
constexpr int kRegMaxWarps = 8;
const void* count_kernel();
// unfused kernels (dtype 0 fp32, 1 bf16, 2 fp16)
const void* stream_kernel_lsm(int dtype);
const void* lsm_generic_kernel(int dtype);
const void* nll_fwd_kernel(int dtype);
const void* nll_bwd_kernel(int dtype);
const void* lsm_bwd_kernel(int dtype);
constexpr int kLsmGenericThreads = 512;
constexpr int kNllThreads = 256;
constexpr int kLsmBwdThreads = 1024;
constexpr int kCountThreads = 256;
constexpr int kCountPerThread = 16;  // targets a count thread loads at once
const void* bwd_kernel(int dtype);

// N-D logits [N, C, inner] (class dimension 1). The forward kernel takes one
// FwdArgs (rows = N * inner, V = C, inner, nd_staged); vec selects 16-byte
// loads of consecutive positions (inner a multiple of 16 / sizeof(T), base
// 16-byte aligned), argmax the first-argmax tracking (predicted tokens,
// accuracy).
constexpr int kNdThreads = 256;
constexpr int kNdWarps = kNdThreads / 32;
// shared memory of an N-D CTA besides its tile: per-warp partials and
// per-position coefficients for `positions` positions
constexpr size_t nd_fixed_smem(int positions) {
    return static_cast<size_t>(2 * kNdWarps + 6) * positions * 4;
}
const void* nd_kernel(int dtype, bool vec, bool softcap, bool argmax);

// The split N-D forward (ce_fwd_nd_split.cuh): the classes of each tile of
// 32 * VP positions in chunks of cc that separate CTAs take. One record
// per (position, chunk): the chunk's statistics of the position.
struct NdRec {
    float m, S, SZ, Wn, xmax;
    int idx;
};
// The gradient's coefficients of one position (merge -> gradient):
// g = (ac exp(z - shift) + bc w_c) dz/dx, and gt, the whole gradient at the
// target class (the one-hot term included).
struct NdCoef {
    float shift, ac, bc, gt;
};
struct NdSplitArgs {
    FwdArgs f;        // rows = N * inner, V = C, inner
    int64_t tiles;    // ceil(rows / (32 VP))
    int nch;          // class chunks a tile
    int cc;           // classes a chunk (the last one may hold fewer)
    NdRec* rec;       // [tiles * 32 VP][nch]
    NdCoef* coef;     // [rows]
    int* tpos;        // [rows]: the counted target, or -1
};
constexpr int kNdSplitThreads = 256;
struct NdSplitFns {
    const void* stats;  // per (tile, chunk): the records
    const void* merge;  // per position: outputs, coefficients, reduced scalars
    const void* grad;   // per (tile, chunk): the gradient in place
    size_t stats_smem;  // dynamic shared memory of a stats CTA
};
NdSplitFns nd_split_fns(int dtype, bool vec, bool softcap, bool argmax, bool smooth);
// A warp a tile of 32 vectors of positions and all C <= kNdWarpClasses
// classes (ce_fwd_nd_split.cuh): FwdArgs as the N-D kernel, 256 threads,
// dynamic shared memory 8 * C * 512 bytes.
constexpr int kNdWarpClasses = 48;
const void* nd_warp_kernel(int dtype, bool softcap, bool argmax);

struct NdBwdArgs {
    const float* g;  // one value, or one per position ([N, inner])
    int per_pos;
    void* x;         // [N, C, inner]
    int64_t N, C, inner;
    int vec_ok;      // inner * sizeof(T) % 16 == 0 and x 16-byte aligned
};
const void* nd_bwd_kernel(int dtype);

}  // namespace gbce
