// Counts of one shard of a batch for the row-sharded "mean": D = the sum of
// w[t_i] over the rows that take part in the loss (w = 1 without class
// weights) and the number of those rows (Liger-Kernel cross-entropy profile,
// §Forward Pass: the mean reduction; tt-mlir pull request #9324 review
// comments: the mean divides by total_weight). A caller all-reduces the two
// numbers of every shard and passes the totals to ce_fwd_shard.
#include "ce_kernels.cuh"

namespace gbce {
namespace {

// Grid-stride over the rows; each CTA adds its rows in double, the CTAs'
// sums go through the scratch's partial slots and the last CTA (atomic
// ticket) adds them in slot order with a fixed lane split and butterfly; a
// launch of one CTA (up to kCountThreads * kCountPerThread rows) writes its
// sums directly.
__global__ void __launch_bounds__(kCountThreads) ce_count_kernel(const __grid_constant__ CountArgs a) {
    constexpr int NW = kCountThreads / 32;
    // a forward launched after this one may start now; it waits for these
    // counts where it first needs them
    pdl_launch_dependents();
    __shared__ double s_d[NW];
    __shared__ long long s_n[NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    double d = 0.0;
    long long n = 0;
    // kCountPerThread targets a thread, all loaded before any is used (one
    // memory round trip a block of them)
    constexpr int PT = kCountPerThread;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kCountThreads * PT;
#pragma unroll 1
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * kCountThreads * PT; base < a.rows;
         base += stride) {
        int64_t t[PT];
#pragma unroll
        for (int j = 0; j < PT; ++j) {
            const int64_t i = base + static_cast<int64_t>(j) * kCountThreads + tid;
            t[j] = i >= a.rows ? a.ignore_index
                   : a.tgt64   ? reinterpret_cast<const int64_t*>(a.target)[i]
                               : static_cast<int64_t>(reinterpret_cast<const int32_t*>(a.target)[i]);
        }
#pragma unroll
        for (int j = 0; j < PT; ++j) {
            if (t[j] != a.ignore_index && t[j] >= 0 && t[j] < a.V) {
                d += a.weight ? static_cast<double>(__ldg(a.weight + t[j])) : 1.0;
                ++n;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        d += __shfl_xor_sync(0xffffffffu, d, o);
        n += __shfl_xor_sync(0xffffffffu, n, o);
    }
    if (lane == 0) {
        s_d[warp] = d;
        s_n[warp] = n;
    }
    __syncthreads();
    if (warp != 0) return;
    if (gridDim.x == 1) {  // one CTA: its sums are the totals
        if (lane == 0) {
            double cd = 0.0;
            long long cn = 0;
            for (int w = 0; w < NW; ++w) {
                cd += s_d[w];
                cn += s_n[w];
            }
            a.counts[0] = cd;
            a.counts[1] = static_cast<double>(cn);
        }
        return;
    }
    Scratch* s = a.scratch;
    int last = 0;
    if (lane == 0) {
        double cd = 0.0;
        long long cn = 0;
        for (int w = 0; w < NW; ++w) {
            cd += s_d[w];
            cn += s_n[w];
        }
        s->partials[blockIdx.x].loss = cd;
        s->partials[blockIdx.x].n_correct = cn;
        __threadfence();
        last = atomicAdd(&s->ticket, 1u) == gridDim.x - 1;
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __threadfence();
    double D = 0.0;
    long long N = 0;
    for (unsigned c = lane; c < gridDim.x; c += 32) {
        D += __ldcg(&s->partials[c].loss);
        N += __ldcg(&s->partials[c].n_correct);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        D += __shfl_xor_sync(0xffffffffu, D, o);
        N += __shfl_xor_sync(0xffffffffu, N, o);
    }
    if (lane == 0) {
        a.counts[0] = D;
        a.counts[1] = static_cast<double>(N);
        s->ticket = 0u;
    }
}

}  // namespace

const void* count_kernel() { return reinterpret_cast<const void*>(&ce_count_kernel); }

}  // namespace gbce
