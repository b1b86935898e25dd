// Device primitives for the sm_103a cross-entropy kernels: mbarriers, bulk
// asynchronous copies (the TMA engine's 1-D form), thread-block-cluster
// barriers and distributed shared memory, bounded waits, and the few fast
// math steps the kernels use. Everything here is inline PTX or CUDA
// intrinsics; nothing is shared with the CPU oracle.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace gbce {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- addresses

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async proxy and to the
// other CTAs of the cluster.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Like mbar_try_wait, but the hardware may suspend the thread up to
// `suspend_ns` nanoseconds inside the instruction while the phase is still
// open, so a waiting warp sleeps instead of spinning.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t suspend_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(suspend_ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of `bar` with the given parity to complete, for at
// most timeout_ns nanoseconds of wall time. Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
#pragma unroll 1
    while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
    return true;
}

// ---------------------------------------------------------------- bulk copy

// L2 policy for data that is read once: evict it first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// L2 policy for data read twice in a row: keep it over other lines.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 16-byte global load with an L2 eviction-policy hint.
__device__ __forceinline__ uint4 ld_v4_hint(const void* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

// 16-byte global store with an L2 eviction-policy hint.
__device__ __forceinline__ void st_v4_hint(void* p, const uint4& v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

// Global -> shared bulk copy that signals `bar` with the bytes it delivers.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// ---------------------------------------------------------------- cluster

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t ncluster_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Cluster-wide barrier: every thread of every CTA of the cluster arrives
// (release) and waits (acquire). Orders shared-memory writes before it with
// distributed-shared-memory reads after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// ---------------------------------------------------------------- math

// 2^x on the special-function unit (flushes subnormal results to zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs: sm_100 and later issue one FFMA2 / FADD2 / FMUL2
// instruction for both lanes (CUDA's float2 builtins, which the compiler
// keeps in register pairs).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// tanh(y) from the identity tanh(y) = 1 - 2 / (exp(2y) + 1), with the
// argument already multiplied by 2*log2(e): tanh_from_2ylog2e(2*y*log2e).
// Absolute error about 1e-7; saturates to +-1 and keeps NaN.
__device__ __forceinline__ float tanh_from_scaled(float two_y_log2e) {
    const float u = ex2(two_y_log2e);
    return fmaf(-2.0f, rcp_approx(u + 1.0f), 1.0f);
}

// Softcap z = s tanh(x/s) through r = 1 / (1 + exp(2x/s)), for a pair of
// logits (k2 = 2 log2(e) / s). With it z = s (1 - 2r) and dz/dx =
// 1 - tanh^2 = 4 r (1 - r), so the exp2 argument (z - m) log2(e) is one FFMA
// of r, c1 r + c0 with c1 = -2 s log2(e) and c0 = (s - m) log2(e), and the
// gradient's factor is one FFMA, r - r^2, the 4 going into the gradient's
// constants. r = 0 for x = +inf, 1 for x = -inf; NaN stays NaN.
__device__ __forceinline__ float2 softcap_r2(float x0, float x1, float k2) {
    const float2 v = fmul2(make_float2(x0, x1), make_float2(k2, k2));
    const float2 u = fadd2(make_float2(ex2(v.x), ex2(v.y)), make_float2(1.f, 1.f));
    return make_float2(rcp_approx(u.x), rcp_approx(u.y));
}

// ---------------------------------------------------------------- storage

template <typename T>
struct Vec;  // one 16-byte vector of logits

template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    // Largest of the 8 values (packed bf16 max, then the two halves).
    __device__ __forceinline__ static float vmax(const uint4& v) {
        __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
        __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
        __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
        __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
        __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
        return fmaxf(__low2float(m), __high2float(m));
    }
    // Running maximum over whole vectors kept as a packed bf16 pair.
    using MaxAcc = __nv_bfloat162;
    __device__ __forceinline__ static MaxAcc max_init() {
        return __halves2bfloat162(__ushort_as_bfloat16(0xFF80u), __ushort_as_bfloat16(0xFF80u));
    }
    __device__ __forceinline__ static MaxAcc max_fold(MaxAcc acc, const uint4& v) {
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
        const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
        const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
        return __hmax2(__hmax2(acc, a), __hmax2(__hmax2(b, c), d));
    }
    __device__ __forceinline__ static float max_value(MaxAcc acc) {
        return fmaxf(__low2float(acc), __high2float(acc));
    }
    __device__ __forceinline__ static float load1(const void* p, int64_t i) {
        const uint16_t b = reinterpret_cast<const uint16_t*>(p)[i];
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
    __device__ __forceinline__ static void store1(void* p, int64_t i, float v) {
        reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
    }
};

template <>
struct Vec<__half> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
        }
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    __device__ __forceinline__ static float vmax(const uint4& v) {
        const __half2 a = *reinterpret_cast<const __half2*>(&v.x);
        const __half2 b = *reinterpret_cast<const __half2*>(&v.y);
        const __half2 c = *reinterpret_cast<const __half2*>(&v.z);
        const __half2 d = *reinterpret_cast<const __half2*>(&v.w);
        const __half2 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
        return fmaxf(__low2float(m), __high2float(m));
    }
    using MaxAcc = __half2;
    __device__ __forceinline__ static MaxAcc max_init() {
        return __halves2half2(__ushort_as_half(0xFC00u), __ushort_as_half(0xFC00u));
    }
    __device__ __forceinline__ static MaxAcc max_fold(MaxAcc acc, const uint4& v) {
        const __half2 a = *reinterpret_cast<const __half2*>(&v.x);
        const __half2 b = *reinterpret_cast<const __half2*>(&v.y);
        const __half2 c = *reinterpret_cast<const __half2*>(&v.z);
        const __half2 d = *reinterpret_cast<const __half2*>(&v.w);
        return __hmax2(__hmax2(acc, a), __hmax2(__hmax2(b, c), d));
    }
    __device__ __forceinline__ static float max_value(MaxAcc acc) {
        return fmaxf(__low2float(acc), __high2float(acc));
    }
    __device__ __forceinline__ static float load1(const void* p, int64_t i) {
        return __half2float(reinterpret_cast<const __half*>(p)[i]);
    }
    __device__ __forceinline__ static void store1(void* p, int64_t i, float v) {
        reinterpret_cast<__half*>(p)[i] = __float2half_rn(v);
    }
};

template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    __device__ __forceinline__ static float vmax(const uint4& v) {
        return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                     fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
    using MaxAcc = float;
    __device__ __forceinline__ static MaxAcc max_init() { return -INFINITY; }
    __device__ __forceinline__ static MaxAcc max_fold(MaxAcc acc, const uint4& v) {
        return fmaxf(fmaxf(acc, __uint_as_float(v.x)),
                     fmaxf(fmaxf(__uint_as_float(v.y), __uint_as_float(v.z)),
                           __uint_as_float(v.w)));
    }
    __device__ __forceinline__ static float max_value(MaxAcc acc) { return acc; }
    __device__ __forceinline__ static float load1(const void* p, int64_t i) {
        return reinterpret_cast<const float*>(p)[i];
    }
    __device__ __forceinline__ static void store1(void* p, int64_t i, float v) {
        reinterpret_cast<float*>(p)[i] = v;
    }
};

// ---------------------------------------------------------------- warp reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// (value, index) maximum: larger value wins, equal values keep the smaller
// index. Same result in every lane.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (ov > v || (ov == v && oi < i)) {
            v = ov;
            i = oi;
        }
    }
}

// Warp-wide maximum of a float and minimum of an int in one instruction
// each (redux.sync on sm_100-class GPUs); every lane gets the result. The
// whole warp must be converged at the call (__syncwarp() after a divergent
// branch).
__device__ __forceinline__ float warp_max_f32(float v) {
    float m;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(v));
    return m;
}

__device__ __forceinline__ int warp_min_s32(int v) {
    // the compiler's own intrinsic for redux.sync.min.s32, which it keeps
    // convergent (an asm statement may be duplicated into divergent paths)
    return __reduce_min_sync(0xffffffffu, v);
}

}  // namespace gbce
