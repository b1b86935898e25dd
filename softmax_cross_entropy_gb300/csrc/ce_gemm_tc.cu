// C[M, N] (fp32, row-major) = A[M, K] @ B[N, K]^T (+ bias[N]), A and B bf16
// or fp16, row-major (K contiguous): the logits GEMM of the fused linear
// cross-entropy (hidden @ lm_weight^T), on the fifth-generation tensor
// cores.
//
// One CTA of 4 warps computes a 128 x 256 tile of C:
//  * lane 0 of warp 0 streams 128 x 64 tiles of A and 256 x 64 tiles of B
//    into a 4-stage shared-memory ring with 2-D TMA copies (128-byte
//    swizzle, the layout the tensor core reads), signalling `full`
//    mbarriers;
//  * lane 0 of warp 1 issues tcgen05.mma (M = 128, N = 256, K = 16, fp32
//    accumulation) into a 256-column accumulator in tensor memory, four per
//    stage, and frees each stage with tcgen05.commit on its `empty`
//    mbarrier; a last commit signals `done`;
//  * all four warps then read the accumulator with tcgen05.ld (warp w owns
//    rows 32 w .. 32 w + 31 of the tile), add the bias and store fp32 rows.
// CTAs run along M first, so the CTAs that share a 256-row slice of B
// (the vocabulary) run together and read it from L2. Every mbarrier wait
// is bounded; a wait that gives up records the timeout in the status word,
// the kernel waits (bounded) for its copies in flight, frees its tensor
// memory and returns.
#include <cuda.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>
#include <string>

#include "ce_kernels.cuh"
#include "gbce.h"

namespace gbce {
ce_status record_cuda_failure(cudaError_t e, const char* what);
void record_message(const std::string& msg);
ce_status library_status_word(cudaStream_t st, unsigned** out);

namespace {

// 4 stages of 128 x 64 + 256 x 64 tiles (192 KB, one CTA an SM): measured
// best of 2 / 3 / 4 / 6 stages and 128- / 256-wide tiles on GB300
constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kTcThreads = 128;
constexpr uint32_t kABytes = kBM * kBK * 2;
constexpr uint32_t kBBytes = kBN * kBK * 2;
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kTmemCols = kBN;
constexpr size_t kTcSmem = static_cast<size_t>(kStages) * kStageBytes + 1024;

struct TcArgs {
    float* C;
    const float* bias;
    int64_t M, N, K;
    uint64_t timeout_ns;
    unsigned* status;  // sticky error word of the scratch (ce_device_status)
    unsigned* abort;   // cleared before the launch; set when a CTA gives up
};

// Shared-memory matrix descriptor of a K-major operand tile stored as
// 128-byte rows with the 128-byte swizzle (8-row atoms of 1024 bytes):
// start address, leading offset (unused for this layout: 1), stride
// between 8-row atoms 1024 bytes, descriptor version 1, swizzle mode 2.
__device__ __forceinline__ uint64_t tc_smem_desc(uint32_t saddr) {
    uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B of the
// given type (0 fp16, 1 bf16), both K-major, N = kBN, M = kBM.
__host__ __device__ constexpr uint32_t tc_idesc(uint32_t ab) {
    return (1u << 4) | (ab << 7) | (ab << 10) | (static_cast<uint32_t>(kBN >> 3) << 17) |
           (static_cast<uint32_t>(kBM >> 4) << 24);
}

// Bounded wait for the producer and MMA threads of the tight GEMM pipeline:
// poll without a suspend hint (a suspended thread may wake late), reading
// the global timer only every 1024 polls.
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
#pragma unroll 1
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 1023u) == 0 && global_timer_ns() - t0 > timeout_ns) return false;
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on `bar` once every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's accumulator row.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

template <uint32_t AB>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_gemm_abt(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
            const __grid_constant__ TcArgs a) {
    extern __shared__ unsigned char tc_smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ __align__(8) uint64_t empty_bar[kStages];
    __shared__ __align__(8) uint64_t done_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ uint32_t s_issued[kStages];  // 0, or 2 + parity of the last copy into the stage
    __shared__ int s_fail;

    // a CTA of this launch already gave up: the others return at once
    // (before any tensor memory is taken)
    if (*reinterpret_cast<volatile unsigned*>(a.abort)) return;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t smem0 = (smem_u32(tc_smem_raw) + 1023u) & ~1023u;  // 1024-byte aligned
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kBM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.y) * kBN;
    const int nk = static_cast<int>((a.K + kBK - 1) / kBK);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
            s_issued[s] = 0;
        }
        mbar_init(smem_u32(&done_bar), 1);
        s_fail = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                smem_u32(&tmem_base_sh)),
            "r"(kTmemCols)
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % kStages;
            const uint32_t ph = static_cast<uint32_t>(kb / kStages) & 1u;
            if (!tc_wait(smem_u32(&empty_bar[s]), ph ^ 1u, a.timeout_ns)) {
                s_fail = 1;
                break;
            }
            const uint32_t fb = smem_u32(&full_bar[s]);
            mbar_arrive_expect_tx(fb, kStageBytes);
            const uint32_t sa = smem0 + static_cast<uint32_t>(s) * kStageBytes;
            tma_load_2d(sa, &mapA, kb * kBK, static_cast<int>(m0), fb);
            tma_load_2d(sa + kABytes, &mapB, kb * kBK, static_cast<int>(n0), fb);
            s_issued[s] = 2u + ph;
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        constexpr uint32_t idesc = tc_idesc(AB);
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % kStages;
            const uint32_t ph = static_cast<uint32_t>(kb / kStages) & 1u;
            if (!tc_wait(smem_u32(&full_bar[s]), ph, a.timeout_ns)) {
                s_fail = 1;
                break;
            }
            tc_fence_after();
            const uint32_t sa = smem0 + static_cast<uint32_t>(s) * kStageBytes;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
                // K step of 16 elements = 32 bytes inside the swizzled 128-byte rows
                tc_mma(tmem, tc_smem_desc(sa + 32u * k), tc_smem_desc(sa + kABytes + 32u * k),
                       idesc, (kb > 0 || k > 0) ? 1u : 0u);
            }
            tc_commit(smem_u32(&empty_bar[s]));
        }
        tc_commit(smem_u32(&done_bar));  // every MMA issued above, also after a failure
    }
    __syncwarp();

    // ---- epilogue: accumulator rows -> fp32 C (+ bias)
    bool ok = mbar_wait_bounded(smem_u32(&done_bar), 0u, a.timeout_ns);
    tc_fence_after();
    __syncthreads();  // s_fail is final
    ok = ok && !s_fail;
    if (ok && nk > 0) {
        const int64_t row = m0 + warp * 32 + lane;
        const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        float* crow = a.C + row * a.N;
        const bool vec = (a.N & 3) == 0;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
            const int64_t n = n0 + c * 32;
            if (n >= a.N) break;  // the same for every thread of the CTA
            float v[32];
            tc_ld32(trow + static_cast<uint32_t>(c * 32), v);
            if (row < a.M) {
                if (a.bias) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (n + i < a.N) v[i] += __ldg(a.bias + n + i);
                }
                if (vec && n + 32 <= a.N) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4*>(crow + n + i) =
                            make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (n + i < a.N) crow[n + i] = v[i];
                }
            }
        }
    }
    if (!ok && threadIdx.x == 0) {
        atomicOr(a.status, kDevErrTimeout);
        atomicExch(a.abort, 1u);
        // copies still in flight land before the shared memory is released
        for (int s = 0; s < kStages; ++s)
            if (s_issued[s])
                (void)mbar_wait_bounded(smem_u32(&full_bar[s]), s_issued[s] & 1u, a.timeout_ns);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_tc_mu;
EncodeTiled g_encode = nullptr;

ce_status encoder(EncodeTiled* out) {
    std::lock_guard<std::mutex> lock(g_tc_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e =
            cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
            record_message("cuTensorMapEncodeTiled is not available");
            return CE_ERR_UNSUPPORTED;
        }
        g_encode = reinterpret_cast<EncodeTiled>(fn);
    }
    *out = g_encode;
    return CE_OK;
}

// 2-D map of a row-major [rows, K] matrix of 16-bit elements, boxes of
// box_rows x 64 elements, 128-byte swizzle, zeros outside the matrix.
ce_status make_map(CUtensorMap* map, const void* p, int dtype, int64_t rows, int64_t K,
                   uint32_t box_rows) {
    EncodeTiled enc = nullptr;
    ce_status rc = encoder(&enc);
    if (rc != CE_OK) return rc;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map,
                           dtype == CE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                           2, const_cast<void*>(p), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        record_message("cuTensorMapEncodeTiled failed (" + std::to_string(static_cast<int>(r)) + ")");
        return CE_ERR_UNSUPPORTED;
    }
    return CE_OK;
}

}  // namespace

// Whether the tensor-core GEMM takes these operands: 16-bit types, 16-byte
// aligned bases and K a multiple of 8 (16-byte row strides for the TMA).
bool tc_gemm_supported(const void* A, const void* B, int dtype, int64_t K) {
    return (dtype == CE_BF16 || dtype == CE_F16) && K % 8 == 0 && K > 0 &&
           (reinterpret_cast<uintptr_t>(A) & 15u) == 0 && (reinterpret_cast<uintptr_t>(B) & 15u) == 0;
}

// C = A @ B^T (+ bias) on `st`; status receives timeouts (device word),
// abort is a device word this launch may use (cleared here first).
ce_status tc_gemm_abt_launch(const void* A, const void* B, int dtype, int64_t M, int64_t N,
                             int64_t K, float* C, const float* bias, unsigned* status,
                             unsigned* abort, cudaStream_t st) {
    if (M <= 0 || N <= 0) return CE_OK;
    if (!tc_gemm_supported(A, B, dtype, K)) return CE_ERR_UNSUPPORTED;
    if (M > INT32_MAX || N > INT32_MAX) return CE_ERR_UNSUPPORTED;
    CUtensorMap ma, mb;
    ce_status rc = make_map(&ma, A, dtype, M, K, kBM);
    if (rc != CE_OK) return rc;
    rc = make_map(&mb, B, dtype, N, K, kBN);
    if (rc != CE_OK) return rc;
    const void* fn = dtype == CE_BF16 ? reinterpret_cast<const void*>(&tc_gemm_abt<1u>)
                                      : reinterpret_cast<const void*>(&tc_gemm_abt<0u>);
    static std::once_flag attr_once[2];
    cudaError_t e = cudaSuccess;
    std::call_once(attr_once[dtype == CE_BF16 ? 1 : 0], [&]() {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kTcSmem));
    });
    if (e != cudaSuccess) return record_cuda_failure(e, "cudaFuncSetAttribute(tensor-core GEMM)");
    const char* tenv = std::getenv("GBCE_WAIT_TIMEOUT_MS");
    const uint64_t tms = (tenv && *tenv) ? static_cast<uint64_t>(std::atoll(tenv)) : 2000ull;
    e = cudaMemsetAsync(abort, 0, sizeof(unsigned), st);
    if (e != cudaSuccess) return record_cuda_failure(e, "cudaMemsetAsync(abort word)");
    TcArgs a{C, bias, M, N, K, tms * 1000000ull, status, abort};
    const dim3 grid(static_cast<unsigned>((M + kBM - 1) / kBM),
                    static_cast<unsigned>((N + kBN - 1) / kBN));
    void* args[] = {&ma, &mb, &a};
    e = cudaLaunchKernel(fn, grid, dim3(kTcThreads), args, kTcSmem, st);
    if (e != cudaSuccess) return record_cuda_failure(e, "tensor-core GEMM launch");
    return CE_OK;
}

}  // namespace gbce

using namespace gbce;

// The GEMM alone, through the C ABI (see include/gbce.h).
extern "C" ce_status ce_gemm_abt(const void* A, const void* B, int dtype, int64_t M, int64_t N,
                                 int64_t K, float* C, const float* bias, ce_stream_t stream) {
    if (dtype != CE_BF16 && dtype != CE_F16) return CE_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K <= 0) return CE_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return CE_OK;
    if (!A || !B || !C) return CE_ERR_INVALID_ARG;
    if (!tc_gemm_supported(A, B, dtype, K)) return CE_ERR_UNSUPPORTED;
    unsigned* status = nullptr;
    ce_status rc = library_status_word(reinterpret_cast<cudaStream_t>(stream), &status);
    if (rc != CE_OK) return rc;
    // the scratch header's spare word after the status word serves as the
    // launch's abort flag
    return tc_gemm_abt_launch(A, B, dtype, M, N, K, C, bias, status, status + 1,
                              reinterpret_cast<cudaStream_t>(stream));
}
