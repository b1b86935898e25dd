// Fused linear cross-entropy: the cross-entropy of the logits
// hidden @ lm_weight^T (+ bias), with the gradients of hidden, lm_weight and
// bias, computed over chunks of rows so that only one chunk of logits
// exists at a time ("Kernel Profile: CrossEntropy", closest_existing_kernel:
// fused_linear_cross_entropy, this kernel with the linear layer fused in).
//
// Per chunk of c rows, on the caller's stream:
//   1. logits [c, V] fp32 = hidden_c @ W^T (+ bias): this library's
//      tcgen05 GEMM (ce_gemm_tc.cu; inputs in the storage type, fp32
//      accumulation in tensor memory);
//   2. the fused forward of this library over the chunk, as one shard of
//      the batch (the batch's D and counted rows from ce_count), writing
//      the gradient of the batch's reduced loss in place over the logits;
//   3. G = that gradient rounded to the storage type;
//   4. grad_hidden_c = G @ W (the same GEMM kernel with W read MN-major,
//      rounded to the storage type), grad_weight (+)= G^T @ hidden_c (both
//      operands MN-major, fp32 written then added to), and grad_bias (+)=
//      the column sums of the fp32 gradient (a column-per-thread kernel).
// fp32 inputs, and 16-bit ones whose rows are not multiples of 8 elements
// (16-byte rows for the TMA), take cuBLAS for the three GEMMs instead
// (GBCE_FLCE_GEMM=cublas forces it for every input).
// The chunks' scalar outputs are added in chunk order at the end, so the
// results are deterministic.
#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>

#include <cublas_v2.h>

#include "ce_kernels.cuh"
#include "gbce.h"

namespace gbce {
ce_status record_cuda_failure(cudaError_t e, const char* what);
void record_message(const std::string& msg);
ce_status library_status_word(cudaStream_t st, unsigned** out);
bool tc_gemm_supported(const void* A, const void* B, int dtype, int64_t K);
ce_status tc_gemm_abt_launch(const void* A, const void* B, int dtype, int64_t M, int64_t N,
                             int64_t K, float* C, const float* bias, unsigned* status,
                             unsigned* abort, cudaStream_t st);
ce_status tc_gemm_launch(const void* A, bool a_mn, const void* B, bool b_mn, int dtype, int64_t M,
                         int64_t N, int64_t K, void* C, int out, const float* bias,
                         unsigned* status, unsigned* abort, cudaStream_t st);
bool tc_operand_ok(const void* p, int dtype, int64_t row_elems);
ce_status fwd_shard_gout(const FwdCall& c, void* gout, int gout_dtype, ce_stream_t stream);

namespace {

constexpr int kFlceThreads = 256;

// logits[r, v] = bias[v] for every row of the chunk (before the GEMM adds
// hidden @ W^T with beta = 1).
__global__ void __launch_bounds__(kFlceThreads)
flce_bias_rows(float* logits, const float* bias, int64_t rows, int64_t V) {
    const int64_t n = rows * V;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kFlceThreads + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * kFlceThreads)
        logits[i] = __ldg(bias + i % V);
}

// out = in rounded to nearest-even into T (the gradient in the storage type).
template <typename T>
__global__ void __launch_bounds__(kFlceThreads)
flce_round(const float* in, T* out, int64_t n) {
    using VT = Vec<T>;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kFlceThreads;
    const int64_t nv = n / 8;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kFlceThreads + threadIdx.x; i < nv;
         i += stride) {
        const float4 a = reinterpret_cast<const float4*>(in)[2 * i];
        const float4 b = reinterpret_cast<const float4*>(in)[2 * i + 1];
        const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        reinterpret_cast<uint4*>(out)[i] = VT::pack(f);
    }
    for (int64_t i = nv * 8 + static_cast<int64_t>(blockIdx.x) * kFlceThreads + threadIdx.x;
         i < n; i += stride)
        VT::store1(out, i, in[i]);
}

// grad_bias[v] (+)= sum over the chunk's rows of g[r, v]: a thread a column
// (consecutive threads, consecutive columns), the rows added in order.
__global__ void __launch_bounds__(kFlceThreads)
flce_colsum(const float* g, float* out, int64_t rows, int64_t V, int accumulate) {
    for (int64_t v = static_cast<int64_t>(blockIdx.x) * kFlceThreads + threadIdx.x; v < V;
         v += static_cast<int64_t>(gridDim.x) * kFlceThreads) {
        float s = accumulate ? out[v] : 0.f;
        for (int64_t r = 0; r < rows; ++r) s += g[r * V + v];
        out[v] = s;
    }
}

// out = in * g rounded into T, g one fp32 value read on the device.
template <typename T>
__global__ void __launch_bounds__(kFlceThreads)
flce_scale_round(const float* in, const float* g, T* out, int64_t n) {
    const float s = __ldg(g);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kFlceThreads + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * kFlceThreads)
        Vec<T>::store1(out, i, in[i] * s);
}

// The scalar outputs: the chunks' shares added in chunk order.
__global__ void flce_sum_chunks(const float* parts, int nchunks, float* loss, float* zloss,
                                float* acc) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    double l = 0.0, z = 0.0, c = 0.0;
    for (int k = 0; k < nchunks; ++k) {
        l += parts[3 * k];
        z += parts[3 * k + 1];
        c += parts[3 * k + 2];
    }
    loss[0] = static_cast<float>(l);
    if (zloss) zloss[0] = static_cast<float>(z);
    if (acc) acc[0] = static_cast<float>(c);
}

std::mutex g_blas_mu;
std::map<int, cublasHandle_t> g_blas;

ce_status blas_for(int dev, cublasHandle_t* out) {
    std::lock_guard<std::mutex> lock(g_blas_mu);
    auto it = g_blas.find(dev);
    if (it != g_blas.end()) {
        *out = it->second;
        return CE_OK;
    }
    cublasHandle_t h = nullptr;
    const cublasStatus_t s = cublasCreate(&h);
    if (s != CUBLAS_STATUS_SUCCESS) {
        record_message(std::string("cublasCreate: ") + cublasGetStatusString(s));
        return CE_ERR_CUDA;
    }
    g_blas[dev] = h;
    *out = h;
    return CE_OK;
}

ce_status blas_check(cublasStatus_t s, const char* what) {
    if (s == CUBLAS_STATUS_SUCCESS) return CE_OK;
    record_message(std::string(what) + ": " + cublasGetStatusString(s));
    return CE_ERR_CUDA;
}

cudaDataType_t blas_type(int dtype) {
    return dtype == CE_F32 ? CUDA_R_32F : dtype == CE_BF16 ? CUDA_R_16BF : CUDA_R_16F;
}

int64_t align256(int64_t b) { return (b + 255) / 256 * 256; }

// Workspace layout: counts (2 doubles) | chunk scalars (3 floats a chunk) |
// logits chunk (fp32) | rounded gradient chunk (storage type, not for fp32).
struct FlceLayout {
    int64_t chunk, nchunks;
    int64_t off_counts, off_parts, off_logits, off_g, total;
};

FlceLayout layout(int dtype, int64_t rows, int64_t V, int64_t chunk_rows) {
    FlceLayout L{};
    int64_t c = chunk_rows;
    // default: about 2 GB of fp32 logits (under 1% of this GPU's memory), in
    // whole 256-row tiles of the tensor-core GEMMs when that leaves any
    if (c <= 0) {
        c = std::max<int64_t>(1, (int64_t{1} << 31) / (V * 4));
        if (c >= 256) c = c / 256 * 256;
    }
    c = std::max<int64_t>(1, std::min<int64_t>(c, std::max<int64_t>(rows, 1)));
    L.chunk = c;
    L.nchunks = rows == 0 ? 0 : (rows + c - 1) / c;
    const int64_t b = dtype == CE_F32 ? 4 : 2;
    L.off_counts = 0;
    L.off_parts = align256(16);
    L.off_logits = L.off_parts + align256(std::max<int64_t>(L.nchunks, 1) * 12);
    L.off_g = L.off_logits + align256(c * V * 4);
    L.total = L.off_g + (dtype == CE_F32 ? 0 : align256(c * V * b));
    return L;
}

}  // namespace
}  // namespace gbce

using namespace gbce;

extern "C" size_t ce_flce_workspace_bytes(int dtype, int64_t rows, int64_t V,
                                          int64_t chunk_rows) {
    if (dtype != CE_F32 && dtype != CE_BF16 && dtype != CE_F16) return 0;
    if (rows < 0 || V <= 0) return 0;
    return static_cast<size_t>(layout(dtype, rows, V, chunk_rows).total);
}

extern "C" ce_status ce_flce(const void* hidden, const void* lm_weight, const float* bias,
                             int dtype, int64_t rows, int64_t H, int64_t V, const void* target,
                             const float* class_weight, int64_t ignore_index,
                             float label_smoothing, float lse_square_scale, float softcap,
                             int reduction, uint32_t flags, float* loss, float* z_loss,
                             float* acc, int64_t* pred, void* grad_hidden, float* grad_weight,
                             float* grad_bias, int64_t chunk_rows, void* workspace,
                             size_t workspace_bytes, ce_stream_t stream) {
    if (dtype != CE_F32 && dtype != CE_BF16 && dtype != CE_F16) return CE_ERR_INVALID_ARG;
    if (rows < 0 || H <= 0 || V <= 0) return CE_ERR_INVALID_ARG;
    if (H > INT32_MAX || V > INT32_MAX - 16 || rows > INT32_MAX) return CE_ERR_UNSUPPORTED;
    if (reduction != CE_RED_NONE && reduction != CE_RED_SUM && reduction != CE_RED_MEAN)
        return CE_ERR_INVALID_ARG;
    if (!loss) return CE_ERR_INVALID_ARG;
    if (rows > 0 && (!hidden || !lm_weight || !target)) return CE_ERR_INVALID_ARG;
    const bool grad = (flags & CE_FLAG_GRAD) != 0;
    const FlceLayout L = layout(dtype, rows, V, chunk_rows);
    if (!workspace || workspace_bytes < static_cast<size_t>(L.total) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return CE_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (rows == 0)  // the empty batch: the forward's own scalars (NaN mean, 0 sum)
        return ce_fwd(nullptr, CE_F32, 0, V, nullptr, class_weight, ignore_index,
                      label_smoothing, lse_square_scale, softcap, reduction,
                      flags & ~static_cast<uint32_t>(CE_FLAG_GRAD), loss, z_loss, acc, pred,
                      stream);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_failure(e, "cudaGetDevice");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return record_cuda_failure(e, "cudaDeviceGetAttribute");
    // The three GEMMs on this library's tcgen05 kernel for 16-bit inputs
    // with rows of multiples of 8 elements; cuBLAS otherwise (or with
    // GBCE_FLCE_GEMM=cublas)
    const char* genv = std::getenv("GBCE_FLCE_GEMM");
    const bool use_tc = !(genv && std::strcmp(genv, "cublas") == 0) && dtype != CE_F32 &&
                        tc_operand_ok(hidden, dtype, H) && tc_operand_ok(lm_weight, dtype, H) &&
                        V % 8 == 0;
    cublasHandle_t blas = nullptr;
    ce_status rc = CE_OK;
    if (!use_tc) {
        rc = blas_for(dev, &blas);
        if (rc != CE_OK) return rc;
        rc = blas_check(cublasSetStream(blas, st), "cublasSetStream");
        if (rc != CE_OK) return rc;
    }

    char* ws = static_cast<char*>(workspace);
    double* counts = reinterpret_cast<double*>(ws + L.off_counts);
    float* parts = reinterpret_cast<float*>(ws + L.off_parts);
    float* logits = reinterpret_cast<float*>(ws + L.off_logits);
    void* gbuf = dtype == CE_F32 ? static_cast<void*>(logits) : static_cast<void*>(ws + L.off_g);
    const int64_t b = dtype == CE_F32 ? 4 : 2;
    const cudaDataType_t dt = blas_type(dtype);
    const uint32_t tflag = flags & static_cast<uint32_t>(CE_FLAG_TARGET_I64);
    const int64_t tbytes = tflag ? 8 : 4;

    // the batch's D and counted rows: every chunk is one shard of the batch
    rc = ce_count(target, class_weight, rows, V, ignore_index, tflag, counts, stream);
    if (rc != CE_OK) return rc;
    unsigned* status = nullptr;
    if (use_tc) {
        rc = library_status_word(st, &status);
        if (rc != CE_OK) return rc;
    }
    const float one = 1.f, zero = 0.f;
    for (int64_t k = 0; k < L.nchunks; ++k) {
        const int64_t r0 = k * L.chunk;
        const int64_t c = std::min<int64_t>(L.chunk, rows - r0);
        const char* hc = static_cast<const char*>(hidden) + r0 * H * b;
        // 1. logits = hidden_c @ W^T (+ bias), column-major [V, c]
        if (use_tc) {
            rc = tc_gemm_abt_launch(hc, lm_weight, dtype, c, V, H, logits, bias, status,
                                    status + 1, st);
            if (rc != CE_OK) return rc;
        } else {
            if (bias) {
                flce_bias_rows<<<static_cast<int>(std::min<int64_t>((c * V + 255) / 256, 8L * sms)),
                                 kFlceThreads, 0, st>>>(logits, bias, c, V);
                e = cudaGetLastError();
                if (e != cudaSuccess) return record_cuda_failure(e, "bias");
            }
            rc = blas_check(cublasGemmEx(blas, CUBLAS_OP_T, CUBLAS_OP_N, static_cast<int>(V),
                                         static_cast<int>(c), static_cast<int>(H), &one, lm_weight,
                                         dt, static_cast<int>(H), hc, dt, static_cast<int>(H),
                                         bias ? &one : &zero, logits, CUDA_R_32F,
                                         static_cast<int>(V), CUBLAS_COMPUTE_32F,
                                         CUBLAS_GEMM_DEFAULT),
                            "logits GEMM");
            if (rc != CE_OK) return rc;
        }
        // 2. the fused forward over the chunk (one shard of the batch); with
        // the tensor-core GEMMs and no grad_bias (which sums the fp32
        // gradient) it writes G in the storage type directly, when its plan
        // allows (the streaming kernel), saving the rounding pass's read
        // and write of the fp32 gradient
        const bool none = reduction == CE_RED_NONE;
        const FwdCall fc{logits, CE_F32, c, V, static_cast<const char*>(target) + r0 * tbytes,
                         class_weight, ignore_index, label_smoothing, lse_square_scale, softcap,
                         reduction, flags, none ? loss + r0 : parts + 3 * k,
                         (flags & CE_FLAG_Z_LOSS) ? (none ? z_loss + r0 : parts + 3 * k + 1)
                                                  : nullptr,
                         (flags & CE_FLAG_ACC) ? (none ? acc + r0 : parts + 3 * k + 2) : nullptr,
                         pred ? pred + r0 : nullptr, counts};
        bool g_done = false;
        if (grad && use_tc && dtype != CE_F32 && !grad_bias &&
            std::getenv("GBCE_FLCE_GOUT") == nullptr) {
            rc = fwd_shard_gout(fc, gbuf, dtype, stream);
            if (rc == CE_OK) g_done = true;
            else if (rc != CE_ERR_UNSUPPORTED) return rc;
        }
        if (!g_done) {
            rc = ce_fwd_shard(fc.logits, CE_F32, c, V, fc.target, class_weight, ignore_index,
                              label_smoothing, lse_square_scale, softcap, reduction, flags,
                              fc.loss, fc.z_loss, fc.acc, fc.pred, counts, stream);
            if (rc != CE_OK) return rc;
        }
        if (!grad) continue;
        // 3. G in the storage type (unless the forward wrote it)
        if (dtype != CE_F32 && !g_done) {
            const int grid = static_cast<int>(std::min<int64_t>((c * V / 8 + 255) / 256 + 1, 8L * sms));
            if (dtype == CE_BF16)
                flce_round<__nv_bfloat16><<<grid, kFlceThreads, 0, st>>>(
                    logits, static_cast<__nv_bfloat16*>(gbuf), c * V);
            else
                flce_round<__half><<<grid, kFlceThreads, 0, st>>>(logits, static_cast<__half*>(gbuf),
                                                                  c * V);
            e = cudaGetLastError();
            if (e != cudaSuccess) return record_cuda_failure(e, "round");
        }
        // 4. gradients
        void* gh = grad_hidden ? static_cast<char*>(grad_hidden) + r0 * H * b : nullptr;
        if (grad_hidden && use_tc) {
            // G [c, V] (K-major) @ W [V, H] (MN-major), rounded to dtype
            rc = tc_gemm_launch(gbuf, false, lm_weight, true, dtype, c, H, V, gh, CE_GEMM_16BIT,
                                nullptr, status, status + 1, st);
            if (rc != CE_OK) return rc;
        } else if (grad_hidden) {
            rc = blas_check(cublasGemmEx(blas, CUBLAS_OP_N, CUBLAS_OP_N, static_cast<int>(H),
                                         static_cast<int>(c), static_cast<int>(V), &one, lm_weight,
                                         dt, static_cast<int>(H), gbuf, dt, static_cast<int>(V),
                                         &zero, static_cast<char*>(grad_hidden) + r0 * H * b, dt,
                                         static_cast<int>(H), CUBLAS_COMPUTE_32F,
                                         CUBLAS_GEMM_DEFAULT),
                            "grad_hidden GEMM");
            if (rc != CE_OK) return rc;
        }
        if (grad_weight && use_tc) {
            // G^T [V, c] (G read MN-major) @ hidden_c [c, H] (MN-major), fp32,
            // written by the first chunk and added to by the others
            rc = tc_gemm_launch(gbuf, true, hc, true, dtype, V, H, c, grad_weight,
                                k == 0 ? CE_GEMM_F32 : CE_GEMM_F32_ADD, nullptr, status,
                                status + 1, st);
            if (rc != CE_OK) return rc;
        } else if (grad_weight) {
            rc = blas_check(cublasGemmEx(blas, CUBLAS_OP_N, CUBLAS_OP_T, static_cast<int>(H),
                                         static_cast<int>(V), static_cast<int>(c), &one, hc, dt,
                                         static_cast<int>(H), gbuf, dt, static_cast<int>(V),
                                         k == 0 ? &zero : &one, grad_weight, CUDA_R_32F,
                                         static_cast<int>(H), CUBLAS_COMPUTE_32F,
                                         CUBLAS_GEMM_DEFAULT),
                            "grad_weight GEMM");
            if (rc != CE_OK) return rc;
        }
        if (grad_bias) {
            const int grid = static_cast<int>(std::min<int64_t>((V + kFlceThreads - 1) / kFlceThreads,
                                                                8L * sms));
            flce_colsum<<<grid, kFlceThreads, 0, st>>>(logits, grad_bias, c, V, k == 0 ? 0 : 1);
            e = cudaGetLastError();
            if (e != cudaSuccess) return record_cuda_failure(e, "grad_bias column sums");
        }
    }
    if (reduction != CE_RED_NONE) {
        flce_sum_chunks<<<1, 32, 0, st>>>(parts, static_cast<int>(L.nchunks), loss,
                                          (flags & CE_FLAG_Z_LOSS) ? z_loss : nullptr,
                                          (flags & CE_FLAG_ACC) ? acc : nullptr);
        e = cudaGetLastError();
        if (e != cudaSuccess) return record_cuda_failure(e, "sum of chunks");
    }
    return CE_OK;
}

extern "C" ce_status ce_scale_round(const float* in, const float* grad_output, void* out,
                                    int dtype, int64_t n, ce_stream_t stream) {
    if (dtype != CE_F32 && dtype != CE_BF16 && dtype != CE_F16) return CE_ERR_INVALID_ARG;
    if (n < 0) return CE_ERR_INVALID_ARG;
    if (n == 0) return CE_OK;
    if (!in || !grad_output || !out) return CE_ERR_INVALID_ARG;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_failure(e, "cudaGetDevice");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return record_cuda_failure(e, "cudaDeviceGetAttribute");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int grid = static_cast<int>(std::min<int64_t>((n + 255) / 256, 8L * sms));
    if (dtype == CE_F32)
        flce_scale_round<float><<<grid, kFlceThreads, 0, st>>>(in, grad_output,
                                                               static_cast<float*>(out), n);
    else if (dtype == CE_BF16)
        flce_scale_round<__nv_bfloat16><<<grid, kFlceThreads, 0, st>>>(
            in, grad_output, static_cast<__nv_bfloat16*>(out), n);
    else
        flce_scale_round<__half><<<grid, kFlceThreads, 0, st>>>(in, grad_output,
                                                                static_cast<__half*>(out), n);
    e = cudaGetLastError();
    if (e != cudaSuccess) return record_cuda_failure(e, "scale and round");
    return CE_OK;
}
