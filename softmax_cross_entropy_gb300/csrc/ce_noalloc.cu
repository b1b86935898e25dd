// ce_fwd_noalloc: the forward call for callers that cannot allocate device
// memory, such as code running inside a custom allocator's callback, a
// memory-capped sandbox, or a framework that forbids allocations after its
// start-up phase. Its scratch (the epilogue's ticket, the status word and
// one partial-sum slot per participating CTA) lives in a fixed file-scope
// device array instead of memory from cudaMalloc.
#include <cstdint>
#include <cstdlib>
#include <map>
#include <mutex>

#include "ce_kernels.cuh"
#include "gbce.h"

namespace gbce {

ce_status fwd_with_scratch(Scratch* scratch, int max_slots, const FwdCall& c, cudaStream_t st);
ce_status record_cuda_failure(cudaError_t e, const char* what);

namespace {

// Room for 2048 partial-sum slots (one per CTA or cluster of a launch): about
// 64 KB, held by every GPU that loads the library until the process exits.
constexpr int kStaticSlots = 2048;
constexpr size_t kStaticScratchBytes = sizeof(Scratch) + (kStaticSlots - 1) * sizeof(Partial);

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
std::map<int, Scratch*> g_static_addr;  // device -> address of g_static_scratch there

// The array's device address on the current device, looked up once per
// device. In host code the symbol is only a stand-in; the device address
// comes from cudaGetSymbolAddress with that device current.
ce_status static_scratch(int dev, Scratch** out) {
    std::lock_guard<std::mutex> lock(g_static_mu);
    auto it = g_static_addr.find(dev);
    if (it != g_static_addr.end()) {
        *out = it->second;
        return CE_OK;
    }
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess || !ptr) return record_cuda_failure(e, "cudaGetSymbolAddress(static scratch)");
    g_static_addr[dev] = static_cast<Scratch*>(ptr);
    *out = static_cast<Scratch*>(ptr);
    return CE_OK;
}

}  // namespace
}  // namespace gbce

using namespace gbce;

namespace gbce {
namespace {

// The number of partial-sum slots a call may use: the array's, or fewer
// when GBCE_TEST_NOALLOC_SLOTS lowers it (a test hook, so that the refusal
// of an oversized launch can be exercised on any GPU).
int usable_slots() {
    const char* v = std::getenv("GBCE_TEST_NOALLOC_SLOTS");
    const int lim = (v && *v) ? std::atoi(v) : 0;
    return lim > 0 && lim < kStaticSlots ? lim : kStaticSlots;
}

}  // namespace
}  // namespace gbce

extern "C" ce_status ce_fwd_noalloc(void* logits, int dtype, int64_t rows, int64_t V,
                                    const void* target, const float* weight,
                                    int64_t ignore_index, float label_smoothing,
                                    float lse_square_scale, float softcap, int reduction,
                                    uint32_t flags, float* loss, float* z_loss, float* acc,
                                    int64_t* pred, ce_stream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_failure(e, "cudaGetDevice");
    Scratch* s = nullptr;
    ce_status rc = static_scratch(dev, &s);
    if (rc != CE_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const FwdCall c{logits, dtype, rows, V, target, weight, ignore_index, label_smoothing,
                    lse_square_scale, softcap, reduction, flags, loss, z_loss, acc, pred, nullptr};
    return fwd_with_scratch(s, usable_slots(), c, st);
}

extern "C" ce_status ce_noalloc_status(ce_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return record_cuda_failure(e, "cudaStreamSynchronize");
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_failure(e, "cudaGetDevice");
    Scratch* s = nullptr;
    const ce_status rc = static_scratch(dev, &s);
    if (rc != CE_OK) return rc;
    // read the sticky word into a host variable, then clear it, in stream
    // order; nothing is allocated
    unsigned status = 0;
    e = cudaMemcpyAsync(&status, &s->status, sizeof status, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(&s->status, 0, sizeof status, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return record_cuda_failure(e, "reading the static scratch status");
    if (status & kDevErrTimeout) return CE_ERR_TIMEOUT;
    if (status & kDevErrTarget) return CE_ERR_TARGET_RANGE;
    return CE_OK;
}
