// C ABI of libgbce.so: argument checks, library-owned scratch, the choice
// of kernel variant and launch shape, and the launches themselves. The
// definitions the calls implement are stated in include/gbce.h.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "ce_kernels.cuh"
#include "gbce.h"

namespace gbce {

// the single-read N-D tile kernel (ce_fwd_nd_tile.cu)
ce_status nd_tile_launch(const FwdArgs& f, int dtype, int64_t N, int64_t C, int64_t inner,
                         int sm_count, int smem_optin, int max_cluster, bool narrow_rows,
                         bool after_count, cudaStream_t st);

namespace {

thread_local std::string g_last_error;

ce_status cuda_failure(cudaError_t e, const char* what) {
    g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
    return CE_ERR_CUDA;
}

struct DeviceInfo {
    int sm_count = 0;
    int smem_per_sm = 0;
    int smem_optin = 0;
};

// A launch plan for one (device, dtype, V, variant): which kernel, how many
// CTAs per row, ring depth, dynamic shared memory and the resident grid.
enum class Kind { General, Staged, Stream, Reg, Tmem };

struct Plan {
    const void* fn = nullptr;
    Kind kind = Kind::General;
    bool staged = false;
    int nt = 0;
    int cluster = 1;
    int stages = 0;
    int slice_vec = 0;
    size_t smem = 0;
    int64_t max_units = 0;  // resident CTAs (cluster == 1) or clusters
    // streaming kernel layout
    int ng = 0, sg = 0, chunk_vec = 0, nchunk = 0, resident = 0;
    int reg_wpr = 0;  // register-resident kernel: warps of a row team
    uint32_t reg_buf_stride = 0;  // register-resident kernel: bytes of a team's row buffer
    int reg_nbuf = 1;             // register-resident kernel: row buffers a team
    int tm_slice_vec = 0, tm_slots = 0;  // tensor-memory kernel: slice of a CTA, ring slots
};

// (device, dtype, V (negative when the logits are not 16-byte aligned),
// softcap (0 off, 1 on, 2 on and at most kTmMaxSoftcap), weighted
// smoothing, weights 16-byte aligned, tuning signature)
using PlanKey = std::tuple<int, int, int64_t, int, bool, bool, std::string>;

// The tensor-memory kernel shifts exp(z) by the softcap s itself; exp(-2 s)
// must stay a normal fp32
constexpr float kTmMaxSoftcap = 40.f;
// N-D logits with at least this many classes take the split form
constexpr int64_t kNdSplitMinClasses = 768;
// ... and the single-read tile form from this many, where one or two CTAs
// hold a tile's classes
constexpr int64_t kNdTileMinClasses = 512;

std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;
std::map<std::pair<int, uintptr_t>, Scratch*> g_scratch;
std::map<PlanKey, Plan> g_plans;

int env_int(const char* name, int fallback) {
    const char* v = std::getenv(name);
    return (v && *v) ? std::atoi(v) : fallback;
}

// Every tuning override that the kernel plans read, as one string: part of
// each plan cache key, so that a plan made under one setting never serves
// another.
std::string tuning_signature() {
    static const char* const kVars[] = {
        "GBCE_KERNEL",        "GBCE_CLUSTER",      "GBCE_CFG",          "GBCE_MAX_STAGES",
        "GBCE_STREAM_GROUPS", "GBCE_STREAM_TWICE", "GBCE_STREAM_SLOTS", "GBCE_STREAM_WARPS",
        "GBCE_REG_MAX_BYTES", "GBCE_REG_NVL",      "GBCE_REG_CLUSTER",  "GBCE_REG_SW",
        "GBCE_REG_NBUF",      "GBCE_TMEM"};
    std::string sig;
    for (const char* name : kVars) {
        const char* v = std::getenv(name);
        if (v) sig += v;
        sig += '|';
    }
    return sig;
}

ce_status device_info(int dev, DeviceInfo* out) {
    auto it = g_devices.find(dev);
    if (it != g_devices.end()) {
        *out = it->second;
        return CE_OK;
    }
    DeviceInfo d;
    cudaError_t e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return cuda_failure(e, "cudaDeviceGetAttribute");
    g_devices[dev] = d;
    *out = d;
    return CE_OK;
}

// Scratch for (device, stream): allocated and zeroed on first use, on the
// caller's stream so the zeroing is ordered before the first kernel.
ce_status scratch_for(int dev, cudaStream_t st, Scratch** out) {
    const auto key = std::make_pair(dev, reinterpret_cast<uintptr_t>(st));
    auto it = g_scratch.find(key);
    if (it != g_scratch.end()) {
        *out = it->second;
        return CE_OK;
    }
    void* p = nullptr;
    cudaError_t e = cudaMalloc(&p, kScratchBytes);
    if (e != cudaSuccess) return cuda_failure(e, "cudaMalloc(scratch)");
    e = cudaMemsetAsync(p, 0, kScratchBytes, st);
    if (e != cudaSuccess) {
        cudaFree(p);
        return cuda_failure(e, "cudaMemsetAsync(scratch)");
    }
    g_scratch[key] = static_cast<Scratch*>(p);
    *out = static_cast<Scratch*>(p);
    return CE_OK;
}

// The split N-D forward's workspace for (device, stream): grown to `bytes`
// when a call needs more (the old buffer is freed first, which waits for
// the device), kept for later calls on the stream.
std::map<std::pair<int, uintptr_t>, std::pair<void*, size_t>> g_nd_work;

ce_status nd_work_for(int dev, cudaStream_t st, size_t bytes, void** out) {
    const auto key = std::make_pair(dev, reinterpret_cast<uintptr_t>(st));
    auto it = g_nd_work.find(key);
    if (it != g_nd_work.end() && it->second.second >= bytes) {
        *out = it->second.first;
        return CE_OK;
    }
    if (it != g_nd_work.end()) {
        cudaError_t e = cudaFree(it->second.first);
        g_nd_work.erase(it);
        if (e != cudaSuccess) return cuda_failure(e, "cudaFree(N-D workspace)");
    }
    void* p = nullptr;
    cudaError_t e = cudaMalloc(&p, bytes);
    if (e != cudaSuccess) return cuda_failure(e, "cudaMalloc(N-D workspace)");
    g_nd_work[key] = std::make_pair(p, bytes);
    *out = p;
    return CE_OK;
}

const void* staged_fn(int dtype, int cfg, bool softcap, bool wsmooth) {
    if (dtype == CE_F16) return nullptr;  // fp16 takes the streaming or the general kernel
    if (dtype == CE_BF16) {
        if (softcap)
            return wsmooth ? staged_kernel_bf16_softcap_wsmooth(cfg)
                           : staged_kernel_bf16_softcap_plain(cfg);
        return wsmooth ? staged_kernel_bf16_nocap_wsmooth(cfg) : staged_kernel_bf16_nocap_plain(cfg);
    }
    if (softcap)
        return wsmooth ? staged_kernel_f32_softcap_wsmooth(cfg) : staged_kernel_f32_softcap_plain(cfg);
    return wsmooth ? staged_kernel_f32_nocap_wsmooth(cfg) : staged_kernel_f32_nocap_plain(cfg);
}

// Evaluates the staged kernel with shape `cfg` and `C` CTAs per row.
// Returns false when the combination does not fit (then other candidates or
// the general path are tried); `occ` receives the CTAs per SM.
bool try_staged(int dtype, int64_t V, bool softcap, bool wsmooth, int C, int cfg,
                const DeviceInfo& dev, Plan* out, int* occ, ce_status* err) {
    const int64_t bytes = dtype == CE_F32 ? 4 : 2;
    const int64_t ve = 16 / bytes;
    const int64_t vec_row = V / ve;
    const int64_t per = (vec_row + C - 1) / C;
    if (C > 1 && per * (C - 1) >= vec_row) return false;  // a CTA would own nothing
    if (static_cast<int64_t>(kStagedCfgs[cfg].nt) * kStagedCfgs[cfg].nv < per) return false;
    const void* fn = staged_fn(dtype, cfg, softcap, wsmooth);
    if (!fn) return false;
    const int nt = kStagedCfgs[cfg].nt;
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) {
        *err = cuda_failure(e, "cudaFuncGetAttributes");
        return false;
    }
    const size_t stage_bytes = static_cast<size_t>(per) * 16;
    const size_t wbytes = wsmooth ? static_cast<size_t>(per) * ve * 4 : 0;
    const size_t max_dyn = static_cast<size_t>(dev.smem_optin) - fa.sharedSizeBytes;
    if (2 * stage_bytes + wbytes > max_dyn) return false;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(max_dyn));
    if (e == cudaSuccess && C > 8)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) {
        *err = cuda_failure(e, "cudaFuncSetAttribute");
        return false;
    }
    // Largest occupancy the registers allow, then the deepest ring that keeps it.
    int occ2 = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ2, fn, nt, 2 * stage_bytes + wbytes);
    if (e != cudaSuccess) {
        *err = cuda_failure(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        return false;
    }
    if (occ2 < 1) return false;
    int stages = 2;
    const int max_stages = std::max(2, std::min(kMaxStages, env_int("GBCE_MAX_STAGES", kMaxStages)));
    for (int s = 3; s <= max_stages; ++s) {
        const size_t dyn = s * stage_bytes + wbytes;
        if (dyn > max_dyn) break;
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, fn, nt, dyn) != cudaSuccess ||
            o < occ2)
            break;
        stages = s;
    }
    const size_t smem = stages * stage_bytes + wbytes;
    int64_t units = static_cast<int64_t>(occ2) * dev.sm_count;
    if (C > 1) {
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(static_cast<unsigned>(C * dev.sm_count));
        lc.blockDim = dim3(static_cast<unsigned>(nt));
        lc.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = static_cast<unsigned>(C);
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        lc.attrs = &attr;
        lc.numAttrs = 1;
        int ncl = 0;
        e = cudaOccupancyMaxActiveClusters(&ncl, fn, &lc);
        if (e != cudaSuccess) {
            // a cluster size this device cannot schedule: not a candidate
            cudaGetLastError();
            return false;
        }
        if (ncl < 1) return false;
        units = ncl;
    }
    units = std::min<int64_t>(units, kMaxUnits);
    out->fn = fn;
    out->staged = true;
    out->nt = nt;
    out->cluster = C;
    out->stages = stages;
    out->slice_vec = static_cast<int>(per);
    out->smem = smem;
    out->max_units = units;
    *occ = occ2;
    return true;
}

// The streaming kernel's layout. NW consumer warps (8 by default, with 8
// vectors a thread a slot, or 16 with 4). A slot holds VPT vectors
// for each thread of a group (or the whole row when it is shorter). A row
// that fits in one slot with room for two more stays resident, with as many
// row groups as the ring holds; otherwise one group of all consumer warps
// streams the row twice.
// ws: class weights with label smoothing; the kernel then keeps the V
// weights in shared memory after the ring, which must leave room for at
// least two slots.
bool try_stream(int dtype, int64_t V, bool softcap, bool ws, const DeviceInfo& dev, Plan* out,
                ce_status* err, bool lsm = false) {
    const int64_t bytes = dtype == CE_F32 ? 4 : 2;
    const int64_t vec_row = V * bytes / 16;
    const int force_ng = env_int("GBCE_STREAM_GROUPS", 0);
    const bool force_twice = env_int("GBCE_STREAM_TWICE", 0) != 0;
    // 16 consumer warps hide latency better than 8 (measured on GB300 at
    // 4096 rows, bf16: 6045 against 5815 GB/s at V = 131072, 3877 against
    // 3561 at V = 16384), except for plain rows of at most 8 KB. The
    // class-weighted smoothing kernel exists with 8 only. GBCE_STREAM_WARPS
    // (8 or 16) overrides.
    const int nw_env = env_int("GBCE_STREAM_WARPS", 0);
    const int nw_auto = (!softcap && V * bytes <= 8192) ? 8 : 16;
    // (the log-softmax mode exists with 16 consumer warps only)
    const int nw = lsm ? 16 : ws ? 8 : (nw_env == 8 || nw_env == 16 ? nw_env : nw_auto);
    const int vpt_res = nw == 8 ? 8 : 4;  // the two compiled shapes
    const size_t wbytes = ws ? static_cast<size_t>((V * 4 + 15) / 16 * 16) : 0;
    Plan p;
    const void* fn = nullptr;
    size_t ring_max = 0;
    auto prepare = [&](int vpt) -> bool {
        fn = lsm  ? stream_kernel_lsm(dtype)
             : ws ? stream_kernel_ws(dtype, softcap)
                  : stream_kernel(dtype, softcap, vpt, nw);
        if (!fn) return false;
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, fn);
        if (e == cudaSuccess) {
            const size_t dyn_max = static_cast<size_t>(dev.smem_optin) - fa.sharedSizeBytes;
            ring_max = dyn_max > wbytes ? dyn_max - wbytes : 0;
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(dyn_max));
        }
        if (e != cudaSuccess) {
            *err = cuda_failure(e, "stream kernel attributes");
            return false;
        }
        return true;
    };
    if (!force_twice) {
        if (!prepare(vpt_res)) return false;
        for (int ng = kStreamMaxGroups; ng >= 1 && !p.ng; ng >>= 1) {
            if (force_ng && ng != force_ng) continue;
            if (nw % ng) continue;
            const int64_t cap = static_cast<int64_t>(vpt_res) * 32 * (nw / ng);
            const int64_t nchunk = (vec_row + cap - 1) / cap;
            const int64_t cvec = nchunk == 1 ? vec_row : cap;
            for (int64_t sg = 3 * nchunk; sg >= 2 * nchunk; --sg) {
                if (ng * sg > kStreamMaxSlots) continue;
                if (static_cast<size_t>(ng * sg * cvec * 16) > ring_max) continue;
                p.ng = ng;
                p.sg = static_cast<int>(sg);
                p.chunk_vec = static_cast<int>(cvec);
                p.nchunk = static_cast<int>(nchunk);
                p.resident = 1;
                break;
            }
        }
    }
    if (!p.ng) {
        const int vpt = vpt_res;
        if (!prepare(vpt)) return false;
        p = Plan();
        // one group by default; GBCE_STREAM_GROUPS splits the warps into
        // groups that stream different rows
        p.ng = (force_ng > 0 && force_ng <= kStreamMaxGroups && nw % force_ng == 0) ? force_ng : 1;
        p.chunk_vec =
            static_cast<int>(std::min<int64_t>(vec_row, 32 * (nw / p.ng) * vpt));
        if (ring_max / (static_cast<size_t>(p.ng) * p.chunk_vec * 16) < 3) {
            // little room left by the weights: smaller slots (a multiple of
            // the group's threads, as the vector ownership needs), three deep
            const int gt = 32 * (nw / p.ng);
            const int64_t fit = static_cast<int64_t>(ring_max / (3 * 16 * static_cast<size_t>(p.ng)));
            const int64_t c = fit / gt * gt;
            if (c >= gt && c < p.chunk_vec) p.chunk_vec = static_cast<int>(c);
        }
        p.nchunk = static_cast<int>((vec_row + p.chunk_vec - 1) / p.chunk_vec);
        p.sg = static_cast<int>(std::min<size_t>(
            kStreamMaxSlots / p.ng, ring_max / (static_cast<size_t>(p.ng) * p.chunk_vec * 16)));
        const int want_slots = env_int("GBCE_STREAM_SLOTS", 0);
        if (want_slots >= 2) p.sg = std::min(p.sg, want_slots);
        p.resident = 0;
        if (p.sg < 2) return false;
    }
    p.fn = fn;
    p.kind = Kind::Stream;
    p.nt = 32 * (nw + 1);
    p.smem = static_cast<size_t>(p.ng) * p.sg * p.chunk_vec * 16 + wbytes;
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, p.nt, p.smem);
    if (e != cudaSuccess) {
        *err = cuda_failure(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        return false;
    }
    if (occ < 1) return false;
    p.max_units = std::min<int64_t>(static_cast<int64_t>(occ) * dev.sm_count, kMaxUnits);
    *out = p;
    return true;
}

// Row buffers of the register-resident kernel `fn` (nt threads, `teams`
// teams, buffers of `stride` bytes, `extra` bytes of shared memory after
// them): one a team. GBCE_REG_NBUF=2 gives each team two (two rows in
// flight a team); that measured slower at every row length on GB300
// (4096 rows bf16, forward alone: V = 4096 27.9 against 26.3 us, 8192 39.2
// against 37.0, 16384 61.9 against 57.9). Sets the kernel's shared-memory
// limit; occ = 0 when nothing fits.
ce_status reg_buffers(const DeviceInfo& dev, const void* fn, int nt, int teams,
                      uint32_t stride, size_t extra, int* nbuf, size_t* smem, int* occ) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, fn);
    const size_t dyn_max = static_cast<size_t>(dev.smem_optin) - fa.sharedSizeBytes;
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(dyn_max));
    if (e != cudaSuccess) return cuda_failure(e, "register kernel attributes");
    int o[3] = {0, 0, 0};
    for (int nb = 1; nb <= 2; ++nb) {
        const size_t sm = static_cast<size_t>(teams) * nb * stride + extra;
        if (sm > dyn_max) continue;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o[nb], fn, nt, sm);
        if (e != cudaSuccess) return cuda_failure(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    }
    const int nb = env_int("GBCE_REG_NBUF", 1) == 2 && o[2] >= 1 ? 2 : 1;
    *nbuf = nb;
    *occ = o[nb];
    *smem = static_cast<size_t>(teams) * nb * stride + extra;
    return CE_OK;
}

// The tensor-memory kernel's plan for rows of vrow 16-byte vectors: a
// cluster of C CTAs a row, CTA c the slice of slice vectors from c * slice,
// each slice's r values within the 128 TMEM columns a consumer thread has;
// a ring of 32 KB slots in the rest of shared memory; as many clusters as
// fit. Leaves `best` alone when the row does not fit a cluster of 8.
ce_status plan_tmem(const DeviceInfo& dev, int dtype, int64_t vrow, Plan* best) {
    const int VE = dtype == CE_F32 ? 4 : 8;
    const int64_t chunk = 32 * kTmWarps * kTmVecPerThread;
    const int64_t max_vec_cta = 32 * kTmWarps * (128 / VE);  // 128 columns a thread
    const int64_t C = (vrow + max_vec_cta - 1) / max_vec_cta;
    const int64_t slice = ((vrow + C - 1) / C + chunk - 1) / chunk * chunk;
    if (C > kTmMaxCluster || slice > max_vec_cta) return CE_OK;
    const void* fn = tmem_kernel(dtype);
    const int nt = 32 * (kTmWarps + 1);
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, fn);
    const size_t dyn_max = static_cast<size_t>(dev.smem_optin) - fa.sharedSizeBytes;
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(dyn_max));
    if (e != cudaSuccess) return cuda_failure(e, "tensor-memory kernel attributes");
    const int slots = static_cast<int>(
        std::min<size_t>(kTmMaxSlots, dyn_max / (static_cast<size_t>(chunk) * 16)));
    const size_t smem = static_cast<size_t>(slots) * chunk * 16;
    // one CTA an SM: each allocates all 512 TMEM columns, and two CTAs of
    // one cluster on one SM would wait on each other. (Two CTAs of 8
    // consumer warps an SM, each with 256 columns, measured slower: 753
    // against 536 us at 4096 x 131072 bf16, softcap 30.)
    if (slots < 2 || 2 * (smem + fa.sharedSizeBytes) <= static_cast<size_t>(dev.smem_per_sm))
        return CE_OK;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(static_cast<unsigned>(C * dev.sm_count));
    lc.blockDim = dim3(static_cast<unsigned>(nt));
    lc.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = static_cast<unsigned>(C);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    lc.attrs = &attr;
    lc.numAttrs = 1;
    int ncl = 0;
    e = cudaOccupancyMaxActiveClusters(&ncl, fn, &lc);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return CE_OK;  // not schedulable here: not a candidate
    }
    if (ncl < 1) return CE_OK;
    best->fn = fn;
    best->kind = Kind::Tmem;
    best->nt = nt;
    best->smem = smem;
    best->cluster = static_cast<int>(C);
    best->tm_slice_vec = static_cast<int>(slice);
    best->tm_slots = slots;
    best->max_units = ncl;
    return CE_OK;
}

ce_status make_plan(int devid, int dtype, int64_t V, bool softcap, bool sc_small, bool wsmooth,
                    bool aligned, bool w_aligned, Plan* out) {
    // Tuning overrides: GBCE_CLUSTER forces the CTAs per row (1, 2, 4, 8 or
    // 16; -1 forces the general path) and GBCE_CFG the CTA shape index.
    const int forced_c = env_int("GBCE_CLUSTER", 0);
    const int forced_cfg = env_int("GBCE_CFG", -1);
    // GBCE_KERNEL: 1 staged, 2 streaming, 3 general, 4 register-resident,
    // 5 register-resident with a cluster of CTAs a row (0: automatic)
    const int forced_kind = env_int("GBCE_KERNEL", 0);
    const PlanKey key(devid, dtype, aligned ? V : -V, softcap ? (sc_small ? 2 : 1) : 0, wsmooth,
                      w_aligned, tuning_signature());
    auto it = g_plans.find(key);
    if (it != g_plans.end()) {
        *out = it->second;
        return CE_OK;
    }
    DeviceInfo dev;
    ce_status rc = device_info(devid, &dev);
    if (rc != CE_OK) return rc;
    Plan best;
    const int64_t bytes = dtype == CE_F32 ? 4 : 2;
    const bool fast_ok = aligned && (V * bytes) % 16 == 0 && forced_c >= 0 && forced_kind != 3;
    // The register-resident kernel for rows of at most GBCE_REG_MAX_BYTES
    // (default and limit 64 KB: 8 warps of 16 vectors a thread). A thread
    // holds 8 or 16 16-byte vectors (GBCE_REG_NVL forces one); a team of
    // the fewest warps that hold a row owns it, and a CTA has as many teams
    // as fit in 8 warps. Its class weights are read as 16-byte vectors.
    const int64_t reg_max = env_int("GBCE_REG_MAX_BYTES", 65536);
    const int64_t vrow = V * bytes / 16;
    // 8 vectors a thread for rows of at most 8 KB, else 16: at 16 and 32 KB
    // bf16 rows 16 vectors a thread (a warp for each 8 KB of the row)
    // measured 3-6% faster than 8; at 8 KB the two are even
    const int nvl_env = env_int("GBCE_REG_NVL", 0);
    const int nvl = (nvl_env == 8 || nvl_env == 16) ? nvl_env : (vrow <= 512 ? 8 : 16);
    const int64_t wpr = (vrow + 32 * nvl - 1) / (32 * nvl);
    // Class-weighted smoothing: the weights in shared memory (one CTA of 16
    // warps an SM, 8 vectors a thread, teams of up to 16 warps) when they
    // fit beside the row buffers; the weights are then read once per CTA
    // instead of twice per element from L1/L2 (GBCE_REG_SW=0 turns it off)
    const int64_t wpr_sw = (vrow + 32 * 8 - 1) / (32 * 8);
    if (fast_ok && wsmooth && w_aligned && wpr_sw <= kRegSwWarps && env_int("GBCE_REG_SW", 1) &&
        (forced_kind == 4 || (forced_kind == 0 && V * bytes <= reg_max))) {
        const void* fn = reg_kernel_sw(dtype, softcap);
        const int teams = kRegSwWarps / static_cast<int>(wpr_sw);
        const int nt = 32 * static_cast<int>(wpr_sw) * teams;
        const uint32_t stride = static_cast<uint32_t>((V * bytes + 127) / 128 * 128);
        int nbuf = 1, occ = 0;
        size_t smem = 0;
        rc = reg_buffers(dev, fn, nt, teams, stride, static_cast<size_t>(V) * 4, &nbuf, &smem, &occ);
        if (rc != CE_OK) return rc;
        if (occ >= 1) {
            best.fn = fn;
            best.kind = Kind::Reg;
            best.nt = nt;
            best.smem = smem;
            best.reg_buf_stride = stride;
            best.reg_nbuf = nbuf;
            best.reg_wpr = static_cast<int>(wpr_sw);
            best.max_units = std::min<int64_t>(
                static_cast<int64_t>(std::min(occ, 8)) * dev.sm_count, kMaxUnits);
        }
    }
    if (best.kind == Kind::General && fast_ok && (!wsmooth || w_aligned) &&
        wpr <= kRegMaxWarps &&
        (forced_kind == 4 || (forced_kind == 0 && V * bytes <= reg_max))) {
        const void* fn = reg_kernel(dtype, softcap, wsmooth, nvl);
        const int teams = kRegMaxWarps / static_cast<int>(wpr);
        const int nt = 32 * static_cast<int>(wpr) * teams;
        // one or two row buffers a team (the next rows' bulk copies)
        const uint32_t stride = static_cast<uint32_t>((V * bytes + 127) / 128 * 128);
        int nbuf = 1, occ = 0;
        size_t smem = 0;
        rc = reg_buffers(dev, fn, nt, teams, stride, 0, &nbuf, &smem, &occ);
        if (rc != CE_OK) return rc;
        if (occ >= 1) {
            best.fn = fn;
            best.kind = Kind::Reg;
            best.nt = nt;
            best.smem = smem;
            best.reg_buf_stride = stride;
            best.reg_nbuf = nbuf;
            best.reg_wpr = static_cast<int>(wpr);
            // at most 8 CTAs an SM: the partial-sum slots of a launch stay
            // within 8 per SM, as for the other kernels
            best.max_units = std::min<int64_t>(
                static_cast<int64_t>(std::min(occ, 8)) * dev.sm_count, kMaxUnits);
        }
    }
    // Rows longer than one CTA of the register-resident kernel holds: a
    // cluster of C CTAs owns a row, each one 8-warp team holding a slice of
    // 32 * 8 * 16 vectors (C <= 8, the portable cluster size).
    const int64_t cl_vpc = 32 * kRegMaxWarps * 16;
    const int64_t cl_C = (vrow + cl_vpc - 1) / cl_vpc;
    if (fast_ok && (!wsmooth || w_aligned) && best.kind == Kind::General && cl_C >= 2 &&
        cl_C <= 8 && (forced_kind == 5 || (forced_kind == 0 && env_int("GBCE_REG_CLUSTER", 0)))) {
        const void* fn = reg_cluster_kernel(dtype, softcap, wsmooth);
        const int nt = 32 * kRegMaxWarps;
        const uint32_t stride = static_cast<uint32_t>(cl_vpc * 16);
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, fn);
        const size_t dyn_max = static_cast<size_t>(dev.smem_optin) - fa.sharedSizeBytes;
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(dyn_max));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
        if (e != cudaSuccess) return cuda_failure(e, "register kernel attributes");
        int ncl = 0;
        if (stride <= dyn_max) {
            cudaLaunchConfig_t lc = {};
            lc.gridDim = dim3(static_cast<unsigned>(cl_C * dev.sm_count));
            lc.blockDim = dim3(static_cast<unsigned>(nt));
            lc.dynamicSmemBytes = stride;
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = static_cast<unsigned>(cl_C);
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            lc.attrs = &attr;
            lc.numAttrs = 1;
            e = cudaOccupancyMaxActiveClusters(&ncl, fn, &lc);
            if (e != cudaSuccess) {
                cudaGetLastError();
                ncl = 0;
            }
        }
        if (ncl >= 1) {
            best.fn = fn;
            best.kind = Kind::Reg;
            best.nt = nt;
            best.smem = stride;
            best.reg_buf_stride = stride;
            best.reg_wpr = kRegMaxWarps;
            best.cluster = static_cast<int>(cl_C);
            // clusters; a launch's CTAs stay within the partial-sum slots
            best.max_units = std::min<int64_t>(ncl, kMaxUnits / cl_C);
        }
    }
    // Softcapped rows longer than the register kernel takes: the
    // tensor-memory kernel (tanh formed once an element and kept in TMEM, a
    // cluster of C CTAs a row), for softcaps up to kTmMaxSoftcap
    // (GBCE_TMEM=0 turns it off; GBCE_KERNEL=6 forces it)
    if (fast_ok && softcap && sc_small && !wsmooth && best.kind == Kind::General &&
        (forced_kind == 6 ||
         (forced_kind == 0 && V * bytes > reg_max && env_int("GBCE_TMEM", 1)))) {
        rc = plan_tmem(dev, dtype, vrow, &best);
        if (rc != CE_OK) return rc;
    }
    if (fast_ok && forced_kind != 1 && best.kind == Kind::General) {
        rc = CE_OK;
        if (!try_stream(dtype, V, softcap, wsmooth, dev, &best, &rc) && rc != CE_OK) return rc;
    }
    if (fast_ok && best.kind == Kind::General && forced_kind != 2) {
        // Candidates: every shape and cluster size that fits. Prefer at
        // least two resident CTAs per SM (latency hiding across rows), then
        // the fewest CTAs per row (cheaper cluster merges), then the deeper
        // ring.
        long best_score = -1;
        for (int C : {1, 2, 4, 8, 16}) {
            if (forced_c && C != forced_c) continue;
            for (int cfg = 0; cfg < kNumStagedCfgs; ++cfg) {
                if (forced_cfg >= 0 && cfg != forced_cfg) continue;
                Plan p;
                int occ = 0;
                rc = CE_OK;
                if (!try_staged(dtype, V, softcap, wsmooth, C, cfg, dev, &p, &occ, &rc)) {
                    if (rc != CE_OK) return rc;
                    continue;
                }
                const long score = std::min(occ, 2) * 100000L + (16 - C) * 1000L +
                                   p.stages * 10L + (kNumStagedCfgs - cfg);
                if (score > best_score) {
                    best_score = score;
                    best = p;
                    best.kind = Kind::Staged;
                }
            }
        }
    }
    if ((forced_kind == 1 && best.kind != Kind::Staged) ||
        (forced_kind == 2 && best.kind != Kind::Stream) ||
        (forced_kind == 4 && best.kind != Kind::Reg) ||
        (forced_kind == 5 && (best.kind != Kind::Reg || best.cluster < 2)) ||
        (forced_kind == 6 && best.kind != Kind::Tmem)) {
        g_last_error = "the kernel forced by GBCE_KERNEL cannot run this shape";
        return CE_ERR_UNSUPPORTED;
    }
    if (best.kind == Kind::General) {
        best.fn = generic_kernel(dtype, softcap);
        best.nt = kGenericThreads;
        best.max_units = std::min<int64_t>(static_cast<int64_t>(dev.sm_count) * 8, kMaxUnits);
    }
    // At most 8 partial-sum slots an SM for every plan (a launch takes one
    // slot per CTA of the register kernel, else one per CTA or cluster), so
    // that a launch on a GB300 needs at most 8 * 152 = 1216 slots, whatever
    // the occupancy calculator allows.
    {
        const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
        const int64_t per_unit =
            (best.kind == Kind::Reg || best.kind == Kind::Tmem) ? best.cluster : 1;
        best.max_units = std::max<int64_t>(1, std::min(best.max_units, cap / per_unit));
    }
    if (env_int("GBCE_VERBOSE", 0))
        std::fprintf(stderr,
                     "gbce plan: dtype=%d V=%lld softcap=%d wsmooth=%d -> %s nt=%d C=%d "
                     "stages=%d slice_vec=%d smem=%zu units=%lld ng=%d sg=%d chunk_vec=%d "
                     "nchunk=%d resident=%d\n",
                     dtype, static_cast<long long>(V), softcap ? 1 : 0, wsmooth ? 1 : 0,
                     best.kind == Kind::Stream   ? "stream"
                     : best.kind == Kind::Staged ? "staged"
                     : best.kind == Kind::Reg    ? "reg"
                     : best.kind == Kind::Tmem   ? "tmem"
                                                 : "general",
                     best.nt, best.cluster, best.stages, best.slice_vec, best.smem,
                     static_cast<long long>(best.max_units), best.ng, best.sg, best.chunk_vec,
                     best.nchunk, best.resident);
    g_plans[key] = best;
    *out = best;
    return CE_OK;
}

// pdl: the launch may begin before the previous launch on the stream has
// finished (programmatic dependent launch); the kernel then waits for it
// (griddepcontrol.wait) before reading what it produced.
ce_status launch(const void* fn, int grid, int nt, size_t smem, int cluster, cudaStream_t st,
                 void* arg, bool pdl = false) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(static_cast<unsigned>(grid));
    lc.blockDim = dim3(static_cast<unsigned>(nt));
    lc.dynamicSmemBytes = smem;
    lc.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (na) {
        lc.attrs = attr;
        lc.numAttrs = na;
    }
    void* args[] = {arg};
    cudaError_t e = cudaLaunchKernelExC(&lc, fn, args);
    if (e != cudaSuccess) return cuda_failure(e, "kernel launch");
    return CE_OK;
}

bool finite(float v) { return std::isfinite(v); }

}  // namespace
}  // namespace gbce

using namespace gbce;

namespace gbce {
namespace {

// Argument checks shared by the forward entry points (CE_OK: go on).
ce_status check_fwd(const FwdCall& c) {
    const uint32_t known =
        CE_FLAG_GRAD | CE_FLAG_Z_LOSS | CE_FLAG_ACC | CE_FLAG_PRED | CE_FLAG_TARGET_I64;
    if (c.dtype != CE_F32 && c.dtype != CE_BF16 && c.dtype != CE_F16) return CE_ERR_INVALID_ARG;
    if (c.rows < 0 || c.V <= 0) return CE_ERR_INVALID_ARG;
    if (c.V > INT32_MAX - 16) return CE_ERR_UNSUPPORTED;
    if (c.reduction != CE_RED_NONE && c.reduction != CE_RED_SUM && c.reduction != CE_RED_MEAN)
        return CE_ERR_INVALID_ARG;
    if (c.flags & ~known) return CE_ERR_INVALID_ARG;
    if (!(c.label_smoothing >= 0.f && c.label_smoothing <= 1.f)) return CE_ERR_INVALID_ARG;
    if (!finite(c.lse_square_scale)) return CE_ERR_INVALID_ARG;
    if (!finite(c.softcap) || c.softcap < 0.f) return CE_ERR_INVALID_ARG;
    if (!c.loss) return CE_ERR_INVALID_ARG;
    if ((c.flags & CE_FLAG_Z_LOSS) && !c.z_loss) return CE_ERR_INVALID_ARG;
    if ((c.flags & CE_FLAG_ACC) && !c.acc) return CE_ERR_INVALID_ARG;
    if ((c.flags & CE_FLAG_PRED) && !c.pred) return CE_ERR_INVALID_ARG;
    if (c.rows > 0 && (!c.logits || !c.target)) return CE_ERR_INVALID_ARG;
    if (c.rows > 0 && c.V > INT64_MAX / c.rows / 4) return CE_ERR_INVALID_ARG;
    return CE_OK;
}

// Plans and launches one checked forward call with `scratch`, whose ticket
// is zero on entry or, with clear_header, cleared here.
// A grid that would need more than max_slots partial-sum slots is refused.
// Called with g_mu held.
ce_status run_fwd(int dev, const FwdCall& c, Scratch* scratch, int64_t max_slots,
                  bool clear_header, cudaStream_t st) {
    FwdArgs a = {};
    a.x = c.logits;
    a.rows = c.rows;
    a.V = c.V;
    a.target = c.target;
    a.tgt64 = (c.flags & CE_FLAG_TARGET_I64) ? 1 : 0;
    a.weight = c.weight;
    a.ignore_index = c.ignore_index;
    a.eps = c.label_smoothing;
    a.lam = c.lse_square_scale;
    const bool sc = c.softcap > 0.f;
    a.softcap = sc ? c.softcap : 0.f;
    a.sc_k2 = sc ? 2.f * kLog2e / c.softcap : 0.f;
    a.sc_slog2e = sc ? c.softcap * kLog2e : 0.f;
    a.reduction = c.reduction;
    a.grad = (c.flags & CE_FLAG_GRAD) ? 1 : 0;
    a.want_z = (c.flags & CE_FLAG_Z_LOSS) ? 1 : 0;
    a.want_acc = (c.flags & CE_FLAG_ACC) ? 1 : 0;
    a.want_pred = (c.flags & CE_FLAG_PRED) ? 1 : 0;
    a.loss = c.loss;
    a.zloss = c.z_loss;
    a.acc = c.acc;
    a.pred = c.pred;
    a.timeout_ns = static_cast<uint64_t>(env_int("GBCE_WAIT_TIMEOUT_MS", 2000)) * 1000000ull;
    a.scratch = scratch;
    a.batch_counts = c.batch_counts;
    a.gout = c.gout;
    a.gout_bf16 = c.gout_dtype == CE_BF16 ? 1 : 0;
    // test hook: the streaming and register kernels leave one copy out, so
    // one bounded wait runs out (GBCE_TEST_STALL_COPY=1)
    a.test_stall = env_int("GBCE_TEST_STALL_COPY", 0) != 0 ? 1 : 0;

    const bool wsmooth = c.weight != nullptr && c.label_smoothing > 0.f;
    const bool aligned = (reinterpret_cast<uintptr_t>(c.logits) % 16) == 0;
    const bool w_aligned = (reinterpret_cast<uintptr_t>(c.weight) % 16) == 0;
    Plan p;
    ce_status rc =
        make_plan(dev, c.dtype, c.V, sc, sc && c.softcap <= kTmMaxSoftcap, wsmooth, aligned,
                  w_aligned, &p);
    if (rc != CE_OK) return rc;
    // a separate 16-bit gradient: fp32 logits on the streaming kernel only
    // (nothing launched otherwise; the caller takes the in-place path)
    const void* gout_fn = nullptr;
    if (c.gout) {
        if (c.dtype != CE_F32 || p.kind != Kind::Stream || wsmooth || !(c.flags & CE_FLAG_GRAD) ||
            (reinterpret_cast<uintptr_t>(c.gout) & 7u) ||
            (c.gout_dtype != CE_BF16 && c.gout_dtype != CE_F16))
            return CE_ERR_UNSUPPORTED;
        const int nw = p.nt / 32 - 1;
        gout_fn = stream_kernel_gout(sc, nw == 8 ? 8 : 4, nw);
        if (!gout_fn) return CE_ERR_UNSUPPORTED;
        static std::map<const void*, bool> ready;  // its shared-memory limit set
        if (!ready[gout_fn]) {
            DeviceInfo di;
            rc = device_info(dev, &di);
            if (rc != CE_OK) return rc;
            cudaFuncAttributes fa;
            cudaError_t e = cudaFuncGetAttributes(&fa, gout_fn);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(
                    gout_fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                    static_cast<int>(static_cast<size_t>(di.smem_optin) - fa.sharedSizeBytes));
            if (e != cudaSuccess) return cuda_failure(e, "stream kernel attributes");
            ready[gout_fn] = true;
        }
    }
    const int64_t units = c.rows == 0 ? 1 : std::min<int64_t>(c.rows, p.max_units);
    // the register kernel's clusters: a partial-sum slot for each CTA
    const int64_t slots =
        records_for((p.kind == Kind::Reg || p.kind == Kind::Tmem) && c.rows > 0
                        ? units * p.cluster
                        : units);
    if (slots > max_slots) {
        g_last_error = "this launch needs " + std::to_string(slots) +
                       " partial-sum slots; the scratch holds " + std::to_string(max_slots);
        return CE_ERR_UNSUPPORTED;
    }
    if (clear_header) {
        // the ticket must start at zero (partial slots are written before
        // they are read); the status word stays sticky until it is read
        const cudaError_t e = cudaMemsetAsync(&scratch->ticket, 0, sizeof(unsigned), st);
        if (e != cudaSuccess) return cuda_failure(e, "cudaMemsetAsync(scratch ticket)");
    }
    if (c.rows == 0)  // empty batch: the general kernel with one CTA writes the scalars
        return launch(generic_kernel(c.dtype, sc), 1, kGenericThreads, 0, 1, st, &a);
    if (p.kind == Kind::Stream) {
        a.ng = p.ng;
        a.sg = p.sg;
        a.chunk_vec = p.chunk_vec;
        a.nchunk = p.nchunk;
        a.resident = p.resident;
        return launch(gout_fn ? gout_fn : p.fn, static_cast<int>(units), p.nt, p.smem, 1, st, &a);
    }
    if (p.kind == Kind::Reg) {
        bool pdl = false;
        // D is needed by "mean" (loss and gradient scale), the counted rows
        // by the accuracy of "sum" and "mean"
        const bool need = c.reduction == CE_RED_MEAN ||
                          (c.reduction == CE_RED_SUM && (c.flags & CE_FLAG_ACC));
        if (need && !c.batch_counts) {
            // D and the counted rows by the count kernel, into the scratch
            // header; the forward overlaps it and waits where it needs them
            CountArgs ca = {};
            ca.target = c.target;
            ca.tgt64 = a.tgt64;
            ca.weight = c.weight;
            ca.rows = c.rows;
            ca.V = c.V;
            ca.ignore_index = c.ignore_index;
            ca.counts = scratch->counts;
            ca.scratch = scratch;
            DeviceInfo info;
            ce_status rc2 = device_info(dev, &info);
            if (rc2 != CE_OK) return rc2;
            constexpr int64_t kPerCta = int64_t{kCountThreads} * kCountPerThread;
            const int64_t want = (c.rows + kPerCta - 1) / kPerCta;
            const int64_t cgrid = std::max<int64_t>(1, std::min<int64_t>(want, info.sm_count));
            rc2 = launch(count_kernel(), static_cast<int>(cgrid), kCountThreads, 0, 1, st, &ca);
            if (rc2 != CE_OK) return rc2;
            a.batch_counts = scratch->counts;
            pdl = true;
        }
        a.reg_wpr = p.reg_wpr;
        a.reg_buf_stride = p.reg_buf_stride;
        a.reg_nbuf = p.reg_nbuf;
        a.reg_cluster = p.cluster;
        return launch(p.fn, static_cast<int>(units * p.cluster), p.nt, p.smem, p.cluster, st, &a,
                      pdl);
    }
    if (p.kind == Kind::Tmem) {
        a.tm_slice_vec = p.tm_slice_vec;
        a.tm_slots = p.tm_slots;
        return launch(p.fn, static_cast<int>(units * p.cluster), p.nt, p.smem, p.cluster, st, &a);
    }
    if (p.kind == Kind::Staged) {
        a.slice_vec = p.slice_vec;
        a.stages = p.stages;
        return launch(p.fn, static_cast<int>(units * p.cluster), p.nt, p.smem, p.cluster, st, &a);
    }
    return launch(p.fn, static_cast<int>(units), p.nt, 0, 1, st, &a);
}

// A forward call with the library's scratch for (current device, stream).
ce_status fwd_library_scratch(const FwdCall& c, ce_stream_t stream) {
    ce_status rc = check_fwd(c);
    if (rc != CE_OK) return rc;
    if (c.rows == 0 && c.reduction == CE_RED_NONE) return CE_OK;  // nothing to write
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_failure(e, "cudaGetDevice");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Scratch* scratch = nullptr;
    rc = scratch_for(dev, st, &scratch);
    if (rc != CE_OK) return rc;
    return run_fwd(dev, c, scratch, kMaxPartials, false, st);
}

}  // namespace

// A shard's forward (ce_fwd_shard) whose gradient goes to gout in bf16 or
// fp16 (gout_dtype) while the fp32 logits stay as they were: the fused
// linear cross-entropy's G without a separate rounding pass.
// CE_ERR_UNSUPPORTED, with nothing launched, when the plan is not the
// streaming kernel.
ce_status fwd_shard_gout(const FwdCall& c, void* gout, int gout_dtype, ce_stream_t stream) {
    if (!c.batch_counts || !gout) return CE_ERR_INVALID_ARG;
    FwdCall g = c;
    g.gout = gout;
    g.gout_dtype = gout_dtype;
    return fwd_library_scratch(g, stream);
}

// The forward call with scratch that the caller provides (the static-scratch
// entry point in ce_noalloc.cu): same checks, plan and launch as ce_fwd, the
// scratch header cleared first; allocates nothing.
ce_status fwd_with_scratch(Scratch* scratch, int max_slots, const FwdCall& c, cudaStream_t st) {
    if (!scratch || max_slots < 1) return CE_ERR_INVALID_ARG;
    ce_status rc = check_fwd(c);
    if (rc != CE_OK) return rc;
    if (c.rows == 0 && c.reduction == CE_RED_NONE) return CE_OK;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_failure(e, "cudaGetDevice");
    return run_fwd(dev, c, scratch, max_slots, true, st);
}

// Records a CUDA error for ce_last_error (for the static-scratch entry point).
ce_status record_cuda_failure(cudaError_t e, const char* what) { return cuda_failure(e, what); }

// Records a message for ce_last_error.
void record_message(const std::string& msg) { g_last_error = msg; }

// The device status word of the library scratch of (current device, stream)
// (allocated on first use, like every other call's scratch).
ce_status library_status_word(cudaStream_t st, unsigned** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_failure(e, "cudaGetDevice");
    Scratch* scratch = nullptr;
    const ce_status rc = scratch_for(dev, st, &scratch);
    if (rc != CE_OK) return rc;
    *out = &scratch->status;
    return CE_OK;
}

}  // namespace gbce

extern "C" ce_status ce_fwd(void* logits, int dtype, int64_t rows, int64_t V, const void* target,
                            const float* weight, int64_t ignore_index, float label_smoothing,
                            float lse_square_scale, float softcap, int reduction, uint32_t flags,
                            float* loss, float* z_loss, float* acc, int64_t* pred,
                            ce_stream_t stream) {
    const FwdCall c{logits, dtype, rows, V, target, weight, ignore_index, label_smoothing,
                    lse_square_scale, softcap, reduction, flags, loss, z_loss, acc, pred, nullptr};
    return fwd_library_scratch(c, stream);
}

extern "C" ce_status ce_fwd_shard(void* logits, int dtype, int64_t rows, int64_t V,
                                  const void* target, const float* weight, int64_t ignore_index,
                                  float label_smoothing, float lse_square_scale, float softcap,
                                  int reduction, uint32_t flags, float* loss, float* z_loss,
                                  float* acc, int64_t* pred, const double* batch_counts,
                                  ce_stream_t stream) {
    if (!batch_counts) return CE_ERR_INVALID_ARG;
    const FwdCall c{logits, dtype, rows, V, target, weight, ignore_index, label_smoothing,
                    lse_square_scale, softcap, reduction, flags, loss, z_loss, acc, pred,
                    batch_counts};
    return fwd_library_scratch(c, stream);
}

extern "C" ce_status ce_count(const void* target, const float* weight, int64_t rows, int64_t V,
                              int64_t ignore_index, uint32_t flags, double* counts,
                              ce_stream_t stream) {
    if (rows < 0 || V <= 0 || !counts) return CE_ERR_INVALID_ARG;
    if (flags & ~static_cast<uint32_t>(CE_FLAG_TARGET_I64)) return CE_ERR_INVALID_ARG;
    if (rows > 0 && !target) return CE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_failure(e, "cudaGetDevice");
    DeviceInfo info;
    ce_status rc = device_info(dev, &info);
    if (rc != CE_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Scratch* scratch = nullptr;
    rc = scratch_for(dev, st, &scratch);
    if (rc != CE_OK) return rc;
    CountArgs a = {};
    a.target = target;
    a.tgt64 = (flags & CE_FLAG_TARGET_I64) ? 1 : 0;
    a.weight = weight;
    a.rows = rows;
    a.V = V;
    a.ignore_index = ignore_index;
    a.counts = counts;
    a.scratch = scratch;
    constexpr int64_t kPerCta = int64_t{kCountThreads} * kCountPerThread;
    const int64_t want = (rows + kPerCta - 1) / kPerCta;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(want, info.sm_count));
    return launch(count_kernel(), static_cast<int>(grid), kCountThreads, 0, 1, st, &a);
}

// ---------------------------------------------------------------- unfused (aten-shaped) ops

namespace gbce {
namespace {

bool dtype_ok(int dtype) { return dtype == CE_F32 || dtype == CE_BF16 || dtype == CE_F16; }
int64_t dtype_bytes(int dtype) { return dtype == CE_F32 ? 4 : 2; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by the unfused entry points.
ce_status check_rows_c(int dtype, int64_t rows, int64_t C) {
    if (!dtype_ok(dtype) || rows < 0 || C <= 0) return CE_ERR_INVALID_ARG;
    if (C > INT32_MAX - 16) return CE_ERR_UNSUPPORTED;
    if (rows > 0 && C > INT64_MAX / rows / 4) return CE_ERR_INVALID_ARG;
    return CE_OK;
}

// The current device, its properties and the (device, stream) scratch.
// Called with g_mu held.
ce_status device_and_scratch(cudaStream_t st, int* dev, DeviceInfo* info, Scratch** scratch) {
    const cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_failure(e, "cudaGetDevice");
    ce_status rc = device_info(*dev, info);
    if (rc != CE_OK) return rc;
    return scratch_for(*dev, st, scratch);
}

std::map<std::tuple<int, int, int64_t, std::string>, Plan> g_lsm_plans;

}  // namespace
}  // namespace gbce

extern "C" ce_status ce_log_softmax(const void* x, void* out, int dtype, int64_t rows, int64_t C,
                                    ce_stream_t stream) {
    ce_status rc = check_rows_c(dtype, rows, C);
    if (rc != CE_OK) return rc;
    if (rows > 0 && (!x || !out)) return CE_ERR_INVALID_ARG;
    if (rows == 0) return CE_OK;
    std::lock_guard<std::mutex> lock(g_mu);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0;
    DeviceInfo info;
    Scratch* scratch = nullptr;
    rc = device_and_scratch(st, &dev, &info, &scratch);
    if (rc != CE_OK) return rc;
    if (aligned16(x) && aligned16(out) && (C * dtype_bytes(dtype)) % 16 == 0) {
        const auto key = std::make_tuple(dev, dtype, C, tuning_signature());
        auto it = g_lsm_plans.find(key);
        if (it == g_lsm_plans.end()) {
            Plan p;
            rc = CE_OK;
            if (!try_stream(dtype, C, false, false, info, &p, &rc, true)) {
                if (rc != CE_OK) return rc;
                p = Plan();  // no streaming plan: the general kernel below
            }
            it = g_lsm_plans.emplace(key, p).first;
        }
        const Plan& p = it->second;
        if (p.kind == Kind::Stream) {
            FwdArgs a = {};
            a.x = const_cast<void*>(x);
            a.out = out;
            a.rows = rows;
            a.V = C;
            a.ignore_index = INT64_MIN;
            a.reduction = CE_RED_NONE;
            a.timeout_ns =
                static_cast<uint64_t>(env_int("GBCE_WAIT_TIMEOUT_MS", 2000)) * 1000000ull;
            a.scratch = scratch;
            a.ng = p.ng;
            a.sg = p.sg;
            a.chunk_vec = p.chunk_vec;
            a.nchunk = p.nchunk;
            a.resident = p.resident;
            const int64_t units = std::min<int64_t>(rows, p.max_units);
            return launch(p.fn, static_cast<int>(units), p.nt, p.smem, 1, st, &a);
        }
    }
    LsmArgs la = {x, out, rows, C};
    const int64_t grid = std::min<int64_t>(rows, static_cast<int64_t>(info.sm_count) * 4);
    return launch(lsm_generic_kernel(dtype), static_cast<int>(grid), kLsmGenericThreads, 0, 1, st,
                  &la);
}

extern "C" ce_status ce_nll_loss_fwd(const void* logp, int dtype, int64_t rows, int64_t C,
                                     const void* target, const float* weight,
                                     int64_t ignore_index, int reduction, uint32_t flags,
                                     float* out, float* total_weight, ce_stream_t stream) {
    ce_status rc = check_rows_c(dtype, rows, C);
    if (rc != CE_OK) return rc;
    if (reduction != CE_RED_NONE && reduction != CE_RED_SUM && reduction != CE_RED_MEAN)
        return CE_ERR_INVALID_ARG;
    if (flags & ~static_cast<uint32_t>(CE_FLAG_TARGET_I64)) return CE_ERR_INVALID_ARG;
    if (!out || !total_weight) return CE_ERR_INVALID_ARG;
    if (rows > 0 && (!logp || !target)) return CE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0;
    DeviceInfo info;
    Scratch* scratch = nullptr;
    rc = device_and_scratch(st, &dev, &info, &scratch);
    if (rc != CE_OK) return rc;
    NllFwdArgs a = {};
    a.logp = logp;
    a.target = target;
    a.tgt64 = (flags & CE_FLAG_TARGET_I64) ? 1 : 0;
    a.weight = weight;
    a.rows = rows;
    a.C = C;
    a.ignore_index = ignore_index;
    a.reduction = reduction;
    a.out = out;
    a.total_weight = total_weight;
    a.scratch = scratch;
    const int64_t want = (rows + kNllThreads - 1) / kNllThreads;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(want, info.sm_count));
    return launch(nll_fwd_kernel(dtype), static_cast<int>(grid), kNllThreads, 0, 1, st, &a);
}

extern "C" ce_status ce_nll_loss_bwd(const float* grad_output, const float* total_weight,
                                     void* grad_input, int dtype, int64_t rows, int64_t C,
                                     const void* target, const float* weight,
                                     int64_t ignore_index, int reduction, uint32_t flags,
                                     ce_stream_t stream) {
    ce_status rc = check_rows_c(dtype, rows, C);
    if (rc != CE_OK) return rc;
    if (reduction != CE_RED_NONE && reduction != CE_RED_SUM && reduction != CE_RED_MEAN)
        return CE_ERR_INVALID_ARG;
    if (flags & ~static_cast<uint32_t>(CE_FLAG_TARGET_I64)) return CE_ERR_INVALID_ARG;
    if (rows > 0 && (!grad_output || !grad_input || !target)) return CE_ERR_INVALID_ARG;
    if (rows > 0 && reduction == CE_RED_MEAN && !total_weight) return CE_ERR_INVALID_ARG;
    if (rows == 0) return CE_OK;
    std::lock_guard<std::mutex> lock(g_mu);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0;
    DeviceInfo info;
    Scratch* scratch = nullptr;
    rc = device_and_scratch(st, &dev, &info, &scratch);
    if (rc != CE_OK) return rc;
    NllBwdArgs a = {};
    a.grad_output = grad_output;
    a.total_weight = total_weight;
    a.grad_input = grad_input;
    a.target = target;
    a.tgt64 = (flags & CE_FLAG_TARGET_I64) ? 1 : 0;
    a.weight = weight;
    a.rows = rows;
    a.C = C;
    a.ignore_index = ignore_index;
    a.reduction = reduction;
    a.vec_ok = (aligned16(grad_input) && (C * dtype_bytes(dtype)) % 16 == 0) ? 1 : 0;
    a.scratch = scratch;
    const int64_t grid = std::min<int64_t>(rows, static_cast<int64_t>(info.sm_count) * 8);
    return launch(nll_bwd_kernel(dtype), static_cast<int>(grid), kNllThreads, 0, 1, st, &a);
}

extern "C" ce_status ce_log_softmax_bwd(const void* grad_output, const void* output,
                                        void* grad_input, int dtype, int64_t rows, int64_t C,
                                        ce_stream_t stream) {
    ce_status rc = check_rows_c(dtype, rows, C);
    if (rc != CE_OK) return rc;
    if (rows > 0 && (!grad_output || !output || !grad_input)) return CE_ERR_INVALID_ARG;
    if (rows == 0) return CE_OK;
    std::lock_guard<std::mutex> lock(g_mu);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_failure(e, "cudaGetDevice");
    DeviceInfo info;
    rc = device_info(dev, &info);
    if (rc != CE_OK) return rc;
    LsmBwdArgs a = {};
    a.dy = grad_output;
    a.y = output;
    a.dx = grad_input;
    a.rows = rows;
    a.C = C;
    a.vec_ok = (aligned16(grad_output) && aligned16(output) && aligned16(grad_input) &&
                (C * dtype_bytes(dtype)) % 16 == 0) ? 1 : 0;
    const int64_t grid = std::min<int64_t>(rows, info.sm_count);
    return launch(lsm_bwd_kernel(dtype), static_cast<int>(grid), kLsmBwdThreads, 0, 1, st, &a);
}

extern "C" ce_status ce_bwd(const float* grad_output, int grad_per_row, void* dlogits, int dtype,
                            int64_t rows, int64_t V, ce_stream_t stream) {
    if (dtype != CE_F32 && dtype != CE_BF16 && dtype != CE_F16) return CE_ERR_INVALID_ARG;
    if (rows < 0 || V <= 0) return CE_ERR_INVALID_ARG;
    if (rows > 0 && (!grad_output || !dlogits)) return CE_ERR_INVALID_ARG;
    if (rows > 0 && V > INT64_MAX / rows / 4) return CE_ERR_INVALID_ARG;
    if (rows == 0) return CE_OK;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_failure(e, "cudaGetDevice");
    DeviceInfo info;
    ce_status rc = device_info(dev, &info);
    if (rc != CE_OK) return rc;
    const int64_t bytes = dtype == CE_F32 ? 4 : 2;
    BwdArgs b = {};
    b.g = grad_output;
    b.per_row = grad_per_row ? 1 : 0;
    b.x = dlogits;
    b.rows = rows;
    b.V = V;
    b.vec_ok = ((V * bytes) % 16 == 0 && reinterpret_cast<uintptr_t>(dlogits) % 16 == 0) ? 1 : 0;
    const int64_t grid = std::min<int64_t>(rows, static_cast<int64_t>(info.sm_count) * 8);
    return launch(bwd_kernel(dtype), static_cast<int>(grid), kBwdThreads, 0, 1,
                  reinterpret_cast<cudaStream_t>(stream), &b, true);
}

extern "C" ce_status ce_device_status(ce_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_failure(e, "cudaStreamSynchronize");
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_failure(e, "cudaGetDevice");
    auto it = g_scratch.find(std::make_pair(dev, reinterpret_cast<uintptr_t>(st)));
    if (it == g_scratch.end()) return CE_OK;
    unsigned status = 0;
    e = cudaMemcpyAsync(&status, &it->second->status, sizeof status, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(&it->second->status, 0, sizeof status, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_failure(e, "reading the device status");
    if (status & kDevErrTimeout) return CE_ERR_TIMEOUT;
    if (status & kDevErrTarget) return CE_ERR_TARGET_RANGE;
    return CE_OK;
}

extern "C" const char* ce_status_string(ce_status s) {
    switch (s) {
    case CE_OK: return "ok";
    case CE_ERR_INVALID_ARG: return "invalid argument";
    case CE_ERR_UNSUPPORTED: return "unsupported argument combination";
    case CE_ERR_CUDA: return "CUDA runtime error";
    case CE_ERR_TARGET_RANGE: return "target index outside [0, V) that is not ignore_index";
    case CE_ERR_TIMEOUT: return "bounded device wait timed out";
    }
    return "unknown status";
}

extern "C" const char* ce_last_error(void) { return g_last_error.c_str(); }

extern "C" int64_t ce_scratch_areas(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    return static_cast<int64_t>(g_scratch.size());
}

// ---------------------------------------------------------------- N-D logits (class dimension 1)

namespace gbce {
namespace {

// Tile layout of the N-D forward: 16-byte vectors of positions or single
// positions, the tile of 32 * VP positions x C classes in shared memory or
// read again from global memory (L2) by phases B and C.
struct NdPlan {
    const void* fn = nullptr;
    bool vec = false;
    bool staged = false;
    size_t smem = 0;
    int64_t max_ctas = 0;
};

std::map<std::tuple<int, int, int64_t, bool, bool, bool, int>, NdPlan> g_nd_plans;

// GBCE_ND_MODE forces a layout: 1 vector staged, 2 vector from global,
// 3 scalar staged, 4 scalar from global (0: automatic). Automatic takes the
// first that fits in this order: vector staged, scalar staged, scalar from
// global; a staged tile may use up to half of an SM's shared memory less
// the fixed part, so two CTAs fit on an SM.
ce_status nd_plan(int dev, const DeviceInfo& info, int dtype, int64_t C, bool vec_ok, bool softcap,
                  bool argmax, NdPlan* out) {
    const int mode = env_int("GBCE_ND_MODE", 0);
    const auto key = std::make_tuple(dev, dtype, C, vec_ok, softcap, argmax, mode);
    auto it = g_nd_plans.find(key);
    if (it != g_nd_plans.end()) {
        *out = it->second;
        return CE_OK;
    }
    const int64_t b = dtype == CE_F32 ? 4 : 2;
    const size_t fixed_vec = nd_fixed_smem(32 * static_cast<int>(16 / b));
    const size_t fixed_one = nd_fixed_smem(32);
    const int64_t tile_vec = C * 32 * 16;
    const int64_t tile_one = C * 32 * b;
    const int64_t half_sm = info.smem_per_sm / 2 - 1024;  // the runtime reserves 1 KB a CTA
    const int64_t cap = info.smem_optin;
    bool vec = false, staged = false;
    switch (mode) {
    case 1: vec = true; staged = true; break;
    case 2: vec = true; break;
    case 3: staged = true; break;
    case 4: break;
    default:
        if (vec_ok && static_cast<int64_t>(fixed_vec) + tile_vec <= half_sm) {
            vec = true;
            staged = true;
        } else if (static_cast<int64_t>(fixed_one) + tile_one <= half_sm) {
            staged = true;
        }
    }
    NdPlan p;
    p.vec = vec;
    p.staged = staged;
    p.smem = (vec ? fixed_vec : fixed_one) + (staged ? (vec ? tile_vec : tile_one) : 0);
    if ((vec && !vec_ok) || static_cast<int64_t>(p.smem) > cap) {
        g_last_error = "the N-D layout forced by GBCE_ND_MODE cannot run this shape";
        return CE_ERR_UNSUPPORTED;
    }
    p.fn = nd_kernel(dtype, vec, softcap, argmax);
    if (!p.fn) return CE_ERR_INVALID_ARG;
    // the largest dynamic size the kernel can take, set once for every plan
    // that uses it (a smaller value would refuse the larger plans' launches)
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, p.fn);
    if (e != cudaSuccess) return cuda_failure(e, "cudaFuncGetAttributes");
    const size_t max_dyn = static_cast<size_t>(cap) - fa.sharedSizeBytes;
    if (p.smem > max_dyn) {
        g_last_error = "the N-D tile does not fit in shared memory";
        return CE_ERR_UNSUPPORTED;
    }
    e = cudaFuncSetAttribute(p.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(max_dyn));
    if (e != cudaSuccess) return cuda_failure(e, "cudaFuncSetAttribute");
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, p.fn, kNdThreads, p.smem);
    if (e != cudaSuccess) return cuda_failure(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (occ < 1) {
        g_last_error = "the N-D kernel does not fit on an SM";
        return CE_ERR_UNSUPPORTED;
    }
    p.max_ctas = static_cast<int64_t>(occ) * info.sm_count;
    g_nd_plans[key] = p;
    *out = p;
    return CE_OK;
}

// Occupancy (CTAs an SM) of an N-D kernel of 256 threads with `smem`
// bytes of dynamic shared memory; the kernel's limit is raised to
// `smem_max` on its first use. Computed once for each (kernel, smem).
int nd_split_occ(const void* fn, size_t smem, size_t smem_max = 0) {
    static std::map<std::pair<const void*, size_t>, int> occ;
    static std::map<const void*, size_t> limit;
    const auto key = std::make_pair(fn, smem);
    auto it = occ.find(key);
    if (it != occ.end()) return it->second;
    int o = 0;
    cudaError_t e = cudaSuccess;
    const size_t want = std::max(smem, smem_max);
    if (limit[fn] < want) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(want));
        if (e == cudaSuccess) limit[fn] = want;
    }
    if (e != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, fn, kNdSplitThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        o = 0;
    }
    occ[key] = o;
    return o;
}

// The split N-D forward (ce_fwd_nd_split.cuh): class chunks of cc classes
// so that the (tile, chunk) items fill GBCE_ND_ITEMS (default 1) waves of
// resident statistics CTAs without starting another, with at least
// GBCE_ND_MIN_CHUNK (default 64) classes a chunk; the records, coefficients
// and counted targets in the stream's N-D workspace.
ce_status nd_split_launch(int dev, const DeviceInfo& info, const FwdArgs& f, int dtype,
                          bool vec_ok, bool softcap, bool argmax, bool after_count,
                          cudaStream_t st) {
    const int64_t b = dtype == CE_F32 ? 4 : 2;
    const int64_t VP = vec_ok ? 16 / b : 1;
    const int64_t P = 32 * VP;
    const int64_t C = f.V;
    NdSplitArgs s = {};
    s.f = f;
    s.tiles = (f.rows + P - 1) / P;
    const NdSplitFns fns = nd_split_fns(dtype, vec_ok, softcap, argmax, f.eps > 0.f);
    if (!fns.stats || !fns.merge || !fns.grad) return CE_ERR_INVALID_ARG;
    const int o1 = nd_split_occ(fns.stats, fns.stats_smem);
    const int o3 = nd_split_occ(fns.grad, 0);
    if (o1 < 1 || o3 < 1) {
        g_last_error = "the split N-D kernels do not fit on an SM";
        return CE_ERR_UNSUPPORTED;
    }
    // as many chunks a tile as keep the items within one wave of resident
    // statistics CTAs (GBCE_ND_ITEMS waves; a partial second wave doubled
    // the launch: 320 items on 304 CTAs at 8 x 4096 x 1024)
    const int64_t want = std::max(1, env_int("GBCE_ND_ITEMS", 1)) * static_cast<int64_t>(o1) *
                         static_cast<int64_t>(info.sm_count);
    const int64_t max_ch = std::max<int64_t>(1, C / std::max(8, env_int("GBCE_ND_MIN_CHUNK", 64)));
    const int64_t nch0 = std::min<int64_t>(max_ch, std::max<int64_t>(1, want / s.tiles));
    const int64_t cc = (C + nch0 - 1) / nch0;
    s.cc = static_cast<int>(cc);
    s.nch = static_cast<int>((C + cc - 1) / cc);
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    const size_t rec_b = up(static_cast<size_t>(s.tiles * P) * s.nch * sizeof(NdRec));
    const size_t coef_b = up(static_cast<size_t>(f.rows) * sizeof(NdCoef));
    const size_t tpos_b = up(static_cast<size_t>(f.rows) * sizeof(int));
    void* ws = nullptr;
    ce_status rc = nd_work_for(dev, st, rec_b + coef_b + tpos_b, &ws);
    if (rc != CE_OK) return rc;
    s.rec = static_cast<NdRec*>(ws);
    s.coef = reinterpret_cast<NdCoef*>(static_cast<char*>(ws) + rec_b);
    s.tpos = reinterpret_cast<int*>(static_cast<char*>(ws) + rec_b + coef_b);
    const int64_t items = s.tiles * s.nch;
    const int64_t g1 = std::min<int64_t>(items, o1 * static_cast<int64_t>(info.sm_count));
    // the statistics overlap the count kernel before them (they do not read
    // its counts; the merge does, launched after both)
    rc = launch(fns.stats, static_cast<int>(g1), kNdSplitThreads, fns.stats_smem, 1, st, &s,
                after_count);
    if (rc != CE_OK) return rc;
    // one warp a position; the merge's CTAs take the partial-sum slots
    const int64_t g2 = std::max<int64_t>(
        1, std::min<int64_t>((f.rows + 7) / 8, std::min<int64_t>(8 * static_cast<int64_t>(info.sm_count),
                                                                 kMaxUnits)));
    rc = launch(fns.merge, static_cast<int>(g2), kNdSplitThreads, 0, 1, st, &s);
    if (rc != CE_OK || !f.grad) return rc;
    const int64_t g3 = std::min<int64_t>(items, o3 * static_cast<int64_t>(info.sm_count));
    return launch(fns.grad, static_cast<int>(g3), kNdSplitThreads, 0, 1, st, &s);
}

}  // namespace
}  // namespace gbce

extern "C" ce_status ce_fwd_nd(void* logits, int dtype, int64_t N, int64_t C, int64_t inner,
                               const void* target, const float* weight, int64_t ignore_index,
                               float label_smoothing, float lse_square_scale, float softcap,
                               int reduction, uint32_t flags, float* loss, float* z_loss,
                               float* acc, int64_t* pred, ce_stream_t stream) {
    if (N < 0 || C <= 0 || inner < 0) return CE_ERR_INVALID_ARG;
    if (inner > 0 && N > INT64_MAX / inner) return CE_ERR_INVALID_ARG;
    const int64_t rows = N * inner;
    const FwdCall c{logits, dtype, rows, C, target, weight, ignore_index, label_smoothing,
                    lse_square_scale, softcap, reduction, flags, loss, z_loss, acc, pred, nullptr};
    ce_status rc = check_fwd(c);
    if (rc != CE_OK) return rc;
    // one class dimension with nothing after it is the 2-D layout; so is an
    // empty batch (which writes only the reduced scalars)
    if (inner == 1 || rows == 0) return fwd_library_scratch(c, stream);
    if (rows > INT32_MAX) return CE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0;
    DeviceInfo info;
    Scratch* scratch = nullptr;
    rc = device_and_scratch(st, &dev, &info, &scratch);
    if (rc != CE_OK) return rc;
    const int64_t b = dtype == CE_F32 ? 4 : 2;
    const bool vec_ok = aligned16(logits) && inner % (16 / b) == 0;
    const bool sc = softcap > 0.f;
    const bool argmax = (flags & (CE_FLAG_ACC | CE_FLAG_PRED)) != 0;
    NdPlan p;
    rc = nd_plan(dev, info, dtype, C, vec_ok, sc, argmax, &p);
    if (rc != CE_OK) return rc;
    if (reduction != CE_RED_NONE) {
        // D and the counted positions first: the gradient's mean scale needs
        // them before any position is finished
        CountArgs ca = {};
        ca.target = target;
        ca.tgt64 = (flags & CE_FLAG_TARGET_I64) ? 1 : 0;
        ca.weight = weight;
        ca.rows = rows;
        ca.V = C;
        ca.ignore_index = ignore_index;
        ca.counts = scratch->counts;
        ca.scratch = scratch;
        constexpr int64_t kPerCta = int64_t{kCountThreads} * kCountPerThread;
        const int64_t want = (rows + kPerCta - 1) / kPerCta;
        const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(want, info.sm_count));
        rc = launch(count_kernel(), static_cast<int>(grid), kCountThreads, 0, 1, st, &ca);
        if (rc != CE_OK) return rc;
    }
    FwdArgs a = {};
    a.x = logits;
    a.rows = rows;
    a.V = C;
    a.target = target;
    a.tgt64 = (flags & CE_FLAG_TARGET_I64) ? 1 : 0;
    a.weight = weight;
    a.ignore_index = ignore_index;
    a.eps = label_smoothing;
    a.lam = lse_square_scale;
    a.softcap = sc ? softcap : 0.f;
    a.sc_k2 = sc ? 2.f * kLog2e / softcap : 0.f;
    a.sc_slog2e = sc ? softcap * kLog2e : 0.f;
    a.reduction = reduction;
    a.grad = (flags & CE_FLAG_GRAD) ? 1 : 0;
    a.want_z = (flags & CE_FLAG_Z_LOSS) ? 1 : 0;
    a.want_acc = (flags & CE_FLAG_ACC) ? 1 : 0;
    a.want_pred = (flags & CE_FLAG_PRED) ? 1 : 0;
    a.loss = loss;
    a.zloss = z_loss;
    a.acc = acc;
    a.pred = pred;
    a.scratch = scratch;
    a.batch_counts = reduction != CE_RED_NONE ? scratch->counts : nullptr;
    a.inner = inner;
    a.timeout_ns = static_cast<uint64_t>(env_int("GBCE_WAIT_TIMEOUT_MS", 2000)) * 1000000ull;
    a.nd_staged = p.staged ? 1 : 0;
    const int64_t P = p.vec ? 32 * (16 / b) : 32;
    const int64_t tiles = (rows + P - 1) / P;
    // The single-kernel form reads a staged tile once, but runs one CTA a
    // tile of every class; when its tile does not fit on chip (it would read
    // the logits three times), there are very few tiles for the SMs (fewer
    // than one for every two SMs; at 256 tiles of 16 x C x 4096 bf16 it was
    // still faster: 23 against 61 us for C = 64, even at 256 and 512), or
    // the classes are many (its serial pass over them then costs more than
    // the split form's second read: 163 against 136 us for C = 1000, 199
    // against 124 for 4 x 2000 x 8192), the split form takes the call
    // (GBCE_ND_SPLIT=0 / 1 forces one or the other)
    const int split_env = env_int("GBCE_ND_SPLIT", -1);
    // The single-read tile kernel (a cluster holds a tile's classes in
    // shared memory), no softcap and no class-weighted smoothing: by default
    // from kNdTileMinClasses classes where one or two CTAs hold a tile's
    // classes in 128-byte rows, the range where it measured faster (bf16,
    // mean: 16 x 512 x 4096 69.9 against 80.3 us for the staged kernel,
    // 16 x 1000 x 4096 98.4 against 135.9 for the split form, 4 x 2000 x
    // 8192 111.8 against 124.6; at 256 classes 55.2 against 52.6, with four
    // CTAs a tile, 8 x 4096 x 1024, 71.4 against 70.4, with sixteen,
    // 8 x 32000 x 512, 445 against 171). GBCE_ND_TILE=0 turns it off, 2
    // takes it for any class count and cluster size.
    const int tile_env = env_int("GBCE_ND_TILE", 1);
    if (tile_env != 0 && !sc && !(weight && label_smoothing > 0.f) &&
        (tile_env == 2 || C >= kNdTileMinClasses) && env_int("GBCE_ND_MODE", 0) == 0 &&
        split_env < 0) {
        rc = nd_tile_launch(a, dtype, N, C, inner, info.sm_count, info.smem_optin,
                            tile_env == 2 ? 16 : 2, tile_env == 2, reduction != CE_RED_NONE, st);
        if (rc != CE_ERR_UNSUPPORTED) return rc;
    }
    const bool split =
        split_env == 1 || (split_env != 0 && env_int("GBCE_ND_MODE", 0) == 0 &&
                           (!p.staged || 2 * tiles < info.sm_count || C >= kNdSplitMinClasses));
    // Few classes with vector positions and enough tiles: a warp a tile
    // (no CTA barrier between its phases; GBCE_ND_WARP=0 turns it off, 2
    // takes it whatever the tile count)
    const int warp_env = env_int("GBCE_ND_WARP", 1);
    if ((warp_env == 2 || (!split && warp_env == 1 && tiles >= 2 * info.sm_count)) && vec_ok &&
        C <= kNdWarpClasses && env_int("GBCE_ND_MODE", 0) == 0 && split_env != 1) {
        const void* fn = nd_warp_kernel(dtype, sc, argmax);
        if (!fn) return CE_ERR_INVALID_ARG;
        const size_t smem = static_cast<size_t>(8) * C * 512;
        const int occ = nd_split_occ(fn, smem, static_cast<size_t>(8) * kNdWarpClasses * 512);
        if (occ >= 1) {
            const int64_t grid = std::min<int64_t>((tiles + 7) / 8,
                                                   std::min<int64_t>(occ * int64_t{info.sm_count}, kMaxUnits));
            return launch(fn, static_cast<int>(grid), 256, smem, 1, st, &a,
                          reduction != CE_RED_NONE);
        }
    }
    if (split)
        return nd_split_launch(dev, info, a, dtype, vec_ok, sc, argmax, reduction != CE_RED_NONE,
                               st);
    const int64_t grid = std::min<int64_t>(tiles, std::min<int64_t>(p.max_ctas, kMaxUnits));
    return launch(p.fn, static_cast<int>(grid), kNdThreads, p.smem, 1, st, &a);
}

extern "C" ce_status ce_bwd_nd(const float* grad_output, int grad_per_position, void* dlogits,
                               int dtype, int64_t N, int64_t C, int64_t inner,
                               ce_stream_t stream) {
    if (dtype != CE_F32 && dtype != CE_BF16 && dtype != CE_F16) return CE_ERR_INVALID_ARG;
    if (N < 0 || C <= 0 || inner < 0) return CE_ERR_INVALID_ARG;
    if (N > 0 && inner > 0 && (C > INT64_MAX / N / inner / 4)) return CE_ERR_INVALID_ARG;
    if (N == 0 || inner == 0) return CE_OK;
    if (!grad_output || !dlogits) return CE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_failure(e, "cudaGetDevice");
    DeviceInfo info;
    ce_status rc = device_info(dev, &info);
    if (rc != CE_OK) return rc;
    const int64_t b = dtype == CE_F32 ? 4 : 2;
    NdBwdArgs a = {};
    a.g = grad_output;
    a.per_pos = grad_per_position ? 1 : 0;
    a.x = dlogits;
    a.N = N;
    a.C = C;
    a.inner = inner;
    a.vec_ok = (aligned16(dlogits) && (inner * b) % 16 == 0) ? 1 : 0;
    int64_t grid;
    if (a.per_pos)
        grid = std::min<int64_t>(N * C, static_cast<int64_t>(info.sm_count) * 8);
    else
        grid = std::max<int64_t>(1, std::min<int64_t>((N * C * inner + 2047) / 2048,
                                                     static_cast<int64_t>(info.sm_count) * 8));
    return launch(nd_bwd_kernel(dtype), static_cast<int>(grid), kBwdThreads, 0, 1,
                  reinterpret_cast<cudaStream_t>(stream), &a, true);
}
