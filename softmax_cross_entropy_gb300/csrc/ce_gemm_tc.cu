// Tensor-core GEMMs of the fused linear cross-entropy (the Liger-Kernel
// cross-entropy kernel profile, §Classification: the closest existing
// kernel is the fused linear cross-entropy, whose logits are hidden @
// lm_head^T) on the fifth-generation tensor cores: C[M, N] = A[M, K] @
// B[K, N] with A and B bf16 or fp16, each operand stored either K-major
// (rows of K contiguous elements:
// A as [M, K], B as [N, K]) or MN-major (A as [K, M], B as [K, N]); C fp32
// written, fp32 added to, or rounded to the operand type (+ bias[N] for the
// fp32 store). The three GEMMs of ce_flce are the three layouts: logits =
// hidden @ W^T (both K-major), grad_hidden = G @ W (B MN-major, 16-bit out),
// grad_weight += G^T @ hidden (both MN-major, fp32 accumulate).
//
// A persistent kernel, one CTA an SM, warp-specialised (6 warps), on tiles
// of 128 or 256 rows x 256 columns (TcTile):
//  * warp 0, lane 0: TMA producer. It walks the CTA's tiles (tile t of the
//    launch goes to CTA t mod grid; consecutive tiles share a tile of the
//    larger operand through L2) and their 64-deep K blocks, and fills a
//    3- or 4-stage shared-memory ring with 2-D TMA copies (128-byte
//    swizzle): one box a K-major operand tile, or boxes of 64 MN elements x
//    64 K rows side by side for an MN-major one;
//  * warp 1, lane 0: MMA issuer. tcgen05.mma (M 128, N 256, K 16, fp32
//    accumulation, one a 128-row half) into tensor memory (512 columns: two
//    256-column accumulators used by turns for 128-row tiles, the two
//    halves of one for 256-row tiles), freeing each stage with
//    tcgen05.commit on its `empty` mbarrier and handing the finished tile
//    to the epilogue with a commit on its `acc_full` mbarrier;
//  * warps 2-5: epilogue. Each reads its 32 accumulator rows of each half
//    (tcgen05.ld), stages them in shared memory and hands them to TMA
//    stores (or reduce-adds), then frees the accumulator (`acc_empty`, 128
//    arrivals); with two accumulators this overlaps the next tile's MMAs.
// Every mbarrier wait is bounded; a wait that gives up records the timeout
// in the status word and sets the launch's abort word, the kernel waits
// (bounded) for its copies in flight, frees its tensor memory and returns.
#include <cuda.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <type_traits>

#include "ce_kernels.cuh"
#include "gbce.h"

namespace gbce {
ce_status record_cuda_failure(cudaError_t e, const char* what);
void record_message(const std::string& msg);
ce_status library_status_word(cudaStream_t st, unsigned** out);

namespace {

// Tiles of BM x 256 (BM = 128 or 256) with K blocks of 64, one CTA an SM:
//  * BM = 128: 4 stages of 128 x 64 + 256 x 64 (48 KB each); two 256-column
//    accumulators, so the epilogue of a tile overlaps the next tile's MMAs;
//  * BM = 256: 3 stages of 256 x 64 + 256 x 64 (64 KB each); the tile's two
//    128-row halves take the 512 columns, the epilogue does not overlap,
//    but each stage's bytes feed twice the MMA work (the TMA latency is
//    what limits the 128-row tiles: a third fewer bytes a flop).
constexpr int kMmaM = 128, kBN = 256, kBK = 64, kMaxStages = 4;
constexpr int kTcThreads = 192;  // producer, MMA issuer, 4 epilogue warps
constexpr uint32_t kBBytes = kBN * kBK * 2;
constexpr uint32_t kHalfA = kMmaM * kBK * 2;  // 128 rows of A (16 KB)
constexpr uint32_t kMnBox = 64 * kBK * 2;  // one 64 (MN) x 64 (K) box of an MN-major tile
constexpr uint32_t kTmemCols = 2 * kBN;    // 512 columns
template <int BM>
struct TcTile {
    static constexpr int kStages = BM == 256 ? 3 : 4;
    static constexpr int kHalves = BM / kMmaM;      // 128-row MMAs a K step
    static constexpr int kAccBufs = BM == 256 ? 1 : 2;
    static constexpr uint32_t kABytes = BM * kBK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
};
constexpr uint32_t kRingBytes = 4 * (kHalfA + kBBytes);  // the same for both BM
static_assert(TcTile<128>::kStages * TcTile<128>::kStageBytes == kRingBytes &&
                  TcTile<256>::kStages * TcTile<256>::kStageBytes == kRingBytes,
              "both tile shapes use the same ring");
// epilogue staging for TMA stores: per epilogue warp two 32-row x 128-byte
// boxes (4 KB each, 128-byte swizzle)
constexpr uint32_t kStageOut = 4096;
constexpr uint32_t kOutBytes = 4 * 2 * kStageOut;
constexpr size_t kTcSmem = static_cast<size_t>(kRingBytes) + kOutBytes + 1024;

// What the epilogue does with the accumulator.
enum : int { kOutF32 = 0, kOutF32Add = 1, kOut16 = 2 };

struct TcArgs {
    void* C;            // [M, N] row-major: fp32, or the operand type for kOut16
    const float* bias;  // [N] or nullptr (kOutF32 only)
    int64_t M, N, K;
    int64_t tiles_m, tiles_n, tiles;
    int m_first;  // tile t runs along M first (1) or along N first (0)
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

// The same for an MN-major operand tile stored as boxes of 64 MN elements
// (one 128-byte swizzled row) x 64 K rows, 8 KB each, side by side along
// MN: 8-row (K) atoms of 1024 bytes, the stride between atoms along K (the
// stride dimension offset) 1024 bytes, between 64-element blocks along MN
// (the leading dimension offset) one box, 8 KB.
__device__ __forceinline__ uint64_t tc_smem_desc_mn(uint32_t saddr) {
    uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(kMnBox >> 4) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B of the
// given type (0 fp16, 1 bf16), A and B K-major (0) or MN-major (1, the
// transpose bits 15 and 16), N = kBN, M = kMmaM.
__host__ __device__ constexpr uint32_t tc_idesc(uint32_t ab, uint32_t a_mn = 0, uint32_t b_mn = 0) {
    return (1u << 4) | (ab << 7) | (ab << 10) | (a_mn << 15) | (b_mn << 16) |
           (static_cast<uint32_t>(kBN >> 3) << 17) | (static_cast<uint32_t>(kMmaM >> 4) << 24);
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

// TMA store and reduce-add of a 2-D box from this CTA's shared memory, in
// a bulk group (commit, then wait for the reads before reusing the buffer)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int x,
                                                  int y) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// at most one bulk group still reading shared memory
__device__ __forceinline__ void bulk_wait_read_1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// this thread's shared-memory writes visible to the TMA (async proxy)
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

// Stores 32 accumulator columns (fp32 v) of row `row` from column n of C.
template <int OUT, uint32_t AB>
__device__ __forceinline__ void tc_store32(const TcArgs& a, int64_t row, int64_t n,
                                           float (&v)[32]) {
    if (OUT == kOutF32 && a.bias) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (n + i < a.N) v[i] += __ldg(a.bias + n + i);
    }
    const bool full = n + 32 <= a.N;
    if constexpr (OUT == kOut16) {
        using T = typename std::conditional<AB == 1u, __nv_bfloat16, __half>::type;
        T* c = static_cast<T*>(a.C) + row * a.N + n;
        if (full && (a.N & 7) == 0) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
                const float f[8] = {v[i], v[i + 1], v[i + 2], v[i + 3],
                                    v[i + 4], v[i + 5], v[i + 6], v[i + 7]};
                *reinterpret_cast<uint4*>(c + i) = Vec<T>::pack(f);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (n + i < a.N) Vec<T>::store1(c, i, v[i]);
        }
    } else {
        float* c = static_cast<float*>(a.C) + row * a.N + n;
        if (full && (a.N & 3) == 0) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                float4 o = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                if (OUT == kOutF32Add) {
                    const float4 p = *reinterpret_cast<const float4*>(c + i);
                    o.x += p.x;
                    o.y += p.y;
                    o.z += p.z;
                    o.w += p.w;
                }
                *reinterpret_cast<float4*>(c + i) = o;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (n + i < a.N) c[i] = OUT == kOutF32Add ? c[i] + v[i] : v[i];
        }
    }
}

// Tile t's row and column of tiles.
__device__ __forceinline__ int64_t tile_m(const TcArgs& a, int64_t t) {
    return a.m_first ? t % a.tiles_m : t / a.tiles_n;
}
__device__ __forceinline__ int64_t tile_n(const TcArgs& a, int64_t t) {
    return a.m_first ? t / a.tiles_m : t % a.tiles_n;
}

// Writes this thread's row of 32 fp32 columns (h = 0), or one half of 64
// 16-bit columns (h = 0, 1), into a 32-row x 128-byte staging box laid out
// as the TMA's 128-byte swizzle wants it: 16-byte chunk j of row r at
// chunk position j ^ (r mod 8). Conflict-free: the 8 threads of a quarter
// warp cover all 32 banks.
template <int OUT, uint32_t AB>
__device__ __forceinline__ void tc_stage32(uint32_t buf, int r, int h, const float (&v)[32]) {
    const uint32_t row = buf + static_cast<uint32_t>(r) * 128u;
    if constexpr (OUT == kOut16) {
        using T = typename std::conditional<AB == 1u, __nv_bfloat16, __half>::type;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float f[8] = {v[8 * j], v[8 * j + 1], v[8 * j + 2], v[8 * j + 3],
                                v[8 * j + 4], v[8 * j + 5], v[8 * j + 6], v[8 * j + 7]};
            const uint4 p = Vec<T>::pack(f);
            const uint32_t at = row + (static_cast<uint32_t>((4 * h + j) ^ (r & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(at), "r"(p.x), "r"(p.y),
                         "r"(p.z), "r"(p.w)
                         : "memory");
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t at = row + (static_cast<uint32_t>(j ^ (r & 7)) << 4);
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(at), "f"(v[4 * j]),
                         "f"(v[4 * j + 1]), "f"(v[4 * j + 2]), "f"(v[4 * j + 3])
                         : "memory");
        }
    }
}

// A_MN / B_MN: the operand is stored MN-major (A as [K, M], B as [K, N]).
// TMAO: C leaves through shared memory with TMA stores (reduce-adds for
// kOutF32Add) of 32-row x 128-byte boxes; else with plain stores (a C
// whose base or row pitch is not a multiple of 16 bytes).
// BM: the tile's rows (TcTile).
template <uint32_t AB, bool A_MN, bool B_MN, int OUT, bool TMAO, int BM>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_gemm(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
        const __grid_constant__ CUtensorMap mapC, const __grid_constant__ TcArgs a) {
    using TT = TcTile<BM>;
    constexpr int kStages = TT::kStages;
    constexpr uint32_t kABytes = TT::kABytes;
    constexpr uint32_t kStageBytes = TT::kStageBytes;
    constexpr int NACC = TT::kAccBufs;
    constexpr int H = TT::kHalves;
    extern __shared__ unsigned char tc_smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ __align__(8) uint64_t acc_full[2];
    __shared__ __align__(8) uint64_t acc_empty[2];
    __shared__ __align__(8) uint64_t done_bar;  // every MMA of the CTA completed
    __shared__ uint32_t tmem_base_sh;
    __shared__ uint32_t s_issued[kMaxStages];  // 0, or 2 + parity of the last copy into the stage
    __shared__ int s_fail;

    // a CTA of this launch already gave up: the others return at once
    // (before any tensor memory is taken)
    if (*reinterpret_cast<volatile unsigned*>(a.abort)) return;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t smem0 = (smem_u32(tc_smem_raw) + 1023u) & ~1023u;  // 1024-byte aligned
    const int nk = static_cast<int>((a.K + kBK - 1) / kBK);
    const int64_t ntiles = a.tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
            s_issued[s] = 0;
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), 128);
        }
        mbar_init(smem_u32(&done_bar), 1);
        s_fail = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
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

    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer: every K block of every tile of this CTA
            int it = 0;  // K blocks issued so far (ring position)
            bool fail = false;
            for (int64_t t = blockIdx.x; t < ntiles && !fail; t += gridDim.x) {
                const int m0 = static_cast<int>(tile_m(a, t) * BM);
                const int n0 = static_cast<int>(tile_n(a, t) * kBN);
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = static_cast<uint32_t>(it / kStages) & 1u;
                    if (!tc_wait(smem_u32(&empty_bar[s]), ph ^ 1u, a.timeout_ns) ||
                        *reinterpret_cast<volatile unsigned*>(a.abort)) {
                        fail = true;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full_bar[s]);
                    mbar_arrive_expect_tx(fb, kStageBytes);
                    const uint32_t sa = smem0 + static_cast<uint32_t>(s) * kStageBytes;
                    const int k0 = kb * kBK;
                    if (A_MN) {
                        for (int j = 0; j < BM / 64; ++j)
                            tma_load_2d(sa + j * kMnBox, &mapA, m0 + 64 * j, k0, fb);
                    } else {
                        tma_load_2d(sa, &mapA, k0, m0, fb);
                    }
                    if (B_MN) {
                        for (int j = 0; j < kBN / 64; ++j)
                            tma_load_2d(sa + kABytes + j * kMnBox, &mapB, n0 + 64 * j, k0, fb);
                    } else {
                        tma_load_2d(sa + kABytes, &mapB, k0, n0, fb);
                    }
                    s_issued[s] = 2u + ph;
                }
            }
            if (fail) s_fail = 1;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer: tile i into accumulator buffer i mod NACC
            constexpr uint32_t idesc = tc_idesc(AB, A_MN ? 1u : 0u, B_MN ? 1u : 0u);
            int it = 0;
            int i = 0;  // tiles of this CTA so far
            bool fail = false;
            for (int64_t t = blockIdx.x; t < ntiles && !fail; t += gridDim.x, ++i) {
                const int b = i % NACC;
                // the epilogue has drained this buffer's previous tile
                if (!tc_wait(smem_u32(&acc_empty[b]),
                             (static_cast<uint32_t>(i / NACC) & 1u) ^ 1u, a.timeout_ns)) {
                    fail = true;
                    break;
                }
                tc_fence_after();
                // half h of the tile (rows 128 h ...) in columns (b H + h) 256
                const uint32_t acc = tmem + static_cast<uint32_t>(b * H * kBN);
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = static_cast<uint32_t>(it / kStages) & 1u;
                    if (!tc_wait(smem_u32(&full_bar[s]), ph, a.timeout_ns)) {
                        fail = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem0 + static_cast<uint32_t>(s) * kStageBytes;
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        // K step of 16: 32 bytes inside a K-major swizzled row, two
                        // 8-row atoms (2 KB) of an MN-major tile
                        const uint64_t db = B_MN ? tc_smem_desc_mn(sa + kABytes + 2048u * k)
                                                 : tc_smem_desc(sa + kABytes + 32u * k);
#pragma unroll
                        for (int h = 0; h < H; ++h) {
                            // rows 128 h of A: 16 KB on in either layout (128
                            // swizzled rows, or two 64-wide boxes)
                            const uint32_t ah = sa + static_cast<uint32_t>(h) * kHalfA;
                            const uint64_t da = A_MN ? tc_smem_desc_mn(ah + 2048u * k)
                                                     : tc_smem_desc(ah + 32u * k);
                            tc_mma(acc + static_cast<uint32_t>(h * kBN), da, db, idesc,
                                   (kb > 0 || k > 0) ? 1u : 0u);
                        }
                    }
                    tc_commit(smem_u32(&empty_bar[s]));
                }
                // every MMA of the tile issued: the epilogue may read it once
                // they complete (also after a failure, so that nothing waits)
                tc_commit(smem_u32(&acc_full[b]));
            }
            if (fail) s_fail = 1;
            tc_commit(smem_u32(&done_bar));  // after every MMA this thread issued
        }
    } else {
        // ---- epilogue: warp w reads accumulator lanes 32 (w mod 4) of
        // each 128-row half of the tile
        const int q = warp & 3;
        // this warp's two staging boxes, used in turn
        const uint32_t stg = smem0 + kRingBytes + static_cast<uint32_t>(q) * 2u * kStageOut;
        uint32_t nst = 0;  // boxes this warp has handed to the TMA
        int i = 0;
        for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
            const int b = i % NACC;
            const bool ok = mbar_wait_bounded(smem_u32(&acc_full[b]),
                                              static_cast<uint32_t>(i / NACC) & 1u, a.timeout_ns);
            if (!ok || *reinterpret_cast<volatile int*>(&s_fail) ||
                *reinterpret_cast<volatile unsigned*>(a.abort)) {
                if (lane == 0) s_fail = 1;
                break;
            }
            tc_fence_after();
            const int64_t n0 = tile_n(a, t) * kBN;
#pragma unroll 1
            for (int hh = 0; hh < H; ++hh) {
                const int64_t m0 = tile_m(a, t) * BM + hh * kMmaM;
                const int64_t row = m0 + q * 32 + lane;
                const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                      static_cast<uint32_t>((b * H + hh) * kBN);
                if constexpr (TMAO) {
                    constexpr int kBoxCols = OUT == kOut16 ? 64 : 32;
                    const bool rows_in = m0 + q * 32 < a.M;  // the same for the whole warp
#pragma unroll 1
                    for (int c = 0; c < kBN / kBoxCols; ++c) {
                        const int64_t n = n0 + c * kBoxCols;
                        if (n >= a.N) break;  // the same for every thread of the warp
                        const uint32_t buf = stg + (nst & 1u) * kStageOut;
                        // the box written two turns ago has been read out of this buffer
                        if (lane == 0) bulk_wait_read_1();
                        __syncwarp();
#pragma unroll
                        for (int h = 0; h < kBoxCols / 32; ++h) {
                            float v[32];
                            tc_ld32(trow + static_cast<uint32_t>(c * kBoxCols + h * 32), v);
                            if (OUT == kOutF32 && a.bias) {
                                const int64_t nb = n + h * 32;
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    if (nb + j < a.N) v[j] += __ldg(a.bias + nb + j);
                            }
                            tc_stage32<OUT, AB>(buf, lane, h, v);
                        }
                        fence_proxy_async_smem();  // the writes, seen by the TMA
                        __syncwarp();
                        if (lane == 0 && rows_in) {
                            // rows past M and columns past N are clipped by the TMA
                            if (OUT == kOutF32Add)
                                tma_reduce_add_2d(&mapC, buf, static_cast<int>(n),
                                                  static_cast<int>(m0 + q * 32));
                            else
                                tma_store_2d(&mapC, buf, static_cast<int>(n),
                                             static_cast<int>(m0 + q * 32));
                        }
                        if (lane == 0) bulk_commit();
                        ++nst;
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < kBN / 32; ++c) {
                        const int64_t n = n0 + c * 32;
                        if (n >= a.N) break;  // the same for every thread of the warp
                        float v[32];
                        tc_ld32(trow + static_cast<uint32_t>(c * 32), v);
                        if (row < a.M) tc_store32<OUT, AB>(a, row, n, v);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&acc_empty[b]));
        }
        // every box written out before the shared memory goes
        if (TMAO && lane == 0) bulk_wait_all();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // every MMA completes before the tensor memory is freed
        const bool done = mbar_wait_bounded(smem_u32(&done_bar), 0u, a.timeout_ns);
        if (s_fail || !done) {
            atomicOr(a.status, kDevErrTimeout);
            atomicExch(a.abort, 1u);
            // copies still in flight land before the shared memory is released
            for (int s = 0; s < kStages; ++s)
                if (s_issued[s])
                    (void)mbar_wait_bounded(smem_u32(&full_bar[s]), s_issued[s] & 1u,
                                            a.timeout_ns);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1)
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

// 2-D map of a row-major [outer, inner] matrix of 16-bit elements, boxes of
// box_outer x 64 elements (128 bytes: the swizzle width), 128-byte
// swizzle, zeros outside the matrix. A K-major operand is [MN, K] with boxes
// of 128 or 256 rows; an MN-major one is [K, MN] with boxes of 64 K rows.
ce_status make_map(CUtensorMap* map, const void* p, int dtype, int64_t outer, int64_t inner,
                   uint32_t box_outer) {
    EncodeTiled enc = nullptr;
    ce_status rc = encoder(&enc);
    if (rc != CE_OK) return rc;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 2};
    const cuuint32_t box[2] = {64u, box_outer};
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

// 2-D map of C [M, N] row-major (fp32, or 16-bit for kOut16) for the
// epilogue's TMA stores: boxes of 32 rows x 128 bytes, 128-byte swizzle.
ce_status make_map_c(CUtensorMap* map, void* C, int dtype, int out, int64_t M, int64_t N) {
    EncodeTiled enc = nullptr;
    ce_status rc = encoder(&enc);
    if (rc != CE_OK) return rc;
    const bool h = out == kOut16;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * (h ? 2 : 4)};
    const cuuint32_t box[2] = {h ? 64u : 32u, 32u};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType t = !h ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                  : dtype == CE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUresult r = enc(map, t, 2, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        record_message("cuTensorMapEncodeTiled (C) failed (" + std::to_string(static_cast<int>(r)) +
                       ")");
        return CE_ERR_UNSUPPORTED;
    }
    return CE_OK;
}

template <uint32_t AB, bool TMAO, int TBM>
const void* gemm_fn_t(bool a_mn, bool b_mn, int out) {
#define GBCE_TC(AM, BMN)                                                              \
    (out == kOutF32      ? (const void*)&tc_gemm<AB, AM, BMN, kOutF32, TMAO, TBM>    \
     : out == kOutF32Add ? (const void*)&tc_gemm<AB, AM, BMN, kOutF32Add, TMAO, TBM> \
                         : (const void*)&tc_gemm<AB, AM, BMN, kOut16, TMAO, TBM>)
    if (!a_mn && !b_mn) return GBCE_TC(false, false);
    if (!a_mn && b_mn) return GBCE_TC(false, true);
    if (a_mn && !b_mn) return GBCE_TC(true, false);
    return GBCE_TC(true, true);
#undef GBCE_TC
}

// The 256-row tiles only with the TMA-store epilogue (a C aligned for it).
template <uint32_t AB>
const void* gemm_fn(bool a_mn, bool b_mn, int out, bool tmao, int bm) {
    if (!tmao) return gemm_fn_t<AB, false, 128>(a_mn, b_mn, out);
    return bm == 256 ? gemm_fn_t<AB, true, 256>(a_mn, b_mn, out)
                     : gemm_fn_t<AB, true, 128>(a_mn, b_mn, out);
}

// Tile rows for an M x N product on `sms` persistent CTAs: the shape with
// the fewer rounds of tiles over the SMs, a round of 256-row tiles counted
// as 1.6 of 128-row ones (measured: 1774 against 1440 TFLOP/s at 8192^3)
// (GBCE_TC_BM = 128 or 256 forces one).
int tile_rows(int64_t M, int64_t N, int sms, bool tmao) {
    if (!tmao) return 128;
    const char* v = std::getenv("GBCE_TC_BM");
    if (v && *v) return std::atoi(v) == 256 ? 256 : 128;
    const int64_t tn = (N + kBN - 1) / kBN, s = std::max(sms, 1);
    const int64_t r256 = ((M + 255) / 256 * tn + s - 1) / s;
    const int64_t r128 = ((M + 127) / 128 * tn + s - 1) / s;
    return 16 * r256 < 10 * r128 ? 256 : 128;
}

}  // namespace

// A 2-D map of a row-major [outer, inner] matrix of `dtype` elements (pitch
// inner elements), boxes of box_inner x box_outer elements, no swizzle,
// zeros outside the matrix (the N-D tile kernel's class rows).
ce_status tensor_map_rows_2d(CUtensorMap* map, int dtype, const void* p, int64_t outer,
                             int64_t inner, uint32_t box_inner, uint32_t box_outer) {
    EncodeTiled enc = nullptr;
    ce_status rc = encoder(&enc);
    if (rc != CE_OK) return rc;
    const int64_t b = dtype == CE_F32 ? 4 : 2;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner * b)};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType t = dtype == CE_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                  : dtype == CE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUresult r = enc(map, t, 2, const_cast<void*>(p), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        record_message("cuTensorMapEncodeTiled (rows) failed (" +
                       std::to_string(static_cast<int>(r)) + ")");
        return CE_ERR_UNSUPPORTED;
    }
    return CE_OK;
}

// Whether the tensor-core GEMM takes an operand: a 16-bit type, a 16-byte
// aligned base and rows of a multiple of 8 elements (16-byte strides for
// the TMA): K for a K-major operand, M or N for an MN-major one.
bool tc_operand_ok(const void* p, int dtype, int64_t row_elems) {
    return (dtype == CE_BF16 || dtype == CE_F16) && row_elems % 8 == 0 && row_elems > 0 &&
           (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

bool tc_gemm_supported(const void* A, const void* B, int dtype, int64_t K) {
    return tc_operand_ok(A, dtype, K) && tc_operand_ok(B, dtype, K);
}

// C = A @ B on `st` (layouts and outputs as ce_gemm); status receives
// timeouts (device word), abort is a device word this launch may use
// (cleared here first).
ce_status tc_gemm_launch(const void* A, bool a_mn, const void* B, bool b_mn, int dtype, int64_t M,
                         int64_t N, int64_t K, void* C, int out, const float* bias,
                         unsigned* status, unsigned* abort, cudaStream_t st) {
    if (M <= 0 || N <= 0) return CE_OK;
    if (K <= 0 || !tc_operand_ok(A, dtype, a_mn ? M : K) || !tc_operand_ok(B, dtype, b_mn ? N : K))
        return CE_ERR_UNSUPPORTED;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return CE_ERR_UNSUPPORTED;
    // C through TMA stores when its base and row pitch are multiples of 16 bytes
    const int64_t cpitch = N * (out == kOut16 ? 2 : 4);
    const bool tmao = (reinterpret_cast<uintptr_t>(C) & 15u) == 0 && cpitch % 16 == 0;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return record_cuda_failure(e, "tensor-core GEMM device");
    const int bm = tile_rows(M, N, sms, tmao);
    CUtensorMap ma, mb;
    ce_status rc = a_mn ? make_map(&ma, A, dtype, K, M, 64)
                        : make_map(&ma, A, dtype, M, K, static_cast<uint32_t>(bm));
    if (rc != CE_OK) return rc;
    rc = b_mn ? make_map(&mb, B, dtype, K, N, 64) : make_map(&mb, B, dtype, N, K, kBN);
    if (rc != CE_OK) return rc;
    CUtensorMap mc;
    std::memset(&mc, 0, sizeof(mc));
    if (tmao) {
        rc = make_map_c(&mc, C, dtype, out, M, N);
        if (rc != CE_OK) return rc;
    }
    const void* fn = dtype == CE_BF16 ? gemm_fn<1u>(a_mn, b_mn, out, tmao, bm)
                                      : gemm_fn<0u>(a_mn, b_mn, out, tmao, bm);
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kTcSmem));
    if (e != cudaSuccess) return record_cuda_failure(e, "tensor-core GEMM attributes");
    const char* tenv = std::getenv("GBCE_WAIT_TIMEOUT_MS");
    const uint64_t tms = (tenv && *tenv) ? static_cast<uint64_t>(std::atoll(tenv)) : 2000ull;
    e = cudaMemsetAsync(abort, 0, sizeof(unsigned), st);
    if (e != cudaSuccess) return record_cuda_failure(e, "cudaMemsetAsync(abort word)");
    const int64_t tm = (M + bm - 1) / bm, tn = (N + kBN - 1) / kBN;
    // consecutive tiles (the CTAs that run together) share a tile of the
    // larger operand, which is then read from DRAM about once: along M first
    // when B is the larger (its tile serves every row of tiles), along N
    // first when A is
    const int m_first = N >= M ? 1 : 0;
    TcArgs a{C,  out == kOutF32 ? bias : nullptr, M, N, K, tm, tn, tm * tn, m_first,
             tms * 1000000ull, status, abort};
    // persistent: one CTA an SM at most
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>(tm * tn, std::max(sms, 1)));
    void* args[] = {&ma, &mb, &mc, &a};
    e = cudaLaunchKernel(fn, dim3(grid), dim3(kTcThreads), args, kTcSmem, st);
    if (e != cudaSuccess) return record_cuda_failure(e, "tensor-core GEMM launch");
    return CE_OK;
}

// C = A @ B^T (+ bias), both K-major, fp32 C: the logits GEMM.
ce_status tc_gemm_abt_launch(const void* A, const void* B, int dtype, int64_t M, int64_t N,
                             int64_t K, float* C, const float* bias, unsigned* status,
                             unsigned* abort, cudaStream_t st) {
    return tc_gemm_launch(A, false, B, false, dtype, M, N, K, C, kOutF32, bias, status, abort, st);
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

extern "C" ce_status ce_gemm(const void* A, int a_mn, const void* B, int b_mn, int dtype,
                             int64_t M, int64_t N, int64_t K, void* C, int c_mode,
                             const float* bias, ce_stream_t stream) {
    if (dtype != CE_BF16 && dtype != CE_F16) return CE_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K <= 0) return CE_ERR_INVALID_ARG;
    if (c_mode != kOutF32 && c_mode != kOutF32Add && c_mode != kOut16) return CE_ERR_INVALID_ARG;
    if (bias && c_mode != kOutF32) return CE_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return CE_OK;
    if (!A || !B || !C) return CE_ERR_INVALID_ARG;
    if (!tc_operand_ok(A, dtype, a_mn ? M : K) || !tc_operand_ok(B, dtype, b_mn ? N : K))
        return CE_ERR_UNSUPPORTED;
    unsigned* status = nullptr;
    ce_status rc = library_status_word(reinterpret_cast<cudaStream_t>(stream), &status);
    if (rc != CE_OK) return rc;
    return tc_gemm_launch(A, a_mn != 0, B, b_mn != 0, dtype, M, N, K, C, c_mode, bias, status,
                          status + 1, reinterpret_cast<cudaStream_t>(stream));
}
