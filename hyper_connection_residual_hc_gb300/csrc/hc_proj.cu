// Projection of the generic path on the 5th-generation tensor cores, for any number of streams hc in
// 1..8 and any width d (a multiple of 8): raw[t][m] = sum_c X'[t][c] w[m][c] over the c < hc*d columns
// of a token's flattened streams, and ssx[t] = sum_c X'[t][c]^2 ("Source layer, pairs pooled" page,
// Block.hc_mixes excerpt: the fp32 projection of the flattened streams onto mix_hc = (2 + hc) * hc
// mixes, and the mean square behind its r). The scaling by r, the split and the norm follow in
// gen_tail_kernel.
//
// The weights are the three bf16 planes of hc_prepare_params, a [3M, hc*d] matrix with
// w = hi + mid + lo exactly (plane_row gives each plane's row). One CTA takes 128 tokens of a chunk
// and streams the hc*d columns in stages of 32: a TMA load of the X' tile [128 x 32] and of all 3M
// plane rows [N x 32] (N = 3M rounded up to 16; rows past 3M and columns past hc*d read as zeros),
// both with the 64-byte swizzle, then two tcgen05.mma kind::f16 (K = 16 each) into a TMEM
// accumulator of N fp32 columns, one per plane row. Each product of two bf16 values is exact in
// fp32, so the projection has the accuracy of an fp32 dot product.
//
// Two accumulators take blocks of 8 stages in turn. While the tensor cores fill one, the four row
// warps (warp q: TMEM lanes and tile rows 32q..32q+31) add the other's columns into their rows'
// running fp32 sums per mix in shared memory: a sum of 256-column partial sums, as the fused kernel
// sums its stages. Between drains they sum the squares of their rows from the same shared tiles.
// Warp 4 issues the loads and warp 5 the MMAs. Every wait is bounded: on expiry the kernel sets a
// bit in its device error word, stops waiting, lets its copies land and frees its tensor memory.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "hc_internal.h"
#include "hc_ptx.cuh"

namespace hc {
namespace {

constexpr int kPjRows = 128;                     // tokens per CTA: the MMA's M
constexpr int kPjCols = 32;                      // columns per stage: one 64-byte row per token
constexpr int kPjATile = kPjRows * kPjCols * 2;  // 8 KB
constexpr int kPjBlock = 8;                      // stages per accumulator block (256 columns)
constexpr int kPjThreads = 192;                  // warps 0-3 rows, 4 loads, 5 MMAs
constexpr int kPjWarpLoad = 4, kPjWarpMma = 5;
constexpr int kPjMaxSlots = 8;
constexpr int kPjSmemBudget = 200 * 1024;
constexpr uint64_t kPjWaitNs = 1000000000ull;  // 1 s
constexpr int kPjMaxDevices = 64;

// device error word of this kernel (bits above the fused kernel's), read with theirs
__device__ unsigned int g_hc_proj_error = 0;
enum : unsigned int { kPjErrLoad = 1u << 16, kPjErrMma = 1u << 17, kPjErrRows = 1u << 18, kPjErrDrain = 1u << 19 };

struct ProjParams {
    float* raw;       // fp32 [m, M]
    float* ssx;       // fp32 [m]
    long long m;      // tokens of the chunk
    int hc;
    int M;            // (2 + hc) * hc
    int N;            // accumulator columns: 3M rounded up to 16
    int stages;       // ceil(hc * d / 32)
    int slots;        // load ring depth
    int tmem_cols;    // allocated TMEM columns (a power of two >= 2N)
};

// shared-memory layout, the same on host and device
struct ProjLayout {
    int slot_bytes, off_sums, off_bars, bytes;
    __host__ __device__ ProjLayout(int N, int M, int slots) {
        slot_bytes = kPjATile + N * kPjCols * 2;
        off_sums = slots * slot_bytes;
        off_bars = (off_sums + M * kPjRows * 4 + 7) & ~7;
        bytes = off_bars + (2 * slots + 5) * 8 + 8;  // full, empty, 2 acc full, 2 acc empty, mma done; tmem + abort
    }
};

struct PjWait {
    volatile uint32_t* abort;
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, unsigned int code) const {
        if (mbar_test(bar, parity)) return true;
        const uint64_t t0 = global_timer_ns();
        while (true) {
            for (int i = 0; i < 32; ++i)
                if (mbar_test(bar, parity)) return true;
            if (*abort) return false;
            if (global_timer_ns() - t0 > kPjWaitNs) {
                *abort = 1u;
                atomicOr(&g_hc_proj_error, code);
                return false;
            }
        }
    }
    // ignores an abort raised elsewhere: used at exit to let copies and MMAs in flight finish
    __device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) const {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_test(bar, parity)) {
            if (global_timer_ns() - t0 > kPjWaitNs) {
                atomicOr(&g_hc_proj_error, kPjErrDrain);
                return;
            }
        }
    }
};

// the mix whose plane sits in plane row j (the inverse of plane_row)
__device__ __forceinline__ int mix_of_row(int hc, int M, int j) {
    return hc == 4 ? 12 * (j / 36) + (j % 36) % 12 : j % M;
}

__global__ void __launch_bounds__(kPjThreads, 1) gen_proj_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                                                                    const __grid_constant__ CUtensorMap tmB,
                                                                    const ProjParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
    const ProjLayout L(p.N, p.M, p.slots);
    float* sums = reinterpret_cast<float*>(smem + L.off_sums);  // [M][128]: mix-major, a row per lane
    const uint32_t bars = sbase + static_cast<uint32_t>(L.off_bars);
    auto full = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
    auto empty = [&](int i) { return bars + 8u * static_cast<uint32_t>(p.slots + i); };
    auto acc_full = [&](int b) { return bars + 8u * static_cast<uint32_t>(2 * p.slots + b); };
    auto acc_empty = [&](int b) { return bars + 8u * static_cast<uint32_t>(2 * p.slots + 2 + b); };
    const uint32_t mma_done = bars + 8u * static_cast<uint32_t>(2 * p.slots + 4);
    uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + L.off_bars + 8 * (2 * p.slots + 5));
    volatile uint32_t* abort_flag = tmem_ptr + 1;
    const PjWait W{abort_flag};
    const int S = p.stages;
    const int nblocks = (S + kPjBlock - 1) / kPjBlock;
    const int row0 = static_cast<int>(blockIdx.x) * kPjRows;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.slots; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), 1 + 4);  // the MMAs' completion + the four row warps' squares
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), 4);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == kPjWarpLoad && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == kPjWarpMma) {
        tmem_alloc(smem_u32(tmem_ptr), static_cast<uint32_t>(p.tmem_cols));
        tmem_relinquish();
    }
    for (int i = static_cast<int>(threadIdx.x); i < p.M * kPjRows; i += kPjThreads) sums[i] = 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_ptr);

    if (warp == kPjWarpLoad) {
        // ===== TMA: stage s into slot s % slots, once the MMAs and the row warps are done with it ====
        if (lane == 0) {
            const uint64_t pol_stream = policy_evict_normal(), pol_keep = policy_evict_last();
            for (int s = 0; s < S; ++s) {
                const int i = s % p.slots, round = s / p.slots;
                if (round > 0) W.wait(empty(i), static_cast<uint32_t>((round - 1) & 1), kPjErrLoad);
                const uint32_t a = sbase + static_cast<uint32_t>(i * L.slot_bytes);
                mbar_arrive_expect_tx(full(i), static_cast<uint32_t>(L.slot_bytes));
                tma_load_2d(a, &tmA, full(i), kPjCols * s, row0, pol_stream);
                tma_load_2d(a + kPjATile, &tmB, full(i), kPjCols * s, 0, pol_keep);
            }
            // every load lands before the CTA may exit (a slot's last load lands after its earlier ones)
            for (int s = S - p.slots > 0 ? S - p.slots : 0; s < S; ++s)
                W.drain(full(s % p.slots), static_cast<uint32_t>((s / p.slots) & 1));
        }
        __syncwarp();
    } else if (warp == kPjWarpMma) {
        // ===== MMA: block b of 16 stages into accumulator b % 2 ======================================
        const uint32_t idesc = idesc_bf16_f32(kPjRows, p.N);
        for (int s = 0; s < S; ++s) {
            const int i = s % p.slots, round = s / p.slots;
            const int b = s / kPjBlock, buf = b & 1;
            // the accumulator's previous block (b - 2) must have been drained by the row warps
            if (s % kPjBlock == 0 && b >= 2) W.wait(acc_empty(buf), static_cast<uint32_t>(((b >> 1) - 1) & 1), kPjErrMma);
            W.wait(full(i), static_cast<uint32_t>(round & 1), kPjErrMma);
            tc_fence_after();
            if (lane == 0) {
                const uint32_t a = sbase + static_cast<uint32_t>(i * L.slot_bytes);
                const uint32_t dcol = tmem + static_cast<uint32_t>(buf * p.N);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    umma_bf16(dcol, sdesc_kmajor_sw64(a + kk * 32), sdesc_kmajor_sw64(a + kPjATile + kk * 32), idesc,
                              (s % kPjBlock != 0 || kk != 0) ? 1u : 0u);
                umma_commit(empty(i));
                if (s % kPjBlock == kPjBlock - 1 || s == S - 1) umma_commit(acc_full(buf));
            }
            __syncwarp();
        }
        if (lane == 0) {
            umma_commit(mma_done);
            W.drain(mma_done, 0u);
        }
        __syncwarp();
    } else {
        // ===== row warps: squares of the rows, and the accumulator blocks into the running sums =====
        const int r = 32 * warp + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * warp) << 16);
        float sq = 0.f;
        int drained = 0;
        auto drain_block = [&](int b) {
            const int buf = b & 1;
            W.wait(acc_full(buf), static_cast<uint32_t>((b >> 1) & 1), kPjErrRows);
            tc_fence_after();
            for (int c0 = 0; c0 < p.N; c0 += 16) {
                uint32_t v[16];
                tmem_ld16_wait(tl + static_cast<uint32_t>(buf * p.N + c0), v);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int j = c0 + e;
                    if (j < 3 * p.M) sums[mix_of_row(p.hc, p.M, j) * kPjRows + r] += __uint_as_float(v[e]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(buf));
        };
        for (int s = 0; s < S; ++s) {
            const int i = s % p.slots, round = s / p.slots;
            W.wait(full(i), static_cast<uint32_t>(round & 1), kPjErrRows);
            // this row's 64 bytes of the tile: 16-byte chunk c sits at chunk c ^ ((r >> 1) & 3)
            const uint32_t rowa = sbase + static_cast<uint32_t>(i * L.slot_bytes + r * 64);
            float part = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 v = ld_smem_v4(rowa + static_cast<uint32_t>((c ^ ((r >> 1) & 3)) << 4));
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xFFFF0000u);
                    part = fmaf(lo, lo, part);
                    part = fmaf(hi, hi, part);
                }
            }
            sq += part;
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(i));
            // block b is drained half a block after it ends, when its MMAs have long completed
            if (s % kPjBlock == kPjBlock / 2 && s >= kPjBlock) drain_block(drained++);
        }
        while (drained < nblocks) drain_block(drained++);
        const long long t = static_cast<long long>(row0) + r;
        if (t < p.m) {
            for (int mm = 0; mm < p.M; ++mm) p.raw[t * p.M + mm] = sums[mm * kPjRows + r];
            p.ssx[t] = sq;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kPjWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, static_cast<uint32_t>(p.tmem_cols));
    }
}

PFN_cuTensorMapEncodeTiled_v12000 proj_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// a 2-D bf16 tensor map [rows, cols] (row stride cols * 2 bytes) with boxes of box_rows x 32 columns
bool encode_rows(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    auto fn = proj_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kPjCols), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int launch_proj_tc(const void* X, const void* planes, int64_t m, int hc, int d, float* raw, float* ssx,
                   cudaStream_t stream) {
    if (m <= 0) return 0;
    const int M = (2 + hc) * hc;
    const int N = (3 * M + 15) / 16 * 16;
    if (hc < 1 || N > 256 || d % 8 != 0) return -2;
    const uint64_t D = static_cast<uint64_t>(hc) * static_cast<uint64_t>(d);
    int slots = kPjMaxSlots;
    while (slots > 2 && ProjLayout(N, M, slots).bytes + 1024 > kPjSmemBudget) --slots;
    const int smem = ProjLayout(N, M, slots).bytes + 1024;
    int tcols = 32;
    while (tcols < 2 * N) tcols *= 2;
    CUtensorMap tmA, tmB;
    if (!encode_rows(&tmA, X, D, static_cast<uint64_t>(m), kPjRows)) return -7;
    if (!encode_rows(&tmB, planes, D, static_cast<uint64_t>(3 * M), static_cast<uint32_t>(N))) return -7;
    ProjParams p;
    p.raw = raw;
    p.ssx = ssx;
    p.m = m;
    p.hc = hc;
    p.M = M;
    p.N = N;
    p.stages = static_cast<int>((D + kPjCols - 1) / kPjCols);
    p.slots = slots;
    p.tmem_cols = tcols;
    {
        // the kernel's shared-memory limit, once per device
        static std::mutex mu;
        static bool done[kPjMaxDevices] = {};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kPjMaxDevices) return -7;
        std::lock_guard<std::mutex> lk(mu);
        if (!done[dev]) {
            if (cudaFuncSetAttribute(gen_proj_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPjSmemBudget) !=
                cudaSuccess)
                return -7;
            done[dev] = true;
        }
    }
    const unsigned grid = static_cast<unsigned>((m + kPjRows - 1) / kPjRows);
    gen_proj_tc_kernel<<<grid, kPjThreads, static_cast<size_t>(smem), stream>>>(tmA, tmB, p);
    return cudaGetLastError() == cudaSuccess ? 0 : -7;
}

int read_proj_error(unsigned int* word, int clear, cudaStream_t stream) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_hc_proj_error, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return -7;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return -7;
    if (clear && v != 0) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbolAsync(g_hc_proj_error, &z, sizeof(z), 0, cudaMemcpyHostToDevice, stream) != cudaSuccess)
            return -7;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return -7;
    }
    *word = v;
    return 0;
}

}  // namespace hc
