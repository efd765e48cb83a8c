// Projection of the generic path on the 5th-generation tensor cores, for any number of streams hc in
// 1..8 and any width d (a multiple of 8): raw[t][m] = sum_c X'[t][c] w[m][c] over the c < hc*d columns
// of a token's flattened streams, and ssx[t] = sum_c X'[t][c]^2 ("Source layer, pairs pooled" page,
// Block.hc_mixes excerpt: the fp32 projection of the flattened streams onto mix_hc = (2 + hc) * hc
// mixes, and the mean square behind its r). The scaling by r, the split and the norm follow in
// gen_tail_kernel.
//
// The weights are the three bf16 planes of hc_prepare_params, a [3M, hc*d] matrix with
// w = hi + mid + lo exactly (plane_row gives each plane's row). One CTA takes 128 tokens of a chunk
// and streams the hc*d columns in stages of 32: a TMA load of the X' tile [128 x 32] and of the plane
// rows [N x 32], both with the 64-byte swizzle, then two tcgen05.mma kind::f16 (K = 16 each) into a
// TMEM accumulator of N fp32 columns. The planes are loaded through a 3-D view (4-D for the grouping
// the fused kernel uses at hc = 4) whose strides put the three planes of a mix side by side, so that
// accumulator column 3 i + pl holds plane pl of mix slot i; the mix slots are the M mixes padded to a
// multiple of 16 (N = 3 * that), and rows past the planes and columns past hc*d read as zeros. Each
// product of two bf16 values is exact in fp32, so the projection has the accuracy of an fp32 dot
// product.
//
// Two accumulators take blocks of 8 stages in turn. While the tensor cores fill one, four drain
// warps (warp 4 + q: TMEM lanes and tile rows 32q..32q+31) add the other's (hi + mid) + lo of every
// mix into running fp32 sums held in registers: a sum of 256-column partial sums, as the fused
// kernel sums its stages. Four square warps sum the squares of the rows from the shared tiles and
// release the slots, so a drain never holds up the loads. Warp 8 issues the loads, warp 9 the MMAs.
// Every wait is bounded: on expiry the kernel sets a bit in its device error word, stops waiting,
// lets its copies land and frees its tensor memory.

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
constexpr int kPjThreads = 320;                  // warps 0-3 squares, 4-7 drains, 8 loads, 9 MMAs
constexpr int kPjWarpDrain = 4, kPjWarpLoad = 8, kPjWarpMma = 9;
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
    int N;            // accumulator columns: 3 per mix slot (M rounded up to 16 slots)
    int stages;       // ceil(hc * d / 32)
    int slots;        // load ring depth
    int tmem_cols;    // allocated TMEM columns (a power of two >= 2N)
};

// shared-memory layout, the same on host and device
struct ProjLayout {
    int slot_bytes, off_bars, bytes;
    __host__ __device__ ProjLayout(int N, int slots) {
        slot_bytes = kPjATile + N * kPjCols * 2;
        off_bars = slots * slot_bytes;
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

// the mix in mix slot i of the accumulator, or -1 for a padding slot: the slots follow the mixes,
// except at hc = 4, where each half of the 24 mixes fills 12 of 16 slots
__device__ __forceinline__ int mix_of_slot(int hc, int M, int i) {
    if (hc == 4) return i % 16 < 12 ? 12 * (i / 16) + i % 16 : -1;
    return i < M ? i : -1;
}

// kMC: mix slots / 16 (the drain warps' running sums, 16 per chunk, live in registers)
template <int kMC>
__global__ void __launch_bounds__(kPjThreads, 1) gen_proj_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                                                                    const __grid_constant__ CUtensorMap tmB,
                                                                    const ProjParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
    const ProjLayout L(p.N, p.slots);
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
            mbar_init(empty(i), 1 + 4);  // the MMAs' completion + the four square warps
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), 4);  // the four drain warps
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_ptr);

    if (warp == kPjWarpLoad) {
        // ===== TMA: stage s into slot s % slots, once the MMAs and the square warps are done with it =
        if (lane == 0) {
            const uint64_t pol_stream = policy_evict_normal(), pol_keep = policy_evict_last();
            for (int s = 0; s < S; ++s) {
                const int i = s % p.slots, round = s / p.slots;
                if (round > 0) W.wait(empty(i), static_cast<uint32_t>((round - 1) & 1), kPjErrLoad);
                const uint32_t a = sbase + static_cast<uint32_t>(i * L.slot_bytes);
                mbar_arrive_expect_tx(full(i), static_cast<uint32_t>(L.slot_bytes));
                tma_load_2d(a, &tmA, full(i), kPjCols * s, row0, pol_stream);
                if (p.hc == 4)
                    tma_load_4d(a + kPjATile, &tmB, full(i), kPjCols * s, 0, 0, 0, pol_keep);
                else
                    tma_load_3d(a + kPjATile, &tmB, full(i), kPjCols * s, 0, 0, pol_keep);
            }
            // every load lands before the CTA may exit (a slot's last load lands after its earlier ones)
            for (int s = S - p.slots > 0 ? S - p.slots : 0; s < S; ++s)
                W.drain(full(s % p.slots), static_cast<uint32_t>((s / p.slots) & 1));
        }
        __syncwarp();
    } else if (warp == kPjWarpMma) {
        // ===== MMA: block b of 8 stages into accumulator b % 2 =======================================
        const uint32_t idesc = idesc_bf16_f32(kPjRows, p.N);
        for (int s = 0; s < S; ++s) {
            const int i = s % p.slots, round = s / p.slots;
            const int b = s / kPjBlock, buf = b & 1;
            // the accumulator's previous block (b - 2) must have been drained
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
    } else if (warp >= kPjWarpDrain) {
        // ===== drain warps: each block's (hi + mid) + lo of every mix into the running sums ==========
        const int q = warp - kPjWarpDrain;
        const int r = 32 * q + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
        float acc[kMC * 16];
#pragma unroll
        for (int i = 0; i < kMC * 16; ++i) acc[i] = 0.f;
        for (int b = 0; b < nblocks; ++b) {
            const int buf = b & 1;
            W.wait(acc_full(buf), static_cast<uint32_t>((b >> 1) & 1), kPjErrRows);
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < kMC; ++c) {
                // mix slots 16c .. 16c + 15: accumulator columns 48c .. 48c + 47, three planes each
                uint32_t v0[16], v1[16], v2[16];
                const uint32_t col = tl + static_cast<uint32_t>(buf * p.N + 48 * c);
                tmem_ld16_wait(col, v0);
                tmem_ld16_wait(col + 16u, v1);
                tmem_ld16_wait(col + 32u, v2);
                // column k of the 48 (a compile-time index once unrolled)
                auto at = [&](int k) { return __uint_as_float(k < 16 ? v0[k & 15] : k < 32 ? v1[k & 15] : v2[k & 15]); };
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[16 * c + i] += (at(3 * i) + at(3 * i + 1)) + at(3 * i + 2);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(buf));
        }
        const long long t = static_cast<long long>(row0) + r;
        if (t < p.m) {
#pragma unroll
            for (int i = 0; i < kMC * 16; ++i) {
                const int mm = mix_of_slot(p.hc, p.M, i);
                if (mm >= 0) p.raw[t * p.M + mm] = acc[i];
            }
        }
    } else {
        // ===== square warps: the squares of the rows, then the slot goes back to the loads ==========
        const int r = 32 * warp + lane;
        float sq = 0.f;
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
        }
        const long long t = static_cast<long long>(row0) + r;
        if (t < p.m) p.ssx[t] = sq;
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

// a bf16 tensor map of `rank` dimensions (dims[0] = columns, the other strides in bytes) whose box is
// 32 columns by box[1..]
bool encode_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                const uint32_t* box_rest) {
    auto fn = proj_encode_fn();
    if (!fn) return false;
    cuuint64_t gd[4], gs[3];
    cuuint32_t bx[4], es[4];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = i == 0 ? static_cast<cuuint32_t>(kPjCols) : box_rest[i - 1];
        es[i] = 1;
        if (i > 0) gs[i - 1] = strides[i - 1];
    }
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gd, gs, bx,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kMC>
int launch_mc(const CUtensorMap& tmA, const CUtensorMap& tmB, const ProjParams& p, unsigned grid, int smem,
              cudaStream_t stream) {
    // the kernel's shared-memory limit, once per device
    static std::mutex mu;
    static bool done[kPjMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kPjMaxDevices) return -7;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!done[dev]) {
            if (cudaFuncSetAttribute(gen_proj_tc_kernel<kMC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kPjSmemBudget) != cudaSuccess)
                return -7;
            done[dev] = true;
        }
    }
    gen_proj_tc_kernel<kMC><<<grid, kPjThreads, static_cast<size_t>(smem), stream>>>(tmA, tmB, p);
    return cudaGetLastError() == cudaSuccess ? 0 : -7;
}

}  // namespace

int launch_proj_tc(const void* X, const void* planes, int64_t m, int hc, int d, float* raw, float* ssx,
                   cudaStream_t stream) {
    if (m <= 0) return 0;
    if (hc < 1 || hc > 8 || d % 8 != 0) return -3;
    const int M = (2 + hc) * hc;
    const int slots_mix = hc == 4 ? 32 : (M + 15) / 16 * 16;  // mix slots, a multiple of 16
    const int N = 3 * slots_mix;                               // at most 240
    const uint64_t D = static_cast<uint64_t>(hc) * static_cast<uint64_t>(d);
    int slots = kPjMaxSlots;
    while (slots > 2 && ProjLayout(N, slots).bytes + 1024 > kPjSmemBudget) --slots;
    const int smem = ProjLayout(N, slots).bytes + 1024;
    int tcols = 32;
    while (tcols < 2 * N) tcols *= 2;
    CUtensorMap tmA, tmB;
    {
        const uint64_t dims[2] = {D, static_cast<uint64_t>(m)};
        const uint64_t str[1] = {D * 2};
        const uint32_t box[1] = {static_cast<uint32_t>(kPjRows)};
        if (!encode_map(&tmA, X, 2, dims, str, box)) return -7;
    }
    if (hc == 4) {
        // plane rows 36 h + 12 pl + i (mix 12 h + i): [h][i][pl] with i padded to 16
        const uint64_t dims[4] = {D, 3, 12, 2};
        const uint64_t str[3] = {12 * D * 2, D * 2, 36 * D * 2};
        const uint32_t box[3] = {3, 16, 2};
        if (!encode_map(&tmB, planes, 4, dims, str, box)) return -7;
    } else {
        // plane rows pl * M + m: [m][pl], m padded to the mix slots
        const uint64_t dims[3] = {D, 3, static_cast<uint64_t>(M)};
        const uint64_t str[2] = {static_cast<uint64_t>(M) * D * 2, D * 2};
        const uint32_t box[2] = {3, static_cast<uint32_t>(slots_mix)};
        if (!encode_map(&tmB, planes, 3, dims, str, box)) return -7;
    }
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
    const unsigned grid = static_cast<unsigned>((m + kPjRows - 1) / kPjRows);
    switch (slots_mix / 16) {
        case 1: return launch_mc<1>(tmA, tmB, p, grid, smem, stream);
        case 2: return launch_mc<2>(tmA, tmB, p, grid, smem, stream);
        case 3: return launch_mc<3>(tmA, tmB, p, grid, smem, stream);
        case 4: return launch_mc<4>(tmA, tmB, p, grid, smem, stream);
        case 5: return launch_mc<5>(tmA, tmB, p, grid, smem, stream);
        default: return -3;
    }
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
