// Fused Hyper-Connection stream step for GB300 (sm_103a).
//
// One launch computes, per token (DeepSeek V4.1 model-atlas pages):
//   [post mode] X' = bf16(post_k * Delta + sum_j comb[j,k] * X_j)      "Write the streams" page,
//                                                                      formula for X'_{n,k}
//   r     = 1/sqrt(mean(X'^2 over all 4*d values) + norm_eps)         "Source layer, pairs pooled"
//   mixes = r * (X'_flat . hc_fn^T)        (24 numbers)                page, Block.hc_mixes excerpt
//   pre / post / comb from mixes: sigmoid, 2*sigmoid, softmax rows     "Reading weights" page,
//            + eps then Sinkhorn column/row normalisation             hc_split_sinkhorn excerpt
//   y        = bf16(sum_j pre_mix_j * X'_j)                            Block.hc_pre excerpt
//   y_normed = bf16(norm_w * y / sqrt(mean(y^2) + norm_eps))           "Final RMSNorm" page,
//                                                                      RMSNorm excerpt
// In pre-step mode X' is the input X itself and nothing is written back to the streams. In expand
// mode (the head of the stack, "Final RMSNorm" page, Transformer.forward excerpt) X' is the
// embedding row h in every stream: h is loaded once per stage, serves as the MMA operand of all
// four streams, is written four times to the streams, and the identity pre_mix (1/4 each)
// collapses the four copies back to h exactly.
//
// Decomposition. A group of kG CTAs (8 for large batches; 16 or 32 for small ones, so that each CTA
// has fewer column stages) owns a tile of up to 128 tokens; CTA `rank` of the group owns d/kG
// columns of every stream, the 32-column chunks rank, rank+kG, rank+2kG, ... (interleaved, so the
// group's loads of one stage cover kG*32 contiguous columns of each row). The 16 warps of a CTA
// have fixed roles:
//   producer (warp 8): per 32-column stage, TMA-loads the four X tiles [tokens x 32 cols] (expand
//     mode: the one embedding tile), the Delta tile (post mode) and the four matching slices of
//     the split projection weights (bf16 planes hi/mid/lo, 72 rows) into a ring of shared-memory
//     slots, 64-byte swizzled: 3 slots in post mode, 4 in pre mode, 6 in expand mode;
//   compute (warps 0-7, thread = token, two warps per TMEM lane quadrant, 16 columns each):
//     compute X' in place (post mode; the other modes read the loaded tile), accumulate sum(X'^2),
//     form and round y, accumulate sum(y^2), store the bf16 y chunk into a ring of 27 chunk slots
//     in tensor memory, and drain the previous stage's accumulator into 12 per-thread fp32 sums
//     (the three planes added back together);
//   MMA (warp 9): one thread issues 8 tcgen05.mma per stage (M=128 tokens, N=80 >= 72 plane
//     rows, K=16) projecting the bf16 X' tile on the three planes into a TMEM accumulator; the
//     products are exact in fp32, so the split projection has fp32-FFMA accuracy;
//   store (warp 10): TMA-stores the X' tile (written once) from the same slot, then frees it;
//   split (warp 11): at each tile end, publishes the CTA's partial sums (28 per token, in a
//     caller-provided global workspace) with a release flag, waits (bounded) for the other flags
//     of the group, gathers the mixes of its own tokens (t % kG == rank) over the group's blocks,
//     and runs their split and Sinkhorn;
//   epilogue (warps 12-15, one per TMEM lane quadrant): turn the group's sums of y^2 into r_y of
//     the warp's rows, read each y chunk back from the ring, scale it by norm_w and r_y into a
//     32-row swizzled staging tile and TMA-store it to y_normed.
// The ring holds a tile's y until the exchange gives r_y, with 7 stages of slack at 20 stages a
// tile: the compute warps stream on into the next tile while the group finishes the previous one.
// The groups are formed in software rather than as hardware clusters because only 15 clusters of
// 8 CTAs fit on a GB300 at once (120 of its 152 SMs); the launch is cooperative, so all CTAs are
// resident together and the flag waits between them cannot deadlock.
//
// Every wait on an mbarrier is bounded in time; on expiry the kernel records an error in a
// device word, stops waiting everywhere, finishes its loops without hanging, frees its tensor
// memory and returns.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <mutex>

#include "hc_internal.h"
#include "hc_ptx.cuh"

namespace hc {

constexpr int kMix = 24;
constexpr int kBRows = 72;        // 3 planes x 24 mixes
constexpr int kUmmaM = 128;
constexpr int kUmmaN = 80;        // smallest legal N >= 72 at M = 128
// A group of kG CTAs (8, 16 or 32, a template parameter) shares one token tile, each CTA taking
// d/kG columns; small batches use larger groups so that each CTA has fewer column stages.
constexpr int kMaxCtas = 256;      // workspace capacity: up to 256 co-resident CTAs
constexpr int kMaxGroups = 32;     // launch counters: group slots (at most 256 / 8)
constexpr int kFlagRanks = 32;     // flags per (group slot, tile parity): the largest group
constexpr int kTileMax = 128;
constexpr int kChunk = 32;        // columns per stage: 64-byte rows
constexpr int kMaxStages = 6;
constexpr int kComputeWarps = 8;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpStore = 10;
constexpr int kWarpSplit = 11;
constexpr int kWarpEpi0 = 12;       // warps 12..15: y_normed epilogue, TMEM lane quadrant = warp % 4
constexpr int kThreads = 16 * 32;
constexpr int kMaxDSlice = 640;   // d <= 5120

constexpr int kXTileBytes = kTileMax * kChunk * 2;            // 8192: 128 rows x 64 B
constexpr int kBTileBytes = kBRows * kChunk * 2;              // 4608: 72 rows x 64 B (the MMA reads
                                                              // 80 rows; rows 72..79 are ignored)
// One CTA's partial sums for one tile: mixes [128 tokens][24] (token-major), then
// sum x^2 [128 tokens][2 column halves], then sum y^2 [128][2] (a token's two halves adjacent).
constexpr int kPartRows = 28;
constexpr int kPartFloats = kPartRows * kTileMax;
constexpr int kPartSx = kMix * kTileMax, kPartSy = kPartSx + 2 * kTileMax;
constexpr int kYStageBytes = 32 * kChunk * 2;                              // 2048
// mbarriers, numbered for up to kMaxStages shared-memory slots
constexpr int kBarFull = 0, kBarXReady = 6, kBarEmpty = 12, kBarAccFull = 18, kBarAccEmpty = 19, kBarMmaDone = 20;
// kBarFlagsSeen[2] (per tile parity): the split warp has seen the group's flags of a tile, so the
// epilogue warps may read its sums of y^2. kBarEpiRead: the epilogue warps have read them (one
// arrival per warp per tile); the split warp publishes the next tile only after that.
constexpr int kBarSplitDone = 21, kBarFlagsSeen = 22, kBarEpiRead = 24, kBarYReady = 25, kBarYFree = 25 + 27;
// kBarPublish: the compute warps have written the CTA's partial sums of a tile (one arrival per
// warp), the split warp waits before publishing them. kBarExit: every warp is done (one arrival per
// warp) before TMEM is freed. The CTA-wide hardware barriers are not used after the set-up: in
// this kernel, whose warps spend most of their time in mbarrier waits, a block-wide bar.sync at
// the end was measured releasing warp 0 while other warps had not reached it; mbarriers hold.
constexpr int kBarPublish = 25 + 2 * 27, kBarExit = kBarPublish + 1;
constexpr int kNumBars = kBarExit + 1;

// Shared-memory layout of each mode, offsets from a 1024-byte aligned base. A slot holds one column
// stage: the stream tiles (four, or the one embedding tile in expand mode), the Delta tile (post
// mode only) and the four weight-plane tiles. The smaller slots of the reading-only modes buy more
// of them, so more loads are in flight while the stage's MMA holds its slot: post 3 x 59392 B,
// pre 4 x 51200 B, expand 6 x 26624 B. After the slots: norm_w of the CTA's columns, the epilogue
// warps' y_normed staging tiles (per warp two 32-row x 64-byte tiles, 64-byte swizzle, filled and
// TMA-stored in turn), the mbarriers, the TMEM address and the abort word.
template <int kMode>
struct Layout {
    static constexpr int kXTiles = kMode == kModeExpand ? 1 : 4;
    static constexpr int kOffX = 0;
    static constexpr int kOffD = kXTiles * kXTileBytes;
    static constexpr int kOffB = kOffD + (kMode == kModePost ? kXTileBytes : 0);
    static constexpr int kStage = kOffB + 4 * kBTileBytes;
    static constexpr int kStages = kMode == kModePost ? 3 : kMode == kModePre ? 4 : 6;
    static constexpr int kOffNormW = kStages * kStage;
    static constexpr int kOffYStage = ((kOffNormW + kMaxDSlice * 4 + 1023) / 1024) * 1024;
    static constexpr int kOffBar = kOffYStage + 4 * 2 * kYStageBytes;
    static constexpr int kOffTmemPtr = kOffBar + kNumBars * 8;
    static constexpr int kOffAbort = kOffTmemPtr + 4;
    static constexpr int kSmemUsed = kOffAbort + 4;
    static constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for aligning the base
    static_assert(kStage % 1024 == 0, "stage buffers keep 1024-byte alignment");
    static_assert(kOffB % 512 == 0 && kBTileBytes % 512 == 0, "B tiles start on 512-byte swizzle atoms");
    static_assert(kStages <= kMaxStages, "barrier numbering");
    static_assert(kSmemBytes <= 232448, "fits the 227 KB opt-in shared memory of one CTA");
    // the MMA of the last B tile of the last slot reads 8 rows (512 B) past it: into norm_w, inside the CTA
    static_assert(kOffB + 3 * kBTileBytes + kUmmaN * 64 + (kStages - 1) * kStage <= kSmemUsed, "B overrun");
};

// global workspace: partial sums [group][tile parity][rank][28][128] fp32 (a block per CTA and
// tile parity), then 64-bit flags [group slot][tile parity][32 ranks], then one 64-bit launch
// counter per group slot. A flag slot is always tagged from the same counter, whatever the group
// size of the launch that writes it, so tags never repeat on one workspace. A flag holds
// (launch number of its group) << 32 | (tile index + 1); the launch number is the group's counter
// + 1, read by every CTA of the group when it starts and stored back by the group's rank-0 CTA
// after its last exchange, when all 8 have read it. The tags therefore come from the device: a
// launch replayed from a CUDA graph tags its flags afresh, and a zero-filled workspace holds no tag.
constexpr size_t kWsPartBytes = static_cast<size_t>(kMaxCtas) * 2 * kPartFloats * 4;
constexpr size_t kWsFlagBytes = static_cast<size_t>(kMaxGroups) * 2 * kFlagRanks * 8;
constexpr size_t kWsCounterBytes = static_cast<size_t>(kMaxGroups) * 8;
constexpr size_t kWorkspaceBytes = kWsPartBytes + kWsFlagBytes + kWsCounterBytes;

static_assert(kWarpEpi0 + 4 == kThreads / 32 && kWarpEpi0 % 4 == 0, "one epilogue warp per TMEM lane quadrant");
static_assert(kWarpSplit + 1 == kWarpEpi0, "warp roles: 8 compute, producer, MMA, store, split, 4 epilogue");

// TMEM: one accumulator (N = 80 columns), then a ring of kRing y chunks of 16 columns each
// (32 rows x 16 bf16 pairs per warp quadrant). A tile has at most 20 stages, so the compute warps
// can run 7 stages into the next tile before they must have stored the previous tile's y.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0, kYCol = 80;
constexpr int kRing = 27;
static_assert(kYCol + kRing * 16 <= kTmemCols, "y ring fits in TMEM");
static_assert(kBarYFree == kBarYReady + kRing, "one ready and one free barrier per ring slot");

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

// L2 handling of the streamed tiles (X, Delta): cache-hint policy of the loads (0 evict_normal,
// 1 evict_first, 2 evict_last) and the L2 promotion of their tensor maps.
#ifndef HC_STREAM_POLICY
#define HC_STREAM_POLICY 0
#endif
#ifndef HC_STREAM_PROMOTION
#define HC_STREAM_PROMOTION CU_TENSOR_MAP_L2_PROMOTION_L2_128B
#endif

// device error word: bit set = which wait gave up
__device__ unsigned int g_hc_error = 0;
enum : unsigned int {
    kErrProducer = 1u, kErrMma = 2u, kErrComputeFull = 4u, kErrComputeAcc = 8u, kErrStore = 16u, kErrDrain = 32u,
    kErrExchange = 64u, kErrSplit = 128u, kErrEpilogue = 256u, kErrComputeY = 512u
};

struct FusedParams {
    const float* post;
    const float* comb;
    const float* pre_mix;
    const float* hc_scale;
    const float* hc_base;
    const float* norm_w;
    float* pre_out;
    float* post_out;
    float* comb_out;
    float* mixes_out;
    void* stream_mean;              // bf16 [n, d] mean of the 4 new streams, or null
    void* y_normed;
    float* ws_part;                 // workspace partial-sum blocks
    unsigned long long* ws_flags;   // workspace flags
    unsigned long long* ws_launch;  // workspace launch counters, one per group
    long long n;
    long long num_tiles;
    int write_y;
    int d;
    int d_slice;
    int stages_per_tile;
    int tile_m;
    int iters;
    float hc_eps;
    float norm_eps;
};

// ---- small helpers ------------------------------------------------------------------------------

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);  // a -> low half
    return *reinterpret_cast<uint32_t*>(&v);
}

// Pairs of adjacent columns travel as float2 through the packed fp32 instructions of sm_100+
// (__ffma2_rn and friends: two independent IEEE operations per instruction, each lane rounded
// exactly like its scalar counterpart).
__device__ __forceinline__ float2 bf2(uint32_t u) { return make_float2(bf_lo(u), bf_hi(u)); }
__device__ __forceinline__ uint32_t pack_bf16(float2 v) { return pack_bf16(v.x, v.y); }
__device__ __forceinline__ float2 bcast(float a) { return make_float2(a, a); }

__device__ __forceinline__ void unpack4(const uint4& v, float2 (&f)[4]) {
    f[0] = bf2(v.x); f[1] = bf2(v.y); f[2] = bf2(v.z); f[3] = bf2(v.w);
}

// Bounded mbarrier wait shared by all roles of one CTA.
struct Waiter {
    volatile uint32_t* abort;
    uint64_t limit_ns = kWaitLimitNs;
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, unsigned int code) const {
        if (mbar_test(bar, parity)) return true;
        const uint64_t t0 = global_timer_ns();
        while (true) {
            for (int i = 0; i < 32; ++i)
                if (mbar_test(bar, parity)) return true;
            if (*abort) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                *abort = 1u;
                atomicOr(&g_hc_error, code);
                return false;
            }
        }
    }
    // Whole warp: lanes 0..g-1 each wait for flag f[lane] to equal `epoch`; returns when all g do.
    __device__ __forceinline__ bool wait_flags_warp(const unsigned long long* f, unsigned long long epoch, int lane,
                                                    int g, unsigned int code) const {
        const uint64_t t0 = global_timer_ns();
        bool mine = lane >= g;
        while (true) {
            if (!mine) mine = ld_acquire_gpu_u64(f + lane) == epoch;
            if (__all_sync(0xffffffffu, mine)) return true;
            const bool aborted = *abort != 0u;
            const bool late = global_timer_ns() - t0 > limit_ns;
            if (__any_sync(0xffffffffu, aborted || late)) {  // one decision for the whole warp
                if (lane == 0 && !aborted) {
                    *abort = 1u;
                    atomicOr(&g_hc_error, code);
                }
                __syncwarp();
                return false;
            }
        }
    }
    // Same as wait, but ignores an abort raised elsewhere: used at exit to let copies in flight land.
    __device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) const {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_test(bar, parity)) {
            if (global_timer_ns() - t0 > limit_ns) {
                atomicOr(&g_hc_error, kErrDrain);
                return;
            }
        }
    }
};

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

// "Reading weights" page, hc_split_sinkhorn kernel excerpt and the formula for p, in fp32. Every
// normalisation multiplies by a reciprocal of its sum taken as the hardware approximation refined
// by one Newton-Raphson step (about 1 ulp; the sums are at least eps or 1, never subnormal): the
// 2 * iters dependent normalisations run several times faster than with correctly rounded
// reciprocals, which matters when a small batch waits for them, and the refinement keeps 50 rounds
// on extreme logits inside the coefficients' 1e-5 tolerance, which the bare approximation did not.
__device__ __forceinline__ void split_sinkhorn(const float (&m)[kMix], const float (&sc)[3], const float (&b)[kMix],
                                               int iters, float eps, float (&pre)[4], float (&post)[4],
                                               float (&C)[16]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) pre[j] = sigmoidf_(m[j] * sc[0] + b[j]) + eps;
#pragma unroll
    for (int j = 0; j < 4; ++j) post[j] = 2.0f * sigmoidf_(m[4 + j] * sc[1] + b[4 + j]);
#pragma unroll
    for (int q = 0; q < 16; ++q) C[q] = m[8 + q] * sc[2] + b[8 + q];
    // softmax over each row (max subtracted), then + eps
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float mx = fmaxf(fmaxf(C[4 * j], C[4 * j + 1]), fmaxf(C[4 * j + 2], C[4 * j + 3]));
        float e0 = expf(C[4 * j] - mx), e1 = expf(C[4 * j + 1] - mx);
        float e2 = expf(C[4 * j + 2] - mx), e3 = expf(C[4 * j + 3] - mx);
        float inv = rcp_refined((e0 + e1) + (e2 + e3));
        C[4 * j] = e0 * inv + eps;
        C[4 * j + 1] = e1 * inv + eps;
        C[4 * j + 2] = e2 * inv + eps;
        C[4 * j + 3] = e3 * inv + eps;
    }
    auto col_norm = [&]() {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float inv = rcp_refined(((C[k] + C[4 + k]) + (C[8 + k] + C[12 + k])) + eps);
            C[k] *= inv;
            C[4 + k] *= inv;
            C[8 + k] *= inv;
            C[12 + k] *= inv;
        }
    };
    auto row_norm = [&]() {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float inv = rcp_refined(((C[4 * j] + C[4 * j + 1]) + (C[4 * j + 2] + C[4 * j + 3])) + eps);
            C[4 * j] *= inv;
            C[4 * j + 1] *= inv;
            C[4 * j + 2] *= inv;
            C[4 * j + 3] *= inv;
        }
    };
    col_norm();
    for (int it = 1; it < iters; ++it) {
        row_norm();
        col_norm();
    }
}

// ---- diagnostic: one bounded wait on an exchange flag ------------------------------------------------
// One warp waits, exactly as the fused kernel's split warp waits for its group, for flags f[0..g-1]
// to equal `value`, giving up after limit_ns: it then records kErrExchange in the device error word
// and returns. Lets a test make a wait run out (on flags nothing sets) and check what the host sees.
__global__ void hc_wait_flag_kernel(const unsigned long long* f, unsigned long long value, int g, uint64_t limit_ns) {
    __shared__ uint32_t abort_word;
    if (threadIdx.x == 0) abort_word = 0u;
    __syncwarp();
    const Waiter W{&abort_word, limit_ns};
    W.wait_flags_warp(f, value, static_cast<int>(threadIdx.x), g, kErrExchange);
}

// ---- the kernel ---------------------------------------------------------------------------------

template <int kMode, int kG>
__global__ void __launch_bounds__(kThreads, 1)
    hc_fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmD,
                    const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmXo,
                    const __grid_constant__ CUtensorMap tmM, const __grid_constant__ CUtensorMap tmY,
                    const __grid_constant__ CUtensorMap tmYr, const FusedParams p) {
    using Lay = Layout<kMode>;
    constexpr int kStages = Lay::kStages, kStageBytes = Lay::kStage;
    constexpr int kOffX = Lay::kOffX, kOffD = Lay::kOffD, kOffB = Lay::kOffB, kOffNormW = Lay::kOffNormW;
    constexpr int kOffYStage = Lay::kOffYStage, kOffBar = Lay::kOffBar, kOffTmemPtr = Lay::kOffTmemPtr;
    constexpr int kOffAbort = Lay::kOffAbort;
    constexpr bool kPost = kMode == kModePost;
    constexpr bool kExpand = kMode == kModeExpand;
    constexpr bool kWriteX = kPost || kExpand;  // X' goes back to the streams
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    static_assert(kG == 8 || kG == 16 || kG == 32, "group sizes");
    const uint32_t rank = blockIdx.x % kG;    // column share of this CTA
    const uint32_t cid = blockIdx.x / kG;     // group: owns tiles cid, cid + ncl, ...
    const uint32_t ncl = gridDim.x / kG;
    // first column of stage s of this CTA: the kG CTAs of a group take interleaved 32-column
    // chunks, so at any moment they read and write kG * 64 contiguous bytes of each stream row
    auto stage_col = [&](int s) -> int { return (s * kG + static_cast<int>(rank)) * kChunk; };
    const int S = p.stages_per_tile;

    auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * static_cast<uint32_t>(i); };
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kOffAbort);
    const Waiter W{abort_flag, kWaitLimitNs};

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(kBarFull + s), 1);
            mbar_init(bar(kBarXReady + s), kComputeWarps);
            mbar_init(bar(kBarEmpty + s), 2);  // MMA completion + X' store done reading
        }
        mbar_init(bar(kBarAccFull), 1);
        mbar_init(bar(kBarAccEmpty), kComputeWarps);
        mbar_init(bar(kBarMmaDone), 1);
        mbar_init(bar(kBarSplitDone), 1);
        for (int b = 0; b < 2; ++b) mbar_init(bar(kBarFlagsSeen + b), 1);
        mbar_init(bar(kBarEpiRead), 4);  // the epilogue warps
        for (int r = 0; r < kRing; ++r) {
            mbar_init(bar(kBarYReady + r), kComputeWarps);
            mbar_init(bar(kBarYFree + r), 4);
        }
        mbar_init(bar(kBarPublish), kComputeWarps);
        mbar_init(bar(kBarExit), kThreads / 32);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == kWarpProducer && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmB);
        if (kWriteX) tma_prefetch_desc(&tmD);
    }
    {
        float* nw = reinterpret_cast<float*>(smem + kOffNormW);
        for (int i = threadIdx.x; i < p.d_slice; i += kThreads) nw[i] = p.norm_w[stage_col(i / kChunk) + i % kChunk];
    }
    if (warp == 0) {
        tmem_alloc(sbase + kOffTmemPtr, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemPtr);

    const long long my_tiles =
        (static_cast<long long>(cid) < p.num_tiles) ? (p.num_tiles - 1 - cid) / ncl + 1 : 0;

    if (warp < kComputeWarps) {
        // ================= compute warps: X', sums, y, accumulator drain ========================
        const int q = warp & 3;             // TMEM lane quadrant = token rows 32q..32q+31
        const int h = warp >> 2;            // column half of each 32-column stage
        const int row = 32 * q + lane;      // token row inside the tile
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
        long long g = 0;        // global stage counter (same sequence in every role)
        // tell the epilogue warps that the y chunk of stage gy is in TMEM
        auto y_ready = [&](long long gy) {
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarYReady + static_cast<int>(gy % kRing)));
        };
        for (long long it = 0; it < my_tiles; ++it) {
            const long long tile = cid + it * ncl;
            const long long t0 = tile * p.tile_m;
            const long long tok = t0 + row;
            const bool valid = (row < p.tile_m) && (tok < p.n);
            // this token's coefficients, each broadcast to both lanes of a float2
            float2 cpost[4], ccomb[16], pm[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) cpost[i] = pm[i] = bcast(0.f);
#pragma unroll
            for (int i = 0; i < 16; ++i) ccomb[i] = bcast(0.f);
            if (kExpand) {
                pm[0] = pm[1] = pm[2] = pm[3] = bcast(0.25f);  // identity pre_mix
            } else if (valid) {
                if (p.pre_mix) {
                    float4 v = __ldg(reinterpret_cast<const float4*>(p.pre_mix) + tok);
                    pm[0] = bcast(v.x); pm[1] = bcast(v.y); pm[2] = bcast(v.z); pm[3] = bcast(v.w);
                }
                if (kPost) {
                    float4 v = __ldg(reinterpret_cast<const float4*>(p.post) + tok);
                    cpost[0] = bcast(v.x); cpost[1] = bcast(v.y); cpost[2] = bcast(v.z); cpost[3] = bcast(v.w);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float4 c = __ldg(reinterpret_cast<const float4*>(p.comb) + tok * 4 + j);
                        ccomb[4 * j] = bcast(c.x); ccomb[4 * j + 1] = bcast(c.y);
                        ccomb[4 * j + 2] = bcast(c.z); ccomb[4 * j + 3] = bcast(c.w);
                    }
                }
            }
            float2 acc[6];  // the 12 mixes of this thread's column half, in pairs
#pragma unroll
            for (int i = 0; i < 6; ++i) acc[i] = bcast(0.f);
            float2 sx[4], sy[2];  // sums of squares, each split over the two lanes
#pragma unroll
            for (int i = 0; i < 4; ++i) sx[i] = bcast(0.f);
            sy[0] = sy[1] = bcast(0.f);

            auto drain = [&](long long gd) {
                W.wait(bar(kBarAccFull), static_cast<uint32_t>(gd & 1), kErrComputeAcc);
                tc_fence_after();
                uint32_t v[36];
                const uint32_t col = kAccCol + 36u * h;
                tmem_ld36_wait(tl + col, tl + col + 32u, v);
                auto f2 = [&](int i) { return make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])); };
#pragma unroll
                for (int i = 0; i < 6; ++i)
                    acc[i] = __fadd2_rn(acc[i], __fadd2_rn(__fadd2_rn(f2(2 * i), f2(12 + 2 * i)), f2(24 + 2 * i)));
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarAccEmpty));
            };

            for (int s = 0; s < S; ++s, ++g) {
                // the y store of the previous stage has had a stage to complete: hand it over
                if (s > 0) y_ready(g - 1);
                // reading-only modes: the MMA of this stage reads the tile as loaded, so it may start
                // as soon as the data lands; drain the previous stage's accumulator first to let it
                if (!kPost && s > 0) drain(g - 1);
                // the ring slot of this stage's y last held the chunk of stage g - kRing
                const long long yround = g / kRing;
                if (yround > 0)
                    W.wait(bar(kBarYFree + static_cast<int>(g % kRing)), static_cast<uint32_t>((yround - 1) & 1),
                           kErrComputeY);
                const int slot = static_cast<int>(g % kStages);
                const uint32_t par = static_cast<uint32_t>((g / kStages) & 1);
                W.wait(bar(kBarFull + slot), par, kErrComputeFull);
                const uint32_t sb = sbase + slot * kStageBytes;
                uint32_t yb[8];
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int c = 2 * h + cc;
                    const uint32_t off = static_cast<uint32_t>(row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
                    float2 xr[4][4];  // X' of the 8 columns, 4 pairs per stream
                    uint4 xv[4];
                    if (kExpand) {
                        xv[0] = ld_smem_v4(sb + kOffX + off);  // h, the same in every stream
                        xv[1] = xv[0];
                        xv[2] = xv[0];
                        xv[3] = xv[0];
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j) xv[j] = ld_smem_v4(sb + kOffX + j * kXTileBytes + off);
                    }
                    if (kPost) {
                        // X'_k = post_k * Delta + sum_j comb[j,k] X_j, in this order for every column
                        float2 dl[4], xf[4][4];
                        unpack4(ld_smem_v4(sb + kOffD + off), dl);
#pragma unroll
                        for (int j = 0; j < 4; ++j) unpack4(xv[j], xf[j]);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            uint32_t o[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                float2 t = __fmul2_rn(cpost[k], dl[e]);
                                t = __ffma2_rn(ccomb[0 * 4 + k], xf[0][e], t);
                                t = __ffma2_rn(ccomb[1 * 4 + k], xf[1][e], t);
                                t = __ffma2_rn(ccomb[2 * 4 + k], xf[2][e], t);
                                t = __ffma2_rn(ccomb[3 * 4 + k], xf[3][e], t);
                                o[e] = pack_bf16(t);
                            }
                            const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
                            st_smem_v4(sb + kOffX + k * kXTileBytes + off, ov);
                            unpack4(ov, xr[k]);
                        }
                        if (p.stream_mean) {
                            // the multi-token-prediction tap: bf16(mean_j X'_j), summed in fp32, written
                            // over this thread's own (already read) Delta chunk; the store warp sends
                            // the tile out with the X' tiles
                            uint32_t o[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                float2 t = __fadd2_rn(__fadd2_rn(__fadd2_rn(xr[0][e], xr[1][e]), xr[2][e]), xr[3][e]);
                                o[e] = pack_bf16(__fmul2_rn(t, bcast(0.25f)));
                            }
                            st_smem_v4(sb + kOffD + off, make_uint4(o[0], o[1], o[2], o[3]));
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j) unpack4(xv[j], xr[j]);
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k)
#pragma unroll
                        for (int e = 0; e < 4; ++e) sx[k] = __ffma2_rn(xr[k][e], xr[k][e], sx[k]);
                    // y = sum_j pre_mix_j X'_j, rounded to bf16; its squares summed from the rounded values
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float2 t = __fmul2_rn(pm[0], xr[0][e]);
                        t = __ffma2_rn(pm[1], xr[1][e], t);
                        t = __ffma2_rn(pm[2], xr[2][e], t);
                        t = __ffma2_rn(pm[3], xr[3][e], t);
                        const uint32_t u = pack_bf16(t);
                        yb[cc * 4 + e] = u;
                        const float2 a = bf2(u);
                        sy[cc] = __ffma2_rn(a, a, sy[cc]);
                    }
                }
                tmem_st8(tl + kYCol + static_cast<uint32_t>((g % kRing) * 16 + h * 8), yb);
                if (kPost) fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarXReady + slot));
                // drain the previous stage's accumulator now: its MMA ran while this stage was
                // computed, so nothing waits here, and the MMA of this stage (which needs the
                // accumulator empty) is issued right after
                if (kPost && s > 0) drain(g - 1);
            }
            drain(g - 1);
            y_ready(g - 1);

            // publish this CTA's partial sums of the tile to the group; the split warp collects them.
            // The block of tile it reuses that of tile it - 2, which the other CTAs of the group may
            // still be reading; each of them publishes tile it - 1 only after it has read tile it - 2,
            // and this CTA's split warp signals split_done(it - 1) only after it has seen all those
            // flags (and read tile it - 1 itself).
            if (it > 0) W.wait(bar(kBarSplitDone), static_cast<uint32_t>((it - 1) & 1), kErrExchange);
            const int buf = static_cast<int>(it & 1);
            float* P = p.ws_part + (static_cast<size_t>(cid * 2 + buf) * kG + rank) * kPartFloats;
            {
                float4* pm4 = reinterpret_cast<float4*>(P + row * kMix + 12 * h);
                pm4[0] = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
                pm4[1] = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
                pm4[2] = make_float4(acc[4].x, acc[4].y, acc[5].x, acc[5].y);
            }
            const float2 sxx = __fadd2_rn(__fadd2_rn(sx[0], sx[1]), __fadd2_rn(sx[2], sx[3]));
            const float2 syy = __fadd2_rn(sy[0], sy[1]);
            P[kPartSx + 2 * row + h] = sxx.x + sxx.y;
            P[kPartSy + 2 * row + h] = syy.x + syy.y;
            // hand the block to the split warp, which publishes it; no waiting here
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarPublish));
        }
    } else if (warp >= kWarpEpi0) {
        // ================= epilogue warps: y_normed = bf16(norm_w * y * r_y), one quadrant each ===
        const int q = warp & 3;
        const int row = 32 * q + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
        const float* nw = reinterpret_cast<const float*>(smem + kOffNormW);
        const float inv_d = 1.0f / static_cast<float>(p.d);
        long long g = 0;
        long long ystores = 0;  // TMA stores this warp has issued (staging tiles alternate)
        for (long long it = 0; it < my_tiles; ++it) {
            const int buf = static_cast<int>(it & 1);
            // r_y of this thread's row from the group's sums of y^2 (2 halves of each of the kG
            // column shares), once the split warp has seen all their flags
            W.wait(bar(kBarFlagsSeen + buf), static_cast<uint32_t>((it >> 1) & 1), kErrEpilogue);
            const float* blk =
                p.ws_part + (static_cast<size_t>(cid * 2 + buf) * kG) * kPartFloats + kPartSy + 2 * row;
            // all kG loads in flight at once (one L2 round trip), summed in share order
            float2 sq[kG];
#pragma unroll
            for (int r = 0; r < kG; ++r) sq[r] = ld_cg_f2(blk + static_cast<size_t>(r) * kPartFloats);
            float ssq = 0.f;
#pragma unroll
            for (int r = 0; r < kG; ++r) ssq += sq[r].x + sq[r].y;
            const float ry = 1.0f / sqrtf(ssq * inv_d + p.norm_eps);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarEpiRead));  // this warp is done with the tile's blocks
            const long long t0 = (cid + it * ncl) * p.tile_m;
            // this warp's rows go out as one TMA tile: 32 rows, or the tile's last tile_m % 32 rows
            // through the second map (rows past n are clipped by the maps; rows past tile_m belong
            // to the next tile and are never stored)
            const int rows_q = p.tile_m - 32 * q;
            const bool store = p.write_y && rows_q > 0;
            const CUtensorMap* ymap = rows_q >= 32 ? &tmY : &tmYr;
            for (int s = 0; s < S; ++s, ++g) {
                const int ys = static_cast<int>(g % kRing);
                W.wait(bar(kBarYReady + ys), static_cast<uint32_t>((g / kRing) & 1), kErrEpilogue);
                tc_fence_after();
                uint32_t yv[16];
                tmem_ld16_wait(tl + kYCol + static_cast<uint32_t>(ys * 16), yv);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarYFree + ys));
                if (store) {
                    // TMEM columns ys*16 + 0..7 hold stage columns 0..15 (half 0), + 8..15 hold 16..31;
                    // y_normed = norm_w * (y * r_y), two columns per instruction
                    const float2* w = reinterpret_cast<const float2*>(nw + s * 32);
                    const float2 ry2 = bcast(ry);
                    uint32_t ov[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) ov[e] = pack_bf16(__fmul2_rn(w[e], __fmul2_rn(bf2(yv[e]), ry2)));
                    // staging tile (alternating): the store issued from it two stages ago must have read it
                    const uint32_t st = sbase + kOffYStage + static_cast<uint32_t>((q * 2 + (ystores & 1)) * kYStageBytes);
                    if (lane == 0 && ystores >= 2) bulk_wait_read<1>();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        st_smem_v4(st + static_cast<uint32_t>(lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)),
                                   make_uint4(ov[4 * j], ov[4 * j + 1], ov[4 * j + 2], ov[4 * j + 3]));
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(ymap, st, stage_col(s), static_cast<int>(t0 + 32 * q));
                        bulk_commit();
                    }
                    ++ystores;
                }
            }
        }
        if (lane == 0) bulk_wait<0>();  // this warp's y_normed stores are complete
        __syncwarp();
    } else if (warp == kWarpProducer) {
        // ================= TMA producer =========================================================
        uint64_t pol_stream = 0, pol_keep = 0;
        if (lane == 0) {
            pol_stream = HC_STREAM_POLICY == 1 ? policy_evict_first()
                         : HC_STREAM_POLICY == 2 ? policy_evict_last() : policy_evict_normal();
            pol_keep = policy_evict_last();
        }
        const uint32_t bytes =
            static_cast<uint32_t>((kExpand ? 1 : 4) * p.tile_m * 64 + (kPost ? p.tile_m * 64 : 0) + 4 * kBTileBytes);
        long long g = 0;
        for (long long it = 0; it < my_tiles; ++it) {
            const long long tile = cid + it * ncl;
            const int t0 = static_cast<int>(tile * p.tile_m);
            for (int s = 0; s < S; ++s, ++g) {
                const int slot = static_cast<int>(g % kStages);
                const long long round = g / kStages;
                if (round > 0) W.wait(bar(kBarEmpty + slot), static_cast<uint32_t>((round - 1) & 1), kErrProducer);
                if (lane == 0) {
                    const uint32_t sb = sbase + slot * kStageBytes;
                    const uint32_t fb = bar(kBarFull + slot);
                    const int col = stage_col(s);
                    mbar_arrive_expect_tx(fb, bytes);
                    if (kExpand) {
                        tma_load_2d(sb + kOffX, &tmD, fb, col, t0, pol_stream);  // h into the stream-0 tile
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tma_load_3d(sb + kOffX + j * kXTileBytes, &tmX, fb, col, j, t0, pol_stream);
                    }
                    if (kPost) tma_load_2d(sb + kOffD, &tmD, fb, col, t0, pol_stream);
#pragma unroll
                    for (int k = 0; k < 4; ++k) tma_load_2d(sb + kOffB + k * kBTileBytes, &tmB, fb, k * p.d + col, 0, pol_keep);
                }
                __syncwarp();
            }
        }
        // let every load issued land before the CTA can exit
        const long long issued = g;
        for (long long gg = (issued > kStages ? issued - kStages : 0); gg < issued; ++gg)
            W.drain(bar(kBarFull + static_cast<int>(gg % kStages)), static_cast<uint32_t>((gg / kStages) & 1));
    } else if (warp == kWarpMma) {
        // ================= MMA issuer ===========================================================
        constexpr uint32_t idesc = idesc_bf16_f32(kUmmaM, kUmmaN);
        long long g = 0;
        for (long long it = 0; it < my_tiles; ++it) {
            for (int s = 0; s < S; ++s, ++g) {
                const int slot = static_cast<int>(g % kStages);
                // the single accumulator must have been drained (stage g - 1)
                if (g > 0) W.wait(bar(kBarAccEmpty), static_cast<uint32_t>((g - 1) & 1), kErrMma);
                // post mode multiplies the X' the compute warps wrote; the other modes the loaded tile
                W.wait(bar((kPost ? kBarXReady : kBarFull) + slot), static_cast<uint32_t>((g / kStages) & 1), kErrMma);
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sb = sbase + slot * kStageBytes;
                    const uint32_t dcol = tmem + kAccCol;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const uint64_t ad = sdesc_kmajor_sw64(sb + kOffX + (kExpand ? 0 : k * kXTileBytes) + kk * 32);
                            const uint64_t bd = sdesc_kmajor_sw64(sb + kOffB + k * kBTileBytes + kk * 32);
                            umma_bf16(dcol, ad, bd, idesc, (k | kk) != 0 ? 1u : 0u);
                        }
                    }
                    umma_commit(bar(kBarEmpty + slot));
                    umma_commit(bar(kBarAccFull));
                }
                __syncwarp();
            }
        }
        if (lane == 0) {
            umma_commit(bar(kBarMmaDone));
            W.drain(bar(kBarMmaDone), 0);
        }
        __syncwarp();
    } else if (warp == kWarpStore) {
        // ================= X' writer (post and expand modes) and slot release ====================
        long long g = 0;
        for (long long it = 0; it < my_tiles; ++it) {
            const long long tile = cid + it * ncl;
            const int t0 = static_cast<int>(tile * p.tile_m);
            for (int s = 0; s < S; ++s, ++g) {
                const int slot = static_cast<int>(g % kStages);
                W.wait(bar(kBarXReady + slot), static_cast<uint32_t>((g / kStages) & 1), kErrStore);
                if (kWriteX && lane == 0) {
                    const uint32_t sb = sbase + slot * kStageBytes;
                    const int col = stage_col(s);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        tma_store_3d(&tmXo, sb + kOffX + (kExpand ? 0 : k * kXTileBytes), col, k, t0);
                    if (kPost && p.stream_mean) tma_store_2d(&tmM, sb + kOffD, col, t0);  // the tap
                    bulk_commit();
                    bulk_wait_read<0>();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarEmpty + slot));
            }
        }
        if (lane == 0) bulk_wait<0>();
    } else {  // warp == kWarpSplit
        // ===== group exchange, r_y of every row, split + Sinkhorn for this CTA's share ==========
        float sc[3], bs[kMix];
#pragma unroll
        for (int i = 0; i < 3; ++i) sc[i] = __ldg(p.hc_scale + i);
#pragma unroll
        for (int i = 0; i < kMix; ++i) bs[i] = __ldg(p.hc_base + i);
        // this launch's number for the group: its counter + 1 (never 0, which a fresh workspace holds)
        unsigned long long launch_no = 0;
        if (lane == 0) launch_no = ld_acquire_gpu_u64(p.ws_launch + cid) + 1ull;
        launch_no = __shfl_sync(0xffffffffu, launch_no, 0);
        const unsigned long long epoch_base = launch_no << 32;
        for (long long it = 0; it < my_tiles; ++it) {
            const int buf = static_cast<int>(it & 1);
            // the compute warps have written this CTA's block of the tile: publish it, then wait for
            // the group (lanes 0..7 poll one flag each)
            W.wait(bar(kBarPublish), static_cast<uint32_t>(it & 1), kErrSplit);
            // a flag also says that this CTA is done reading the group's blocks of the previous tile
            // (whose buffer the group reuses after this tile): the split warp read them in its last
            // iteration, the epilogue warps read the sums of y^2
            if (it >= 1) W.wait(bar(kBarEpiRead), static_cast<uint32_t>((it - 1) & 1), kErrSplit);
            unsigned long long* flg = p.ws_flags + static_cast<size_t>(cid * 2 + buf) * kFlagRanks;
            const unsigned long long epoch = epoch_base + static_cast<unsigned long long>(it) + 1ull;
            if (lane == 0) {
                fence_acq_rel_gpu();  // after the barrier: the compute threads' block writes come first
                st_release_gpu_u64(flg + rank, epoch);
            }
            W.wait_flags_warp(flg, epoch, lane, kG, kErrExchange);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarFlagsSeen + buf));  // the epilogue warps may read the sums of y^2
            const long long tile = cid + it * ncl;
            const long long t0 = tile * p.tile_m;
            const float* blk = p.ws_part + (static_cast<size_t>(cid * 2 + buf) * kG) * kPartFloats;
            // the owned tokens t = rank + kG i (i < kT = 128 / kG). The kParts = 32 / kT lanes of token
            // i (lane = part * kT + i) each sum the token's 24 mixes and sum x^2 over kG / kParts = 4
            // of the group's blocks (shares part, part + kParts, ...: every load in flight at once);
            // a reduce-scatter across those lanes then leaves lane `part` with mixes part * kMP ..
            // part * kMP + kMP - 1 summed over all kG blocks, and an all-reduce gives each the sum x^2
            constexpr int kT = kTileMax / kG, kParts = 32 / kT, kMP = kMix / kParts;
            constexpr int kShares = kG / kParts, kLog = kParts == 8 ? 3 : kParts == 4 ? 2 : 1;
            static_assert(kShares * kParts == kG && (1 << kLog) == kParts, "gather split");
            const int oi = lane % kT, part = lane / kT;
            const int r_tok = static_cast<int>(rank) + kG * oi;
            const bool mine = r_tok < p.tile_m && t0 + r_tok < p.n;
            float c[kMix];
#pragma unroll
            for (int i = 0; i < kMix; ++i) c[i] = 0.f;
            float sxt = 0.f;
            if (mine) {
                float4 u[kShares][kMix / 4];
                float2 sxr[kShares];
#pragma unroll
                for (int j = 0; j < kShares; ++j) {
                    const float* Pr = blk + static_cast<size_t>(part + kParts * j) * kPartFloats;
#pragma unroll
                    for (int q = 0; q < kMix / 4; ++q) u[j][q] = ld_cg_f4(Pr + r_tok * kMix + 4 * q);
                    sxr[j] = ld_cg_f2(Pr + kPartSx + 2 * r_tok);
                }
#pragma unroll
                for (int j = 0; j < kShares; ++j) {
#pragma unroll
                    for (int q = 0; q < kMix / 4; ++q) {
                        c[4 * q] += u[j][q].x; c[4 * q + 1] += u[j][q].y;
                        c[4 * q + 2] += u[j][q].z; c[4 * q + 3] += u[j][q].w;
                    }
                    sxt += sxr[j].x + sxr[j].y;
                }
            }
            // reduce-scatter: at level l the lanes split by bit (kLog - 1 - l) of `part`, each keeping
            // one half of its current span and adding the partner's copy of that half
#pragma unroll
            for (int l = 0; l < kLog; ++l) {
                const int half = (kMix >> l) / 2;
                const int mask = kT << (kLog - 1 - l);
                const bool upper = (lane & mask) != 0;
#pragma unroll
                for (int i = 0; i < half; ++i) {
                    const float send = upper ? c[i] : c[i + half];
                    const float keep = upper ? c[i + half] : c[i];
                    c[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
                }
            }
#pragma unroll
            for (int l = 0; l < kLog; ++l) sxt += __shfl_xor_sync(0xffffffffu, sxt, kT << l);
            const float* v = c;  // this lane's kMP mixes
            float m[kMix];
#pragma unroll
            for (int q = 0; q < kParts; ++q)
#pragma unroll
                for (int i = 0; i < kMP; ++i) m[q * kMP + i] = __shfl_sync(0xffffffffu, v[i], q * kT + oi);
            const bool oh = part != 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarSplitDone));  // the blocks of this tile may be reused
            if (mine && oh == 0) {
                const long long tok = t0 + r_tok;
                const float rr = 1.0f / sqrtf(sxt / static_cast<float>(4 * p.d) + p.norm_eps);
#pragma unroll
                for (int i = 0; i < kMix; ++i) m[i] *= rr;
                if (p.mixes_out) {
                    float4* mo = reinterpret_cast<float4*>(p.mixes_out + tok * kMix);
#pragma unroll
                    for (int i = 0; i < kMix / 4; ++i) mo[i] = make_float4(m[4 * i], m[4 * i + 1], m[4 * i + 2], m[4 * i + 3]);
                }
                if (p.pre_out) {
                    float pre[4], post[4], C[16];
                    split_sinkhorn(m, sc, bs, p.iters, p.hc_eps, pre, post, C);
                    reinterpret_cast<float4*>(p.pre_out)[tok] = make_float4(pre[0], pre[1], pre[2], pre[3]);
                    reinterpret_cast<float4*>(p.post_out)[tok] = make_float4(post[0], post[1], post[2], post[3]);
                    float4* co = reinterpret_cast<float4*>(p.comb_out) + tok * 4;
#pragma unroll
                    for (int j = 0; j < 4; ++j) co[j] = make_float4(C[4 * j], C[4 * j + 1], C[4 * j + 2], C[4 * j + 3]);
                }
            }
            __syncwarp();
        }
        // every CTA of the group has read the counter (each published a flag of the last tile,
        // which this warp has seen): advance it for the group's next launch
        if (rank == 0 && lane == 0 && my_tiles > 0) st_release_gpu_u64(p.ws_launch + cid, launch_no);
        __syncwarp();
    }

    // every warp is done with TMEM (and with everything else) before warp 0 frees it
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kBarExit));
    W.drain(bar(kBarExit), 0);
    __syncwarp();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---- host side ----------------------------------------------------------------------------------

namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

bool encode(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
            const uint32_t* box, CUtensorMapSwizzle sw,
            CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_128B) {
    auto fn = get_encode();
    if (!fn) return false;
    uint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base),
                    reinterpret_cast<const cuuint64_t*>(dims), reinterpret_cast<const cuuint64_t*>(strides_bytes),
                    reinterpret_cast<const cuuint32_t*>(box), reinterpret_cast<const cuuint32_t*>(estr),
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, promo,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct DeviceState {
    bool ready = false;
    int ctas = 0;
};

constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

// every instantiation of the fused kernel: [mode][group size 8, 16, 32]
template <int kMode>
void kernels_of_mode(const void** k) {
    k[0] = reinterpret_cast<const void*>(&hc_fused_kernel<kMode, 8>);
    k[1] = reinterpret_cast<const void*>(&hc_fused_kernel<kMode, 16>);
    k[2] = reinterpret_cast<const void*>(&hc_fused_kernel<kMode, 32>);
}

int prepare_device(int* ctas) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -7;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
        const void* kernels[9];
        kernels_of_mode<kModePre>(kernels);
        kernels_of_mode<kModePost>(kernels + 3);
        kernels_of_mode<kModeExpand>(kernels + 6);
        const int k_smem[9] = {Layout<kModePre>::kSmemBytes,    Layout<kModePre>::kSmemBytes,
                               Layout<kModePre>::kSmemBytes,    Layout<kModePost>::kSmemBytes,
                               Layout<kModePost>::kSmemBytes,   Layout<kModePost>::kSmemBytes,
                               Layout<kModeExpand>::kSmemBytes, Layout<kModeExpand>::kSmemBytes,
                               Layout<kModeExpand>::kSmemBytes};
        int per_sm = 1 << 30;
        for (int i = 0; i < 9; ++i) {
            const void* k = kernels[i];
            const int smem = k_smem[i];
            if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return -7;
            int b = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k, kThreads, smem) != cudaSuccess || b < 1)
                return -7;
            per_sm = std::min(per_sm, b);
        }
        int sms = 0, coop = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -7;
        if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop) return -3;
        st.ctas = std::min(kMaxCtas, sms * per_sm);
        if (st.ctas < 8) return -3;
        st.ready = true;
    }
    *ctas = st.ctas;
    return 0;
}

}  // namespace

// Launch plan: for each group size g (d a multiple of 32 g) and tile height m (32, 64, 96, 128, a
// balanced height of 96..128 for batches of several waves, or n when n < 32), groups = ctas / g groups run at once; a launch takes ceil(tiles / groups) waves of S =
// d / (32 g) column stages each, plus a per-tile cost (group exchange, y_normed epilogue tail).
// A stage costs the larger of its latency floor and a fixed part plus a part per token row; the
// constants were measured on GB300 (2.1 us per 128-token stage of the prefill step, about 0.8 us
// for a stage of a small batch, about 4 us per tile).
void plan_tiles(int64_t n, int d, int ctas, int only_group, int* group, int* tile_m, int64_t* num_tiles) {
    *group = 8;
    *tile_m = kTileMax;
    *num_tiles = 0;
    if (n <= 0) return;
    constexpr double kStageFloorUs = 0.8, kStageFixedUs = 0.5, kStagePerRowUs = 1.6 / kTileMax, kTileUs = 4.0;
    double best = -1.0;
    const int gs[3] = {8, 16, 32};
    for (int g : gs) {
        if (d % (kChunk * g) != 0 || (only_group != 0 && g != only_group)) continue;
        const int groups = ctas / g;
        if (groups < 1) continue;
        const int S = d / (kChunk * g);
        // tile heights, largest first (ties keep the larger tile and the smaller group), then for
        // batches of several waves the height that spreads the tokens evenly over the waves
        // 128-token tiles would take (16,384 tokens: 133 tiles of 124 fill 7 waves of 19 groups,
        // where 128 tiles of 128 leave 5 groups idle in the last); only from 96 rows up, where a
        // stage's time still follows its rows (shorter balanced tiles measured slower)
        const int64_t waves128 = ((n + kTileMax - 1) / kTileMax + groups - 1) / groups;
        const int m_even = static_cast<int>((n + groups * waves128 - 1) / (groups * waves128));
        const int ms[6] = {128, 96, 64, 32, n < 32 ? static_cast<int>(n) : 0,
                           waves128 > 1 && m_even >= 96 ? m_even : 0};
        for (int m : ms) {
            if (m < 1) continue;
            const int64_t tiles = (n + m - 1) / m;
            const int64_t waves = (tiles + groups - 1) / groups;
            const double stage = std::max(kStageFloorUs, kStageFixedUs + m * kStagePerRowUs);
            const double cost = static_cast<double>(waves) * (S * stage + kTileUs);
            if (best < 0.0 || cost < best - 1e-9) {
                best = cost;
                *group = g;
                *tile_m = m;
                *num_tiles = tiles;
            }
        }
    }
}

int fused_ctas(int* ctas) { return prepare_device(ctas); }

size_t workspace_bytes() { return kWorkspaceBytes; }

int launch_fused(const FusedArgs& a, cudaStream_t stream) {
    int ctas = 0;
    const int st = prepare_device(&ctas);
    if (st != 0) return st;
    int group = 8, tile_m = 0;
    int64_t num_tiles = 0;
    plan_tiles(a.n, a.d, ctas, a.group, &group, &tile_m, &num_tiles);
    if (num_tiles == 0) return 0;

    const uint64_t n = static_cast<uint64_t>(a.n), d = static_cast<uint64_t>(a.d);
    // maps a mode does not use are encoded on a buffer of the right shape and never touched:
    // tmX (streams read) on X, or on X_out in expand mode; tmXo (streams written) on X_out, or on X
    // in pre mode; tmD ([n, d] rows read) on delta, on the embedding, or on X in pre mode
    const bool write_x = a.mode != kModePre;
    const void* x_in = a.mode == kModeExpand ? a.X_out : a.X;
    const void* rows = a.mode == kModePost ? a.delta : a.mode == kModeExpand ? a.embed : a.X;
    CUtensorMap tmX, tmD, tmB, tmXo, tmM, tmY, tmYr;
    {
        const uint64_t dims[3] = {d, 4, n};
        const uint64_t str[2] = {d * 2, 4 * d * 2};
        const uint32_t box[3] = {kChunk, 1, static_cast<uint32_t>(tile_m)};
        if (!encode(&tmX, x_in, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B, HC_STREAM_PROMOTION)) return -7;
        if (!encode(&tmXo, write_x ? a.X_out : a.X, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B)) return -7;
    }
    {
        const uint64_t dims[2] = {d, n};
        const uint64_t str[1] = {d * 2};
        const uint32_t box[2] = {kChunk, static_cast<uint32_t>(tile_m)};
        if (!encode(&tmD, rows, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B, HC_STREAM_PROMOTION)) return -7;
        // the tap's rows (encoded on the read rows when there is no tap: never used then)
        if (!encode(&tmM, a.stream_mean ? a.stream_mean : rows, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B)) return -7;
        // y_normed in 32-row tiles, one per epilogue warp (encoded on the read rows when it is not written)
        const uint32_t ybox[2] = {kChunk, 32};
        if (!encode(&tmY, a.y_normed ? a.y_normed : rows, 2, dims, str, ybox, CU_TENSOR_MAP_SWIZZLE_64B)) return -7;
        // and the last rows of a tile whose height is not a multiple of 32
        const uint32_t yrbox[2] = {kChunk, static_cast<uint32_t>(tile_m % 32 ? tile_m % 32 : 32)};
        if (!encode(&tmYr, a.y_normed ? a.y_normed : rows, 2, dims, str, yrbox, CU_TENSOR_MAP_SWIZZLE_64B)) return -7;
    }
    {
        const uint64_t dims[2] = {4 * d, static_cast<uint64_t>(kBRows)};
        const uint64_t str[1] = {4 * d * 2};
        const uint32_t box[2] = {kChunk, static_cast<uint32_t>(kBRows)};
        if (!encode(&tmB, a.planes, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B)) return -7;
    }

    FusedParams p;
    p.post = a.post;
    p.comb = a.comb;
    p.pre_mix = a.pre_mix;
    p.hc_scale = a.hc_scale;
    p.hc_base = a.hc_base;
    p.norm_w = a.norm_w;
    p.pre_out = a.pre_out;
    p.post_out = a.post_out;
    p.comb_out = a.comb_out;
    p.mixes_out = a.mixes_out;
    p.stream_mean = a.stream_mean;
    p.y_normed = a.y_normed;
    p.ws_part = reinterpret_cast<float*>(a.workspace);
    p.ws_flags = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(a.workspace) + kWsPartBytes);
    p.ws_launch =
        reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(a.workspace) + kWsPartBytes + kWsFlagBytes);
    p.n = a.n;
    p.num_tiles = num_tiles;
    p.write_y = a.y_normed != nullptr;
    p.d = a.d;
    p.d_slice = a.d / group;
    p.stages_per_tile = p.d_slice / kChunk;
    p.tile_m = tile_m;
    p.iters = a.iters;
    p.hc_eps = a.hc_eps;
    p.norm_eps = a.norm_eps;

    const int64_t grid_groups = std::min<int64_t>(num_tiles, ctas / group);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident together: the group flags can be awaited
    attr[0].val.cooperative = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid_groups * group), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = a.mode == kModePost     ? Layout<kModePost>::kSmemBytes
                           : a.mode == kModeExpand ? Layout<kModeExpand>::kSmemBytes
                                                   : Layout<kModePre>::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaErrorInvalidValue;
    auto go = [&](auto kernel) { e = cudaLaunchKernelEx(&cfg, kernel, tmX, tmD, tmB, tmXo, tmM, tmY, tmYr, p); };
    if (a.mode == kModePost) {
        if (group == 8) go(hc_fused_kernel<kModePost, 8>);
        else if (group == 16) go(hc_fused_kernel<kModePost, 16>);
        else go(hc_fused_kernel<kModePost, 32>);
    } else if (a.mode == kModeExpand) {
        if (group == 8) go(hc_fused_kernel<kModeExpand, 8>);
        else if (group == 16) go(hc_fused_kernel<kModeExpand, 16>);
        else go(hc_fused_kernel<kModeExpand, 32>);
    } else {
        if (group == 8) go(hc_fused_kernel<kModePre, 8>);
        else if (group == 16) go(hc_fused_kernel<kModePre, 16>);
        else go(hc_fused_kernel<kModePre, 32>);
    }
    return e == cudaSuccess ? 0 : -7;
}

// ---- scratch that needs no allocation ------------------------------------------------------------
// The workspace of hc_post_then_pre_noalloc: a fixed array in the library's device image, one per
// GPU that loads the library, zero at load and kept until the process exits. Its size is the same
// kWorkspaceBytes (7,356,672 bytes: room for 256 co-resident CTAs) that hc_workspace_size reports.
static __device__ __align__(256) unsigned char g_noalloc_workspace[kWorkspaceBytes];
// A launch never needs more scratch than this: the fused kernel runs at most kMaxCtas CTAs (the
// device's resident count is capped there) and the generic path works through its tokens in chunks
// sized to kWorkspaceBytes, so no call is ever refused for want of room in the array.
static_assert(sizeof(g_noalloc_workspace) >= kWorkspaceBytes && kWorkspaceBytes >= kWsPartBytes &&
                  kWsPartBytes == static_cast<size_t>(kMaxCtas) * 2 * kPartFloats * 4,
              "the fixed scratch holds the partial sums of kMaxCtas CTAs, their flags and counters");

namespace {
void* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;
}  // namespace

int noalloc_workspace(void** ptr, size_t* capacity) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -7;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        // host code only knows the array by its host-side stand-in: ask the runtime for the
        // address of this device's copy, once, with this device current
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || !p) return -7;
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    *capacity = sizeof(g_noalloc_workspace);
    return 0;
}

int launch_wait_flag(const unsigned long long* flags, unsigned long long value, int g, uint64_t limit_ns,
                     cudaStream_t stream) {
    hc_wait_flag_kernel<<<1, 32, 0, stream>>>(flags, value, g, limit_ns);
    return cudaGetLastError() == cudaSuccess ? 0 : -7;
}

int read_device_error(unsigned int* word, int clear, cudaStream_t stream) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_hc_error, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return -7;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return -7;
    if (clear) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbolAsync(g_hc_error, &z, sizeof(z), 0, cudaMemcpyHostToDevice, stream) != cudaSuccess)
            return -7;
        if (v != 0) {
            // A kernel gave up a wait: a CTA of its group that had not yet read the group's launch
            // counter when the counter advanced would tag its flags like the group's next launch. The
            // library's fixed scratch (hc_post_then_pre_noalloc) therefore starts afresh from zero; a
            // memset is not an allocation. Caller workspaces are the caller's to zero (hc.h).
            int dev = 0;
            if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -7;
            void* scratch = nullptr;
            {
                std::lock_guard<std::mutex> lk(g_noalloc_mu);
                scratch = g_noalloc_ptr[dev];
            }
            if (scratch && cudaMemsetAsync(scratch, 0, sizeof(g_noalloc_workspace), stream) != cudaSuccess) return -7;
        }
        if (cudaStreamSynchronize(stream) != cudaSuccess) return -7;
    }
    *word = v;
    return 0;
}

}  // namespace hc
