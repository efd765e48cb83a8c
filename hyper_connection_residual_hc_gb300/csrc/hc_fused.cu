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
// has fewer column stages) owns a tile of up to 128 tokens (groups of 16 and 32: up to 64); CTA
// `rank` of the group owns d/kG columns of every stream, the 32-column chunks rank, rank+kG,
// rank+2kG, ... (interleaved, so the group's loads of one stage cover kG*32 contiguous columns of
// each row). Groups of 8 make one pass per 32-column stage. Groups of 16 and 32 fold their tiles:
// a pass holds two column stages, the second in rows 64..127 of each tile, so that the 128-row MMA
// and all compute warps do useful work on small batches. The 16 warps of a CTA have fixed roles:
//   producer (warp 8): per pass, TMA-loads the four X tiles [tokens x 32 cols] (expand mode: the
//     one embedding tile), the Delta tile (post mode) and the matching slices of the split
//     projection weights (bf16 planes hi/mid/lo, 72 rows per stream and stage) into a ring of
//     shared-memory slots, 64-byte swizzled: 3 slots in post mode, 4 in pre mode, 6 in expand mode
//     (folded: 2, 2, 4); a folded pass of 64-token tiles takes one box per tensor. The first slots'
//     loads are issued by thread 0 as soon as the kernel ahead on the stream has completed;
//   compute (warps 0-7, thread = token row, two warps per TMEM lane quadrant, 16 columns each):
//     compute X' in place (post mode; the other modes read the loaded tile), accumulate sum(X'^2),
//     form and round y, accumulate sum(y^2), store the bf16 y chunk into a ring of chunk slots in
//     tensor memory, and drain the previous pass's accumulator into 12 per-thread fp32 sums (the
//     three planes added back together); folded, the warps of rows 64..127 hand their sums of a
//     tile to those of rows 0..63 (same tokens) through shared memory;
//   MMA (warp 9): one thread issues 8 tcgen05.mma per pass (M=128 rows, N=80 >= 72 plane rows, or
//     N=144 for the two stages of a folded pass, K=16) projecting the bf16 X' tile on the three
//     planes into a TMEM accumulator; the products are exact in fp32, so the split projection has
//     fp32-FFMA accuracy;
//   store (warp 10): TMA-stores the X' tile (written once) from the same slot, then frees it;
//   split (warp 11): at each tile end, publishes the CTA's partial sums (28 per token, in a
//     caller-provided global workspace) by a release add to the group's arrival counter, waits
//     (bounded) until the counter shows every CTA of the group, gathers the mixes of its own tokens
//     (t % kG == rank) over the group's blocks, and runs their split and Sinkhorn;
//   epilogue (warps 12-15, one per TMEM lane quadrant): load norm_w of the CTA's columns, turn the
//     group's sums of y^2 into r_y of the warp's rows, read each y chunk back from the ring, scale
//     it by norm_w and r_y into a 32-row swizzled staging tile and TMA-store it to y_normed.
// The ring holds a tile's y until the exchange gives r_y, with 7 stages of slack at 20 stages a
// tile: the compute warps stream on into the next tile while the group finishes the previous one.
// The groups are formed in software rather than as hardware clusters because only 15 clusters of
// 8 CTAs fit on a GB300 at once (120 of its 152 SMs); the launch is cooperative, so all CTAs are
// resident together and the counter waits between them cannot deadlock. It is also a programmatic
// dependent launch: the set-up (barriers, tensor memory, descriptors, an L2 prefetch of the first
// weight planes) overlaps the end of the kernel ahead, and every access to global memory follows
// griddepcontrol.wait.
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
constexpr int kMaxGroups = 32;     // group slots (at most 256 / 8): one arrival counter and one base each
constexpr int kCounterStride = 16; // 64-bit words between arrival counters: one 128-byte line each
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
// Folded tiles (groups of 16 and 32, tiles of at most 64 tokens): rows 64..127 of every tile in a
// slot hold the same tokens at the next column stage, so one 128-row MMA and all compute warps
// serve two stages. The weight-plane tile then holds both stages' planes, rows 0..71 and 72..143,
// and one MMA of N = 144 gives rows 0..63 their projection in accumulator columns 0..71 and rows
// 64..127 theirs in columns 72..143 (the other blocks of the product are not read). A pass of two
// stages on 64-token tiles is loaded with one box per tensor: the four streams' two stages of X
// [stream][stage][token][32 columns], the two of Delta, the four streams' two stages of planes
// (4-D and 3-D views whose "stage" dimension steps by the group's column stride), 3 TMA issues
// instead of 18 (each issue costs a thread about 57 cycles, the first about 390).
constexpr int kFoldRows = 64;                                 // tokens per folded tile at most
constexpr int kFoldXHalf = kFoldRows * kChunk * 2;            // 4096: the second stage's rows
constexpr int kUmmaNFold = 144;
constexpr int kFoldBRow1 = kBRows;                            // first plane row of the second stage
constexpr int kBTileBytesFold = kUmmaNFold * kChunk * 2;      // 9216
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
// kBarNormW: the epilogue warps have put norm_w of the CTA's columns in shared memory (one arrival per
// epilogue warp; only they read it, long after the stage loop has started)
constexpr int kBarNormW = kBarExit + 1;
// folded tiles alternate between two accumulators: the full and empty barriers of the second
constexpr int kBarAccFull2 = kBarExit + 2, kBarAccEmpty2 = kBarExit + 3;
// kBarPartEmpty: the split warp has copied a tile's partial sums out of their shared-memory block
// (every mode but unfolded pre, one arrival per tile)
constexpr int kBarPartEmpty = kBarExit + 4;
constexpr int kNumBars = kBarExit + 5;

// Shared-memory layout of each mode, offsets from a 1024-byte aligned base. A slot holds one column
// stage (a folded slot two): the stream tiles (four, or the one embedding tile in expand mode), the
// Delta tile (post mode only) and the four weight-plane tiles. The smaller slots of the
// reading-only modes buy more of them, so more loads are in flight while the stage's MMA holds its
// slot: post 3 x 59392 B, pre 4 x 51200 B, expand 6 x 26624 B; folded post 2 x 81920 B, pre
// 2 x 73728 B, expand 4 x 49152 B. After the slots: norm_w of the CTA's columns, the epilogue warps'
// y_normed staging tiles (per warp two 32-row x 64-byte tiles, 64-byte swizzle, filled and
// TMA-stored in turn), the folded tiles' scratch, the mbarriers, the TMEM address and the abort word.
template <int kMode, bool kFold>
struct Layout {
    static constexpr int kXTiles = kMode == kModeExpand ? 1 : 4;
    static constexpr int kBTile = kFold ? kBTileBytesFold : kBTileBytes;
    static constexpr int kOffX = 0;
    static constexpr int kOffD = kXTiles * kXTileBytes;
    static constexpr int kOffB = kOffD + (kMode == kModePost ? kXTileBytes : 0);
    static constexpr int kStage = kOffB + 4 * kBTile;
    static constexpr int kStages = kFold ? (kMode == kModeExpand ? 4 : 2)
                                         : (kMode == kModePost ? 3 : kMode == kModePre ? 4 : 6);
    // folded post and pre modes: a slot of its own for the compact one-stage pass that ends a tile of
    // an odd stage count: four 64-row X tiles 4 KB apart, the Delta tile, four plane tiles 4,608 B apart
    static constexpr bool kHasC = kFold && kMode != kModeExpand;
    static constexpr int kCOffD = 4 * kFoldXHalf;                  // 16384
    static constexpr int kCOffB = kCOffD + kFoldXHalf;             // 20480
    static constexpr int kCSlot = kCOffB + 4 * kBTileBytes;        // 38912
    static constexpr int kOffC = kStages * kStage;
    static constexpr int kOffNormW = kOffC + (kHasC ? kCSlot : 0);
    static constexpr int kOffYStage = ((kOffNormW + kMaxDSlice * 4 + 1023) / 1024) * 1024;
    // Tiles hand their partial sums to the split warp in a shared-memory block, which the split warp
    // writes to the workspace. Folded tiles have it here: rows 64..127 (the same tokens at the odd
    // stages) are added to rows 0..63 as it is copied. Unfolded post and expand tiles have it after
    // the split warp's scratch. Unfolded pre mode has no room for it, so its compute warps write the
    // workspace themselves. Holding the tile's last slot for the block instead measured slower
    // (152 -> 154 us at the prefill batch), as did publishing a tile one pass late.
    static constexpr bool kPartInSmem = kFold || kMode != kModePre;
    static constexpr int kOffFoldPart = kOffYStage + 4 * 2 * kYStageBytes;
    // the split warp's gather scratch: per owned token (at most 16) its 24 mixes and sum of x^2; then
    // hc_scale and hc_base (27 floats, 32 reserved)
    static constexpr int kOffSplit = kOffFoldPart + (kFold ? kPartFloats * 4 : 0);
    static constexpr int kOffSplitPrm = kOffSplit + (kTileMax / 8) * 7 * 16;
    static constexpr int kOffPart = kFold ? kOffFoldPart : kOffSplitPrm + 32 * 4;
    static constexpr int kOffBar = kOffSplitPrm + 32 * 4 + ((kPartInSmem && !kFold) ? kPartFloats * 4 : 0);
    static constexpr int kOffTmemPtr = kOffBar + kNumBars * 8;
    static constexpr int kOffAbort = kOffTmemPtr + 4;
    static constexpr int kSmemUsed = kOffAbort + 4;
    static constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for aligning the base
    static_assert(kStage % 1024 == 0, "stage buffers keep 1024-byte alignment");
    static_assert(kOffB % 512 == 0 && kBTileBytes % 512 == 0, "B tiles start on 512-byte swizzle atoms");
    static_assert(kStages + (kHasC ? 1 : 0) <= kMaxStages, "barrier numbering");
    static_assert(kCOffB % 512 == 0 && kCSlot % 1024 == 0, "compact slot on swizzle atoms");
    // the compact slot's MMA reads past its last X tile (into its Delta and plane tiles) and past its
    // last plane tile (into norm_w and the staging tiles): inside the CTA's shared memory
    static_assert(!kHasC || kOffC + kCOffB + 3 * kBTileBytes + kUmmaNFold * 64 <= kSmemUsed, "compact overrun");
    static_assert(kSmemBytes <= 232448, "fits the 227 KB opt-in shared memory of one CTA");
    // unfolded: the MMA of the last B tile of the last slot reads 8 rows (512 B) past it: into norm_w,
    // inside the CTA (a folded B tile is exactly the 160 rows its MMA reads)
    static_assert(kOffB + 3 * kBTile + (kFold ? kUmmaNFold : kUmmaN) * 64 + (kStages - 1) * kStage <= kSmemUsed,
                  "B overrun");
    static_assert(kFoldXHalf % 512 == 0 && (kFoldBRow1 * 64) % 512 == 0, "second stage on swizzle atoms");
    static_assert(kOffPart % 16 == 0, "partial-sum block: 16-byte aligned");
};

// global workspace: partial sums [group][tile parity][rank][28][128] fp32 (a block per CTA and
// tile parity), then one 64-bit arrival counter per group slot (each on its own 128-byte line),
// then one 64-bit base per group slot. When a CTA has written its block of a tile it adds 1 to its
// group's arrival counter (release); the tile's exchange is complete when the counter reaches
// base + kG * (tile index + 1), the base being the counter's value when the launch started. Every
// CTA of the group reads the base when it starts, and the group's rank-0 CTA stores the counter's
// final value as the next base after its last exchange, when all its group has read the base and
// added its last arrival. A group slot keeps counting across launches of any group size, so the
// targets never repeat on one workspace; they come from the device, so a launch replayed from a
// CUDA graph waits for its own arrivals, and a zero-filled workspace starts at 0. One counter per
// group, polled by one lane per CTA, keeps the exchange off a contended line: with one flag per
// CTA, polled by every lane of every CTA of a group (1024 pollers on two 128-byte lines), some
// groups of a 256-token launch saw their flags 3-4 us after the last one was published.
constexpr size_t kWsPartBytes = static_cast<size_t>(kMaxCtas) * 2 * kPartFloats * 4;
constexpr size_t kWsFlagBytes = static_cast<size_t>(kMaxGroups) * kCounterStride * 8;
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
// folded tiles: two 144-column accumulators used in turn (the MMA of a pass need not wait for the
// previous pass's drain), then 13 ring slots (a folded tile has at most 5 passes)
constexpr uint32_t kYColFold = 2 * 144;
constexpr int kRingFold = 13;
static_assert(kYColFold + kRingFold * 16 <= kTmemCols, "folded y ring fits in TMEM");
static_assert(kBarYFree == kBarYReady + kRing, "one ready and one free barrier per ring slot");

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

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
    unsigned long long* ws_arrivals;  // workspace arrival counters, one per group slot
    unsigned long long* ws_launch;  // workspace launch counters, one per group
    long long n;
    long long num_tiles;
    int write_y;
    int d;
    int d_slice;
    int stages_per_tile;
    int tile_m;
    int combined;                   // folded 64-token tiles: one box per tensor for a two-stage pass
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
    // Whole warp: lanes 0..g-1 each wait for the 64-bit counter c[lane] to reach `target`; returns
    // when all g do. The fused kernel waits on one counter (g = 1): that of its group.
    __device__ __forceinline__ bool wait_count(const unsigned long long* c, unsigned long long target, int lane,
                                               int g, unsigned int code) const {
        const uint64_t t0 = global_timer_ns();
        bool mine = lane >= g;
        while (true) {
            if (!mine) mine = ld_acquire_gpu_u64(c + lane) >= target;
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
// The 4x4 matrix is passed as row pairs (C2[2j] = columns 0-1 of row j, C2[2j+1] = columns 2-3); a
// row's sum is (C[j0] + C[j2]) + (C[j1] + C[j3]).

// The Sinkhorn rounds on the softmax matrix C2 (row j: C2[2j] holds columns 0 and 1, C2[2j + 1]
// columns 2 and 3): one column normalisation, then iters - 1 times a row and a column one. Scalar
// operations, in the order the fp32x2 form had (a column sum is (c0 + c1) + (c2 + c3) over the rows,
// a row sum (c0 + c2) + (c1 + c3) over the columns), so the values are the same bits; the scalar form
// takes about 153 cycles a round against 163 for the fp32x2 one (the pairs cost moves).
__device__ __forceinline__ void sinkhorn_rounds(float2 (&C2)[8], int iters, float eps) {
    float C[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        C[j][0] = C2[2 * j].x;
        C[j][1] = C2[2 * j].y;
        C[j][2] = C2[2 * j + 1].x;
        C[j][3] = C2[2 * j + 1].y;
    }
    auto col_norm = [&]() {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float inv = rcp_refined(((C[0][k] + C[1][k]) + (C[2][k] + C[3][k])) + eps);
#pragma unroll
            for (int j = 0; j < 4; ++j) C[j][k] *= inv;
        }
    };
    auto row_norm = [&]() {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float inv = rcp_refined(((C[j][0] + C[j][2]) + (C[j][1] + C[j][3])) + eps);
#pragma unroll
            for (int k = 0; k < 4; ++k) C[j][k] *= inv;
        }
    };
    col_norm();
    for (int it = 1; it < iters; ++it) {
        row_norm();
        col_norm();
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        C2[2 * j] = make_float2(C[j][0], C[j][1]);
        C2[2 * j + 1] = make_float2(C[j][2], C[j][3]);
    }
}

__device__ __forceinline__ void split_sinkhorn(const float (&m)[kMix], const float (&sc)[3], const float (&b)[kMix],
                                               int iters, float eps, float (&pre)[4], float (&post)[4],
                                               float (&C)[16]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) pre[j] = sigmoidf_(fmaf(m[j], sc[0], b[j])) + eps;
#pragma unroll
    for (int j = 0; j < 4; ++j) post[j] = 2.0f * sigmoidf_(fmaf(m[4 + j], sc[1], b[4 + j]));
    float2 C2[8];
    const float2 e2 = make_float2(eps, eps);
    // softmax over each row (max subtracted), then + eps
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float l[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) l[k] = fmaf(m[8 + 4 * j + k], sc[2], b[8 + 4 * j + k]);
        const float mx = fmaxf(fmaxf(l[0], l[1]), fmaxf(l[2], l[3]));
        const float2 x01 = make_float2(expf(l[0] - mx), expf(l[1] - mx));
        const float2 x23 = make_float2(expf(l[2] - mx), expf(l[3] - mx));
        const float inv = rcp_refined((x01.x + x01.y) + (x23.x + x23.y));
        C2[2 * j] = __ffma2_rn(x01, make_float2(inv, inv), e2);
        C2[2 * j + 1] = __ffma2_rn(x23, make_float2(inv, inv), e2);
    }
    sinkhorn_rounds(C2, iters, eps);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        C[4 * j] = C2[2 * j].x;
        C[4 * j + 1] = C2[2 * j].y;
        C[4 * j + 2] = C2[2 * j + 1].x;
        C[4 * j + 3] = C2[2 * j + 1].y;
    }
}

// ---- diagnostic: one bounded wait on an exchange counter ---------------------------------------------
// One warp waits, exactly as the fused kernel's split warp waits for its group, for the counters
// f[0..g-1] to reach `value`, giving up after limit_ns: it then records kErrExchange in the device
// error word and returns. Lets a test make a wait run out (on counters nothing advances) and check
// what the host sees.
__global__ void hc_wait_flag_kernel(const unsigned long long* f, unsigned long long value, int g, uint64_t limit_ns) {
    __shared__ uint32_t abort_word;
    if (threadIdx.x == 0) abort_word = 0u;
    __syncwarp();
    const Waiter W{&abort_word, limit_ns};
    W.wait_count(f, value, static_cast<int>(threadIdx.x), g, kErrExchange);
}

// ---- the kernel ---------------------------------------------------------------------------------

template <int kMode, int kG, bool kFold>
__global__ void __launch_bounds__(kThreads, 1)
    hc_fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmD,
                    const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmXo,
                    const __grid_constant__ CUtensorMap tmM, const __grid_constant__ CUtensorMap tmY,
                    const __grid_constant__ CUtensorMap tmYr, const __grid_constant__ CUtensorMap tmX4,
                    const __grid_constant__ CUtensorMap tmXo4, const __grid_constant__ CUtensorMap tmD3,
                    const __grid_constant__ CUtensorMap tmM3, const __grid_constant__ CUtensorMap tmB4,
                    const __grid_constant__ CUtensorMap tmX3s, const __grid_constant__ CUtensorMap tmXo3s,
                    const __grid_constant__ CUtensorMap tmB3, const FusedParams p) {
    using Lay = Layout<kMode, kFold>;
    constexpr int kStages = Lay::kStages, kStageBytes = Lay::kStage, kBTile = Lay::kBTile;
    constexpr int kRingN = kFold ? kRingFold : kRing;
    constexpr uint32_t kYColN = kFold ? kYColFold : kYCol;
    constexpr int kOffX = Lay::kOffX, kOffD = Lay::kOffD, kOffB = Lay::kOffB, kOffNormW = Lay::kOffNormW;
    constexpr int kOffYStage = Lay::kOffYStage, kOffBar = Lay::kOffBar, kOffTmemPtr = Lay::kOffTmemPtr;
    constexpr int kOffAbort = Lay::kOffAbort, kOffSplit = Lay::kOffSplit;
    constexpr int kOffSplitPrm = Lay::kOffSplitPrm, kOffPart = Lay::kOffPart;
    constexpr bool kPartInSmem = Lay::kPartInSmem;
    constexpr int kNumSlots = kStages + (Lay::kHasC ? 1 : 0);
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
    // passes over a tile: one per column stage, or one per pair of stages when folded (stage 2f in
    // rows 0..63, stage 2f + 1, if any, in rows 64..127)
    const int SP = kFold ? (S + 1) / 2 : S;
    // A folded pass with one stage on 64-token tiles (the last pass of an odd stage count) is loaded
    // compact, one box per tensor: the four streams' 64 rows 4 KB apart and their plane tiles 4,608
    // bytes apart, so the 128-row MMA of stream k reads stream k + 1 as its rows 64..127 (products
    // that land in accumulator cells nobody drains) and all reads stay inside the slot.
    auto compact = [&](int sp) { return kFold && p.combined && 2 * sp + 1 >= S; };
    auto x_pitch = [&](int sp) -> uint32_t { return compact(sp) ? static_cast<uint32_t>(kFoldXHalf) : kXTileBytes; };
    auto b_pitch = [&](int sp) -> uint32_t { return compact(sp) ? static_cast<uint32_t>(kBTileBytes) : kBTile; };
    // Shared-memory slot of pass sp of the CTA's tile `it` (the same function in every role). With an
    // odd stage count in post and pre modes the compact last pass takes the slot after the ring, so
    // that all passes of a tile can be loaded at once; the other passes take the ring in order.
    const bool use_c = Lay::kHasC && p.combined && (S & 1) != 0;
    const int nring = use_c ? SP - 1 : SP;
    struct Slot {
        int idx;         // barrier index (kStages: the compact slot)
        uint32_t base;   // shared-memory address
        long long round; // how many passes used this slot before
        uint32_t offd, offb;
    };
    auto slot_at = [&](long long it, int sp) -> Slot {
        Slot r;
        if (use_c && sp == SP - 1) {
            r.idx = kStages;
            r.base = sbase + static_cast<uint32_t>(Lay::kOffC);
            r.round = it;
            r.offd = static_cast<uint32_t>(Lay::kCOffD);
            r.offb = static_cast<uint32_t>(Lay::kCOffB);
        } else {
            const long long gr = it * nring + sp;
            r.idx = static_cast<int>(gr % kStages);
            r.base = sbase + static_cast<uint32_t>(r.idx) * kStageBytes;
            r.round = gr / kStages;
            r.offd = static_cast<uint32_t>(kOffD);
            r.offb = static_cast<uint32_t>(kOffB);
        }
        return r;
    };

    auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * static_cast<uint32_t>(i); };
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kOffAbort);
    const Waiter W{abort_flag, kWaitLimitNs};
    // accumulators: one, or two used in turn when folded (pass g uses g % kNAcc)
    constexpr int kNAcc = kFold ? 2 : 1;
    auto acc_full = [&](long long g) { return bar((g % kNAcc) ? kBarAccFull2 : kBarAccFull); };
    auto acc_empty = [&](long long g) { return bar((g % kNAcc) ? kBarAccEmpty2 : kBarAccEmpty); };
    auto acc_col = [&](long long g) { return kAccCol + static_cast<uint32_t>((g % kNAcc) * kUmmaNFold); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNumSlots; ++s) {
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
        mbar_init(bar(kBarNormW), 4);
        mbar_init(bar(kBarAccFull2), 1);
        mbar_init(bar(kBarAccEmpty2), kComputeWarps);
        mbar_init(bar(kBarPartEmpty), 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    const long long my_tiles =
        (static_cast<long long>(cid) < p.num_tiles) ? (p.num_tiles - 1 - cid) / ncl + 1 : 0;
    // bytes of one column stage; a folded pass loads two (rows 64.. of each tile, plane rows 80..)
    const uint32_t stage_bytes =
        static_cast<uint32_t>((kExpand ? 1 : 4) * p.tile_m * 64 + (kPost ? p.tile_m * 64 : 0) + 4 * kBTileBytes);
    // one thread: the TMA loads of pass s of the tile starting at token t0 into slot sl
    auto issue_pass = [&](const Slot& sl, int s, int t0, uint64_t pol_stream, uint64_t pol_keep) {
        const uint32_t sb = sl.base;
        const uint32_t fb = bar(kBarFull + sl.idx);
        const int halves = (kFold && 2 * s + 1 < S) ? 2 : 1;
        mbar_arrive_expect_tx(fb, stage_bytes * static_cast<uint32_t>(halves));
        if (kFold && halves == 2 && p.combined) {
            const int col = stage_col(2 * s);
            if (kExpand)
                tma_load_3d(sb + kOffX, &tmD3, fb, col, t0, 0, pol_stream);
            else
                tma_load_4d(sb + kOffX, &tmX4, fb, col, t0, 0, 0, pol_stream);
            if (kPost) tma_load_3d(sb + kOffD, &tmD3, fb, col, t0, 0, pol_stream);
            tma_load_4d(sb + kOffB, &tmB4, fb, col, 0, 0, 0, pol_keep);
            return;
        }
        if (compact(s)) {
            const int col = stage_col(2 * s);
            if (kExpand)
                tma_load_2d(sb + kOffX, &tmD, fb, col, t0, pol_stream);
            else
                tma_load_3d(sb + kOffX, &tmX3s, fb, col, t0, 0, pol_stream);
            if (kPost) tma_load_2d(sb + sl.offd, &tmD, fb, col, t0, pol_stream);
            tma_load_3d(sb + sl.offb, &tmB3, fb, col, 0, 0, pol_keep);
            return;
        }
        for (int hf = 0; hf < halves; ++hf) {
            const int col = stage_col(kFold ? 2 * s + hf : s);
            const uint32_t xo = static_cast<uint32_t>(hf * kFoldXHalf);
            const uint32_t bo = static_cast<uint32_t>(hf * kFoldBRow1 * 64);
            if (kExpand) {
                tma_load_2d(sb + kOffX + xo, &tmD, fb, col, t0, pol_stream);  // h into the stream-0 tile
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    tma_load_3d(sb + kOffX + j * kXTileBytes + xo, &tmX, fb, col, j, t0, pol_stream);
            }
            if (kPost) tma_load_2d(sb + kOffD + xo, &tmD, fb, col, t0, pol_stream);
            if (!kFold) {
                tma_load_3d(sb + kOffB, &tmB3, fb, col, 0, 0, pol_keep);  // the four streams' planes, one box
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    tma_load_2d(sb + kOffB + k * kBTile + bo, &tmB, fb, k * p.d + col, 0, pol_keep);
            }
        }
    };
    // the passes of the first tile that fill the empty slots: issued as soon as the kernel ahead has
    // completed, by the thread that initialised the barriers and before the CTA-wide barrier below
    // (the producer warp skips them)
    auto early = [&](long long it, int sp) { return my_tiles > 0 && it == 0 && sp < nring && sp < kStages; };
    if (warp == kWarpProducer && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmB);
        if (kWriteX) tma_prefetch_desc(&tmD);
        // the weight-plane tiles of the first stages into L2 while the previous kernel may still run
        // (a prefetch into L2, the point of coherence, returns nothing stale to the loads that follow
        // the wait below)
        if (my_tiles > 0)
            for (int s = 0; s < S && s < (kFold ? 2 : 1) * kStages; ++s)
                for (int k = 0; k < 4; ++k) tma_prefetch_l2_2d(&tmB, k * p.d + stage_col(s), 0);
    }
    if (warp == 0) {
        tmem_alloc(sbase + kOffTmemPtr, kTmemCols);
        tmem_relinquish();
    }
    // Launched with programmatic stream serialization: the set-up above (barriers, tensor memory,
    // descriptors, L2 prefetch) overlaps the end of the kernel ahead on the stream; every read and
    // write of global memory comes after this wait for that kernel to complete. The next kernel may
    // start its own set-up as soon as every CTA of this one has got here.
    if (threadIdx.x == 0) griddep_launch_dependents();
    griddep_wait();
    if (threadIdx.x == 0) {
        // the streamed tiles (X, Delta) keep the normal L2 policy: evict_first dropped the unused
        // half of each 128-byte line and re-read it (356 MB more per prefill step)
        const uint64_t pol_stream = policy_evict_normal(), pol_keep = policy_evict_last();
        for (int s = 0; s < SP; ++s)
            if (early(0, s)) issue_pass(slot_at(0, s), s, static_cast<int>(cid * p.tile_m), pol_stream, pol_keep);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemPtr);

    if (warp < kComputeWarps) {
        // ================= compute warps: X', sums, y, accumulator drain ========================
        const int q = warp & 3;             // TMEM lane quadrant = tile rows 32q..32q+31
        const int h = warp >> 2;            // column half of each 32-column stage
        const int row = 32 * q + lane;      // row of the tile (and TMEM lane)
        // folded: rows 64..127 (sub = 1) hold the tokens of rows 0..63 at the pass's second stage
        const int sub = kFold ? (q >> 1) : 0;
        const int trow = kFold ? (row & (kFoldRows - 1)) : row;  // token row inside the tile
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
        long long g = 0;        // global pass counter (same sequence in every role)
        // does pass sp of a tile hold a stage for this warp's rows (folded: not the second half of
        // the last pass when the stages are odd)
        auto pass_ok = [&](int sp) { return !kFold || 2 * sp + sub < S; };
        // tell the epilogue warps that the y chunk of pass gy is in TMEM
        auto y_ready = [&](long long gy) {
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarYReady + static_cast<int>(gy % kRingN)));
        };
        // this token's coefficients of the current tile, each broadcast to both lanes of a float2
        float2 cpost[4], ccomb[16], pm[4];
        auto load_coefs = [&](long long it) {
            const long long tok = (cid + it * ncl) * p.tile_m + trow;
            const bool valid = (trow < p.tile_m) && (tok < p.n);
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
        };
        if (my_tiles > 0) load_coefs(0);
        for (long long it = 0; it < my_tiles; ++it) {
            float2 acc[6];  // the 12 mixes of this thread's column half, in pairs
#pragma unroll
            for (int i = 0; i < 6; ++i) acc[i] = bcast(0.f);
            float2 sx[4], sy[2];  // sums of squares, each split over the two lanes
#pragma unroll
            for (int i = 0; i < 4; ++i) sx[i] = bcast(0.f);
            sy[0] = sy[1] = bcast(0.f);

            // drain pass gd's accumulator (the three planes added back together) into acc; a folded
            // pass with no stage for these rows is waited for and released but not added
            auto drain = [&](long long gd, bool add) {
                W.wait(acc_full(gd), static_cast<uint32_t>((gd / kNAcc) & 1), kErrComputeAcc);
                tc_fence_after();
                if (add) {
                    uint32_t v[36];
                    const uint32_t col = acc_col(gd) + (sub ? static_cast<uint32_t>(kFoldBRow1) : 0u) + 36u * h;
                    tmem_ld36_wait(tl + col, tl + col + 32u, v);
                    auto f2 = [&](int i) { return make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])); };
#pragma unroll
                    for (int i = 0; i < 6; ++i)
                        acc[i] = __fadd2_rn(acc[i], __fadd2_rn(__fadd2_rn(f2(2 * i), f2(12 + 2 * i)), f2(24 + 2 * i)));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty(gd));
            };

            for (int s = 0; s < SP; ++s, ++g) {
                // the y store of the previous pass has had a pass to complete: hand it over
                if (s > 0) y_ready(g - 1);
                // reading-only modes: the MMA of this pass reads the tile as loaded, so it may start
                // as soon as the data lands; drain the previous pass's accumulator first to let it
                if (!kPost && s > 0) drain(g - 1, pass_ok(s - 1));
                // the ring slot of this pass's y last held the chunk of pass g - kRingN
                const long long yround = g / kRingN;
                if (yround > 0)
                    W.wait(bar(kBarYFree + static_cast<int>(g % kRingN)), static_cast<uint32_t>((yround - 1) & 1),
                           kErrComputeY);
                // three passes before the tile ends (the first, in a shorter tile), the next tile's
                // coefficient lines into L2: loaded from DRAM at the tile's end, under the stream's
                // load, they took 1.3-2.2 us to land, which the next tile's first pass waited for
                if (kPost && h == 0 && s == (SP > 3 ? SP - 3 : 0) && it + 1 < my_tiles) {
                    const long long ntok = (cid + (it + 1) * ncl) * p.tile_m + trow;
                    if (trow < p.tile_m && ntok < p.n) {
                        prefetch_l2_evict_last(p.post + ntok * 4);
                        prefetch_l2_evict_last(p.comb + ntok * 16);
                        if (p.pre_mix) prefetch_l2_evict_last(p.pre_mix + ntok * 4);
                    }
                }
                const Slot sl = slot_at(it, s);
                W.wait(bar(kBarFull + sl.idx), static_cast<uint32_t>(sl.round & 1), kErrComputeFull);
                const uint32_t sb = sl.base;
                const uint32_t offd = sl.offd;
                const bool here = pass_ok(s);  // warp-uniform
                const uint32_t xp = x_pitch(s);  // bytes between the streams' tiles in this pass
                uint32_t yb[8];
                if (here) {
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
                        for (int j = 0; j < 4; ++j) xv[j] = ld_smem_v4(sb + kOffX + j * xp + off);
                    }
                    if (kPost) {
                        // X'_k = post_k * Delta + sum_j comb[j,k] X_j, in this order for every column
                        float2 dl[4], xf[4][4];
                        unpack4(ld_smem_v4(sb + offd + off), dl);
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
                            st_smem_v4(sb + kOffX + k * xp + off, ov);
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
                            st_smem_v4(sb + offd + off, make_uint4(o[0], o[1], o[2], o[3]));
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
                tmem_st8(tl + kYColN + static_cast<uint32_t>((g % kRingN) * 16 + h * 8), yb);
                }
                if (kPost) fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarXReady + sl.idx));
                // drain the previous pass's accumulator now: its MMA ran while this pass was
                // computed, so nothing waits here, and the MMA of this pass (which needs the
                // accumulator empty) is issued right after
                if (kPost && s > 0) drain(g - 1, pass_ok(s - 1));
            }
            drain(g - 1, pass_ok(SP - 1));
            y_ready(g - 1);
            // the next tile's coefficients, loaded now (this tile's are no longer read) so that their
            // latency passes while the partial sums below are written and published: the publishing
            // arrive waits for this thread's stores, and the next tile's first pass would wait for
            // these loads
            if (it + 1 < my_tiles) load_coefs(it + 1);

            // this CTA's partial sums of the tile, for the split warp to publish to the group. The
            // workspace block of tile it reuses that of tile it - 2, which the other CTAs of the group
            // may still be reading; each of them publishes tile it - 1 only after it has read tile
            // it - 2, and this CTA's split warp signals split_done(it - 1) only after it has seen all
            // those arrivals (and read tile it - 1 itself). Compute warps that write the workspace
            // therefore wait for split_done(it - 1); where the split warp writes it, its own order
            // gives the same.
            const float2 sxx = __fadd2_rn(__fadd2_rn(sx[0], sx[1]), __fadd2_rn(sx[2], sx[3]));
            const float2 syy = __fadd2_rn(sy[0], sy[1]);
            float sxs = sxx.x + sxx.y, sys = syy.x + syy.y;
            float* P;
            int prow = trow;  // the block's row of this thread's sums
            if constexpr (kPartInSmem) {
                // into shared memory; the split warp writes the block to the workspace, so the arrive
                // below has no global stores to wait for (a memory round trip per tile otherwise).
                // Folded, rows 64..127 keep their own row: the split warp adds them to rows 0..63
                if (it > 0) W.wait(bar(kBarPartEmpty), static_cast<uint32_t>((it - 1) & 1), kErrComputeAcc);
                P = reinterpret_cast<float*>(smem + kOffPart);
                prow = row;
            } else {
                if (it > 0) W.wait(bar(kBarSplitDone), static_cast<uint32_t>((it - 1) & 1), kErrExchange);
                P = p.ws_part + (static_cast<size_t>(cid * 2 + static_cast<int>(it & 1)) * kG + rank) * kPartFloats;
            }
            {
                float4* pm4 = reinterpret_cast<float4*>(P + prow * kMix + 12 * h);
                pm4[0] = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
                pm4[1] = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
                pm4[2] = make_float4(acc[4].x, acc[4].y, acc[5].x, acc[5].y);
            }
            P[kPartSx + 2 * prow + h] = sxs;
            P[kPartSy + 2 * prow + h] = sys;
            // hand the block to the split warp, which publishes it (the arrive is a release: in
            // unfolded pre mode it waits for this warp's workspace stores)
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarPublish));
        }
    } else if (warp >= kWarpEpi0) {
        // ================= epilogue warps: y_normed = bf16(norm_w * y * r_y), one quadrant each ===
        const int q = warp & 3;
        // folded: quadrants 2 and 3 hold the tokens of quadrants 0 and 1 at each pass's second stage
        const int sub = kFold ? (q >> 1) : 0;
        const int qt = kFold ? (q & 1) : q;   // this warp's 32 token rows: 32 qt .. 32 qt + 31
        const int trow = 32 * qt + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
        float* nw = reinterpret_cast<float*>(smem + kOffNormW);
        // norm_w of this CTA's columns, loaded by the epilogue warps themselves: off the path to the
        // first loads, and needed only once a tile's exchange is complete
        for (int i = threadIdx.x - kWarpEpi0 * 32; i < p.d_slice; i += 4 * 32)
            nw[i] = p.norm_w[stage_col(i / kChunk) + i % kChunk];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarNormW));
        W.wait(bar(kBarNormW), 0u, kErrEpilogue);
        const float inv_d = 1.0f / static_cast<float>(p.d);
        long long g = 0;
        long long ystores = 0;  // TMA stores this warp has issued (staging tiles alternate)
        for (long long it = 0; it < my_tiles; ++it) {
            const int buf = static_cast<int>(it & 1);
            // r_y of this thread's row from the group's sums of y^2 (2 halves of each of the kG
            // column shares), once the split warp has seen the group's arrivals for the tile
            W.wait(bar(kBarFlagsSeen + buf), static_cast<uint32_t>((it >> 1) & 1), kErrEpilogue);
            const float* blk =
                p.ws_part + (static_cast<size_t>(cid * 2 + buf) * kG) * kPartFloats + kPartSy + 2 * trow;
            // all kG loads in flight at once (one L2 round trip), summed in share order
            float2 sq[kG];
#pragma unroll
            for (int r = 0; r < kG; ++r) sq[r] = ld_cg_f2(blk + static_cast<size_t>(r) * kPartFloats);
            float ssq = 0.f;
#pragma unroll
            for (int r = 0; r < kG; ++r) ssq += sq[r].x + sq[r].y;
            const float ry = rsqrtf(ssq * inv_d + p.norm_eps);  // the norm's rsqrt of mean(y^2) + eps
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarEpiRead));  // this warp is done with the tile's blocks
            const long long t0 = (cid + it * ncl) * p.tile_m;
            // this warp's rows go out as one TMA tile: 32 rows, or the tile's last tile_m % 32 rows
            // through the second map (rows past n are clipped by the maps; rows past tile_m belong
            // to the next tile and are never stored)
            const int rows_q = p.tile_m - 32 * qt;
            const bool store = p.write_y && rows_q > 0;
            const CUtensorMap* ymap = rows_q >= 32 ? &tmY : &tmYr;
            for (int s = 0; s < SP; ++s, ++g) {
                const int cs = kFold ? 2 * s + sub : s;  // the column stage of this warp's rows
                const int ys = static_cast<int>(g % kRingN);
                W.wait(bar(kBarYReady + ys), static_cast<uint32_t>((g / kRingN) & 1), kErrEpilogue);
                tc_fence_after();
                uint32_t yv[16];
                tmem_ld16_wait(tl + kYColN + static_cast<uint32_t>(ys * 16), yv);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarYFree + ys));
                if (store && cs < S) {
                    // TMEM columns ys*16 + 0..7 hold stage columns 0..15 (half 0), + 8..15 hold 16..31;
                    // y_normed = norm_w * (y * r_y), two columns per instruction
                    const float2* w = reinterpret_cast<const float2*>(nw + cs * 32);
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
                        tma_store_2d(ymap, st, stage_col(cs), static_cast<int>(t0 + 32 * qt));
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
            pol_stream = policy_evict_normal();
            pol_keep = policy_evict_last();
        }
        long long last_round[kMaxStages];  // the latest pass loaded into each slot
#pragma unroll
        for (int i = 0; i < kMaxStages; ++i) last_round[i] = -1;
        for (long long it = 0; it < my_tiles; ++it) {
            const long long tile = cid + it * ncl;
            const int t0 = static_cast<int>(tile * p.tile_m);
            for (int s = 0; s < SP; ++s) {
                const Slot sl = slot_at(it, s);
                last_round[sl.idx] = sl.round;
                if (early(it, s)) continue;  // issued at the start
                if (sl.round > 0)
                    W.wait(bar(kBarEmpty + sl.idx), static_cast<uint32_t>((sl.round - 1) & 1), kErrProducer);
                if (lane == 0) issue_pass(sl, s, t0, pol_stream, pol_keep);
                __syncwarp();
            }
        }
        // let every load issued land before the CTA can exit (a slot's latest load lands after its
        // earlier ones, which the compute warps consumed before the slot was reused)
#pragma unroll
        for (int i = 0; i < kMaxStages; ++i)
            if (i < kNumSlots && last_round[i] >= 0) W.drain(bar(kBarFull + i), static_cast<uint32_t>(last_round[i] & 1));
    } else if (warp == kWarpMma) {
        // ================= MMA issuer ===========================================================
        constexpr uint32_t idesc = idesc_bf16_f32(kUmmaM, kFold ? kUmmaNFold : kUmmaN);
        long long g = 0;
        for (long long it = 0; it < my_tiles; ++it) {
            for (int s = 0; s < SP; ++s, ++g) {
                const Slot sl = slot_at(it, s);
                // this pass's accumulator must have been drained (pass g - kNAcc)
                if (g >= kNAcc) W.wait(acc_empty(g), static_cast<uint32_t>((g / kNAcc - 1) & 1), kErrMma);
                // post mode multiplies the X' the compute warps wrote; the other modes the loaded tile
                W.wait(bar((kPost ? kBarXReady : kBarFull) + sl.idx), static_cast<uint32_t>(sl.round & 1), kErrMma);
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sb = sl.base;
                    const uint32_t dcol = tmem + acc_col(g);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const uint64_t ad = sdesc_kmajor_sw64(sb + kOffX + (kExpand ? 0 : k * x_pitch(s)) + kk * 32);
                            const uint64_t bd = sdesc_kmajor_sw64(sb + sl.offb + k * b_pitch(s) + kk * 32);
                            umma_bf16(dcol, ad, bd, idesc, (k | kk) != 0 ? 1u : 0u);
                        }
                    }
                    umma_commit(bar(kBarEmpty + sl.idx));
                    umma_commit(acc_full(g));
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
            for (int s = 0; s < SP; ++s, ++g) {
                const Slot sl = slot_at(it, s);
                W.wait(bar(kBarXReady + sl.idx), static_cast<uint32_t>(sl.round & 1), kErrStore);
                if (kWriteX && lane == 0) {
                    const uint32_t sb = sl.base;
                    const int halves = (kFold && 2 * s + 1 < S) ? 2 : 1;
                    if (kPost && halves == 2 && p.combined) {
                        // both stages of the four streams in one box, the tap's two in another
                        tma_store_4d(&tmXo4, sb + kOffX, stage_col(2 * s), t0, 0, 0);
                        if (p.stream_mean) tma_store_3d(&tmM3, sb + sl.offd, stage_col(2 * s), t0, 0);
                    } else if (kPost && compact(s)) {
                        tma_store_3d(&tmXo3s, sb + kOffX, stage_col(2 * s), t0, 0);  // the compact tiles
                        if (p.stream_mean) tma_store_2d(&tmM, sb + sl.offd, stage_col(2 * s), t0);
                    } else {
                        for (int hf = 0; hf < halves; ++hf) {
                            const int col = stage_col(kFold ? 2 * s + hf : s);
                            const uint32_t xo = static_cast<uint32_t>(hf * kFoldXHalf);
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                tma_store_3d(&tmXo, sb + kOffX + (kExpand ? 0 : k * kXTileBytes) + xo, col, k, t0);
                            if (kPost && p.stream_mean) tma_store_2d(&tmM, sb + sl.offd + xo, col, t0);  // the tap
                        }
                    }
                    bulk_commit();
                    bulk_wait_read<0>();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarEmpty + sl.idx));
            }
        }
        if (lane == 0) bulk_wait<0>();
    } else {  // warp == kWarpSplit
        // ===== group exchange, r_y of every row, split + Sinkhorn for this CTA's share ==========
        // hc_scale and hc_base into shared memory now, read from there by each split (not held in
        // registers through the gather)
        float* prm = reinterpret_cast<float*>(smem + kOffSplitPrm);
        if (lane < 3) prm[lane] = __ldg(p.hc_scale + lane);
        if (lane < kMix) prm[3 + lane] = __ldg(p.hc_base + lane);
        __syncwarp();
        // the group's arrival counter and its value when this launch started
        unsigned long long* arrivals = p.ws_arrivals + static_cast<size_t>(cid) * kCounterStride;
        unsigned long long base = 0;
        if (lane == 0) base = ld_acquire_gpu_u64(p.ws_launch + cid);
        base = __shfl_sync(0xffffffffu, base, 0);
        for (long long it = 0; it < my_tiles; ++it) {
            const int buf = static_cast<int>(it & 1);
            // the compute warps have written this CTA's block of the tile: publish it, then wait for
            // the group (lane 0 polls the group's arrival counter)
            W.wait(bar(kBarPublish), static_cast<uint32_t>(it & 1), kErrSplit);
            // an arrival also says that this CTA is done reading the group's blocks of the previous
            // tile (whose buffer the group reuses after this tile): the split warp read them in its
            // last iteration, the epilogue warps read the sums of y^2
            if (it >= 1) W.wait(bar(kBarEpiRead), static_cast<uint32_t>((it - 1) & 1), kErrSplit);
            if constexpr (kPartInSmem) {
                // the CTA's block from shared memory to its place in the workspace. That place held tile
                // it - 2, which every CTA of the group had read before it added its arrival of tile
                // it - 1, which this warp has seen. Each store consumes its load, so when the last store
                // has issued the block may be reused (a relaxed arrival: the stores need not complete)
                const float4* src = reinterpret_cast<const float4*>(smem + kOffPart);
                float4* dst = reinterpret_cast<float4*>(p.ws_part + (static_cast<size_t>(cid * 2 + buf) * kG + rank) * kPartFloats);
                if constexpr (kFold) {
                    // rows 0..63 (each pass's first stage) plus rows 64..127 (the same tokens at its
                    // second stage), in that order: the mixes are float4 i < 384 (row i / 6) with the
                    // partner 384 further on; the sums of x^2 and of y^2 are 32 float4 each (two rows'
                    // halves per float4) with the partner 32 further on. Rows 64..127 of the workspace
                    // block are not read.
                    constexpr int kMixV = kFoldRows * kMix / 4, kSumV = kFoldRows * 2 / 4;
                    static_assert((kMixV + 2 * kSumV) % 32 == 0, "whole warps");
#pragma unroll 7
                    for (int i = lane; i < kMixV + 2 * kSumV; i += 32) {
                        const int a = i < kMixV ? i
                                      : i < kMixV + kSumV ? kPartSx / 4 + (i - kMixV)
                                                           : kPartSy / 4 + (i - kMixV - kSumV);
                        const int b = a + (i < kMixV ? kMixV : kSumV);
                        const float4 u = src[a], v = src[b];
                        dst[a] = make_float4(u.x + v.x, u.y + v.y, u.z + v.z, u.w + v.w);
                    }
                } else {
                    constexpr int kPer = kPartFloats / 4 / 32, kChunkV = 7;  // 28 float4 per lane, 7 at a time
                    static_assert(kPer % kChunkV == 0, "copy chunks");
#pragma unroll
                    for (int c0 = 0; c0 < kPer; c0 += kChunkV) {
                        float4 v[kChunkV];
#pragma unroll
                        for (int c = 0; c < kChunkV; ++c) v[c] = src[lane + 32 * (c0 + c)];
#pragma unroll
                        for (int c = 0; c < kChunkV; ++c) dst[lane + 32 * (c0 + c)] = v[c];
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed(bar(kBarPartEmpty), 1u);
            }
            // the block's writes happen before the add (the publish mbarrier, or this warp's own stores
            // and __syncwarp, order them within the CTA; the add's release orders them at GPU scope)
            if (lane == 0) red_release_gpu_add_u64(arrivals, 1ull);
            const unsigned long long target = base + static_cast<unsigned long long>(kG) * static_cast<unsigned long long>(it + 1);
            W.wait_count(arrivals, target, lane, 1, kErrExchange);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarFlagsSeen + buf));  // the epilogue warps may read the sums of y^2
            const long long tile = cid + it * ncl;
            const long long t0 = tile * p.tile_m;
            const float* blk = p.ws_part + (static_cast<size_t>(cid * 2 + buf) * kG) * kPartFloats;
            // the owned tokens t = rank + kG i (i < kT = 128 / kG, the first kTv of them in the tile). One
            // load instruction of the warp covers four shares' rows of one token: lane 4q + j (q < 6)
            // loads float4 q of the token's 24 mixes and lane 24 + j its two sums of x^2, from shares
            // j, j + 4, j + 8, ... (about four 128-byte lines per instruction, where one lane per share
            // and token scattered the loads over 16 to 32 lines). Each lane sums its shares in order, two
            // shuffle levels add the four phases, and the token's 24 mixes and sum of x^2 go through the
            // warp's shared-memory scratch to lane i, which runs the token's split. kBatch tokens' loads
            // are in flight at once (kBatch * kG / 4 = 16 per lane).
            constexpr int kT = kTileMax / kG, kPhases = 4, kPerPhase = kG / kPhases, kBatch = 64 / kG;
            static_assert(kBatch * kPerPhase == 16 && kT % kBatch == 0, "gather batches");
            int kTv = 0;  // owned tokens in this tile
            for (int i = 0; i < kT; ++i)
                if (static_cast<int>(rank) + kG * i < p.tile_m && t0 + rank + kG * i < p.n) kTv = i + 1;
            const int gq = lane >> 2, gj = lane & 3;  // float4 index (6: the sums of x^2), phase
            float* scr = reinterpret_cast<float*>(smem + kOffSplit);
            for (int i0 = 0; i0 < kTv; i0 += kBatch) {
                float4 u[kBatch][kPerPhase];
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    const int tok_row = static_cast<int>(rank) + kG * (i0 + b);
#pragma unroll
                    for (int m = 0; m < kPerPhase; ++m) {
                        u[b][m] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (i0 + b < kTv && lane < 28) {
                            const float* Pr = blk + static_cast<size_t>(kPhases * m + gj) * kPartFloats;
                            if (gq < 6) {
                                u[b][m] = ld_cg_f4(Pr + tok_row * kMix + 4 * gq);
                            } else {
                                const float2 v = ld_cg_f2(Pr + kPartSx + 2 * tok_row);
                                u[b][m] = make_float4(v.x, v.y, 0.f, 0.f);
                            }
                        }
                    }
                }
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    float4 a = u[b][0];
#pragma unroll
                    for (int m = 1; m < kPerPhase; ++m) {
                        a.x += u[b][m].x; a.y += u[b][m].y; a.z += u[b][m].z; a.w += u[b][m].w;
                    }
#pragma unroll
                    for (int x = 1; x <= 2; x <<= 1) {
                        a.x += __shfl_xor_sync(0xffffffffu, a.x, x);
                        a.y += __shfl_xor_sync(0xffffffffu, a.y, x);
                        a.z += __shfl_xor_sync(0xffffffffu, a.z, x);
                        a.w += __shfl_xor_sync(0xffffffffu, a.w, x);
                    }
                    if (gj == 0 && lane < 28 && i0 + b < kTv)
                        reinterpret_cast<float4*>(scr)[(i0 + b) * 7 + gq] =
                            gq < 6 ? a : make_float4(a.x + a.y, 0.f, 0.f, 0.f);
                }
            }
            __syncwarp();
            if constexpr (kFold) {
                // At most 64 / kG = 4 owned tokens. The steps of the split before its Sinkhorn rounds
                // (logits, sigmoids, row softmax) run with one lane per mix (lanes 0..23), each value
                // by the same operations as in split_sinkhorn: the row max and sum combine the four
                // lanes of a row as (0,1),(2,3) then the two pairs, as split_sinkhorn does. On one lane
                // those 24 exponentials and 8 divisions took about 1,600 of its 4,900 cycles. Token i's
                // rounds then run on lane i, which gathers its 16 softmax values by shuffles.
                constexpr int kOwn = kFoldRows / kG;
                static_assert(kOwn >= 1 && kOwn <= 4, "owned tokens of a folded tile");
                float mv[kOwn];  // lane k < 24: mix k of each owned token
#pragma unroll
                for (int i = 0; i < kOwn; ++i) {
                    mv[i] = 0.f;
                    if (i < kTv && lane < kMix) {
                        const float rr = rsqrtf(scr[i * 28 + 24] / static_cast<float>(4 * p.d) + p.norm_eps);
                        mv[i] = scr[i * 28 + lane] * rr;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarSplitDone));  // the blocks of this tile may be reused
                if (p.mixes_out && lane < kMix) {
#pragma unroll
                    for (int i = 0; i < kOwn; ++i)
                        if (i < kTv) p.mixes_out[(t0 + static_cast<int>(rank) + kG * i) * kMix + lane] = mv[i];
                }
                if (p.pre_out) {
                    const float bk = lane < kMix ? prm[3 + lane] : 0.f;
                    const float sck = prm[lane < 4 ? 0 : lane < 8 ? 1 : 2];
                    float cv[kOwn];  // lanes 8..23: entry lane - 8 of each token's softmax, + eps
#pragma unroll
                    for (int i = 0; i < kOwn; ++i) {
                        const float l = fmaf(mv[i], sck, bk);
                        float mx = fmaxf(l, __shfl_xor_sync(0xffffffffu, l, 1));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                        const float x = expf(l - mx);
                        float sm = x + __shfl_xor_sync(0xffffffffu, x, 1);
                        sm = sm + __shfl_xor_sync(0xffffffffu, sm, 2);
                        cv[i] = fmaf(x, rcp_refined(sm), p.hc_eps);
                        if (i < kTv && lane < 8) {
                            const long long tok = t0 + static_cast<int>(rank) + kG * i;
                            if (lane < 4)
                                p.pre_out[tok * 4 + lane] = sigmoidf_(l) + p.hc_eps;
                            else
                                p.post_out[tok * 4 + (lane - 4)] = 2.0f * sigmoidf_(l);
                        }
                    }
                    float2 C2[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        float a = 0.f, b = 0.f;
#pragma unroll
                        for (int i = 0; i < kOwn; ++i) {
                            const float va = __shfl_sync(0xffffffffu, cv[i], 8 + 2 * q);
                            const float vb = __shfl_sync(0xffffffffu, cv[i], 9 + 2 * q);
                            if (lane == i) { a = va; b = vb; }
                        }
                        C2[q] = make_float2(a, b);
                    }
                    if (lane < kTv) {
                        sinkhorn_rounds(C2, p.iters, p.hc_eps);
                        const long long tok = t0 + static_cast<int>(rank) + kG * lane;
                        float4* co = reinterpret_cast<float4*>(p.comb_out) + tok * 4;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            co[j] = make_float4(C2[2 * j].x, C2[2 * j].y, C2[2 * j + 1].x, C2[2 * j + 1].y);
                    }
                }
            } else {
                const int oi = lane;  // lane i runs the split of owned token i
                const int r_tok = static_cast<int>(rank) + kG * oi;
                const bool mine = oi < kTv;
                float m[kMix];
                float sxt = 0.f;
                if (mine) {
                    const float4* sv = reinterpret_cast<const float4*>(scr) + oi * 7;
    #pragma unroll
                    for (int k = 0; k < 6; ++k) {
                        const float4 v = sv[k];
                        m[4 * k] = v.x; m[4 * k + 1] = v.y; m[4 * k + 2] = v.z; m[4 * k + 3] = v.w;
                    }
                    sxt = sv[6].x;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarSplitDone));  // the blocks of this tile may be reused
                if (mine) {
                    const long long tok = t0 + r_tok;
                    const float rr = rsqrtf(sxt / static_cast<float>(4 * p.d) + p.norm_eps);  // rsqrt of mean(x^2) + eps
    #pragma unroll
                    for (int i = 0; i < kMix; ++i) m[i] *= rr;
                    if (p.mixes_out) {
                        float4* mo = reinterpret_cast<float4*>(p.mixes_out + tok * kMix);
    #pragma unroll
                        for (int i = 0; i < kMix / 4; ++i) mo[i] = make_float4(m[4 * i], m[4 * i + 1], m[4 * i + 2], m[4 * i + 3]);
                    }
                    if (p.pre_out) {
                        float pre[4], post[4], C[16];
                        float sc[3], bs[kMix];
    #pragma unroll
                        for (int i = 0; i < 3; ++i) sc[i] = prm[i];
    #pragma unroll
                        for (int i = 0; i < kMix; ++i) bs[i] = prm[3 + i];
                        split_sinkhorn(m, sc, bs, p.iters, p.hc_eps, pre, post, C);
                        reinterpret_cast<float4*>(p.pre_out)[tok] = make_float4(pre[0], pre[1], pre[2], pre[3]);
                        reinterpret_cast<float4*>(p.post_out)[tok] = make_float4(post[0], post[1], post[2], post[3]);
                        float4* co = reinterpret_cast<float4*>(p.comb_out) + tok * 4;
    #pragma unroll
                        for (int j = 0; j < 4; ++j) co[j] = make_float4(C[4 * j], C[4 * j + 1], C[4 * j + 2], C[4 * j + 3]);
                    }
                }
            }
            __syncwarp();
        }
        // every CTA of the group has read the base and added its last arrival (the counter reached
        // the last tile's target, which this warp has seen): store the final count as the next base
        if (rank == 0 && lane == 0 && my_tiles > 0)
            st_release_gpu_u64(p.ws_launch + cid,
                               base + static_cast<unsigned long long>(kG) * static_cast<unsigned long long>(my_tiles));
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
    uint32_t estr[4] = {1, 1, 1, 1};
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

// every instantiation of the fused kernel: [mode][group size 8, 16, 32]; groups of 16 and 32 always
// fold their tiles (at most 64 tokens), groups of 8 never, so that a token's mixes (the order in
// which its partial sums meet) depend on the group size alone
constexpr bool fold_of(int group) { return group != 8; }

template <int kMode>
void kernels_of_mode(const void** k, int* smem) {
    k[0] = reinterpret_cast<const void*>(&hc_fused_kernel<kMode, 8, fold_of(8)>);
    k[1] = reinterpret_cast<const void*>(&hc_fused_kernel<kMode, 16, fold_of(16)>);
    k[2] = reinterpret_cast<const void*>(&hc_fused_kernel<kMode, 32, fold_of(32)>);
    smem[0] = Layout<kMode, fold_of(8)>::kSmemBytes;
    smem[1] = Layout<kMode, fold_of(16)>::kSmemBytes;
    smem[2] = Layout<kMode, fold_of(32)>::kSmemBytes;
}

template <int kMode>
int smem_of(int group) {
    return group == 8 ? Layout<kMode, fold_of(8)>::kSmemBytes
                      : group == 16 ? Layout<kMode, fold_of(16)>::kSmemBytes : Layout<kMode, fold_of(32)>::kSmemBytes;
}

int prepare_device(int* ctas) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -7;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
        const void* kernels[9];
        int k_smem[9];
        kernels_of_mode<kModePre>(kernels, k_smem);
        kernels_of_mode<kModePost>(kernels + 3, k_smem + 3);
        kernels_of_mode<kModeExpand>(kernels + 6, k_smem + 6);
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

// Launch plan: for each group size g (d a multiple of 32 g) and tile height m, groups = ctas / g
// groups run at once; a launch takes ceil(tiles / groups) waves, each of P passes over a tile plus
// a per-tile cost (group exchange, y_normed epilogue tail). Groups of 8 take tiles of 32, 64, 96 or
// 128 tokens (or a balanced height of 96..128 for batches of several waves, or n when n < 32) and
// make one pass per column stage, P = S = d / (32 g). Groups of 16 and 32 fold: tiles of 64 tokens,
// two column stages per pass in the 128 rows of the MMA, P = ceil(S / 2), every pass loaded with one
// box per tensor (a folded pass costs the same whatever the tokens of its tile).
// A pass costs the larger of its latency floor and a fixed part plus a part per row in use (a folded
// pass uses all 128 rows); the constants were measured on GB300 (2.1 us per 128-row pass of the
// prefill step, about 0.8 us for a pass of a small batch, about 4 us per tile).
void plan_tiles(int64_t n, int d, int ctas, int only_group, int* group, int* tile_m, int64_t* num_tiles) {
    *group = 8;
    *tile_m = kTileMax;
    *num_tiles = 0;
    if (n <= 0) return;
    constexpr double kPassFloorUs = 0.8, kPassFixedUs = 0.5, kPassPerRowUs = 1.6 / kTileMax, kTileUs = 4.0;
    double best = -1.0;
    const int gs[3] = {8, 16, 32};
    for (int g : gs) {
        if (d % (kChunk * g) != 0 || (only_group != 0 && g != only_group)) continue;
        const int groups = ctas / g;
        if (groups < 1) continue;
        const bool fold = fold_of(g);
        const int S = d / (kChunk * g);
        const int P = fold ? (S + 1) / 2 : S;
        // tile heights, largest first (ties keep the larger tile and the smaller group), then for
        // unfolded batches of several waves the height that spreads the tokens evenly over the waves
        // 128-token tiles would take (16,384 tokens: 133 tiles of 124 fill 7 waves of 19 groups,
        // where 128 tiles of 128 leave 5 groups idle in the last); only from 96 rows up, where a
        // stage's time still follows its rows (shorter balanced tiles measured slower)
        const int64_t waves128 = ((n + kTileMax - 1) / kTileMax + groups - 1) / groups;
        const int m_even = static_cast<int>((n + groups * waves128 - 1) / (groups * waves128));
        const int ms[6] = {fold ? 0 : 128, fold ? 0 : 96, 64, fold ? 0 : 32, !fold && n < 32 ? static_cast<int>(n) : 0,
                           !fold && waves128 > 1 && m_even >= 96 ? m_even : 0};
        for (int m : ms) {
            if (m < 1) continue;
            const int64_t tiles = (n + m - 1) / m;
            const int64_t waves = (tiles + groups - 1) / groups;
            // a folded pass runs all 128 rows of the tile in every compute warp
            const int rows = fold ? kTileMax : m;
            const double pass = std::max(kPassFloorUs, kPassFixedUs + rows * kPassPerRowUs);
            const double cost = static_cast<double>(waves) * (P * pass + kTileUs);
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
        if (!encode(&tmX, x_in, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B)) return -7;
        if (!encode(&tmXo, write_x ? a.X_out : a.X, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B)) return -7;
    }
    {
        const uint64_t dims[2] = {d, n};
        const uint64_t str[1] = {d * 2};
        const uint32_t box[2] = {kChunk, static_cast<uint32_t>(tile_m)};
        if (!encode(&tmD, rows, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B)) return -7;
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
    // Folded 64-token tiles load a pass of two stages with one box per tensor: views with a "stage"
    // dimension of 2 whose stride is the group's column step (a CTA's stages are kG * 32 columns
    // apart); the box lands as [stream][stage][token][32 columns], which is the folded slot's layout.
    // These maps are used only for passes whose two stages exist, so no box reaches past a row. For
    // other launches they are placeholders, never read.
    const bool combined = fold_of(group) && tile_m == kFoldRows;
    CUtensorMap tmX4 = tmX, tmXo4 = tmXo, tmD3 = tmD, tmM3 = tmM, tmB4 = tmB, tmX3s = tmX, tmXo3s = tmXo, tmB3 = tmB;
    {
        // the four streams' plane tiles of one stage in one box, 4,608 bytes apart
        const uint64_t dims[3] = {d, static_cast<uint64_t>(kBRows), 4};
        const uint64_t str[2] = {4 * d * 2, d * 2};
        const uint32_t box[3] = {kChunk, static_cast<uint32_t>(kBRows), 4};
        if (!encode(&tmB3, a.planes, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B)) return -7;
    }
    if (combined) {
        {
            // a compact one-stage pass: the four streams' 64 rows, 4 KB apart
            const uint64_t dims[3] = {d, n, 4};
            const uint64_t str[2] = {4 * d * 2, d * 2};
            const uint32_t box[3] = {kChunk, static_cast<uint32_t>(kFoldRows), 4};
            if (!encode(&tmX3s, x_in, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B)) return -7;
            if (!encode(&tmXo3s, write_x ? a.X_out : a.X, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B)) return -7;
        }
        const uint64_t cs = static_cast<uint64_t>(group) * kChunk * 2;
        {
            const uint64_t dims[4] = {d, n, 2, 4};
            const uint64_t str[3] = {4 * d * 2, cs, d * 2};
            const uint32_t box[4] = {kChunk, static_cast<uint32_t>(kFoldRows), 2, 4};
            if (!encode(&tmX4, x_in, 4, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B)) return -7;
            if (!encode(&tmXo4, write_x ? a.X_out : a.X, 4, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B)) return -7;
        }
        {
            const uint64_t dims[3] = {d, n, 2};
            const uint64_t str[2] = {d * 2, cs};
            const uint32_t box[3] = {kChunk, static_cast<uint32_t>(kFoldRows), 2};
            if (!encode(&tmD3, rows, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B)) return -7;
            if (!encode(&tmM3, a.stream_mean ? a.stream_mean : rows, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B))
                return -7;
        }
        {
            const uint64_t dims[4] = {d, static_cast<uint64_t>(kBRows), 2, 4};
            const uint64_t str[3] = {4 * d * 2, cs, d * 2};
            const uint32_t box[4] = {kChunk, static_cast<uint32_t>(kBRows), 2, 4};
            if (!encode(&tmB4, a.planes, 4, dims, str, box, CU_TENSOR_MAP_SWIZZLE_64B)) return -7;
        }
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
    p.ws_arrivals = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(a.workspace) + kWsPartBytes);
    p.ws_launch =
        reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(a.workspace) + kWsPartBytes + kWsFlagBytes);
    p.n = a.n;
    p.num_tiles = num_tiles;
    p.write_y = a.y_normed != nullptr;
    p.d = a.d;
    p.d_slice = a.d / group;
    p.stages_per_tile = p.d_slice / kChunk;
    p.tile_m = tile_m;
    p.combined = combined ? 1 : 0;
    p.iters = a.iters;
    p.hc_eps = a.hc_eps;
    p.norm_eps = a.norm_eps;

    const int64_t grid_groups = std::min<int64_t>(num_tiles, ctas / group);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident together: the group counters can be awaited
    attr[0].val.cooperative = 1;
    // programmatic dependent launch: the kernel's set-up may overlap the end of the kernel ahead
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid_groups * group), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = a.mode == kModePost     ? smem_of<kModePost>(group)
                           : a.mode == kModeExpand ? smem_of<kModeExpand>(group)
                                                   : smem_of<kModePre>(group);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaErrorInvalidValue;
    auto go = [&](auto kernel) {
        e = cudaLaunchKernelEx(&cfg, kernel, tmX, tmD, tmB, tmXo, tmM, tmY, tmYr, tmX4, tmXo4, tmD3, tmM3, tmB4, tmX3s,
                               tmXo3s, tmB3, p);
    };
    if (a.mode == kModePost) {
        if (group == 8) go(hc_fused_kernel<kModePost, 8, fold_of(8)>);
        else if (group == 16) go(hc_fused_kernel<kModePost, 16, fold_of(16)>);
        else go(hc_fused_kernel<kModePost, 32, fold_of(32)>);
    } else if (a.mode == kModeExpand) {
        if (group == 8) go(hc_fused_kernel<kModeExpand, 8, fold_of(8)>);
        else if (group == 16) go(hc_fused_kernel<kModeExpand, 16, fold_of(16)>);
        else go(hc_fused_kernel<kModeExpand, 32, fold_of(32)>);
    } else {
        if (group == 8) go(hc_fused_kernel<kModePre, 8, fold_of(8)>);
        else if (group == 16) go(hc_fused_kernel<kModePre, 16, fold_of(16)>);
        else go(hc_fused_kernel<kModePre, 32, fold_of(32)>);
    }
    return e == cudaSuccess ? 0 : -7;
}

// ---- scratch that needs no allocation ------------------------------------------------------------
// The workspace of hc_post_then_pre_noalloc: a fixed array in the library's device image, one per
// GPU that loads the library, zero at load and kept until the process exits. Its size is the same
// kWorkspaceBytes (7,344,384 bytes: room for 256 co-resident CTAs) that hc_workspace_size reports.
static __device__ __align__(256) unsigned char g_noalloc_workspace[kWorkspaceBytes];
// A launch never needs more scratch than this: the fused kernel runs at most kMaxCtas CTAs (the
// device's resident count is capped there) and the generic path works through its tokens in chunks
// sized to kWorkspaceBytes, so no call is ever refused for want of room in the array.
static_assert(sizeof(g_noalloc_workspace) >= kWorkspaceBytes && kWorkspaceBytes >= kWsPartBytes &&
                  kWsPartBytes == static_cast<size_t>(kMaxCtas) * 2 * kPartFloats * 4,
              "the fixed scratch holds the partial sums of kMaxCtas CTAs and the groups' counters");

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
            // A kernel gave up a wait: a CTA of its group may still add arrivals to the group's
            // counter after the group's base has moved on, and the group's next launch would count
            // them as its own. The library's fixed scratch (hc_post_then_pre_noalloc) therefore
            // starts afresh from zero; a memset is not an allocation. Caller workspaces are the
            // caller's to zero (hc.h).
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
