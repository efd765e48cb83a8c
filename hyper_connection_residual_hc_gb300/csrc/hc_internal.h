// Host-side declarations shared by the library's translation units (not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace hc {

// What the fused kernel does before the reading half.
enum FusedMode : int {
    kModePre = 0,     // hc_pre_step: the reading half of X as it is
    kModePost = 1,    // hc_post_then_pre: X' = hc_post(delta, X, post, comb) first, written to X_out
    kModeExpand = 2,  // hc_expand_pre_step: X' = the embedding in every stream, written to X_out,
                      // read with the identity pre_mix
};

// Everything one fused launch needs. Device pointers; optional ones may be null.
struct FusedArgs {
    int mode;                // FusedMode
    const void* X;           // bf16 [n, 4, d]           (pre and post modes)
    const void* embed;       // bf16 [n, d]              (expand mode)
    const void* delta;       // bf16 [n, d]            (post mode)
    const float* post;       // fp32 [n, 4]            (post mode)
    const float* comb;       // fp32 [n, 4, 4]         (post mode)
    const float* pre_mix;    // fp32 [n, 4]            (null: zeros, diagnostic use; ignored in expand mode)
    const void* planes;      // bf16 [72, 4d]
    const float* hc_scale;   // fp32 [3]
    const float* hc_base;    // fp32 [24]
    const float* norm_w;     // fp32 [d]
    void* X_out;             // bf16 [n, 4, d]         (post and expand modes)
    void* y_normed;          // bf16 [n, d]            (null: not written)
    float* pre_out;          // fp32 [n, 4]            (null: not written)
    float* post_out;         // fp32 [n, 4]
    float* comb_out;         // fp32 [n, 4, 4]
    float* mixes_out;        // fp32 [n, 24]           (null: not written)
    void* stream_mean;       // bf16 [n, d]            (post mode; null: not written)
    void* workspace;         // workspace_bytes(), zero-filled before its first use
    int64_t n;
    int d;
    int iters;
    float hc_eps;
    float norm_eps;
    int group;               // CTAs per token tile: 0 = the launch plan's choice, else 8, 16 or 32
};

// Launch plan of the fused kernel for n tokens of width d when `ctas` CTAs can be resident at once:
// CTAs per token tile (8, 16 or 32), tokens per tile and number of tiles.
// only_group: 0 = any group size; 8, 16 or 32 = that one only (no tiles if d does not allow it)
void plan_tiles(int64_t n, int d, int ctas, int only_group, int* group, int* tile_m, int64_t* num_tiles);

// Launches the fused kernel; returns 0, -7 (CUDA failure) or -3 (no cooperative launch).
int launch_fused(const FusedArgs& a, cudaStream_t stream);

// Everything one launch of the tail-of-stack kernel needs (device pointers).
struct FinalArgs {
    const void* X;           // bf16 [n, 4, d]
    const void* delta;       // bf16 [n, d]   null: no writing half (hc_final)
    const float* post;       // fp32 [n, 4]   (with delta)
    const float* comb;       // fp32 [n, 4, 4] (with delta)
    const float* pre_mix;    // fp32 [n, 4]
    const float* norm_w;     // fp32 [d]
    void* X_out;             // bf16 [n, 4, d] or null (with delta)
    void* z;                 // bf16 [n, d]
    int64_t n;
    int d;                   // multiple of 8, at most kFinalMaxD
    float norm_eps;
};
constexpr int kFinalMaxD = 5120;

// Launches the tail-of-stack kernel; returns 0 or -7.
int launch_final(const FinalArgs& a, cudaStream_t stream);

// Row of the prepared weight planes that holds plane pl (0 hi, 1 mid, 2 lo) of mix m, for hc
// streams and M = (2 + hc) * hc mixes: the fused kernel's grouping at hc = 4 (row 36h + 12 pl + i
// for mix 12h + i, so that one warp drains one half of the mixes from contiguous accumulator
// columns), plane-major (row pl * M + m) for any other hc.
__host__ __device__ inline int plane_row(int hc, int M, int pl, int m) {
    return hc == 4 ? 36 * (m / 12) + 12 * pl + m % 12 : pl * M + m;
}

// The generic path (any hc in 1..8, any d multiple of 8): plain CUDA-core kernels for the shapes
// the fused kernel does not take.
struct GenericArgs {
    const void* X;           // bf16 [n, hc, d]: the streams the reading half reads
    const float* pre_mix;    // fp32 [n, hc], unless identity
    int identity;            // 1: pre_mix is 1/hc for every stream (head of the stack)
    const void* planes;      // bf16 planes of hc_prepare_params
    const float* hc_scale;
    const float* hc_base;
    const float* norm_w;
    void* y_normed;          // bf16 [n, d], or null (debug mixes)
    float* pre_out;
    float* post_out;
    float* comb_out;
    float* mixes_out;        // fp32 [n, M]: debug mixes instead of the coefficients, or null
    void* workspace;         // workspace_bytes(): raw mixes and sums of squares, a chunk of tokens at a time
    int64_t n;
    int hc;
    int d;
    int iters;
    float hc_eps;
    float norm_eps;
};
size_t generic_tokens_per_chunk(int hc);
int launch_generic_post(const void* X, const void* delta, const float* post, const float* comb, void* X_out,
                        void* mean_out, int64_t n, int hc, int d, cudaStream_t stream);
int launch_generic_expand(const void* h, void* X_out, int64_t n, int hc, int d, cudaStream_t stream);
int launch_generic_reading(const GenericArgs& a, cudaStream_t stream);
// The generic path's projection on the tensor cores (csrc/hc_proj.cu): raw [m, M] and ssx [m] of the
// m tokens of X (bf16 [m, hc * d]) against the prepared planes; returns 0, -3 (a shape it does not
// take: hc outside 1..8 or d not a multiple of 8) or -7 (CUDA).
int launch_proj_tc(const void* X, const void* planes, int64_t m, int hc, int d, float* raw, float* ssx,
                   cudaStream_t stream);
// The projection kernel's device error word (read, and cleared if asked); returns 0 or -7.
int read_proj_error(unsigned int* word, int clear, cudaStream_t stream);
int launch_generic_final(const void* X, const void* delta, const float* post, const float* comb,
                         const float* pre_mix, const float* norm_w, void* X_out, void* z, int64_t n, int hc, int d,
                         float eps, cudaStream_t stream);

// Diagnostic: one bounded wait (limit_ns) for flags[0..g-1] to equal value; 0 or -7.
int launch_wait_flag(const unsigned long long* flags, unsigned long long value, int g, uint64_t limit_ns,
                     cudaStream_t stream);

// Reads (and optionally clears) the device error word of the current device.
int read_device_error(unsigned int* word, int clear, cudaStream_t stream);

// CTAs of the fused kernel that can be resident at once on the current device (cached per device).
int fused_ctas(int* ctas);

// Bytes of the workspace the fused kernel exchanges partial sums through.
size_t workspace_bytes();

// Device address and size of the library's own fixed workspace on the current device (resolved
// once per device); returns 0 or -7.
int noalloc_workspace(void** ptr, size_t* capacity);

}  // namespace hc
