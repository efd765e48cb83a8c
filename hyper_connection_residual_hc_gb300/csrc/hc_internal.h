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
};

// Launch plan of the fused kernel for n tokens of width d when `ctas` CTAs can be resident at once:
// CTAs per token tile (8, 16 or 32), tokens per tile and number of tiles.
void plan_tiles(int64_t n, int d, int ctas, int* group, int* tile_m, int64_t* num_tiles);

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
