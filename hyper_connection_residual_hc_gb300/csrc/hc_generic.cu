// Hyper-Connection step for any number of streams hc (1..8) and any stream width d (a multiple of
// 8): plain CUDA-core kernels. The fused tcgen05 kernel covers the model's own shape (hc = 4, d a
// multiple of 256 up to 5120); these kernels make the same calls work for every other shape the
// formulas allow ("Source layer, pairs pooled" page: mix_hc = (2 + hc) * hc from Block.__init__;
// "Reading weights" page: hc_split_sinkhorn written for any hc_mult).
//
//   writing half   gen_post_kernel      X' = bf16(post_k * Delta + sum_j comb[j,k] X_j) (+ stream mean)
//   head           gen_expand_kernel    X' = the embedding in every stream
//   projection     gen_proj_tc_kernel   raw mixes sum_c X'_c w_mc and sum_c X'_c^2 on the tensor cores
//                                       (csrc/hc_proj.cu), 128 tokens per CTA
//   rest           gen_tail_kernel      r, split + Sinkhorn, y = bf16(sum_j pre_mix_j X'_j), RMSNorm
//   tail           gen_final_kernel     [hc_post], collapse, final RMSNorm
// The weights come from the bf16 planes of hc_prepare_params: w = hi + (mid + lo) is exact in fp32.
// Arithmetic orders match the fused kernel where it has one (X', y); sums run in fp32.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "hc_internal.h"
#include "hc_ptx.cuh"

namespace hc {
namespace {

constexpr int kGMaxHc = 8;
constexpr int kGMaxMix = (2 + kGMaxHc) * kGMaxHc;  // 80

__device__ __forceinline__ float gbf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float gbf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t gpack(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ void gunpack(const uint4& v, float (&f)[8]) {
    f[0] = gbf_lo(v.x); f[1] = gbf_hi(v.x); f[2] = gbf_lo(v.y); f[3] = gbf_hi(v.y);
    f[4] = gbf_lo(v.z); f[5] = gbf_hi(v.z); f[6] = gbf_lo(v.w); f[7] = gbf_hi(v.w);
}
__device__ __forceinline__ uint4 gpack8(const float (&o)[8]) {
    return make_uint4(gpack(o[0], o[1]), gpack(o[2], o[3]), gpack(o[4], o[5]), gpack(o[6], o[7]));
}
__device__ __forceinline__ float bf16f(const uint16_t* p, long long i) { return __uint_as_float(static_cast<uint32_t>(p[i]) << 16); }

// ---- writing half ------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gen_post_kernel(const uint4* __restrict__ X, const uint4* __restrict__ delta,
                                                       const float* __restrict__ post, const float* __restrict__ comb,
                                                       uint4* __restrict__ X_out, uint4* __restrict__ mean_out,
                                                       long long n, int hc, int dv) {
    const long long total = n * dv;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const float inv_hc = 1.0f / static_cast<float>(hc);
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const long long t = idx / dv, i = idx - (idx / dv) * dv;
        float dl[8], x[kGMaxHc][8];
        gunpack(__ldcs(delta + t * dv + i), dl);
#pragma unroll
        for (int j = 0; j < kGMaxHc; ++j)
            if (j < hc) gunpack(__ldcs(X + (t * hc + j) * dv + i), x[j]);
        float ms[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < kGMaxHc; ++k) {
            if (k >= hc) break;
            const float pk = __ldg(post + t * hc + k);
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = pk * dl[e];
#pragma unroll
            for (int j = 0; j < kGMaxHc; ++j) {
                if (j < hc) {
                    const float c = __ldg(comb + (t * hc + j) * hc + k);
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = fmaf(c, x[j][e], o[e]);
                }
            }
            const uint4 ov = gpack8(o);
            __stcs(X_out + (t * hc + k) * dv + i, ov);
            if (mean_out) {
                float r[8];
                gunpack(ov, r);
#pragma unroll
                for (int e = 0; e < 8; ++e) ms[e] += r[e];
            }
        }
        if (mean_out) {
#pragma unroll
            for (int e = 0; e < 8; ++e) ms[e] = hc == 4 ? ms[e] * 0.25f : ms[e] * inv_hc;
            __stcs(mean_out + t * dv + i, gpack8(ms));
        }
    }
}

// ---- head of the stack: the embedding in every stream --------------------------------------------
__global__ void __launch_bounds__(256) gen_expand_kernel(const uint4* __restrict__ h, uint4* __restrict__ X_out,
                                                         long long n, int hc, int dv) {
    const long long total = n * dv;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const long long t = idx / dv, i = idx - (idx / dv) * dv;
        const uint4 v = __ldcs(h + t * dv + i);
        for (int j = 0; j < hc; ++j) __stcs(X_out + (t * hc + j) * dv + i, v);
    }
}

// ---- split + Sinkhorn for any hc <= 8 ("Reading weights" page, hc_split_sinkhorn kernel) ----------
__device__ void gen_split_sinkhorn(int hc, const float* m, const float* sc, const float* b, int iters, float eps,
                                   float* pre, float* post, float* C) {
    for (int j = 0; j < hc; ++j) pre[j] = 1.0f / (1.0f + expf(-(m[j] * sc[0] + b[j]))) + eps;
    for (int j = 0; j < hc; ++j) post[j] = 2.0f * (1.0f / (1.0f + expf(-(m[hc + j] * sc[1] + b[hc + j]))));
    for (int q = 0; q < hc * hc; ++q) C[q] = m[2 * hc + q] * sc[2] + b[2 * hc + q];
    for (int j = 0; j < hc; ++j) {
        float mx = C[j * hc];
        for (int k = 1; k < hc; ++k) mx = fmaxf(mx, C[j * hc + k]);
        float s = 0.f;
        for (int k = 0; k < hc; ++k) {
            C[j * hc + k] = expf(C[j * hc + k] - mx);
            s += C[j * hc + k];
        }
        const float inv = rcp_refined(s);
        for (int k = 0; k < hc; ++k) C[j * hc + k] = C[j * hc + k] * inv + eps;
    }
    for (int it = 0; it < iters; ++it) {
        if (it > 0) {
            for (int j = 0; j < hc; ++j) {
                float s = 0.f;
                for (int k = 0; k < hc; ++k) s += C[j * hc + k];
                const float inv = rcp_refined(s + eps);
                for (int k = 0; k < hc; ++k) C[j * hc + k] *= inv;
            }
        }
        for (int k = 0; k < hc; ++k) {
            float s = 0.f;
            for (int j = 0; j < hc; ++j) s += C[j * hc + k];
            const float inv = rcp_refined(s + eps);
            for (int j = 0; j < hc; ++j) C[j * hc + k] *= inv;
        }
    }
}

// ---- rest of the reading half, one CTA per token ----------------------------------------------------
constexpr int kTThreads = 256;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float s = 0.f;
    for (int i = 0; i < kTThreads / 32; ++i) s += red[i];  // fixed order: deterministic
    return s;
}

// y = bf16(sum_j pm_j X_j) at column i of token row Xt (hc streams of width d)
__device__ __forceinline__ float collapse(const uint16_t* Xt, const float* pm, int hc, int d, int i) {
    float s = pm[0] * bf16f(Xt, i);
    for (int j = 1; j < hc; ++j) s = fmaf(pm[j], bf16f(Xt, static_cast<long long>(j) * d + i), s);
    return __bfloat162float(__float2bfloat16_rn(s));
}

__global__ void __launch_bounds__(kTThreads) gen_tail_kernel(const uint16_t* __restrict__ X,
                                                             const float* __restrict__ pre_mix, int identity,
                                                             const float* __restrict__ hc_scale,
                                                             const float* __restrict__ hc_base,
                                                             const float* __restrict__ norm_w,
                                                             const float* __restrict__ raw, const float* __restrict__ ssx,
                                                             int hc, int d, int iters, float hc_eps, float norm_eps,
                                                             uint16_t* __restrict__ y_normed, float* __restrict__ pre,
                                                             float* __restrict__ post, float* __restrict__ comb,
                                                             float* __restrict__ mixes_out) {
    __shared__ float red[kTThreads / 32];
    __shared__ float pm[kGMaxHc];
    const long long t = blockIdx.x;
    const int M = (2 + hc) * hc;
    const uint16_t* Xt = X + t * hc * static_cast<long long>(d);
    if (threadIdx.x < hc)
        pm[threadIdx.x] = identity ? 1.0f / static_cast<float>(hc) : pre_mix ? pre_mix[t * hc + threadIdx.x] : 0.f;
    if (threadIdx.x == 0) {
        // coefficients: r over all hc*d values, mixes = raw * r, then the split
        float m[kGMaxMix], sc[3], bs[kGMaxMix];
        const float r = 1.0f / sqrtf(ssx[t] / static_cast<float>(hc * d) + norm_eps);
        for (int i = 0; i < M; ++i) m[i] = raw[t * M + i] * r;
        if (mixes_out) {
            for (int i = 0; i < M; ++i) mixes_out[t * M + i] = m[i];
        } else {
            for (int i = 0; i < 3; ++i) sc[i] = hc_scale[i];
            for (int i = 0; i < M; ++i) bs[i] = hc_base[i];
            float pr[kGMaxHc], po[kGMaxHc], C[kGMaxHc * kGMaxHc];
            gen_split_sinkhorn(hc, m, sc, bs, iters, hc_eps, pr, po, C);
            for (int j = 0; j < hc; ++j) {
                pre[t * hc + j] = pr[j];
                post[t * hc + j] = po[j];
            }
            for (int q = 0; q < hc * hc; ++q) comb[t * hc * hc + q] = C[q];
        }
    }
    __syncthreads();
    if (!y_normed) return;
    float sy = 0.f;
    for (int i = threadIdx.x; i < d; i += kTThreads) {
        const float y = collapse(Xt, pm, hc, d, i);
        sy = fmaf(y, y, sy);
    }
    const float ry = 1.0f / sqrtf(block_sum(sy, red) / static_cast<float>(d) + norm_eps);
    for (int i = threadIdx.x; i < d; i += kTThreads) {
        const float y = collapse(Xt, pm, hc, d, i);
        y_normed[t * d + i] = __bfloat16_as_ushort(__float2bfloat16_rn(norm_w[i] * (y * ry)));
    }
}

// ---- tail of the stack: [hc_post], collapse, final RMSNorm, one CTA per token -------------------------
__global__ void __launch_bounds__(kTThreads) gen_final_kernel(const uint16_t* __restrict__ X,
                                                              const uint16_t* __restrict__ delta,
                                                              const float* __restrict__ post,
                                                              const float* __restrict__ comb,
                                                              const float* __restrict__ pre_mix,
                                                              const float* __restrict__ norm_w,
                                                              uint16_t* __restrict__ X_out, uint16_t* __restrict__ z,
                                                              int hc, int d, float eps) {
    __shared__ float red[kTThreads / 32];
    __shared__ float cf[kGMaxHc + kGMaxHc * kGMaxHc + kGMaxHc];  // post, comb, pre_mix
    const long long t = blockIdx.x;
    const long long D = static_cast<long long>(hc) * d;
    if (threadIdx.x < hc) {
        cf[threadIdx.x] = delta ? post[t * hc + threadIdx.x] : 0.f;
        cf[kGMaxHc + kGMaxHc * kGMaxHc + threadIdx.x] = pre_mix[t * hc + threadIdx.x];
    }
    if (delta && threadIdx.x < hc * hc) cf[kGMaxHc + threadIdx.x] = comb[t * hc * hc + threadIdx.x];
    __syncthreads();
    const float* pm = cf + kGMaxHc + kGMaxHc * kGMaxHc;
    auto y_at = [&](int i, bool write_x) -> float {
        float xp[kGMaxHc];
        for (int k = 0; k < hc; ++k) {
            if (delta) {
                float o = cf[k] * bf16f(delta, t * d + i);
                for (int j = 0; j < hc; ++j) o = fmaf(cf[kGMaxHc + j * hc + k], bf16f(X, t * D + j * static_cast<long long>(d) + i), o);
                const __nv_bfloat16 ob = __float2bfloat16_rn(o);
                if (write_x) X_out[t * D + k * static_cast<long long>(d) + i] = __bfloat16_as_ushort(ob);
                xp[k] = __bfloat162float(ob);
            } else {
                xp[k] = bf16f(X, t * D + k * static_cast<long long>(d) + i);
            }
        }
        float s = pm[0] * xp[0];
        for (int j = 1; j < hc; ++j) s = fmaf(pm[j], xp[j], s);
        return __bfloat162float(__float2bfloat16_rn(s));
    };
    float sy = 0.f;
    for (int i = threadIdx.x; i < d; i += kTThreads) {
        const float y = y_at(i, X_out != nullptr);
        sy = fmaf(y, y, sy);
    }
    const float ry = 1.0f / sqrtf(block_sum(sy, red) / static_cast<float>(d) + eps);
    for (int i = threadIdx.x; i < d; i += kTThreads) {
        const float y = y_at(i, false);
        z[t * d + i] = __bfloat16_as_ushort(__float2bfloat16_rn(norm_w[i] * (y * ry)));
    }
}

int grid_of(long long work, int per_block) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long blocks = (work + per_block - 1) / per_block;
    const long long cap = static_cast<long long>(sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

int status_of(cudaError_t e) { return e == cudaSuccess ? 0 : -7; }

}  // namespace

size_t generic_tokens_per_chunk(int hc) {
    const size_t M = static_cast<size_t>(2 + hc) * hc;
    return workspace_bytes() / ((M + 1) * sizeof(float));
}

int launch_generic_post(const void* X, const void* delta, const float* post, const float* comb, void* X_out,
                        void* mean_out, int64_t n, int hc, int d, cudaStream_t stream) {
    if (n <= 0) return 0;
    const int dv = d / 8;
    gen_post_kernel<<<grid_of(n * dv, 256), 256, 0, stream>>>(
        static_cast<const uint4*>(X), static_cast<const uint4*>(delta), post, comb, static_cast<uint4*>(X_out),
        static_cast<uint4*>(mean_out), n, hc, dv);
    return status_of(cudaGetLastError());
}

int launch_generic_expand(const void* h, void* X_out, int64_t n, int hc, int d, cudaStream_t stream) {
    if (n <= 0) return 0;
    const int dv = d / 8;
    gen_expand_kernel<<<grid_of(n * dv, 256), 256, 0, stream>>>(static_cast<const uint4*>(h),
                                                                  static_cast<uint4*>(X_out), n, hc, dv);
    return status_of(cudaGetLastError());
}

int launch_generic_reading(const GenericArgs& a, cudaStream_t stream) {
    const int M = (2 + a.hc) * a.hc;
    const int64_t chunk = static_cast<int64_t>(generic_tokens_per_chunk(a.hc));
    float* raw = static_cast<float*>(a.workspace);
    float* ssx = raw + static_cast<size_t>(chunk) * M;
    const size_t D = static_cast<size_t>(a.hc) * a.d;
    for (int64_t t0 = 0; t0 < a.n; t0 += chunk) {
        const int64_t m = a.n - t0 < chunk ? a.n - t0 : chunk;
        const uint16_t* Xc = static_cast<const uint16_t*>(a.X) + t0 * D;
        const int st = launch_proj_tc(Xc, a.planes, m, a.hc, a.d, raw, ssx, stream);
        if (st != 0) return st;
        gen_tail_kernel<<<static_cast<unsigned>(m), kTThreads, 0, stream>>>(
            Xc, a.pre_mix ? a.pre_mix + t0 * a.hc : nullptr, a.identity, a.hc_scale, a.hc_base, a.norm_w, raw, ssx,
            a.hc, a.d, a.iters, a.hc_eps, a.norm_eps,
            a.y_normed ? static_cast<uint16_t*>(a.y_normed) + t0 * a.d : nullptr,
            a.pre_out ? a.pre_out + t0 * a.hc : nullptr, a.post_out ? a.post_out + t0 * a.hc : nullptr,
            a.comb_out ? a.comb_out + t0 * a.hc * a.hc : nullptr, a.mixes_out ? a.mixes_out + t0 * M : nullptr);
        if (cudaGetLastError() != cudaSuccess) return -7;
    }
    return 0;
}

int launch_generic_final(const void* X, const void* delta, const float* post, const float* comb,
                         const float* pre_mix, const float* norm_w, void* X_out, void* z, int64_t n, int hc, int d,
                         float eps, cudaStream_t stream) {
    if (n <= 0) return 0;
    gen_final_kernel<<<static_cast<unsigned>(n), kTThreads, 0, stream>>>(
        static_cast<const uint16_t*>(X), static_cast<const uint16_t*>(delta), post, comb, pre_mix, norm_w,
        static_cast<uint16_t*>(X_out), static_cast<uint16_t*>(z), hc, d, eps);
    return status_of(cudaGetLastError());
}

}  // namespace hc
