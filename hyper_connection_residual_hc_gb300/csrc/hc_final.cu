// Tail of the Hyper-Connection stack for GB300 (sm_103a): after the last block the streams are
// collapsed once more with the last pre_mix and pass through the final RMSNorm ("Final RMSNorm"
// page, Transformer.forward excerpt, RMSNorm excerpt and the m_2 formula), optionally after the
// last sublayer's writing half ("Write the streams" page, formula for X'):
//   [post] X'_k = bf16(post_k * Delta + sum_j comb[j,k] * X_j)     (written to X_out if given)
//   y = bf16(sum_j pre_mix_j * X'_j)
//   z = bf16(norm_w * (y * r)),  r = 1/sqrt(mean(y^2) + eps)        (eps 1e-20 on the page)
//
// Streaming and HBM-bound: per token it reads 4*d bf16 stream values (+ d of Delta) and writes d
// values of z. One CTA of 128 threads per token; thread i holds the 8-column groups i, i + 128,
// ... (at most 5 for d <= 5120) of y in registers between the two passes the norm needs (sum of
// y^2, then scale). All loads of a thread are issued before any arithmetic, so each CTA has its
// whole token (up to 51 KB) in flight.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "hc_internal.h"

namespace hc {
namespace {

constexpr int kFinalThreads = 128;
constexpr int kFinalVec = kFinalMaxD / 8 / kFinalThreads;  // 8-column groups per thread (5)
static_assert(kFinalVec * 8 * kFinalThreads == kFinalMaxD, "d <= 5120 is covered by 128 threads x 5 groups");

__device__ __forceinline__ float flo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float fhi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);  // a -> low half
    return *reinterpret_cast<uint32_t*>(&v);
}
// 8 bf16 columns as column pairs: f[m] = columns 2m, 2m + 1
__device__ __forceinline__ void unpack(const uint4& v, float2 (&f)[4]) {
    f[0] = make_float2(flo(v.x), fhi(v.x)); f[1] = make_float2(flo(v.y), fhi(v.y));
    f[2] = make_float2(flo(v.z), fhi(v.z)); f[3] = make_float2(flo(v.w), fhi(v.w));
}
__device__ __forceinline__ uint4 pack8(const float2 (&o)[4]) {
    return make_uint4(pack2(o[0].x, o[0].y), pack2(o[1].x, o[1].y), pack2(o[2].x, o[2].y), pack2(o[3].x, o[3].y));
}
__device__ __forceinline__ float2 bcast2(float a) { return make_float2(a, a); }

// X' without its store is held to 128 registers (4 blocks per SM): left free it took 130 and 3 blocks
template <bool kPost, bool kStoreX>
__global__ void __launch_bounds__(kFinalThreads, (kPost && !kStoreX) ? 4 : 0) hc_final_kernel(
    const uint4* __restrict__ X, const uint4* __restrict__ delta, const float4* __restrict__ post,
    const float4* __restrict__ comb, const float4* __restrict__ pre_mix, const float* __restrict__ norm_w,
    uint4* __restrict__ X_out, uint4* __restrict__ z, int dv, float inv_d, float eps) {
    __shared__ float red[kFinalThreads / 32];
    const long long t = blockIdx.x;
    const int tid = threadIdx.x;

    // issue every load of this thread first
    uint4 xs[kFinalVec][4], ds[kFinalVec];
#pragma unroll
    for (int v = 0; v < kFinalVec; ++v) {
        const int i = tid + v * kFinalThreads;
        if (i < dv) {
#pragma unroll
            for (int j = 0; j < 4; ++j) xs[v][j] = __ldcs(X + (t * 4 + j) * dv + i);
            if (kPost) ds[v] = __ldcs(delta + t * dv + i);
        }
    }
    const float4 pmv = __ldg(pre_mix + t);
    const float pm[4] = {pmv.x, pmv.y, pmv.z, pmv.w};
    float pv[4] = {0.f, 0.f, 0.f, 0.f}, c[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) c[q] = 0.f;
    if (kPost) {
        const float4 p4 = __ldg(post + t);
        pv[0] = p4.x; pv[1] = p4.y; pv[2] = p4.z; pv[3] = p4.w;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 cv = __ldg(comb + t * 4 + j);
            c[4 * j] = cv.x; c[4 * j + 1] = cv.y; c[4 * j + 2] = cv.z; c[4 * j + 3] = cv.w;
        }
    }

    // pass 1: X' (post), y rounded to bf16, sum of y^2. Column pairs go through the packed fp32
    // instructions (two IEEE operations each, rounded per lane as the scalar ones), in the order
    // of the formulas above.
    uint32_t yb[kFinalVec][4];
    float ss = 0.f;
#pragma unroll
    for (int v = 0; v < kFinalVec; ++v) {
        const int i = tid + v * kFinalThreads;
        if (i < dv) {
            float2 x[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) unpack(xs[v][j], x[j]);
            if (kPost) {
                float2 dl[4];
                unpack(ds[v], dl);
                float2 xp[4][4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float2 o[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        float2 s = __fmul2_rn(bcast2(pv[k]), dl[m]);
                        s = __ffma2_rn(bcast2(c[0 * 4 + k]), x[0][m], s);
                        s = __ffma2_rn(bcast2(c[1 * 4 + k]), x[1][m], s);
                        s = __ffma2_rn(bcast2(c[2 * 4 + k]), x[2][m], s);
                        s = __ffma2_rn(bcast2(c[3 * 4 + k]), x[3][m], s);
                        o[m] = s;
                    }
                    const uint4 ov = pack8(o);
                    if (kStoreX) __stcs(X_out + (t * 4 + k) * dv + i, ov);
                    unpack(ov, xp[k]);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int m = 0; m < 4; ++m) x[k][m] = xp[k][m];
            }
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                float2 s = __fmul2_rn(bcast2(pm[0]), x[0][m]);
                s = __ffma2_rn(bcast2(pm[1]), x[1][m], s);
                s = __ffma2_rn(bcast2(pm[2]), x[2][m], s);
                s = __ffma2_rn(bcast2(pm[3]), x[3][m], s);
                const uint32_t u = pack2(s.x, s.y);
                yb[v][m] = u;
                const float a0 = flo(u), a1 = fhi(u);
                ss = fmaf(a0, a0, ss);
                ss = fmaf(a1, a1, ss);
            }
        }
    }

    // block sum of y^2 in a fixed order (deterministic)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    const float total = (red[0] + red[1]) + (red[2] + red[3]);
    const float r = 1.0f / sqrtf(total * inv_d + eps);

    // pass 2: z = bf16(norm_w * (y * r))
#pragma unroll
    for (int v = 0; v < kFinalVec; ++v) {
        const int i = tid + v * kFinalThreads;
        if (i < dv) {
            const float4 w0 = __ldg(reinterpret_cast<const float4*>(norm_w) + 2 * i);
            const float4 w1 = __ldg(reinterpret_cast<const float4*>(norm_w) + 2 * i + 1);
            const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            float2 o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                o[e] = __fmul2_rn(make_float2(w[2 * e], w[2 * e + 1]),
                                  __fmul2_rn(make_float2(flo(yb[v][e]), fhi(yb[v][e])), bcast2(r)));
            __stcs(z + t * dv + i, pack8(o));
        }
    }
}

}  // namespace

int launch_final(const FinalArgs& a, cudaStream_t stream) {
    if (a.n <= 0) return 0;
    const int dv = a.d / 8;
    const dim3 grid(static_cast<unsigned>(a.n)), block(kFinalThreads);
    const float inv_d = 1.0f / static_cast<float>(a.d);
    const uint4* X = static_cast<const uint4*>(a.X);
    const uint4* D = static_cast<const uint4*>(a.delta);
    const float4* P = reinterpret_cast<const float4*>(a.post);
    const float4* C = reinterpret_cast<const float4*>(a.comb);
    const float4* M = reinterpret_cast<const float4*>(a.pre_mix);
    uint4* Xo = static_cast<uint4*>(a.X_out);
    uint4* Z = static_cast<uint4*>(a.z);
    if (!a.delta)
        hc_final_kernel<false, false><<<grid, block, 0, stream>>>(X, D, P, C, M, a.norm_w, Xo, Z, dv, inv_d,
                                                                  a.norm_eps);
    else if (!a.X_out)
        hc_final_kernel<true, false><<<grid, block, 0, stream>>>(X, D, P, C, M, a.norm_w, Xo, Z, dv, inv_d,
                                                                 a.norm_eps);
    else
        hc_final_kernel<true, true><<<grid, block, 0, stream>>>(X, D, P, C, M, a.norm_w, Xo, Z, dv, inv_d,
                                                                a.norm_eps);
    return cudaGetLastError() == cudaSuccess ? 0 : -7;
}

}  // namespace hc
