// C ABI of libhc.so (declared in include/hc.h): host-side argument validation, the two
// elementwise kernels (standalone writing half, weight splitting) and dispatch to the fused
// reading-half kernel (hc_fused.cu) and the tail-of-stack kernel (hc_final.cu).

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "../../include/hc.h"
#include "hc_internal.h"

namespace hc {
namespace {

constexpr int kHC = 4;         // the fused kernel's number of streams
constexpr int kMaxHc = 8;      // the generic path's limits
constexpr int kMaxD = 65536;

// ---- writing half: X' = bf16(post_k * delta + sum_j comb[j,k] X_j) ---------------------------
// "Write the streams" page, formula for X'_{n,k}; "Source layer, pairs pooled" page, Block.hc_post
// excerpt. One thread per (token, 8 columns); all four streams of those columns, so X_out may be X.

__device__ __forceinline__ float lo16(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float hi16(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pk(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(256, 3) hc_post_kernel(const uint4* __restrict__ X, const uint4* __restrict__ delta,
                                                      const float4* __restrict__ post, const float4* __restrict__ comb,
                                                      uint4* X_out, long long n, int dv) {
    const long long total = n * dv;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const long long t = idx / dv;
        const long long i = idx - t * dv;
        const float4 pst = __ldg(post + t);
        float c[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 v = __ldg(comb + t * 4 + j);
            c[4 * j] = v.x; c[4 * j + 1] = v.y; c[4 * j + 2] = v.z; c[4 * j + 3] = v.w;
        }
        const float pv[4] = {pst.x, pst.y, pst.z, pst.w};
        float x[4][8], dl[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 v = __ldcs(X + (t * 4 + j) * dv + i);
            x[j][0] = lo16(v.x); x[j][1] = hi16(v.x); x[j][2] = lo16(v.y); x[j][3] = hi16(v.y);
            x[j][4] = lo16(v.z); x[j][5] = hi16(v.z); x[j][6] = lo16(v.w); x[j][7] = hi16(v.w);
        }
        {
            const uint4 v = __ldcs(delta + t * dv + i);
            dl[0] = lo16(v.x); dl[1] = hi16(v.x); dl[2] = lo16(v.y); dl[3] = hi16(v.y);
            dl[4] = lo16(v.z); dl[5] = hi16(v.z); dl[6] = lo16(v.w); dl[7] = hi16(v.w);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float s = pv[k] * dl[e];
                s = fmaf(c[0 * 4 + k], x[0][e], s);
                s = fmaf(c[1 * 4 + k], x[1][e], s);
                s = fmaf(c[2 * 4 + k], x[2][e], s);
                s = fmaf(c[3 * 4 + k], x[3][e], s);
                o[e] = s;
            }
            __stcs(X_out + (t * 4 + k) * dv + i, make_uint4(pk(o[0], o[1]), pk(o[2], o[3]), pk(o[4], o[5]), pk(o[6], o[7])));
        }
    }
}

// ---- weight split: hc_fn = hi + mid + lo, three bf16 planes ----------------------------------
// Plane rows follow plane_row(): grouped for the fused kernel's accumulator drain at hc = 4 (row
// 36*h + 12*p + i holds plane p (0 hi, 1 mid, 2 lo) of mix 12*h + i), plane-major otherwise.
__global__ void __launch_bounds__(256) hc_prepare_kernel(const float* __restrict__ fn, __nv_bfloat16* planes,
                                                         int hc, long long D) {
    const int M = (2 + hc) * hc;
    const long long total = static_cast<long long>(M) * D;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const long long m = idx / D;
        const long long c = idx - m * D;
        const float w = fn[idx];
        const __nv_bfloat16 hi = __float2bfloat16_rn(w);
        const float r1 = w - __bfloat162float(hi);  // exact (Sterbenz)
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);  // exact; at most 8 significant bits remain
        const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
        const int mm = static_cast<int>(m);
        planes[plane_row(hc, M, 0, mm) * D + c] = hi;
        planes[plane_row(hc, M, 1, mm) * D + c] = mid;
        planes[plane_row(hc, M, 2, mm) * D + c] = lo;
    }
}

int grid_for(long long work, int per_block) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long blocks = (work + per_block - 1) / per_block;
    const long long cap = static_cast<long long>(sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

// Blocks of hc_post_kernel resident at once on the current device (SMs x blocks per SM), found once
// per device: its grid-stride loop then runs as a single wave (at 3 blocks per SM, the earlier cap of
// 8 blocks per SM left a partial last wave)
int post_grid(long long work) {
    static std::atomic<int> resident[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return grid_for(work, 256);
    int r = resident[dev].load(std::memory_order_relaxed);
    if (r == 0) {
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, hc_post_kernel, 256, 0) != cudaSuccess ||
            sms < 1 || per_sm < 1)
            return grid_for(work, 256);
        r = sms * per_sm;
        resident[dev].store(r, std::memory_order_relaxed);
    }
    const long long blocks = (work + 255) / 256;
    return static_cast<int>(blocks < r ? (blocks < 1 ? 1 : blocks) : r);
}

// ---- validation ---------------------------------------------------------------------------------

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na && nb && x < y + nb && y < x + na;
}

// Shape rules of every call: hc in 1..8 and d a positive multiple of 8 up to 65536 (the fused
// kernel takes hc = 4 with d a multiple of 256 up to 5120, the generic kernels the rest).
int check_shape(int64_t n, const hc_shape_t& s, bool reading) {
    if (n < 0 || n > 0x7FFFFFFFLL) return HC_ERR_SHAPE;
    if (s.hc < 1 || s.d < 1 || s.d % 8 != 0) return HC_ERR_SHAPE;
    if (s.hc > kMaxHc || s.d > kMaxD) return HC_ERR_UNSUPPORTED;
    if (reading && s.sinkhorn_iters < 1) return HC_ERR_ARG;
    if (reading && (!std::isfinite(s.hc_eps) || s.hc_eps < 0.f)) return HC_ERR_ARG;
    if (!std::isfinite(s.norm_eps) || s.norm_eps < 0.f) return HC_ERR_ARG;
    return HC_OK;
}

bool fused_shape(const hc_shape_t& s) { return s.hc == kHC && s.d % 256 == 0 && s.d <= 5120; }

// byte sizes of the per-token arrays of n tokens
struct Sizes {
    size_t x, y, c, k;  // streams [n, hc, d] bf16, rows [n, d] bf16, [n, hc] fp32, [n, hc, hc] fp32
    Sizes(int64_t n, const hc_shape_t& s) {
        const size_t N = static_cast<size_t>(n), H = static_cast<size_t>(s.hc), D = static_cast<size_t>(s.d);
        x = N * H * D * 2;
        y = N * D * 2;
        c = N * H * 4;
        k = N * H * H * 4;
    }
};

// true if any output overlaps an input or another output (null entries are skipped)
bool any_overlap(const void* const* outs, const size_t* osz, int no, const void* const* ins, const size_t* isz,
                 int ni) {
    for (int i = 0; i < no; ++i) {
        if (!outs[i]) continue;
        for (int j = 0; j < ni; ++j)
            if (ins[j] && overlap(outs[i], osz[i], ins[j], isz[j])) return true;
        for (int j = i + 1; j < no; ++j)
            if (outs[j] && overlap(outs[i], osz[i], outs[j], osz[j])) return true;
    }
    return false;
}

int check_params(const hc_params_t& p) {
    if (!p.hc_fn_planes || !p.hc_scale || !p.hc_base || !p.norm_w) return HC_ERR_NULL;
    if (!aligned16(p.hc_fn_planes) || !aligned16(p.hc_scale) || !aligned16(p.hc_base) || !aligned16(p.norm_w))
        return HC_ERR_ALIGN;
    return HC_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? HC_OK : HC_ERR_CUDA; }

int launch_status(int internal) { return internal == 0 ? HC_OK : internal == -3 ? HC_ERR_UNSUPPORTED : HC_ERR_CUDA; }

}  // namespace
}  // namespace hc

using namespace hc;

// the reading half of one sublayer on streams X (hc_pre_step; the second half of the post calls)
static int reading_half(const void* X, const float* pre_mix, bool identity, const hc_params_t& p, int64_t n,
                        const hc_shape_t& s, void* y_normed, float* pre, float* post, float* comb, float* mixes,
                        void* workspace, cudaStream_t stream) {
    GenericArgs g = {};
    g.X = X;
    g.pre_mix = pre_mix;
    g.identity = identity ? 1 : 0;
    g.planes = p.hc_fn_planes;
    g.hc_scale = p.hc_scale;
    g.hc_base = p.hc_base;
    g.norm_w = p.norm_w;
    g.y_normed = y_normed;
    g.pre_out = pre;
    g.post_out = post;
    g.comb_out = comb;
    g.mixes_out = mixes;
    g.workspace = workspace;
    g.n = n;
    g.hc = s.hc;
    g.d = s.d;
    g.iters = s.sinkhorn_iters;
    g.hc_eps = s.hc_eps;
    g.norm_eps = s.norm_eps;
    return launch_generic_reading(g, stream);
}

static int post_then_pre_impl(const void* delta, const void* X, const float* post, const float* comb,
                              const float* pre_mix, hc_params_t next, int64_t n, hc_shape_t s, void* X_out,
                              void* y_normed, float* pre_out, float* post_out, float* comb_out, void* stream_mean,
                              void* workspace, bool noalloc, hc_stream_t stream) {
    if (!delta || !X || !post || !comb || !pre_mix || !X_out || !y_normed || !pre_out || !post_out || !comb_out ||
        (!workspace && !noalloc))
        return HC_ERR_NULL;
    int st = check_params(next);
    if (st != HC_OK) return st;
    st = check_shape(n, s, true);
    if (st != HC_OK) return st;
    const void* ptrs[10] = {delta, X, post, comb, pre_mix, X_out, y_normed, pre_out, post_out, comb_out};
    for (const void* q : ptrs)
        if (!aligned16(q)) return HC_ERR_ALIGN;
    if ((workspace && !aligned16(workspace)) || (stream_mean && !aligned16(stream_mean))) return HC_ERR_ALIGN;
    const Sizes z(n, s);
    const void* ins[5] = {delta, X, post, comb, pre_mix};
    const size_t isz[5] = {z.y, z.x, z.c, z.k, z.c};
    const void* outs[7] = {X_out, y_normed, pre_out, post_out, comb_out, workspace, stream_mean};
    const size_t osz[7] = {z.x, z.y, z.c, z.c, z.k, workspace_bytes(), z.y};
    if (any_overlap(outs, osz, 7, ins, isz, 5)) return HC_ERR_ALIAS;
    if (n == 0) return HC_OK;
    if (noalloc) {
        // the scratch is the library's fixed array: find this device's copy (first call only); it is
        // as large as any launch needs (a compile-time check beside the array)
        size_t capacity = 0;
        if (noalloc_workspace(&workspace, &capacity) != 0) return HC_ERR_CUDA;
    }
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (!fused_shape(s)) {
        st = launch_generic_post(X, delta, post, comb, X_out, stream_mean, n, s.hc, s.d, cs);
        if (st != 0) return launch_status(st);
        return launch_status(reading_half(X_out, pre_mix, false, next, n, s, y_normed, pre_out, post_out, comb_out,
                                          nullptr, workspace, cs));
    }
    FusedArgs a = {};
    a.mode = kModePost;
    a.X = X;
    a.delta = delta;
    a.post = post;
    a.comb = comb;
    a.pre_mix = pre_mix;
    a.planes = next.hc_fn_planes;
    a.hc_scale = next.hc_scale;
    a.hc_base = next.hc_base;
    a.norm_w = next.norm_w;
    a.X_out = X_out;
    a.y_normed = y_normed;
    a.pre_out = pre_out;
    a.post_out = post_out;
    a.comb_out = comb_out;
    a.stream_mean = stream_mean;
    a.workspace = workspace;
    a.n = n;
    a.d = s.d;
    a.iters = s.sinkhorn_iters;
    a.hc_eps = s.hc_eps;
    a.norm_eps = s.norm_eps;
    return launch_status(launch_fused(a, cs));
}

extern "C" {

const char* hc_status_string(int status) {
    switch (status) {
        case HC_OK: return "ok";
        case HC_ERR_NULL: return "a required pointer is NULL";
        case HC_ERR_SHAPE: return "invalid shape (n < 0, or hc < 1, or d not a positive multiple of 8)";
        case HC_ERR_UNSUPPORTED: return "configuration not implemented (hc > 8, d > 65536, or no cooperative launch)";
        case HC_ERR_ALIGN: return "a device pointer is not 16-byte aligned";
        case HC_ERR_ALIAS: return "an output overlaps an input or another output";
        case HC_ERR_ARG: return "invalid scalar argument (sinkhorn_iters < 1, or an eps negative or not finite)";
        case HC_ERR_CUDA: return "a CUDA call or kernel launch failed";
        case HC_ERR_DEVICE: return "a kernel gave up a bounded wait";
        default: return "unknown status";
    }
}

int hc_prepare_params_size(int hc, int d, size_t* bytes) {
    if (!bytes) return HC_ERR_NULL;
    if (hc < 1 || d < 1) return HC_ERR_SHAPE;
    *bytes = static_cast<size_t>(3) * static_cast<size_t>((2 + hc) * hc) * static_cast<size_t>(hc) *
             static_cast<size_t>(d) * 2u;
    return HC_OK;
}

int hc_prepare_params(const float* hc_fn, int hc, int d, void* planes, hc_stream_t stream) {
    if (!hc_fn || !planes) return HC_ERR_NULL;
    if (hc < 1 || d < 1 || d % 8 != 0) return HC_ERR_SHAPE;
    if (hc > kMaxHc || d > kMaxD) return HC_ERR_UNSUPPORTED;
    if (!aligned16(hc_fn) || !aligned16(planes)) return HC_ERR_ALIGN;
    const long long D = static_cast<long long>(hc) * d;
    const long long M = static_cast<long long>(2 + hc) * hc;
    if (overlap(hc_fn, static_cast<size_t>(M * D) * 4, planes, static_cast<size_t>(3 * M * D) * 2))
        return HC_ERR_ALIAS;
    const long long work = M * D;
    hc_prepare_kernel<<<grid_for(work, 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        hc_fn, static_cast<__nv_bfloat16*>(planes), hc, D);
    return cuda_status(cudaGetLastError());
}

int hc_post(const void* delta, const void* X, const float* post, const float* comb, int64_t n, hc_shape_t s,
            void* X_out, hc_stream_t stream) {
    if (!delta || !X || !post || !comb || !X_out) return HC_ERR_NULL;
    if (n < 0 || s.hc < 1 || s.d < 1 || s.d % 8 != 0 || n > (1LL << 40)) return HC_ERR_SHAPE;
    if (s.hc > kMaxHc || s.d > kMaxD) return HC_ERR_UNSUPPORTED;
    if (!aligned16(delta) || !aligned16(X) || !aligned16(post) || !aligned16(comb) || !aligned16(X_out))
        return HC_ERR_ALIGN;
    const Sizes z(n, s);
    if ((X_out != X && overlap(X_out, z.x, X, z.x)) || overlap(X_out, z.x, delta, z.y) ||
        overlap(X_out, z.x, post, z.c) || overlap(X_out, z.x, comb, z.k))
        return HC_ERR_ALIAS;
    if (n == 0) return HC_OK;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (s.hc != kHC) return launch_status(launch_generic_post(X, delta, post, comb, X_out, nullptr, n, s.hc, s.d, cs));
    const int dv = s.d / 8;
    hc_post_kernel<<<post_grid(n * dv), 256, 0, cs>>>(
        static_cast<const uint4*>(X), static_cast<const uint4*>(delta), reinterpret_cast<const float4*>(post),
        reinterpret_cast<const float4*>(comb), static_cast<uint4*>(X_out), n, dv);
    return cuda_status(cudaGetLastError());
}

int hc_workspace_size(size_t* bytes) {
    if (!bytes) return HC_ERR_NULL;
    *bytes = workspace_bytes();
    return HC_OK;
}

int hc_pre_step(const void* X, const float* pre_mix, hc_params_t p, int64_t n, hc_shape_t s, void* y_normed,
                float* pre, float* post, float* comb, void* workspace, hc_stream_t stream) {
    if (!X || !pre_mix || !y_normed || !pre || !post || !comb || !workspace) return HC_ERR_NULL;
    int st = check_params(p);
    if (st != HC_OK) return st;
    st = check_shape(n, s, true);
    if (st != HC_OK) return st;
    if (!aligned16(X) || !aligned16(pre_mix) || !aligned16(y_normed) || !aligned16(pre) || !aligned16(post) ||
        !aligned16(comb) || !aligned16(workspace))
        return HC_ERR_ALIGN;
    const Sizes z(n, s);
    const void* outs[5] = {y_normed, pre, post, comb, workspace};
    const size_t osz[5] = {z.y, z.c, z.c, z.k, workspace_bytes()};
    const void* ins[2] = {X, pre_mix};
    const size_t isz[2] = {z.x, z.c};
    if (any_overlap(outs, osz, 5, ins, isz, 2)) return HC_ERR_ALIAS;
    if (n == 0) return HC_OK;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (!fused_shape(s))
        return launch_status(reading_half(X, pre_mix, false, p, n, s, y_normed, pre, post, comb, nullptr, workspace, cs));
    FusedArgs a = {};
    a.mode = kModePre;
    a.X = X;
    a.pre_mix = pre_mix;
    a.planes = p.hc_fn_planes;
    a.hc_scale = p.hc_scale;
    a.hc_base = p.hc_base;
    a.norm_w = p.norm_w;
    a.y_normed = y_normed;
    a.pre_out = pre;
    a.post_out = post;
    a.comb_out = comb;
    a.workspace = workspace;
    a.n = n;
    a.d = s.d;
    a.iters = s.sinkhorn_iters;
    a.hc_eps = s.hc_eps;
    a.norm_eps = s.norm_eps;
    return launch_status(launch_fused(a, cs));
}

int hc_post_then_pre(const void* delta, const void* X, const float* post, const float* comb, const float* pre_mix,
                     hc_params_t next, int64_t n, hc_shape_t s, void* X_out, void* y_normed, float* pre_out,
                     float* post_out, float* comb_out, void* workspace, hc_stream_t stream) {
    return post_then_pre_impl(delta, X, post, comb, pre_mix, next, n, s, X_out, y_normed, pre_out, post_out,
                              comb_out, nullptr, workspace, false, stream);
}

int hc_post_then_pre_tap(const void* delta, const void* X, const float* post, const float* comb,
                         const float* pre_mix, hc_params_t next, int64_t n, hc_shape_t s, void* X_out,
                         void* y_normed, float* pre_out, float* post_out, float* comb_out, void* stream_mean,
                         void* workspace, hc_stream_t stream) {
    if (!stream_mean) return HC_ERR_NULL;
    return post_then_pre_impl(delta, X, post, comb, pre_mix, next, n, s, X_out, y_normed, pre_out, post_out,
                              comb_out, stream_mean, workspace, false, stream);
}

int hc_post_then_pre_noalloc(const void* delta, const void* X, const float* post, const float* comb,
                             const float* pre_mix, hc_params_t next, int64_t n, hc_shape_t s, void* X_out,
                             void* y_normed, float* pre_out, float* post_out, float* comb_out, hc_stream_t stream) {
    return post_then_pre_impl(delta, X, post, comb, pre_mix, next, n, s, X_out, y_normed, pre_out, post_out,
                              comb_out, nullptr, nullptr, true, stream);
}

int hc_expand_pre_step(const void* h, hc_params_t p, int64_t n, hc_shape_t s, void* X_out, void* y_normed, float* pre,
                       float* post, float* comb, void* workspace, hc_stream_t stream) {
    if (!h || !X_out || !y_normed || !pre || !post || !comb || !workspace) return HC_ERR_NULL;
    int st = check_params(p);
    if (st != HC_OK) return st;
    st = check_shape(n, s, true);
    if (st != HC_OK) return st;
    const void* ptrs[7] = {h, X_out, y_normed, pre, post, comb, workspace};
    for (const void* q : ptrs)
        if (!aligned16(q)) return HC_ERR_ALIGN;
    const Sizes z(n, s);
    const void* ins[1] = {h};
    const size_t isz[1] = {z.y};
    const void* outs[6] = {X_out, y_normed, pre, post, comb, workspace};
    const size_t osz[6] = {z.x, z.y, z.c, z.c, z.k, workspace_bytes()};
    if (any_overlap(outs, osz, 6, ins, isz, 1)) return HC_ERR_ALIAS;
    if (n == 0) return HC_OK;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (!fused_shape(s)) {
        st = launch_generic_expand(h, X_out, n, s.hc, s.d, cs);
        if (st != 0) return launch_status(st);
        return launch_status(reading_half(X_out, nullptr, true, p, n, s, y_normed, pre, post, comb, nullptr,
                                          workspace, cs));
    }
    FusedArgs a = {};
    a.mode = kModeExpand;
    a.embed = h;
    a.planes = p.hc_fn_planes;
    a.hc_scale = p.hc_scale;
    a.hc_base = p.hc_base;
    a.norm_w = p.norm_w;
    a.X_out = X_out;
    a.y_normed = y_normed;
    a.pre_out = pre;
    a.post_out = post;
    a.comb_out = comb;
    a.workspace = workspace;
    a.n = n;
    a.d = s.d;
    a.iters = s.sinkhorn_iters;
    a.hc_eps = s.hc_eps;
    a.norm_eps = s.norm_eps;
    return launch_status(launch_fused(a, cs));
}

// the tail of the stack: the 4-stream kernel for hc = 4 and d <= 5120, the generic one otherwise
static int final_impl(const void* delta, const void* X, const float* post, const float* comb, const float* pre_mix,
                      const float* norm_w, int64_t n, const hc_shape_t& s, void* X_out, void* z, cudaStream_t cs) {
    if (s.hc != kHC || s.d > kFinalMaxD)
        return launch_status(launch_generic_final(X, delta, post, comb, pre_mix, norm_w, X_out, z, n, s.hc, s.d,
                                                  s.norm_eps, cs));
    FinalArgs a = {};
    a.X = X;
    a.delta = delta;
    a.post = post;
    a.comb = comb;
    a.pre_mix = pre_mix;
    a.norm_w = norm_w;
    a.X_out = X_out;
    a.z = z;
    a.n = n;
    a.d = s.d;
    a.norm_eps = s.norm_eps;
    return launch_status(launch_final(a, cs));
}

int hc_final(const void* X, const float* pre_mix, const float* norm_w, int64_t n, hc_shape_t s, void* z,
             hc_stream_t stream) {
    if (!X || !pre_mix || !norm_w || !z) return HC_ERR_NULL;
    int st = check_shape(n, s, false);
    if (st != HC_OK) return st;
    if (!aligned16(X) || !aligned16(pre_mix) || !aligned16(norm_w) || !aligned16(z)) return HC_ERR_ALIGN;
    const Sizes q(n, s);
    const void* ins[3] = {X, pre_mix, norm_w};
    const size_t isz[3] = {q.x, q.c, static_cast<size_t>(s.d) * 4};
    const void* outs[1] = {z};
    const size_t osz[1] = {q.y};
    if (any_overlap(outs, osz, 1, ins, isz, 3)) return HC_ERR_ALIAS;
    if (n == 0) return HC_OK;
    return final_impl(nullptr, X, nullptr, nullptr, pre_mix, norm_w, n, s, nullptr, z,
                      reinterpret_cast<cudaStream_t>(stream));
}

int hc_post_then_final(const void* delta, const void* X, const float* post, const float* comb, const float* pre_mix,
                       const float* norm_w, int64_t n, hc_shape_t s, void* X_out, void* z, hc_stream_t stream) {
    if (!delta || !X || !post || !comb || !pre_mix || !norm_w || !z) return HC_ERR_NULL;
    int st = check_shape(n, s, false);
    if (st != HC_OK) return st;
    const void* ptrs[7] = {delta, X, post, comb, pre_mix, norm_w, z};
    for (const void* q : ptrs)
        if (!aligned16(q)) return HC_ERR_ALIGN;
    if (X_out && !aligned16(X_out)) return HC_ERR_ALIGN;
    const Sizes q(n, s);
    const void* ins[6] = {delta, X, post, comb, pre_mix, norm_w};
    const size_t isz[6] = {q.y, q.x, q.c, q.k, q.c, static_cast<size_t>(s.d) * 4};
    const void* outs[2] = {z, X_out};
    const size_t osz[2] = {q.y, q.x};
    if (any_overlap(outs, osz, 2, ins, isz, 6)) return HC_ERR_ALIAS;
    if (n == 0) return HC_OK;
    return final_impl(delta, X, post, comb, pre_mix, norm_w, n, s, X_out, z, reinterpret_cast<cudaStream_t>(stream));
}

int hc_debug_mixes(const void* X, hc_params_t p, int64_t n, hc_shape_t s, int group, float* mixes, void* workspace,
                   hc_stream_t stream) {
    if (!X || !mixes || !p.hc_fn_planes || !workspace) return HC_ERR_NULL;
    hc_shape_t s2 = s;
    if (s2.sinkhorn_iters < 1) s2.sinkhorn_iters = 1;
    int st = check_shape(n, s2, true);
    if (st != HC_OK) return st;
    if (group != 0 && group != 8 && group != 16 && group != 32) return HC_ERR_ARG;
    if (fused_shape(s2) && group != 0 && s2.d % (32 * group) != 0) return HC_ERR_ARG;
    if (!aligned16(X) || !aligned16(mixes) || !aligned16(p.hc_fn_planes) || !aligned16(workspace))
        return HC_ERR_ALIGN;
    const Sizes z(n, s);
    const size_t mb = static_cast<size_t>(n) * (2 + s.hc) * s.hc * 4;
    if (overlap(mixes, mb, X, z.x) || overlap(workspace, workspace_bytes(), X, z.x) ||
        overlap(workspace, workspace_bytes(), mixes, mb))
        return HC_ERR_ALIAS;
    if (n == 0) return HC_OK;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (!fused_shape(s2))
        return launch_status(reading_half(X, nullptr, false, p, n, s2, nullptr, nullptr, nullptr, nullptr, mixes,
                                          workspace, cs));
    // the kernel reads scale/base/norm_w unconditionally: point them at the planes (never used)
    FusedArgs a = {};
    a.mode = kModePre;
    a.X = X;
    a.planes = p.hc_fn_planes;
    a.hc_scale = static_cast<const float*>(p.hc_fn_planes);
    a.hc_base = static_cast<const float*>(p.hc_fn_planes);
    a.norm_w = static_cast<const float*>(p.hc_fn_planes);
    a.mixes_out = mixes;
    a.workspace = workspace;
    a.n = n;
    a.d = s2.d;
    a.iters = s2.sinkhorn_iters;
    a.hc_eps = s2.hc_eps;
    a.norm_eps = s2.norm_eps;
    a.group = group;
    return launch_status(launch_fused(a, cs));
}

int hc_plan_tiles(int64_t n, int d, int ctas, int* group, int* tile_m, int64_t* num_tiles) {
    if (!group || !tile_m || !num_tiles) return HC_ERR_NULL;
    if (n < 0 || d < 1 || d % 256 != 0 || ctas < 8) return HC_ERR_SHAPE;
    plan_tiles(n, d, ctas, 0, group, tile_m, num_tiles);
    return HC_OK;
}

int hc_fused_ctas(int* ctas) {
    if (!ctas) return HC_ERR_NULL;
    return launch_status(fused_ctas(ctas));
}

int hc_debug_wait_flag(const unsigned long long* flags, int count, unsigned long long value, int64_t limit_ns,
                       hc_stream_t stream) {
    if (!flags) return HC_ERR_NULL;
    if (count < 1 || count > 32) return HC_ERR_SHAPE;
    if (limit_ns < 0 || limit_ns > 1000000000LL) return HC_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(flags) & 7u) return HC_ERR_ALIGN;
    return launch_status(launch_wait_flag(flags, value, count, static_cast<uint64_t>(limit_ns),
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int hc_device_error(unsigned int* word, int clear, hc_stream_t stream) {
    if (!word) return HC_ERR_NULL;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    unsigned int fused = 0, proj = 0;
    if (read_device_error(&fused, clear, cs) != 0 || read_proj_error(&proj, clear, cs) != 0) return HC_ERR_CUDA;
    *word = fused | proj;
    return HC_OK;
}

}  // extern "C"
