// Host-buffer executor of libhc.so (declared in include/hc.h): runs hc_post_then_pre on per-token
// arrays that live in host memory. The tokens go through in chunks; each chunk's inputs are copied
// in on one stream, the fused step runs on the caller's stream, and the chunk's results are copied
// out on a second stream, so the copies of neighbouring chunks in both directions and the kernels
// overlap. On a GB300 the host link, not the GPU, bounds such a call: about 210 GB/s host to
// device and 190 GB/s back with the copy engines, about 170 GB/s each way when both run at once
// (copies driven by SM loads and stores from mapped memory measured the same), against a fused
// step that moves the same bytes through HBM some 30 times faster.
//
// Ordering, per staging buffer b (kDepth of them, chunk i uses b = i mod kDepth):
//   copy-in stream:  wait in_free[b] (the kernel of chunk i - kDepth has read its inputs),
//                    copy the inputs of chunk i, record in_ready[b]
//   caller's stream: wait in_ready[b] and out_free[b] (chunk i - kDepth's results are out),
//                    hc_post_then_pre on the staging buffer, record in_free[b]
//   copy-out stream: wait in_free[b], copy the results of chunk i out, record out_free[b]
// Every copy has a fixed cost on the link, about 20 us per chunk once both directions are busy,
// which the coefficient arrays (16 to 256 bytes a token) would pay for a few kilobytes each. When
// hc is a multiple of 4 (every chunk's rows of them then start 16-byte aligned), they move once per
// segment of consecutive chunks instead (up to max(chunk, 65536) tokens): post, comb and pre_mix
// in before the segment's first chunk, pre, post and comb out after its last, through two segment
// buffers used in turn (events seg_in_free / seg_out_free, as for the chunk buffers).
// A call starts after the caller's earlier work on its stream and after the previous call on the
// same executor (its `done` event), and the caller's stream waits for the last copy-out, so the
// call is ordered on `stream` like every other entry point.

#include <cuda_runtime.h>

#include <cstdint>
#include <new>

#include "../../include/hc.h"

namespace {

constexpr int kDepth = 3;                  // staging buffers in flight
constexpr int64_t kDefaultChunk = 1024;    // tokens per chunk when the caller passes 0 (measured best)
constexpr int64_t kMaxChunk = 1 << 20;
constexpr int64_t kMinSegment = 65536;     // tokens per segment of coefficient copies (at least a chunk)
constexpr int kMaxHc = 8;
constexpr int kMaxD = 65536;

size_t round_up(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// byte sizes of the per-token arrays of m tokens
struct Bytes {
    size_t x, y, c, k;  // streams [m, hc, d] bf16; rows [m, d] bf16; [m, hc] fp32; [m, hc, hc] fp32
    Bytes(int64_t m, int hc, int d) {
        const size_t M = static_cast<size_t>(m), H = static_cast<size_t>(hc), D = static_cast<size_t>(d);
        x = M * H * D * 2;
        y = M * D * 2;
        c = M * H * 4;
        k = M * H * H * 4;
    }
};

// offsets of the ten arrays inside one staging buffer of `chunk` tokens
struct Layout {
    size_t delta, X, post, comb, pre_mix, X_out, y, pre_o, post_o, comb_o, total;
    Layout(int64_t chunk, int hc, int d) {
        const Bytes b(chunk, hc, d);
        size_t o = 0;
        auto take = [&](size_t n) {
            const size_t at = o;
            o += round_up(n);
            return at;
        };
        delta = take(b.y);
        X = take(b.x);
        post = take(b.c);
        comb = take(b.k);
        pre_mix = take(b.c);
        X_out = take(b.x);
        y = take(b.y);
        pre_o = take(b.c);
        post_o = take(b.c);
        comb_o = take(b.k);
        total = o;
    }
};

// The chunks of one call, in order. Between ramps of halving size at both ends (C/2, C/4, ...,
// down to the last size of at least max(128, C/32) tokens) run chunks of C (the last of them
// shorter), so that the first copy-in and the last copy-out, which nothing overlaps, are short
// while most of the tokens go in a few large copies (each copy costs a fixed time on the link).
// A call too small for both ramps and one full chunk, or an executor with chunks under 256 tokens,
// is cut into equal chunks instead: at most C tokens each, and up to 8 of them when they keep 32
// tokens or more.
struct ChunkPlan {
    static constexpr int kMaxRamp = 5;
    int64_t n, C, count;
    int64_t ramp[kMaxRamp];  // ramp[j] = C >> (j + 1): the head runs ramp[nramp-1] ... ramp[0]
    int nramp;
    int64_t head;                   // tokens in one ramp
    int64_t mid, mid_chunks;        // tokens and chunks between the ramps
    int64_t eq_base, eq_rem;        // equal split: eq_base tokens, one more in the first eq_rem chunks
    ChunkPlan(int64_t n_, int64_t C_)
        : n(n_), C(C_), count(0), ramp{}, nramp(0), head(0), mid(0), mid_chunks(0), eq_base(0), eq_rem(0) {
        if (n <= 0) return;
        const int64_t floor_size = C / 32 > 128 ? C / 32 : 128;
        int levels = 0;
        for (int j = 0; j < kMaxRamp && (C >> (j + 1)) >= floor_size; ++j) levels = j + 1;
        int64_t h = 0;
        for (int j = 0; j < levels; ++j) h += C >> (j + 1);
        if (levels > 0 && n >= 2 * h + C) {
            nramp = levels;
            for (int j = 0; j < levels; ++j) ramp[j] = C >> (j + 1);
            head = h;
            mid = n - 2 * h;
            mid_chunks = (mid + C - 1) / C;
            count = 2 * nramp + mid_chunks;
        } else {
            int64_t k = (n + C - 1) / C;
            const int64_t eight = n / 32 < 8 ? n / 32 : 8;
            if (k < eight) k = eight;
            if (k < 1) k = 1;
            count = k;
            eq_base = n / k;
            eq_rem = n % k;
        }
    }
    // first token and size of chunk i (0 <= i < count)
    void chunk(int64_t i, int64_t* t0, int64_t* m) const {
        if (nramp == 0) {
            *t0 = i * eq_base + (i < eq_rem ? i : eq_rem);
            *m = eq_base + (i < eq_rem ? 1 : 0);
            return;
        }
        if (i < nramp) {  // rising: ramp[nramp-1], ..., ramp[0]; before chunk i lie the smaller ones
            const int j = nramp - 1 - static_cast<int>(i);
            int64_t before = 0;
            for (int q = j + 1; q < nramp; ++q) before += ramp[q];
            *t0 = before;
            *m = ramp[j];
        } else if (i < nramp + mid_chunks) {
            const int64_t k = i - nramp;
            *t0 = head + k * C;
            *m = k + 1 < mid_chunks ? C : mid - k * C;
        } else {  // falling: ramp[0], ..., ramp[nramp-1]
            const int j = static_cast<int>(i - nramp - mid_chunks);
            int64_t before = 0;
            for (int q = 0; q < j; ++q) before += ramp[q];
            *t0 = head + mid + before;
            *m = ramp[j];
        }
    }
};

// offsets of the six coefficient arrays inside one segment buffer of `tokens` tokens
struct SegLayout {
    size_t post, comb, pre_mix, pre_o, post_o, comb_o, total;
    SegLayout(int64_t tokens, int hc) {
        const Bytes b(tokens, hc, 8);
        size_t o = 0;
        auto take = [&](size_t n) {
            const size_t at = o;
            o += round_up(n);
            return at;
        };
        post = take(b.c);
        comb = take(b.k);
        pre_mix = take(b.c);
        pre_o = take(b.c);
        post_o = take(b.c);
        comb_o = take(b.k);
        total = o;
    }
};

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na && nb && x < y + nb && y < x + na;
}

}  // namespace

struct hc_host_pipeline {
    int hc = 0, d = 0, device = 0;
    int64_t chunk = 0;
    size_t buffer_bytes = 0;
    char* staging = nullptr;   // kDepth buffers of buffer_bytes
    int64_t seg_tokens = 0;    // tokens per segment buffer (0: coefficients move with each chunk)
    size_t seg_bytes = 0;
    char* seg = nullptr;       // 2 segment buffers of seg_bytes: post, comb, pre_mix in; pre, post, comb out
    cudaEvent_t seg_in_free[2] = {}, seg_out_free[2] = {};
    void* workspace = nullptr; // hc_workspace_size bytes, zeroed at creation
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t entry = nullptr, done = nullptr;
    cudaEvent_t in_ready[kDepth] = {}, in_free[kDepth] = {}, out_free[kDepth] = {};
};

namespace {

void release(hc_host_pipeline* p) {
    if (p->staging) cudaFree(p->staging);
    if (p->seg) cudaFree(p->seg);
    for (int b = 0; b < 2; ++b) {
        if (p->seg_in_free[b]) cudaEventDestroy(p->seg_in_free[b]);
        if (p->seg_out_free[b]) cudaEventDestroy(p->seg_out_free[b]);
    }
    if (p->workspace) cudaFree(p->workspace);
    if (p->s_in) cudaStreamDestroy(p->s_in);
    if (p->s_out) cudaStreamDestroy(p->s_out);
    if (p->entry) cudaEventDestroy(p->entry);
    if (p->done) cudaEventDestroy(p->done);
    for (int b = 0; b < kDepth; ++b) {
        if (p->in_ready[b]) cudaEventDestroy(p->in_ready[b]);
        if (p->in_free[b]) cudaEventDestroy(p->in_free[b]);
        if (p->out_free[b]) cudaEventDestroy(p->out_free[b]);
    }
    delete p;
}

}  // namespace

extern "C" {

int hc_host_pipeline_create(int hc, int d, int64_t chunk_tokens, hc_host_pipeline_t** out) {
    if (!out) return HC_ERR_NULL;
    *out = nullptr;
    if (hc < 1 || d < 1 || d % 8 != 0 || chunk_tokens < 0) return HC_ERR_SHAPE;
    if (hc > kMaxHc || d > kMaxD) return HC_ERR_UNSUPPORTED;
    const int64_t chunk = chunk_tokens == 0 ? kDefaultChunk : chunk_tokens;
    if (chunk > kMaxChunk) return HC_ERR_SHAPE;
    hc_host_pipeline* p = new (std::nothrow) hc_host_pipeline;
    if (!p) return HC_ERR_CUDA;
    p->hc = hc;
    p->d = d;
    p->chunk = chunk;
    p->buffer_bytes = Layout(chunk, hc, d).total;
    if (hc % 4 == 0) {
        p->seg_tokens = chunk > kMinSegment ? chunk : kMinSegment;
        p->seg_bytes = SegLayout(p->seg_tokens, hc).total;
    }
    size_t ws = 0;
    hc_workspace_size(&ws);
    bool ok = cudaGetDevice(&p->device) == cudaSuccess &&
              cudaMalloc(reinterpret_cast<void**>(&p->staging), kDepth * p->buffer_bytes) == cudaSuccess &&
              (p->seg_tokens == 0 || cudaMalloc(reinterpret_cast<void**>(&p->seg), 2 * p->seg_bytes) == cudaSuccess) &&
              cudaMalloc(&p->workspace, ws) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p->entry, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&p->done, cudaEventDisableTiming) == cudaSuccess &&
              cudaMemsetAsync(p->workspace, 0, ws, p->s_in) == cudaSuccess;
    for (int b = 0; ok && b < kDepth; ++b)
        ok = cudaEventCreateWithFlags(&p->in_ready[b], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->in_free[b], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->out_free[b], cudaEventDisableTiming) == cudaSuccess;
    for (int b = 0; ok && b < 2; ++b)
        ok = cudaEventCreateWithFlags(&p->seg_in_free[b], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->seg_out_free[b], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventRecord(p->seg_in_free[b], p->s_in) == cudaSuccess &&
             cudaEventRecord(p->seg_out_free[b], p->s_in) == cudaSuccess;
    // every event starts recorded (on the idle copy-in stream), so the first waits pass at once
    for (int b = 0; ok && b < kDepth; ++b)
        ok = cudaEventRecord(p->in_ready[b], p->s_in) == cudaSuccess &&
             cudaEventRecord(p->in_free[b], p->s_in) == cudaSuccess &&
             cudaEventRecord(p->out_free[b], p->s_in) == cudaSuccess;
    ok = ok && cudaEventRecord(p->entry, p->s_in) == cudaSuccess &&
         cudaEventRecord(p->done, p->s_in) == cudaSuccess && cudaStreamSynchronize(p->s_in) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        release(p);
        return HC_ERR_CUDA;
    }
    *out = p;
    return HC_OK;
}

int hc_host_pipeline_destroy(hc_host_pipeline_t* p) {
    if (!p) return HC_OK;
    int st = HC_OK;
    if (cudaEventSynchronize(p->done) != cudaSuccess) st = HC_ERR_CUDA;
    release(p);
    return st;
}

int hc_host_pipeline_chunk_tokens(const hc_host_pipeline_t* p, int64_t* chunk_tokens) {
    if (!p || !chunk_tokens) return HC_ERR_NULL;
    *chunk_tokens = p->chunk;
    return HC_OK;
}

int hc_host_chunk_plan(int64_t n, int64_t chunk_tokens, int64_t index, int64_t* count, int64_t* t0,
                       int64_t* tokens) {
    if (!count) return HC_ERR_NULL;
    if (n < 0 || chunk_tokens < 0) return HC_ERR_SHAPE;
    const int64_t C = chunk_tokens == 0 ? kDefaultChunk : chunk_tokens;
    if (C > kMaxChunk) return HC_ERR_SHAPE;
    const ChunkPlan plan(n, C);
    *count = plan.count;
    if (index < 0) return HC_OK;
    if (!t0 || !tokens) return HC_ERR_NULL;
    if (index >= plan.count) return HC_ERR_ARG;
    plan.chunk(index, t0, tokens);
    return HC_OK;
}

int hc_host_post_then_pre(hc_host_pipeline_t* p, const void* delta, const void* X, const float* post,
                          const float* comb, const float* pre_mix, hc_params_t next, int64_t n, hc_shape_t s,
                          void* X_out, void* y_normed, float* pre_out, float* post_out, float* comb_out,
                          hc_stream_t stream) {
    if (!p || !delta || !X || !post || !comb || !pre_mix || !X_out || !y_normed || !pre_out || !post_out ||
        !comb_out)
        return HC_ERR_NULL;
    if (!next.hc_fn_planes || !next.hc_scale || !next.hc_base || !next.norm_w) return HC_ERR_NULL;
    if (n < 0 || s.hc != p->hc || s.d != p->d) return HC_ERR_SHAPE;
    if (s.sinkhorn_iters < 1 || !(s.hc_eps >= 0.f && s.hc_eps <= 3.4e38f) ||
        !(s.norm_eps >= 0.f && s.norm_eps <= 3.4e38f))
        return HC_ERR_ARG;
    // host arrays: no output may overlap an input or another output
    const Bytes z(n, s.hc, s.d);
    const void* ins[5] = {delta, X, post, comb, pre_mix};
    const size_t isz[5] = {z.y, z.x, z.c, z.k, z.c};
    const void* outs[5] = {X_out, y_normed, pre_out, post_out, comb_out};
    const size_t osz[5] = {z.x, z.y, z.c, z.c, z.k};
    for (int i = 0; i < 5; ++i) {
        for (int j = 0; j < 5; ++j)
            if (overlap(outs[i], osz[i], ins[j], isz[j])) return HC_ERR_ALIAS;
        for (int j = i + 1; j < 5; ++j)
            if (overlap(outs[i], osz[i], outs[j], osz[j])) return HC_ERR_ALIAS;
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return HC_ERR_CUDA;
    if (dev != p->device) return HC_ERR_ARG;
    if (n == 0) return HC_OK;

    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const Layout L(p->chunk, s.hc, s.d);
    auto in_host = [](const void* base, size_t row_bytes, int64_t t0) {
        return static_cast<const char*>(base) + static_cast<size_t>(t0) * row_bytes;
    };
    auto out_host = [](void* base, size_t row_bytes, int64_t t0) {
        return static_cast<char*>(base) + static_cast<size_t>(t0) * row_bytes;
    };
    const Bytes one(1, s.hc, s.d);  // bytes per token of each array
    bool ok = cudaStreamWaitEvent(cs, p->done, 0) == cudaSuccess &&
              cudaEventRecord(p->entry, cs) == cudaSuccess &&
              cudaStreamWaitEvent(p->s_in, p->entry, 0) == cudaSuccess &&
              cudaStreamWaitEvent(p->s_out, p->entry, 0) == cudaSuccess;
    int st = ok ? HC_OK : HC_ERR_CUDA;
    const ChunkPlan plan(n, p->chunk);
    const bool segmented = p->seg_tokens > 0;
    const SegLayout SL(segmented ? p->seg_tokens : 0, s.hc);
    int64_t seg_t0 = 0, seg_end = 0;  // token range of the current segment
    int64_t g = -1;                   // segment number
    char* sbuf = nullptr;             // its buffer
    auto h2d = [&](void* dst, const void* src, size_t bytes) {
        return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, p->s_in) == cudaSuccess;
    };
    auto d2h = [&](void* dst, const void* src, size_t bytes) {
        return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, p->s_out) == cudaSuccess;
    };
    for (int64_t i = 0; st == HC_OK && i < plan.count; ++i) {
        const int b = static_cast<int>(i % kDepth);
        int64_t t0 = 0, m = 0;
        plan.chunk(i, &t0, &m);
        const Bytes c(m, s.hc, s.d);
        char* buf = p->staging + static_cast<size_t>(b) * p->buffer_bytes;
        ok = true;
        if (segmented && t0 >= seg_end) {
            // a segment starts with this chunk: the whole chunks from here that fit in a segment buffer
            ++g;
            const int sb = static_cast<int>(g & 1);
            sbuf = p->seg + static_cast<size_t>(sb) * p->seg_bytes;
            seg_t0 = t0;
            seg_end = t0;
            for (int64_t j = i; j < plan.count; ++j) {
                int64_t a = 0, k = 0;
                plan.chunk(j, &a, &k);
                if (a + k - seg_t0 > p->seg_tokens) break;
                seg_end = a + k;
            }
            const Bytes sg(seg_end - seg_t0, s.hc, s.d);
            // its coefficients in, once segment g - 2's kernels have read that buffer; its kernels
            // write their coefficients there only after segment g - 2's have been copied out
            ok = cudaStreamWaitEvent(p->s_in, p->seg_in_free[sb], 0) == cudaSuccess &&
                 h2d(sbuf + SL.post, in_host(post, one.c, seg_t0), sg.c) &&
                 h2d(sbuf + SL.comb, in_host(comb, one.k, seg_t0), sg.k) &&
                 h2d(sbuf + SL.pre_mix, in_host(pre_mix, one.c, seg_t0), sg.c) &&
                 cudaStreamWaitEvent(cs, p->seg_out_free[sb], 0) == cudaSuccess;
        }
        // the chunk's coefficient arrays: in the segment buffer, or in the chunk buffer
        const size_t so = static_cast<size_t>(t0 - seg_t0);
        char* c_post = segmented ? sbuf + SL.post + so * one.c : buf + L.post;
        char* c_comb = segmented ? sbuf + SL.comb + so * one.k : buf + L.comb;
        char* c_pre_mix = segmented ? sbuf + SL.pre_mix + so * one.c : buf + L.pre_mix;
        char* c_pre_o = segmented ? sbuf + SL.pre_o + so * one.c : buf + L.pre_o;
        char* c_post_o = segmented ? sbuf + SL.post_o + so * one.c : buf + L.post_o;
        char* c_comb_o = segmented ? sbuf + SL.comb_o + so * one.k : buf + L.comb_o;
        // inputs in
        ok = ok && cudaStreamWaitEvent(p->s_in, p->in_free[b], 0) == cudaSuccess &&
             h2d(buf + L.delta, in_host(delta, one.y, t0), c.y) && h2d(buf + L.X, in_host(X, one.x, t0), c.x) &&
             (segmented || (h2d(c_post, in_host(post, one.c, t0), c.c) && h2d(c_comb, in_host(comb, one.k, t0), c.k) &&
                            h2d(c_pre_mix, in_host(pre_mix, one.c, t0), c.c))) &&
             cudaEventRecord(p->in_ready[b], p->s_in) == cudaSuccess;
        // the step on the chunk
        ok = ok && cudaStreamWaitEvent(cs, p->in_ready[b], 0) == cudaSuccess &&
             cudaStreamWaitEvent(cs, p->out_free[b], 0) == cudaSuccess;
        if (!ok) {
            st = HC_ERR_CUDA;
            break;
        }
        st = hc_post_then_pre(buf + L.delta, buf + L.X, reinterpret_cast<const float*>(c_post),
                              reinterpret_cast<const float*>(c_comb), reinterpret_cast<const float*>(c_pre_mix), next,
                              m, s, buf + L.X_out, buf + L.y, reinterpret_cast<float*>(c_pre_o),
                              reinterpret_cast<float*>(c_post_o), reinterpret_cast<float*>(c_comb_o), p->workspace,
                              stream);
        if (st != HC_OK) break;
        const bool seg_last = segmented && t0 + m == seg_end;
        // results out
        ok = cudaEventRecord(p->in_free[b], cs) == cudaSuccess &&
             (!seg_last || cudaEventRecord(p->seg_in_free[g & 1], cs) == cudaSuccess) &&
             cudaStreamWaitEvent(p->s_out, p->in_free[b], 0) == cudaSuccess &&
             d2h(out_host(X_out, one.x, t0), buf + L.X_out, c.x) && d2h(out_host(y_normed, one.y, t0), buf + L.y, c.y) &&
             (segmented || (d2h(out_host(pre_out, one.c, t0), c_pre_o, c.c) &&
                            d2h(out_host(post_out, one.c, t0), c_post_o, c.c) &&
                            d2h(out_host(comb_out, one.k, t0), c_comb_o, c.k))) &&
             cudaEventRecord(p->out_free[b], p->s_out) == cudaSuccess;
        if (ok && seg_last) {
            // the segment's last kernel has run (the caller's stream is in order): its coefficients out
            const Bytes sg(seg_end - seg_t0, s.hc, s.d);
            ok = d2h(out_host(pre_out, one.c, seg_t0), sbuf + SL.pre_o, sg.c) &&
                 d2h(out_host(post_out, one.c, seg_t0), sbuf + SL.post_o, sg.c) &&
                 d2h(out_host(comb_out, one.k, seg_t0), sbuf + SL.comb_o, sg.k) &&
                 cudaEventRecord(p->seg_out_free[g & 1], p->s_out) == cudaSuccess;
        }
        if (!ok) st = HC_ERR_CUDA;
    }
    // the caller's stream continues once every result is in host memory; the next call on this
    // executor starts after that point too (also after a failure part-way, for what was enqueued)
    const bool closed = cudaEventRecord(p->done, p->s_out) == cudaSuccess &&
                        cudaStreamWaitEvent(cs, p->done, 0) == cudaSuccess;
    if (st == HC_OK && !closed) st = HC_ERR_CUDA;
    return st;
}

}  // extern "C"
