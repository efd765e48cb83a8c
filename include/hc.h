/*
 * hc.h -- C ABI of the GB300 (sm_103a) Hyper-Connection stream-step library (libhc.so).
 *
 * The Hyper-Connection residual keeps hc parallel copies ("streams") of the hidden state.
 * Around every sublayer the model (DeepSeek V4.1 model-atlas pages) does, per token:
 *   writing half  ("Write the streams" page, formula for X'_{n,k}; "Source layer, pairs pooled"
 *                  page, Block.hc_post excerpt):
 *       X'_k = post_k * Delta + sum_j comb[j,k] * X_j            (fp32 math, cast to bf16)
 *   reading half  (same page, Block.hc_mixes and Block.hc_pre excerpts; "Reading weights" page,
 *                  hc_split_sinkhorn kernel excerpt and the formula for p; "Final RMSNorm" page,
 *                  RMSNorm excerpt):
 *       r      = 1 / sqrt(mean over all hc*d values of X'^2 + norm_eps)
 *       mixes  = r * (X'_flat . hc_fn^T)                      24 numbers at hc = 4
 *       pre    = sigmoid(s0*mixes[0:hc] + base) + hc_eps
 *       post   = 2*sigmoid(s1*mixes[hc:2hc] + base)
 *       comb   = Sinkhorn(softmax_rows(s2*mixes[2hc:] + base) + hc_eps), sinkhorn_iters rounds
 *       y      = bf16(sum_j pre_mix_j * X'_j)                 pre_mix = the INCOMING reading mix
 *       y_normed = bf16(norm_w * y / sqrt(mean(y^2) + norm_eps))
 * Block.forward ("Source layer, pairs pooled" page) hands the (pre, post, comb) computed by one
 * sublayer to the next: the returned pre is the next call's pre_mix, post/comb are the next
 * call's post/comb.
 *
 * Conventions for every entry point
 *   - Pointers marked [device] are CUDA device pointers in the current device's context; the
 *     caller allocates and owns every buffer. The library never allocates or frees device memory
 *     and never synchronises the stream, except hc_device_error and the host-buffer executor
 *     (hc_host_pipeline_*, which owns its staging memory; documented there).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *   - All arrays are contiguous row-major; tokens are flattened, n = batch * positions.
 *   - bf16 is IEEE bfloat16 (16-bit storage); fp32 is IEEE binary32.
 *   - Layouts: X, X_out [n, hc, d] bf16; delta, y_normed [n, d] bf16; pre_mix, pre, post [n, hc]
 *     fp32; comb [n, hc, hc] fp32 with comb[t, j, k]: j = source stream (summed over in the
 *     writing half), k = destination stream. mixes order: [pre hc | post hc | comb hc*hc, row j
 *     then column k].
 *   - Every device pointer must be 16-byte aligned (HC_ERR_ALIGN otherwise).
 *   - n == 0 is a no-op that returns HC_OK. n < 0 returns HC_ERR_SHAPE.
 *   - Arguments are validated on the host before anything is launched; a failed check returns a
 *     negative status and leaves every output untouched. No exception crosses the ABI.
 *   - Floating-point specials (NaN, Inf) in the data propagate; they are never trapped.
 */
#ifndef HC_GB300_H
#define HC_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* hc_stream_t; /* identical to cudaStream_t */

/* Status codes. */
enum {
    HC_OK = 0,
    HC_ERR_NULL = -1,        /* a required pointer is NULL */
    HC_ERR_SHAPE = -2,       /* n < 0, or hc < 1, or d not a positive multiple of 8 */
    HC_ERR_UNSUPPORTED = -3, /* a valid configuration not implemented (hc > 8, d > 65536, no cooperative launch) */
    HC_ERR_ALIGN = -4,       /* a device pointer is not 16-byte aligned */
    HC_ERR_ALIAS = -5,       /* an output overlaps an input or another output (see each call) */
    HC_ERR_ARG = -6,         /* sinkhorn_iters < 1, or an eps negative or not finite */
    HC_ERR_CUDA = -7,        /* a CUDA runtime/driver call or kernel launch failed */
    HC_ERR_DEVICE = -8       /* a kernel gave up a bounded wait (see hc_device_error) */
};

/* Problem shape and scalar constants. The model's values ("Router" page, config.json excerpt):
 * hc = 4 (hc_mult), d = 5120 (dim), sinkhorn_iters = 20, hc_eps = 1e-6, norm_eps = 1e-20. */
typedef struct {
    int hc;             /* streams, 1..8. hc = 4 with d a multiple of 256 up to 5120 (the model's shape)
                           runs on the fused tensor-core kernel; every other shape on the generic
                           kernels (the projection on the tensor cores, the other steps on CUDA cores),
                           within the same tolerances (slower) */
    int d;              /* width of one stream: a multiple of 8, at most 65536 */
    int sinkhorn_iters; /* >= 1: one softmax + column normalisation, then iters-1 row+column rounds */
    float hc_eps;       /* >= 0, finite: the eps of pre and of the Sinkhorn normalisations */
    float norm_eps;     /* >= 0, finite: used by both the mixes statistic and the sublayer RMSNorm */
} hc_shape_t;

/* One sublayer's HC parameters ("Source layer, pairs pooled" page, Block.__init__ excerpt:
 * hc_fn [mix_hc, hc*d], hc_base [mix_hc], hc_scale [3], mix_hc = (2+hc)*hc; the sublayer's
 * RMSNorm weight [d]). All [device].
 * The projection weights come as the planes hc_prepare_params makes from the fp32 hc_fn, not as
 * hc_fn itself: the split is done once per parameter set instead of in every call, and the planes
 * are laid out for the kernel's loads. The caller guarantees that the planes were prepared with
 * the (hc, d) of the call's hc_shape_t and from the hc_fn in use. A device buffer carries neither
 * its size nor its source, so the library cannot check this: planes of another shape are read out
 * of bounds, and planes of an older hc_fn give that hc_fn's mixes. */
typedef struct {
    const void* hc_fn_planes; /* bf16 [3*mix_hc, hc*d]: hc_fn split by hc_prepare_params. Required. */
    const float* hc_scale;    /* fp32 [3] */
    const float* hc_base;     /* fp32 [mix_hc] */
    const float* norm_w;      /* fp32 [d] */
} hc_params_t;

/* Size in bytes of the buffer hc_prepare_params fills: 3 * (2+hc)*hc * hc*d * 2.
 * Returns HC_ERR_NULL / HC_ERR_SHAPE on bad arguments. Host-only, no CUDA call. */
int hc_prepare_params_size(int hc, int d, size_t* bytes);

/* Split an fp32 hc_fn [(2+hc)*hc, hc*d] [device] into three bf16 planes hi + mid + lo whose sum
 * equals every fp32 weight exactly, laid out for the tensor-core projections, into `planes`
 * [device] (hc_prepare_params_size bytes, 16-byte aligned): [3*mix_hc, hc*d] rows, at hc = 4 row
 * 36h + 12p + i holding plane p of mix 12h + i, at any other hc row p*mix_hc + m holding plane p
 * of mix m. Run it once per parameter set (weights are static); the planes stay valid while hc_fn
 * is unchanged. No counterpart on the pages: it is this library's weight packing. hc in 1..8. */
int hc_prepare_params(const float* hc_fn, int hc, int d, void* planes, hc_stream_t stream);

/* Size in bytes of the workspace the fused calls (hc_pre_step, hc_post_then_pre,
 * hc_post_then_pre_tap, hc_expand_pre_step, hc_debug_mixes) need: the CTAs that share a token tile
 * (8, 16 or 32 of them, as the launch plan of hc_plan_tiles chooses) exchange their per-token
 * partial sums through it (about 14 KB per CTA per tile, L2-resident) together with one 64-bit
 * arrival counter per group of CTAs, which counts the blocks published, and the counter's value at
 * the start of the group's next launch (both kept on the device, so launches replayed from a CUDA
 * graph wait for their own arrivals too). It has room for 256 co-resident CTAs: 7,344,384 bytes.
 * The caller allocates it once [device], 16-byte aligned, fills it with zeros before its first use
 * and then keeps passing it unchanged (no re-zeroing needed). Calls that may run at the same time on
 * the GPU must not share a workspace. One exception to "no re-zeroing": after a kernel gave up a
 * bounded wait (HC_ERR_DEVICE, a nonzero hc_device_error word), the counters may no longer match
 * (a late CTA may add its arrival after the group moved on); zero the workspace again before reusing
 * it. Host-only, no CUDA call. */
int hc_workspace_size(size_t* bytes);

/* Reading half of one sublayer ("Source layer, pairs pooled" page, Block.forward excerpt, the
 * lines up to the sublayer's norm): hc_mixes of X with `p`, hc_pre of X with pre_mix, RMSNorm.
 *   X        [device] bf16 [n, hc, d]      the incoming streams
 *   pre_mix  [device] fp32 [n, hc]         the reading mix handed over by the previous sublayer
 *   p        this sublayer's parameters
 *   y_normed [device] bf16 [n, d]          out: the sublayer's input
 *   pre, post [device] fp32 [n, hc]; comb [device] fp32 [n, hc, hc]   out: this sublayer's
 *            coefficients (pre goes to the next sublayer, post/comb to this one's hc_post)
 *   workspace [device]                     see hc_workspace_size
 * Outputs and the workspace must not overlap each other or any input (HC_ERR_ALIAS). The launch
 * is cooperative (all its CTAs resident at once); HC_ERR_UNSUPPORTED if the device cannot. */
int hc_pre_step(const void* X, const float* pre_mix, hc_params_t p, int64_t n, hc_shape_t s,
                void* y_normed, float* pre, float* post, float* comb, void* workspace,
                hc_stream_t stream);

/* Writing half of a sublayer, then the reading half of the next one, fused in one pass:
 *   X_out = hc_post(delta, X, post, comb)   ("Write the streams" page, formula for X')
 *   (y_normed, pre_out, post_out, comb_out) = hc_pre_step(X_out, pre_mix, next)
 *   delta [device] bf16 [n, d]      the sublayer's output
 *   X     [device] bf16 [n, hc, d]  the streams the sublayer read (its residual)
 *   post, comb [device] fp32        this sublayer's writing coefficients
 *   pre_mix [device] fp32 [n, hc]   the reading mix for the next sublayer (the pre returned by
 *                                   the call that produced post/comb)
 *   next                            the next sublayer's parameters
 *   workspace [device]              see hc_workspace_size
 * X_out is written once. Outputs and the workspace must not overlap each other or any input
 * (HC_ERR_ALIAS). Cooperative launch, as hc_pre_step. */
int hc_post_then_pre(const void* delta, const void* X, const float* post, const float* comb,
                     const float* pre_mix, hc_params_t next, int64_t n, hc_shape_t s, void* X_out,
                     void* y_normed, float* pre_out, float* post_out, float* comb_out,
                     void* workspace, hc_stream_t stream);

/* hc_post_then_pre that also writes the mean of the four new streams, the input of the
 * multi-token-prediction head ("Final RMSNorm" page, Transformer.forward excerpt: at the head's
 * target layers, 37-39 of the "Router" page's config.json, the model keeps the mean over the hc
 * streams entering the layer, cast to the stream dtype):
 *   stream_mean [device] bf16 [n, d] = bf16(mean_j X_out[:, j, :])   (summed in fp32)
 * computed from the X' values the call already holds, so it costs only its own 2*d bytes of writes
 * per token. stream_mean must not overlap any other argument (HC_ERR_ALIAS); everything else as
 * hc_post_then_pre. */
int hc_post_then_pre_tap(const void* delta, const void* X, const float* post, const float* comb,
                         const float* pre_mix, hc_params_t next, int64_t n, hc_shape_t s, void* X_out,
                         void* y_normed, float* pre_out, float* post_out, float* comb_out, void* stream_mean,
                         void* workspace, hc_stream_t stream);

/* hc_post_then_pre for callers that cannot allocate device memory. Some callers can never call
 * cudaMalloc (or any allocator) at the point where they run this step: a plugin hosted by an
 * engine that owns all device memory and hands it no workspace, a runtime whose memory plan is
 * frozen after start-up, or a program that must not risk an allocation failing mid-run. This
 * entry point takes the same arguments as hc_post_then_pre minus the workspace, and computes the
 * same results: its scratch is a fixed array inside the library's device image, 7,344,384 bytes
 * (the hc_workspace_size figure), which every GPU that loads the library keeps until the process
 * exits. It allocates nothing and calls no allocating routine.
 *   - The first call on a device looks up that device's copy of the array (a runtime query, no
 *     allocation); make that first call before any stream capture.
 *   - No call needs more scratch than the array holds: the library launches at most 256 CTAs
 *     whatever the GPU, and the shapes outside the fused kernel work through their tokens in
 *     chunks that fit. Sizes are refused only as for hc_post_then_pre (n above 2^31 - 1:
 *     HC_ERR_SHAPE; hc > 8 or d > 65536: HC_ERR_UNSUPPORTED).
 *   - All calls share the one array. It needs no clearing between calls: it is zero at load and
 *     every call tags its exchange flags with a new launch number. But two calls whose kernels
 *     could run at the same time on the GPU (other streams, other threads) race on it and produce
 *     wrong results; serialise them, or use hc_post_then_pre with separate workspaces.
 *   - After a kernel gave up a bounded wait (HC_ERR_DEVICE, a nonzero hc_device_error word), the
 *     array's exchange counters may no longer match: hc_device_error with `clear` zeroes the array
 *     of the current device too, so the next call starts afresh.
 * The pages have no counterpart to this call: it is a packaging of hc_post_then_pre only. */
int hc_post_then_pre_noalloc(const void* delta, const void* X, const float* post, const float* comb,
                             const float* pre_mix, hc_params_t next, int64_t n, hc_shape_t s,
                             void* X_out, void* y_normed, float* pre_out, float* post_out,
                             float* comb_out, hc_stream_t stream);

/* Writing half alone ("Write the streams" page): X_out = bf16(post_k*delta + sum_j comb[j,k]*X_j).
 * For the last sublayer of a stack and for boundaries where another module edits the streams
 * before the next reading half. s.sinkhorn_iters and the eps fields are ignored; d is a multiple
 * of 8. X_out may be exactly X (in place); any other overlap with X or delta is HC_ERR_ALIAS. */
int hc_post(const void* delta, const void* X, const float* post, const float* comb, int64_t n,
            hc_shape_t s, void* X_out, hc_stream_t stream);

/* Head of the stack ("Final RMSNorm" page, Transformer.forward excerpt: the embedding row is copied
 * into each of the hc streams and the first block reads them with the identity pre_mix), fused
 * with the first sublayer's reading half:
 *   X_out[t, j, :] = h[t, :] for every stream j
 *   (y_normed, pre, post, comb) = hc_pre_step(X_out, identity pre_mix, p)
 *   h      [device] bf16 [n, d]      the embedding rows
 *   X_out  [device] bf16 [n, hc, d]  out: the expanded streams (the first sublayer's residual)
 *   the other arguments as hc_pre_step.
 * The pages do not print the identity pre_mix; this call weights every stream by 1/hc. Any
 * weights summing to 1 collapse identical streams to h exactly, so the choice changes no output.
 * h is read once and the streams are written once. Outputs and the workspace must not overlap
 * each other or h (HC_ERR_ALIAS). Cooperative launch, as hc_pre_step. */
int hc_expand_pre_step(const void* h, hc_params_t p, int64_t n, hc_shape_t s, void* X_out,
                       void* y_normed, float* pre, float* post, float* comb, void* workspace,
                       hc_stream_t stream);

/* Tail of the stack ("Final RMSNorm" page: Transformer.forward excerpt, RMSNorm excerpt and the
 * m_2 formula): after the last block the streams are collapsed once more with the last pre_mix
 * and go through the final RMSNorm:
 *   y = bf16(sum_j pre_mix_j * X_j)
 *   z = bf16(norm_w * y / sqrt(mean(y^2) + s.norm_eps))     (the page's eps is 1e-20)
 *   X       [device] bf16 [n, hc, d]   the streams after the last block
 *   pre_mix [device] fp32 [n, hc]      the pre returned by the last reading half
 *   norm_w  [device] fp32 [d]          the final norm's gain
 *   z       [device] bf16 [n, d]       out
 * s.sinkhorn_iters and s.hc_eps are ignored; d is a multiple of 8 and at most 5120. z must not
 * overlap an input (HC_ERR_ALIAS). */
int hc_final(const void* X, const float* pre_mix, const float* norm_w, int64_t n, hc_shape_t s,
             void* z, hc_stream_t stream);

/* The last sublayer's writing half fused with hc_final:
 *   X' = bf16(post_k * delta + sum_j comb[j,k] * X_j), then z = hc_final(X', pre_mix, norm_w)
 *   delta, X, post, comb as hc_post_then_pre; pre_mix, norm_w, z as hc_final.
 *   X_out [device] bf16 [n, hc, d] or NULL: receives X' when given. The model reads the streams
 *         no more after the final collapse, so NULL saves their 2*hc*d bytes per token of writes.
 * Outputs must not overlap each other or any input (HC_ERR_ALIAS). Other rules as hc_final. */
int hc_post_then_final(const void* delta, const void* X, const float* post, const float* comb,
                       const float* pre_mix, const float* norm_w, int64_t n, hc_shape_t s,
                       void* X_out, void* z, hc_stream_t stream);

/* ---- Host-buffer executor ---------------------------------------------------------------------
 * For callers whose per-token arrays live in host memory: the executor streams the tokens through
 * the GPU in chunks, copying one chunk in while the fused step runs on another and a third is
 * copied back, on its own two copy streams. On a GB300 the host link bounds such a call, so the
 * overlap of the two copy directions is what it buys. No counterpart on the pages: it is this
 * library's host-side runtime around hc_post_then_pre. */
typedef struct hc_host_pipeline hc_host_pipeline_t;

/* Create an executor for calls of shape (hc, d) on the current device. It allocates, and owns
 * until hc_host_pipeline_destroy: device staging for 3 chunks of `chunk_tokens` tokens of every
 * input and output of hc_post_then_pre (3 * chunk_tokens * (2*hc*d*2 + 2*d*2 + 3*hc*4 + 2*hc*hc*4)
 * bytes, plus alignment; 0 = 1024 tokens, at most 1 << 20); when hc is a multiple of 4, two
 * segment buffers for the coefficient arrays of S = max(chunk_tokens, 65536) tokens each
 * (2 * S * (4*hc*4 + 2*hc*hc*4) bytes), which then move once per segment of up to S tokens instead
 * of once per chunk; its own zero-filled workspace; two non-blocking streams and its events. It
 * synchronises its own copy stream once. Returns HC_ERR_NULL (out NULL), HC_ERR_SHAPE (hc < 1, d
 * not a positive multiple of 8, chunk_tokens out of range), HC_ERR_UNSUPPORTED (hc > 8,
 * d > 65536) or HC_ERR_CUDA (an allocation or a stream or event creation failed; nothing is left
 * allocated). */
int hc_host_pipeline_create(int hc, int d, int64_t chunk_tokens, hc_host_pipeline_t** out);

/* Tokens per chunk of an executor. */
int hc_host_pipeline_chunk_tokens(const hc_host_pipeline_t* p, int64_t* chunk_tokens);

/* How a call on n tokens is cut into chunks by an executor of chunk_tokens (0 = the default, see
 * hc_host_pipeline_create) tokens per chunk, C. Between ramps of halving size at both ends (C/2,
 * C/4, ... down to the last size of at least max(128, C/32) tokens, five sizes at most) run chunks
 * of C, the last of them shorter: the first copy-in and the last copy-out, which nothing overlaps,
 * stay short, and most tokens move in a few large copies. When n is below both ramps plus one
 * chunk, or C < 256, the tokens are cut into equal chunks of at most C tokens, and into up to 8
 * when each keeps 32 tokens or more. Writes the number of chunks to *count; for 0 <= index < *count
 * also the chunk's first token and size. index < 0 asks for the count only (t0 and tokens may then
 * be NULL). Host-only, no CUDA call. Returns HC_ERR_NULL, HC_ERR_SHAPE (n < 0, chunk_tokens out of
 * range) or HC_ERR_ARG (index >= count). */
int hc_host_chunk_plan(int64_t n, int64_t chunk_tokens, int64_t index, int64_t* count, int64_t* t0,
                       int64_t* tokens);

/* Wait for every call enqueued on the executor to finish (host-side wait), then free what it owns.
 * NULL is a no-op. Returns HC_ERR_CUDA if that wait reported an error (everything is freed anyway). */
int hc_host_pipeline_destroy(hc_host_pipeline_t* p);

/* hc_post_then_pre with every per-token array in HOST memory (delta, X, post, comb, pre_mix in;
 * X_out, y_normed, pre_out, post_out, comb_out out; same layouts as hc_post_then_pre). The results
 * are those of hc_post_then_pre applied to each chunk of hc_host_chunk_plan: X_out equals a single
 * call on all n tokens bit for bit (it is per element); y_normed and the coefficients may differ
 * from it in the last bits, since the order in which the mixes' partial sums meet follows the tile
 * plan of the chunk's size. `next` holds [device] pointers, as for hc_post_then_pre. Host arrays
 * need no alignment; page-locked ones (cudaHostAlloc, cudaHostRegister, torch pin_memory) let the
 * copies run asynchronously and overlap; pageable ones work, but each copy then blocks the calling
 * thread. The call enqueues everything and returns: the results are in host memory once `stream`
 * has passed the call (e.g. after cudaStreamSynchronize(stream)); until then the host arrays must
 * stay allocated and the inputs unchanged. The call starts after the earlier work on `stream` and
 * after the previous call on the same executor. One executor serves one call at a time: calls on
 * it from several host threads must be serialised by the caller. s.hc and s.d must be the
 * executor's (HC_ERR_SHAPE otherwise); the current device must be the executor's (HC_ERR_ARG
 * otherwise); no output may overlap an input or another output (HC_ERR_ALIAS). A failure part-way
 * (HC_ERR_CUDA, or a status of the per-chunk hc_post_then_pre) leaves the outputs incomplete. */
int hc_host_post_then_pre(hc_host_pipeline_t* p, const void* delta, const void* X, const float* post,
                          const float* comb, const float* pre_mix, hc_params_t next, int64_t n,
                          hc_shape_t s, void* X_out, void* y_normed, float* pre_out, float* post_out,
                          float* comb_out, hc_stream_t stream);

/* Diagnostic: the 24 mix numbers r * (X_flat . hc_fn^T) [device] fp32 [n, (2+hc)*hc] exactly as the
 * fused reading half computes them (same kernel, same tensor-core projection), for checking the
 * projection on its own. p.hc_scale, p.hc_base and p.norm_w are not read. A token's mixes depend on
 * the group size of the launch (how many CTAs split its columns, so in which order their partial
 * sums meet), not on which other tokens share its tile: `group` 0 takes the launch plan for n
 * tokens; 8, 16 or 32 forces that group size (d a multiple of 32 * group), so that the mixes of
 * sampled tokens reproduce bit for bit those of a call on more tokens (its group: hc_plan_tiles).
 * The generic path (shapes the fused kernel does not take) ignores `group`. HC_ERR_ARG for another
 * group value. */
int hc_debug_mixes(const void* X, hc_params_t p, int64_t n, hc_shape_t s, int group, float* mixes,
                   void* workspace, hc_stream_t stream);

/* Launch plan of the fused calls for n tokens of stream width d when `ctas` CTAs of the fused
 * kernel can be resident at once (hc_fused_ctas): the CTAs that share one token tile (`group`: 8,
 * 16 or 32, each taking d/group columns; small batches use larger groups, so each CTA has fewer
 * column stages), the tokens per tile and the number of tiles. Groups of 8 take tiles of 32, 64, 96
 * or 128 tokens (for batches of several waves possibly the height between 96 and 128 that spreads
 * the tiles evenly over the waves; n itself when n < 32). Groups of 16 and 32 take tiles of 64 tokens
 * and process two column stages per pass, in the two halves of the 128-row tensor-core tile. Host-only, no CUDA call. Returns HC_ERR_NULL / HC_ERR_SHAPE (n < 0, d
 * not a positive multiple of 256, ctas < 8) on bad arguments. */
int hc_plan_tiles(int64_t n, int d, int ctas, int* group, int* tile_m, int64_t* num_tiles);

/* How many CTAs of the fused kernel can be resident on the current device at once (one per SM on
 * GB300: 152), capped at 256. */
int hc_fused_ctas(int* ctas);

/* Diagnostic for the bounded waits: one warp waits, exactly as the fused kernel waits for the other
 * CTAs of its group, for each of the 64-bit counters flags[0..count-1] [device] (8-byte aligned,
 * count 1..32) to reach at least `value` (the fused kernel waits on one: its group's arrival
 * counter), and gives up after limit_ns (0..1e9) nanoseconds: it then sets the exchange bit of the
 * device error word (hc_device_error) and returns, leaving the context usable. The fused kernel
 * gives up after one second on every wait in the same way. No counterpart on the pages. */
int hc_debug_wait_flag(const unsigned long long* flags, int count, unsigned long long value, int64_t limit_ns,
                       hc_stream_t stream);

/* Read the device-side error word of the current device: nonzero when a kernel gave up a
 * bounded wait (it then returned early and its outputs are not valid); bits 0-15 are the fused
 * kernel's waits, bits 16-19 those of the generic path's projection. Synchronises `stream`.
 * If `clear` is nonzero the word is reset to 0, and, when it was nonzero, the library's own fixed
 * scratch of hc_post_then_pre_noalloc on this device is zeroed as well (on `stream`; no call using it
 * may still be running). Returns HC_OK, HC_ERR_NULL or HC_ERR_CUDA. */
int hc_device_error(unsigned int* word, int clear, hc_stream_t stream);

/* Static description of a status code (never NULL). */
const char* hc_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* HC_GB300_H */
