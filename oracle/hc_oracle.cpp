// Plain CPU oracle for the Hyper-Connection (HC) stream step.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or call this file:
// only the tests, the smoke check and the CPU-baseline / reference arm of the benchmark do.
// It shares no code, header, table or helper with the CUDA path.
//
// Every quantity is computed in double precision, step by step, in the order the source pages
// give, and rounded to bfloat16 (round to nearest, ties to even) exactly where the model casts:
// the written streams X', the collapsed sublayer input y and the normalised sublayer input.
//
// Sources (DeepSeek V4.1 model-atlas pages):
//   [SL]  "Source layer, pairs pooled" page, Code section: the Block.__init__, Block.forward and
//         Block.hc_mixes / hc_pre / hc_post excerpts; Parameters table (stream weights 491,547).
//   [RW]  "Reading weights" page: the formula for p_{n+1,j}, and the Code section's
//         hc_split_sinkhorn kernel excerpt and its wrapper.
//   [FN]  "Final RMSNorm" page: the m_2(x) formula (with its epsilon of 1e-20), the RMSNorm
//         excerpt, and the Transformer.forward excerpt (the embedding copied into the hc streams
//         before the first block; after the last block one more collapse with the last pre_mix,
//         then the final norm).
//   [WS]  "Write the streams" page: the formula for X'_{n,k} and its in/out shapes.
//   [RT]  "Router" page, config.json excerpt: hc_mult 4, hc_sinkhorn_iters 20, hc_eps 1e-6,
//         norm_eps 1e-20, dim 5120.
//
// Layouts (all contiguous, row-major, tokens flattened to n = B*T):
//   X       [n, hc, d]  bf16 bits      delta  [n, d]  bf16 bits
//   post    [n, hc]     fp32           comb   [n, hc, hc] fp32, comb[t, j, k]: j = source stream
//                                                             (summed over), k = destination
//   pre_mix [n, hc]     fp32           hc_fn  [(2+hc)*hc, hc*d] fp32, column c = j*d + i
//   hc_scale [3] fp32, hc_base [(2+hc)*hc] fp32, norm_w [d] fp32
//   mixes   [n, (2+hc)*hc] double: [pre logits hc | post logits hc | comb logits hc*hc (row j, col k)]

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>

namespace {

// ---- bfloat16 conversions, from the format's definition ------------------------------------
// bfloat16 = the top 16 bits of an IEEE binary32: 1 sign bit, 8 exponent bits, 7 fraction bits.
// So it has binary32's exponent range (normal down to 2^-126, subnormal down to 2^-133) and an
// 8-bit significand.

double bf16_to_double(uint16_t b) {
    uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return static_cast<double>(f);
}

// Round a double to the nearest bfloat16, ties to even, overflow to infinity, NaN to a quiet NaN.
uint16_t double_to_bf16(double x) {
    if (std::isnan(x)) return 0x7FC0;
    const bool neg = std::signbit(x);
    const uint16_t sign = neg ? 0x8000 : 0x0000;
    double a = std::fabs(x);
    if (std::isinf(a)) return sign | 0x7F80;
    if (a == 0.0) return sign;
    int E;
    std::frexp(a, &E);                    // a = f * 2^E, f in [0.5, 1): a in [2^(E-1), 2^E)
    int qexp = std::max(E - 8, -133);     // spacing of bf16 values around a (8 significant bits)
    double q = std::ldexp(1.0, qexp);
    double t = a / q;                     // exact: scaling by a power of two
    double r = std::floor(t);
    double frac = t - r;
    if (frac > 0.5 || (frac == 0.5 && std::fmod(r, 2.0) != 0.0)) r += 1.0;
    double v = r * q;
    // largest finite bf16 is (2 - 2^-7) * 2^127; anything that rounds beyond it is infinite
    if (v >= std::ldexp(1.0, 128)) return sign | 0x7F80;
    float vf = static_cast<float>(v);     // exact: v has at most 8 significant bits in range
    uint32_t u;
    std::memcpy(&u, &vf, 4);
    return sign | static_cast<uint16_t>(u >> 16);
}

double sigmoid(double z) { return 1.0 / (1.0 + std::exp(-z)); }

template <class F>
void parallel_for(int64_t n, int threads, F&& body) {
    if (threads <= 0) threads = static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));
    if (n <= 0) return;
    if (threads == 1 || n < 2) {
        for (int64_t t = 0; t < n; ++t) body(t);
        return;
    }
    int64_t nt = std::min<int64_t>(threads, n);
    std::vector<std::thread> pool;
    pool.reserve(nt);
    for (int64_t w = 0; w < nt; ++w) {
        int64_t lo = n * w / nt, hi = n * (w + 1) / nt;
        pool.emplace_back([lo, hi, &body]() {
            for (int64_t t = lo; t < hi; ++t) body(t);
        });
    }
    for (auto& th : pool) th.join();
}

// ---- one token of each step -----------------------------------------------------------------

// [WS] formula X'_{n,k} = u_k * Delta + sum_j C_jk X_{n,j}; [SL] hc_post excerpt: the sum runs over
// the comb index that multiplies the residual's stream (dim 2 of comb), the result is cast to the
// stream dtype.
// Optionally also returns the value before rounding and the sum of the terms' magnitudes (the
// scale of any fp32 evaluation's rounding error, used by tolerances).
void post_token(int hc, int d, const uint16_t* X, const uint16_t* delta, const float* post,
                const float* comb, uint16_t* X_out, double* exact, double* abssum) {
    for (int k = 0; k < hc; ++k) {
        for (int i = 0; i < d; ++i) {
            double acc = static_cast<double>(post[k]) * bf16_to_double(delta[i]);
            double mag = std::fabs(acc);
            for (int j = 0; j < hc; ++j) {
                double term = static_cast<double>(comb[j * hc + k]) * bf16_to_double(X[j * d + i]);
                acc += term;
                mag += std::fabs(term);
            }
            X_out[k * d + i] = double_to_bf16(acc);
            if (exact) exact[k * d + i] = acc;
            if (abssum) abssum[k * d + i] = mag;
        }
    }
}

// [SL] hc_mixes excerpt: flatten the hc streams to hc*d values, r = 1/sqrt(mean(x^2) + norm_eps)
// over all hc*d of them, mixes = (x . hc_fn[m]) * r. Also returns S[m] = r * sum |x_c hc_fn[m,c]|,
// the scale of the dot product's rounding error.
void mixes_token(int hc, int d, const uint16_t* X, const float* hc_fn, double norm_eps,
                 double* mixes, double* r_out, double* S) {
    const int D = hc * d;
    const int M = (2 + hc) * hc;
    double ss = 0.0;
    for (int c = 0; c < D; ++c) {
        double x = bf16_to_double(X[c]);
        ss += x * x;
    }
    double r = 1.0 / std::sqrt(ss / D + norm_eps);
    for (int m = 0; m < M; ++m) {
        const float* w = hc_fn + static_cast<int64_t>(m) * D;
        double dot = 0.0, absdot = 0.0;
        for (int c = 0; c < D; ++c) {
            double p = bf16_to_double(X[c]) * static_cast<double>(w[c]);
            dot += p;
            absdot += std::fabs(p);
        }
        mixes[m] = dot * r;
        if (S) S[m] = absdot * r;
    }
    if (r_out) *r_out = r;
}

// [RW] hc_split_sinkhorn kernel excerpt and the p_{n+1,j} formula:
//   pre_j  = sigmoid(s0 * m_j + b_j) + eps
//   post_j = 2 * sigmoid(s1 * m_{hc+j} + b_{hc+j})
//   L_jk   = s2 * m_{2hc + j*hc + k} + b_{2hc + j*hc + k}
//   C = softmax over each row of L (max subtracted), then + eps
//   C_jk /= (column sum_k + eps)
//   then (iters - 1) times: C_jk /= (row sum_j + eps); C_jk /= (column sum_k + eps)
void split_token(int hc, const double* m, const float* hc_scale, const float* hc_base, int iters,
                 double eps, double* pre, double* post, double* comb) {
    const double s0 = hc_scale[0], s1 = hc_scale[1], s2 = hc_scale[2];
    for (int j = 0; j < hc; ++j) pre[j] = sigmoid(m[j] * s0 + hc_base[j]) + eps;
    for (int j = 0; j < hc; ++j) post[j] = 2.0 * sigmoid(m[hc + j] * s1 + hc_base[hc + j]);
    std::vector<double> C(static_cast<size_t>(hc) * hc), rs(hc), cs(hc);
    for (int j = 0; j < hc; ++j)
        for (int k = 0; k < hc; ++k)
            C[j * hc + k] = m[2 * hc + j * hc + k] * s2 + hc_base[2 * hc + j * hc + k];
    // row softmax, then + eps
    for (int j = 0; j < hc; ++j) {
        double mx = C[j * hc];
        for (int k = 1; k < hc; ++k) mx = std::max(mx, C[j * hc + k]);
        double sum = 0.0;
        for (int k = 0; k < hc; ++k) {
            C[j * hc + k] = std::exp(C[j * hc + k] - mx);
            sum += C[j * hc + k];
        }
        for (int k = 0; k < hc; ++k) C[j * hc + k] = C[j * hc + k] / sum + eps;
    }
    auto col_normalise = [&]() {
        for (int k = 0; k < hc; ++k) {
            double s = 0.0;
            for (int j = 0; j < hc; ++j) s += C[j * hc + k];
            cs[k] = s;
        }
        for (int j = 0; j < hc; ++j)
            for (int k = 0; k < hc; ++k) C[j * hc + k] = C[j * hc + k] / (cs[k] + eps);
    };
    auto row_normalise = [&]() {
        for (int j = 0; j < hc; ++j) {
            double s = 0.0;
            for (int k = 0; k < hc; ++k) s += C[j * hc + k];
            rs[j] = s;
        }
        for (int j = 0; j < hc; ++j)
            for (int k = 0; k < hc; ++k) C[j * hc + k] = C[j * hc + k] / (rs[j] + eps);
    };
    col_normalise();
    for (int it = 0; it < iters - 1; ++it) {
        row_normalise();
        col_normalise();
    }
    for (int q = 0; q < hc * hc; ++q) comb[q] = C[q];
}

// [SL] hc_pre excerpt: y = sum_j pre_mix_j * X_j in float, cast back to the stream dtype.
void pre_token(int hc, int d, const uint16_t* X, const float* pre_mix, uint16_t* y, double* y_exact,
               double* y_abssum) {
    for (int i = 0; i < d; ++i) {
        double acc = 0.0, mag = 0.0;
        for (int j = 0; j < hc; ++j) {
            double term = static_cast<double>(pre_mix[j]) * bf16_to_double(X[j * d + i]);
            acc += term;
            mag += std::fabs(term);
        }
        if (y_exact) y_exact[i] = acc;
        if (y_abssum) y_abssum[i] = mag;
        y[i] = double_to_bf16(acc);
    }
}

// [FN] RMSNorm excerpt and formula: m2 = mean(x^2) over d, out = w * x / sqrt(m2 + eps), cast back
// to the input dtype.
void rmsnorm_token(int d, const uint16_t* x, const float* w, double eps, uint16_t* out, double* out_exact) {
    double ss = 0.0;
    for (int i = 0; i < d; ++i) {
        double v = bf16_to_double(x[i]);
        ss += v * v;
    }
    double r = 1.0 / std::sqrt(ss / d + eps);
    for (int i = 0; i < d; ++i) {
        double v = static_cast<double>(w[i]) * (bf16_to_double(x[i]) * r);
        if (out_exact) out_exact[i] = v;
        out[i] = double_to_bf16(v);
    }
}

// [FN] Transformer.forward excerpt: the embedding row h [d] becomes hc identical streams.
void expand_token(int hc, int d, const uint16_t* h, uint16_t* X) {
    for (int j = 0; j < hc; ++j) std::copy(h, h + d, X + static_cast<int64_t>(j) * d);
}

// The identity pre_mix the same excerpt hands to the first block is not printed on the pages. On
// hc identical streams every set of weights summing to 1 collapses them to the embedding itself;
// the oracle takes the uniform weights 1/hc (exact in binary for hc = 2, 4, 8).
void identity_pre_mix(int hc, float* pm) {
    for (int j = 0; j < hc; ++j) pm[j] = 1.0f / static_cast<float>(hc);
}

}  // namespace

extern "C" {

uint16_t oracle_double_to_bf16(double x) { return double_to_bf16(x); }
double oracle_bf16_to_double(uint16_t b) { return bf16_to_double(b); }

void oracle_round_bf16(int64_t count, const double* x, uint16_t* out) {
    for (int64_t q = 0; q < count; ++q) out[q] = double_to_bf16(x[q]);
}

void oracle_hc_post(int64_t n, int hc, int d, const uint16_t* X, const uint16_t* delta, const float* post,
                    const float* comb, uint16_t* X_out, int threads) {
    parallel_for(n, threads, [&](int64_t t) {
        post_token(hc, d, X + t * hc * d, delta + t * d, post + t * hc, comb + t * hc * hc, X_out + t * hc * d,
                   nullptr, nullptr);
    });
}

void oracle_hc_post_detail(int64_t n, int hc, int d, const uint16_t* X, const uint16_t* delta, const float* post,
                           const float* comb, uint16_t* X_out, double* exact, double* abssum, int threads) {
    parallel_for(n, threads, [&](int64_t t) {
        post_token(hc, d, X + t * hc * d, delta + t * d, post + t * hc, comb + t * hc * hc, X_out + t * hc * d,
                   exact + t * hc * d, abssum + t * hc * d);
    });
}

void oracle_hc_mixes(int64_t n, int hc, int d, const uint16_t* X, const float* hc_fn, double norm_eps,
                     double* mixes, double* r, double* S, int threads) {
    const int M = (2 + hc) * hc;
    parallel_for(n, threads, [&](int64_t t) {
        mixes_token(hc, d, X + t * hc * d, hc_fn, norm_eps, mixes + t * M, r ? r + t : nullptr,
                    S ? S + t * M : nullptr);
    });
}

void oracle_split_sinkhorn(int64_t n, int hc, const double* mixes, const float* hc_scale, const float* hc_base,
                           int iters, double eps, double* pre, double* post, double* comb, int threads) {
    const int M = (2 + hc) * hc;
    parallel_for(n, threads, [&](int64_t t) {
        split_token(hc, mixes + t * M, hc_scale, hc_base, iters, eps, pre + t * hc, post + t * hc,
                    comb + t * hc * hc);
    });
}

void oracle_hc_pre(int64_t n, int hc, int d, const uint16_t* X, const float* pre_mix, uint16_t* y,
                   double* y_exact, double* y_abssum, int threads) {
    parallel_for(n, threads, [&](int64_t t) {
        pre_token(hc, d, X + t * hc * d, pre_mix + t * hc, y + t * d, y_exact ? y_exact + t * d : nullptr,
                  y_abssum ? y_abssum + t * d : nullptr);
    });
}

void oracle_rmsnorm(int64_t n, int d, const uint16_t* x, const float* w, double eps, uint16_t* out,
                    double* out_exact, int threads) {
    parallel_for(n, threads, [&](int64_t t) {
        rmsnorm_token(d, x + t * d, w, eps, out + t * d, out_exact ? out_exact + t * d : nullptr);
    });
}

// [SL] Block.forward excerpt, one sublayer's reading half: the coefficients come from hc_mixes of
// the incoming streams with this sublayer's parameters; the streams are collapsed with the pre_mix
// handed over by the previous sublayer; the collapse goes through the sublayer's RMSNorm.
// Outputs: y_normed [n,d] bf16; pre, post [n,hc]; comb [n,hc,hc]; optional mixes [n,M], r [n],
// S [n,M] and y (the collapsed, bf16-rounded input to the norm) [n,d].
void oracle_hc_pre_step(int64_t n, int hc, int d, const uint16_t* X, const float* pre_mix, const float* hc_fn,
                        const float* hc_scale, const float* hc_base, const float* norm_w, int iters,
                        double hc_eps, double norm_eps, uint16_t* y_normed, double* pre, double* post,
                        double* comb, double* mixes_out, double* r_out, double* S_out, uint16_t* y_out,
                        int threads) {
    const int M = (2 + hc) * hc;
    parallel_for(n, threads, [&](int64_t t) {
        const uint16_t* Xt = X + t * hc * d;
        std::vector<double> m(M), S(M);
        double r;
        mixes_token(hc, d, Xt, hc_fn, norm_eps, m.data(), &r, S.data());
        split_token(hc, m.data(), hc_scale, hc_base, iters, hc_eps, pre + t * hc, post + t * hc,
                    comb + t * hc * hc);
        std::vector<uint16_t> y(d);
        pre_token(hc, d, Xt, pre_mix + t * hc, y.data(), nullptr, nullptr);
        rmsnorm_token(d, y.data(), norm_w, norm_eps, y_normed + t * d, nullptr);
        if (mixes_out) std::copy(m.begin(), m.end(), mixes_out + t * M);
        if (S_out) std::copy(S.begin(), S.end(), S_out + t * M);
        if (r_out) r_out[t] = r;
        if (y_out) std::copy(y.begin(), y.end(), y_out + t * d);
    });
}

// [SL] Block.forward excerpt, the writing half of one sublayer followed by the reading half of the
// next: hc_post with this sublayer's post/comb gives X'; then oracle_hc_pre_step on X' with the
// next sublayer's parameters and the pre_mix this sublayer's predecessor handed over.
void oracle_hc_post_then_pre(int64_t n, int hc, int d, const uint16_t* delta, const uint16_t* X,
                             const float* post_in, const float* comb_in, const float* pre_mix,
                             const float* hc_fn, const float* hc_scale, const float* hc_base,
                             const float* norm_w, int iters, double hc_eps, double norm_eps, uint16_t* X_out,
                             uint16_t* y_normed, double* pre, double* post, double* comb, int threads) {
    oracle_hc_post(n, hc, d, X, delta, post_in, comb_in, X_out, threads);
    oracle_hc_pre_step(n, hc, d, X_out, pre_mix, hc_fn, hc_scale, hc_base, norm_w, iters, hc_eps, norm_eps,
                       y_normed, pre, post, comb, nullptr, nullptr, nullptr, nullptr, threads);
}

// [FN] Transformer.forward excerpt, the head of the stack: expand the embedding h [n,d] into hc
// streams (X_out [n,hc,d]) and run the first sublayer's reading half on them with the identity
// pre_mix (uniform 1/hc). Outputs as oracle_hc_pre_step.
void oracle_hc_expand(int64_t n, int hc, int d, const uint16_t* h, uint16_t* X_out, int threads) {
    parallel_for(n, threads, [&](int64_t t) { expand_token(hc, d, h + t * d, X_out + t * hc * d); });
}

void oracle_hc_expand_pre_step(int64_t n, int hc, int d, const uint16_t* h, const float* hc_fn,
                               const float* hc_scale, const float* hc_base, const float* norm_w, int iters,
                               double hc_eps, double norm_eps, uint16_t* X_out, uint16_t* y_normed, double* pre,
                               double* post, double* comb, int threads) {
    oracle_hc_expand(n, hc, d, h, X_out, threads);
    std::vector<float> pm(static_cast<size_t>(n) * hc);
    for (int64_t t = 0; t < n; ++t) identity_pre_mix(hc, pm.data() + t * hc);
    oracle_hc_pre_step(n, hc, d, X_out, pm.data(), hc_fn, hc_scale, hc_base, norm_w, iters, hc_eps, norm_eps,
                       y_normed, pre, post, comb, nullptr, nullptr, nullptr, nullptr, threads);
}

// [FN] Transformer.forward excerpt, the tail of the stack: collapse the streams X [n,hc,d] once more
// with the pre_mix the last sublayer produced (hc_pre, cast to bf16), then the final RMSNorm with
// its gain norm_w [d] and epsilon norm_eps (1e-20 on the page's formula). z [n,d] bf16; optional
// y [n,d] (the bf16 collapse) and z before rounding.
void oracle_hc_final(int64_t n, int hc, int d, const uint16_t* X, const float* pre_mix, const float* norm_w,
                     double norm_eps, uint16_t* z, uint16_t* y_out, double* z_exact, int threads) {
    parallel_for(n, threads, [&](int64_t t) {
        std::vector<uint16_t> y(d);
        pre_token(hc, d, X + t * hc * d, pre_mix + t * hc, y.data(), nullptr, nullptr);
        rmsnorm_token(d, y.data(), norm_w, norm_eps, z + t * d, z_exact ? z_exact + t * d : nullptr);
        if (y_out) std::copy(y.begin(), y.end(), y_out + t * d);
    });
}

// The last sublayer's writing half (hc_post, X_out [n,hc,d]) followed by oracle_hc_final on X_out.
void oracle_hc_post_then_final(int64_t n, int hc, int d, const uint16_t* delta, const uint16_t* X,
                               const float* post, const float* comb, const float* pre_mix, const float* norm_w,
                               double norm_eps, uint16_t* X_out, uint16_t* z, int threads) {
    oracle_hc_post(n, hc, d, X, delta, post, comb, X_out, threads);
    oracle_hc_final(n, hc, d, X_out, pre_mix, norm_w, norm_eps, z, nullptr, nullptr, threads);
}

// [FN] Transformer.forward excerpt: at the multi-token-prediction head's target layers the model
// keeps h.mean over the hc streams entering the layer (the streams after the previous sublayer's
// hc_post), cast to the stream dtype. out [n, d] bf16 = bf16(mean_j X[t, j, :]).
void oracle_stream_mean(int64_t n, int hc, int d, const uint16_t* X, uint16_t* out, double* exact, int threads) {
    parallel_for(n, threads, [&](int64_t t) {
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int j = 0; j < hc; ++j) acc += bf16_to_double(X[(t * hc + j) * d + i]);
            const double m = acc / hc;
            if (exact) exact[t * d + i] = m;
            out[t * d + i] = double_to_bf16(m);
        }
    });
}

int oracle_hardware_threads() {
    return static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));
}

}  // extern "C"
