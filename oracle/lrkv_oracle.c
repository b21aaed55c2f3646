/*
 * lrkv_oracle.c -- plain fp64 CPU oracle for attention over an LRKV-compressed
 * KV cache.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load this library.  It shares no code, header, table or
 * helper with the CUDA library; the two only ever see the same input bits.
 *
 * What it computes (source: "Low-Rank Key Value Attention", O'Neill, Clancy,
 * Matskevichus, Reid, arXiv:2601.11471v3, as presented in the slide deck
 * "Low-Rank Key Value Attention: shared projections, specialized heads"):
 *
 *   Eqs. (2)-(3), frame "LRKV constrains differences between heads":
 *       W_h^{K,V} = W_shared^{K,V} + U_h^{K,V} (B_h^{K,V})^T,
 *       W_shared in R^{d x d_h}, U_h in R^{d x r}, B_h in R^{d_h x r}.
 *   Eqs. (4)-(5), frame "Cache shared features and compact per-head latents":
 *       K_s = X W_shared^K, V_s = X W_shared^V (L x d_h),
 *       R_h^K = X U_h^K,   R_h^V = X U_h^V   (L x r),
 *       implied full features K_h = K_s + R_h^K (B_h^K)^T, V_h likewise.
 *   Frame "Compute logits without expanding historical keys":
 *       a_h = softmax(q_h K_h^T / sqrt(d_h) + causal mask).
 *   Frame "Aggregate values before the residual up-projection", Eq. (7):
 *       o_h = a_h V_h  (= a_h V_s + (a_h R_h^V)(B_h^V)^T).
 *
 * The oracle deliberately takes the EXPANDED road: it forms W_h (or K_h, V_h)
 * explicitly and runs textbook softmax attention.  The factored road of
 * Eqs. (6)-(7) is what the GPU takes; the slides state the two are equal for
 * the linear model (frame "Training learns the base and residuals together",
 * block "Two different notions of equivalence").
 *
 * Readings where the pages leave a step open:
 *   - no position encoding and no normalisation inside attention;
 *   - decode: the query attends to all seq_len cached tokens (it is the newest
 *     position and is already in the cache); prefill: query at absolute
 *     position p attends to keys j <= p;
 *   - softmax scale 1/sqrt(d_h) unless the caller passes another;
 *   - cache values are produced by an fp64 sum, rounded to fp32 (nearest) and
 *     then to bf16 (nearest, ties to even).
 *
 * Training: forward and backward of one expanded projection K_h = X (W_shared + U_h B_h^T)
 * (frame "Training learns the base and residuals together"), by the chain rule.
 *
 * Second workload: multi-head latent attention ("Embeddings II: MLA & Architectural
 * Choices", weight absorption and decoupled RoPE), absorbed (attention over the cached
 * rows [c_t | k^R_t], values c_t) and expanded (per-head keys and values reconstructed
 * through W^UK, W^UV) -- the associativity of the LRKV slides' backup frame "MLA also
 * admits associative computation".
 *
 * Everything is fp64; bf16 inputs are widened exactly.  Parallelism is plain
 * OpenMP over independent (sequence, head) pairs or token rows; no blocking,
 * fusion or reordering of any sum.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef LRKV_ORACLE_MUTANT
#define LRKV_ORACLE_MUTANT 0 /* planted-mistake builds used by the pin tests */
#endif

/* ---------------------------------------------------------------- scalars */

static double bf(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* fp32 -> bf16, round to nearest with ties to even on the 16 dropped bits. */
static uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u); /* quiet NaN */
    uint32_t keep_lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7fffu + keep_lsb) >> 16);
}

/* fp64 value -> fp32 (round to nearest) -> bf16 (round to nearest even). */
uint16_t oracle_round_to_cache(double v) { return f32_to_bf16((float)v); }

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- softmax */

/* Textbook softmax: p_t = exp(l_t - max) / sum_u exp(l_u - max). */
void oracle_softmax(int n, const double* logits, double* p) {
    if (n <= 0) return;
    double m = logits[0];
    for (int t = 1; t < n; ++t) if (logits[t] > m) m = logits[t];
    double s = 0.0;
    for (int t = 0; t < n; ++t) { p[t] = exp(logits[t] - m); s += p[t]; }
    for (int t = 0; t < n; ++t) p[t] /= s;
}

/* Single-head attention over explicit keys and values:
 *   out = softmax(q K^T * scale) V,  K: [L][dk], V: [L][dv] row-major. */
static void attend_kv(int L, int dk, int dv, const double* q, const double* K, const double* V, double scale,
                      double* out) {
    for (int i = 0; i < dv; ++i) out[i] = 0.0;
    if (L <= 0) return;
    double* logits = (double*)malloc(sizeof(double) * (size_t)L);
    double* p = (double*)malloc(sizeof(double) * (size_t)L);
    for (int t = 0; t < L; ++t) {
        double acc = 0.0;
        for (int i = 0; i < dk; ++i) acc += q[i] * K[(size_t)t * dk + i];
        logits[t] = acc * scale;
    }
    oracle_softmax(L, logits, p);
    for (int t = 0; t < L; ++t)
        for (int i = 0; i < dv; ++i) out[i] += p[t] * V[(size_t)t * dv + i];
    free(logits);
    free(p);
}

void oracle_attend(int L, int d_h, const double* q, const double* K, const double* V,
                   double scale, double* out) {
    attend_kv(L, d_h, d_h, q, K, V, scale, out);
}

/* Rotary position encoding of a d_rope-wide vector at position pos: each pair
 * (2i, 2i+1) is rotated by the angle pos * base^(-2i / d_rope). */
static void rope_rotate(double* v, int d_rope, int pos, double base) {
    for (int i = 0; i < d_rope / 2; ++i) {
#if LRKV_ORACLE_MUTANT == 8
        const double a = -(double)pos * pow(base, -2.0 * i / d_rope); /* planted: rotation reversed */
#else
        const double a = (double)pos * pow(base, -2.0 * i / d_rope);
#endif
        const double c = cos(a), sn = sin(a), x0 = v[2 * i], x1 = v[2 * i + 1];
        v[2 * i] = x0 * c - x1 * sn;
        v[2 * i + 1] = x0 * sn + x1 * c;
    }
}

static double default_scale(double scale, int d_h) {
#if LRKV_ORACLE_MUTANT == 3
    return scale != 0.0 ? scale : 1.0 / (double)d_h; /* planted: wrong scale */
#else
    return scale != 0.0 ? scale : 1.0 / sqrt((double)d_h);
#endif
}

/* Element (i, j) of B_h (d_h x r, row-major [H][d_h][r]). */
static double b_elem(const uint16_t* Bm, int h, int d_h, int r, int i, int j) {
#if LRKV_ORACLE_MUTANT == 6
    /* planted: factor read as if stored transposed ([r][d_h]) */
    return bf(Bm[(size_t)h * d_h * r + (size_t)j * d_h + i]);
#else
    return bf(Bm[((size_t)h * d_h + i) * r + j]);
#endif
}

/* ---------------------------------------------------------------- Eqs. (4)-(5) */

/* Cache contents for n token rows of X [n][d]:
 *   sK = [X W_shared^K | RoPE(X W^KR)], sV = X W_shared^V   -> [n][d_h + d_rope], [n][d_h]
 *   zK[:,h,:] = X U_h^K, zV[:,h,:] = X U_h^V                 -> [n][H][r]
 * The optional decoupled positional key (d_rope > 0; frame "Decoupled RoPE, derived" of
 * the MLA lesson: one small key per token, shared by all heads, that alone carries the
 * rotation) is rotated at the token's position before rounding.
 * Weights: Ws* [d][d_h]; WKR [d][d_rope]; U* [H][d][r].  Each element is an fp64 sum over
 * d, rounded to fp32 and then to bf16 (the reference rounding of the cache). */
void oracle_append_rope(int n, int d, int d_h, int H, int r, int d_rope, double rope_base, const uint16_t* X,
                        const uint16_t* WsK, const uint16_t* WKR, const uint16_t* WsV, const uint16_t* UK,
                        const uint16_t* UV, const int32_t* positions, uint16_t* sK, uint16_t* sV, uint16_t* zK,
                        uint16_t* zV) {
    const int dk = d_h + d_rope;
    #pragma omp parallel for schedule(dynamic)
    for (int t = 0; t < n; ++t) {
        const uint16_t* x = X + (size_t)t * d;
        for (int i = 0; i < d_h; ++i) {
            double ak = 0.0, av = 0.0;
            for (int k = 0; k < d; ++k) {
                ak += bf(x[k]) * bf(WsK[(size_t)k * d_h + i]);
                av += bf(x[k]) * bf(WsV[(size_t)k * d_h + i]);
            }
            sK[(size_t)t * dk + i] = oracle_round_to_cache(ak);
            sV[(size_t)t * d_h + i] = oracle_round_to_cache(av);
        }
        if (d_rope > 0) {
            double kr[256];
            for (int i = 0; i < d_rope && i < 256; ++i) {
                double a = 0.0;
                for (int k = 0; k < d; ++k) a += bf(x[k]) * bf(WKR[(size_t)k * d_rope + i]);
                kr[i] = a;
            }
            rope_rotate(kr, d_rope, positions[t], rope_base);
            for (int i = 0; i < d_rope && i < 256; ++i) sK[(size_t)t * dk + d_h + i] = oracle_round_to_cache(kr[i]);
        }
        for (int h = 0; h < H; ++h)
            for (int j = 0; j < r; ++j) {
                double ak = 0.0, av = 0.0;
                for (int k = 0; k < d; ++k) {
                    ak += bf(x[k]) * bf(UK[((size_t)h * d + k) * r + j]);
                    av += bf(x[k]) * bf(UV[((size_t)h * d + k) * r + j]);
                }
                zK[((size_t)t * H + h) * r + j] = oracle_round_to_cache(ak);
                zV[((size_t)t * H + h) * r + j] = oracle_round_to_cache(av);
            }
    }
}

void oracle_append(int n, int d, int d_h, int H, int r, const uint16_t* X,
                   const uint16_t* WsK, const uint16_t* WsV, const uint16_t* UK, const uint16_t* UV,
                   uint16_t* sK, uint16_t* sV, uint16_t* zK, uint16_t* zV) {
    oracle_append_rope(n, d, d_h, H, r, 0, 0.0, X, WsK, NULL, WsV, UK, UV, NULL, sK, sV, zK, zV);
}

/* ---------------------------------------------------------------- Eqs. (2)-(3) */

/* W_h = W_shared + U_h B_h^T, explicitly, as a d x d_h fp64 matrix. */
static void form_w_h(int d, int d_h, int r, int h, const uint16_t* Ws, const uint16_t* U,
                     const uint16_t* Bm, double* W) {
    for (int k = 0; k < d; ++k)
        for (int i = 0; i < d_h; ++i) {
            double w = bf(Ws[(size_t)k * d_h + i]);
#if LRKV_ORACLE_MUTANT == 5
            w = 0.0; /* planted: shared projection dropped */
#endif
            for (int j = 0; j < r; ++j) {
#if LRKV_ORACLE_MUTANT != 1
                w += bf(U[((size_t)h * d + k) * r + j]) * b_elem(Bm, h, d_h, r, i, j);
#endif
            }
            W[(size_t)k * d_h + i] = w;
        }
}

/* Rows [0, L) of X_b W (X_b: [L][d]) into F [L][d_h]. */
static void project(int L, int d, int d_h, const uint16_t* Xb, const double* W, double* F) {
    for (int t = 0; t < L; ++t)
        for (int i = 0; i < d_h; ++i) {
            double acc = 0.0;
            for (int k = 0; k < d; ++k) acc += bf(Xb[(size_t)t * d + k]) * W[(size_t)k * d_h + i];
            F[(size_t)t * d_h + i] = acc;
        }
}

/* Implied full features from the cache of one token slot:
 *   K_h[t] = s^K_t + B_h^K z^K_{h,t}   (row t of K_s + R_h^K (B_h^K)^T). */
static void expand_from_cache(int d_h, int s_stride, int H, int r, int h, int64_t slot, const uint16_t* s_pool,
                              const uint16_t* z_pool, const uint16_t* Bm, double* row) {
    for (int i = 0; i < d_h; ++i) {
        double v = bf(s_pool[slot * s_stride + i]);
#if LRKV_ORACLE_MUTANT == 5
        v = 0.0;
#endif
        for (int j = 0; j < r; ++j) {
#if LRKV_ORACLE_MUTANT != 1
            v += b_elem(Bm, h, d_h, r, i, j) * bf(z_pool[(slot * H + h) * r + j]);
#endif
        }
        row[i] = v;
    }
}

/* ---------------------------------------------------------------- decode */

/* E1 (expanded from weights).  For each sequence b with ctx_len[b] context
 * rows X[b][0:ctx_len[b]][d] (row stride Lmax*d per sequence) and each head h:
 * form W_h^K and W_h^V, K_h = X W_h^K, V_h = X W_h^V, then
 * out[b][h] = softmax(q[b][h] K_h^T * scale) V_h.
 * want: optional [B][H] mask of the pairs to compute (NULL = all).
 * Returns 0, or -1 for a bad argument. */
int oracle_decode_expanded(int B, int H, int d_h, int r, int d, int Lmax, const int32_t* ctx_len,
                           const uint16_t* X, const uint16_t* WsK, const uint16_t* WsV,
                           const uint16_t* UK, const uint16_t* UV, const uint16_t* BK,
                           const uint16_t* BV, const uint16_t* q, double scale,
                           const uint8_t* want, double* out) {
    for (int b = 0; b < B; ++b)
        if (ctx_len[b] < 0 || ctx_len[b] > Lmax) return -1;
    scale = default_scale(scale, d_h);
    int bad = 0;
    #pragma omp parallel for schedule(dynamic)
    for (int bh = 0; bh < B * H; ++bh) {
        int b = bh / H, h = bh % H;
        if (want && !want[bh]) continue;
        int L = ctx_len[b];
        double* WK = (double*)malloc(sizeof(double) * (size_t)d * d_h);
        double* WV = (double*)malloc(sizeof(double) * (size_t)d * d_h);
        double* K = (double*)malloc(sizeof(double) * (size_t)(L ? L : 1) * d_h);
        double* V = (double*)malloc(sizeof(double) * (size_t)(L ? L : 1) * d_h);
        double qd[512];
        if (!WK || !WV || !K || !V || d_h > 512) {
            #pragma omp atomic write
            bad = 1;
        } else {
            form_w_h(d, d_h, r, h, WsK, UK, BK, WK);
            form_w_h(d, d_h, r, h, WsV, UV, BV, WV);
            const uint16_t* Xb = X + (size_t)b * Lmax * d;
            project(L, d, d_h, Xb, WK, K);
            project(L, d, d_h, Xb, WV, V);
            for (int i = 0; i < d_h; ++i) qd[i] = bf(q[((size_t)b * H + h) * d_h + i]);
            oracle_attend(L, d_h, qd, K, V, scale, out + ((size_t)b * H + h) * d_h);
        }
        free(WK); free(WV); free(K); free(V);
    }
    return bad ? -1 : 0;
}

/* E2 (expanded from the paged cache).  Pools: sK[num_blocks*bs][d_h + d_rope],
 * sV[num_blocks*bs][d_h], z*[num_blocks*bs][H][r]; token t of sequence b lives in slot
 * block_table[b][t / bs] * bs + t % bs.  For each (b, h): materialise
 *   K_h[t] = [s^K_t + B_h^K z^K_{h,t} | k^R_t]   (k^R: the shared positional key, if any)
 *   V_h[t] = s^V_t + B_h^V z^V_{h,t}
 * for t < seq_lens[b] and run textbook attention with q [B][H][d_h + d_rope] at scale
 * 1/sqrt(d_h + d_rope) (the width of the dotted vectors) unless one is given.
 * Returns 0, or -1 when a block id or length is out of range. */
int oracle_decode_cache_rope(int B, int H, int d_h, int r, int d_rope, int bs, int num_blocks,
                             const uint16_t* sK, const uint16_t* sV, const uint16_t* zK, const uint16_t* zV,
                             const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                             const uint16_t* BK, const uint16_t* BV, const uint16_t* q, double scale,
                             const uint8_t* want, double* out) {
    for (int b = 0; b < B; ++b) {
        if (seq_lens[b] < 0 || seq_lens[b] > max_pages * bs) return -1;
        for (int p = 0; p < (seq_lens[b] + bs - 1) / bs; ++p) {
            int32_t blk = block_table[(size_t)b * max_pages + p];
            if (blk < 0 || blk >= num_blocks) return -1;
        }
    }
    const int dk = d_h + d_rope;
#if LRKV_ORACLE_MUTANT == 9
    scale = default_scale(scale, d_h); /* planted: scale of the content width only */
#else
    scale = default_scale(scale, dk);
#endif
    int bad = 0;
    #pragma omp parallel for schedule(dynamic)
    for (int bh = 0; bh < B * H; ++bh) {
        int b = bh / H, h = bh % H;
        if (want && !want[bh]) continue;
        int L = seq_lens[b];
        double* K = (double*)malloc(sizeof(double) * (size_t)(L ? L : 1) * dk);
        double* V = (double*)malloc(sizeof(double) * (size_t)(L ? L : 1) * d_h);
        double qd[768];
        if (!K || !V || dk > 768) {
            #pragma omp atomic write
            bad = 1;
        } else {
            for (int t = 0; t < L; ++t) {
                int64_t slot = (int64_t)block_table[(size_t)b * max_pages + t / bs] * bs + t % bs;
#if LRKV_ORACLE_MUTANT == 2
                expand_from_cache(d_h, dk, H, r, h, slot, sK, zK, BK, K + (size_t)t * dk);
                expand_from_cache(d_h, d_h, H, r, h, slot, sV, zV, BK, V + (size_t)t * d_h); /* planted */
#else
                expand_from_cache(d_h, dk, H, r, h, slot, sK, zK, BK, K + (size_t)t * dk);
                expand_from_cache(d_h, d_h, H, r, h, slot, sV, zV, BV, V + (size_t)t * d_h);
#endif
                for (int i = 0; i < d_rope; ++i) K[(size_t)t * dk + d_h + i] = bf(sK[slot * dk + d_h + i]);
            }
            for (int i = 0; i < dk; ++i) qd[i] = bf(q[((size_t)b * H + h) * dk + i]);
            attend_kv(L, dk, d_h, qd, K, V, scale, out + ((size_t)b * H + h) * d_h);
        }
        free(K); free(V);
    }
    return bad ? -1 : 0;
}

int oracle_decode_cache(int B, int H, int d_h, int r, int bs, int num_blocks,
                        const uint16_t* sK, const uint16_t* sV, const uint16_t* zK, const uint16_t* zV,
                        const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                        const uint16_t* BK, const uint16_t* BV, const uint16_t* q, double scale,
                        const uint8_t* want, double* out) {
    return oracle_decode_cache_rope(B, H, d_h, r, 0, bs, num_blocks, sK, sV, zK, zV, block_table, max_pages,
                                    seq_lens, BK, BV, q, scale, want, out);
}

/* Decode with absorbed weights (both absorptions folded into the caller's projections,
 * frame "Compute logits without expanding historical keys" step 1 and Eq. (7)): the query
 * arrives as [q_h | q~_h] (q~_h = x W_h^Q B_h^K) and the result is returned before the
 * residual up-projection.  Written out plainly, that is single-head softmax attention over
 * concatenated features, with the scale of the (d_h + d_rope)-wide dot product:
 *     keys [s^K_t | k^R_t | z^K_{h,t}],  values [s^V_t | z^V_{h,t}],  query [q_h | q~_h],
 *     out_h = softmax_t(query . key * scale) value
 * (k^R, the shared positional key, is present when d_rope > 0; q_h then carries the
 * caller's rotated positional query in its last d_rope entries).
 * out: [B][H][d_h + r].  Returns 0, or -1 when a block id or length is out of range. */
int oracle_decode_fused_rope(int B, int H, int d_h, int r, int d_rope, int bs, int num_blocks,
                             const uint16_t* sK, const uint16_t* sV, const uint16_t* zK, const uint16_t* zV,
                             const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                             const uint16_t* q, const uint16_t* qt, double scale, const uint8_t* want,
                             double* out) {
    for (int b = 0; b < B; ++b) {
        if (seq_lens[b] < 0 || seq_lens[b] > max_pages * bs) return -1;
        for (int p = 0; p < (seq_lens[b] + bs - 1) / bs; ++p) {
            int32_t blk = block_table[(size_t)b * max_pages + p];
            if (blk < 0 || blk >= num_blocks) return -1;
        }
    }
    const int ds = d_h + d_rope;      /* shared key width */
    const int wk = ds + r, wv = d_h + r;
    scale = default_scale(scale, ds);
    int bad = 0;
    #pragma omp parallel for schedule(dynamic)
    for (int bh = 0; bh < B * H; ++bh) {
        int b = bh / H, h = bh % H;
        if (want && !want[bh]) continue;
        int L = seq_lens[b];
        double* K = (double*)malloc(sizeof(double) * (size_t)(L ? L : 1) * wk);
        double* V = (double*)malloc(sizeof(double) * (size_t)(L ? L : 1) * wv);
        double* qc = (double*)malloc(sizeof(double) * (size_t)wk);
        if (!K || !V || !qc) {
            #pragma omp atomic write
            bad = 1;
        } else {
            for (int t = 0; t < L; ++t) {
                int64_t slot = (int64_t)block_table[(size_t)b * max_pages + t / bs] * bs + t % bs;
                for (int i = 0; i < ds; ++i) K[(size_t)t * wk + i] = bf(sK[slot * ds + i]);
                for (int i = 0; i < d_h; ++i) V[(size_t)t * wv + i] = bf(sV[slot * d_h + i]);
                for (int j = 0; j < r; ++j) {
                    K[(size_t)t * wk + ds + j] = bf(zK[(slot * H + h) * r + j]);
#if LRKV_ORACLE_MUTANT == 7
                    V[(size_t)t * wv + d_h + j] = 0.0; /* planted: residual values dropped */
#else
                    V[(size_t)t * wv + d_h + j] = bf(zV[(slot * H + h) * r + j]);
#endif
                }
            }
            for (int i = 0; i < ds; ++i) qc[i] = bf(q[((size_t)b * H + h) * ds + i]);
            for (int j = 0; j < r; ++j) qc[ds + j] = bf(qt[((size_t)b * H + h) * r + j]);
            attend_kv(L, wk, wv, qc, K, V, scale, out + ((size_t)b * H + h) * wv);
        }
        free(K); free(V); free(qc);
    }
    return bad ? -1 : 0;
}

int oracle_decode_fused(int B, int H, int d_h, int r, int bs, int num_blocks,
                        const uint16_t* sK, const uint16_t* sV, const uint16_t* zK, const uint16_t* zV,
                        const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                        const uint16_t* q, const uint16_t* qt, double scale, const uint8_t* want, double* out) {
    return oracle_decode_fused_rope(B, H, d_h, r, 0, bs, num_blocks, sK, sV, zK, zV, block_table, max_pages,
                                    seq_lens, q, qt, scale, want, out);
}

/* ---------------------------------------------------------------- prefill */

/* Causal limit: query at absolute position pos sees keys j <= pos. */
static int visible(int pos) {
#if LRKV_ORACLE_MUTANT == 4
    return pos; /* planted: diagonal excluded */
#else
    return pos + 1;
#endif
}

/* E1 causal prefill.  Queries q[b][i][h][d_h] for i < Tq sit at absolute
 * positions q_start[b] + i; context rows X[b][0:q_start[b]+Tq][d] (stride
 * Lmax*d).  out[b][i][h] = softmax over keys j <= q_start[b]+i. */
int oracle_prefill_expanded(int B, int Tq, int H, int d_h, int r, int d, int Lmax,
                            const int32_t* q_start, const uint16_t* X, const uint16_t* WsK,
                            const uint16_t* WsV, const uint16_t* UK, const uint16_t* UV,
                            const uint16_t* BK, const uint16_t* BV, const uint16_t* q,
                            double scale, const uint8_t* want, double* out) {
    for (int b = 0; b < B; ++b)
        if (q_start[b] < 0 || q_start[b] + Tq > Lmax) return -1;
    scale = default_scale(scale, d_h);
    int bad = 0;
    #pragma omp parallel for schedule(dynamic)
    for (int bh = 0; bh < B * H; ++bh) {
        int b = bh / H, h = bh % H;
        if (want && !want[bh]) continue;
        int L = q_start[b] + Tq;
        double* WK = (double*)malloc(sizeof(double) * (size_t)d * d_h);
        double* WV = (double*)malloc(sizeof(double) * (size_t)d * d_h);
        double* K = (double*)malloc(sizeof(double) * (size_t)(L ? L : 1) * d_h);
        double* V = (double*)malloc(sizeof(double) * (size_t)(L ? L : 1) * d_h);
        double qd[512];
        if (!WK || !WV || !K || !V || d_h > 512) {
            #pragma omp atomic write
            bad = 1;
        } else {
            form_w_h(d, d_h, r, h, WsK, UK, BK, WK);
            form_w_h(d, d_h, r, h, WsV, UV, BV, WV);
            const uint16_t* Xb = X + (size_t)b * Lmax * d;
            project(L, d, d_h, Xb, WK, K);
            project(L, d, d_h, Xb, WV, V);
            for (int i = 0; i < Tq; ++i) {
                const uint16_t* qi = q + (((size_t)b * Tq + i) * H + h) * d_h;
                for (int c = 0; c < d_h; ++c) qd[c] = bf(qi[c]);
                oracle_attend(visible(q_start[b] + i), d_h, qd, K, V, scale,
                              out + (((size_t)b * Tq + i) * H + h) * d_h);
            }
        }
        free(WK); free(WV); free(K); free(V);
    }
    return bad ? -1 : 0;
}

/* E2 causal prefill from the paged cache (layout as oracle_decode_cache_rope): query i of
 * sequence b, at absolute position q_start[b] + i, attends to keys j <= that position.
 * q [B][Tq][H][d_h + d_rope] (the positional part already rotated by the caller). */
int oracle_prefill_cache_rope(int B, int Tq, int H, int d_h, int r, int d_rope, int bs, int num_blocks,
                              const uint16_t* sK, const uint16_t* sV, const uint16_t* zK,
                              const uint16_t* zV, const int32_t* block_table, int max_pages,
                              const int32_t* q_start, const uint16_t* BK, const uint16_t* BV,
                              const uint16_t* q, double scale, const uint8_t* want, double* out) {
    for (int b = 0; b < B; ++b) {
        int L = q_start[b] + Tq;
        if (q_start[b] < 0 || L > max_pages * bs) return -1;
        for (int p = 0; p < (L + bs - 1) / bs; ++p) {
            int32_t blk = block_table[(size_t)b * max_pages + p];
            if (blk < 0 || blk >= num_blocks) return -1;
        }
    }
    const int dk = d_h + d_rope;
    scale = default_scale(scale, dk);
    int bad = 0;
    #pragma omp parallel for schedule(dynamic)
    for (int bh = 0; bh < B * H; ++bh) {
        int b = bh / H, h = bh % H;
        if (want && !want[bh]) continue;
        int L = q_start[b] + Tq;
        double* K = (double*)malloc(sizeof(double) * (size_t)(L ? L : 1) * dk);
        double* V = (double*)malloc(sizeof(double) * (size_t)(L ? L : 1) * d_h);
        double qd[768];
        if (!K || !V || dk > 768) {
            #pragma omp atomic write
            bad = 1;
        } else {
            for (int t = 0; t < L; ++t) {
                int64_t slot = (int64_t)block_table[(size_t)b * max_pages + t / bs] * bs + t % bs;
                expand_from_cache(d_h, dk, H, r, h, slot, sK, zK, BK, K + (size_t)t * dk);
                expand_from_cache(d_h, d_h, H, r, h, slot, sV, zV, BV, V + (size_t)t * d_h);
                for (int c = 0; c < d_rope; ++c) K[(size_t)t * dk + d_h + c] = bf(sK[slot * dk + d_h + c]);
            }
            for (int i = 0; i < Tq; ++i) {
                const uint16_t* qi = q + (((size_t)b * Tq + i) * H + h) * dk;
                for (int c = 0; c < dk; ++c) qd[c] = bf(qi[c]);
                attend_kv(visible(q_start[b] + i), dk, d_h, qd, K, V, scale,
                          out + (((size_t)b * Tq + i) * H + h) * d_h);
            }
        }
        free(K); free(V);
    }
    return bad ? -1 : 0;
}

int oracle_prefill_cache(int B, int Tq, int H, int d_h, int r, int bs, int num_blocks,
                         const uint16_t* sK, const uint16_t* sV, const uint16_t* zK,
                         const uint16_t* zV, const int32_t* block_table, int max_pages,
                         const int32_t* q_start, const uint16_t* BK, const uint16_t* BV,
                         const uint16_t* q, double scale, const uint8_t* want, double* out) {
    return oracle_prefill_cache_rope(B, Tq, H, d_h, r, 0, bs, num_blocks, sK, sV, zK, zV, block_table, max_pages,
                                     q_start, BK, BV, q, scale, want, out);
}

/* E2 causal prefill with absorbed weights (the associativity of the LRKV slides' frame
 * "Compute logits without expanding historical keys" and of Eq. (7), applied to a chunk of
 * queries): query i of sequence b, at absolute position q_start[b] + i, brings q~_i = q_i B_h^K
 * already projected, and head h returns the aggregate before the residual up-projection,
 *     out = sum_{j <= q_start[b] + i} p_j [s^V_j | z^V_{h,j}],
 *     p = softmax_j([q_i | q~_i] . [s^K_j | z^K_{h,j}] * scale)
 * i.e. causal single-head attention over the concatenated features (with a positional key,
 * [q | q^R | q~] . [s^K | k^R | z^K_h]).  q [B][Tq][H][d_h + d_rope], qt [B][Tq][H][r],
 * out [B][Tq][H][d_h + r].  Returns 0, or -1 when a block id or length is out of range. */
int oracle_prefill_fused_rope(int B, int Tq, int H, int d_h, int r, int d_rope, int bs, int num_blocks,
                              const uint16_t* sK, const uint16_t* sV, const uint16_t* zK,
                              const uint16_t* zV, const int32_t* block_table, int max_pages,
                              const int32_t* q_start, const uint16_t* q, const uint16_t* qt, double scale,
                              const uint8_t* want, double* out) {
    for (int b = 0; b < B; ++b) {
        int L = q_start[b] + Tq;
        if (q_start[b] < 0 || L > max_pages * bs) return -1;
        for (int p = 0; p < (L + bs - 1) / bs; ++p) {
            int32_t blk = block_table[(size_t)b * max_pages + p];
            if (blk < 0 || blk >= num_blocks) return -1;
        }
    }
    const int ds = d_h + d_rope;      /* shared key width */
    const int wk = ds + r, wv = d_h + r;
    scale = default_scale(scale, ds);
    int bad = 0;
    #pragma omp parallel for schedule(dynamic)
    for (int bh = 0; bh < B * H; ++bh) {
        int b = bh / H, h = bh % H;
        if (want && !want[bh]) continue;
        int L = q_start[b] + Tq;
        double* K = (double*)malloc(sizeof(double) * (size_t)(L ? L : 1) * wk);
        double* V = (double*)malloc(sizeof(double) * (size_t)(L ? L : 1) * wv);
        double* qc = (double*)malloc(sizeof(double) * (size_t)wk);
        if (!K || !V || !qc) {
            #pragma omp atomic write
            bad = 1;
        } else {
            for (int t = 0; t < L; ++t) {
                int64_t slot = (int64_t)block_table[(size_t)b * max_pages + t / bs] * bs + t % bs;
                for (int i = 0; i < ds; ++i) K[(size_t)t * wk + i] = bf(sK[slot * ds + i]);
                for (int i = 0; i < d_h; ++i) V[(size_t)t * wv + i] = bf(sV[slot * d_h + i]);
                for (int j = 0; j < r; ++j) {
                    K[(size_t)t * wk + ds + j] = bf(zK[(slot * H + h) * r + j]);
                    V[(size_t)t * wv + d_h + j] = bf(zV[(slot * H + h) * r + j]);
                }
            }
            for (int i = 0; i < Tq; ++i) {
                const size_t row = ((size_t)b * Tq + i) * H + h;
                for (int c = 0; c < ds; ++c) qc[c] = bf(q[row * ds + c]);
#if LRKV_ORACLE_MUTANT == 13
                /* planted: q~ of the next head */
                for (int j = 0; j < r; ++j) qc[ds + j] = bf(qt[(row - h + (h + 1) % H) * r + j]);
#else
                for (int j = 0; j < r; ++j) qc[ds + j] = bf(qt[row * r + j]);
#endif
                attend_kv(visible(q_start[b] + i), wk, wv, qc, K, V, scale, out + row * wv);
            }
        }
        free(K); free(V); free(qc);
    }
    return bad ? -1 : 0;
}

/* ---------------------------------------------------------------- MLA, absorbed and expanded */
/*
 * Multi-head latent attention as the MLA lesson ("Embeddings II: MLA & Architectural
 * Choices") builds it, in the associative form of the LRKV slides' backup frame "MLA
 * also admits associative computation": per token the cache holds the latent
 * c_t = x_t W^DKV (width d_c) and the decoupled positional key k^R_t (width d_rope, shared
 * by all heads, rotated at the token's position), stored as one row [c_t | k^R_t].
 * Head i's key and value are k_{i,t} = [c_t W^UK_i | k^R_t] and v_{i,t} = c_t W^UV_i
 * (W^UK_i, W^UV_i: d_c x d_head), its query [q^C_i | q^R_i], and the logit scale
 * 1/sqrt(d_head + d_rope) -- the width of the vectors actually dotted (section
 * "the softmax denominator changes too").
 */

/* Absorbed: W^UK_i folded into the query (q~_i = q^C_i (W^UK_i)^T, width d_c) and W^UV_i into
 * the output projection, so head i attends with [q~_i | q^R_i] against the cache rows and
 * returns o_i = sum_t p_t c_t (width d_c), before W^UV_i.
 *   kv [num_blocks][bs][d_c + d_rope], q [B][H][d_c + d_rope], out [B][H][d_c]. */
int oracle_mla_decode(int B, int H, int d_c, int d_rope, int d_head, int bs, int num_blocks, const uint16_t* kv,
                      const int32_t* block_table, int max_pages, const int32_t* seq_lens, const uint16_t* q,
                      double scale, const uint8_t* want, double* out) {
    for (int b = 0; b < B; ++b) {
        if (seq_lens[b] < 0 || seq_lens[b] > max_pages * bs) return -1;
        for (int p = 0; p < (seq_lens[b] + bs - 1) / bs; ++p) {
            int32_t blk = block_table[(size_t)b * max_pages + p];
            if (blk < 0 || blk >= num_blocks) return -1;
        }
    }
    const int dk = d_c + d_rope;
    if (dk > 1024) return -1;
#if LRKV_ORACLE_MUTANT == 10
    scale = default_scale(scale, dk); /* planted: scale over the cached row's width */
#else
    scale = default_scale(scale, d_head + d_rope);
#endif
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        int L = seq_lens[b];
        double* K = (double*)malloc(sizeof(double) * (size_t)(L ? L : 1) * dk);
        double* V = (double*)malloc(sizeof(double) * (size_t)(L ? L : 1) * d_c);
        if (!K || !V) {
            bad = 1;
        } else {
            for (int t = 0; t < L; ++t) {
                int64_t slot = (int64_t)block_table[(size_t)b * max_pages + t / bs] * bs + t % bs;
                for (int i = 0; i < dk; ++i) K[(size_t)t * dk + i] = bf(kv[slot * dk + i]);
#if LRKV_ORACLE_MUTANT == 11
                for (int i = 0; i < d_c; ++i) V[(size_t)t * d_c + i] = bf(kv[slot * dk + d_rope + i]); /* planted */
#else
                for (int i = 0; i < d_c; ++i) V[(size_t)t * d_c + i] = bf(kv[slot * dk + i]);
#endif
            }
            /* heads are independent: one query row each against the same keys and values */
            #pragma omp parallel for schedule(dynamic)
            for (int h = 0; h < H; ++h) {
                if (want && !want[(size_t)b * H + h]) continue;
                double qd[1024];
                for (int i = 0; i < dk && i < 1024; ++i) qd[i] = bf(q[((size_t)b * H + h) * dk + i]);
                attend_kv(L, dk, d_c, qd, K, V, scale, out + ((size_t)b * H + h) * d_c);
            }
        }
        free(K); free(V);
    }
    return bad ? -1 : 0;
}

/* Expanded ("reconstruct, then attend"): per head the full keys and values are formed from
 * the cached rows and the up-projections, then textbook attention.
 *   rows [B][Lmax][d_c + d_rope], qC [B][H][d_head], qR [B][H][d_rope],
 *   WUK, WUV [H][d_c][d_head], out [B][H][d_head]. */
int oracle_mla_decode_expanded(int B, int H, int d_c, int d_rope, int d_head, int Lmax, const int32_t* ctx_len,
                               const uint16_t* rows, const uint16_t* qC, const uint16_t* qR, const uint16_t* WUK,
                               const uint16_t* WUV, double scale, double* out) {
    for (int b = 0; b < B; ++b)
        if (ctx_len[b] < 0 || ctx_len[b] > Lmax) return -1;
    const int dk = d_c + d_rope, wk = d_head + d_rope;
    scale = default_scale(scale, wk);
    int bad = 0;
    #pragma omp parallel for schedule(dynamic)
    for (int bh = 0; bh < B * H; ++bh) {
        int b = bh / H, h = bh % H, L = ctx_len[b];
        double* K = (double*)malloc(sizeof(double) * (size_t)(L ? L : 1) * wk);
        double* V = (double*)malloc(sizeof(double) * (size_t)(L ? L : 1) * d_head);
        double* qd = (double*)malloc(sizeof(double) * (size_t)wk);
        if (!K || !V || !qd) {
            #pragma omp atomic write
            bad = 1;
        } else {
            for (int t = 0; t < L; ++t) {
                const uint16_t* row = rows + ((size_t)b * Lmax + t) * dk;
                for (int e = 0; e < d_head; ++e) {
                    double ak = 0.0, av = 0.0;
                    for (int c = 0; c < d_c; ++c) {
                        ak += bf(row[c]) * bf(WUK[((size_t)h * d_c + c) * d_head + e]);
                        av += bf(row[c]) * bf(WUV[((size_t)h * d_c + c) * d_head + e]);
                    }
                    K[(size_t)t * wk + e] = ak;
                    V[(size_t)t * d_head + e] = av;
                }
                for (int e = 0; e < d_rope; ++e) K[(size_t)t * wk + d_head + e] = bf(row[d_c + e]);
            }
            for (int e = 0; e < d_head; ++e) qd[e] = bf(qC[((size_t)b * H + h) * d_head + e]);
            for (int e = 0; e < d_rope; ++e) qd[d_head + e] = bf(qR[((size_t)b * H + h) * d_rope + e]);
            attend_kv(L, wk, d_head, qd, K, V, scale, out + ((size_t)b * H + h) * d_head);
        }
        free(K); free(V); free(qd);
    }
    return bad ? -1 : 0;
}

/* ---------------------------------------------------------------- training: expanded projections */
/*
 * "Low-Rank Key Value Attention", frame "Training learns the base and residuals together":
 * during training the full per-head features are materialised, K_h = X W_h with
 * W_h = W_shared + U_h B_h^T (Eqs. (2)-(3)), and the base and residual factors receive
 * gradients through that product.  Forward and backward of one such projection (keys or
 * values alike), by the plain definition and the chain rule:
 *   K_h    = X W_h                          [n][H][d_h]
 *   dX     = sum_h dK_h W_h^T               [n][d]
 *   dW_s   = X^T sum_h dK_h                 [d][d_h]
 *   dU_h   = X^T (dK_h B_h)                 [H][d][r]
 *   dB_h   = dK_h^T (X U_h)                 [H][d_h][r]
 * X [n][d], Ws [d][d_h], U [H][d][r], B [H][d_h][r], dK [n][H][d_h] (bf16); outputs fp64.
 */
void oracle_train_forward(int n, int d, int d_h, int H, int r, const uint16_t* X, const uint16_t* Ws,
                          const uint16_t* U, const uint16_t* Bm, double* K) {
    #pragma omp parallel for schedule(dynamic)
    for (int h = 0; h < H; ++h) {
        double* W = (double*)malloc(sizeof(double) * (size_t)d * d_h);
        double* F = (double*)malloc(sizeof(double) * (size_t)n * d_h);
        if (W && F) {
            form_w_h(d, d_h, r, h, Ws, U, Bm, W);
            project(n, d, d_h, X, W, F);
            for (int t = 0; t < n; ++t)
                for (int i = 0; i < d_h; ++i) K[((size_t)t * H + h) * d_h + i] = F[(size_t)t * d_h + i];
        }
        free(W); free(F);
    }
}

void oracle_train_backward(int n, int d, int d_h, int H, int r, const uint16_t* X, const uint16_t* Ws,
                           const uint16_t* U, const uint16_t* Bm, const uint16_t* dK, double* dX, double* dWs,
                           double* dU, double* dB) {
    /* dX = sum_h dK_h W_h^T, with W_h formed explicitly */
    for (size_t i = 0; i < (size_t)n * d; ++i) dX[i] = 0.0;
    double* W = (double*)malloc(sizeof(double) * (size_t)d * d_h);
    for (int h = 0; h < H && W; ++h) {
        form_w_h(d, d_h, r, h, Ws, U, Bm, W);
        #pragma omp parallel for schedule(static)
        for (int t = 0; t < n; ++t)
            for (int k = 0; k < d; ++k) {
                double acc = 0.0;
                for (int i = 0; i < d_h; ++i) acc += bf(dK[((size_t)t * H + h) * d_h + i]) * W[(size_t)k * d_h + i];
                dX[(size_t)t * d + k] += acc;
            }
    }
    free(W);
    /* dW_s = X^T sum_h dK_h */
    #pragma omp parallel for schedule(static)
    for (int k = 0; k < d; ++k)
        for (int i = 0; i < d_h; ++i) {
            double acc = 0.0;
            for (int t = 0; t < n; ++t) {
                double g = 0.0;
                for (int h = 0; h < H; ++h) g += bf(dK[((size_t)t * H + h) * d_h + i]);
                acc += bf(X[(size_t)t * d + k]) * g;
            }
            dWs[(size_t)k * d_h + i] = acc;
        }
    /* dU_h = X^T (dK_h B_h),  dB_h = dK_h^T (X U_h) */
    #pragma omp parallel for schedule(dynamic)
    for (int h = 0; h < H; ++h) {
        double* dR = (double*)malloc(sizeof(double) * (size_t)n * r);
        double* R = (double*)malloc(sizeof(double) * (size_t)n * r);
        if (dR && R) {
            for (int t = 0; t < n; ++t)
                for (int j = 0; j < r; ++j) {
                    double a = 0.0, c = 0.0;
                    for (int i = 0; i < d_h; ++i) a += bf(dK[((size_t)t * H + h) * d_h + i]) * b_elem(Bm, h, d_h, r, i, j);
                    for (int k = 0; k < d; ++k) c += bf(X[(size_t)t * d + k]) * bf(U[((size_t)h * d + k) * r + j]);
                    dR[(size_t)t * r + j] = a;
                    R[(size_t)t * r + j] = c;
                }
            for (int k = 0; k < d; ++k)
                for (int j = 0; j < r; ++j) {
                    double acc = 0.0;
                    for (int t = 0; t < n; ++t) acc += bf(X[(size_t)t * d + k]) * dR[(size_t)t * r + j];
                    dU[((size_t)h * d + k) * r + j] = acc;
                }
            for (int i = 0; i < d_h; ++i)
                for (int j = 0; j < r; ++j) {
                    double acc = 0.0;
#if LRKV_ORACLE_MUTANT == 12
                    for (int t = 0; t < n; ++t) acc += bf(dK[((size_t)t * H + h) * d_h + i]) * dR[(size_t)t * r + j]; /* planted */
#else
                    for (int t = 0; t < n; ++t) acc += bf(dK[((size_t)t * H + h) * d_h + i]) * R[(size_t)t * r + j];
#endif
                    dB[((size_t)h * d_h + i) * r + j] = acc;
                }
        }
        free(dR); free(R);
    }
}
