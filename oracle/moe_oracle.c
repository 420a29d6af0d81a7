/*
 * Plain fp64 CPU oracle for the W4A16 routed-expert MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY. It exists to check the CUDA library, and only the
 * tests, the entry module's smoke check and the benchmark's CPU-baseline leg
 * may load it. It shares no code, header or table with the CUDA path.
 *
 * Each function writes out the plain definition of one step, with no
 * blocking, fusion or reordering beyond that definition:
 *
 *   weights  - symmetric INT4, group size 128 along K, "pack-quantized":
 *              eight values per int32, lowest nibble first, each stored as
 *              q + 8 so that q lies in [-8, 7]; one bf16 scale per row and
 *              128-wide K group; W = q * scale.
 *              (model card "Minachist/Qwen3.8-Flash-Next-INT4-Mixed-AutoRound",
 *              "What is quantized", group A; the int8 analogue of the packing,
 *              four values per word, least significant first, stored as
 *              value + 128, is in "Running 125B MoE on Three 3090s - vLLM
 *              Optimization Edition", section 3.3 "Hyper-connection".)
 *   routing  - logits = x . Wr^T (+ bias); softmax over all experts; the k
 *              largest logits are selected, ties going to the lower expert id;
 *              the selected probabilities are renormalised to sum to one.
 *              (Optimization Edition, section 3.3 "MoE block": the router GEMV,
 *              topk_softmax, norm_topk_prob, and the lower-id tie rule.)
 *   permute  - per-expert counts, exclusive prefix sum, and the assignments
 *              (t, j) listed expert by expert in increasing t*k + j.
 *              (section 3.3: moe_align_block_size, here without padding.)
 *   experts  - per assignment: g = W1[0:I] x, u = W1[I:2I] x,
 *              h = SiLU(g) * u, y = W2 h; out[t] += w_j * y.
 *              (section 3.3: fused Marlin MoE gate_up, SiluAndMul, down,
 *              moe_sum.)
 *   stack    - next layer input = bf16(r / sqrt(mean(r^2) + eps)), r = x + out.
 *   shared   - the shared expert beside the routed ones: its gate logit
 *              g = x . wg is one more row of the router GEMV, and the layer
 *              output is routed + sigmoid(g) * SwiGLU_shared(x).
 *              (section 3.3 "MoE block": the router and the shared expert gate
 *              as one GEMV of 512 + 1 rows; the final combine, routed +
 *              sigmoid(gate) x shared.)
 *   W8A16    - INT8 weights, four per int32 word, least significant byte
 *              first, stored as q + 128, one bf16 scale per 64 or 128 values
 *              of a row; y = x . W^T. (section 3.3 "Hyper-connection
 *              (decode-04)": the INT8 GEMVs and the W8A16 GEMM; model card
 *              "What is quantized", groups C and D.)
 *   quantise - round-to-nearest INT4, group size 128, symmetric, with a
 *              per-group search for the clip that minimises the squared error.
 *              (section 7 "Putting MTP on the GPU": make_mtp_int4.py.)
 *
 * Parity of the expert outputs themselves is pinned only by brute force,
 * closed forms and invariants in the tests; the pages print no worked example
 * of output values.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_GROUP 128

/* bf16 bit pattern -> double (exact). */
static double bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* double -> float (round to nearest even) -> bf16 (round to nearest even). */
static uint16_t f64_to_bf16(double v)
{
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) /* NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- INT4 storage ------------------------------------------------------- */

/* q[n][c] in [-8, 7] from packed[n][c/8]: nibble c%8 of the word, minus 8. */
void oracle_unpack_int4(const int32_t *packed, int64_t N, int64_t K, int8_t *q)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t c = 0; c < K; ++c) {
            uint32_t word = (uint32_t)packed[n * (K / 8) + c / 8];
            int nib = (int)((word >> (4 * (c % 8))) & 0xFu);
            q[n * K + c] = (int8_t)(nib - 8);
        }
}

/* Inverse of oracle_unpack_int4. Returns -1 if some q lies outside [-8, 7]. */
int oracle_pack_int4(const int8_t *q, int64_t N, int64_t K, int32_t *packed)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t w = 0; w < K / 8; ++w) {
            uint32_t word = 0;
            for (int i = 0; i < 8; ++i) {
                int v = q[n * K + w * 8 + i];
                if (v < -8 || v > 7) return -1;
                word |= (uint32_t)(v + 8) << (4 * i);
            }
            packed[n * (K / 8) + w] = (int32_t)word;
        }
    return 0;
}

/* One dequantised weight: W[n][c] = q[n][c] * scale[n][c / 128]. */
static double weight(const int32_t *packed, const uint16_t *scales, int64_t K,
                     int64_t n, int64_t c)
{
    uint32_t word = (uint32_t)packed[n * (K / 8) + c / 8];
    int q = (int)((word >> (4 * (c % 8))) & 0xFu) - 8;
    return (double)q * bf16_to_f64(scales[n * (K / ORACLE_GROUP) + c / ORACLE_GROUP]);
}

/* W[N][K] in fp64. */
void oracle_dequant(const int32_t *packed, const uint16_t *scales, int64_t N,
                    int64_t K, double *W)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t c = 0; c < K; ++c) W[n * K + c] = weight(packed, scales, K, n, c);
}

/* ---- routing ------------------------------------------------------------ */

/* logits[t][e] = sum_h x[t][h] * Wr[e][h] (+ bias[e]); bias may be NULL. */
void oracle_router_logits(const uint16_t *x, const uint16_t *wr, const float *bias,
                          int T, int H, int E, double *logits, int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double s = 0.0;
            for (int h = 0; h < H; ++h)
                s += bf16_to_f64(x[(int64_t)t * H + h]) * bf16_to_f64(wr[(int64_t)e * H + h]);
            if (bias) s += (double)bias[e];
            logits[(int64_t)t * E + e] = s;
        }
}

/*
 * From logits [T][E]: ids [T][k] in order of descending logit (ties: lower
 * id first) and weights [T][k] = p_id / sum over the selected p, p being the
 * softmax over all E experts. Returns -1 if k > E.
 */
int oracle_topk_softmax(const double *logits, int T, int E, int k, int32_t *ids,
                        double *w)
{
    if (k > E || k <= 0) return -1;
    char *taken = (char *)malloc((size_t)E);
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    if (!taken || !p) { free(taken); free(p); return -2; }
    for (int t = 0; t < T; ++t) {
        const double *l = logits + (int64_t)t * E;
        double mx = l[0];
        for (int e = 1; e < E; ++e) if (l[e] > mx) mx = l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) { p[e] = exp(l[e] - mx); z += p[e]; }
        for (int e = 0; e < E; ++e) p[e] /= z;

        memset(taken, 0, (size_t)E);
        double psel = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e; /* strict: ties keep the lower id */
            }
            taken[best] = 1;
            ids[(int64_t)t * k + j] = best;
            psel += p[best];
        }
        for (int j = 0; j < k; ++j) w[(int64_t)t * k + j] = p[ids[(int64_t)t * k + j]] / psel;
    }
    free(taken);
    free(p);
    return 0;
}

/* ---- permute ------------------------------------------------------------ */

/*
 * offsets[E+1]: exclusive prefix sum of per-expert counts;
 * perm[T*k]: assignment indices a = t*k + j grouped by expert, increasing a
 * within an expert. Returns -1 on an id outside [0, E).
 */
int oracle_permute(const int32_t *ids, int T, int k, int E, int32_t *offsets,
                   int32_t *perm)
{
    int64_t n = (int64_t)T * k;
    for (int e = 0; e <= E; ++e) offsets[e] = 0;
    for (int64_t a = 0; a < n; ++a) {
        if (ids[a] < 0 || ids[a] >= E) return -1;
        offsets[ids[a] + 1] += 1;
    }
    for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    if (!cursor) return -2;
    for (int e = 0; e < E; ++e) cursor[e] = offsets[e];
    for (int64_t a = 0; a < n; ++a) perm[cursor[ids[a]]++] = (int32_t)a;
    free(cursor);
    return 0;
}

/* ---- experts ------------------------------------------------------------ */

/*
 * out[T][H] = sum_j topk_w[t][j] * W2[e] (SiLU(W1[e][0:I] x_t) * W1[e][I:2I] x_t),
 * e = ids[t][j].
 *
 * Weight arrays hold `n_held` experts; expert e is found at row
 * expert_row[e] of them (expert_row may be NULL: row e). Returns -1 if an id
 * is outside [0, E) or its expert is not held.
 *
 * Layouts: x bf16 [T][H]; w1_packed int32 [n_held][2I][H/8];
 * w1_scales bf16 [n_held][2I][H/128]; w2_packed int32 [n_held][H][I/8];
 * w2_scales bf16 [n_held][H][I/128].
 */
int oracle_expert_forward(const uint16_t *x, const int32_t *ids, const float *topk_w,
                          const int32_t *w1_packed, const uint16_t *w1_scales,
                          const int32_t *w2_packed, const uint16_t *w2_scales,
                          const int32_t *expert_row, int n_held,
                          int T, int H, int E, int k, int I, double *out, int nthreads)
{
    for (int64_t a = 0; a < (int64_t)T * k; ++a) {
        int e = ids[a];
        if (e < 0 || e >= E) return -1;
        int r = expert_row ? expert_row[e] : e;
        if (r < 0 || r >= n_held) return -1;
    }
    const int64_t w1_rows = 2 * (int64_t)I, w2_rows = H;
    const int64_t w1_words = w1_rows * (H / 8), w1_groups = w1_rows * (H / ORACLE_GROUP);
    const int64_t w2_words = w2_rows * (I / 8), w2_groups = w2_rows * (I / ORACLE_GROUP);
    int failed = 0;
    set_threads(nthreads);
#pragma omp parallel
    {
        double *xt = (double *)malloc(sizeof(double) * (size_t)H);
        double *h = (double *)malloc(sizeof(double) * (size_t)I);
        if (!xt || !h) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic)
            for (int t = 0; t < T; ++t) {
                for (int c = 0; c < H; ++c) xt[c] = bf16_to_f64(x[(int64_t)t * H + c]);
                double *o = out + (int64_t)t * H;
                for (int n = 0; n < H; ++n) o[n] = 0.0;
                for (int j = 0; j < k; ++j) {
                    int e = ids[(int64_t)t * k + j];
                    int r = expert_row ? expert_row[e] : e;
                    const int32_t *p1 = w1_packed + r * w1_words;
                    const uint16_t *s1 = w1_scales + r * w1_groups;
                    const int32_t *p2 = w2_packed + r * w2_words;
                    const uint16_t *s2 = w2_scales + r * w2_groups;
                    for (int i = 0; i < I; ++i) {
                        double g = 0.0, u = 0.0;
                        for (int c = 0; c < H; ++c) {
                            g += weight(p1, s1, H, i, c) * xt[c];
                            u += weight(p1, s1, H, (int64_t)I + i, c) * xt[c];
                        }
                        h[i] = g / (1.0 + exp(-g)) * u;
                    }
                    double wj = (double)topk_w[(int64_t)t * k + j];
                    for (int n = 0; n < H; ++n) {
                        double y = 0.0;
                        for (int i = 0; i < I; ++i) y += weight(p2, s2, I, n, i) * h[i];
                        o[n] += wj * y;
                    }
                }
            }
        }
        free(xt);
        free(h);
    }
    return failed ? -2 : 0;
}

/* ---- stack -------------------------------------------------------------- */

/*
 * Next layer input of the 48-layer stack: r = x + out,
 * x_next = bf16(r / sqrt(mean_h(r^2) + eps)) (no learned weight).
 * Writes the bf16 bits to x_next and, if x_next_f64 is not NULL, the value
 * before rounding.
 */
void oracle_residual_rms(const uint16_t *x, const double *out, int T, int H, double eps,
                         uint16_t *x_next, double *x_next_f64)
{
    for (int t = 0; t < T; ++t) {
        double ss = 0.0;
        for (int c = 0; c < H; ++c) {
            double r = bf16_to_f64(x[(int64_t)t * H + c]) + out[(int64_t)t * H + c];
            ss += r * r;
        }
        double inv = 1.0 / sqrt(ss / H + eps);
        for (int c = 0; c < H; ++c) {
            double r = bf16_to_f64(x[(int64_t)t * H + c]) + out[(int64_t)t * H + c];
            double v = r * inv;
            x_next[(int64_t)t * H + c] = f64_to_bf16(v);
            if (x_next_f64) x_next_f64[(int64_t)t * H + c] = v;
        }
    }
}

/* bf16 rounding of doubles through float, for tests of the helper itself. */
void oracle_round_bf16(const double *v, int64_t n, uint16_t *bits)
{
    for (int64_t i = 0; i < n; ++i) bits[i] = f64_to_bf16(v[i]);
}

/* ---- shared expert ---------------------------------------------------------- */

/*
 * The shared expert of one layer, for every token:
 *   gate[t] = sum_h x[t][h] * wg[h]                  (the router's extra row)
 *   y[t]    = W2s (SiLU(W1s[0:I] x_t) * W1s[I:2I] x_t)   (unweighted)
 * Weights in the routed experts' storage: w1p int32 [2I][H/8], w1s bf16
 * [2I][H/128], w2p int32 [H][I/8], w2s bf16 [H][I/128].
 */
void oracle_shared_expert(const uint16_t *x, const uint16_t *wg, const int32_t *w1p, const uint16_t *w1s,
                          const int32_t *w2p, const uint16_t *w2s, int T, int H, int I, double *gate,
                          double *y, int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel
    {
        double *xt = (double *)malloc(sizeof(double) * (size_t)H);
        double *h = (double *)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(dynamic)
        for (int t = 0; t < T; ++t) {
            if (!xt || !h) continue;
            double g0 = 0.0;
            for (int c = 0; c < H; ++c) {
                xt[c] = bf16_to_f64(x[(int64_t)t * H + c]);
                g0 += xt[c] * bf16_to_f64(wg[c]);
            }
            gate[t] = g0;
            for (int i = 0; i < I; ++i) {
                double g = 0.0, u = 0.0;
                for (int c = 0; c < H; ++c) {
                    g += weight(w1p, w1s, H, i, c) * xt[c];
                    u += weight(w1p, w1s, H, (int64_t)I + i, c) * xt[c];
                }
                h[i] = g / (1.0 + exp(-g)) * u;
            }
            for (int n = 0; n < H; ++n) {
                double s = 0.0;
                for (int i = 0; i < I; ++i) s += weight(w2p, w2s, I, n, i) * h[i];
                y[(int64_t)t * H + n] = s;
            }
        }
        free(xt);
        free(h);
    }
}

/* out[t][n] = routed[t][n] + sigmoid(gate[t]) * y[t][n]. */
void oracle_shared_combine(const double *routed, const double *gate, const double *y, int T, int H,
                           double *out)
{
    for (int t = 0; t < T; ++t) {
        double sg = 1.0 / (1.0 + exp(-gate[t]));
        for (int n = 0; n < H; ++n) out[(int64_t)t * H + n] = routed[(int64_t)t * H + n] + sg * y[(int64_t)t * H + n];
    }
}

/* ---- INT4 quantiser ----------------------------------------------------------- */

/*
 * Round to nearest, symmetric, one scale per 128 consecutive values of a row.
 * For a group with amax = max |w| and clip ratio c_j = (100 - j) / 100
 * (j = 0 .. nclip-1; nclip = 1 is plain round-to-nearest):
 *   s_j = bf16(c_j * amax / 7)            (the stored scale; fp32 arithmetic,
 *                                          each step rounded to nearest)
 *   q_i = clamp(rint(w_i / s_j), -8, 7)   (fp32 division; q = 0 if s_j = 0)
 *   err_j = sum_i (w_i - q_i * s_j)^2     (fp64)
 * The group takes the j with the smallest err_j, the lowest j on a tie.
 * The rounding decisions are made in fp32, the precision of the kernel.
 *
 * w bf16 [N][K] (K a multiple of 128); err f64 [N][K/128][nclip] (may be
 * NULL); packed int32 [N][K/8] and scales bf16 [N][K/128] (may be NULL: then
 * only err is written); choice int32 [N][K/128] (may be NULL).
 */
static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint16_t f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float clip_scale(float amax, int j)
{
    volatile float c = (float)(100 - j) / 100.0f;   /* volatile: each step rounded to fp32 */
    volatile float t = c * amax;
    volatile float s = t / 7.0f;
    return bf16_to_f32(f32_to_bf16(s));
}

static int quant_one(float w, float s)
{
    if (s == 0.0f) return 0;
    volatile float r = w / s;
    float q = rintf(r);
    if (q < -8.0f) q = -8.0f;
    if (q > 7.0f) q = 7.0f;
    return (int)q;
}

int oracle_quantize_int4(const uint16_t *w, int64_t N, int64_t K, int nclip, double *err,
                         int32_t *packed, uint16_t *scales, int32_t *choice)
{
    if (K % ORACLE_GROUP || nclip < 1 || nclip > 100) return -1;
    const int64_t G = K / ORACLE_GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t rg = 0; rg < N * G; ++rg) {
        const int64_t n = rg / G, g = rg % G;
        const uint16_t *wv = w + n * K + g * ORACLE_GROUP;
        float amax = 0.0f;
        for (int i = 0; i < ORACLE_GROUP; ++i) {
            float a = fabsf(bf16_to_f32(wv[i]));
            if (a > amax) amax = a;
        }
        int best = 0;
        double best_err = 0.0;
        for (int j = 0; j < nclip; ++j) {
            const float s = clip_scale(amax, j);
            double e = 0.0;
            for (int i = 0; i < ORACLE_GROUP; ++i) {
                const double wi = (double)bf16_to_f32(wv[i]);
                const double d = wi - (double)quant_one(bf16_to_f32(wv[i]), s) * (double)s;
                e += d * d;
            }
            if (err) err[rg * nclip + j] = e;
            if (j == 0 || e < best_err) {
                best = j;
                best_err = e;
            }
        }
        if (choice) choice[rg] = best;
        if (!packed || !scales) continue;
        const float s = clip_scale(amax, best);
        scales[rg] = f32_to_bf16(s);
        for (int wd = 0; wd < ORACLE_GROUP / 8; ++wd) {
            uint32_t word = 0;
            for (int i = 0; i < 8; ++i)
                word |= (uint32_t)(quant_one(bf16_to_f32(wv[8 * wd + i]), s) + 8) << (4 * i);
            packed[n * (K / 8) + g * (ORACLE_GROUP / 8) + wd] = (int32_t)word;
        }
    }
    return 0;
}

/* ---- INT8 weights (W8A16) --------------------------------------------------- */
/*
 * compressed-tensors INT8 pack-quantized ("vLLM Optimization Edition",
 * section 3.3 "Hyper-connection (decode-04)"; model card "What is quantized",
 * groups C and D): four values per int32 word, least significant byte first,
 * each stored as q + 128, so q lies in [-128, 127]; one bf16 scale per row
 * and group of gs (64 or 128) consecutive values along K.
 */

/* q[n][c] = byte c%4 of packed[n][c/4], minus 128. */
void oracle_unpack_int8(const int32_t *packed, int64_t N, int64_t K, int16_t *q)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t c = 0; c < K; ++c) {
            uint32_t word = (uint32_t)packed[n * (K / 4) + c / 4];
            q[n * K + c] = (int16_t)((int)((word >> (8 * (c % 4))) & 0xFFu) - 128);
        }
}

/* Inverse of oracle_unpack_int8. Returns -1 if some q lies outside [-128, 127]. */
int oracle_pack_int8(const int16_t *q, int64_t N, int64_t K, int32_t *packed)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t w = 0; w < K / 4; ++w) {
            uint32_t word = 0;
            for (int i = 0; i < 4; ++i) {
                int v = q[n * K + w * 4 + i];
                if (v < -128 || v > 127) return -1;
                word |= (uint32_t)(v + 128) << (8 * i);
            }
            packed[n * (K / 4) + w] = (int32_t)word;
        }
    return 0;
}

/*
 * y[t][n] = sum_c x[t][c] * W[n][c], W[n][c] = q[n][c] * scale[n][c / gs]
 * (fp64). x bf16 [T][K], packed int32 [N][K/4], scales bf16 [N][K/gs], y f64
 * [T][N]. Returns -1 unless gs is 64 or 128 and divides K.
 */
int oracle_w8a16_linear(const uint16_t *x, const int32_t *packed, const uint16_t *scales, int gs, int T,
                        int64_t N, int64_t K, double *y, int nthreads)
{
    if ((gs != 64 && gs != 128) || K % gs) return -1;
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int t = 0; t < T; ++t) {
            double s = 0.0;
            for (int64_t c = 0; c < K; ++c) {
                uint32_t word = (uint32_t)packed[n * (K / 4) + c / 4];
                int q = (int)((word >> (8 * (c % 4))) & 0xFFu) - 128;
                double w = (double)q * bf16_to_f64(scales[n * (K / gs) + c / gs]);
                s += bf16_to_f64(x[(int64_t)t * K + c]) * w;
            }
            y[(int64_t)t * N + n] = s;
        }
    }
    return 0;
}
