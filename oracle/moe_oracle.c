/*
 * CPU oracle for the single-GPU MoE layer hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or constant with the CUDA library.
 *
 * Every function is the plain definition of one step, written out in fp64 with
 * no blocking, fusion or reordering beyond what the definition states.  Sources:
 *
 *  [BLOG]  "Lower latency and higher throughput with multi-node DeepSeek
 *          deployment" (Perplexity blog).
 *            §Expert Parallelism: a MoE layer has 256 routed experts and one
 *              shared expert; each token goes to 8 distinct routed experts whose
 *              outputs are summed with weights, and the shared expert's output
 *              is added.
 *            §Roofline / GEMM: a Linear layer is the product [m,k]x[k,n].
 *            §MoE Router: top-k of the router scores, keeping the indices of the
 *              selected elements; dense dispatch needs the routing aggregated per
 *              expert instead of per token.
 *            §Quantization: the activation is SiLU (DeepSeek-V3/R1).
 *  [CANN]  "DeepSeek-R1 prefill inference optimisation on Atlas A3"
 *          (cann-recipes-infer), §MoE deployment strategy (Double-Routing):
 *            step 1, init-routing expands each token and sorts the copies,
 *              returning expanded_x, expanded_row_idx (used to restore the
 *              original order) and tokens_per_expert;
 *            step 6, the inverse permutation is the argsort of the permutation;
 *            step 8, finalize-routing restores the original order through
 *              expanded_src_to_dst_row, applies scales=topk_weight and adds the
 *              shared expert output passed as skip1.
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes): selection is on fp32 scores s_e = fl32(logit_e + bias_e) with
 * ties going to the lower expert id; slots are in descending score order;
 * source rows are token-major (src = t*k + j); the sort is stable (ascending
 * src inside an expert); no token is dropped or padded; the SwiGLU expert is
 * W2 (silu(Wgate v) * (Wup v)); the shared experts' outputs are summed and form
 * one skip tensor.
 *
 * Rounding points (dt = storage dtype, RNE): logits are stored as fp32; the
 * expert hidden h, the expert output y and the shared output are stored in dt;
 * the layer output is rounded once to dt.  All sums are fp64.
 *
 * dtype codes: 0 = fp32 (float), 1 = bf16 (uint16 bit pattern).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1 };

/* ---- storage conversions ------------------------------------------------ */

/* bf16 bit pattern -> value: the bf16 bits are the top half of an fp32. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* fp32 -> bf16 bits, round to nearest, ties to even (finite inputs). */
static uint16_t float_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* Value of element i of an array stored in dtype dt. */
static double load(const void* p, int dt, size_t i) {
    if (dt == OR_BF16) return bf16_bits_to_double(((const uint16_t*)p)[i]);
    return (double)((const float*)p)[i];
}

/* Round a double to the storage dtype and return the stored value.  bf16 goes
 * through fp32 first (fp64 -> fp32 -> bf16, each RNE). */
static double round_to(double v, int dt) {
    float f = (float)v;
    if (dt == OR_BF16) return bf16_bits_to_double(float_to_bf16_bits(f));
    return (double)f;
}

static void store(void* p, int dt, size_t i, double v) {
    if (dt == OR_BF16) ((uint16_t*)p)[i] = float_to_bf16_bits((float)v);
    else ((float*)p)[i] = (float)v;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Exposed so that tests can pin the rounding helper against a library cast. */
void oracle_round_array(const double* in, int dt, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = round_to(in[i], dt);
}

/* ---- FP8 (e4m3) block quantisation ------------------------------------------
 * [BLOG §Quantization]: DeepSeek-V3/R1 uses per-block FP8 quantisation, with
 * weights quantised statically and activations on the fly; scales are computed
 * per 128-element vector for activations and per 128x128 tile for weights.
 * Readings (the page does not fix them): the FP8 format is e4m3 (1 sign bit,
 * 4 exponent bits with bias 7, 3 mantissa bits, largest finite 448, no
 * infinities); a block's scale is amax/448 in fp32 (1 for an all-zero block);
 * a value's code is round-to-nearest-even of fl32(v / scale) onto the e4m3
 * grid, saturating at +-448.                                                   */

/* e4m3 code -> value. */
double oracle_e4m3_decode(uint8_t code) {
    int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double v = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
    return sign ? -v : v;
}

/* value -> e4m3 code, round to nearest even on the e4m3 grid, saturating. */
uint8_t oracle_e4m3_encode(float f) {
    double v = (double)f;
    int sign = v < 0 || (v == 0 && signbit(v));
    double a = fabs(v);
    if (isnan(v)) return 0x7F;
    if (a >= 448.0) return (uint8_t)((sign << 7) | 0x7E);
    /* spacing of the grid around a: 2^-9 below 2^-6 (subnormals), else 2^(E-3) */
    int E = a > 0 ? (int)floor(log2(a)) : -10;
    if (E < -6) E = -6;
    double q = ldexp(1.0, E - 3);
    double n = a / q;                 /* exact: q is a power of two */
    double r = floor(n);
    double frac = n - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) == 1.0)) r += 1.0;
    double val = r * q;
    if (val > 448.0) val = 448.0;
    /* encode val */
    uint8_t code;
    if (val < ldexp(1.0, -6)) {
        code = (uint8_t)(int)(val / ldexp(1.0, -9));                /* subnormal: e = 0 */
    } else {
        int e2 = (int)floor(log2(val));
        int mant = (int)(val / ldexp(1.0, e2 - 3)) - 8;            /* 0..7 */
        code = (uint8_t)(((e2 + 7) << 3) | mant);
    }
    return (uint8_t)((sign << 7) | code);
}

/* Scale of one block from its largest magnitude (fp32 arithmetic). */
static float block_scale(float amax) { return amax > 0.0f ? amax / 448.0f : 1.0f; }

/* Power-of-two block scales (the second scale format).  [BLOG §Quantization]
 * fixes per-block scales but not their number format; this reading stores each
 * scale as a power of two, an 8-bit exponent with no mantissa, which is what
 * block-scaled tensor-core instructions take.  A block's scale is the smallest
 * power of two s with amax / s <= 448, so the block's largest magnitude lands
 * in (224, 448] (1 for an all-zero block; exponent at least -127).  Dividing by
 * s is exact, so a code is round-to-nearest-even of v / s.                    */
static float block_scale_pow2(float amax) {
    if (!(amax > 0.0f)) return 1.0f;
    int e = (int)ceil(log2((double)amax / 448.0));
    while (e > -127 && ldexp(448.0, e - 1) >= (double)amax) --e; /* smallest e with amax <= 448 * 2^e */
    while (ldexp(448.0, e) < (double)amax) ++e;
    if (e < -127) e = -127;
    return (float)ldexp(1.0, e);
}

static float scale_of(float amax, int pow2) { return pow2 ? block_scale_pow2(amax) : block_scale(amax); }

/* Rows of a [rows, cols] matrix (dtype dt) quantised in 1 x 128 blocks along
 * the columns: codes [rows, cols], scales [rows, ceil(cols/128)] fp32 (powers
 * of two when pow2 != 0).                                                    */
void oracle_quantize_rows_fp8(const void* a, int dt, int64_t rows, int cols, uint8_t* codes, float* scales,
                              int pow2) {
    int kb = (cols + 127) / 128;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int b = 0; b < kb; ++b) {
            int c0 = b * 128, c1 = c0 + 128 < cols ? c0 + 128 : cols;
            float amax = 0.0f;
            for (int c = c0; c < c1; ++c) {
                float v = (float)load(a, dt, (size_t)r * cols + c);
                if (fabsf(v) > amax) amax = fabsf(v);
            }
            float s = scale_of(amax, pow2);
            scales[(size_t)r * kb + b] = s;
            for (int c = c0; c < c1; ++c)
                codes[(size_t)r * cols + c] = oracle_e4m3_encode((float)load(a, dt, (size_t)r * cols + c) / s);
        }
    }
}

/* A weight [n_out, k_in] (dtype dt) quantised in 128 x 128 tiles:
 * codes [n_out, k_in], scales [ceil(n_out/128), ceil(k_in/128)] fp32 (powers
 * of two when pow2 != 0).                                                    */
void oracle_quantize_tiles_fp8(const void* w, int dt, int n_out, int k_in, uint8_t* codes, float* scales, int pow2) {
    int nb = (n_out + 127) / 128, kb = (k_in + 127) / 128;
    #pragma omp parallel for schedule(static) collapse(2)
    for (int bn = 0; bn < nb; ++bn) {
        for (int bk = 0; bk < kb; ++bk) {
            int n1 = bn * 128 + 128 < n_out ? bn * 128 + 128 : n_out;
            int k1 = bk * 128 + 128 < k_in ? bk * 128 + 128 : k_in;
            float amax = 0.0f;
            for (int n = bn * 128; n < n1; ++n)
                for (int k = bk * 128; k < k1; ++k) {
                    float v = (float)load(w, dt, (size_t)n * k_in + k);
                    if (fabsf(v) > amax) amax = fabsf(v);
                }
            float s = scale_of(amax, pow2);
            scales[(size_t)bn * kb + bk] = s;
            for (int n = bn * 128; n < n1; ++n)
                for (int k = bk * 128; k < k1; ++k)
                    codes[(size_t)n * k_in + k] = oracle_e4m3_encode((float)load(w, dt, (size_t)n * k_in + k) / s);
        }
    }
}

/* ---- gate GEMM ------------------------------------------------------------
 * [BLOG §Roofline / GEMM]: logits = x [T,H] times the router weight; the
 * router weight is stored like a Linear weight, wg [E,H] (H contiguous), so
 *   logits[t,e] = sum_h x[t,h] * wg[e,h].                                    */
void oracle_gate_logits(const void* x, const void* wg, int dt, int T, int H, int E,
                        double* logits) {
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += load(x, dt, (size_t)t * H + h) * load(wg, dt, (size_t)e * H + h);
            logits[(size_t)t * E + e] = acc;
        }
    }
}

/* ---- top-k routing --------------------------------------------------------
 * [BLOG §MoE Router]: per token, the k experts with the highest scores, with
 * their indices.  Score s_e = fl32(logits[t,e] + bias[e]) (bias may be NULL).
 * Selection order: descending s, ties to the lower expert id; this is a full
 * stable sort of the experts by (-s, e) truncated to k, written as k passes of
 * "pick the best remaining".
 * Weights: softmax over all E scores, then the k selected probabilities; with
 * renorm != 0 they are divided by their sum (the full softmax denominator
 * cancels, leaving a softmax over the selected scores).                      */
void oracle_route_topk(const float* logits, const float* bias, int T, int E, int k,
                       int renorm, int32_t* ids, double* w) {
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        float* s = (float*)malloc(sizeof(float) * (size_t)E);
        char* taken = (char*)calloc((size_t)E, 1);
        for (int e = 0; e < E; ++e) {
            float b = bias ? bias[e] : 0.0f;
            s[e] = logits[(size_t)t * E + e] + b; /* one fp32 add */
        }
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || s[e] > s[best]) best = e; /* strict: ties keep lower id */
            }
            taken[best] = 1;
            ids[(size_t)t * k + j] = best;
        }
        /* softmax over all E scores (shifted by the max for range only). */
        double smax = -INFINITY;
        for (int e = 0; e < E; ++e) if ((double)s[e] > smax) smax = (double)s[e];
        double denom_all = 0.0;
        for (int e = 0; e < E; ++e) denom_all += exp((double)s[e] - smax);
        double sel_sum = 0.0;
        for (int j = 0; j < k; ++j) {
            double p = exp((double)s[ids[(size_t)t * k + j]] - smax) / denom_all;
            w[(size_t)t * k + j] = p;
            sel_sum += p;
        }
        if (renorm)
            for (int j = 0; j < k; ++j) w[(size_t)t * k + j] /= sel_sum;
        free(s);
        free(taken);
    }
}

/* ---- group-limited top-k ------------------------------------------------------
 * [BLOG §MoE Router]: flat top-k is the special case of DeepSeek routing in
 * which the selected group is all experts.  Steps, per token:
 *   1. s_e = fl32(logits[t,e] + bias[e])                        (as above)
 *   2. the E experts form n_group contiguous groups of E/n_group;
 *      group score = the largest s in the group (rule 0), or the sum of the
 *      two largest s in the group as one fp32 add (rule 1);
 *   3. the topk_group groups with the highest group score are kept (ties to
 *      the lower group index);
 *   4. top-k over the experts of the kept groups, descending s, ties to the
 *      lower expert id;
 *   5. weights: softmax over all E scores at the selected experts, divided
 *      by their sum when renorm != 0 (as in the flat router).
 * Every decision (2-4) is taken on fp32 values with fp32 arithmetic.       */
void oracle_route_topk_grouped(const float* logits, const float* bias, int T, int E, int k, int n_group,
                               int topk_group, int rule, int renorm, int32_t* ids, double* w) {
    const int gs = E / n_group;
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        float* s = (float*)malloc(sizeof(float) * (size_t)E);
        float* gscore = (float*)malloc(sizeof(float) * (size_t)n_group);
        char* gkept = (char*)calloc((size_t)n_group, 1);
        char* taken = (char*)calloc((size_t)E, 1);
        for (int e = 0; e < E; ++e) s[e] = logits[(size_t)t * E + e] + (bias ? bias[e] : 0.0f);
        for (int g = 0; g < n_group; ++g) {
            float m1 = -INFINITY, m2 = -INFINITY;  /* largest, second largest */
            for (int e = g * gs; e < (g + 1) * gs; ++e) {
                if (s[e] > m1) { m2 = m1; m1 = s[e]; }
                else if (s[e] > m2) { m2 = s[e]; }
            }
            gscore[g] = rule == 1 ? m1 + m2 : m1;
        }
        for (int r = 0; r < topk_group; ++r) {
            int best = -1;
            for (int g = 0; g < n_group; ++g) {
                if (gkept[g]) continue;
                if (best < 0 || gscore[g] > gscore[best]) best = g;
            }
            gkept[best] = 1;
        }
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e] || !gkept[e / gs]) continue;
                if (best < 0 || s[e] > s[best]) best = e;
            }
            taken[best] = 1;
            ids[(size_t)t * k + j] = best;
        }
        double smax = -INFINITY;
        for (int e = 0; e < E; ++e) if ((double)s[e] > smax) smax = (double)s[e];
        double denom_all = 0.0;
        for (int e = 0; e < E; ++e) denom_all += exp((double)s[e] - smax);
        double sel_sum = 0.0;
        for (int j = 0; j < k; ++j) {
            double p = exp((double)s[ids[(size_t)t * k + j]] - smax) / denom_all;
            w[(size_t)t * k + j] = p;
            sel_sum += p;
        }
        if (renorm)
            for (int j = 0; j < k; ++j) w[(size_t)t * k + j] /= sel_sum;
        free(s);
        free(gscore);
        free(gkept);
        free(taken);
    }
}

/* ---- init-routing -----------------------------------------------------------
 * [CANN §MoE deployment, Double-Routing step 1] + [BLOG §MoE Router]
 * (aggregation per expert).  Source row src = t*k + j (token-major).
 *   tokens_per_expert[e] = #{src : ids[src] == e}
 *   expert_offsets       = exclusive prefix sum of tokens_per_expert ([E+1])
 *   expanded_row_idx[src] = expert_offsets[ids[src]]
 *                           + #{src' < src : ids[src'] == ids[src]}
 *   expanded_x[expanded_row_idx[src], :] = x[src / k, :]
 * i.e. a stable sort of the source rows by expert id.  Ids outside [0,E) get
 * expanded_row_idx = -1, are not counted and the function returns the number
 * of such ids.                                                               */
int oracle_init_routing(const int32_t* ids, int T, int k, int E, const void* x, int dt,
                        int H, void* expanded_x, int32_t* expanded_row_idx,
                        int32_t* tokens_per_expert, int32_t* expert_offsets) {
    int64_t R = (int64_t)T * k;
    int bad = 0;
    for (int e = 0; e < E; ++e) tokens_per_expert[e] = 0;
    for (int64_t src = 0; src < R; ++src) {
        int e = ids[src];
        if (e < 0 || e >= E) { ++bad; continue; }
        tokens_per_expert[e] += 1;
    }
    expert_offsets[0] = 0;
    for (int e = 0; e < E; ++e) expert_offsets[e + 1] = expert_offsets[e] + tokens_per_expert[e];
    int32_t* seen = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int64_t src = 0; src < R; ++src) {
        int e = ids[src];
        if (e < 0 || e >= E) { expanded_row_idx[src] = -1; continue; }
        expanded_row_idx[src] = expert_offsets[e] + seen[e];
        seen[e] += 1;
    }
    free(seen);
    if (expanded_x) {
        size_t esz = dt == OR_BF16 ? 2 : 4;
        for (int64_t src = 0; src < R; ++src) {
            int32_t dst = expanded_row_idx[src];
            if (dst < 0) continue;
            memcpy((char*)expanded_x + (size_t)dst * H * esz,
                   (const char*)x + (size_t)(src / k) * H * esz, (size_t)H * esz);
        }
    }
    return bad;
}

/* ---- re-routing (second routing of Double-Routing) ---------------------------
 * [CANN §MoE deployment, Double-Routing steps 3-4]: a rank receives, from each
 * of W source ranks in rank order, that source's rows for the rank's E_local
 * experts, grouped by expert in expert order (counts[p*E_local + e] rows from
 * source p for local expert e).  Re-routing sorts the received rows by local
 * expert, stable (source order, then arrival order, inside an expert):
 *   x_sorted[i, :] = x_recv[gathered_ids_unsort[i], :]
 *   tokens_per_local_expert[e] = sum_p counts[p, e]; local_offsets = exclusive scan.
 * Written as: enumerate the received rows in arrival order with their local
 * expert, then a counting sort by expert.                                      */
void oracle_re_routing(const void* x_recv, int dt, const int32_t* counts, int W, int E_local, int H,
                       void* x_sorted, int32_t* gathered_ids_unsort, int32_t* tokens_per_local_expert,
                       int32_t* local_offsets) {
    int64_t N = 0;
    for (int i = 0; i < W * E_local; ++i) N += counts[i];
    int32_t* expert_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N > 0 ? N : 1));
    int64_t r = 0;
    for (int p = 0; p < W; ++p)
        for (int e = 0; e < E_local; ++e)
            for (int i = 0; i < counts[p * E_local + e]; ++i) expert_of[r++] = e;
    for (int e = 0; e < E_local; ++e) tokens_per_local_expert[e] = 0;
    for (int64_t i = 0; i < N; ++i) tokens_per_local_expert[expert_of[i]] += 1;
    local_offsets[0] = 0;
    for (int e = 0; e < E_local; ++e) local_offsets[e + 1] = local_offsets[e] + tokens_per_local_expert[e];
    int32_t* next = (int32_t*)malloc(sizeof(int32_t) * (size_t)E_local);
    for (int e = 0; e < E_local; ++e) next[e] = local_offsets[e];
    size_t esz = dt == OR_BF16 ? 2 : 4;
    for (int64_t i = 0; i < N; ++i) {
        int32_t dst = next[expert_of[i]]++;
        gathered_ids_unsort[dst] = (int32_t)i;
        if (x_sorted)
            memcpy((char*)x_sorted + (size_t)dst * H * esz, (const char*)x_recv + (size_t)i * H * esz,
                   (size_t)H * esz);
    }
    free(next);
    free(expert_of);
}

/* [CANN step 6]: rows back in received order, out[gathered_ids_unsort[i]] =
 * y_sorted[i] (the page's index_select with the argsort of gathered_ids_unsort). */
void oracle_unsort_rows(const void* y_sorted, int dt, const int32_t* gathered_ids_unsort, int64_t N, int H,
                        void* out) {
    size_t esz = dt == OR_BF16 ? 2 : 4;
    for (int64_t i = 0; i < N; ++i)
        memcpy((char*)out + (size_t)gathered_ids_unsort[i] * H * esz, (const char*)y_sorted + (size_t)i * H * esz,
               (size_t)H * esz);
}

/* ---- one SwiGLU expert on one row ------------------------------------------
 * [BLOG §Expert Parallelism] (expert FFN) and [BLOG §Quantization] (SiLU):
 *   g = wgate v,  u = wup v          (wgate, wup: [I,H], H contiguous)
 *   h_i = silu(g_i) * u_i,  silu(z) = z / (1 + exp(-z))
 *   y = w2 h                          (w2: [H,I], I contiguous)
 * h is rounded to dt when round_h != 0 (the stored intermediate); y is
 * returned unrounded.                                                        */
static void expert_ffn_row(const void* v, size_t v_off, int dt, const void* wgate,
                           const void* wup, const void* w2, size_t wgu_off, size_t w2_off,
                           int H, int I, int round_h, double* hbuf, double* y) {
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) {
            double vh = load(v, dt, v_off + h);
            g += load(wgate, dt, wgu_off + (size_t)i * H + h) * vh;
            u += load(wup, dt, wgu_off + (size_t)i * H + h) * vh;
        }
        double hi = g / (1.0 + exp(-g)) * u;
        hbuf[i] = round_h ? round_to(hi, dt) : hi;
    }
    for (int o = 0; o < H; ++o) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += load(w2, dt, w2_off + (size_t)o * I + i) * hbuf[i];
        y[o] = acc;
    }
}

/* Expert FFN applied to n rows of a [*,H] matrix: rows[r] = FFN_{expert[r]}(a[r]).
 * Weights: wgate/wup [E,I,H], w2 [E,H,I].  The output of each row is rounded to
 * dt (the stored expert output).  Rows with expert < 0 are left untouched.   */
void oracle_expert_ffn_rows(const void* a, int dt, int64_t n, const int32_t* expert,
                            const void* wgate, const void* wup, const void* w2, int H, int I,
                            double* y) {
    #pragma omp parallel
    {
        double* hbuf = (double*)malloc(sizeof(double) * (size_t)I);
        double* yr = (double*)malloc(sizeof(double) * (size_t)H);
        #pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n; ++r) {
            int e = expert[r];
            if (e < 0) continue;
            expert_ffn_row(a, (size_t)r * H, dt, wgate, wup, w2, (size_t)e * I * H,
                           (size_t)e * H * I, H, I, dt == OR_BF16, hbuf, yr);
            for (int o = 0; o < H; ++o) y[(size_t)r * H + o] = round_to(yr[o], dt);
        }
        free(hbuf);
        free(yr);
    }
}

/* ---- finalize-routing --------------------------------------------------------
 * [CANN §MoE deployment, Double-Routing step 8]:
 *   out[t,:] = skip[t,:] + sum_j scales[t,j] * y[expanded_src_to_dst_row[t*k+j], :]
 * skip may be NULL; rows whose index is outside [0, n_rows) are skipped.  The
 * result is returned unrounded (fp64).                                       */
void oracle_finalize_routing(const void* y, int dt, int64_t n_rows, const void* skip,
                             const double* scales, const int32_t* expanded_row_idx, int T,
                             int H, int k, double* out) {
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int o = 0; o < H; ++o) {
            double acc = skip ? load(skip, dt, (size_t)t * H + o) : 0.0;
            for (int j = 0; j < k; ++j) {
                int32_t r = expanded_row_idx[(size_t)t * k + j];
                if (r < 0 || r >= n_rows) continue;
                acc += scales[(size_t)t * k + j] * load(y, dt, (size_t)r * H + o);
            }
            out[(size_t)t * H + o] = acc;
        }
    }
}

/* ---- FP8 block-scaled GEMM and SwiGLU expert ---------------------------------
 * [BLOG §Quantization]: with scales per 1x128 activation vector and per 128x128
 * weight tile, a product [M,K]x[K,N] (weights stored [N,K]) is
 *   C[m,n] = sum_b sa[m,b] * sb[n/128, b] * sum_{k in block b} qa[m,k] * qb[n,k]
 * with qa, qb the e4m3 values.  Sums in fp64.                                 */
static double E4M3[256];
static void init_e4m3(void) {
    static int done = 0;
    if (done) return;
    for (int c = 0; c < 256; ++c) E4M3[c] = oracle_e4m3_decode((uint8_t)c);
    done = 1;
}

static double fp8_dot(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb_row, int K) {
    int kb = (K + 127) / 128;
    double acc = 0.0;
    for (int b = 0; b < kb; ++b) {
        double part = 0.0;
        int k1 = b * 128 + 128 < K ? b * 128 + 128 : K;
        for (int k = b * 128; k < k1; ++k) part += E4M3[qa[k]] * E4M3[qb[k]];
        acc += (double)sa[b] * (double)sb_row[b] * part;
    }
    return acc;
}

void oracle_gemm_fp8(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb, int M, int N, int K,
                     double* c) {
    init_e4m3();
    int kb = (K + 127) / 128;
    #pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n)
            c[(size_t)m * N + n] = fp8_dot(qa + (size_t)m * K, sa + (size_t)m * kb, qb + (size_t)n * K,
                                           sb + (size_t)(n / 128) * kb, K);
}

/* One SwiGLU expert on one quantised row (bf16 layer with FP8 weights):
 *   g, u   = FP8 products of the row with the gate and up weights
 *   h      = silu(g) * u, stored in bf16, then quantised in 1x128 blocks
 *            (power-of-two scales when pow2 != 0)
 *   y      = FP8 product of h with the down weight (returned unrounded)
 * Weights of the expert: gq/uq [I,H] with scales [I/128][H/128]; dq [H,I]
 * with scales [H/128][I/128].                                                 */
static void expert_ffn_row_fp8(const uint8_t* xq, const float* xs, const uint8_t* gq, const float* gs,
                               const uint8_t* uq, const float* us, const uint8_t* dq, const float* ds, int H,
                               int I, double* hbuf, uint8_t* hq, float* hs, double* y, int pow2) {
    int kbh = (H + 127) / 128, kbi = (I + 127) / 128;
    for (int i = 0; i < I; ++i) {
        double g = fp8_dot(xq, xs, gq + (size_t)i * H, gs + (size_t)(i / 128) * kbh, H);
        double u = fp8_dot(xq, xs, uq + (size_t)i * H, us + (size_t)(i / 128) * kbh, H);
        hbuf[i] = round_to(g / (1.0 + exp(-g)) * u, OR_BF16);
    }
    for (int b = 0; b < kbi; ++b) {
        int i1 = b * 128 + 128 < I ? b * 128 + 128 : I;
        float amax = 0.0f;
        for (int i = b * 128; i < i1; ++i) if (fabsf((float)hbuf[i]) > amax) amax = fabsf((float)hbuf[i]);
        float sc = scale_of(amax, pow2);
        hs[b] = sc;
        for (int i = b * 128; i < i1; ++i) hq[i] = oracle_e4m3_encode((float)hbuf[i] / sc);
    }
    for (int o = 0; o < H; ++o) y[o] = fp8_dot(hq, hs, dq + (size_t)o * I, ds + (size_t)(o / 128) * kbi, I);
}

/* Expert FFN on quantised rows: y[r] = FFN_fp8_{expert[r]}(xq[r]) stored in bf16
 * (rows with expert < 0 untouched).  xs [n][ceil(H/128)]; weights per expert as
 * in oracle_layer_fp8.                                                        */
void oracle_expert_ffn_rows_fp8(const uint8_t* xq, const float* xs, int64_t n, const int32_t* expert,
                                const uint8_t* gq, const float* gs, const uint8_t* uq, const float* us,
                                const uint8_t* dq, const float* ds, int H, int I, double* y, int pow2) {
    init_e4m3();
    const int kbh = (H + 127) / 128, kbi = (I + 127) / 128;
    const size_t gsz = (size_t)kbi * kbh;
    #pragma omp parallel
    {
        double* hbuf = (double*)malloc(sizeof(double) * (size_t)I);
        uint8_t* hq = (uint8_t*)malloc((size_t)I);
        float* hs = (float*)malloc(sizeof(float) * (size_t)kbi);
        double* yr = (double*)malloc(sizeof(double) * (size_t)H);
        #pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n; ++r) {
            int e = expert[r];
            if (e < 0) continue;
            expert_ffn_row_fp8(xq + (size_t)r * H, xs + (size_t)r * kbh, gq + (size_t)e * I * H, gs + e * gsz,
                               uq + (size_t)e * I * H, us + e * gsz, dq + (size_t)e * H * I, ds + e * gsz, H, I,
                               hbuf, hq, hs, yr, pow2);
            for (int o = 0; o < H; ++o) y[(size_t)r * H + o] = round_to(yr[o], OR_BF16);
        }
        free(hbuf); free(hq); free(hs); free(yr);
    }
}

/* The layer with FP8 expert weights (bf16 activations and outputs), brute force
 * per token: bf16 gate logits and routing exactly as oracle_layer, x quantised
 * in 1x128 blocks, each expert (routed and shared) through expert_ffn_row_fp8,
 * the shared outputs summed and stored in bf16, each routed output stored in
 * bf16, the weighted sum rounded once to bf16.
 * Per-expert weight arrays: gq, uq [E][I][H], gs, us [E][I/128][H/128],
 * dq [E][H][I], ds [E][H/128][I/128]; the shared ones likewise with S.  With
 * pow2 != 0 the activations (x and h) get power-of-two block scales; the weight
 * codes and scales are whatever the caller quantised them with.              */
void oracle_layer_fp8(const void* x, int T, int H, int E, int k, int I, int S, int renorm, const void* wg,
                      const float* bias, const uint8_t* gq, const float* gs, const uint8_t* uq, const float* us,
                      const uint8_t* dq, const float* ds, const uint8_t* sgq, const float* sgs, const uint8_t* suq,
                      const float* sus, const uint8_t* sdq, const float* sds, const int32_t* tokens, int n_tok,
                      double* logits64, int32_t* ids, double* w, double* out, int n_group, int topk_group,
                      int group_rule, int pow2) {
    init_e4m3();
    if (!tokens) n_tok = T;
    const int kbh = (H + 127) / 128, kbi = (I + 127) / 128;
    const size_t gsz = (size_t)kbi * kbh;  /* scale blocks of one [I,H] weight */
    #pragma omp parallel
    {
        float* l32 = (float*)malloc(sizeof(float) * (size_t)E);
        uint8_t* xq = (uint8_t*)malloc((size_t)H);
        float* xs = (float*)malloc(sizeof(float) * (size_t)kbh);
        double* hbuf = (double*)malloc(sizeof(double) * (size_t)I);
        uint8_t* hq = (uint8_t*)malloc((size_t)I);
        float* hs = (float*)malloc(sizeof(float) * (size_t)kbi);
        double* yr = (double*)malloc(sizeof(double) * (size_t)H);
        double* ysh = (double*)malloc(sizeof(double) * (size_t)H);
        #pragma omp for schedule(dynamic, 1)
        for (int n = 0; n < n_tok; ++n) {
            int t = tokens ? tokens[n] : n;
            size_t xo = (size_t)t * H;
            for (int e = 0; e < E; ++e) {
                double acc = 0.0;
                for (int h = 0; h < H; ++h) acc += load(x, OR_BF16, xo + h) * load(wg, OR_BF16, (size_t)e * H + h);
                l32[e] = (float)acc;
                if (logits64) logits64[(size_t)n * E + e] = acc;
            }
            if (n_group > 1)
                oracle_route_topk_grouped(l32, bias, 1, E, k, n_group, topk_group, group_rule, renorm,
                                          ids + (size_t)n * k, w + (size_t)n * k);
            else
                oracle_route_topk(l32, bias, 1, E, k, renorm, ids + (size_t)n * k, w + (size_t)n * k);
            oracle_quantize_rows_fp8((const char*)x + xo * 2, OR_BF16, 1, H, xq, xs, pow2);
            for (int o = 0; o < H; ++o) ysh[o] = 0.0;
            for (int s2 = 0; s2 < S; ++s2) {
                expert_ffn_row_fp8(xq, xs, sgq + (size_t)s2 * I * H, sgs + s2 * gsz, suq + (size_t)s2 * I * H,
                                   sus + s2 * gsz, sdq + (size_t)s2 * H * I, sds + s2 * gsz, H, I, hbuf, hq, hs, yr,
                                   pow2);
                for (int o = 0; o < H; ++o) ysh[o] += yr[o];
            }
            double* orow = out + (size_t)n * H;
            for (int o = 0; o < H; ++o) orow[o] = round_to(ysh[o], OR_BF16);
            for (int j = 0; j < k; ++j) {
                int e = ids[(size_t)n * k + j];
                expert_ffn_row_fp8(xq, xs, gq + (size_t)e * I * H, gs + e * gsz, uq + (size_t)e * I * H,
                                   us + e * gsz, dq + (size_t)e * H * I, ds + e * gsz, H, I, hbuf, hq, hs, yr,
                                   pow2);
                double wj = w[(size_t)n * k + j];
                for (int o = 0; o < H; ++o) orow[o] += wj * round_to(yr[o], OR_BF16);
            }
            for (int o = 0; o < H; ++o) orow[o] = round_to(orow[o], OR_BF16);
        }
        free(l32); free(xq); free(xs); free(hbuf); free(hq); free(hs); free(yr); free(ysh);
    }
}

/* ---- the whole layer, brute force per token ---------------------------------
 * [BLOG §Expert Parallelism]: out[t] = shared(x_t) + sum_j w_j * FFN_{e_j}(x_t)
 * with e_j, w_j from the router on the gate logits (flat, or group-limited when
 * n_group > 1).  S shared experts (weights
 * sgate/sup [S,I,H], s2 [S,H,I]) are summed into one shared output, stored in
 * dt; each routed expert output is stored in dt; the final sum is rounded to dt.
 * Only the tokens listed in tokens[0..n_tok) are evaluated (all when tokens is
 * NULL, n_tok = T).  Returns for those tokens: logits64 [n_tok,E] (fp64, before
 * the fp32 store; may be NULL), ids [n_tok,k], w [n_tok,k], out [n_tok,H]
 * (already rounded to dt, returned as double).                               */
void oracle_layer(const void* x, int dt, int T, int H, int E, int k, int I, int S, int renorm,
                  const void* wg, const float* bias, const void* wgate, const void* wup,
                  const void* w2, const void* sgate, const void* sup, const void* s2,
                  const int32_t* tokens, int n_tok, double* logits64, int32_t* ids, double* w,
                  double* out, int n_group, int topk_group, int group_rule) {
    if (!tokens) n_tok = T;
    #pragma omp parallel
    {
        double* l64 = (double*)malloc(sizeof(double) * (size_t)E);
        float* l32 = (float*)malloc(sizeof(float) * (size_t)E);
        double* hbuf = (double*)malloc(sizeof(double) * (size_t)I);
        double* yr = (double*)malloc(sizeof(double) * (size_t)H);
        double* ysh = (double*)malloc(sizeof(double) * (size_t)H);
        #pragma omp for schedule(dynamic, 1)
        for (int n = 0; n < n_tok; ++n) {
            int t = tokens ? tokens[n] : n;
            size_t xo = (size_t)t * H;
            /* gate logits for this token, stored as fp32 */
            for (int e = 0; e < E; ++e) {
                double acc = 0.0;
                for (int h = 0; h < H; ++h) acc += load(x, dt, xo + h) * load(wg, dt, (size_t)e * H + h);
                l64[e] = acc;
                l32[e] = (float)acc;
                if (logits64) logits64[(size_t)n * E + e] = acc;
            }
            if (n_group > 1)
                oracle_route_topk_grouped(l32, bias, 1, E, k, n_group, topk_group, group_rule, renorm,
                                          ids + (size_t)n * k, w + (size_t)n * k);
            else
                oracle_route_topk(l32, bias, 1, E, k, renorm, ids + (size_t)n * k, w + (size_t)n * k);
            /* shared experts: one summed output, stored in dt */
            for (int o = 0; o < H; ++o) ysh[o] = 0.0;
            for (int s = 0; s < S; ++s) {
                expert_ffn_row(x, xo, dt, sgate, sup, s2, (size_t)s * I * H, (size_t)s * H * I, H, I,
                               dt == OR_BF16, hbuf, yr);
                for (int o = 0; o < H; ++o) ysh[o] += yr[o];
            }
            double* orow = out + (size_t)n * H;
            for (int o = 0; o < H; ++o) orow[o] = round_to(ysh[o], dt);
            /* routed experts, each output stored in dt, weighted sum */
            for (int j = 0; j < k; ++j) {
                int e = ids[(size_t)n * k + j];
                expert_ffn_row(x, xo, dt, wgate, wup, w2, (size_t)e * I * H, (size_t)e * H * I, H, I,
                               dt == OR_BF16, hbuf, yr);
                double wj = w[(size_t)n * k + j];
                for (int o = 0; o < H; ++o) orow[o] += wj * round_to(yr[o], dt);
            }
            for (int o = 0; o < H; ++o) orow[o] = round_to(orow[o], dt);
        }
        free(l64);
        free(l32);
        free(hbuf);
        free(yr);
        free(ysh);
    }
}
