/*
 * moe_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of what the MoE expert-FFN forward
 * computes.  Only tests/, the smoke check and the benchmark's CPU-baseline
 * leg load this file; the product library never does, and this file shares
 * no code, header, table or constant with the CUDA path.
 *
 * Sources (cited by page title and section):
 *  [P3]  "factor_moe_fused_gemm.cu" (ex_engine, Factor 2: MOE_FUSED_GEMM):
 *        the header comment "Current PyTorch path" is the definition of the
 *        forward; fused_silu_gate_kernel fixes gate = first half of the w13
 *        rows, up = second half and SiLU(g) = g / (1 + exp(-g));
 *        build_expert_map_kernel fixes the expert histogram / CSR offsets.
 *  [P1]  "moe triton kernel use tma" (LightLLM pull request 1100): the
 *        summary's mblocks_to_tuple_info (expert id, M-index, token start
 *        per M-block) and the review comment on TOKEN_INPUT_USE_TMA /
 *        MUL_ROUTED_WEIGHT (routing weight multiplies in the down projection).
 *  [P2]  "MOE Bmm1 Fused Gather" (Triton Gluon example): load_activations
 *        (padded rows of a block are masked), pack_e4m3x2 (fp32 -> e4m3 with
 *        round-to-nearest-even and saturation), init_routing_data (the gather
 *        row of an assignment is its flat index divided by top-k).
 *
 * Readings where the pages are silent are listed with each function.
 * Parity is pinned by tests/test_oracle_pins.py (brute force, closed forms,
 * invariants, special cases), not by this file agreeing with itself.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* element storage codes used by the oracle's own interface */
#define ORC_F32 0   /* IEEE binary32                                   */
#define ORC_BF16 1  /* bfloat16 (upper half of a binary32)             */
#define ORC_MXFP4 3 /* OCP MX: e2m1 pairs packed low-nibble-first, one */
                    /* e8m0 scale per 32 consecutive K elements         */

#define ORC_ACT_SILU 0          /* a = SiLU(g) * u                        */
#define ORC_ACT_SWIGLU_CLAMP 1  /* [P2]'s GPT-OSS SwiGLU (clamped, alpha)   */

#define ORC_EXACT 0   /* no intermediate rounding                        */
#define ORC_EMULATE 1 /* round the activation a_j to its storage type    */

typedef struct {
    int T, H, I, E, K;
    int x_dtype;     /* ORC_F32 or ORC_BF16                               */
    int w_dtype;     /* ORC_F32, ORC_BF16 or ORC_MXFP4                    */
    int quantize_x;  /* 1: x goes through the per-row e4m3 step first     */
    int h_e4m3;      /* 1: h is stored as e4m3(a / h_scale) (EMULATE)     */
    double h_scale;  /* scale of the e4m3 h (1.0 when unused)             */
    int expert_base;   /* expert-parallel shard: first expert held here     */
    int local_experts; /* experts held (weights hold these only); 0 = all E */
    int activation;           /* ORC_ACT_SILU or ORC_ACT_SWIGLU_CLAMP        */
    double swiglu_alpha;      /* sigmoid slope of ORC_ACT_SWIGLU_CLAMP       */
    double swiglu_limit;      /* clamp of ORC_ACT_SWIGLU_CLAMP               */
    int gate_up_interleaved;  /* w13 rows 2j = gate j, 2j+1 = up j           */
    const float* w13_bias;    /* (experts held, 2I) in w13's row order, or 0 */
    const float* w2_bias;     /* (experts held, H), or 0                     */
} orc_problem;

/* Experts of the shard (all E when local_experts is 0). */
static int shard_size(const orc_problem* p) {
    return p->local_experts > 0 ? p->local_experts : p->E;
}

/* ------------------------------------------------------------------ */
/* Number formats, decoded from their definitions                      */
/* ------------------------------------------------------------------ */

static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* OCP FP8 E4M3 (the "fn" variant: no infinities, S.1111.111 is NaN):
 * bias 7, exponent field 0 is subnormal with value m/8 * 2^-6. */
double orc_e4m3_to_double(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* OCP MX FP4 E2M1: bias 1, exponent field 0 is subnormal with value m/2. */
double orc_e2m1_to_double(uint8_t nib) {
    int s = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* OCP MX E8M0 scale: 2^(v - 127); 255 is NaN. */
double orc_e8m0_to_double(uint8_t v) {
    if (v == 255) return NAN;
    return ldexp(1.0, (int)v - 127);
}

/* fp32 -> e4m3 code, round to nearest, ties to even code, saturating to
 * +-448 (what cvt.rn.satfinite.e4m3x2.f32 in pack_e4m3x2 [P2] does).
 * Written as a search over every finite code: slow, but it is the
 * definition of "nearest representable value". */
uint8_t orc_float_to_e4m3(float f) {
    if (isnan(f)) return 0x7F;
    double v = (double)f;
    int neg = signbit(f) ? 1 : 0;
    double a = fabs(v);
    if (a >= 448.0) return (uint8_t)((neg << 7) | 0x7E);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double err = fabs(orc_e4m3_to_double((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)((neg << 7) | best);
}

/* double -> nearest bfloat16 value (ties to even), rounded once from the
 * double (EMULATE mode only).  bf16 keeps 8 significant bits: the spacing of
 * the values around v is 2^(e-8) for v = m 2^e with 0.5 <= |m| < 1, and
 * 2^-133 at the bottom of the subnormal range; rint rounds half to even.
 * Values past the largest finite bf16, (2 - 2^-7) 2^127, become infinite. */
static double round_to_bf16(double v) {
    if (!isfinite(v) || v == 0.0) return v;
    int e;
    frexp(v, &e);
    int q = e - 8;
    if (q < -133) q = -133;
    double r = ldexp(rint(ldexp(v, -q)), q);
    if (fabs(r) > ldexp(2.0 - ldexp(1.0, -7), 127)) r = copysign(INFINITY, v);
    return r;
}

/* ------------------------------------------------------------------ */
/* Element access                                                      */
/* ------------------------------------------------------------------ */

static double load_act(const void* p, int dtype, size_t idx) {
    if (dtype == ORC_BF16) return bf16_to_double(((const uint16_t*)p)[idx]);
    return (double)((const float*)p)[idx];
}

/* Decode row `row` (0 <= row < R) of expert e of a weight tensor stored as
 * (E, R, C) with C along K, into dst[0..C). */
static void load_weight_row(const void* w, const uint8_t* scale, int dtype, int R, int C, int e,
                            int row, double* dst) {
    size_t r = (size_t)e * (size_t)R + (size_t)row;
    if (dtype == ORC_F32) {
        const float* src = (const float*)w + r * (size_t)C;
        for (int c = 0; c < C; ++c) dst[c] = (double)src[c];
    } else if (dtype == ORC_BF16) {
        const uint16_t* src = (const uint16_t*)w + r * (size_t)C;
        for (int c = 0; c < C; ++c) dst[c] = bf16_to_double(src[c]);
    } else { /* ORC_MXFP4 */
        const uint8_t* src = (const uint8_t*)w + r * (size_t)(C / 2);
        const uint8_t* sc = scale + r * (size_t)(C / 32);
        for (int c = 0; c < C; ++c) {
            uint8_t byte = src[c / 2];
            uint8_t nib = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
            dst[c] = orc_e2m1_to_double(nib) * orc_e8m0_to_double(sc[c / 32]);
        }
    }
}

static double dot(const double* a, const double* b, int n) {
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* ------------------------------------------------------------------ */
/* fp8 activation step (used when quantize_x is set)                  */
/* ------------------------------------------------------------------ */

/* Per-row symmetric e4m3 quantisation of x: s_t = amax_t / 448 (1 when the
 * row is all zero), code = e4m3_rn_satfinite(x / s_t).  Both the scale and
 * the quotient are formed in fp32, so that the rounding decision is taken
 * in the same precision the GPU takes it.  Reading: [P2] uses one scalar
 * x scale; the workload asks for one scale per row. */
void orc_quantize_x_fp8(const void* x, int x_dtype, int T, int H, uint8_t* xq, float* row_scale) {
    for (int t = 0; t < T; ++t) {
        float amax = 0.0f;
        for (int h = 0; h < H; ++h) {
            float v = (float)load_act(x, x_dtype, (size_t)t * H + h);
            if (fabsf(v) > amax) amax = fabsf(v);
        }
        float s = (amax > 0.0f) ? amax / 448.0f : 1.0f;
        row_scale[t] = s;
        for (int h = 0; h < H; ++h) {
            float v = (float)load_act(x, x_dtype, (size_t)t * H + h);
            xq[(size_t)t * H + h] = orc_float_to_e4m3(v / s);
        }
    }
}

/* The activation row of token t as the method sees it: x itself, or the
 * dequantised e4m3 codes times the row scale. */
static void load_token_row(const orc_problem* p, const void* x, int t, double* dst) {
    if (!p->quantize_x) {
        for (int h = 0; h < p->H; ++h) dst[h] = load_act(x, p->x_dtype, (size_t)t * p->H + h);
        return;
    }
    uint8_t* q = (uint8_t*)malloc((size_t)p->H);
    float s;
    orc_quantize_x_fp8((const char*)x + (size_t)t * p->H * (p->x_dtype == ORC_BF16 ? 2 : 4),
                       p->x_dtype, 1, p->H, q, &s);
    for (int h = 0; h < p->H; ++h) dst[h] = orc_e4m3_to_double(q[h]) * (double)s;
    free(q);
}

/* Round an activation a_j to what the GPU stores between the two GEMMs
 * (EMULATE mode; EXACT keeps it). */
static double store_hidden(const orc_problem* p, int mode, double a) {
    if (mode != ORC_EMULATE) return a;
    if (p->h_e4m3) {
        float q = (float)(a / p->h_scale);
        return orc_e4m3_to_double(orc_float_to_e4m3(q)) * p->h_scale;
    }
    if (p->x_dtype == ORC_BF16) return round_to_bf16(a);
    return (double)(float)a;
}

/* ------------------------------------------------------------------ */
/* One expert FFN on one token row                                     */
/* ------------------------------------------------------------------ */

/* Rows of gate j and up j in w13.  [P3] (fused_silu_gate_kernel,
 * "gate_up.chunk(2)" in the PyTorch path) puts gate in the first half of the
 * rows and up in the second; [P2]'s GPT-OSS layout interleaves them (its
 * epilogue unpacks adjacent (gate, linear) column pairs). */
static int gate_row(const orc_problem* p, int j) { return p->gate_up_interleaved ? 2 * j : j; }
static int up_row(const orc_problem* p, int j) {
    return p->gate_up_interleaved ? 2 * j + 1 : p->I + j;
}

/* [P2] _swiglu_step1 / _swiglu_step2: the gate is clamped from above at
 * `limit`, the linear branch to [-limit, limit], and
 * out = gate * sigmoid(alpha * gate) * (linear + 1). */
static double swiglu_clamped(const orc_problem* p, double g, double u) {
    g = fmin(g, p->swiglu_limit);
    u = fmax(fmin(u, p->swiglu_limit), -p->swiglu_limit);
    return g / (1.0 + exp(-p->swiglu_alpha * g)) * (u + 1.0);
}

/* a_j = act(W13[e, gate_row(j), :] . xrow + b13[gate_row(j)],
 *           W13[e, up_row(j), :] . xrow + b13[up_row(j)]), j < I,
 * act(g, u) = SiLU(g) * u ([P3]) or the clamped SwiGLU above ([P2]); the
 * bias (per expert and w13 row, [P2] apply_bias_and_scale) is added to the
 * accumulator before the activation. */
static void expert_hidden(const orc_problem* p, const void* w13, const uint8_t* w13_scale, int e,
                          const double* xrow, double* a, double* wrow) {
    const float* b13 = p->w13_bias ? p->w13_bias + (size_t)e * 2 * p->I : NULL;
    for (int j = 0; j < p->I; ++j) {
        load_weight_row(w13, w13_scale, p->w_dtype, 2 * p->I, p->H, e, gate_row(p, j), wrow);
        double g = dot(wrow, xrow, p->H) + (b13 ? (double)b13[gate_row(p, j)] : 0.0);
        load_weight_row(w13, w13_scale, p->w_dtype, 2 * p->I, p->H, e, up_row(p, j), wrow);
        double u = dot(wrow, xrow, p->H) + (b13 ? (double)b13[up_row(p, j)] : 0.0);
        if (p->activation == ORC_ACT_SWIGLU_CLAMP)
            a[j] = swiglu_clamped(p, g, u);
        else
            a[j] = silu(g) * u;
    }
}

/* y_c = W2[e, c, :] . a + b2[e, c], c < H (the bias, when given, belongs to
 * the expert's second projection, before the routing weight). */
static void expert_out(const orc_problem* p, const void* w2, const uint8_t* w2_scale, int e,
                       const double* a, double* y, double* wrow) {
    for (int c = 0; c < p->H; ++c) {
        load_weight_row(w2, w2_scale, p->w_dtype, p->H, p->I, e, c, wrow);
        y[c] = dot(wrow, a, p->I) + (p->w2_bias ? (double)p->w2_bias[(size_t)e * p->H + c] : 0.0);
    }
}

static int max_int(int a, int b) { return a > b ? a : b; }

/* ------------------------------------------------------------------ */
/* The forward, loop over tokens then their top-k slots                */
/* ------------------------------------------------------------------ */

/* out[r, c] for token t = tokens[r] (all tokens when tokens == NULL):
 *   out[t, :] = sum_{k=0..K-1} w[t,k] * W2[e] (SiLU(W13g[e] x_t) * (W13u[e] x_t)),
 *   e = ids[t,k], accumulated in k order, fp64.
 * This is the "Current PyTorch path" of [P3] written per token; the routing
 * weight multiplies the down-projection output ([P1] MUL_ROUTED_WEIGHT).
 * Expert-parallel shard ([P2] init_routing_data: a shard keeps the
 * histogram of its local experts only, make_expt_dict_uniform gives each
 * shard a contiguous range): slots routed to an expert outside
 * [expert_base, expert_base + local_experts) contribute nothing, and the
 * weights are indexed by e - expert_base.  The shards' outputs sum to the
 * unsharded output.
 * Returns 0, or -1 when an expert id is outside [0, E). */
int orc_moe_forward(const orc_problem* p, int mode, const void* x, const int32_t* ids,
                    const float* topk_w, const void* w13, const uint8_t* w13_scale, const void* w2,
                    const uint8_t* w2_scale, const int32_t* tokens, int n_tokens, double* out) {
    int n = tokens ? n_tokens : p->T;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int r = 0; r < n; ++r) {
        int t = tokens ? tokens[r] : r;
        double* xrow = (double*)malloc(sizeof(double) * p->H);
        double* wrow = (double*)malloc(sizeof(double) * max_int(p->H, p->I));
        double* a = (double*)malloc(sizeof(double) * p->I);
        double* y = (double*)malloc(sizeof(double) * p->H);
        double* o = out + (size_t)r * p->H;
        for (int c = 0; c < p->H; ++c) o[c] = 0.0;
        load_token_row(p, x, t, xrow);
        for (int k = 0; k < p->K; ++k) {
            int e = ids[(size_t)t * p->K + k];
            if (e < 0 || e >= p->E) {
                bad = 1;
                continue;
            }
            if (e < p->expert_base || e >= p->expert_base + shard_size(p)) continue;
            e -= p->expert_base; /* index into this shard's weights */
            double w = (double)topk_w[(size_t)t * p->K + k];
            expert_hidden(p, w13, w13_scale, e, xrow, a, wrow);
            for (int j = 0; j < p->I; ++j) a[j] = store_hidden(p, mode, a[j]);
            expert_out(p, w2, w2_scale, e, a, y, wrow);
            for (int c = 0; c < p->H; ++c) o[c] += w * y[c];
        }
        free(xrow);
        free(wrow);
        free(a);
        free(y);
    }
    return bad ? -1 : 0;
}

/* The same forward in the per-expert loop order of [P3]'s PyTorch path:
 * for each expert, take its (token, slot) pairs in ascending flat index,
 * run the FFN, and index-add weight * output into the token rows.  Used
 * only to check that the two loop orders agree. */
int orc_moe_forward_by_expert(const orc_problem* p, int mode, const void* x, const int32_t* ids,
                              const float* topk_w, const void* w13, const uint8_t* w13_scale,
                              const void* w2, const uint8_t* w2_scale, double* out) {
    size_t na = (size_t)p->T * p->K;
    for (size_t i = 0; i < (size_t)p->T * p->H; ++i) out[i] = 0.0;
    for (size_t i = 0; i < na; ++i)
        if (ids[i] < 0 || ids[i] >= p->E) return -1;
    double* xrow = (double*)malloc(sizeof(double) * p->H);
    double* wrow = (double*)malloc(sizeof(double) * max_int(p->H, p->I));
    double* a = (double*)malloc(sizeof(double) * p->I);
    double* y = (double*)malloc(sizeof(double) * p->H);
    for (int e = p->expert_base; e < p->expert_base + shard_size(p); ++e) {
        int el = e - p->expert_base;
        for (size_t i = 0; i < na; ++i) {
            if (ids[i] != e) continue;
            int t = (int)(i / (size_t)p->K);
            load_token_row(p, x, t, xrow);
            expert_hidden(p, w13, w13_scale, el, xrow, a, wrow);
            for (int j = 0; j < p->I; ++j) a[j] = store_hidden(p, mode, a[j]);
            expert_out(p, w2, w2_scale, el, a, y, wrow);
            for (int c = 0; c < p->H; ++c) out[(size_t)t * p->H + c] += (double)topk_w[i] * y[c];
        }
    }
    free(xrow);
    free(wrow);
    free(a);
    free(y);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Per-stage definitions (for stage-level parity)                      */
/* ------------------------------------------------------------------ */

/* GEMM1 + SiLU*up on sorted slots: h[r, :] = a(token of slot rows[r]) for
 * expert expert_of_row[r].  The token of a flat index i is i / K ([P2]
 * init_routing_data: gather_indx = combine_indx // k).  Slots holding the
 * sentinel (i >= T*K) give no row (h left untouched). */
void orc_gemm1_silu_rows(const orc_problem* p, int mode, const void* x, const void* w13,
                         const uint8_t* w13_scale, const int32_t* sorted_ids,
                         const int32_t* expert_of_row, const int32_t* rows, int n_rows, double* h) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < n_rows; ++r) {
        int i = sorted_ids[rows[r]];
        if (i < 0 || i >= p->T * p->K) continue;
        double* xrow = (double*)malloc(sizeof(double) * p->H);
        double* wrow = (double*)malloc(sizeof(double) * max_int(p->H, p->I));
        double* a = (double*)malloc(sizeof(double) * p->I);
        load_token_row(p, x, i / p->K, xrow);
        expert_hidden(p, w13, w13_scale, expert_of_row[r], xrow, a, wrow);
        for (int j = 0; j < p->I; ++j) h[(size_t)r * p->I + j] = store_hidden(p, mode, a[j]);
        free(xrow);
        free(wrow);
        free(a);
    }
}

/* GEMM2 + routing weight on sorted slots: y[r, :] = w_i * W2[e] . hin[row],
 * where hin is an (rows_total, I) activation tensor stored as `h_dtype`
 * (ORC_F32 / ORC_BF16, or 2 for e4m3 codes times h_scale). */
void orc_gemm2_weighted_rows(const orc_problem* p, const void* hin, int h_dtype, const void* w2,
                             const uint8_t* w2_scale, const float* topk_w,
                             const int32_t* sorted_ids, const int32_t* expert_of_row,
                             const int32_t* rows, int n_rows, double* y) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < n_rows; ++r) {
        int i = sorted_ids[rows[r]];
        if (i < 0 || i >= p->T * p->K) continue;
        double* a = (double*)malloc(sizeof(double) * p->I);
        double* wrow = (double*)malloc(sizeof(double) * max_int(p->H, p->I));
        double* yr = (double*)malloc(sizeof(double) * p->H);
        size_t base = (size_t)rows[r] * p->I;
        for (int j = 0; j < p->I; ++j) {
            if (h_dtype == 2)
                a[j] = orc_e4m3_to_double(((const uint8_t*)hin)[base + j]) * p->h_scale;
            else
                a[j] = load_act(hin, h_dtype, base + j);
        }
        expert_out(p, w2, w2_scale, expert_of_row[r], a, yr, wrow);
        for (int c = 0; c < p->H; ++c) y[(size_t)r * p->H + c] = (double)topk_w[i] * yr[c];
        free(a);
        free(wrow);
        free(yr);
    }
}

/* Combine: out[t, :] = sum_{k} y[inv_perm[t*K + k], :] summed in k order
 * (the index_add of [P3]'s PyTorch path, in a fixed order).  A negative
 * slot (an assignment to another shard's expert) contributes nothing. */
void orc_combine(const float* y, const int32_t* inv_perm, int T, int K, int H, double* out) {
    for (int t = 0; t < T; ++t)
        for (int c = 0; c < H; ++c) {
            double s = 0.0;
            for (int k = 0; k < K; ++k) {
                int slot = inv_perm[(size_t)t * K + k];
                if (slot >= 0) s += (double)y[(size_t)slot * H + c];
            }
            out[(size_t)t * H + c] = s;
        }
}

/* ------------------------------------------------------------------ */
/* Router                                                              */
/* ------------------------------------------------------------------ */

/* Top-K routing of T tokens over E experts from their router logits
 * (logit_dtype ORC_F32 or ORC_BF16, (T, E) row-major): ids[t, 0..K-1] are
 * the experts of the K largest logits in descending order, an equal logit
 * going to the lower expert id; weights[t, k] is the softmax over the
 * experts, renormalised over the K chosen ones, which equals the softmax
 * over the K chosen logits alone:
 *   w_k = exp(l_k - l_0) / sum_j exp(l_j - l_0).
 * Source: "MOE Bmm1 Fused Gather", init_routing_data (topk with
 * apply_softmax over the router logits, whose histogram feeds the ragged
 * metadata).  The softmax is monotone, so ranking the logits ranks the
 * probabilities; ranking the logits keeps the choice exact.  Computed in
 * fp64.  Returns 0, or -1 when K is outside [1, E]. */
int orc_route(const void* logits, int logit_dtype, int T, int E, int K, int32_t* ids,
              double* weights) {
    if (K < 1 || K > E) return -1;
    char* taken = (char*)malloc((size_t)E);
    double* v = (double*)malloc(sizeof(double) * (size_t)K);
    for (int t = 0; t < T; ++t) {
        memset(taken, 0, (size_t)E);
        for (int k = 0; k < K; ++k) {
            int best = -1;
            double bv = 0.0;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                double l = load_act(logits, logit_dtype, (size_t)t * E + e);
                if (best < 0 || l > bv) { /* strictly larger: ties keep the lower id */
                    best = e;
                    bv = l;
                }
            }
            taken[best] = 1;
            ids[(size_t)t * K + k] = best;
            v[k] = bv;
        }
        double sum = 0.0;
        for (int k = 0; k < K; ++k) sum += exp(v[k] - v[0]);
        for (int k = 0; k < K; ++k) weights[(size_t)t * K + k] = exp(v[k] - v[0]) / sum;
    }
    free(taken);
    free(v);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Align                                                               */
/* ------------------------------------------------------------------ */

/* Capacity of the padded sorted list: every active expert wastes at most
 * bm-1 slots, and at most min(E, T*K) experts are active. */
long orc_align_capacity(int T, int K, int E, int bm) {
    long na = (long)T * K;
    long act = na < E ? na : E;
    return na + act * (bm - 1);
}

/* Align top-k ids into per-expert, bm-padded lists.  With i = t*K + k:
 *   counts[e]          = #{i : ids[i] = e}              ([P3] build_expert_map_kernel)
 *   offsets            = exclusive prefix sum of counts (CSR offsets, length E+1)
 *   padded_offsets     = exclusive prefix sum of ceil(counts/bm)*bm
 *   sorted_ids[po[e]+r]= the r-th smallest i with ids[i] = e   (reading: stable,
 *                        ascending flat index; [P3] leaves the order to atomics)
 *   every other slot < cap holds the sentinel T*K         ([P2] load_activations
 *                        masks padded rows)
 *   inv_perm[i]        = the slot of i
 *   block_info[b]      = (expert, m-index, first slot, valid rows) for the
 *                        num_blocks = po[E]/bm blocks in expert order ([P1]
 *                        mblocks_to_tuple_info); (-1, 0, 0, 0) past them.
 * Expert-parallel shard of L experts from `base` ([P2] init_routing_data
 * keeps the local experts' histogram): every per-expert array above runs
 * over the local experts e - base, ids of other experts are left out of
 * the lists and get inv_perm[i] = -1, and the capacity counts min(L, T*K)
 * active experts.  base = 0, L = E is the plain align.
 * The sorted order is built by scanning i in ascending order once per expert.
 * Returns 0, or -1 when an id is outside [0, E). */
int orc_align_local(const int32_t* ids, int T, int K, int E, int base, int L, int bm,
                    int32_t* counts, int32_t* offsets, int32_t* padded_offsets,
                    int32_t* sorted_ids, int32_t* inv_perm, int32_t* block_info,
                    int32_t* num_blocks) {
    long na = (long)T * K;
    long cap = orc_align_capacity(T, K, L, bm);
    for (long i = 0; i < na; ++i)
        if (ids[i] < 0 || ids[i] >= E) return -1;
    for (int e = 0; e < L; ++e) counts[e] = 0;
    for (long i = 0; i < na; ++i) {
        inv_perm[i] = -1;
        if (ids[i] >= base && ids[i] < base + L) counts[ids[i] - base] += 1;
    }
    offsets[0] = 0;
    padded_offsets[0] = 0;
    for (int e = 0; e < L; ++e) {
        offsets[e + 1] = offsets[e] + counts[e];
        padded_offsets[e + 1] = padded_offsets[e] + (counts[e] + bm - 1) / bm * bm;
    }
    for (long s = 0; s < cap; ++s) sorted_ids[s] = (int32_t)na;
    for (int e = base; e < base + L; ++e) {
        int r = 0;
        for (long i = 0; i < na; ++i) {
            if (ids[i] != e) continue;
            sorted_ids[padded_offsets[e - base] + r] = (int32_t)i;
            inv_perm[i] = padded_offsets[e - base] + r;
            ++r;
        }
    }
    int nb = padded_offsets[L] / bm;
    *num_blocks = nb;
    long max_blocks = cap / bm;
    for (long b = 0; b < max_blocks; ++b) {
        int32_t* bi = block_info + 4 * b;
        bi[0] = -1;
        bi[1] = 0;
        bi[2] = 0;
        bi[3] = 0;
    }
    int b = 0;
    for (int e = 0; e < L; ++e) {
        int nblk = (padded_offsets[e + 1] - padded_offsets[e]) / bm;
        for (int m = 0; m < nblk; ++m, ++b) {
            int32_t* bi = block_info + 4 * (long)b;
            int left = counts[e] - m * bm;
            bi[0] = e;
            bi[1] = m;
            bi[2] = b * bm;
            bi[3] = left < bm ? left : bm;
        }
    }
    return 0;
}

/* The plain align: one shard holding all E experts. */
int orc_align(const int32_t* ids, int T, int K, int E, int bm, int32_t* counts, int32_t* offsets,
              int32_t* padded_offsets, int32_t* sorted_ids, int32_t* inv_perm, int32_t* block_info,
              int32_t* num_blocks) {
    return orc_align_local(ids, T, K, E, 0, E, bm, counts, offsets, padded_offsets, sorted_ids,
                           inv_perm, block_info, num_blocks);
}
