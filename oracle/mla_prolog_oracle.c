/*
 * Plain CPU oracle of the fused MLA attention prolog.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code with the CUDA library.
 *
 * It is deliberately slow and literal: plain loops over tokens and columns,
 * the steps in the order the pages give them, no blocking and no fusion.
 * OpenMP splits the independent token rows over host threads; the arithmetic
 * of one row does not depend on the thread count.
 *
 * Precision of each step:
 *   - GEMM dot products: the pages fix only the output type (BF16 for the
 *     compression and KV expansion projections), so the oracle forms the
 *     plain definition -- the sum of exact BF16 x BF16 products -- in float64
 *     and rounds it once to the output type.
 *   - RMSNorm: FP32 throughout, as the pages fix it ("PyPTO-Gym 算子设计模式
 *     AT-10", section 三, variant B: x^2, times 1/L, sum, + eps, sqrt, 1/std,
 *     x * rstd), then * gamma in FP32 and a cast to BF16 (section 五).
 *   - RoPE: FP32 rotate-half, out = x*cos + rotate_half(x)*sin, with
 *     rotate_half(x1, x2) = (-x2, x1) (DeepSeek-V3.2-Exp PyPTO article,
 *     section 3.3 QuantRope; V2-Lite migration guide, section "精度验证").
 *   - Per-token INT8 quant: FP32 chain amax = max|y|, inv = 127/amax,
 *     code = rint(y * inv) (round half to even), clamp to +-127,
 *     scale = amax / 127 (DeepSeek-V3.2-Exp PyPTO article, section 3.1
 *     PrologQuant; grouped_matmul_swiglu_quant article, sections "数学公式" and
 *     "5. 量化流水线的数值细节").
 *
 *   - Variants (flags): ORACLE_ROPE_INTERLEAVED de-interleaves each rope
 *     slice before the rotate-half RoPE (QuantRope3D, DeepSeek-V3.2-Exp
 *     PyPTO article, section 3.3); ORACLE_Q_HEAD_NORM applies a per-head FP32
 *     RMSNorm without gamma to every q head before its RoPE (AT-10 article,
 *     section 九, the DeepSeek-V4 q path); ORACLE_QUANT_PER_HEAD quantises
 *     each (token, head) row of Dn + R values with its own scale (the quant
 *     formula of section 3.1 applied per head row).
 *
 *   - W8A8 projections (oracle_mla_prolog_w8a8): the INT8 mode of the Linear
 *     step (PyPTO-Gym AT-10 article, section 四, AT-09 "INT8 W8A8"):
 *     the activation row is quantised per token with the formula above
 *     (AT-05), the product is the exact integer sum of code x code
 *     (int32 result; formed here in int64, which cannot overflow), and AT-06
 *     turns it back into FP32 as ((float)y_int32 * a_scale) * w_scale, one
 *     correctly rounded FP32 operation per step.  Every projection of the
 *     prolog runs that way: x -> compression (then the BF16 cast the BF16
 *     mode also has), the normed c_q / c_kv rows (after their BF16 cast) ->
 *     q and KV expansion; with a quantised Linear the norm block becomes
 *     RMSNorm + Linear + Quant (AT-11, V -> C -> V).
 *
 * Readings where the pages are silent (the pages fix none of these; each is
 * the plainest reading that the passages cited above support):
 *   - W8A8: one FP32 weight scale per output row of each weight matrix; the
 *     quantised matmul input is the tensor the BF16 mode feeds to the
 *     matmul (x; the normed rows after their BF16 cast); AT-06 multiplies
 *     left to right: (y * a_scale) * w_scale;
 *   - a zero row (amax == 0) yields codes 0 and scale 0;
 *   - a position outside [0, max_pos) zero-fills every output of that token
 *     and is reported in the return value;
 *   - q is kept in FP32 after its projection and RoPE; the quant reads FP32.
 *
 * Build: cc -O2 -ffp-contract=off -fopenmp -fPIC -shared (no -ffast-math),
 * so every FP32 operation below is one IEEE-754 operation, rounded to nearest.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_QUANT_Q 1u
#define ORACLE_ROPE_INTERLEAVED 2u
#define ORACLE_Q_HEAD_NORM 4u
#define ORACLE_QUANT_PER_HEAD 8u
#define ORACLE_W8A8 16u

typedef struct {
    int32_t T, D, q_lora_rank, kv_lora_rank, rope_dim, num_heads, nope_dim, v_dim, max_pos;
    float eps;
    uint32_t flags;
} oracle_dims;

/* ---------------------------------------------------------------- BF16 -- */

/* Widen BF16 bits to FP32: the BF16 bits are the upper half of the FP32. */
static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* FP32 -> BF16, round to nearest, ties to even, on the bit pattern. */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) /* NaN: keep it quiet */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* float64 -> BF16 with a single rounding: the value rounded to 8 significant
 * bits (to nearest, ties to even), or to a multiple of 2^-133 in BF16's
 * subnormal range. */
uint16_t oracle_f64_to_bf16(double v) {
    if (isnan(v)) return 0x7fc0u;
    if (v == 0.0) return signbit(v) ? 0x8000u : 0x0000u;
    int e;
    (void)frexp(v, &e);                 /* v = m * 2^e, 0.5 <= |m| < 1 */
    int q = e - 8;                      /* quantum exponent for 8 significant bits */
    if (q < -133) q = -133;             /* BF16 subnormal spacing */
    double r = nearbyint(ldexp(v, -q)); /* default rounding mode: to nearest even */
    double w = ldexp(r, q);
    if (fabs(w) >= 0x1p128) return signbit(v) ? 0xff80u : 0x7f80u; /* overflow to inf */
    float f = (float)w;                 /* exact: w has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------ steps ----- */

/* One output of a projection with weights in [N, K] layout:
 * sum_k a[k] * w[n, k] in float64 (each BF16 x BF16 product is exact). */
static double dot_bf16_f64(const uint16_t* a, const uint16_t* w_row, int K) {
    double acc = 0.0;
    for (int k = 0; k < K; ++k)
        acc += (double)bf16_to_f32(a[k]) * (double)bf16_to_f32(w_row[k]);
    return acc;
}

/* Compression projection of one token row, rounded to BF16:
 * c[n] = bf16( sum_k x[k] * W_a[n, k] ), n in [0, N). */
void oracle_project_bf16(const uint16_t* x_row, const uint16_t* W, int N, int K, uint16_t* out) {
    for (int n = 0; n < N; ++n)
        out[n] = oracle_f64_to_bf16(dot_bf16_f64(x_row, W + (size_t)n * K, K));
}

/* Expansion projection of one normed row, rounded to FP32. */
void oracle_project_f32(const uint16_t* a_row, const uint16_t* W, int N, int K, float* out) {
    for (int n = 0; n < N; ++n)
        out[n] = (float)dot_bf16_f64(a_row, W + (size_t)n * K, K);
}

/* RMSNorm of one row of L BF16 values with BF16 gamma, FP32 inside.
 * y_f32 (optional) receives x * rstd * gamma before the BF16 cast. */
void oracle_rmsnorm_row(const uint16_t* x, const uint16_t* gamma, int L, float eps,
                        float* y_f32, uint16_t* y_bf16) {
    const float inv_L = (float)(1.0 / (double)L);
    float ms = 0.0f;
    for (int i = 0; i < L; ++i) {
        float v = bf16_to_f32(x[i]);
        float sq = v * v;
        ms += sq * inv_L;
    }
    float var = ms + eps;
    float stdv = sqrtf(var);
    float rstd = 1.0f / stdv;
    for (int i = 0; i < L; ++i) {
        float y = bf16_to_f32(x[i]) * rstd;
        y = y * (gamma ? bf16_to_f32(gamma[i]) : 1.0f);
        if (y_f32) y_f32[i] = y;
        if (y_bf16) y_bf16[i] = oracle_f32_to_bf16(y);
    }
}

/* Rotate-half RoPE of R values in FP32 with the table row (cos | sin):
 * out[i]       = x[i] * c_i + (-x[i + R/2]) * s_i
 * out[i + R/2] = x[i + R/2] * c_i + x[i] * s_i,   i < R/2. */
void oracle_rope_f32(const float* x, const float* cs_row, int R, float* out) {
    const int h = R / 2;
    for (int i = 0; i < h; ++i) {
        float c = cs_row[i], s = cs_row[h + i];
        float x1 = x[i], x2 = x[h + i];
        float a = x1 * c;
        float b = (-x2) * s;
        float e = x2 * c;
        float f = x1 * s;
        out[i] = a + b;
        out[h + i] = e + f;
    }
}

/* The de-interleave of QuantRope3D (DeepSeek-V3.2-Exp PyPTO article,
 * section 3.3 and section 2.3): the R rope values are viewed as [R/2, 2]
 * (chunks of 2) and transposed to [2, R/2], so out[i] = x[2i] and
 * out[R/2 + i] = x[2i + 1]; the rotate-half RoPE then pairs the values that
 * sat next to each other.  The result stays in the transposed order. */
void oracle_deinterleave(const float* x, int R, float* out) {
    const int h = R / 2;
    for (int i = 0; i < h; ++i) {
        out[i] = x[2 * i];
        out[h + i] = x[2 * i + 1];
    }
}

/* RMSNorm of one FP32 row without gamma, FP32 in and out: the second,
 * per-head RMSNorm of the DeepSeek-V4 q path (PyPTO-Gym AT-10 article,
 * section 九: q_b_proj, reshape to (heads, head_dim), RMSNorm again; the
 * no-gamma variant rms_norm_new of the same section), with the variant-B
 * steps of section 三: x^2, times 1/L, sum, + eps, sqrt, 1/std, x * rstd. */
void oracle_rmsnorm_f32_row(const float* x, int L, float eps, float* out) {
    const float inv_l = 1.0f / (float)L;
    float ms = 0.0f;
    for (int i = 0; i < L; ++i) {
        float sq = x[i] * x[i];
        ms += sq * inv_l;
    }
    float var = ms + eps;
    float sd = sqrtf(var);
    float rstd = 1.0f / sd;
    for (int i = 0; i < L; ++i) out[i] = x[i] * rstd;
}

/* Per-token symmetric INT8 quantisation of one FP32 row. */
void oracle_quant_row(const float* y, int n, int8_t* codes, float* scale) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(y[i]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
        for (int i = 0; i < n; ++i) codes[i] = 0;
        *scale = 0.0f;
        return;
    }
    float inv = 127.0f / amax;
    for (int i = 0; i < n; ++i) {
        float v = y[i] * inv;
        float r = rintf(v); /* round half to even (default rounding mode) */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        codes[i] = (int8_t)r;
    }
    *scale = amax / 127.0f;
}

/* Exact integer product of two INT8 code rows of length K (the int32 matmul
 * of the W8A8 Linear, PyPTO-Gym AT-10 article, section 四): the sum of
 * code x code in int64, which holds it exactly for any K used here. */
int64_t oracle_dot_i8(const int8_t* a, const int8_t* w_row, int K) {
    int64_t acc = 0;
    for (int k = 0; k < K; ++k) acc += (int64_t)a[k] * (int64_t)w_row[k];
    return acc;
}

/* AT-06 dequantisation of one int32 product: FP32 (y * a_scale) * w_scale,
 * the int32 -> FP32 conversion rounded to nearest. */
float oracle_dequant(int32_t y, float a_scale, float w_scale) {
    float f = (float)y;
    float g = f * a_scale;
    return g * w_scale;
}

/* One W8A8 projection of a quantised row: out[n] = AT-06(sum_k a[k] W[n,k],
 * a_scale, w_scale[n]), n in [0, N), W INT8 codes in [N, K] layout. */
void oracle_project_w8a8(const int8_t* a_codes, const int8_t* W, int N, int K, float a_scale,
                         const float* w_scale, float* out) {
    for (int n = 0; n < N; ++n)
        out[n] = oracle_dequant((int32_t)oracle_dot_i8(a_codes, W + (size_t)n * K, K), a_scale, w_scale[n]);
}

/* The W8A8 operands and taps of one prolog run (NULL in the BF16 mode). */
typedef struct {
    const int8_t* W_a;     /* [NA, D] codes                                     */
    const int8_t* W_b;     /* W_q_b [NQ, Lq] codes, then W_kv_b [NKV, Lkv]       */
    const float* w_scale;  /* [NA + (Lq > 0 ? NQ : 0) + NKV]: one per weight row */
    int8_t* x_codes;       /* taps (NULL to skip): x codes [n, D]               */
    float* x_scale;        /*   x scales [n]                                    */
    int8_t* n_codes;       /*   normed c_q | c_kv codes [n, Lq + Lkv]           */
    float* n_scale;        /*   their scales [n, 2] = (c_q, c_kv)               */
    const int8_t* given_codes; /* optional [n, Lq + Lkv]: the expansions take   */
    const float* given_scale;  /*   these codes and [n, 2] scales instead       */
} oracle_w8a8;

/* ------------------------------------------------------------ whole op -- */

/*
 * Runs the whole prolog for the tokens listed in `tokens` (all T tokens when
 * `tokens` is NULL, n_tokens then ignored).  Output rows are compact: row j
 * of every output belongs to token tokens[j].
 *
 * Optional taps (NULL to skip), also compact by selected token:
 *   c_out      BF16 [n, Lq+Lkv+R]  compression output after the BF16 cast
 *   normed_out BF16 [n, Lq+Lkv]    normed c_q | c_kv after gamma and the cast
 *   q_out      FP32 [n, H*(Dn+R)]  q after projection and RoPE (the quant input)
 *
 * Returns the number of selected tokens whose position was out of range
 * (their outputs are zero-filled), or -1 on bad arguments.
 */
static int prolog(const oracle_dims* d,
                  const uint16_t* x, const uint16_t* gamma,
                  const uint16_t* W_a, const uint16_t* W_b, const oracle_w8a8* w8,
                  const int32_t* positions, const float* cos_sin,
                  const int32_t* tokens, int32_t n_tokens,
                  uint16_t* out_k, uint16_t* out_v, uint16_t* out_kpe,
                  int8_t* out_q_int8, float* out_scale,
                  uint16_t* c_out, uint16_t* normed_out, float* q_out) {
    if (!d || !x || !positions || !cos_sin || !out_k || !out_v || !out_kpe) return -1;
    if (w8 ? (!w8->W_a || !w8->W_b || !w8->w_scale || W_a || W_b) : (!W_a || !W_b)) return -1;
    if (((d->flags & ORACLE_W8A8) != 0) != (w8 != NULL)) return -1;
    const int T = d->T, D = d->D, Lq = d->q_lora_rank, Lkv = d->kv_lora_rank, R = d->rope_dim;
    const int H = d->num_heads, Dn = d->nope_dim, Dv = d->v_dim;
    const int NA = Lq + Lkv + R, NQ = H * (Dn + R);
    const int quant = (d->flags & ORACLE_QUANT_Q) != 0;
    const int interleaved = (d->flags & ORACLE_ROPE_INTERLEAVED) != 0;
    const int head_norm = (d->flags & ORACLE_Q_HEAD_NORM) != 0;
    const int per_head = (d->flags & ORACLE_QUANT_PER_HEAD) != 0;
    if (T < 0 || D <= 0 || Lq < 0 || Lkv <= 0 || R <= 0 || (R & 1) || H <= 0 || Dn < 0 || Dv < 0)
        return -1;
    if ((Lq + Lkv) > 0 && !gamma) return -1;
    if (Lq > 0 && (!quant || !out_q_int8 || !out_scale)) return -1;
    const int n = tokens ? n_tokens : T;
    if (n < 0) return -1;
    const uint16_t* W_qb = W_b;                                   /* [NQ, Lq]  */
    const uint16_t* W_kvb = W_b ? W_b + (size_t)NQ * Lq : NULL;  /* [NKV, Lkv] */
    const int NKV = H * (Dn + Dv);
    const int NQw = Lq > 0 ? NQ : 0;  /* rows of W_q_b */
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (int j = 0; j < n; ++j) {
        const int t = tokens ? tokens[j] : j;
        uint16_t* ok = out_k + (size_t)j * H * (Dn + R);
        uint16_t* ov = out_v + (size_t)j * H * Dv;
        uint16_t* okpe = out_kpe + (size_t)j * R;
        if (t < 0 || t >= T) { bad += 1; continue; }
        /* W8A8, AT-05 on x: the per-token codes of the compression's input
         * (they do not depend on the position). */
        int8_t* xq = NULL;
        float sx = 0.0f;
        if (w8) {
            float* xf = (float*)malloc(sizeof(float) * (size_t)D);
            xq = (int8_t*)malloc((size_t)D);
            for (int k = 0; k < D; ++k) xf[k] = bf16_to_f32(x[(size_t)t * D + k]);
            oracle_quant_row(xf, D, xq, &sx);
            if (w8->x_codes) memcpy(w8->x_codes + (size_t)j * D, xq, (size_t)D);
            if (w8->x_scale) w8->x_scale[j] = sx;
            free(xf);
        }
        const int32_t pos = positions[t];
        if (pos < 0 || pos >= d->max_pos) {
            free(xq);
            if (w8 && w8->n_codes) memset(w8->n_codes + (size_t)j * (Lq + Lkv), 0, (size_t)(Lq + Lkv));
            if (w8 && w8->n_scale) w8->n_scale[2 * j] = w8->n_scale[2 * j + 1] = 0.0f;
            memset(ok, 0, sizeof(uint16_t) * (size_t)H * (Dn + R));
            memset(ov, 0, sizeof(uint16_t) * (size_t)H * Dv);
            memset(okpe, 0, sizeof(uint16_t) * (size_t)R);
            if (Lq > 0) {
                memset(out_q_int8 + (size_t)j * NQ, 0, (size_t)NQ);
                if (per_head)
                    memset(out_scale + (size_t)j * H, 0, sizeof(float) * (size_t)H);
                else
                    out_scale[j] = 0.0f;
            }
            if (c_out) memset(c_out + (size_t)j * NA, 0, sizeof(uint16_t) * (size_t)NA);
            if (normed_out) memset(normed_out + (size_t)j * (Lq + Lkv), 0, sizeof(uint16_t) * (size_t)(Lq + Lkv));
            if (q_out) memset(q_out + (size_t)j * NQ, 0, sizeof(float) * (size_t)NQ);
            bad += 1;
            continue;
        }
        const float* cs = cos_sin + (size_t)pos * R;
        uint16_t* c = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)NA);
        uint16_t* nrm = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(Lq + Lkv));
        float* kpe_f = (float*)malloc(sizeof(float) * (size_t)R);
        float* kpe_r = (float*)malloc(sizeof(float) * (size_t)R);

        /* Step 1: compression projection x . W_a^T, each output rounded to BF16
         * (W8A8: the integer product of the codes, dequantised, then rounded). */
        if (w8) {
            float* cf = (float*)malloc(sizeof(float) * (size_t)NA);
            oracle_project_w8a8(xq, w8->W_a, NA, D, sx, w8->w_scale, cf);
            for (int i = 0; i < NA; ++i) c[i] = oracle_f32_to_bf16(cf[i]);
            free(cf);
        } else {
            oracle_project_bf16(x + (size_t)t * D, W_a, NA, D, c);
        }
        /* Step 2: split -- c_q = c[0, Lq), c_kv = c[Lq, Lq+Lkv), k_pe = c[Lq+Lkv, NA). */
        /* Step 3: RMSNorm of c_q and c_kv with their gammas, then BF16. */
        if (Lq > 0) oracle_rmsnorm_row(c, gamma, Lq, d->eps, NULL, nrm);
        oracle_rmsnorm_row(c + Lq, gamma + Lq, Lkv, d->eps, NULL, nrm + Lq);
        /* W8A8 (AT-11): the normed BF16 rows c_q and c_kv, each quantised per
         * token, are the expansions' inputs. */
        int8_t* nq = NULL;
        float sq = 0.0f, skv = 0.0f;
        if (w8) {
            float* nf = (float*)malloc(sizeof(float) * (size_t)(Lq + Lkv));
            nq = (int8_t*)malloc((size_t)(Lq + Lkv));
            for (int i = 0; i < Lq + Lkv; ++i) nf[i] = bf16_to_f32(nrm[i]);
            if (Lq > 0) oracle_quant_row(nf, Lq, nq, &sq);
            oracle_quant_row(nf + Lq, Lkv, nq + Lq, &skv);
            if (w8->n_codes) memcpy(w8->n_codes + (size_t)j * (Lq + Lkv), nq, (size_t)(Lq + Lkv));
            if (w8->n_scale) w8->n_scale[2 * j] = sq, w8->n_scale[2 * j + 1] = skv;
            /* Given codes (a candidate's own normed-row codes and scales):
             * every step after the quantisation runs on them instead. */
            if (w8->given_codes) {
                memcpy(nq, w8->given_codes + (size_t)j * (Lq + Lkv), (size_t)(Lq + Lkv));
                sq = w8->given_scale[2 * j];
                skv = w8->given_scale[2 * j + 1];
            }
            free(nf);
        }
        /* Step 4 (k_pe RoPE): rotate-half in FP32 with this token's table row
         * (after the de-interleave in the interleaved variant). */
        for (int i = 0; i < R; ++i) kpe_f[i] = bf16_to_f32(c[Lq + Lkv + i]);
        if (interleaved) {
            oracle_deinterleave(kpe_f, R, kpe_r);
            memcpy(kpe_f, kpe_r, sizeof(float) * (size_t)R);
        }
        oracle_rope_f32(kpe_f, cs, R, kpe_r);
        for (int i = 0; i < R; ++i) okpe[i] = oracle_f32_to_bf16(kpe_r[i]);
        /* Steps 5-7: KV expansion, split per head into k_nope | value, assemble
         * K = [k_nope | k_pe_rot] with the rotated k_pe shared by every head. */
        float* kvf = NULL;
        if (w8) {
            kvf = (float*)malloc(sizeof(float) * (size_t)NKV);
            oracle_project_w8a8(nq + Lq, w8->W_b + (size_t)NQw * Lq, NKV, Lkv, skv, w8->w_scale + NA + NQw, kvf);
        }
        for (int h = 0; h < H; ++h) {
            const uint16_t* Wh = w8 ? NULL : W_kvb + (size_t)h * (Dn + Dv) * Lkv;
            for (int i = 0; i < Dn; ++i)
                ok[(size_t)h * (Dn + R) + i] =
                    w8 ? oracle_f32_to_bf16(kvf[(size_t)h * (Dn + Dv) + i])
                       : oracle_f64_to_bf16(dot_bf16_f64(nrm + Lq, Wh + (size_t)i * Lkv, Lkv));
            for (int i = 0; i < Dv; ++i)
                ov[(size_t)h * Dv + i] =
                    w8 ? oracle_f32_to_bf16(kvf[(size_t)h * (Dn + Dv) + Dn + i])
                       : oracle_f64_to_bf16(dot_bf16_f64(nrm + Lq, Wh + (size_t)(Dn + i) * Lkv, Lkv));
            for (int i = 0; i < R; ++i) ok[(size_t)h * (Dn + R) + Dn + i] = okpe[i];
        }
        free(kvf);
        /* q path: expansion, (per-head RMSNorm,) RoPE on each head's rope
         * slice, INT8 quant per token (or per head row). */
        if (Lq > 0) {
            float* q = (float*)malloc(sizeof(float) * (size_t)NQ);
            float* hb = (float*)malloc(sizeof(float) * (size_t)(Dn + R));
            if (w8)
                oracle_project_w8a8(nq, w8->W_b, NQ, Lq, sq, w8->w_scale + NA, q);
            else
                oracle_project_f32(nrm, W_qb, NQ, Lq, q);
            for (int h = 0; h < H; ++h) {
                float* qh = q + (size_t)h * (Dn + R);
                if (head_norm) {
                    oracle_rmsnorm_f32_row(qh, Dn + R, d->eps, hb);
                    memcpy(qh, hb, sizeof(float) * (size_t)(Dn + R));
                }
                float* qr = qh + Dn;
                if (interleaved)
                    oracle_deinterleave(qr, R, kpe_f);
                else
                    memcpy(kpe_f, qr, sizeof(float) * (size_t)R);
                oracle_rope_f32(kpe_f, cs, R, qr);
            }
            if (q_out) memcpy(q_out + (size_t)j * NQ, q, sizeof(float) * (size_t)NQ);
            if (per_head) {
                for (int h = 0; h < H; ++h)
                    oracle_quant_row(q + (size_t)h * (Dn + R), Dn + R, out_q_int8 + (size_t)j * NQ + (size_t)h * (Dn + R),
                                     out_scale + (size_t)j * H + h);
            } else {
                oracle_quant_row(q, NQ, out_q_int8 + (size_t)j * NQ, out_scale + j);
            }
            free(hb);
            free(q);
        }
        if (c_out) memcpy(c_out + (size_t)j * NA, c, sizeof(uint16_t) * (size_t)NA);
        if (normed_out) memcpy(normed_out + (size_t)j * (Lq + Lkv), nrm, sizeof(uint16_t) * (size_t)(Lq + Lkv));
        free(c); free(nrm); free(kpe_f); free(kpe_r); free(xq); free(nq);
    }
    return bad;
}

int oracle_mla_prolog(const oracle_dims* d,
                      const uint16_t* x, const uint16_t* gamma,
                      const uint16_t* W_a, const uint16_t* W_b,
                      const int32_t* positions, const float* cos_sin,
                      const int32_t* tokens, int32_t n_tokens,
                      uint16_t* out_k, uint16_t* out_v, uint16_t* out_kpe,
                      int8_t* out_q_int8, float* out_scale,
                      uint16_t* c_out, uint16_t* normed_out, float* q_out) {
    return prolog(d, x, gamma, W_a, W_b, NULL, positions, cos_sin, tokens, n_tokens, out_k, out_v, out_kpe,
                  out_q_int8, out_scale, c_out, normed_out, q_out);
}

/*
 * The prolog with W8A8 projections (dims flag ORACLE_W8A8): arguments as
 * oracle_mla_prolog, with the INT8 weights and their row scales in place of
 * the BF16 weights, and four more optional taps (x codes and scales, the
 * normed rows' codes and scales; see oracle_w8a8).  normed_out still
 * receives the normed BF16 values, before their quantisation.
 *
 * given_codes / given_scale (optional, compact by selected token like the
 * outputs): normed-row codes [n, Lq + Lkv] and scales [n, 2] that the two
 * expansion projections take in place of the oracle's own.  A candidate whose
 * normed rows legitimately differ (the RMSNorm's FP32 sum of squares may run
 * in another order) is then checked step for step after that point: the
 * integer products, AT-06, RoPE, the split / assemble and the q quant.  The
 * n_codes / n_scale taps still report the oracle's own codes.
 */
int oracle_mla_prolog_w8a8(const oracle_dims* d,
                           const uint16_t* x, const uint16_t* gamma,
                           const int8_t* W_a, const int8_t* W_b, const float* w_scale,
                           const int32_t* positions, const float* cos_sin,
                           const int32_t* tokens, int32_t n_tokens,
                           uint16_t* out_k, uint16_t* out_v, uint16_t* out_kpe,
                           int8_t* out_q_int8, float* out_scale,
                           uint16_t* c_out, uint16_t* normed_out, float* q_out,
                           int8_t* x_codes, float* x_scale, int8_t* n_codes, float* n_scale,
                           const int8_t* given_codes, const float* given_scale) {
    if ((given_codes == NULL) != (given_scale == NULL)) return -1;
    const oracle_w8a8 w8 = {W_a, W_b, w_scale, x_codes, x_scale, n_codes, n_scale, given_codes, given_scale};
    return prolog(d, x, gamma, NULL, NULL, &w8, positions, cos_sin, tokens, n_tokens, out_k, out_v, out_kpe,
                  out_q_int8, out_scale, c_out, normed_out, q_out);
}

/* Threads OpenMP will use for the next parallel region (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
