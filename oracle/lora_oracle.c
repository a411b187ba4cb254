/*
 * CPU oracle for the batched multi-adapter LoRA side branch.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may link,
 * load or call this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or constant with the CUDA
 * library: it is a plain, slow restatement of what the pages define, in double
 * precision, with no blocking, fusion or reordering.
 *
 * Notation (PEFT orientation, vLLM LoRA deep-dive page, §1 "LoRA 数学原理" and
 * §4 "完整推理流程": lora_a is (r, k), lora_b is (d, r)):
 *   x     [T, k]      input rows, one per token
 *   A_s,i [r_s, k]    down projection of slot s, output slice i
 *   B_s,i [d_i, r_s]  up projection of slot s, output slice i
 *   y     [T, d]      output rows; slice i occupies columns [o_i, o_i + d_i)
 *
 * Branch (llama.cpp LoRA adapter page, §"为什么低秩增量可以「后加」" and
 * §"真正的核心:建图时如何把低秩分支拼进去"; vLLM book ch. 16, §16.1.3
 * "推理时的叠加式计算"; TensorRT-LLM LoRA serving page, §"与基座并行:
 * forward_with_base", add_lora_result): for every token t whose slot
 * s = slot_ids[t] is in [0, S) with r_s > 0, for every slice i and column m:
 *     y[t, o_i + m] = y_in[t, o_i + m]
 *                     + scale_s * sum_j ( sum_c x[t,c] * A_s,i[j,c] ) * B_s,i[m,j]
 * Every other row is left as it was.  Slot -1 means "no adapter" (vLLM book
 * ch. 16, §16.4.2, token_lora_mapping).
 *
 * Index (TensorRT-LLM LoRA serving page, §"一次 decode 批次的路由", steps 2
 * and 4: sorted ids, bincount, cumsum with one extra entry holding the total;
 * vLLM book ch. 16, §16.4.3, the five LoRAKernelMeta tensors):
 *   key(t) = slot_ids[t] if 0 <= slot_ids[t] < S, else S (the "no adapter"
 *            bucket, placed last like TensorRT-LLM's sentinel slot);
 *   sorted_ids = tokens 0..T-1 in ascending key order, ties in ascending token
 *                index;
 *   seg_offsets[b] = #{t : key(t) < b} for b = 0..S+1;
 *   active = [count, s_1 < s_2 < ...] for slots with >= 1 token and r_s > 0.
 * A slot id outside [-1, S) is an error; the token goes to the last bucket and
 * is left unchanged by the branch.
 *
 * parity: pinned by tests/test_oracle_pins.py (library matmul, merged-weight
 * identity, closed forms, brute force over all permutations of tiny inputs).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_SLOT_RANGE 1

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_bf16_to_double(uint16_t bits) { return bf16_value(bits); }

/*
 * Round a double to the nearest bf16 (8 significant bits, binary32 exponent
 * range), ties to even, written from the format's definition: split off the
 * exponent, scale the significand to an integer grid, round half-to-even.
 */
uint16_t oracle_round_bf16(double v)
{
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);                 /* a = m * 2^e, 0.5 <= m < 1 */
    int q_exp = e - 8;                  /* quantum of an 8-bit significand */
    if (q_exp < -133) q_exp = -133;     /* subnormal quantum 2^(-126-7) */
    double scaled = ldexp(a, -q_exp);   /* exact: only the exponent changes */
    double fl = floor(scaled);
    double frac = scaled - fl;
    double q;
    if (frac > 0.5) q = fl + 1.0;
    else if (frac < 0.5) q = fl;
    else q = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double r = ldexp(q, q_exp);
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80); /* overflow to inf */
    float f = (float)r;                 /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

/*
 * Per-slot scale.  llama.cpp's get_scale (llama.cpp LoRA adapter page,
 * §"缩放系数到底乘在哪"): alpha ? adapter_scale * alpha / rank : adapter_scale.
 * rsLoRA (vLLM LoRA deep-dive page, §1, "rsLoRA 变体"): alpha / sqrt(rank).
 * The runtime strength multiplies either rule; alpha == 0 means "alpha/r is 1".
 */
double oracle_scale(double alpha, int32_t rank, int32_t rslora, double adapter_scale)
{
    if (alpha == 0.0 || rank <= 0) return adapter_scale;
    if (rslora) return adapter_scale * alpha / sqrt((double)rank);
    return adapter_scale * alpha / (double)rank;
}

/* Fold a scale into B (vLLM LoRA deep-dive page, §1 "推理优化:预合并 scaling",
 * LoRALayerWeights.optimize: lora_b *= scaling): bf16(s * B), nearest-even. */
void oracle_premultiply(const uint16_t *b, int64_t n, double s, uint16_t *out)
{
    for (int64_t e = 0; e < n; ++e) out[e] = oracle_round_bf16(s * bf16_value(b[e]));
}

typedef struct { int32_t key; int32_t t; } key_token_t;

static int cmp_key_token(const void *pa, const void *pb)
{
    const key_token_t *a = (const key_token_t *)pa, *b = (const key_token_t *)pb;
    if (a->key != b->key) return a->key < b->key ? -1 : 1;
    return a->t < b->t ? -1 : (a->t > b->t ? 1 : 0);
}

/* Returns ORACLE_OK or ORACLE_ERR_SLOT_RANGE (first error); outputs are always
 * written.  A comparison sort on unique (key, token) pairs gives the stable
 * order; the offsets are counted straight from their definition. */
int oracle_build_index(const int32_t *slot_ids, int32_t T, int32_t S, const int32_t *ranks,
                       int32_t *sorted_ids, int32_t *seg_offsets, int32_t *active)
{
    int status = ORACLE_OK;
    key_token_t *pairs = (key_token_t *)malloc(sizeof(key_token_t) * (size_t)(T > 0 ? T : 1));
    int32_t *key = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    for (int32_t t = 0; t < T; ++t) {
        int32_t s = slot_ids[t];
        if (s >= 0 && s < S) {
            key[t] = s;
        } else {
            key[t] = S;
            if (s != -1) status = ORACLE_ERR_SLOT_RANGE;
        }
        pairs[t].key = key[t];
        pairs[t].t = t;
    }
    qsort(pairs, (size_t)T, sizeof(key_token_t), cmp_key_token);
    for (int32_t p = 0; p < T; ++p) sorted_ids[p] = pairs[p].t;
    for (int32_t b = 0; b <= S + 1; ++b) {
        int32_t c = 0;
        for (int32_t t = 0; t < T; ++t) c += (key[t] < b);
        seg_offsets[b] = c;
    }
    int32_t n_active = 0;
    for (int32_t s = 0; s < S; ++s) {
        int32_t count = 0;
        for (int32_t t = 0; t < T; ++t) count += (key[t] == s);
        if (count > 0 && ranks[s] > 0) active[1 + n_active++] = s;
    }
    active[0] = n_active;
    free(pairs);
    free(key);
    return status;
}

/*
 * Shrink for a list of rows: xa[q][i][j] = sum_c x[t,c] * A_s,i[j,c] with
 * t = rows[q], s = slot_ids[t], j < r_s; entries j >= r_s and rows without an
 * active slot are left as they were.  A is indexed [s * n_slices + i].
 * *macs is increased by the multiply-adds performed.
 */
void oracle_shrink(const uint16_t *x, int64_t ldx, int32_t k, int32_t n_slices,
                   const int32_t *slot_ids, int32_t S, const int32_t *ranks,
                   const uint16_t *const *A, const int32_t *rows, int32_t n_rows,
                   int32_t r_max, double *xa, int64_t *macs)
{
    for (int32_t q = 0; q < n_rows; ++q) {
        int32_t t = rows[q];
        int32_t s = slot_ids[t];
        if (s < 0 || s >= S || ranks[s] <= 0) continue;
        const uint16_t *xt = x + (int64_t)t * ldx;
        for (int32_t i = 0; i < n_slices; ++i) {
            const uint16_t *a = A[(int64_t)s * n_slices + i];
            for (int32_t j = 0; j < ranks[s]; ++j) {
                double acc = 0.0;
                for (int32_t c = 0; c < k; ++c) acc += bf16_value(xt[c]) * bf16_value(a[(int64_t)j * k + c]);
                xa[((int64_t)q * n_slices + i) * r_max + j] = acc;
                *macs += k;
            }
        }
    }
}

/*
 * Full branch for a list of rows: y_out[q][:] is row rows[q] of the result, in
 * double, before any rounding to bf16.  y_in may be NULL (zeros).  scales are
 * per slot.  B is indexed [s * n_slices + i].  Returns ORACLE_ERR_SLOT_RANGE if
 * a listed row carries a slot id outside [-1, S).
 */
int oracle_apply(const uint16_t *x, int64_t ldx, const uint16_t *y_in, int64_t ldy,
                 int32_t k, int32_t n_slices, const int32_t *slice_offsets,
                 const int32_t *slot_ids, int32_t S, const int32_t *ranks, const double *scales,
                 const uint16_t *const *A, const uint16_t *const *B,
                 const int32_t *rows, int32_t n_rows, double *y_out, int64_t *macs)
{
    int status = ORACLE_OK;
    int32_t d = slice_offsets[n_slices];
    double *xa = (double *)malloc(sizeof(double) * 512);
    for (int32_t q = 0; q < n_rows; ++q) {
        int32_t t = rows[q];
        double *yo = y_out + (int64_t)q * d;
        for (int32_t m = 0; m < d; ++m) yo[m] = y_in ? bf16_value(y_in[(int64_t)t * ldy + m]) : 0.0;
        int32_t s = slot_ids[t];
        if (s != -1 && (s < 0 || s >= S)) { status = ORACLE_ERR_SLOT_RANGE; continue; }
        if (s < 0 || ranks[s] <= 0) continue;
        int32_t r = ranks[s];
        if (r > 512) { free(xa); xa = (double *)malloc(sizeof(double) * (size_t)r); }
        const uint16_t *xt = x + (int64_t)t * ldx;
        for (int32_t i = 0; i < n_slices; ++i) {
            const uint16_t *a = A[(int64_t)s * n_slices + i];
            const uint16_t *b = B[(int64_t)s * n_slices + i];
            /* shrink: xa_j = x_t . A_j */
            for (int32_t j = 0; j < r; ++j) {
                double acc = 0.0;
                for (int32_t c = 0; c < k; ++c) acc += bf16_value(xt[c]) * bf16_value(a[(int64_t)j * k + c]);
                xa[j] = acc;
                *macs += k;
            }
            /* expand: y += scale * B xa over this slice's columns */
            int32_t o = slice_offsets[i];
            int32_t di = slice_offsets[i + 1] - slice_offsets[i];
            for (int32_t m = 0; m < di; ++m) {
                double acc = 0.0;
                for (int32_t j = 0; j < r; ++j) acc += xa[j] * bf16_value(b[(int64_t)m * r + j]);
                yo[o + m] += scales[s] * acc;
                *macs += r;
            }
        }
        if (r > 512) { free(xa); xa = (double *)malloc(sizeof(double) * 512); }
    }
    free(xa);
    return status;
}

/*
 * FP8 adapters (TensorRT-LLM LoRA serving page, §"第五步:FP8 特判" and the
 * "data_type" check at the start of the forward pass): the adapter weights stay
 * in float8_e4m3fn, the runtime activation x is clamped to the FP8 range and
 * converted to it, and the branch then multiplies FP8 values.
 *
 * float8_e4m3fn: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; exponent 0 holds the subnormals m * 2^-9; the
 * largest finite value is 448.
 */
double oracle_e4m3_to_double(uint8_t code)
{
    int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = m * ldexp(1.0, -9);
    else v = (1.0 + m / 8.0) * ldexp(1.0, e - 7);
    return sign ? -v : v;
}

/*
 * x.clamp(-448, 448).to(float8_e4m3fn): the finite code nearest to the clamped
 * value, ties to the code with an even mantissa; found by comparing against
 * every non-negative finite code (0x00 .. 0x7E).
 */
uint8_t oracle_e4m3_round(double v)
{
    if (isnan(v)) return 0x7F;
    int neg = signbit(v) != 0;
    double a = fabs(v);
    if (a > 448.0) a = 448.0;
    int best = 0;
    double best_d = a;
    for (int c = 1; c <= 0x7E; ++c) {
        double d = fabs(oracle_e4m3_to_double((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) { best = c; best_d = d; }
    }
    return (uint8_t)(best | (neg ? 0x80 : 0));
}

/* The pages' load-time scale for FP8 B: (b.to(bf16) * s).clamp(-448, 448).to(fp8),
 * the product rounded to bf16 first. */
void oracle_premultiply_e4m3(const uint8_t *b, int64_t n, double s, uint8_t *out)
{
    for (int64_t e = 0; e < n; ++e)
        out[e] = oracle_e4m3_round(bf16_value(oracle_round_bf16(oracle_e4m3_to_double(b[e]) * s)));
}

/*
 * oracle_apply with FP8 operands: every x value is rounded to e4m3 as above
 * before the shrink; A and B hold e4m3 codes.  Sums and y as in oracle_apply.
 */
int oracle_apply_e4m3(const uint16_t *x, int64_t ldx, const uint16_t *y_in, int64_t ldy,
                      int32_t k, int32_t n_slices, const int32_t *slice_offsets,
                      const int32_t *slot_ids, int32_t S, const int32_t *ranks, const double *scales,
                      const uint8_t *const *A, const uint8_t *const *B,
                      const int32_t *rows, int32_t n_rows, double *y_out)
{
    int status = ORACLE_OK;
    int32_t d = slice_offsets[n_slices];
    double *xq = (double *)malloc(sizeof(double) * (size_t)k);
    for (int32_t q = 0; q < n_rows; ++q) {
        int32_t t = rows[q];
        double *yo = y_out + (int64_t)q * d;
        for (int32_t m = 0; m < d; ++m) yo[m] = y_in ? bf16_value(y_in[(int64_t)t * ldy + m]) : 0.0;
        int32_t s = slot_ids[t];
        if (s != -1 && (s < 0 || s >= S)) { status = ORACLE_ERR_SLOT_RANGE; continue; }
        if (s < 0 || ranks[s] <= 0) continue;
        int32_t r = ranks[s];
        for (int32_t c = 0; c < k; ++c)
            xq[c] = oracle_e4m3_to_double(oracle_e4m3_round(bf16_value(x[(int64_t)t * ldx + c])));
        double *xa = (double *)malloc(sizeof(double) * (size_t)r);
        for (int32_t i = 0; i < n_slices; ++i) {
            const uint8_t *a = A[(int64_t)s * n_slices + i];
            const uint8_t *b = B[(int64_t)s * n_slices + i];
            for (int32_t j = 0; j < r; ++j) {
                double acc = 0.0;
                for (int32_t c = 0; c < k; ++c) acc += xq[c] * oracle_e4m3_to_double(a[(int64_t)j * k + c]);
                xa[j] = acc;
            }
            int32_t o = slice_offsets[i];
            int32_t di = slice_offsets[i + 1] - slice_offsets[i];
            for (int32_t m = 0; m < di; ++m) {
                double acc = 0.0;
                for (int32_t j = 0; j < r; ++j) acc += xa[j] * oracle_e4m3_to_double(b[(int64_t)m * r + j]);
                yo[o + m] += scales[s] * acc;
            }
        }
        free(xa);
    }
    free(xq);
    return status;
}

/*
 * Routed-expert (MoE) LoRA.  llama.cpp LoRA adapter page, "MoE 专属的
 * build_lora_mm_id": the A product and the B product are both routed by the
 * token's expert ids, so every (token, chosen expert) pair uses that expert's
 * A and B.  TensorRT-LLM LoRA serving page, "MoE LoRA": an adapter holds one
 * (A, B) pair per expert, stored as A [E][r][k] and B [E][d_i][r], expert e's
 * pair starting e * dim * rank elements into each.
 *
 * Pairs p = t K + j of T tokens with K choices each; token t has adapter
 * slot_ids[t] (-1: none) and pair p expert expert_ids[p].  For each requested
 * pair p (rows[]):
 *   y_out[p][o_i + m] = y_in[p][o_i + m]
 *                       + scale_s * sum_j B_{s,e,i}[m][j] sum_c x[row][c] A_{s,e,i}[j][c]
 * with row = t when x_per_token (the layer input shared by the token's experts)
 * and p otherwise.  A[s n + i] and B[s n + i] point at adapter s's [E][r_s][k]
 * and [E][d_i][r_s] arrays.  A slot id outside [-1, S) or, for a token with an
 * adapter, an expert id outside [0, E) sets ORACLE_ERR_SLOT_RANGE and leaves
 * the pair's row unchanged.
 */
int oracle_apply_moe(const uint16_t *x, int64_t ldx, int32_t x_per_token, const uint16_t *y_in, int64_t ldy,
                     int32_t k, int32_t n_slices, const int32_t *slice_offsets, const int32_t *slot_ids,
                     const int32_t *expert_ids, int32_t K, int32_t E, int32_t S, const int32_t *ranks,
                     const double *scales, const uint16_t *const *A, const uint16_t *const *B,
                     const int32_t *rows, int32_t n_rows, double *y_out)
{
    int status = ORACLE_OK;
    int32_t d = slice_offsets[n_slices];
    for (int32_t q = 0; q < n_rows; ++q) {
        int32_t p = rows[q];
        int32_t t = p / K;
        double *yo = y_out + (int64_t)q * d;
        for (int32_t m = 0; m < d; ++m) yo[m] = y_in ? bf16_value(y_in[(int64_t)p * ldy + m]) : 0.0;
        int32_t s = slot_ids[t];
        if (s == -1) continue;
        if (s < 0 || s >= S) { status = ORACLE_ERR_SLOT_RANGE; continue; }
        int32_t e = expert_ids[p];
        if (e < 0 || e >= E) { status = ORACLE_ERR_SLOT_RANGE; continue; }
        int32_t r = ranks[s];
        if (r <= 0) continue;
        const uint16_t *xr = x + (int64_t)(x_per_token ? t : p) * ldx;
        double *xa = (double *)malloc(sizeof(double) * (size_t)r);
        for (int32_t i = 0; i < n_slices; ++i) {
            int32_t o = slice_offsets[i];
            int32_t di = slice_offsets[i + 1] - o;
            /* expert e's pair: e * dim * rank elements into the adapter's arrays */
            const uint16_t *a = A[(int64_t)s * n_slices + i] + (int64_t)e * k * r;
            const uint16_t *b = B[(int64_t)s * n_slices + i] + (int64_t)e * di * r;
            for (int32_t j = 0; j < r; ++j) {
                double acc = 0.0;
                for (int32_t c = 0; c < k; ++c) acc += bf16_value(xr[c]) * bf16_value(a[(int64_t)j * k + c]);
                xa[j] = acc;
            }
            for (int32_t m = 0; m < di; ++m) {
                double acc = 0.0;
                for (int32_t j = 0; j < r; ++j) acc += xa[j] * bf16_value(b[(int64_t)m * r + j]);
                yo[o + m] += scales[s] * acc;
            }
        }
        free(xa);
    }
    return status;
}
