/*
 * wo_oracle.c -- plain, slow, obviously correct CPU oracle for the weight-only
 * quantized fpA.intB GEMM  C[m,n] = A[m,k] . dequant(B)^T + bias  and for the
 * grouped weight-only MoE FFN built from it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links or calls this file;
 * only the tests, the smoke check and the bench's CPU-baseline leg load it.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * Sources (pages):
 *   [acext]   "acext User Guide (v1.7)", sections 1.2.1 (fpAintB GEMM runner:
 *             gemm(A, B, scales, zeros, biases, C, m, n, k, group_size)),
 *             1.3.1 (Int8 weight-only: one scale per output channel),
 *             1.3.3 (Int4 group-wise: one scale per group along K, zero points
 *             when asymmetric), 1.2.3 (MoE runner: gating -> top-k -> fc1 ->
 *             activation -> fc2 -> weighted combine).
 *   [cpu_int4] vLLM-Omni "cpu_int4.py", module docstring (checkpoint layout:
 *             byte j = w[2j] | w[2j+1] << 4; w = (q - 8) * scale + zero) and
 *             functions pack_nibbles / unpack_nibbles.
 *   [allspark] "[Misc][Kernel]: Add GPTQAllSpark Quantization": A16W8,
 *             group_size = -1 (per channel), no act-order; its kernel
 *             choice names desc_act / has_g_idx (GPTQ act-order, a group
 *             index per input channel) as the case it leaves out, which
 *             oracle_gemm_gidx covers.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - int8 codes are stored as uint8 0..255 and dequantise as (q - 128) * s
 *     (+ z when zeros are given); the pages store "int8" and call it
 *     symmetric, which this offset encoding is (signed = q ^ 0x80).
 *   - B is [n, k] (output channel major), C = A . W^T.
 *   - group_size of -1 or k both mean one scale per output channel.
 *   - bias is added in full precision before the single final rounding.
 *   - dequantisation is done in fp32 (separately rounded multiply and add,
 *     no contraction: build with -ffp-contract=off), every product and sum of
 *     the contraction in fp64, summed in ascending k.
 *   - MoE: top-k on the raw fp32 logits, ties to the lower expert id; the
 *     routing weight of a chosen expert is its softmax probability over all
 *     experts (fp64), optionally renormalised over the chosen ones; the gate
 *     is the first half of fc1's outputs and h = silu(gate) * up is rounded
 *     to the activation dtype (it is fc2's A operand); combine in fp64.
 *
 * Parity status of every function here is pinned by tests that do not call
 * the function they check against itself (see the oracle pin tests).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_BAD 1

#define OR_F16 0
#define OR_BF16 1

/* ------------------------------------------------------------------------ */
/* IEEE binary16 / bfloat16 decoding and round-to-nearest-even encoding,    */
/* written from the formats' definitions.                                   */
/* ------------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* 1.f * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round a double to the nearest value of a binary format with `sig_bits`
 * significand bits (hidden bit included) and `exp_bits` exponent bits, ties
 * to even, with gradual underflow and overflow to infinity.  Returns the
 * 16-bit encoding.
 */
static uint16_t encode_rne(double x, int sig_bits, int exp_bits)
{
    const int frac_bits = sig_bits - 1;
    const int bias = (1 << (exp_bits - 1)) - 1;
    const int emin = 1 - bias;
    const uint32_t exp_all = (1u << exp_bits) - 1u;
    const uint16_t sign = signbit(x) ? (uint16_t)0x8000 : (uint16_t)0;
    if (isnan(x))
        return (uint16_t)(sign | (exp_all << frac_bits) | (1u << (frac_bits - 1)));
    double a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | (exp_all << frac_bits));
    if (a == 0.0)
        return sign;
    int e2;
    (void)frexp(a, &e2);      /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;           /* a = 1.xxx * 2^E                */
    int qexp = (E < emin ? emin : E) - frac_bits; /* exponent of one ulp */
    double r = nearbyint(ldexp(a, -qexp)); /* exact scaling, then RNE   */
    uint64_t R = (uint64_t)r;
    uint32_t biased;
    if (E < emin) {
        /* subnormal range; a carry reaches the smallest normal */
        if (R >= (1ull << frac_bits)) {
            biased = 1;
            R -= (1ull << frac_bits);
        } else {
            biased = 0;
        }
    } else {
        if (R >= (1ull << sig_bits)) { /* rounding carried into the exponent */
            R >>= 1;
            E += 1;
        }
        biased = (uint32_t)(E + bias);
        R -= (1ull << frac_bits);
    }
    if (biased >= exp_all)
        return (uint16_t)(sign | (exp_all << frac_bits));
    return (uint16_t)(sign | (biased << frac_bits) | (uint32_t)R);
}

uint16_t oracle_double_to_half(double x) { return encode_rne(x, 11, 5); }
uint16_t oracle_double_to_bf16(double x) { return encode_rne(x, 8, 8); }

static double decode_act(uint16_t v, int dtype)
{
    return dtype == OR_BF16 ? oracle_bf16_to_double(v) : oracle_half_to_double(v);
}

static uint16_t encode_act(double x, int dtype)
{
    return dtype == OR_BF16 ? oracle_double_to_bf16(x) : oracle_double_to_half(x);
}

/* Round `count` doubles to the activation dtype (RNE). */
void oracle_round(const double* x, size_t count, int dtype, uint16_t* out)
{
    for (size_t i = 0; i < count; ++i)
        out[i] = encode_act(x[i], dtype);
}

void oracle_decode(const uint16_t* v, size_t count, int dtype, double* out)
{
    for (size_t i = 0; i < count; ++i)
        out[i] = decode_act(v[i], dtype);
}

/* ------------------------------------------------------------------------ */
/* Codes: the row-major storage the pages define.                           */
/* ------------------------------------------------------------------------ */

/*
 * Unpack row-major stored codes into integers q[n][k].
 *   bits 8: B is [n, k], one code per byte (0..255).
 *   bits 4: B is [n, k/2]; byte j of a row holds code 2j in its low nibble
 *           and code 2j+1 in its high nibble ([cpu_int4] module docstring,
 *           checkpoint layout; unpack_nibbles).
 */
int oracle_unpack_codes(const uint8_t* B, int n, int k, int bits, int32_t* q)
{
    if (n < 0 || k < 0 || (bits != 4 && bits != 8) || (bits == 4 && (k & 1)))
        return OR_BAD;
    for (int r = 0; r < n; ++r) {
        for (int c = 0; c < k; ++c) {
            int32_t v;
            if (bits == 8) {
                v = B[(size_t)r * k + c];
            } else {
                uint8_t byte = B[(size_t)r * (k / 2) + c / 2];
                v = (c % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
            }
            q[(size_t)r * k + c] = v;
        }
    }
    return OR_OK;
}

/*
 * Pack integer codes q[n][k] (0..15) two per byte, low nibble first:
 * byte j = q[2j] | q[2j+1] << 4 ([cpu_int4] pack_nibbles).
 */
int oracle_pack_nibbles(const int32_t* q, int n, int k, uint8_t* B)
{
    if (n < 0 || k < 0 || (k & 1))
        return OR_BAD;
    for (int r = 0; r < n; ++r)
        for (int j = 0; j < k / 2; ++j) {
            int32_t lo = q[(size_t)r * k + 2 * j];
            int32_t hi = q[(size_t)r * k + 2 * j + 1];
            if (lo < 0 || lo > 15 || hi < 0 || hi > 15)
                return OR_BAD;
            B[(size_t)r * (k / 2) + j] = (uint8_t)(lo | (hi << 4));
        }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Dequantisation.                                                          */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint8_t* B;       /* row-major codes, see oracle_unpack_codes */
    const uint16_t* scales; /* [n, G] (G = k / group) in sz_dtype        */
    const uint16_t* zeros;  /* [n, G] or NULL (= 0)                     */
    const int32_t* g_idx;   /* [k] group of each input channel, or NULL  */
    int n, k, group, G, bits, sz_dtype;
} wdesc;

static int make_wdesc(wdesc* d, const uint8_t* B, const uint16_t* scales,
                      const uint16_t* zeros, int n, int k, int group_size,
                      int bits, int sz_dtype)
{
    if (n < 0 || k < 0 || (bits != 4 && bits != 8) || (bits == 4 && (k & 1)))
        return OR_BAD;
    if (sz_dtype != OR_F16 && sz_dtype != OR_BF16)
        return OR_BAD;
    int group = (group_size == -1 || group_size == k) ? k : group_size;
    if (k > 0 && (group <= 0 || k % group != 0))
        return OR_BAD;
    d->B = B;
    d->scales = scales;
    d->zeros = zeros;
    d->g_idx = NULL;
    d->n = n;
    d->k = k;
    d->group = group;
    d->G = k > 0 ? k / group : 0;
    d->bits = bits;
    d->sz_dtype = sz_dtype;
    return OR_OK;
}

/*
 * One dequantised weight row w[r][0..k) in fp32:
 *   bits 4: w = (q - 8) * scale[r][g(c)] + zero[r][g(c)]
 *           ([cpu_int4] module docstring; [acext] 1.3.3 group-wise scales);
 *   bits 8: w = (q - 128) * scale[r][g(c)] (+ zero when given)
 *           ([acext] 1.3.1: one scale per output channel; the 128 offset is
 *           the uint8 storage of a symmetric int8 code).
 * g(c) = c / group, or g_idx[c] when a GPTQ act-order group index is given
 * ([allspark] names desc_act / has_g_idx as the case its kernel excludes:
 * each input channel c carries its own group number instead of c / group).
 * The product and the sum are separate fp32 operations.
 */
static void dequant_row(const wdesc* d, int r, float* w)
{
    const int off = d->bits == 4 ? 8 : 128;
    for (int c = 0; c < d->k; ++c) {
        int32_t q;
        if (d->bits == 8) {
            q = d->B[(size_t)r * d->k + c];
        } else {
            uint8_t byte = d->B[(size_t)r * (d->k / 2) + c / 2];
            q = (c % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
        }
        const int g = d->g_idx ? d->g_idx[c] : c / d->group;
        size_t gi = (size_t)r * d->G + (size_t)g;
        float s = (float)decode_act(d->scales[gi], d->sz_dtype);
        float prod = (float)(q - off) * s;
        float z = d->zeros ? (float)decode_act(d->zeros[gi], d->sz_dtype) : 0.0f;
        w[c] = prod + z;
    }
}

/* Attach a per-channel group index: every entry must name a group. */
static int set_g_idx(wdesc* d, const int32_t* g_idx)
{
    if (!g_idx)
        return OR_OK;
    for (int c = 0; c < d->k; ++c)
        if (g_idx[c] < 0 || g_idx[c] >= d->G)
            return OR_BAD;
    d->g_idx = g_idx;
    return OR_OK;
}

int oracle_dequant(const uint8_t* B, const uint16_t* scales, const uint16_t* zeros,
                   int n, int k, int group_size, int bits, int sz_dtype, float* w)
{
    wdesc d;
    if (make_wdesc(&d, B, scales, zeros, n, k, group_size, bits, sz_dtype) != OR_OK)
        return OR_BAD;
    for (int r = 0; r < n; ++r)
        dequant_row(&d, r, w + (size_t)r * k);
    return OR_OK;
}

/* oracle_dequant with a GPTQ act-order group index g_idx[k] (see dequant_row). */
int oracle_dequant_gidx(const uint8_t* B, const uint16_t* scales, const uint16_t* zeros,
                        const int32_t* g_idx, int n, int k, int group_size, int bits,
                        int sz_dtype, float* w)
{
    wdesc d;
    if (make_wdesc(&d, B, scales, zeros, n, k, group_size, bits, sz_dtype) != OR_OK ||
        set_g_idx(&d, g_idx) != OR_OK)
        return OR_BAD;
    for (int r = 0; r < n; ++r)
        dequant_row(&d, r, w + (size_t)r * k);
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* GEMM: C[i][j] = sum_k A[i][k] * w[j][k] + bias[j], fp64, ascending k.    */
/* ------------------------------------------------------------------------ */

typedef struct {
    wdesc d;
    const double* A; /* decoded activations [m][k] */
    const double* bias; /* decoded [n] or NULL */
    int m;
    int j0, j1;      /* output-channel range of this worker */
    double* C;
} gemm_job;

static void* gemm_worker(void* arg)
{
    gemm_job* job = (gemm_job*)arg;
    const int k = job->d.k;
    const int n = job->d.n;
    float* w = (float*)malloc(sizeof(float) * (size_t)(k > 0 ? k : 1));
    if (!w)
        return (void*)1;
    for (int j = job->j0; j < job->j1; ++j) {
        dequant_row(&job->d, j, w);
        for (int i = 0; i < job->m; ++i) {
            const double* a = job->A + (size_t)i * k;
            double acc = 0.0;
            for (int c = 0; c < k; ++c)
                acc += a[c] * (double)w[c];
            if (job->bias)
                acc += job->bias[j];
            job->C[(size_t)i * n + j] = acc;
        }
    }
    free(w);
    return NULL;
}

/*
 * The fpA.intB GEMM ([acext] 1.2.1 gemm with weight_scales,
 * weight_zero_points, biases, group_size).  A and bias are in act_dtype
 * (fp16/bf16 bits), scales and zeros in act_dtype too.  C is fp64 [m][n].
 * nthreads > 1 splits the output channels across threads; each element is
 * still one ascending-k sum, so the result does not depend on nthreads.
 */
static int gemm_common(const uint16_t* A, int act_dtype, const uint8_t* B,
                       const uint16_t* scales, const uint16_t* zeros, const int32_t* g_idx,
                       const uint16_t* bias, int m, int n, int k, int group_size, int bits,
                       int nthreads, double* C)
{
    gemm_job base;
    if (make_wdesc(&base.d, B, scales, zeros, n, k, group_size, bits, act_dtype) != OR_OK ||
        set_g_idx(&base.d, g_idx) != OR_OK)
        return OR_BAD;
    if (m < 0)
        return OR_BAD;
    if (m == 0 || n == 0)
        return OR_OK;
    double* Ad = (double*)malloc(sizeof(double) * (size_t)m * (size_t)(k > 0 ? k : 1));
    double* bd = bias ? (double*)malloc(sizeof(double) * (size_t)n) : NULL;
    if (!Ad || (bias && !bd)) {
        free(Ad);
        free(bd);
        return OR_BAD;
    }
    oracle_decode(A, (size_t)m * k, act_dtype, Ad);
    if (bias)
        oracle_decode(bias, (size_t)n, act_dtype, bd);
    base.A = Ad;
    base.bias = bd;
    base.m = m;
    base.C = C;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > n)
        nthreads = n;
    gemm_job* jobs = (gemm_job*)malloc(sizeof(gemm_job) * (size_t)nthreads);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int rc = OR_OK;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].j0 = (int)((long long)n * t / nthreads);
        jobs[t].j1 = (int)((long long)n * (t + 1) / nthreads);
    }
    if (nthreads == 1) {
        if (gemm_worker(&jobs[0]))
            rc = OR_BAD;
    } else {
        for (int t = 0; t < nthreads; ++t)
            pthread_create(&th[t], NULL, gemm_worker, &jobs[t]);
        for (int t = 0; t < nthreads; ++t) {
            void* ret = NULL;
            pthread_join(th[t], &ret);
            if (ret)
                rc = OR_BAD;
        }
    }
    free(jobs);
    free(th);
    free(Ad);
    free(bd);
    return rc;
}

int oracle_gemm(const uint16_t* A, int act_dtype, const uint8_t* B,
                const uint16_t* scales, const uint16_t* zeros, const uint16_t* bias,
                int m, int n, int k, int group_size, int bits, int nthreads, double* C)
{
    return gemm_common(A, act_dtype, B, scales, zeros, NULL, bias, m, n, k, group_size, bits,
                       nthreads, C);
}

/*
 * The GEMM of a GPTQ act-order checkpoint ([allspark]: desc_act, has_g_idx):
 * B, A and C keep the original input-channel order, and input channel c
 * takes the scale and zero of group g_idx[c] (0 <= g_idx[c] < k / group).
 * No permutation is applied anywhere: the sum still runs over c ascending.
 */
int oracle_gemm_gidx(const uint16_t* A, int act_dtype, const uint8_t* B,
                     const uint16_t* scales, const uint16_t* zeros, const int32_t* g_idx,
                     const uint16_t* bias, int m, int n, int k, int group_size, int bits,
                     int nthreads, double* C)
{
    if (!g_idx)
        return OR_BAD;
    return gemm_common(A, act_dtype, B, scales, zeros, g_idx, bias, m, n, k, group_size, bits,
                       nthreads, C);
}

/* ------------------------------------------------------------------------ */
/* Grouped weight-only MoE FFN ([acext] 1.2.3 MoE GEMM: gating output ->    */
/* top-k experts per row -> fc1 -> activation -> fc2 -> scale-weighted     */
/* sum of the k expert outputs).                                            */
/* ------------------------------------------------------------------------ */

/*
 * Routing of one token.  ids[j] = the j-th largest logit's expert (ties to
 * the lower id); weights[j] = softmax probability of that expert over all
 * E logits, computed in fp64; with renormalize the k chosen probabilities
 * are divided by their sum.
 */
static void route_token(const float* logits, int E, int topk, int renormalize,
                        int32_t* ids, double* weights)
{
    for (int j = 0; j < topk; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            int taken = 0;
            for (int p = 0; p < j; ++p)
                if (ids[p] == e)
                    taken = 1;
            if (taken)
                continue;
            if (best < 0 || logits[e] > logits[best])
                best = e; /* strict '>' keeps the lower id on ties */
        }
        ids[j] = best;
    }
    double mx = -INFINITY;
    for (int e = 0; e < E; ++e)
        if ((double)logits[e] > mx)
            mx = (double)logits[e];
    double denom = 0.0;
    for (int e = 0; e < E; ++e)
        denom += exp((double)logits[e] - mx);
    double chosen = 0.0;
    for (int j = 0; j < topk; ++j) {
        weights[j] = exp((double)logits[ids[j]] - mx) / denom;
        chosen += weights[j];
    }
    if (renormalize)
        for (int j = 0; j < topk; ++j)
            weights[j] /= chosen;
}

int oracle_moe_route(const float* logits, int T, int E, int topk, int renormalize,
                     int32_t* ids, double* weights)
{
    if (T < 0 || E <= 0 || topk <= 0 || topk > E)
        return OR_BAD;
    for (int t = 0; t < T; ++t)
        route_token(logits + (size_t)t * E, E, topk, renormalize,
                    ids + (size_t)t * topk, weights + (size_t)t * topk);
    return OR_OK;
}

static double silu(double x) { return x / (1.0 + exp(-x)); }

typedef struct {
    /* shared, read-only */
    const double* A;         /* decoded activations of the chosen tokens [S][H] */
    const uint8_t* fc1;      /* [E][2I][H] uint8 codes */
    const uint16_t* fc1_s;   /* [E][2I] */
    const uint8_t* fc2;      /* [E][H][I] uint8 codes */
    const uint16_t* fc2_s;   /* [E][H] */
    int H, I, E, act_dtype;
    const int32_t* pair_tok; /* [P] index into the chosen tokens */
    const int32_t* pair_exp; /* [P] expert id */
    const double* pair_w;    /* [P] routing weight */
    int P;
    /* work split: experts e0..e1 */
    int e0, e1;
    double* y;               /* [P][H] expert outputs (written per pair) */
} moe_job;

static void* moe_worker(void* arg)
{
    moe_job* jb = (moe_job*)arg;
    const int H = jb->H, I = jb->I;
    float* w = (float*)malloc(sizeof(float) * (size_t)(H > I ? H : I));
    int32_t* mine = (int32_t*)malloc(sizeof(int32_t) * (size_t)jb->P);
    double* x1 = (double*)malloc(sizeof(double) * (size_t)2 * I * jb->P);
    double* h = (double*)malloc(sizeof(double) * (size_t)I * jb->P);
    if (!w || !mine || !x1 || !h) {
        free(w); free(mine); free(x1); free(h);
        return (void*)1;
    }
    for (int e = jb->e0; e < jb->e1; ++e) {
        /* the (token, slot) pairs routed to expert e */
        int Pe = 0;
        for (int p = 0; p < jb->P; ++p)
            if (jb->pair_exp[p] == e)
                mine[Pe++] = p;
        if (Pe == 0)
            continue;
        wdesc d1, d2;
        make_wdesc(&d1, jb->fc1 + (size_t)e * 2 * I * H, jb->fc1_s + (size_t)e * 2 * I,
                   NULL, 2 * I, H, -1, 8, jb->act_dtype);
        make_wdesc(&d2, jb->fc2 + (size_t)e * H * I, jb->fc2_s + (size_t)e * H,
                   NULL, H, I, -1, 8, jb->act_dtype);
        /* fc1: x1[q][r] = sum_c a_q[c] * w1[r][c] */
        for (int r = 0; r < 2 * I; ++r) {
            dequant_row(&d1, r, w);
            for (int q = 0; q < Pe; ++q) {
                const double* a = jb->A + (size_t)jb->pair_tok[mine[q]] * H;
                double acc = 0.0;
                for (int c = 0; c < H; ++c)
                    acc += a[c] * (double)w[c];
                x1[(size_t)q * 2 * I + r] = acc;
            }
        }
        /* gated activation: gate = first I outputs, up = last I; rounded to
         * the activation dtype because it is fc2's A operand */
        for (int q = 0; q < Pe; ++q)
            for (int i = 0; i < I; ++i) {
                double g = x1[(size_t)q * 2 * I + i];
                double u = x1[(size_t)q * 2 * I + I + i];
                h[(size_t)q * I + i] =
                    decode_act(encode_act(silu(g) * u, jb->act_dtype), jb->act_dtype);
            }
        /* fc2: y[p][r] = sum_i h_q[i] * w2[r][i] */
        for (int r = 0; r < H; ++r) {
            dequant_row(&d2, r, w);
            for (int q = 0; q < Pe; ++q) {
                const double* hq = h + (size_t)q * I;
                double acc = 0.0;
                for (int i = 0; i < I; ++i)
                    acc += hq[i] * (double)w[i];
                jb->y[(size_t)mine[q] * H + r] = acc;
            }
        }
    }
    free(w); free(mine); free(x1); free(h);
    return NULL;
}

/*
 * MoE FFN for the tokens listed in `tokens` (n_tokens of them; NULL means
 * all T).  out is fp64 [n_tokens][H]:
 *   out[t] = sum_j weight[t][j] * fc2_e(round(silu(g) * u)),
 *   [g | u] = A[t] . dequant(fc1_e)^T, e = ids[t][j].
 * fc1 is [E][2I][H] and fc2 [E][H][I], int8 per-channel codes (uint8,
 * w = (q - 128) * s) with scales [E][2I] and [E][H] in act_dtype.
 */
int oracle_moe_ffn(const uint16_t* A, int act_dtype, const float* logits,
                   const uint8_t* fc1, const uint16_t* fc1_scales,
                   const uint8_t* fc2, const uint16_t* fc2_scales,
                   int T, int H, int I, int E, int topk, int renormalize,
                   const int32_t* tokens, int n_tokens, int nthreads, double* out)
{
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || topk <= 0 || topk > E)
        return OR_BAD;
    if (act_dtype != OR_F16 && act_dtype != OR_BF16)
        return OR_BAD;
    int S = tokens ? n_tokens : T;
    if (S < 0)
        return OR_BAD;
    if (S == 0)
        return OR_OK;
    int P = S * topk;
    double* Ad = (double*)malloc(sizeof(double) * (size_t)S * H);
    int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)P);
    double* wts = (double*)malloc(sizeof(double) * (size_t)P);
    int32_t* ptok = (int32_t*)malloc(sizeof(int32_t) * (size_t)P);
    double* y = (double*)malloc(sizeof(double) * (size_t)P * H);
    if (!Ad || !ids || !wts || !ptok || !y) {
        free(Ad); free(ids); free(wts); free(ptok); free(y);
        return OR_BAD;
    }
    int rc = OR_OK;
    for (int s = 0; s < S; ++s) {
        int t = tokens ? tokens[s] : s;
        if (t < 0 || t >= T) {
            rc = OR_BAD;
            break;
        }
        oracle_decode(A + (size_t)t * H, (size_t)H, act_dtype, Ad + (size_t)s * H);
        route_token(logits + (size_t)t * E, E, topk, renormalize, ids + (size_t)s * topk,
                    wts + (size_t)s * topk);
        for (int j = 0; j < topk; ++j)
            ptok[s * topk + j] = s;
    }
    if (rc == OR_OK) {
        if (nthreads < 1)
            nthreads = 1;
        if (nthreads > E)
            nthreads = E;
        moe_job* jobs = (moe_job*)malloc(sizeof(moe_job) * (size_t)nthreads);
        pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
        for (int w = 0; w < nthreads; ++w) {
            moe_job j;
            j.A = Ad; j.fc1 = fc1; j.fc1_s = fc1_scales; j.fc2 = fc2; j.fc2_s = fc2_scales;
            j.H = H; j.I = I; j.E = E; j.act_dtype = act_dtype;
            j.pair_tok = ptok; j.pair_exp = ids; j.pair_w = wts; j.P = P;
            j.e0 = (int)((long long)E * w / nthreads);
            j.e1 = (int)((long long)E * (w + 1) / nthreads);
            j.y = y;
            jobs[w] = j;
        }
        if (nthreads == 1) {
            if (moe_worker(&jobs[0]))
                rc = OR_BAD;
        } else {
            for (int w = 0; w < nthreads; ++w)
                pthread_create(&th[w], NULL, moe_worker, &jobs[w]);
            for (int w = 0; w < nthreads; ++w) {
                void* ret = NULL;
                pthread_join(th[w], &ret);
                if (ret)
                    rc = OR_BAD;
            }
        }
        free(jobs);
        free(th);
    }
    if (rc == OR_OK) {
        /* combine in ascending j */
        for (int s = 0; s < S; ++s)
            for (int r = 0; r < H; ++r) {
                double acc = 0.0;
                for (int j = 0; j < topk; ++j)
                    acc += wts[s * topk + j] * y[(size_t)(s * topk + j) * H + r];
                out[(size_t)s * H + r] = acc;
            }
    }
    free(Ad); free(ids); free(wts); free(ptok); free(y);
    return rc;
}
