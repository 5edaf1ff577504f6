/*
 * attn_oracle.c -- CPU oracle for the exact attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. The product path (the
 * CUDA library under exact_attention_forward_14_b300/) never calls it and
 * shares no code with it.
 *
 * Source of the method: "FlashAttention-3 deep dive: asynchronous TMA and
 * WGMMA on NVIDIA Hopper H100 ..." (techknowgenie.com/posts/109164421204410442),
 * referred to below as [FA3]. Sections cited by their heading:
 *   [FA3 intro]   standard attention materialises the S x S score matrix;
 *                 FlashAttention computes the same result tile by tile with an
 *                 online softmax (the method is exact).
 *   [FA3 s2]      "3-stage asynchronous software pipelining": S = Q K^T,
 *                 softmax with running max / sum statistics, O = P V.
 *   [FA3 s4]      "FP8 low-precision arithmetic and numerical stability",
 *                 sub-section "block quantisation and dynamic scaling":
 *                 independent scale factors per small tile block, taken from
 *                 the block's local maximum.
 *
 * Because the method is exact, the oracle is the plain definition of the
 * result, evaluated in fp64 with two passes over the keys of each query row:
 *
 *   s_ij  = scale * sum_k q[b,i,hq,k] * k[b,j,hkv,k]      for j in V_i
 *   m_i   = max_j s_ij                                     (pass 1)
 *   l_i   = sum_j exp(s_ij - m_i)                          (pass 2)
 *   O_i   = sum_j exp(s_ij - m_i) * v[b,j,hkv,:] / l_i
 *   LSE_i = m_i + ln(l_i)
 *
 * Readings where the pages are silent (the pages define neither GQA, causal
 * alignment, the LSE output nor the tensor layouts):
 *   - layouts: Q, O are [B, Sq, Hq, d]; K, V are [B, Sk, Hkv, d]; LSE is
 *     [B, Hq, Sq]; all contiguous;
 *   - GQA: hkv = hq / (Hq / Hkv) (consecutive query heads share a KV head);
 *   - causal: bottom-right alignment, V_i = { j : j <= i + Sk - Sq };
 *   - a row with no visible key has O = 0 and LSE = -inf;
 *   - LSE is the natural logarithm.
 *
 * FP16 inputs (the page's own benchmark precision, section 6): element value =
 * the IEEE binary16 value of the bits.
 *
 * FP8 inputs: element value = decode_e4m3(code) * scale[b, h, row / 64], the
 * block being 64 consecutive sequence rows of one head times all d columns.
 * The quantiser that produces these codes follows [FA3 s4]: per block,
 * s = amax / 448 (s = 1 when amax = 0), code = RNE_saturate_e4m3(x / s); the
 * division and the amax are evaluated in fp32, the precision in which the
 * quantised code is decided.
 *
 * Backward (oracle_attn_bwd): the pages give no backward algorithm; the
 * gradients of sum(dO * O) are the chain rule through the definition above,
 * written out in fp64 per (query row, visible key) pair:
 *   P_ij = exp(s_ij - LSE_i),  dP_ij = dO_i . v_j,  D_i = dO_i . O_i,
 *   dS_ij = P_ij (dP_ij - D_i),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,
 *   dV_j = sum_i P_ij dO_i,
 * GQA query heads summing into their KV head; rows with no visible key get
 * dQ = 0 and contribute nothing.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC attn_oracle.c -o liboracle.so -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_DTYPE_BF16 0
#define ORACLE_DTYPE_E4M3 1
#define ORACLE_DTYPE_F16 2
#define ORACLE_FP8_BLOCK_ROWS 64

/* ---------------------------------------------------------------- codecs -- */

/* bfloat16 is the upper half of an IEEE binary32 value. */
static double bf16_bits_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits with bias 15, 10 fraction
 * bits; exponent field 0 encodes subnormals f * 2^-24; field 31 is inf / NaN. */
double oracle_f16_decode(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double mag;
    if (e == 0x1F) mag = f ? NAN : INFINITY;
    else if (e == 0) mag = ldexp((double)f, -24);
    else mag = ldexp(1.0 + (double)f / 1024.0, e - 15);
    return sign ? -mag : mag;
}

/* OCP 8-bit floating point, E4M3 ("fn" variant): 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits; exponent field 0 encodes subnormals
 * m * 2^-9; the all-ones pattern S.1111.111 is NaN; there is no infinity, so
 * the largest finite magnitude is 1.110 * 2^8 = 448. */
double oracle_e4m3_decode(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0) mag = ldexp((double)m, -9);
    else mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Round-to-nearest-even into E4M3 with saturation to +-448 (values beyond the
 * largest finite magnitude become that magnitude). NaN input gives 0x7F. */
uint8_t oracle_e4m3_encode(float x) {
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (isnan(x)) return 0x7F;
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: a multiple of 2^-9, 0..8 (8 is the smallest normal,
         * whose code 0x08 follows on from the subnormal codes) */
        double q = nearbyint(ldexp(a, 9)); /* default rounding: ties to even */
        return sign | (uint8_t)q;
    }
    int e;
    double fr = frexp(a, &e); /* a = fr * 2^e, fr in [0.5, 1) */
    int ue = e - 1;            /* a = (2 fr) * 2^ue, 2 fr in [1, 2) */
    double mant = nearbyint((2.0 * fr - 1.0) * 8.0);
    if (mant >= 8.0) { mant = 0.0; ue += 1; }
    int field = ue + 7;
    if (field > 15 || (field == 15 && mant > 6.0)) return sign | 0x7E;
    return sign | (uint8_t)((field << 3) | (int)mant);
}

/* -------------------------------------------------- FP8 block quantiser -- */

/* x: fp32 [B, S, H, d]; codes: u8 [B, S, H, d]; scales: fp32 [B, H, nblk]
 * with nblk = ceil(S / 64). [FA3 s4] block quantisation. */
void oracle_quantize_fp8_e4m3(const float* x, uint8_t* codes, float* scales,
                              int B, int S, int H, int d) {
    int nblk = (S + ORACLE_FP8_BLOCK_ROWS - 1) / ORACLE_FP8_BLOCK_ROWS;
#pragma omp parallel for collapse(3) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int blk = 0; blk < nblk; ++blk) {
                int r0 = blk * ORACLE_FP8_BLOCK_ROWS;
                int r1 = r0 + ORACLE_FP8_BLOCK_ROWS;
                if (r1 > S) r1 = S;
                float amax = 0.0f;
                for (int r = r0; r < r1; ++r) {
                    const float* row = x + (((size_t)b * S + r) * H + h) * (size_t)d;
                    for (int c = 0; c < d; ++c) {
                        float a = fabsf(row[c]);
                        if (a > amax) amax = a;
                    }
                }
                float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
                scales[((size_t)b * H + h) * nblk + blk] = s;
                for (int r = r0; r < r1; ++r) {
                    size_t off = (((size_t)b * S + r) * H + h) * (size_t)d;
                    for (int c = 0; c < d; ++c) {
                        float t = x[off + c] / s; /* fp32 IEEE division */
                        codes[off + c] = oracle_e4m3_encode(t);
                    }
                }
            }
}

/* --------------------------------------------------- QK RMSNorm (heads) -- */

/* "QKNorm across heads" (SGLang PR 21503 analysis, secrett2633 blog): RMSNorm
 * of each token's whole hidden vector, all heads together, before attention:
 *     y[t, h, c] = x[t, h, c] / sqrt(eps + (1/(H d)) sum_{h', c'} x[t, h', c']^2)
 *                  * w[h d + c]
 * x: [T, H, d] 16-bit bits (bf16 or IEEE fp16, `dtype`), w: [H d] same type.
 * y: fp64 [T, H, d] (not rounded; the caller compares against its own
 * rounding). Q and K are normalised independently with their own weights. */
void oracle_rmsnorm_heads(const uint16_t* x, const uint16_t* w, int dtype, double* y,
                          long long T, int H, int d, double eps) {
    const long long n = (long long)H * d;
#pragma omp parallel for schedule(static)
    for (long long t = 0; t < T; ++t) {
        const uint16_t* row = x + t * n;
        double ss = 0.0;
        for (long long i = 0; i < n; ++i) {
            double v = dtype == ORACLE_DTYPE_F16 ? oracle_f16_decode(row[i])
                                                 : bf16_bits_to_double(row[i]);
            ss += v * v;
        }
        const double r = 1.0 / sqrt(eps + ss / (double)n);
        for (long long i = 0; i < n; ++i) {
            double v = dtype == ORACLE_DTYPE_F16 ? oracle_f16_decode(row[i])
                                                 : bf16_bits_to_double(row[i]);
            double wi = dtype == ORACLE_DTYPE_F16 ? oracle_f16_decode(w[i])
                                                  : bf16_bits_to_double(w[i]);
            y[t * n + i] = v * r * wi;
        }
    }
}

/* ------------------------------------------------------------ attention -- */

typedef struct {
    const void* q;
    const void* k;
    const void* v;
    const float* q_scale;
    const float* k_scale;
    const float* v_scale;
    int dtype;
    int B, Hq, Hkv, Sq, Sk, d;
} oracle_inputs;

/* Value of element [b, s, h, c] of a [B, S, H, d] operand, decoded exactly to
 * fp64. For E4M3 the block scale of (b, h, s/64) multiplies the code. */
static double load_elem(const oracle_inputs* in, const void* base, const float* scale,
                        int S, int H, int b, int s, int h, int c) {
    size_t idx = (((size_t)b * S + s) * H + h) * (size_t)in->d + c;
    if (in->dtype == ORACLE_DTYPE_BF16) return bf16_bits_to_double(((const uint16_t*)base)[idx]);
    if (in->dtype == ORACLE_DTYPE_F16) return oracle_f16_decode(((const uint16_t*)base)[idx]);
    int nblk = (S + ORACLE_FP8_BLOCK_ROWS - 1) / ORACLE_FP8_BLOCK_ROWS;
    double sc = (double)scale[((size_t)b * H + h) * nblk + s / ORACLE_FP8_BLOCK_ROWS];
    return oracle_e4m3_decode(((const uint8_t*)base)[idx]) * sc;
}

/* The d values of row [b, s, h, :] of an operand, decoded exactly to fp64
 * into out[d]: the same values load_elem gives, element by element. E4M3
 * codes are decoded through `e4m3` (oracle_e4m3_decode of every code) and
 * multiplied by the row's block scale. */
static void load_row(const oracle_inputs* in, const void* base, const float* scale,
                     const double* e4m3, int S, int H, int b, int s, int h, double* out) {
    const int d = in->d;
    size_t idx = (((size_t)b * S + s) * H + h) * (size_t)d;
    if (in->dtype == ORACLE_DTYPE_BF16) {
        const uint16_t* p = (const uint16_t*)base + idx;
        for (int c = 0; c < d; ++c) out[c] = bf16_bits_to_double(p[c]);
    } else if (in->dtype == ORACLE_DTYPE_F16) {
        const uint16_t* p = (const uint16_t*)base + idx;
        for (int c = 0; c < d; ++c) out[c] = oracle_f16_decode(p[c]);
    } else {
        int nblk = (S + ORACLE_FP8_BLOCK_ROWS - 1) / ORACLE_FP8_BLOCK_ROWS;
        double sc = (double)scale[((size_t)b * H + h) * nblk + s / ORACLE_FP8_BLOCK_ROWS];
        const uint8_t* p = (const uint8_t*)base + idx;
        for (int c = 0; c < d; ++c) out[c] = e4m3[p[c]] * sc;
    }
}

/* One query row (b, hq, i): writes d outputs to o_row and returns LSE.
 * work: scratch of Sk + 3*d doubles; e4m3: decode table (E4M3 inputs). */
static double attn_row(const oracle_inputs* in, const double* e4m3, int causal, double scale,
                       int b, int hq, int i, double* o_row, double* work) {
    const int d = in->d;
    const int group = in->Hq / in->Hkv;
    const int hkv = hq / group;
    long jmax = in->Sk - 1; /* last visible key */
    if (causal) {
        long lim = (long)i + (long)in->Sk - (long)in->Sq;
        if (lim < jmax) jmax = lim;
    }
    if (jmax < 0) {
        for (int c = 0; c < d; ++c) o_row[c] = 0.0;
        return -INFINITY;
    }
    double* s = work;             /* Sk scores */
    double* qrow = work + in->Sk; /* d */
    double* acc = qrow + d;       /* d */
    double* kv = acc + d;         /* d: one decoded key or value row */
    load_row(in, in->q, in->q_scale, e4m3, in->Sq, in->Hq, b, i, hq, qrow);

    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (long j = 0; j <= jmax; ++j) {
        load_row(in, in->k, in->k_scale, e4m3, in->Sk, in->Hkv, b, (int)j, hkv, kv);
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += qrow[c] * kv[c];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    /* pass 2: normaliser and weighted sum of values */
    double l = 0.0;
    for (int c = 0; c < d; ++c) acc[c] = 0.0;
    for (long j = 0; j <= jmax; ++j) {
        double w = exp(s[j] - m);
        l += w;
        load_row(in, in->v, in->v_scale, e4m3, in->Sk, in->Hkv, b, (int)j, hkv, kv);
        for (int c = 0; c < d; ++c) acc[c] += w * kv[c];
    }
    for (int c = 0; c < d; ++c) o_row[c] = acc[c] / l;
    return m + log(l);
}

static int check_dims_bwd(int B, int Hq, int Hkv, int Sq, int Sk, int d) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || d <= 0) return 1;
    return Hq % Hkv != 0;
}

/* ------------------------------------------------------------- backward -- */

/* Gradient of the loss L = sum(dO * O) through O = softmax(scale Q K^T + mask) V
 * (the pages give no backward algorithm; this is the chain rule written out):
 *   P_ij  = exp(s_ij - LSE_i)                          (visible j, else 0)
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . V_j
 *   D_i   = sum_j P_ij dP_ij  (= dO_i . O_i)
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale sum_j dS_ij K_j,   dK_j = scale sum_i dS_ij Q_i
 * with GQA query heads summed into their KV head's dK and dV. Inputs as for
 * oracle_attn_fwd (16-bit bits: bf16 or fp16), dO with O's shape; outputs fp64:
 * dq [B,Sq,Hq,d], dk / dv [B,Sk,Hkv,d]. Recomputes LSE itself in fp64. */
int oracle_attn_bwd(const void* q, const void* k, const void* v, const void* d_o, int dtype,
                    double* dq, double* dk, double* dv,
                    int B, int Hq, int Hkv, int Sq, int Sk, int d, int causal, double scale) {
    if (check_dims_bwd(B, Hq, Hkv, Sq, Sk, d)) return 1;
    if (dtype != ORACLE_DTYPE_BF16 && dtype != ORACLE_DTYPE_F16) return 1;
    oracle_inputs in = {q, k, v, NULL, NULL, NULL, dtype, B, Hq, Hkv, Sq, Sk, d};
    oracle_inputs gin = {d_o, NULL, NULL, NULL, NULL, NULL, dtype, B, Hq, Hkv, Sq, Sk, d};
    const int group = Hq / Hkv;
    memset(dk, 0, sizeof(double) * (size_t)B * Sk * Hkv * d);
    memset(dv, 0, sizeof(double) * (size_t)B * Sk * Hkv * d);
    /* one (b, hkv) per task: its query heads' contributions go to its dk / dv */
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b)
        for (int hk = 0; hk < Hkv; ++hk) {
            double* o_row = (double*)malloc(sizeof(double) * 2 * (size_t)d);
            double* work = (double*)malloc(sizeof(double) * ((size_t)Sk + 3 * (size_t)d));
            double* dorow = o_row + d;
            for (int hq = hk * group; hq < (hk + 1) * group; ++hq)
                for (int i = 0; i < Sq; ++i) {
                    double lse = attn_row(&in, NULL, causal, scale, b, hq, i, o_row, work);
                    double* dqrow = dq + (((size_t)b * Sq + i) * Hq + hq) * (size_t)d;
                    for (int c = 0; c < d; ++c) {
                        dqrow[c] = 0.0;
                        dorow[c] = load_elem(&gin, d_o, NULL, Sq, Hq, b, i, hq, c);
                    }
                    if (lse == -INFINITY) continue; /* no visible key: zero gradient */
                    long jmax = Sk - 1;
                    if (causal && (long)i + Sk - Sq < jmax) jmax = (long)i + Sk - Sq;
                    double D = 0.0;
                    for (int c = 0; c < d; ++c) D += dorow[c] * o_row[c];
                    for (long j = 0; j <= jmax; ++j) {
                        double dot = 0.0, dp = 0.0;
                        for (int c = 0; c < d; ++c) {
                            double qv = load_elem(&in, q, NULL, Sq, Hq, b, i, hq, c);
                            dot += qv * load_elem(&in, k, NULL, Sk, Hkv, b, (int)j, hk, c);
                            dp += dorow[c] * load_elem(&in, v, NULL, Sk, Hkv, b, (int)j, hk, c);
                        }
                        const double p = exp(scale * dot - lse);
                        const double ds = p * (dp - D);
                        double* dkrow = dk + (((size_t)b * Sk + j) * Hkv + hk) * (size_t)d;
                        double* dvrow = dv + (((size_t)b * Sk + j) * Hkv + hk) * (size_t)d;
                        for (int c = 0; c < d; ++c) {
                            dqrow[c] += scale * ds * load_elem(&in, k, NULL, Sk, Hkv, b, (int)j, hk, c);
                            dkrow[c] += scale * ds * load_elem(&in, q, NULL, Sq, Hq, b, i, hq, c);
                            dvrow[c] += p * dorow[c];
                        }
                    }
                }
            free(o_row);
            free(work);
        }
    return 0;
}

/* Sampled form of oracle_attn_bwd, for inputs too large to differentiate
 * whole: dq for the query rows qrows[r] = (b Hq + hq) Sq + i (out [nq, d]) and
 * dk, dv for the keys krows[r] = (b Hkv + hk) Sk + j (out [nk, d]; krows
 * sorted ascending). Same formulas as oracle_attn_bwd; LSE_i and D_i are
 * recomputed for every row of the query heads a sampled key's KV head serves. */
int oracle_attn_bwd_sampled(const void* q, const void* k, const void* v, const void* d_o,
                            int dtype, int B, int Hq, int Hkv, int Sq, int Sk, int d, int causal,
                            double scale, const int64_t* qrows, int64_t nq, const int64_t* krows,
                            int64_t nk, double* dq, double* dk, double* dv) {
    if (check_dims_bwd(B, Hq, Hkv, Sq, Sk, d)) return 1;
    if (dtype != ORACLE_DTYPE_BF16 && dtype != ORACLE_DTYPE_F16) return 1;
    for (int64_t r = 0; r < nq; ++r)
        if (qrows[r] < 0 || qrows[r] >= (int64_t)B * Hq * Sq) return 1;
    for (int64_t r = 0; r < nk; ++r) {
        if (krows[r] < 0 || krows[r] >= (int64_t)B * Hkv * Sk) return 1;
        if (r > 0 && krows[r] < krows[r - 1]) return 1;
    }
    oracle_inputs in = {q, k, v, NULL, NULL, NULL, dtype, B, Hq, Hkv, Sq, Sk, d};
    oracle_inputs gin = {d_o, NULL, NULL, NULL, NULL, NULL, dtype, B, Hq, Hkv, Sq, Sk, d};
    const int group = Hq / Hkv;
    const long off = (long)Sk - (long)Sq; /* key j visible to row i iff j <= i + off */

    /* dq rows */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nq; ++r) {
        const int i = (int)(qrows[r] % Sq);
        const int bh = (int)(qrows[r] / Sq);
        const int b = bh / Hq, hq = bh % Hq, hk = hq / group;
        double* o_row = (double*)malloc(sizeof(double) * 2 * (size_t)d);
        double* work = (double*)malloc(sizeof(double) * ((size_t)Sk + 3 * (size_t)d));
        double* dorow = o_row + d;
        double* out = dq + (size_t)r * d;
        const double lse = attn_row(&in, NULL, causal, scale, b, hq, i, o_row, work);
        double D = 0.0;
        for (int c = 0; c < d; ++c) {
            out[c] = 0.0;
            dorow[c] = load_elem(&gin, d_o, NULL, Sq, Hq, b, i, hq, c);
            D += dorow[c] * o_row[c];
        }
        if (lse != -INFINITY) {
            long jmax = Sk - 1;
            if (causal && (long)i + off < jmax) jmax = (long)i + off;
            for (long j = 0; j <= jmax; ++j) {
                double dot = 0.0, dp = 0.0;
                for (int c = 0; c < d; ++c) {
                    dot += load_elem(&in, q, NULL, Sq, Hq, b, i, hq, c) *
                           load_elem(&in, k, NULL, Sk, Hkv, b, (int)j, hk, c);
                    dp += dorow[c] * load_elem(&in, v, NULL, Sk, Hkv, b, (int)j, hk, c);
                }
                const double ds = exp(scale * dot - lse) * (dp - D);
                for (int c = 0; c < d; ++c)
                    out[c] += scale * ds * load_elem(&in, k, NULL, Sk, Hkv, b, (int)j, hk, c);
            }
        }
        free(o_row);
        free(work);
    }

    /* dk, dv keys, grouped by (b, hk) */
    double* lse_all = (double*)malloc(sizeof(double) * (size_t)group * Sq);
    double* D_all = (double*)malloc(sizeof(double) * (size_t)group * Sq);
    int64_t r0 = 0;
    while (r0 < nk) {
        const int64_t bhk = krows[r0] / Sk;
        int64_t r1 = r0;
        while (r1 < nk && krows[r1] / Sk == bhk) ++r1;
        const int b = (int)(bhk / Hkv), hk = (int)(bhk % Hkv);
        /* row statistics of every query head served by this KV head */
#pragma omp parallel for schedule(dynamic, 16)
        for (long gi = 0; gi < (long)group * Sq; ++gi) {
            const int g = (int)(gi / Sq), i = (int)(gi % Sq);
            const int hq = hk * group + g;
            double* o_row = (double*)malloc(sizeof(double) * (size_t)d);
            double* work = (double*)malloc(sizeof(double) * ((size_t)Sk + 3 * (size_t)d));
            lse_all[gi] = attn_row(&in, NULL, causal, scale, b, hq, i, o_row, work);
            double D = 0.0;
            for (int c = 0; c < d; ++c) D += load_elem(&gin, d_o, NULL, Sq, Hq, b, i, hq, c) * o_row[c];
            D_all[gi] = D;
            free(o_row);
            free(work);
        }
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t r = r0; r < r1; ++r) {
            const int j = (int)(krows[r] % Sk);
            double* ok = dk + (size_t)r * d;
            double* ov = dv + (size_t)r * d;
            for (int c = 0; c < d; ++c) ok[c] = ov[c] = 0.0;
            for (int g = 0; g < group; ++g) {
                const int hq = hk * group + g;
                for (int i = 0; i < Sq; ++i) {
                    if (causal && (long)j > (long)i + off) continue;
                    const double lse = lse_all[(size_t)g * Sq + i];
                    if (lse == -INFINITY) continue;
                    double dot = 0.0, dp = 0.0;
                    for (int c = 0; c < d; ++c) {
                        dot += load_elem(&in, q, NULL, Sq, Hq, b, i, hq, c) *
                               load_elem(&in, k, NULL, Sk, Hkv, b, j, hk, c);
                        dp += load_elem(&gin, d_o, NULL, Sq, Hq, b, i, hq, c) *
                              load_elem(&in, v, NULL, Sk, Hkv, b, j, hk, c);
                    }
                    const double p = exp(scale * dot - lse);
                    const double ds = p * (dp - D_all[(size_t)g * Sq + i]);
                    for (int c = 0; c < d; ++c) {
                        ok[c] += scale * ds * load_elem(&in, q, NULL, Sq, Hq, b, i, hq, c);
                        ov[c] += p * load_elem(&gin, d_o, NULL, Sq, Hq, b, i, hq, c);
                    }
                }
            }
        }
        r0 = r1;
    }
    free(lse_all);
    free(D_all);
    return 0;
}

static int check_dims(int B, int Hq, int Hkv, int Sq, int Sk, int d) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || d <= 0) return 1;
    if (Hq % Hkv != 0) return 1;
    return 0;
}

/* Full evaluation. o: fp64 [B, Sq, Hq, d]; lse: fp64 [B, Hq, Sq].
 * If rows != NULL, only the nrows listed rows are evaluated: rows[r] is the
 * flat index (b * Hq + hq) * Sq + i, o receives nrows x d values and lse
 * nrows values, in list order. Returns 0, or 1 on bad dimensions. */
int oracle_attn_fwd(const void* q, const void* k, const void* v,
                    const float* q_scale, const float* k_scale, const float* v_scale,
                    int dtype, double* o, double* lse,
                    int B, int Hq, int Hkv, int Sq, int Sk, int d, int causal, double scale,
                    const int64_t* rows, int64_t nrows) {
    if (check_dims(B, Hq, Hkv, Sq, Sk, d)) return 1;
    if (dtype != ORACLE_DTYPE_BF16 && dtype != ORACLE_DTYPE_E4M3 && dtype != ORACLE_DTYPE_F16)
        return 1;
    if (dtype == ORACLE_DTYPE_E4M3 && (!q_scale || !k_scale || !v_scale)) return 1;
    oracle_inputs in = {q, k, v, q_scale, k_scale, v_scale, dtype, B, Hq, Hkv, Sq, Sk, d};
    int64_t total = rows ? nrows : (int64_t)B * Hq * Sq;
    double e4m3[256];
    for (int c = 0; c < 256; ++c) e4m3[c] = oracle_e4m3_decode((uint8_t)c);
#pragma omp parallel
    {
        double* work = (double*)malloc(sizeof(double) * ((size_t)Sk + 3 * (size_t)d));
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < total; ++r) {
            int64_t flat = rows ? rows[r] : r;
            int i = (int)(flat % Sq);
            int64_t bh = flat / Sq;
            int hq = (int)(bh % Hq);
            int b = (int)(bh / Hq);
            double* o_row = rows ? o + (size_t)r * d
                                 : o + (((size_t)b * Sq + i) * Hq + hq) * (size_t)d;
            double val = attn_row(&in, e4m3, causal, scale, b, hq, i, o_row, work);
            lse[rows ? r : flat] = val;
        }
        free(work);
    }
    return 0;
}
