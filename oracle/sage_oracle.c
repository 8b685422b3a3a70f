/*
 * sage_oracle.c -- CPU oracle for SageAttention-style quantized attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously-correct
 * statement of what the quantize-then-attend path computes.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or constant generator with the CUDA path.
 *
 * Sources (web pages describing the method):
 *  [I15014]  diffusers issue #15014 "gfx1201 (RDNA4) SageAttention attention
 *            backend: aiter package or Hub kernel?", section "Is your feature
 *            request related to a problem?" (kernel contract bullets):
 *            INT8 QK^T and FP8 PV with FP32 accumulation; Q/K quantized per
 *            32-row block, V per channel; BF16 [B, S, H, 128], equal Q/K/V
 *            shapes, no mask, non-causal.
 *  [P15060]  diffusers PR #15060 "Add aiter_sage_hub attention backend for AMD
 *            RDNA4 (gfx1201)", section "What does this PR do?": INT8 QK^T,
 *            FP8 PV, head dim 128, the kernel returns no LSE.
 *
 * Readings of points the pages leave open (each one is fixed here once):
 *  R1  one FP32 scale per 32 consecutive tokens of one (batch, head); blocks
 *      start at token 0 and never cross heads; the last block may be short.
 *  R2  Q/K symmetric INT8: scale = amax / 127 (fp32 division, RNE),
 *      code = clamp(rint(x / scale), -127, 127) with x / scale an fp32 RNE
 *      division; an all-zero block has scale 0 and codes 0.
 *  R3  FP8 is OCP E4M3FN (bias 7, max 448, subnormal quantum 2^-9, no Inf);
 *      conversion is round-to-nearest-even with saturation to +-448.
 *  R4  V per channel = per (batch, head, d) over all S tokens;
 *      sv = amax / 448, code = e4m3(v / sv); an all-zero channel has sv = 0.
 *  R5  QK^T: integer products summed exactly.  |acc| <= 128 * 127^2 < 2^24,
 *      so FP32 accumulation of these products is exact too and equals INT32.
 *  R6  scores in the base-2 domain, fp32, in this order:
 *      c = fl(softmax_scale * L2E) (L2E = the fp32 value nearest log2 e),
 *      c_row = fl(sq * c), cb_j = fl(c_row * sk_{j/32}), x_j = fl(acc_j * cb_j),
 *      so that exp(s_j - s_k) = 2^(x_j - x_k) with s = acc * sq * sk *
 *      softmax_scale.  The kernel takes the FP8 decisions of R8 from these
 *      same fp32 values, so both sides decide every P code in one precision.
 *  R7  online softmax in FP32 over KV tiles of T keys (keys [T t, T t + T)
 *      that exist): the running max m_t = max(m_{t-1}, max_{j in t} x_j)
 *      (m_{-1} = -inf); bias_t = fl(m_t - LOG2_448) with LOG2_448 =
 *      fp32(log2 448); p_j = fp32(2^fmaf(acc_j, cb_j, -bias_t)) (2^ in double,
 *      rounded once), so p_j <= 448 is 448 * exp(s_j - running max);
 *      alpha_t = fp32(2^fl(m_{t-1} - m_t)) rescales what was accumulated
 *      (alpha_0 = 0).  The pages fix no tile: T is an argument.  T = 96 (three
 *      K blocks) follows the CUDA kernel's tile and is the default the parity
 *      tests compare against bit for bit; T = 0 means one tile holding every
 *      key, which is the exact two-pass softmax (m = the row's true max, every
 *      p_j = 448 exp(s_j - m), no rescale).  The bound of R16 links the two.
 *  R8  P to FP8 per tile, against the running max: code_j = e4m3(p_j).
 *  R9  normaliser L = alpha_t * L + sum_{j in t} dec(code_j) (the applied
 *      quantised weights, in double); l_mode = 1 selects the alternative
 *      L = alpha_t * L + sum_{j in t} p_j (the unquantised FP32 weights).
 *  R10 PV: O[d] = alpha_t * O[d] + sum_{j in t} dec(code_j) dec(vcode_jd) in
 *      double.  Within a tile every product is a multiple of 2^-18 below
 *      2^18, so each tile's sum is exact and independent of key order.
 *  R11 out[d] = bf16_rne((float)(O[d] * sv[d] / L)), layout [B, S, H, D].
 *  R13 (LSE, optional output) lse = ln 2 * (m + log2 L - log2 448) in double,
 *      with m the final running max (fp32, base 2) and L the normaliser of R9:
 *      the natural log of sum_j exp(scores) as this quantised computation
 *      estimates it (p_j = 448 * 2^(x_j - m), so sum_j 2^(x_j) ~ 2^m L / 448).
 *      Tie bound for lse: ln(L / (L - T)).
 *  R15 (K smoothing, optional) before K is quantised, each (batch, head,
 *      channel d) of K loses its mean over the S tokens: mean_d =
 *      fp32(sum_s k_sd / S), the sum taken in double (exact for bf16 inputs
 *      whose magnitudes span fewer than 45 - log2 S binary orders: any exact
 *      method gives the same mean) and the division in double, rounded once;
 *      k'_sd = fl32(k_sd - mean_d); k' is
 *      then quantised as R1/R2.  Every score of a query row moves by the
 *      same q . mean, so the softmax is unchanged in exact arithmetic.
 *  R14 (cross-attention) Q may have Sq rows and K, V S != Sq rows: each is
 *      quantised over its own 32-row blocks (Q, K) or its own tokens (V);
 *      every step above runs over the S keys unchanged.
 *
 *  R16 (bound between tilings)  For a tile T and the two-pass form (T = 0)
 *      the scores x_j, the final max m and every fp32 step are the same; a key
 *      in a tile at or after the one that holds the row max gets the same p_j,
 *      the same code and no later rescale (alpha = 2^0 = 1) in both, so only
 *      the keys of earlier tiles ("early" keys) weigh differently.  With
 *      y_j = 2^(acc_j cb_j - m + LOG2_448) exact, each applied weight w_j
 *      (code value times the product of later alphas) satisfies
 *      |w_j - y_j| <= b_j: the E4M3 rounding error of p_j in its tile's units
 *      (2^-4 p relative at or above 2^-6, at most min(p, 2^-10) below) scaled
 *      back by 2^(m_t - m), plus a relative slack eta_j for the fp32 roundings
 *      (bias, fma, 2^x, alphas).  Since o(w) - o(w') = sum_j (w_j - w'_j)
 *      (v_j - o(w')) / sum_j w_j for any two weightings,
 *        |out_T[d] - out_0[d]| <= spread_d * G,
 *        G = sum_{j early} (b_j(T) + b_j(0)) / (sum_j y_j - sum_j b_j(T)),
 *      with spread_d = max_j v_jd - min_j v_jd of the dequantised V, plus one
 *      BF16 ulp for the two final roundings.  oracle_requant_bound returns G.
 *
 *  Tie bound.  A P code whose p_j lies within 2^-19 (relative) of a
 *  rounding midpoint of the E4M3 grid is a tie: an implementation whose 2^x
 *  differs from the correctly rounded one by a few ulp may round it the other
 *  way, and both results are correct.  For each row the oracle reports
 *  bound = T * 2 * vmax / (L - T), with T the weight (in final units) such
 *  ties could move and vmax = 448 * max_d sv[d]: the most any such flip can
 *  change any output of the row.  Rows without ties have bound 0.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fno-fast-math -shared -fPIC
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- BF16 -- */

static float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round an fp32 value to the nearest bf16, ties to even (NaN kept quiet). */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7fffu + lsb) >> 16);
}

/* ------------------------------------------------------------ E4M3FN -- */

/* Value of an E4M3FN code: (-1)^s * 2^(e-7) * (1 + m/8) for e > 0,
 * (-1)^s * 2^-6 * (m/8) for e == 0; e == 15 && m == 7 is NaN. */
double oracle_e4m3_decode(uint8_t c) {
    int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m, -9);
    else mag = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Round y to E4M3FN, nearest-even, saturating to +-448 (R3).  The grid step
 * in the binade [2^e, 2^(e+1)) is 2^(e-3); below 2^-6 the step is 2^-9. */
uint8_t oracle_e4m3_encode(float y) {
    if (isnan(y)) return 0x7f;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    if (a >= 448.0) return sign | 0x7e;
    int e;
    if (a == 0.0) return sign;
    (void)frexp(a, &e);          /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                      /* floor(log2 a) */
    if (e < -6) e = -6;
    double quantum = ldexp(1.0, e - 3);
    double r = nearbyint(a / quantum) * quantum;   /* a/quantum is exact */
    if (r > 448.0) r = 448.0;
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -6))      /* subnormal: r = m * 2^-9, m in 1..7 */
        return sign | (uint8_t)(r / ldexp(1.0, -9));
    int er;
    (void)frexp(r, &er);
    er -= 1;                     /* rounding may have moved r up one binade */
    int mant = (int)(r / ldexp(1.0, er) * 8.0) - 8;
    return sign | (uint8_t)(((er + 7) << 3) | mant);
}

/* ------------------------------------------------- Q/K quantisation -- */

/* x: bf16 [B, S, H, D].  codes: int8 [B, H, S_pad, D] (rows >= S are 0).
 * scale: fp32 [B, H, nb], nb = ceil(S / 32).  [I15014] bullet 1; R1, R2. */
void oracle_quantize_qk(const uint16_t *x, int B, int S, int H, int D,
                        int S_pad, int8_t *codes, float *scale) {
    int nb = (S + 31) / 32;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            int8_t *dst = codes + ((size_t)b * H + h) * S_pad * D;
            memset(dst, 0, (size_t)S_pad * D);
            for (int blk = 0; blk < nb; ++blk) {
                int r0 = blk * 32, r1 = r0 + 32 < S ? r0 + 32 : S;
                float amax = 0.0f;
                for (int s = r0; s < r1; ++s)
                    for (int d = 0; d < D; ++d) {
                        float v = fabsf(bf16_to_f32(x[(((size_t)b * S + s) * H + h) * D + d]));
                        if (v > amax) amax = v;
                    }
                float sc = amax / 127.0f;
                scale[((size_t)b * H + h) * nb + blk] = sc;
                if (sc == 0.0f) continue;
                for (int s = r0; s < r1; ++s)
                    for (int d = 0; d < D; ++d) {
                        float v = bf16_to_f32(x[(((size_t)b * S + s) * H + h) * D + d]);
                        float r = rintf(v / sc);
                        if (r > 127.0f) r = 127.0f;
                        if (r < -127.0f) r = -127.0f;
                        dst[(size_t)s * D + d] = (int8_t)r;
                    }
            }
        }
}

/* ---------------------------------------------------- V quantisation -- */

/* v: bf16 [B, S, H, D].  vt: e4m3 [B, H, D, S_pad] (V transposed, columns
 * >= S are 0).  vscale: fp32 [B, H, D].  [I15014] bullet 1 ("V per
 * channel"), [P15060] ("FP8 PV"); R3, R4. */
void oracle_quantize_v(const uint16_t *v, int B, int S, int H, int D,
                       int S_pad, uint8_t *vt, float *vscale) {
#pragma omp parallel for collapse(3) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int d = 0; d < D; ++d) {
                uint8_t *dst = vt + (((size_t)b * H + h) * D + d) * S_pad;
                memset(dst, 0, (size_t)S_pad);
                float amax = 0.0f;
                for (int s = 0; s < S; ++s) {
                    float a = fabsf(bf16_to_f32(v[(((size_t)b * S + s) * H + h) * D + d]));
                    if (a > amax) amax = a;
                }
                float sv = amax / 448.0f;
                vscale[((size_t)b * H + h) * D + d] = sv;
                if (sv == 0.0f) continue;
                for (int s = 0; s < S; ++s) {
                    float x = bf16_to_f32(v[(((size_t)b * S + s) * H + h) * D + d]);
                    dst[s] = oracle_e4m3_encode(x / sv);
                }
            }
}

/* ------------------------------------------------------------ QK^T -- */

/* Exact integer Q K^T for every (b, h): s_out int32 [B, H, S, S].
 * Returns 0, or -1 if a sum does not fit int32 (cannot happen for codes in
 * [-127, 127] and D <= 128).  R5. */
int oracle_qk_int32(const int8_t *q, const int8_t *k, int B, int S, int H,
                    int D, int S_pad, int32_t *s_out) {
    int bad = 0;
#pragma omp parallel for collapse(3) schedule(static) reduction(| : bad)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int i = 0; i < S; ++i) {
                const int8_t *qi = q + (((size_t)b * H + h) * S_pad + i) * D;
                for (int j = 0; j < S; ++j) {
                    const int8_t *kj = k + (((size_t)b * H + h) * S_pad + j) * D;
                    int64_t acc = 0;
                    for (int c = 0; c < D; ++c) acc += (int64_t)qi[c] * kj[c];
                    if (acc > INT32_MAX || acc < INT32_MIN) bad = 1;
                    s_out[(((size_t)b * H + h) * S + i) * S + j] = (int32_t)acc;
                }
            }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------- attention -- */

/* The fp32 value nearest log2(e), and fp32(log2(448)). */
#define ORACLE_L2E 1.44269502162933349609375f
#define ORACLE_LOG2_448 8.80735492706298828125f
#define ORACLE_KV_TILE 96   /* default T of R7: the CUDA kernel's tile */
#define ORACLE_TIE_REL 1.9073486328125e-06 /* 2^-19 */

/* Distance of an E4M3 code's value to the other side of the nearest rounding
 * midpoint: if y (the fp32 value encoded) is within ORACLE_TIE_REL of a
 * midpoint, returns |value of the neighbouring code - value of code|, else 0. */
static double tie_step(float y, uint8_t code) {
    double a = fabs((double)y);
    if (a >= 448.0 || a == 0.0) return 0.0;
    int e;
    (void)frexp(a, &e);
    e -= 1;
    if (e < -6) e = -6;
    double quantum = ldexp(1.0, e - 3);
    double f = a / quantum;
    double mid = floor(f) + 0.5;
    if (fabs(f - mid) * quantum > ORACLE_TIE_REL * a) return 0.0;
    double v = fabs(oracle_e4m3_decode(code));
    double other = (v >= mid * quantum) ? floor(f) * quantum : (floor(f) + 1.0) * quantum;
    if (other > 448.0) other = 448.0;
    return fabs(other - v);
}

/* One query row (b, h, i) of Q (Sq rows, padded to Sq_pad) against S keys
 * and values (padded to S_pad): S = Sq for self-attention, S != Sq for
 * cross-attention (reading R14).  Writes D bf16 outputs to out_row.  If pcodes is
 * not NULL it receives the S FP8 codes of P (each against the running max of
 * its tile) and *L_out the normaliser; *tie_out (if not NULL) the row's tie
 * bound.  vdec is this head's decoded V, [S][D] floats (exact); acc is
 * scratch for one tile's integer scores (S entries).  kv_tile is T of R7
 * (0: one tile of all S keys, the two-pass form).  R6..R11. */
static void attend_row(const int8_t *q, const float *qs, const int8_t *k,
                       const float *ks, const float *vdec, const float *vs,
                       int b, int h, int i, int Sq, int S, int H, int D, int Sq_pad, int S_pad,
                       float softmax_scale, int l_mode, int kv_tile, float *sbuf,
                       int32_t *acc, uint8_t *cbuf, double *obuf, uint16_t *out_row,
                       uint8_t *pcodes, double *L_out, double *tie_out,
                       double *lse_out, double *lse_tie_out) {
    int nb = (S + 31) / 32, nbq = (Sq + 31) / 32;
    const int8_t *qi = q + (((size_t)b * H + h) * Sq_pad + i) * D;
    const float *vsh = vs + ((size_t)b * H + h) * D;
    float sq = qs[((size_t)b * H + h) * nbq + i / 32];
    float c = softmax_scale * ORACLE_L2E;
    float c_row = sq * c;
    double L = 0.0, T = 0.0;
    float m_run = -INFINITY;
    for (int d = 0; d < D; ++d) obuf[d] = 0.0;
    int tile = (kv_tile <= 0 || kv_tile > S) ? S : kv_tile;   /* R7: 0 = one tile */
    for (int j0 = 0; j0 < S; j0 += tile) {
        int j1 = j0 + tile < S ? j0 + tile : S;
        /* integer scores (R5) and their base-2 values (R6); sbuf keeps cb_j */
        float m_tile = -INFINITY;
        for (int j = j0; j < j1; ++j) {
            const int8_t *kj = k + (((size_t)b * H + h) * S_pad + j) * D;
            int32_t a = 0;
            for (int cc = 0; cc < D; ++cc) a += (int32_t)qi[cc] * (int32_t)kj[cc];
            float cb = c_row * ks[((size_t)b * H + h) * nb + j / 32];
            float x = (float)a * cb;
            acc[j - j0] = a;
            sbuf[j] = cb;
            if (x > m_tile) m_tile = x;
        }
        /* running max, rescale of what was accumulated (R7, R9, R10) */
        float m_new = m_run > m_tile ? m_run : m_tile;
        double alpha = (m_run == -INFINITY) ? 0.0 : (double)(float)exp2((double)(m_run - m_new));
        float bias = m_new - ORACLE_LOG2_448;
        L *= alpha;
        T *= alpha;
        for (int d = 0; d < D; ++d) obuf[d] *= alpha;
        for (int j = j0; j < j1; ++j) {
            float p = (float)exp2((double)fmaf((float)acc[j - j0], sbuf[j], -bias));
            uint8_t code = oracle_e4m3_encode(p);           /* R8 */
            double w = oracle_e4m3_decode(code);
            cbuf[j] = code;
            L += l_mode ? (double)p : w;
            T += tie_step(p, code);
            if (w == 0.0) continue;
            const float *vj = vdec + (size_t)j * D;
            for (int d = 0; d < D; ++d) obuf[d] += w * (double)vj[d];
        }
        m_run = m_new;
    }
    /* epilogue (R11) */
    double vmax = 0.0;
    for (int d = 0; d < D; ++d) {
        double o = obuf[d] * (double)vsh[d] / L;
        out_row[d] = f32_to_bf16_rne((float)o);
        if (448.0 * (double)vsh[d] > vmax) vmax = 448.0 * (double)vsh[d];
    }
    if (pcodes) memcpy(pcodes, cbuf, (size_t)S);
    if (L_out) *L_out = L;
    if (tie_out) *tie_out = (T > 0.0 && L > T) ? T * 2.0 * vmax / (L - T) : (T > 0.0 ? INFINITY : 0.0);
    /* R13 */
    if (lse_out) *lse_out = log(2.0) * ((double)m_run + log2(L) - log2(448.0));
    if (lse_tie_out) *lse_tie_out = (T > 0.0 && L > T) ? log(L / (L - T)) : (T > 0.0 ? INFINITY : 0.0);
}

/* K smoothing (R15): per (b, h) channel means over the S tokens (fp32,
 * [B, H, D]) and INT8 codes / block scales of k - mean, layouts as
 * oracle_quantize_qk. */
void oracle_quantize_k_smooth(const uint16_t *x, int B, int S, int H, int D,
                              int S_pad, int8_t *codes, float *scale, float *mean) {
    int nb = (S + 31) / 32;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            float *mu = mean + ((size_t)b * H + h) * D;
            for (int d = 0; d < D; ++d) {
                double sum = 0.0;
                for (int s = 0; s < S; ++s)
                    sum += (double)bf16_to_f32(x[(((size_t)b * S + s) * H + h) * D + d]);
                mu[d] = (float)(sum / (double)S);
            }
            int8_t *dst = codes + ((size_t)b * H + h) * S_pad * D;
            memset(dst, 0, (size_t)S_pad * D);
            for (int blk = 0; blk < nb; ++blk) {
                int r0 = blk * 32, r1 = r0 + 32 < S ? r0 + 32 : S;
                float amax = 0.0f;
                for (int s = r0; s < r1; ++s)
                    for (int d = 0; d < D; ++d) {
                        float v = bf16_to_f32(x[(((size_t)b * S + s) * H + h) * D + d]) - mu[d];
                        if (fabsf(v) > amax) amax = fabsf(v);
                    }
                float sc = amax / 127.0f;
                scale[((size_t)b * H + h) * nb + blk] = sc;
                if (sc == 0.0f) continue;
                for (int s = r0; s < r1; ++s)
                    for (int d = 0; d < D; ++d) {
                        float v = bf16_to_f32(x[(((size_t)b * S + s) * H + h) * D + d]) - mu[d];
                        float r = rintf(v / sc);
                        if (r > 127.0f) r = 127.0f;
                        if (r < -127.0f) r = -127.0f;
                        dst[(size_t)s * D + d] = (int8_t)r;
                    }
            }
        }
}

/* Decode one head's V^T codes into [S][D] floats (e4m3 values are exact in
 * fp32). */
static void decode_v_head(const uint8_t *vt, int b, int h, int S, int H, int D,
                          int S_pad, float *vdec) {
    for (int d = 0; d < D; ++d) {
        const uint8_t *row = vt + (((size_t)b * H + h) * D + d) * S_pad;
        for (int s = 0; s < S; ++s) vdec[(size_t)s * D + d] = (float)oracle_e4m3_decode(row[s]);
    }
}

/* Attention output for a list of query rows.  rows: n triples (b, h, i).
 * out: bf16 [n, D] in the order of rows.  Every (b, h) named in rows must
 * appear; heads are decoded once.  ties (may be NULL): double [n], each
 * row's tie bound.  lse, lse_ties (may be NULL): double [n], each row's
 * log-sum-exp (R13) and its tie bound.  kv_tile: T of R7 (0: two-pass).
 * Returns 0, or -1 on allocation failure.  [I15014] bullets 1-2, [P15060] ("no LSE"): the kernel contract's
 * output is the normalised attention; the LSE is the optional extra output. */
int oracle_attend_rows_cross(const int8_t *q, const float *qs, const int8_t *k,
                             const float *ks, const uint8_t *vt, const float *vs,
                             int B, int Sq, int S, int H, int D, int Sq_pad, int S_pad,
                             float softmax_scale, int l_mode, int kv_tile,
                             const int32_t *rows, int64_t n, uint16_t *out, double *ties,
                             double *lse, double *lse_ties) {
    /* decode the heads in use */
    int nheads = B * H;
    float **vdec = (float **)calloc((size_t)nheads, sizeof(float *));
    if (!vdec) return -1;
    int fail = 0;
    for (int64_t r = 0; r < n; ++r) {
        int bh = rows[3 * r] * H + rows[3 * r + 1];
        if (!vdec[bh]) {
            vdec[bh] = (float *)malloc((size_t)S * D * sizeof(float));
            if (!vdec[bh]) { fail = 1; break; }
        }
    }
    if (!fail) {
#pragma omp parallel for schedule(static)
        for (int bh = 0; bh < nheads; ++bh)
            if (vdec[bh]) decode_v_head(vt, bh / H, bh % H, S, H, D, S_pad, vdec[bh]);
#pragma omp parallel
        {
            float *sbuf = (float *)malloc((size_t)S * sizeof(float));
            int32_t *abuf = (int32_t *)malloc((size_t)S * sizeof(int32_t));
            uint8_t *cbuf = (uint8_t *)malloc((size_t)S);
            double *obuf = (double *)malloc((size_t)D * sizeof(double));
            if (!sbuf || !abuf || !cbuf || !obuf) {
#pragma omp atomic write
                fail = 1;
            } else {
#pragma omp for schedule(dynamic, 4)
                for (int64_t r = 0; r < n; ++r) {
                    int b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
                    attend_row(q, qs, k, ks, vdec[b * H + h], vs, b, h, i, Sq, S, H, D,
                               Sq_pad, S_pad, softmax_scale, l_mode, kv_tile, sbuf, abuf,
                               cbuf, obuf,
                               out + (size_t)r * D, NULL, NULL, ties ? ties + r : NULL,
                               lse ? lse + r : NULL, lse_ties ? lse_ties + r : NULL);
                }
            }
            free(sbuf); free(abuf); free(cbuf); free(obuf);
        }
    }
    for (int bh = 0; bh < nheads; ++bh) free(vdec[bh]);
    free(vdec);
    return fail ? -1 : 0;
}

/* Self-attention: Q, K and V share the length S. */
int oracle_attend_rows(const int8_t *q, const float *qs, const int8_t *k,
                       const float *ks, const uint8_t *vt, const float *vs,
                       int B, int S, int H, int D, int S_pad,
                       float softmax_scale, int l_mode, int kv_tile, const int32_t *rows,
                       int64_t n, uint16_t *out, double *ties, double *lse,
                       double *lse_ties) {
    return oracle_attend_rows_cross(q, qs, k, ks, vt, vs, B, S, S, H, D, S_pad, S_pad,
                                    softmax_scale, l_mode, kv_tile, rows, n, out, ties, lse,
                                    lse_ties);
}

/* Single row with its FP8 P codes and normaliser exposed (for the pins on
 * the softmax/normaliser readings R7-R9). */
int oracle_attend_row_debug(const int8_t *q, const float *qs, const int8_t *k,
                            const float *ks, const uint8_t *vt, const float *vs,
                            int B, int S, int H, int D, int S_pad,
                            float softmax_scale, int l_mode, int kv_tile, int b, int h,
                            int i, uint16_t *out_row, uint8_t *pcodes, double *L_out,
                            double *tie_out) {
    (void)B;
    float *vdec = (float *)malloc((size_t)S * D * sizeof(float));
    float *sbuf = (float *)malloc((size_t)S * sizeof(float));
    int32_t *abuf = (int32_t *)malloc((size_t)S * sizeof(int32_t));
    uint8_t *cbuf = (uint8_t *)malloc((size_t)S);
    double *obuf = (double *)malloc((size_t)D * sizeof(double));
    int rc = -1;
    if (vdec && sbuf && abuf && cbuf && obuf) {
        decode_v_head(vt, b, h, S, H, D, S_pad, vdec);
        attend_row(q, qs, k, ks, vdec, vs, b, h, i, S, S, H, D, S_pad, S_pad, softmax_scale,
                   l_mode, kv_tile, sbuf, abuf, cbuf, obuf, out_row, pcodes, L_out, tie_out,
                   NULL, NULL);
        rc = 0;
    }
    free(vdec); free(sbuf); free(abuf); free(cbuf); free(obuf);
    return rc;
}

/* Bound on |dec(e4m3(p)) - p| for p >= 0 (R3): half a step, 2^-4 p, in the
 * normal range (p >= 2^-6, saturation at 448 included); below it half the
 * subnormal quantum, 2^-10, or p itself where p rounds to zero. */
static double e4m3_err_bound(double p) {
    if (p >= 0x1p-6) return 0x1p-4 * p;
    return p < 0x1p-10 ? p : 0x1p-10;
}

/* R16: per query row, G with |out_T[d] - out_0[d]| <= spread_d * G (plus one
 * BF16 ulp), where out_T is the output with KV tiles of kv_tile keys and
 * out_0 the two-pass output.  Operands as oracle_attend_rows_cross; G: double
 * [n].  Every term is computed from the exact scores, not from either
 * output.  Returns 0, or -1 on allocation failure. */
int oracle_requant_bound(const int8_t *q, const float *qs, const int8_t *k,
                         const float *ks, int B, int Sq, int S, int H, int D, int Sq_pad,
                         int S_pad, float softmax_scale, int kv_tile, const int32_t *rows,
                         int64_t n, double *G) {
    (void)B;
    int fail = 0;
    int tile = (kv_tile <= 0 || kv_tile > S) ? S : kv_tile;
    int n_tiles = (S + tile - 1) / tile;
    int nb = (S + 31) / 32, nbq = (Sq + 31) / 32;
#pragma omp parallel
    {
        int32_t *acc = (int32_t *)malloc((size_t)S * sizeof(int32_t));
        float *cb = (float *)malloc((size_t)S * sizeof(float));
        float *mt = (float *)malloc((size_t)n_tiles * sizeof(float));
        if (!acc || !cb || !mt) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < n; ++r) {
                int b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
                const int8_t *qi = q + (((size_t)b * H + h) * Sq_pad + i) * D;
                float c_row = qs[((size_t)b * H + h) * nbq + i / 32] * (softmax_scale * ORACLE_L2E);
                /* scores of R6 and the running max of R7 at the end of each tile */
                float m = -INFINITY;
                for (int j = 0; j < S; ++j) {
                    const int8_t *kj = k + (((size_t)b * H + h) * S_pad + j) * D;
                    int32_t a = 0;
                    for (int c = 0; c < D; ++c) a += (int32_t)qi[c] * (int32_t)kj[c];
                    acc[j] = a;
                    cb[j] = c_row * ks[((size_t)b * H + h) * nb + j / 32];
                    float x = (float)a * cb[j];
                    if (x > m) m = x;
                    if ((j + 1) % tile == 0 || j == S - 1) mt[j / tile] = m;
                }
                int t_star = 0;
                while (mt[t_star] != m) ++t_star;
                double sum_y = 0.0, sum_b = 0.0, early = 0.0;
                for (int j = 0; j < S; ++j) {
                    int t = j / tile;
                    double prod = (double)acc[j] * (double)cb[j];   /* exact */
                    double x = fabs((double)((float)acc[j] * cb[j]));
                    double y = exp2(prod - (double)m + (double)ORACLE_LOG2_448);
                    /* relative slack of the fp32 steps: the bias, the fma and the
                     * rounding of 2^x (each <= 2^-24 of its magnitude), and for
                     * the tiled form the n_tiles alphas and their arguments */
                    double eta0 = 0x1p-23 * (2.0 + x + 2.0 * (fabs((double)m) + 9.0));
                    double eta = 0x1p-23 * (2.0 + x + 2.0 * (fabs((double)mt[t]) + 9.0) + n_tiles +
                                            ((double)m - (double)mt[t]));
                    double y_tile = exp2(prod - (double)mt[t] + (double)ORACLE_LOG2_448);
                    double back = exp2((double)mt[t] - (double)m);   /* <= 1 */
                    double b_t = e4m3_err_bound(y_tile * (1.0 + eta)) * (1.0 + eta) * back + 3.0 * eta * y;
                    double b_0 = e4m3_err_bound(y * (1.0 + eta0)) * (1.0 + eta0) + 3.0 * eta0 * y;
                    sum_y += y;
                    sum_b += b_t;
                    if (t < t_star) early += b_t + b_0;
                }
                double den = sum_y - sum_b;
                G[r] = early == 0.0 ? 0.0 : (den > 0.0 ? early / den : INFINITY);
            }
        }
        free(acc); free(cb); free(mt);
    }
    return fail ? -1 : 0;
}

/* Threads the OpenMP runtime will use (for the benchmark's core count). */
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
#else
int oracle_num_threads(void) { return 1; }
#endif

/* Element-wise E4M3FN conversion over arrays (for the format pins). */
void oracle_e4m3_encode_array(const float *y, int64_t n, uint8_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(y[i]);
}
void oracle_e4m3_decode_array(const uint8_t *c, int64_t n, double *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(c[i]);
}
