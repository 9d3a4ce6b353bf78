/*
 * qhead_oracle.c -- the fp64 CPU oracle for the fused quantized LM-head.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * execute this file: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it computes is the plain definition of the method described on the
 * page "mlx-bun 0.0.4 -> 0.0.6" (src/train/flash-cce.ts): the per-token
 * response log-prob  logp = z[target] - logsumexp_v z[v]  where z is the
 * (optionally soft-capped) logit of token h against vocab row v of a frozen
 * affine-quantized head, and the frozen-head gradient
 * dh = d(sum_t dlogp_t * logp_t)/dh.  Every step is written out directly in
 * double precision; there is no vocab blocking, no online softmax and no
 * fusion.  The only concession to speed is an OpenMP loop over independent
 * outputs, which does not change any arithmetic.
 *
 * Layout (the head type FlashCceHead on the same page):
 *   wq      uint32 [V, H*bits/32]  packed codes, least-significant field first
 *   scales  [V, H/group]           per-group affine scale (fed here as fp64)
 *   biases  [V, H/group]           per-group affine bias  (fed here as fp64)
 *   h       [M, H]                 hidden states (fed here as fp64)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- widening */

/* bf16 is the upper half of an IEEE-754 binary32, so widening is a shift. */
void oracle_widen_bf16(const uint16_t *src, double *dst, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u = ((uint32_t)src[i]) << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        dst[i] = (double)f;
    }
}

/* IEEE-754 binary16 -> double from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
void oracle_widen_f16(const uint16_t *src, double *dst, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        const uint16_t b = src[i];
        const int sign = (b >> 15) & 1;
        const int expo = (b >> 10) & 31;
        const int frac = b & 1023;
        double v;
        if (expo == 0)
            v = ldexp((double)frac, -24);                 /* subnormal: frac * 2^-24 */
        else if (expo == 31)
            v = frac ? NAN : INFINITY;
        else
            v = ldexp((double)(1024 + frac), expo - 25);  /* (1 + frac/1024) * 2^(expo-15) */
        dst[i] = sign ? -v : v;
    }
}

/* ------------------------------------------------------------ quantization */

/* Code q[v,d]: the page's forward kernel reads word d / (32/bits) of row v and
 * takes field d mod (32/bits), counting from the least significant bits. */
static inline uint32_t code_at(const uint32_t *row, int bits, int64_t d) {
    const int per_word = 32 / bits;
    const uint32_t word = row[d / per_word];
    const int field = (int)(d % per_word);
    const uint32_t mask = (bits == 32) ? 0xffffffffu : ((1u << bits) - 1u);
    return (word >> (bits * field)) & mask;
}

void oracle_codes(const uint32_t *wq, int64_t V, int64_t H, int bits, uint32_t *codes) {
    const int64_t wpr = H * bits / 32;
    for (int64_t v = 0; v < V; ++v)
        for (int64_t d = 0; d < H; ++d)
            codes[v * H + d] = code_at(wq + v * wpr, bits, d);
}

/* Affine dequantization  w[v,d] = scale[v, d/group] * q[v,d] + bias[v, d/group]. */
static void dequant_row(const uint32_t *wq, const double *scales, const double *biases,
                        int64_t v, int64_t H, int bits, int group, double *w) {
    const int64_t wpr = H * bits / 32;
    const int64_t gpr = H / group;
    const uint32_t *row = wq + v * wpr;
    for (int64_t d = 0; d < H; ++d) {
        const double s = scales[v * gpr + d / group];
        const double b = biases[v * gpr + d / group];
        w[d] = s * (double)code_at(row, bits, d) + b;
    }
}

void oracle_dequant(const uint32_t *wq, const double *scales, const double *biases,
                    int64_t V, int64_t H, int bits, int group, double *w) {
    for (int64_t v = 0; v < V; ++v) dequant_row(wq, scales, biases, v, H, bits, group, w + v * H);
}

/* --------------------------------------------------------------- forward */

static int pick_threads(int nthreads) {
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

int oracle_num_threads(int nthreads) { return pick_threads(nthreads); }

/* raw[m,v] = sum_d h[m,d] * w[v,d]   (the logit, before any soft cap). */
void oracle_logits(int64_t M, int64_t H, int64_t V, int bits, int group,
                   const double *h, const uint32_t *wq, const double *scales,
                   const double *biases, double *raw, int nthreads) {
    const int nt = pick_threads(nthreads);
#pragma omp parallel num_threads(nt)
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(static)
        for (int64_t v = 0; v < V; ++v) {
            dequant_row(wq, scales, biases, v, H, bits, group, w);
            for (int64_t m = 0; m < M; ++m) {
                const double *hm = h + m * H;
                double acc = 0.0;
                for (int64_t d = 0; d < H; ++d) acc += hm[d] * w[d];
                raw[m * V + v] = acc;
            }
        }
        free(w);
    }
}

/* Final-logit soft cap: z = cap * tanh(raw / cap) when cap > 0, else z = raw. */
static inline double capped(double raw, double cap) {
    return cap > 0.0 ? cap * tanh(raw / cap) : raw;
}

/*
 * Per-row statistics from the full logits row (no blocking):
 *   lse    = log sum_v exp(z[v])           (max-shifted for range only)
 *   logp   = z[target] - lse               (only when targets != NULL)
 *   argmax = lowest v attaining max_v raw[v]
 *   gap    = largest z minus second-largest z (0 when the maximum is tied)
 *   zmax   = max_v z[v]
 * Rows with mask[m] == 0 are not computed: logp = lse = gap = zmax = 0 and
 * argmax = -1.
 */
void oracle_row_stats(int64_t M, int64_t V, double softcap, const double *raw,
                      const int32_t *targets, const uint8_t *mask, double *logp,
                      double *lse, int64_t *argmax, double *gap, double *zmax,
                      int nthreads) {
    const int nt = pick_threads(nthreads);
#pragma omp parallel for schedule(static) num_threads(nt)
    for (int64_t m = 0; m < M; ++m) {
        if (mask && !mask[m]) {
            if (logp) logp[m] = 0.0;
            lse[m] = 0.0;
            argmax[m] = -1;
            gap[m] = 0.0;
            if (zmax) zmax[m] = 0.0;
            continue;
        }
        const double *r = raw + m * V;
        double zbest = -INFINITY, zsecond = -INFINITY, rbest = -INFINITY;
        int64_t ibest = -1;
        for (int64_t v = 0; v < V; ++v) {
            const double z = capped(r[v], softcap);
            if (z > zbest) {
                zsecond = zbest;
                zbest = z;
            } else if (z > zsecond) {
                zsecond = z;
            }
            if (r[v] > rbest) {
                rbest = r[v];
                ibest = v;
            }
        }
        double sum = 0.0;
        for (int64_t v = 0; v < V; ++v) sum += exp(capped(r[v], softcap) - zbest);
        const double l = zbest + log(sum);
        lse[m] = l;
        argmax[m] = ibest;
        gap[m] = (V > 1) ? (zbest - zsecond) : INFINITY;
        if (zmax) zmax[m] = zbest;
        if (logp) logp[m] = targets ? capped(r[targets[m]], softcap) - l : 0.0;
    }
}

/* -------------------------------------------------------------- backward */

/*
 * coeff[m,v] = dlogp[m] * (1[v == target_m] - exp(z[m,v] - lse[m])) * sech2[m,v]
 * with sech2 = 1 - tanh^2(raw/cap) when the cap is on (1 otherwise), as in the
 * backward kernel on the same page.  Masked rows get coeff = 0.
 * Overwrites `raw` in place with coeff.
 */
void oracle_coeff(int64_t M, int64_t V, double softcap, double *raw, const double *lse,
                  const int32_t *targets, const uint8_t *mask, const double *dlogp,
                  int nthreads) {
    const int nt = pick_threads(nthreads);
#pragma omp parallel for schedule(static) num_threads(nt)
    for (int64_t m = 0; m < M; ++m) {
        double *r = raw + m * V;
        if (mask && !mask[m]) {
            for (int64_t v = 0; v < V; ++v) r[v] = 0.0;
            continue;
        }
        for (int64_t v = 0; v < V; ++v) {
            double z = r[v], sech2 = 1.0;
            if (softcap > 0.0) {
                const double th = tanh(r[v] / softcap);
                z = softcap * th;
                sech2 = 1.0 - th * th;
            }
            const double p = exp(z - lse[m]);
            const double onehot = (v == (int64_t)targets[m]) ? 1.0 : 0.0;
            r[v] = dlogp[m] * (onehot - p) * sech2;
        }
    }
}

/* dW[v,d] = sum_m coeff[m,v] * h[m,d]: the gradient of sum_m dlogp[m] * logp[m]
 * with respect to the dequantized head (the classifier gradient of the
 * Apple CCE reference, which the pages leave out because their head is
 * frozen).  Each output row is owned by one thread and summed over m in
 * ascending order, so the result does not depend on the thread count. */
void oracle_dw(int64_t M, int64_t H, int64_t V, const double *coeff, const double *h, double *dw,
               int nthreads) {
    const int nt = pick_threads(nthreads);
#pragma omp parallel for schedule(static) num_threads(nt)
    for (int64_t v = 0; v < V; ++v) {
        double *o = dw + v * H;
        for (int64_t d = 0; d < H; ++d) o[d] = 0.0;
        for (int64_t m = 0; m < M; ++m) {
            const double c = coeff[m * V + v];
            if (c == 0.0) continue;
            const double *hm = h + m * H;
            for (int64_t d = 0; d < H; ++d) o[d] += c * hm[d];
        }
    }
}

/* dh[m,d] = sum_v coeff[m,v] * w[v,d]; each output column is owned by one
 * thread and summed over v in ascending order, so the result does not depend
 * on the thread count. */
void oracle_dh(int64_t M, int64_t H, int64_t V, int bits, int group, const uint32_t *wq,
               const double *scales, const double *biases, const double *coeff, double *dh,
               int nthreads) {
    const int nt = pick_threads(nthreads);
    for (int64_t i = 0; i < M * H; ++i) dh[i] = 0.0;
    const int64_t ngroups = H / group;
    const int64_t wpr = H * bits / 32;
#pragma omp parallel num_threads(nt)
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(static)
        for (int64_t g = 0; g < ngroups; ++g) {
            const int64_t d0 = g * group, d1 = d0 + group;
            for (int64_t v = 0; v < V; ++v) {
                const double s = scales[v * ngroups + g];
                const double b = biases[v * ngroups + g];
                for (int64_t d = d0; d < d1; ++d) w[d] = s * (double)code_at(wq + v * wpr, bits, d) + b;
                for (int64_t m = 0; m < M; ++m) {
                    const double c = coeff[m * V + v];
                    double *o = dh + m * H;
                    for (int64_t d = d0; d < d1; ++d) o[d] += c * w[d];
                }
            }
        }
        free(w);
    }
}
