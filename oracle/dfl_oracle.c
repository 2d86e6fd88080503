/*
 * dfl_oracle.c -- numeric core of the ORACLE for the DFlash speculative-decode step.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU-baseline leg load
 * this file's library. It shares no code, header, table or constant with the CUDA path.
 *
 * Everything is a plain loop in IEEE double precision, reductions in ascending index order, and a
 * result is rounded to float (the pages' "floats") only where it is stored. OpenMP splits only the
 * independent outputs of a product (one output column per iteration), so every number is the same
 * for any thread count. Build with -ffp-contract=off so no multiply-add is fused on any host.
 *
 * Formats (stated readings; the pages give none):
 *  - Q4_1 block ("5 bits per weight with scales and minimums", model card "Nemotron-3.5-Bolt-E4B-
 *    DFlash-NPU2", spec table): 32 weights along the reduction dimension of one output column; bytes
 *    0-1 the fp16 scale d, bytes 2-3 the fp16 minimum m, then 16 bytes of 4-bit codes q, element i in
 *    byte 4 + i/2, low nibble for even i. Weight value w = d*q + m, the exact real number (it is
 *    exact in double: d*q has at most 15 significant bits).
 *  - bf16: the upper half of an IEEE binary32; rounding to bf16 is round-to-nearest, ties to even.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- number formats ------------------------------------------------------------------------ */

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_value(uint16_t h)
{
    int sign = (h >> 15) & 1, e = (h >> 10) & 31, f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* zero or subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);    /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bf16 bits are the upper 16 bits of a binary32. */
static double bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 value (8 significant bits), ties to even, returned as float.
 * Written from the format's definition: the spacing of bf16 values near |x| is 2^(e-7) where
 * 2^e <= |x| < 2^(e+1), and 2^-133 below the normal range. */
static float round_bf16(double x)
{
    if (x == 0.0 || isnan(x) || isinf(x))
        return (float)x;
    int E;
    frexp(x, &E);                                  /* |x| = f * 2^E, f in [0.5, 1) */
    int e = E - 1;
    if (e < -126)
        e = -126;
    double ulp = ldexp(1.0, e - 7);
    double r = nearbyint(x / ulp) * ulp;           /* current rounding mode: to nearest, ties even */
    return (float)r;                               /* exact: r has at most 8 significant bits */
}

/* ---- exported: formats ----------------------------------------------------------------------- */

void orc_bf16_round(const float *x, float *y, long n)
{
    for (long i = 0; i < n; i++)
        y[i] = round_bf16((double)x[i]);
}

void orc_bf16_decode(const uint16_t *b, float *y, long n)
{
    for (long i = 0; i < n; i++)
        y[i] = (float)bf16_value(b[i]);
}

void orc_half_decode(const uint16_t *h, double *y, long n)
{
    for (long i = 0; i < n; i++)
        y[i] = half_value(h[i]);
}

/* One Q4_1 block -> its 32 weights w_i = d*q_i + m (exact). */
static void q41_block(const uint8_t *blk, double *w)
{
    uint16_t dh, mh;
    memcpy(&dh, blk, 2);
    memcpy(&mh, blk + 2, 2);
    double d = half_value(dh), m = half_value(mh);
    for (int i = 0; i < 32; i++) {
        int q = (blk[4 + i / 2] >> ((i & 1) ? 4 : 0)) & 15;
        w[i] = d * (double)q + m;
    }
}

void orc_q41_dequant(const uint8_t *blocks, long nblocks, double *w)
{
    for (long b = 0; b < nblocks; b++)
        q41_block(blocks + 20 * b, w + 32 * b);
}

/* ---- exported: products ---------------------------------------------------------------------- */

/* y[r][n] = sum_k x[r][k] * w[n][k] for a Q4_1 matrix W of N output columns, each K/32 blocks
 * (uint8 [N][K/32][20]). x holds R rows of K floats; the sum runs k = 0..K-1 in order, in double,
 * and is rounded to float once. Row r's result does not depend on R. */
void orc_linear_q41(const float *x, int R, int K, const uint8_t *W, int N, float *y)
{
    const int nb = K / 32;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        double acc[64];
        double w[32];
        for (int r0 = 0; r0 < R; r0 += 64) {
            int rr = R - r0 < 64 ? R - r0 : 64;
            for (int r = 0; r < rr; r++)
                acc[r] = 0.0;
            for (int b = 0; b < nb; b++) {
                q41_block(W + ((long)n * nb + b) * 20, w);
                for (int r = 0; r < rr; r++) {
                    const float *xr = x + (long)(r0 + r) * K + 32 * b;
                    double a = acc[r];
                    for (int i = 0; i < 32; i++)
                        a += (double)xr[i] * w[i];
                    acc[r] = a;
                }
            }
            for (int r = 0; r < rr; r++)
                y[(long)(r0 + r) * N + n] = (float)acc[r];
        }
    }
}

/* Same product for a bf16 matrix stored [N][K] (one output column per row of K values). */
void orc_linear_bf16(const float *x, int R, int K, const uint16_t *W, int N, float *y)
{
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        const uint16_t *wn = W + (long)n * K;
        for (int r = 0; r < R; r++) {
            const float *xr = x + (long)r * K;
            double a = 0.0;
            for (int k = 0; k < K; k++)
                a += (double)xr[k] * bf16_value(wn[k]);
            y[(long)r * N + n] = (float)a;
        }
    }
}

/* ---- exported: sampling ------------------------------------------------------------------------ */

/* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014):
 * the finaliser applied to state + golden gamma. */
static uint64_t splitmix64(uint64_t x)
{
    uint64_t z = x + 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* The uniform in [0, 1) drawn for the token at absolute position pos: the top 53 bits of
 * splitmix64(seed XOR (pos * golden gamma)), times 2^-53. */
/* ---- exported: threads of the products (results do not depend on them) ----------------------- */

void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

double orc_uniform(uint64_t seed, int64_t pos)
{
    uint64_t z = splitmix64(seed ^ ((uint64_t)pos * 0x9E3779B97F4A7C15ULL));
    return (double)(z >> 11) * (1.0 / 9007199254740992.0);
}

/* Sampled token from logits at temperature T: p_j = exp((l_j - max)/T); the token is the smallest j
 * whose running sum of p exceeds u * sum(p) (sums in ascending j, double). *rel_gap receives the
 * distance from u * sum(p) to the nearer edge of the chosen token's interval, divided by sum(p), so a
 * caller can tell a draw that fell next to a boundary. */
int orc_sample(const float *logits, int V, double T, double u, double *rel_gap)
{
    double mx = -INFINITY;
    for (int j = 0; j < V; j++)
        if ((double)logits[j] > mx)
            mx = (double)logits[j];
    double Z = 0.0;
    for (int j = 0; j < V; j++)
        Z += exp(((double)logits[j] - mx) / T);
    double thr = u * Z, c = 0.0;
    int last = 0;
    for (int j = 0; j < V; j++) {
        double p = exp(((double)logits[j] - mx) / T);
        if (p > 0.0)
            last = j;
        double prev = c;
        c += p;
        if (c > thr) {
            if (rel_gap) {
                double g0 = thr - prev, g1 = c - thr;
                *rel_gap = (g0 < g1 ? g0 : g1) / Z;
            }
            return j;
        }
    }
    if (rel_gap)
        *rel_gap = 0.0;
    return last;
}
