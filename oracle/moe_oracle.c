/*
 * CPU oracle kernels for the DeepSeek-style Mixture-of-Experts decode layer.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
 * CPU-baseline leg are the only callers.  Nothing here is shared with the
 * CUDA path: no header, helper, table or constant of that path is used, and
 * that path never calls into this file.
 *
 * Three plain loops live here because they are too slow in numpy at the
 * DeepSeek-R1 shape (hidden 7168, 256 experts); every other step of the
 * oracle is Python in oracle/*.py.
 *
 *   oracle_gate_logits  gate logits l[t,e] = sum_h x[t,h] * Wg[e,h] in fp32,
 *                       in the fixed summation order that makes the routing
 *                       decision reproducible (see the function comment).
 *                       Source: Moreh report "21K output tokens/s DeepSeek
 *                       inference on MI300X with Expert Parallelism",
 *                       section "Overview": a light gating network picks a
 *                       small subset of experts per token.
 *   oracle_matmul_fp8   out[v,n] = sum_k a[v,k] * (q[n,k] * s[n/128,k/128])
 *                       in fp64: an FP8 e4m3 weight matrix with one fp32
 *                       scale per 128x128 block, applied to fp64 vectors.
 *   oracle_matmul_bf16  out[v,n] = sum_k a[v,k] * w[n,k] in fp64 for a bf16
 *                       weight matrix.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no fast-math, so
 * every float operation is the IEEE operation written).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE binary32: widening is a 16-bit shift. */
static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * FP8 e4m3 ("fn" variant, the OCP FP8 E4M3 format): 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN.
 *   exponent field 0  : subnormal, value = m/8 * 2^-6 = m * 2^-9
 *   exponent field e>0: normal,    value = (1 + m/8) * 2^(e-7)
 */
static double e4m3_value(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10);
    return sign ? -v : v;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Gate logits in fp32 with a fixed summation order.
 *
 * The pages give no formula for the gate; the plainest reading is a linear
 * map l = x Wg^T.  Because the selected experts (an integer decision) depend
 * on the low bits of l, the summation order is part of the definition here:
 *   - the hidden index h belongs to slice s = (h / 8) mod 32;
 *   - partial p_s accumulates x[h]*Wg[e,h] over its slice in increasing h,
 *     each step one fp32 fused multiply-add;
 *   - the 32 partials are combined by a butterfly: for o = 16, 8, 4, 2, 1,
 *     v_s <- v_s + v_(s xor o) (all v_s end equal);
 *   - an optional per-expert offset is then added in fp32.
 * A bf16 x bf16 product is exact in fp32, so each fused step equals an
 * exact product followed by one rounded fp32 addition.
 */
void oracle_gate_logits(int64_t T, int64_t E, int64_t H,
                        const uint16_t *x, const uint16_t *wg,
                        const float *offset, float *logits)
{
    int64_t te;
#pragma omp parallel for schedule(static)
    for (te = 0; te < T * E; ++te) {
        int64_t t = te / E, e = te % E;
        const uint16_t *xr = x + t * H;
        const uint16_t *wr = wg + e * H;
        float part[32];
        float next[32];
        int s, o;
        int64_t h;
        for (s = 0; s < 32; ++s)
            part[s] = 0.0f;
        for (h = 0; h < H; ++h) {
            s = (int)((h / 8) % 32);
            part[s] = fmaf(bf16_bits_to_float(xr[h]), bf16_bits_to_float(wr[h]), part[s]);
        }
        for (o = 16; o >= 1; o /= 2) {
            for (s = 0; s < 32; ++s)
                next[s] = part[s] + part[s ^ o];
            memcpy(part, next, sizeof part);
        }
        logits[t * E + e] = offset ? part[0] + offset[e] : part[0];
    }
}

/*
 * out[v, n] = sum_k a[v, k] * (value(q[n, k]) * s[n / 128, k / 128]), fp64.
 * q is row-major [N, K] (K contiguous), s is row-major [N/128, K/128].
 */
void oracle_matmul_fp8(int64_t nvec, int64_t N, int64_t K,
                       const double *a, const uint8_t *q, const float *s,
                       double *out)
{
    double table[256];
    int c;
    int64_t vn;
    for (c = 0; c < 256; ++c)
        table[c] = e4m3_value((uint8_t)c);
#pragma omp parallel for schedule(static)
    for (vn = 0; vn < nvec * N; ++vn) {
        int64_t v = vn / N, n = vn % N, k;
        const double *av = a + v * K;
        const uint8_t *qn = q + n * K;
        const float *sn = s + (n / 128) * (K / 128);
        double acc = 0.0;
        for (k = 0; k < K; ++k)
            acc += av[k] * (table[qn[k]] * (double)sn[k / 128]);
        out[v * N + n] = acc;
    }
}

/* out[v, n] = sum_k a[v, k] * w[n, k], fp64, w bf16 row-major [N, K]. */
void oracle_matmul_bf16(int64_t nvec, int64_t N, int64_t K,
                        const double *a, const uint16_t *w, double *out)
{
    int64_t vn;
#pragma omp parallel for schedule(static)
    for (vn = 0; vn < nvec * N; ++vn) {
        int64_t v = vn / N, n = vn % N, k;
        const double *av = a + v * K;
        const uint16_t *wn = w + n * K;
        double acc = 0.0;
        for (k = 0; k < K; ++k)
            acc += av[k] * (double)bf16_bits_to_float(wn[k]);
        out[v * N + n] = acc;
    }
}
