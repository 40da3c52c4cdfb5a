/*
 * kv_oracle.c -- plain fp64 CPU oracle for the shared multi-agent KV codec.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or constant with the
 * CUDA library; the two agree only through the byte formats they both write.
 *
 * Everything here is deliberately slow and literal: every value is carried in
 * double precision, every rounding to a storage format (bf16, fp16, fp32) is
 * written out from the IEEE-754 definition of round-to-nearest-even, and the
 * steps follow the order in which the pages describe them.
 *
 * Sources (web pages, cited by title and section):
 *  [PolyKV]   "PolyKV: A Shared Asymmetrically-Compressed KV Cache Pool for
 *             Multi-Agent LLM Inference" -- 2.A core architecture
 *             (SharedKVPool, PooledAgent), 2.B asymmetric compression
 *             (1. keys, 2. values: rotation / quantization / dequantization),
 *             compression-ratio equation.
 *  [QKVShare] "QKVShare: Quantized KV-Cache Handoff for Multi-Agent On-Device
 *             LLMs" -- Methodology 1 (per-token bitwidth from {2,4,8,FP16}),
 *             2 (CacheCard: quantized groups, per-token bitwidths, metadata
 *             seq_len / model_id / position offset), 3 (injection: rebuild
 *             16-bit past_key_values).
 *
 * Choices the pages leave open, fixed here (the same readings the library
 * documents): one K scale per layer tensor, symmetric range [-127,127];
 * Sylvester-order FWHT without random signs; sigma = ||v||/sqrt(d) stored as
 * fp16; the 8-level Lloyd-Max N(0,1) codebook +-0.2451/0.7560/1.3440/2.1520
 * with midpoint thresholds (upper bin on a tie); 8 codes packed little-endian
 * into 3 bytes; CacheCard groups of 32 along head_dim with fp16 scale and
 * fp16 zero point (z = group minimum); 16-bit tokens stored verbatim.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* Threads                                                                    */
/* ------------------------------------------------------------------------- */

void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------- */
/* Storage formats, from the IEEE-754 definitions                             */
/* ------------------------------------------------------------------------- */

/* Round x to a binary format with p significand bits (leading bit included)
 * and minimum normal exponent emin, ties to even.  Overflow is left to the
 * caller (the result may be one binade above the format's largest finite). */
static double round_to_format(double x, int p, int emin)
{
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    frexp(x, &e);                 /* |x| in [2^(e-1), 2^e) */
    int lead = e - 1;
    if (lead < emin) lead = emin; /* subnormal range: fixed quantum */
    int qexp = lead - (p - 1);    /* exponent of one unit in the last place */
    double scaled = ldexp(x, -qexp);  /* exact: power-of-two scaling */
    double r = nearbyint(scaled);     /* default rounding mode: to nearest, ties even */
    return ldexp(r, qexp);
}

double orc_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* bf16: 8 significand bits, emin -126, largest finite (2-2^-7)*2^127. */
uint16_t orc_f64_to_bf16(double x)
{
    if (isnan(x)) return 0x7FC0;
    double r = round_to_format(x, 8, -126);
    if (fabs(r) >= ldexp(1.0, 128)) r = copysign(INFINITY, x);
    float f = (float)r;           /* exact: every bf16 value is an fp32 value */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1F;
    int man = h & 0x3FF;
    double v;
    if (ex == 0x1F) v = man ? NAN : INFINITY;
    else if (ex == 0) v = ldexp((double)man, -24);
    else v = ldexp((double)(man | 0x400), ex - 25);
    return sign ? -v : v;
}

/* fp16: 11 significand bits, emin -14, largest finite 65504. */
uint16_t orc_f64_to_f16(double x)
{
    if (isnan(x)) return 0x7E00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double r = fabs(round_to_format(x, 11, -14));
    if (r >= 65536.0) return sign | 0x7C00;
    if (r == 0.0) return sign;
    int e;
    frexp(r, &e);
    int lead = e - 1;
    if (lead < -14) {
        return sign | (uint16_t)ldexp(r, 24);           /* subnormal: r / 2^-24 */
    }
    uint16_t man = (uint16_t)(ldexp(r, -lead) * 1024.0 - 1024.0);
    return sign | (uint16_t)((lead + 15) << 10) | man;
}

/* ------------------------------------------------------------------------- */
/* Walsh-Hadamard transform                                                   */
/* ------------------------------------------------------------------------- */

/* In-place unnormalised Walsh-Hadamard transform in Sylvester (natural)
 * order: y[i] = sum_j (-1)^popcount(i&j) x[j].  Butterflies over each index
 * bit in turn.  [PolyKV] 2.B.2 rotation. */
void orc_fwht(double *x, int d)
{
    for (int h = 1; h < d; h <<= 1)
        for (int i = 0; i < d; i += 2 * h)
            for (int j = i; j < i + h; j++) {
                double a = x[j], b = x[j + h];
                x[j] = a + b;
                x[j + h] = a - b;
            }
}

/* ------------------------------------------------------------------------- */
/* Lloyd-Max quantizer for N(0,1)                                             */
/* ------------------------------------------------------------------------- */

static double phi(double x) { return exp(-0.5 * x * x) / sqrt(2.0 * M_PI); }
static double Phi(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

/* Lloyd iteration for the `levels`-level minimum-MSE scalar quantizer of a
 * standard normal: thresholds at midpoints of adjacent centroids, centroids
 * at the conditional mean of each cell, E[X | a<X<b] = (phi(a)-phi(b)) /
 * (Phi(b)-Phi(a)).  Returns the iterations used; writes the centroids and the
 * resulting mean squared error.  [PolyKV] 2.B.2 quantization names the
 * Lloyd-Max centroids for N(0,1). */
int orc_lloyd_max_gauss(int levels, int max_iter, double tol, double *c, double *mse)
{
    for (int i = 0; i < levels; i++)            /* spread start over +-2 */
        c[i] = -2.0 + 4.0 * (i + 0.5) / levels;
    int it;
    for (it = 1; it <= max_iter; it++) {
        double delta = 0.0;
        for (int i = 0; i < levels; i++) {
            double a = (i == 0) ? -INFINITY : 0.5 * (c[i - 1] + c[i]);
            double b = (i == levels - 1) ? INFINITY : 0.5 * (c[i] + c[i + 1]);
            double pa = isinf(a) ? 0.0 : phi(a), pb = isinf(b) ? 0.0 : phi(b);
            double m = (pa - pb) / (Phi(b) - Phi(a));
            delta = fmax(delta, fabs(m - c[i]));
            c[i] = m;
        }
        if (delta < tol) break;
    }
    /* E[(X-Q(X))^2] = 1 - sum_i c_i^2 P_i at a fixed point (centroid condition);
     * computed here from the cell integrals directly:
     * int_a^b (x-c)^2 phi = [P + a phi(a) - b phi(b)] - 2c[phi(a)-phi(b)] + c^2 P. */
    double e = 0.0;
    for (int i = 0; i < levels; i++) {
        double a = (i == 0) ? -INFINITY : 0.5 * (c[i - 1] + c[i]);
        double b = (i == levels - 1) ? INFINITY : 0.5 * (c[i] + c[i + 1]);
        double P = Phi(b) - Phi(a);
        double pa = isinf(a) ? 0.0 : phi(a), pb = isinf(b) ? 0.0 : phi(b);
        double apa = isinf(a) ? 0.0 : a * pa, bpb = isinf(b) ? 0.0 : b * pb;
        e += (P + apa - bpb) - 2.0 * c[i] * (pa - pb) + c[i] * c[i] * P;
    }
    *mse = e;
    return it;
}

/* ------------------------------------------------------------------------- */
/* Codebook used by the codec                                                 */
/* ------------------------------------------------------------------------- */

/* The 8-level Lloyd-Max codebook for N(0,1), to four decimals, ascending. */
static const double CENTROID[8] = {
    -2.1520, -1.3440, -0.7560, -0.2451, 0.2451, 0.7560, 1.3440, 2.1520
};

void orc_centroids(double *out)
{
    for (int i = 0; i < 8; i++) out[i] = CENTROID[i];
}

/* Decision thresholds: midpoints of adjacent centroids. */
void orc_thresholds(double *out)
{
    for (int i = 0; i < 7; i++) out[i] = 0.5 * (CENTROID[i] + CENTROID[i + 1]);
}

/* Code of one rotated, normalised coordinate u: the number of thresholds
 * t_j with t_j <= u (a value on a threshold goes to the upper cell). */
int orc_v_code(double u)
{
    double t[7];
    orc_thresholds(t);
    int code = 0;
    for (int j = 0; j < 7; j++)
        if (t[j] <= u) code++;
    return code;
}

/* ------------------------------------------------------------------------- */
/* Error bits written into the pool / card header                             */
/* ------------------------------------------------------------------------- */

#define ORC_FLAG_NONFINITE 1u  /* an input element was Inf or NaN            */
#define ORC_FLAG_RANGE 2u      /* a scale or zero point overflowed fp16      */
#define ORC_FLAG_BITS 4u       /* a CacheCard bitwidth outside {2,4,8,16}    */

/* ------------------------------------------------------------------------- */
/* Keys: per-tensor symmetric int8.  [PolyKV] 2.B.1                           */
/* ------------------------------------------------------------------------- */

/* Largest |k| over one layer's key tensor (all heads, tokens, dims), exact.
 * Sets *nonfinite if any element is Inf/NaN (those are skipped). */
double orc_k_absmax(const uint16_t *k, size_t n, int *nonfinite)
{
    double m = 0.0;
    int bad = 0;
    for (size_t i = 0; i < n; i++) {
        double a = fabs(orc_bf16_to_f64(k[i]));
        if (!isfinite(a)) { bad = 1; continue; }
        if (a > m) m = a;
    }
    if (nonfinite) *nonfinite = bad;
    return m;
}

/* s = m / 127 rounded once to fp32.  The fp64 quotient rounded to fp32 is
 * the correctly rounded fp32 quotient (53 >= 2*24+2, double rounding is
 * innocuous for division). */
float orc_k_scale(double m)
{
    return (float)(m / 127.0);
}

/* Code of one key element: the integer nearest to the real k/s, ties to
 * even, clamped to [-127,127]; 0 when s == 0.  For fp32 s and bf16 k the
 * fp64 quotient lands on the same side of every half-integer as the real
 * quotient, and exactly on it only when the real quotient is on it. */
int orc_k_code(uint16_t kbits, float s)
{
    if (s == 0.0f) return 0;
    double k = orc_bf16_to_f64(kbits);
    if (!isfinite(k)) return 0;
    double q = nearbyint(k / (double)s);
    if (q > 127.0) q = 127.0;
    if (q < -127.0) q = -127.0;
    return (int)q;
}

/* Key reconstruction: q*s (exact in fp64) rounded to bf16. */
uint16_t orc_k_decode(int q, float s)
{
    return orc_f64_to_bf16((double)q * (double)s);
}

/* Keys in q8_0 blocks, the format [PolyKV] 2.B.1 names by its label "q8_0":
 * every 32 consecutive elements of a key vector (along d) share one fp16
 * scale s_b = fp16(max|k| / 127) (round to nearest even), and each element
 * is the int8 code nearest to k / s_b (ties to even) clamped to [-127, 127]
 * -- the clamp only bites when s_b is an fp16 subnormal, rounded down by
 * more than a half code.  s_b = 0 (every |k| below 127 * 2^-25) gives codes
 * 0.  Sets *nonfinite for Inf/NaN elements (skipped, code 0) and *range when
 * finite input overflows the fp16 scale. */
uint16_t orc_k_block_scale(const uint16_t *k32, int *nonfinite, int *range)
{
    double m = orc_k_absmax(k32, 32, nonfinite);
    uint16_t sb = orc_f64_to_f16(m / 127.0);
    if (range) *range = (sb & 0x7C00u) == 0x7C00u;
    return sb;
}

int orc_k_block_code(uint16_t kbits, uint16_t sbits)
{
    double s = orc_f16_to_f64(sbits);
    if (s == 0.0 || !isfinite(s)) return 0;
    double k = orc_bf16_to_f64(kbits);
    if (!isfinite(k)) return 0;
    double q = nearbyint(k / s);
    if (q > 127.0) q = 127.0;
    if (q < -127.0) q = -127.0;
    return (int)q;
}

/* Block key reconstruction: q * s_b (exact in fp64) rounded to bf16. */
uint16_t orc_k_block_decode(int q, uint16_t sbits)
{
    return orc_f64_to_bf16((double)q * orc_f16_to_f64(sbits));
}

/* ------------------------------------------------------------------------- */
/* Values: FWHT rotation + Lloyd-Max 3-bit codes.  [PolyKV] 2.B.2             */
/* ------------------------------------------------------------------------- */

/* Encode one value vector of d bf16 elements.
 *  1. rotate: y = H_d v (Sylvester, unnormalised; the orthonormal rotation
 *     is y / sqrt(d)),
 *  2. normalise: sigma = ||v|| / sqrt(d), so the orthonormal coordinates
 *     divided by sigma, u_i = y_i / ||v||, are near N(0,1),
 *  3. quantize: code_i = cell of u_i in the Lloyd-Max codebook.
 * Writes d codes (0..7), the fp16 bits of sigma, and optionally the u_i.
 * A zero vector gets u = 0, every code 4 (the cell just above 0), sigma 0.
 * Returns error flags (NONFINITE for Inf/NaN input, RANGE if sigma
 * overflows fp16). */
uint32_t orc_v_encode_vec(const uint16_t *v, int d, uint8_t *codes,
                          uint16_t *sigma_h, double *u_out)
{
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    double n2 = 0.0;
    uint32_t flags = 0;
    for (int i = 0; i < d; i++) {
        y[i] = orc_bf16_to_f64(v[i]);
        if (!isfinite(y[i])) flags |= ORC_FLAG_NONFINITE;
        n2 += y[i] * y[i];
    }
    double nrm = sqrt(n2);
    orc_fwht(y, d);
    double sigma = nrm / sqrt((double)d);
    uint16_t sh = orc_f64_to_f16(sigma);
    /* RANGE: a finite vector whose sigma is beyond fp16; a non-finite input
     * is reported as NONFINITE only. */
    if (!(flags & ORC_FLAG_NONFINITE) && (sh & 0x7C00) == 0x7C00) flags |= ORC_FLAG_RANGE;
    *sigma_h = sh;
    for (int i = 0; i < d; i++) {
        double u = (nrm > 0.0 && isfinite(nrm)) ? y[i] / nrm : 0.0;
        if (u_out) u_out[i] = u;
        codes[i] = (uint8_t)orc_v_code(u);
    }
    free(y);
    return flags;
}

/* 3-bit packing: each run of 8 codes c_0..c_7 is the 24-bit little-endian
 * word sum_j c_j << 3j, stored as 3 bytes.  d must be a multiple of 8. */
void orc_pack3(const uint8_t *codes, int d, uint8_t *out)
{
    for (int g = 0; g < d / 8; g++) {
        uint32_t w = 0;
        for (int j = 0; j < 8; j++) w |= (uint32_t)(codes[8 * g + j] & 7u) << (3 * j);
        out[3 * g + 0] = (uint8_t)(w & 0xFF);
        out[3 * g + 1] = (uint8_t)((w >> 8) & 0xFF);
        out[3 * g + 2] = (uint8_t)((w >> 16) & 0xFF);
    }
}

void orc_unpack3(const uint8_t *in, int d, uint8_t *codes)
{
    for (int g = 0; g < d / 8; g++) {
        uint32_t w = (uint32_t)in[3 * g] | ((uint32_t)in[3 * g + 1] << 8) |
                     ((uint32_t)in[3 * g + 2] << 16);
        for (int j = 0; j < 8; j++) codes[8 * g + j] = (uint8_t)((w >> (3 * j)) & 7u);
    }
}

/* Decode one value vector: centroid lookup, inverse rotation (the
 * orthonormal FWHT is its own inverse: H_d c / sqrt(d)), rescale by the
 * stored fp16 sigma, round to bf16.  [PolyKV] 2.B.2 dequantization. */
void orc_v_decode_vec(const uint8_t *codes, uint16_t sigma_h, int d, uint16_t *out)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)d);
    for (int i = 0; i < d; i++) z[i] = CENTROID[codes[i] & 7];
    orc_fwht(z, d);
    double sig = orc_f16_to_f64(sigma_h);
    double rs = sqrt((double)d);
    for (int i = 0; i < d; i++) out[i] = orc_f64_to_bf16(sig * z[i] / rs);
    free(z);
}

/* ------------------------------------------------------------------------- */
/* SharedKVPool byte image.  [PolyKV] 2.A: computed once, compressed, stored  */
/* as one object whose size does not depend on the number of agents.         */
/* ------------------------------------------------------------------------- */
/*
 * Layout (all integers little-endian, every section 256-byte aligned):
 *   [0,256)        header: u32 magic 'KVPL', u32 version 1, i32 L, H, d, T,
 *                  u32 error bits, u32 key format (0: one scale per layer
 *                  tensor, 1: q8_0 blocks), u64 off_scales, off_layers,
 *                  layer_stride, sec_v, sec_sigma, total_bytes, zero pad
 *   off_scales     fp32 s[L]          (format 1: zero)
 *   off_layers + l*layer_stride:
 *                  +0         int8 K codes  [H][T][d]
 *                  +sec_v     u8 V codes    [H][T][3d/8]
 *                  +sec_sigma fp16 sigma    [H][T]
 *   off_kscales    format 1 only: fp16 block scales [L][H][T][d/32]
 */

static uint64_t al256(uint64_t x) { return (x + 255u) & ~(uint64_t)255u; }

typedef struct {
    uint64_t off_scales, off_layers, layer_stride, sec_v, sec_sigma, total, off_kscales, total_q8;
} orc_pool_geom;

static orc_pool_geom pool_geom(int L, int H, int d, int T)
{
    orc_pool_geom g;
    uint64_t nv = (uint64_t)H * (uint64_t)T;
    g.off_scales = 256;
    g.off_layers = al256(256 + 4ull * (uint64_t)L);
    g.sec_v = al256(nv * (uint64_t)d);
    g.sec_sigma = al256(g.sec_v + nv * (uint64_t)(3 * d / 8));
    g.layer_stride = al256(g.sec_sigma + 2ull * nv);
    g.total = g.off_layers + (uint64_t)L * g.layer_stride;
    g.off_kscales = g.total;
    g.total_q8 = g.off_kscales + al256((uint64_t)L * nv * (uint64_t)(d / 32) * 2u);
    return g;
}

size_t orc_pool_bytes(int L, int H, int d, int T)
{
    return (size_t)pool_geom(L, H, d, T).total;
}

/* Pool bytes for key format k_mode (0: per-tensor scale, 1: q8_0 blocks). */
size_t orc_pool_bytes_mode(int L, int H, int d, int T, int k_mode)
{
    orc_pool_geom g = pool_geom(L, H, d, T);
    return (size_t)(k_mode == 1 ? g.total_q8 : g.total);
}

void orc_pool_geometry(int L, int H, int d, int T, uint64_t *out6)
{
    orc_pool_geom g = pool_geom(L, H, d, T);
    out6[0] = g.off_scales; out6[1] = g.off_layers; out6[2] = g.layer_stride;
    out6[3] = g.sec_v; out6[4] = g.sec_sigma; out6[5] = g.total;
}

/* off_kscales and the format-1 total. */
void orc_pool_geometry_q8(int L, int H, int d, int T, uint64_t *out2)
{
    orc_pool_geom g = pool_geom(L, H, d, T);
    out2[0] = g.off_kscales; out2[1] = g.total_q8;
}

static void put32(uint8_t *p, uint32_t v) { memcpy(p, &v, 4); }
static void put64(uint8_t *p, uint64_t v) { memcpy(p, &v, 8); }
static uint32_t get32(const uint8_t *p) { uint32_t v; memcpy(&v, p, 4); return v; }
static uint64_t get64(const uint8_t *p) { uint64_t v; memcpy(&v, p, 8); return v; }

/* Encode every layer into a zero-initialised pool image of orc_pool_bytes()
 * bytes.  k[l], v[l] point at layer l's bf16 [H][T][d] tensors.  If u_out is
 * given it receives the fp64 rotated coordinates u (layer-major, [L][H][T][d])
 * used to decide each V code.  Returns the error bits (also in the header). */
uint32_t orc_pool_encode_mode(int L, int H, int d, int T, int k_mode, const uint16_t *const *k,
                              const uint16_t *const *v, uint8_t *pool, double *u_out);

uint32_t orc_pool_encode(int L, int H, int d, int T, const uint16_t *const *k,
                         const uint16_t *const *v, uint8_t *pool, double *u_out)
{
    return orc_pool_encode_mode(L, H, d, T, 0, k, v, pool, u_out);
}

/* As orc_pool_encode, with the key format chosen by k_mode: 0 one scale per
 * layer tensor, 1 q8_0 blocks (scales in the off_kscales region, s[L] left
 * zero).  The image is orc_pool_bytes_mode() bytes. */
uint32_t orc_pool_encode_mode(int L, int H, int d, int T, int k_mode, const uint16_t *const *k,
                              const uint16_t *const *v, uint8_t *pool, double *u_out)
{
    orc_pool_geom g = pool_geom(L, H, d, T);
    uint64_t nv = (uint64_t)H * (uint64_t)T;
    uint64_t ne = nv * (uint64_t)d;
    uint32_t flags = 0;

    put32(pool + 0, 0x4C50564Bu);      /* "KVPL" */
    put32(pool + 4, 1u);
    put32(pool + 8, (uint32_t)L);
    put32(pool + 12, (uint32_t)H);
    put32(pool + 16, (uint32_t)d);
    put32(pool + 20, (uint32_t)T);
    put64(pool + 32, g.off_scales);
    put64(pool + 40, g.off_layers);
    put64(pool + 48, g.layer_stride);
    put64(pool + 56, g.sec_v);
    put64(pool + 64, g.sec_sigma);
    put32(pool + 28, (uint32_t)k_mode);
    put64(pool + 72, k_mode == 1 ? g.total_q8 : g.total);

    for (int l = 0; l < L; l++) {
        uint8_t *lay = pool + g.off_layers + (uint64_t)l * g.layer_stride;
        int8_t *kc = (int8_t *)lay;
        const uint16_t *kl = k[l];
        if (k_mode == 1) {
            const uint64_t nb = ne / 32u;
            uint8_t *ks = pool + g.off_kscales + (uint64_t)l * nb * 2u;
            uint32_t kflags = 0;
#pragma omp parallel for schedule(static) reduction(| : kflags)
            for (int64_t b = 0; b < (int64_t)nb; b++) {
                int bad = 0, range = 0;
                uint16_t sb = orc_k_block_scale(kl + (uint64_t)b * 32u, &bad, &range);
                if (bad) kflags |= ORC_FLAG_NONFINITE;
                else if (range) kflags |= ORC_FLAG_RANGE;
                memcpy(ks + 2u * (uint64_t)b, &sb, 2);
                for (int i = 0; i < 32; i++)
                    kc[(uint64_t)b * 32u + (uint64_t)i] = (int8_t)orc_k_block_code(kl[(uint64_t)b * 32u + (uint64_t)i], sb);
            }
            flags |= kflags;
        } else {
            int bad = 0;
            double m = orc_k_absmax(kl, (size_t)ne, &bad);
            if (bad) flags |= ORC_FLAG_NONFINITE;
            float s = orc_k_scale(m);
            memcpy(pool + g.off_scales + 4u * (uint64_t)l, &s, 4);
#pragma omp parallel for schedule(static)
            for (int64_t i = 0; i < (int64_t)ne; i++) kc[i] = (int8_t)orc_k_code(kl[i], s);
        }

        uint8_t *vc = lay + g.sec_v;
        uint8_t *sg = lay + g.sec_sigma;
        const uint16_t *vl = v[l];
        uint32_t vflags = 0;
#pragma omp parallel for schedule(static) reduction(| : vflags)
        for (int64_t n = 0; n < (int64_t)nv; n++) {
            uint8_t codes[128];
            uint16_t sh;
            double *uo = u_out ? u_out + ((uint64_t)l * nv + (uint64_t)n) * (uint64_t)d : NULL;
            vflags |= orc_v_encode_vec(vl + (uint64_t)n * d, d, codes, &sh, uo);
            orc_pack3(codes, d, vc + (uint64_t)n * (uint64_t)(3 * d / 8));
            memcpy(sg + 2u * (uint64_t)n, &sh, 2);
        }
        flags |= vflags;
    }
    put32(pool + 24, flags);
    return flags;
}

/* PooledAgent read, [PolyKV] 2.A: decode layers [lb, le) of the pool once and
 * store each decoded vector into every agent's cache.  k_dst/v_dst hold
 * n_agents*L pointers, agent-major (index a*L + l), each a bf16 [H][T][d]
 * tensor.  Returns 0, or -1 if the header is not a version-1 pool. */
int orc_pool_decode_into(const uint8_t *pool, int lb, int le, int n_agents,
                         uint16_t *const *k_dst, uint16_t *const *v_dst)
{
    if (get32(pool) != 0x4C50564Bu || get32(pool + 4) != 1u) return -1;
    int L = (int)get32(pool + 8), H = (int)get32(pool + 12);
    int d = (int)get32(pool + 16), T = (int)get32(pool + 20);
    const int k_mode = (int)get32(pool + 28);
    if (k_mode != 0 && k_mode != 1) return -1;
    orc_pool_geom g = pool_geom(L, H, d, T);
    uint64_t nv = (uint64_t)H * (uint64_t)T;
    for (int l = lb; l < le; l++) {
        const uint8_t *lay = pool + g.off_layers + (uint64_t)l * g.layer_stride;
        float s;
        memcpy(&s, pool + g.off_scales + 4u * (uint64_t)l, 4);
        const int8_t *kc = (const int8_t *)lay;
        const uint8_t *vc = lay + g.sec_v;
        const uint8_t *sg = lay + g.sec_sigma;
        const uint8_t *ks = pool + g.off_kscales + (uint64_t)l * nv * (uint64_t)(d / 32) * 2u;
#pragma omp parallel for schedule(static)
        for (int64_t n = 0; n < (int64_t)nv; n++) {
            uint16_t kk[128], vv[128];
            uint8_t codes[128];
            uint16_t sh;
            for (int i = 0; i < d; i++) {
                const int q = kc[(uint64_t)n * d + i];
                if (k_mode == 1) {
                    uint16_t sb;
                    memcpy(&sb, ks + 2u * ((uint64_t)n * (uint64_t)(d / 32) + (uint64_t)(i / 32)), 2);
                    kk[i] = orc_k_block_decode(q, sb);
                } else {
                    kk[i] = orc_k_decode(q, s);
                }
            }
            orc_unpack3(vc + (uint64_t)n * (uint64_t)(3 * d / 8), d, codes);
            memcpy(&sh, sg + 2u * (uint64_t)n, 2);
            orc_v_decode_vec(codes, sh, d, vv);
            for (int a = 0; a < n_agents; a++) {
                memcpy(k_dst[(size_t)a * L + l] + (uint64_t)n * d, kk, 2u * (unsigned)d);
                memcpy(v_dst[(size_t)a * L + l] + (uint64_t)n * d, vv, 2u * (unsigned)d);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* CacheCard.  [QKVShare] Methodology 1-3                                      */
/* ------------------------------------------------------------------------- */
/*
 * Layout (little-endian):
 *   [0,128)     header: u32 magic 'KVCC', u32 version 1, i32 seq_len T, L, H,
 *               d, group 32, dtype 1 (bf16), u64 model_id, i64 pos_offset,
 *               u64 off_bits, off_offsets, off_layers, layer_stride,
 *               total_bytes, u32 error bits, zero pad
 *   off_bits    u8 bits[T]           (= 128)
 *   off_offsets u32 off[T]           (16-byte aligned): byte offset of token
 *               t's record inside a layer, exclusive prefix sum of sizes
 *   off_layers  (256-aligned) L layers of layer_stride bytes each.
 * Token record, b in {2,4,8}: K codes [H][d] at b bits, V codes [H][d],
 *   K (fp16 scale, fp16 zero) [H][d/32], V (scale, zero) [H][d/32]; the codes
 *   of one group of 32 form a little-endian bit string, code j at bits
 *   j*b .. j*b+b-1.  b = 16: K then V as raw 16-bit [H][d].  Every record is
 *   padded to a multiple of 16 bytes.
 */

static int valid_bits(int b) { return b == 2 || b == 4 || b == 8 || b == 16; }

uint64_t orc_card_record_bytes(int b, int H, int d)
{
    uint64_t r;
    if (b == 16) r = 2ull * (uint64_t)H * (uint64_t)d * 2ull;
    else r = 2ull * ((uint64_t)H * (uint64_t)d * (uint64_t)b / 8ull + (uint64_t)H * (uint64_t)(d / 32) * 4ull);
    return (r + 15u) & ~(uint64_t)15u;
}

typedef struct {
    uint64_t off_bits, off_offsets, off_layers, layer_stride, total;
} orc_card_geom;

/* Returns -1 if some bitwidth is invalid. */
static int card_geom(int L, int H, int d, int T, const uint8_t *bits, orc_card_geom *g)
{
    uint64_t sum = 0;
    for (int t = 0; t < T; t++) {
        if (!valid_bits(bits[t])) return -1;
        sum += orc_card_record_bytes(bits[t], H, d);
    }
    g->off_bits = 128;
    g->off_offsets = (128u + (uint64_t)T + 15u) & ~(uint64_t)15u;
    g->off_layers = al256(g->off_offsets + 4ull * (uint64_t)T);
    g->layer_stride = al256(sum);
    g->total = g->off_layers + (uint64_t)L * g->layer_stride;
    return 0;
}

/* Exact card size for these bitwidths, or 0 if a bitwidth is invalid. */
size_t orc_card_bytes(int L, int H, int d, int T, const uint8_t *bits)
{
    orc_card_geom g;
    if (card_geom(L, H, d, T, bits, &g)) return 0;
    return (size_t)g.total;
}

void orc_card_geometry(int L, int H, int d, int T, const uint8_t *bits, uint64_t *out5)
{
    orc_card_geom g;
    memset(&g, 0, sizeof g);
    card_geom(L, H, d, T, bits, &g);
    out5[0] = g.off_bits; out5[1] = g.off_offsets; out5[2] = g.off_layers;
    out5[3] = g.layer_stride; out5[4] = g.total;
}

/* Quantize one group of 32 values x[0..31] at b bits, asymmetric min/max:
 * s = (max-min)/(2^b-1) and z = min, both rounded to fp16; code =
 * clamp(nearest integer to (x - z_h)/s_h, 0, 2^b-1), ties to even, 0 when
 * s_h = 0.  Writes the codes, the fp16 bits of s and z, and optionally
 * r = (x - z_h)/s_h.  Returns error flags. */
uint32_t orc_group_quant(const double *x, int b, uint8_t *q, uint16_t *s_h, uint16_t *z_h, double *r_out)
{
    uint32_t flags = 0;
    double mn = x[0], mx = x[0];
    for (int i = 0; i < 32; i++) {
        if (!isfinite(x[i])) flags |= ORC_FLAG_NONFINITE;
        if (x[i] < mn) mn = x[i];
        if (x[i] > mx) mx = x[i];
    }
    double qmax = (double)((1 << b) - 1);
    uint16_t sb = orc_f64_to_f16((mx - mn) / qmax);
    uint16_t zb = orc_f64_to_f16(mn);
    if (!(flags & ORC_FLAG_NONFINITE) && ((sb & 0x7C00) == 0x7C00 || (zb & 0x7C00) == 0x7C00))
        flags |= ORC_FLAG_RANGE;
    *s_h = sb;
    *z_h = zb;
    double s = orc_f16_to_f64(sb), z = orc_f16_to_f64(zb);
    for (int i = 0; i < 32; i++) {
        double r = (s > 0.0 && isfinite(s)) ? (x[i] - z) / s : 0.0;
        if (r_out) r_out[i] = r;
        double c = (s > 0.0 && isfinite(s)) ? nearbyint(r) : 0.0;
        if (!(c >= 0.0)) c = 0.0;     /* also catches NaN */
        if (c > qmax) c = qmax;
        q[i] = (uint8_t)c;
    }
    return flags;
}

/* Store 32 codes of b bits as a little-endian bit string of 4*b bytes. */
static void pack_group(const uint8_t *q, int b, uint8_t *out)
{
    memset(out, 0, (size_t)(4 * b));
    for (int j = 0; j < 32; j++)
        for (int k = 0; k < b; k++)
            if ((q[j] >> k) & 1) {
                int bit = j * b + k;
                out[bit >> 3] |= (uint8_t)(1u << (bit & 7));
            }
}

static void unpack_group(const uint8_t *in, int b, uint8_t *q)
{
    for (int j = 0; j < 32; j++) {
        unsigned c = 0;
        for (int k = 0; k < b; k++) {
            int bit = j * b + k;
            c |= (unsigned)((in[bit >> 3] >> (bit & 7)) & 1) << k;
        }
        q[j] = (uint8_t)c;
    }
}

/* Pack a CacheCard: header, per-token bitwidths, offsets and every layer's
 * token records into a zero-initialised buffer of orc_card_bytes() bytes.
 * If r_out is given it receives r = (x - z_h)/s_h for every quantized
 * element, laid out [L][T][2 (K,V)][H][d] (0 for 16-bit tokens).  Returns the
 * error bits (BITS alone, with nothing written, for an invalid bitwidth). */
uint32_t orc_card_pack(int L, int H, int d, int T, uint64_t model_id, int64_t pos_offset,
                       const uint8_t *bits, const uint16_t *const *k, const uint16_t *const *v,
                       uint8_t *card, double *r_out)
{
    orc_card_geom g;
    if (card_geom(L, H, d, T, bits, &g)) return ORC_FLAG_BITS;
    put32(card + 0, 0x4343564Bu);      /* "KVCC" */
    put32(card + 4, 1u);
    put32(card + 8, (uint32_t)T);
    put32(card + 12, (uint32_t)L);
    put32(card + 16, (uint32_t)H);
    put32(card + 20, (uint32_t)d);
    put32(card + 24, 32u);
    put32(card + 28, 1u);
    put64(card + 32, model_id);
    put64(card + 40, (uint64_t)pos_offset);
    put64(card + 48, g.off_bits);
    put64(card + 56, g.off_offsets);
    put64(card + 64, g.off_layers);
    put64(card + 72, g.layer_stride);
    put64(card + 80, g.total);

    uint64_t acc = 0;
    for (int t = 0; t < T; t++) {
        card[g.off_bits + (uint64_t)t] = bits[t];
        put32(card + g.off_offsets + 4ull * (uint64_t)t, (uint32_t)acc);
        acc += orc_card_record_bytes(bits[t], H, d);
    }

    uint32_t flags = 0;
    const int ng = d / 32;
    for (int l = 0; l < L; l++) {
        uint8_t *lay = card + g.off_layers + (uint64_t)l * g.layer_stride;
#pragma omp parallel for schedule(static) reduction(| : flags)
        for (int t = 0; t < T; t++) {
            int b = bits[t];
            uint8_t *rec = lay + get32(card + g.off_offsets + 4ull * (uint64_t)t);
            for (int kv = 0; kv < 2; kv++) {
                const uint16_t *src = kv ? v[l] : k[l];
                if (b == 16) {
                    uint8_t *dst = rec + (uint64_t)kv * (uint64_t)H * (uint64_t)d * 2u;
                    for (int h = 0; h < H; h++)
                        memcpy(dst + (uint64_t)h * d * 2u, src + ((uint64_t)h * T + (uint64_t)t) * d, 2u * (unsigned)d);
                    continue;
                }
                uint64_t code_bytes = (uint64_t)H * (uint64_t)d * (uint64_t)b / 8u;
                uint8_t *codes = rec + (uint64_t)kv * code_bytes;
                uint8_t *par = rec + 2u * code_bytes + (uint64_t)kv * (uint64_t)H * (uint64_t)ng * 4u;
                for (int h = 0; h < H; h++) {
                    const uint16_t *row = src + ((uint64_t)h * T + (uint64_t)t) * d;
                    for (int gi = 0; gi < ng; gi++) {
                        double x[32];
                        uint8_t q[32];
                        uint16_t sb, zb;
                        for (int i = 0; i < 32; i++) x[i] = orc_bf16_to_f64(row[32 * gi + i]);
                        double *ro = r_out ? r_out + ((((uint64_t)l * T + (uint64_t)t) * 2u + (uint64_t)kv) * H + (uint64_t)h) * d + 32u * (uint64_t)gi : NULL;
                        flags |= orc_group_quant(x, b, q, &sb, &zb, ro);
                        pack_group(q, b, codes + ((uint64_t)h * ng + (uint64_t)gi) * 4u * (uint64_t)b);
                        uint8_t *pp = par + ((uint64_t)h * ng + (uint64_t)gi) * 4u;
                        memcpy(pp, &sb, 2);
                        memcpy(pp + 2, &zb, 2);
                    }
                }
            }
        }
    }
    put32(card + 88, flags);
    return flags;
}

/* Receiver injection, [QKVShare] Methodology 3: rebuild every layer's 16-bit
 * K and V ([H][T][d] bf16) from the card.  x = q*s_h + z_h rounded to bf16;
 * 16-bit tokens are copied verbatim.  Returns 0, or -1 on a bad header. */
int orc_card_unpack(const uint8_t *card, uint16_t *const *k_out, uint16_t *const *v_out)
{
    if (get32(card) != 0x4343564Bu || get32(card + 4) != 1u) return -1;
    int T = (int)get32(card + 8), L = (int)get32(card + 12);
    int H = (int)get32(card + 16), d = (int)get32(card + 20);
    uint64_t off_bits = get64(card + 48), off_offsets = get64(card + 56);
    uint64_t off_layers = get64(card + 64), stride = get64(card + 72);
    const int ng = d / 32;
    for (int l = 0; l < L; l++) {
        const uint8_t *lay = card + off_layers + (uint64_t)l * stride;
#pragma omp parallel for schedule(static)
        for (int t = 0; t < T; t++) {
            int b = card[off_bits + (uint64_t)t];
            const uint8_t *rec = lay + get32(card + off_offsets + 4ull * (uint64_t)t);
            for (int kv = 0; kv < 2; kv++) {
                uint16_t *dst = kv ? v_out[l] : k_out[l];
                if (b == 16) {
                    const uint8_t *src = rec + (uint64_t)kv * (uint64_t)H * (uint64_t)d * 2u;
                    for (int h = 0; h < H; h++)
                        memcpy(dst + ((uint64_t)h * T + (uint64_t)t) * d, src + (uint64_t)h * d * 2u, 2u * (unsigned)d);
                    continue;
                }
                uint64_t code_bytes = (uint64_t)H * (uint64_t)d * (uint64_t)b / 8u;
                const uint8_t *codes = rec + (uint64_t)kv * code_bytes;
                const uint8_t *par = rec + 2u * code_bytes + (uint64_t)kv * (uint64_t)H * (uint64_t)ng * 4u;
                for (int h = 0; h < H; h++) {
                    uint16_t *row = dst + ((uint64_t)h * T + (uint64_t)t) * d;
                    for (int gi = 0; gi < ng; gi++) {
                        uint8_t q[32];
                        uint16_t sb, zb;
                        unpack_group(codes + ((uint64_t)h * ng + (uint64_t)gi) * 4u * (uint64_t)b, b, q);
                        memcpy(&sb, par + ((uint64_t)h * ng + (uint64_t)gi) * 4u, 2);
                        memcpy(&zb, par + ((uint64_t)h * ng + (uint64_t)gi) * 4u + 2, 2);
                        double s = orc_f16_to_f64(sb), z = orc_f16_to_f64(zb);
                        for (int i = 0; i < 32; i++) row[32 * gi + i] = orc_f64_to_bf16((double)q[i] * s + z);
                    }
                }
            }
        }
    }
    return 0;
}

/* Receiver injection at other positions.  A CacheCard carries the position
 * of its first token in the sender's sequence ([QKVShare] "CacheCard
 * representation": sequence length, model id, position offset), and a
 * shared segment's keys are moved to the receiving agent's positions before
 * reuse ([KVCMAS] "How it is used": the source cache's key positions are
 * re-aligned to the target's).  With rotary position embedding -- dims i and
 * i + d/2 form a pair turned through the angle p * w_i at position p, as the
 * Hugging Face Llama implementation pairs them -- a key turned for position
 * p0 + t becomes the key for p1 + t by one further turn through
 * (p1 - p0) * w_i, because plane rotations add their angles.
 *
 * K of every layer, head and token is dequantized exactly (16-bit tokens:
 * their bf16 value), turned in fp64 and rounded to bf16 once; V is decoded
 * exactly as orc_card_unpack does.  w: d/2 frequencies in radians per
 * position.  Returns 0, or -1 on a bad header. */
int orc_card_unpack_at(const uint8_t *card, int64_t pos_dst, const float *w, uint16_t *const *k_out,
                       uint16_t *const *v_out)
{
    if (get32(card) != 0x4343564Bu || get32(card + 4) != 1u) return -1;
    int T = (int)get32(card + 8), L = (int)get32(card + 12);
    int H = (int)get32(card + 16), d = (int)get32(card + 20);
    int64_t pos_src = (int64_t)get64(card + 40);
    uint64_t off_bits = get64(card + 48), off_offsets = get64(card + 56);
    uint64_t off_layers = get64(card + 64), stride = get64(card + 72);
    const int ng = d / 32, half = d / 2;
    double cs[64], sn[64];
    const double delta = (double)(pos_dst - pos_src);
    for (int i = 0; i < half; i++) {
        double phi = delta * (double)w[i];
        cs[i] = cos(phi);
        sn[i] = sin(phi);
    }
    for (int l = 0; l < L; l++) {
        const uint8_t *lay = card + off_layers + (uint64_t)l * stride;
#pragma omp parallel for schedule(static)
        for (int t = 0; t < T; t++) {
            int b = card[off_bits + (uint64_t)t];
            const uint8_t *rec = lay + get32(card + off_offsets + 4ull * (uint64_t)t);
            for (int kv = 0; kv < 2; kv++) {
                uint16_t *dst = kv ? v_out[l] : k_out[l];
                for (int h = 0; h < H; h++) {
                    double x[128];
                    if (b == 16) {
                        const uint8_t *src = rec + (uint64_t)kv * (uint64_t)H * (uint64_t)d * 2u + (uint64_t)h * d * 2u;
                        for (int i = 0; i < d; i++) {
                            uint16_t u;
                            memcpy(&u, src + 2 * i, 2);
                            x[i] = orc_bf16_to_f64(u);
                        }
                    } else {
                        uint64_t code_bytes = (uint64_t)H * (uint64_t)d * (uint64_t)b / 8u;
                        const uint8_t *codes = rec + (uint64_t)kv * code_bytes;
                        const uint8_t *par = rec + 2u * code_bytes + (uint64_t)kv * (uint64_t)H * (uint64_t)ng * 4u;
                        for (int gi = 0; gi < ng; gi++) {
                            uint8_t q[32];
                            uint16_t sb, zb;
                            unpack_group(codes + ((uint64_t)h * ng + (uint64_t)gi) * 4u * (uint64_t)b, b, q);
                            memcpy(&sb, par + ((uint64_t)h * ng + (uint64_t)gi) * 4u, 2);
                            memcpy(&zb, par + ((uint64_t)h * ng + (uint64_t)gi) * 4u + 2, 2);
                            double sc = orc_f16_to_f64(sb), z = orc_f16_to_f64(zb);
                            for (int i = 0; i < 32; i++) x[32 * gi + i] = (double)q[i] * sc + z;
                        }
                    }
                    uint16_t *row = dst + ((uint64_t)h * T + (uint64_t)t) * d;
                    if (kv == 0) {
                        for (int i = 0; i < half; i++) {
                            double a = x[i], c = x[i + half];
                            row[i] = orc_f64_to_bf16(a * cs[i] - c * sn[i]);
                            row[i + half] = orc_f64_to_bf16(a * sn[i] + c * cs[i]);
                        }
                    } else {
                        for (int i = 0; i < d; i++) row[i] = orc_f64_to_bf16(x[i]);
                    }
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Attention over the pool without materialising the caches.                  */
/* [QKVShare] "Significance": a fully fused attention kernel over the          */
/* quantized cache, deferred by the page; [PolyKV] 2.A: agents read the one    */
/* shared pool.                                                                */
/* ------------------------------------------------------------------------- */

/* Keys and values of every KV head of one pool layer, dequantized exactly:
 * k = q * s_l (format 1: q * s_b of the key's 32-key block) and
 * v = sigma_h * (H_d c) / sqrt(d), as fp64 [H][T][d] arrays (caller frees). */
static void attend_dequant(const uint8_t *pool, orc_pool_geom g, int layer, int H, int d, int T, int k_mode,
                           double **kf_out, double **vf_out)
{
    const uint8_t *lay = pool + g.off_layers + (uint64_t)layer * g.layer_stride;
    const uint8_t *ks = pool + g.off_kscales + (uint64_t)layer * (uint64_t)H * T * (uint64_t)(d / 32) * 2u;
    float s;
    memcpy(&s, pool + g.off_scales + 4u * (uint64_t)layer, 4);
    const int8_t *kc = (const int8_t *)lay;
    const uint8_t *vc = lay + g.sec_v;
    const uint8_t *sg = lay + g.sec_sigma;
    double *kf = (double *)malloc(sizeof(double) * (size_t)H * T * d);
    double *vf = (double *)malloc(sizeof(double) * (size_t)H * T * d);
    for (int64_t n = 0; n < (int64_t)H * T; n++) {
        uint8_t codes[128];
        uint16_t sh;
        double z[128];
        for (int i = 0; i < d; i++) {
            double sk = (double)s;
            if (k_mode == 1) {
                uint16_t sb;
                memcpy(&sb, ks + 2u * ((uint64_t)n * (uint64_t)(d / 32) + (uint64_t)(i / 32)), 2);
                sk = orc_f16_to_f64(sb);
            }
            kf[n * d + i] = (double)kc[n * d + i] * sk;
        }
        orc_unpack3(vc + (uint64_t)n * (uint64_t)(3 * d / 8), d, codes);
        memcpy(&sh, sg + 2u * (uint64_t)n, 2);
        for (int i = 0; i < d; i++) z[i] = CENTROID[codes[i]];
        orc_fwht(z, d);
        double sig = orc_f16_to_f64(sh);
        for (int i = 0; i < d; i++) vf[n * d + i] = sig * z[i] / sqrt((double)d);
    }
    *kf_out = kf;
    *vf_out = vf;
}

/* One decode step of attention for n_agents agents against layer `layer` of
 * the pool: for agent a and query head j (GQA: query head j reads KV head
 * j / (n_q_heads / H)),
 *   s_t   = scale * (q . k_t),        k_t = q_t * s_l  (q8_0 pools: q_t * s_b
 *                                     per 32-element block; exact, fp64)
 *   p_t   = exp(s_t - max s) / sum,   v_t = sigma_h * (H_d c_t) / sqrt(d)
 *   out   = sum_t p_t v_t,            lse = log(sum_t exp(s_t))
 * over the T pooled tokens.  q: bf16 [n_agents][n_q_heads][d]; out:
 * [n_agents][n_q_heads][d]; lse: [n_agents][n_q_heads].  Keys and values are
 * dequantized exactly (no bf16 rounding).  Returns 0, or -1 on a bad header
 * or head count. */
int orc_pool_attend(const uint8_t *pool, int layer, int n_agents, int n_q_heads, const uint16_t *q,
                    double scale, double *out, double *lse)
{
    if (get32(pool) != 0x4C50564Bu || get32(pool + 4) != 1u) return -1;
    int L = (int)get32(pool + 8), H = (int)get32(pool + 12);
    int d = (int)get32(pool + 16), T = (int)get32(pool + 20);
    if (layer < 0 || layer >= L || n_q_heads % H != 0) return -1;
    const int k_mode = (int)get32(pool + 28);
    if (k_mode != 0 && k_mode != 1) return -1;
    orc_pool_geom g = pool_geom(L, H, d, T);
    const int grp = n_q_heads / H;
    /* dequantized keys and values of every KV head, exact */
    double *kf, *vf;
    attend_dequant(pool, g, layer, H, d, T, k_mode, &kf, &vf);
#pragma omp parallel for schedule(static)
    for (int aj = 0; aj < n_agents * n_q_heads; aj++) {
        const int j = aj % n_q_heads;
        const int h = j / grp;
        const uint16_t *qv = q + (uint64_t)aj * d;
        double *sc = (double *)malloc(sizeof(double) * (size_t)T);
        double mx = -INFINITY;
        for (int t = 0; t < T; t++) {
            const double *kt = kf + ((uint64_t)h * T + t) * d;
            double dot = 0.0;
            for (int i = 0; i < d; i++) dot += orc_bf16_to_f64(qv[i]) * kt[i];
            sc[t] = scale * dot;
            if (sc[t] > mx) mx = sc[t];
        }
        double sum = 0.0;
        for (int t = 0; t < T; t++) { sc[t] = exp(sc[t] - mx); sum += sc[t]; }
        double *o = out + (uint64_t)aj * d;
        for (int i = 0; i < d; i++) o[i] = 0.0;
        for (int t = 0; t < T; t++) {
            const double *vt = vf + ((uint64_t)h * T + t) * d;
            const double p = sc[t] / sum;
            for (int i = 0; i < d; i++) o[i] += p * vt[i];
        }
        lse[aj] = mx + log(sum);
        free(sc);
    }
    free(kf);
    free(vf);
    return 0;
}

/* Attention over the pool with a shared low-rank value cache, "LRAgent"
 * (2. Sharing Schemes, BaseLRShared; 3. Flash-LoRA-Attention): every agent's
 * values are the shared base values plus its own LoRA term,
 *   v_{a,h,t} = vbase_{h,t} + sum_k vlr_{t,k} * B_a[k][h*d + i],
 * with vbase the pool's decoded values (exact dequantization), vlr the
 * layer's shared low-rank cache (X A, bf16 [T][rank]) and B_a agent a's
 * up-projection (bf16 [rank][H*d]).  This is the definition written out:
 * each agent's values are formed first and attended over as in
 * orc_pool_attend (the kernel's reordering P vbase + (P vlr) B is what it
 * is checked against).  Returns 0, or -1 on a bad header or head count. */
int orc_pool_attend_lora(const uint8_t *pool, int layer, int n_agents, int n_q_heads, const uint16_t *q,
                         double scale, int rank, const uint16_t *vlr, const uint16_t *lora_b, double *out,
                         double *lse)
{
    if (get32(pool) != 0x4C50564Bu || get32(pool + 4) != 1u) return -1;
    int H = (int)get32(pool + 12), d = (int)get32(pool + 16), T = (int)get32(pool + 20);
    if (n_q_heads % H != 0 || rank < 1) return -1;
    const int grp = n_q_heads / H;
    int L = (int)get32(pool + 8);
    if (layer < 0 || layer >= L) return -1;
    const int k_mode = (int)get32(pool + 28);
    if (k_mode != 0 && k_mode != 1) return -1;
    orc_pool_geom g = pool_geom(L, H, d, T);
    double *kf, *vb;  /* keys and base values, dequantized exactly */
    attend_dequant(pool, g, layer, H, d, T, k_mode, &kf, &vb);
#pragma omp parallel for schedule(static)
    for (int aj = 0; aj < n_agents * n_q_heads; aj++) {
        const int a = aj / n_q_heads, j = aj % n_q_heads;
        const int h = j / grp;
        const uint16_t *qv = q + (uint64_t)aj * d;
        const uint16_t *ba = lora_b + (uint64_t)a * (uint64_t)rank * (uint64_t)H * d;
        double *sc = (double *)malloc(sizeof(double) * (size_t)T);
        double *vt = (double *)malloc(sizeof(double) * (size_t)d);
        double mx = -INFINITY;
        for (int t = 0; t < T; t++) {
            const double *kt = kf + ((uint64_t)h * T + t) * d;
            double dot = 0.0;
            for (int i = 0; i < d; i++) dot += orc_bf16_to_f64(qv[i]) * kt[i];
            sc[t] = scale * dot;
            if (sc[t] > mx) mx = sc[t];
        }
        double sum = 0.0;
        for (int t = 0; t < T; t++) { sc[t] = exp(sc[t] - mx); sum += sc[t]; }
        double *o = out + (uint64_t)aj * d;
        for (int i = 0; i < d; i++) o[i] = 0.0;
        for (int t = 0; t < T; t++) {
            /* agent a's value of token t at head h */
            for (int i = 0; i < d; i++) {
                double v = vb[((uint64_t)h * T + t) * d + i];
                for (int k = 0; k < rank; k++)
                    v += orc_bf16_to_f64(vlr[(uint64_t)t * rank + k]) *
                         orc_bf16_to_f64(ba[(uint64_t)k * H * d + (uint64_t)h * d + i]);
                vt[i] = v;
            }
            const double p = sc[t] / sum;
            for (int i = 0; i < d; i++) o[i] += p * vt[i];
        }
        lse[aj] = mx + log(sum);
        free(sc);
        free(vt);
    }
    free(kf);
    free(vb);
    return 0;
}
