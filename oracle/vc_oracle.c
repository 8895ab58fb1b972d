/*
 * vc_oracle.c -- plain, slow, obviously-correct CPU oracle for the VeriCache
 * draft-and-verify hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the test-suite, the smoke check and the benchmark's CPU
 * baseline leg load it.  It shares no code, header, table or constant with the
 * CUDA path.
 *
 * What it follows (pages: "VeriCache: Turning Lossy KV Cache into Lossless LLM
 * Inference", the neuraltrendhub paper page, section "What the paper found",
 * and the abstract on the same page and on pith.science):
 *   - drafting runs the target model on a compressed KV cache (quantized
 *     KIVI-style, or token-dropped); verification re-runs the drafted block on
 *     the full KV cache; greedy output equals full-KV greedy decoding.
 *   - KIVI (cited as source 4 on the podparley page, ref [42] on pith.science):
 *     K is quantized per channel, V per token, each group with its own scale and
 *     zero-point.  The pages give only the name; the exact rounding rule used
 *     here is the reading recorded in the design notes (directed-rounded fp16
 *     meta so that the dequantization error is at most half a step).
 *   - token dropping (H2O, source 3 on the podparley page; KVzip 4x on the paper
 *     page): keep the highest accumulated-score tokens plus a recent window.
 *
 * Every floating-point result below is computed in fp64 unless the rule itself
 * fixes a narrower precision (the quantizer's fp32/fp16 steps).
 * Build: gcc -O2 -ffp-contract=off -frounding-math -fopenmp -fPIC -shared.
 */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#pragma STDC FENV_ACCESS ON

enum { ORC_RN = 0, ORC_RD = 1, ORC_RU = 2 };

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 / bfloat16, written from the format definitions.        */
/* ------------------------------------------------------------------------ */

/* Exact value of a binary16 bit pattern (1 sign, 5 exponent, 10 fraction). */
double orc_f16_value(uint16_t h)
{
    int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Exact value of a bfloat16 bit pattern: the top half of a binary32. */
float orc_bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Encode a magnitude that is exactly representable in binary16 (or is the
 * overflow marker) into its bit pattern. */
static uint16_t f16_encode_mag(double m, int sign)
{
    uint16_t bits;
    if (isinf(m)) {
        bits = 0x7C00;
    } else if (m < ldexp(1.0, -14)) {
        bits = (uint16_t)(m / ldexp(1.0, -24));    /* 1024 here lands on 0x0400 */
    } else {
        int E;
        double f = frexp(m, &E);                   /* m = f * 2^E, f in [0.5,1) */
        int ebias = E - 1 + 15;
        int mant = (int)(f * 2048.0) - 1024;
        bits = (uint16_t)((ebias << 10) | mant);
    }
    return (uint16_t)(bits | (sign ? 0x8000 : 0));
}

/* Round a finite binary32 value to binary16 under the given IEEE rounding
 * direction (nearest-even, toward -inf, toward +inf). */
uint16_t orc_f32_to_f16(float x, int mode)
{
    int sign = signbit(x) ? 1 : 0;
    double a = fabs((double)x);
    if (a == 0.0)
        return (uint16_t)(sign ? 0x8000 : 0);
    double u;                                      /* spacing of binary16 at a */
    if (a < ldexp(1.0, -14)) {
        u = ldexp(1.0, -24);
    } else {
        int E;
        frexp(a, &E);                              /* 2^(E-1) <= a < 2^E */
        u = ldexp(1.0, E - 1 - 10);
    }
    double q = a / u;                              /* exact: power-of-two scale */
    double fl = floor(q), k;
    int away;                                      /* round magnitude up? */
    if (mode == ORC_RN) {
        double fr = q - fl;
        if (fr > 0.5) away = 1;
        else if (fr < 0.5) away = 0;
        else away = (fmod(fl, 2.0) != 0.0);        /* tie: to even */
    } else if (mode == ORC_RD) {
        away = sign ? (q != fl) : 0;
    } else {
        away = sign ? 0 : (q != fl);
    }
    k = away ? fl + 1.0 : fl;
    double m = k * u;
    if (m > 65504.0) {
        /* overflow: to infinity when rounding away from zero, else max finite */
        int to_inf = (mode == ORC_RN) || (mode == ORC_RU && !sign) || (mode == ORC_RD && sign);
        m = to_inf ? INFINITY : 65504.0;
    }
    return f16_encode_mag(m, sign);
}

/* binary32 subtraction and division under a directed rounding mode. */
static float f32_sub_dir(float a, float b, int dir)
{
    int old = fegetround();
    fesetround(dir);
    volatile float va = a, vb = b;
    volatile float r = va - vb;
    fesetround(old);
    return r;
}

static float f32_div_dir(float a, float b, int dir)
{
    int old = fegetround();
    fesetround(dir);
    volatile float va = a, vb = b;
    volatile float r = va / vb;
    fesetround(old);
    return r;
}

/* ------------------------------------------------------------------------ */
/* KIVI-style asymmetric group quantization (reading of the pages' "KIVI").  */
/* ------------------------------------------------------------------------ */

/* Quantize one group x[0..n) (elements x[i*stride]) to `bits`-bit codes.
 *   zero  z = fp16 round-down of the group minimum
 *   scale s = fp16 round-up of  (max - z) / (2^bits - 1), both fp32 steps
 *             rounded upward
 *   code    = clamp(round-half-even((x - z) / s), 0, 2^bits - 1), fp32 steps
 *             rounded to nearest; code = 0 when s == 0
 *   dequant x^ = code * s + z
 * Directed rounding makes z <= min and z + (2^bits-1) s >= max, so every
 * element lies inside the quantization grid and |x - x^| <= s/2 up to the
 * rounding of the fp32 quotient. */
void orc_quantize_group(const float *x, int n, long stride, int bits,
                        uint8_t *codes, long code_stride,
                        uint16_t *s_bits, uint16_t *z_bits)
{
    float mn = x[0], mx = x[0];
    for (int i = 1; i < n; i++) {
        float v = x[(long)i * stride];
        if (v < mn) mn = v;
        if (v > mx) mx = v;
    }
    int qmax = (1 << bits) - 1;
    uint16_t zb = orc_f32_to_f16(mn, ORC_RD);
    float z = (float)orc_f16_value(zb);
    float range = f32_sub_dir(mx, z, FE_UPWARD);
    float step = f32_div_dir(range, (float)qmax, FE_UPWARD);
    uint16_t sb = orc_f32_to_f16(step, ORC_RU);
    float s = (float)orc_f16_value(sb);
    for (int i = 0; i < n; i++) {
        int c = 0;
        if (s != 0.0f) {
            volatile float diff = x[(long)i * stride] - z;   /* nearest */
            volatile float qv = diff / s;                    /* nearest */
            float r = nearbyintf(qv);                        /* half-even */
            if (r < 0.0f) r = 0.0f;
            if (r > (float)qmax) r = (float)qmax;
            c = (int)r;
        }
        codes[(long)i * code_stride] = (uint8_t)c;
    }
    *s_bits = sb;
    *z_bits = zb;
}

/* Quantize a whole cache.  k, v: [B][H][L][d] fp32 (exact images of the
 * bf16/fp32 inputs).  The first nq = floor(max(L - R, 0) / G) * G tokens are
 * quantized; the rest stays full precision.
 * Outputs (logical, unpermuted):
 *   kcode [B][H][nq][d]        per-channel K codes over token groups of G
 *   kscale/kzero [B][H][nq/G][d]
 *   vcode [B][H][nq][d]        per-token V codes over channel groups of G
 *   vscale/vzero [B][H][nq][d/G]
 * Returns nq. */
long orc_kivi_quantize(const float *k, const float *v, int B, int H, int L, int d,
                       int bits, int G, int R,
                       uint8_t *kcode, uint16_t *kscale, uint16_t *kzero,
                       uint8_t *vcode, uint16_t *vscale, uint16_t *vzero)
{
    long nq = (L - R > 0) ? (long)((L - R) / G) * G : 0;
    long ng = nq / G;
    int ncg = d / G;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; b++)
        for (int h = 0; h < H; h++) {
            long bh = (long)b * H + h;
            const float *kb = k + bh * L * d;
            const float *vb = v + bh * L * d;
            /* K: per channel, groups of G consecutive tokens. */
            for (long g = 0; g < ng; g++)
                for (int c = 0; c < d; c++)
                    orc_quantize_group(kb + g * G * d + c, G, d, bits,
                                       kcode + (bh * nq + g * G) * d + c, d,
                                       kscale + (bh * ng + g) * d + c,
                                       kzero + (bh * ng + g) * d + c);
            /* V: per token, groups of G consecutive channels. */
            for (long t = 0; t < nq; t++)
                for (int gc = 0; gc < ncg; gc++)
                    orc_quantize_group(vb + t * d + gc * G, G, 1, bits,
                                       vcode + (bh * nq + t) * d + gc * G, 1,
                                       vscale + (bh * nq + t) * ncg + gc,
                                       vzero + (bh * nq + t) * ncg + gc);
        }
    return nq;
}

/* ------------------------------------------------------------------------ */
/* Packed group-record reader (the library's documented storage format).    */
/* ------------------------------------------------------------------------ */

/* One record per (sequence, kv head, token group of G=32):
 *   [K codes: G*d*bits/8][V codes: G*d*bits/8][K meta: 4d][V meta: 4d] bytes.
 * Code sections.  Lane l in [0,32) owns W = d*bits/32 little-endian 32-bit
 * words; word w of lane l sits at byte 16*(32*(w/4) + l) + 4*(w%4) (16-byte
 * chunks interleaved across lanes).  A lane holds d/2 code pairs; pair
 * (mt, ks, r) covers the two elements hh = 0, 1 of the m16n8k16 operand
 * fragment register r (PTX ISA fragment layout: row = lane/4 + 8*(r&1),
 * col = 2*(lane%4) + hh + 8*(r>>1)):
 *   K (A = codes, rows = tokens):  mt in {0,1}, ks in [0,d/16):
 *       token = 16 mt + lane/4 + 8 (r&1), channel = 16 ks + 2 (lane%4) + hh + 8 (r>>1);
 *       class kappa = 2 ks + (r>>1), member mu = 2 mt + (r&1)
 *   V (A = codes^T, rows = channels): mt in [0,d/16), ks in {0,1}:
 *       channel = 16 mt + lane/4 + 8 (r&1), token = 16 ks + 2 (lane%4) + hh + 8 (r>>1);
 *       class kappa = 2 mt + (r&1), member mu = 2 ks + (r>>1)
 * Pair (kappa, mu) sits in word `word`, slot `slot` (first element at bit
 * bits*slot, second at bit 16 + bits*slot):
 *   bits = 2 (h = W/2, q = W/4): kappa < 3h: e = kappa / h, i = kappa % h,
 *       word = 2 i + mu/2, slot = e + 5 (mu%2); else k2 = kappa - 3h:
 *       e = 3 + k2 / q, i = k2 % q, word = 4 i + mu, slot = e.
 *   bits = 4 (h = W/2): e = kappa / h, i = kappa % h, word = 2 i + mu/2,
 *       slot = e + 2 (mu%2).
 * K meta section.  For lane quad j in [0,4) and k-step ks in [0,d/16) the
 * 16 bytes at 16*(4 ks + j) hold, for rr = 0 then rr = 1, the fp16 zero-point
 * pair (z[c0], z[c0+1]) followed by the scale pair (s[c0], s[c0+1]),
 * c0 = 16 ks + 2 j + 8 rr (zero pair at +8 rr, scale pair at +8 rr + 4).
 * V meta section.  For lane quad j the library stores a sequence of fp16
 * pairs; pair n of quad j sits at byte 16*(4*(n/4) + j) + 4*(n%4) of the
 * scale region, and the matching zero-point pair at the same offset + 2d:
 *   n = (2 ks + rr)*(d/32) + gc, pair = (s[t0][gc], s[t0+1][gc]),
 *   t0 = 16 ks + 2 j + 8 rr.
 * This reader implements the map directly from that statement; it shares
 * nothing with the GPU writer. */
static void pair_pos(int bits, int d, int kappa, int mu, int *word, int *slot)
{
    int W = d * bits / 32;
    if (bits == 2) {
        int h = W / 2, q = W / 4;
        if (kappa < 3 * h) {
            int e = kappa / h, i = kappa % h;
            *word = 2 * i + mu / 2;
            *slot = e + 5 * (mu % 2);
        } else {
            int k2 = kappa - 3 * h;
            int e = 3 + k2 / q, i = k2 % q;
            *word = 4 * i + mu;
            *slot = e;
        }
    } else {
        int h = W / 2;
        int e = kappa / h, i = kappa % h;
        *word = 2 * i + mu / 2;
        *slot = e + 2 * (mu % 2);
    }
}

static uint32_t rd_u32(const uint8_t *p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

static int rec_code(const uint8_t *sec, int lane, int word, int slot, int hh, int bits)
{
    uint32_t w = rd_u32(sec + 16 * (32 * (word / 4) + lane) + 4 * (word % 4));
    int shift = bits * slot + (hh ? 16 : 0);
    return (int)((w >> shift) & ((1u << bits) - 1));
}

static uint16_t rd_u16(const uint8_t *p)
{
    return (uint16_t)(p[0] | (p[1] << 8));
}

static const uint8_t *meta_pair(const uint8_t *region, int j, int n)
{
    return region + 16 * (4 * (n / 4) + j) + 4 * (n % 4);
}

long orc_record_bytes(int bits, int d, int G)
{
    return (long)2 * G * d * bits / 8 + 4L * d + 4L * G * (d / G);
}

/* Unpack n_rec consecutive records (each one group of G=32 tokens) into the
 * logical arrays: kcode/vcode [n_rec][G][d] (token-major), kscale/kzero
 * [n_rec][d], vscale/vzero [n_rec][G][d/32]. */
int orc_unpack_records(const uint8_t *rec, long n_rec, int bits, int d, int G,
                       uint8_t *kcode, uint16_t *kscale, uint16_t *kzero,
                       uint8_t *vcode, uint16_t *vscale, uint16_t *vzero)
{
    if (G != 32 || (d != 64 && d != 128) || (bits != 2 && bits != 4))
        return -1;
    long rb = orc_record_bytes(bits, d, G);
    int KS = d / 16, ncg = d / 32;
    for (long g = 0; g < n_rec; g++) {
        const uint8_t *r0 = rec + g * rb;
        const uint8_t *kc = r0;
        const uint8_t *vc = r0 + (long)G * d * bits / 8;
        const uint8_t *km = vc + (long)G * d * bits / 8;
        const uint8_t *vm = km + 4L * d;
        for (int lane = 0; lane < 32; lane++) {
            int gid = lane / 4, tig = lane % 4;
            for (int r = 0; r < 4; r++)
                for (int hh = 0; hh < 2; hh++) {
                    int word, slot;
                    /* K */
                    for (int mt = 0; mt < 2; mt++)
                        for (int ks = 0; ks < KS; ks++) {
                            pair_pos(bits, d, 2 * ks + (r >> 1), 2 * mt + (r & 1), &word, &slot);
                            int t = 16 * mt + gid + 8 * (r & 1);
                            int c = 16 * ks + 2 * tig + hh + 8 * (r >> 1);
                            kcode[(g * G + t) * d + c] = (uint8_t)rec_code(kc, lane, word, slot, hh, bits);
                        }
                    /* V */
                    for (int mt = 0; mt < KS; mt++)
                        for (int ks = 0; ks < 2; ks++) {
                            pair_pos(bits, d, 2 * mt + (r & 1), 2 * ks + (r >> 1), &word, &slot);
                            int c = 16 * mt + gid + 8 * (r & 1);
                            int t = 16 * ks + 2 * tig + hh + 8 * (r >> 1);
                            vcode[(g * G + t) * d + c] = (uint8_t)rec_code(vc, lane, word, slot, hh, bits);
                        }
                }
        }
        for (int j = 0; j < 4; j++) {
            for (int ks = 0; ks < KS; ks++)
                for (int rr = 0; rr < 2; rr++) {
                    int c0 = 16 * ks + 2 * j + 8 * rr;
                    const uint8_t *zp = km + 16 * (4 * ks + j) + 8 * rr;
                    const uint8_t *sp = zp + 4;
                    kscale[g * d + c0] = rd_u16(sp);
                    kscale[g * d + c0 + 1] = rd_u16(sp + 2);
                    kzero[g * d + c0] = rd_u16(zp);
                    kzero[g * d + c0 + 1] = rd_u16(zp + 2);
                }
            for (int ks = 0; ks < 2; ks++)
                for (int rr = 0; rr < 2; rr++)
                    for (int gc = 0; gc < ncg; gc++) {
                        int t0 = 16 * ks + 2 * j + 8 * rr;
                        const uint8_t *sp = meta_pair(vm, j, (2 * ks + rr) * ncg + gc);
                        const uint8_t *zp = sp + 2 * d;
                        vscale[(g * G + t0) * ncg + gc] = rd_u16(sp);
                        vscale[(g * G + t0 + 1) * ncg + gc] = rd_u16(sp + 2);
                        vzero[(g * G + t0) * ncg + gc] = rd_u16(zp);
                        vzero[(g * G + t0 + 1) * ncg + gc] = rd_u16(zp + 2);
                    }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Attention, fp64, straight from the definition o = softmax(q k^T * scale) v */
/* ------------------------------------------------------------------------ */

/* One query row against keys K[0..n), values V[0..n) (row-major, d wide).
 * Max-subtracted softmax in fp64. */
static void attend_row(const double *q, int d, long n, double scale,
                       const double *K, const double *V, double *out, double *sbuf)
{
    if (n <= 0) {                     /* no keys: the empty sum, defined as 0 */
        for (int c = 0; c < d; c++) out[c] = 0.0;
        return;
    }
    double m = -INFINITY;
    for (long i = 0; i < n; i++) {
        double s = 0.0;
        for (int c = 0; c < d; c++)
            s += q[c] * K[i * d + c];
        s *= scale;
        sbuf[i] = s;
        if (s > m) m = s;
    }
    double l = 0.0;
    for (int c = 0; c < d; c++) out[c] = 0.0;
    for (long i = 0; i < n; i++) {
        double p = exp(sbuf[i] - m);
        l += p;
        for (int c = 0; c < d; c++)
            out[c] += p * V[i * d + c];
    }
    for (int c = 0; c < d; c++) out[c] /= l;
}

/* Single-query decode attention over the KIVI cache of one layer.
 * Query head qh reads kv head qh / (Hq/Hkv).  Tokens [0, nq) come from the
 * logical codes/meta (dequantized x^ = code*s + z in fp64); tokens [nq, len)
 * from the full-precision residual kres/vres [B][Hkv][len][d] (positions nq..).
 * q [B][Hq][d] (fp32 images), out [B][Hq][d] fp64. */
void orc_kivi_decode_attn(const float *q, int B, int Hq, int Hkv, int d, int G,
                          long nq, long len, double scale,
                          const uint8_t *kcode, const uint16_t *kscale, const uint16_t *kzero,
                          const uint8_t *vcode, const uint16_t *vscale, const uint16_t *vzero,
                          const float *kres, const float *vres, double *out)
{
    int grp = Hq / Hkv, ncg = d / G;
    long nres = len - nq, ng = nq / G;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; b++)
        for (int kh = 0; kh < Hkv; kh++) {
            long bh = (long)b * Hkv + kh;
            double *K = (double *)malloc(sizeof(double) * len * d);
            double *V = (double *)malloc(sizeof(double) * len * d);
            double *sb = (double *)malloc(sizeof(double) * len);
            double *qd = (double *)malloc(sizeof(double) * d);
            for (long t = 0; t < nq; t++) {
                long g = t / G;
                for (int c = 0; c < d; c++) {
                    K[t * d + c] = kcode[(bh * nq + t) * d + c] *
                                       orc_f16_value(kscale[(bh * ng + g) * d + c]) +
                                   orc_f16_value(kzero[(bh * ng + g) * d + c]);
                    V[t * d + c] = vcode[(bh * nq + t) * d + c] *
                                       orc_f16_value(vscale[(bh * nq + t) * ncg + c / G]) +
                                   orc_f16_value(vzero[(bh * nq + t) * ncg + c / G]);
                }
            }
            for (long t = 0; t < nres; t++)
                for (int c = 0; c < d; c++) {
                    K[(nq + t) * d + c] = kres[(bh * nres + t) * d + c];
                    V[(nq + t) * d + c] = vres[(bh * nres + t) * d + c];
                }
            for (int j = 0; j < grp; j++) {
                int qh = kh * grp + j;
                for (int c = 0; c < d; c++) qd[c] = q[((long)b * Hq + qh) * d + c];
                attend_row(qd, d, len, scale, K, V, out + ((long)b * Hq + qh) * d, sb);
            }
            free(K); free(V); free(sb); free(qd);
        }
}

/* Single-query decode attention over a plain cache k, v [B][Hkv][Ls][d]
 * (fp32 images), sequence b attends to its first len[b] tokens. */
void orc_dense_decode_attn(const float *q, const float *k, const float *v,
                           const int *len, int B, int Hq, int Hkv, int d, long Ls,
                           double scale, double *out)
{
    int grp = Hq / Hkv;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; b++)
        for (int qh = 0; qh < Hq; qh++) {
            long bh = (long)b * Hkv + qh / grp;
            long n = len[b];
            double *K = (double *)malloc(sizeof(double) * (n ? n : 1) * d);
            double *V = (double *)malloc(sizeof(double) * (n ? n : 1) * d);
            double *sb = (double *)malloc(sizeof(double) * (n ? n : 1));
            double qd[512];
            for (long i = 0; i < n * d; i++) {
                K[i] = k[bh * Ls * d + i];
                V[i] = v[bh * Ls * d + i];
            }
            for (int c = 0; c < d; c++) qd[c] = q[((long)b * Hq + qh) * d + c];
            attend_row(qd, d, n, scale, K, V, out + ((long)b * Hq + qh) * d, sb);
            free(K); free(V); free(sb);
        }
}

/* Causal block (verify) attention.  q [B][Dq][Hq][d]; k, v [B][Hkv][Ls][d];
 * query i of sequence b sits at position ctx[b] + i and attends keys
 * 0 .. ctx[b] + i inclusive.  out [B][Dq][Hq][d] fp64.
 * `units`/`n_units` optionally restrict the work to a list of (b*Hkv + kh)
 * units (NULL = all); rows of skipped units are left untouched. */
void orc_verify_attn(const float *q, const float *k, const float *v, const int *ctx,
                     int B, int Dq, int Hq, int Hkv, int d, long Ls, double scale,
                     const int *units, int n_units, double *out)
{
    int grp = Hq / Hkv;
    int nu = units ? n_units : B * Hkv;
#pragma omp parallel for schedule(dynamic)
    for (int ui = 0; ui < nu; ui++) {
        int u = units ? units[ui] : ui;
        int b = u / Hkv, kh = u % Hkv;
        long bh = (long)b * Hkv + kh;
        long nmax = (long)ctx[b] + Dq;
        double *K = (double *)malloc(sizeof(double) * nmax * d);
        double *V = (double *)malloc(sizeof(double) * nmax * d);
        double *sb = (double *)malloc(sizeof(double) * nmax);
        double qd[512];
        for (long i = 0; i < nmax * d; i++) {
            K[i] = k[bh * Ls * d + i];
            V[i] = v[bh * Ls * d + i];
        }
        for (int i = 0; i < Dq; i++)
            for (int j = 0; j < grp; j++) {
                int qh = kh * grp + j;
                long row = (((long)b * Dq + i) * Hq + qh) * d;
                for (int c = 0; c < d; c++) qd[c] = q[row + c];
                attend_row(qd, d, (long)ctx[b] + i + 1, scale, K, V, out + row, sb);
            }
        free(K); free(V); free(sb);
    }
}

/* ------------------------------------------------------------------------ */
/* Greedy acceptance (speculative decoding's greedy rule, source 2 on the    */
/* podparley page): longest prefix whose verify argmax equals the drafts.    */
/* ------------------------------------------------------------------------ */

/* argmax with the lowest index winning ties; -0 and +0 compare equal. */
static long argmax_row(const float *x, long n)
{
    long best = 0;
    for (long i = 1; i < n; i++)
        if (x[i] > x[best]) best = i;
    return best;
}

/* logits [B][D+1][V] (fp32 images), drafts [B][D].
 * n_acc[b] = first i in [0,D) with argmax(row i) != drafts[b][i], else D.
 * next[b]  = argmax(row n_acc[b]).  Returns -1 on a non-finite logit. */
int orc_accept(const float *logits, const int *drafts, int B, int D, long V,
               int *n_acc, int *next, int *row_argmax)
{
    for (long i = 0; i < (long)B * (D + 1) * V; i++)
        if (!isfinite(logits[i])) return -1;
    for (int b = 0; b < B; b++) {
        int n = D;
        for (int i = 0; i <= D; i++) {
            long a = argmax_row(logits + ((long)b * (D + 1) + i) * V, V);
            if (row_argmax) row_argmax[b * (D + 1) + i] = (int)a;
        }
        for (int i = 0; i < D; i++) {
            long a = argmax_row(logits + ((long)b * (D + 1) + i) * V, V);
            if (a != drafts[b * D + i]) { n = i; break; }
        }
        n_acc[b] = n;
        next[b] = (int)argmax_row(logits + ((long)b * (D + 1) + n) * V, V);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Token dropping by accumulated score (H2O / KVzip-like).                  */
/* ------------------------------------------------------------------------ */

static const float *g_sort_scores;
static int cmp_score_desc_pos_asc(const void *a, const void *b)
{
    int i = *(const int *)a, j = *(const int *)b;
    float si = g_sort_scores[i], sj = g_sort_scores[j];
    if (si > sj) return -1;
    if (si < sj) return 1;
    return (i > j) - (i < j);
}
static int cmp_int_asc(const void *a, const void *b)
{
    int i = *(const int *)a, j = *(const int *)b;
    return (i > j) - (i < j);
}

/* scores [B][H][L].  Per (b,h): keep the recent window [L-R, L) and the top
 * keep_top positions of [0, L-R) ranked by (score descending, position
 * ascending); write them ascending to kept [B][H][n_keep] where
 * n_keep = min(keep_top, max(L-R,0)) + min(R, L).  Returns n_keep.
 * (Single-threaded: the comparator reads a file-scope pointer.) */
long orc_drop_select(const float *scores, int B, int H, long L, long keep_top,
                     long keep_recent, int *kept)
{
    long R = keep_recent < L ? keep_recent : L;
    long cand = L - R;
    long k = keep_top < cand ? keep_top : cand;
    long n_keep = k + R;
    int *idx = (int *)malloc(sizeof(int) * (cand > 0 ? cand : 1));
    for (long bh = 0; bh < (long)B * H; bh++) {
        const float *s = scores + bh * L;
        for (long i = 0; i < cand; i++) idx[i] = (int)i;
        g_sort_scores = s;
        qsort(idx, (size_t)cand, sizeof(int), cmp_score_desc_pos_asc);
        int *out = kept + bh * n_keep;
        for (long i = 0; i < k; i++) out[i] = idx[i];
        qsort(out, (size_t)k, sizeof(int), cmp_int_asc);
        for (long i = 0; i < R; i++) out[k + i] = (int)(cand + i);
    }
    free(idx);
    return n_keep;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
