/*
 * rc_oracle.c -- the oracle for the write-time FP8 ring KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, fp64 restatement of
 * what the cache computes.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load it.  It shares no code, header,
 * table or constant generator with the CUDA library, and it includes nothing
 * from it.
 *
 * Sources (web pages about "Runway Characters: Serving a 57B Video Diffusion
 * Transformer for Real-Time Conversation", arXiv 2611.05642):
 *   - paperdot mirror of the arXiv abstract: a ring cache; keys take RoPE
 *     and FP8 quantisation a single time, when written; resetting the
 *     positions rotates the stored keys by the difference; each chunk's 240
 *     attention calls read 5,788 slots, 757 of them new.
 *   - cpdf.ai blog, section "Como rodar 57B em tempo real com batch size 1":
 *     rotary positions and FP8 quantisation are applied when a frame enters
 *     the cache, and the cache is a ring so the window advances without
 *     copies.
 *   - cpdf.ai blog, section "Blackwell, escalabilidade e limites do
 *     decodificador": the FP8 attention uses per-head scales.
 * Where the pages are silent, the readings used here are:
 *   - E4M3 is the OCP 8-bit float (bias 7, max 448, no infinities, NaN =
 *     S.1111.111, subnormal step 2^-9); encoding rounds to nearest even and
 *     saturates to +-448.
 *   - One fp32 scale per (layer, head, write call), separately for K and V:
 *     s = fl32(amax / 448); s = 1 when amax = 0.  A code is enc(fl32(x / s)):
 *     the quotient is rounded once to fp32 and that fp32 value is encoded,
 *     so the integer decision is taken in the kernel's precision (fp32); the
 *     pages fix no precision for it.
 *   - RoPE uses interleaved pairs (2i, 2i+1), theta_i = base^(-2i/d), the
 *     pair (a, b) at angle phi becomes (a cos phi - b sin phi,
 *     a sin phi + b cos phi).  Keys are rotated before quantisation; values
 *     are not rotated.
 *   - slot(p) = floormod(p - delta_total, C).
 *   - Delta rotation dequantises each write group, rotates it by delta,
 *     recomputes the group's amax and scale, and requantises.
 *   - Attention: the layer's last-write queries, rotated at their (shifted)
 *     positions, attend to every occupied slot with no mask; scale 1/sqrt(d).
 *
 * Everything here is fp64 except the stored fp32 scales and the 8-bit codes,
 * which are part of the state the method defines.  Every floating-point
 * operation is done in the order written, with no blocking or fusion.
 *
 * The end of the file holds a second state machine, the same ring with bf16
 * storage (the non-FP8 cache of the pages' comparison), prefixed orc_b_.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_EMPTY INT64_MIN

/* ---------------------------------------------------------------- E4M3 */

/* Decode one OCP E4M3 code. */
double orc_e4m3_decode(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);          /* subnormal: m * 2^-9 */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);   /* normal: 1.m * 2^(e-7) */
    return sign ? -v : v;
}

/* Encode x as OCP E4M3: round to nearest, ties to even; saturate to +-448. */
uint8_t orc_e4m3_encode(double x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0)
        return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; q == 8 is the smallest normal */
        double q = rint(ldexp(a, 9));
        return sign | (uint8_t)q;
    }
    int e;
    frexp(a, &e);
    e -= 1;                                  /* a = f * 2^e, f in [1, 2) */
    double q = rint(ldexp(a, 3 - e));        /* 8 .. 16: 1.mmm in units of 1/8 */
    if (q == 16.0) {
        q = 8.0;
        e += 1;
    }
    return sign | (uint8_t)(((e + 7) << 3) | ((int)q - 8));
}

/* ---------------------------------------------------------------- bf16 */

double orc_bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------------------- RoPE */

double orc_rope_theta(int i, int d, double base)
{
    return pow(base, -2.0 * (double)i / (double)d);
}

/* Rotate one d-vector in place by position p (angle p * theta_i per pair). */
void orc_rope_rotate(double *x, int d, int64_t p, double base)
{
    for (int i = 0; i < d / 2; ++i) {
        double ang = (double)p * orc_rope_theta(i, d, base);
        double c = cos(ang), s = sin(ang);
        double a = x[2 * i], b = x[2 * i + 1];
        x[2 * i] = a * c - b * s;
        x[2 * i + 1] = a * s + b * c;
    }
}

/* Rotate n rows of d values; row t by pos[t]. */
void orc_rope_rows(double *x, int n, int d, const int64_t *pos, double base)
{
    for (int t = 0; t < n; ++t)
        orc_rope_rotate(x + (size_t)t * d, d, pos[t], base);
}

/* ---------------------------------------------------------------- scale */

/* Scale of a group with absolute maximum amax: fl32(amax / 448), or 1. */
float orc_scale_from_amax(double amax)
{
    if (amax == 0.0)
        return 1.0f;
    return (float)(amax / 448.0);
}

/* ---------------------------------------------------------------- attention */

/*
 * Softmax attention of n query rows (already rotated, fp64, [n][d]) over the
 * m key/value rows khat, vhat ([m][d], fp64).  out is [n][d].
 * scores s_j = q . k_j / sqrt(d); weights exp(s_j - max s); out = sum w v / sum w.
 */
void orc_attention_rows(const double *q, int n, const double *khat,
                        const double *vhat, int m, int d, double *out)
{
    double inv_sqrt_d = 1.0 / sqrt((double)d);
#pragma omp parallel for schedule(dynamic, 4)
    for (int r = 0; r < n; ++r) {
        double *s = (double *)malloc(sizeof(double) * (size_t)(m > 0 ? m : 1));
        const double *qr = q + (size_t)r * d;
        double mx = -INFINITY;
        for (int j = 0; j < m; ++j) {
            const double *kj = khat + (size_t)j * d;
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += qr[c] * kj[c];
            s[j] = acc * inv_sqrt_d;
            if (s[j] > mx)
                mx = s[j];
        }
        double l = 0.0;
        for (int j = 0; j < m; ++j) {
            s[j] = exp(s[j] - mx);
            l += s[j];
        }
        double *o = out + (size_t)r * d;
        for (int c = 0; c < d; ++c)
            o[c] = 0.0;
        for (int j = 0; j < m; ++j) {
            const double *vj = vhat + (size_t)j * d;
            for (int c = 0; c < d; ++c)
                o[c] += s[j] * vj[c];
        }
        for (int c = 0; c < d; ++c)
            o[c] /= l;
        free(s);
    }
}

/* ---------------------------------------------------------------- state */

typedef struct orc_cache {
    int L, H, d, C;
    double base;
    uint8_t *kc, *vc;      /* [L][H][C][d] E4M3 codes */
    float *sk, *sv;        /* [L][H][C] per-slot scale (the slot's write group scale) */
    int64_t *pos;          /* [L][C] position of the stored token, or ORC_EMPTY */
    int64_t *gid;          /* [L][C] serial number of the write that filled the slot */
    int64_t *last_pos;     /* [L][C] positions of the layer's last write */
    int *last_n;           /* [L] size of the layer's last write (0: none) */
    int64_t delta_total;
    int64_t next_gid;
} orc_cache;

#define IDX_CODE(c, l, h, s) ((((size_t)(l) * (c)->H + (h)) * (c)->C + (s)) * (c)->d)
#define IDX_SCALE(c, l, h, s) (((size_t)(l) * (c)->H + (h)) * (c)->C + (s))

orc_cache *orc_create(int L, int H, int d, int C, double base)
{
    if (L <= 0 || H <= 0 || d <= 0 || (d % 2) != 0 || C <= 0)
        return NULL;
    orc_cache *c = (orc_cache *)calloc(1, sizeof *c);
    c->L = L; c->H = H; c->d = d; c->C = C; c->base = base;
    size_t ncode = (size_t)L * H * C * d, nsc = (size_t)L * H * C;
    c->kc = (uint8_t *)calloc(ncode, 1);
    c->vc = (uint8_t *)calloc(ncode, 1);
    c->sk = (float *)calloc(nsc, sizeof(float));
    c->sv = (float *)calloc(nsc, sizeof(float));
    c->pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)L * C);
    c->gid = (int64_t *)malloc(sizeof(int64_t) * (size_t)L * C);
    c->last_pos = (int64_t *)calloc((size_t)L * C, sizeof(int64_t));
    c->last_n = (int *)calloc((size_t)L, sizeof(int));
    for (size_t i = 0; i < (size_t)L * C; ++i) {
        c->pos[i] = ORC_EMPTY;
        c->gid[i] = ORC_EMPTY;
    }
    return c;
}

void orc_destroy(orc_cache *c)
{
    if (!c) return;
    free(c->kc); free(c->vc); free(c->sk); free(c->sv);
    free(c->pos); free(c->gid); free(c->last_pos); free(c->last_n);
    free(c);
}

static int64_t floormod(int64_t a, int64_t m)
{
    int64_t r = a % m;
    return r < 0 ? r + m : r;
}

int64_t orc_slot_of(const orc_cache *c, int64_t p)
{
    return floormod(p - c->delta_total, c->C);
}

/*
 * Quantise a group of `rows` rows of d fp64 values (row-major) into codes with
 * one scale: returns the scale and writes codes[rows][d].
 */
static float quantise_group(const double *x, size_t rows, int d, uint8_t *codes)
{
    double amax = 0.0;
    for (size_t i = 0; i < rows * (size_t)d; ++i) {
        double a = fabs(x[i]);
        if (a > amax) amax = a;
    }
    float s = orc_scale_from_amax(amax);
    for (size_t i = 0; i < rows * (size_t)d; ++i) {
        float q = (float)(x[i] / (double)s);   /* the fp32 quotient */
        codes[i] = orc_e4m3_encode((double)q);
    }
    return s;
}

/*
 * The write proper, from fp64 rows: K, V [n][H][d] (values, not yet rotated);
 * positions[n].  Returns 0, or -1 on bad arguments (n out of range, layer out
 * of range, two tokens on one slot).
 */
static int write_rows(orc_cache *c, int l, const double *K, const double *V,
                      const int64_t *positions, int n)
{
    if (!c || l < 0 || l >= c->L || n <= 0 || n > c->C)
        return -1;
    int H = c->H, d = c->d;
    int64_t *slot = (int64_t *)malloc(sizeof(int64_t) * n);
    char *seen = (char *)calloc((size_t)c->C, 1);
    for (int t = 0; t < n; ++t) {
        slot[t] = orc_slot_of(c, positions[t]);
        if (seen[slot[t]]) {
            free(slot); free(seen);
            return -1;
        }
        seen[slot[t]] = 1;
    }
    free(seen);
    double *xk = (double *)malloc(sizeof(double) * (size_t)n * d);
    double *xv = (double *)malloc(sizeof(double) * (size_t)n * d);
    uint8_t *ck = (uint8_t *)malloc((size_t)n * d);
    uint8_t *cv = (uint8_t *)malloc((size_t)n * d);
    for (int h = 0; h < H; ++h) {
        for (int t = 0; t < n; ++t)
            for (int i = 0; i < d; ++i) {
                size_t src = ((size_t)t * H + h) * d + i;
                xk[(size_t)t * d + i] = K[src];
                xv[(size_t)t * d + i] = V[src];
            }
        orc_rope_rows(xk, n, d, positions, c->base);
        float sk = quantise_group(xk, (size_t)n, d, ck);
        float sv = quantise_group(xv, (size_t)n, d, cv);
        for (int t = 0; t < n; ++t) {
            memcpy(c->kc + IDX_CODE(c, l, h, slot[t]), ck + (size_t)t * d, d);
            memcpy(c->vc + IDX_CODE(c, l, h, slot[t]), cv + (size_t)t * d, d);
            c->sk[IDX_SCALE(c, l, h, slot[t])] = sk;
            c->sv[IDX_SCALE(c, l, h, slot[t])] = sv;
        }
    }
    for (int t = 0; t < n; ++t) {
        c->pos[(size_t)l * c->C + slot[t]] = positions[t];
        c->gid[(size_t)l * c->C + slot[t]] = c->next_gid;
        c->last_pos[(size_t)l * c->C + t] = positions[t];
    }
    c->last_n[l] = n;
    c->next_gid += 1;
    free(xk); free(xv); free(ck); free(cv); free(slot);
    return 0;
}

/*
 * Write n new tokens to layer l.  K, V are bf16 bit patterns [n][H][d];
 * positions[n].  Returns 0, or -1 on bad arguments.
 */
int orc_write(orc_cache *c, int l, const uint16_t *K, const uint16_t *V,
              const int64_t *positions, int n)
{
    if (!c || n <= 0 || n > c->C)
        return -1;
    size_t m = (size_t)n * c->H * c->d;
    double *k = (double *)malloc(sizeof(double) * m);
    double *v = (double *)malloc(sizeof(double) * m);
    for (size_t i = 0; i < m; ++i) {
        k[i] = orc_bf16_to_double(K[i]);
        v[i] = orc_bf16_to_double(V[i]);
    }
    int r = write_rows(c, l, k, v, positions, n);
    free(k); free(v);
    return r;
}

/*
 * The write fused into the K/V projection (the single-GPU half of the pages'
 * fused FP8 GEMM; paperdot abstract and cpdf.ai blog): X [n][hidden],
 * Wk and Wv [H*d][hidden] are E4M3 codes with one scale each, and
 *   K[t][h][i] = xs * wks * sum_k X[t][k] Wk[h*d + i][k]
 * (V alike with Wv, wvs) is the exact product of the decoded operands (a sum
 * of at most 2^13 products of two E4M3 values needs fewer than 53 bits, so
 * fp64 holds it exactly).  Those fp64 rows are then written as orc_write
 * writes its inputs: no bf16 rounding in between.
 */
int orc_write_proj(orc_cache *c, int l, const uint8_t *X, double xs, const uint8_t *Wk, double wks,
                   const uint8_t *Wv, double wvs, int hidden, const int64_t *positions, int n)
{
    if (!c || n <= 0 || n > c->C || hidden <= 0)
        return -1;
    int F = c->H * c->d;
    double *xd = (double *)malloc(sizeof(double) * (size_t)n * hidden);
    double *wk = (double *)malloc(sizeof(double) * (size_t)F * hidden);
    double *wv = (double *)malloc(sizeof(double) * (size_t)F * hidden);
    for (size_t i = 0; i < (size_t)n * hidden; ++i) xd[i] = orc_e4m3_decode(X[i]);
    for (size_t i = 0; i < (size_t)F * hidden; ++i) {
        wk[i] = orc_e4m3_decode(Wk[i]);
        wv[i] = orc_e4m3_decode(Wv[i]);
    }
    double *k = (double *)malloc(sizeof(double) * (size_t)n * F);
    double *v = (double *)malloc(sizeof(double) * (size_t)n * F);
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < n; ++t)
        for (int f = 0; f < F; ++f) {
            const double *xr = xd + (size_t)t * hidden;
            const double *kr = wk + (size_t)f * hidden, *vr = wv + (size_t)f * hidden;
            double sk = 0.0, sv = 0.0;
            for (int q = 0; q < hidden; ++q) {
                sk += xr[q] * kr[q];
                sv += xr[q] * vr[q];
            }
            k[(size_t)t * F + f] = sk * xs * wks;
            v[(size_t)t * F + f] = sv * xs * wvs;
        }
    int r = write_rows(c, l, k, v, positions, n);
    free(xd); free(wk); free(wv); free(k); free(v);
    return r;
}

/*
 * Delta rotation: every occupied slot of every layer holds a key rotated at
 * position p; afterwards it holds the key rotated at p + delta.  Each write
 * group is dequantised, rotated by delta, and requantised with a fresh scale.
 */
void orc_delta_rotate(orc_cache *c, int64_t delta)
{
    int C = c->C, d = c->d;
    int64_t *members = (int64_t *)malloc(sizeof(int64_t) * C);
    char *done = (char *)malloc((size_t)C);
    double *x = (double *)malloc(sizeof(double) * (size_t)C * d);
    uint8_t *codes = (uint8_t *)malloc((size_t)C * d);
    for (int l = 0; l < c->L; ++l) {
        memset(done, 0, (size_t)C);
        const int64_t *gid = c->gid + (size_t)l * C;
        for (int s0 = 0; s0 < C; ++s0) {
            if (done[s0] || c->pos[(size_t)l * C + s0] == ORC_EMPTY)
                continue;
            int64_t g = gid[s0];
            size_t m = 0;
            for (int s = s0; s < C; ++s)
                if (!done[s] && c->pos[(size_t)l * C + s] != ORC_EMPTY && gid[s] == g) {
                    members[m++] = s;
                    done[s] = 1;
                }
            for (int h = 0; h < c->H; ++h) {
                for (size_t j = 0; j < m; ++j) {
                    const uint8_t *src = c->kc + IDX_CODE(c, l, h, members[j]);
                    double sc = (double)c->sk[IDX_SCALE(c, l, h, members[j])];
                    for (int i = 0; i < d; ++i)
                        x[j * d + i] = orc_e4m3_decode(src[i]) * sc;
                    orc_rope_rotate(x + j * d, d, delta, c->base);
                }
                float s_new = quantise_group(x, m, d, codes);
                for (size_t j = 0; j < m; ++j) {
                    memcpy(c->kc + IDX_CODE(c, l, h, members[j]), codes + j * d, d);
                    c->sk[IDX_SCALE(c, l, h, members[j])] = s_new;
                }
            }
        }
        for (int s = 0; s < C; ++s)
            if (c->pos[(size_t)l * C + s] != ORC_EMPTY)
                c->pos[(size_t)l * C + s] += delta;
        for (int t = 0; t < c->last_n[l]; ++t)
            c->last_pos[(size_t)l * C + t] += delta;
    }
    c->delta_total += delta;
    free(members); free(done); free(x); free(codes);
}

/*
 * Attention over an explicit cache image of one layer: codes [H][C][d],
 * scales [H][C], pos [C] (ORC_EMPTY = free).  Q is bf16 bits [n][H][d],
 * rotated here at qpos[n].  out is fp64 [n][H][d].  Returns the number of
 * occupied slots, or -1 if there are none.
 */
int orc_attend_image(int H, int d, int C, double base,
                     const uint8_t *kc, const float *sk,
                     const uint8_t *vc, const float *sv,
                     const int64_t *pos, const uint16_t *Q,
                     const int64_t *qpos, int n, double *out)
{
    int m = 0;
    for (int s = 0; s < C; ++s)
        if (pos[s] != ORC_EMPTY) ++m;
    if (m == 0)
        return -1;
    double *khat = (double *)malloc(sizeof(double) * (size_t)m * d);
    double *vhat = (double *)malloc(sizeof(double) * (size_t)m * d);
    double *q = (double *)malloc(sizeof(double) * (size_t)n * d);
    double *o = (double *)malloc(sizeof(double) * (size_t)n * d);
    for (int h = 0; h < H; ++h) {
        int j = 0;
        for (int s = 0; s < C; ++s) {
            if (pos[s] == ORC_EMPTY) continue;
            size_t base_idx = ((size_t)h * C + s) * d;
            double ks = (double)sk[(size_t)h * C + s];
            double vs = (double)sv[(size_t)h * C + s];
            for (int i = 0; i < d; ++i) {
                khat[(size_t)j * d + i] = orc_e4m3_decode(kc[base_idx + i]) * ks;
                vhat[(size_t)j * d + i] = orc_e4m3_decode(vc[base_idx + i]) * vs;
            }
            ++j;
        }
        for (int t = 0; t < n; ++t)
            for (int i = 0; i < d; ++i)
                q[(size_t)t * d + i] = orc_bf16_to_double(Q[((size_t)t * H + h) * d + i]);
        orc_rope_rows(q, n, d, qpos, base);
        orc_attention_rows(q, n, khat, vhat, m, d, o);
        for (int t = 0; t < n; ++t)
            memcpy(out + ((size_t)t * H + h) * d, o + (size_t)t * d, sizeof(double) * d);
    }
    free(khat); free(vhat); free(q); free(o);
    return m;
}

/*
 * Attention call of layer l: the layer's last-write tokens (n of them) attend
 * with queries Q (bf16 bits [n][H][d]).  Returns 0, -1 on bad arguments,
 * -2 if n differs from the layer's last write or the layer is empty.
 */
int orc_attend(const orc_cache *c, int l, const uint16_t *Q, int n, double *out)
{
    if (!c || l < 0 || l >= c->L || n <= 0)
        return -1;
    if (c->last_n[l] == 0 || n != c->last_n[l])
        return -2;
    size_t off = (size_t)l * c->H * c->C;
    int m = orc_attend_image(c->H, c->d, c->C, c->base,
                             c->kc + off * c->d, c->sk + off,
                             c->vc + off * c->d, c->sv + off,
                             c->pos + (size_t)l * c->C, Q,
                             c->last_pos + (size_t)l * c->C, n, out);
    return m < 0 ? -2 : 0;
}

/* ---------------------------------------------------------------- state I/O */

/* Copy layer l's state out: codes [H][C][d], scales [H][C], pos/gid [C]. */
void orc_export(const orc_cache *c, int l, uint8_t *kc, float *sk, uint8_t *vc,
                float *sv, int64_t *pos, int64_t *gid)
{
    size_t off = (size_t)l * c->H * c->C;
    size_t nc = (size_t)c->H * c->C;
    if (kc) memcpy(kc, c->kc + off * c->d, nc * c->d);
    if (vc) memcpy(vc, c->vc + off * c->d, nc * c->d);
    if (sk) memcpy(sk, c->sk + off, nc * sizeof(float));
    if (sv) memcpy(sv, c->sv + off, nc * sizeof(float));
    if (pos) memcpy(pos, c->pos + (size_t)l * c->C, sizeof(int64_t) * c->C);
    if (gid) memcpy(gid, c->gid + (size_t)l * c->C, sizeof(int64_t) * c->C);
}

/* Replace layer l's state (used to run one oracle step from another state). */
void orc_import(orc_cache *c, int l, const uint8_t *kc, const float *sk,
                const uint8_t *vc, const float *sv, const int64_t *pos,
                const int64_t *gid, const int64_t *last_pos, int last_n)
{
    size_t off = (size_t)l * c->H * c->C;
    size_t nc = (size_t)c->H * c->C;
    memcpy(c->kc + off * c->d, kc, nc * c->d);
    memcpy(c->vc + off * c->d, vc, nc * c->d);
    memcpy(c->sk + off, sk, nc * sizeof(float));
    memcpy(c->sv + off, sv, nc * sizeof(float));
    memcpy(c->pos + (size_t)l * c->C, pos, sizeof(int64_t) * c->C);
    memcpy(c->gid + (size_t)l * c->C, gid, sizeof(int64_t) * c->C);
    if (last_n > 0)
        memcpy(c->last_pos + (size_t)l * c->C, last_pos, sizeof(int64_t) * last_n);
    c->last_n[l] = last_n;
}

void orc_set_counters(orc_cache *c, int64_t delta_total, int64_t next_gid)
{
    c->delta_total = delta_total;
    c->next_gid = next_gid;
}

int64_t orc_delta_total(const orc_cache *c) { return c->delta_total; }
int orc_last_n(const orc_cache *c, int l) { return c->last_n[l]; }
void orc_last_pos(const orc_cache *c, int l, int64_t *out)
{
    memcpy(out, c->last_pos + (size_t)l * c->C, sizeof(int64_t) * c->last_n[l]);
}

/*
 * Read-time quantisation of one layer (the original design the pages describe:
 * RoPE and FP8 quantisation of the whole cache in every call).  kraw, vraw are
 * the unrotated bf16 rows of every slot ([H][C][d] bits), pos[C] their
 * positions (ORC_EMPTY = free).  One scale per head for K and one for V over
 * all occupied slots; codes of free slots are 0 with scale 0.
 */
void orc_readtime_image(int H, int d, int C, double base, const uint16_t *kraw,
                        const uint16_t *vraw, const int64_t *pos,
                        uint8_t *kc, float *sk, uint8_t *vc, float *sv)
{
    double *xk = (double *)malloc(sizeof(double) * (size_t)C * d);
    double *xv = (double *)malloc(sizeof(double) * (size_t)C * d);
    int *occ = (int *)malloc(sizeof(int) * (size_t)C);
    for (int h = 0; h < H; ++h) {
        size_t m = 0;
        for (int s = 0; s < C; ++s) {
            if (pos[s] == ORC_EMPTY) continue;
            occ[m] = s;
            for (int i = 0; i < d; ++i) {
                size_t src = ((size_t)h * C + s) * d + i;
                xk[m * d + i] = orc_bf16_to_double(kraw[src]);
                xv[m * d + i] = orc_bf16_to_double(vraw[src]);
            }
            orc_rope_rotate(xk + m * d, d, pos[s], base);
            ++m;
        }
        uint8_t *ck = (uint8_t *)malloc(m * (size_t)d + 1);
        uint8_t *cv = (uint8_t *)malloc(m * (size_t)d + 1);
        float fk = quantise_group(xk, m, d, ck);
        float fv = quantise_group(xv, m, d, cv);
        memset(kc + (size_t)h * C * d, 0, (size_t)C * d);
        memset(vc + (size_t)h * C * d, 0, (size_t)C * d);
        for (int s = 0; s < C; ++s) {
            sk[(size_t)h * C + s] = 0.0f;
            sv[(size_t)h * C + s] = 0.0f;
        }
        for (size_t j = 0; j < m; ++j) {
            memcpy(kc + ((size_t)h * C + occ[j]) * d, ck + j * d, d);
            memcpy(vc + ((size_t)h * C + occ[j]) * d, cv + j * d, d);
            sk[(size_t)h * C + occ[j]] = fk;
            sv[(size_t)h * C + occ[j]] = fv;
        }
        free(ck); free(cv);
    }
    free(xk); free(xv); free(occ);
}

/* ================================================================ bf16 cache
 *
 * The same ring with bf16 storage instead of E4M3 codes and scales: the
 * non-FP8 cache that the pages compare the FP8 cache against (cpdf.ai blog,
 * section "Blackwell, escalabilidade e limites do decodificador").  A write
 * stores RoPE(K) rounded once from fp64 to bf16 (nearest, ties to even) and
 * V as given (already bf16); a delta rotation decodes each stored key,
 * rotates it by delta in fp64 and rounds it back to bf16; attention reads the
 * stored values.  The slot, position and write-serial bookkeeping is that of
 * the FP8 cache above.
 */

/* bf16 bits of x rounded to nearest, ties to even (8 significant bits; the
   bf16 subnormals below 2^-126 step by 2^-133).  Magnitudes that round to
   2^128 or more give infinity. */
uint16_t orc_bf16_encode(double x)
{
    if (x != x)
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);                      /* a = m 2^e, m in [0.5, 1) */
    int qe = e - 8;                    /* bf16 step in the binade [2^(e-1), 2^e) */
    if (qe < -133)
        qe = -133;                     /* subnormal range: fixed step 2^-133 */
    double q = ldexp(a, -qe);          /* exact: a / step */
    double r = nearbyint(q);           /* ties to even in the default mode */
    double v = ldexp(r, qe);
    if (v >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80);
    float f = (float)v;                /* exact: at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

typedef struct orc_bcache {
    int L, H, d, C;
    double base;
    uint16_t *kb, *vb;     /* [L][H][C][d] bf16 bits */
    int64_t *pos;          /* [L][C] position of the stored token, or ORC_EMPTY */
    int64_t *gid;          /* [L][C] serial number of the write that filled the slot */
    int64_t *last_pos;     /* [L][C] positions of the layer's last write */
    int *last_n;           /* [L] */
    int64_t delta_total;
    int64_t next_gid;
} orc_bcache;

orc_bcache *orc_b_create(int L, int H, int d, int C, double base)
{
    if (L <= 0 || H <= 0 || d <= 0 || (d % 2) != 0 || C <= 0)
        return NULL;
    orc_bcache *c = (orc_bcache *)calloc(1, sizeof *c);
    c->L = L; c->H = H; c->d = d; c->C = C; c->base = base;
    size_t nval = (size_t)L * H * C * d;
    c->kb = (uint16_t *)calloc(nval, sizeof(uint16_t));
    c->vb = (uint16_t *)calloc(nval, sizeof(uint16_t));
    c->pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)L * C);
    c->gid = (int64_t *)malloc(sizeof(int64_t) * (size_t)L * C);
    c->last_pos = (int64_t *)calloc((size_t)L * C, sizeof(int64_t));
    c->last_n = (int *)calloc((size_t)L, sizeof(int));
    for (size_t i = 0; i < (size_t)L * C; ++i) {
        c->pos[i] = ORC_EMPTY;
        c->gid[i] = ORC_EMPTY;
    }
    return c;
}

void orc_b_destroy(orc_bcache *c)
{
    if (!c) return;
    free(c->kb); free(c->vb); free(c->pos); free(c->gid); free(c->last_pos); free(c->last_n);
    free(c);
}

#define IDX_B(c, l, h, s) ((((size_t)(l) * (c)->H + (h)) * (c)->C + (s)) * (c)->d)

/* Write n tokens to layer l (K, V bf16 bits [n][H][d]).  Returns 0, or -1 on
   bad arguments (n or layer out of range, two tokens on one slot). */
int orc_b_write(orc_bcache *c, int l, const uint16_t *K, const uint16_t *V, const int64_t *positions, int n)
{
    if (!c || l < 0 || l >= c->L || n <= 0 || n > c->C)
        return -1;
    int H = c->H, d = c->d;
    int64_t *slot = (int64_t *)malloc(sizeof(int64_t) * n);
    char *seen = (char *)calloc((size_t)c->C, 1);
    for (int t = 0; t < n; ++t) {
        slot[t] = floormod(positions[t] - c->delta_total, c->C);
        if (seen[slot[t]]) {
            free(slot); free(seen);
            return -1;
        }
        seen[slot[t]] = 1;
    }
    free(seen);
    double *x = (double *)malloc(sizeof(double) * d);
    for (int t = 0; t < n; ++t)
        for (int h = 0; h < H; ++h) {
            size_t src = ((size_t)t * H + h) * d;
            for (int i = 0; i < d; ++i)
                x[i] = orc_bf16_to_double(K[src + i]);
            orc_rope_rotate(x, d, positions[t], c->base);
            uint16_t *kd = c->kb + IDX_B(c, l, h, slot[t]);
            for (int i = 0; i < d; ++i)
                kd[i] = orc_bf16_encode(x[i]);
            memcpy(c->vb + IDX_B(c, l, h, slot[t]), V + src, sizeof(uint16_t) * d);
        }
    for (int t = 0; t < n; ++t) {
        c->pos[(size_t)l * c->C + slot[t]] = positions[t];
        c->gid[(size_t)l * c->C + slot[t]] = c->next_gid;
        c->last_pos[(size_t)l * c->C + t] = positions[t];
    }
    c->last_n[l] = n;
    c->next_gid += 1;
    free(x); free(slot);
    return 0;
}

/* Every stored key of every layer: decode, rotate by delta (fp64), round to bf16. */
void orc_b_delta_rotate(orc_bcache *c, int64_t delta)
{
    int C = c->C, d = c->d;
    double *x = (double *)malloc(sizeof(double) * d);
    for (int l = 0; l < c->L; ++l) {
        for (int s = 0; s < C; ++s) {
            if (c->pos[(size_t)l * C + s] == ORC_EMPTY) continue;
            for (int h = 0; h < c->H; ++h) {
                uint16_t *kd = c->kb + IDX_B(c, l, h, s);
                for (int i = 0; i < d; ++i)
                    x[i] = orc_bf16_to_double(kd[i]);
                orc_rope_rotate(x, d, delta, c->base);
                for (int i = 0; i < d; ++i)
                    kd[i] = orc_bf16_encode(x[i]);
            }
            c->pos[(size_t)l * C + s] += delta;
        }
        for (int t = 0; t < c->last_n[l]; ++t)
            c->last_pos[(size_t)l * C + t] += delta;
    }
    c->delta_total += delta;
    free(x);
}

/* Attention of layer l's last-write queries Q (bf16 bits [n][H][d]) over the
   stored values; out fp64 [n][H][d].  Returns 0, -1 on bad arguments, -2 if
   n differs from the layer's last write or the layer is empty. */
int orc_b_attend(const orc_bcache *c, int l, const uint16_t *Q, int n, double *out)
{
    if (!c || l < 0 || l >= c->L || n <= 0)
        return -1;
    if (c->last_n[l] == 0 || n != c->last_n[l])
        return -2;
    int H = c->H, d = c->d, C = c->C, m = 0;
    for (int s = 0; s < C; ++s)
        if (c->pos[(size_t)l * C + s] != ORC_EMPTY) ++m;
    double *k = (double *)malloc(sizeof(double) * (size_t)m * d);
    double *v = (double *)malloc(sizeof(double) * (size_t)m * d);
    double *q = (double *)malloc(sizeof(double) * (size_t)n * d);
    double *o = (double *)malloc(sizeof(double) * (size_t)n * d);
    for (int h = 0; h < H; ++h) {
        int j = 0;
        for (int s = 0; s < C; ++s) {
            if (c->pos[(size_t)l * C + s] == ORC_EMPTY) continue;
            const uint16_t *kd = c->kb + IDX_B(c, l, h, s), *vd = c->vb + IDX_B(c, l, h, s);
            for (int i = 0; i < d; ++i) {
                k[(size_t)j * d + i] = orc_bf16_to_double(kd[i]);
                v[(size_t)j * d + i] = orc_bf16_to_double(vd[i]);
            }
            ++j;
        }
        for (int t = 0; t < n; ++t)
            for (int i = 0; i < d; ++i)
                q[(size_t)t * d + i] = orc_bf16_to_double(Q[((size_t)t * H + h) * d + i]);
        orc_rope_rows(q, n, d, c->last_pos + (size_t)l * C, c->base);
        orc_attention_rows(q, n, k, v, m, d, o);
        for (int t = 0; t < n; ++t)
            memcpy(out + ((size_t)t * H + h) * d, o + (size_t)t * d, sizeof(double) * d);
    }
    free(k); free(v); free(q); free(o);
    return 0;
}

/* Layer l's state: K, V bf16 bits [H][C][d], pos/gid [C]. */
void orc_b_export(const orc_bcache *c, int l, uint16_t *kb, uint16_t *vb, int64_t *pos, int64_t *gid)
{
    size_t nv = (size_t)c->H * c->C * c->d;
    if (kb) memcpy(kb, c->kb + IDX_B(c, l, 0, 0), nv * sizeof(uint16_t));
    if (vb) memcpy(vb, c->vb + IDX_B(c, l, 0, 0), nv * sizeof(uint16_t));
    if (pos) memcpy(pos, c->pos + (size_t)l * c->C, sizeof(int64_t) * c->C);
    if (gid) memcpy(gid, c->gid + (size_t)l * c->C, sizeof(int64_t) * c->C);
}

int orc_b_last_n(const orc_bcache *c, int l) { return c->last_n[l]; }
void orc_b_last_pos(const orc_bcache *c, int l, int64_t *out)
{
    memcpy(out, c->last_pos + (size_t)l * c->C, sizeof(int64_t) * c->last_n[l]);
}
