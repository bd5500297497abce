/*
 * fp64 CPU oracle for causal multi-head self-attention with parameter-free
 * QK RMSNorm and rotary position embeddings (RoPE).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code with
 * the CUDA path: it is the plain definition written out in double precision,
 * one loop per step, with no tiling, fusion or reordering.
 *
 * What it follows (the pages print no formula; the readings are the plainest
 * ones the pages support):
 *  - QK-norm: queries and keys are normalised (usually RMSNorm) before the dot
 *    product -- ai.flicky.cc, "nanochat: свой ChatGPT от токенизатора до чата",
 *    section "Модель: что изменилось со времён GPT-2" (QK-norm bullet) and
 *    adg.csdn.net "4小时100美元！...nanochat...", section "1. 极致精简的技术架构".
 *  - RMSNorm is x / sqrt(mean(x^2) + eps) * g and nanochat uses it without
 *    trainable parameters (g = 1) -- same ai.flicky.cc section, RMSNorm bullet.
 *    Read here per head vector over D.
 *  - Rotary embeddings replace positional embeddings -- same section, first
 *    bullet.  Read here as the original RoPE: theta_i = base^(-2i/D),
 *    i < D/2, pair (i, i + D/2) rotated by angle p * theta_i (the "rotate-half"
 *    pairing), norm first, then rotation.
 *  - Causal softmax(QK^T / sqrt(D)) V per head; the log-sum-exp is natural log.
 *  - Decode: generation with a KV cache (ai.flicky.cc, section
 *    "Карта репозитория", engine.py row; 7minutos.es "Andrej Karpathy lanza
 *    nanochat ...", section "Entrenamiento medio, SFT y uso de herramientas").
 *  - Grouped-query attention: fewer key/value heads than query heads is an
 *    option of the model (ai.flicky.cc, section "Модель: что изменилось со
 *    времён GPT-2", GQA bullet).  Read here as: with Hkv key/value heads,
 *    query head h uses key/value head h / (H / Hkv) (consecutive query heads
 *    share one); the key and value gradients sum over the group.
 *  - Sliding windows: most layers attend through a short window of a quarter
 *    of the context (ai.flicky.cc, section "Модель: что изменилось со времён
 *    GPT-2", window-pattern bullet).  Read here as: with window W > 0, query
 *    i sees key j exactly when 0 <= i - j < W (W keys, itself included);
 *    W <= 0 means the plain causal mask.
 *
 * Layout: q, k, v, o, dout, dq, dk, dv are [B, T, H, D] row-major; lse is
 * [B, H, T]; rms factors are [B, T, H].  pos is [T] (NULL means 0..T-1).
 * flags: bit 0 = apply RMSNorm, bit 1 = apply RoPE (both on for the method;
 * off only to reduce to plain causal attention in the tests).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORC_NORM 1
#define ORC_ROPE 2

/* Is key j visible from query i?  Causal, and inside the window when W > 0. */
static int visible(int i, int j, int W) { return j <= i && (W <= 0 || i - j < W); }

static size_t at4(int b, int t, int h, int d, int T, int H, int D)
{
    return (((size_t)b * T + t) * H + h) * D + d;
}

static int position(const int *pos, int t) { return pos ? pos[t] : t; }

/* RMS factor r = sqrt(mean_d(x_d^2) + eps) of one head vector. */
static double rms_of(const double *x, int D, double eps)
{
    double ss = 0.0;
    for (int d = 0; d < D; ++d) ss += x[d] * x[d];
    return sqrt(ss / D + eps);
}

/* RoPE angle of pair i at position p: p * base^(-2i/D). */
static double rope_angle(int p, int i, int D, double base)
{
    return (double)p * pow(base, -2.0 * i / D);
}

/* Rotate pair (i, i + D/2) of one head vector by +angle(p) (sign = +1) or
 * by -angle(p) (sign = -1, the transpose used in the backward). */
static void rotate(double *x, int p, int D, double base, int sign)
{
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
        double th = sign * rope_angle(p, i, D, base);
        double c = cos(th), s = sin(th);
        double a = x[i], b = x[i + half];
        x[i] = a * c - b * s;
        x[i + half] = a * s + b * c;
    }
}

/* Step 1 + 2: xhat = RoPE(x / r, pos), r per head vector.
 * xhat [B,T,H,D]; r [B,T,H] (may be NULL). */
void orc_norm_rope(const double *x, const int *pos, int B, int T, int H, int D,
                   double eps, double base, int flags, double *xhat, double *r)
{
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t)
            for (int h = 0; h < H; ++h) {
                const double *xi = x + at4(b, t, h, 0, T, H, D);
                double *yo = xhat + at4(b, t, h, 0, T, H, D);
                double rr = (flags & ORC_NORM) ? rms_of(xi, D, eps) : 1.0;
                for (int d = 0; d < D; ++d) yo[d] = xi[d] / rr;
                if (flags & ORC_ROPE) rotate(yo, position(pos, t), D, base, +1);
                if (r) r[((size_t)b * T + t) * H + h] = rr;
            }
}

static double dot(const double *a, const double *b, int n)
{
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

/* E4M3 rounding (the OCP 8-bit float with 4 exponent bits, bias 7 and 3
 * mantissa bits, "fn" variant: no infinities, largest finite value 448):
 * round to nearest, ties to even, with saturation to +-448.  Normal numbers
 * are (1 + m/8) 2^(e-7), e = 1..15; subnormals m/8 2^-6; so the spacing of
 * representable values is 2^(E-3) in the binade [2^E, 2^(E+1)), E >= -6, and
 * 2^-9 below 2^-6. */
double orc_e4m3(double x)
{
    if (x != x) return x;
    double a = fabs(x);
    if (a == 0.0) return x;
    int E;
    frexp(a, &E);          /* a = f 2^E with f in [0.5, 1): binade [2^(E-1), 2^E) */
    E -= 1;
    if (E < -6) E = -6;    /* subnormal spacing below 2^-6 */
    double quantum = ldexp(1.0, E - 3);
    double r = nearbyint(a / quantum) * quantum;  /* default rounding mode: ties to even */
    if (r > 448.0) r = 448.0;
    return x < 0 ? -r : r;
}

/* Step 3 for one (b, h): probabilities P[i][j] (zero where j is not
 * visible from i), outputs o and log-sum-exp.  P is T*T, row-major.
 * pquant (the fp8 reading only): each probability p = exp(s - max) is
 * replaced by E4M3(p 2^8) 2^-8 before it weights v, the output divides by
 * the sum of those quantised weights, and lse uses the sum of the exact p. */
static void attend_head_q(const double *qh, const double *kh, const double *v,
                          int b, int h, int T, int H, int Hkv, int D, int W, int pquant, double *P,
                          double *o, double *lse)
{
    int hk = h / (H / Hkv);  /* the key/value head of query head h */
    double scale = 1.0 / sqrt((double)D);
    for (int i = 0; i < T; ++i) {
        double *row = P + (size_t)i * T;
        const double *qi = qh + at4(b, i, h, 0, T, H, D);
        double m = -INFINITY;
        for (int j = 0; j < T; ++j) {
            if (!visible(i, j, W)) continue;
            row[j] = dot(qi, kh + at4(b, j, hk, 0, T, Hkv, D), D) * scale;
            if (row[j] > m) m = row[j];
        }
        double l = 0.0, lexact = 0.0;
        for (int j = 0; j < T; ++j) {
            if (!visible(i, j, W)) {
                row[j] = 0.0;
                continue;
            }
            row[j] = exp(row[j] - m);
            lexact += row[j];
            if (pquant) row[j] = orc_e4m3(row[j] * 256.0) / 256.0;
            l += row[j];
        }
        for (int j = 0; j < T; ++j) row[j] /= l;
        double *oi = o + at4(b, i, h, 0, T, H, D);
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int j = 0; j < T; ++j) acc += row[j] * v[at4(b, j, hk, d, T, Hkv, D)];
            oi[d] = acc;
        }
        if (lse) lse[((size_t)b * H + h) * T + i] = m + log(lexact);
    }
}

static void attend_head(const double *qh, const double *kh, const double *v,
                        int b, int h, int T, int H, int Hkv, int D, int W, double *P,
                        double *o, double *lse)
{
    attend_head_q(qh, kh, v, b, h, T, H, Hkv, D, W, 0, P, o, lse);
}

/* Forward: o = softmax(qhat khat^T / sqrt(D) + mask) v; lse [B,H,T].  The
 * mask is causal, banded to the last W keys when W > 0. */
int orc_attn_fwd(const double *q, const double *k, const double *v, const int *pos,
                 int B, int T, int H, int Hkv, int D, double eps, double base, int flags, int W,
                 double *o, double *lse)
{
    size_t n = (size_t)B * T * H * D, nk = (size_t)B * T * Hkv * D;
    double *qh = malloc(n * sizeof(double)), *kh = malloc(nk * sizeof(double));
    if (!qh || !kh) { free(qh); free(kh); return -1; }
    orc_norm_rope(q, pos, B, T, H, D, eps, base, flags, qh, NULL);
    orc_norm_rope(k, pos, B, T, Hkv, D, eps, base, flags, kh, NULL);
    int err = 0;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            double *P = malloc((size_t)T * T * sizeof(double));
            if (!P) { err = -1; continue; }
            attend_head(qh, kh, v, b, h, T, H, Hkv, D, W, P, o, lse);
            free(P);
        }
    free(qh);
    free(kh);
    return err;
}

/* FP8 forward (this library's reading of fp8 attention; the pages name an
 * fp8 training path and give no attention scheme).  With quant = 1:
 *   qhat8 = E4M3(qhat 2^5) 2^-5, khat8 likewise (QK-norm bounds every element
 *     by sqrt(D) <= 11.32, so 2^5 keeps them within E4M3's 448);
 *   v8 = E4M3(v 2^tau) 2^-tau per (batch, key/value head), tau the largest
 *     integer with max |v| 2^tau <= 448 (0 for an all-zero head);
 *   s = qhat8 . khat8 / sqrt(D); p = exp(s - max over the row's visible keys);
 *   P8 = E4M3(p 2^8) 2^-8; o = sum P8 v8 / sum P8; lse = max + ln sum p.
 * quant = 0 skips every rounding: the function is then orc_attn_fwd. */
int orc_attn_fwd_fp8(const double *q, const double *k, const double *v, const int *pos,
                     int B, int T, int H, int Hkv, int D, double eps, double base, int W, int quant,
                     double *o, double *lse)
{
    size_t n = (size_t)B * T * H * D, nk = (size_t)B * T * Hkv * D;
    double *qh = malloc(n * sizeof(double)), *kh = malloc(nk * sizeof(double));
    double *vq = malloc(nk * sizeof(double));
    if (!qh || !kh || !vq) { free(qh); free(kh); free(vq); return -1; }
    orc_norm_rope(q, pos, B, T, H, D, eps, base, ORC_NORM | ORC_ROPE, qh, NULL);
    orc_norm_rope(k, pos, B, T, Hkv, D, eps, base, ORC_NORM | ORC_ROPE, kh, NULL);
    memcpy(vq, v, nk * sizeof(double));
    if (quant) {
        for (size_t e = 0; e < n; ++e) qh[e] = orc_e4m3(qh[e] * 32.0) / 32.0;
        for (size_t e = 0; e < nk; ++e) kh[e] = orc_e4m3(kh[e] * 32.0) / 32.0;
        for (int b = 0; b < B; ++b)
            for (int g = 0; g < Hkv; ++g) {
                double mx = 0.0;
                for (int t = 0; t < T; ++t)
                    for (int d = 0; d < D; ++d) {
                        double a = fabs(v[at4(b, t, g, d, T, Hkv, D)]);
                        if (a > mx) mx = a;
                    }
                int tau = 0;
                if (mx > 0.0) {
                    tau = (int)floor(log2(448.0 / mx));
                    while (ldexp(mx, tau) > 448.0) --tau;  /* guard the log2 rounding */
                    while (ldexp(mx, tau + 1) <= 448.0) ++tau;
                }
                for (int t = 0; t < T; ++t)
                    for (int d = 0; d < D; ++d) {
                        size_t e = at4(b, t, g, d, T, Hkv, D);
                        vq[e] = ldexp(orc_e4m3(ldexp(v[e], tau)), -tau);
                    }
            }
    }
    int err = 0;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            double *P = malloc((size_t)T * T * sizeof(double));
            if (!P) { err = -1; continue; }
            attend_head_q(qh, kh, vq, b, h, T, H, Hkv, D, W, quant, P, o, lse);
            free(P);
        }
    free(qh);
    free(kh);
    free(vq);
    return err;
}

/* Backward of one head vector through RoPE and RMSNorm:
 * u = R(p)^T g, then dx = (u - y <u, y> / D) / r with y = x / r (the
 * normalised vector before rotation). */
static void norm_rope_backward(const double *x, const double *g, int p, int D,
                               double eps, double base, int flags, double *dx)
{
    double *u = malloc((size_t)D * sizeof(double));
    memcpy(u, g, (size_t)D * sizeof(double));
    if (flags & ORC_ROPE) rotate(u, p, D, base, -1);
    if (flags & ORC_NORM) {
        double r = rms_of(x, D, eps);
        double uy = 0.0;
        for (int d = 0; d < D; ++d) uy += u[d] * (x[d] / r);
        for (int d = 0; d < D; ++d) dx[d] = (u[d] - (x[d] / r) * uy / D) / r;
    } else {
        memcpy(dx, u, (size_t)D * sizeof(double));
    }
    free(u);
}

/* Step 4, by hand (no autograd), with P zero where j is not visible from i:
 *   dv_j  = sum_i P_ij do_i
 *   dP_ij = <do_i, v_j>,  Delta_i = <do_i, o_i>
 *   dS_ij = P_ij (dP_ij - Delta_i)
 *   dqhat_i = sum_j dS_ij khat_j / sqrt(D),  dkhat_j = sum_i dS_ij qhat_i / sqrt(D)
 * then back through RoPE and RMSNorm to dq, dk. */
int orc_attn_bwd(const double *q, const double *k, const double *v, const double *dout,
                 const int *pos, int B, int T, int H, int Hkv, int D, double eps, double base,
                 int flags, int W, double *dq, double *dk, double *dv)
{
    size_t n = (size_t)B * T * H * D, nk = (size_t)B * T * Hkv * D;
    int G = H / Hkv;
    double *qh = malloc(n * sizeof(double)), *kh = malloc(nk * sizeof(double));
    double *o = malloc(n * sizeof(double));
    double *dqh = calloc(n, sizeof(double)), *dkh = calloc(nk, sizeof(double));
    if (!qh || !kh || !o || !dqh || !dkh) {
        free(qh); free(kh); free(o); free(dqh); free(dkh);
        return -1;
    }
    orc_norm_rope(q, pos, B, T, H, D, eps, base, flags, qh, NULL);
    orc_norm_rope(k, pos, B, T, Hkv, D, eps, base, flags, kh, NULL);
    memset(dv, 0, nk * sizeof(double));
    double scale = 1.0 / sqrt((double)D);
    int err = 0;
    /* one key/value head per task; its group's query heads in turn, so the
     * sums over the group into dk and dv need no synchronisation */
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
        for (int hk = 0; hk < Hkv; ++hk) {
            double *P = malloc((size_t)T * T * sizeof(double));
            double *dS = malloc((size_t)T * T * sizeof(double));
            if (!P || !dS) { free(P); free(dS); err = -1; continue; }
            for (int h = hk * G; h < (hk + 1) * G; ++h) {
                attend_head(qh, kh, v, b, h, T, H, Hkv, D, W, P, o, NULL);
                for (int i = 0; i < T; ++i) {
                    const double *doi = dout + at4(b, i, h, 0, T, H, D);
                    double delta = dot(doi, o + at4(b, i, h, 0, T, H, D), D);
                    for (int j = 0; j < T; ++j) {
                        double pij = P[(size_t)i * T + j];
                        double dpij = visible(i, j, W) ? dot(doi, v + at4(b, j, hk, 0, T, Hkv, D), D) : 0.0;
                        dS[(size_t)i * T + j] = pij * (dpij - delta);
                    }
                }
                for (int j = 0; j < T; ++j)
                    for (int d = 0; d < D; ++d) {
                        double acc = 0.0;
                        for (int i = j; i < T; ++i)
                            acc += P[(size_t)i * T + j] * dout[at4(b, i, h, d, T, H, D)];
                        dv[at4(b, j, hk, d, T, Hkv, D)] += acc;
                    }
                for (int i = 0; i < T; ++i)
                    for (int d = 0; d < D; ++d) {
                        double acc = 0.0;
                        for (int j = 0; j <= i; ++j)
                            acc += dS[(size_t)i * T + j] * kh[at4(b, j, hk, d, T, Hkv, D)];
                        dqh[at4(b, i, h, d, T, H, D)] = acc * scale;
                    }
                for (int j = 0; j < T; ++j)
                    for (int d = 0; d < D; ++d) {
                        double acc = 0.0;
                        for (int i = j; i < T; ++i)
                            acc += dS[(size_t)i * T + j] * qh[at4(b, i, h, d, T, H, D)];
                        dkh[at4(b, j, hk, d, T, Hkv, D)] += acc * scale;
                    }
                for (int t = 0; t < T; ++t) {
                    size_t off = at4(b, t, h, 0, T, H, D);
                    norm_rope_backward(q + off, dqh + off, position(pos, t), D, eps, base, flags, dq + off);
                }
            }
            for (int t = 0; t < T; ++t) {
                size_t off = at4(b, t, hk, 0, T, Hkv, D);
                norm_rope_backward(k + off, dkh + off, position(pos, t), D, eps, base, flags, dk + off);
            }
            free(P);
            free(dS);
        }
    free(qh); free(kh); free(o); free(dqh); free(dkh);
    return err;
}

/* Step 5, decode: one new query per stream b at position p = lens[b] - 1,
 * attending over the cache slots j <= p visible from p (all of them, or the
 * last W when W > 0).  Keys are given RAW: slot j is
 * normalised and rotated at position j here, exactly as a prefill over the
 * same raw keys would have stored it; the new token's raw key sits at slot p.
 * q [B,H,D]; k_raw, v [B,Tcap,Hkv,D]; out [B,H,D]. */
int orc_attn_decode(const double *q, const double *k_raw, const double *v, const int *lens,
                    int B, int H, int Hkv, int D, int Tcap, double eps, double base, int flags, int W,
                    double *out)
{
    int G = H / Hkv;
    double scale = 1.0 / sqrt((double)D);
    int err = 0;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            int L = lens[b];
            if (L < 1 || L > Tcap) { err = -2; continue; }
            double *qh = malloc((size_t)D * sizeof(double));
            double *kh = malloc((size_t)D * sizeof(double));
            double *s = malloc((size_t)L * sizeof(double));
            const double *qi = q + ((size_t)b * H + h) * D;
            double rq = (flags & ORC_NORM) ? rms_of(qi, D, eps) : 1.0;
            for (int d = 0; d < D; ++d) qh[d] = qi[d] / rq;
            if (flags & ORC_ROPE) rotate(qh, L - 1, D, base, +1);
            double m = -INFINITY;
            for (int j = 0; j < L; ++j) {
                s[j] = -INFINITY;
                if (!visible(L - 1, j, W)) continue;
                const double *kj = k_raw + at4(b, j, h / G, 0, Tcap, Hkv, D);
                double rk = (flags & ORC_NORM) ? rms_of(kj, D, eps) : 1.0;
                for (int d = 0; d < D; ++d) kh[d] = kj[d] / rk;
                if (flags & ORC_ROPE) rotate(kh, j, D, base, +1);
                s[j] = dot(qh, kh, D) * scale;
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            for (int j = 0; j < L; ++j) {
                s[j] = exp(s[j] - m);  /* exp(-inf) = 0 for the slots outside the window */
                l += s[j];
            }
            double *oi = out + ((size_t)b * H + h) * D;
            for (int d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int j = 0; j < L; ++j) acc += s[j] / l * v[at4(b, j, h / G, d, Tcap, Hkv, D)];
                oi[d] = acc;
            }
            free(qh); free(kh); free(s);
        }
    return err;
}

/* Prefill of a chunk: C new tokens per stream b at positions start[b] ..
 * start[b] + C - 1, each attending (causally, inside the window when W > 0)
 * over the cache slots 0 .. its own position.  Keys are given RAW for every
 * slot up to start[b] + C - 1 (the chunk's own keys in its slots): slot j is
 * normalised and rotated at position j, as the cache holds it.  This is
 * rows start[b] .. start[b] + C - 1 of the forward over the whole sequence.
 * q, out [B,C,H,D]; k_raw, v [B,Tcap,Hkv,D] (query head h reads key/value
 * head h / (H / Hkv)); lse [B,H,C] (may be NULL). */
int orc_attn_prefill(const double *q, const double *k_raw, const double *v, const int *start,
                     int B, int C, int H, int Hkv, int D, int Tcap, double eps, double base, int flags, int W,
                     double *out, double *lse)
{
    if (Hkv < 1 || H % Hkv) return -1;
    const int G = H / Hkv;
    double scale = 1.0 / sqrt((double)D);
    int err = 0;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            int s0 = start[b];
            if (s0 < 0 || s0 + C > Tcap) { err = -2; continue; }
            int L = s0 + C;
            double *qh = malloc((size_t)D * sizeof(double));
            double *kh = malloc((size_t)L * D * sizeof(double));
            double *s = malloc((size_t)L * sizeof(double));
            for (int j = 0; j < L; ++j) {
                const double *kj = k_raw + at4(b, j, h / G, 0, Tcap, Hkv, D);
                double rk = (flags & ORC_NORM) ? rms_of(kj, D, eps) : 1.0;
                for (int d = 0; d < D; ++d) kh[(size_t)j * D + d] = kj[d] / rk;
                if (flags & ORC_ROPE) rotate(kh + (size_t)j * D, j, D, base, +1);
            }
            for (int t = 0; t < C; ++t) {
                int p = s0 + t;
                const double *qi = q + at4(b, t, h, 0, C, H, D);
                double rq = (flags & ORC_NORM) ? rms_of(qi, D, eps) : 1.0;
                for (int d = 0; d < D; ++d) qh[d] = qi[d] / rq;
                if (flags & ORC_ROPE) rotate(qh, p, D, base, +1);
                double m = -INFINITY;
                for (int j = 0; j < L; ++j) {
                    s[j] = -INFINITY;
                    if (!visible(p, j, W)) continue;
                    s[j] = dot(qh, kh + (size_t)j * D, D) * scale;
                    if (s[j] > m) m = s[j];
                }
                double l = 0.0;
                for (int j = 0; j < L; ++j) {
                    s[j] = exp(s[j] - m);
                    l += s[j];
                }
                double *oi = out + at4(b, t, h, 0, C, H, D);
                for (int d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (int j = 0; j < L; ++j) acc += s[j] / l * v[at4(b, j, h / G, d, Tcap, Hkv, D)];
                    oi[d] = acc;
                }
                if (lse) lse[((size_t)b * H + h) * C + t] = m + log(l);
            }
            free(qh); free(kh); free(s);
        }
    return err;
}

