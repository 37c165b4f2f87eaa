/*
 * mtp_oracle.c -- plain float64 CPU oracle for MTP rejection-sampling
 * verification, per-position row statistics and the end-to-end TV loss.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links or calls this
 * file: only the test suite, the package smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; it is written from the method's definitions, one row at a
 * time, with no blocking, fusion or reordering beyond what they state.
 *
 * Sources (cited by page title and section):
 *   [BB]  "Breaking Entropy Bounds: Accelerating RL Training via MTP with
 *         Rejection Sampling" (paperlayer.ai summary of arXiv 2606.12370).
 *   [BBz] The same paper, Chinese summary (paper.rainbus.top), sections
 *         "前置知识" (background) and "核心方法" / "技术新颖性" (method).
 *   [EM]  "EntMTP: Accelerating LLM Inference with Entropy Guided Multi Token
 *         Prediction", Related Work, "Speculative Decoding".
 *
 * Readings of points the pages leave open (each one is listed with its reason
 * in the design notes of the repository):
 *   - One temperature T per sequence scales both target and draft logits.
 *   - Accept test is the strict comparison u*q(y) < p(y), u in [0,1).
 *   - u[b, 0..gamma-1] are the accept tests; u[b, gamma] is the single final
 *     draw (residual or bonus).  Uniforms after the stop are not used.
 *   - The bonus token after gamma accepts is the residual draw with q = 0,
 *     i.e. a draw from p_gamma.
 *   - Inverse CDF: ascending vocabulary index, smallest v with C(v) > u*R; if
 *     rounding leaves no such v, the last v with r_v > 0.  R == 0 at a
 *     rejection (only reachable through rounding) draws from p_j and sets the
 *     ZERO_MASS flag.
 *   - TV-gradient indicator 1[q <= p] as the pages write it (tie_le = 1);
 *     tie_le = 0 selects the strict 1[q < p].
 *   - e2e loss l = -sum_{k=1..gamma} prod_{i<=k} alpha_i, unnormalised.
 *   - T == 0 is greedy decoding: p and q are one-hot at the row's arg max
 *     (ties to the smallest index), so a draft is accepted iff it is the
 *     target's arg max and the replacement / bonus token is the arg max.
 *     Statistics need T > 0.  T < 0, NaN or inf is a bad temperature.
 *   - Target-only acceptance: the draft token is the arg max of the draft
 *     logits (ties to the smallest index), accepted iff u < p(y); at the
 *     first rejection the replacement is drawn from p with y removed, i.e.
 *     the residual of rejection sampling with a one-hot draft.
 *   - Gumbel-max final draw ([BB] App. G.2): the acceptance chain is the
 *     same; the residual (or bonus) token is arg max_v [ln w_v + G_v] over
 *     the v with w_v > 0, G_v = -ln(-ln U_v) standard Gumbel noise.  U_v
 *     comes from the counter-based generator Philox4x32-10 (Salmon, Moraes,
 *     Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011)
 *     with key (seed_lo, seed_hi) and counter (v / 4, i, b, offset), word
 *     v mod 4, where b is the sequence and i the row drawn from (the
 *     rejected position, or gamma for the bonus): U_v = (floor(x / 2^8) +
 *     1/2) / 2^24, exact in single precision and strictly inside (0, 1).
 *     u[b, gamma] is not used.
 *   - Shared target rows (the MTP layout): with target [N + gamma - 1, V],
 *     pair (t, k) uses target row t + k, the target model's distribution at
 *     the token that draft step k of position t predicts.
 *   - Top-K target (App. F): the target of a pair is given as its K largest
 *     logits and their indices; the target distribution is their softmax,
 *     renormalised over the K entries; the draft keeps its full softmax.
 *   - App. F clamped loss: per position the sum over steps of clamp(1 -
 *     alpha_k, 0, tau_max); its derivative in alpha_k is -1 strictly inside
 *     (0, tau_max) and 0 elsewhere (the subgradient 0 at the two kinks).
 *
 * Logit storage codes: 0 = float32, 1 = bfloat16 (uint16 bit patterns),
 * 2 = float64.  Every element is widened exactly to double before use.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_F32 0
#define OR_BF16 1
#define OR_F64 2

/* Row flag bits (same meanings as the library's documented flags). */
#define OR_ROW_NONFINITE 1
#define OR_ROW_BAD_ID 2
#define OR_ROW_BAD_TEMP 4
#define OR_ROW_ZERO_MASS 8
#define OR_ROW_BAD_UNIFORM 16
#define OR_ERROR_BITS (OR_ROW_NONFINITE | OR_ROW_BAD_ID | OR_ROW_BAD_TEMP | OR_ROW_BAD_UNIFORM)

/* Exact widening of one stored logit to double. */
static double load_logit(const void *base, int dtype, size_t idx)
{
    if (dtype == OR_F64) return ((const double *)base)[idx];
    if (dtype == OR_F32) return (double)((const float *)base)[idx];
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * p = softmax(z / T) over one row of V logits starting at element `off`.
 * Temperature-scaled softmax [BB, §7 "Temperature and generation position";
 * App. G.2 caches temperature-scaled logits].  Max subtraction only guards
 * exp() against overflow.  Returns 0 on success, OR_ROW_NONFINITE if a logit
 * is NaN or +inf or every logit is -inf (no probability can be formed).
 */
static int softmax_row(const void *z, int dtype, size_t off, int V, double T, double *p)
{
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double x = load_logit(z, dtype, off + (size_t)v);
        if (isnan(x) || (isinf(x) && x > 0)) return OR_ROW_NONFINITE;
        x = x / T;
        p[v] = x;
        if (x > m) m = x;
    }
    if (isinf(m)) return OR_ROW_NONFINITE; /* all -inf */
    double s = 0.0;
    for (int v = 0; v < V; ++v) {
        p[v] = exp(p[v] - m);
        s += p[v];
    }
    for (int v = 0; v < V; ++v) p[v] /= s;
    return 0;
}

/* Exported for tests: softmax of `rows` rows of length V at temperature T. */
int oracle_softmax(const void *z, int dtype, int rows, int V, double T, double *p)
{
    int bad = 0;
    for (int r = 0; r < rows; ++r)
        bad |= softmax_row(z, dtype, (size_t)r * V, V, T, p + (size_t)r * V);
    return bad;
}

/* alpha = sum_v min(p_v, q_v): the RS acceptance probability, equal to the
 * TV overlap [BB, §3 "Rejection Sampling"; §8 "Total Variation Distance"]. */
static double overlap(const double *p, const double *q, int V)
{
    double a = 0.0;
    for (int v = 0; v < V; ++v) a += (p[v] < q[v]) ? p[v] : q[v];
    return a;
}

/* d_TV(p, q) = 1/2 sum_v |p_v - q_v| [BBz, 前置知识 "Total Variation Distance"].
 * Computed independently of overlap() so tests can check alpha = 1 - TV. */
static double tv_distance(const double *p, const double *q, int V)
{
    double d = 0.0;
    for (int v = 0; v < V; ++v) d += fabs(p[v] - q[v]);
    return 0.5 * d;
}

/* H(p) = -sum_v p_v log p_v, in nats, terms with p_v = 0 omitted
 * [BBz, 前置知识 "Entropy"]. */
static double entropy(const double *p, int V)
{
    double h = 0.0;
    for (int v = 0; v < V; ++v)
        if (p[v] > 0.0) h -= p[v] * log(p[v]);
    return h;
}

/*
 * Index of the largest logit of one row (smallest index among equals);
 * -1 if a logit is NaN or +inf or every logit is -inf.  Greedy decoding and
 * target-only draft selection take the arg max [BB, App. D.2 "Target-Only
 * Sampling": the draft token is arg max_y q(y), and arg max of the softmax
 * is the arg max of the logits].
 */
static int argmax_row(const void *z, int dtype, size_t off, int V)
{
    int best = -1;
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double x = load_logit(z, dtype, off + (size_t)v);
        if (isnan(x) || (isinf(x) && x > 0)) return -1;
        if (x > m) {
            m = x;
            best = v;
        }
    }
    return best;
}

/* D_KL(q || p) = sum_{q_v > 0} q_v log(q_v / p_v), in nats; +inf where some
 * q_v > 0 has p_v = 0 [BB, §9 "Distributional effects of TV loss"]. */
static double kl_qp(const double *q, const double *p, int V)
{
    double d = 0.0;
    for (int v = 0; v < V; ++v) {
        if (q[v] > 0.0) {
            if (!(p[v] > 0.0)) return INFINITY;
            d += q[v] * log(q[v] / p[v]);
        }
    }
    return d;
}

/*
 * Inverse-CDF draw from the unnormalised weights r[0..V-1] with uniform u:
 * C(v) = sum_{w<=v} r_w, R = C(V-1); returns the smallest v with C(v) > u*R,
 * or the last v with r_v > 0 if rounding leaves none.  This is the residual
 * resampling step [EM, "Speculative Decoding": draw from
 * norm(max(0, p - q))] done as a two-pass CDF inversion [BB, App. G.1]:
 * pass one sums R, pass two walks the CDF.  *margin receives
 * min(u*R - C(v-1), C(v) - u*R) / R, the distance of the draw from the
 * nearest CDF breakpoint (0 when R == 0).
 */
static int cdf_draw(const double *r, int V, double u, double *margin)
{
    double R = 0.0;
    for (int v = 0; v < V; ++v) R += r[v];
    double t = u * R;
    double c = 0.0;
    for (int v = 0; v < V; ++v) {
        double prev = c;
        c += r[v];
        if (c > t) {
            double a = t - prev, b = c - t;
            *margin = (R > 0.0) ? ((a < b) ? a : b) / R : 0.0;
            return v;
        }
    }
    int last = -1;
    for (int v = 0; v < V; ++v)
        if (r[v] > 0.0) last = v;
    *margin = 0.0;
    return last;
}

/*
 * One sequence of the verify step.  target: gamma+1 rows, draft: gamma rows,
 * row-major [., V] starting at the given element offsets.
 *
 * Steps [BB, §2 "Acceptance methods"; App. G.1; EM, "Speculative Decoding"]:
 * for i = 0..gamma-1 compute p_i = softmax(target_i / T), q_i =
 * softmax(draft_i / T) and accept draft y_i iff u_i * q_i(y_i) < p_i(y_i),
 * i.e. with probability min(1, p_i(y_i)/q_i(y_i)); stop at the first
 * rejection j and draw the replacement from norm(max(0, p_j - q_j)).  If all
 * gamma drafts are accepted, draw the bonus token from p_gamma.
 *
 * With want_stats, alpha_i, TV_i (i < gamma) and H_i (i <= gamma) are formed
 * for every position, including positions after the stop.
 */
/*
 * Philox4x32-10 [Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
 * easy as 1, 2, 3", SC 2011]: ten rounds of the Philox S-box on a 4 x 32-bit
 * counter.  A round multiplies counter words 0 and 2 by the two round
 * multipliers (full 64-bit products), and forms the new counter (hi(M1 c2)
 * ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)); the key is bumped
 * by the two Weyl constants between rounds.
 */
static void philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u, W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)M0 * c0, p1 = (uint64_t)M1 * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n1 = (uint32_t)p1;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        const uint32_t n3 = (uint32_t)p0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
        k0 += W0;
        k1 += W1;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

int oracle_philox4x32_10(const uint32_t *ctr, const uint32_t *key, uint32_t *out)
{
    philox4x32_10(ctr, key, out);
    return 0;
}

/* Key and counter words of one Gumbel stream (one sequence). */
struct gumbel_ctx {
    uint32_t seed_lo, seed_hi, offset, b;
};

/* U_v in (0, 1) for vocabulary index v of row i (see the header). */
static double gumbel_uniform(const struct gumbel_ctx *g, int i, int v)
{
    const uint32_t ctr[4] = {(uint32_t)v >> 2, (uint32_t)i, g->b, g->offset};
    const uint32_t key[2] = {g->seed_lo, g->seed_hi};
    uint32_t x[4];
    philox4x32_10(ctr, key, x);
    return ((double)(x[v & 3] >> 8) + 0.5) / 16777216.0;
}

/* Standard Gumbel noise G = -ln(-ln U). */
static double gumbel_noise(const struct gumbel_ctx *g, int i, int v)
{
    return -log(-log(gumbel_uniform(g, i, v)));
}

int oracle_gumbel_noise(uint32_t seed_lo, uint32_t seed_hi, uint32_t offset, uint32_t b, int i, int v0, int n,
                        double *out)
{
    const struct gumbel_ctx g = {seed_lo, seed_hi, offset, b};
    for (int j = 0; j < n; ++j) out[j] = gumbel_noise(&g, i, v0 + j);
    return 0;
}

/*
 * Gumbel-max draw from the unnormalised weights w[0..V-1] of row i [BB, App.
 * G.2]: arg max over w_v > 0 of ln w_v + G_v (-1 if every weight is 0).
 * *margin receives the gap between the best and the second best key (+inf
 * with a single candidate): the decision is exact unless rounding of the
 * keys exceeds it.
 */
static int gumbel_draw(const double *w, int V, const struct gumbel_ctx *g, int i, double *margin)
{
    double best = -INFINITY, second = -INFINITY;
    int arg = -1;
    for (int v = 0; v < V; ++v) {
        if (!(w[v] > 0.0)) continue;
        const double key = log(w[v]) + gumbel_noise(g, i, v);
        if (arg < 0 || key > best) {
            second = best;
            best = key;
            arg = v;
        } else if (key > second) {
            second = key;
        }
    }
    *margin = arg < 0 ? 0.0 : best - second;
    return arg;
}

static void verify_one(const void *target, const void *draft, int dtype, size_t toff, size_t doff,
                       const int32_t *ids, double T, const double *u, int gamma, int V, int want_stats,
                       int32_t *tokens, int32_t *accept_len, double *alpha, double *tv, double *ent,
                       int32_t *flags, double *acc_margin, double *cdf_margin, double *p, double *q,
                       double *r, const struct gumbel_ctx *gumbel)
{
    int f = 0;
    for (int i = 0; i <= gamma; ++i) tokens[i] = -1;
    for (int i = 0; i < gamma; ++i) acc_margin[i] = NAN;
    *cdf_margin = NAN;
    if (want_stats) {
        for (int i = 0; i < gamma; ++i) alpha[i] = tv[i] = NAN;
        for (int i = 0; i <= gamma; ++i) ent[i] = NAN;
    }
    if (!(T >= 0.0) || isinf(T) || (T == 0.0 && want_stats)) f |= OR_ROW_BAD_TEMP;
    for (int i = 0; i < gamma; ++i)
        if (ids[i] < 0 || ids[i] >= V) f |= OR_ROW_BAD_ID;
    for (int i = 0; i < gamma + (gumbel ? 0 : 1); ++i)  /* the Gumbel draw uses no u[gamma] */
        if (!(u[i] >= 0.0 && u[i] < 1.0)) f |= OR_ROW_BAD_UNIFORM;
    if (f) {
        *accept_len = -1;
        *flags = f;
        return;
    }

    /* Greedy (T == 0): accept while the draft is the target's arg max, then
     * emit the target's arg max.  No probability is formed. */
    if (T == 0.0) {
        int n = 0;
        for (int i = 0; i <= gamma; ++i) {
            int a = argmax_row(target, dtype, toff + (size_t)i * V, V);
            if (a < 0) {
                for (int j = 0; j <= gamma; ++j) tokens[j] = -1;
                *accept_len = -1;
                *flags = OR_ROW_NONFINITE;
                return;
            }
            if (i < gamma) acc_margin[i] = INFINITY;
            if (i < gamma && ids[i] == a) {
                tokens[i] = a;
                ++n;
                continue;
            }
            tokens[i] = a;
            break;
        }
        *cdf_margin = INFINITY;
        *accept_len = n;
        *flags = 0;
        return;
    }

    /* Stats pass: every position, independent of the decisions. */
    if (want_stats) {
        for (int i = 0; i <= gamma; ++i) {
            f |= softmax_row(target, dtype, toff + (size_t)i * V, V, T, p);
            if (f) break;
            ent[i] = entropy(p, V);
            if (i < gamma) {
                f |= softmax_row(draft, dtype, doff + (size_t)i * V, V, T, q);
                if (f) break;
                alpha[i] = overlap(p, q, V);
                tv[i] = tv_distance(p, q, V);
            }
        }
        if (f) {
            for (int i = 0; i < gamma; ++i) alpha[i] = tv[i] = NAN;
            for (int i = 0; i <= gamma; ++i) ent[i] = NAN;
            *accept_len = -1;
            *flags = f;
            return;
        }
    }

    /* Accept chain: left to right, stop at the first rejection. */
    int n = 0, rejected = 0;
    for (int i = 0; i < gamma; ++i) {
        f |= softmax_row(target, dtype, toff + (size_t)i * V, V, T, p);
        f |= softmax_row(draft, dtype, doff + (size_t)i * V, V, T, q);
        if (f) break;
        double py = p[ids[i]], qy = q[ids[i]];
        double ratio = (qy > 0.0) ? py / qy : (py > 0.0 ? INFINITY : NAN);
        acc_margin[i] = isnan(ratio) ? 0.0 : fabs(u[i] - ratio);
        if (u[i] * qy < py) {
            tokens[i] = ids[i];
            ++n;
            continue;
        }
        rejected = 1;
        break;
    }
    if (f) {
        for (int i = 0; i <= gamma; ++i) tokens[i] = -1;
        *accept_len = -1;
        *flags = f;
        return;
    }

    /* Final draw: residual at the rejection, or bonus from p_gamma. */
    if (rejected) {
        double R = 0.0;
        for (int v = 0; v < V; ++v) {
            double d = p[v] - q[v];
            r[v] = d > 0.0 ? d : 0.0;
            R += r[v];
        }
        if (!(R > 0.0)) {
            f |= OR_ROW_ZERO_MASS;
            memcpy(r, p, sizeof(double) * (size_t)V);
        }
    } else {
        f |= softmax_row(target, dtype, toff + (size_t)gamma * V, V, T, p);
        if (f) {
            for (int i = 0; i <= gamma; ++i) tokens[i] = -1;
            *accept_len = -1;
            *flags = f;
            return;
        }
        memcpy(r, p, sizeof(double) * (size_t)V);
    }
    tokens[n] = gumbel ? gumbel_draw(r, V, gumbel, n, cdf_margin) : cdf_draw(r, V, u[gamma], cdf_margin);
    *accept_len = n;
    *flags = f;
}

/*
 * Batched verify over B sequences (OpenMP over sequences).
 *   target  [B, gamma+1, V], draft [B, gamma, V] in storage `dtype`
 *   ids     [B, gamma] int32, temp [B] (double), u [B, gamma+1] (double)
 * Outputs: tokens [B, gamma+1] (-1 padded), accept_len [B] (-1 if flagged),
 *   flags [B]; with want_stats alpha, tv [B, gamma] and ent [B, gamma+1]
 *   (may be NULL otherwise); acc_margin [B, gamma] = |u_i - p_i(y)/q_i(y)|
 *   for every decision taken (NaN where none), cdf_margin [B].
 */
int oracle_verify(const void *target, const void *draft, int dtype, const int32_t *ids, const double *temp,
                  const double *u, int B, int gamma, int V, int want_stats, int32_t *tokens,
                  int32_t *accept_len, double *alpha, double *tv, double *ent, int32_t *flags,
                  double *acc_margin, double *cdf_margin)
{
    if (B < 0 || gamma < 1 || V < 1) return 1;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        double *buf = (double *)malloc(sizeof(double) * (size_t)V * 3);
        if (!buf) {
#pragma omp atomic write
            fail = 1;
            continue;
        }
        verify_one(target, draft, dtype, (size_t)b * (gamma + 1) * V, (size_t)b * gamma * V, ids + (size_t)b * gamma,
                   temp[b], u + (size_t)b * (gamma + 1), gamma, V, want_stats, tokens + (size_t)b * (gamma + 1),
                   accept_len + b, want_stats ? alpha + (size_t)b * gamma : NULL,
                   want_stats ? tv + (size_t)b * gamma : NULL, want_stats ? ent + (size_t)b * (gamma + 1) : NULL,
                   flags + b, acc_margin + (size_t)b * gamma, cdf_margin + b, buf, buf + V, buf + 2 * (size_t)V,
                   NULL);
        free(buf);
    }
    return fail ? 2 : 0;
}

/*
 * Batched verify with the Gumbel-max final draw [BB, App. G.2]: the
 * acceptance chain of oracle_verify, then the residual (or bonus) token by
 * gumbel_draw with the stream (seed, offset, b).  u [B, gamma+1]: only
 * u[b, 0..gamma-1] are used.  gumbel_margin [B] receives the gap between the
 * best and second best key of the final draw (+inf for greedy rows).
 */
int oracle_gumbel_verify(const void *target, const void *draft, int dtype, const int32_t *ids, const double *temp,
                         const double *u, uint32_t seed_lo, uint32_t seed_hi, uint32_t offset, int B, int gamma,
                         int V, int32_t *tokens, int32_t *accept_len, int32_t *flags, double *acc_margin,
                         double *gumbel_margin)
{
    if (B < 0 || gamma < 1 || V < 1) return 1;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        double *buf = (double *)malloc(sizeof(double) * (size_t)V * 3);
        if (!buf) {
#pragma omp atomic write
            fail = 1;
            continue;
        }
        const struct gumbel_ctx g = {seed_lo, seed_hi, offset, (uint32_t)b};
        verify_one(target, draft, dtype, (size_t)b * (gamma + 1) * V, (size_t)b * gamma * V, ids + (size_t)b * gamma,
                   temp[b], u + (size_t)b * (gamma + 1), gamma, V, 0, tokens + (size_t)b * (gamma + 1),
                   accept_len + b, NULL, NULL, NULL, flags + b, acc_margin + (size_t)b * gamma, gumbel_margin + b,
                   buf, buf + V, buf + 2 * (size_t)V, &g);
        free(buf);
    }
    return fail ? 2 : 0;
}

/*
 * One sequence of target-only verification [BB, §2 "Acceptance methods":
 * the draft token is selected greedily and accepted with probability p(y);
 * App. D.2]: for i = 0..gamma-1, y_i = arg max of draft row i, p_i =
 * softmax(target_i / T); accept iff u_i < p_i(y_i); at the first rejection j
 * draw the replacement from p_j with y_j removed (the residual of rejection
 * sampling with a one-hot draft, so the output law stays p); after gamma
 * accepts draw the bonus from p_gamma.  With T == 0: accept iff y_i is the
 * target's arg max, and emit the target's arg max.  yhat[i] receives y_i
 * for every position the chain reached (-1 elsewhere).
 */
static void to_verify_one(const void *target, const void *draft, int dtype, size_t toff, size_t doff, double T,
                          const double *u, int gamma, int V, int32_t *tokens, int32_t *accept_len, int32_t *yhat,
                          int32_t *flags, double *acc_margin, double *cdf_margin, double *p, double *r)
{
    for (int i = 0; i <= gamma; ++i) tokens[i] = -1;
    for (int i = 0; i < gamma; ++i) {
        acc_margin[i] = NAN;
        yhat[i] = -1;
    }
    *cdf_margin = NAN;
    int f = 0;
    if (!(T >= 0.0) || isinf(T)) f |= OR_ROW_BAD_TEMP;
    for (int i = 0; i <= gamma; ++i)
        if (!(u[i] >= 0.0 && u[i] < 1.0)) f |= OR_ROW_BAD_UNIFORM;
    if (f) {
        *accept_len = -1;
        *flags = f;
        return;
    }
    int n = 0, rejected = 0, yj = -1;
    for (int i = 0; i < gamma; ++i) {
        int y = argmax_row(draft, dtype, doff + (size_t)i * V, V);
        if (y < 0) {
            f |= OR_ROW_NONFINITE;
            break;
        }
        yhat[i] = y;
        if (T == 0.0) {
            int a = argmax_row(target, dtype, toff + (size_t)i * V, V);
            if (a < 0) {
                f |= OR_ROW_NONFINITE;
                break;
            }
            acc_margin[i] = INFINITY;
            if (y == a) {
                tokens[i] = y;
                ++n;
                continue;
            }
            tokens[i] = a;
            *cdf_margin = INFINITY;
            *accept_len = n;
            *flags = 0;
            return;
        }
        f |= softmax_row(target, dtype, toff + (size_t)i * V, V, T, p);
        if (f) break;
        acc_margin[i] = fabs(u[i] - p[y]);
        if (u[i] < p[y]) {
            tokens[i] = y;
            ++n;
            continue;
        }
        rejected = 1;
        yj = y;
        break;
    }
    if (!f && !rejected) {
        if (T == 0.0) {
            int a = argmax_row(target, dtype, toff + (size_t)gamma * V, V);
            if (a < 0) {
                f |= OR_ROW_NONFINITE;
            } else {
                tokens[gamma] = a;
                *cdf_margin = INFINITY;
                *accept_len = n;
                *flags = 0;
                return;
            }
        } else {
            f |= softmax_row(target, dtype, toff + (size_t)gamma * V, V, T, p);
        }
    }
    if (f) {
        for (int i = 0; i <= gamma; ++i) tokens[i] = -1;
        *accept_len = -1;
        *flags = f;
        return;
    }
    memcpy(r, p, sizeof(double) * (size_t)V);
    if (rejected) {
        r[yj] = 0.0;
        double R = 0.0;
        for (int v = 0; v < V; ++v) R += r[v];
        if (!(R > 0.0)) { /* p(y) rounds to 1: draw from p, as for rejection sampling */
            f |= OR_ROW_ZERO_MASS;
            memcpy(r, p, sizeof(double) * (size_t)V);
        }
    }
    tokens[n] = cdf_draw(r, V, u[gamma], cdf_margin);
    *accept_len = n;
    *flags = f;
}

/*
 * Batched target-only verification (OpenMP over sequences).
 *   target [B, gamma+1, V], draft [B, gamma, V], temp [B], u [B, gamma+1]
 * Outputs: tokens [B, gamma+1], accept_len [B], yhat [B, gamma], flags [B],
 *   acc_margin [B, gamma] = |u_i - p_i(y_i)|, cdf_margin [B].
 */
int oracle_to_verify(const void *target, const void *draft, int dtype, const double *temp, const double *u, int B,
                     int gamma, int V, int32_t *tokens, int32_t *accept_len, int32_t *yhat, int32_t *flags,
                     double *acc_margin, double *cdf_margin)
{
    if (B < 0 || gamma < 1 || V < 1) return 1;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        double *buf = (double *)malloc(sizeof(double) * (size_t)V * 2);
        if (!buf) {
#pragma omp atomic write
            fail = 1;
            continue;
        }
        to_verify_one(target, draft, dtype, (size_t)b * (gamma + 1) * V, (size_t)b * gamma * V, temp[b],
                      u + (size_t)b * (gamma + 1), gamma, V, tokens + (size_t)b * (gamma + 1), accept_len + b,
                      yhat + (size_t)b * gamma, flags + b, acc_margin + (size_t)b * gamma, cdf_margin + b, buf,
                      buf + V);
        free(buf);
    }
    return fail ? 2 : 0;
}

/*
 * Per-position acceptance diagnostics, every position (no decisions).  For
 * draft position i < gamma with p = softmax(target_i / T), q =
 * softmax(draft_i / T): alpha_i = sum min(p, q), tv_i = d_TV(p, q), ent_q_i =
 * H(q), kl_i = D_KL(q || p), yhat_i = arg max of the draft logits, p_yhat_i
 * = p(yhat_i), and rs_better_i = [d_TV(p, q) < 1 - p(yhat_i)], the boundary
 * below which rejection sampling accepts more than target-only sampling
 * [BB, App. E "Rejection Sampling Decision Boundary Derivation"; §8
 * "Robustness of acceptance methods"].  ent_p_i = H(p_i) for i <= gamma.
 * boundary_margin_i = |d_TV - (1 - p(yhat))| for the parity rule.
 */
int oracle_diagnostics(const void *target, const void *draft, int dtype, const double *temp, int B, int gamma, int V,
                       double *alpha, double *tv, double *ent_q, double *kl, int32_t *yhat, double *p_yhat,
                       int32_t *rs_better, double *boundary_margin, double *ent_p, int32_t *flags)
{
    if (B < 0 || gamma < 1 || V < 1) return 1;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        double *p = (double *)malloc(sizeof(double) * (size_t)V * 2);
        if (!p) {
#pragma omp atomic write
            fail = 1;
            continue;
        }
        double *q = p + V;
        double T = temp[b];
        int f = (!(T > 0.0) || isinf(T)) ? OR_ROW_BAD_TEMP : 0;
        size_t toff = (size_t)b * (gamma + 1) * V, doff = (size_t)b * gamma * V;
        for (int i = 0; i <= gamma && !f; ++i) {
            f |= softmax_row(target, dtype, toff + (size_t)i * V, V, T, p);
            if (f) break;
            ent_p[(size_t)b * (gamma + 1) + i] = entropy(p, V);
            if (i < gamma) {
                size_t o = (size_t)b * gamma + i;
                f |= softmax_row(draft, dtype, doff + (size_t)i * V, V, T, q);
                if (f) break;
                int y = argmax_row(draft, dtype, doff + (size_t)i * V, V);
                alpha[o] = overlap(p, q, V);
                tv[o] = tv_distance(p, q, V);
                ent_q[o] = entropy(q, V);
                kl[o] = kl_qp(q, p, V);
                yhat[o] = y;
                p_yhat[o] = p[y];
                rs_better[o] = tv[o] < 1.0 - p[y];
                boundary_margin[o] = fabs(tv[o] - (1.0 - p[y]));
            }
        }
        if (f) {
            for (int i = 0; i < gamma; ++i) {
                size_t o = (size_t)b * gamma + i;
                alpha[o] = tv[o] = ent_q[o] = kl[o] = p_yhat[o] = boundary_margin[o] = NAN;
                yhat[o] = -1;
                rs_better[o] = -1;
            }
            for (int i = 0; i <= gamma; ++i) ent_p[(size_t)b * (gamma + 1) + i] = NAN;
        }
        flags[b] = f;
        free(p);
    }
    return fail ? 2 : 0;
}

/*
 * Per-position row statistics (no decisions): alpha_i = sum min(p_i, q_i) and
 * TV_i for i < gamma, H(p_i) for i <= gamma [BB, §3 "Rejection Sampling";
 * BBz, 前置知识 "Entropy"].  Flagged sequences get NaN statistics.
 */
int oracle_row_stats(const void *target, const void *draft, int dtype, const double *temp, int B, int gamma,
                     int V, double *alpha, double *tv, double *ent, int32_t *flags)
{
    if (B < 0 || gamma < 1 || V < 1) return 1;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        double *p = (double *)malloc(sizeof(double) * (size_t)V * 2);
        if (!p) {
#pragma omp atomic write
            fail = 1;
            continue;
        }
        double *q = p + V;
        double T = temp[b];
        int f = (!(T > 0.0) || isinf(T)) ? OR_ROW_BAD_TEMP : 0;
        size_t toff = (size_t)b * (gamma + 1) * V, doff = (size_t)b * gamma * V;
        for (int i = 0; i <= gamma && !f; ++i) {
            f |= softmax_row(target, dtype, toff + (size_t)i * V, V, T, p);
            if (f) break;
            ent[(size_t)b * (gamma + 1) + i] = entropy(p, V);
            if (i < gamma) {
                f |= softmax_row(draft, dtype, doff + (size_t)i * V, V, T, q);
                if (f) break;
                alpha[(size_t)b * gamma + i] = overlap(p, q, V);
                tv[(size_t)b * gamma + i] = tv_distance(p, q, V);
            }
        }
        if (f) {
            for (int i = 0; i < gamma; ++i) alpha[(size_t)b * gamma + i] = tv[(size_t)b * gamma + i] = NAN;
            for (int i = 0; i <= gamma; ++i) ent[(size_t)b * (gamma + 1) + i] = NAN;
        }
        flags[b] = f;
        free(p);
    }
    return fail ? 2 : 0;
}

/*
 * End-to-end TV loss forward and backward for N token positions, gamma draft
 * steps each.  target, draft: [N, gamma, V]; p is detached [BB, App. A].
 *
 *   alpha_k = sum_v min(p_kv, q_kv)                 [BB, §8]
 *   S_k     = sum_v 1[q_kv <= p_kv] q_kv            [BB, App. A]
 *   l_t     = -sum_{m=1..gamma} prod_{i<=m} alpha_i [BB, §4 "End-to-end TV
 *             loss": expected acceptance length, multiplicative over steps]
 *   g_k     = dl_t/dalpha_k = -sum_{m>=k} prod_{i<=m, i!=k} alpha_i
 *   dalpha_k/dz_j = (1/T) q_kj (1[q_kj <= p_kj] - S_k)   [BB, App. A; the
 *             1/T is the chain rule through q = softmax(z/T)]
 *   grad[t,k,j] = grad_scale * g_k * dalpha_k/dz_j.
 *
 * Outputs: loss [N], alpha [N, gamma], S [N, gamma], g [N, gamma], flags [N],
 * and grad [N, gamma, V] unless grad is NULL.  Flagged positions get NaN.
 */
/*
 * The TV-loss variants of [BB] App. F and of the MTP layout, as options of
 * the same computation:
 *   shared_target = 1: target is [N + gamma - 1, V], one row per token
 *     position, and pair (t, k) uses target row t + k (the target model's
 *     distribution at the token that draft step k of position t predicts);
 *     shared_target = 0: target is [N, gamma, V] like the draft.
 *   loss_kind = 1: the per-step clamped loss of App. F summed over the
 *     steps, l_t = sum_k clamp(1 - alpha_k, 0, tau_max), whose derivative
 *     dl_t/dalpha_k is -1 where 0 < 1 - alpha_k < tau_max and 0 elsewhere
 *     (the subgradient 0 at the kinks); loss_kind = 0: the e2e loss above.
 */
int oracle_tv_loss_ex(const void *target, const void *draft, int dtype, double T, int N, int gamma, int V,
                      double grad_scale, int tie_le, int shared_target, int loss_kind, double tau_max,
                      double *loss, double *alpha, double *S, double *g, double *grad, int32_t *flags);

int oracle_tv_loss(const void *target, const void *draft, int dtype, double T, int N, int gamma, int V,
                   double grad_scale, int tie_le, double *loss, double *alpha, double *S, double *g,
                   double *grad, int32_t *flags)
{
    return oracle_tv_loss_ex(target, draft, dtype, T, N, gamma, V, grad_scale, tie_le, 0, 0, 0.0, loss, alpha, S,
                             g, grad, flags);
}

int oracle_tv_loss_ex(const void *target, const void *draft, int dtype, double T, int N, int gamma, int V,
                      double grad_scale, int tie_le, int shared_target, int loss_kind, double tau_max,
                      double *loss, double *alpha, double *S, double *g, double *grad, int32_t *flags)
{
    if (N < 0 || gamma < 1 || V < 1) return 1;
    if (loss_kind == 1 && !(tau_max >= 0.0)) return 1;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < N; ++t) {
        double *p = (double *)malloc(sizeof(double) * (size_t)V * 2);
        if (!p) {
#pragma omp atomic write
            fail = 1;
            continue;
        }
        double *q = p + V;
        int f = (!(T > 0.0) || isinf(T)) ? OR_ROW_BAD_TEMP : 0;
        double *a = alpha + (size_t)t * gamma, *s = S + (size_t)t * gamma, *gk = g + (size_t)t * gamma;
        for (int k = 0; k < gamma && !f; ++k) {
            size_t off = ((size_t)t * gamma + k) * V;
            size_t toff = shared_target ? (size_t)(t + k) * V : off;
            f |= softmax_row(target, dtype, toff, V, T, p);
            f |= softmax_row(draft, dtype, off, V, T, q);
            if (f) break;
            a[k] = overlap(p, q, V);
            double sk = 0.0;
            for (int v = 0; v < V; ++v)
                if (tie_le ? (q[v] <= p[v]) : (q[v] < p[v])) sk += q[v];
            s[k] = sk;
        }
        flags[t] = f;
        if (f) {
            loss[t] = NAN;
            for (int k = 0; k < gamma; ++k) a[k] = s[k] = gk[k] = NAN;
            if (grad)
                for (size_t e = 0; e < (size_t)gamma * V; ++e) grad[(size_t)t * gamma * V + e] = NAN;
            free(p);
            continue;
        }
        double l = 0.0;
        if (loss_kind == 1) {
            /* Clamped per-step loss and its (sub)gradient. */
            for (int k = 0; k < gamma; ++k) {
                const double d = 1.0 - a[k];
                l += d < 0.0 ? 0.0 : (d > tau_max ? tau_max : d);
                gk[k] = (d > 0.0 && d < tau_max) ? -1.0 : 0.0;
            }
            loss[t] = l;
        } else {
            /* Loss: sum over the gamma prefix products. */
            for (int m = 0; m < gamma; ++m) {
                double prod = 1.0;
                for (int i = 0; i <= m; ++i) prod *= a[i];
                l -= prod;
            }
            loss[t] = l;
            /* dl/dalpha_k: each product containing alpha_k, with alpha_k removed. */
            for (int k = 0; k < gamma; ++k) {
                double d = 0.0;
                for (int m = k; m < gamma; ++m) {
                    double prod = 1.0;
                    for (int i = 0; i <= m; ++i)
                        if (i != k) prod *= a[i];
                    d -= prod;
                }
                gk[k] = d;
            }
        }
        if (grad) {
            for (int k = 0; k < gamma; ++k) {
                size_t off = ((size_t)t * gamma + k) * V;
                size_t toff = shared_target ? (size_t)(t + k) * V : off;
                softmax_row(target, dtype, toff, V, T, p);
                softmax_row(draft, dtype, off, V, T, q);
                for (int v = 0; v < V; ++v) {
                    double ind = (tie_le ? (q[v] <= p[v]) : (q[v] < p[v])) ? 1.0 : 0.0;
                    grad[off + v] = grad_scale * gk[k] * (1.0 / T) * q[v] * (ind - s[k]);
                }
            }
        }
        free(p);
    }
    return fail ? 2 : 0;
}

/*
 * Draft sampling, the step before verification [BB, App. G "Rejection
 * Sampling Inference Implementation": production rejection sampling draws the
 * draft tokens from q; G.1 multinomial (SGLang), G.2 Gumbel-max (vLLM)]:
 * for row r of logits [R, V], q = softmax(z_r / T_r) and
 *   method 0: the inverse-CDF draw with u[r] (cdf_draw: the smallest v with
 *             C(v) > u R);
 *   method 1: the Gumbel-max draw arg max_v [ln q_v + G_v] with the noise of
 *             row 0 of sequence r (counter (v / 4, 0, r, offset)), i.e. the
 *             bonus draw of a one-row sequence; u is not used.
 * T_r == 0 is greedy (arg max, ties to the smallest index).  margin[r] is the
 * draw's distance to a decision boundary: the CDF margin, the gap between
 * the two best Gumbel keys, or +inf for greedy rows.
 */
int oracle_draft_sample(const void *logits, int dtype, const double *temp, const double *u, int method,
                        uint32_t seed_lo, uint32_t seed_hi, uint32_t offset, int R, int V, int32_t *ids,
                        int32_t *flags, double *margin)
{
    if (R < 0 || V < 1 || (method != 0 && method != 1)) return 1;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < R; ++r) {
        double *q = (double *)malloc(sizeof(double) * (size_t)V);
        if (!q) {
#pragma omp atomic write
            fail = 1;
            continue;
        }
        const double T = temp[r];
        int f = 0;
        ids[r] = -1;
        margin[r] = NAN;
        if (!(T >= 0.0) || isinf(T)) f |= OR_ROW_BAD_TEMP;
        /* the uniform is checked on every row, greedy ones included, like the
         * final uniform of verification */
        if (method == 0 && !(u[r] >= 0.0 && u[r] < 1.0)) f |= OR_ROW_BAD_UNIFORM;
        if (!f && T == 0.0) {
            ids[r] = argmax_row(logits, dtype, (size_t)r * V, V);
            margin[r] = INFINITY;
            if (ids[r] < 0) f |= OR_ROW_NONFINITE;
        } else if (!f) {
            f |= softmax_row(logits, dtype, (size_t)r * V, V, T, q);
            if (!f) {
                if (method == 0) {
                    ids[r] = cdf_draw(q, V, u[r], &margin[r]);
                } else {
                    const struct gumbel_ctx g = {seed_lo, seed_hi, offset, (uint32_t)r};
                    ids[r] = gumbel_draw(q, V, &g, 0, &margin[r]);
                }
            }
        }
        if (f) ids[r] = -1;
        flags[r] = f;
        free(q);
    }
    return fail ? 2 : 0;
}

/*
 * Top-K TV loss [BB, App. F: "an optional top-K path reduces memory from
 * O(|V|) to O(K)"]: the detached target of pair (t, k) is cached as its K
 * largest logits (values [N, gamma, K] in storage `dtype`) and their
 * vocabulary indices (idx [N, gamma, K], distinct, in [0, V)).  The target
 * distribution is the softmax over those K entries at temperature T,
 * renormalised (p~ = 0 elsewhere); q = softmax(z_d / T) over the full row.
 * alpha~_k = sum_e min(p~_e, q_{idx_e}), S~_k = sum over entries with
 * q_{idx_e} <= p~_e of q_{idx_e}; the loss (e2e, or the clamped per-step
 * loss) and the gradient are those of oracle_tv_loss_ex with p~ in place of
 * p: grad_j = scale g_k (1/T) q_j (1[j is an entry with q_j <= p~_j] - S~_k).
 * An index outside [0, V) sets BAD_ID; a NaN / +inf value or draft logit, or
 * an all -inf row, sets NONFINITE.
 */
int oracle_tv_loss_topk(const void *values, const int32_t *idx, const void *draft, int dtype, double T, int N,
                        int gamma, int K, int V, double grad_scale, int tie_le, int loss_kind, double tau_max,
                        double *loss, double *alpha, double *S, double *g, double *grad, int32_t *flags)
{
    if (N < 0 || gamma < 1 || V < 1 || K < 1) return 1;
    if (loss_kind == 1 && !(tau_max >= 0.0)) return 1;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < N; ++t) {
        double *q = (double *)malloc(sizeof(double) * ((size_t)V + (size_t)K));
        if (!q) {
#pragma omp atomic write
            fail = 1;
            continue;
        }
        double *pk = q + V;
        int f = (!(T > 0.0) || isinf(T)) ? OR_ROW_BAD_TEMP : 0;
        double *a = alpha + (size_t)t * gamma, *s = S + (size_t)t * gamma, *gk = g + (size_t)t * gamma;
        for (int k = 0; k < gamma && !f; ++k) {
            const size_t base = ((size_t)t * gamma + k) * K;
            for (int e = 0; e < K; ++e)
                if (idx[base + e] < 0 || idx[base + e] >= V) f |= OR_ROW_BAD_ID;
            if (f) break;
            f |= softmax_row(values, dtype, base, K, T, pk);
            f |= softmax_row(draft, dtype, ((size_t)t * gamma + k) * V, V, T, q);
            if (f) break;
            double ak = 0.0, sk = 0.0;
            for (int e = 0; e < K; ++e) {
                const double qv = q[idx[base + e]];
                ak += qv < pk[e] ? qv : pk[e];
                if (tie_le ? (qv <= pk[e]) : (qv < pk[e])) sk += qv;
            }
            a[k] = ak;
            s[k] = sk;
        }
        flags[t] = f;
        if (f) {
            loss[t] = NAN;
            for (int k = 0; k < gamma; ++k) a[k] = s[k] = gk[k] = NAN;
            if (grad)
                for (size_t e = 0; e < (size_t)gamma * V; ++e) grad[(size_t)t * gamma * V + e] = NAN;
            free(q);
            continue;
        }
        double l = 0.0;
        if (loss_kind == 1) {
            for (int k = 0; k < gamma; ++k) {
                const double d = 1.0 - a[k];
                l += d < 0.0 ? 0.0 : (d > tau_max ? tau_max : d);
                gk[k] = (d > 0.0 && d < tau_max) ? -1.0 : 0.0;
            }
        } else {
            for (int m = 0; m < gamma; ++m) {
                double prod = 1.0;
                for (int i = 0; i <= m; ++i) prod *= a[i];
                l -= prod;
            }
            for (int k = 0; k < gamma; ++k) {
                double d = 0.0;
                for (int m = k; m < gamma; ++m) {
                    double prod = 1.0;
                    for (int i = 0; i <= m; ++i)
                        if (i != k) prod *= a[i];
                    d -= prod;
                }
                gk[k] = d;
            }
        }
        loss[t] = l;
        if (grad) {
            for (int k = 0; k < gamma; ++k) {
                const size_t off = ((size_t)t * gamma + k) * V, base = ((size_t)t * gamma + k) * K;
                softmax_row(values, dtype, base, K, T, pk);
                softmax_row(draft, dtype, off, V, T, q);
                for (int v = 0; v < V; ++v) grad[off + v] = grad_scale * gk[k] * (1.0 / T) * q[v] * (0.0 - s[k]);
                for (int e = 0; e < K; ++e) {
                    const int v = idx[base + e];
                    const double ind = (tie_le ? (q[v] <= pk[e]) : (q[v] < pk[e])) ? 1.0 : 0.0;
                    grad[off + v] = grad_scale * gk[k] * (1.0 / T) * q[v] * (ind - s[k]);
                }
            }
        }
        free(q);
    }
    return fail ? 2 : 0;
}

/* Thread count of later parallel regions (timing runs on a stated number
 * of cores; n <= 0 leaves it unchanged).  No arithmetic depends on it. */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oracle_num_threads(void)
{
    int n = 1;
#ifdef _OPENMP
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
#endif
    return n;
}
