/*
 * attn_oracle.c -- plain fp64 CPU oracle for masked training attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (row-materialised, no tiling, no online rescaling):
 *
 *   SpecForge long-context post, "EAGLE3 Training":
 *       attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V
 *   CS336 README, "Flash Attention (Triton)": the forward keeps the per-row
 *       logsumexp L and the backward recomputes the weights from L.
 *   HOT-Step flash-attn-training, section 1 ("What exists"): forward emits O
 *       and LSE, backward emits dQ, dK, dV; section 6 trap 9: a query row that
 *       sees no key gets O = 0 and LSE = 0.
 *
 * Visibility (mask) follows the SpecForge post, "Flex Attention": the eagle3
 * mask_mod is or(causal_mask, suffix_mask) with shift_left = t (the number of
 * appended TTT segments), Q_LEN = Sq and KV_LEN = (t+1)*Sq.  Its padding
 * terms take the per-batch key length seq_lengths[b] (kv < seq_lengths[b] in
 * the causal part, kv % Q_LEN < seq_lengths[b] in the suffix part); without
 * lengths every key is inside.  The same key-length bound applies to the
 * full, causal and window masks.  The window mask (the band of the HOT-Step
 * page's self-attention over a window, section 4, read as q - left <= kv <=
 * q + right) takes its two extents from the caller.
 *
 * Additive mask (HOT-Step section 3: its ops accept an arbitrary additive
 * mask shaped [S_kv, S], or [S_kv, S, 1, B] with broadcast): an optional M[b][q][kv] added to
 * the scaled scores of the pairs the mask kind admits; M = -inf hides the
 * pair.  One M per batch entry (or one for all), shared by every head.
 *
 * For every (b, h) and query row q:
 *     s[kv]  = scale * sum_d Q[q,d] K[kv,d]        (visible kv only)
 *     LSE[q] = log sum_kv exp(s[kv])               (two-pass: max, then sum)
 *     P[kv]  = exp(s[kv] - LSE[q])
 *     O[q,:] = sum_kv P[kv] V[kv,:]
 * Backward with upstream dO:
 *     dP[kv] = sum_d dO[q,d] V[kv,d]
 *     Delta  = sum_d dO[q,d] O[q,d]                (O recomputed here in fp64)
 *     dS[kv] = P[kv] (dP[kv] - Delta)
 *     dQ[q,:] = scale * sum_kv dS[kv] K[kv,:]
 *     dK[kv,:] += scale * dS[kv] Q[q,:]             (summed over the q heads of
 *     dV[kv,:] += P[kv] dO[q,:]                      the kv head, ascending h)
 *
 * GQA: kv head of q head h is h / (Hq / Hkv) (contiguous groups).
 * Layout of every array: contiguous [B][H][S][D] fp64; LSE is [B][Hq][Sq].
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MASK_FULL 0
#define ORACLE_MASK_CAUSAL 1
#define ORACLE_MASK_TTT 2
#define ORACLE_MASK_WINDOW 3

/* Visibility of key kv to query q.  Returns 1 if visible.
 *   t       TTT step (shift_left and number of suffix segments), TTT only
 *   wl, wr  window extents (kv in [q - wl, q + wr]), window mask only
 *   len     key length of this batch (seq_lengths[b]); negative = no padding */
int oracle_visible(int mask, int t, long wl, long wr, long len, long Sq, long Skv, long q,
                   long kv)
{
    if (q < 0 || q >= Sq || kv < 0 || kv >= Skv) return 0;
    if (mask == ORACLE_MASK_TTT) {
        long S = Sq;
        long seq_len = len < 0 ? S : len;
        /* causal_mask: q_idx - shift_left >= kv_idx, padding kv_idx < seq_lengths[b] */
        int causal_part = (q - t >= kv) && (kv < seq_len);
        /* suffix_mask: kv_idx >= Q_LEN, kv_idx % Q_LEN < seq_lengths[b],
         *              (kv_idx - q_idx) % Q_LEN == 0 */
        int suffix_part = (kv >= S) && (kv < (long)(t + 1) * S) && (kv % S < seq_len) &&
                          (((kv - q) % S) == 0);
        return causal_part || suffix_part;
    }
    if (len >= 0 && kv >= len) return 0; /* padding: kv_idx < seq_lengths[b] */
    if (mask == ORACLE_MASK_FULL) return 1;
    if (mask == ORACLE_MASK_CAUSAL) return kv <= q;
    if (mask == ORACLE_MASK_WINDOW) return (kv >= q - wl) && (kv <= q + wr);
    return 0;
}

/* Dense visibility bitmap out[q*Skv + kv] in {0,1} for one batch entry. */
void oracle_mask(int mask, int t, long wl, long wr, long len, long Sq, long Skv,
                 unsigned char *out)
{
    for (long q = 0; q < Sq; ++q)
        for (long kv = 0; kv < Skv; ++kv)
            out[q * Skv + kv] = (unsigned char)oracle_visible(mask, t, wl, wr, len, Sq, Skv, q, kv);
}

/* The mask parameters that travel together through the passes. */
typedef struct {
    int mask, t;
    long wl, wr;
    const int *seq_lengths; /* [B] or NULL */
    const double *add;      /* additive mask [B or 1][Sq][Skv], or NULL */
    long add_sb;            /* batch stride of add in elements (0: one for all) */
} geom_t;

static long batch_len(const geom_t *g, int b)
{
    return g->seq_lengths ? (long)g->seq_lengths[b] : -1;
}

/* One query row: fills s[] (scaled scores, -INFINITY where invisible) and
 * returns the number of visible keys; *lse gets log sum exp(s) (0 if none). */
static long row_scores(const double *qrow, const double *Kh, long Skv, int D, double scale,
                       const geom_t *g, int b, long len, long Sq, long q, double *s, double *lse)
{
    long nvis = 0;
    double mx = -INFINITY;
    const double *arow = g->add ? g->add + (long)b * g->add_sb + q * Skv : NULL;
    for (long kv = 0; kv < Skv; ++kv) {
        if (!oracle_visible(g->mask, g->t, g->wl, g->wr, len, Sq, Skv, q, kv) ||
            (arow && arow[kv] == -INFINITY)) {
            s[kv] = -INFINITY;
            continue;
        }
        const double *krow = Kh + kv * (long)D;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += qrow[d] * krow[d];
        s[kv] = scale * acc + (arow ? arow[kv] : 0.0);
        if (s[kv] > mx) mx = s[kv];
        ++nvis;
    }
    if (nvis == 0) {
        *lse = 0.0;
        return 0;
    }
    double sum = 0.0;
    for (long kv = 0; kv < Skv; ++kv)
        if (s[kv] != -INFINITY) sum += exp(s[kv] - mx);
    *lse = mx + log(sum);
    return nvis;
}

static int check_shape(int B, int Hq, int Hkv, long Sq, long Skv, int D, const geom_t *g)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || D <= 0) return 1;
    if (Hq % Hkv != 0) return 1;
    if (g->mask < 0 || g->mask > 3) return 1;
    if (g->mask == ORACLE_MASK_TTT && (g->t < 0 || Skv != (long)(g->t + 1) * Sq)) return 1;
    if (g->mask == ORACLE_MASK_WINDOW && (g->wl < 0 || g->wr < 0)) return 1;
    if (g->seq_lengths)
        for (int b = 0; b < B; ++b)
            if (g->seq_lengths[b] < 0) return 1;
    return 0;
}

/* Forward over query rows [q_begin, q_end) of every (b, h): O [B,Hq,Sq,D],
 * LSE [B,Hq,Sq] (other rows untouched).  Returns 0 on success. */
int oracle_fwd_rows(int B, int Hq, int Hkv, long Sq, long Skv, int D, int mask, int t, long wl,
                    long wr, const int *seq_lengths, const double *add, long add_sb, double scale,
                    const double *Q, const double *K, const double *V, double *O, double *LSE,
                    long q_begin, long q_end)
{
    const geom_t g = {mask, t, wl, wr, seq_lengths, add, add_sb};
    if (check_shape(B, Hq, Hkv, Sq, Skv, D, &g)) return 1;
    if (q_begin < 0 || q_end > Sq || q_begin > q_end) return 1;
    const int G = Hq / Hkv;
    int ok = 1;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Skv);
        if (!s) {
#pragma omp atomic write
            ok = 0;
        }
#pragma omp for schedule(dynamic) collapse(2)
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < Hq; ++h) {
                if (!s) continue;
                const int hk = h / G;
                const double *Qh = Q + ((long)b * Hq + h) * Sq * D;
                const double *Kh = K + ((long)b * Hkv + hk) * Skv * D;
                const double *Vh = V + ((long)b * Hkv + hk) * Skv * D;
                double *Oh = O + ((long)b * Hq + h) * Sq * D;
                double *Lh = LSE + ((long)b * Hq + h) * Sq;
                for (long q = q_begin; q < q_end; ++q) {
                    double lse;
                    long nvis = row_scores(Qh + q * D, Kh, Skv, D, scale, &g, b, batch_len(&g, b),
                                           Sq, q, s, &lse);
                    double *orow = Oh + q * D;
                    for (int d = 0; d < D; ++d) orow[d] = 0.0;
                    Lh[q] = lse;
                    if (nvis == 0) continue;
                    for (long kv = 0; kv < Skv; ++kv) {
                        if (s[kv] == -INFINITY) continue;
                        const double p = exp(s[kv] - lse);
                        const double *vrow = Vh + kv * (long)D;
                        for (int d = 0; d < D; ++d) orow[d] += p * vrow[d];
                    }
                }
            }
        free(s);
    }
    return ok ? 0 : 2;
}

/* Forward over every row. */
int oracle_fwd(int B, int Hq, int Hkv, long Sq, long Skv, int D, int mask, int t, long wl, long wr,
               const int *seq_lengths, const double *add, long add_sb, double scale,
               const double *Q, const double *K, const double *V, double *O, double *LSE)
{
    return oracle_fwd_rows(B, Hq, Hkv, Sq, Skv, D, mask, t, wl, wr, seq_lengths, add, add_sb, scale,
                           Q, K, V, O, LSE, 0, Sq);
}

/* Backward over query rows [q_begin, q_end): dQ of those rows, and the dK /
 * dV contributions of those rows (the full gradients when the range is
 * [0, Sq)).  dQ [B,Hq,Sq,D], dK and dV [B,Hkv,Skv,D].  Recomputes P and O
 * itself.  dK/dV are accumulated per q head and then summed over the group in
 * ascending head order.  Returns 0 on success. */
int oracle_bwd_rows(int B, int Hq, int Hkv, long Sq, long Skv, int D, int mask, int t, long wl,
                    long wr, const int *seq_lengths, const double *add, long add_sb, double scale,
                    const double *Q, const double *K, const double *V, const double *dO,
                    double *dQ, double *dK, double *dV, long q_begin, long q_end)
{
    const geom_t g = {mask, t, wl, wr, seq_lengths, add, add_sb};
    if (check_shape(B, Hq, Hkv, Sq, Skv, D, &g)) return 1;
    if (q_begin < 0 || q_end > Sq || q_begin > q_end) return 1;
    const int G = Hq / Hkv;
    const size_t head_kv = (size_t)Skv * D;
    double *dKh_all = (double *)calloc((size_t)B * Hq * head_kv, sizeof(double));
    double *dVh_all = (double *)calloc((size_t)B * Hq * head_kv, sizeof(double));
    if (!dKh_all || !dVh_all) {
        free(dKh_all);
        free(dVh_all);
        return 2;
    }
    int ok = 1;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Skv);
        double *orow = (double *)malloc(sizeof(double) * (size_t)D);
        if (!s || !orow) {
#pragma omp atomic write
            ok = 0;
        }
#pragma omp for schedule(dynamic) collapse(2)
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < Hq; ++h) {
                if (!s || !orow) continue;
                const int hk = h / G;
                const double *Qh = Q + ((long)b * Hq + h) * Sq * D;
                const double *dOh = dO + ((long)b * Hq + h) * Sq * D;
                const double *Kh = K + ((long)b * Hkv + hk) * Skv * D;
                const double *Vh = V + ((long)b * Hkv + hk) * Skv * D;
                double *dQh = dQ + ((long)b * Hq + h) * Sq * D;
                double *dKh = dKh_all + ((size_t)b * Hq + h) * head_kv;
                double *dVh = dVh_all + ((size_t)b * Hq + h) * head_kv;
                for (long q = q_begin; q < q_end; ++q) {
                    double lse;
                    const double *qrow = Qh + q * D;
                    const double *dorow = dOh + q * D;
                    double *dqrow = dQh + q * D;
                    long nvis = row_scores(qrow, Kh, Skv, D, scale, &g, b, batch_len(&g, b), Sq, q,
                                           s, &lse);
                    for (int d = 0; d < D; ++d) dqrow[d] = 0.0;
                    if (nvis == 0) continue;
                    /* P in place of s; O row in fp64 */
                    for (int d = 0; d < D; ++d) orow[d] = 0.0;
                    for (long kv = 0; kv < Skv; ++kv) {
                        if (s[kv] == -INFINITY) {
                            s[kv] = 0.0;
                            continue;
                        }
                        s[kv] = exp(s[kv] - lse);
                        const double *vrow = Vh + kv * (long)D;
                        for (int d = 0; d < D; ++d) orow[d] += s[kv] * vrow[d];
                    }
                    double delta = 0.0;
                    for (int d = 0; d < D; ++d) delta += dorow[d] * orow[d];
                    for (long kv = 0; kv < Skv; ++kv) {
                        const double p = s[kv];
                        if (p == 0.0) continue;
                        const double *vrow = Vh + kv * (long)D;
                        const double *krow = Kh + kv * (long)D;
                        double dp = 0.0;
                        for (int d = 0; d < D; ++d) dp += dorow[d] * vrow[d];
                        const double ds = p * (dp - delta);
                        double *dkrow = dKh + kv * (long)D;
                        double *dvrow = dVh + kv * (long)D;
                        for (int d = 0; d < D; ++d) {
                            dqrow[d] += scale * ds * krow[d];
                            dkrow[d] += scale * ds * qrow[d];
                            dvrow[d] += p * dorow[d];
                        }
                    }
                }
            }
        free(s);
        free(orow);
    }
    /* fixed-order group reduction: dK[b,hk] = sum_{g=0..G-1} dK_h[b, hk*G+g] */
    for (int b = 0; b < B; ++b)
        for (int hk = 0; hk < Hkv; ++hk) {
            double *dKo = dK + ((size_t)b * Hkv + hk) * head_kv;
            double *dVo = dV + ((size_t)b * Hkv + hk) * head_kv;
            memset(dKo, 0, sizeof(double) * head_kv);
            memset(dVo, 0, sizeof(double) * head_kv);
            for (int g = 0; g < G; ++g) {
                const double *a = dKh_all + ((size_t)b * Hq + (size_t)hk * G + g) * head_kv;
                const double *c = dVh_all + ((size_t)b * Hq + (size_t)hk * G + g) * head_kv;
                for (size_t i = 0; i < head_kv; ++i) {
                    dKo[i] += a[i];
                    dVo[i] += c[i];
                }
            }
        }
    free(dKh_all);
    free(dVh_all);
    return ok ? 0 : 2;
}

/* Backward over every row. */
int oracle_bwd(int B, int Hq, int Hkv, long Sq, long Skv, int D, int mask, int t, long wl, long wr,
               const int *seq_lengths, const double *add, long add_sb, double scale,
               const double *Q, const double *K, const double *V, const double *dO, double *dQ,
               double *dK, double *dV)
{
    return oracle_bwd_rows(B, Hq, Hkv, Sq, Skv, D, mask, t, wl, wr, seq_lengths, add, add_sb, scale,
                           Q, K, V, dO, dQ, dK, dV, 0, Sq);
}

/* Exact count of visible (q, kv) pairs for one (b, h); used to pin the
 * mask-aware FLOP counter. */
long long oracle_count_visible(int mask, int t, long wl, long wr, long len, long Sq, long Skv)
{
    long long n = 0;
    for (long q = 0; q < Sq; ++q)
        for (long kv = 0; kv < Skv; ++kv) n += oracle_visible(mask, t, wl, wr, len, Sq, Skv, q, kv);
    return n;
}

/* Number of threads the OpenMP runtime will use (reported by the benchmark). */
int oracle_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}
