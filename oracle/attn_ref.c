/*
 * fp64 oracle for causal attention over packed rows with a document-level
 * (block-diagonal causal) mask, and its exact gradient.
 *
 * TEST INFRASTRUCTURE ONLY: called from tests/ and from the CPU-baseline leg of
 * bench.py through ctypes. It shares nothing with the CUDA library.
 *
 * What it computes (plain definitions, no tiling, no online softmax):
 *
 *   mask(i, j)  = seg(i) == seg(j) && j <= i
 *       the block-diagonal causal mask: one lower-triangular block per
 *       document, so a packed row is the same as its documents attended
 *       separately (page "Sample Packing: attention problems of long-sequence
 *       LLM training", section 3 "Attention Mask"); segments are the
 *       cu_seqlens ranges (InternEvo page "Data loading and flow", section
 *       "Fetching data from the Dataloader").
 *   group       = Hq / Hkv;  q head h reads kv head h / group
 *       (InternEvo page "Data loading and flow", section "Computing
 *       attention": qkv viewed as [.., num_kv_heads, group + 2, head_dim],
 *       q takes the first group slots of each kv head).
 *   S_ij        = scale * sum_c q[i,h,c] k[j,g,c]          for mask(i,j)
 *   LSE_i       = log sum_j exp(S_ij)                      (natural log)
 *   O_i         = sum_j exp(S_ij - LSE_i) v[j,g]
 *
 *   backward, with P_ij = exp(S_ij - LSE_i), dP_ij = dO_i . v_j,
 *   D_i = sum_j P_ij dP_ij (= dO_i . O_i):
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale sum_j dS_ij k_j
 *   dK_j  = scale sum_{h in g} sum_i dS_ij q_i
 *   dV_j  = sum_{h in g} sum_i P_ij dO_i
 *
 * Inputs are bf16 bit patterns (uint16), widened exactly to double. Layouts:
 * q / out / dout [T, Hq, d], k / v [T, Hkv, d], cu_seqlens int32 [nsegs + 1].
 * Every row has its diagonal, so no row is empty and no NaN policy is needed.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double widen(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q, *k, *v, *dout;
    const int32_t *cu;
    int32_t nsegs;
    int64_t T;
    int Hq, Hkv, d;
    double scale;
    int32_t *seg;   /* segment id of every token */
} problem;

static int setup(problem *p)
{
    if (p->Hq <= 0 || p->Hkv <= 0 || p->Hq % p->Hkv != 0 || p->d <= 0) return -1;
    if (p->cu[0] != 0 || p->cu[p->nsegs] != p->T) return -1;
    p->seg = (int32_t *)malloc(sizeof(int32_t) * (size_t)(p->T > 0 ? p->T : 1));
    if (!p->seg) return -1;
    for (int32_t s = 0; s < p->nsegs; ++s) {
        if (p->cu[s + 1] <= p->cu[s]) { free(p->seg); return -1; }
        for (int64_t i = p->cu[s]; i < p->cu[s + 1]; ++i) p->seg[i] = s;
    }
    return 0;
}

static int masked_in(const problem *p, int64_t i, int64_t j)
{
    return p->seg[i] == p->seg[j] && j <= i;
}

static double qk(const problem *p, int64_t i, int h, int64_t j, int g)
{
    const uint16_t *qi = p->q + ((size_t)i * p->Hq + h) * p->d;
    const uint16_t *kj = p->k + ((size_t)j * p->Hkv + g) * p->d;
    double acc = 0.0;
    for (int c = 0; c < p->d; ++c) acc += widen(qi[c]) * widen(kj[c]);
    return p->scale * acc;
}

static double dot_dout_v(const problem *p, int64_t i, int h, int64_t j, int g)
{
    const uint16_t *oi = p->dout + ((size_t)i * p->Hq + h) * p->d;
    const uint16_t *vj = p->v + ((size_t)j * p->Hkv + g) * p->d;
    double acc = 0.0;
    for (int c = 0; c < p->d; ++c) acc += widen(oi[c]) * widen(vj[c]);
    return acc;
}

/* One query row: fills s[] with S_ij over its segment (index j - a), returns
 * LSE_i and, if o != NULL, O_i. */
static double row_forward(const problem *p, int64_t i, int h, double *s, double *o)
{
    int g = h / (p->Hq / p->Hkv);
    int64_t a = p->cu[p->seg[i]], b = p->cu[p->seg[i] + 1];
    double m = -INFINITY;
    for (int64_t j = a; j < b; ++j) {
        if (!masked_in(p, i, j)) { s[j - a] = -INFINITY; continue; }
        s[j - a] = qk(p, i, h, j, g);
        if (s[j - a] > m) m = s[j - a];
    }
    double l = 0.0;
    for (int64_t j = a; j < b; ++j)
        if (masked_in(p, i, j)) l += exp(s[j - a] - m);
    double lse = m + log(l);
    if (o) {
        for (int c = 0; c < p->d; ++c) o[c] = 0.0;
        for (int64_t j = a; j < b; ++j) {
            if (!masked_in(p, i, j)) continue;
            double pij = exp(s[j - a] - lse);
            const uint16_t *vj = p->v + ((size_t)j * p->Hkv + g) * p->d;
            for (int c = 0; c < p->d; ++c) o[c] += pij * widen(vj[c]);
        }
    }
    return lse;
}

static int32_t max_seg_len(const problem *p)
{
    int32_t mx = 1;
    for (int32_t s = 0; s < p->nsegs; ++s)
        if (p->cu[s + 1] - p->cu[s] > mx) mx = p->cu[s + 1] - p->cu[s];
    return mx;
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/*
 * Forward for a list of (head, row) items, item = h * T + i; items == NULL
 * means every row of every head in [Hq, T] order. out [nitems, d], lse
 * [nitems]. Returns 0, or -1 on bad arguments.
 */
int spd_oracle_attn_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        const int32_t *cu, int32_t nsegs, int64_t T, int Hq, int Hkv,
                        int d, double scale, int64_t nitems, const int64_t *items,
                        double *out, double *lse, int nthreads)
{
    problem p = {q, k, v, NULL, cu, nsegs, T, Hq, Hkv, d, scale, NULL};
    if (setup(&p)) return -1;
    if (!items) nitems = (int64_t)Hq * T;
    int32_t L = max_seg_len(&p);
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        if (!s) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t it = 0; it < nitems; ++it) {
            if (!s) continue;
            int64_t key = items ? items[it] : it;
            int h = (int)(key / T);
            int64_t i = key % T;
            lse[it] = row_forward(&p, i, h, s, out + (size_t)it * d);
        }
        free(s);
    }
    free(p.seg);
    return err ? -1 : 0;
}

/* Row-side backward terms for one query row: LSE_i and D_i (through the exact
 * O_i) and, if dq != NULL, dQ_i. s and dp are scratch of the segment length. */
static void row_backward(const problem *p, int64_t i, int h, double *s, double *o,
                         double *lse_out, double *D_out, double *dq)
{
    int g = h / (p->Hq / p->Hkv);
    int64_t a = p->cu[p->seg[i]], b = p->cu[p->seg[i] + 1];
    double lse = row_forward(p, i, h, s, o);
    const uint16_t *doi = p->dout + ((size_t)i * p->Hq + h) * p->d;
    double D = 0.0;
    for (int c = 0; c < p->d; ++c) D += widen(doi[c]) * o[c];
    if (lse_out) *lse_out = lse;
    if (D_out) *D_out = D;
    if (!dq) return;
    for (int c = 0; c < p->d; ++c) dq[c] = 0.0;
    for (int64_t j = a; j < b; ++j) {
        if (!masked_in(p, i, j)) continue;
        double pij = exp(s[j - a] - lse);
        double ds = pij * (dot_dout_v(p, i, h, j, g) - D);
        const uint16_t *kj = p->k + ((size_t)j * p->Hkv + g) * p->d;
        for (int c = 0; c < p->d; ++c) dq[c] += p->scale * ds * widen(kj[c]);
    }
}

/*
 * dQ for a list of (head, row) items (item = h * T + i). dq [nitems, d].
 */
int spd_oracle_attn_dq_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const uint16_t *dout, const int32_t *cu, int32_t nsegs,
                            int64_t T, int Hq, int Hkv, int d, double scale,
                            int64_t nitems, const int64_t *items, double *dq, int nthreads)
{
    problem p = {q, k, v, dout, cu, nsegs, T, Hq, Hkv, d, scale, NULL};
    if (setup(&p)) return -1;
    int32_t L = max_seg_len(&p);
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !o) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t it = 0; it < nitems; ++it) {
            if (!s || !o) continue;
            int h = (int)(items[it] / T);
            int64_t i = items[it] % T;
            row_backward(&p, i, h, s, o, NULL, NULL, dq + (size_t)it * d);
        }
        free(s);
        free(o);
    }
    free(p.seg);
    return err ? -1 : 0;
}

/*
 * Full gradient over a list of whole segments (sel == NULL: all segments).
 * Outputs are compact: the rows of the selected segments, in list order,
 * dq [rows, Hq, d], dk / dv [rows, Hkv, d]. Two passes per segment: rows
 * (LSE_i, D_i, dQ_i), then columns (dK_j, dV_j summed over the group's heads
 * and over i). Both passes are parallel over independent rows.
 */
int spd_oracle_attn_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        const uint16_t *dout, const int32_t *cu, int32_t nsegs, int64_t T,
                        int Hq, int Hkv, int d, double scale, int32_t nsel,
                        const int32_t *sel, double *dq, double *dk, double *dv, int nthreads)
{
    problem p = {q, k, v, dout, cu, nsegs, T, Hq, Hkv, d, scale, NULL};
    if (setup(&p)) return -1;
    if (!sel) nsel = nsegs;
    int32_t L = max_seg_len(&p);
    int group = Hq / Hkv;
    set_threads(nthreads);
    double *lse = (double *)malloc(sizeof(double) * (size_t)L * Hq);
    double *D = (double *)malloc(sizeof(double) * (size_t)L * Hq);
    if (!lse || !D) { free(lse); free(D); free(p.seg); return -1; }
    int err = 0;
    int64_t base = 0;  /* first compact row of the current segment */
    for (int32_t si = 0; si < nsel; ++si) {
        int32_t s = sel ? sel[si] : si;
        if (s < 0 || s >= nsegs) { err = 1; break; }
        int64_t a = cu[s], b = cu[s + 1], n = b - a;
        /* pass 1: rows */
#pragma omp parallel
        {
            double *sc = (double *)malloc(sizeof(double) * (size_t)L);
            double *o = (double *)malloc(sizeof(double) * (size_t)d);
            if (!sc || !o) {
#pragma omp atomic write
                err = 1;
            }
#pragma omp for schedule(dynamic, 4) collapse(2)
            for (int h = 0; h < Hq; ++h)
                for (int64_t r = 0; r < n; ++r) {
                    if (!sc || !o) continue;
                    row_backward(&p, a + r, h, sc, o, &lse[(size_t)h * n + r],
                                 &D[(size_t)h * n + r],
                                 dq + ((size_t)(base + r) * Hq + h) * d);
                }
            free(sc);
            free(o);
        }
        /* pass 2: columns */
#pragma omp parallel for schedule(dynamic, 4) collapse(2)
        for (int g = 0; g < Hkv; ++g)
            for (int64_t c = 0; c < n; ++c) {
                int64_t j = a + c;
                double *dkj = dk + ((size_t)(base + c) * Hkv + g) * d;
                double *dvj = dv + ((size_t)(base + c) * Hkv + g) * d;
                for (int e = 0; e < d; ++e) { dkj[e] = 0.0; dvj[e] = 0.0; }
                for (int h = g * group; h < (g + 1) * group; ++h)
                    for (int64_t i = a; i < b; ++i) {
                        if (!masked_in(&p, i, j)) continue;
                        double pij = exp(qk(&p, i, h, j, g) - lse[(size_t)h * n + (i - a)]);
                        double ds = pij * (dot_dout_v(&p, i, h, j, g) - D[(size_t)h * n + (i - a)]);
                        const uint16_t *qi = q + ((size_t)i * Hq + h) * d;
                        const uint16_t *doi = dout + ((size_t)i * Hq + h) * d;
                        for (int e = 0; e < d; ++e) {
                            dkj[e] += scale * ds * widen(qi[e]);
                            dvj[e] += pij * widen(doi[e]);
                        }
                    }
            }
        base += n;
    }
    free(lse);
    free(D);
    free(p.seg);
    return err ? -1 : 0;
}
