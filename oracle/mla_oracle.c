/*
 * CPU oracle for DDTree verify attention, MLA in absorbed form.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, float64 statement
 * of what the verify path computes.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or helper with the CUDA library, and the CUDA library never calls it.
 *
 * What it computes (one query row = one draft-tree node i of sequence b, seen
 * through one head h):
 *
 *   visible(b, i) = { prefix positions 0 .. P_b-1 }
 *                 u { tree position P_b + t : node t is node i or one of its
 *                     ancestors in the draft tree }
 *   s_j   = scale * ( sum_{d<512} q_lat[b,i,h,d] * kv_c[slot_j, d]
 *                   + sum_{d<64}  q_pe [b,i,h,d] * k_pe[slot_j, d] )
 *   m     = max_j s_j ,  Z = sum_j exp(s_j - m)
 *   lse   = m + ln Z                                    (natural log)
 *   out_d = sum_j exp(s_j - m) / Z * kv_c[slot_j, d]    (d < 512)
 *
 * Sources: "Ground Truth in Silicon: The Role of the Python Reference in
 * Custom CUDA Kernel Development", section "The Message in Full" (the KV cache
 * holds a per-token latent kv_c of width 512 and a rope key k_pe of width 64,
 * shared across heads) and section "Input Knowledge Required ...", items 2
 * (absorbed query; latent shared by all heads) and 3 (softmax over the full
 * prefix plus the tree-structured tail under a custom visibility mask);
 * "Reading the Reference: How a Single File-Read Message Anchored a Complex
 * CUDA Kernel Implementation", section "Output Knowledge Created by This
 * Message" (mask = prefix visibility + tree-tail visibility).  The pages do
 * not print the formula; the readings taken here are: the scale multiplies
 * both score terms; the value vector is kv_c alone (width 512); lse is in
 * natural log; node t of the tree sits at logical position P_b + t; a parent
 * of -1 hangs the node directly off the prefix; a row with nothing visible
 * gets out = 0 and lse = -inf.
 *
 * Inputs are widened exactly to double (bf16 bit patterns, float32 or float64),
 * and every sum runs in double in position order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_DL 512
#define ORACLE_DR 64

enum { ORACLE_BF16 = 0, ORACLE_FP32 = 1, ORACLE_FP64 = 2 };

typedef struct {
    int B, Q, H;
    int dtype;                 /* element type of q_lat, q_pe, kv_c, k_pe */
    const void *q_lat;         /* [B][Q][H][512] */
    const void *q_pe;          /* [B][Q][H][64]  */
    const void *kv_c;          /* row r at element offset r * kv_c_stride */
    const void *k_pe;          /* row r at element offset r * k_pe_stride */
    int64_t kv_c_stride, k_pe_stride, pool_slots;
    int page_size;             /* 1: kv_indptr/kv_indices; >1: block_table */
    const int32_t *kv_indptr;  /* [B+1] */
    const int32_t *kv_indices; /* [kv_indptr[B]] */
    const int32_t *block_table;/* [B][max_pages] */
    int max_pages;
    const int32_t *prefix_lens;/* [B] */
    const int32_t *tree_parent;/* [B][Q] */
    double scale;
} oracle_problem;

static double elem(const void *base, int dtype, int64_t idx)
{
    if (dtype == ORACLE_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    if (dtype == ORACLE_FP32)
        return (double)((const float *)base)[idx];
    return ((const double *)base)[idx];
}

/* Ancestor-or-self bit sets of one tree: bit t of anc[i] is set when node t is
 * node i or an ancestor of it.  Nodes come in topological order, so a parent's
 * set is complete before its children read it.  Returns 0, or -1 when a parent
 * index is outside [-1, i-1] or the tree has more than 64 nodes. */
int oracle_tree_anc(int B, int Q, const int32_t *tree_parent, uint64_t *anc)
{
    if (Q < 0 || Q > 64)
        return -1;
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i < Q; ++i) {
            int p = tree_parent[(int64_t)b * Q + i];
            if (p < -1 || p >= i)
                return -1;
            uint64_t self = (uint64_t)1 << i;
            anc[(int64_t)b * Q + i] = (p < 0) ? self : (anc[(int64_t)b * Q + p] | self);
        }
    }
    return 0;
}

/* Pool slot of logical position p of sequence b; -1 if a table entry is out
 * of range. */
static int64_t slot_of(const oracle_problem *pr, int b, int64_t p)
{
    int64_t s;
    if (pr->page_size == 1) {
        s = pr->kv_indices[(int64_t)pr->kv_indptr[b] + p];
    } else {
        int64_t page_idx = p / pr->page_size;
        if (page_idx >= pr->max_pages)
            return -1;
        int64_t page = pr->block_table[(int64_t)b * pr->max_pages + page_idx];
        if (page < 0)
            return -1;
        s = page * pr->page_size + p % pr->page_size;
    }
    if (s < 0 || s >= pr->pool_slots)
        return -1;
    return s;
}

/* Every sequence's slots in position order, sequences back to back
 * (sum_b (P_b + Q) entries).  Returns that count, or -1 on a bad entry. */
int64_t oracle_resolve_slots(const oracle_problem *pr, int32_t *slots)
{
    int64_t k = 0;
    for (int b = 0; b < pr->B; ++b) {
        int64_t n = (int64_t)pr->prefix_lens[b] + pr->Q;
        if (pr->page_size == 1 && (int64_t)pr->kv_indptr[b + 1] - pr->kv_indptr[b] != n)
            return -1;
        for (int64_t p = 0; p < n; ++p) {
            int64_t s = slot_of(pr, b, p);
            if (s < 0)
                return -1;
            slots[k++] = (int32_t)s;
        }
    }
    return k;
}

/* Attention for a list of rows (b, i, h).  out: [n_rows][512], lse: [n_rows],
 * n_visible (may be NULL): [n_rows].  Returns 0, or -1 on bad input. */
int oracle_verify_rows(const oracle_problem *pr, int n_rows, const int32_t *rows,
                       double *out, double *lse, int64_t *n_visible)
{
    const int B = pr->B, Q = pr->Q, H = pr->H;
    if (Q > 64)
        return -1;
    uint64_t *anc = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(B * (int64_t)Q + 1));
    if (!anc)
        return -1;
    if (oracle_tree_anc(B, Q, pr->tree_parent, anc) != 0) {
        free(anc);
        return -1;
    }
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < n_rows; ++r) {
        const int b = rows[3 * r + 0], i = rows[3 * r + 1], h = rows[3 * r + 2];
        double *o = out + (int64_t)r * ORACLE_DL;
        for (int d = 0; d < ORACLE_DL; ++d)
            o[d] = 0.0;
        if (b < 0 || b >= B || i < 0 || i >= Q || h < 0 || h >= H) {
            /* written by several threads, only ever to 1 */
#pragma omp atomic write
            bad = 1;
            continue;
        }
        const int64_t P = pr->prefix_lens[b];
        const uint64_t mask = anc[(int64_t)b * Q + i];

        /* The visible positions, in increasing order. */
        int64_t nv = P;
        for (int t = 0; t < Q; ++t)
            if ((mask >> t) & 1)
                ++nv;
        int64_t *pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nv + 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(nv + 1));
        if (!pos || !s) {
            free(pos);
            free(s);
            /* written by several threads, only ever to 1 */
#pragma omp atomic write
            bad = 1;
            continue;
        }
        int64_t k = 0;
        for (int64_t p = 0; p < P; ++p)
            pos[k++] = p;
        for (int t = 0; t < Q; ++t)
            if ((mask >> t) & 1)
                pos[k++] = P + t;

        const int64_t qrow = ((int64_t)b * Q + i) * H + h;
        int row_bad = 0;

        /* Scores. */
        for (int64_t j = 0; j < nv; ++j) {
            int64_t slot = slot_of(pr, b, pos[j]);
            if (slot < 0) {
                row_bad = 1;
                break;
            }
            double dot_lat = 0.0, dot_pe = 0.0;
            for (int d = 0; d < ORACLE_DL; ++d)
                dot_lat += elem(pr->q_lat, pr->dtype, qrow * ORACLE_DL + d) *
                           elem(pr->kv_c, pr->dtype, slot * pr->kv_c_stride + d);
            for (int d = 0; d < ORACLE_DR; ++d)
                dot_pe += elem(pr->q_pe, pr->dtype, qrow * ORACLE_DR + d) *
                          elem(pr->k_pe, pr->dtype, slot * pr->k_pe_stride + d);
            s[j] = pr->scale * (dot_lat + dot_pe);
        }
        if (row_bad) {
            /* written by several threads, only ever to 1 */
#pragma omp atomic write
            bad = 1;
            free(pos);
            free(s);
            continue;
        }

        /* Softmax statistics. */
        double m = -INFINITY;
        for (int64_t j = 0; j < nv; ++j)
            if (s[j] > m)
                m = s[j];
        double Z = 0.0;
        for (int64_t j = 0; j < nv; ++j)
            Z += exp(s[j] - m);
        lse[r] = (nv > 0) ? m + log(Z) : -INFINITY;

        /* Weighted sum of the visible latent rows. */
        for (int64_t j = 0; j < nv; ++j) {
            const double w = exp(s[j] - m) / Z;
            const int64_t slot = slot_of(pr, b, pos[j]);
            for (int d = 0; d < ORACLE_DL; ++d)
                o[d] += w * elem(pr->kv_c, pr->dtype, slot * pr->kv_c_stride + d);
        }
        if (n_visible)
            n_visible[r] = nv;
        free(pos);
        free(s);
    }
    free(anc);
    return bad ? -1 : 0;
}

/* Threads an OpenMP region of this library will use. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
