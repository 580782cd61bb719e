/*
 * bss_oracle.c -- slow, plain, fp64 CPU oracle for block-sparse spatio-temporal
 * attention.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the product library never does.
 * It shares no code, header or table with the CUDA path.
 *
 * Source: "Accelerating Spatio-Temporal Attention for Video Diffusion on TPUs"
 * (Google Developers blog).  Each function names the passage it follows.
 *
 * Notation: F frames, S = Hs*Ws raster positions per frame, N = F*S tokens.
 *   frame-major (F,H,W) index     t = f*S + s
 *   temporal-major (H,W,F) index  p = s*F + f
 * Mask kinds:
 *   0  spatial, (F,H,W) layout
 *   1  temporal, (H,W,F) layout, keys in a "virtual" space
 *      [0, S_pad) sink segment (v < S is the frame-0 key at raster v),
 *      [S_pad, S_pad + N) band segment (v - S_pad is a permuted row)
 *   2  temporal, (F,H,W) layout (in-kernel indexing comparator)
 *   3  dense (every real pair retained)
 *
 * Everything is written from coordinates with div/mod, one pair at a time;
 * there is no interval arithmetic, tiling trick or fusion here.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_FULL 0
#define ORC_BOUNDARY 1
#define ORC_PAD 2
#define ORC_COLUMNS 3 /* kept tile of which some real columns are dropped (see orc_classify) */
#define ORC_SKIP 4

typedef struct {
    int64_t F, S, N;       /* frames, positions per frame, tokens */
    int64_t wf;            /* spatial head: |f_k - f_q| <= wf */
    int64_t ws;            /* temporal head: |s_k - s_q| <= ws */
    int64_t sink_frames;   /* frames [0, sink_frames) are an attention sink */
    int64_t S_pad;         /* kind 1: sink segment length (S rounded up to BKV) */
} orc_geom;

static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the parallel loops that follow (timing on fewer cores). */
void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Token permutation (F,H,W) -> (H,W,F): the blog's section "Arrange tokens for
 * efficient temporal access" and Figure 9.  Token t = f*S + s goes to p = s*F + f. */
int64_t orc_perm_index(int64_t t, int64_t F, int64_t S) {
    int64_t f = t / S, s = t % S;
    return s * F + f;
}

int64_t orc_unperm_index(int64_t p, int64_t F, int64_t S) {
    int64_t s = p / F, f = p % F;
    return f * S + s;
}

/* Per-head permutation of a [H][N][d] bf16 tensor, driven by per-head flags
 * (section "Support dynamic routing with fixed tensor shapes": flagged heads
 * switch layout, unflagged heads keep their order, shapes never change). */
void orc_permute(const uint16_t *in, uint16_t *out, int64_t H, int64_t F, int64_t S,
                 int64_t d, const uint8_t *flags, int inverse) {
    int64_t N = F * S;
    for (int64_t h = 0; h < H; ++h) {
        const uint16_t *src = in + h * N * d;
        uint16_t *dst = out + h * N * d;
        for (int64_t t = 0; t < N; ++t) {
            int64_t u = t;
            if (flags[h]) u = inverse ? orc_unperm_index(t, F, S) : orc_perm_index(t, F, S);
            /* forward: out[perm(t)] = in[t]; inverse: out[unperm(t)] = in[t] */
            for (int64_t c = 0; c < d; ++c) dst[u * d + c] = src[t * d + c];
        }
    }
}

static int64_t iabs64(int64_t x) { return x < 0 ? -x : x; }

/* Is virtual/layout column k a real key (not padding)? */
static int orc_col_real(int kind, const orc_geom *g, int64_t k) {
    if (k < 0) return 0;
    if (kind == 1) {
        if (k < g->S_pad) return k < g->S;
        return k - g->S_pad < g->N;
    }
    return k < g->N;
}

/* The retention predicate for query q (layout index) and key column k.
 *   spatial: keys in the same or nearby frames plus the first-frame sink
 *            (blog: spatial heads attend within close-by frames; Figure 3 left;
 *             both masks keep full attention to frame F00).
 *   temporal: keys at nearby raster positions across all frames plus the sink
 *            (blog: a small spatial region across many frames; Figure 3 right).
 * Reading: the temporal region is a band in the raster index s = h*W + w. */
int orc_retained(int kind, const orc_geom *g, int64_t q, int64_t k) {
    if (q < 0 || q >= g->N || !orc_col_real(kind, g, k)) return 0;
    switch (kind) {
    case 0: { /* spatial, (F,H,W) */
        int64_t fq = q / g->S, fk = k / g->S;
        return iabs64(fk - fq) <= g->wf || fk < g->sink_frames;
    }
    case 2: { /* temporal, (F,H,W) */
        int64_t sq = q % g->S, fk = k / g->S, sk = k % g->S;
        return iabs64(sk - sq) <= g->ws || fk < g->sink_frames;
    }
    case 1: { /* temporal, (H,W,F) with a sink segment in front of the band */
        int64_t sq = q / g->F;
        if (k < g->S_pad) {
            /* frame-0 key at raster k, kept here only when the band misses it */
            return iabs64(k - sq) > g->ws;
        }
        int64_t pk = k - g->S_pad;
        int64_t sk = pk / g->F;
        return iabs64(sk - sq) <= g->ws;
    }
    case 3:
        return 1;
    }
    return 0;
}

/* Map a key column to the physical row of the layout tensor it reads. */
static int64_t orc_key_row(int kind, const orc_geom *g, int64_t k) {
    if (kind == 1) return k < g->S_pad ? k * g->F : k - g->S_pad;
    return k;
}

int64_t orc_num_cols(int kind, const orc_geom *g) {
    return kind == 1 ? g->S_pad + g->N : g->N;
}

/* Tile classification (section "Logical sparsity is not physical sparsity":
 * full / boundary / skipped tiles; section "Align the sparse mask with final
 * execution": tile-aligned rounding, masking only for padding).  Brute force:
 * every pair of every tile in q-tile rows [qt0, qt1) is tested with
 * orc_retained.  Outputs per tile (row-major over [qt1-qt0][nkv]):
 *   counts[] = retained real pairs c, cls[] = ORC_* class.
 * Rules: exact     c == 0 -> SKIP; all columns real and c == real_rows*BKV
 *                  -> FULL; otherwise BOUNDARY.
 *        rounded   kept iff real_area > 0 and 2c >= real_area (reading of the
 *                  "balanced" rounding: at least half the tile is retained);
 *                  kept tiles with a padding column -> PAD, else FULL.
 *        naive     (mode 2, the blog's B1 naive traversal) c == 0 -> SKIP;
 *                  every visited tile -> BOUNDARY.
 * Rounded temporal (H,W,F) maps, kind 1: the rounded result is attention over
 * the SET of physical (query, key) pairs that the kept tiles cover.  In the
 * virtual key space the frame-0 key at raster v has two columns, sink column v
 * and band column S_pad + v*F (permuted row v*F), so a q tile can keep both.
 * The copy in the sink segment is then dropped: a kept sink tile loses every
 * real column whose band twin lies in a kept tile of the same q tile, and
 * becomes COLUMNS (some real columns left) or SKIP (none left). */
void orc_classify(int kind, const orc_geom *g, int64_t BQ, int64_t BKV, int rounding,
                  int64_t qt0, int64_t qt1, int64_t *counts, int8_t *cls) {
    int64_t ncols = orc_num_cols(kind, g);
    int64_t nkv = (ncols + BKV - 1) / BKV;
    int64_t ntiles = (qt1 - qt0) * nkv;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t idx = 0; idx < ntiles; ++idx) {
        int64_t I = qt0 + idx / nkv, J = idx % nkv;
        int64_t real_rows = 0, real_cols = 0, c = 0;
        for (int64_t q = I * BQ; q < (I + 1) * BQ; ++q) real_rows += (q < g->N);
        for (int64_t k = J * BKV; k < (J + 1) * BKV; ++k) real_cols += orc_col_real(kind, g, k);
        for (int64_t q = I * BQ; q < (I + 1) * BQ; ++q)
            for (int64_t k = J * BKV; k < (J + 1) * BKV; ++k) c += orc_retained(kind, g, q, k);
        int8_t cl;
        if (rounding == 2) {
            cl = c == 0 ? ORC_SKIP : ORC_BOUNDARY;
        } else if (!rounding) {
            if (c == 0) cl = ORC_SKIP;
            else if (real_cols == BKV && c == real_rows * BKV) cl = ORC_FULL;
            else cl = ORC_BOUNDARY;
        } else {
            int64_t area = real_rows * real_cols;
            if (area > 0 && 2 * c >= area) cl = (real_cols < BKV) ? ORC_PAD : ORC_FULL;
            else cl = ORC_SKIP;
        }
        counts[idx] = c;
        cls[idx] = cl;
    }
    if (kind == 1 && rounding == 1) {
        int64_t nsink = g->S_pad / BKV;
        for (int64_t I = qt0; I < qt1; ++I) {
            int8_t *row = cls + (I - qt0) * nkv;
            for (int64_t J = 0; J < nsink; ++J) {
                if (row[J] == ORC_SKIP) continue;
                int64_t real = 0, dropped = 0;
                for (int64_t v = J * BKV; v < (J + 1) * BKV && v < g->S; ++v) {
                    int64_t twin = g->S_pad + v * g->F; /* band column of the same key */
                    ++real;
                    if (row[twin / BKV] != ORC_SKIP) ++dropped;
                }
                if (dropped == real) row[J] = ORC_SKIP;
                else if (dropped > 0) row[J] = ORC_COLUMNS;
            }
        }
    }
}

/* Exact softmax attention for a list of query rows of ONE head, in fp64.
 * SoftMax(Q K^T * scale) V over the retained keys only; excluded pairs carry
 * zero weight (blog section "Logical sparsity is not physical sparsity": scores
 * of excluded pairs are set to -inf before the softmax).
 *   Q, K, V : [N][d] bf16 in the head's layout (already permuted for kind 1)
 *   rows    : layout query indices
 *   kept    : NULL for the exact mask, else per-tile keep flags for rounded
 *             masks, indexed [q_tile][kv_tile] over the whole map; the row
 *             then keeps every physical key that some real column of a kept
 *             tile reads, each key once (a set of pairs, not a multiset)
 *   O       : [nrows][d] fp64, lse : [nrows] fp64 (natural log)
 * A row with no retained key gets O = 0 and lse = -inf. */
void orc_attention(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int64_t d,
                   int kind, const orc_geom *g, double scale, const int8_t *kept,
                   int64_t BQ, int64_t BKV, const int64_t *rows, int64_t nrows,
                   double *O, double *lse) {
    int64_t ncols = orc_num_cols(kind, g);
    int64_t nkv = (ncols + BKV - 1) / BKV;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)ncols);
        int64_t *key = (int64_t *)malloc(sizeof(int64_t) * (size_t)ncols);
        double *q = (double *)malloc(sizeof(double) * (size_t)d);
        char *taken = (char *)calloc((size_t)(g->N > 0 ? g->N : 1), 1); /* physical key rows seen */
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            int64_t qi = rows[r];
            for (int64_t c = 0; c < d; ++c) q[c] = bf16_to_double(Q[qi * d + c]);
            int64_t n = 0;
            for (int64_t k = 0; k < ncols; ++k) {
                int keep;
                if (kept) {
                    keep = orc_col_real(kind, g, k) && kept[(qi / BQ) * nkv + k / BKV];
                } else {
                    keep = orc_retained(kind, g, qi, k);
                }
                if (!keep) continue;
                int64_t kr = orc_key_row(kind, g, k);
                if (taken[kr]) continue; /* the same key through another column */
                taken[kr] = 1;
                double acc = 0.0;
                for (int64_t c = 0; c < d; ++c) acc += q[c] * bf16_to_double(K[kr * d + c]);
                s[n] = acc * scale;
                key[n] = kr;
                ++n;
            }
            for (int64_t j = 0; j < n; ++j) taken[key[j]] = 0;
            double *o = O + r * d;
            for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
            if (n == 0) {
                lse[r] = -INFINITY;
                continue;
            }
            double m = s[0];
            for (int64_t j = 1; j < n; ++j) m = s[j] > m ? s[j] : m;
            double l = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                double w = exp(s[j] - m);
                l += w;
                const uint16_t *vr = V + key[j] * d;
                for (int64_t c = 0; c < d; ++c) o[c] += w * bf16_to_double(vr[c]);
            }
            for (int64_t c = 0; c < d; ++c) o[c] /= l;
            lse[r] = m + log(l);
        }
        free(s);
        free(key);
        free(q);
        free(taken);
    }
}
