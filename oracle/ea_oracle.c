/*
 * ea_oracle.c - plain, slow, fp64 CPU oracle for Elastic Attention's hybrid-head
 * attention path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path may link, load or call
 * this file; only the tests, the package's smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header, table or helper with the
 * CUDA library: it is written from the definitions on the pages, and every
 * function below cites the passage it follows.
 *
 * Sources (page titles as printed):
 *   [EN]  "Paper Reading - Elastic Attention: Test-time Adaptive Sparsity Ratios"
 *         (English reading notes)
 *   [ZH]  "论文精读 - Elastic Attention: 测试时自适应稀疏比的 Transformer 高效推理"
 *         (Chinese reading notes; the only page with eqs. 4-5 written out)
 *   [HA]  hyper.ai summary page "Elastic Attention" (arXiv 2601.17367)
 *
 * Conventions (readings of points the pages leave open):
 *   - scores are scale * <q, k> with scale given by the caller (1/sqrt(d));
 *   - every mode is causal (j <= i);
 *   - SSA (streaming sparse attention = attention sink + local window, [EN]
 *     Glossary "SSA"; sink/local sizes in [EN] §07 Table 8) keeps key j for query
 *     i iff j < sink or i - j < window, token-exact;
 *   - BLOCK keeps key j for query i iff the caller's 128x128 block mask entry
 *     [i/T][j/T] is non-zero ([EN] Glossary "XA", §04 Algorithm 1(b));
 *   - a row with no kept key has O = 0 and LSE = -inf;
 *   - inputs are bf16 bit patterns (uint16) converted exactly to double.
 *
 * Every floating point step is done in double, in the order the definition
 * states; no blocking, fusion or reordering.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_FULL 0
#define ORACLE_SSA 1
#define ORACLE_BLOCK 2

/* bf16 -> double: a bf16 value is the upper half of an IEEE binary32. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * The dense mask of one KV head: may query i attend to key j?
 * FA: plain causal attention, [EN] §02 eq. (1).
 * SA: attention over a reduced key set, [EN] §02 eq. (2), in its two forms:
 *     SSA (sink + window) and BLOCK (block mask).
 * Returns 1/0, or -1 for an unknown mode.
 */
static int oracle_allowed(int mode, int64_t i, int64_t j, int64_t sink, int64_t window,
                          const uint8_t *bm_head, int64_t nB, int64_t T)
{
    if (j > i)
        return 0;
    if (mode == ORACLE_FULL)
        return 1;
    if (mode == ORACLE_SSA)
        return (j < sink) || (i - j < window);
    if (mode == ORACLE_BLOCK)
        return bm_head[(i / T) * nB + (j / T)] != 0;
    return -1;
}

/*
 * One output row of the hybrid-head prefill.  [EN] §02 eqs. (1)-(3):
 *   s_j  = scale * sum_k q_k K[j,k]          for every kept key j
 *   p_j  = exp(s_j - max) / sum_l exp(s_l - max)
 *   O    = sum_j p_j V[j,:]
 *   LSE  = ln sum_j exp(s_j)
 * Query head qh reads KV head qh / (Hq/Hkv) (GQA grouping, [EN] §03 "every KV
 * head"), and its output lands in column block qh of O (eq. 3 concatenation).
 *
 * Q strides qs[4] and K/V strides kvs[4] are in elements over (b, s, h, dim).
 * rows[n][3] = (b, qh, i).  O is [n][d] doubles, LSE is [n].
 * Returns 0, or -1 on a bad argument or mode.
 */
int ea_oracle_prefill_rows(const uint16_t *Q, const int64_t *qs,
                           const uint16_t *K, const uint16_t *V, const int64_t *kvs,
                           int B, int S, int Hq, int Hkv, int d, double scale,
                           const uint8_t *modes, int sink, int window,
                           const uint8_t *block_mask, int T,
                           int64_t n_rows, const int64_t *rows,
                           double *O, double *LSE)
{
    if (B <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0 || T <= 0)
        return -1;
    const int64_t g = Hq / Hkv;
    const int64_t nB = ((int64_t)S + T - 1) / T;
    int bad = 0;

#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)S);
        char *keep = (char *)malloc((size_t)S);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r) {
            const int64_t b = rows[3 * r + 0], qh = rows[3 * r + 1], i = rows[3 * r + 2];
            double *o = O + r * d;
            if (b < 0 || b >= B || qh < 0 || qh >= Hq || i < 0 || i >= S || !s || !keep) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            const int64_t h = qh / g;
            const int mode = modes[b * Hkv + h];
            const uint8_t *bm = NULL;
            if (mode == ORACLE_BLOCK) {
                if (!block_mask) {
#pragma omp atomic write
                    bad = 1;
                    continue;
                }
                bm = block_mask + (b * Hkv + h) * nB * nB;
            }
            const uint16_t *q = Q + b * qs[0] + i * qs[1] + qh * qs[2];
            /* scores over the kept keys */
            double mx = -INFINITY;
            int any = 0;
            for (int64_t j = 0; j < S; ++j) {
                int a = oracle_allowed(mode, i, j, sink, window, bm, nB, T);
                if (a < 0) {
#pragma omp atomic write
                    bad = 1;
                    a = 0;
                }
                keep[j] = (char)a;
                if (!a)
                    continue;
                const uint16_t *k = K + b * kvs[0] + j * kvs[1] + h * kvs[2];
                double dot = 0.0;
                for (int c = 0; c < d; ++c)
                    dot += bf16_to_double(q[c * qs[3]]) * bf16_to_double(k[c * kvs[3]]);
                s[j] = scale * dot;
                if (s[j] > mx)
                    mx = s[j];
                any = 1;
            }
            for (int c = 0; c < d; ++c)
                o[c] = 0.0;
            if (!any) {
                LSE[r] = -INFINITY;
                continue;
            }
            /* softmax denominator */
            double denom = 0.0;
            for (int64_t j = 0; j < S; ++j)
                if (keep[j])
                    denom += exp(s[j] - mx);
            /* O = sum_j p_j V_j */
            for (int64_t j = 0; j < S; ++j) {
                if (!keep[j])
                    continue;
                const double p = exp(s[j] - mx) / denom;
                const uint16_t *v = V + b * kvs[0] + j * kvs[1] + h * kvs[2];
                for (int c = 0; c < d; ++c)
                    o[c] += p * bf16_to_double(v[c * kvs[3]]);
            }
            LSE[r] = mx + log(denom);
        }
        free(s);
        free(keep);
    }
    return bad ? -1 : 0;
}

/*
 * Decode: one new query per sequence attends to its cached keys [0, L), with
 * L = seqlens[b] (the cache already holds the current token).  The routing
 * decision made at prefill is reused ([EN] §08 Commentary, stated limit ③:
 * routing is decided once per request, at prefill).  The query is the
 * sequence's position L - 1 and keeps exactly the keys the prefill's row L - 1
 * keeps under the same mask (oracle_allowed above): FA every key; SSA
 * j < sink or (L-1) - j < window; BLOCK the keys of the blocks kept in row
 * (L-1) / T of the head's block mask, which covers nB = ceil(Lmax / T) blocks
 * and is reused across decode steps (the pages give no other decode reading).
 * A query with no kept key gets O = 0 and LSE = -inf.
 * q strides qs[3] over (b, h, dim); cache strides kvs[4] over (b, pos, h, dim).
 * block_mask: [B][Hkv][nB][nB] bytes, required if any mode is BLOCK.
 * O is [B][Hq][d] doubles, LSE is [B][Hq].
 */
int ea_oracle_decode(const uint16_t *q, const int64_t *qs,
                     const uint16_t *Kc, const uint16_t *Vc, const int64_t *kvs,
                     const int32_t *seqlens, int B, int Hq, int Hkv, int d, int Lmax,
                     double scale, const uint8_t *modes, int sink, int window,
                     const uint8_t *block_mask, int T, double *O, double *LSE)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0 || Lmax <= 0 || T <= 0)
        return -1;
    const int64_t nB = ((int64_t)Lmax + T - 1) / T;
    for (int b = 0; b < B; ++b) {
        if (seqlens[b] < 0 || seqlens[b] > Lmax)
            return -1;
        for (int h = 0; h < Hkv; ++h) {
            const int mode = modes[b * Hkv + h];
            if (mode == ORACLE_BLOCK && !block_mask)
                return -2;
            if (mode != ORACLE_FULL && mode != ORACLE_SSA && mode != ORACLE_BLOCK)
                return -1;
        }
    }
    const int64_t g = Hq / Hkv;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        for (int qh = 0; qh < Hq; ++qh) {
            const int64_t L = seqlens[b];
            const int64_t h = qh / g;
            const int mode = modes[b * Hkv + h];
            const uint16_t *qv = q + (int64_t)b * qs[0] + (int64_t)qh * qs[1];
            double *o = O + ((int64_t)b * Hq + qh) * d;
            for (int c = 0; c < d; ++c)
                o[c] = 0.0;
            double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
            double mx = -INFINITY;
            const uint8_t *bm = mode == ORACLE_BLOCK ? block_mask + ((int64_t)b * Hkv + h) * nB * nB
                                                     : NULL;
            for (int64_t j = 0; j < L; ++j) {
                const int keep = oracle_allowed(mode, L - 1, j, sink, window, bm, nB, T);
                if (!keep) {
                    s[j] = NAN;
                    continue;
                }
                const uint16_t *k = Kc + (int64_t)b * kvs[0] + j * kvs[1] + h * kvs[2];
                double dot = 0.0;
                for (int c = 0; c < d; ++c)
                    dot += bf16_to_double(qv[c * qs[2]]) * bf16_to_double(k[c * kvs[3]]);
                s[j] = scale * dot;
                if (s[j] > mx)
                    mx = s[j];
            }
            if (L == 0 || mx == -INFINITY) {
                LSE[(int64_t)b * Hq + qh] = -INFINITY;
                free(s);
                continue;
            }
            double denom = 0.0;
            for (int64_t j = 0; j < L; ++j)
                if (!isnan(s[j]))
                    denom += exp(s[j] - mx);
            for (int64_t j = 0; j < L; ++j) {
                if (isnan(s[j]))
                    continue;
                const double p = exp(s[j] - mx) / denom;
                const uint16_t *v = Vc + (int64_t)b * kvs[0] + j * kvs[1] + h * kvs[2];
                for (int c = 0; c < d; ++c)
                    o[c] += p * bf16_to_double(v[c * kvs[3]]);
            }
            LSE[(int64_t)b * Hq + qh] = mx + log(denom);
            free(s);
        }
    }
    return 0;
}

/*
 * Visited tiles: tile (qb, kb) of a KV head is visited iff at least one
 * (query, key) element inside it is kept by the dense mask above.  Brute force
 * over the elements (queries i < S only).  Covers q-block rows
 * [qb_begin, qb_end); vis is [B][Hkv][qb_end - qb_begin][nB] bytes (0/1).
 * This is the set of tiles a block-sparse kernel must touch ([EN] §04,
 * Algorithm 1(b): each head's branch over its own key blocks).
 */
int ea_oracle_visited(int B, int S, int Hkv, const uint8_t *modes, int sink, int window,
                      const uint8_t *block_mask, int T, int qb_begin, int qb_end, uint8_t *vis)
{
    const int64_t nB = ((int64_t)S + T - 1) / T;
    if (qb_begin < 0 || qb_end > nB || qb_begin > qb_end)
        return -1;
    const int64_t nq = qb_end - qb_begin;
    int bad = 0;
#pragma omp parallel for collapse(3) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hkv; ++h)
            for (int64_t qq = 0; qq < nq; ++qq) {
                const int64_t qb = qb_begin + qq;
                const int mode = modes[b * Hkv + h];
                const uint8_t *bm = NULL;
                if (mode == ORACLE_BLOCK) {
                    if (!block_mask) {
#pragma omp atomic write
                        bad = 1;
                        continue;
                    }
                    bm = block_mask + ((int64_t)b * Hkv + h) * nB * nB;
                }
                for (int64_t kb = 0; kb < nB; ++kb) {
                    int found = 0;
                    for (int64_t i = qb * T; i < (qb + 1) * T && i < S && !found; ++i)
                        for (int64_t j = kb * T; j < (kb + 1) * T && j < S && !found; ++j) {
                            const int a = oracle_allowed(mode, i, j, sink, window, bm, nB, T);
                            if (a < 0) {
#pragma omp atomic write
                                bad = 1;
                            }
                            found = a > 0;
                        }
                    vis[(((int64_t)b * Hkv + h) * nq + qq) * nB + kb] = (uint8_t)found;
                }
            }
    return bad ? -1 : 0;
}

/*
 * Attention Router, inference forward ([EN] §03 "Method: the Attention Router";
 * [ZH] §04 Method, "Router 怎么工作"):
 *   1. boundary pooling: mean of K over the first pool_head and the last
 *      pool_tail tokens of each KV head (100 + 100 on the pages); a token in both
 *      ranges (S < pool_head + pool_tail) is counted once;
 *   2. a stack of dense layers (dims[0] = d ... dims[n_layers] = 2) with ReLU
 *      between layers, weights shared across heads; logits z in R^{H x 2};
 *   3. hard routing r = argmax_c z_c ([EN] eq. 6), first maximum on a tie,
 *      0 = FA, 1 = SA; m = r ? sa_impl : fa_impl.
 * W_all / b_all hold the layers back to back, layer l as a dims[l+1] x dims[l]
 * row-major float matrix and a dims[l+1] vector.  All arithmetic in double.
 * K strides ks[4] over (b, s, h, dim).  logits [B][Hkv][2]; pooled (nullable)
 * [B][Hkv][d].
 */
int ea_oracle_route(const uint16_t *K, const int64_t *ks, int B, int S, int Hkv, int d,
                    int pool_head, int pool_tail, int n_layers, const int *dims,
                    const float *W_all, const float *b_all, int fa_impl, int sa_impl,
                    uint8_t *r, uint8_t *m, double *logits, double *pooled)
{
    if (B <= 0 || S <= 0 || Hkv <= 0 || d <= 0 || n_layers < 1 || dims[0] != d ||
        dims[n_layers] != 2 || pool_head < 0 || pool_tail < 0 || pool_head + pool_tail == 0)
        return -1;
    int maxw = 0;
    for (int l = 0; l <= n_layers; ++l) {
        if (dims[l] <= 0)
            return -1;
        if (dims[l] > maxw)
            maxw = dims[l];
    }
    const int64_t head_end = pool_head < S ? pool_head : S;
    const int64_t tail_begin = (S - pool_tail) > head_end ? (S - pool_tail) : head_end;
    const int64_t count = head_end + (S - tail_begin);

    double *x = (double *)malloc(sizeof(double) * (size_t)maxw);
    double *y = (double *)malloc(sizeof(double) * (size_t)maxw);
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hkv; ++h) {
            /* 1. boundary mean pooling */
            for (int c = 0; c < d; ++c)
                x[c] = 0.0;
            for (int64_t t = 0; t < S; ++t) {
                if (!(t < head_end || t >= tail_begin))
                    continue;
                const uint16_t *k = K + (int64_t)b * ks[0] + t * ks[1] + (int64_t)h * ks[2];
                for (int c = 0; c < d; ++c)
                    x[c] += bf16_to_double(k[c * ks[3]]);
            }
            for (int c = 0; c < d; ++c)
                x[c] /= (double)count;
            if (pooled)
                for (int c = 0; c < d; ++c)
                    pooled[((int64_t)b * Hkv + h) * d + c] = x[c];
            /* 2. dense layers, ReLU between them */
            const float *W = W_all;
            const float *bias = b_all;
            for (int l = 0; l < n_layers; ++l) {
                const int nin = dims[l], nout = dims[l + 1];
                for (int o = 0; o < nout; ++o) {
                    double acc = (double)bias[o];
                    for (int c = 0; c < nin; ++c)
                        acc += (double)W[(int64_t)o * nin + c] * x[c];
                    y[o] = acc;
                }
                if (l + 1 < n_layers)
                    for (int o = 0; o < nout; ++o)
                        y[o] = y[o] > 0.0 ? y[o] : 0.0;
                memcpy(x, y, sizeof(double) * (size_t)nout);
                W += (int64_t)nout * nin;
                bias += nout;
            }
            /* 3. hard routing */
            logits[((int64_t)b * Hkv + h) * 2 + 0] = x[0];
            logits[((int64_t)b * Hkv + h) * 2 + 1] = x[1];
            const int dec = x[1] > x[0] ? 1 : 0;
            r[b * Hkv + h] = (uint8_t)dec;
            m[b * Hkv + h] = (uint8_t)(dec ? sa_impl : fa_impl);
        }
    free(x);
    free(y);
    return 0;
}

/*
 * Sparsity ratios of one model over one input ([ZH] §02 eqs. (4)-(5); [EN] §02
 * "Two sparsity measures"):
 *   Omega_MSR = (1/(H L)) sum_{l,h} 1[pi(l,h) = SA]           (r[l][h] == 1)
 *   Omega_ESR = (1/(H L)) sum_{l,h} rho(l,h)
 * with rho = the share of causal (query, key) pairs the head prunes: 0 for a
 * head that keeps every causal pair, 0.9 when it keeps 10% ([ZH] §02 text under
 * eq. 5).  rho is taken from the mode m actually executed (a BLOCK head routed
 * to FA still prunes).  Pairs are counted by brute force over the dense mask;
 * because every head shares the same causal count, sum rho / (H L) equals the
 * single division (sum of pruned pairs) / (H L causal), which is what is
 * returned, so the result is the correctly rounded value of that rational.
 * block_masks: [L][Hkv][nB][nB] bytes, required if any m == BLOCK.
 * kept (nullable) receives the per-head kept-pair counts [L][Hkv].
 */
int ea_oracle_sparsity_ratios(const uint8_t *r, const uint8_t *m, int L, int Hkv, int S,
                              int sink, int window, const uint8_t *block_masks, int T,
                              double *msr, double *esr, int64_t *kept)
{
    if (L <= 0 || Hkv <= 0 || S <= 0 || T <= 0)
        return -1;
    const int64_t nB = ((int64_t)S + T - 1) / T;
    const int64_t causal = (int64_t)S * (S + 1) / 2;
    int64_t n_sa = 0, pruned_total = 0;
    int bad = 0;
    for (int l = 0; l < L; ++l)
        for (int h = 0; h < Hkv; ++h) {
            const int mode = m[l * Hkv + h];
            if (r[l * Hkv + h] > 1)
                return -1;
            n_sa += r[l * Hkv + h] == 1;
            const uint8_t *bm = NULL;
            if (mode == ORACLE_BLOCK) {
                if (!block_masks)
                    return -1;
                bm = block_masks + ((int64_t)l * Hkv + h) * nB * nB;
            }
            int64_t k = 0;
#pragma omp parallel for reduction(+ : k) schedule(dynamic, 64)
            for (int64_t i = 0; i < S; ++i)
                for (int64_t j = 0; j <= i; ++j) {
                    const int a = oracle_allowed(mode, i, j, sink, window, bm, nB, T);
                    if (a < 0) {
#pragma omp atomic write
                        bad = 1;
                    }
                    k += a > 0;
                }
            if (kept)
                kept[l * Hkv + h] = k;
            pruned_total += causal - k;
        }
    if (bad)
        return -1;
    *msr = (double)n_sa / ((double)L * (double)Hkv);
    *esr = (double)pruned_total / ((double)L * (double)Hkv * (double)causal);
    return 0;
}

/*
 * XA block scores of one (b, KV head): antidiagonal scoring.
 * The pages name XA as XAttention, a training-free block-sparse attention that
 * picks key blocks by antidiagonal scoring ([EN] Glossary "XA"; [ZH] glossary
 * "XA"), with stride 16 and threshold 0.9 ([EN] §07 Table 8, "stride/threshold
 * 16/0.9"; [HA] experiments, "XA, tau=0.9"), but do not write the scoring out.
 * This follows the plainest reading of those words:
 *   - the score matrix is cut into s x s cells (s = stride): cell (a, c) holds
 *     queries a*s .. a*s+s-1 and keys c*s .. c*s+s-1;
 *   - a cell's score is the mean of the scaled logits on its antidiagonal
 *     (query offset u pairs with key offset s-1-u):
 *       A[a][c] = (scale / s) * sum_{u<s} <q[a*s+u], k[c*s+s-1-u]>;
 *   - every downsampled query row a is normalised by a softmax over its causal
 *     cells c <= a:  P[a][c] = exp(A[a][c]) / sum_{c'<=a} exp(A[a][c']);
 *   - block (qb, kb) of the T x T block grid scores the sum of P over the cells
 *     inside it and over the query heads that read this KV head (the block mask
 *     is per KV head).
 * Tokens at or beyond S contribute nothing to a cell's sum; cell rows and
 * columns are the ceil(S/s) cells that hold at least one token.  T must be a
 * multiple of s.
 * W receives [nB][nB] (nB = ceil(S/T)), zero above the diagonal; when qb_sel
 * (bytes [nB]) is given, only the rows qb with qb_sel[qb] != 0 are computed and
 * the others stay zero.
 * Q strides qs[4] and K strides ks[4] are in elements over (b, s, h, dim).
 */
int ea_oracle_xa_block_scores(const uint16_t *Q, const int64_t *qs, const uint16_t *K,
                              const int64_t *ks, int S, int Hq, int Hkv, int d, double scale,
                              int stride, int T, int b, int h, const uint8_t *qb_sel, double *W)
{
    if (S <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || stride <= 0 || T <= 0 ||
        T % stride || h < 0 || h >= Hkv)
        return -1;
    const int g = Hq / Hkv;
    const int64_t s = stride;
    const int64_t nA = ((int64_t)S + s - 1) / s;
    const int64_t nB = ((int64_t)S + T - 1) / T;
    memset(W, 0, sizeof(double) * nB * nB);
    double *A = (double *)malloc(sizeof(double) * nA);
    if (!A)
        return -2;
    for (int qi = 0; qi < g; ++qi) {
        const int qh = h * g + qi;
        for (int64_t a = 0; a < nA; ++a) {
            if (qb_sel && !qb_sel[a * s / T])
                continue;
            /* antidiagonal means of row a, for every causal cell c <= a */
#pragma omp parallel for schedule(static)
            for (int64_t c = 0; c <= a; ++c) {
                double sum = 0.0;
                for (int64_t u = 0; u < s; ++u) {
                    const int64_t i = a * s + u, j = c * s + (s - 1 - u);
                    if (i >= S || j >= S)
                        continue;
                    const uint16_t *q = Q + b * qs[0] + i * qs[1] + qh * qs[2];
                    const uint16_t *k = K + b * ks[0] + j * ks[1] + h * ks[2];
                    double dot = 0.0;
                    for (int x = 0; x < d; ++x)
                        dot += bf16_to_double(q[x * qs[3]]) * bf16_to_double(k[x * ks[3]]);
                    sum += dot;
                }
                A[c] = scale * sum / (double)s;
            }
            /* softmax over c <= a */
            double mx = -INFINITY;
            for (int64_t c = 0; c <= a; ++c)
                if (A[c] > mx)
                    mx = A[c];
            double den = 0.0;
            for (int64_t c = 0; c <= a; ++c)
                den += exp(A[c] - mx);
            const int64_t qb = a * s / T;
            for (int64_t c = 0; c <= a; ++c)
                W[qb * nB + c * s / T] += exp(A[c] - mx) / den;
        }
    }
    free(A);
    return 0;
}

typedef struct {
    double w;
    int64_t kb;
} oracle_xa_entry;

/* Highest score first; equal scores by lower key block first. */
static int oracle_xa_cmp(const void *x, const void *y)
{
    const oracle_xa_entry *p = (const oracle_xa_entry *)x, *q = (const oracle_xa_entry *)y;
    if (p->w > q->w)
        return -1;
    if (p->w < q->w)
        return 1;
    return (p->kb > q->kb) - (p->kb < q->kb);
}

/*
 * XA threshold selection over the block scores of one head (same reading as
 * above; the threshold is [EN] §07 Table 8's 0.9): in every query-block row qb,
 * order the causal key blocks kb <= qb by score, highest first (ties: lower kb
 * first), and keep the shortest leading run whose scores add up to at least
 * tau times the row's total.  If rounding leaves every run short of that, every
 * block with a positive score is kept.  The diagonal block is always kept (every
 * query attends to its own key).
 * W: [nB][nB]; mask receives [nB][nB] bytes (1 = keep), zero above the diagonal;
 * when qb_sel (bytes [nB]) is given only the rows with qb_sel[qb] != 0 are
 * selected (the others stay zero).
 */
int ea_oracle_xa_select(const double *W, int64_t nB, double tau, const uint8_t *qb_sel,
                        uint8_t *mask)
{
    if (nB <= 0 || !(tau >= 0.0))
        return -1;
    oracle_xa_entry *e = (oracle_xa_entry *)malloc(sizeof(oracle_xa_entry) * nB);
    if (!e)
        return -2;
    memset(mask, 0, (size_t)(nB * nB));
    for (int64_t qb = 0; qb < nB; ++qb) {
        if (qb_sel && !qb_sel[qb])
            continue;
        const double *row = W + qb * nB;
        uint8_t *out = mask + qb * nB;
        double total = 0.0;
        for (int64_t kb = 0; kb <= qb; ++kb) {
            e[kb].w = row[kb];
            e[kb].kb = kb;
            total += row[kb];
        }
        qsort(e, (size_t)(qb + 1), sizeof(oracle_xa_entry), oracle_xa_cmp);
        const double target = tau * total;
        double run = 0.0;
        int64_t n = -1;
        for (int64_t k = 0; k <= qb; ++k) {
            if (run >= target) {
                n = k;
                break;
            }
            run += e[k].w;
        }
        if (n < 0 && run >= target)
            n = qb + 1;
        if (n < 0) {
            for (int64_t kb = 0; kb <= qb; ++kb)
                out[kb] = row[kb] > 0.0;
        } else {
            for (int64_t k = 0; k < n; ++k)
                out[e[k].kb] = 1;
        }
        out[qb] = 1;
    }
    free(e);
    return 0;
}
