/*
 * Parity oracle for the speculative-decoding verification step.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, fp64 CPU statement of
 * what the verification step computes.  It shares no code with the CUDA
 * library; only the test suite, the smoke check and the benchmark's CPU
 * baseline leg may load it.  The product path never calls it.
 *
 * Sources (web pages on speculative decoding):
 *  - "Co-Designing AI Models Using Speculative Decoding for Faster LLM
 *    Inference" (NVIDIA Technical Blog; Chinese translation), sections
 *    "What is speculative decoding" (AL in [1, 1+D]), "Draft length and
 *    performance of linear layers" (GEMM-M grows from M to M(1+D)) and
 *    "Draft length and attention performance" (drafts reuse the KV cache,
 *    attention GEMM-M = G(1+D)).
 *  - "How does speculative decoding speed up LLM inference?" (llm-digest),
 *    sections "Mechanism" and "Math intuition": accept x with probability
 *    min(1, p(x)/q(x)); at the first rejection resample from
 *    max(0, p - q) renormalised.
 *  - LLM inference handbook, "Speculative decoding", section "How
 *    speculative decoding works": accept the longest agreeing prefix, then
 *    emit one more token from the target.
 *
 * Readings where the pages are silent (each restated where it is used):
 *  R1 kv_len[b] counts the 1+D verify tokens; query row i sees keys
 *     j < kv_len[b] - D + i (drafts see the prefix, earlier drafts and
 *     themselves).  D = 0 is plain decode over kv_len[b] keys.
 *  R2 softmax scale is a caller argument (1/sqrt(head_dim) by default).
 *  R3 accept test is strict u * q(x) < p(x), evaluated exactly.
 *  R4 residual/bonus draw: smallest v (ascending id) with C(v) > u * Z where
 *     C is the running sum and Z the total.
 *  R5 if Z <= 0 after a rejection, draw from p of that row instead.
 *  R6 greedy ties resolve to the lowest index.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static void set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------
 * Verify attention, one query row.
 *
 * Row (b, i, h, g): query head hq = h*G + g, draft position i in [0, D].
 * Visible keys j in [0, kv_len[b] - D + i) (reading R1).  With fp64 scores
 * s_j = scale * sum_c q_c K_jc, m = max_j s_j, w_j = exp(s_j - m):
 *   o = sum_j w_j V_j / sum_j w_j,   lse = m + ln(sum_j w_j).
 * Key j of sequence b lives in page block_table[b][j / page_size] at slot
 * j % page_size.  Returns 0, or -1 if a page id is outside [0, num_pages).
 * ---------------------------------------------------------------------- */
static int attention_row(const uint16_t *q, const uint16_t *kp, const uint16_t *vp,
                         const int32_t *block_table, int max_pages, const int32_t *kv_len,
                         int D, int Hkv, int G, int d, int page_size, double scale,
                         int64_t num_pages, int b, int i, int h, int g,
                         double *out, double *lse, double *scratch)
{
    const int Hq = Hkv * G;
    const uint16_t *qrow = q + (((int64_t)b * (1 + D) + i) * Hq + (int64_t)h * G + g) * d;
    const int64_t n_keys = (int64_t)kv_len[b] - D + i;
    double m = -INFINITY;
    for (int64_t j = 0; j < n_keys; ++j) {
        int32_t page = block_table[(int64_t)b * max_pages + j / page_size];
        if (page < 0 || page >= num_pages) return -1;
        const uint16_t *krow = kp + (((int64_t)page * page_size + j % page_size) * Hkv + h) * d;
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += bf16_to_f64(qrow[c]) * bf16_to_f64(krow[c]);
        s *= scale;
        scratch[j] = s;
        if (s > m) m = s;
    }
    double l = 0.0;
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
        int32_t page = block_table[(int64_t)b * max_pages + j / page_size];
        const uint16_t *vrow = vp + (((int64_t)page * page_size + j % page_size) * Hkv + h) * d;
        double w = exp(scratch[j] - m);
        l += w;
        for (int c = 0; c < d; ++c) out[c] += w * bf16_to_f64(vrow[c]);
    }
    for (int c = 0; c < d; ++c) out[c] /= l;
    if (lse) *lse = m + log(l);
    return 0;
}

/* rows == NULL: every row, out laid out [B][1+D][Hq][d], lse [B][1+D][Hq].
 * rows != NULL: n_rows entries (b, i, h, g); out [n_rows][d], lse [n_rows]. */
int oracle_verify_attention(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                            const int32_t *block_table, int max_pages_per_seq,
                            const int32_t *kv_len, int B, int D, int Hkv, int G,
                            int head_dim, int page_size, double softmax_scale,
                            int64_t num_pages, int n_rows, const int32_t *rows,
                            double *out, double *lse, int num_threads)
{
    if (B < 0 || D < 0 || Hkv < 1 || G < 1 || head_dim < 1 || page_size < 1) return -2;
    for (int b = 0; b < B; ++b)
        if (kv_len[b] < 1 + D || (int64_t)kv_len[b] > (int64_t)max_pages_per_seq * page_size)
            return -3;
    const int Hq = Hkv * G;
    const int64_t total = rows ? (int64_t)n_rows : (int64_t)B * (1 + D) * Hq;
    int64_t max_len = 1;
    for (int b = 0; b < B; ++b) if (kv_len[b] > max_len) max_len = kv_len[b];
    int err = 0;
    set_threads(num_threads);
#pragma omp parallel
    {
        double *scratch = (double *)malloc(sizeof(double) * (size_t)max_len);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < total; ++r) {
            int b, i, h, g;
            if (rows) {
                b = rows[4 * r]; i = rows[4 * r + 1]; h = rows[4 * r + 2]; g = rows[4 * r + 3];
            } else {
                int64_t t = r;
                g = (int)(t % G); t /= G;
                h = (int)(t % Hkv); t /= Hkv;
                i = (int)(t % (1 + D)); t /= (1 + D);
                b = (int)t;
            }
            int rc = attention_row(q, k_pages, v_pages, block_table, max_pages_per_seq, kv_len,
                                   D, Hkv, G, head_dim, page_size, softmax_scale, num_pages,
                                   b, i, h, g, out + r * head_dim, lse ? lse + r : NULL, scratch);
            if (rc) {
#pragma omp atomic write
                err = rc;
            }
        }
        free(scratch);
    }
    return err;
}

/* ------------------------------------------------------------------------
 * Verify GEMM: y[m][n] = sum_k x[m][k] * w[n][k] in fp64, x [M][K] and
 * w [N][K] bf16 (both K-contiguous).  GEMM-M = B(1+D) is the batch of
 * verified tokens.  samples == NULL: full y [M][N]; else y[s] for the n
 * pairs (m, n) in samples.
 * ---------------------------------------------------------------------- */
int oracle_gemm(const uint16_t *x, const uint16_t *w, int M, int N, int K,
                int n_samples, const int32_t *samples, double *y, int num_threads)
{
    if (M < 0 || N < 0 || K < 0) return -2;
    const int64_t total = samples ? (int64_t)n_samples : (int64_t)M * N;
    set_threads(num_threads);
#pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < total; ++s) {
        int m, n;
        if (samples) { m = samples[2 * s]; n = samples[2 * s + 1]; }
        else { m = (int)(s / N); n = (int)(s % N); }
        const uint16_t *xr = x + (int64_t)m * K;
        const uint16_t *wr = w + (int64_t)n * K;
        double acc = 0.0;
        for (int k = 0; k < K; ++k) acc += bf16_to_f64(xr[k]) * bf16_to_f64(wr[k]);
        y[s] = acc;
    }
    return 0;
}

/* Lowest index of the maximum of row[0..V) (reading R6). */
static int argmax_row(const float *row, int V)
{
    int best = 0;
    double bv = (double)row[0];
    for (int v = 1; v < V; ++v) {
        double x = (double)row[v];
        if (x > bv) { bv = x; best = v; }
    }
    return best;
}

/* ------------------------------------------------------------------------
 * Greedy acceptance.  Target token t_i = argmax_v p[b][i][v].  Drafts are
 * accepted in order until the first i with draft[b][i] != t_i; n_acc = that
 * i (or D if all match); the emitted extra token is t_{n_acc}.  Accepted
 * length AL = n_acc + 1 lies in [1, 1+D].
 * ---------------------------------------------------------------------- */
int oracle_accept_greedy(const float *p, const int32_t *draft, int B, int D, int V,
                         int32_t *n_accepted, int32_t *token, int num_threads)
{
    if (B < 0 || D < 0 || V < 1) return -2;
    set_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        const float *pb = p + (int64_t)b * (1 + D) * V;
        int n = D;
        for (int i = 0; i < D; ++i) {
            if (draft[(int64_t)b * D + i] != argmax_row(pb + (int64_t)i * V, V)) { n = i; break; }
        }
        n_accepted[b] = n;
        token[b] = argmax_row(pb + (int64_t)n * V, V);
    }
    return 0;
}

/* Draw from weights r (computed on the fly): smallest v with C(v) > u * Z,
 * C the ascending running sum, Z = C(V-1) (reading R4).  Also returns the
 * boundary margin min_v |u*Z - C(v)| / Z.  kind 0: r = p; kind 1:
 * r = max(0, p - q).  Returns -1 if Z <= 0. */
static int draw_residual(const float *p, const float *q, int V, int kind, double u,
                         double *margin)
{
    double Z = 0.0;
    for (int v = 0; v < V; ++v) {
        double r = kind ? fmax(0.0, (double)p[v] - (double)q[v]) : (double)p[v];
        Z += r;
    }
    if (!(Z > 0.0)) return -1;
    const double T = u * Z;
    double C = 0.0, mg = INFINITY;
    int pick = -1;
    for (int v = 0; v < V; ++v) {
        double r = kind ? fmax(0.0, (double)p[v] - (double)q[v]) : (double)p[v];
        C += r;
        double gap = fabs(T - C);
        if (gap < mg) mg = gap;
        if (pick < 0 && C > T) pick = v;
    }
    if (pick < 0) { /* rounding left T >= Z: take the last token with mass */
        for (int v = V - 1; v >= 0; --v) {
            double r = kind ? fmax(0.0, (double)p[v] - (double)q[v]) : (double)p[v];
            if (r > 0.0) { pick = v; break; }
        }
    }
    if (margin) *margin = mg / Z;
    return pick;
}

/* ------------------------------------------------------------------------
 * Stochastic acceptance (modified rejection sampling).  For i = 0..D-1 with
 * x = draft[b][i]: accept iff u_acc[b][i] * q[b][i][x] < p[b][i][x] (reading
 * R3; the fp32 inputs make the fp64 product exact).  At the first
 * rejection j, emit a draw from max(0, p[b][j] - q[b][j]) renormalised with
 * uniform u_res[b]; if none is rejected, emit a draw from p[b][D] (the bonus
 * token).  n_acc = j (or D).  Outputs per sequence: n_accepted, token, the
 * boundary margin (min over the accept tests of |u - p/q| and over the draw
 * of the CDF gap / Z) and a flag set when reading R5's fallback was taken.
 * ---------------------------------------------------------------------- */
int oracle_accept_sample(const float *p, const float *q, const int32_t *draft,
                         const float *u_acc, const float *u_res, int B, int D, int V,
                         int32_t *n_accepted, int32_t *token, double *margin,
                         int32_t *fallback, int num_threads)
{
    if (B < 0 || D < 0 || V < 1) return -2;
    int err = 0;
    set_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        const float *pb = p + (int64_t)b * (1 + D) * V;
        const float *qb = q + (int64_t)b * D * V;
        double mg = INFINITY;
        int j = D;
        for (int i = 0; i < D; ++i) {
            int x = draft[(int64_t)b * D + i];
            if (x < 0 || x >= V) {
#pragma omp atomic write
                err = -4;
                x = 0;
            }
            double px = (double)pb[(int64_t)i * V + x];
            double qx = (double)qb[(int64_t)i * V + x];
            double u = (double)u_acc[(int64_t)b * D + i];
            if (qx > 0.0) {
                double gap = fabs(u - px / qx);
                if (gap < mg) mg = gap;
            }
            if (!(u * qx < px)) { j = i; break; }
        }
        int fb = 0, tok;
        double dm = INFINITY;
        if (j < D) {
            tok = draw_residual(pb + (int64_t)j * V, qb + (int64_t)j * V, V, 1,
                                (double)u_res[b], &dm);
            if (tok < 0) {
                fb = 1;
                tok = draw_residual(pb + (int64_t)j * V, NULL, V, 0, (double)u_res[b], &dm);
            }
        } else {
            tok = draw_residual(pb + (int64_t)D * V, NULL, V, 0, (double)u_res[b], &dm);
        }
        if (tok < 0) { tok = 0; }
        if (dm < mg) mg = dm;
        n_accepted[b] = j;
        token[b] = tok;
        if (margin) margin[b] = mg;
        if (fallback) fallback[b] = fb;
    }
    return err;
}

/* ------------------------------------------------------------------------
 * Tree verification (Medusa / EAGLE-2 style draft trees).
 *
 * Candidate continuations form a tree that the target scores in one pass,
 * with an attention mask keeping every branch causal; the longest accepted
 * candidate prefix is carried into the next step (LLM inference handbook,
 * "Speculative decoding", section on Medusa; EAGLE-2's dynamic draft tree
 * in the same section).
 *
 * The tree of sequence b has T = 1 + D nodes in topological order:
 * parent[b][0] = -1 (node 0 is the last accepted token, the root) and
 * 0 <= parent[b][k] < k for k >= 1.  Node k's K/V occupy cache position
 * kv_len[b] - T + k.
 *  R7 node k's query attends to the prefix keys j < kv_len[b] - T and to
 *     the tree keys of the nodes on its root-to-k path (its ancestors and
 *     itself).  A chain (parent[k] = k - 1) is reading R1.
 *  R8 greedy tree acceptance: from the root, repeatedly move to the child
 *     whose token equals the target argmax at the current node (the lowest
 *     node index if several siblings carry it); stop when no child matches.
 *     n_acc = the depth reached, the emitted token is the argmax at the
 *     last node, and the path lists the accepted nodes in order.  A chain
 *     whose node k carries draft k-1 is the greedy acceptance above.
 *  R12 stochastic tree acceptance: see oracle_accept_tree_sample.
 * ---------------------------------------------------------------------- */

/* Whether parent[0..T) is a valid tree in topological order. */
static int tree_valid(const int32_t *parent, int T)
{
    if (T < 1 || parent[0] != -1) return 0;
    for (int k = 1; k < T; ++k)
        if (parent[k] < 0 || parent[k] >= k) return 0;
    return 1;
}

static int tree_attention_row(const uint16_t *q, const uint16_t *kp, const uint16_t *vp,
                              const int32_t *block_table, int max_pages, const int32_t *kv_len,
                              const int32_t *parent, int D, int Hkv, int G, int d, int page_size,
                              double scale, int64_t num_pages, int b, int k, int h, int g,
                              double *out, double *lse, double *scratch, int64_t *keys)
{
    const int T = 1 + D, Hq = Hkv * G;
    const int32_t *par = parent + (int64_t)b * T;
    const int64_t P = (int64_t)kv_len[b] - T;   /* prefix keys */
    /* visible keys, ascending: the prefix, then the tree path root..k */
    int onpath[64];
    for (int a = 0; a < T; ++a) onpath[a] = 0;
    for (int a = k; a >= 0; a = par[a]) onpath[a] = 1;
    int64_t n = 0;
    for (int64_t j = 0; j < P; ++j) keys[n++] = j;
    for (int a = 0; a < T; ++a) if (onpath[a]) keys[n++] = P + a;
    const uint16_t *qrow = q + (((int64_t)b * T + k) * Hq + (int64_t)h * G + g) * d;
    double m = -INFINITY;
    for (int64_t x = 0; x < n; ++x) {
        const int64_t j = keys[x];
        int32_t page = block_table[(int64_t)b * max_pages + j / page_size];
        if (page < 0 || page >= num_pages) return -1;
        const uint16_t *krow = kp + (((int64_t)page * page_size + j % page_size) * Hkv + h) * d;
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += bf16_to_f64(qrow[c]) * bf16_to_f64(krow[c]);
        s *= scale;
        scratch[x] = s;
        if (s > m) m = s;
    }
    double l = 0.0;
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    for (int64_t x = 0; x < n; ++x) {
        const int64_t j = keys[x];
        int32_t page = block_table[(int64_t)b * max_pages + j / page_size];
        const uint16_t *vrow = vp + (((int64_t)page * page_size + j % page_size) * Hkv + h) * d;
        double w = exp(scratch[x] - m);
        l += w;
        for (int c = 0; c < d; ++c) out[c] += w * bf16_to_f64(vrow[c]);
    }
    for (int c = 0; c < d; ++c) out[c] /= l;
    if (lse) *lse = m + log(l);
    return 0;
}

/* Tree verify attention; arguments as oracle_verify_attention plus
 * parent [B][1+D] (1 + D <= 64).  Returns -4 for an invalid tree. */
int oracle_tree_attention(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                          const int32_t *block_table, int max_pages_per_seq,
                          const int32_t *kv_len, const int32_t *parent, int B, int D, int Hkv,
                          int G, int head_dim, int page_size, double softmax_scale,
                          int64_t num_pages, int n_rows, const int32_t *rows, double *out,
                          double *lse, int num_threads)
{
    if (B < 0 || D < 0 || D > 63 || Hkv < 1 || G < 1 || head_dim < 1 || page_size < 1) return -2;
    for (int b = 0; b < B; ++b) {
        if (kv_len[b] < 1 + D || (int64_t)kv_len[b] > (int64_t)max_pages_per_seq * page_size)
            return -3;
        if (!tree_valid(parent + (int64_t)b * (1 + D), 1 + D)) return -4;
    }
    const int Hq = Hkv * G;
    const int64_t total = rows ? (int64_t)n_rows : (int64_t)B * (1 + D) * Hq;
    int64_t max_len = 1;
    for (int b = 0; b < B; ++b) if (kv_len[b] > max_len) max_len = kv_len[b];
    int err = 0;
    set_threads(num_threads);
#pragma omp parallel
    {
        double *scratch = (double *)malloc(sizeof(double) * (size_t)max_len);
        int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)max_len);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < total; ++r) {
            int b, k, h, g;
            if (rows) {
                b = rows[4 * r]; k = rows[4 * r + 1]; h = rows[4 * r + 2]; g = rows[4 * r + 3];
            } else {
                int64_t t = r;
                g = (int)(t % G); t /= G;
                h = (int)(t % Hkv); t /= Hkv;
                k = (int)(t % (1 + D)); t /= (1 + D);
                b = (int)t;
            }
            int rc = tree_attention_row(q, k_pages, v_pages, block_table, max_pages_per_seq,
                                        kv_len, parent, D, Hkv, G, head_dim, page_size,
                                        softmax_scale, num_pages, b, k, h, g,
                                        out + r * head_dim, lse ? lse + r : NULL, scratch, keys);
            if (rc) {
#pragma omp atomic write
                err = rc;
            }
        }
        free(scratch);
        free(keys);
    }
    return err;
}

/* Greedy tree acceptance (reading R8).  p [B][1+D][V] target probabilities
 * at every node, tokens [B][1+D] the node tokens (node 0's is unused),
 * parent [B][1+D].  Outputs n_accepted [B], token [B] and path [B][D]
 * (accepted node ids in order, -1 after the last).  Returns -4 for an
 * invalid tree. */
int oracle_accept_tree_greedy(const float *p, const int32_t *tokens, const int32_t *parent, int B,
                              int D, int V, int32_t *n_accepted, int32_t *token, int32_t *path,
                              int num_threads)
{
    if (B < 0 || D < 0 || D > 63 || V < 1) return -2;
    for (int b = 0; b < B; ++b)
        if (!tree_valid(parent + (int64_t)b * (1 + D), 1 + D)) return -4;
    set_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        const int T = 1 + D;
        const float *pb = p + (int64_t)b * T * V;
        const int32_t *par = parent + (int64_t)b * T, *tok = tokens + (int64_t)b * T;
        for (int x = 0; x < D; ++x) path[(int64_t)b * D + x] = -1;
        int cur = 0, depth = 0, t;
        for (;;) {
            t = argmax_row(pb + (int64_t)cur * V, V);
            int next = -1;
            for (int c = cur + 1; c < T; ++c)
                if (par[c] == cur && tok[c] == t) { next = c; break; }
            if (next < 0) break;
            path[(int64_t)b * D + depth] = next;
            ++depth;
            cur = next;
        }
        n_accepted[b] = depth;
        token[b] = t;
    }
    return 0;
}

/* Stochastic tree acceptance (reading R12).  The children of node k (the
 * nodes whose parent is k, in increasing index) carry tokens drafted from
 * q[b][k].  From the root, at the current node v the working row r starts
 * as p[b][v]; child c with token x is accepted iff u_acc[b][c] * q[b][v][x]
 * < r(x) (the walk then moves to c), otherwise r becomes max(0, r -
 * q[b][v]) divided by its sum (left unchanged, and flagged, when that sum is
 * 0) and the next child is tried.  When no child of v is accepted, or v has
 * none, the token is drawn from r with u_res[b]: the smallest v with
 * sum_{w <= v} r(w) > u_res[b] * sum_w r(w).  For a chain whose node k
 * carries draft k - 1 this is the stochastic acceptance above.
 * p, q [B][1+D][V] (q's rows of leaves are not read), tokens, parent,
 * u_acc [B][1+D] (entry 0 unused), u_res [B].  Outputs n_accepted (the
 * depth reached), token, path [B][D] (accepted nodes, -1 after the last),
 * margin (min over the tests of |u - r(x)/q(x)| and over the draw of the
 * CDF gap / sum r) and flag (1 when an empty residual was left as it
 * was).  Returns -4 for an invalid tree or token. */
static int draw_row_f64(const double *r, int V, double u, double *margin)
{
    double Z = 0.0;
    for (int v = 0; v < V; ++v) Z += r[v];
    if (!(Z > 0.0)) return -1;
    const double T = u * Z;
    double C = 0.0, mg = INFINITY;
    int pick = -1;
    for (int v = 0; v < V; ++v) {
        C += r[v];
        const double gap = fabs(T - C);
        if (gap < mg) mg = gap;
        if (pick < 0 && C > T) pick = v;
    }
    if (pick < 0)
        for (int v = V - 1; v >= 0; --v)
            if (r[v] > 0.0) { pick = v; break; }
    if (margin) *margin = mg / Z;
    return pick;
}

int oracle_accept_tree_sample(const float *p, const float *q, const int32_t *tokens, const int32_t *parent,
                              const float *u_acc, const float *u_res, int B, int D, int V,
                              int32_t *n_accepted, int32_t *token, int32_t *path, double *margin,
                              int32_t *flag, int num_threads)
{
    if (B < 0 || D < 0 || D > 63 || V < 1) return -2;
    const int T = 1 + D;
    for (int b = 0; b < B; ++b) {
        if (!tree_valid(parent + (int64_t)b * T, T)) return -4;
        for (int k = 1; k < T; ++k) {
            const int32_t x = tokens[(int64_t)b * T + k];
            if (x < 0 || x >= V) return -4;
        }
    }
    int err = 0;
    set_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        const float *pb = p + (int64_t)b * T * V, *qb = q + (int64_t)b * T * V;
        const int32_t *par = parent + (int64_t)b * T, *tok = tokens + (int64_t)b * T;
        double *r = (double *)malloc((size_t)V * sizeof(double));
        if (!r) {
#pragma omp atomic write
            err = -3;
            continue;
        }
        for (int x = 0; x < D; ++x) path[(int64_t)b * D + x] = -1;
        int cur = 0, depth = 0, fl = 0;
        double mg = INFINITY;
        for (;;) {
            const float *pv = pb + (int64_t)cur * V, *qv = qb + (int64_t)cur * V;
            for (int v = 0; v < V; ++v) r[v] = (double)pv[v];
            int next = -1;
            for (int c = cur + 1; c < T && next < 0; ++c) {
                if (par[c] != cur) continue;
                const int x = tok[c];
                const double u = (double)u_acc[(int64_t)b * T + c];
                const double qx = (double)qv[x];
                if (qx > 0.0) {
                    const double gap = fabs(u - r[x] / qx);
                    if (gap < mg) mg = gap;
                }
                if (u * qx < r[x]) { next = c; break; }
                double Z = 0.0;
                for (int v = 0; v < V; ++v) Z += fmax(0.0, r[v] - (double)qv[v]);
                if (Z > 0.0) {
                    for (int v = 0; v < V; ++v) r[v] = fmax(0.0, r[v] - (double)qv[v]) / Z;
                } else {
                    fl = 1;
                }
            }
            if (next < 0) break;
            path[(int64_t)b * D + depth] = next;
            ++depth;
            cur = next;
        }
        double dm = INFINITY;
        int t = draw_row_f64(r, V, (double)u_res[b], &dm);
        if (t < 0) t = 0;
        if (dm < mg) mg = dm;
        n_accepted[b] = depth;
        token[b] = t;
        if (margin) margin[b] = mg;
        if (flag) flag[b] = fl;
        free(r);
    }
    return err;
}

/* ------------------------------------------------------------------------
 * Acceptance from logits (the fused form of the stochastic acceptance).
 *
 * The acceptance of the llm-digest page ("Mechanism": x is kept with
 * probability min(1, p(x)/q(x))) with p = softmax(target logits / T),
 * q = softmax(draft logits / T), and the uniforms drawn by Philox4x32-10
 * from a seed.
 *  R9  one temperature T > 0 for both models.
 *  R10 the target turns its logits into next-token probabilities
 *      (llm-digest, "Mechanism"): p_v = exp((z_v - m) / T) / sum_w exp((z_w - m) / T),
 *      m = max_v z_v, all in fp64, then rounded to the nearest fp32 -- the
 *      same fp32 probability rows the probability form of the acceptance
 *      takes (the batched-acceptance workload's "fp32 target probs from
 *      softmax").  A row holding NaN or +inf, or no finite entry, has no
 *      softmax and reads as all-zero probabilities.
 *  R11 u_acc[b][i] = Philox4x32-10(key = seed, counter (b, i, 0, 0)) and
 *      u_res[b] = Philox4x32-10(key = seed, counter (b, 0, 1, 0)): word 0's
 *      top 24 bits times 2^-24 (Salmon et al., "Parallel random numbers: as
 *      easy as 1, 2, 3", SC'11: the Philox S-box, 10 rounds, Weyl key
 *      schedule).
 * Then the acceptance is oracle_accept_sample on these p, q, u.
 * ---------------------------------------------------------------------- */
static void philox4x32_10(uint32_t c[4], uint64_t key)
{
    uint32_t k0 = (uint32_t)key, k1 = (uint32_t)(key >> 32);
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c[1] ^ k0;
        const uint32_t n1 = (uint32_t)p1;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c[3] ^ k1;
        const uint32_t n3 = (uint32_t)p0;
        c[0] = n0; c[1] = n1; c[2] = n2; c[3] = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
}

static float philox_u(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t stream)
{
    uint32_t c[4] = {c0, c1, stream, 0u};
    philox4x32_10(c, seed);
    return (float)((double)(c[0] >> 8) * 0x1p-24);
}

/* m = max_v z_v and Z = sum_v exp((z_v - m) / T) in fp64 (reading R10).
 * Returns 1, with m = 0 and Z = +inf, for a row without a softmax. */
static int softmax_row_stats(const float *z, int V, double T, float *m_out, double *Z_out)
{
    int bad = 0;
    float m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        if (isnan(z[v]) || z[v] == INFINITY) bad = 1;
        else if (z[v] > m) m = z[v];
    }
    if (bad || m == -INFINITY) {
        *m_out = 0.0f;
        *Z_out = INFINITY;
        return 1;
    }
    double Z = 0.0;
    for (int v = 0; v < V; ++v) Z += exp(((double)z[v] - (double)m) / T);
    *m_out = m;
    *Z_out = Z;
    return 0;
}

static int softmax_to_f32(const float *z, int V, double T, float *p)
{
    float m;
    double Z;
    const int bad = softmax_row_stats(z, V, T, &m, &Z);
    for (int v = 0; v < V; ++v) p[v] = bad ? 0.0f : (float)(exp(((double)z[v] - (double)m) / T) / Z);
    return bad;
}

/* Probabilities and uniforms of the logits form (readings R9-R11), for the
 * acceptance oracle and for the tests: p [B][1+D][V], q [B][D][V],
 * u_acc [B][D], u_res [B]. */
int oracle_logits_to_probs(const float *zp, const float *zq, float temperature, uint64_t seed,
                           int B, int D, int V, float *p, float *q, float *u_acc, float *u_res,
                           int num_threads)
{
    if (B < 0 || D < 0 || V < 1 || !(temperature > 0.0f)) return -2;
    const double T = temperature;
    set_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < (int64_t)B * (2 * D + 1); ++r) {
        const int64_t b = r / (2 * D + 1), k = r % (2 * D + 1);
        if (k <= D)
            softmax_to_f32(zp + (b * (1 + D) + k) * V, V, T, p + (b * (1 + D) + k) * V);
        else
            softmax_to_f32(zq + (b * D + (k - D - 1)) * V, V, T, q + (b * D + (k - D - 1)) * V);
    }
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i < D; ++i) u_acc[(int64_t)b * D + i] = philox_u(seed, (uint32_t)b, (uint32_t)i, 0u);
        u_res[b] = philox_u(seed, (uint32_t)b, 0u, 1u);
    }
    return 0;
}

/* The row statistics (m, Z) of reading R10 for the B (2D + 1) rows, row
 * b (2D + 1) + k being target row k for k <= D and draft row k - D - 1
 * otherwise.  Returns the number of rows without a softmax. */
int oracle_logits_row_stats(const float *zp, const float *zq, float temperature, int B, int D, int V,
                            float *m, double *Z, int num_threads)
{
    if (B < 0 || D < 0 || V < 1 || !(temperature > 0.0f)) return -2;
    const double T = temperature;
    int nbad = 0;
    set_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : nbad)
    for (int64_t r = 0; r < (int64_t)B * (2 * D + 1); ++r) {
        const int64_t b = r / (2 * D + 1), k = r % (2 * D + 1);
        const float *z = k <= D ? zp + (b * (1 + D) + k) * V : zq + (b * D + (k - D - 1)) * V;
        nbad += softmax_row_stats(z, V, T, m + r, Z + r);
    }
    return nbad;
}

/* ------------------------------------------------------------------------
 * AdaSD relaxed acceptance ("Adaptive speculative decoding" article,
 * section AdaSD): two thresholds taken from runtime statistics -- the
 * entropy of the draft distribution decides where the drafter stops, and
 * the Jensen-Shannon distance between the draft and target distributions
 * decides whether a draft token is close enough to be accepted even where
 * the min(1, p/q) rule would reject it (so the method is lossy); both act
 * on the token distributions of a shared vocabulary.  Readings:
 *  R12 entropy H(q) = -sum_v q(v) ln q(v) (natural log, 0 ln 0 = 0); the
 *      drafter stops at the first position whose draft distribution is too
 *      uncertain: D_eff = min{ i : H(q_i) > tau_H }, else D; drafts from
 *      D_eff on are not proposed.
 *  R13 JS distance = sqrt(JSD), JSD(p, q) = (KL(p || m) + KL(q || m)) / 2,
 *      m = (p + q) / 2, natural log: a value in [0, sqrt(ln 2)].
 *  R14 draft i < D_eff is accepted iff u_acc * q(x) < p(x) (the exact rule of
 *      the stochastic acceptance) or JS(p_i, q_i) <= tau_JS.  At the first
 *      failure j the token is drawn from max(0, p_j - q_j) renormalised (R5's
 *      fallback to p_j when that is zero); if all D_eff are accepted, from
 *      p_{D_eff}.  n_accepted = j or D_eff.
 *  R15 the thresholds are inputs of the call; the per-row statistics H and
 *      JS are outputs, from which the caller adapts the thresholds.
 * ---------------------------------------------------------------------- */
static double xlnx(double x) { return x > 0.0 ? x * log(x) : 0.0; }

static void adasd_row_stats(const float *p, const float *q, int V, double *H, double *JS)
{
    double h = 0.0, jsd = 0.0;
    for (int v = 0; v < V; ++v) {
        const double pv = (double)p[v], qv = (double)q[v];
        const double m = 0.5 * (pv + qv);
        h -= xlnx(qv);
        /* p ln(p/m) + q ln(q/m), each term 0 where its weight is 0 */
        if (pv > 0.0) jsd += pv * log(pv / m);
        if (qv > 0.0) jsd += qv * log(qv / m);
    }
    *H = h;
    *JS = sqrt(fmax(0.0, 0.5 * jsd));
}

/* H [B][D] and JS [B][D] of every draft position's (p_i, q_i). */
int oracle_adasd_stats(const float *p, const float *q, int B, int D, int V, double *H, double *JS,
                       int num_threads)
{
    if (B < 0 || D < 0 || V < 1) return -2;
    set_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < (int64_t)B * D; ++r) {
        const int64_t b = r / D, i = r % D;
        adasd_row_stats(p + (b * (1 + D) + i) * V, q + (b * D + i) * V, V, H + r, JS + r);
    }
    return 0;
}

/* Readings R12-R14 with the statistics above.  Outputs per sequence:
 * n_accepted, token, d_eff, margin_u (as oracle_accept_sample's margin, over
 * the uniform-based decisions and the draw), margin_stat (min over the
 * decisive threshold comparisons of |H - tau_H| and |JS - tau_JS|) and the
 * R5 fallback flag. */
int oracle_accept_adasd(const float *p, const float *q, const int32_t *draft, const float *u_acc,
                        const float *u_res, float tau_h, float tau_js, int B, int D, int V,
                        int32_t *n_accepted, int32_t *token, int32_t *d_eff, double *margin_u,
                        double *margin_stat, int32_t *fallback, int num_threads)
{
    if (B < 0 || D < 0 || V < 1) return -2;
    int err = 0;
    set_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        const float *pb = p + (int64_t)b * (1 + D) * V;
        const float *qb = q + (int64_t)b * D * V;
        double mu = INFINITY, ms = INFINITY;
        int de = D;
        for (int i = 0; i < D; ++i) {
            double H, JS;
            adasd_row_stats(pb + (int64_t)i * V, qb + (int64_t)i * V, V, &H, &JS);
            if (fabs(H - (double)tau_h) < ms) ms = fabs(H - (double)tau_h);
            if (H > (double)tau_h) { de = i; break; }
        }
        int j = de;
        for (int i = 0; i < de; ++i) {
            int x = draft[(int64_t)b * D + i];
            if (x < 0 || x >= V) {
#pragma omp atomic write
                err = -4;
                x = 0;
            }
            const double px = (double)pb[(int64_t)i * V + x], qx = (double)qb[(int64_t)i * V + x];
            const double u = (double)u_acc[(int64_t)b * D + i];
            if (qx > 0.0 && fabs(u - px / qx) < mu) mu = fabs(u - px / qx);
            if (u * qx < px) continue;                 /* the exact rule accepts */
            double H, JS;
            adasd_row_stats(pb + (int64_t)i * V, qb + (int64_t)i * V, V, &H, &JS);
            if (fabs(JS - (double)tau_js) < ms) ms = fabs(JS - (double)tau_js);
            if (JS <= (double)tau_js) continue;        /* close enough: accepted anyway */
            j = i;
            break;
        }
        int fb = 0, tok;
        double dm = INFINITY;
        if (j < de) {
            tok = draw_residual(pb + (int64_t)j * V, qb + (int64_t)j * V, V, 1, (double)u_res[b], &dm);
            if (tok < 0) {
                fb = 1;
                tok = draw_residual(pb + (int64_t)j * V, NULL, V, 0, (double)u_res[b], &dm);
            }
        } else {
            tok = draw_residual(pb + (int64_t)de * V, NULL, V, 0, (double)u_res[b], &dm);
        }
        if (tok < 0) tok = 0;
        if (dm < mu) mu = dm;
        n_accepted[b] = j;
        token[b] = tok;
        if (d_eff) d_eff[b] = de;
        if (margin_u) margin_u[b] = mu;
        if (margin_stat) margin_stat[b] = ms;
        if (fallback) fallback[b] = fb;
    }
    return err;
}
