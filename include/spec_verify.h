/*
 * spec_verify.h -- C ABI of the speculative-decoding verification step on
 * one GB300 (sm_103a) GPU.
 *
 * The verification step runs the target model once over B x (1 + D)
 * tokens: for every sequence, the last accepted token plus D draft tokens
 * ("What is speculative decoding", co-design blog).  This library provides
 * the three data-parallel parts of that step:
 *
 *   spec_verify_attention  GQA attention of the B(1+D) query tokens over a
 *                          paged bf16 KV cache, causal among the drafts.
 *   spec_verify_gemm       a linear layer of the verify pass, GEMM-M = B(1+D).
 *   spec_accept_greedy     greedy longest-prefix acceptance.
 *   spec_accept_sample     stochastic min(1, p/q) acceptance with residual
 *                          resampling.
 *   spec_accept_sample_logits   the same from logits, temperature and seed.
 *   spec_accept_adasd      AdaSD relaxed acceptance (draft-entropy stop,
 *                          Jensen-Shannon distance threshold).
 *
 * Conventions shared by every entry point:
 *  - Pointers marked "device" are CUDA device pointers owned by the caller;
 *    the library never frees or retains them and allocates no device memory.
 *    Scratch space is the caller's `workspace` (size from the matching
 *    *_workspace_size call).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    enqueued asynchronously; the call returns once it is enqueued.
 *  - Arguments are validated on the host before anything is enqueued; an
 *    invalid call returns an error status and launches nothing.
 *  - Conditions only the device can see (a page id outside the pool, a
 *    kv_len outside its range, a token id outside [0, V), a uniform outside
 *    [0, 1), a bounded wait that expired) are OR-ed into *dev_status when
 *    dev_status is non-NULL (a device uint32_t the caller zeroes and reads
 *    after synchronising).  Kernels never trap.
 *  - All entry points are thread-safe; calls on one stream execute in order.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1,   /* NULL/misaligned pointer, negative size, ... */
    SPEC_ERR_UNSUPPORTED = 2,   /* valid but outside the supported set        */
    SPEC_ERR_WORKSPACE = 3,     /* workspace missing or too small             */
    SPEC_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed          */
    SPEC_ERR_TIMEOUT = 5        /* reserved: bounded device wait expired      */
} spec_status_t;

/* Bits OR-ed into *dev_status by the kernels. */
#define SPEC_DEV_ERR_PAGE_ID     0x00000001u /* block_table entry outside [0, num_pages) */
#define SPEC_DEV_ERR_KV_LEN      0x00000002u /* kv_len[b] < 1+D or > max_pages*page_size */
#define SPEC_DEV_ERR_TIMEOUT     0x00000004u /* a bounded mbarrier wait expired          */
#define SPEC_DEV_ERR_TOKEN_ID    0x00000008u /* draft token outside [0, V)               */
#define SPEC_DEV_ERR_UNIFORM     0x00000010u /* uniform outside [0, 1)                   */
#define SPEC_DEV_ERR_ZERO_MASS   0x00000020u /* a row to sample from has zero total mass */
#define SPEC_DEV_ERR_LAUNCH      0x00000040u /* launched without the cluster shape it
                                                needs (e.g. replayed by a tool): did nothing */
#define SPEC_DEV_ERR_TREE        0x00000080u /* draft tree not in topological order */
#define SPEC_DEV_ERR_LOGITS      0x00000100u /* a logits row holding NaN or +inf, or no
                                                finite entry: all its probabilities 0 */
#define SPEC_DEV_ERR_PROB        0x00000200u /* the row the stochastic acceptance draws
                                                from holds a value its exact masses cannot
                                                represent (negative, NaN, 2 or more) or sums
                                                to about 8 or more: the draw is undefined */
#define SPEC_DEV_INFO_ZERO_RESIDUAL 0x00010000u /* informational: max(0,p-q) summed to 0
                                                   after a rejection; drew from p instead */

/* Human-readable name of a status code (static storage). */
const char *spec_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int spec_version(void);

/* ------------------------------------------------------------------------
 * Verify attention.
 *
 * Defined by "Draft length and attention performance" (co-design blog): the
 * D draft tokens reuse the same KV cache, so each KV head serves G(1+D)
 * query rows and the attention GEMM-M is G(1+D).  For sequence b, KV head
 * h, draft position i in [0, D] and group member g in [0, G):
 *
 *     o = softmax(softmax_scale * q K^T) V over keys j < kv_len[b] - D + i
 *
 * i.e. kv_len[b] counts the 1 + D verify tokens, whose K/V the preceding
 * projection has already written into the cache; row i sees the prefix,
 * the earlier drafts and itself.  D = 0 is ordinary decode attention.
 *
 * Layouts (all row-major, innermost last):
 *   q_bf16        device, bf16 [B][1+D][Hkv*G][head_dim]; query head h*G+g
 *                 belongs to KV head h.  16-byte aligned.
 *   k_pages_bf16,
 *   v_pages_bf16  device, bf16 [num_pages][page_size][Hkv][head_dim].
 *                 16-byte aligned.  V is used as stored (bf16 operand of
 *                 the P.V product, P carried as a bf16 hi + lo pair).
 *   block_table   device, int32 [B][max_pages_per_seq]; key j of sequence b
 *                 is slot j % page_size of page block_table[b][j/page_size].
 *                 Entries past a sequence's last page are never read.
 *   kv_len        device, int32 [B]; 1 + D <= kv_len[b] <=
 *                 max_pages_per_seq * page_size.
 *   out_f32       device, fp32 [B][1+D][Hkv*G][head_dim]; 16-byte aligned.
 *   lse_f32       device, fp32 [B][1+D][Hkv*G] or NULL: natural-log
 *                 partition function log(sum_j exp(softmax_scale q.k_j)).
 * Contiguous caches are passed as pages with an identity block table.
 *
 * Supported set: head_dim in {64, 128}; page_size a multiple of 16;
 * 0 <= D <= 63; G >= 1 with G*(1+D) <= 1024.  Other values return
 * SPEC_ERR_UNSUPPORTED.  workspace must hold
 * spec_verify_attention_workspace_size(...) bytes (device, 256-byte
 * aligned); its contents need no initialisation and are scratch only.
 * Rows of a sequence whose kv_len is out of range are not written and set
 * SPEC_DEV_ERR_KV_LEN.
 * ---------------------------------------------------------------------- */
size_t spec_verify_attention_workspace_size(int B, int D, int Hkv, int G, int head_dim,
                                            int max_kv_len);

spec_status_t spec_verify_attention(const void *q_bf16, const void *k_pages_bf16,
                                    const void *v_pages_bf16, int num_pages,
                                    const int32_t *block_table, int max_pages_per_seq,
                                    const int32_t *kv_len, int B, int D, int Hkv, int G,
                                    int head_dim, int page_size, float softmax_scale,
                                    float *out_f32, float *lse_f32, void *workspace,
                                    size_t workspace_bytes, uint32_t *dev_status,
                                    void *stream);

/* ------------------------------------------------------------------------
 * Verify attention without a caller workspace: allocates nothing.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot hand the library a device buffer -- for example a plugin in
 * an inference engine whose own memory pool owns all device memory and
 * forbids other allocations, or a latency-critical loop in which
 * cudaMalloc / cudaFree would synchronise the device.  It computes exactly
 * what spec_verify_attention computes, with the same arguments minus the
 * workspace pair, but takes its scratch from a fixed device array of
 * SPEC_NOALLOC_SCRATCH_BYTES built into the library (every GPU that loads
 * the library holds that array until the process exits) and calls no
 * allocator of any kind.
 *  - A problem whose spec_verify_attention_workspace_size(...) exceeds
 *    SPEC_NOALLOC_SCRATCH_BYTES is rejected with SPEC_ERR_WORKSPACE before
 *    anything is launched.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture.
 *  - Every call shares the one array, whose contents persist between calls
 *    but need no clearing.  Calls that can overlap on the GPU (two streams,
 *    or host threads without ordering between them) race on the array and
 *    must be serialised by the caller.
 * ---------------------------------------------------------------------- */
#define SPEC_NOALLOC_SCRATCH_BYTES (24u << 20)

spec_status_t spec_verify_attention_noalloc(const void *q_bf16, const void *k_pages_bf16,
                                            const void *v_pages_bf16, int num_pages,
                                            const int32_t *block_table, int max_pages_per_seq,
                                            const int32_t *kv_len, int B, int D, int Hkv, int G,
                                            int head_dim, int page_size, float softmax_scale,
                                            float *out_f32, float *lse_f32, uint32_t *dev_status,
                                            void *stream);

/* ------------------------------------------------------------------------
 * Verify GEMM.
 *
 * Defined by "Draft length and performance of linear layers" (co-design
 * blog): with speculation every linear layer of the target runs with
 * GEMM-M = M(1+D) instead of M; the representative expert GEMM is
 * N = K = 6144.
 *
 *     y[m][n] = sum_k x[m][k] * w[n][k]     (fp32 accumulate, bf16 out)
 *
 *   x_bf16   device, bf16 [M][K] row-major, 16-byte aligned.
 *   w_bf16   device, bf16 [N][K] row-major (nn.Linear weight layout),
 *            16-byte aligned.
 *   y_bf16   device, bf16 [M][N] row-major, 16-byte aligned.
 *   dev_status  device uint32 or NULL: SPEC_DEV_ERR_TIMEOUT (a bounded wait
 *            expired; y is then incomplete) or SPEC_DEV_ERR_LAUNCH.
 * Supported set: 1 <= M <= 65536, N a multiple of 128, K a multiple of 64.
 * M <= 256 (weight streaming) splits the K range of each 128-row block of
 * w between CTAs.  When every block's CTAs fit on the device at once (a
 * thread-block cluster per block or, for M > 64, per pair of blocks whose
 * MMAs CTA pairs share), the pieces are added in shared memory across the
 * cluster and the workspace is not touched; otherwise (stream-K) they are
 * added through it.  Either
 * way pass spec_verify_gemm_workspace_size(M, N, K) bytes of device memory,
 * 256-byte aligned, owned by the caller.  It holds the arrival counters of
 * the tiles cut between CTAs (the first 4096 bytes) and the fp32 partial
 * tiles: zero it once before its first use (cudaMemset); every call that
 * completes leaves the counters zero again, also under CUDA-graph replay.
 * A call that sets any dev_status bit may leave counters non-zero: zero the
 * workspace again before the next call.  Calls that share a workspace must
 * not overlap in time.  A smaller workspace returns SPEC_ERR_WORKSPACE.
 * M > 256 (pairs of CTAs sharing each MMA, whole tiles) needs no workspace
 * (its size is 0 and workspace may be NULL).  The size depends on the
 * current device's SM count (without a device it is sized for 256 SMs).
 * ---------------------------------------------------------------------- */
size_t spec_verify_gemm_workspace_size(int M, int N, int K);

spec_status_t spec_verify_gemm(const void *x_bf16, const void *w_bf16, void *y_bf16, int M,
                               int N, int K, void *workspace, size_t workspace_bytes,
                               uint32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Greedy acceptance.
 *
 * The target keeps the longest draft prefix it agrees with and adds one
 * token of its own (LLM inference handbook, "How speculative decoding
 * works"; co-design blog, "What is speculative decoding").  With
 * t_i = argmax_v p[b][i][v] (lowest index on ties):
 *     n_accepted[b] = first i < D with draft[b][i] != t_i, else D
 *     token[b]      = t_{n_accepted[b]}
 * so the accepted length AL = n_accepted + 1 lies in [1, 1 + D].  Only the
 * rows 0..n_accepted[b] of p are read.
 *
 *   p        device, fp32 [B][1+D][V] target probabilities (or logits: only
 *            their order matters).  NaN-free.
 *   draft    device, int32 [B][D].
 *   n_accepted, token   device, int32 [B].
 *   dev_status  device uint32 or NULL (SPEC_DEV_ERR_TIMEOUT).
 * Supported set: B >= 0, 0 <= D <= 63, 1 <= V <= 2^26.
 * ---------------------------------------------------------------------- */
spec_status_t spec_accept_greedy(const float *p, const int32_t *draft, int B, int D, int V,
                                 int32_t *n_accepted, int32_t *token, uint32_t *dev_status,
                                 void *stream);

/* ------------------------------------------------------------------------
 * Tree verification.
 *
 * Multi-head and feature-level drafters propose a tree of candidate
 * continuations; the target scores the whole tree in one pass with a mask
 * that keeps each branch causal, and the longest accepted candidate prefix
 * is kept (LLM inference handbook, "Speculative decoding", Medusa; EAGLE-2's
 * dynamic draft tree in the same section).
 *
 * A draft tree of sequence b has 1 + D nodes in topological order:
 *   tree_parent  device, int32 [B][1+D]; tree_parent[b][0] = -1 (the root:
 *                the last accepted token), 0 <= tree_parent[b][k] < k.
 * Node k's K/V sit at cache position kv_len[b] - (1+D) + k, and its query
 * is q[b][k].  Malformed trees set SPEC_DEV_ERR_TREE (their nodes then see
 * the prefix and themselves only).
 *
 * spec_verify_tree_attention: as spec_verify_attention, except that node k
 * attends to keys j < kv_len[b] - (1+D) and to the tree keys of the nodes
 * on its root-to-k path (its ancestors and itself).  The chain
 * tree_parent[b][k] = k - 1 gives exactly spec_verify_attention.  workspace:
 * spec_verify_tree_attention_workspace_size(...) bytes (the chain workspace
 * plus 8 bytes per node), scratch only.
 * ---------------------------------------------------------------------- */
size_t spec_verify_tree_attention_workspace_size(int B, int D, int Hkv, int G, int head_dim,
                                                 int max_kv_len);

spec_status_t spec_verify_tree_attention(const void *q_bf16, const void *k_pages_bf16,
                                         const void *v_pages_bf16, int num_pages,
                                         const int32_t *block_table, int max_pages_per_seq,
                                         const int32_t *kv_len, const int32_t *tree_parent, int B,
                                         int D, int Hkv, int G, int head_dim, int page_size,
                                         float softmax_scale, float *out_f32, float *lse_f32,
                                         void *workspace, size_t workspace_bytes,
                                         uint32_t *dev_status, void *stream);

/* spec_accept_tree_greedy: with t_k = argmax_v p[b][k][v] (lowest index on
 * ties), start at the root and repeatedly move to the child of the current
 * node whose token equals t_(current) -- the lowest node index if several
 * siblings carry it -- until no child does.
 *   p          device, fp32 [B][1+D][V] target probabilities at every node.
 *   tokens     device, int32 [B][1+D]; tokens[b][k] is node k's draft token
 *              (tokens[b][0] is not read).
 *   n_accepted device, int32 [B]: the depth reached (accepted drafts).
 *   token      device, int32 [B]: t at the last node reached.
 *   path       device, int32 [B][D] or NULL: the accepted node ids in order,
 *              then -1.
 * Only the rows of the nodes on the accepted path are read.  The chain with
 * node k carrying draft k - 1 gives exactly spec_accept_greedy.
 * ---------------------------------------------------------------------- */
spec_status_t spec_accept_tree_greedy(const float *p, const int32_t *tokens, const int32_t *parent,
                                      int B, int D, int V, int32_t *n_accepted, int32_t *token,
                                      int32_t *path, uint32_t *dev_status, void *stream);

/* spec_accept_tree_sample: stochastic acceptance over a draft tree (the
 * lossless rule of the stochastic acceptance below, generalised to
 * siblings).  The children of node k (nodes whose parent is k, in
 * increasing index) carry tokens drafted from q[b][k].  From the root, at
 * the current node the working row r starts as p[b][node]; a child with
 * token x is accepted iff u_acc[b][child] * q[b][node][x] < r(x), and the
 * walk moves to it; otherwise r becomes max(0, r - q[b][node]) divided by
 * its sum (left as it is, with SPEC_DEV_INFO_ZERO_RESIDUAL, when that sum is
 * 0) and the next child is tried.  When no child is accepted, or the node
 * has none, the token is the smallest v with sum_{w <= v} r(w) > u_res[b] *
 * sum_w r(w).  A chain whose node k carries draft k - 1 is
 * spec_accept_sample.
 *   p, q       device, fp32 [B][1+D][V]; q[b][k] is the draft distribution
 *              node k's children were drawn from (rows of leaves are not
 *              read).  Probabilities in [0, 1].
 *   tokens     device, int32 [B][1+D]; tokens[b][0] is not read.
 *   parent     device, int32 [B][1+D], as for tree attention.
 *   u_acc      device, fp32 [B][1+D] in [0, 1): the uniform of node k's
 *              test (u_acc[b][0] is not read).
 *   u_res      device, fp32 [B] in [0, 1): the uniform of the final draw.
 *   n_accepted, token, path  as for spec_accept_tree_greedy.
 * Arithmetic: the row after j rejections is kept unnormalised (R_j =
 * max(0, R_(j-1) - S_(j-1) q) with S_0 = 1 and S_j the sum of R_j), which
 * unrolls to R_j = max(0, p - c_j q) with c_j = S_0 + ... + S_(j-1); each
 * element is evaluated in that form (c_j summed in fp64 and rounded to fp32
 * once, then one fp32 fused multiply-add), and the sums are exact in 2^-61
 * fixed point; a test after j rejections is u q(x) S_j < R_j(x) in fp64.  A
 * cluster of CTAs per sequence (vocabulary slices whose exact sums are
 * exchanged through distributed shared memory); each rejection and the
 * final draw read the node's p and q rows once (from HBM the first time,
 * mostly from L2 after).
 * Supported: D <= 63, V <= 2^22.  A malformed tree (SPEC_DEV_ERR_TREE) or a
 * token outside [0, V) (SPEC_DEV_ERR_TOKEN_ID) makes the walk stop at the
 * root; uniforms outside [0, 1) are clamped (SPEC_DEV_ERR_UNIFORM).
 * ---------------------------------------------------------------------- */
spec_status_t spec_accept_tree_sample(const float *p, const float *q, const int32_t *tokens,
                                      const int32_t *parent, const float *u_acc, const float *u_res,
                                      int B, int D, int V, int32_t *n_accepted, int32_t *token,
                                      int32_t *path, uint32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Stochastic acceptance (modified rejection sampling).
 *
 * From "How does speculative decoding speed up LLM inference?" (llm-digest,
 * sections "Mechanism" and "Math intuition"): walk the drafts left to
 * right, accept draft x with probability min(1, p(x)/q(x)); at the first
 * rejection discard the rest and resample that position from
 * max(0, p - q) renormalised; the emitted tokens then follow p exactly.
 * With explicit uniforms:
 *     accept draft i  iff  u_acc[b][i] * q[b][i][x] < p[b][i][x]   (exact)
 *     j = first rejected i, else D;  n_accepted[b] = j
 *     r(v) = max(0, p[b][j][v] - q[b][j][v])  if j < D,  else p[b][D][v]
 *     token[b] = smallest v with sum_{w<=v} r(w) > u_res[b] * sum_w r(w)
 * If r sums to zero after a rejection, r = p[b][j] is used instead and
 * SPEC_DEV_INFO_ZERO_RESIDUAL is set.  The sums are carried out exactly
 * (fixed point with 2^-61 resolution), so the result does not depend on
 * summation order.
 *
 *   p        device, fp32 [B][1+D][V], entries in [0, 1], row sums < 8.
 *   q        device, fp32 [B][D][V], same constraints (may be NULL if D=0).
 *            The values a sequence draws from are checked: a residual
 *            max(0, p - q), or a bonus-row p, that is negative (other than
 *            -0), NaN or 2 or more, or a row whose values sum to about 8 or
 *            more (the 64-bit sums of its 2^-61 masses would wrap), sets
 *            SPEC_DEV_ERR_PROB.
 *   draft    device, int32 [B][D].
 *   u_acc    device, fp32 [B][D] in [0, 1).
 *   u_res    device, fp32 [B] in [0, 1).
 *   n_accepted, token   device, int32 [B].
 *   workspace  device, spec_accept_sample_workspace_size(B, V) bytes,
 *              256-byte aligned, owned by the caller; scratch only (the
 *              first rejected draft and the exact masses of every 512- and
 *              128-element slice of the needed rows), needs no
 *              initialisation.  Calls sharing a workspace must not overlap
 *              in time.
 * Supported set: B >= 0, 0 <= D <= 63, 1 <= V <= 2^26.
 * ---------------------------------------------------------------------- */
size_t spec_accept_sample_workspace_size(int B, int V);

spec_status_t spec_accept_sample(const float *p, const float *q, const int32_t *draft,
                                 const float *u_acc, const float *u_res, int B, int D, int V,
                                 int32_t *n_accepted, int32_t *token, void *workspace,
                                 size_t workspace_bytes, uint32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * AdaSD relaxed acceptance (lossy).
 *
 * From "Adaptive speculative decoding" (section AdaSD): two thresholds act
 * on the token distributions of the shared vocabulary -- the entropy of the
 * draft distribution decides where the drafter stops, and the
 * Jensen-Shannon distance between draft and target distributions decides
 * whether a draft token is close enough to be accepted even where the
 * min(1, p/q) rule would reject it.  Per sequence b and position i < D:
 *     H[b][i]  = -sum_v q ln q                   (natural log, 0 ln 0 = 0)
 *     JS[b][i] = sqrt((KL(p || m) + KL(q || m)) / 2),  m = (p + q) / 2
 *     d_eff    = first i with H[b][i] > tau_entropy, else D
 *     draft i < d_eff accepted iff u_acc * q(x) < p(x) (exact, as in
 *         spec_accept_sample) or JS[b][i] <= tau_js
 *     at the first failure j: n_accepted = j and the token is drawn from
 *     max(0, p[j] - q[j]) renormalised (p[j] if that is zero); if all d_eff
 *     drafts pass: n_accepted = d_eff and the token is drawn from p[d_eff].
 * tau_entropy = +inf and tau_js < 0 give exactly spec_accept_sample.  The
 * thresholds are the caller's (it adapts them from the statistics this call
 * returns).  H and JS are computed in fp32 with the hardware logarithm
 * (absolute error about 1e-5 against exact arithmetic at V = 131072), so a
 * decision can differ from the exact one only for a statistic that close
 * to its threshold.  Every p_i and q_i row with i < D is read once for the
 * statistics, then the gathered draft entries and the one row each sequence
 * draws from.
 *
 *   p, q, draft, u_acc, u_res, n_accepted, token   as in spec_accept_sample.
 *   tau_entropy, tau_js   thresholds (not NaN).
 *   draft_len    device int32 [B] or NULL: d_eff.
 *   entropy, js_distance  device fp32 [B][D] or NULL: H and JS of every
 *                position (all D, also past d_eff).
 *   workspace  device, spec_accept_adasd_workspace_size(B, D, V) bytes,
 *              256-byte aligned, scratch only, needs no initialisation.
 * Supported set: B <= 65535, 0 <= D <= 63, 1 <= V <= 2^26.
 * ---------------------------------------------------------------------- */
size_t spec_accept_adasd_workspace_size(int B, int D, int V);

spec_status_t spec_accept_adasd(const float *p, const float *q, const int32_t *draft, const float *u_acc,
                                const float *u_res, float tau_entropy, float tau_js, int B, int D, int V,
                                int32_t *n_accepted, int32_t *token, int32_t *draft_len, float *entropy,
                                float *js_distance, void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                                void *stream);

/* ------------------------------------------------------------------------
 * Stochastic acceptance from logits.
 *
 * The acceptance above with p = softmax(target_logits / T) and
 * q = softmax(draft_logits / T) taken inside the library, and the uniforms
 * drawn from `seed` by Philox4x32-10 (Salmon, Moraes, Dror and Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3", SC'11; key = seed, word 0
 * of the output, u = (word >> 8) * 2^-24):
 *     u_acc[b][i] from counter (b, i, 0, 0),  u_res[b] from (b, 0, 1, 0).
 * The probabilities are the fp32 roundings of the exact softmax, the rows
 * spec_accept_sample would take:
 *  - the row each sequence draws from (max(0, p_j - q_j) after a rejection
 *    at j, else p_D) is evaluated to double-float accuracy and rounded once,
 *    so each of its entries is the nearest fp32 to softmax(z / T) unless
 *    the exact value lies within about 2^-33 (relative) of a rounding tie;
 *  - the accept tests use a fast evaluation (hardware base-2 exponential,
 *    fp32 row sums), relative error about 1e-7 (up to 1e-6 for logits far
 *    below the row maximum): a decision can differ from the exact one only
 *    when u_acc lies that close to p(x) / q(x).
 * Every logit is read from HBM once for the row statistics; afterwards only
 * the gathered draft entries and the one or two rows each sequence draws
 * from are read again (twice: for their exact sums, then for the draw).
 *
 *   target_logits  device, fp32 [B][1+D][V]; finite or -inf.
 *   draft_logits   device, fp32 [B][D][V] (may be NULL if D = 0).
 *   temperature    T, finite and > 0.
 *   draft, n_accepted, token   as in spec_accept_sample.
 *   workspace  device, spec_accept_sample_logits_workspace_size(B, D, V)
 *              bytes, 256-byte aligned; scratch only (first the row
 *              statistics (m = max_v z_v, Zf = sum_v 2^((z_v - m) log2(e) /
 *              T) in fp32) of the B (2D + 1) rows as fp32 pairs, row
 *              b (2D + 1) + k being target row k for k <= D and draft row
 *              k - D - 1 otherwise; then the draw rows' exact partial sums and
 *              the scratch of spec_accept_sample), needs no initialisation.
 * A row holding NaN or +inf, or only -inf, sets SPEC_DEV_ERR_LOGITS and
 * reads as all-zero probabilities.
 * Supported set: B <= 65535, 0 <= D <= 63, 1 <= V <= 2^26.
 * ---------------------------------------------------------------------- */
size_t spec_accept_sample_logits_workspace_size(int B, int D, int V);

spec_status_t spec_accept_sample_logits(const float *target_logits, const float *draft_logits,
                                        const int32_t *draft, float temperature, uint64_t seed, int B, int D,
                                        int V, int32_t *n_accepted, int32_t *token, void *workspace,
                                        size_t workspace_bytes, uint32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Host-side planning helper (no GPU work).
 *
 * Reports how spec_verify_attention splits the KV stream across CTAs for
 * the given host copy of kv_len and CTA-group count: segment s covers key
 * tiles [tile_begin, tile_end) (SPEC_ATTENTION_KEY_TILE keys per tile) of
 * unit (b, h), processed
 * by group `group` and written to partial slot `slot` (-1 when the segment
 * covers the whole unit and is written straight to the output).  Writes up
 * to max_segments records of 6 int32 (group, b, h, tile_begin, tile_end,
 * slot) and returns the number of segments, or -1 on invalid arguments.
 * ---------------------------------------------------------------------- */
#define SPEC_ATTENTION_KEY_TILE 128

int spec_verify_attention_plan(int B, const int32_t *kv_len_host, int D, int Hkv,
                               int num_groups, int32_t *segments, int max_segments);

/* ------------------------------------------------------------------------
 * Host-side view of how spec_verify_gemm splits the work (no counterpart
 * on the pages; launches nothing, needs no device).
 *
 * The work is split into units over at most num_sms SMs, one CTA per SM.
 *  - M > 256: a unit is a pair of CTAs (a thread-block cluster of 2) that
 *    runs one MMA of 256 rows; output tile t covers rows
 *    (t % tiles_m) * 256 .. + 255, tiles_m = ceil(M / 256), and column tile
 *    t / tiles_m.  The N columns are cut into tiles_n column tiles, in
 *    32-column units, whose widths differ by at most 32 (the wider ones
 *    first); pair c takes tiles c, c + pairs, ... whole (all k-blocks).
 *  - M <= 256: a unit is one CTA; tile t covers the 128 w rows (output
 *    columns) t * 128 .. t * 128 + 127 for all M rows, which are padded to
 *    BN in {32, 64, 128, 256} on the MMA side.  Each unit walks a list of
 *    segments (a tile and a range [kb0, kb1) of its 64-wide k-blocks).
 *    With split K over clusters (spec_verify_gemm_plan_cluster returns
 *    their size C >= 2 for M <= 256), each unit has one segment: either
 *    S = C single CTAs per tile (unit c = t S + r takes [r K/S,
 *    (r + 1) K/S) of tile t) or, for 64 < M <= 256, S = C / 2 CTA pairs
 *    per 256-row pair tile T (unit c = T C + 2p + h takes [p K/S,
 *    (p + 1) K/S) of tile 2T + h), in k-blocks of 64.
 * Writes, for each segment in unit order, the row (unit, tile, kb0, kb1,
 * last, BN) into segments[6 * i ..] (int32, host memory), where last is,
 * for a segment with kb0 == 0, the last unit holding a later piece of the
 * same tile (the unit itself when the tile is whole), and -1 otherwise, and
 * BN is the tile's width (M > 256) or the padded rows of x (M <= 256).
 * Returns the number of segments (rows beyond max_segments are counted, not
 * written), or -1 for invalid arguments.
 * ---------------------------------------------------------------------- */
int spec_verify_gemm_plan(int M, int N, int K, int num_sms, int32_t *segments,
                          int max_segments);

/* The cluster size of the launch that spec_verify_gemm_plan describes: 2
 * for CTA pairs when M > 256; for M <= 256, 1 for stream-K weight
 * streaming and C in [2, 8] for split K over clusters of C CTAs (unit c is
 * CTA c of the grid, rank c % C of its cluster; the CTAs of a cluster that
 * hold the same tile split its k-blocks in rank order).  Planned for
 * num_sms SMs holding num_sms / C clusters of C (a device may hold fewer
 * and plan otherwise); -1 for invalid arguments.  No device needed. */
int spec_verify_gemm_plan_cluster(int M, int N, int K, int num_sms);

/* ------------------------------------------------------------------------
 * Self-test of the bounded device wait (no counterpart on the pages).
 *
 * Every mbarrier wait in the library's kernels is bounded: when it runs out
 * the kernel ORs SPEC_DEV_ERR_TIMEOUT into *dev_status, stops its other
 * roles, waits (bounded) for its own copies and MMAs in flight and returns,
 * so the CUDA context stays usable.  This entry point runs that same wait
 * in a one-CTA kernel so that a test can make it run out on purpose:
 * warp 0 waits on an mbarrier, limited to wait_limit_ns; one thread of
 * warp 1 arrives on it after arrive_after_ns, or never when
 * arrive_after_ns is UINT64_MAX.  No copy or MMA is in flight.
 *   result     device, uint64 [3], 8-byte aligned: [0] 1 if the wait saw the
 *              barrier complete, 0 if it gave up; [1] the kernel's abort flag
 *              after the wait; [2] how long the wait took, in ns.
 *   dev_status device uint32 or NULL: SPEC_DEV_ERR_TIMEOUT when it gave up.
 * 0 < wait_limit_ns <= 10 s and arrive_after_ns <= 10 s (or UINT64_MAX),
 * else SPEC_ERR_INVALID_ARG; the kernel ends within about
 * max(wait_limit_ns, arrive_after_ns).
 * ---------------------------------------------------------------------- */
spec_status_t spec_selftest_bounded_wait(uint64_t wait_limit_ns, uint64_t arrive_after_ns,
                                         uint64_t *result, uint32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Adaptive draft length (host only; no counterpart kernels).
 *
 * SGLang's controller tracks an exponential moving average of the accept
 * length after every round and switches among a few fixed draft lengths
 * (by default 1, 3 and 7), each with a CUDA graph captured in advance (LLM
 * inference handbook, "Adaptive speculative decoding").  Rule (the pages
 * leave it open): the next round uses the
 * smallest tier D >= EMA(AL), AL = n_accepted + 1, else the largest tier;
 * EMA_1 = mean AL of the first round, EMA_r = beta * EMA_(r-1) +
 * (1 - beta) * mean AL.
 *
 * spec_adaptive_init: tiers strictly increasing draft lengths in [0, 63]
 *   (host array, n_tiers <= SPEC_ADAPTIVE_MAX_TIERS), 0 <= beta < 1.  The
 *   controller starts at the largest tier.
 * spec_adaptive_update: n_accepted host int32 [B] of the round just
 *   verified; returns the draft length for the next round (-1 on bad
 *   arguments).  B = 0 re-evaluates the tier without a new sample.
 * spec_adaptive_draft_len: the current tier's draft length.
 * ---------------------------------------------------------------------- */
#define SPEC_ADAPTIVE_MAX_TIERS 8

typedef struct {
    float ema;       /* moving average of the accept length */
    float beta;      /* weight of the previous average */
    int rounds;      /* rounds seen */
    int n_tiers;
    int current;     /* index of the tier in use */
    int tiers[SPEC_ADAPTIVE_MAX_TIERS];
} spec_adaptive_t;

spec_status_t spec_adaptive_init(spec_adaptive_t *s, const int32_t *tiers, int n_tiers, float beta);
int spec_adaptive_update(spec_adaptive_t *s, const int32_t *n_accepted, int B);
int spec_adaptive_draft_len(const spec_adaptive_t *s);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
