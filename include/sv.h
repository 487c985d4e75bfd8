/*
 * sv.h -- C ABI of the GB300 (sm_103a) verify-and-accept library for
 * speculative decoding: Leviathan rejection sampling along a draft chain or
 * the best-scored path of an EAGLE-style draft tree, residual / bonus
 * sampling, the tree's ancestor attention mask, and KV-cache rollback /
 * compaction.
 *
 * Sources (web pages; cited by title and section):
 *   [Lesson] "Decodificação Especulativa e EAGLE-3" (ai-engineering.academy,
 *            Phase 10 Lesson 15; the same lesson in Persian on nextadmin.net).
 *   [Blog]   "投机解码发展" (caijizhuo.github.io).  The blog swaps the letters;
 *            this header uses the lesson's: p = draft, q = verifier.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is owned by the caller and points to memory the
 *    current device can address: its own device (or managed) memory, or
 *    page-locked host memory (cudaHostAlloc / cudaHostRegister).  Host
 *    buffers are read and written in place by the kernels over the host link
 *    (on GB300, NVLink-C2C), so a round whose logits sit in host memory moves
 *    only the rows it actually reads.  Pageable host memory and another
 *    device's memory are refused with SV_ERR_INVALID_ARG before anything is
 *    enqueued.  The library never allocates, frees or synchronises; scratch
 *    memory is the caller's `workspace`, sized by the matching *_workspace()
 *    query (device memory is the fast choice).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  All work is enqueued asynchronously on it.
 *  - `accept_event` (verify calls; a cudaEvent_t as void*, or NULL): when
 *    given, it is recorded on `stream` as soon as the accept walk is done --
 *    out_accept_len, out_path_nodes and the accepted tokens are final -- and
 *    before the correction / bonus sampling runs.  Work that needs only the
 *    accepted prefix (the KV compaction) can wait on it from another stream
 *    and overlap the sampling.  out_tokens[a], out_margin's gap and the
 *    SV_ROW_RESID_ZERO bit are written after it.
 *  - Argument errors are detected on the host before anything is enqueued;
 *    the call then returns a non-OK sv_status and sv_last_error() says why.
 *    A failed kernel launch returns SV_ERR_CUDA.  No C++ exception crosses
 *    the ABI.
 *  - Data faults found on the device never abort: they set bits in the
 *    per-sequence out_status word and produce the defined fallback outputs.
 *  - Logit rows are row-major [rows][V], element type sv_dtype; rows need no
 *    alignment beyond the element size (16-byte-aligned rows take the
 *    vectorised path).
 *  - Random numbers: Philox4x32-10 (Salmon et al., SC'11) keyed on `seed`,
 *    counter (position, draw, sequence, step mod 2^32); u = (x0 >> 8) 2^-24.
 *    draw 0 = accept test at a position, draw 1 = residual / bonus sample.
 *    A round is a pure function of its inputs, seed and step.
 */
#ifndef SV_H
#define SV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1, /* bad pointer, size, dtype or workspace */
  SV_ERR_UNSUPPORTED = 2, /* valid but beyond this build's limits */
  SV_ERR_CUDA = 3,        /* a CUDA call failed; sv_last_error() has it */
  SV_ERR_TIMEOUT = 4      /* reserved: no call of this build waits on the device */
} sv_status;

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/* Bits of the per-sequence out_status word. */
#define SV_ROW_NAN 1u        /* a used logit row holds NaN or +inf, or is all -inf */
#define SV_ROW_BAD_TOKEN 2u  /* a draft token outside [0, V) */
#define SV_ROW_RESID_ZERO 4u /* residual mass was 0; the correction came from q */
#define SV_ROW_P_ZERO 8u     /* a tested draft token had p(d) = 0 (draft logit -inf) and was accepted */
#define SV_ROW_BAD_TREE 16u  /* parent/score arrays do not describe a tree */
#define SV_ROW_BAD_BASE 32u  /* sv_tree_attention: base < 0 or base + T > S */
#define SV_ROW_TIMEOUT 64u   /* a bounded wait on the device ran out (row pass, sampling, attention) */

/* Build limits. */
#define SV_MAX_VOCAB (1 << 22)  /* fixed-point sampling sums stay below 2^63 */
#define SV_MAX_POSITIONS 1024   /* N (chain) or max_depth (tree) */
#define SV_MAX_TREE_NODES 1024  /* T */

/* ---------------------------------------------------------------------------
 * sv_verify_chain -- verify N drafted tokens per sequence in one call.
 * [Lesson] "O invariante" (Leviathan rejection sampling; the chained form),
 * Passo 1 (accept rule), Passo 2 (residual), Passo 3 (one speculative step);
 * [Blog] section 2 (draft / verify / accept) and section 4 (spec_decode).
 *
 * For sequence b and position i = 0..N-1 the draft token d = draft_tokens[b][i]
 * is judged by q_{i+1} = softmax(vlogits[b][i] / temperature) and
 * p_{i+1} = softmax(dlogits[b][i] / temperature): accepted iff
 * u < min(1, q(d)/p(d)) (or p(d) = 0), left to right.  At the first rejection
 * a < N a correction token is drawn from (q_{a+1} - p_{a+1})_+ normalised (q
 * itself if that mass is 0); if all N pass, a bonus token is drawn from
 * q_{N+1} = softmax(vlogits[b][N]).
 *
 *   vlogits      [B][N+1][V] verifier logits (row i = distribution after input
 *                position i, i.e. over the token that follows it)
 *   dlogits      [B][N][V]   draft logits (may be NULL when N == 0)
 *   draft_tokens [B][N] int32
 *   temperature  >= 0, finite.  Probabilities are softmax(logits / T).
 *                T = 0 is greedy verification, the T -> 0 limit of the rule
 *                (every softmax a point mass at the row's arg max, ties to
 *                the lowest token id): a draft token is accepted iff it is
 *                the verifier row's arg max, the first mismatch emits that
 *                arg max, full acceptance emits the last row's arg max.  Only
 *                verifier rows are read and nothing is sampled; out_q_prob
 *                holds 1 or 0, out_p_prob and out_margin NaN.  The same
 *                holds for sv_verify_tree along the best path.
 * Outputs (device, caller-owned):
 *   out_tokens     [B][N+1]  accepted drafts then the correction/bonus token;
 *                            -1 after it.  emitted = out_accept_len + 1.
 *   out_accept_len [B]       a, the number of accepted drafts.
 *   out_q_prob     [B][N] or NULL: q_{i+1}(d_{i+1}) for every position.
 *   out_p_prob     [B][N] or NULL: p_{i+1}(d_{i+1}).
 *   out_margin     [B][N+1] or NULL: [i] = min(1, q/p) - u at position i;
 *                  [N] = distance of the correction/bonus threshold to the
 *                  nearest CDF boundary, as a fraction of the sampled mass.
 *   out_status     [B]       SV_ROW_* bits.  On NAN / BAD_TOKEN the sequence
 *                  emits nothing: accept_len 0, tokens all -1.
 * The correction/bonus choice uses exact 64-bit fixed-point prefix sums of
 * weights computed with a fixed sequence of IEEE fp32 operations, so the
 * chosen token does not depend on how the sum is split across threads: a
 * draw from q (the bonus, or a zero residual) takes the weights
 * floor(e_v 2^40), e_v = exp(x_v / T - max_v x_v / T) in that arithmetic; a
 * residual takes floor(max(0, q_v - p_v) 2^62) with q, p normalised by those
 * sums.  The row pass's and the sampler's device waits are bounded; one that
 * runs out (which a working device never does) sets SV_ROW_TIMEOUT for the
 * sequences concerned: a row-pass segment it left unread also faults the
 * sequence as SV_ROW_NAN (accept_len 0, tokens -1); a sampler wait leaves
 * the correction/bonus token at -1.
 * --------------------------------------------------------------------------- */
size_t sv_verify_chain_workspace(int B, int N, int V);
/* A larger workspace for logits in page-locked host memory: with it, every
 * logit row the round reads crosses the host link once (the row statistics
 * keep a device copy that the accept walk and the sampler read); with the
 * plain size those steps read the host rows again.  Returns 0 on bad sizes. */
size_t sv_verify_chain_workspace_host(int B, int N, int V, sv_dtype dt);
sv_status sv_verify_chain(const void *vlogits, const void *dlogits, sv_dtype dt,
                          const int32_t *draft_tokens, int B, int N, int V,
                          float temperature, uint64_t seed, uint64_t step,
                          int32_t *out_tokens, int32_t *out_accept_len,
                          float *out_q_prob, float *out_p_prob,
                          float *out_margin, uint32_t *out_status,
                          void *workspace, size_t workspace_bytes,
                          void *stream, void *accept_event);

/* ---------------------------------------------------------------------------
 * sv_verify_chain_early_exit -- sv_verify_chain reading only the rows the walk
 * reaches.  [Lesson] Passo 3 and [Blog] section 4 spec_decode: the walk ends
 * at the first rejection, so the rows after it are never needed.
 *
 * Same arguments, workspace sizes, outputs and accepted / emitted tokens as
 * sv_verify_chain, with these differences:
 *   - temperature must be > 0 (SV_ERR_UNSUPPORTED otherwise: greedy
 *     verification already reads only the verifier rows);
 *   - rows are scheduled position by position; once a sequence's position i
 *     has been judged a rejection (or a fault), the rows of its later
 *     positions that have not been scheduled yet are not read.  How many rows
 *     are skipped depends on scheduling, never the results;
 *   - faults follow the walk: at the first position whose verifier or draft
 *     row has no finite positive softmax sum, or whose token is outside
 *     [0, V), the sequence faults with the bits found there (accept_len 0,
 *     tokens -1); a bad row or token after the first rejection is not seen.
 *     The bonus row faults the sequence only when every position passes;
 *   - out_q_prob, out_p_prob and out_margin are NaN after the first
 *     rejecting position.
 * The workspace may be that of sv_verify_chain_workspace or
 * sv_verify_chain_workspace_host for the same B, N, V.
 * --------------------------------------------------------------------------- */
sv_status sv_verify_chain_early_exit(const void *vlogits, const void *dlogits, sv_dtype dt,
                                     const int32_t *draft_tokens, int B, int N, int V,
                                     float temperature, uint64_t seed, uint64_t step,
                                     int32_t *out_tokens, int32_t *out_accept_len,
                                     float *out_q_prob, float *out_p_prob,
                                     float *out_margin, uint32_t *out_status,
                                     void *workspace, size_t workspace_bytes,
                                     void *stream, void *accept_event);

/* ---------------------------------------------------------------------------
 * sv_verify_tree -- verify a flattened draft tree per sequence.
 * [Blog] section 3 "为什么要树，以及树怎么一次验完" (flattened tree verified in
 * one pass), section 4 eagle_round (walk along best_child with the same
 * accept rule; residual on rejection; bonus at the end), section 5 (EAGLE-2
 * path score = product of draft probabilities).
 *
 * Node 0 of each tree is the root = the last committed token.  parent[b][0] =
 * -1; parent[b][c] in [0, c) for a node; -2 for an unused slot.  token[b][c]
 * is the token of node c; score[b][c] its path score.  The walk starts at the
 * root and repeatedly takes the child with the highest score (ties: the lower
 * slot), at most max_depth steps; this gives path n_0 = 0, n_1..n_D.  Step
 * k = 1..D tests token[n_k] with q = softmax(vlogits[b][n_{k-1}]) and
 * p = softmax(dlogits[b][n_{k-1}]); the bonus comes from vlogits[b][n_D].
 * Only the path's rows are read.
 *
 *   vlogits, dlogits [B][T][V]; parent, token int32 [B][T]; score f32 [B][T].
 * Outputs: out_path_nodes [B][max_depth+1] = n_0..n_a then -1 (n_0 = 0 even
 * for a faulty sequence: the root row is always kept); out_tokens
 * [B][max_depth+1]; out_accept_len [B]; out_q_prob / out_p_prob [B][max_depth]
 * or NULL; out_margin [B][max_depth+1] or NULL (gap at index max_depth);
 * out_status [B] (SV_ROW_BAD_TREE: accept_len 0, tokens -1).
 * A single-path tree gives bit-identical results to sv_verify_chain.
 * --------------------------------------------------------------------------- */
size_t sv_verify_tree_workspace(int B, int T, int max_depth, int V);
/* As sv_verify_chain_workspace_host, for trees. */
size_t sv_verify_tree_workspace_host(int B, int T, int max_depth, int V, sv_dtype dt);
sv_status sv_verify_tree(const void *vlogits, const void *dlogits, sv_dtype dt,
                         const int32_t *parent, const int32_t *token,
                         const float *score, int B, int T, int max_depth,
                         int V, float temperature, uint64_t seed,
                         uint64_t step, int32_t *out_path_nodes,
                         int32_t *out_tokens, int32_t *out_accept_len,
                         float *out_q_prob, float *out_p_prob,
                         float *out_margin, uint32_t *out_status,
                         void *workspace, size_t workspace_bytes,
                         void *stream, void *accept_event);

/* ---------------------------------------------------------------------------
 * sv_tree_build_mask -- the tree attention mask.
 * [Blog] section 3 (each flattened node sees only itself and its ancestors,
 * never its siblings); [Lesson] "Reversão de KV cache" (the verifier runs a
 * non-causal mask that follows the tree).
 *   parent  int32 [B][T] as for sv_verify_tree.
 *   out_mask  uint64 [B][T][(T+63)/64]: bit j of word j/64 of node n is set
 *             iff j == n or j is an ancestor of n.
 *   out_depth int32  [B][T]: number of ancestors; -1 for unused slots.
 * An invalid tree gets an all-zero mask and depth -1 everywhere.
 * --------------------------------------------------------------------------- */
sv_status sv_tree_build_mask(const int32_t *parent, int B, int T,
                             uint64_t *out_mask, int32_t *out_depth,
                             void *stream);

/* ---------------------------------------------------------------------------
 * sv_kv_compact -- KV rollback / compaction.
 * [Lesson] "Reversão de KV cache" (scratch buffer committed on acceptance, or
 * a physical cache with a logical length truncated on rejection) and Passo 4;
 * [Blog] section 3 (copy the accepted path's KV rows together, drop the other
 * branches) and compact_kv in section 4.
 *
 * Cache layout [L][2][B][S][H][D], elem_bytes per element; one token row is
 * H*D*elem_bytes contiguous bytes.  For every sequence b, layer and K/V:
 *   dst row dst_base[b]+k  <-  src row src_base[b]+rows[b][k],  k < n,
 * with n = n_rows[b] + n_rows_add, all reads before any write.  rows == NULL
 * means rows[b][k] = k.  out_kv_len[b] = dst_base[b] + n, or -1 with nothing
 * moved when n is outside [0, P] or above 4096, a row is out of range, or an
 * in-place call (src_kv == dst_kv) has dst_base != src_base or rows not
 * strictly increasing with rows[k] >= k (an accepted tree path always
 * satisfies both).  In place,
 * rows with rows[k] == k are not copied.  src_kv and dst_kv must be the same
 * buffer or not overlap.
 * Typical uses: tree compaction with rows = out_path_nodes, n_rows =
 * out_accept_len, n_rows_add = 1; chain rollback (rows NULL, in place: no
 * bytes move, only the length); scratch commit (src = scratch, src_base 0).
 * --------------------------------------------------------------------------- */
sv_status sv_kv_compact(const void *src_kv, void *dst_kv, int L, int B,
                        int S_src, int S_dst, int H, int D, int elem_bytes,
                        const int32_t *src_base, const int32_t *dst_base,
                        const int32_t *rows, const int32_t *n_rows,
                        int n_rows_add, int P, int32_t *out_kv_len,
                        void *stream);

/* ---------------------------------------------------------------------------
 * sv_verify_chain_noalloc -- sv_verify_chain without a caller workspace.
 * The pages have no counterpart to this call; it exists for callers that must
 * not allocate device memory at all: a plugin inside a host program that owns
 * every device allocation through its own pool, a caller whose memory budget
 * is fixed once at start-up, or code that may run where an allocation would
 * synchronise the device.  Such callers still pass every input and output.
 *
 * Scratch comes from one file-scope static device array of
 * sv_verify_chain_noalloc_max_bytes() bytes (16 MiB), which every GPU that
 * loads this library keeps until the process exits.  It holds the workspace
 * of any call with sv_verify_chain_workspace(B, N, V) <= 16 MiB: for example
 * B = 256, N = 7, V = 128256 (about 9.6 MB), or up to B = 447 at that N and
 * V.
 * The argument checks of sv_verify_chain come first, in its order; then a
 * call whose workspace exceeds the array returns SV_ERR_UNSUPPORTED with a
 * message and enqueues nothing.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress, with that device
 * current); make that first call before any stream capture.  Nothing here
 * calls cudaMalloc, cudaFree or any allocating routine.
 * All calls on a device share the one array, which keeps the previous call's
 * contents; the kernels write every scratch word before reading it, so nothing
 * has to start at zero.  Calls that overlap on the GPU (for example on two
 * streams at once) race on the array: serialise them.
 * Arguments, outputs and errors are otherwise those of sv_verify_chain.
 * --------------------------------------------------------------------------- */
size_t sv_verify_chain_noalloc_max_bytes(void);
sv_status sv_verify_chain_noalloc(const void *vlogits, const void *dlogits,
                                  sv_dtype dt, const int32_t *draft_tokens,
                                  int B, int N, int V, float temperature,
                                  uint64_t seed, uint64_t step,
                                  int32_t *out_tokens, int32_t *out_accept_len,
                                  float *out_q_prob, float *out_p_prob,
                                  float *out_margin, uint32_t *out_status,
                                  void *stream, void *accept_event);

/* ---------------------------------------------------------------------------
 * Dynamic draft tree (EAGLE-2).  [Blog] section 5 (三代之间的变化): the tree
 * grows where the draft is confident; a node's score is the product of the
 * draft probabilities along its path; the best-scored nodes are expanded and
 * the tree is pruned to a node budget.  The caller runs the draft model level
 * by level and calls, per level, sv_tree_expand on the frontier's draft rows
 * and sv_tree_select on the level's candidates; sv_tree_finalize turns all
 * candidates into the [B][T] parent / token / score arrays of sv_verify_tree.
 *
 * sv_tree_expand -- per frontier row (dlogits [B][F][V], sv_dtype dt; the
 * path score of the node it belongs to in frontier_score [B][F]) the K
 * tokens with the largest logits, equal logits in ascending token id
 * (out_token [B][F][K], descending), and their child scores
 * frontier_score * softmax(x / T)[token] (out_score [B][F][K], fp32).
 * T = 0: probability 1 for the first arg max, 0 for the others.  A row with
 * a NaN or +inf logit, or all -inf, or a NaN frontier score (an empty
 * frontier entry) proposes nothing: tokens -1, scores -inf.  1 <= K <= 16 and K <= V (else SV_ERR_INVALID_ARG / UNSUPPORTED).
 * --------------------------------------------------------------------------- */
sv_status sv_tree_expand(const void *dlogits, sv_dtype dt, int B, int F, int V,
                         float temperature, const float *frontier_score, int K,
                         int32_t *out_token, float *out_score, void *stream);

/* sv_tree_select -- per sequence, the indices (out_index [B][K]) of the K
 * best of C candidates (cand_score / cand_token [B][C]): score descending,
 * equal scores in ascending index; a candidate with token -1 is never chosen;
 * missing picks are -1.  C <= 2048. */
sv_status sv_tree_select(const float *cand_score, const int32_t *cand_token, int B,
                         int C, int K, int32_t *out_index, void *stream);

/* sv_tree_finalize -- per sequence, the T-slot tree from C candidates
 * (cand_parent: index of the parent candidate, -1 for candidate 0 = the
 * root; cand_token; cand_score; cand_level, all [B][ldc], the first C
 * columns used; ldc >= C, ldc = C for packed arrays).  The kept nodes are
 * the T first in (score descending, level ascending, index ascending) among
 * the root and the candidates with a token; slots number them in (level
 * ascending, score descending, index ascending).  out_parent [B][T] = slot of
 * the parent candidate (-1 for the root; -2 if it was not kept, which cannot
 * happen when child scores never exceed their parent's); out_token,
 * out_score [B][T]; unused slots: parent -2, token -1, score 0.  C <= 2048,
 * T <= SV_MAX_TREE_NODES. */
sv_status sv_tree_finalize(const int32_t *cand_parent, const int32_t *cand_token,
                           const float *cand_score, const int32_t *cand_level, int B,
                           int C, int ldc, int T, int32_t *out_parent, int32_t *out_token,
                           float *out_score, void *stream);

/* sv_tree_level -- one level of a build, with every step in the library's
 * kernels: sv_tree_expand of the frontier's rows and sv_tree_select of their
 * children, reading and writing a caller-owned candidate table
 * cand_parent / cand_token / cand_score / cand_level, all [B][ldc]
 * (ldc <= 2048), device memory.  Candidate 0 is the root; level l's children
 * are appended at columns [n0, n0 + F*K).
 *   level 1: expands the root (F = 1, n0 = 1, dlogits [B][1][V]) and also
 *            writes candidate 0 (parent -1, token 0, score 1, level 0);
 *            frontier is output only;
 *   level l > 1: frontier [B][K] holds the candidate ids of the F <= K rows
 *            of dlogits [B][F][V] (-1, or an id outside [0, n0): an empty
 *            entry, which proposes nothing); a row's score is read from
 *            cand_score.
 * Each child gets parent = its row's candidate id (-1 for an empty entry),
 * the token and score of sv_tree_expand, and level = l.  On return (in stream
 * order) frontier [B][K] holds the ids of the next frontier, the K best
 * children as sv_tree_select orders them (-1 where there are fewer).  The
 * caller's next n0 is n0 + F*K; after the last level, sv_tree_finalize with
 * C = that n0 and the same ldc builds the tree.
 * Errors, returned before anything is enqueued: SV_ERR_INVALID_ARG for
 * B < 0, F < 1, V < 1, K outside [1, V], a negative or non-finite
 * temperature, level < 1, level 1 with F != 1 or n0 != 1, level > 1 with
 * F > K or n0 < 2, a full table (n0 + F*K > ldc), a null or misaligned
 * pointer, or one the device cannot address; SV_ERR_UNSUPPORTED for K > 16,
 * ldc > 2048 or V above SV_MAX_VOCAB.  B = 0 returns SV_OK with no launch. */
sv_status sv_tree_level(const void *dlogits, sv_dtype dt, int B, int F, int V,
                        float temperature, int K, int level, int n0, int ldc,
                        int32_t *frontier, int32_t *cand_parent, int32_t *cand_token,
                        float *cand_score, int32_t *cand_level, void *stream);

/* ---------------------------------------------------------------------------
 * sv_tree_attention -- tree-masked verifier attention, one layer.
 * [Blog] section 3 (the flattened draft tree is scored in one verifier pass;
 * each node attends to the committed context and to itself and its ancestors,
 * never to a sibling or another branch); [Lesson] "Reversão de KV cache" (the
 * tree pass runs a non-causal mask that follows the tree).  Grouped-query
 * heads: query head h reads KV head h / (Hq / Hkv).
 *
 *   q     bf16 [B][T][Hq][D]      queries of the T tree nodes (node 0 = root)
 *   kv    bf16 [2][B][S][Hkv][D]  this layer of the cache, K then V (one layer
 *                                 of the [L][2][B][S][H][D] layout that
 *                                 sv_kv_compact moves); node n's own K/V row
 *                                 is slot base[b] + n
 *   base  int32 [B]               committed length of each sequence
 *   mask  uint64 [B][T][(T+63)/64] ancestor bitmask (sv_tree_build_mask)
 *   scale > 0, finite             softmax scale (usually 1/sqrt(D))
 *   out   bf16 [B][T][Hq][D]      softmax(scale * q K^T) V over the visible
 *                                 keys
 *   out_lse   fp32 [B][T][Hq] or NULL: natural log of sum exp(scale * q.k)
 *   out_status uint32 [B] or NULL: SV_ROW_BAD_BASE / SV_ROW_TIMEOUT bits are
 *                                 OR-ed in (zero it before the call)
 * Row (b, n, h) sees key slots j < base[b] and base[b] + m for each m < T
 * whose bit is set in node n's mask.  A row with no visible key gets 0 and
 * lse -inf; a sequence with base < 0 or base + T > S gets NaN rows and
 * SV_ROW_BAD_BASE.  Slots at or past base + T are never read into a result
 * (they may hold anything); slots below it must be finite.
 * D = 128 only, Hq / Hkv must divide 128 (else SV_ERR_UNSUPPORTED).  q and kv
 * must be device memory (they are read by tensor-map copies) and q, kv, out
 * 16-byte aligned.  The kernel keeps every wait bounded (2 s); a wait that
 * runs out sets SV_ROW_TIMEOUT and the sequence's rows are left unwritten.
 * --------------------------------------------------------------------------- */
sv_status sv_tree_attention(const void *q, const void *kv, const int32_t *base,
                            const uint64_t *mask, int B, int T, int Hq, int Hkv,
                            int D, int S, float scale, void *out, float *out_lse,
                            uint32_t *out_status, void *stream);
/* sv_tree_attention with the limit of each pipeline wait given: wait_ns
 * nanoseconds (0: the default 2 s).  The pages have no counterpart; it makes
 * the timeout path reachable.  After a wait runs out, the kernel still lets
 * every copy and product it has issued complete (each of those waits bounded
 * by 2 s) before it releases tensor memory and exits, so the context stays
 * usable; the affected sequences get SV_ROW_TIMEOUT. */
sv_status sv_tree_attention_ex(const void *q, const void *kv, const int32_t *base,
                               const uint64_t *mask, int B, int T, int Hq, int Hkv,
                               int D, int S, float scale, void *out, float *out_lse,
                               uint32_t *out_status, uint64_t wait_ns, void *stream);

/* Thread-local message for the last non-OK status returned on this thread. */
const char *sv_last_error(void);

/* ---------------------------------------------------------------------------
 * Launch accounting and tracing (host-side; no device memory).
 * sv_launch_count: kernels this library has launched since it was loaded.
 * sv_trace_enable(1) starts recording a CUDA event pair around every kernel
 * the library launches (on the launching stream); sv_trace_collect waits for
 * the recorded events, writes up to `max` per-kernel aggregates and clears
 * the record.  Returns the number of entries written, or -1 on a CUDA error.
 * --------------------------------------------------------------------------- */
typedef struct {
  char name[40];
  int64_t launches;
  double total_ms;
} sv_trace_entry;

uint64_t sv_launch_count(void);
sv_status sv_trace_enable(int on);
int sv_trace_collect(sv_trace_entry *out, int max);

#ifdef __cplusplus
}
#endif

#endif /* SV_H */
