/*
 * spec_verify.h - C ABI of libspecverify, the GB300 (sm_103a) implementation
 * of the target-model verification step of speculative decoding.
 *
 * The method is the one stated on these pages:
 *   "【大模型基础设施工程】15：推测解码与 MTP" (juejin.cn), §2.1 "算法骨架":
 *     accept draft x_i with probability min(1, p_i(x_i) / q_i(x_i)); at the
 *     first rejection draw one token from norm(max(0, p_i - q_i)) and stop;
 *     if all K drafts are accepted draw one extra token from p_{K+1}.
 *   the same page, "1.2 正确性保证" (inside part 2): the emitted tokens are
 *     distributed exactly as sampling from the target;
 *   the same page, §2.3: 1 <= accept length <= K+1;
 *   the same page, §3.3 "Tree Attention": candidate trees, each node sees only
 *     its ancestors, the longest accepted root path wins;
 *   the same page, §11: greedy (do_sample=False) output equals plain decoding;
 *   "投机解码" (FastDeploy docs), "高效投机解码框架设计": per-sample parallel
 *     sampling+verification; output tokens located by batch id through
 *     padding-free indexing instead of copies and slices.
 *
 * Conventions shared by every entry point
 *   - Tensor pointers are DEVICE pointers to caller-owned, contiguous,
 *     row-major memory.  The library never allocates, frees or retains them;
 *     it reads inputs and writes outputs on `stream`.
 *   - Calls are asynchronous and stream-ordered: they return after queueing
 *     the kernels; nothing is synchronised.  `stream` is a cudaStream_t
 *     (NULL = the legacy default stream).
 *   - The return value reports ARGUMENT errors found on the host before any
 *     launch (nothing is queued then), or SV_ERR_CUDA if a launch failed.
 *   - DATA errors found on the device never trap or hang: they set bits in
 *     the request's status word (SV_REQ_*), and that request emits nothing
 *     (accept_len 0, all token slots -1).
 *   - Token ids are int32.  Unused output token slots hold -1.
 *   - Logits are bfloat16 or IEEE fp32 (sv_dtype).  Every logit must be finite
 *     or -inf (masking); each row that the rule needs must hold at least one
 *     finite logit.  NaN or +inf in a needed row is a data error.  |logit / T|
 *     must be representable in fp32.
 *   - A workspace (device memory, >= spec_verify_workspace_size bytes,
 *     256-byte aligned) holds per-call scratch: chunk records, row summaries
 *     and arrival counters.  Zero-fill a newly allocated workspace once with
 *     spec_verify_workspace_init.  The counters must be zero when a call
 *     starts; every call leaves them zero, and when a workspace is used with a
 *     different (B, K, mode) than on its previous call, the library first
 *     zero-fills the counter region on the call's stream (one small
 *     cudaMemsetAsync).  Calls that share a workspace must be ordered on one
 *     stream: concurrent calls need separate workspaces.
 */
#ifndef SPEC_VERIFY_H_
#define SPEC_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* sv_stream_t;

typedef enum sv_status {
  SV_OK = 0,
  SV_ERR_NULL = 1,        /* a required pointer is NULL */
  SV_ERR_SHAPE = 2,       /* B, K, V, N or max_depth outside the supported range */
  SV_ERR_DTYPE = 3,       /* unknown sv_dtype */
  SV_ERR_TEMPERATURE = 4, /* temperature negative, NaN or infinite */
  SV_ERR_TREE = 5,        /* tree parent stride neither 0 nor N */
  SV_ERR_WORKSPACE = 6,   /* workspace NULL, not 256-byte aligned, or too small */
  SV_ERR_CUDA = 7,        /* a CUDA runtime call or kernel launch failed */
  SV_ERR_FILTER = 8       /* top_k negative, top_p outside (0, 1], or eps / delta negative */
} sv_status;

typedef enum sv_dtype { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/* Per-request device status bits (out_status). */
#define SV_REQ_BAD_TOKEN 1     /* a draft / tree token outside [0, V) */
#define SV_REQ_BAD_LOGITS 2    /* a needed row has NaN or +inf, or no finite logit */
#define SV_REQ_BAD_DRAFT_LEN 4 /* draft_lens[b] outside [0, K] */
#define SV_REQ_TIMEOUT 8       /* a bounded wait for staged logits gave up (device fault, or
                                  the limit of spec_verify_set_wait_limit_ns ran out) */
#define SV_REQ_BAD_TREE 16     /* the request's parent array is not a tree of depth <= max_depth */

/* Limits. */
#define SV_MAX_K 31             /* draft positions per request */
#define SV_MAX_B 65536          /* requests per call */
#define SV_MAX_V (1 << 24)      /* vocabulary size */
#define SV_MAX_TREE_NODES 256   /* candidate nodes per tree (root excluded) */
#define SV_MAX_NGRAM 32         /* longest n-gram the proposer matches */

/* Bytes of workspace that spec_verify_sample / _greedy need for B requests
 * of K draft positions over a vocabulary of V (the dense-draft sampling case,
 * the largest).  spec_verify_tree needs none.  Returns 0 if out of range. */
size_t spec_verify_workspace_size(int B, int K, int V);

/* Zero-fill a workspace on `stream` (one cudaMemsetAsync).  Needed once per
 * workspace before its first use. */
sv_status spec_verify_workspace_init(void* workspace, size_t ws_bytes, sv_stream_t stream);

/* Rejection-sampling verification ("推测解码与 MTP" §2.1).
 *
 *   target_logits  [B, K+1, V] dtype: row i < K scores draft position i,
 *                  row K is the extra (bonus) position.
 *   draft_logits   [B, K, V] dtype, or NULL.  Given: q_i = softmax(d_i / T),
 *                  the same temperature as the target (the drafts are assumed
 *                  sampled from exactly that q).  NULL: one-hot drafts from a
 *                  deterministic proposer (n-gram / prompt lookup), q_i is the
 *                  point mass at x_i: acceptance probability p_i(x_i), residual
 *                  p_i with x_i removed and renormalised.
 *   draft_tokens   [B, K] int32, the drafts x_i.  May be NULL when K == 0.
 *   uniforms       [B, K+1] fp32 in [0, 1): column i < K drives the test at
 *                  position i (accept iff u_i * q_i(x_i) < p_i(x_i)); column K
 *                  drives the residual or bonus draw: the emitted token is the
 *                  smallest j whose cumulative weight exceeds u_K times the total.
 *   temperature    T > 0: p_i = softmax(target_i / T).  T == 0 selects the greedy
 *                  rule of spec_verify_greedy (draft_logits and uniforms unused;
 *                  out_accept_prob reports 1 for a match and 0 for a mismatch).
 *   out_tokens     [B, K+1] int32: x_0 .. x_{n-1}, then the drawn token, then -1.
 *   out_accept_len [B] int32: n + 1 emitted tokens (1 <= n+1 <= K_b+1), or 0 for
 *                  a request with a data error.
 *   dtype, B, K, V 1 <= B <= SV_MAX_B, 0 <= K <= SV_MAX_K, 1 <= V <= SV_MAX_V.
 *   draft_lens     [B] int32 or NULL: per-request draft count K_b <= K (ragged
 *                  drafts).  Rows beyond K_b are never read; the bonus position
 *                  of request b is row K_b; the draw still uses column K.
 *   out_cu_accept  [B+1] int32 or NULL: exclusive prefix sum of out_accept_len.
 *   out_packed     [B*(K+1)] int32 or NULL: the emitted tokens of all requests
 *                  back to back (request b at out_cu_accept[b]..), then -1.
 *   out_batch_id   [B*(K+1)] int32 or NULL: the request of each packed token, -1
 *                  past the end.  (Any of the three packed outputs may be given
 *                  alone; out_cu_accept is computed either way.)
 *   out_accept_prob [B, K] fp32 or NULL: min(1, p_i(x_i)/q_i(x_i)) at each
 *                  tested position (i <= n, i < K_b), -1 elsewhere.
 *   out_status     [B] int32 or NULL: SV_REQ_* bits per request.
 *   workspace, ws_bytes  see the conventions above.
 */
sv_status spec_verify_sample(const void* target_logits, const void* draft_logits,
                             const int32_t* draft_tokens, const float* uniforms,
                             float temperature, int32_t* out_tokens, int32_t* out_accept_len,
                             sv_dtype dtype, int B, int K, int V, const int32_t* draft_lens,
                             int32_t* out_cu_accept, int32_t* out_packed,
                             int32_t* out_batch_id, float* out_accept_prob,
                             int32_t* out_status, void* workspace, size_t ws_bytes,
                             sv_stream_t stream);

/* Greedy verification ("推测解码与 MTP" §11, temperature 0): x_i is accepted
 * while it equals the argmax of target row i (lowest index among equal
 * maxima; -0.0 == +0.0); the first mismatch emits that argmax; if all K_b
 * match, the argmax of row K_b is the extra token.  Arguments as in
 * spec_verify_sample.  Bit-exact: the argmax is taken on the stored values. */
sv_status spec_verify_greedy(const void* target_logits, const int32_t* draft_tokens,
                             int32_t* out_tokens, int32_t* out_accept_len, sv_dtype dtype,
                             int B, int K, int V, const int32_t* draft_lens,
                             int32_t* out_cu_accept, int32_t* out_packed,
                             int32_t* out_batch_id, int32_t* out_status, void* workspace,
                             size_t ws_bytes, sv_stream_t stream);

/* Grammar-constrained verification ("Speculative Decoding" (LMDeploy docs),
 * "投机解码与结构化输出" / "工作原理"): with structured output (a JSON schema, a
 * regular expression) each position may only emit the tokens its grammar
 * state allows.  The mask of position i is applied to target row i - and to
 * draft row i, since the draft was proposed under the same mask - before the
 * rule runs: a ruled-out token has probability 0, so it is never accepted,
 * drawn or taken as the argmax.  The masks of positions 1..K depend on the
 * drafts before them; the caller's grammar matcher computes them all (on a
 * fork advanced through the drafts) before the call.
 *
 *   token_mask  [B, K+1, ceil(V/32)] 32-bit words, 4-byte aligned: request b,
 *               position i allows token j iff bit j % 32 of word j / 32 of row
 *               (b, i) is set.  Bits at j >= V are ignored.  When the rows are
 *               16-byte aligned (16-byte aligned base and ceil(V/32) a multiple
 *               of 4) the words travel with the logits in the same bulk copies;
 *               otherwise they are read word by word.
 * A needed position whose mask leaves no finite logit is a data error
 * (SV_REQ_BAD_LOGITS).  NULL or misaligned token_mask: SV_ERR_NULL.  All other
 * arguments, results and the workspace size are those of spec_verify_sample
 * and spec_verify_greedy. */
sv_status spec_verify_sample_masked(const void* target_logits, const void* draft_logits,
                                    const int32_t* draft_tokens, const float* uniforms,
                                    float temperature, const uint32_t* token_mask,
                                    int32_t* out_tokens, int32_t* out_accept_len, sv_dtype dtype,
                                    int B, int K, int V, const int32_t* draft_lens,
                                    int32_t* out_cu_accept, int32_t* out_packed,
                                    int32_t* out_batch_id, float* out_accept_prob,
                                    int32_t* out_status, void* workspace, size_t ws_bytes,
                                    sv_stream_t stream);
sv_status spec_verify_greedy_masked(const void* target_logits, const int32_t* draft_tokens,
                                    const uint32_t* token_mask, int32_t* out_tokens,
                                    int32_t* out_accept_len, sv_dtype dtype, int B, int K, int V,
                                    const int32_t* draft_lens, int32_t* out_cu_accept,
                                    int32_t* out_packed, int32_t* out_batch_id,
                                    int32_t* out_status, void* workspace, size_t ws_bytes,
                                    sv_stream_t stream);

/* Verification of top-k / top-p filtered sampling (the vLLM Ascend guide's
 * examples sample with SamplingParams(temperature=0.8, top_p=0.95); "推测解码与
 * MTP" §8.3 non-greedy decoding with wide top-p).  Every sampled
 * distribution - target rows and, with dense drafts, draft rows - is the
 * tempered softmax of the (grammar-masked) logits filtered as follows, and
 * the drafts are assumed drawn from the filtered draft distributions:
 *   top_k > 0 keeps the tokens whose logit is >= the k-th largest logit of
 *     the row (counted with multiplicity, so ties at the cut are all kept),
 *     then renormalises; top_k = 0 (or >= V) switches it off;
 *   top_p < 1 then keeps a token when the probability mass of the tokens
 *     with a strictly larger logit is below top_p (the smallest set of
 *     leading logit values whose mass reaches top_p, ties kept together),
 *     then renormalises; top_p = 1 switches it off.
 * The acceptance test, the residual norm(max(0, p' - q')) and the bonus draw
 * use the filtered p', q'.  temperature == 0 is the greedy rule (filters do
 * not change the argmax).  token_mask: as in spec_verify_sample_masked, or
 * NULL.  Each row of a filtered call is taken by one CTA: V * sizeof(logit)
 * must not exceed 512 KB (V <= 262144 for bf16, 131072 for fp32), else
 * SV_ERR_SHAPE.  SV_ERR_FILTER for a negative top_k or
 * top_p outside (0, 1].
 *   out_cut   [B, R] fp32 or NULL, R = K+1 (one-hot drafts) or 2K+1 (draft
 *             logits): the lowest logit each filtered distribution keeps -
 *             row i <= K target position i, row K+1+i the draft of position
 *             i; NaN for rows the request does not need (beyond K_b, or a
 *             request with a bad draft length); -inf for a row without a
 *             finite max.  Written only when a filter is active (top_k in
 *             (0, V) or top_p < 1).  With top-p the cut is where the fp32
 *             mass of the leading value classes reaches top_p; it tells a
 *             caller (or a test) which value classes were kept.
 * All other arguments, results and the workspace size are those of
 * spec_verify_sample. */
sv_status spec_verify_sample_filtered(const void* target_logits, const void* draft_logits,
                                      const int32_t* draft_tokens, const float* uniforms,
                                      float temperature, int top_k, float top_p,
                                      const uint32_t* token_mask, int32_t* out_tokens,
                                      int32_t* out_accept_len, sv_dtype dtype, int B, int K, int V,
                                      const int32_t* draft_lens, int32_t* out_cu_accept,
                                      int32_t* out_packed, int32_t* out_batch_id,
                                      float* out_accept_prob, float* out_cut,
                                      int32_t* out_status, void* workspace, size_t ws_bytes,
                                      sv_stream_t stream);

/* Typical acceptance ("推测解码与 MTP" §10.4: the rule of the original Medusa,
 * an approximation that is not exactly lossless, also offered by EAGLE).
 * Draft x_i passes when p_i(x_i) > min(eps, delta * exp(-H(p_i))), with p_i
 * the tempered target distribution of position i and H its entropy in nats;
 * positions are tested in order, and at the first failure n (or at K_b when
 * all pass) one token is drawn from p_n itself with uniforms[b, K] (inverse
 * CDF: the smallest j whose cumulative probability exceeds u).  There is no
 * residual: the output follows the rule, not the target distribution.
 *   eps, delta      the rule's two thresholds (Medusa's defaults are 0.09 and
 *                   0.3), finite and >= 0, else SV_ERR_FILTER.
 *   temperature     T > 0; T == 0 applies the greedy rule instead.
 *   out_accept_prob p_i(x_i) at each tested position, -1 elsewhere.
 * Drafts are one-hot (no draft logits).  uniforms [B, K+1], of which only
 * column K is used.  All other arguments, results and the workspace size are
 * those of spec_verify_sample. */
sv_status spec_verify_typical(const void* target_logits, const int32_t* draft_tokens,
                              const float* uniforms, float temperature, float eps, float delta,
                              int32_t* out_tokens, int32_t* out_accept_len, sv_dtype dtype, int B,
                              int K, int V, const int32_t* draft_lens, int32_t* out_cu_accept,
                              int32_t* out_packed, int32_t* out_batch_id, float* out_accept_prob,
                              int32_t* out_status, void* workspace, size_t ws_bytes,
                              sv_stream_t stream);

/* Typical acceptance on a candidate tree (§10.4 with §3.3).  Node n passes
 * when its parent passed (the root always does) and its token passes the
 * typical test under its parent's distribution; the result is the deepest
 * passing node (the lowest id among equally deep ones): the tokens of its
 * root path, then one token drawn from its own distribution with
 * uniforms[b].  Rows of passing nodes must be valid (SV_REQ_BAD_LOGITS).
 *   target_logits, tree_parent, parent_stride, tree_tokens, out_tokens,
 *   out_path, out_accept_len, out_status, max_depth: as in spec_verify_tree.
 *   uniforms [B] fp32 in [0, 1).  temperature > 0; eps, delta as in
 *   spec_verify_typical.  workspace: >= spec_verify_tree_workspace_size(B, N,
 *   V) bytes, 256-byte aligned, zero-filled once (spec_verify_workspace_init).
 * Every row of the tree is read once (all candidate rows are reduced in
 * parallel). */
size_t spec_verify_tree_workspace_size(int B, int N, int V);
sv_status spec_verify_tree_typical(const void* target_logits, const int32_t* tree_parent,
                                   int parent_stride, const int32_t* tree_tokens,
                                   const float* uniforms, float temperature, float eps,
                                   float delta, int32_t* out_tokens, int32_t* out_accept_len,
                                   sv_dtype dtype, int B, int N, int V, int max_depth,
                                   int32_t* out_path, int32_t* out_status, void* workspace,
                                   size_t ws_bytes, sv_stream_t stream);

/* Lossless tree verification by rejection sampling ("推测解码与 MTP" §10.4:
 * the methods that verify by rejection sampling, EAGLE among them, are
 * lossless; the candidate trees of §3.3 "Tree Attention" and §4.2, whose
 * nodes are each head's top-k candidates).  Every candidate is a
 * deterministic (one-hot) draft of the distribution at its parent.  From the
 * root: with p the tempered target distribution at the current node and w = p,
 * the node's children are tested in increasing id - child c with token x_c
 * is accepted iff u_c < w(x_c) / sum(w), and a rejected child's token leaves
 * w (w(x_c) = 0); the first accepted child's token is emitted and the walk
 * moves to it; when no child is accepted (or at a leaf) one token is drawn
 * from w / sum(w) with u_0 (the smallest j whose cumulative weight exceeds
 * u_0 times the total) and the walk ends.  Each emitted token is distributed
 * exactly as the target's distribution at its node; a token repeated among
 * siblings has no mass left when its turn comes and is rejected.
 *   uniforms  [B, N+1] fp32 in [0, 1): column c (1..N) drives the test of
 *             node c, column 0 the final draw.
 *   temperature  T > 0; T == 0 runs the greedy walk of spec_verify_tree
 *             (uniforms and workspace unused).
 *   target_logits, tree_parent, parent_stride, tree_tokens, out_tokens,
 *   out_path, out_accept_len, out_status, max_depth: as in spec_verify_tree
 *   (out_tokens: the accepted candidates' tokens, then the drawn token).
 *   workspace: >= spec_verify_tree_workspace_size(B, N, V) bytes, as for
 *   spec_verify_tree_typical.
 * Every row of the tree is read once (all candidate rows are reduced in
 * parallel, each row's sums leaving out its children's tokens); only the
 * walked rows must be valid (SV_REQ_BAD_LOGITS). */
sv_status spec_verify_tree_sample(const void* target_logits, const int32_t* tree_parent,
                                  int parent_stride, const int32_t* tree_tokens,
                                  const float* uniforms, float temperature, int32_t* out_tokens,
                                  int32_t* out_accept_len, sv_dtype dtype, int B, int N, int V,
                                  int max_depth, int32_t* out_path, int32_t* out_status,
                                  void* workspace, size_t ws_bytes, sv_stream_t stream);

/* Greedy tree verification (Medusa / EAGLE; "推测解码与 MTP" §3.3).
 *
 *   target_logits  [B, N+1, V] dtype: row 0 is the root (the last committed
 *                  token), row n the target's logits after candidate node n.
 *   tree_parent    [N] or [B, N] int32 (device): parent of node n (n = 1..N)
 *                  at index n-1; a tree needs 0 <= parent < n (an earlier
 *                  node; breadth-first order qualifies) and no node deeper
 *                  than max_depth - a request whose array breaks this gets
 *                  SV_REQ_BAD_TREE and emits nothing.
 *   parent_stride  0: every request shares the one [N] tree; N: request b's
 *                  tree is tree_parent[b*N .. b*N+N) (EAGLE-2's dynamic trees,
 *                  built per request on the device, §4.3).  Other values:
 *                  SV_ERR_TREE.
 *   tree_tokens    [B, N] int32: the candidate token of node n at index n-1.
 *   out_tokens     [B, max_depth+1] int32: the target argmax at each node of the
 *                  accepted path (root first): the accepted node tokens followed
 *                  by the extra token; -1 after.
 *   out_accept_len [B] int32: accepted nodes + 1, or 0 on a data error.
 *   N, max_depth   0 <= N <= SV_MAX_TREE_NODES; max_depth >= the tree's depth.
 *   out_path       [B, max_depth+1] int32 or NULL: node ids of the path from the
 *                  root (0) on, -1 after.
 *   out_status     [B] int32 or NULL: SV_REQ_* bits.
 * A node is accepted when its token equals the argmax at its parent and its
 * parent is accepted.  With distinct sibling tokens (top-k candidates) the
 * accepted nodes form one chain and the walk returns the longest accepted
 * path; if a caller repeats a token among siblings, the lowest node id wins.
 * Only the rows on the accepted path are read. */
sv_status spec_verify_tree(const void* target_logits, const int32_t* tree_parent,
                           int parent_stride, const int32_t* tree_tokens, int32_t* out_tokens,
                           int32_t* out_accept_len, sv_dtype dtype, int B, int N, int V,
                           int max_depth, int32_t* out_path, int32_t* out_status,
                           sv_stream_t stream);

/* The longest time a kernel waits for logits it staged in shared memory
 * before it gives up: the call then marks every request SV_REQ_TIMEOUT (the
 * workspace stays usable; the next call starts clean).  Default 2 s, which
 * only a device fault can exhaust; a serving loop with a watchdog may set
 * less.  0 makes the waits give up at once, without polling - every call
 * then reports SV_REQ_TIMEOUT, which is how the timeout path is tested.
 * Process-wide; applies to the calls queued after it.  Always SV_OK. */
sv_status spec_verify_set_wait_limit_ns(uint64_t limit_ns);
uint64_t spec_verify_wait_limit_ns(void);

/* n-gram (prompt-lookup) proposer: the step before verification that makes
 * the one-hot drafts ("投机解码" (FastDeploy docs), "使用 Ngram 解码": drafts
 * come from matching an n-gram window against the prompt and the generated
 * tokens; the vLLM Ascend guide's n-gram example, prompt_lookup_max = 4 and 5
 * speculative tokens; "推测解码与 MTP" §9.1 prompt lookup).
 *
 * For n = n_max down to n_min, the last n tokens of request b's context
 * c = tokens[b, 0 .. lens[b]) are looked up earlier in c: the match is the
 * EARLIEST start s with c[s .. s+n) equal to them and at least one token
 * after it (s + n < lens[b]).  The first n that matches decides; the drafts
 * are the tokens after the match, c[s+n .. min(s+n+K, lens[b])).
 *
 *   tokens          [B, L] int32: request b's context in its first lens[b]
 *                   entries (prompt then generated tokens); the rest is never
 *                   read.  Any int32 values (they are only compared).
 *   lens            [B] int32, 0 <= lens[b] <= L; outside that range the
 *                   request gets no drafts and SV_REQ_BAD_DRAFT_LEN.
 *   n_min, n_max    1 <= n_min <= n_max <= SV_MAX_NGRAM.
 *   K               0 <= K <= SV_MAX_K drafts per request.
 *   out_drafts      [B, K] int32: the drafts, -1 after them.
 *   out_draft_lens  [B] int32: how many (0..K); pass it as draft_lens to
 *                   spec_verify_sample with draft_logits = NULL.
 *   out_match       [B] int32 or NULL: the start s, or -1 without a match.
 *   out_status      [B] int32 or NULL: SV_REQ_* bits.
 * B * L < 2^31.  One pass over each context; no workspace. */
sv_status spec_ngram_propose(const int32_t* tokens, const int32_t* lens, int B, int L,
                             int n_min, int n_max, int K, int32_t* out_drafts,
                             int32_t* out_draft_lens, int32_t* out_match, int32_t* out_status,
                             sv_stream_t stream);

/* Allocation-free variant of spec_verify_sample.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory - for example an inference runtime that reserves the
 * whole device for its own pool and hands a plugin only its input and output
 * buffers, or a path on which a cudaMalloc (which may synchronise the device)
 * is not allowed.
 *
 * Arguments and results are those of spec_verify_sample, without the
 * workspace.  Its scratch is one fixed device array of
 * SV_NOALLOC_SCRATCH_BYTES inside the library, held by every GPU that loads
 * the library until the process exits; the call itself allocates nothing.
 *   - Limit: spec_verify_workspace_size(B, K, V) must not exceed
 *     SV_NOALLOC_SCRATCH_BYTES; larger problems return SV_ERR_WORKSPACE with
 *     nothing queued.  (B = 256, K = 5, V = 152064 needs about 3.4 MB.)
 *   - Each call looks up the array's device address on the current device
 *     (cudaGetSymbolAddress; it queues no work, and a device reset that
 *     reloads the module cannot leave a stale address behind).  The first
 *     call on a device may load the library's module there: make that first
 *     call before any stream capture.
 *   - Every call on a device uses the same array, which keeps the previous
 *     call's contents; each call first clears, on its stream, the counters
 *     that must start at zero.  Calls that overlap on the GPU (different
 *     streams, or different host threads without ordering) race on the
 *     array and give wrong results: order them on one stream. */
#define SV_NOALLOC_SCRATCH_BYTES (8u << 20)
sv_status spec_verify_sample_noalloc(const void* target_logits, const void* draft_logits,
                                     const int32_t* draft_tokens, const float* uniforms,
                                     float temperature, int32_t* out_tokens,
                                     int32_t* out_accept_len, sv_dtype dtype, int B, int K, int V,
                                     const int32_t* draft_lens, int32_t* out_cu_accept,
                                     int32_t* out_packed, int32_t* out_batch_id,
                                     float* out_accept_prob, int32_t* out_status,
                                     sv_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char* spec_verify_status_string(sv_status status);

/* Library ABI version: 100 * major + minor. */
int spec_verify_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H_ */
