/*
 * spec_oracle.c - plain fp64 CPU oracle for the speculative-decoding
 * verification step.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package's smoke check and
 * the benchmark's CPU-baseline leg may load this code.  The product path
 * (the CUDA library) never calls it, shares no source with it and does not
 * fall back to it.
 *
 * What it computes follows these pages:
 *   [SD]   "【大模型基础设施工程】15：推测解码与 MTP" (juejin.cn)
 *          §2.1 "算法骨架" (the verification rule), the following "1.2 正确性
 *          保证" (exactness), §2.3 (1 <= accept length <= K+1),
 *          §3.3 "Tree Attention" (ancestor-only paths, longest accepted path),
 *          §11 (the hand-written sketch: softmax over the K+1 target positions,
 *          strict "r < min(1, p/q)" test, clamp-then-normalise residual).
 *   [FD]   "投机解码" (FastDeploy docs), "高效投机解码框架设计"
 *          (per-sample parallel verify; padding-free batch-id lookup).
 *   [LD]   "Speculative Decoding" (LMDeploy docs), "投机解码与结构化输出",
 *          "工作原理" (grammar masks applied to the target logits of every
 *          verified position, and to the draft's).
 *   [VA]   "Speculative Decoding Guide" (vLLM Ascend docs): the examples'
 *          SamplingParams(temperature=0.8, top_p=0.95) (top-p filtering of
 *          the sampled distributions), with "推测解码与 MTP" §8.3 (non-greedy
 *          decoding with wide top-p).
 *   [SD] §10.4 also names typical acceptance, the approximate (not exactly
 *          lossless) rule of the original Medusa, offered by EAGLE too; and
 *          says that the methods which verify by rejection sampling, EAGLE
 *          among them, are lossless - with EAGLE's candidate trees (§4.2
 *          "结合 tree attention"; §4.3 dynamic trees that differ per request).
 *
 * Every quantity is computed in double precision, one request at a time,
 * with plain serial loops: no blocking, fusion or reordering.  Where the
 * pages leave a step open, the reading taken is named R1..R21 in the
 * comments (the same labels are used in the design notes).
 *
 * Logit storage: dtype 0 = IEEE fp32, dtype 1 = bfloat16 given as raw
 * 16-bit patterns.  Both are widened exactly to double before any
 * arithmetic.
 *
 * Per-request status bits (0 = valid request):
 *   1  a draft / tree token outside [0, V)
 *   2  a needed logit row holds NaN or +inf, or holds no finite value
 *   4  a draft length outside [0, K]
 *   16 a parent array that is not a tree of depth <= max_depth (a parent
 *      that is not an earlier node)
 * A request with a nonzero status emits nothing: accept_len = 0 and all its
 * token slots are -1.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_BAD_TOKEN 1
#define OR_BAD_LOGITS 2
#define OR_BAD_DRAFT_LEN 4
#define OR_BAD_TREE 16

#define OR_FLAG_ACCEPT 1 /* u within 1e-5 (relative) of the acceptance threshold */
#define OR_FLAG_CDF 2    /* u*W within 1e-5*W of a CDF step around the chosen token */
#define OR_FLAG_CUT 4    /* a top-p cut of the position's rows within 1e-5 of moving */

#define OR_FLAG_TOL 1e-5

/* ------------------------------------------------------------------ */
/* input decoding                                                      */
/* ------------------------------------------------------------------ */

static double load_logit(const void* base, int dtype, size_t idx) {
  if (dtype == 0) return (double)((const float*)base)[idx];
  /* bfloat16 is the top half of an IEEE binary32 word */
  uint32_t word = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &word, sizeof f);
  return (double)f;
}

static void load_row(const void* base, int dtype, size_t row, int V, double* out) {
  for (int j = 0; j < V; ++j) out[j] = load_logit(base, dtype, row * (size_t)V + (size_t)j);
}

/* R12: a row is usable when every entry is finite or -inf (masking) and at
 * least one entry is finite. */
static int row_is_valid(const double* l, int V) {
  int any_finite = 0;
  for (int j = 0; j < V; ++j) {
    if (isnan(l[j])) return 0;
    if (isinf(l[j]) && l[j] > 0) return 0;
    if (isfinite(l[j])) any_finite = 1;
  }
  return any_finite;
}

/* Grammar mask [LD "工作原理"]: the mask of position i is applied to the
 * logits of position i before anything else is computed from them.  R18:
 * one row of ceil(V/32) 32-bit words per position; token j is allowed when
 * bit (j mod 32) of word floor(j/32) is set.  A disallowed token's logit
 * becomes -inf, so it has probability 0 and never wins an argmax; a row
 * left with no finite logit is unusable (R12).  mask_row NULL: no mask. */
static void apply_token_mask(double* l, int V, const uint32_t* mask_row) {
  if (!mask_row) return;
  for (int j = 0; j < V; ++j)
    if (!((mask_row[j / 32] >> (j % 32)) & 1u)) l[j] = -INFINITY;
}

/* The mask row of position i of request b (R18: draft row i shares it). */
static const uint32_t* mask_row_of(const uint32_t* mask, int K, int V, size_t b, int i) {
  if (!mask) return NULL;
  const size_t words = ((size_t)V + 31) / 32;
  return mask + (b * (size_t)(K + 1) + (size_t)i) * words;
}

/* ------------------------------------------------------------------ */
/* the steps                                                           */
/* ------------------------------------------------------------------ */

/* Tempered softmax [SD §11: softmax over the vocabulary at each target
 * position; temperature as in the SamplingParams of the vLLM guide]:
 *   p[j] = exp(l[j]/T - M) / sum_k exp(l[k]/T - M),  M = max_k l[k]/T.
 * Subtracting M does not change the value; it keeps exp() in range. */
void sv_oracle_tempered_softmax(const double* l, int V, double T, double* p) {
  double M = -INFINITY;
  for (int j = 0; j < V; ++j) {
    double s = l[j] / T;
    if (s > M) M = s;
  }
  double Z = 0.0;
  for (int j = 0; j < V; ++j) {
    p[j] = exp(l[j] / T - M);
    Z += p[j];
  }
  for (int j = 0; j < V; ++j) p[j] /= Z;
}

/* Argmax with the lowest index among equal maxima (R8; -0.0 == +0.0). */
int sv_oracle_argmax(const double* l, int V) {
  int best = 0;
  for (int j = 1; j < V; ++j)
    if (l[j] > l[best]) best = j;
  return best;
}

/* Inverse-CDF draw from non-negative weights w (unnormalised):
 *   C_j = sum_{k<=j} w_k,  W = C_{V-1},
 *   token = the smallest j with C_j > u*W;
 *   if no j qualifies (only through rounding), the largest j with w_j > 0 (R4).
 * *margin receives min(|u*W - C_{t-1}|, |u*W - C_t|) / W, the distance of
 * the draw to the nearer edge of the chosen token's CDF step. */
int sv_oracle_inverse_cdf(const double* w, int V, double u, double* margin) {
  double W = 0.0;
  for (int j = 0; j < V; ++j) W += w[j];
  double target = u * W;
  double C = 0.0, C_prev = 0.0;
  int t = -1;
  for (int j = 0; j < V; ++j) {
    C_prev = C;
    C += w[j];
    if (C > target) {
      t = j;
      break;
    }
  }
  if (t < 0) {
    for (int j = V - 1; j >= 0; --j)
      if (w[j] > 0) {
        t = j;
        break;
      }
    C_prev = W - (t >= 0 ? w[t] : 0.0);
    C = W;
  }
  if (margin) {
    double a = fabs(target - C_prev), b = fabs(target - C);
    *margin = (W > 0) ? (a < b ? a : b) / W : 0.0;
  }
  return t;
}

/* The normalised CDF step [C_{t-1}/W, C_t/W) that token t occupies in a
 * draw from weights w (NaN if t is out of range or there is no mass): the
 * window a draw made elsewhere is checked against. */
static void cdf_step(const double* w, int V, int32_t t, double* out) {
  double W = 0.0, below = 0.0;
  for (int j = 0; j < V; ++j) {
    if (j < t) below += w[j];
    W += w[j];
  }
  int ok = t >= 0 && t < V && W > 0;
  out[0] = ok ? below / W : NAN;
  out[1] = ok ? (below + w[t]) / W : NAN;
}

/* Top-k / top-p filtering of one row's distribution [VA: SamplingParams
 * with top_p; SD §8.3].  R20: l are the row's logits (after any grammar
 * mask), p its tempered softmax; both filters keep whole value classes
 * (tokens with equal logits are kept or dropped together):
 *   top_k > 0: keep the tokens whose logit is >= the k-th largest logit,
 *     counted with multiplicity; renormalise;
 *   top_p < 1: over what is left, keep the tokens for which the mass of
 *     tokens with a strictly larger logit is < top_p (so the smallest set of
 *     leading value classes whose mass reaches top_p); renormalise.
 * The cut is flagged (return OR_FLAG_CUT) when the mass in front of the
 * last kept class, or in front of the first dropped one, lies within
 * OR_FLAG_TOL of top_p: an fp32 evaluation may keep one class more or less.
 * order: scratch of V ints.
 *
 * Forced cut (checking a cut made elsewhere): when `forced` is not NaN, the
 * top-k step runs as above and then the tokens with a logit >= forced are
 * kept (renormalised) instead of the top-p rule's own choice, and no flag is
 * returned.  *margin then receives how far that cut is from the rule:
 *   0    it is the rule's own cut;
 *   d    it differs, and d is the largest distance |F - top_p| over the
 *        classes it decides the other way (F = the mass of the strictly
 *        larger logits): F(forced) - top_p when it keeps classes the rule
 *        drops, top_p - F(next class) when it drops classes the rule keeps;
 *   NaN  it is not admissible: not the logit of a token the top-k step
 *        keeps, a top-k-only cut other than the k-th largest value, or a
 *        distance beyond OR_FLAG_TOL. */
static _Thread_local const double* g_sort_key; /* qsort has no context argument */
static int by_logit_desc(const void* a, const void* b) {
  double x = g_sort_key[*(const int*)a], y = g_sort_key[*(const int*)b];
  if (x > y) return -1;
  if (x < y) return 1;
  return (*(const int*)a > *(const int*)b) - (*(const int*)a < *(const int*)b);
}

static int filter_top_k_top_p(const double* l, double* p, int V, int top_k, double top_p,
                              int* order, double forced, double* margin) {
  int use_k = top_k > 0 && top_k < V, use_p = top_p < 1.0;
  if (!use_k && !use_p) return 0;
  for (int j = 0; j < V; ++j) order[j] = j;
  g_sort_key = l;
  qsort(order, (size_t)V, sizeof(int), by_logit_desc);
  double vk = -INFINITY;
  if (use_k) {
    vk = l[order[top_k - 1]];
    double Z = 0.0;
    for (int j = 0; j < V; ++j) {
      if (l[j] < vk) p[j] = 0.0;
      Z += p[j];
    }
    for (int j = 0; j < V; ++j) p[j] /= Z;
  }
  if (!isnan(forced)) {
    /* the rule's own cut: the lowest kept value class */
    double own = vk;
    if (use_p) {
      double above = 0.0;
      for (int t = 0; t < V;) {
        int e = t;
        double mass = 0.0;
        while (e < V && l[order[e]] == l[order[t]]) mass += p[order[e++]];
        if (!(above < top_p) || l[order[t]] < vk) break;
        own = l[order[t]];
        above += mass;
        t = e;
      }
    }
    int is_class = 0;
    double front = 0.0, through = 0.0;
    for (int j = 0; j < V; ++j) {
      if (l[j] == forced && l[j] >= vk) is_class = 1;
      if (l[j] > forced) front += p[j];
      if (l[j] >= forced) through += p[j];
    }
    double d = NAN;
    if (is_class && forced == own)
      d = 0.0;
    else if (is_class && use_p)
      d = forced < own ? front - top_p : top_p - through;
    if (!(d <= OR_FLAG_TOL)) d = NAN;
    if (margin) *margin = d;
    if (use_p) {
      double Z = 0.0;
      for (int j = 0; j < V; ++j) {
        if (l[j] < forced) p[j] = 0.0;
        Z += p[j];
      }
      for (int j = 0; j < V; ++j) p[j] /= Z;
    }
    return 0;
  }
  int flag = 0;
  if (use_p) {
    double above = 0.0; /* mass of the classes before the current one */
    int t = 0, dropping = 0;
    while (t < V) {
      int e = t;
      double mass = 0.0;
      while (e < V && l[order[e]] == l[order[t]]) mass += p[order[e++]];
      if (!dropping && above < top_p) {
        if (top_p - above <= OR_FLAG_TOL) flag = OR_FLAG_CUT;
      } else {
        if (!dropping && above - top_p <= OR_FLAG_TOL) flag = OR_FLAG_CUT;
        dropping = 1;
        for (int r = t; r < e; ++r) p[order[r]] = 0.0;
      }
      above += mass;
      t = e;
    }
    double Z = 0.0;
    for (int j = 0; j < V; ++j) Z += p[j];
    for (int j = 0; j < V; ++j) p[j] /= Z;
  }
  return flag;
}

/* Acceptance threshold theta = min(1, p/q) [SD §2.1].  R2: q = 0 < p gives
 * 1 (always accept under the strict test below); p = q = 0 gives 0. */
static double accept_threshold(double p, double q) {
  if (q > 0) return p / q < 1.0 ? p / q : 1.0;
  return p > 0 ? 1.0 : 0.0;
}

/* ------------------------------------------------------------------ */
/* greedy verification                                                 */
/* ------------------------------------------------------------------ */

static void clear_request(int32_t* tokens, int width, int32_t* accept_len) {
  for (int k = 0; k < width; ++k) tokens[k] = -1;
  *accept_len = 0;
}

/* Greedy verify (temperature 0) [SD §11: do_sample=False gives output
 * identical to plain decoding]: draft x_i is accepted while it equals the
 * argmax of target row i; the first mismatch emits that argmax; if all
 * drafts match, the argmax of the last row is the bonus token.  The argmax
 * is taken on the raw logits, so the temperature plays no part. */
static int greedy_request(const void* target, int dtype, const int32_t* draft_tokens,
                          const uint32_t* mask, int K, int K_b, int V, size_t b, double* row,
                          int32_t* tokens, int32_t* accept_len, double* accept_prob) {
  for (int i = 0; i < K_b; ++i) {
    int32_t x = draft_tokens[b * (size_t)K + (size_t)i];
    if (x < 0 || x >= V) return OR_BAD_TOKEN;
  }
  int n = K_b;
  int emitted = -1;
  for (int i = 0; i <= K_b; ++i) {
    load_row(target, dtype, b * (size_t)(K + 1) + (size_t)i, V, row);
    apply_token_mask(row, V, mask_row_of(mask, K, V, b, i));
    if (!row_is_valid(row, V)) return OR_BAD_LOGITS;
    int a = sv_oracle_argmax(row, V);
    if (i == K_b) {
      emitted = a;
      break;
    }
    int32_t x = draft_tokens[b * (size_t)K + (size_t)i];
    if (accept_prob) accept_prob[i] = (x == a) ? 1.0 : 0.0;
    if (x != a) {
      n = i;
      emitted = a;
      break;
    }
  }
  for (int i = 0; i < n; ++i) tokens[i] = draft_tokens[b * (size_t)K + (size_t)i];
  tokens[n] = emitted;
  *accept_len = n + 1;
  return 0;
}

int sv_oracle_greedy(const void* target, int dtype, const int32_t* draft_tokens,
                     const int32_t* draft_lens, int B, int K, int V, int b_begin, int b_end,
                     int32_t* out_tokens, int32_t* out_accept_len, int32_t* out_status,
                     const uint32_t* token_mask) {
  if (B < 0 || K < 0 || V < 1 || b_begin < 0 || b_end > B) return -1;
  double* row = (double*)malloc(sizeof(double) * (size_t)V);
  if (!row) return -2;
  for (int b = b_begin; b < b_end; ++b) {
    int32_t* tokens = out_tokens + (size_t)b * (size_t)(K + 1);
    clear_request(tokens, K + 1, &out_accept_len[b]);
    int K_b = draft_lens ? draft_lens[b] : K;
    int st = 0;
    if (K_b < 0 || K_b > K)
      st = OR_BAD_DRAFT_LEN;
    else
      st = greedy_request(target, dtype, draft_tokens, token_mask, K, K_b, V, (size_t)b, row,
                          tokens, &out_accept_len[b], NULL);
    if (st) clear_request(tokens, K + 1, &out_accept_len[b]);
    out_status[b] = st;
  }
  free(row);
  return 0;
}

/* ------------------------------------------------------------------ */
/* rejection-sampling verification                                     */
/* ------------------------------------------------------------------ */

/* One request of the verification rule [SD §2.1]:
 *   for i = 0..K_b-1 in order: accept x_i iff u_i * q_i(x_i) < p_i(x_i)
 *     (the strict "r < min(1, p/q)" of the §11 sketch, written without a
 *     division; R2);
 *   at the first rejection n: draw from norm(max(0, p_n - q_n)) and stop;
 *   if all K_b are accepted (n = K_b): draw the bonus token from p_{K_b}.
 * Dense drafts: q_i = tempered softmax of the draft logits with the same T
 * (R1).  One-hot drafts (deterministic proposer): q_i = delta at x_i, so the
 * residual is p_n with x_n removed (R9).  If the residual has no mass (only
 * through rounding, since max(0, p - q) sums to 0 only when p = q), draw
 * from p_n instead (R3).  The draw uses uniform u_K (R5).
 * Checking hooks (no effect when NULL): flip[i] != 0 inverts the outcome of
 * the test at position i (to follow the other branch of a test whose
 * uniform lies within rounding distance of its threshold); cut[r] (not NaN)
 * replaces the top-p rule's cut of row r (r = i for target row i, K+1+i for
 * draft row i) by the given logit value, and cut_margin[r] reports how far
 * that cut is from the rule (filter_top_k_top_p). */
static int sample_request(const void* target, const void* draft, int dtype,
                          const int32_t* draft_tokens, const uint32_t* mask,
                          const double* uniforms, double T, int top_k, double top_p, int K,
                          int K_b, int V, size_t b, double* lrow, double* p, double* q,
                          double* w, int* order, int32_t* tokens, int32_t* accept_len,
                          double* accept_prob, int32_t* flags, double* margins, int32_t probe,
                          double* probe_out, const uint8_t* flip, const double* cut,
                          double* cut_margin) {
  for (int i = 0; i < K_b; ++i) {
    int32_t x = draft_tokens[b * (size_t)K + (size_t)i];
    if (x < 0 || x >= V) return OR_BAD_TOKEN;
  }
  const double* u = uniforms + b * (size_t)(K + 1);
  int n = K_b;
  for (int i = 0; i < K_b; ++i) {
    int32_t x = draft_tokens[b * (size_t)K + (size_t)i];
    load_row(target, dtype, b * (size_t)(K + 1) + (size_t)i, V, lrow);
    apply_token_mask(lrow, V, mask_row_of(mask, K, V, b, i));
    if (!row_is_valid(lrow, V)) return OR_BAD_LOGITS;
    sv_oracle_tempered_softmax(lrow, V, T, p);
    flags[i] |= filter_top_k_top_p(lrow, p, V, top_k, top_p, order, cut ? cut[i] : NAN,
                                   cut_margin ? &cut_margin[i] : NULL);
    double qx = 1.0;
    if (draft) {
      load_row(draft, dtype, b * (size_t)K + (size_t)i, V, lrow);
      apply_token_mask(lrow, V, mask_row_of(mask, K, V, b, i));
      if (!row_is_valid(lrow, V)) return OR_BAD_LOGITS;
      sv_oracle_tempered_softmax(lrow, V, T, q);
      flags[i] |= filter_top_k_top_p(lrow, q, V, top_k, top_p, order,
                                     cut ? cut[K + 1 + i] : NAN,
                                     cut_margin ? &cut_margin[K + 1 + i] : NULL);
      qx = q[x];
    }
    double theta = accept_threshold(p[x], qx);
    if (accept_prob) accept_prob[i] = theta;
    if (margins) margins[i] = theta > 0 ? fabs(u[i] - theta) / theta : INFINITY;
    if (fabs(u[i] - theta) <= OR_FLAG_TOL * theta) flags[i] |= OR_FLAG_ACCEPT;
    int accept = u[i] * qx < p[x];
    if (flip && flip[i]) accept = !accept;
    if (!accept) {
      n = i;
      /* residual weights max(0, p - q) */
      for (int j = 0; j < V; ++j) {
        double qj = draft ? q[j] : (j == x ? 1.0 : 0.0);
        double r = p[j] - qj;
        w[j] = r > 0 ? r : 0.0;
      }
      break;
    }
  }
  if (n == K_b) {
    load_row(target, dtype, b * (size_t)(K + 1) + (size_t)K_b, V, lrow);
    apply_token_mask(lrow, V, mask_row_of(mask, K, V, b, K_b));
    if (!row_is_valid(lrow, V)) return OR_BAD_LOGITS;
    sv_oracle_tempered_softmax(lrow, V, T, p);
    flags[K_b] |= filter_top_k_top_p(lrow, p, V, top_k, top_p, order, cut ? cut[K_b] : NAN,
                                     cut_margin ? &cut_margin[K_b] : NULL);
    for (int j = 0; j < V; ++j) w[j] = p[j];
  } else {
    double W = 0.0;
    for (int j = 0; j < V; ++j) W += w[j];
    if (!(W > 0)) /* R3 */
      for (int j = 0; j < V; ++j) w[j] = p[j];
  }
  if (probe_out) cdf_step(w, V, probe, probe_out);
  double margin = 0.0;
  int t = sv_oracle_inverse_cdf(w, V, u[K], &margin);
  if (margins) margins[K] = margin;
  if (margin <= OR_FLAG_TOL) flags[n] |= OR_FLAG_CDF;
  for (int i = 0; i < n; ++i) tokens[i] = draft_tokens[b * (size_t)K + (size_t)i];
  tokens[n] = t;
  *accept_len = n + 1;
  return 0;
}

/* Batched entry over requests [b_begin, b_end).  Requests are independent
 * (R6: the per-sample parallel verify of the FastDeploy design; the sketch's
 * batch-wide ".all()" is not followed).
 *   target       [B, K+1, V]   draft  [B, K, V] or NULL (one-hot drafts)
 *   draft_tokens [B, K]        draft_lens [B] or NULL (all K)
 *   uniforms     [B, K+1] doubles: column i < K for the acceptance test of
 *                position i, column K for the residual / bonus draw (R5)
 *   temperature  0 selects greedy verification; otherwise > 0 and finite
 *   outputs: tokens [B, K+1] (-1 padded), accept_len [B] (R7: accepted
 *   drafts + 1), accept_prob [B, K] (min(1, p/q) at the tested positions,
 *   -1 elsewhere), flags [B, K+1], margins [B, K+1] or NULL (relative
 *   distances of u_i to theta_i at i < K, and of the draw to the nearer edge
 *   of its CDF step at K), status [B].
 *   probe_tokens [B] / probe_interval [B, 2] (both optional): for a request
 *   whose draw happened, the normalised CDF step [C_{t-1}/W, C_t/W) that
 *   token t = probe_tokens[b] occupies in that draw's distribution (NaN if
 *   t is out of range).  Used to check a draw made elsewhere.
 *   token_mask [B, K+1, ceil(V/32)] words or NULL: grammar masks (R18).
 *   top_k (0 = off), top_p (1 = off): filters of every sampled distribution,
 *   target and dense draft alike (R20); the greedy rule ignores them.
 *   flip [B, K] bytes or NULL: invert the outcome of the marked tests.
 *   cut_logits [B, R] or NULL (R = K+1, plus K with draft logits; NaN = the
 *   rule's own cut): forced top-p cuts per row; cut_margin [B, R] or NULL
 *   receives each forced row's distance from the rule (see
 *   filter_top_k_top_p; rows the request never reached keep their value).
 * Returns 0, or a negative code for arguments outside the domain. */
int sv_oracle_sample(const void* target, const void* draft, int dtype,
                     const int32_t* draft_tokens, const int32_t* draft_lens,
                     const double* uniforms, double temperature, int B, int K, int V,
                     int b_begin, int b_end, int32_t* out_tokens, int32_t* out_accept_len,
                     double* out_accept_prob, int32_t* out_flags, double* out_margins,
                     int32_t* out_status, const int32_t* probe_tokens, double* probe_interval,
                     const uint32_t* token_mask, int top_k, double top_p, const uint8_t* flip,
                     const double* cut_logits, double* cut_margin) {
  if (B < 0 || K < 0 || V < 1 || b_begin < 0 || b_end > B) return -1;
  if (!(temperature >= 0) || isinf(temperature)) return -3;
  if (top_k < 0 || !(top_p > 0.0 && top_p <= 1.0)) return -5;
  double* buf = (double*)malloc(sizeof(double) * (size_t)V * 4);
  int* order = (int*)malloc(sizeof(int) * (size_t)V);
  if (!buf || !order) {
    free(buf);
    free(order);
    return -2;
  }
  const size_t R = (size_t)(K + 1) + (draft ? (size_t)K : 0);
  double *lrow = buf, *p = buf + V, *q = buf + 2 * (size_t)V, *w = buf + 3 * (size_t)V;
  for (int b = b_begin; b < b_end; ++b) {
    int32_t* tokens = out_tokens + (size_t)b * (size_t)(K + 1);
    int32_t* flags = out_flags + (size_t)b * (size_t)(K + 1);
    double* aprob = out_accept_prob + (size_t)b * (size_t)K;
    double* margins = out_margins ? out_margins + (size_t)b * (size_t)(K + 1) : NULL;
    clear_request(tokens, K + 1, &out_accept_len[b]);
    for (int i = 0; i <= K; ++i) flags[i] = 0;
    for (int i = 0; i < K; ++i) aprob[i] = -1.0;
    if (margins)
      for (int i = 0; i <= K; ++i) margins[i] = INFINITY;
    int K_b = draft_lens ? draft_lens[b] : K;
    int st;
    if (K_b < 0 || K_b > K)
      st = OR_BAD_DRAFT_LEN;
    else if (temperature == 0)
      st = greedy_request(target, dtype, draft_tokens, token_mask, K, K_b, V, (size_t)b, lrow,
                          tokens, &out_accept_len[b], aprob);
    else
      st = sample_request(target, draft, dtype, draft_tokens, token_mask, uniforms, temperature,
                          top_k, top_p, K, K_b,
                          V, (size_t)b, lrow, p, q, w, order, tokens, &out_accept_len[b], aprob,
                          flags, margins, probe_tokens ? probe_tokens[b] : -1,
                          probe_interval ? probe_interval + 2 * (size_t)b : NULL,
                          flip ? flip + (size_t)b * (size_t)K : NULL,
                          cut_logits ? cut_logits + (size_t)b * R : NULL,
                          cut_margin ? cut_margin + (size_t)b * R : NULL);
    if (st) {
      clear_request(tokens, K + 1, &out_accept_len[b]);
      for (int i = 0; i < K; ++i) aprob[i] = -1.0;
      for (int i = 0; i <= K; ++i) flags[i] = 0;
    }
    out_status[b] = st;
  }
  free(buf);
  free(order);
  return 0;
}

/* ------------------------------------------------------------------ */
/* greedy tree verification                                            */
/* ------------------------------------------------------------------ */

/* Depth of every node of a parent array (parent[n-1] = parent of node n,
 * n = 1..N; the root is node 0).  A tree needs every parent to be an earlier
 * node (0 <= parent < n, so the links cannot cycle) and no node deeper than
 * max_depth; otherwise OR_BAD_TREE. */
static int tree_depths(const int32_t* parent, int N, int max_depth, int* depth) {
  depth[0] = 0;
  for (int n = 1; n <= N; ++n) {
    int pa = parent[n - 1];
    if (pa < 0 || pa >= n) return OR_BAD_TREE;
    depth[n] = depth[pa] + 1;
    if (depth[n] > max_depth) return OR_BAD_TREE;
  }
  return 0;
}

/* Medusa / EAGLE tree [SD §3.3]: candidate nodes form a tree under the root
 * (node 0, the last committed token); each node's target row was computed
 * seeing only its ancestors.  A node is accepted when its token equals the
 * target argmax at its parent and its parent is accepted; the result is the
 * longest accepted root path plus the argmax at its last node.
 *   parent [N] shared by all requests (parent_stride 0), or [B, N] with one
 *     tree per request (parent_stride N; EAGLE-2's dynamic trees, [SD]
 *     §4.3): parent of node n (n = 1..N) at index n-1, with parent < n.
 *   tokens [B, N]: token of node n at index n-1.
 *   target [B, N+1, V]: row n holds node n's logits.
 * Outputs: tokens [B, max_depth+1] (argmax along the path, -1 padded),
 * accept_len [B] = accepted nodes + 1, path [B, max_depth+1] (node ids from
 * the root, -1 padded), status [B] (OR_BAD_TREE for a parent array that is
 * not a tree of depth <= max_depth).
 * With distinct sibling tokens (top-k candidates) at most one child of a
 * node can match, so walking from the root finds the longest path; when a
 * caller repeats a token among siblings, the lowest node index wins (R11). */
int sv_oracle_tree(const void* target, int dtype, const int32_t* parent, int parent_stride,
                   const int32_t* node_tokens, int B, int N, int V, int max_depth,
                   int b_begin, int b_end, int32_t* out_tokens, int32_t* out_accept_len,
                   int32_t* out_path, int32_t* out_status) {
  if (B < 0 || N < 0 || V < 1 || max_depth < 0 || b_begin < 0 || b_end > B) return -1;
  if (parent_stride != 0 && parent_stride != N) return -1;
  int* depth = (int*)malloc(sizeof(int) * (size_t)(N + 1));
  double* row = (double*)malloc(sizeof(double) * (size_t)V);
  if (!depth || !row) {
    free(depth);
    free(row);
    return -2;
  }
  int width = max_depth + 1;
  for (int b = b_begin; b < b_end; ++b) {
    const int32_t* par = parent + (size_t)b * (size_t)parent_stride;
    int32_t* tokens = out_tokens + (size_t)b * (size_t)width;
    int32_t* path = out_path + (size_t)b * (size_t)width;
    clear_request(tokens, width, &out_accept_len[b]);
    for (int k = 0; k < width; ++k) path[k] = -1;
    int st = tree_depths(par, N, max_depth, depth);
    for (int n = 1; n <= N && !st; ++n) {
      int32_t t = node_tokens[(size_t)b * (size_t)N + (size_t)(n - 1)];
      if (t < 0 || t >= V) st = OR_BAD_TOKEN;
    }
    int node = 0, len = 0;
    while (!st) {
      load_row(target, dtype, (size_t)b * (size_t)(N + 1) + (size_t)node, V, row);
      if (!row_is_valid(row, V)) {
        st = OR_BAD_LOGITS;
        break;
      }
      int a = sv_oracle_argmax(row, V);
      path[len] = node;
      tokens[len] = a;
      ++len;
      int next = -1;
      for (int c = 1; c <= N; ++c)
        if (par[c - 1] == node &&
            node_tokens[(size_t)b * (size_t)N + (size_t)(c - 1)] == a) {
          next = c;
          break;
        }
      if (next < 0) break;
      node = next;
    }
    if (st) {
      clear_request(tokens, width, &out_accept_len[b]);
      for (int k = 0; k < width; ++k) path[k] = -1;
    } else {
      out_accept_len[b] = len;
    }
    out_status[b] = st;
  }
  free(depth);
  free(row);
  return 0;
}

/* ------------------------------------------------------------------ */
/* lossless tree verification by rejection sampling                    */
/* ------------------------------------------------------------------ */

/* R22 (rejection sampling over a candidate tree: [SD] §10.4 - EAGLE verified
 * by rejection sampling is lossless - with the candidate trees of §3.3 and
 * §4.2; the pages state the requirement, not the steps).  The candidates
 * are deterministic (each head's top-k, §3.3), so every candidate is a
 * one-hot draft (R9) of the distribution at its parent.  From the root:
 *   p = the tempered target distribution at the current node, w = p;
 *   the node's children c, in increasing id, are tested in turn: with
 *     theta_c = w(x_c) / sum(w), x_c accepted iff u_c < theta_c; an
 *     accepted child's token is emitted and the walk moves to it; a
 *     rejected child's token leaves the residual (w(x_c) = 0, the one-hot
 *     residual of R9, applied once per rejected candidate);
 *   when no child is accepted (or the node is a leaf) one token is drawn
 *     from w, normalised, with u_0 (inverse CDF as everywhere; all mass gone
 *     - rounding only - draws from p, R3), and the walk ends.
 * Each token emitted this way is distributed as p at its node: candidate k
 * is emitted with probability prod_{j<k}(1 - theta_j) theta_k = p(x_k)
 * (distinct tokens), and the draw gives the rest of p.  A repeated sibling
 * token has no mass left when its turn comes and is always rejected.
 *   uniforms [B, N+1]: column c (1..N) for the test of node c, column 0
 *     for the final draw.  The rows needed are those of the walked nodes.
 *   Outputs: tokens / path [B, max_depth+1] as sv_oracle_tree (tokens[k] is
 *   the token emitted after path[k]); accept_len [B] = accepted nodes + 1;
 *   accept_prob [B, N+1] (theta of the tested nodes, -1 elsewhere);
 *   node_flags [B, N+1] (OR_FLAG_ACCEPT for a test within 1e-5 (relative)
 *   of theta); flags [B] (OR_FLAG_CDF for the draw); margins [B] (the
 *   draw's distance to its CDF step's nearer edge); status [B].
 *   flip [B, N+1] or NULL inverts the outcome of the marked tests;
 *   probe_tokens / probe_interval [B] / [B, 2] (optional): the CDF step of
 *   a given token in the final draw. */
int sv_oracle_tree_sample(const void* target, int dtype, const int32_t* parent,
                          int parent_stride, const int32_t* node_tokens, const double* uniforms,
                          double T, int B, int N, int V, int max_depth, int b_begin, int b_end,
                          const uint8_t* flip, int32_t* out_tokens, int32_t* out_accept_len,
                          int32_t* out_path, double* out_accept_prob, int32_t* out_node_flags,
                          int32_t* out_flags, double* out_margins, int32_t* out_status,
                          const int32_t* probe_tokens, double* probe_interval) {
  if (B < 0 || N < 0 || V < 1 || max_depth < 0 || b_begin < 0 || b_end > B) return -1;
  if (parent_stride != 0 && parent_stride != N) return -1;
  if (!(T > 0) || isinf(T)) return -3;
  int* depth = (int*)malloc(sizeof(int) * (size_t)(N + 1));
  double* buf = (double*)malloc(sizeof(double) * (size_t)V * 3);
  if (!depth || !buf) {
    free(depth);
    free(buf);
    return -2;
  }
  double *l = buf, *p = buf + V, *w = buf + 2 * (size_t)V;
  int width = max_depth + 1;
  for (int b = b_begin; b < b_end; ++b) {
    const int32_t* par = parent + (size_t)b * (size_t)parent_stride;
    const int32_t* tok = node_tokens + (size_t)b * (size_t)N;
    const double* u = uniforms + (size_t)b * (size_t)(N + 1);
    int32_t* tokens = out_tokens + (size_t)b * (size_t)width;
    int32_t* path = out_path + (size_t)b * (size_t)width;
    double* aprob = out_accept_prob + (size_t)b * (size_t)(N + 1);
    int32_t* nflags = out_node_flags + (size_t)b * (size_t)(N + 1);
    clear_request(tokens, width, &out_accept_len[b]);
    for (int k = 0; k < width; ++k) path[k] = -1;
    for (int n = 0; n <= N; ++n) {
      aprob[n] = -1.0;
      nflags[n] = 0;
    }
    out_flags[b] = 0;
    if (out_margins) out_margins[b] = INFINITY;
    int st = tree_depths(par, N, max_depth, depth);
    for (int n = 1; n <= N && !st; ++n)
      if (tok[n - 1] < 0 || tok[n - 1] >= V) st = OR_BAD_TOKEN;
    int node = 0, len = 0;
    while (!st) {
      load_row(target, dtype, (size_t)b * (size_t)(N + 1) + (size_t)node, V, l);
      if (!row_is_valid(l, V)) {
        st = OR_BAD_LOGITS;
        break;
      }
      sv_oracle_tempered_softmax(l, V, T, p);
      for (int j = 0; j < V; ++j) w[j] = p[j];
      int next = -1;
      for (int c = 1; c <= N && next < 0; ++c) {
        if (par[c - 1] != node) continue;
        int32_t x = tok[c - 1];
        double W = 0.0;
        for (int j = 0; j < V; ++j) W += w[j];
        double theta = W > 0 ? w[x] / W : 0.0;
        aprob[c] = theta;
        if (fabs(u[c] - theta) <= OR_FLAG_TOL * theta) nflags[c] |= OR_FLAG_ACCEPT;
        int accept = u[c] < theta;
        if (flip && flip[(size_t)b * (size_t)(N + 1) + (size_t)c]) accept = !accept;
        if (accept)
          next = c;
        else
          w[x] = 0.0;
      }
      path[len] = node;
      if (next >= 0) {
        tokens[len++] = tok[next - 1];
        node = next;
        continue;
      }
      double W = 0.0;
      for (int j = 0; j < V; ++j) W += w[j];
      if (!(W > 0)) /* R3 */
        for (int j = 0; j < V; ++j) w[j] = p[j];
      double margin = 0.0;
      tokens[len++] = sv_oracle_inverse_cdf(w, V, u[0], &margin);
      if (margin <= OR_FLAG_TOL) out_flags[b] |= OR_FLAG_CDF;
      if (out_margins) out_margins[b] = margin;
      if (probe_tokens && probe_interval) cdf_step(w, V, probe_tokens[b], probe_interval + 2 * (size_t)b);
      break;
    }
    if (st) {
      clear_request(tokens, width, &out_accept_len[b]);
      for (int k = 0; k < width; ++k) path[k] = -1;
      for (int n = 0; n <= N; ++n) {
        aprob[n] = -1.0;
        nflags[n] = 0;
      }
      out_flags[b] = 0;
    } else {
      out_accept_len[b] = len;
    }
    out_status[b] = st;
  }
  free(depth);
  free(buf);
  return 0;
}

/* ------------------------------------------------------------------ */
/* typical acceptance                                                  */
/* ------------------------------------------------------------------ */

/* Entropy in nats, H = -sum p ln p (a zero probability adds nothing). */
static double entropy_nats(const double* p, int V) {
  double H = 0.0;
  for (int j = 0; j < V; ++j)
    if (p[j] > 0) H -= p[j] * log(p[j]);
  return H;
}

/* R21 (typical acceptance, [SD] §10.4; the pages name it only): a draft x
 * at a position whose target distribution is p is accepted when
 *   p(x) > min(eps, delta * exp(-H(p))),
 * H the entropy of p in nats, eps and delta the rule's two parameters (the
 * posterior threshold and alpha of the Medusa implementation).  The test
 * runs in position order; the emitted token at the first failing position
 * n (or at K_b when all pass) is drawn from p_n itself by inverse CDF with
 * u_K - this rule has no residual.  accept_prob reports p_i(x_i) at every
 * tested position; a test with |p(x) - threshold| <= 1e-5 * threshold is
 * flagged. */
static double typical_threshold(const double* p, int V, double eps, double delta) {
  double t = delta * exp(-entropy_nats(p, V));
  return t < eps ? t : eps;
}

/* Typical acceptance on chains (R21).  flip [B, K] or NULL inverts the
 * outcome of the marked tests; margins [B] or NULL receives the draw's
 * distance to the nearer edge of its CDF step (relative to the total);
 * probe_tokens / probe_interval [B] / [B, 2] (optional) as for
 * sv_oracle_sample. */
int sv_oracle_typical(const void* target, int dtype, const int32_t* draft_tokens,
                      const int32_t* draft_lens, const double* uniforms, double T, double eps,
                      double delta, int B, int K, int V, int b_begin, int b_end,
                      int32_t* out_tokens, int32_t* out_accept_len, double* out_accept_prob,
                      int32_t* out_flags, int32_t* out_status, const uint8_t* flip,
                      double* out_margins, const int32_t* probe_tokens, double* probe_interval) {
  if (B < 0 || K < 0 || V < 1 || b_begin < 0 || b_end > B) return -1;
  if (!(T > 0) || isinf(T) || !(eps >= 0) || !(delta >= 0)) return -3;
  double* buf = (double*)malloc(sizeof(double) * (size_t)V * 2);
  if (!buf) return -2;
  double *l = buf, *p = buf + V;
  for (int b = b_begin; b < b_end; ++b) {
    int32_t* tokens = out_tokens + (size_t)b * (size_t)(K + 1);
    int32_t* flags = out_flags + (size_t)b * (size_t)(K + 1);
    double* aprob = out_accept_prob + (size_t)b * (size_t)K;
    const double* u = uniforms + (size_t)b * (size_t)(K + 1);
    clear_request(tokens, K + 1, &out_accept_len[b]);
    for (int i = 0; i <= K; ++i) flags[i] = 0;
    for (int i = 0; i < K; ++i) aprob[i] = -1.0;
    if (out_margins) out_margins[b] = INFINITY;
    int K_b = draft_lens ? draft_lens[b] : K;
    int st = 0;
    if (K_b < 0 || K_b > K) st = OR_BAD_DRAFT_LEN;
    for (int i = 0; i < K_b && !st; ++i) {
      int32_t x = draft_tokens[(size_t)b * (size_t)K + (size_t)i];
      if (x < 0 || x >= V) st = OR_BAD_TOKEN;
    }
    int n = K_b;
    for (int i = 0; i < K_b && !st; ++i) {
      int32_t x = draft_tokens[(size_t)b * (size_t)K + (size_t)i];
      load_row(target, dtype, (size_t)b * (size_t)(K + 1) + (size_t)i, V, l);
      if (!row_is_valid(l, V)) {
        st = OR_BAD_LOGITS;
        break;
      }
      sv_oracle_tempered_softmax(l, V, T, p);
      double thr = typical_threshold(p, V, eps, delta);
      aprob[i] = p[x];
      if (fabs(p[x] - thr) <= OR_FLAG_TOL * thr) flags[i] |= OR_FLAG_ACCEPT;
      int pass = p[x] > thr;
      if (flip && flip[(size_t)b * (size_t)K + (size_t)i]) pass = !pass;
      if (!pass) {
        n = i;
        break;
      }
    }
    if (!st) {
      load_row(target, dtype, (size_t)b * (size_t)(K + 1) + (size_t)n, V, l);
      if (!row_is_valid(l, V)) st = OR_BAD_LOGITS;
    }
    if (!st) {
      sv_oracle_tempered_softmax(l, V, T, p);
      double margin = 0.0;
      int t = sv_oracle_inverse_cdf(p, V, u[K], &margin);
      if (margin <= OR_FLAG_TOL) flags[n] |= OR_FLAG_CDF;
      if (out_margins) out_margins[b] = margin;
      if (probe_tokens && probe_interval) cdf_step(p, V, probe_tokens[b], probe_interval + 2 * (size_t)b);
      for (int i = 0; i < n; ++i) tokens[i] = draft_tokens[(size_t)b * (size_t)K + (size_t)i];
      tokens[n] = t;
      out_accept_len[b] = n + 1;
    } else {
      clear_request(tokens, K + 1, &out_accept_len[b]);
      for (int i = 0; i < K; ++i) aprob[i] = -1.0;
      for (int i = 0; i <= K; ++i) flags[i] = 0;
    }
    out_status[b] = st;
  }
  free(buf);
  return 0;
}

/* Typical acceptance on a candidate tree (R21 with [SD] §3.3): node n is
 * accepted when its parent is (the root always is) and its token passes the
 * typical test under the parent's distribution; the result is the deepest
 * accepted node (the lowest id among equally deep ones), the tokens along
 * its root path and one token drawn from its own distribution with u[b].
 * Only the rows of accepted nodes are needed (their validity is checked).
 *   parent / parent_stride as sv_oracle_tree; uniforms [B]; outputs as
 *   sv_oracle_tree, plus flags [B] (OR_FLAG_ACCEPT when any test made is
 *   within 1e-5 of its threshold, OR_FLAG_CDF for the draw), node_flags
 *   [B, N+1] (OR_FLAG_ACCEPT per flagged node test) and margins [B] (the
 *   draw's distance to its CDF step's nearer edge).  flip [B, N+1] or NULL
 *   inverts the outcome of the marked node tests; probe_tokens /
 *   probe_interval (optional) as sv_oracle_sample. */
int sv_oracle_tree_typical(const void* target, int dtype, const int32_t* parent,
                           int parent_stride, const int32_t* node_tokens,
                           const double* uniforms, double T, double eps, double delta, int B,
                           int N, int V, int max_depth, int b_begin, int b_end,
                           int32_t* out_tokens, int32_t* out_accept_len, int32_t* out_path,
                           int32_t* out_flags, int32_t* out_status, const uint8_t* flip,
                           int32_t* out_node_flags, double* out_margins,
                           const int32_t* probe_tokens, double* probe_interval) {
  if (B < 0 || N < 0 || V < 1 || max_depth < 0 || b_begin < 0 || b_end > B) return -1;
  if (parent_stride != 0 && parent_stride != N) return -1;
  if (!(T > 0) || isinf(T) || !(eps >= 0) || !(delta >= 0)) return -3;
  int* depth = (int*)malloc(sizeof(int) * (size_t)(N + 1));
  int* acc = (int*)malloc(sizeof(int) * (size_t)(N + 1));
  double* thr = (double*)malloc(sizeof(double) * (size_t)(N + 1));
  double* l = (double*)malloc(sizeof(double) * (size_t)V);
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* pp = (double*)malloc(sizeof(double) * (size_t)V * (size_t)(N + 1));
  if (!depth || !acc || !thr || !l || !p || !pp) {
    free(depth); free(acc); free(thr); free(l); free(p); free(pp);
    return -2;
  }
  int width = max_depth + 1;
  for (int b = b_begin; b < b_end; ++b) {
    const int32_t* par = parent + (size_t)b * (size_t)parent_stride;
    int32_t* tokens = out_tokens + (size_t)b * (size_t)width;
    int32_t* path = out_path + (size_t)b * (size_t)width;
    int32_t* nflags = out_node_flags ? out_node_flags + (size_t)b * (size_t)(N + 1) : NULL;
    const uint8_t* fl = flip ? flip + (size_t)b * (size_t)(N + 1) : NULL;
    clear_request(tokens, width, &out_accept_len[b]);
    for (int k = 0; k < width; ++k) path[k] = -1;
    out_flags[b] = 0;
    if (nflags)
      for (int n = 0; n <= N; ++n) nflags[n] = 0;
    if (out_margins) out_margins[b] = INFINITY;
    int st = tree_depths(par, N, max_depth, depth);
    for (int n = 1; n <= N && !st; ++n) {
      int32_t t = node_tokens[(size_t)b * (size_t)N + (size_t)(n - 1)];
      if (t < 0 || t >= V) st = OR_BAD_TOKEN;
    }
    /* the distribution and threshold of every accepted node, parents first */
    acc[0] = 1;
    for (int n = 0; n <= N && !st; ++n) {
      if (n > 0) {
        int pa = par[n - 1];
        int32_t t = node_tokens[(size_t)b * (size_t)N + (size_t)(n - 1)];
        acc[n] = 0;
        if (acc[pa]) {
          double px = pp[(size_t)pa * (size_t)V + (size_t)t];
          if (fabs(px - thr[pa]) <= OR_FLAG_TOL * thr[pa]) {
            out_flags[b] |= OR_FLAG_ACCEPT;
            if (nflags) nflags[n] |= OR_FLAG_ACCEPT;
          }
          acc[n] = px > thr[pa];
          if (fl && fl[n]) acc[n] = !acc[n];
        }
      }
      if (!acc[n]) continue;
      load_row(target, dtype, (size_t)b * (size_t)(N + 1) + (size_t)n, V, l);
      if (!row_is_valid(l, V)) {
        st = OR_BAD_LOGITS;
        break;
      }
      sv_oracle_tempered_softmax(l, V, T, pp + (size_t)n * (size_t)V);
      thr[n] = typical_threshold(pp + (size_t)n * (size_t)V, V, eps, delta);
    }
    if (!st) {
      int best = 0;
      for (int n = 1; n <= N; ++n)
        if (acc[n] && depth[n] > depth[best]) best = n;
      int len = depth[best] + 1;
      for (int n = best, d = depth[best]; d >= 0; --d) {
        path[d] = n;
        if (d > 0) tokens[d - 1] = node_tokens[(size_t)b * (size_t)N + (size_t)(n - 1)];
        n = d > 0 ? par[n - 1] : 0;
      }
      for (int j = 0; j < V; ++j) p[j] = pp[(size_t)best * (size_t)V + (size_t)j];
      double margin = 0.0;
      tokens[len - 1] = sv_oracle_inverse_cdf(p, V, uniforms[b], &margin);
      if (margin <= OR_FLAG_TOL) out_flags[b] |= OR_FLAG_CDF;
      if (out_margins) out_margins[b] = margin;
      if (probe_tokens && probe_interval) cdf_step(p, V, probe_tokens[b], probe_interval + 2 * (size_t)b);
      out_accept_len[b] = len;
    } else {
      clear_request(tokens, width, &out_accept_len[b]);
      for (int k = 0; k < width; ++k) path[k] = -1;
      out_flags[b] = 0;
      if (nflags)
        for (int n = 0; n <= N; ++n) nflags[n] = 0;
    }
    out_status[b] = st;
  }
  free(depth); free(acc); free(thr); free(l); free(p); free(pp);
  return 0;
}

/* ------------------------------------------------------------------ */
/* padding-free output layout                                          */
/* ------------------------------------------------------------------ */

/* [FD "高效投机解码框架设计": locate each output token's batch id without
 * copies or slices]: cu[0] = 0, cu[b+1] = cu[b] + accept_len[b]; the
 * emitted tokens of request b sit at packed[cu[b] .. cu[b+1]-1] and
 * batch_id there is b.  Slots from cu[B] to B*width-1 hold -1. */
void sv_oracle_compact(const int32_t* tokens, const int32_t* accept_len, int B, int width,
                       int32_t* cu, int32_t* packed, int32_t* batch_id) {
  cu[0] = 0;
  for (int b = 0; b < B; ++b) cu[b + 1] = cu[b] + accept_len[b];
  for (size_t s = 0; s < (size_t)B * (size_t)width; ++s) {
    packed[s] = -1;
    batch_id[s] = -1;
  }
  for (int b = 0; b < B; ++b)
    for (int k = 0; k < accept_len[b]; ++k) {
      packed[cu[b] + k] = tokens[(size_t)b * (size_t)width + (size_t)k];
      batch_id[cu[b] + k] = b;
    }
}

/* ------------------------------------------------------------------ */
/* n-gram (prompt-lookup) proposer                                     */
/* ------------------------------------------------------------------ */

/* The deterministic proposer whose drafts the one-hot verification checks
 * ["投机解码" (FastDeploy docs), "使用 Ngram 解码": drafts come from matching an
 * n-gram window against the prompt and the tokens generated so far; the vLLM
 * Ascend guide's n-gram example and "推测解码与 MTP" §9.1: prompt lookup with
 * prompt_lookup_max = 4 and num_speculative_tokens = 5].
 * R19: for n = n_max down to n_min, the pattern is the last n tokens of the
 * request's context c[0..len); the match is the EARLIEST start s with
 * c[s..s+n) equal to the pattern and at least one token after it
 * (s + n < len, so the pattern's own position never counts); the drafts
 * are the up to K tokens that follow, c[s+n .. min(s+n+K, len)).  The first
 * n (longest) that matches decides; with no match there are no drafts.
 *   tokens [B, L] int32 (row b holds its context in the first lens[b]
 *   entries), lens [B].
 *   Outputs: drafts [B, K] (-1 padded), draft_lens [B] (0..K), match [B]
 *   (the start s, or -1), ngram [B] (the n that matched, or 0), status [B]
 *   (4 when lens[b] is outside [0, L]: no drafts).
 * Returns 0, or -1 for arguments outside the domain. */
int sv_oracle_ngram(const int32_t* tokens, const int32_t* lens, int B, int L, int n_min,
                    int n_max, int K, int32_t* drafts, int32_t* draft_lens, int32_t* match,
                    int32_t* ngram, int32_t* status) {
  if (B < 0 || L < 0 || n_min < 1 || n_max < n_min || K < 0) return -1;
  for (int b = 0; b < B; ++b) {
    const int32_t* c = tokens + (size_t)b * (size_t)L;
    int len = lens[b];
    for (int k = 0; k < K; ++k) drafts[(size_t)b * (size_t)K + (size_t)k] = -1;
    draft_lens[b] = 0;
    match[b] = -1;
    ngram[b] = 0;
    status[b] = 0;
    if (len < 0 || len > L) {
      status[b] = OR_BAD_DRAFT_LEN;
      continue;
    }
    for (int n = n_max; n >= n_min; --n) {
      if (len < n + 1) continue;
      const int32_t* pattern = c + (len - n);
      int found = -1;
      for (int s = 0; s + n < len && found < 0; ++s) {
        int equal = 1;
        for (int t = 0; t < n; ++t)
          if (c[s + t] != pattern[t]) {
            equal = 0;
            break;
          }
        if (equal) found = s;
      }
      if (found >= 0) {
        int k = len - (found + n);
        if (k > K) k = K;
        for (int t = 0; t < k; ++t) drafts[(size_t)b * (size_t)K + (size_t)t] = c[found + n + t];
        draft_lens[b] = k;
        match[b] = found;
        ngram[b] = n;
        break;
      }
    }
  }
  return 0;
}
