/*
 * eagle_oracle.c -- plain CPU oracle for the EAGLE draft-tree verify step.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  The product path never
 * does, and this file shares no code, header, table or constant with the CUDA
 * library: it is written from the pages' definitions alone.
 *
 * Arithmetic is float64 throughout.  Inputs are read from the very bytes the GPU
 * reads: float32, or bfloat16 widened exactly to float.  Every loop is the plain
 * definition; nothing is blocked, fused or reordered.
 *
 * Sources (page title, section):
 *   tree attention  -- EAGLE review (zenmind), terms "tree attention": each draft
 *                      candidate attends only to its own ancestors; lesson
 *                      "Speculative decoding and EAGLE-3", glossary "Tree attention".
 *   acceptance      -- EAGLE review, section 3.3 + appendix A.2 / Algorithm 1
 *                      (multi-round speculative sampling: accept if r < p/p_hat,
 *                      else p <- norm(max(0, p - p_hat)), next candidate; sample
 *                      from the adjusted p only when all are rejected); lesson
 *                      steps 1-2 (accept rule with the p_draft <= 0 case, residual
 *                      with the zero-sum fallback), "bonus token".
 *   dynamic tree    -- EAGLE-3 visual reading, "EAGLE-2: dynamic draft tree"
 *                      (draft confidence ~ acceptance, so the tree keeps the most
 *                      confident candidates); EAGLE review section 3.1 /
 *                      appendix A.1 (top-k children per node, k = 4 at the root).
 *   static tree     -- EAGLE review appendix A.1: greedy -> top-k children,
 *                      non-greedy -> k sampled children.
 *
 * Readings where the pages are silent are stated at each function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_BAD_ARG 1
#define OR_NO_MEM 2

/* A decision is a near-tie when fp32 and fp64 arithmetic could resolve it
 * differently: |u - p/q| < 1e-5 for an accept test; a draw landing within
 * 1e-7 * sum(w) of a bin edge; two scores at a selection boundary closer than
 * 1e-5 (unless they are siblings with the same logit, an exact tie both sides
 * break by pool index). */
#define NEAR_TIE_EPS 1e-5
#define ICDF_NEAR_EPS 1e-7

/* Element types of the input buffers. */
#define OR_F32 0
#define OR_BF16 1

static double elem(const void* base, size_t i, int dtype) {
  if (dtype == OR_F32) return (double)((const float*)base)[i];
  uint32_t u = ((uint32_t)((const uint16_t*)base)[i]) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ------------------------------------------------------------------ helpers */

/* w[v] = exp((x_v - max x) / T) for one row, returns the sum of w. */
static double softmax_weights(const void* row, size_t off, int V, int dtype, double T, double* w) {
  double mx = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double x = elem(row, off + v, dtype);
    if (x > mx) mx = x;
  }
  double s = 0.0;
  for (int v = 0; v < V; ++v) {
    w[v] = exp((elem(row, off + v, dtype) - mx) / T);
    s += w[v];
  }
  return s;
}

/* ln softmax(x)[v] at T = 1 for one row (the draft confidence, in log form). */
static void log_softmax(const void* row, size_t off, int V, int dtype, double* out) {
  double mx = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double x = elem(row, off + v, dtype);
    if (x > mx) mx = x;
  }
  double s = 0.0;
  for (int v = 0; v < V; ++v) s += exp(elem(row, off + v, dtype) - mx);
  double ls = log(s);
  for (int v = 0; v < V; ++v) out[v] = (elem(row, off + v, dtype) - mx) - ls;
}

/* Inverse CDF: smallest i with w_0 + ... + w_i > u * sum(w).  If rounding leaves
 * no such i, the last i with w_i > 0.  *near is set when u*sum(w) lies within
 * 1e-7 * sum(w) of either edge of the chosen bin. */
static int icdf(const double* w, int V, double u, int* near) {
  double W = 0.0;
  for (int v = 0; v < V; ++v) W += w[v];
  double target = u * W, c = 0.0;
  for (int v = 0; v < V; ++v) {
    double prev = c;
    c += w[v];
    if (c > target) {
      if (near && (target - prev < ICDF_NEAR_EPS * W || c - target < ICDF_NEAR_EPS * W)) *near = 1;
      return v;
    }
  }
  for (int v = V - 1; v >= 0; --v)
    if (w[v] > 0.0) {
      if (near) *near = 1;
      return v;
    }
  return 0;
}

/* Sort keys for top-k: (value desc, id asc). */
typedef struct {
  double val;
  int id;
} vid_t;

static int cmp_vid(const void* a, const void* b) {
  const vid_t* x = (const vid_t*)a;
  const vid_t* y = (const vid_t*)b;
  if (x->val > y->val) return -1;
  if (x->val < y->val) return 1;
  return (x->id > y->id) - (x->id < y->id);
}

/* The c best tokens of one row by (logit desc, token id asc): a full sort. */
static int row_topk(const void* row, size_t off, int V, int dtype, int c, int* out) {
  vid_t* t = (vid_t*)malloc(sizeof(vid_t) * (size_t)V);
  if (!t) return OR_NO_MEM;
  for (int v = 0; v < V; ++v) {
    t[v].val = elem(row, off + v, dtype);
    t[v].id = v;
  }
  qsort(t, (size_t)V, sizeof(vid_t), cmp_vid);
  for (int j = 0; j < c; ++j) out[j] = t[j].id;
  free(t);
  return OR_OK;
}

/* Sort keys for the rerank: (score desc, pool index asc). */
static int cmp_score(const void* a, const void* b) { return cmp_vid(a, b); }

/* ------------------------------------------------------------------ tree attention
 *
 * For request b, node i, query head hq (KV head hq / G):
 *   keys = prefix positions j < seq_len[b]  U  tree nodes on the root..i path,
 *   x_j  = scale * <q, k_j>,   out = sum_j softmax(x)_j v_j,   lse = ln sum_j exp(x_j).
 * The ancestor set is found by walking parent[] from i to the root.
 */
int oracle_tree_attn(int B, int R, int Hq, int Hkv, int D, int P_max, double scale, int dtype,
                     const void* q, const void* k_cache, const void* v_cache, const void* tree_k,
                     const void* tree_v, const int32_t* seq_len, const int32_t* parent, double* out,
                     double* lse) {
  if (B <= 0 || R <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv) return OR_BAD_ARG;
  const int G = Hq / Hkv;
  int max_len = 0;
  for (int b = 0; b < B; ++b) {
    if (seq_len[b] < 0 || seq_len[b] > P_max) return OR_BAD_ARG;
    if (seq_len[b] > max_len) max_len = seq_len[b];
  }
  double* x = (double*)malloc(sizeof(double) * (size_t)(max_len + R));
  int* anc = (int*)malloc(sizeof(int) * (size_t)R);
  if (!x || !anc) {
    free(x);
    free(anc);
    return OR_NO_MEM;
  }
  for (int b = 0; b < B; ++b) {
    for (int i = 0; i < R; ++i) {
      int n_anc = 0;
      for (int a = i; a >= 0; a = parent[(size_t)b * R + a]) {
        if (n_anc >= R || (a > 0 && parent[(size_t)b * R + a] >= a)) {
          free(x);
          free(anc);
          return OR_BAD_ARG;
        }
        anc[n_anc++] = a;
      }
      const int L = seq_len[b];
      for (int hq = 0; hq < Hq; ++hq) {
        const int h = hq / G;
        const size_t qoff = (((size_t)b * R + i) * Hq + hq) * D;
        for (int j = 0; j < L; ++j) {
          const size_t koff = (((size_t)b * Hkv + h) * P_max + j) * D;
          double s = 0.0;
          for (int d = 0; d < D; ++d) s += elem(q, qoff + d, dtype) * elem(k_cache, koff + d, dtype);
          x[j] = scale * s;
        }
        for (int t = 0; t < n_anc; ++t) {
          const size_t koff = (((size_t)b * Hkv + h) * R + anc[t]) * D;
          double s = 0.0;
          for (int d = 0; d < D; ++d) s += elem(q, qoff + d, dtype) * elem(tree_k, koff + d, dtype);
          x[L + t] = scale * s;
        }
        const int n = L + n_anc;
        double mx = -INFINITY;
        for (int j = 0; j < n; ++j)
          if (x[j] > mx) mx = x[j];
        double sum = 0.0;
        for (int j = 0; j < n; ++j) sum += exp(x[j] - mx);
        double* o = out + qoff;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (int j = 0; j < L; ++j) {
          const double p = exp(x[j] - mx) / sum;
          const size_t voff = (((size_t)b * Hkv + h) * P_max + j) * D;
          for (int d = 0; d < D; ++d) o[d] += p * elem(v_cache, voff + d, dtype);
        }
        for (int t = 0; t < n_anc; ++t) {
          const double p = exp(x[L + t] - mx) / sum;
          const size_t voff = (((size_t)b * Hkv + h) * R + anc[t]) * D;
          for (int d = 0; d < D; ++d) o[d] += p * elem(tree_v, voff + d, dtype);
        }
        if (lse) lse[((size_t)b * R + i) * Hq + hq] = mx + log(sum);
      }
    }
  }
  free(x);
  free(anc);
  return OR_OK;
}

/* ------------------------------------------------------------------ acceptance
 *
 * Per request, starting at the root (node 0):
 *   T == 0 (greedy): a = argmax target[cur] (lowest id on ties); if a child of cur
 *     carries token a, accept it and move there; otherwise emit a and stop.
 *   T > 0: p = softmax(target[cur] / T).  For the children of cur in index order,
 *     with d = the child's token and q its proposal distribution:
 *       accept iff q(d) <= 0 or u_accept[child] < p(d) / q(d);
 *       else p <- norm(max(0, p - q)), keeping p when that sum is 0.
 *     The first accepted child becomes cur.  When every child is rejected (or cur
 *     is a leaf) emit icdf(p, u_final) and stop.
 * Proposal q (reading of the pages, which state the rule for drawn candidates):
 *   proposal 1 (SAMPLED): q = softmax(draft[cur] / T), the distribution the
 *     children were drawn from; it stays fixed across siblings.
 *   proposal 0 (DELTA): the children were chosen deterministically (top-k), so
 *     each child's proposal is the point mass on its own token: q = onehot(d).
 * Outputs: n_acc accepted drafts, path (node ids, root first), out_tok (the
 * accepted tokens then the emitted one), near_tie = 1 when a decision had
 * |u - p/q| < 1e-5 or an inverse-CDF draw landed within 1e-5 of a bin edge.
 */
int oracle_accept(int B, int R, int V, int dtype, double T, int proposal, int max_path,
                  const void* target, const void* draft, const int32_t* tokens, const int32_t* parent,
                  const float* u_accept, const float* u_final, int32_t* n_acc, int32_t* path,
                  int32_t* out_tok, int32_t* near_tie, double* ratio_out) {
  if (B <= 0 || R <= 0 || V <= 0 || max_path <= 0) return OR_BAD_ARG;
  if (T > 0 && proposal == 1 && !draft) return OR_BAD_ARG;
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  double* r = (double*)malloc(sizeof(double) * (size_t)V);
  if (!p || !q || !r) {
    free(p);
    free(q);
    free(r);
    return OR_NO_MEM;
  }
  for (int b = 0; b < B; ++b) {
    const int32_t* tok = tokens + (size_t)b * R;
    const int32_t* par = parent + (size_t)b * R;
    int32_t* pb = path + (size_t)b * max_path;
    int32_t* ob = out_tok + (size_t)b * max_path;
    for (int j = 0; j < max_path; ++j) pb[j] = ob[j] = -1;
    if (ratio_out)
      for (int j = 0; j < R; ++j) ratio_out[(size_t)b * R + j] = NAN;
    int near = 0, len = 1, cur = 0, emitted = -1;
    pb[0] = 0;
    for (;;) {
      const size_t roff = ((size_t)b * R + cur) * V;
      int next = -1;
      if (T <= 0.0) {
        double best = -INFINITY;
        int a = 0;
        for (int v = 0; v < V; ++v) {
          double x = elem(target, roff + v, dtype);
          if (x > best) {
            best = x;
            a = v;
          }
        }
        for (int c = cur + 1; c < R; ++c)
          if (par[c] == cur && tok[c] == a) {
            next = c;
            break;
          }
        if (next < 0) {
          emitted = a;
          break;
        }
      } else {
        double s = softmax_weights(target, roff, V, dtype, T, p);
        for (int v = 0; v < V; ++v) p[v] /= s;
        if (proposal == 1) {
          double sq = softmax_weights(draft, roff, V, dtype, T, q);
          for (int v = 0; v < V; ++v) q[v] /= sq;
        }
        for (int c = cur + 1; c < R; ++c) {
          if (par[c] != cur) continue;
          const int d = tok[c];
          const double qd = (proposal == 1) ? q[d] : 1.0;
          const double ratio = (qd > 0.0) ? p[d] / qd : INFINITY;
          const double u = (double)u_accept[(size_t)b * R + c];
          if (ratio_out) ratio_out[(size_t)b * R + c] = ratio;
          if (fabs(u - ratio) < NEAR_TIE_EPS) near = 1;
          if (qd <= 0.0 || u < ratio) {
            next = c;
            break;
          }
          double rs = 0.0;
          for (int v = 0; v < V; ++v) {
            const double qv = (proposal == 1) ? q[v] : (v == d ? 1.0 : 0.0);
            r[v] = p[v] - qv > 0.0 ? p[v] - qv : 0.0;
            rs += r[v];
          }
          if (rs > 0.0)
            for (int v = 0; v < V; ++v) p[v] = r[v] / rs;
        }
        if (next < 0) {
          emitted = icdf(p, V, (double)u_final[b], &near);
          break;
        }
      }
      if (len >= max_path) {
        free(p);
        free(q);
        free(r);
        return OR_BAD_ARG; /* tree deeper than max_path - 1 */
      }
      pb[len++] = next;
      cur = next;
    }
    n_acc[b] = len - 1;
    for (int j = 1; j < len; ++j) ob[j - 1] = tok[pb[j]];
    ob[len - 1] = emitted;
    if (near_tie) near_tie[b] = near;
  }
  free(p);
  free(q);
  free(r);
  return OR_OK;
}

/* ------------------------------------------------------------------ dynamic tree
 *
 * Reading of the EAGLE-2 dynamic tree (the pages give the idea, not the steps):
 *   level 1: the root's top-k tokens become candidates with score ln q_root(t);
 *            they are the first frontier.
 *   level d: each frontier node f adds its top-k tokens with score
 *            s_f + ln q_f(t) (q at temperature 1: the draft confidence).  The next
 *            frontier is the best k of these F*k new candidates.
 *   final:   the best N candidates of the whole pool form the tree.
 * "Best" is (score desc, pool index asc).  Pool indices are handed out level by
 * level, frontier slot by frontier slot, child rank by child rank, so a parent
 * always precedes its children.  A frontier is kept in pool-index order.
 * Top-k within a row is (logit desc, token id asc).
 * near_tie counts selection boundaries where the last kept and the first dropped
 * scores differ by less than 1e-5.
 */
int oracle_tree_level_dynamic(int B, int V, int dtype, int k, int level, const void* logits,
                              int pool_cap, int32_t* pool_tok, int32_t* pool_parent,
                              double* pool_score, int32_t* pool_depth, int32_t* n_pool,
                              int32_t* frontier, int32_t* near_tie) {
  if (B <= 0 || V <= 0 || k <= 0 || k > V || level < 1) return OR_BAD_ARG;
  const int F = (level == 1) ? 1 : k;
  double* lq = (double*)malloc(sizeof(double) * (size_t)V);
  int* top = (int*)malloc(sizeof(int) * (size_t)k);
  vid_t* cand = (vid_t*)malloc(sizeof(vid_t) * (size_t)F * k);
  if (!lq || !top || !cand) {
    free(lq);
    free(top);
    free(cand);
    return OR_NO_MEM;
  }
  int rc = OR_OK;
  for (int b = 0; b < B && rc == OR_OK; ++b) {
    int32_t* ptok = pool_tok + (size_t)b * pool_cap;
    int32_t* ppar = pool_parent + (size_t)b * pool_cap;
    double* psc = pool_score + (size_t)b * pool_cap;
    int32_t* pdep = pool_depth + (size_t)b * pool_cap;
    int32_t* fr = frontier + (size_t)b * k;
    if (level == 1) n_pool[b] = 0;
    const int base = n_pool[b];
    if (base + F * k > pool_cap) {
      rc = OR_BAD_ARG;
      break;
    }
    for (int f = 0; f < F; ++f) {
      const int pidx = (level == 1) ? -1 : fr[f];
      const double s_par = (pidx < 0) ? 0.0 : psc[pidx];
      const size_t off = ((size_t)b * F + f) * V;
      log_softmax(logits, off, V, dtype, lq);
      if ((rc = row_topk(logits, off, V, dtype, k, top)) != OR_OK) break;
      for (int r = 0; r < k; ++r) {
        const int i = base + f * k + r;
        ptok[i] = top[r];
        ppar[i] = pidx;
        psc[i] = s_par + lq[top[r]];
        pdep[i] = level;
      }
    }
    n_pool[b] = base + F * k;
    /* next frontier: the best k of the new candidates, kept in pool-index order */
    for (int j = 0; j < F * k; ++j) {
      cand[j].val = psc[base + j];
      cand[j].id = base + j;
    }
    qsort(cand, (size_t)F * k, sizeof(vid_t), cmp_score);
    if (F * k > k && fabs(cand[k - 1].val - cand[k].val) < NEAR_TIE_EPS &&
        !(cand[k - 1].val == cand[k].val && ppar[cand[k - 1].id] == ppar[cand[k].id]))
      near_tie[b] += 1;
    for (int j = 0; j < k; ++j) fr[j] = cand[j].id;
    for (int a = 1; a < k; ++a) /* insertion sort by pool index */
      for (int j = a; j > 0 && fr[j - 1] > fr[j]; --j) {
        int t = fr[j];
        fr[j] = fr[j - 1];
        fr[j - 1] = t;
      }
  }
  free(lq);
  free(top);
  free(cand);
  return rc;
}

/* Final rerank: keep the best N of the pool, order them by pool index (so parents
 * precede children), prepend the root, and emit the tree arrays.
 * anc_mask[i] bit j is set iff node j is node i or one of its ancestors. */
int oracle_tree_finalize_dynamic(int B, int N, int pool_cap, const int32_t* pool_tok,
                                 const int32_t* pool_parent, const double* pool_score,
                                 const int32_t* pool_depth, const int32_t* n_pool,
                                 const int32_t* root_tok, const int32_t* seq_len, int W,
                                 int32_t* tokens, int32_t* parent, int32_t* depth, int32_t* pos_id,
                                 uint64_t* anc_mask, double* score, int32_t* near_tie) {
  const int R = N + 1;
  if (B <= 0 || N <= 0 || W * 64 < R) return OR_BAD_ARG;
  vid_t* cand = (vid_t*)malloc(sizeof(vid_t) * (size_t)pool_cap);
  int* sel = (int*)malloc(sizeof(int) * (size_t)N);
  int* tree_of = (int*)malloc(sizeof(int) * (size_t)pool_cap);
  if (!cand || !sel || !tree_of) {
    free(cand);
    free(sel);
    free(tree_of);
    return OR_NO_MEM;
  }
  int rc = OR_OK;
  for (int b = 0; b < B; ++b) {
    const int np = n_pool[b];
    if (np < N) {
      rc = OR_BAD_ARG;
      break;
    }
    const size_t po = (size_t)b * pool_cap;
    for (int j = 0; j < np; ++j) {
      cand[j].val = pool_score[po + j];
      cand[j].id = j;
      tree_of[j] = -1;
    }
    qsort(cand, (size_t)np, sizeof(vid_t), cmp_score);
    if (np > N && fabs(cand[N - 1].val - cand[N].val) < NEAR_TIE_EPS &&
        !(cand[N - 1].val == cand[N].val &&
          pool_parent[po + cand[N - 1].id] == pool_parent[po + cand[N].id]))
      near_tie[b] += 1;
    for (int j = 0; j < N; ++j) sel[j] = cand[j].id;
    for (int a = 1; a < N; ++a)
      for (int j = a; j > 0 && sel[j - 1] > sel[j]; --j) {
        int t = sel[j];
        sel[j] = sel[j - 1];
        sel[j - 1] = t;
      }
    int32_t* tk = tokens + (size_t)b * R;
    int32_t* pa = parent + (size_t)b * R;
    int32_t* de = depth + (size_t)b * R;
    int32_t* ps = pos_id + (size_t)b * R;
    uint64_t* am = anc_mask + (size_t)b * R * W;
    double* sc = score + (size_t)b * R;
    memset(am, 0, sizeof(uint64_t) * (size_t)R * W);
    tk[0] = root_tok[b];
    pa[0] = -1;
    de[0] = 0;
    ps[0] = seq_len[b];
    sc[0] = 0.0;
    am[0] = 1ull;
    for (int i = 1; i < R; ++i) {
      const int j = sel[i - 1];
      tree_of[j] = i;
      const int pp = pool_parent[po + j];
      const int t_par = (pp < 0) ? 0 : tree_of[pp];
      if (t_par < 0) { /* parent not kept: the set is not ancestor-closed */
        rc = OR_BAD_ARG;
        break;
      }
      tk[i] = pool_tok[po + j];
      pa[i] = t_par;
      de[i] = pool_depth[po + j];
      ps[i] = seq_len[b] + de[i];
      sc[i] = pool_score[po + j];
      for (int w = 0; w < W; ++w) am[(size_t)i * W + w] = am[(size_t)t_par * W + w];
      am[(size_t)i * W + i / 64] |= 1ull << (i % 64);
    }
    if (rc != OR_OK) break;
  }
  free(cand);
  free(sel);
  free(tree_of);
  return rc;
}

/* ------------------------------------------------------------------ static tree
 *
 * The shape is fixed: parent[] per node, nodes ordered by depth, root = node 0.
 * Level d expands the nodes of depth d-1; frontier row f is the f-th such node in
 * index order.  A node's children, in index order, receive
 *   sampled == 0: its 1st, 2nd, ... best tokens (logit desc, id asc);
 *   sampled == 1: icdf(softmax(row / T), u_draft[child]) each, drawn
 *                 independently (with replacement: duplicates stay distinct nodes).
 * score[child] = score[node] + ln softmax(row)[token] (temperature 1).
 */
int oracle_tree_level_static(int B, int V, int dtype, int R, const int32_t* static_parent, int level,
                             int sampled, double T, const void* logits, const float* u_draft,
                             int32_t* tokens, double* score, int32_t* near_tie) {
  if (B <= 0 || V <= 0 || R <= 0 || level < 1) return OR_BAD_ARG;
  int* dep = (int*)malloc(sizeof(int) * (size_t)R);
  double* lq = (double*)malloc(sizeof(double) * (size_t)V);
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  int* top = (int*)malloc(sizeof(int) * (size_t)R);
  if (!dep || !lq || !w || !top) {
    free(dep);
    free(lq);
    free(w);
    free(top);
    return OR_NO_MEM;
  }
  int rc = OR_OK;
  dep[0] = 0;
  for (int i = 1; i < R; ++i) {
    if (static_parent[i] < 0 || static_parent[i] >= i) rc = OR_BAD_ARG;
    else dep[i] = dep[static_parent[i]] + 1;
  }
  int F = 0;
  for (int i = 0; i < R && rc == OR_OK; ++i)
    if (dep[i] == level - 1) ++F;
  for (int b = 0; b < B && rc == OR_OK; ++b) {
    if (level == 1) score[(size_t)b * R] = 0.0;
    int f = 0;
    for (int n = 0; n < R && rc == OR_OK; ++n) {
      if (dep[n] != level - 1) continue;
      const size_t off = ((size_t)b * F + f) * V;
      ++f;
      int c = 0;
      for (int ch = n + 1; ch < R; ++ch)
        if (static_parent[ch] == n) ++c;
      if (c == 0) continue;
      if (c > V) {
        rc = OR_BAD_ARG;
        break;
      }
      log_softmax(logits, off, V, dtype, lq);
      if (!sampled) {
        if ((rc = row_topk(logits, off, V, dtype, c, top)) != OR_OK) break;
      } else {
        softmax_weights(logits, off, V, dtype, T, w);
      }
      int j = 0;
      for (int ch = n + 1; ch < R; ++ch) {
        if (static_parent[ch] != n) continue;
        int t;
        if (!sampled) {
          t = top[j];
        } else {
          int near = 0;
          t = icdf(w, V, (double)u_draft[(size_t)b * R + ch], &near);
          if (near) near_tie[b] += 1;
        }
        tokens[(size_t)b * R + ch] = t;
        score[(size_t)b * R + ch] = score[(size_t)b * R + n] + lq[t];
        ++j;
      }
    }
  }
  free(dep);
  free(lq);
  free(w);
  free(top);
  return rc;
}
