// abi.cu -- the extern "C" entry points of libeagle: host-side argument checks, then
// the launches on the caller's stream.  Every check runs before anything is
// enqueued; a failed check launches nothing.
#include <math.h>
#include <string.h>

#include "common.cuh"
#include "launch.h"

using namespace eagle;

namespace {

thread_local cudaError_t t_last_cuda = cudaSuccess;

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return EAGLE_OK;
  t_last_cuda = e;
  return EAGLE_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool dtype_ok(int t) { return t == EAGLE_F32 || t == EAGLE_BF16; }

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 152;
  }
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    return 152;
  }
  return n;
}

int check_tree_desc(const eagle_tree_desc* d) {
  if (!d) return EAGLE_ERR_INVALID_ARG;
  if (d->batch < 1 || d->vocab < 1) return EAGLE_ERR_INVALID_ARG;
  if (!dtype_ok(d->dtype) || d->vocab > kMaxTreeChunks * kVocabChunk) return EAGLE_ERR_UNSUPPORTED;
  if (d->mode == EAGLE_TREE_DYNAMIC) {
    if (d->depth < 1 || d->top_k < 1 || d->total_tokens < 1) return EAGLE_ERR_INVALID_ARG;
    if (d->depth > kMaxDepth || d->top_k > kMaxTopK || d->top_k > d->vocab) return EAGLE_ERR_UNSUPPORTED;
    const long long pool = d->top_k + static_cast<long long>(d->depth - 1) * d->top_k * d->top_k;
    if (pool > kMaxPool || d->total_tokens + 1 > kMaxRows) return EAGLE_ERR_UNSUPPORTED;
    if (d->total_tokens > pool) return EAGLE_ERR_INVALID_ARG;
    return EAGLE_OK;
  }
  if (d->mode != EAGLE_TREE_STATIC_TOPK && d->mode != EAGLE_TREE_STATIC_SAMPLED) return EAGLE_ERR_INVALID_ARG;
  if (d->n_static < 1 || !d->static_parent) return EAGLE_ERR_INVALID_ARG;
  if (d->n_static + 1 > kMaxRows) return EAGLE_ERR_UNSUPPORTED;
  if (d->mode == EAGLE_TREE_STATIC_SAMPLED && !(d->temperature > 0.f && isfinite(d->temperature)))
    return EAGLE_ERR_INVALID_ARG;
  const int R = d->n_static + 1;
  int depth[kMaxRows], kids[kMaxRows];
  depth[0] = 0;
  kids[0] = 0;
  for (int i = 1; i < R; ++i) {
    const int p = d->static_parent[i];
    if (p < 0 || p >= i) return EAGLE_ERR_INVALID_ARG;
    depth[i] = depth[p] + 1;
    if (depth[i] < depth[i - 1]) return EAGLE_ERR_INVALID_ARG;  // nodes ordered by depth
    kids[i] = 0;
    if (++kids[p] > kMaxTopK) return EAGLE_ERR_UNSUPPORTED;
    if (d->mode == EAGLE_TREE_STATIC_TOPK && kids[p] > d->vocab) return EAGLE_ERR_INVALID_ARG;
  }
  if (depth[R - 1] > kMaxDepth) return EAGLE_ERR_UNSUPPORTED;
  return EAGLE_OK;
}

int check_attn_desc(const eagle_attn_desc* d) {
  if (!d) return EAGLE_ERR_INVALID_ARG;
  if (d->batch < 1 || d->rows < 1 || d->n_q_heads < 1 || d->n_kv_heads < 1 || d->max_seq < 1)
    return EAGLE_ERR_INVALID_ARG;
  if (d->num_splits < 0 || !(d->scale > 0.f) || !isfinite(d->scale)) return EAGLE_ERR_INVALID_ARG;
  if (d->n_q_heads % d->n_kv_heads) return EAGLE_ERR_UNSUPPORTED;
  if (static_cast<long long>(d->batch) * d->n_kv_heads > 65535) return EAGLE_ERR_UNSUPPORTED;  // grid z
  if (d->head_dim != 64 && d->head_dim != 128) return EAGLE_ERR_UNSUPPORTED;
  if (d->rows > kMaxRows || !dtype_ok(d->dtype) || !dtype_ok(d->out_dtype)) return EAGLE_ERR_UNSUPPORTED;
  if (d->dtype == EAGLE_F32 && d->out_dtype != EAGLE_F32) return EAGLE_ERR_UNSUPPORTED;
  if (d->precision != EAGLE_ATTN_PRECISE && d->precision != EAGLE_ATTN_FAST) return EAGLE_ERR_INVALID_ARG;
  if (d->fault_test != 0 && d->fault_test != 1) return EAGLE_ERR_INVALID_ARG;
  return EAGLE_OK;
}

int check_ttt_desc(const eagle_ttt_desc* d) {
  if (!d) return EAGLE_ERR_INVALID_ARG;
  if (d->steps < 1 || d->seq < 1 || d->n_q_heads < 1 || d->n_kv_heads < 1 || !(d->scale > 0.f) ||
      !isfinite(d->scale))
    return EAGLE_ERR_INVALID_ARG;
  if (d->head_dim != 128 || d->n_q_heads % d->n_kv_heads || 128 % (d->n_q_heads / d->n_kv_heads))
    return EAGLE_ERR_UNSUPPORTED;
  if (d->out_dtype != EAGLE_BF16 && d->out_dtype != EAGLE_F32) return EAGLE_ERR_UNSUPPORTED;
  if (static_cast<long long>(d->steps) * d->n_kv_heads > 65535) return EAGLE_ERR_UNSUPPORTED;  // grid z
  return EAGLE_OK;
}

int check_accept_desc(const eagle_accept_desc* d) {
  if (!d) return EAGLE_ERR_INVALID_ARG;
  if (d->batch < 1 || d->rows < 1 || d->vocab < 1 || d->max_depth < 0) return EAGLE_ERR_INVALID_ARG;
  if (!(d->temperature >= 0.f) || !isfinite(d->temperature)) return EAGLE_ERR_INVALID_ARG;
  if (d->proposal != EAGLE_PROPOSAL_DELTA && d->proposal != EAGLE_PROPOSAL_SAMPLED) return EAGLE_ERR_INVALID_ARG;
  if (d->rows > kMaxRows || d->max_depth >= kMaxRows || !dtype_ok(d->dtype)) return EAGLE_ERR_UNSUPPORTED;
  if (d->vocab > kMaxVocabTiles * kVocabChunk) return EAGLE_ERR_UNSUPPORTED;
  return EAGLE_OK;
}

}  // namespace

// Records a CUDA error for eagle_last_cuda_error() and returns EAGLE_ERR_CUDA (EAGLE_OK
// for cudaSuccess); for entry points defined in other translation units.
int eagle::report_cuda_error(cudaError_t e) { return cuda_status(e); }

extern "C" {

const char* eagle_version(void) { return "eagle-tree-gb300 0.1 (sm_103a)"; }

int eagle_last_cuda_error(void) { return static_cast<int>(t_last_cuda); }

const char* eagle_last_cuda_error_string(void) { return cudaGetErrorName(t_last_cuda); }

const char* eagle_status_string(int status) {
  switch (status) {
    case EAGLE_OK: return "EAGLE_OK";
    case EAGLE_ERR_INVALID_ARG: return "EAGLE_ERR_INVALID_ARG: bad pointer, size or shape";
    case EAGLE_ERR_UNSUPPORTED: return "EAGLE_ERR_UNSUPPORTED: outside the supported envelope";
    case EAGLE_ERR_ALIGNMENT: return "EAGLE_ERR_ALIGNMENT: a device buffer is not 16-byte aligned";
    case EAGLE_ERR_WORKSPACE: return "EAGLE_ERR_WORKSPACE: workspace missing or too small";
    case EAGLE_ERR_CUDA: return "EAGLE_ERR_CUDA: kernel launch failed";
    default: return "unknown eagle status";
  }
}

size_t eagle_workspace_size(int which, const void* desc) {
  if (!desc) return 0;
  switch (which) {
    case EAGLE_WS_TREE_BUILD: {
      const eagle_tree_desc* d = static_cast<const eagle_tree_desc*>(desc);
      if (check_tree_desc(d) != EAGLE_OK) return 0;
      TreeBuildPlan p;
      plan_tree_build(d, &p);
      return p.total;
    }
    case EAGLE_WS_TREE_ATTN: {
      const eagle_attn_desc* d = static_cast<const eagle_attn_desc*>(desc);
      if (check_attn_desc(d) != EAGLE_OK) return 0;
      AttnPlan p;
      plan_tree_attn(d, num_sms(), &p);
      return p.total > 0 ? p.total : 16;
    }
    case EAGLE_WS_ACCEPT: {
      const eagle_accept_desc* d = static_cast<const eagle_accept_desc*>(desc);
      if (check_accept_desc(d) != EAGLE_OK) return 0;
      AcceptPlan p;
      plan_accept(d, &p);
      return p.total;
    }
    case EAGLE_WS_TTT_ATTN:
      return check_ttt_desc(static_cast<const eagle_ttt_desc*>(desc)) == EAGLE_OK ? 256 : 0;
    default: return 0;
  }
}

int eagle_tree_frontier_rows(const eagle_tree_desc* d, int level) {
  if (check_tree_desc(d) != EAGLE_OK) return -1;
  TreeBuildPlan p;
  plan_tree_build(d, &p);
  return frontier_rows(p, level);
}

int eagle_tree_max_frontier(const eagle_tree_desc* d) {
  if (check_tree_desc(d) != EAGLE_OK) return -1;
  TreeBuildPlan p;
  plan_tree_build(d, &p);
  return p.f_max;
}

int eagle_tree_attn_plan(const eagle_attn_desc* d, int32_t* splits, int32_t* kernels) {
  if (!d) return EAGLE_ERR_INVALID_ARG;
  const int st = check_attn_desc(d);
  if (st != EAGLE_OK) return st;
  AttnPlan p;
  plan_tree_attn(d, num_sms(), &p);
  if (splits) *splits = p.splits;
  if (kernels) *kernels = (p.splits > 1 && !p.coop) ? 2 : 1;
  return EAGLE_OK;
}

int eagle_tree_build(const eagle_tree_desc* d, int level, const void* frontier_logits, const float* u_draft,
                     const int32_t* root_tok, const int32_t* seq_len, void* ws, size_t ws_bytes,
                     const eagle_tree* out, void* stream) {
  int rc = check_tree_desc(d);
  if (rc != EAGLE_OK) return rc;
  TreeBuildPlan p;
  plan_tree_build(d, &p);
  if (level < 1 || level > p.depth) return EAGLE_ERR_INVALID_ARG;
  if (!frontier_logits || !root_tok || !seq_len || !out) return EAGLE_ERR_INVALID_ARG;
  if (d->mode == EAGLE_TREE_STATIC_SAMPLED && !u_draft) return EAGLE_ERR_INVALID_ARG;
  if (!out->tokens || !out->parent || !out->depth || !out->pos_id || !out->anc_mask || !out->score ||
      !out->frontier_tok || !out->frontier_slot || !out->near_tie)
    return EAGLE_ERR_INVALID_ARG;
  if (!aligned(frontier_logits, 16) || !aligned(ws, 16) || !aligned(out->anc_mask, 8) ||
      (u_draft && !aligned(u_draft, 4)))
    return EAGLE_ERR_ALIGNMENT;
  if (!ws || ws_bytes < p.total) return EAGLE_ERR_WORKSPACE;
  return cuda_status(launch_tree_build(p, level, frontier_logits, u_draft, root_tok, seq_len, ws, *out,
                           static_cast<cudaStream_t>(stream)));
}

int eagle_tree_build_head(const eagle_tree_desc* d, int level, const void* hidden, const void* head_weight,
                          int32_t hidden_dim, const int32_t* root_tok, const int32_t* seq_len, void* ws,
                          size_t ws_bytes, const eagle_tree* out, uint32_t* status, void* stream) {
  int rc = check_tree_desc(d);
  if (rc != EAGLE_OK) return rc;
  if (d->mode == EAGLE_TREE_STATIC_SAMPLED) return EAGLE_ERR_UNSUPPORTED;  // draws read the logits
  TreeBuildPlan p;
  plan_tree_build(d, &p);
  if (level < 1 || level > p.depth) return EAGLE_ERR_INVALID_ARG;
  if (hidden_dim < 64 || hidden_dim % 64 != 0) return hidden_dim < 1 ? EAGLE_ERR_INVALID_ARG : EAGLE_ERR_UNSUPPORTED;
  if (static_cast<long long>(d->batch) * p.f_max > 128) return EAGLE_ERR_UNSUPPORTED;  // one M-tile of rows
  if (!hidden || !head_weight || !root_tok || !seq_len || !out || !status) return EAGLE_ERR_INVALID_ARG;
  if (!out->tokens || !out->parent || !out->depth || !out->pos_id || !out->anc_mask || !out->score ||
      !out->frontier_tok || !out->frontier_slot || !out->near_tie)
    return EAGLE_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(head_weight, 16) || !aligned(ws, 16) || !aligned(out->anc_mask, 8) ||
      !aligned(status, 4))
    return EAGLE_ERR_ALIGNMENT;
  if (!ws || ws_bytes < p.total) return EAGLE_ERR_WORKSPACE;
  return cuda_status(launch_tree_build_head(p, level, hidden, head_weight, hidden_dim, root_tok, seq_len, ws, *out,
                                            status, static_cast<cudaStream_t>(stream)));
}

int eagle_tree_attn(const eagle_attn_desc* d, const void* q, const void* k_cache, const void* v_cache,
                    const void* tree_k, const void* tree_v, const int32_t* seq_len, const int32_t* n_nodes,
                    const uint64_t* anc_mask, void* out, float* lse, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_attn_desc(d);
  if (rc != EAGLE_OK) return rc;
  if (!q || !k_cache || !v_cache || !tree_k || !tree_v || !seq_len || !anc_mask || !out)
    return EAGLE_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(tree_k, 16) ||
      !aligned(tree_v, 16) || !aligned(out, 16) || !aligned(anc_mask, 8) || (lse && !aligned(lse, 4)) ||
      (n_nodes && !aligned(n_nodes, 4)) ||
      (ws && !aligned(ws, 16)))
    return EAGLE_ERR_ALIGNMENT;
  AttnPlan p;
  plan_tree_attn(d, num_sms(), &p);
  if (p.total > 0 && (!ws || ws_bytes < p.total)) return EAGLE_ERR_WORKSPACE;
  return cuda_status(launch_tree_attn(p, q, k_cache, v_cache, tree_k, tree_v, seq_len, n_nodes, anc_mask, out, lse, ws,
                          static_cast<cudaStream_t>(stream)));
}

int eagle_accept(const eagle_accept_desc* d, const void* target_logits, const void* draft_logits,
                 const int32_t* tree_tokens, const int32_t* tree_parent, const float* u_accept,
                 const float* u_final, const eagle_accept_out* out, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_accept_desc(d);
  if (rc != EAGLE_OK) return rc;
  const bool need_draft = d->temperature > 0.f && d->proposal == EAGLE_PROPOSAL_SAMPLED;
  if (!target_logits || (need_draft && !draft_logits) || !tree_tokens || !tree_parent || !u_accept || !u_final ||
      !out)
    return EAGLE_ERR_INVALID_ARG;
  if (!out->n_acc || !out->path || !out->out_tok || !out->near_tie || !out->status) return EAGLE_ERR_INVALID_ARG;
  if (!aligned(target_logits, 16) || (draft_logits && !aligned(draft_logits, 16)) || !aligned(ws, 16))
    return EAGLE_ERR_ALIGNMENT;
  AcceptPlan p;
  plan_accept(d, &p);
  if (!ws || ws_bytes < p.total) return EAGLE_ERR_WORKSPACE;
  return cuda_status(launch_accept(p, target_logits, need_draft ? draft_logits : nullptr, tree_tokens, tree_parent, u_accept,
                       u_final, *out, ws, static_cast<cudaStream_t>(stream)));
}

int eagle_kv_commit(const eagle_commit_desc* d, void* const* k_cache_layers, void* const* v_cache_layers,
                    const void* const* tree_k_layers, const void* const* tree_v_layers, const int32_t* n_acc,
                    const int32_t* path, int32_t* seq_len, int32_t* commit_pos, void* feat_cache,
                    const void* tree_feat, uint32_t* status, void* stream) {
  if (!d) return EAGLE_ERR_INVALID_ARG;
  if (d->layers < 1 || d->batch < 1 || d->n_kv_heads < 1 || d->head_dim < 1 || d->rows < 1 || d->max_seq < 1 ||
      d->max_depth < 0 || d->feat_dim < 0)
    return EAGLE_ERR_INVALID_ARG;
  if (d->layers > kMaxLayers || d->rows > kMaxRows || d->max_depth >= kMaxRows || !dtype_ok(d->dtype) ||
      (d->feat_dim > 0 && !dtype_ok(d->feat_dtype)))
    return EAGLE_ERR_UNSUPPORTED;
  const int esz = d->dtype == EAGLE_F32 ? 4 : 2;
  if ((d->head_dim * esz) % 16) return EAGLE_ERR_UNSUPPORTED;
  if (!k_cache_layers || !v_cache_layers || !tree_k_layers || !tree_v_layers || !n_acc || !path || !seq_len)
    return EAGLE_ERR_INVALID_ARG;
  if (d->feat_dim > 0 && (!feat_cache || !tree_feat)) return EAGLE_ERR_INVALID_ARG;
  CommitArgs a;
  memset(&a, 0, sizeof a);
  for (int l = 0; l < d->layers; ++l) {
    if (!k_cache_layers[l] || !v_cache_layers[l] || !tree_k_layers[l] || !tree_v_layers[l])
      return EAGLE_ERR_INVALID_ARG;
    if (!aligned(k_cache_layers[l], 16) || !aligned(v_cache_layers[l], 16) || !aligned(tree_k_layers[l], 16) ||
        !aligned(tree_v_layers[l], 16))
      return EAGLE_ERR_ALIGNMENT;
    a.k_cache[l] = k_cache_layers[l];
    a.v_cache[l] = v_cache_layers[l];
    a.tree_k[l] = tree_k_layers[l];
    a.tree_v[l] = tree_v_layers[l];
  }
  if (d->feat_dim > 0) {
    const int fsz = d->feat_dtype == EAGLE_F32 ? 4 : 2;
    const size_t rb = static_cast<size_t>(d->feat_dim) * fsz;
    if (rb % 16 == 0 && (!aligned(feat_cache, 16) || !aligned(tree_feat, 16))) return EAGLE_ERR_ALIGNMENT;
  }
  return cuda_status(launch_kv_commit(d, a, n_acc, path, seq_len, commit_pos, feat_cache, tree_feat, status,
                          static_cast<cudaStream_t>(stream)));
}


int eagle_ttt_attn(const eagle_ttt_desc* d, const void* q, const void* k_trunk, const void* v_trunk,
                   const void* k_branch, const void* v_branch, void* out, float* lse, void* ws, size_t ws_bytes,
                   void* stream) {
  const int rc = check_ttt_desc(d);
  if (rc != EAGLE_OK) return rc;
  if (!q || !k_trunk || !v_trunk || !out || (d->steps > 1 && (!k_branch || !v_branch))) return EAGLE_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_trunk, 16) || !aligned(v_trunk, 16) || !aligned(out, 16) ||
      (k_branch && !aligned(k_branch, 16)) || (v_branch && !aligned(v_branch, 16)) || (lse && !aligned(lse, 4)) ||
      (ws && !aligned(ws, 16)))
    return EAGLE_ERR_ALIGNMENT;
  if (!ws || ws_bytes < 256) return EAGLE_ERR_WORKSPACE;
  return cuda_status(launch_ttt_attn_tc(d->steps, d->seq, d->n_q_heads, d->n_kv_heads, d->scale,
                                        d->out_dtype == EAGLE_F32, q, k_trunk, v_trunk, k_branch, v_branch, out, lse,
                                        ws, static_cast<cudaStream_t>(stream)));
}

int eagle_lmhead_stats(const eagle_lmhead_desc* d, const void* hidden, const void* weight,
                       const int32_t* tree_tokens, const int32_t* tree_parent, eagle_vocab_record* records,
                       float* child_logit, uint32_t* status, void* stream) {
  if (!d || !hidden || !weight || !records || !status) return EAGLE_ERR_INVALID_ARG;
  if (d->rows < 1 || d->tree_rows < 1 || d->hidden < 1 || d->vocab < 1 || d->rows % d->tree_rows)
    return EAGLE_ERR_INVALID_ARG;
  if (!isfinite(d->temperature)) return EAGLE_ERR_INVALID_ARG;
  if ((tree_tokens == nullptr) != (tree_parent == nullptr) || (tree_tokens && !child_logit))
    return EAGLE_ERR_INVALID_ARG;
  if (d->rows > 128 || d->hidden % 64) return EAGLE_ERR_UNSUPPORTED;
  if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(records, 16)) return EAGLE_ERR_ALIGNMENT;
  return cuda_status(launch_lmhead_stats(d->rows, d->hidden, d->vocab, d->tree_rows, d->temperature, hidden, weight,
                                         tree_tokens, tree_parent, records, tree_tokens ? child_logit : nullptr,
                                         status, num_sms(), static_cast<cudaStream_t>(stream)));
}

int eagle_selftest_ff_log(const float* z_hi, const float* z_lo, float* out_hi, float* out_lo, int32_t n,
                          void* stream) {
  if (n < 0 || (n > 0 && (!z_hi || !z_lo || !out_hi || !out_lo))) return EAGLE_ERR_INVALID_ARG;
  return cuda_status(launch_ff_log_selftest(z_hi, z_lo, out_hi, out_lo, n, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
