// launch.h -- internal launcher interface between the C-ABI layer (abi.cu) and the
// kernel files.  Launchers assume arguments were validated on the host.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/eagle.h"

namespace eagle {

// ------------------------------------------------------------------ tree build
struct StaticShape {
  int32_t rows;
  int8_t parent[128];
  int8_t depth[128];
  uint8_t lrank[128];  // a node's rank among the nodes of its depth, in index order
};

struct TreeBuildPlan {
  int B, V, mode, depth, k, N, R, W, dtype;
  float temperature;
  int n_chunks;   // vocabulary chunks per row
  int f_max;      // widest frontier
  int kc;         // entries of each chunk's top list that a level can use (top-k modes)
  int pool_cap;   // dynamic pool capacity per request
  StaticShape shape;
  // workspace carve-up (byte offsets)
  size_t off_pool_tok, off_pool_par, off_pool_score, off_pool_depth, off_state, off_front,
      off_part, off_node_tok, off_node_score, off_ticket, off_front_score, off_best_score, off_best_idx, total;
};
void plan_tree_build(const eagle_tree_desc* d, TreeBuildPlan* p);
int frontier_rows(const TreeBuildPlan& p, int level);
// One tree level from the draft model's hidden states of the frontier rows and its LM
// head (dynamic and static top-k trees): the head kernel writes the rows' records, the
// finishers select as from logits.
cudaError_t launch_tree_build_head(const TreeBuildPlan& plan, int level, const void* hidden, const void* weight,
                                   int hidden_dim, const int32_t* root_tok, const int32_t* seq_len, void* ws,
                                   const eagle_tree& out, uint32_t* status, cudaStream_t s);
cudaError_t launch_tree_build(const TreeBuildPlan& p, int level, const void* logits, const float* u_draft,
                              const int32_t* root_tok, const int32_t* seq_len, void* ws, const eagle_tree& out,
                              cudaStream_t s);

// The tree build's float-float natural logarithm on n values (self-test entry).
cudaError_t launch_ff_log_selftest(const float* z_hi, const float* z_lo, float* out_hi, float* out_lo, int n,
                                   cudaStream_t s);

// ------------------------------------------------------------------ tree attention
struct AttnPlan {
  int B, R, Hq, Hkv, G, D, P, dtype, W, out_dtype;
  bool precise;
  bool tc;           // tcgen05 kernel
  float scale;
  int rows_per_cta;  // query rows (node x head-in-group) per CTA
  int row_blocks;
  int splits;
  int rows_pad;      // row_blocks * rows_per_cta
  bool coop;         // tcgen05, splits > 1, grid fits on the SMs at once: the splits of a
                     // (request, KV head, row block) merge their partials in the kernel
  bool fault_test;   // test hook: the in-kernel split group waits for a split that never comes
  int tps;           // tcgen05 without coop: tile units per split (0: even splits)
  bool lpt;          // tcgen05 without coop, B > 1: longest requests dispatched first
  size_t off_err, off_cnt, off_o, off_ml, total;
};
// Records a CUDA error for eagle_last_cuda_error(); EAGLE_ERR_CUDA (EAGLE_OK on success).
int report_cuda_error(cudaError_t e);

void plan_tree_attn(const eagle_attn_desc* d, int num_sms, AttnPlan* p);
// Merge split partials into out / lse (shared by the mma.sync and tcgen05 kernels).
// pdl: programmatic launch (waits for the preceding kernel inside, lets the next start early)
cudaError_t launch_tree_attn_combine(const AttnPlan& p, const int32_t* seq_len, const int32_t* n_nodes, void* out,
                                     float* lse, const float* part_o, const float* part_ml, cudaStream_t s,
                                     bool pdl = false);
// The tcgen05 kernel (plan.tc); ws holds the error word and the partials.
cudaError_t launch_tree_attn_tc(const AttnPlan& p, const void* q, const void* k_cache, const void* v_cache,
                                const void* tree_k, const void* tree_v, const int32_t* seq_len,
                                const int32_t* n_nodes, const uint64_t* anc_mask, void* out, float* lse, void* ws,
                                cudaStream_t s);
cudaError_t launch_tree_attn(const AttnPlan& p, const void* q, const void* k_cache, const void* v_cache,
                             const void* tree_k, const void* tree_v, const int32_t* seq_len, const int32_t* n_nodes,
                             const uint64_t* anc_mask, void* out, float* lse, void* ws, cudaStream_t s);

// Training-time-test attention on the tcgen05 kernel (see eagle.h: eagle_ttt_attn).
cudaError_t launch_ttt_attn_tc(int steps, int S, int Hq, int Hkv, float scale, bool out_f32, const void* q,
                               const void* k_trunk, const void* v_trunk, const void* k_branch, const void* v_branch,
                               void* out, float* lse, void* ws, cudaStream_t s);

// ------------------------------------------------------------------ accept
struct AcceptPlan {
  int B, R, V, dtype, proposal, max_depth;
  float temperature;
  int n_chunks;
  int n_sources;  // 1 (target) or 2 (target + draft)
  size_t off_cnt, off_part, total;
};
void plan_accept(const eagle_accept_desc* d, AcceptPlan* p);
cudaError_t launch_accept(const AcceptPlan& p, const void* target, const void* draft, const int32_t* tokens,
                          const int32_t* parent, const float* u_accept, const float* u_final,
                          const eagle_accept_out& out, void* ws, cudaStream_t s);

// ------------------------------------------------------------------ LM-head statistics
int lmhead_tiles(int vocab);

// A tree-build vocabulary record of one frontier row: the best 16 (value desc, id asc)
// of the tokens it covers, sum exp(x - m) and sum exp((x - m) / T) as float-float pairs,
// and the max m.  Written by the tree build's chunk pass (one 4096-token chunk) or by the
// LM-head kernel (the tiles one persistent CTA covered).
struct TreeChunkRecord {
  float tv[16];
  int ti[16];
  float s1_hi, s1_lo, sT_hi, sT_lo;
  float m;
  float pad[3];
};
static_assert(sizeof(TreeChunkRecord) == 160, "tree chunk records are 160 bytes");

// Records per frontier row when the tree build reads the draft LM head (one per
// persistent CTA of the head kernel).
constexpr int kHeadRecords = 144;

// Draft LM head for a tree level: for hidden rows r = b F + f (M = B F <= 128), the
// record of row r for CTA c goes to trec[(b f_max + f) n_rec + c], c < n_rec.
cudaError_t launch_lmhead_tree_records(int M, int h, int V, int F, int f_max, int n_rec, const void* hidden,
                                       const void* weight, TreeChunkRecord* trec, uint32_t* status, cudaStream_t s);
cudaError_t launch_lmhead_stats(int M, int h, int V, int R, float temperature, const void* hidden, const void* weight,
                                const int32_t* tokens, const int32_t* parent, eagle_vocab_record* rec, float* child,
                                uint32_t* status, int num_sms, cudaStream_t s);

// ------------------------------------------------------------------ commit
constexpr int kMaxLayers = 128;
struct CommitArgs {
  void* k_cache[kMaxLayers];
  void* v_cache[kMaxLayers];
  const void* tree_k[kMaxLayers];
  const void* tree_v[kMaxLayers];
};
cudaError_t launch_kv_commit(const eagle_commit_desc* d, const CommitArgs& a, const int32_t* n_acc,
                             const int32_t* path, int32_t* seq_len, int32_t* commit_pos, void* feat_cache,
                             const void* tree_feat, uint32_t* status, cudaStream_t s);

}  // namespace eagle
