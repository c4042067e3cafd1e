/*
 * eagle.h -- C ABI of the EAGLE draft-tree verify step on one GB300 (sm_103a).
 *
 * One verify step of EAGLE-style lossless speculative decoding has four stages,
 * one entry point each:
 *
 *   eagle_tree_build  draft-tree construction, one draft level per call
 *                     (EAGLE review (zenmind), section 3.1 and appendix A.1:
 *                     top-k children per node, k = 4 at the root, static tree;
 *                     EAGLE-3 visual reading, "EAGLE-2": dynamic tree that keeps
 *                     the most confident candidates, draft confidence tracking
 *                     acceptance, Figures 4 and 6).
 *   eagle_tree_attn   attention of every tree node over the prefix KV cache and
 *                     its own ancestors in the tree (EAGLE review, terms "tree
 *                     attention" and section 3.3; lesson "Speculative decoding
 *                     and EAGLE-3", glossary "Tree attention": a flash-attention
 *                     call with a tree mask).
 *   eagle_accept      multi-round speculative sampling down the tree, greedy
 *                     argmax matching at temperature 0 (EAGLE review, section 3.3
 *                     and appendix A.2 / Algorithm 1; lesson steps 1-2, "bonus
 *                     token").
 *   eagle_kv_commit   compaction of the accepted path's K/V (and feature rows)
 *                     into the contiguous cache (EAGLE review, section 3.3 and
 *                     data path step 7; lesson "KV cache rollback", step 4).
 *
 * Conventions shared by every call
 *   - All buffer pointers are DEVICE pointers unless the comment says HOST.
 *     The caller owns every buffer; the library allocates nothing, keeps no
 *     state between calls and is reentrant.  Scratch memory comes from the
 *     caller's `ws` buffer, sized by eagle_workspace_size().  The one exception
 *     is eagle_accept_noalloc, which takes its scratch from a fixed device array
 *     inside the library instead (see there: one array per device, shared by
 *     every call, so its calls on a device must not overlap).
 *   - A workspace belongs to one descriptor: calls whose descriptors differ may
 *     lay their scratch out differently, so give each its own workspace (or
 *     re-zero it between them).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *     only enqueues work on it and returns; nothing synchronises.  Outputs are
 *     valid once the stream has reached the call's work.  No call does a
 *     device-to-host copy, so a whole verify step can be captured in one graph.
 *   - Argument errors are detected on the host before anything is enqueued and
 *     returned as EAGLE_ERR_*; nothing is launched in that case.  Conditions that
 *     depend on device data (a malformed tree, a full cache) set bits in a device
 *     status word that the caller reads after the stream completes.  No call
 *     traps, asserts or prints on the device.
 *   - Element types: EAGLE_F32 or EAGLE_BF16.  Every accumulation is fp32.
 *   - Device buffers must be 16-byte aligned (EAGLE_ERR_ALIGNMENT otherwise).
 *
 * Shapes (B batch, R tree rows including the root, V vocabulary, Hq / Hkv query /
 * KV heads, G = Hq / Hkv, D head dim, P cache capacity per request, W = ceil(R/64))
 *   tree tokens / parent / depth / pos_id   int32  [B][R]   row 0 = root, parent[0] = -1,
 *                                                           parent[i] < i (parents first)
 *   ancestor mask                           uint64 [B][R][W] bit j of row i set iff node j
 *                                                           is node i or an ancestor of i
 *   q, attention out                        [B][R][Hq][D]
 *   KV cache (per layer)                    [B][Hkv][P][D]
 *   tree K/V (per layer)                    [B][Hkv][R][D]
 *   logits                                  [B][R][V]
 */
#ifndef EAGLE_H
#define EAGLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status codes */
enum {
  EAGLE_OK = 0,
  EAGLE_ERR_INVALID_ARG = 1, /* NULL pointer, non-positive size, inconsistent shape */
  EAGLE_ERR_UNSUPPORTED = 2, /* outside the supported envelope (see each call) */
  EAGLE_ERR_ALIGNMENT = 3,   /* a device buffer is not 16-byte aligned */
  EAGLE_ERR_WORKSPACE = 4,   /* ws is NULL or smaller than eagle_workspace_size() */
  EAGLE_ERR_CUDA = 5         /* a kernel launch failed; cudaGetLastError() has the cause */
};

/* Bits of the device status word written by eagle_accept / eagle_kv_commit.
 * The caller zeroes the word; the library only ORs bits into it. */
#define EAGLE_STATUS_BAD_TREE 0x1u      /* a row's parent is not an earlier row, or a path node is out of range */
#define EAGLE_STATUS_PATH_OVERFLOW 0x2u /* accepted path deeper than max_depth: truncated */
#define EAGLE_STATUS_CACHE_FULL 0x4u    /* seq_len + n_acc + 1 > max_seq: that request was not committed */
#define EAGLE_STATUS_BAD_TOKEN 0x8u     /* a draft token outside [0, V): treated as rejected */
#define EAGLE_STATUS_TIMEOUT 0x10u      /* eagle_accept: a bounded wait between the CTAs of a request
                                           gave up (2 s); that request's outputs were not written */

/* Element types */
enum { EAGLE_F32 = 0, EAGLE_BF16 = 1 };

/* Tree modes */
enum {
  EAGLE_TREE_DYNAMIC = 0,       /* EAGLE-2: top-k per frontier node, rerank by cumulative confidence */
  EAGLE_TREE_STATIC_TOPK = 1,   /* fixed shape; a node's children are its best tokens in rank order */
  EAGLE_TREE_STATIC_SAMPLED = 2 /* fixed shape; children drawn i.i.d. from the draft distribution */
};

/* What distribution a draft candidate was proposed from (used by eagle_accept). */
enum {
  EAGLE_PROPOSAL_DELTA = 0,  /* deterministic candidates (top-k / dynamic trees): q = point mass */
  EAGLE_PROPOSAL_SAMPLED = 1 /* candidates drawn from softmax(draft / T): q = that softmax */
};

/* Precision of the attention PV product (bf16 path) */
enum {
  EAGLE_ATTN_PRECISE = 0, /* default: P enters the PV product as two bf16 terms (hi + lo, about 16
                             significant bits; one extra MMA per PV step) and split partials stay
                             fp32, so the only bf16 rounding after the inputs is that of a bf16
                             output: max abs error 2e-3 + 2^-8 |O| against exact arithmetic */
  EAGLE_ATTN_FAST = 1     /* P rounded to bf16 once (8 significant bits), as flash attention does:
                             cheaper, but on sharply peaked rows the rounding of P moves O by up to
                             2^-8 max|v| */
};

/* Attention kernel selection.  The tcgen05 kernel covers bf16 inputs with head_dim 128
 * and 128 % (Hq / Hkv) == 0; everything else runs the mma.sync (bf16) or SIMT (fp32)
 * kernels. */
enum { EAGLE_ENGINE_AUTO = 0, EAGLE_ENGINE_MMA_SYNC = 1 };

/* Workspace kinds for eagle_workspace_size() */
enum { EAGLE_WS_TREE_BUILD = 1, EAGLE_WS_TREE_ATTN = 2, EAGLE_WS_ACCEPT = 3, EAGLE_WS_TTT_ATTN = 4 };

/* ---------------------------------------------------------------- tree build */
typedef struct {
  int32_t batch;              /* B >= 1 */
  int32_t vocab;              /* 1 <= V <= 524288 (128 chunks of 4096 tokens) */
  int32_t mode;               /* EAGLE_TREE_* */
  int32_t depth;              /* draft levels D, 1..16 (dynamic), or the static shape's depth */
  int32_t top_k;              /* dynamic: children per frontier node and frontier width, 1..16 */
  int32_t total_tokens;       /* dynamic: drafts kept N; rows R = N + 1 <= 128 and N <= the pool size */
  int32_t n_static;           /* static: number of draft nodes; R = n_static + 1 <= 128 */
  const int32_t* static_parent; /* static: HOST array [R], parent[0] = -1, parent[i] < i, nodes
                                   ordered by depth; at most 16 children per node */
  int32_t dtype;              /* element type of the draft logits */
  float temperature;          /* STATIC_SAMPLED: draw temperature (> 0) */
} eagle_tree_desc;

typedef struct {             /* all DEVICE pointers, caller-allocated */
  int32_t* tokens;           /* [B][R]   written after the last level */
  int32_t* parent;           /* [B][R]   written after the last level */
  int32_t* depth;            /* [B][R]   written after the last level */
  int32_t* pos_id;           /* [B][R]   = seq_len[b] + depth, written after the last level */
  uint64_t* anc_mask;        /* [B][R][W] written after the last level */
  float* score;              /* [B][R]   cumulative ln draft confidence (root 0) */
  int32_t* frontier_tok;     /* [B][F_max] tokens of the nodes whose draft rows feed the next level */
  int32_t* frontier_slot;    /* [B][F_max] each such node's parent row in this level's input */
  int32_t* near_tie;         /* [B]      1 if a selection boundary fell between two scores less
                                           than 1e-5 apart (siblings with equal logits excepted: both
                                           sides break those by index), or a draw landed within 1e-7 of
                                           the row's mass from a bin edge */
} eagle_tree;

/* Rows the frontier_logits of `level` must have: 1 at level 1; then top_k (dynamic)
 * or the number of depth level-1 nodes (static).  -1 on a bad argument. */
int eagle_tree_frontier_rows(const eagle_tree_desc* d, int level);

/* Widest frontier over all levels (the F_max of eagle_tree.frontier_*). */
int eagle_tree_max_frontier(const eagle_tree_desc* d);

/* Run draft level `level` (1..depth) of the tree build.
 *   frontier_logits  [B][F][V] draft logits of the current frontier rows, in the
 *                    order eagle_tree.frontier_tok listed them after the previous
 *                    level (level 1: the root row).
 *   u_draft          [B][R] fp32 uniforms in [0,1), one per node (STATIC_SAMPLED;
 *                    else may be NULL).  Node i's token is drawn with u_draft[b][i].
 *   root_tok, seq_len [B] int32: the pending token and the prefix length (used by
 *                    the last level).
 *   ws               scratch of eagle_workspace_size(EAGLE_WS_TREE_BUILD, d) bytes.
 *                    It carries the candidate pool from level to level: pass the
 *                    same ws, untouched, to levels 1..depth of one build.  Level 1
 *                    clears its counters (one memset on the stream), so it need not be
 *                    zero-filled.
 * After each level frontier_tok / frontier_slot name the next level's rows.  The
 * last level writes the tree.  Ties inside a row go to the lower token id;
 * cumulative scores are float-float (about 48 bits) with the pool index breaking
 * ties.  One kernel launch per level (after level 1's memset): the last CTA to
 * finish a frontier row merges that row, and the last row of a request selects. */
int eagle_tree_build(const eagle_tree_desc* d, int level, const void* frontier_logits,
                     const float* u_draft, const int32_t* root_tok, const int32_t* seq_len,
                     void* ws, size_t ws_bytes, const eagle_tree* out, void* stream);

/* One draft level of the tree build from the draft model's hidden states instead of its
 * logits: the draft LM head fused with tree expansion (EAGLE review, section 3.1: the
 * draft maps its predicted feature to tokens through the frozen LM head; EAGLE-3 visual
 * reading, "EAGLE-2": the dynamic tree keeps the most confident candidates).  For each
 * frontier row, logits x = hidden W^T (bf16 x bf16, fp32 accumulation, on the tensor
 * cores) are reduced to the row's softmax statistics (T = 1) and its best tokens by
 * (logit desc, id asc) without being written; the level then selects exactly as
 * eagle_tree_build does from logits with those values.
 *   hidden       [B][F][hidden_dim] bf16 DEVICE: the draft's last hidden states of the
 *                frontier rows, in eagle_tree.frontier_tok order (level 1: the root).
 *   head_weight  [V][hidden_dim] bf16 DEVICE, row-major (the frozen LM head).
 *   status       DEVICE uint32: EAGLE_STATUS_TIMEOUT is ORed in when a bounded wait of
 *                the head kernel gives up (2 s); the caller clears it.
 *   ws, out      as eagle_tree_build (the same workspace size; level 1 clears its
 *                counters).  Levels from logits and from hidden states may be mixed.
 * Modes: EAGLE_TREE_DYNAMIC and EAGLE_TREE_STATIC_TOPK (STATIC_SAMPLED draws need the
 * logits: EAGLE_ERR_UNSUPPORTED).  Unsupported: hidden_dim not a multiple of 64,
 * B x (widest frontier) > 128.  Near-ties as eagle_tree_build. */
int eagle_tree_build_head(const eagle_tree_desc* d, int level, const void* hidden, const void* head_weight,
                          int32_t hidden_dim, const int32_t* root_tok, const int32_t* seq_len, void* ws,
                          size_t ws_bytes, const eagle_tree* out, uint32_t* status, void* stream);

/* ---------------------------------------------------------------- tree attention */
typedef struct {
  int32_t batch;       /* B */
  int32_t rows;        /* R = tree rows incl. root, 1..128 */
  int32_t n_q_heads;   /* Hq, a multiple of n_kv_heads */
  int32_t n_kv_heads;  /* Hkv */
  int32_t head_dim;    /* D: 64 or 128 */
  int32_t max_seq;     /* P: cache capacity per request (rows of the K/V cache) */
  float scale;         /* softmax scale, usually 1/sqrt(D) */
  int32_t dtype;       /* element type of q, caches and tree K/V */
  int32_t num_splits;  /* prefix splits per (request, KV head); 0 = choose: from the SM count
                          when the grid fits on the SMs at once, else key pieces of a fixed
                          number of tiles per request */
  int32_t out_dtype;   /* element type of out: EAGLE_F32, or EAGLE_BF16 when dtype is EAGLE_BF16 */
  int32_t precision;   /* EAGLE_ATTN_PRECISE (0, default) or EAGLE_ATTN_FAST (ignored for fp32 inputs) */
  int32_t engine;      /* EAGLE_ENGINE_AUTO (tensor-core tcgen05 kernel where supported) or
                          EAGLE_ENGINE_MMA_SYNC (the legacy warp-level MMA kernel) */
  int32_t fault_test;  /* 0 in normal use.  1 is a test hook for the failure path of the
                          tcgen05 kernel's in-kernel split merge: each split group waits for
                          one split more than exist and gives up after 1 ms, so the call
                          returns with bit 0x100 set in the workspace error word and the
                          outputs unwritten (re-zero the workspace afterwards).  No effect
                          when the splits do not merge in the kernel. */
} eagle_attn_desc;

/* One layer of tree attention.  Row i of request b, query head hq attends to the
 * prefix keys j < seq_len[b] of KV head hq / G and to the tree keys a < n_nodes[b]
 * whose bit is set in anc_mask[b][i]:
 *     out = softmax(scale * q k^T) v,   lse = ln sum exp(scale * q k^T)  (natural log)
 *   q [B][R][Hq][D]; k_cache, v_cache [B][Hkv][P][D]; tree_k, tree_v [B][Hkv][R][D];
 *   seq_len [B] int32 (0 <= seq_len <= P); anc_mask [B][R][W]; out [B][R][Hq][D];
 *   lse [B][R][Hq] fp32, may be NULL.
 *   n_nodes [B] int32, may be NULL (every request has R rows): request b's tree has
 *   n_nodes[b] rows (clamped to [0, R]), so requests with trees of different sizes
 *   share one call; rows i >= n_nodes[b] of out and lse are left untouched and the
 *   tree keys >= n_nodes[b] are ignored whatever their mask bits say.
 * ws: eagle_workspace_size(EAGLE_WS_TREE_ATTN, d) bytes (split partials and, for the
 * tcgen05 kernel, an error word and split-group counters), zero-filled by the caller
 * before its first use; every call leaves the counters at zero again.  The tcgen05
 * kernel ORs a bit into the error word (the first 4 bytes of ws) when a bounded wait
 * inside it gives up; the word stays set until the caller clears it, and the outputs
 * of the calls made since it was last zero are not valid (re-zero the whole workspace
 * before further use).  When the splits merge inside the kernel its launch is
 * cooperative (all CTAs resident at once, one per SM).  The tcgen05 launch is
 * programmatic: its setup may overlap the preceding kernel in the stream, and it reads
 * its inputs (and ws) only once that kernel has completed.
 * Unsupported: head_dim not 64/128, R > 128, Hq % Hkv != 0, B * Hkv > 65535, bf16 out
 * with fp32 inputs. */
int eagle_tree_attn(const eagle_attn_desc* d, const void* q, const void* k_cache, const void* v_cache,
                    const void* tree_k, const void* tree_v, const int32_t* seq_len, const int32_t* n_nodes,
                    const uint64_t* anc_mask, void* out, float* lse, void* ws, size_t ws_bytes,
                    void* stream);

/* How eagle_tree_attn runs a descriptor on the current device (no counterpart in the
 * method's description; it reports the launch plan): *splits = prefix splits per
 * (request, KV head, row block), *kernels = kernel launches one call makes (1, or 2
 * when a separate kernel merges the splits).  Either pointer may be NULL.  Returns
 * EAGLE_OK, or the status eagle_tree_attn would return for a bad descriptor. */
int eagle_tree_attn_plan(const eagle_attn_desc* d, int32_t* splits, int32_t* kernels);

/* ---------------------------------------------------------------- acceptance */
typedef struct {
  int32_t batch;       /* B */
  int32_t rows;        /* R, 1..128 */
  int32_t vocab;       /* V */
  float temperature;   /* T; 0 = greedy argmax matching */
  int32_t proposal;    /* EAGLE_PROPOSAL_* (ignored when T == 0) */
  int32_t dtype;       /* element type of the logits */
  int32_t max_depth;   /* path arrays hold max_depth + 1 entries */
} eagle_accept_desc;

typedef struct {       /* all DEVICE pointers, caller-allocated */
  int32_t* n_acc;      /* [B] accepted drafts */
  int32_t* path;       /* [B][max_depth+1] accepted node rows, root first, -1 padded */
  int32_t* out_tok;    /* [B][max_depth+1] accepted tokens then the emitted token, -1 padded */
  int32_t* near_tie;   /* [B] 1 if an accept decision had |u - p/q| < 1e-5, or the final draw
                          landed within 1e-7 of the distribution's mass from a bin edge */
  uint32_t* status;    /* [1] EAGLE_STATUS_* bits (ORed) */
} eagle_accept_out;

/* Walk the tree from the root.  T == 0: the child whose token is the target argmax
 * (lowest id on ties) is accepted, else the argmax is emitted.  T > 0: with
 * p = softmax(target[cur] / T), the children of cur are tried in row order:
 * child d is accepted iff u_accept[b][child] < p(d) / q(d); otherwise
 * p <- norm(max(0, p - q)) and the next child is tried; when all are rejected, or
 * cur is a leaf, icdf(p, u_final[b]) is emitted (the smallest index whose running
 * sum exceeds u * sum).  q is a point mass on d for EAGLE_PROPOSAL_DELTA and
 * softmax(draft[cur] / T) for EAGLE_PROPOSAL_SAMPLED.
 *   target_logits, draft_logits [B][R][V] (draft only for SAMPLED, else NULL);
 *   tree_tokens, tree_parent [B][R]; u_accept [B][R]; u_final [B] (fp32 in [0,1)).
 * ws: eagle_workspace_size(EAGLE_WS_ACCEPT, d) bytes. */
int eagle_accept(const eagle_accept_desc* d, const void* target_logits, const void* draft_logits,
                 const int32_t* tree_tokens, const int32_t* tree_parent, const float* u_accept,
                 const float* u_final, const eagle_accept_out* out, void* ws, size_t ws_bytes,
                 void* stream);

/* eagle_accept without a caller workspace.  The method's description has no
 * counterpart: this is a deployment convenience for callers that cannot allocate
 * device memory when they verify a draft (memory reserved up front, an allocator
 * that is not reachable from the calling thread, plain C code with no device
 * allocator).  Same arguments, semantics and kernels as eagle_accept, minus ws and
 * ws_bytes: the scratch eagle_accept would take from ws lives in a device array of
 * EAGLE_ACCEPT_NOALLOC_SCRATCH_BYTES inside the library (one per device).  The call
 * allocates nothing.
 *   - A descriptor whose scratch (eagle_workspace_size(EAGLE_WS_ACCEPT, d)) exceeds
 *     EAGLE_ACCEPT_NOALLOC_SCRATCH_BYTES is rejected with EAGLE_ERR_WORKSPACE before
 *     anything is launched.  4 MiB is 768 bytes per tree row and proposal source at
 *     vocab 128256: up to 89 requests of 61 rows with one source, 44 with the draft
 *     logits as a second source.
 *   - The first call on each device looks the buffer's address up (a CUDA runtime
 *     query, done once per device with that device current); make that first call
 *     outside any stream capture.  The address is kept for the life of the process:
 *     a device reset (cudaDeviceReset, or anything else that destroys the primary
 *     context) after the first call is not supported, since later calls would
 *     launch with the old address.
 *   - The buffer needs no clearing: each call zeroes the counters it uses and
 *     writes every other entry before reading it.
 *   - One buffer per device: calls on the same device must not overlap in time
 *     (concurrent streams or host threads would race on it). */
#define EAGLE_ACCEPT_NOALLOC_SCRATCH_BYTES (4u << 20)
int eagle_accept_noalloc(const eagle_accept_desc* d, const void* target_logits, const void* draft_logits,
                         const int32_t* tree_tokens, const int32_t* tree_parent, const float* u_accept,
                         const float* u_final, const eagle_accept_out* out, void* stream);

/* ---------------------------------------------------------------- training-time-test attention */
/* The attention of EAGLE-3's training-time test (EAGLE-3 visual reading, "训练时的
 * Attention Mask 设计"; Didi EAGLE-3 article, sections 5.2-5.3): the draft model is
 * trained on its own k-step rollouts, and TTT step j's prediction at position t attends
 * causally to the original sequence (trunk keys t' <= t) and, through the diagonal
 * mask, only to its own predecessors at the same position in the earlier steps (branch
 * keys (i, t), 1 <= i <= j), all under one softmax:
 *     out = softmax(scale * q [K_trunk(<= t); K_branch(1..j, t)]^T) [V_trunk(<= t); V_branch(1..j, t)]
 *     lse = ln sum exp(...)
 * The trunk runs on the tensor cores (the causal keys, tile by tile, with the tree
 * attention kernel's machinery); the j branch keys of a row are a few dot products
 * folded into the row's softmax at the end (the streaming-softmax fusion of trunk and
 * branch).  bf16 inputs, fp32 accumulation, P split into two bf16 terms in the PV
 * product (as EAGLE_ATTN_PRECISE).
 *   q [k][S][Hq][128]; k_trunk, v_trunk [Hkv][S][128] (the original sequence's keys,
 *   shared by every step); k_branch, v_branch [k][Hkv][S][128] (step i's predictions'
 *   keys; step 0's entries are not read); out [k][S][Hq][128] (bf16 or fp32 by
 *   out_dtype); lse [k][S][Hq] fp32, may be NULL.
 * ws: eagle_workspace_size(EAGLE_WS_TTT_ATTN, d) bytes, zero-filled; its first 4 bytes
 * are an error word that a bounded wait ORs a bit into when it gives up (2 s).
 * Unsupported: head_dim != 128, 128 % (Hq / Hkv) != 0, Hq % Hkv != 0. */
typedef struct {
  int32_t steps;       /* k >= 1 */
  int32_t seq;         /* S >= 1 */
  int32_t n_q_heads;   /* Hq */
  int32_t n_kv_heads;  /* Hkv */
  int32_t head_dim;    /* 128 */
  float scale;         /* usually 1/sqrt(128) */
  int32_t out_dtype;   /* EAGLE_BF16 or EAGLE_F32 */
} eagle_ttt_desc;

int eagle_ttt_attn(const eagle_ttt_desc* d, const void* q, const void* k_trunk, const void* v_trunk,
                   const void* k_branch, const void* v_branch, void* out, float* lse, void* ws, size_t ws_bytes,
                   void* stream);

/* ---------------------------------------------------------------- LM-head statistics */
/* What acceptance needs from the target model's distribution at every tree node,
 * computed from the verify pass's hidden states and the frozen LM head without
 * writing the [rows][V] logits (EAGLE review, "GPU / system data path" steps 3 and 6:
 * the LM head gives the distribution at each node; section 3.3 / Algorithm 1: the
 * multi-round test reads each child's token probability under its parent, the bonus
 * draw reads the distribution).  logits x = hidden W^T, fp32 accumulation. */
#define EAGLE_LMHEAD_TILE 128 /* vocabulary entries per record */

typedef struct {
  int32_t rows;        /* M = B * R hidden rows, 1..128: row b * R + i is node i of request b */
  int32_t tree_rows;   /* R, rows per request (M a multiple of R) */
  int32_t hidden;      /* h, a multiple of 64 */
  int32_t vocab;       /* V */
  float temperature;   /* T of the sums (T <= 0 counts as 1) */
} eagle_lmhead_desc;

typedef struct {       /* one row's statistics over one tile of EAGLE_LMHEAD_TILE tokens */
  float max;           /* max logit */
  int32_t argmax;      /* its token (lowest id on ties) */
  float sum_hi, sum_lo; /* sum exp((x - max) / T) over the tile, as the float pair hi + lo */
} eagle_vocab_record;

/* hidden [M][h] bf16, weight [V][h] bf16 (row v = token v's output embedding), both
 * 16-byte aligned with h * 2 a multiple of 16.  records [M][ceil(V / 128)] (DEVICE).
 * tree_tokens, tree_parent [B][R] int32 (may both be NULL): then child_logit [M] gets,
 * for every node i >= 1 of request b, the logit of its token under its parent's row
 * (entry b * R + i; roots and nodes whose token is out of range are left untouched).
 * status [1] (DEVICE): EAGLE_STATUS_TIMEOUT is ORed in when a bounded wait inside the
 * kernel gives up (2 s); the outputs are then incomplete.  Allocates nothing.
 * Unsupported: rows > 128, h not a multiple of 64. */
int eagle_lmhead_stats(const eagle_lmhead_desc* d, const void* hidden, const void* weight,
                       const int32_t* tree_tokens, const int32_t* tree_parent, eagle_vocab_record* records,
                       float* child_logit, uint32_t* status, void* stream);

/* ---------------------------------------------------------------- KV commit */
typedef struct {
  int32_t layers;      /* L, 1..128 */
  int32_t batch;       /* B */
  int32_t n_kv_heads;  /* Hkv */
  int32_t head_dim;    /* D (any, with D * element size a multiple of 16 bytes) */
  int32_t rows;        /* R */
  int32_t max_seq;     /* P */
  int32_t max_depth;   /* path arrays hold max_depth + 1 entries */
  int32_t dtype;       /* K/V element type */
  int32_t feat_dim;    /* feature row width; 0 = no feature rows */
  int32_t feat_dtype;  /* feature element type */
} eagle_commit_desc;

/* For every layer l, request b, KV head h and m = 0..n_acc[b]: copy tree row
 * path[b][m] of tree_k/v_layers[l] to cache row seq_len[b] + m of
 * k/v_cache_layers[l]; copy feature row path[b][m] of tree_feat [B][R][F] to
 * feat_cache [B][P][F] row seq_len[b] + m; set commit_pos[b][m] = seq_len[b] + m
 * (-1 beyond n_acc); then seq_len[b] += n_acc[b] + 1.  A request whose commit
 * would pass max_seq is left untouched and flagged EAGLE_STATUS_CACHE_FULL.
 *   k_cache_layers, v_cache_layers, tree_k_layers, tree_v_layers: HOST arrays of
 *   `layers` DEVICE pointers; each cache [B][Hkv][P][D], each tree [B][Hkv][R][D].
 *   n_acc [B], path [B][max_depth+1] as written by eagle_accept; seq_len [B] in/out;
 *   commit_pos [B][max_depth+1]; feat_cache / tree_feat may be NULL (feat_dim 0).
 * Source and destination never overlap (tree K/V is its own buffer). */
int eagle_kv_commit(const eagle_commit_desc* d, void* const* k_cache_layers, void* const* v_cache_layers,
                    const void* const* tree_k_layers, const void* const* tree_v_layers,
                    const int32_t* n_acc, const int32_t* path, int32_t* seq_len, int32_t* commit_pos,
                    void* feat_cache, const void* tree_feat, uint32_t* status, void* stream);

/* ---------------------------------------------------------------- misc */
/* Scratch bytes a call needs (which = EAGLE_WS_*, desc = the matching desc); 0 on a
 * bad argument. */
size_t eagle_workspace_size(int which, const void* desc);

/* A static string naming a status code. */
const char* eagle_status_string(int status);

/* Library version string. */
const char* eagle_version(void);

/* Self-test of an internal routine (no counterpart in the method's description):
 * evaluates the float-float natural logarithm that eagle_tree_build uses for the
 * log-normaliser ln Z of a draft row, on n values z = z_hi[i] + z_lo[i] (DEVICE
 * arrays of n floats, z > 0, |z_lo| <= ulp(z_hi) / 2), writing ln z as
 * out_hi[i] + out_lo[i].  Asynchronous on `stream`.  EAGLE_ERR_INVALID_ARG for n < 0
 * or a NULL array. */
int eagle_selftest_ff_log(const float* z_hi, const float* z_lo, float* out_hi, float* out_lo, int32_t n,
                          void* stream);

/* The CUDA error behind the calling thread's most recent EAGLE_ERR_CUDA (a
 * cudaError_t value, 0 if none), and its name.  Thread-local, like cudaGetLastError. */
int eagle_last_cuda_error(void);
const char* eagle_last_cuda_error_string(void);

#ifdef __cplusplus
}
#endif
#endif /* EAGLE_H */
