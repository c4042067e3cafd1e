// tree_build.cu -- draft-tree construction, one draft level per call.
//
// Dynamic mode (EAGLE-2 dynamic draft tree; EAGLE-3 visual reading "EAGLE-2": the
// tree keeps the candidates the draft is most confident in, confidence tracking
// acceptance):
//   level 1: the root's top-k tokens join the pool with score ln q_root(t);
//   level d: each of the k frontier nodes adds its top-k tokens with score
//            s_parent + ln q(t); the next frontier is the best k of those k*k;
//   last level: the best N of the pool, ordered by pool index, form the tree.
// "Best" = (score desc, pool index asc); in-row ties go to the lower token id; q is
// the draft softmax at temperature 1.
// Static mode (EAGLE review appendix A.1): fixed shape; a node's children are its
// best tokens in rank order (greedy) or i.i.d. inverse-CDF draws from
// softmax(row / T) (non-greedy).
//
// Kernels
//   tree_chunk_kernel   one CTA per (request x frontier row, 4096-token chunk):
//                       chunk max, sum exp (T = 1 and T), and the chunk's top-16 by
//                       (logit desc, id asc) -- one streaming pass over the logits.
//   tree_select_kernel  one CTA per request: merges the chunk results per row,
//                       extends the pool, picks the frontier (bitonic sort in shared
//                       memory) and, at the last level, emits the tree arrays.
//
// Precision: chunk sums are compensated fp32, merged in double; cumulative scores
// are kept in double so that fp32 and fp64 selections agree unless two scores at a
// boundary are within 1e-5 (reported as a near-tie).
#include <limits.h>

#include "common.cuh"
#include "launch.h"

namespace eagle {
namespace {

constexpr int kThreads = 256;
constexpr int K = kMaxTopK;
constexpr double kIcdfNearEps = 1e-7;

struct ChunkPart {
  float m;        // chunk max logit
  float pad;
  double s1;      // sum exp(x - m)
  double sT;      // sum exp((x - m) / T)
  float tv[K];    // top-K logits of the chunk, best first
  int ti[K];      // their token ids (INT_MAX = empty)
};

struct BuildArgs {
  const void* logits;
  const float* u_draft;
  const int32_t* root_tok;
  const int32_t* seq_len;
  uint8_t* ws;
  eagle_tree out;
  int level, F;
};

__device__ __forceinline__ ChunkPart* parts(const TreeBuildPlan& p, uint8_t* ws) {
  return reinterpret_cast<ChunkPart*>(ws + p.off_part);
}

// ------------------------------------------------------------------ chunk pass
template <bool TOPK>
__global__ void __launch_bounds__(kThreads) tree_chunk_kernel(const TreeBuildPlan p, const BuildArgs a) {
  const int bf = blockIdx.x, c = blockIdx.y;
  const int b = bf / a.F, f = bf % a.F;
  const int lo = c * kVocabChunk;
  const int hi = min(p.V, lo + kVocabChunk);
  const size_t row = static_cast<size_t>(bf) * p.V;
  const float invT = 1.f / (p.temperature > 0.f ? p.temperature : 1.f);

  float m = -INFINITY;
  CSum s1, sT;
  float tv[K];
  int ti[K];
#pragma unroll
  for (int j = 0; j < K; ++j) {
    tv[j] = -INFINITY;
    ti[j] = INT_MAX;
  }
  for (int v = lo + threadIdx.x; v < hi; v += kThreads) {
    const float x = load_elem(a.logits, row + v, p.dtype);
    if (x > m) {
      if (m != -INFINITY) {
        s1.scale(expf(m - x));
        sT.scale(expf((m - x) * invT));
      }
      m = x;
    }
    s1.add(expf(x - m));
    sT.add(expf((x - m) * invT));
    if (TOPK && before(x, v, tv[K - 1], ti[K - 1])) {
      float cv = x;
      int ci = v;
#pragma unroll
      for (int j = 0; j < K; ++j) {
        const bool bt = before(cv, ci, tv[j], ti[j]);
        const float ov = tv[j];
        const int oi = ti[j];
        tv[j] = bt ? cv : ov;
        ti[j] = bt ? ci : oi;
        cv = bt ? ov : cv;
        ci = bt ? oi : ci;
      }
    }
  }
  // block reduction of (m, s1, sT): sums rescaled to the warp max, in double
  __shared__ float sm[kThreads / 32];
  __shared__ double ss1[kThreads / 32], ssT[kThreads / 32];
  __shared__ float wv[kThreads / 32];
  __shared__ int wi[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float M = warp_max(m);
  double d1 = (m == -INFINITY) ? 0.0 : s1.total() * static_cast<double>(expf(m - M));
  double dT = (m == -INFINITY) ? 0.0 : sT.total() * static_cast<double>(expf((m - M) * invT));
  d1 = warp_sum_d(d1);
  dT = warp_sum_d(dT);
  if (lane == 0) {
    sm[warp] = M;
    ss1[warp] = d1;
    ssT[warp] = dT;
  }
  __syncthreads();
  ChunkPart* out = parts(p, a.ws) + (static_cast<size_t>(b) * p.f_max + f) * p.n_chunks + c;
  if (threadIdx.x == 0) {
    float BM = -INFINITY;
    for (int w = 0; w < kThreads / 32; ++w) BM = fmaxf(BM, sm[w]);
    double t1 = 0.0, tT = 0.0;
    for (int w = 0; w < kThreads / 32; ++w) {
      if (sm[w] == -INFINITY) continue;
      t1 += ss1[w] * static_cast<double>(expf(sm[w] - BM));
      tT += ssT[w] * static_cast<double>(expf((sm[w] - BM) * invT));
    }
    out->m = BM;
    out->s1 = t1;
    out->sT = tT;
  }
  if constexpr (TOPK) {
    // block top-K: K rounds of block argmax over the threads' list heads
    for (int r = 0; r < K; ++r) {
      float bv = tv[0];
      int bi = ti[0];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
        if (before(v2, i2, bv, bi)) {
          bv = v2;
          bi = i2;
        }
      }
      __syncthreads();
      if (lane == 0) {
        wv[warp] = bv;
        wi[warp] = bi;
      }
      __syncthreads();
      bv = wv[0];
      bi = wi[0];
      for (int w = 1; w < kThreads / 32; ++w)
        if (before(wv[w], wi[w], bv, bi)) {
          bv = wv[w];
          bi = wi[w];
        }
      if (threadIdx.x == 0) {
        out->tv[r] = bv;
        out->ti[r] = bi;
      }
      if (bi != INT_MAX && ti[0] == bi) {  // the owner pops its head
#pragma unroll
        for (int j = 0; j < K - 1; ++j) {
          tv[j] = tv[j + 1];
          ti[j] = ti[j + 1];
        }
        tv[K - 1] = -INFINITY;
        ti[K - 1] = INT_MAX;
      }
    }
  }
}

// ------------------------------------------------------------------ select helpers
// Block bitonic sort of n2 (power of two) entries, best first by (key desc, idx asc).
__device__ void bitonic_sort(double* key, int* idx, int n2) {
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const bool up = (i & k) == 0;
          const bool sw = up ? before(key[ixj], idx[ixj], key[i], idx[i]) : before(key[i], idx[i], key[ixj], idx[ixj]);
          if (sw) {
            const double tk = key[i];
            key[i] = key[ixj];
            key[ixj] = tk;
            const int t = idx[i];
            idx[i] = idx[ixj];
            idx[ixj] = t;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Row statistics merged over chunks by one warp: M, ln Z (T = 1) and the mass at
// temperature T (for draws), in double.
struct RowStats {
  float M;
  double lnZ1, WT;
};

__device__ RowStats row_stats(const ChunkPart* cp, int n_chunks, float invT) {
  float M = -INFINITY;
  for (int c = threadIdx.x & 31; c < n_chunks; c += 32) M = fmaxf(M, cp[c].m);
  M = warp_max(M);
  double z1 = 0.0, zT = 0.0;
  for (int c = threadIdx.x & 31; c < n_chunks; c += 32) {
    if (cp[c].m == -INFINITY) continue;
    z1 += cp[c].s1 * static_cast<double>(expf(cp[c].m - M));
    zT += cp[c].sT * static_cast<double>(expf((cp[c].m - M) * invT));
  }
  RowStats r;
  r.M = M;
  r.lnZ1 = log(warp_sum_d(z1));
  r.WT = warp_sum_d(zT);
  return r;
}

// Warp merge of the chunks' top-K lists: writes the best `cnt` (token ids) to tok[].
__device__ void merge_topk(const ChunkPart* cp, int n_chunks, int cnt, int* tok, float* val) {
  const int lane = threadIdx.x & 31;
  int head[4] = {0, 0, 0, 0};  // per owned chunk (lane, lane+32, ...)
  for (int r = 0; r < cnt; ++r) {
    float bv = -INFINITY;
    int bi = INT_MAX, bslot = -1;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int c = lane + 32 * s;
      if (c < n_chunks && head[s] < K) {
        const float v = cp[c].tv[head[s]];
        const int i = cp[c].ti[head[s]];
        if (before(v, i, bv, bi)) {
          bv = v;
          bi = i;
          bslot = s;
        }
      }
    }
    float wv2 = bv;
    int wi2 = bi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, wv2, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, wi2, o);
      if (before(v2, i2, wv2, wi2)) {
        wv2 = v2;
        wi2 = i2;
      }
    }
    if (bslot >= 0 && bi == wi2 && bi != INT_MAX) head[bslot] += 1;
    if (lane == 0) {
      tok[r] = wi2;
      val[r] = wv2;
    }
  }
  __syncwarp();
}

// Warp inverse-CDF draw over one logit row with weights exp((x - M) / T): the chunk
// masses pick the chunk that holds the crossing, then the lanes scan that chunk
// (lane offsets in double, local running sums in fp32).  Returns the token; *near =
// 1 when the draw lands within 1e-7 of the mass of a bin edge.
__device__ int warp_draw(const void* logits, size_t row, int dtype, int V, const ChunkPart* cp, int n_chunks, float M,
                         float invT, double W, float u, int* near) {
  const int lane = threadIdx.x & 31;
  const double target = static_cast<double>(u) * W;
  int cstar = -1, fallback = 0;
  double base = 0.0;
  if (lane == 0) {
    double cum = 0.0;
    int last_pos = -1;
    for (int c = 0; c < n_chunks; ++c) {
      const double w = (cp[c].m == -INFINITY) ? 0.0 : cp[c].sT * static_cast<double>(expf((cp[c].m - M) * invT));
      if (w > 0.0) last_pos = c;
      if (cum + w > target) {
        cstar = c;
        base = cum;
        break;
      }
      cum += w;
    }
    if (cstar < 0) {  // nothing crosses (rounding): the last positive weight
      cstar = last_pos < 0 ? 0 : last_pos;
      fallback = 1;
    }
  }
  cstar = __shfl_sync(0xffffffffu, cstar, 0);
  fallback = __shfl_sync(0xffffffffu, fallback, 0);
  base = __shfl_sync(0xffffffffu, base, 0);
  const int lo = cstar * kVocabChunk, hi = min(V, lo + kVocabChunk);
  const int n = hi - lo;
  const int seg = (n + 31) / 32;
  const int a0 = lo + lane * seg, a1 = min(hi, a0 + seg);
  double my = 0.0;
  for (int v = a0; v < a1; ++v) my += static_cast<double>(expf((load_elem(logits, row + v, dtype) - M) * invT));
  double incl = my;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const double lbase = base + incl - my;
  const double rel = fallback ? INFINITY : target - lbase;
  double cum = 0.0;
  int found = -1;
  double prev_edge = 0.0, next_edge = 0.0;
  int last_pos = -1;
  for (int v = a0; v < a1; ++v) {
    const float w = expf((load_elem(logits, row + v, dtype) - M) * invT);
    if (w > 0.f) last_pos = v;
    const double nc = cum + static_cast<double>(w);
    if (found < 0 && w > 0.f && nc > rel) {
      found = v;
      prev_edge = lbase + cum;
      next_edge = lbase + nc;
    }
    cum = nc;
  }
  const unsigned ball = __ballot_sync(0xffffffffu, found >= 0);
  int tok;
  int nr = 0;
  if (ball) {
    const int src = __ffs(ball) - 1;
    tok = __shfl_sync(0xffffffffu, found, src);
    const double pe = __shfl_sync(0xffffffffu, prev_edge, src);
    const double ne = __shfl_sync(0xffffffffu, next_edge, src);
    nr = (target - pe < kIcdfNearEps * W || ne - target < kIcdfNearEps * W) ? 1 : 0;
  } else {
    const unsigned bl = __ballot_sync(0xffffffffu, last_pos >= 0);
    const int src = bl ? 31 - __clz(bl) : 0;
    tok = __shfl_sync(0xffffffffu, last_pos, src);
    if (tok < 0) tok = lo;
    nr = 1;
  }
  *near = nr;
  return tok;
}

__global__ void __launch_bounds__(kThreads) tree_select_kernel(const TreeBuildPlan p, const BuildArgs a) {
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int NW = kThreads / 32;
  uint8_t* ws = a.ws;
  int32_t* state = reinterpret_cast<int32_t*>(ws + p.off_state) + b * 4;  // [0] n_pool, [1] near
  const ChunkPart* cps = parts(p, ws) + static_cast<size_t>(b) * p.f_max * p.n_chunks;
  const float invT = 1.f / (p.temperature > 0.f ? p.temperature : 1.f);

  __shared__ double skey[kMaxPool];
  __shared__ int sidx[kMaxPool];
  __shared__ int srow[kMaxPool];
  __shared__ int stok[NW][K];
  __shared__ float sval[NW][K];
  __shared__ int s_near;
  __shared__ uint64_t smask[kMaxRows][2];
  __shared__ int spar[kMaxRows];

  if (threadIdx.x == 0) {
    if (a.level == 1) {
      state[0] = 0;
      state[1] = 0;
    }
    s_near = 0;
  }
  __syncthreads();

  if (p.mode == EAGLE_TREE_DYNAMIC) {
    int32_t* ptok = reinterpret_cast<int32_t*>(ws + p.off_pool_tok) + static_cast<size_t>(b) * p.pool_cap;
    int32_t* ppar = reinterpret_cast<int32_t*>(ws + p.off_pool_par) + static_cast<size_t>(b) * p.pool_cap;
    double* psc = reinterpret_cast<double*>(ws + p.off_pool_score) + static_cast<size_t>(b) * p.pool_cap;
    int32_t* pdep = reinterpret_cast<int32_t*>(ws + p.off_pool_depth) + static_cast<size_t>(b) * p.pool_cap;
    int32_t* front = reinterpret_cast<int32_t*>(ws + p.off_front) + static_cast<size_t>(b) * K;
    const int base = state[0];
    const int k = p.k;
    // extend the pool: one warp per frontier row
    for (int f = warp; f < a.F; f += NW) {
      const ChunkPart* cp = cps + static_cast<size_t>(f) * p.n_chunks;
      const RowStats rs = row_stats(cp, p.n_chunks, invT);
      merge_topk(cp, p.n_chunks, k, stok[warp], sval[warp]);
      const int pidx = (a.level == 1) ? -1 : front[f];
      const double spar_score = (pidx < 0) ? 0.0 : psc[pidx];
      if (lane < k) {
        const int i = base + f * k + lane;
        ptok[i] = stok[warp][lane];
        ppar[i] = pidx;
        psc[i] = spar_score + (static_cast<double>(sval[warp][lane] - rs.M) - rs.lnZ1);
        pdep[i] = a.level;
      }
      __syncwarp();
    }
    __syncthreads();
    const int n_new = a.F * k;
    // next frontier: best k of the new candidates, kept in pool order
    int n2 = 1;
    while (n2 < n_new) n2 <<= 1;
    for (int j = threadIdx.x; j < n2; j += kThreads) {
      skey[j] = j < n_new ? psc[base + j] : -INFINITY;
      sidx[j] = j < n_new ? base + j : INT_MAX;
    }
    __syncthreads();
    bitonic_sort(skey, sidx, n2);
    // a near-tie at the boundary, unless it is an exact tie between siblings (same
    // parent, same logit), which both fp32 and fp64 break by pool index
    if (threadIdx.x == 0 && n_new > k && skey[k - 1] - skey[k] < kNearTieEps &&
        !(skey[k - 1] == skey[k] && ppar[sidx[k - 1]] == ppar[sidx[k]]))
      s_near += 1;
    for (int j = threadIdx.x; j < n_new; j += kThreads) srow[j] = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < k; j += kThreads) srow[sidx[j] - base] = 1;
    __syncthreads();
    if (threadIdx.x == 0) {
      int slot = 0;
      for (int j = 0; j < n_new; ++j) {
        if (!srow[j]) continue;
        front[slot] = base + j;
        a.out.frontier_tok[static_cast<size_t>(b) * p.f_max + slot] = ptok[base + j];
        a.out.frontier_slot[static_cast<size_t>(b) * p.f_max + slot] = j / k;
        ++slot;
      }
      state[0] = base + n_new;
      state[1] += s_near;
      s_near = 0;
    }
    __syncthreads();
    if (a.level != p.depth) return;

    // ---- last level: best N of the pool, rows in pool order
    const int np = state[0];
    const int N = p.N;
    n2 = 1;
    while (n2 < np) n2 <<= 1;
    for (int j = threadIdx.x; j < n2; j += kThreads) {
      skey[j] = j < np ? psc[j] : -INFINITY;
      sidx[j] = j < np ? j : INT_MAX;
    }
    __syncthreads();
    bitonic_sort(skey, sidx, n2);
    if (threadIdx.x == 0 && np > N && skey[N - 1] - skey[N] < kNearTieEps &&
        !(skey[N - 1] == skey[N] && ppar[sidx[N - 1]] == ppar[sidx[N]]))
      state[1] += 1;
    for (int j = threadIdx.x; j < np; j += kThreads) srow[j] = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < N; j += kThreads) srow[sidx[j]] = 1;
    __syncthreads();
    if (threadIdx.x == 0) {  // rows in pool order (one pass over the pool)
      int r = 1;
      for (int j = 0; j < np; ++j) srow[j] = srow[j] ? r++ : -1;
    }
    __syncthreads();
    const size_t ob = static_cast<size_t>(b) * p.R;
    const int L = a.seq_len[b];
    for (int j = threadIdx.x; j < np; j += kThreads) {
      const int r = srow[j];
      if (r < 0) continue;
      const int pp = ppar[j];
      const int pr = (pp < 0) ? 0 : (srow[pp] > 0 ? srow[pp] : 0);
      spar[r] = pr;
      a.out.tokens[ob + r] = ptok[j];
      a.out.parent[ob + r] = pr;
      a.out.depth[ob + r] = pdep[j];
      a.out.pos_id[ob + r] = L + pdep[j];
      a.out.score[ob + r] = static_cast<float>(psc[j]);
    }
    if (threadIdx.x == 0) {
      spar[0] = -1;
      a.out.tokens[ob] = a.root_tok[b];
      a.out.parent[ob] = -1;
      a.out.depth[ob] = 0;
      a.out.pos_id[ob] = L;
      a.out.score[ob] = 0.f;
    }
    __syncthreads();
  } else {
    // ---- static shape
    int32_t* ntok = reinterpret_cast<int32_t*>(ws + p.off_node_tok) + static_cast<size_t>(b) * p.R;
    double* nsc = reinterpret_cast<double*>(ws + p.off_node_score) + static_cast<size_t>(b) * p.R;
    const bool sampled = p.mode == EAGLE_TREE_STATIC_SAMPLED;
    if (a.level == 1 && threadIdx.x == 0) {
      ntok[0] = a.root_tok[b];
      nsc[0] = 0.0;
    }
    __syncthreads();
    // frontier row f = the f-th node of depth level-1; one warp per row
    int near_local = 0;
    for (int f = warp; f < a.F; f += NW) {
      int n = -1, cnt = -1;
      for (int i = 0; i < p.R; ++i)
        if (p.shape.depth[i] == a.level - 1 && ++cnt == f) {
          n = i;
          break;
        }
      if (n < 0) continue;
      int kids = 0;
      for (int i = n + 1; i < p.R; ++i) kids += (p.shape.parent[i] == n);
      if (kids == 0) continue;
      const ChunkPart* cp = cps + static_cast<size_t>(f) * p.n_chunks;
      const RowStats rs = row_stats(cp, p.n_chunks, invT);
      const size_t row = (static_cast<size_t>(b) * a.F + f) * p.V;
      if (!sampled) merge_topk(cp, p.n_chunks, kids, stok[warp], sval[warp]);
      int j = 0;
      for (int ch = n + 1; ch < p.R; ++ch) {
        if (p.shape.parent[ch] != n) continue;
        int tok;
        if (!sampled) {
          tok = stok[warp][j];
        } else {
          int nr = 0;
          tok = warp_draw(a.logits, row, p.dtype, p.V, cp, p.n_chunks, rs.M, invT, rs.WT,
                          a.u_draft[static_cast<size_t>(b) * p.R + ch], &nr);
          near_local += nr;
        }
        if (lane == 0) {
          ntok[ch] = tok;
          nsc[ch] = nsc[n] + (static_cast<double>(load_elem(a.logits, row + tok, p.dtype) - rs.M) - rs.lnZ1);
        }
        ++j;
      }
      __syncwarp();
    }
    if (lane == 0 && near_local) atomicAdd(&s_near, near_local);
    __syncthreads();
    if (threadIdx.x == 0) {
      state[1] += s_near;
      // next frontier: the nodes of depth `level`, with their parent's row in this level's input
      int slot = 0;
      for (int i = 0; i < p.R; ++i) {
        if (p.shape.depth[i] != a.level) continue;
        const int par = p.shape.parent[i];
        int prow = 0;
        for (int q = 0; q < par; ++q) prow += (p.shape.depth[q] == a.level - 1);
        a.out.frontier_tok[static_cast<size_t>(b) * p.f_max + slot] = ntok[i];
        a.out.frontier_slot[static_cast<size_t>(b) * p.f_max + slot] = prow;
        ++slot;
      }
    }
    __syncthreads();
    if (a.level != p.depth) return;
    const size_t ob = static_cast<size_t>(b) * p.R;
    const int L = a.seq_len[b];
    for (int i = threadIdx.x; i < p.R; i += kThreads) {
      spar[i] = p.shape.parent[i];
      a.out.tokens[ob + i] = (i == 0) ? a.root_tok[b] : ntok[i];
      a.out.parent[ob + i] = p.shape.parent[i];
      a.out.depth[ob + i] = p.shape.depth[i];
      a.out.pos_id[ob + i] = L + p.shape.depth[i];
      a.out.score[ob + i] = static_cast<float>(nsc[i]);
    }
    __syncthreads();
  }
  // ancestor masks: row i = row parent(i) | bit i (parents come first)
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.R; ++i) {
      uint64_t w0 = 0, w1 = 0;
      if (i > 0) {
        w0 = smask[spar[i]][0];
        w1 = smask[spar[i]][1];
      }
      if (i < 64)
        w0 |= 1ull << i;
      else
        w1 |= 1ull << (i - 64);
      smask[i][0] = w0;
      smask[i][1] = w1;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < p.R; i += kThreads) {
    a.out.anc_mask[(static_cast<size_t>(b) * p.R + i) * p.W] = smask[i][0];
    if (p.W > 1) a.out.anc_mask[(static_cast<size_t>(b) * p.R + i) * p.W + 1] = smask[i][1];
  }
  if (threadIdx.x == 0) a.out.near_tie[b] = state[1];
}

}  // namespace

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

void plan_tree_build(const eagle_tree_desc* d, TreeBuildPlan* p) {
  p->B = d->batch;
  p->V = d->vocab;
  p->mode = d->mode;
  p->dtype = d->dtype;
  p->temperature = d->temperature;
  p->n_chunks = (d->vocab + kVocabChunk - 1) / kVocabChunk;
  if (d->mode == EAGLE_TREE_DYNAMIC) {
    p->depth = d->depth;
    p->k = d->top_k;
    p->N = d->total_tokens;
    p->R = d->total_tokens + 1;
    p->f_max = d->top_k;
    p->pool_cap = d->top_k + (d->depth - 1) * d->top_k * d->top_k;
    p->shape.rows = 0;
  } else {
    p->R = d->n_static + 1;
    p->N = d->n_static;
    p->k = 0;
    p->pool_cap = 0;
    p->shape.rows = p->R;
    int maxd = 0;
    for (int i = 0; i < p->R && i < kMaxRows; ++i) {
      const int par = (i == 0) ? -1 : d->static_parent[i];
      p->shape.parent[i] = static_cast<int8_t>(par);
      p->shape.depth[i] = static_cast<int8_t>(i == 0 ? 0 : p->shape.depth[par] + 1);
      if (p->shape.depth[i] > maxd) maxd = p->shape.depth[i];
    }
    p->depth = maxd;
    int fmax = 1;
    for (int dd = 0; dd <= maxd; ++dd) {
      int c = 0;
      for (int i = 0; i < p->R; ++i) c += (p->shape.depth[i] == dd);
      if (c > fmax) fmax = c;
    }
    p->f_max = fmax;
  }
  p->W = (p->R + 63) / 64;
  size_t off = 0;
  const size_t cap = static_cast<size_t>(p->B) * (p->pool_cap > 0 ? p->pool_cap : 1);
  p->off_pool_tok = off;
  off = align256(off + cap * 4);
  p->off_pool_par = off;
  off = align256(off + cap * 4);
  p->off_pool_score = off;
  off = align256(off + cap * 8);
  p->off_pool_depth = off;
  off = align256(off + cap * 4);
  p->off_state = off;
  off = align256(off + static_cast<size_t>(p->B) * 4 * 4);
  p->off_front = off;
  off = align256(off + static_cast<size_t>(p->B) * K * 4);
  p->off_part = off;
  off = align256(off + static_cast<size_t>(p->B) * p->f_max * p->n_chunks * sizeof(ChunkPart));
  p->off_node_tok = off;
  off = align256(off + static_cast<size_t>(p->B) * p->R * 4);
  p->off_node_score = off;
  off = align256(off + static_cast<size_t>(p->B) * p->R * 8);
  p->total = off;
}

int frontier_rows(const TreeBuildPlan& p, int level) {
  if (level < 1 || level > p.depth) return -1;
  if (p.mode == EAGLE_TREE_DYNAMIC) return level == 1 ? 1 : p.k;
  int c = 0;
  for (int i = 0; i < p.R; ++i) c += (p.shape.depth[i] == level - 1);
  return c;
}

cudaError_t launch_tree_build(const TreeBuildPlan& p, int level, const void* logits, const float* u_draft,
                              const int32_t* root_tok, const int32_t* seq_len, void* ws, const eagle_tree& out,
                              cudaStream_t s) {
  BuildArgs a;
  a.logits = logits;
  a.u_draft = u_draft;
  a.root_tok = root_tok;
  a.seq_len = seq_len;
  a.ws = static_cast<uint8_t*>(ws);
  a.out = out;
  a.level = level;
  a.F = frontier_rows(p, level);
  dim3 grid(p.B * a.F, p.n_chunks);
  if (p.mode == EAGLE_TREE_STATIC_SAMPLED)
    tree_chunk_kernel<false><<<grid, kThreads, 0, s>>>(p, a);
  else
    tree_chunk_kernel<true><<<grid, kThreads, 0, s>>>(p, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  tree_select_kernel<<<p.B, kThreads, 0, s>>>(p, a);
  return cudaGetLastError();
}

}  // namespace eagle
