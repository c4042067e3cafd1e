// accept.cu -- multi-round speculative sampling down the draft tree.
//
// The rule (EAGLE review, section 3.3 and appendix A.2 / Algorithm 1; lesson steps
// 1-2): at the current node, with p = softmax(target / T), try the children in row
// order; child d is accepted iff u < p(d) / q(d), else p <- norm(max(0, p - q)) and
// the next child is tried; when every child is rejected (or the node is a leaf)
// the emitted token is drawn from p (the bonus token when the whole path was
// accepted).  T = 0 is greedy: the child carrying the target argmax is accepted,
// else the argmax is emitted.  q is the candidate's proposal distribution: a point
// mass on d for deterministic (top-k) candidates, softmax(draft / T) for drawn
// ones.
//
// Kernels
//   accept_rowstats_kernel  one CTA per (4096-token chunk, tree row, source): chunk
//                           max, sum exp((x - m) / T) and argmax -- a single
//                           streaming pass over every target (and draft) row.
//   accept_walk_kernel      one CTA per request: merges the chunk statistics of the
//                           rows it visits, applies the rule, and draws the emitted
//                           token by inverse CDF.  Point-mass residuals only zero a
//                           few tokens, so the draw skips to the chunk that holds
//                           the crossing; drawn-proposal residuals take full passes.
#include <limits.h>

#include "common.cuh"
#include "launch.h"

namespace eagle {
namespace {

constexpr int kThreads = 256;
constexpr int kPer = kVocabChunk / kThreads;  // 16 elements per thread per tile

struct RowPart {
  float m;    // chunk max
  float s;    // sum exp2((x - m) * cT)
  float av;   // chunk argmax value
  int ai;     // chunk argmax index (lowest on ties)
};

struct WalkArgs {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const int32_t* parent;
  const float* u_accept;
  const float* u_final;
  eagle_accept_out out;
  const RowPart* part;  // [source][B*R][n_chunks]
};

__global__ void __launch_bounds__(kThreads) accept_rowstats_kernel(const AcceptPlan p, const void* target,
                                                                   const void* draft, RowPart* part) {
  const int c = blockIdx.x, row = blockIdx.y, src = blockIdx.z;
  const void* base = src == 0 ? target : draft;
  const size_t off = static_cast<size_t>(row) * p.V;
  const int lo = c * kVocabChunk, hi = min(p.V, lo + kVocabChunk);
  const float cT = kLog2e / (p.temperature > 0.f ? p.temperature : 1.f);
  float m = -INFINITY, s = 0.f, av = -INFINITY;
  int ai = INT_MAX;
  for (int v = lo + threadIdx.x; v < hi; v += kThreads) {
    const float x = load_elem(base, off + v, p.dtype);
    if (x > m) {
      if (m != -INFINITY) s *= exp2f((m - x) * cT);
      m = x;
    }
    s += exp2f((x - m) * cT);
    if (before(x, v, av, ai)) {
      av = x;
      ai = v;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float v2 = __shfl_xor_sync(0xffffffffu, av, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, ai, o);
    const float M = fmaxf(m, m2);
    if (M != -INFINITY) s = s * exp2f((m - M) * cT) + s2 * exp2f((m2 - M) * cT);
    m = M;
    if (before(v2, i2, av, ai)) {
      av = v2;
      ai = i2;
    }
  }
  __shared__ RowPart wp[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) wp[warp] = RowPart{m, s, av, ai};
  __syncthreads();
  if (threadIdx.x == 0) {
    RowPart r = wp[0];
    for (int w = 1; w < kThreads / 32; ++w) {
      const RowPart q = wp[w];
      const float M = fmaxf(r.m, q.m);
      if (M != -INFINITY) r.s = r.s * exp2f((r.m - M) * cT) + q.s * exp2f((q.m - M) * cT);
      r.m = M;
      if (before(q.av, q.ai, r.av, r.ai)) {
        r.av = q.av;
        r.ai = q.ai;
      }
    }
    part[(static_cast<size_t>(src) * gridDim.y + row) * gridDim.x + c] = r;
  }
}

// ------------------------------------------------------------------ block helpers
struct DrawScratch {
  float wsum[kThreads / 32];
  int found;
  int last;
  float prev_edge, next_edge, total;
};

// One tile of an inverse-CDF draw: elements [lo, hi) (hi - lo <= 4096), running sum
// `base` before lo.  Sets ds.found to the first index whose running sum exceeds
// `target` (INT_MAX if none), ds.last to the last index with positive weight
// (-1 if none) and ds.total to the tile's weight sum.
template <class WF>
__device__ void block_draw_tile(int lo, int hi, float base, float target, WF wf, DrawScratch& ds) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a0 = lo + threadIdx.x * kPer;
  float w[kPer];
  float mine = 0.f;
  int last = -1;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int v = a0 + e;
    w[e] = (v < hi) ? wf(v) : 0.f;
    mine += w[e];
    if (w[e] > 0.f) last = v;
  }
  float incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();  // earlier readers of ds are done
  if (threadIdx.x == 0) {
    ds.found = INT_MAX;
    ds.last = -1;
  }
  if (lane == 31) ds.wsum[warp] = incl;
  __syncthreads();
  float wbase = 0.f, tot = 0.f;
  for (int i = 0; i < kThreads / 32; ++i) {
    if (i < warp) wbase += ds.wsum[i];
    tot += ds.wsum[i];
  }
  float cum = base + wbase + incl - mine;
  int found = INT_MAX;
  float pe = 0.f, ne = 0.f;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const float nc = cum + w[e];
    if (found == INT_MAX && a0 + e < hi && nc > target) {
      found = a0 + e;
      pe = cum;
      ne = nc;
    }
    cum = nc;
  }
  if (found != INT_MAX) atomicMin(&ds.found, found);
  if (last >= 0) atomicMax(&ds.last, last);
  __syncthreads();
  if (found != INT_MAX && found == ds.found) {
    ds.prev_edge = pe;
    ds.next_edge = ne;
  }
  if (threadIdx.x == 0) ds.total = tot;
  __syncthreads();
}

// Block sum of wf(v) over [0, V).
template <class WF>
__device__ float block_sum(int V, WF wf, float* red) {
  float s = 0.f;
  for (int v = threadIdx.x; v < V; v += kThreads) s += wf(v);
  s = warp_sum(s);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = s;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < kThreads / 32; ++i) t += red[i];
  __syncthreads();
  return t;
}

__global__ void __launch_bounds__(kThreads) accept_walk_kernel(const AcceptPlan p, const WalkArgs a) {
  const int b = blockIdx.x;
  const int R = p.R, V = p.V, C = p.n_chunks;
  const bool greedy = !(p.temperature > 0.f);
  const bool sampled = !greedy && p.proposal == EAGLE_PROPOSAL_SAMPLED;
  const float cT = kLog2e / (greedy ? 1.f : p.temperature);
  const int32_t* tok = a.tokens + static_cast<size_t>(b) * R;
  const int32_t* par = a.parent + static_cast<size_t>(b) * R;
  const int maxp = p.max_depth + 1;

  __shared__ int s_path[kMaxRows + 1];
  __shared__ int s_kids[kMaxRows];
  __shared__ int s_nk, s_len, s_cur, s_next, s_emit, s_done, s_near;
  __shared__ unsigned s_status;
  __shared__ int s_rej[kMaxRows];
  __shared__ int s_nrej;
  __shared__ float s_Z[kMaxRows];
  __shared__ int s_nz;
  __shared__ float s_M, s_Zt, s_Mq, s_Zq, s_rejmass;
  __shared__ int s_amax;
  __shared__ float red[kThreads / 32];
  __shared__ DrawScratch ds;

  if (threadIdx.x == 0) {
    s_len = 1;
    s_path[0] = 0;
    s_cur = 0;
    s_done = 0;
    s_near = 0;
    s_status = 0;
    s_emit = -1;
  }
  __syncthreads();

  const size_t row_base = static_cast<size_t>(b) * R;
  for (int iter = 0; iter <= R && !s_done; ++iter) {
    const int cur = s_cur;
    const size_t xrow = (row_base + cur) * V;
    if (threadIdx.x == 0) {
      int nk = 0;
      for (int c = cur + 1; c < R; ++c) {
        const int pc = par[c];
        if (pc >= c || pc < -1 || (c > 0 && pc < 0)) s_status |= EAGLE_STATUS_BAD_TREE;
        if (pc == cur) s_kids[nk++] = c;
      }
      s_nk = nk;
      // merge the target row's chunk statistics
      const RowPart* rp = a.part + (row_base + cur) * C;
      float M = -INFINITY, av = -INFINITY;
      int ai = INT_MAX;
      for (int c = 0; c < C; ++c) {
        M = fmaxf(M, rp[c].m);
        if (before(rp[c].av, rp[c].ai, av, ai)) {
          av = rp[c].av;
          ai = rp[c].ai;
        }
      }
      float Z = 0.f;
      for (int c = 0; c < C; ++c)
        if (rp[c].m != -INFINITY) Z += rp[c].s * exp2f((rp[c].m - M) * cT);
      s_M = M;
      s_Zt = Z;
      s_amax = ai;
      if (sampled) {
        const RowPart* dp = a.part + (static_cast<size_t>(p.B) * R + row_base + cur) * C;
        float Mq = -INFINITY;
        for (int c = 0; c < C; ++c) Mq = fmaxf(Mq, dp[c].m);
        float Zq = 0.f;
        for (int c = 0; c < C; ++c)
          if (dp[c].m != -INFINITY) Zq += dp[c].s * exp2f((dp[c].m - Mq) * cT);
        s_Mq = Mq;
        s_Zq = Zq;
      }
      s_next = -1;
      s_nrej = 0;
      s_nz = 0;
      s_rejmass = 0.f;
    }
    __syncthreads();
    const float M = s_M, Zt = s_Zt;
    const float Mq = s_Mq, Zq = s_Zq;
    auto p_of = [&](int v) { return exp2f((load_elem(a.target, xrow + v, p.dtype) - M) * cT) / Zt; };
    auto q_of = [&](int v) { return exp2f((load_elem(a.draft, xrow + v, p.dtype) - Mq) * cT) / Zq; };
    // residual chain for drawn proposals: p_j = max(0, p_{j-1} - q) / Z_j
    auto pres_of = [&](int v, int nz) {
      float pv = p_of(v);
      if (nz == 0) return pv;
      const float qv = q_of(v);
      for (int i = 0; i < nz; ++i) pv = fmaxf(pv - qv, 0.f) / s_Z[i];
      return pv;
    };

    if (greedy) {
      if (threadIdx.x == 0) {
        const int am = s_amax;
        for (int i = 0; i < s_nk; ++i)
          if (tok[s_kids[i]] == am) {
            s_next = s_kids[i];
            break;
          }
        if (s_next < 0) {
          s_emit = am;
          s_done = 1;
        }
      }
      __syncthreads();
    } else if (!sampled) {
      // point-mass proposals: p_res(d) = p(d) / (1 - mass of the rejected tokens)
      if (threadIdx.x == 0) {
        for (int i = 0; i < s_nk; ++i) {
          const int c = s_kids[i];
          const int d = tok[c];
          if (d < 0 || d >= V) {
            s_status |= EAGLE_STATUS_BAD_TOKEN;
            continue;
          }
          bool dup = false;
          for (int r = 0; r < s_nrej; ++r) dup |= (s_rej[r] == d);
          const float pd = dup ? 0.f : p_of(d);
          const float denom = 1.f - s_rejmass;
          const float ratio = denom > 0.f ? pd / denom : 0.f;
          const float u = a.u_accept[row_base + c];
          if (fabsf(u - ratio) < kNearTieEps) s_near = 1;
          if (u < ratio) {
            s_next = c;
            break;
          }
          if (!dup) {
            s_rej[s_nrej++] = d;
            s_rejmass += pd;
          }
        }
      }
      __syncthreads();
    } else {
      // drawn proposals (SpecInfer multi-round): q fixed across siblings
      for (int i = 0; i < s_nk; ++i) {
        const int c = s_kids[i];
        const int nz = s_nz;
        if (threadIdx.x == 0) {
          const int d = tok[c];
          s_rej[0] = 0;  // flag: 1 = rejected, residual needed
          if (d < 0 || d >= V) {
            s_status |= EAGLE_STATUS_BAD_TOKEN;
          } else {
            const float qd = q_of(d);
            const float pd = pres_of(d, nz);
            const float ratio = qd > 0.f ? pd / qd : INFINITY;
            const float u = a.u_accept[row_base + c];
            if (qd > 0.f && fabsf(u - ratio) < kNearTieEps) s_near = 1;
            if (!(qd > 0.f) || u < ratio)
              s_next = c;
            else
              s_rej[0] = 1;
          }
        }
        __syncthreads();
        if (s_next >= 0) break;
        if (s_rej[0]) {
          const float z = block_sum(V, [&](int v) { return fmaxf(pres_of(v, nz) - q_of(v), 0.f); }, red);
          if (threadIdx.x == 0 && z > 0.f) s_Z[s_nz++] = z;
        }
        __syncthreads();
      }
    }

    if (s_next >= 0) {
      if (threadIdx.x == 0) {
        if (s_len >= maxp) {  // deeper than the path arrays: emit the accepted token and stop
          s_status |= EAGLE_STATUS_PATH_OVERFLOW;
          s_emit = tok[s_next];
          s_done = 1;
        } else {
          s_path[s_len++] = s_next;
          s_cur = s_next;
        }
      }
      __syncthreads();
      continue;
    }
    if (s_done) break;

    // ---- draw the emitted token from the (residual) target distribution
    const float u = a.u_final[b];
    if (sampled && s_nz > 0) {
      const int nz = s_nz;
      // full passes, tile by tile; W = the residual's sum, taken in the same pass order
      float W = 0.f;
      for (int lo = 0; lo < V; lo += kVocabChunk) {
        block_draw_tile(lo, min(V, lo + kVocabChunk), W, INFINITY, [&](int v) { return pres_of(v, nz); }, ds);
        W += ds.total;
      }
      const float target = u * W;
      float run = 0.f;
      int emit = -1, last = -1;
      for (int lo = 0; lo < V; lo += kVocabChunk) {
        block_draw_tile(lo, min(V, lo + kVocabChunk), run, target, [&](int v) { return pres_of(v, nz); }, ds);
        if (ds.last >= 0) last = ds.last;
        if (ds.found != INT_MAX) {
          emit = ds.found;
          if (threadIdx.x == 0 &&
              (target - ds.prev_edge < kNearTieEps * W || ds.next_edge - target < kNearTieEps * W))
            s_near = 1;
          break;
        }
        run += ds.total;
      }
      if (threadIdx.x == 0) {
        if (emit < 0) {
          emit = last < 0 ? 0 : last;
          s_near = 1;
        }
        s_emit = emit;
      }
    } else {
      // untouched p, or p with the rejected point-mass tokens zeroed: skip to the chunk
      const int nrej = s_nrej;
      auto w_of = [&](int v) {
        for (int r = 0; r < nrej; ++r)
          if (s_rej[r] == v) return 0.f;
        return exp2f((load_elem(a.target, xrow + v, p.dtype) - M) * cT);
      };
      __shared__ int s_chunk, s_fallback;
      __shared__ float s_base, s_W;
      if (threadIdx.x == 0) {
        const RowPart* rp = a.part + (row_base + cur) * C;
        float W = 0.f;
        for (int c = 0; c < C; ++c)
          if (rp[c].m != -INFINITY) W += rp[c].s * exp2f((rp[c].m - M) * cT);
        for (int r = 0; r < nrej; ++r) W -= exp2f((load_elem(a.target, xrow + s_rej[r], p.dtype) - M) * cT);
        const float target = u * W;
        float cum = 0.f;
        int cs = -1, lastc = -1;
        float bs = 0.f;
        for (int c = 0; c < C; ++c) {
          float wc = (rp[c].m == -INFINITY) ? 0.f : rp[c].s * exp2f((rp[c].m - M) * cT);
          for (int r = 0; r < nrej; ++r)
            if (s_rej[r] / kVocabChunk == c)
              wc -= exp2f((load_elem(a.target, xrow + s_rej[r], p.dtype) - M) * cT);
          if (wc > 0.f) lastc = c;
          if (cs < 0 && cum + wc > target) {
            cs = c;
            bs = cum;
          }
          cum += wc;
        }
        s_fallback = cs < 0;  // nothing crosses (rounding): take the last positive weight
        if (cs < 0) cs = lastc < 0 ? 0 : lastc;
        s_chunk = cs;
        s_base = bs;
        s_W = W;
      }
      __syncthreads();
      const int lo = s_chunk * kVocabChunk;
      const float W = s_W, target = s_fallback ? INFINITY : u * W;
      block_draw_tile(lo, min(V, lo + kVocabChunk), s_base, target, w_of, ds);
      if (threadIdx.x == 0) {
        int emit = ds.found;
        if (emit == INT_MAX) {
          emit = ds.last < 0 ? lo : ds.last;
          s_near = 1;
        } else if (target - ds.prev_edge < kNearTieEps * W || ds.next_edge - target < kNearTieEps * W) {
          s_near = 1;
        }
        s_emit = emit;
      }
    }
    __syncthreads();
    break;
  }

  // ---- outputs
  if (threadIdx.x == 0) {
    const int len = s_len;
    const int na = len - 1;
    int32_t* pb = a.out.path + static_cast<size_t>(b) * maxp;
    int32_t* ob = a.out.out_tok + static_cast<size_t>(b) * maxp;
    for (int j = 0; j < maxp; ++j) {
      pb[j] = j < len ? s_path[j] : -1;
      ob[j] = j < na ? tok[s_path[j + 1]] : (j == na ? s_emit : -1);
    }
    a.out.n_acc[b] = na;
    a.out.near_tie[b] = s_near;
    if (s_status) atomicOr(a.out.status, s_status);
  }
}

}  // namespace

void plan_accept(const eagle_accept_desc* d, AcceptPlan* p) {
  p->B = d->batch;
  p->R = d->rows;
  p->V = d->vocab;
  p->dtype = d->dtype;
  p->proposal = d->proposal;
  p->max_depth = d->max_depth;
  p->temperature = d->temperature;
  p->n_chunks = (d->vocab + kVocabChunk - 1) / kVocabChunk;
  p->n_sources = (d->temperature > 0.f && d->proposal == EAGLE_PROPOSAL_SAMPLED) ? 2 : 1;
  p->off_part = 0;
  p->total = static_cast<size_t>(p->n_sources) * p->B * p->R * p->n_chunks * sizeof(RowPart);
}

cudaError_t launch_accept(const AcceptPlan& p, const void* target, const void* draft, const int32_t* tokens,
                          const int32_t* parent, const float* u_accept, const float* u_final,
                          const eagle_accept_out& out, void* ws, cudaStream_t s) {
  RowPart* part = reinterpret_cast<RowPart*>(static_cast<uint8_t*>(ws) + p.off_part);
  dim3 grid(p.n_chunks, p.B * p.R, p.n_sources);
  accept_rowstats_kernel<<<grid, kThreads, 0, s>>>(p, target, draft, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  WalkArgs a;
  a.target = target;
  a.draft = draft;
  a.tokens = tokens;
  a.parent = parent;
  a.u_accept = u_accept;
  a.u_final = u_final;
  a.out = out;
  a.part = part;
  accept_walk_kernel<<<p.B, kThreads, 0, s>>>(p, a);
  return cudaGetLastError();
}

}  // namespace eagle
