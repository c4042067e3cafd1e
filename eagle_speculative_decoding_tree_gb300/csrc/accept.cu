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
//   accept_rowstats_kernel  one CTA per (tree row, 4096-token chunk, source): chunk
//                           max, sum exp((x - m) / T) and argmax -- a single
//                           streaming pass over every target (and draft) row.
//   accept_walk_kernel      one CTA per request: merges the chunk statistics of the
//                           rows it visits, applies the rule, and draws the emitted
//                           token by inverse CDF.  Point-mass residuals only zero a
//                           few tokens, so the draw skips to the chunk that holds
//                           the crossing; drawn-proposal residuals take full passes.
//
// Precision: weights are expf((x - m) / T) in fp32; per-thread sums are compensated
// (Neumaier) and every sum across threads, chunks or tiles is taken in double, so a
// running sum is within about 2e-7 of the total mass of its exact value.  Draws are
// reported as near-ties when they land within 1e-7 of the mass of a bin edge.
#include <limits.h>

#include "common.cuh"
#include "launch.h"

namespace eagle {
namespace {

constexpr int kThreads = 256;
constexpr int kPer = kVocabChunk / kThreads;  // 16 elements per thread per tile
constexpr double kIcdfNearEps = 1e-7;

struct RowPart {
  float m;    // chunk max
  float av;   // chunk argmax value
  int ai;     // chunk argmax index (lowest on ties)
  int pad;
  double s;   // sum exp((x - m) / T)
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
  const int row = blockIdx.x, c = blockIdx.y, src = blockIdx.z;
  const int rows = gridDim.x, n_chunks = gridDim.y;
  const void* base = src == 0 ? target : draft;
  const size_t off = static_cast<size_t>(row) * p.V;
  const int lo = c * kVocabChunk, hi = min(p.V, lo + kVocabChunk);
  const float invT = 1.f / (p.temperature > 0.f ? p.temperature : 1.f);
  float m = -INFINITY, av = -INFINITY;
  int ai = INT_MAX;
  CSum acc;
  for (int v = lo + threadIdx.x; v < hi; v += kThreads) {
    const float x = load_elem(base, off + v, p.dtype);
    if (x > m) {
      if (m != -INFINITY) acc.scale(expf((m - x) * invT));
      m = x;
    }
    acc.add(expf((x - m) * invT));
    if (before(x, v, av, ai)) {
      av = x;
      ai = v;
    }
  }
  // warp max / argmax, then the sums rescaled to the warp max, in double
  double s = acc.total();
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float v2 = __shfl_xor_sync(0xffffffffu, av, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, ai, o);
    if (before(v2, i2, av, ai)) {
      av = v2;
      ai = i2;
    }
  }
  s = (m == -INFINITY) ? 0.0 : s * static_cast<double>(expf((m - M) * invT));
  s = warp_sum_d(s);
  __shared__ RowPart wp[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) wp[warp] = RowPart{M, av, ai, 0, s};
  __syncthreads();
  if (threadIdx.x == 0) {
    RowPart r = wp[0];
    for (int w = 1; w < kThreads / 32; ++w) r.m = fmaxf(r.m, wp[w].m);
    double t = 0.0;
    for (int w = 0; w < kThreads / 32; ++w) {
      if (wp[w].m != -INFINITY) t += wp[w].s * static_cast<double>(expf((wp[w].m - r.m) * invT));
      if (w > 0 && before(wp[w].av, wp[w].ai, r.av, r.ai)) {
        r.av = wp[w].av;
        r.ai = wp[w].ai;
      }
    }
    r.s = t;
    part[(static_cast<size_t>(src) * rows + row) * n_chunks + c] = r;
  }
}

// ------------------------------------------------------------------ block helpers
struct DrawScratch {
  double wsum[kThreads / 32];
  int found;
  int last;
  double prev_edge, next_edge, total;
};

// One tile of an inverse-CDF draw: elements [lo, hi) (hi - lo <= 4096), running mass
// `base` before lo.  Each thread takes 16 consecutive elements; its running sum and
// the thread offsets are taken in double.  Sets ds.found to the first index whose running mass
// exceeds `target` (INT_MAX if none), ds.last to the last index with positive
// weight (-1 if none) and ds.total to the tile's mass.
template <class WF>
__device__ void block_draw_tile(int lo, int hi, double base, double target, WF wf, DrawScratch& ds) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a0 = lo + threadIdx.x * kPer;
  float w[kPer];
  double my = 0.0;
  int last = -1;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int v = a0 + e;
    w[e] = (v < hi) ? wf(v) : 0.f;
    my += static_cast<double>(w[e]);
    if (w[e] > 0.f) last = v;
  }
  double incl = my;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();  // earlier readers of ds are done
  if (threadIdx.x == 0) {
    ds.found = INT_MAX;
    ds.last = -1;
  }
  if (lane == 31) ds.wsum[warp] = incl;
  __syncthreads();
  double wbase = 0.0, tot = 0.0;
  for (int i = 0; i < kThreads / 32; ++i) {
    if (i < warp) wbase += ds.wsum[i];
    tot += ds.wsum[i];
  }
  const double tbase = base + wbase + incl - my;  // mass before this thread's first element
  const double rel = target - tbase;
  int found = INT_MAX;
  double pe = 0.0, ne = 0.0;
  {
    double cum = 0.0;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const double nc = cum + static_cast<double>(w[e]);
      if (found == INT_MAX && a0 + e < hi && w[e] > 0.f && nc > rel) {
        found = a0 + e;
        pe = tbase + cum;
        ne = tbase + nc;
      }
      cum = nc;
    }
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

// Block sum of wf(v) over [lo, hi): compensated per thread, double across threads.
template <class WF>
__device__ double block_sum(int lo, int hi, WF wf, double* red) {
  CSum acc;
  for (int v = lo + threadIdx.x; v < hi; v += kThreads) acc.add(wf(v));
  double s = warp_sum_d(acc.total());
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = s;
  __syncthreads();
  double t = 0.0;
  for (int i = 0; i < kThreads / 32; ++i) t += red[i];
  __syncthreads();
  return t;
}

__global__ void __launch_bounds__(kThreads) accept_walk_kernel(const AcceptPlan p, const WalkArgs a) {
  const int b = blockIdx.x;
  const int R = p.R, V = p.V, C = p.n_chunks;
  const bool greedy = !(p.temperature > 0.f);
  const bool sampled = !greedy && p.proposal == EAGLE_PROPOSAL_SAMPLED;
  const float invT = 1.f / (greedy ? 1.f : p.temperature);
  const int32_t* tok = a.tokens + static_cast<size_t>(b) * R;
  const int32_t* par = a.parent + static_cast<size_t>(b) * R;
  const int maxp = p.max_depth + 1;

  __shared__ int s_path[kMaxRows + 1];
  __shared__ int s_kids[kMaxRows];
  __shared__ int s_nk, s_len, s_cur, s_next, s_emit, s_done, s_near, s_flag;
  __shared__ unsigned s_status;
  __shared__ int s_rej[kMaxRows];
  __shared__ int s_nrej;
  __shared__ double s_Z[kMaxRows];
  __shared__ int s_nz;
  __shared__ float s_M, s_Mq;
  __shared__ double s_Zt, s_Zq, s_rejmass;
  __shared__ int s_amax;
  __shared__ double red[kThreads / 32];
  __shared__ DrawScratch ds;
  __shared__ int s_chunk, s_fallback;
  __shared__ double s_base, s_W;
  __shared__ double s_tile[kMaxVocabTiles];

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
        if (pc >= c || pc < 0) s_status |= EAGLE_STATUS_BAD_TREE;
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
      double Z = 0.0;
      for (int c = 0; c < C; ++c)
        if (rp[c].m != -INFINITY) Z += rp[c].s * static_cast<double>(expf((rp[c].m - M) * invT));
      s_M = M;
      s_Zt = Z;
      s_amax = ai;
      if (sampled) {
        const RowPart* dp = a.part + (static_cast<size_t>(p.B) * R + row_base + cur) * C;
        float Mq = -INFINITY;
        for (int c = 0; c < C; ++c) Mq = fmaxf(Mq, dp[c].m);
        double Zq = 0.0;
        for (int c = 0; c < C; ++c)
          if (dp[c].m != -INFINITY) Zq += dp[c].s * static_cast<double>(expf((dp[c].m - Mq) * invT));
        s_Mq = Mq;
        s_Zq = Zq;
      }
      s_next = -1;
      s_nrej = 0;
      s_nz = 0;
      s_rejmass = 0.0;
    }
    __syncthreads();
    const float M = s_M, Mq = s_Mq;
    const float invZt = static_cast<float>(1.0 / s_Zt);
    const float invZq = sampled ? static_cast<float>(1.0 / s_Zq) : 0.f;
    auto w_target = [&](int v) { return expf((load_elem(a.target, xrow + v, p.dtype) - M) * invT); };
    auto p_of = [&](int v) { return w_target(v) * invZt; };
    auto q_of = [&](int v) { return expf((load_elem(a.draft, xrow + v, p.dtype) - Mq) * invT) * invZq; };
    // residual chain for drawn proposals: p_j = max(0, p_{j-1} - q) / Z_j
    auto pres_of = [&](int v, int nz) {
      float pv = p_of(v);
      if (nz == 0) return pv;
      const float qv = q_of(v);
      for (int i = 0; i < nz; ++i) pv = static_cast<float>(fmaxf(pv - qv, 0.f) / s_Z[i]);
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
          const double pd = dup ? 0.0 : static_cast<double>(w_target(d)) / s_Zt;
          const double denom = 1.0 - s_rejmass;
          const double ratio = denom > 0.0 ? pd / denom : 0.0;
          const double u = a.u_accept[row_base + c];
          if (fabs(u - ratio) < static_cast<double>(kNearTieEps)) s_near = 1;
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
          s_flag = 0;  // 1: rejected, residual needed
          if (d < 0 || d >= V) {
            s_status |= EAGLE_STATUS_BAD_TOKEN;
          } else {
            const double qd = q_of(d);
            const double pd = pres_of(d, nz);
            const double ratio = qd > 0.0 ? pd / qd : INFINITY;
            const double u = a.u_accept[row_base + c];
            if (qd > 0.0 && fabs(u - ratio) < static_cast<double>(kNearTieEps)) s_near = 1;
            if (!(qd > 0.0) || u < ratio)
              s_next = c;
            else
              s_flag = 1;
          }
        }
        __syncthreads();
        if (s_next >= 0) break;
        if (s_flag) {
          const double z = block_sum(0, V, [&](int v) { return fmaxf(pres_of(v, nz) - q_of(v), 0.f); }, red);
          if (threadIdx.x == 0 && z > 0.0) s_Z[s_nz++] = z;
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
    const double u = a.u_final[b];
    if (sampled && s_nz > 0) {
      // residual of drawn proposals: a mass per 4096-token tile, then the crossing
      // tile is scanned element by element
      const int nz = s_nz;
      auto wres = [&](int v) { return pres_of(v, nz); };
      const int n_tiles = (V + kVocabChunk - 1) / kVocabChunk;
      for (int t = 0; t < n_tiles; ++t) {
        const double m = block_sum(t * kVocabChunk, min(V, (t + 1) * kVocabChunk), wres, red);
        if (threadIdx.x == 0) s_tile[t] = m;
      }
      if (threadIdx.x == 0) {
        double W = 0.0;
        for (int t = 0; t < n_tiles; ++t) W += s_tile[t];
        const double target = u * W;
        double cum = 0.0, bs = 0.0;
        int ts = -1, lastt = -1;
        for (int t = 0; t < n_tiles; ++t) {
          if (s_tile[t] > 0.0) lastt = t;
          if (ts < 0 && cum + s_tile[t] > target) {
            ts = t;
            bs = cum;
          }
          cum += s_tile[t];
        }
        s_fallback = ts < 0;
        if (ts < 0) ts = lastt < 0 ? 0 : lastt;
        s_chunk = ts;
        s_base = bs;
        s_W = W;
      }
      __syncthreads();
      const int lo = s_chunk * kVocabChunk;
      const double W = s_W, target = s_fallback ? INFINITY : u * W;
      block_draw_tile(lo, min(V, lo + kVocabChunk), s_base, target, wres, ds);
      if (threadIdx.x == 0) {
        int emit = ds.found;
        if (emit == INT_MAX) {
          emit = ds.last < 0 ? lo : ds.last;
          s_near = 1;
        } else if (target - ds.prev_edge < kIcdfNearEps * W || ds.next_edge - target < kIcdfNearEps * W) {
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
        return w_target(v);
      };
      if (threadIdx.x == 0) {
        const RowPart* rp = a.part + (row_base + cur) * C;
        double W = 0.0;
        for (int c = 0; c < C; ++c)
          if (rp[c].m != -INFINITY) W += rp[c].s * static_cast<double>(expf((rp[c].m - M) * invT));
        for (int r = 0; r < nrej; ++r) W -= static_cast<double>(w_target(s_rej[r]));
        const double target = u * W;
        double cum = 0.0, bs = 0.0;
        int cs = -1, lastc = -1;
        for (int c = 0; c < C; ++c) {
          double wc = (rp[c].m == -INFINITY) ? 0.0 : rp[c].s * static_cast<double>(expf((rp[c].m - M) * invT));
          for (int r = 0; r < nrej; ++r)
            if (s_rej[r] / kVocabChunk == c) wc -= static_cast<double>(w_target(s_rej[r]));
          if (wc > 0.0) lastc = c;
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
      const double W = s_W, target = s_fallback ? INFINITY : u * W;
      block_draw_tile(lo, min(V, lo + kVocabChunk), s_base, target, w_of, ds);
      if (threadIdx.x == 0) {
        int emit = ds.found;
        if (emit == INT_MAX) {
          emit = ds.last < 0 ? lo : ds.last;
          s_near = 1;
        } else if (target - ds.prev_edge < kIcdfNearEps * W || ds.next_edge - target < kIcdfNearEps * W) {
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
  dim3 grid(p.B * p.R, p.n_chunks, p.n_sources);
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
