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
//   accept_coop_kernel      the walk as one cooperative launch: a group of CTAs per
//                           request, each owning a slice of the vocabulary (whole
//                           4096-token chunks).  At each node the walk reaches, every
//                           CTA reads its slice of that node's row once (chunk max,
//                           sum exp((x - m) / T), argmax), the group exchanges the
//                           chunk records through a bounded per-request barrier, and
//                           every CTA merges them and takes the same decision; a
//                           rejected drawn proposal adds one more slice pass (the
//                           residual's mass).  The emitted token is drawn by the CTA
//                           whose chunk holds the crossing.  Only the rows the walk
//                           visits are read.
//   accept_rowstats_kernel  (when a cooperative grid of the requests does not fit)
//   + accept_walk_kernel    one CTA per (tree row, chunk, source) for every row's
//                           statistics, then one CTA per request walks, merging the
//                           chunk statistics of the rows it visits.  Point-mass
//                           residuals only zero a few tokens, so a draw skips to the
//                           chunk that holds the crossing; drawn-proposal residuals
//                           take full passes.
//
// Precision: weights are expf((x - m) / T) in fp32; per-thread sums are compensated
// (Neumaier) and every sum across threads, chunks or tiles is float-float (about 48
// significant bits, on the fp32 pipe: this GPU's fp64 pipe is too narrow for it), so a
// running sum stays orders of magnitude within 1e-7 of the total mass of its exact
// value.  Draws are reported as near-ties when they land within 1e-7 of the mass of a
// bin edge; acceptance ratios (fp32) when within 1e-5 of u.
#include <limits.h>

#include "common.cuh"
#include "launch.h"
#include "sm100.cuh"

namespace eagle {
namespace {

constexpr int kThreads = 256;
constexpr int kPer = kVocabChunk / kThreads;  // 16 elements per thread per tile
constexpr float kIcdfNearEps = 1e-7f;

struct RowPart {
  float m;    // chunk max
  float av;   // chunk argmax value
  int ai;     // chunk argmax index (lowest on ties)
  int pad;
  ff s;       // sum exp((x - m) / T), float-float
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

// The 16 elements thread t takes of a 4096-token chunk starting at lo (each index of
// the chunk exactly once): bf16 rows whose length is a multiple of 8 read two 16-byte
// groups 2048 tokens apart, fp32 rows (length a multiple of 4) four groups 1024
// apart, anything else one token per 256.  Out-of-range tokens read as -inf.  All the
// loads are issued before any value is used.
__device__ __forceinline__ void load_chunk(const void* base, size_t off, int lo, int hi, int dtype, int V, float (&x)[kPer],
                                           int (&xi)[kPer]) {
  const int t = threadIdx.x;
  if (dtype == EAGLE_BF16 && (V & 7) == 0) {
    uint4 u[2];
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const int i0 = lo + g * 2048 + 8 * t;
      u[g] = (i0 + 8 <= hi) ? __ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(base) + off + i0))
                            : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);  // bf16 -inf pairs
    }
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      x[8 * g + 0] = __uint_as_float(u[g].x << 16);
      x[8 * g + 1] = __uint_as_float(u[g].x & 0xffff0000u);
      x[8 * g + 2] = __uint_as_float(u[g].y << 16);
      x[8 * g + 3] = __uint_as_float(u[g].y & 0xffff0000u);
      x[8 * g + 4] = __uint_as_float(u[g].z << 16);
      x[8 * g + 5] = __uint_as_float(u[g].z & 0xffff0000u);
      x[8 * g + 6] = __uint_as_float(u[g].w << 16);
      x[8 * g + 7] = __uint_as_float(u[g].w & 0xffff0000u);
#pragma unroll
      for (int j = 0; j < 8; ++j) xi[8 * g + j] = lo + g * 2048 + 8 * t + j;
    }
  } else if (dtype == EAGLE_F32 && (V & 3) == 0) {
    float4 f[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int i0 = lo + g * 1024 + 4 * t;
      f[g] = (i0 + 4 <= hi) ? __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + off + i0))
                            : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      x[4 * g + 0] = f[g].x;
      x[4 * g + 1] = f[g].y;
      x[4 * g + 2] = f[g].z;
      x[4 * g + 3] = f[g].w;
#pragma unroll
      for (int j = 0; j < 4; ++j) xi[4 * g + j] = lo + g * 1024 + 4 * t + j;
    }
  } else {
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      xi[k] = lo + k * kThreads + t;
      x[k] = xi[k] < hi ? load_elem(base, off + xi[k], dtype) : -INFINITY;
    }
  }
}

// Block-wide statistics of chunk c of one row (elements [c 4096, min(V, (c + 1) 4096))):
// max, argmax (lowest index on ties) and sum exp((x - m) / T) as float-float.  Every
// thread of the block calls it; the returned record is valid in thread 0.
__device__ RowPart chunk_rowpart(const AcceptPlan& p, const void* base, size_t off, int c, float invT,
                                float* keep = nullptr) {
  const int lo = c * kVocabChunk, hi = min(p.V, lo + kVocabChunk);
  float x[kPer];
  int xi[kPer];
  load_chunk(base, off, lo, hi, p.dtype, p.V, x, xi);
  if (keep) {  // the chunk's values, by position in the chunk, for a later draw
#pragma unroll
    for (int k = 0; k < kPer; ++k) keep[xi[k] - lo] = x[k];
  }
  // this thread's max and argmax (lowest index on ties), then its sum of
  // exp((x - m) / T), compensated
  float m = -INFINITY, av = -INFINITY;
  int ai = INT_MAX;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    if (xi[k] >= hi) continue;
    m = fmaxf(m, x[k]);
    if (before(x[k], xi[k], av, ai)) {
      av = x[k];
      ai = xi[k];
    }
  }
  CSum acc;
  if (m != -INFINITY) {
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      if (xi[k] < hi) acc.add(expf((x[k] - m) * invT));
  }
  // warp max / argmax, then the sums rescaled to the warp max, float-float
  ff s = csum_ff(acc);
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
  s = (m == -INFINITY) ? ff_make(0.f) : ff_mul(s, expf((m - M) * invT));
  s = warp_sum_ff(s);
  __shared__ RowPart wp[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // earlier readers of wp are done
  if (lane == 0) wp[warp] = RowPart{M, av, ai, 0, s};
  __syncthreads();
  RowPart r = wp[0];
  if (threadIdx.x == 0) {
    for (int w = 1; w < kThreads / 32; ++w) r.m = fmaxf(r.m, wp[w].m);
    ff t = ff_make(0.f);
    for (int w = 0; w < kThreads / 32; ++w) {
      if (wp[w].m != -INFINITY) t = ff_add(t, ff_mul(wp[w].s, expf((wp[w].m - r.m) * invT)));
      if (w > 0 && before(wp[w].av, wp[w].ai, r.av, r.ai)) {
        r.av = wp[w].av;
        r.ai = wp[w].ai;
      }
    }
    r.s = t;
  }
  return r;
}

__global__ void __launch_bounds__(kThreads, 4) accept_rowstats_kernel(const AcceptPlan p, const void* target,
                                                                   const void* draft, RowPart* part) {
  const int row = blockIdx.x, c = blockIdx.y, src = blockIdx.z;
  const int rows = gridDim.x, n_chunks = gridDim.y;
  const void* base = src == 0 ? target : draft;
  const float invT = 1.f / (p.temperature > 0.f ? p.temperature : 1.f);
  const RowPart r = chunk_rowpart(p, base, static_cast<size_t>(row) * p.V, c, invT);
  if (threadIdx.x == 0) part[(static_cast<size_t>(src) * rows + row) * n_chunks + c] = r;
}

// ------------------------------------------------------------------ block helpers
struct DrawScratch {
  ff wsum[kThreads / 32];
  int found;
  int last;
  ff prev_edge, next_edge, total;
};

__device__ __forceinline__ ff ff_shfl_up(ff v, int o) {
  return ff{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}

// One tile of an inverse-CDF draw: elements [lo, hi) (lo < hi <= lo + 4096), running
// mass `base` before lo.  Each thread takes 16 consecutive elements: ld(v) fetches an
// element's raw values (all 16 requested before any is used), wt(v, raw) gives its
// weight.  Its running sum and the thread offsets are float-float.  Sets ds.found to
// the first index whose running mass exceeds `target` (INT_MAX if none), ds.last to the
// last index with positive weight (-1 if none) and ds.total to the tile's mass.
// The n_ex indices in ex[] (shared memory) get weight 0.
template <class LD, class WT>
__device__ void block_draw_tile(int lo, int hi, ff base, ff target, LD ld, WT wt, const int* ex, int n_ex,
                                DrawScratch& ds) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a0 = lo + threadIdx.x * kPer;
  float2 raw[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) raw[e] = ld(min(a0 + e, hi - 1));
  uint32_t exm = 0;  // excluded elements of this thread, one bit each
  for (int r = 0; r < n_ex; ++r) {
    const int d = ex[r] - a0;
    if (d >= 0 && d < kPer) exm |= 1u << d;
  }
  float w[kPer];
  ff my = ff_make(0.f);
  int last = -1;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int v = a0 + e;
    w[e] = (v < hi && !((exm >> e) & 1u)) ? wt(v, raw[e]) : 0.f;
    my = ff_add(my, w[e]);
    if (w[e] > 0.f) last = v;
  }
  ff incl = my;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff t = ff_shfl_up(incl, o);
    if (lane >= o) incl = ff_add(incl, t);
  }
  __syncthreads();  // earlier readers of ds are done
  if (threadIdx.x == 0) {
    ds.found = INT_MAX;
    ds.last = -1;
  }
  if (lane == 31) ds.wsum[warp] = incl;
  __syncthreads();
  ff wbase = ff_make(0.f), tot = ff_make(0.f);
  for (int i = 0; i < kThreads / 32; ++i) {
    if (i < warp) wbase = ff_add(wbase, ds.wsum[i]);
    tot = ff_add(tot, ds.wsum[i]);
  }
  const ff tbase = ff_sub(ff_add(ff_add(base, wbase), incl), my);  // mass before this thread's first element
  const ff rel = ff_sub(target, tbase);
  int found = INT_MAX;
  ff pe = ff_make(0.f), ne = ff_make(0.f);
  {
    ff cum = ff_make(0.f);
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const ff nc = ff_add(cum, w[e]);
      if (found == INT_MAX && a0 + e < hi && w[e] > 0.f && ff_gt(nc, rel)) {
        found = a0 + e;
        pe = ff_add(tbase, cum);
        ne = ff_add(tbase, nc);
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

// Block sum of wf(v) over [lo, hi): compensated per thread, float-float across threads.
template <class WF>
__device__ ff block_sum(int lo, int hi, WF wf, ff* red) {
  CSum acc;
  for (int v = lo + threadIdx.x; v < hi; v += kThreads) acc.add(wf(v));
  const ff s = warp_sum_ff(csum_ff(acc));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = s;
  __syncthreads();
  ff t = ff_make(0.f);
  for (int i = 0; i < kThreads / 32; ++i) t = ff_add(t, red[i]);
  __syncthreads();
  return t;
}

// Block-wide merge of one row's chunk statistics: M = max chunk max, the argmax (lowest
// index on ties), and the mass of each chunk relative to M, wc = s_c exp((m_c - M) / T)
// (into tile_mass when non-null), summed as float-float.  Every thread returns the
// totals.
struct RowStats {
  float M;
  int amax;
  ff Z;
};

// A chunk record read from L2 (.cg): records are rewritten between the barrier phases of
// one launch by other CTAs, so this SM's L1 may hold an older copy.
__device__ __forceinline__ RowPart load_rowpart(const RowPart* rp) {
  RowPart r;
  r.m = __ldcg(&rp->m);
  r.av = __ldcg(&rp->av);
  r.ai = __ldcg(&rp->ai);
  r.pad = 0;
  r.s = ff{__ldcg(&rp->s.hi), __ldcg(&rp->s.lo)};
  return r;
}

__device__ RowStats merge_row_stats(const RowPart* rp, int C, float invT, ff* tile_mass, float* rf, int* ri,
                                    ff* rd) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float m = -INFINITY, av = -INFINITY;
  int ai = INT_MAX;
  // this thread's first record stays in registers for the mass pass below (C <= 256
  // needs no second read)
  const RowPart r0 = threadIdx.x < C ? load_rowpart(rp + threadIdx.x) : RowPart{-INFINITY, -INFINITY, INT_MAX, 0, {0.f, 0.f}};
  for (int c = threadIdx.x; c < C; c += kThreads) {
    const RowPart r = c == threadIdx.x ? r0 : load_rowpart(rp + c);
    m = fmaxf(m, r.m);
    if (before(r.av, r.ai, av, ai)) {
      av = r.av;
      ai = r.ai;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float v2 = __shfl_xor_sync(0xffffffffu, av, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, ai, o);
    if (before(v2, i2, av, ai)) {
      av = v2;
      ai = i2;
    }
  }
  __syncthreads();  // earlier readers of the scratch are done
  if (lane == 0) {
    rf[warp] = m;
    rf[kThreads / 32 + warp] = av;
    ri[warp] = ai;
  }
  __syncthreads();
  RowStats st;
  st.M = rf[0];
  av = rf[kThreads / 32];
  ai = ri[0];
  for (int w = 1; w < kThreads / 32; ++w) {
    st.M = fmaxf(st.M, rf[w]);
    if (before(rf[kThreads / 32 + w], ri[w], av, ai)) {
      av = rf[kThreads / 32 + w];
      ai = ri[w];
    }
  }
  st.amax = ai;
  ff z = ff_make(0.f);
  for (int c = threadIdx.x; c < C; c += kThreads) {
    const RowPart r = c == threadIdx.x ? r0 : load_rowpart(rp + c);
    const ff wc = (r.m == -INFINITY) ? ff_make(0.f) : ff_mul(r.s, expf((r.m - st.M) * invT));
    if (tile_mass) tile_mass[c] = wc;
    z = ff_add(z, wc);
  }
  z = warp_sum_ff(z);
  if (lane == 0) rd[warp] = z;
  __syncthreads();
  st.Z = ff_make(0.f);
  for (int w = 0; w < kThreads / 32; ++w) st.Z = ff_add(st.Z, rd[w]);
  return st;
}

__global__ void __launch_bounds__(kThreads, 1) accept_walk_kernel(const AcceptPlan p, const WalkArgs a) {
  const int b = blockIdx.x;
  const int R = p.R, V = p.V, C = p.n_chunks;
  const bool greedy = !(p.temperature > 0.f);
  const bool sampled = !greedy && p.proposal == EAGLE_PROPOSAL_SAMPLED;
  const float invT = 1.f / (greedy ? 1.f : p.temperature);
  const int maxp = p.max_depth + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  __shared__ int s_path[kMaxRows + 1];
  __shared__ int s_par[kMaxRows], s_tokr[kMaxRows];
  __shared__ uint32_t s_kidmask[kMaxRows / 32];
  __shared__ int s_kids[kMaxRows];
  __shared__ float s_wk[kMaxRows];  // point-mass proposals: exp((x_d - M) / T) of each child's token
  __shared__ float s_uk[kMaxRows];  // the children's acceptance uniforms
  __shared__ int s_nk, s_len, s_cur, s_next, s_emit, s_done, s_near, s_flag;
  __shared__ unsigned s_status;
  __shared__ int s_rej[kMaxRows];
  __shared__ float s_rejw[kMaxRows];
  __shared__ int s_nrej;
  __shared__ float s_Z[kMaxRows];  // drawn proposals: normalisers of the residual chain
  __shared__ int s_nz;
  __shared__ float s_M, s_Mq;
  __shared__ ff s_Zt, s_Zq;
  __shared__ int s_amax;
  __shared__ ff red[kThreads / 32];
  __shared__ float s_rf[kThreads / 16];
  __shared__ int s_ri[kThreads / 32];
  __shared__ DrawScratch ds;
  __shared__ int s_chunk, s_fallback;
  __shared__ ff s_base, s_W;
  __shared__ ff s_tile[kMaxVocabTiles];

  // the request's tree arrays, once; a parent that does not precede its row is a bad tree
  for (int c = threadIdx.x; c < R; c += kThreads) {
    s_par[c] = a.parent[static_cast<size_t>(b) * R + c];
    s_tokr[c] = a.tokens[static_cast<size_t>(b) * R + c];
  }
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
  {
    bool bad = false;
    for (int c = 1 + threadIdx.x; c < R; c += kThreads) bad |= (s_par[c] >= c || s_par[c] < 0);
    if (__syncthreads_or(bad) && threadIdx.x == 0) s_status |= EAGLE_STATUS_BAD_TREE;
  }

  const size_t row_base = static_cast<size_t>(b) * R;
  const int32_t* tok = s_tokr;
  for (int iter = 0; iter <= R && !s_done; ++iter) {
    const int cur = s_cur;
    const size_t xrow = (row_base + cur) * V;
    // children of cur in row order: a ballot per 32 rows
    if (warp < kMaxRows / 32) {
      const int c = warp * 32 + lane;
      const uint32_t mk = __ballot_sync(0xffffffffu, c > cur && c < R && s_par[c] == cur);
      if (lane == 0) s_kidmask[warp] = mk;
    }
    // the target row's statistics (and the draft row's for drawn proposals)
    const RowStats ts = merge_row_stats(a.part + (row_base + cur) * C, C, invT, s_tile, s_rf, s_ri, red);
    RowStats qs{};
    if (sampled)
      qs = merge_row_stats(a.part + (static_cast<size_t>(p.B) * R + row_base + cur) * C, C, invT, nullptr, s_rf,
                           s_ri, red);
    if (threadIdx.x == 0) {
      int nk = 0;
      for (int w = 0; w < kMaxRows / 32; ++w) {
        uint32_t mk = s_kidmask[w];
        while (mk) {
          s_kids[nk++] = w * 32 + __ffs(mk) - 1;
          mk &= mk - 1;
        }
      }
      s_nk = nk;
      s_M = ts.M;
      s_Zt = ts.Z;
      s_amax = ts.amax;
      s_Mq = qs.M;
      s_Zq = qs.Z;
      s_next = -1;
      s_nrej = 0;
      s_nz = 0;
    }
    __syncthreads();
    const float M = s_M, Mq = s_Mq;
    const float invZt = 1.f / ff_float(s_Zt);
    const float invZq = sampled ? 1.f / ff_float(s_Zq) : 0.f;
    auto w_target = [&](int v) { return expf((load_elem(a.target, xrow + v, p.dtype) - M) * invT); };
    auto p_of = [&](int v) { return w_target(v) * invZt; };
    auto q_of = [&](int v) { return expf((load_elem(a.draft, xrow + v, p.dtype) - Mq) * invT) * invZq; };
    // residual chain for drawn proposals: p_j = max(0, p_{j-1} - q) / Z_j
    auto pres_of = [&](int v, int nz) {
      float pv = p_of(v);
      if (nz == 0) return pv;
      const float qv = q_of(v);
      for (int i = 0; i < nz; ++i) pv = fmaxf(pv - qv, 0.f) / s_Z[i];
      return pv;
    };
    // the children's uniforms (and, for point-mass proposals, their target weights)
    for (int i = threadIdx.x; i < s_nk; i += kThreads) {
      const int c = s_kids[i];
      const int d = tok[c];
      s_uk[i] = a.u_accept[row_base + c];
      s_wk[i] = (!greedy && !sampled && d >= 0 && d < V) ? w_target(d) : 0.f;
    }
    __syncthreads();

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
        const float invZ = 1.f / ff_float(s_Zt);
        ff rejmass = ff_make(0.f);
        for (int i = 0; i < s_nk; ++i) {
          const int c = s_kids[i];
          const int d = tok[c];
          if (d < 0 || d >= V) {
            s_status |= EAGLE_STATUS_BAD_TOKEN;
            continue;
          }
          bool dup = false;
          for (int r = 0; r < s_nrej; ++r) dup |= (s_rej[r] == d);
          const float pd = dup ? 0.f : s_wk[i] * invZ;
          const float denom = ff_float(ff_sub(ff_make(1.f), rejmass));
          const float ratio = denom > 0.f ? __fdividef(pd, denom) : 0.f;
          const float u = s_uk[i];
          if (fabsf(u - ratio) < kNearTieEps) s_near = 1;
          if (u < ratio) {
            s_next = c;
            break;
          }
          if (!dup) {
            s_rejw[s_nrej] = s_wk[i];
            s_rej[s_nrej++] = d;
            rejmass = ff_add(rejmass, pd);
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
            const float qd = q_of(d);
            const float pd = pres_of(d, nz);
            const float ratio = qd > 0.f ? pd / qd : INFINITY;
            const float u = s_uk[i];
            if (qd > 0.f && fabsf(u - ratio) < kNearTieEps) s_near = 1;
            if (!(qd > 0.f) || u < ratio)
              s_next = c;
            else
              s_flag = 1;
          }
        }
        __syncthreads();
        if (s_next >= 0) break;
        if (s_flag) {
          const ff z = block_sum(0, V, [&](int v) { return fmaxf(pres_of(v, nz) - q_of(v), 0.f); }, red);
          if (threadIdx.x == 0 && z.hi > 0.f) s_Z[s_nz++] = ff_float(z);
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

    // ---- draw the emitted token from the (residual) target distribution: a mass per
    // 4096-token tile, the tile holding the crossing, then that tile element by element
    const float u = a.u_final[b];
    const bool residual = sampled && s_nz > 0;
    const int nz = s_nz, nrej = s_nrej;
    auto wres = [&](int v) { return pres_of(v, nz); };
    if (residual) {
      const int n_tiles = (V + kVocabChunk - 1) / kVocabChunk;
      for (int t = 0; t < n_tiles; ++t) {
        const ff m = block_sum(t * kVocabChunk, min(V, (t + 1) * kVocabChunk), wres, red);
        if (threadIdx.x == 0) s_tile[t] = m;
      }
    } else {
      // the row's chunk masses less the rejected point-mass tokens
      for (int c = threadIdx.x; c < C; c += kThreads) {
        ff wc = s_tile[c];
        for (int r = 0; r < nrej; ++r)
          if (s_rej[r] / kVocabChunk == c) wc = ff_sub(wc, ff_make(s_rejw[r]));
        s_tile[c] = wc;
      }
    }
    __syncthreads();
    if (warp == 0) {
      // total mass W, then the first tile whose running mass exceeds u W: an inclusive
      // float-float scan over 32 tiles at a time, the crossing found by ballot
      ff W = ff_make(0.f);
      if (residual) {
        for (int c = lane; c < C; c += 32) W = ff_add(W, s_tile[c]);
        W = warp_sum_ff(W);
      } else {
        W = s_Zt;
        for (int r = 0; r < nrej; ++r) W = ff_sub(W, ff_make(s_rejw[r]));
      }
      const ff target = ff_mul(W, u);
      ff carry = ff_make(0.f), bs = ff_make(0.f);
      int cs = -1, lastc = -1;
      for (int c0 = 0; c0 < C; c0 += 32) {
        const int c = c0 + lane;
        const ff wc = c < C ? s_tile[c] : ff_make(0.f);
        ff incl = wc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const ff t = ff_shfl_up(incl, o);
          if (lane >= o) incl = ff_add(incl, t);
        }
        const ff cum = ff_add(carry, incl);
        const unsigned pos = __ballot_sync(0xffffffffu, c < C && wc.hi > 0.f);
        if (pos) lastc = c0 + 31 - __clz(pos);
        const unsigned cross = __ballot_sync(0xffffffffu, c < C && ff_gt(cum, target));
        const ff excl = ff_sub(cum, wc);
        if (cs < 0 && cross) {
          const int l = __ffs(cross) - 1;
          cs = c0 + l;
          bs = ff{__shfl_sync(0xffffffffu, excl.hi, l), __shfl_sync(0xffffffffu, excl.lo, l)};
        }
        carry = ff_add(carry, ff{__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)});
      }
      if (lane == 0) {
        s_fallback = cs < 0;  // nothing crosses (rounding): take the last positive weight
        s_chunk = cs < 0 ? (lastc < 0 ? 0 : lastc) : cs;
        s_base = bs;
        s_W = W;
      }
    }
    __syncthreads();
    const int lo = s_chunk * kVocabChunk;
    const ff W = s_W;
    const ff target = s_fallback ? ff{INFINITY, 0.f} : ff_mul(W, u);
    if (residual) {
      block_draw_tile(
          lo, min(V, lo + kVocabChunk), s_base, target,
          [&](int v) {
            return make_float2(load_elem(a.target, xrow + v, p.dtype), load_elem(a.draft, xrow + v, p.dtype));
          },
          [&](int v, float2 x) {
            float pv = expf((x.x - M) * invT) * invZt;
            const float qv = expf((x.y - Mq) * invT) * invZq;
            for (int i = 0; i < nz; ++i) pv = fmaxf(pv - qv, 0.f) / s_Z[i];
            return pv;
          },
          s_rej, 0, ds);
    } else {
      block_draw_tile(
          lo, min(V, lo + kVocabChunk), s_base, target,
          [&](int v) { return make_float2(load_elem(a.target, xrow + v, p.dtype), 0.f); },
          [&](int, float2 x) { return expf((x.x - M) * invT); }, s_rej, nrej, ds);
    }
    if (threadIdx.x == 0) {
      int emit = ds.found;
      const float win = kIcdfNearEps * ff_float(W);
      if (emit == INT_MAX) {
        emit = ds.last < 0 ? lo : ds.last;
        s_near = 1;
      } else if (ff_float(ff_sub(target, ds.prev_edge)) < win || ff_float(ff_sub(ds.next_edge, target)) < win) {
        s_near = 1;
      }
      s_emit = emit;
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
      ob[j] = j < na ? s_tokr[s_path[j + 1]] : (j == na ? s_emit : -1);
    }
    a.out.n_acc[b] = na;
    a.out.near_tie[b] = s_near;
    if (s_status) atomicOr(a.out.status, s_status);
  }
}

// ------------------------------------------------------------------ cooperative walk
struct CoopArgs {
  WalkArgs w;  // w.part: chunk records [B][2 slots][2 sources][C]
  int* cnt;    // [B] arrivals at the per-request barrier, zeroed before each launch
  int cpr;     // CTAs per request
};

// Per-request barrier: thread 0 counts this CTA in and waits (at most 2 s) until the
// request has `target` arrivals; then the block syncs.  False on a timeout.
__device__ bool req_barrier(int* cnt, int target) {
  __shared__ int s_ok;
  __syncthreads();  // this CTA's record writes come before its count
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(cnt, 1);
    int ok = 1;
    if (sm100::ld_acquire_gpu(cnt) < target) {
      const uint64_t t0 = sm100::global_ns();
      while (sm100::ld_acquire_gpu(cnt) < target) {
        if (sm100::global_ns() - t0 > 2000000000ull) {
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Float-float sum of the s fields of C chunk records (every thread returns it).
__device__ ff sum_records(const RowPart* rp, int C, ff* red) {
  ff z = ff_make(0.f);
  for (int c = threadIdx.x; c < C; c += kThreads) z = ff_add(z, ff{__ldcg(&rp[c].s.hi), __ldcg(&rp[c].s.lo)});
  z = warp_sum_ff(z);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = z;
  __syncthreads();
  ff t = ff_make(0.f);
  for (int i = 0; i < kThreads / 32; ++i) t = ff_add(t, red[i]);
  __syncthreads();
  return t;
}

// The walk's mode is a template argument (greedy, point-mass or drawn proposals), so that
// each launch carries only its own path: the walk runs most of its code once per launch,
// from a cold instruction cache, and a smaller kernel misses less.
enum { kWalkGreedy = 0, kWalkDelta = 1, kWalkSampled = 2 };

template <int MODE>
__global__ void __launch_bounds__(kThreads, 2) accept_coop_kernel(const AcceptPlan p, const CoopArgs ca) {
  const WalkArgs& a = ca.w;
  const int b = blockIdx.y, cta = blockIdx.x, cpr = ca.cpr;
  const int R = p.R, V = p.V, C = p.n_chunks;
  constexpr bool greedy = MODE == kWalkGreedy;
  constexpr bool sampled = MODE == kWalkSampled;
  const float invT = 1.f / (greedy ? 1.f : p.temperature);
  const int maxp = p.max_depth + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* cnt = ca.cnt + b;
  // chunk records of slot s (alternating between barrier phases) and source (0 target, 1 draft)
  auto rec = [&](int slot, int src) { return const_cast<RowPart*>(a.part) + ((static_cast<size_t>(b) * 2 + slot) * 2 + src) * C; };
  int phase = 0;  // barrier phases this request has passed

  __shared__ int s_path[kMaxRows + 1];
  __shared__ int s_par[kMaxRows], s_tokr[kMaxRows];
  __shared__ uint32_t s_kidmask[kMaxRows / 32];
  __shared__ int s_kids[kMaxRows];
  __shared__ float s_wk[kMaxRows];
  __shared__ float s_uk[kMaxRows];
  __shared__ int s_nk, s_len, s_cur, s_next, s_emit, s_done, s_near, s_flag, s_abort, s_write;
  __shared__ unsigned s_status;
  __shared__ int s_rej[kMaxRows];
  __shared__ float s_rejw[kMaxRows];
  __shared__ int s_nrej;
  __shared__ float s_Z[kMaxRows];
  __shared__ int s_nz;
  __shared__ float s_M, s_Mq;
  __shared__ ff s_Zt, s_Zq;
  __shared__ int s_amax;
  __shared__ ff red[kThreads / 32];
  __shared__ float s_rf[kThreads / 16];
  __shared__ int s_ri[kThreads / 32];
  __shared__ DrawScratch ds;
  __shared__ int s_chunk, s_fallback;
  __shared__ ff s_base, s_W;
  __shared__ ff s_tile[kMaxVocabTiles];
  __shared__ float s_xk[kMaxRows];  // the target logits of the children's tokens
  // one chunk per CTA: the target (and draft) values of that chunk of the current row,
  // kept from the statistics pass for the residual passes and the draw in this CTA
  __shared__ float s_vals[kVocabChunk];
  __shared__ float s_dvals[kVocabChunk];
  const bool keep = cpr == C;
  const int own_lo = cta * kVocabChunk;

  // the request's tree and uniforms, once: later levels read them from shared memory
  __shared__ float s_ua[kMaxRows];
  __shared__ float s_uf;
  for (int c = threadIdx.x; c < R; c += kThreads) {
    s_par[c] = a.parent[static_cast<size_t>(b) * R + c];
    s_tokr[c] = a.tokens[static_cast<size_t>(b) * R + c];
    s_ua[c] = a.u_accept[static_cast<size_t>(b) * R + c];
  }
  if (threadIdx.x == 0) s_uf = a.u_final[b];
  if (threadIdx.x == 0) {
    s_len = 1;
    s_path[0] = 0;
    s_cur = 0;
    s_done = 0;
    s_near = 0;
    s_status = 0;
    s_emit = -1;
    s_abort = 0;
    s_write = cta == 0;  // the writer of the outputs unless a draw names another CTA
  }
  __syncthreads();
  {
    bool bad = false;
    for (int c = 1 + threadIdx.x; c < R; c += kThreads) bad |= (s_par[c] >= c || s_par[c] < 0);
    if (__syncthreads_or(bad) && threadIdx.x == 0) s_status |= EAGLE_STATUS_BAD_TREE;
  }

  const size_t row_base = static_cast<size_t>(b) * R;
  const int32_t* tok = s_tokr;
  for (int iter = 0; iter <= R && !s_done && !s_abort; ++iter) {
    const int cur = s_cur;
    const size_t xrow = (row_base + cur) * V;
    if (warp < kMaxRows / 32) {
      const int c = warp * 32 + lane;
      const uint32_t mk = __ballot_sync(0xffffffffu, c > cur && c < R && s_par[c] == cur);
      if (lane == 0) s_kidmask[warp] = mk;
    }
    __syncthreads();
    // the children of cur, their uniforms and their tokens' target logits, fetched
    // while the row's statistics load
    if (threadIdx.x == 0) {
      int nk = 0;
      for (int w = 0; w < kMaxRows / 32; ++w) {
        uint32_t mk = s_kidmask[w];
        while (mk) {
          s_kids[nk++] = w * 32 + __ffs(mk) - 1;
          mk &= mk - 1;
        }
      }
      s_nk = nk;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < s_nk; i += kThreads) {
      const int c = s_kids[i];
      const int d = tok[c];
      s_uk[i] = s_ua[c];
      s_xk[i] = (!greedy && !sampled && d >= 0 && d < V) ? load_elem(a.target, xrow + d, p.dtype) : 0.f;
    }
    // this CTA's slice of the node's target (and draft) row, exchanged with the group
    const int slot = phase & 1;
    for (int c = cta; c < C; c += cpr) {
      const RowPart r = chunk_rowpart(p, a.target, xrow, c, invT, keep ? s_vals : nullptr);
      if (threadIdx.x == 0) rec(slot, 0)[c] = r;
      if (sampled) {
        const RowPart q = chunk_rowpart(p, a.draft, xrow, c, invT, keep ? s_dvals : nullptr);
        if (threadIdx.x == 0) rec(slot, 1)[c] = q;
      }
    }
    if (!req_barrier(cnt, ++phase * cpr)) {
      if (threadIdx.x == 0) s_abort = 1;
      __syncthreads();
      break;
    }
    const RowStats ts = merge_row_stats(rec(slot, 0), C, invT, s_tile, s_rf, s_ri, red);
    RowStats qs{};
    if (sampled) qs = merge_row_stats(rec(slot, 1), C, invT, nullptr, s_rf, s_ri, red);
    if (threadIdx.x == 0) {
      s_M = ts.M;
      s_Zt = ts.Z;
      s_amax = ts.amax;
      s_Mq = qs.M;
      s_Zq = qs.Z;
      s_next = -1;
      s_nrej = 0;
      s_nz = 0;
    }
    __syncthreads();
    const float M = s_M, Mq = s_Mq;
    const float invZt = 1.f / ff_float(s_Zt);
    const float invZq = sampled ? 1.f / ff_float(s_Zq) : 0.f;
    auto w_target = [&](int v) { return expf((load_elem(a.target, xrow + v, p.dtype) - M) * invT); };
    auto p_of = [&](int v) { return w_target(v) * invZt; };
    auto q_of = [&](int v) { return expf((load_elem(a.draft, xrow + v, p.dtype) - Mq) * invT) * invZq; };
    auto pres_of = [&](int v, int nz) {
      float pv = p_of(v);
      if (nz == 0) return pv;
      const float qv = q_of(v);
      for (int i = 0; i < nz; ++i) pv = fmaxf(pv - qv, 0.f) / s_Z[i];
      return pv;
    };
    // the same for a token of this CTA's own chunk, from the kept values
    auto pres_own = [&](int v, int nz) {
      if (!keep) return pres_of(v, nz);
      float pv = expf((s_vals[v - own_lo] - M) * invT) * invZt;
      if (nz == 0) return pv;
      const float qv = expf((s_dvals[v - own_lo] - Mq) * invT) * invZq;
      for (int i = 0; i < nz; ++i) pv = fmaxf(pv - qv, 0.f) / s_Z[i];
      return pv;
    };
    auto q_own = [&](int v) { return keep ? expf((s_dvals[v - own_lo] - Mq) * invT) * invZq : q_of(v); };
    for (int i = threadIdx.x; i < s_nk; i += kThreads) {
      const int d = tok[s_kids[i]];
      s_wk[i] = (!greedy && !sampled && d >= 0 && d < V) ? expf((s_xk[i] - M) * invT) : 0.f;
    }
    __syncthreads();

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
      // point-mass proposals: p_res(d) = p(d) / (1 - mass of the rejected tokens).  Child
      // i is tested only when every earlier child was rejected, so its residual mass is
      // 1 minus the masses of the distinct valid tokens before it: one lane per child, an
      // exclusive scan of those masses, and the first child whose test passes is the one
      // accepted (a node has at most 16 children; more take the serial loop)
      const int nk = s_nk;
      if (nk <= 32 && warp == 0) {
        const float invZ = 1.f / ff_float(s_Zt);
        const bool valid = lane < nk;
        const int c = valid ? s_kids[lane] : 0;
        const int d = valid ? tok[c] : -1;
        const bool bad = valid && (d < 0 || d >= V);
        bool dup = false;  // an earlier valid child with the same token (its mass is gone)
        for (int j = 0; j < lane && j < nk; ++j) {
          const int dj = tok[s_kids[j]];
          dup |= (dj >= 0 && dj < V && dj == d);
        }
        const bool live = valid && !bad && !dup;
        const float pd = live ? s_wk[lane] * invZ : 0.f;
        ff incl = ff_make(pd);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const ff t = ff_shfl_up(incl, o);
          if (lane >= o) incl = ff_add(incl, t);
        }
        const ff rejmass = ff_sub(incl, ff_make(pd));  // exclusive: the children before this one
        const float denom = ff_float(ff_sub(ff_make(1.f), rejmass));
        const float ratio = denom > 0.f ? __fdividef(pd, denom) : 0.f;
        const float u = valid ? s_uk[lane] : 2.f;
        const bool tested = valid && !bad;
        const unsigned acc = __ballot_sync(0xffffffffu, tested && u < ratio);
        const int first = acc ? __ffs(acc) - 1 : 32;  // children after it are never tested
        const bool seen = lane <= first;
        const bool near = __any_sync(0xffffffffu, seen && tested && fabsf(u - ratio) < kNearTieEps);
        const bool anybad = __any_sync(0xffffffffu, seen && bad && lane != first);
        // the rejected tokens and their weights, in child order, when none is accepted
        const unsigned rj = __ballot_sync(0xffffffffu, live && lane < first);
        if (live && lane < first) {
          const int slot = __popc(rj & ((1u << lane) - 1u));
          s_rej[slot] = d;
          s_rejw[slot] = s_wk[lane];
        }
        if (lane == 0) {
          if (near) s_near = 1;
          if (anybad) s_status |= EAGLE_STATUS_BAD_TOKEN;
          s_nrej = __popc(rj);
          if (first < 32) s_next = s_kids[first];
        }
      } else if (nk > 32 && threadIdx.x == 0) {
        const float invZ = 1.f / ff_float(s_Zt);
        ff rejmass = ff_make(0.f);
        for (int i = 0; i < s_nk; ++i) {
          const int c = s_kids[i];
          const int d = tok[c];
          if (d < 0 || d >= V) {
            s_status |= EAGLE_STATUS_BAD_TOKEN;
            continue;
          }
          bool dup = false;
          for (int r = 0; r < s_nrej; ++r) dup |= (s_rej[r] == d);
          const float pd = dup ? 0.f : s_wk[i] * invZ;
          const float denom = ff_float(ff_sub(ff_make(1.f), rejmass));
          const float ratio = denom > 0.f ? __fdividef(pd, denom) : 0.f;
          const float u = s_uk[i];
          if (fabsf(u - ratio) < kNearTieEps) s_near = 1;
          if (u < ratio) {
            s_next = c;
            break;
          }
          if (!dup) {
            s_rejw[s_nrej] = s_wk[i];
            s_rej[s_nrej++] = d;
            rejmass = ff_add(rejmass, pd);
          }
        }
      }
      __syncthreads();
    } else {
      // drawn proposals (SpecInfer multi-round): q fixed across siblings; a rejection
      // needs the residual's normaliser, one more slice pass of the group
      for (int i = 0; i < s_nk; ++i) {
        const int c = s_kids[i];
        const int nz = s_nz;
        if (threadIdx.x == 0) {
          const int d = tok[c];
          s_flag = 0;
          if (d < 0 || d >= V) {
            s_status |= EAGLE_STATUS_BAD_TOKEN;
          } else {
            const float qd = q_of(d);
            const float pd = pres_of(d, nz);
            const float ratio = qd > 0.f ? pd / qd : INFINITY;
            const float u = s_uk[i];
            if (qd > 0.f && fabsf(u - ratio) < kNearTieEps) s_near = 1;
            if (!(qd > 0.f) || u < ratio)
              s_next = c;
            else
              s_flag = 1;
          }
        }
        __syncthreads();
        if (s_next >= 0) break;
        if (s_flag) {
          const int slot2 = phase & 1;
          for (int cc = cta; cc < C; cc += cpr) {
            const int lo = cc * kVocabChunk, hi = min(V, lo + kVocabChunk);
            const ff z = block_sum(lo, hi, [&](int v) { return fmaxf(pres_own(v, nz) - q_own(v), 0.f); }, red);
            if (threadIdx.x == 0) rec(slot2, 0)[cc] = RowPart{0.f, 0.f, 0, 0, z};
          }
          if (!req_barrier(cnt, ++phase * cpr)) {
            if (threadIdx.x == 0) s_abort = 1;
            __syncthreads();
            break;
          }
          const ff z = sum_records(rec(slot2, 0), C, red);
          if (threadIdx.x == 0 && z.hi > 0.f) s_Z[s_nz++] = ff_float(z);
        }
        __syncthreads();
      }
      if (s_abort) break;
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

    // ---- draw the emitted token from the (residual) target distribution: the chunk
    // masses (the group's slice passes for a drawn-proposal residual), the chunk holding
    // the crossing, then that chunk element by element in the CTA that owns it
    const float u = s_uf;
    const bool residual = sampled && s_nz > 0;
    const int nz = s_nz, nrej = s_nrej;
    if (residual) {
      const int slot2 = phase & 1;
      for (int cc = cta; cc < C; cc += cpr) {
        const int lo = cc * kVocabChunk, hi = min(V, lo + kVocabChunk);
        const ff m = block_sum(lo, hi, [&](int v) { return pres_own(v, nz); }, red);
        if (threadIdx.x == 0) rec(slot2, 0)[cc] = RowPart{0.f, 0.f, 0, 0, m};
      }
      if (!req_barrier(cnt, ++phase * cpr)) {
        if (threadIdx.x == 0) s_abort = 1;
        __syncthreads();
        break;
      }
      for (int c = threadIdx.x; c < C; c += kThreads) s_tile[c] = ff{__ldcg(&rec(slot2, 0)[c].s.hi), __ldcg(&rec(slot2, 0)[c].s.lo)};
    } else {
      for (int c = threadIdx.x; c < C; c += kThreads) {
        ff wc = s_tile[c];
        for (int r = 0; r < nrej; ++r)
          if (s_rej[r] / kVocabChunk == c) wc = ff_sub(wc, ff_make(s_rejw[r]));
        s_tile[c] = wc;
      }
    }
    __syncthreads();
    if (warp == 0) {
      ff W = ff_make(0.f);
      if (residual) {
        for (int c = lane; c < C; c += 32) W = ff_add(W, s_tile[c]);
        W = warp_sum_ff(W);
      } else {
        W = s_Zt;
        for (int r = 0; r < nrej; ++r) W = ff_sub(W, ff_make(s_rejw[r]));
      }
      const ff target = ff_mul(W, u);
      ff carry = ff_make(0.f), bs = ff_make(0.f);
      int cs = -1, lastc = -1;
      for (int c0 = 0; c0 < C; c0 += 32) {
        const int c = c0 + lane;
        const ff wc = c < C ? s_tile[c] : ff_make(0.f);
        ff incl = wc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const ff t = ff_shfl_up(incl, o);
          if (lane >= o) incl = ff_add(incl, t);
        }
        const ff cum = ff_add(carry, incl);
        const unsigned pos = __ballot_sync(0xffffffffu, c < C && wc.hi > 0.f);
        if (pos) lastc = c0 + 31 - __clz(pos);
        const unsigned cross = __ballot_sync(0xffffffffu, c < C && ff_gt(cum, target));
        const ff excl = ff_sub(cum, wc);
        if (cs < 0 && cross) {
          const int l = __ffs(cross) - 1;
          cs = c0 + l;
          bs = ff{__shfl_sync(0xffffffffu, excl.hi, l), __shfl_sync(0xffffffffu, excl.lo, l)};
        }
        carry = ff_add(carry, ff{__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)});
      }
      if (lane == 0) {
        s_fallback = cs < 0;
        s_chunk = cs < 0 ? (lastc < 0 ? 0 : lastc) : cs;
        s_base = bs;
        s_W = W;
        s_write = (s_chunk % cpr) == cta;  // the chunk's owner draws and writes the outputs
      }
    }
    __syncthreads();
    if (!s_write) break;
    const int lo = s_chunk * kVocabChunk;
    const ff W = s_W;
    const ff target = s_fallback ? ff{INFINITY, 0.f} : ff_mul(W, u);
    if (residual) {
      block_draw_tile(
          lo, min(V, lo + kVocabChunk), s_base, target,
          [&](int v) {
            return keep ? make_float2(s_vals[v - lo], s_dvals[v - lo])
                        : make_float2(load_elem(a.target, xrow + v, p.dtype), load_elem(a.draft, xrow + v, p.dtype));
          },
          [&](int v, float2 x) {
            float pv = expf((x.x - M) * invT) * invZt;
            const float qv = expf((x.y - Mq) * invT) * invZq;
            for (int i = 0; i < nz; ++i) pv = fmaxf(pv - qv, 0.f) / s_Z[i];
            return pv;
          },
          s_rej, 0, ds);
    } else {
      block_draw_tile(
          lo, min(V, lo + kVocabChunk), s_base, target,
          [&](int v) { return make_float2(keep ? s_vals[v - lo] : load_elem(a.target, xrow + v, p.dtype), 0.f); },
          [&](int, float2 x) { return expf((x.x - M) * invT); }, s_rej, nrej, ds);
    }
    if (threadIdx.x == 0) {
      int emit = ds.found;
      const float win = kIcdfNearEps * ff_float(W);
      if (emit == INT_MAX) {
        emit = ds.last < 0 ? lo : ds.last;
        s_near = 1;
      } else if (ff_float(ff_sub(target, ds.prev_edge)) < win || ff_float(ff_sub(ds.next_edge, target)) < win) {
        s_near = 1;
      }
      s_emit = emit;
    }
    __syncthreads();
    break;
  }

  // ---- outputs, from one CTA of the request
  if (threadIdx.x == 0) {
    if (s_abort) {
      atomicOr(a.out.status, EAGLE_STATUS_TIMEOUT | s_status);
    } else if (s_write) {
      const int len = s_len;
      const int na = len - 1;
      int32_t* pb = a.out.path + static_cast<size_t>(b) * maxp;
      int32_t* ob = a.out.out_tok + static_cast<size_t>(b) * maxp;
      for (int j = 0; j < maxp; ++j) {
        pb[j] = j < len ? s_path[j] : -1;
        ob[j] = j < na ? s_tokr[s_path[j + 1]] : (j == na ? s_emit : -1);
      }
      a.out.n_acc[b] = na;
      a.out.near_tie[b] = s_near;
      if (s_status) atomicOr(a.out.status, s_status);
    }
  }
}

// Co-resident CTAs of the cooperative walk on the current device (0 when unknown);
// cached per device.
int coop_capacity() {
  static int cached[64];
  static unsigned long long known = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  if (dev < 64 && (__atomic_load_n(&known, __ATOMIC_ACQUIRE) & (1ull << dev))) return cached[dev];
  int per_sm = 0, sms = 0, o1 = 0, o2 = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, accept_coop_kernel<kWalkGreedy>, kThreads, 0) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o1, accept_coop_kernel<kWalkDelta>, kThreads, 0) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o2, accept_coop_kernel<kWalkSampled>, kThreads, 0) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    per_sm = sms = 0;
  }
  per_sm = per_sm < o1 ? per_sm : o1;  // the co-resident grid of the smallest occupancy
  per_sm = per_sm < o2 ? per_sm : o2;
  (void)cudaGetLastError();
  const int n = per_sm * sms;
  if (dev < 64) {
    cached[dev] = n;
    __atomic_fetch_or(&known, 1ull << dev, __ATOMIC_RELEASE);
  }
  return n;
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
  // the workspace holds either launch form: the cooperative walk's barrier counters and
  // chunk records [B][2][2][C], or every row's chunk statistics for the two-kernel form
  p->off_cnt = 0;
  p->off_part = (static_cast<size_t>(p->B) * sizeof(int) + 255) / 256 * 256;
  const size_t coop = static_cast<size_t>(p->B) * 4 * p->n_chunks * sizeof(RowPart);
  const size_t rows = static_cast<size_t>(p->n_sources) * p->B * p->R * p->n_chunks * sizeof(RowPart);
  p->total = p->off_part + (coop > rows ? coop : rows);
}

cudaError_t launch_accept(const AcceptPlan& p, const void* target, const void* draft, const int32_t* tokens,
                          const int32_t* parent, const float* u_accept, const float* u_final,
                          const eagle_accept_out& out, void* ws, cudaStream_t s) {
  RowPart* part = reinterpret_cast<RowPart*>(static_cast<uint8_t*>(ws) + p.off_part);
  // the cooperative walk when a group of CTAs per request fits on the device at once
  const int cap = coop_capacity();
  const int cpr = cap / p.B < p.n_chunks ? cap / p.B : p.n_chunks;
  if (cpr >= 1) {
    int* cnt = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + p.off_cnt);
    cudaError_t e = cudaMemsetAsync(cnt, 0, static_cast<size_t>(p.B) * sizeof(int), s);
    if (e != cudaSuccess) return e;
    CoopArgs ca;
    ca.w.target = target;
    ca.w.draft = draft;
    ca.w.tokens = tokens;
    ca.w.parent = parent;
    ca.w.u_accept = u_accept;
    ca.w.u_final = u_final;
    ca.w.out = out;
    ca.w.part = part;
    ca.cnt = cnt;
    ca.cpr = cpr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cpr, p.B, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!(p.temperature > 0.f))
      e = cudaLaunchKernelEx(&cfg, accept_coop_kernel<kWalkGreedy>, p, ca);
    else if (p.proposal == EAGLE_PROPOSAL_SAMPLED)
      e = cudaLaunchKernelEx(&cfg, accept_coop_kernel<kWalkSampled>, p, ca);
    else
      e = cudaLaunchKernelEx(&cfg, accept_coop_kernel<kWalkDelta>, p, ca);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
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
