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
// One launch per level: tree_level_kernel, one CTA per (request x frontier row,
// 4096-token chunk).
//   chunk pass    every CTA: the chunk max, sum exp(x - m) (and sum exp((x - m) / T)
//                 for draws) and the chunk's best kc by (logit desc, id asc), from one
//                 read of the logits held in registers (16 per thread).
//   row finisher  the last CTA of a row to finish (an atomic ticket): merges the row's
//                 chunk records (M, ln Z, top-k or draws) and adds its candidates to the
//                 pool (dynamic) or its children to the shape (static).
//   request       the last row finisher of a request (a second ticket): picks the
//                 next frontier (rank counting), merges the level's ranked candidates
//                 into the request's sorted list of the best N + 1 so far, and after the
//                 last level writes the tree from that list's first N.
// No CTA waits for another; the tickets return to zero for the next level, and level 1
// clears them with a memset first.
//
// Precision: chunk sums are compensated fp32, merged as float-float (about 48
// significant bits on the fp32 pipe; this GPU's fp64 pipe is narrow), and ln Z is a
// float-float logarithm.  Cumulative scores are float-float, so that the selections
// agree with an fp64 computation unless two scores at a boundary are within 1e-5
// (reported as a near-tie).
#include <limits.h>
#include <stddef.h>

#include "common.cuh"
#include "launch.h"

namespace eagle {
namespace {

constexpr int kThreads = 256;
constexpr int NW = kThreads / 32;
constexpr int K = kMaxTopK;
constexpr int kPer = kVocabChunk / kThreads;  // logits per thread in the chunk pass
constexpr float kIcdfNearEps = 1e-7f;
static_assert(kPer == K, "the chunk pass sorts one thread's logits as a K-entry list");
static_assert(K * K <= kThreads, "a level's dynamic candidates are one per thread of the request's finisher");

struct __align__(16) ChunkPart {
  float tv[K];    // top-K logits of the chunk, best first
  int ti[K];      // their token ids (INT_MAX = empty)
  ff s1;          // sum exp(x - m)
  ff sT;          // sum exp((x - m) / T)
  float m;        // chunk max logit
  float pad[3];
};
static_assert(sizeof(ChunkPart) % 16 == 0, "chunk lists are read as 16-byte vectors");
static_assert(sizeof(ChunkPart) == sizeof(TreeChunkRecord) && offsetof(ChunkPart, s1) == offsetof(TreeChunkRecord, s1_hi) &&
                  offsetof(ChunkPart, sT) == offsetof(TreeChunkRecord, sT_hi) && offsetof(ChunkPart, m) == offsetof(TreeChunkRecord, m),
              "the LM-head kernel writes chunk records in this layout");
static_assert(kHeadRecords <= 160, "a warp merges at most 160 chunk lists");

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

// (value desc, id asc) order without short-circuit evaluation (no branches).
__device__ __forceinline__ bool before_nb(float va, int ia, float vb, int ib) {
  return (va > vb) | ((va == vb) & (ia < ib));
}

// Compare-exchange of two list entries so that entry i comes before entry j.
__device__ __forceinline__ void cas(float& vi, int& ii, float& vj, int& ij) {
  const bool sw = before_nb(vj, ij, vi, ii);
  const float tv = sw ? vj : vi;
  const int t = sw ? ij : ii;
  vj = sw ? vi : vj;
  ij = sw ? ii : ij;
  vi = tv;
  ii = t;
}

// Bitonic sorting network over K registers, best first (indices are compile-time
// constants once the loops unroll, so the arrays stay in registers).
__device__ __forceinline__ void sort_regs(float (&v)[K], int (&id)[K]) {
#pragma unroll
  for (int k = 2; k <= K; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int i = 0; i < K; ++i) {
        const int l = i ^ j;
        if (l > i) {
          if ((i & k) == 0)
            cas(v[i], id[i], v[l], id[l]);
          else
            cas(v[l], id[l], v[i], id[i]);
        }
      }
    }
  }
}

// Order-preserving unsigned images of floats (-0 taken as +0, so equal floats map to
// equal keys): a larger key is a larger value.
__device__ __forceinline__ uint32_t ord32(float f) {
  uint32_t u = __float_as_uint(f);
  u = (u == 0x80000000u) ? 0u : u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unord32(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
// The same for a bf16 value (its 16 bits), and back.
__device__ __forceinline__ uint32_t ord16(uint32_t b) {
  b = (b == 0x8000u) ? 0u : b;
  return (b & 0x8000u) ? (~b & 0xffffu) : (b | 0x8000u);
}
__device__ __forceinline__ float unord16(uint32_t o) {
  return __uint_as_float(((o & 0x8000u) ? (o & 0x7fffu) : (~o & 0xffffu)) << 16);
}

// Descending sorting network over K packed keys in registers.
__device__ __forceinline__ void sort_keys(uint32_t (&k)[K]) {
#pragma unroll
  for (int s = 2; s <= K; s <<= 1) {
#pragma unroll
    for (int j = s >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int i = 0; i < K; ++i) {
        const int l = i ^ j;
        if (l > i) {
          const uint32_t a = k[i], b = k[l];
          const bool first = (i & s) == 0;  // i takes the larger key
          k[i] = first ? max(a, b) : min(a, b);
          k[l] = first ? min(a, b) : max(a, b);
        }
      }
    }
  }
}

// A thread's kPer logits of the chunk [lo, hi) and their ids (-inf / INT_MAX past hi):
// bf16 as two runs of 8 (lo + 2048 g + 8 t ..), fp32 as four runs of 4 (lo + 1024 g +
// 4 t ..), each run one 16-byte load when `vec` (the row base is 16-byte aligned).
template <bool BF16>
__device__ __forceinline__ void load_chunk(const void* logits, size_t row, int lo, int hi, bool vec, float (&x)[kPer],
                                           int (&xi)[kPer]) {
  constexpr int RUN = BF16 ? 8 : 4;
  constexpr int NRUN = kPer / RUN;
#pragma unroll
  for (int g = 0; g < NRUN; ++g) {
    const int v0 = lo + g * kThreads * RUN + RUN * threadIdx.x;
    if (vec && v0 + RUN <= hi) {
      if constexpr (BF16) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(logits) + row + v0));
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          x[g * RUN + 2 * j] = __uint_as_float(u[j] << 16);
          x[g * RUN + 2 * j + 1] = __uint_as_float(u[j] & 0xffff0000u);
        }
      } else {
        const float4 w = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(logits) + row + v0));
        x[g * RUN] = w.x;
        x[g * RUN + 1] = w.y;
        x[g * RUN + 2] = w.z;
        x[g * RUN + 3] = w.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < RUN; ++j) {
        const int v = v0 + j;
        x[g * RUN + j] = v < hi ? load_elem(logits, row + v, BF16 ? EAGLE_BF16 : EAGLE_F32) : -INFINITY;
      }
    }
#pragma unroll
    for (int j = 0; j < RUN; ++j) xi[g * RUN + j] = (v0 + j < hi) ? v0 + j : INT_MAX;
  }
}

// ------------------------------------------------------------------ chunk pass
// One CTA's (frontier row, chunk) record: the chunk max, sum exp(x - m) (and, for draws,
// sum exp((x - m) / T)) and the chunk's best kc by (logit desc, id asc).
template <bool TOPK, bool BF16>
__device__ __forceinline__ void chunk_pass(const TreeBuildPlan& p, const BuildArgs& a) {
  const int bf = blockIdx.x, c = blockIdx.y;
  const int b = bf / a.F, f = bf % a.F;
  const int lo = c * kVocabChunk;
  const int hi = min(p.V, lo + kVocabChunk);
  const size_t row = static_cast<size_t>(bf) * p.V;
  const float invT = 1.f / (p.temperature > 0.f ? p.temperature : 1.f);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  __shared__ float sm[NW];
  __shared__ ff ss1[NW], ssT[NW];
  __shared__ float wlv[NW][K];
  __shared__ int wli[NW][K];
  __shared__ uint32_t wlk[NW][K];

  // all loads first
  float x[kPer];
  int xi[kPer];
  const bool vec = (reinterpret_cast<uintptr_t>(a.logits) & 15u) == 0 && (p.V % (BF16 ? 8 : 4)) == 0;
  load_chunk<BF16>(a.logits, row, lo, hi, vec, x, xi);
  // chunk max (two passes over registers: no online rescale)
  float m = x[0];
#pragma unroll
  for (int e = 1; e < kPer; ++e) m = fmaxf(m, x[e]);
  m = warp_max(m);
  if (lane == 0) sm[warp] = m;
  __syncthreads();
  float BM = sm[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) BM = fmaxf(BM, sm[w]);
  CSum s1, sT;
  if (BM != -INFINITY) {
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      s1.add(expf(x[e] - BM));
      if constexpr (!TOPK) sT.add(expf((x[e] - BM) * invT));  // the mass at T only feeds draws
    }
  }
  const ff d1 = warp_sum_ff(csum_ff(s1));
  const ff dT = TOPK ? d1 : warp_sum_ff(csum_ff(sT));
  if (lane == 0) {
    ss1[warp] = d1;
    ssT[warp] = dT;
  }
  ChunkPart* out = parts(p, a.ws) + (static_cast<size_t>(b) * p.f_max + f) * p.n_chunks + c;
  if constexpr (TOPK && BF16) {
    // bf16: one 32-bit key per logit, (order-preserving bf16 bits << 12) | (4095 -
    // offset in the chunk): a larger key is a larger logit, or an equal one with a
    // lower id; 0 = empty.  Each thread sorts its keys, each warp takes its best kc by
    // kc rounds of a warp max (redux) over the list heads, and the chunk's best kc of
    // the warp lists are found by rank, as on the fp32 path below.
    uint32_t key[K];
#pragma unroll
    for (int e = 0; e < kPer; ++e)
      key[e] = (xi[e] == INT_MAX) ? 0u : ((ord16(__float_as_uint(x[e]) >> 16) << 12) | (4095u - (xi[e] - lo)));
    sort_keys(key);
    const int kc = p.kc;
#pragma unroll 1
    for (int r = 0; r < kc; ++r) {
      const uint32_t best = __reduce_max_sync(0xffffffffu, key[0]);
      if (lane == 0) wlk[warp][r] = best;
      if (best != 0u && key[0] == best) {  // the owner pops its head
#pragma unroll
        for (int j = 0; j < K - 1; ++j) key[j] = key[j + 1];
        key[K - 1] = 0u;
      }
    }
    for (int r = kc + lane; r < K; r += 32) wlk[warp][r] = 0u;
    if (threadIdx.x < K) {
      out->tv[threadIdx.x] = -INFINITY;
      out->ti[threadIdx.x] = INT_MAX;
    }
  } else if constexpr (TOPK) {
    // each thread sorts its K logits; each warp takes its best kc by kc rounds of warp
    // argmax over the lanes' list heads (a level takes at most kc tokens of a row, so
    // at most kc of one chunk); the chunk's best kc of the NW warp lists are found by
    // rank: an entry's rank is the count of entries before it in every list.
    sort_regs(x, xi);
    const int kc = p.kc;
#pragma unroll 1
    for (int r = 0; r < kc; ++r) {
      float bv = x[0];
      int bi = xi[0];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
        const bool tk = before_nb(v2, i2, bv, bi);
        bv = tk ? v2 : bv;
        bi = tk ? i2 : bi;
      }
      if (lane == 0) {
        wlv[warp][r] = bv;
        wli[warp][r] = bi;
      }
      if (bi != INT_MAX && xi[0] == bi) {  // the owner pops its head
#pragma unroll
        for (int j = 0; j < K - 1; ++j) {
          x[j] = x[j + 1];
          xi[j] = xi[j + 1];
        }
        x[K - 1] = -INFINITY;
        xi[K - 1] = INT_MAX;
      }
    }
    for (int r = kc + lane; r < K; r += 32) {  // the warp list past kc: empty
      wlv[warp][r] = -INFINITY;
      wli[warp][r] = INT_MAX;
    }
    if (threadIdx.x < K) {  // slots no real entry reaches stay empty
      out->tv[threadIdx.x] = -INFINITY;
      out->ti[threadIdx.x] = INT_MAX;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    ff t1 = ff_make(0.f), tT = ff_make(0.f);
    for (int w = 0; w < NW; ++w) {
      t1 = ff_add(t1, ss1[w]);
      tT = ff_add(tT, ssT[w]);
    }
    out->m = BM;
    out->s1 = t1;
    out->sT = tT;
  }
  if constexpr (TOPK && BF16) {
    if (threadIdx.x < NW * K) {
      const int w0 = threadIdx.x / K, r0 = threadIdx.x % K;
      const uint32_t ck = wlk[w0][r0];
      if (ck != 0u) {
        int rank = r0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          int n = 0;  // keys of list w above ck: binary search of a descending list
#pragma unroll
          for (int step = K / 2; step > 0; step >>= 1) n += (wlk[w][n + step - 1] > ck) ? step : 0;
          n += (n == K - 1 && wlk[w][K - 1] > ck) ? 1 : 0;
          rank += (w == w0) ? 0 : n;
        }
        if (rank < p.kc) {
          out->tv[rank] = unord16(ck >> 12);
          out->ti[rank] = lo + 4095 - static_cast<int>(ck & 4095u);
        }
      }
    }
  } else if constexpr (TOPK) {
    if (threadIdx.x < NW * K) {
      const int w0 = threadIdx.x / K, r0 = threadIdx.x % K;
      const float cv = wlv[w0][r0];
      const int ci = wli[w0][r0];
      if (ci != INT_MAX) {
        int rank = r0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          int n = 0;  // entries of list w before (cv, ci): binary search of a sorted list
#pragma unroll
          for (int step = K / 2; step > 0; step >>= 1)
            n += before_nb(wlv[w][n + step - 1], wli[w][n + step - 1], cv, ci) ? step : 0;
          n += (n == K - 1 && before_nb(wlv[w][K - 1], wli[w][K - 1], cv, ci)) ? 1 : 0;
          rank += (w == w0) ? 0 : n;
        }
        if (rank < p.kc) {
          out->tv[rank] = cv;
          out->ti[rank] = ci;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ select helpers
// Exclusive ranks, in index order, of the entries of fr[0, n) that are non-zero:
// fr[i] becomes that rank, or -1 for a zero entry.  Block-wide; ends synchronised.
__device__ void block_flag_ranks(int* fr, int n, int* s_cnt) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int running = 0;
  for (int base = 0; base < n; base += kThreads) {
    const int i = base + threadIdx.x;
    const int fl = (i < n) ? fr[i] : 0;
    const unsigned bal = __ballot_sync(0xffffffffu, fl != 0);
    __syncthreads();  // readers of s_cnt from the previous chunk are done
    if (lane == 0) s_cnt[warp] = __popc(bal);
    __syncthreads();
    int off = running, tot = 0;
    for (int w = 0; w < NW; ++w) {
      if (w < warp) off += s_cnt[w];
      tot += s_cnt[w];
    }
    if (i < n) fr[i] = fl ? off + __popc(bal & ((1u << lane) - 1u)) : -1;
    running += tot;
  }
  __syncthreads();
}

// Float-float constants split on the host: hi = the nearest float, lo = the rest.
__host__ __device__ constexpr float split_hi(double d) { return static_cast<float>(d); }
__host__ __device__ constexpr float split_lo(double d) {
  return static_cast<float>(d - static_cast<double>(static_cast<float>(d)));
}
constexpr double kLn2 = 0.693147180559945309417232121458;


// ln z for a float-float z > 0 (finite, normal), as float-float, on the fp32 pipe.
// z = 2^k w with w in [1/sqrt 2, sqrt 2); ln z = k ln 2 + ln w and, with
// t = (w - 1) / (w + 1) (|t| < 0.172), ln w = 2 atanh t = 2 (t + t^3/3 + t^5/5 + ...);
// the series stops after t^17 (remainder below 1e-15 of ln w).
__device__ __forceinline__ ff ff_log(ff z) {
  // compile-time constants: they become instruction immediates, so the logarithm reads
  // no constant memory (whose first touch on an SM costs a round trip to L2)
  constexpr float kLogSeries[9][2] = {
      {split_hi(1.0), split_lo(1.0)},           {split_hi(1.0 / 3), split_lo(1.0 / 3)},
      {split_hi(1.0 / 5), split_lo(1.0 / 5)},   {split_hi(1.0 / 7), split_lo(1.0 / 7)},
      {split_hi(1.0 / 9), split_lo(1.0 / 9)},   {split_hi(1.0 / 11), split_lo(1.0 / 11)},
      {split_hi(1.0 / 13), split_lo(1.0 / 13)}, {split_hi(1.0 / 15), split_lo(1.0 / 15)},
      {split_hi(1.0 / 17), split_lo(1.0 / 17)}};
  constexpr float kLn2Split[2] = {split_hi(kLn2), split_lo(kLn2)};
  int e;
  float w_hi = frexpf(z.hi, &e);  // z.hi = w_hi 2^e, w_hi in [0.5, 1)
  int k = e;
  if (w_hi < 0.70710678f) {
    w_hi *= 2.f;
    k -= 1;
  }
  const ff w = ff{w_hi, ldexpf(z.lo, -k)};
  const ff t = ff_div(ff_add(w, -1.f), ff_add(w, 1.f));
  const ff t2 = ff_mul(t, t);
  ff sum = ff{kLogSeries[8][0], kLogSeries[8][1]};
#pragma unroll
  for (int i = 7; i >= 0; --i) sum = ff_add(ff_mul(sum, t2), ff{kLogSeries[i][0], kLogSeries[i][1]});
  const ff lnw = ff_mul(ff_mul(t, sum), 2.f);
  return ff_add(ff_mul(ff{kLn2Split[0], kLn2Split[1]}, static_cast<float>(k)), lnw);
}

// Row statistics merged over chunks by one warp: M, ln Z (T = 1) and the mass at
// temperature T (for draws), as float-float.
struct RowStats {
  float M;
  ff lnZ1, WT;
};

__device__ RowStats row_stats(const ChunkPart* cp, int n_chunks, float invT) {
  float M = -INFINITY;
  for (int c = threadIdx.x & 31; c < n_chunks; c += 32) M = fmaxf(M, cp[c].m);
  M = warp_max(M);
  ff z1 = ff_make(0.f), zT = ff_make(0.f);
  for (int c = threadIdx.x & 31; c < n_chunks; c += 32) {
    const ChunkPart& q = cp[c];
    if (q.m == -INFINITY) continue;
    z1 = ff_add(z1, ff_mul(q.s1, expf(q.m - M)));
    zT = ff_add(zT, ff_mul(q.sT, expf((q.m - M) * invT)));
  }
  RowStats r;
  r.M = M;
  r.lnZ1 = ff_log(warp_sum_ff(z1));
  r.WT = warp_sum_ff(zT);
  return r;
}

// ln q(t) = (x_t - M) - ln Z for a logit x_t of the row (x - M exact as float-float).
__device__ __forceinline__ ff log_q(float x, const RowStats& rs) { return ff_sub(two_sum(x, -rs.M), rs.lnZ1); }

// Warp merge of the chunks' top-K lists: writes the best `cnt` (token ids) to tok[].
__device__ void merge_topk(const ChunkPart* cp, int n_chunks, int cnt, int* tok, float* val) {
  const int lane = threadIdx.x & 31;
  if (n_chunks <= 32) {
    // lane c holds chunk c's whole list in registers (read once, 16-byte vectors)
    float lv[K];
    int li[K];
    if (lane < n_chunks) {
      const float4* pv = reinterpret_cast<const float4*>(cp[lane].tv);
      const int4* pi = reinterpret_cast<const int4*>(cp[lane].ti);
#pragma unroll
      for (int q = 0; q < K / 4; ++q) {
        const float4 v = pv[q];
        const int4 i = pi[q];
        lv[4 * q] = v.x;
        lv[4 * q + 1] = v.y;
        lv[4 * q + 2] = v.z;
        lv[4 * q + 3] = v.w;
        li[4 * q] = i.x;
        li[4 * q + 1] = i.y;
        li[4 * q + 2] = i.z;
        li[4 * q + 3] = i.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < K; ++j) {
        lv[j] = -INFINITY;
        li[j] = INT_MAX;
      }
    }
    for (int r = 0; r < cnt; ++r) {
      // the best head: the largest value (warp max of its order-preserving image), then
      // among equal values the lowest id
      const uint32_t kv = ord32(lv[0]);
      const uint32_t best = __reduce_max_sync(0xffffffffu, kv);
      const uint32_t bid = __reduce_min_sync(0xffffffffu, kv == best ? static_cast<uint32_t>(li[0]) : 0xffffffffu);
      const int bi = static_cast<int>(bid);
      if (lane == 0) {
        tok[r] = bi;
        val[r] = unord32(best);
      }
      if (bi != INT_MAX && kv == best && li[0] == bi) {  // the owner pops its head
#pragma unroll
        for (int j = 0; j < K - 1; ++j) {
          lv[j] = lv[j + 1];
          li[j] = li[j + 1];
        }
        lv[K - 1] = -INFINITY;
        li[K - 1] = INT_MAX;
      }
    }
    __syncwarp();
    return;
  }
  int head[5] = {0, 0, 0, 0, 0};  // per owned chunk (lane, lane+32, ...): up to 160 chunks
  for (int r = 0; r < cnt; ++r) {
    float bv = -INFINITY;
    int bi = INT_MAX, bslot = -1;
#pragma unroll
    for (int s = 0; s < 5; ++s) {
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

__device__ __forceinline__ ff ff_shfl(ff v, int src) {
  return ff{__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}
__device__ __forceinline__ ff ff_shfl_up(ff v, int o) {
  return ff{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}

// Warp inclusive scan of a float-float value over the lanes.
__device__ __forceinline__ ff warp_incl_scan(ff v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff t = ff_shfl_up(v, o);
    if (lane >= o) v = ff_add(v, t);
  }
  return v;
}

// Warp inverse-CDF draw over one logit row with weights w_v = exp((x_v - M) / T): the
// smallest v whose running mass exceeds u W.  Three warp-parallel levels, each a scan over
// the lanes with float-float sums: the chunk masses (32 chunks at a time) pick the
// 4096-token chunk; 32 runs of <= 128 tokens of that chunk pick the run; 32 groups of <= 4
// tokens of that run pick the group, whose lane finds the token.  The levels add the same
// weights in different orders, which moves a sum by about 1e-14 of it; a draw that close to
// an edge is flagged near anyway.  Returns the token; *near = 1 when u W lies
// within 1e-7 W of an edge of the chosen bin, or when no bin crosses (rounding: the last
// token with positive weight is taken).
__device__ int warp_draw(const void* logits, size_t row, int dtype, int V, const ChunkPart* cp, int n_chunks, float M,
                         float invT, ff W, float u, int* near) {
  const int lane = threadIdx.x & 31;
  const ff target = ff_mul(W, u);
  auto wt = [&](int v) { return expf((load_elem(logits, row + v, dtype) - M) * invT); };
  auto group4 = [&](int g0, int g1) {  // mass of tokens [g0, g1), g1 - g0 <= 4, in order
    ff m = ff_make(0.f);
#pragma unroll
    for (int k = 0; k < 4; ++k) m = ff_add(m, (g0 + k < g1) ? wt(g0 + k) : 0.f);
    return m;
  };
  // level 1: the chunk
  int cstar = -1, last_chunk = -1;
  ff base = ff_make(0.f), run = ff_make(0.f);
  for (int c0 = 0; c0 < n_chunks; c0 += 32) {
    const int c = c0 + lane;
    const ff w = (c < n_chunks && cp[c].m != -INFINITY) ? ff_mul(cp[c].sT, expf((cp[c].m - M) * invT)) : ff_make(0.f);
    const ff incl = ff_add(run, warp_incl_scan(w));
    const unsigned pos = __ballot_sync(0xffffffffu, w.hi > 0.f);
    if (pos) last_chunk = c0 + 31 - __clz(pos);
    const unsigned cross = __ballot_sync(0xffffffffu, c < n_chunks && ff_gt(incl, target));
    if (cross) {
      const int src = __ffs(cross) - 1;
      cstar = c0 + src;
      base = ff_shfl(ff_sub(incl, w), src);
      break;
    }
    run = ff_shfl(incl, 31);
  }
  bool fallback = cstar < 0;
  if (fallback) cstar = last_chunk < 0 ? 0 : last_chunk;
  const int lo = cstar * kVocabChunk, hi = min(V, lo + kVocabChunk);
  // level 2: 32 runs of 128 tokens (32 groups of 4 each)
  const int r0 = min(hi, lo + 128 * lane), r1 = min(hi, r0 + 128);
  ff acc[4] = {ff_make(0.f), ff_make(0.f), ff_make(0.f), ff_make(0.f)};  // four chains of groups
#pragma unroll 4
  for (int q = 0; q < 32; ++q) {
    const int g = r0 + 4 * q;
    if (g < r1) acc[q & 3] = ff_add(acc[q & 3], group4(g, min(r1, g + 4)));
  }
  const ff my = ff_add(ff_add(acc[0], acc[1]), ff_add(acc[2], acc[3]));
  const ff incl2 = ff_add(base, warp_incl_scan(my));
  const unsigned cross2 = fallback ? 0u : __ballot_sync(0xffffffffu, my.hi > 0.f && ff_gt(incl2, target));
  int tok = -1, nr = 0;
  if (cross2) {
    const int src = __ffs(cross2) - 1;
    const ff rbase = ff_shfl(ff_sub(incl2, my), src);  // mass before the run
    // level 3: the run's 32 groups of 4
    const int s0 = lo + 128 * src, s1 = min(hi, s0 + 128);
    const int g0 = min(s1, s0 + 4 * lane), g1 = min(s1, g0 + 4);
    const ff gm = group4(g0, g1);
    const ff incl3 = ff_add(rbase, warp_incl_scan(gm));
    const unsigned cross3 = __ballot_sync(0xffffffffu, gm.hi > 0.f && ff_gt(incl3, target));
    if (cross3) {
      const int src3 = __ffs(cross3) - 1;
      int found = -1;
      ff pe = ff_make(0.f), ne = ff_make(0.f);
      if (lane == src3) {
        ff cum = ff_sub(incl3, gm);
        for (int v = g0; v < g1; ++v) {
          const float w = wt(v);
          const ff nc = ff_add(cum, w);
          if (found < 0 && w > 0.f && ff_gt(nc, target)) {
            found = v;
            pe = cum;
            ne = nc;
          }
          cum = nc;
        }
      }
      found = __shfl_sync(0xffffffffu, found, src3);
      pe = ff_shfl(pe, src3);
      ne = ff_shfl(ne, src3);
      if (found >= 0) {
        tok = found;
        const float win = kIcdfNearEps * ff_float(W);
        nr = (ff_float(ff_sub(target, pe)) < win || ff_float(ff_sub(ne, target)) < win) ? 1 : 0;
      }
    }
  }
  if (tok < 0) {  // nothing crosses (rounding): the last token of the chunk with positive weight
    int last = -1;
    for (int v = r0; v < r1; ++v)
      if (wt(v) > 0.f) last = v;
    const unsigned bl = __ballot_sync(0xffffffffu, last >= 0);
    tok = bl ? __shfl_sync(0xffffffffu, last, 31 - __clz(bl)) : lo;
    nr = 1;
  }
  *near = nr;
  return tok;
}

// ------------------------------------------------------------------ the level's finishers
// The CTAs of a level finish in any order.  The last chunk CTA of a frontier row (an
// atomic ticket per row) merges that row's chunk records; the last row to finish in a
// request (a ticket per request) selects the request's next frontier and, at the last
// level, writes the tree.  Nobody waits for anybody: a CTA that is not last returns.
// Records written in the same launch by other CTAs are read from L2 (ld.global.cg)
// after the ticket, never through this SM's L1.

// Pool entries before level `level` of a dynamic tree: level 1 adds k, every later
// level k * k.
__device__ __forceinline__ int pool_base(const TreeBuildPlan& p, int level) {
  return level == 1 ? 0 : p.k + (level - 2) * p.k * p.k;
}

// Workspace views of one request.
struct ReqView {
  int32_t* state;   // [1] near-ties so far (zeroed before level 1)
  int32_t* ptok;    // dynamic pool: token, parent pool index, score, depth
  int32_t* ppar;
  ff* psc;
  int32_t* pdep;
  int32_t* front;   // pool index of each frontier slot
  ff* fsc;          // and its score
  int32_t* ntok;    // static shape: node tokens and scores
  ff* nsc;
};

__device__ __forceinline__ ReqView req_view(const TreeBuildPlan& p, uint8_t* ws, int b) {
  ReqView v;
  v.state = reinterpret_cast<int32_t*>(ws + p.off_state) + b * 4;
  const size_t pc = static_cast<size_t>(b) * p.pool_cap;
  v.ptok = reinterpret_cast<int32_t*>(ws + p.off_pool_tok) + pc;
  v.ppar = reinterpret_cast<int32_t*>(ws + p.off_pool_par) + pc;
  v.psc = reinterpret_cast<ff*>(ws + p.off_pool_score) + pc;
  v.pdep = reinterpret_cast<int32_t*>(ws + p.off_pool_depth) + pc;
  v.front = reinterpret_cast<int32_t*>(ws + p.off_front) + static_cast<size_t>(b) * K;
  v.fsc = reinterpret_cast<ff*>(ws + p.off_front_score) + static_cast<size_t>(b) * K;
  v.ntok = reinterpret_cast<int32_t*>(ws + p.off_node_tok) + static_cast<size_t>(b) * p.R;
  v.nsc = reinterpret_cast<ff*>(ws + p.off_node_score) + static_cast<size_t>(b) * p.R;
  return v;
}

// Device-scope acquire-release fetch-and-add (a ticket).
__device__ __forceinline__ int atom_add_acq_rel(int* ptr, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(ptr), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ ff ldcg_ff(const ff* q) {
  const float2 v = __ldcg(reinterpret_cast<const float2*>(q));
  return ff{v.x, v.y};
}

// The finishers' shared memory: a row's chunk records while a row is merged, then the
// request's selection arrays.
constexpr int kFinParts = (kMaxTreeChunks > kHeadRecords ? kMaxTreeChunks : kHeadRecords) * static_cast<int>(sizeof(ChunkPart));
constexpr int kFinSelect = (2 * kThreads + 2 * kMaxRows) * 8 + (kThreads + 2 * kMaxRows + kMaxPool) * 4;
constexpr int kFinBytes = kFinParts > kFinSelect ? kFinParts : kFinSelect;

// Copies the row's chunk records from L2 into shared memory (the whole CTA).
__device__ void stage_parts(const ChunkPart* g, ChunkPart* sp, int n_chunks) {
  const uint4* src = reinterpret_cast<const uint4*>(g);
  uint4* dst = reinterpret_cast<uint4*>(sp);
  const int n = n_chunks * static_cast<int>(sizeof(ChunkPart) / 16);
  for (int i = threadIdx.x; i < n; i += kThreads) dst[i] = __ldcg(src + i);
  __syncthreads();
}

// Dynamic tree, frontier row f of request b: the row's statistics (warp 0) and top-k
// (warp 1) from its chunk records, then its k candidates join the pool with
// score s_parent + ln q(t).
__device__ __forceinline__ void finish_row_dynamic(const TreeBuildPlan& p, const BuildArgs& a, int b, int f,
                                                uint8_t* s_fin) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ int stok[K];
  __shared__ float sval[K];
  ChunkPart* sp = reinterpret_cast<ChunkPart*>(s_fin);
  const ReqView v = req_view(p, a.ws, b);
  // the parent (written by the previous level), loaded while the records are staged
  const int pidx = (a.level == 1) ? -1 : __ldcg(v.front + f);
  const ff sp_score = (a.level == 1) ? ff_make(0.f) : ldcg_ff(v.fsc + f);
  stage_parts(parts(p, a.ws) + (static_cast<size_t>(b) * p.f_max + f) * p.n_chunks, sp, p.n_chunks);
  RowStats rs;
  if (warp == 0) rs = row_stats(sp, p.n_chunks, 1.f);
  if (warp == 1) merge_topk(sp, p.n_chunks, p.k, stok, sval);
  __syncthreads();
  if (warp == 0 && lane < p.k) {
    const int i = pool_base(p, a.level) + f * p.k + lane;
    v.ptok[i] = stok[lane];
    v.ppar[i] = pidx;
    v.psc[i] = ff_add(sp_score, log_q(sval[lane], rs));
    v.pdep[i] = a.level;
  }
}

// Static shape, frontier row f (the f-th node n of depth level - 1): the children of n
// are its best tokens in rank order (top-k) or draws from softmax(row / T), one warp per
// child; node scores are s_n + ln q(t) at T = 1.
__device__ __forceinline__ void finish_row_static(const TreeBuildPlan& p, const BuildArgs& a, int b, int f,
                                               uint8_t* s_fin) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool sampled = p.mode == EAGLE_TREE_STATIC_SAMPLED;
  const float invT = 1.f / (p.temperature > 0.f ? p.temperature : 1.f);
  __shared__ int stok[K];
  __shared__ float sval[K];
  __shared__ RowStats s_rs;
  int n = -1;
  for (int i = 0; i < p.R; ++i)
    if (p.shape.depth[i] == a.level - 1 && p.shape.lrank[i] == f) {
      n = i;
      break;
    }
  int kids = 0;
  for (int i = n + 1; n >= 0 && i < p.R; ++i) kids += (p.shape.parent[i] == n);
  if (kids == 0) return;  // uniform over the CTA
  ChunkPart* sp = reinterpret_cast<ChunkPart*>(s_fin);
  stage_parts(parts(p, a.ws) + (static_cast<size_t>(b) * p.f_max + f) * p.n_chunks, sp, p.n_chunks);
  const ReqView v = req_view(p, a.ws, b);
  if (warp == 0) {
    const RowStats rs = row_stats(sp, p.n_chunks, invT);
    if (lane == 0) s_rs = rs;
  }
  if (warp == 1 && !sampled) merge_topk(sp, p.n_chunks, kids, stok, sval);
  __syncthreads();
  const RowStats rs = s_rs;
  const size_t row = (static_cast<size_t>(b) * a.F + f) * p.V;
  const ff s_par = (n == 0) ? ff_make(0.f) : ldcg_ff(v.nsc + n);
  int near_local = 0, j = 0;
  for (int ch = n + 1; ch < p.R; ++ch) {
    if (p.shape.parent[ch] != n) continue;
    if ((j++ % NW) != warp) continue;
    int tok;
    float x;  // the token's logit
    if (!sampled) {
      tok = stok[j - 1];
      x = sval[j - 1];
    } else {
      int nr = 0;
      tok = warp_draw(a.logits, row, p.dtype, p.V, sp, p.n_chunks, rs.M, invT, rs.WT,
                      a.u_draft[static_cast<size_t>(b) * p.R + ch], &nr);
      near_local += nr;
      x = load_elem(a.logits, row + tok, p.dtype);
    }
    if (lane == 0) {
      v.ntok[ch] = tok;
      v.nsc[ch] = ff_add(s_par, log_q(x, rs));
    }
  }
  if (lane == 0 && near_local) atomicAdd(v.state + 1, near_local);
}

// Ancestor masks: row i has bits i and those of its ancestors (each row walks up the
// parent chain; parents come first, so at most R steps).
__device__ void write_masks(const TreeBuildPlan& p, const BuildArgs& a, int b, const int* spar) {
  const size_t mb = static_cast<size_t>(b) * p.R;
  for (int i = threadIdx.x; i < p.R; i += kThreads) {
    uint64_t w0 = 0, w1 = 0;
    int j = i;
    for (int steps = 0; j >= 0 && steps < p.R; ++steps) {
      if (j < 64)
        w0 |= 1ull << j;
      else
        w1 |= 1ull << (j - 64);
      j = spar[j];
    }
    a.out.anc_mask[(mb + i) * p.W] = w0;
    if (p.W > 1) a.out.anc_mask[(mb + i) * p.W + 1] = w1;
  }
}

// The order of pool entries as one 64-bit key: (score desc) as the float-float pair's
// order-preserving images, high part first (the pairs are normalised, so this is the
// order of their values); ties go to the lower pool index.
__device__ __forceinline__ uint64_t score_key(ff s) {
  return (static_cast<uint64_t>(ord32(s.hi)) << 32) | ord32(s.lo);
}

__device__ __forceinline__ ff key_score(uint64_t key) {
  return ff{unord32(static_cast<uint32_t>(key >> 32)), unord32(static_cast<uint32_t>(key))};
}

// Leading entries of a descending list (key, index) that come before (x, ix).
__device__ __forceinline__ int count_before(const uint64_t* key, const int* idx, int n, uint64_t x, int ix) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (key[mid] > x || (key[mid] == x && idx[mid] < ix))
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
}

// Dynamic tree, request b, after all its rows: the next frontier is the best k of the
// level's F k candidates (kept in pool order).  The request also keeps, from level to
// level, the best N + 1 entries of the pool so far as a sorted list (the level's
// candidates, ranked, are merged into it), so that after the last level the best N of
// the pool, in pool order, form the tree without sorting the whole pool.
__device__ __forceinline__ void finish_request_dynamic(const TreeBuildPlan& p, const BuildArgs& a, int b,
                                                       uint8_t* s_fin) {
  // shared memory: the level's candidates, the incoming and outgoing best lists, flags
  uint64_t* ck = reinterpret_cast<uint64_t*>(s_fin);      // [256] candidate keys, by candidate
  uint64_t* bk = ck + kThreads;                            // [256] candidate keys, by rank
  uint64_t* lk = bk + kThreads;                            // [128] best list in
  uint64_t* nk = lk + kMaxRows;                            // [128] best list out
  int* bi = reinterpret_cast<int*>(nk + kMaxRows);         // [256] pool index, by rank
  int* li = bi + kThreads;                                 // [128]
  int* ni = li + kMaxRows;                                 // [128]
  int* srow = ni + kMaxRows;                               // [kMaxPool] flags / parents
  __shared__ int s_cnt[NW];
  __shared__ int s_bnd[2];
  __shared__ int spar[kMaxRows];
  const ReqView v = req_view(p, a.ws, b);
  ff* best_sc = reinterpret_cast<ff*>(a.ws + p.off_best_score) + static_cast<size_t>(b) * kMaxRows;
  int32_t* best_ix = reinterpret_cast<int32_t*>(a.ws + p.off_best_idx) + static_cast<size_t>(b) * kMaxRows;
  const int base = pool_base(p, a.level);
  const int k = p.k;
  const int n_new = a.F * k;  // <= 256 = kThreads: one candidate per thread
  const int M = p.N + 1;      // the best list: the N kept and the first dropped
  const int nA = base < M ? base : M;
  const int nL = (base + n_new) < M ? base + n_new : M;
  const int j = threadIdx.x;
  // every load of the level at once: the candidates (written by the row finishers) and
  // the best list (written by the previous level)
  ff kj = ff_make(-INFINITY);
  int tj = 0, pj = 0;
  if (j < n_new) {
    kj = ldcg_ff(v.psc + base + j);
    tj = __ldcg(v.ptok + base + j);
    pj = __ldcg(v.ppar + base + j);
  }
  ff la = ff_make(-INFINITY);
  int lix = 0;
  if (j < nA) {
    la = ldcg_ff(best_sc + j);
    lix = __ldcg(best_ix + j);
    lk[j] = score_key(la);
    li[j] = lix;
  }
  const uint64_t kkey = score_key(kj);
  if (j < n_new) {
    ck[j] = kkey;
    srow[j] = pj;
  }
  __syncthreads();
  // a candidate's rank among the level's: the candidates before it by (score desc,
  // pool index asc)
  int r = n_new;
  if (j < n_new) {
    r = 0;
    int i = 0;
    for (; i + 4 <= n_new; i += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint64_t ki = ck[i + u];
        r += (ki > kkey || (ki == kkey && i + u < j)) ? 1 : 0;
      }
    }
    for (; i < n_new; ++i) r += (ck[i] > kkey || (ck[i] == kkey && i < j)) ? 1 : 0;
    bk[r] = kkey;
    bi[r] = base + j;
    if (r == k - 1 || r == k) s_bnd[r - (k - 1)] = j;  // the two candidates at the boundary
  }
  __syncthreads();
  // a near-tie at the frontier boundary, unless it is an exact tie between siblings (same
  // parent, same logit), which both sides break by pool index
  if (threadIdx.x == 0 && n_new > k) {
    const int ja = s_bnd[0], jb = s_bnd[1];
    if (ff_float(ff_sub(key_score(ck[ja]), key_score(ck[jb]))) < kNearTieEps &&
        !(ck[ja] == ck[jb] && srow[ja] == srow[jb]))
      atomicAdd(v.state + 1, 1);
  }
  // the merged best list: an entry's position is its rank in its own list plus the
  // entries of the other list before it
  if (j < nA) {
    const int pos = j + count_before(bk, bi, n_new, lk[j], lix);
    if (pos < M) {
      nk[pos] = lk[j];
      ni[pos] = lix;
      best_sc[pos] = la;
      best_ix[pos] = lix;
    }
  }
  if (j < n_new) {
    const int pos = r + count_before(lk, li, nA, kkey, base + j);
    if (pos < M) {
      nk[pos] = kkey;
      ni[pos] = base + j;
      best_sc[pos] = kj;
      best_ix[pos] = base + j;
    }
  }
  __syncthreads();
  if (j < n_new) srow[j] = r < k ? 1 : 0;
  block_flag_ranks(srow, n_new, s_cnt);
  if (j < n_new && srow[j] >= 0) {
    const int slot = srow[j];
    v.front[slot] = base + j;
    v.fsc[slot] = kj;
    a.out.frontier_tok[static_cast<size_t>(b) * p.f_max + slot] = tj;
    a.out.frontier_slot[static_cast<size_t>(b) * p.f_max + slot] = j / k;
  }
  __syncthreads();
  if (a.level != p.depth) return;

  // ---- last level: the best N of the pool, rows in pool order
  const int np = base + n_new;
  const int N = p.N;
  if (threadIdx.x == 0 && np > N) {  // the selection boundary: the N-th and the first dropped
    const int ia = ni[N - 1], ib = ni[N];
    if (ff_float(ff_sub(key_score(nk[N - 1]), key_score(nk[N]))) < kNearTieEps &&
        !(nk[N - 1] == nk[N] && __ldcg(v.ppar + ia) == __ldcg(v.ppar + ib)))
      atomicAdd(v.state + 1, 1);
  }
  for (int jj = threadIdx.x; jj < np; jj += kThreads) srow[jj] = 0;
  __syncthreads();
  for (int jj = threadIdx.x; jj < N && jj < nL; jj += kThreads) srow[ni[jj]] = 1;
  __syncthreads();
  block_flag_ranks(srow, np, s_cnt);  // row of a selected pool entry = its rank + 1
  const size_t ob = static_cast<size_t>(b) * p.R;
  const int L = a.seq_len[b];
  for (int jj = threadIdx.x; jj < np; jj += kThreads) {
    if (srow[jj] < 0) continue;
    const int pp = __ldcg(v.ppar + jj), dep = __ldcg(v.pdep + jj), tok = __ldcg(v.ptok + jj);
    const ff sc = ldcg_ff(v.psc + jj);
    const int rr = srow[jj] + 1;
    const int pr = (pp < 0) ? 0 : (srow[pp] >= 0 ? srow[pp] + 1 : 0);
    spar[rr] = pr;
    a.out.tokens[ob + rr] = tok;
    a.out.parent[ob + rr] = pr;
    a.out.depth[ob + rr] = dep;
    a.out.pos_id[ob + rr] = L + dep;
    a.out.score[ob + rr] = ff_float(sc);
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
  write_masks(p, a, b, spar);
  __syncthreads();
  if (threadIdx.x == 0) a.out.near_tie[b] = atomicAdd(v.state + 1, 0);
}

// Static shape, request b, after all its rows: the next frontier is the nodes of depth
// `level` in index order; after the last level the tree arrays.
__device__ __forceinline__ void finish_request_static(const TreeBuildPlan& p, const BuildArgs& a, int b) {
  __shared__ int spar[kMaxRows];
  const ReqView v = req_view(p, a.ws, b);
  for (int i = threadIdx.x; i < p.R; i += kThreads) {
    if (p.shape.depth[i] != a.level) continue;
    const int slot = p.shape.lrank[i];
    a.out.frontier_tok[static_cast<size_t>(b) * p.f_max + slot] = __ldcg(v.ntok + i);
    a.out.frontier_slot[static_cast<size_t>(b) * p.f_max + slot] = p.shape.lrank[p.shape.parent[i]];
  }
  if (a.level != p.depth) return;
  const size_t ob = static_cast<size_t>(b) * p.R;
  const int L = a.seq_len[b];
  for (int i = threadIdx.x; i < p.R; i += kThreads) {
    spar[i] = p.shape.parent[i];
    a.out.tokens[ob + i] = (i == 0) ? a.root_tok[b] : __ldcg(v.ntok + i);
    a.out.parent[ob + i] = p.shape.parent[i];
    a.out.depth[ob + i] = p.shape.depth[i];
    a.out.pos_id[ob + i] = L + p.shape.depth[i];
    a.out.score[ob + i] = (i == 0) ? 0.f : ff_float(ldcg_ff(v.nsc + i));
  }
  __syncthreads();
  write_masks(p, a, b, spar);
  if (threadIdx.x == 0) a.out.near_tie[b] = atomicAdd(v.state + 1, 0);
}

// A frontier row's finisher, then (by the request ticket) the request's.  The tree mode
// is a template argument: the finishers run once per level from a cold instruction
// cache, so each kernel carries only its own mode's code.
template <bool DYN>
__device__ __forceinline__ void finish_row_and_request(const TreeBuildPlan& p, const BuildArgs& a, int b, int f,
                                                       uint8_t* s_fin, int* req_ticket, int* s_ticket) {
  if constexpr (DYN)
    finish_row_dynamic(p, a, b, f, s_fin);
  else
    finish_row_static(p, a, b, f, s_fin);
  __syncthreads();
  if (threadIdx.x == 0) *s_ticket = atom_add_acq_rel(req_ticket, 1);
  __syncthreads();
  if (*s_ticket != a.F - 1) return;
  if constexpr (DYN)
    finish_request_dynamic(p, a, b, s_fin);
  else
    finish_request_static(p, a, b);
  if (threadIdx.x == 0) *req_ticket = 0;  // ready for the next level
}

// ------------------------------------------------------------------ one draft level
// One CTA per (request x frontier row, 4096-token chunk): the chunk pass, then the
// tickets: the row's last chunk CTA merges the row, the request's last row selects.
template <bool TOPK, bool BF16, bool DYN>
__global__ void __launch_bounds__(kThreads, 2)
    tree_level_kernel(const TreeBuildPlan p, const BuildArgs a) {
  __shared__ __align__(16) uint8_t s_fin[kFinBytes];
  __shared__ int s_ticket;
  chunk_pass<TOPK, BF16>(p, a);
  const int b = blockIdx.x / a.F, f = blockIdx.x % a.F;
  int* row_ticket = reinterpret_cast<int*>(a.ws + p.off_ticket) + b * p.f_max + f;
  int* req_ticket = reinterpret_cast<int*>(a.ws + p.off_ticket) + p.B * p.f_max + b;
  // the ticket: the barrier orders the CTA's record writes before thread 0's atomic,
  // whose release makes them visible with it at device scope and whose acquire orders
  // the last CTA's reads of the other CTAs' records after it
  __syncthreads();
  if (threadIdx.x == 0) s_ticket = atom_add_acq_rel(row_ticket, 1);
  __syncthreads();
  if (s_ticket != p.n_chunks - 1) return;
  if (threadIdx.x == 0) *row_ticket = 0;  // ready for the next level
  finish_row_and_request<DYN>(p, a, b, f, s_fin, req_ticket, &s_ticket);
}

// The finishers of a level whose records the LM-head kernel wrote (kHeadRecords per
// row): one CTA per (request, frontier row) merges its row, the request's last selects.
template <bool DYN>
__global__ void __launch_bounds__(kThreads, 1) tree_head_finish_kernel(const TreeBuildPlan p, const BuildArgs a) {
  __shared__ __align__(16) uint8_t s_fin[kFinBytes];
  __shared__ int s_ticket;
  const int b = blockIdx.x / a.F, f = blockIdx.x % a.F;
  int* req_ticket = reinterpret_cast<int*>(a.ws + p.off_ticket) + p.B * p.f_max + b;
  finish_row_and_request<DYN>(p, a, b, f, s_fin, req_ticket, &s_ticket);
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
    p->kc = d->top_k;
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
    int seen[kMaxRows] = {0};
    for (int i = 0; i < p->R && i < kMaxRows; ++i) p->shape.lrank[i] = static_cast<uint8_t>(seen[p->shape.depth[i]]++);
    int fmax = 1;
    for (int dd = 0; dd <= maxd; ++dd) {
      int c = 0;
      for (int i = 0; i < p->R; ++i) c += (p->shape.depth[i] == dd);
      if (c > fmax) fmax = c;
    }
    p->f_max = fmax;
    int kmax = 1;  // most children of one node
    for (int i = 0; i < p->R; ++i) {
      int c = 0;
      for (int j = i + 1; j < p->R; ++j) c += (p->shape.parent[j] == i);
      if (c > kmax) kmax = c;
    }
    p->kc = kmax < K ? kmax : K;
  }
  p->W = (p->R + 63) / 64;
  size_t off = 0;
  const size_t cap = static_cast<size_t>(p->B) * (p->pool_cap > 0 ? p->pool_cap : 1);
  p->off_pool_tok = off;
  off = align256(off + cap * 4);
  p->off_pool_par = off;
  off = align256(off + cap * 4);
  p->off_pool_score = off;
  off = align256(off + cap * sizeof(ff));
  p->off_pool_depth = off;
  off = align256(off + cap * 4);
  p->off_state = off;  // state [B][4], then the row tickets [B][f_max] and request tickets [B]
  off += static_cast<size_t>(p->B) * 4 * 4;
  p->off_ticket = off;
  off = align256(off + static_cast<size_t>(p->B) * (p->f_max + 1) * 4);
  p->off_front = off;
  off = align256(off + static_cast<size_t>(p->B) * K * 4);
  p->off_front_score = off;
  off = align256(off + static_cast<size_t>(p->B) * K * sizeof(ff));
  p->off_best_score = off;  // the best N + 1 of the pool so far, per request
  off = align256(off + static_cast<size_t>(p->B) * kMaxRows * sizeof(ff));
  p->off_best_idx = off;
  off = align256(off + static_cast<size_t>(p->B) * kMaxRows * 4);
  p->off_part = off;  // room for the chunk pass's records or the LM head's, whichever is more
  const int n_rec = p->n_chunks > kHeadRecords ? p->n_chunks : kHeadRecords;
  off = align256(off + static_cast<size_t>(p->B) * p->f_max * n_rec * sizeof(ChunkPart));
  p->off_node_tok = off;
  off = align256(off + static_cast<size_t>(p->B) * p->R * 4);
  p->off_node_score = off;
  off = align256(off + static_cast<size_t>(p->B) * p->R * sizeof(ff));
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
  if (level == 1) {  // a new build: zero the per-request state and the tickets
    const cudaError_t e = cudaMemsetAsync(a.ws + p.off_state, 0,
                                          p.off_ticket - p.off_state + static_cast<size_t>(p.B) * (p.f_max + 1) * 4, s);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(p.B * a.F, p.n_chunks);
  const bool bf16 = p.dtype != EAGLE_F32;
  if (p.mode == EAGLE_TREE_STATIC_SAMPLED) {
    if (bf16)
      tree_level_kernel<false, true, false><<<grid, kThreads, 0, s>>>(p, a);
    else
      tree_level_kernel<false, false, false><<<grid, kThreads, 0, s>>>(p, a);
  } else if (p.mode == EAGLE_TREE_DYNAMIC) {
    if (bf16)
      tree_level_kernel<true, true, true><<<grid, kThreads, 0, s>>>(p, a);
    else
      tree_level_kernel<true, false, true><<<grid, kThreads, 0, s>>>(p, a);
  } else {
    if (bf16)
      tree_level_kernel<true, true, false><<<grid, kThreads, 0, s>>>(p, a);
    else
      tree_level_kernel<true, false, false><<<grid, kThreads, 0, s>>>(p, a);
  }
  return cudaGetLastError();
}

cudaError_t launch_tree_build_head(const TreeBuildPlan& plan, int level, const void* hidden, const void* weight,
                                   int hidden_dim, const int32_t* root_tok, const int32_t* seq_len, void* ws,
                                   const eagle_tree& out, uint32_t* status, cudaStream_t s) {
  TreeBuildPlan p = plan;
  p.n_chunks = kHeadRecords;  // the finishers read the head kernel's records
  BuildArgs a;
  a.logits = nullptr;
  a.u_draft = nullptr;
  a.root_tok = root_tok;
  a.seq_len = seq_len;
  a.ws = static_cast<uint8_t*>(ws);
  a.out = out;
  a.level = level;
  a.F = frontier_rows(p, level);
  if (level == 1) {
    const cudaError_t e = cudaMemsetAsync(a.ws + p.off_state, 0,
                                          p.off_ticket - p.off_state + static_cast<size_t>(p.B) * (p.f_max + 1) * 4, s);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch_lmhead_tree_records(p.B * a.F, hidden_dim, p.V, a.F, p.f_max, kHeadRecords, hidden, weight,
                                             reinterpret_cast<TreeChunkRecord*>(a.ws + p.off_part), status, s);
  if (e != cudaSuccess) return e;
  if (p.mode == EAGLE_TREE_DYNAMIC)
    tree_head_finish_kernel<true><<<p.B * a.F, kThreads, 0, s>>>(p, a);
  else
    tree_head_finish_kernel<false><<<p.B * a.F, kThreads, 0, s>>>(p, a);
  return cudaGetLastError();
}

namespace {
// Evaluates the float-float logarithm on n inputs (one thread each).
__global__ void ff_log_selftest_kernel(const float* z_hi, const float* z_lo, float* out_hi, float* out_lo, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const ff r = ff_log(ff{z_hi[i], z_lo[i]});
  out_hi[i] = r.hi;
  out_lo[i] = r.lo;
}
}  // namespace

cudaError_t launch_ff_log_selftest(const float* z_hi, const float* z_lo, float* out_hi, float* out_lo, int n,
                                   cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  ff_log_selftest_kernel<<<(n + 255) / 256, 256, 0, s>>>(z_hi, z_lo, out_hi, out_lo, n);
  return cudaGetLastError();
}

}  // namespace eagle
