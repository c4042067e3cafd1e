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
//   tree_chunk_kernel   one CTA per (request x frontier row, 4096-token chunk): the
//                       chunk max, sum exp (T = 1 and T) and the chunk's top-16 by
//                       (logit desc, id asc), from one read of the logits held in
//                       registers (16 per thread).
//   tree_select_kernel  one CTA per request: merges the chunk results per row,
//                       extends the pool, picks the frontier (bitonic sort in shared
//                       memory) and, at the last level, emits the tree arrays.
//
// Precision: chunk sums are compensated fp32, merged as float-float (about 48
// significant bits on the fp32 pipe; this GPU's fp64 pipe is narrow), and ln Z is a
// float-float logarithm.  Cumulative scores are float-float, so that the selections
// agree with an fp64 computation unless two scores at a boundary are within 1e-5
// (reported as a near-tie).
#include <limits.h>

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

struct __align__(16) ChunkPart {
  float tv[K];    // top-K logits of the chunk, best first
  int ti[K];      // their token ids (INT_MAX = empty)
  ff s1;          // sum exp(x - m)
  ff sT;          // sum exp((x - m) / T)
  float m;        // chunk max logit
  float pad[3];
};
static_assert(sizeof(ChunkPart) % 16 == 0, "chunk lists are read as 16-byte vectors");

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

// Order of (value, id) pairs: best first.  Two float-float values compare as reals.
__device__ __forceinline__ bool ff_eq(ff a, ff b) { return a.hi == b.hi && a.lo == b.lo; }
__device__ __forceinline__ bool before_ff(ff va, int ia, ff vb, int ib) {
  return ff_gt(va, vb) || (ff_eq(va, vb) && ia < ib);
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
template <bool TOPK, bool BF16>
__global__ void __launch_bounds__(kThreads, 2) tree_chunk_kernel(const TreeBuildPlan p, const BuildArgs a) {
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
      sT.add(expf((x[e] - BM) * invT));
    }
  }
  const ff d1 = warp_sum_ff(csum_ff(s1));
  const ff dT = warp_sum_ff(csum_ff(sT));
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
// Block bitonic sort of n2 (power of two) entries, best first by (key desc, idx asc).
__device__ void bitonic_sort(ff* key, int* idx, int n2) {
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const bool up = (i & k) == 0;
          const ff ki = key[i], kj = key[ixj];
          const int ii = idx[i], ij = idx[ixj];
          const bool sw = up ? before_ff(kj, ij, ki, ii) : before_ff(ki, ii, kj, ij);
          if (sw) {
            key[i] = kj;
            key[ixj] = ki;
            idx[i] = ij;
            idx[ixj] = ii;
          }
        }
      }
      __syncthreads();
    }
  }
}

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
constexpr float split_hi(double d) { return static_cast<float>(d); }
constexpr float split_lo(double d) { return static_cast<float>(d - static_cast<double>(static_cast<float>(d))); }
constexpr double kLn2 = 0.693147180559945309417232121458;
__constant__ float kLogSeries[9][2] = {
    {split_hi(1.0), split_lo(1.0)},           {split_hi(1.0 / 3), split_lo(1.0 / 3)},
    {split_hi(1.0 / 5), split_lo(1.0 / 5)},   {split_hi(1.0 / 7), split_lo(1.0 / 7)},
    {split_hi(1.0 / 9), split_lo(1.0 / 9)},   {split_hi(1.0 / 11), split_lo(1.0 / 11)},
    {split_hi(1.0 / 13), split_lo(1.0 / 13)}, {split_hi(1.0 / 15), split_lo(1.0 / 15)},
    {split_hi(1.0 / 17), split_lo(1.0 / 17)}};
__constant__ float kLn2Split[2] = {split_hi(kLn2), split_lo(kLn2)};

// ln z for a float-float z > 0 (finite, normal), as float-float, on the fp32 pipe.
// z = 2^k w with w in [1/sqrt 2, sqrt 2); ln z = k ln 2 + ln w and, with
// t = (w - 1) / (w + 1) (|t| < 0.172), ln w = 2 atanh t = 2 (t + t^3/3 + t^5/5 + ...);
// the series stops after t^17 (remainder below 1e-15 of ln w).
__device__ __forceinline__ ff ff_log(ff z) {
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

__global__ void __launch_bounds__(kThreads, 1) tree_select_kernel(const TreeBuildPlan p, const BuildArgs a) {
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ws = a.ws;
  int32_t* state = reinterpret_cast<int32_t*>(ws + p.off_state) + b * 4;  // [0] n_pool, [1] near
  const ChunkPart* cps = parts(p, ws) + static_cast<size_t>(b) * p.f_max * p.n_chunks;
  const float invT = 1.f / (p.temperature > 0.f ? p.temperature : 1.f);

  __shared__ ff skey[kMaxPool];
  __shared__ int sidx[kMaxPool];
  __shared__ int srow[kMaxPool];
  __shared__ int stok[NW][K];
  __shared__ float sval[NW][K];
  __shared__ int s_cnt[NW];
  __shared__ int s_near;
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
    ff* psc = reinterpret_cast<ff*>(ws + p.off_pool_score) + static_cast<size_t>(b) * p.pool_cap;
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
      const ff spar_score = (pidx < 0) ? ff_make(0.f) : psc[pidx];
      if (lane < k) {
        const int i = base + f * k + lane;
        ptok[i] = stok[warp][lane];
        ppar[i] = pidx;
        psc[i] = ff_add(spar_score, log_q(sval[warp][lane], rs));
        pdep[i] = a.level;
      }
      __syncwarp();
    }
    __syncthreads();
    const int n_new = a.F * k;
    // next frontier: best k of the new candidates, kept in pool order.  A candidate's
    // rank is the number of candidates before it by (score desc, pool index asc).
    for (int j = threadIdx.x; j < n_new; j += kThreads) skey[j] = psc[base + j];
    __syncthreads();
    for (int j = threadIdx.x; j < n_new; j += kThreads) {
      const ff kj = skey[j];
      int r = 0;
      for (int i = 0; i < n_new; ++i) r += before_ff(skey[i], i, kj, j) ? 1 : 0;
      if (r == k - 1 || r == k) sidx[r - (k - 1)] = j;  // the two candidates at the boundary
      srow[j] = r < k ? 1 : 0;
    }
    __syncthreads();
    // a near-tie at the boundary, unless it is an exact tie between siblings (same
    // parent, same logit), which both sides break by pool index
    if (threadIdx.x == 0 && n_new > k) {
      const ff ka = skey[sidx[0]], kb = skey[sidx[1]];
      if (ff_float(ff_sub(ka, kb)) < kNearTieEps && !(ff_eq(ka, kb) && ppar[base + sidx[0]] == ppar[base + sidx[1]]))
        s_near += 1;
    }
    block_flag_ranks(srow, n_new, s_cnt);
    for (int j = threadIdx.x; j < n_new; j += kThreads) {
      const int slot = srow[j];
      if (slot < 0) continue;
      front[slot] = base + j;
      a.out.frontier_tok[static_cast<size_t>(b) * p.f_max + slot] = ptok[base + j];
      a.out.frontier_slot[static_cast<size_t>(b) * p.f_max + slot] = j / k;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      state[0] = base + n_new;
      state[1] += s_near;
      s_near = 0;
    }
    __syncthreads();
    if (a.level != p.depth) return;

    // ---- last level: best N of the pool, rows in pool order
    const int np = base + n_new;
    const int N = p.N;
    int n2 = 1;
    while (n2 < np) n2 <<= 1;
    for (int j = threadIdx.x; j < n2; j += kThreads) {
      skey[j] = j < np ? psc[j] : ff_make(-INFINITY);
      sidx[j] = j < np ? j : INT_MAX;
    }
    __syncthreads();
    bitonic_sort(skey, sidx, n2);
    if (threadIdx.x == 0 && np > N && ff_float(ff_sub(skey[N - 1], skey[N])) < kNearTieEps &&
        !(ff_eq(skey[N - 1], skey[N]) && ppar[sidx[N - 1]] == ppar[sidx[N]]))
      state[1] += 1;
    for (int j = threadIdx.x; j < np; j += kThreads) srow[j] = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < N; j += kThreads) srow[sidx[j]] = 1;
    __syncthreads();
    block_flag_ranks(srow, np, s_cnt);  // row of a selected pool entry = its rank + 1
    const size_t ob = static_cast<size_t>(b) * p.R;
    const int L = a.seq_len[b];
    for (int j = threadIdx.x; j < np; j += kThreads) {
      if (srow[j] < 0) continue;
      const int r = srow[j] + 1;
      const int pp = ppar[j];
      const int pr = (pp < 0) ? 0 : (srow[pp] >= 0 ? srow[pp] + 1 : 0);
      spar[r] = pr;
      a.out.tokens[ob + r] = ptok[j];
      a.out.parent[ob + r] = pr;
      a.out.depth[ob + r] = pdep[j];
      a.out.pos_id[ob + r] = L + pdep[j];
      a.out.score[ob + r] = ff_float(psc[j]);
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
    ff* nsc = reinterpret_cast<ff*>(ws + p.off_node_score) + static_cast<size_t>(b) * p.R;
    const bool sampled = p.mode == EAGLE_TREE_STATIC_SAMPLED;
    if (a.level == 1 && threadIdx.x == 0) {
      ntok[0] = a.root_tok[b];
      nsc[0] = ff_make(0.f);
    }
    __syncthreads();
    // frontier row f = the f-th node of depth level-1; one warp per row
    int near_local = 0;
    for (int f = warp; f < a.F; f += NW) {
      int n = -1;
      for (int i = 0; i < p.R; ++i)
        if (p.shape.depth[i] == a.level - 1 && p.shape.lrank[i] == f) {
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
          nsc[ch] = ff_add(nsc[n], log_q(load_elem(a.logits, row + tok, p.dtype), rs));
        }
        ++j;
      }
      __syncwarp();
    }
    if (lane == 0 && near_local) atomicAdd(&s_near, near_local);
    __syncthreads();
    // next frontier: the nodes of depth `level` in index order, with their parent's
    // row in this level's input (the parent's rank within its depth)
    for (int i = threadIdx.x; i < p.R; i += kThreads) {
      if (p.shape.depth[i] != a.level) continue;
      const int slot = p.shape.lrank[i];
      a.out.frontier_tok[static_cast<size_t>(b) * p.f_max + slot] = ntok[i];
      a.out.frontier_slot[static_cast<size_t>(b) * p.f_max + slot] = p.shape.lrank[p.shape.parent[i]];
    }
    if (threadIdx.x == 0) state[1] += s_near;
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
      a.out.score[ob + i] = ff_float(nsc[i]);
    }
    __syncthreads();
  }
  // ancestor masks: row i has bits i and those of its ancestors (each row walks up
  // the parent chain; parents come first, so at most R steps)
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
  p->off_state = off;
  off = align256(off + static_cast<size_t>(p->B) * 4 * 4);
  p->off_front = off;
  off = align256(off + static_cast<size_t>(p->B) * K * 4);
  p->off_part = off;
  off = align256(off + static_cast<size_t>(p->B) * p->f_max * p->n_chunks * sizeof(ChunkPart));
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
  dim3 grid(p.B * a.F, p.n_chunks);
  const bool bf16 = p.dtype != EAGLE_F32;
  if (p.mode == EAGLE_TREE_STATIC_SAMPLED) {
    if (bf16)
      tree_chunk_kernel<false, true><<<grid, kThreads, 0, s>>>(p, a);
    else
      tree_chunk_kernel<false, false><<<grid, kThreads, 0, s>>>(p, a);
  } else {
    if (bf16)
      tree_chunk_kernel<true, true><<<grid, kThreads, 0, s>>>(p, a);
    else
      tree_chunk_kernel<true, false><<<grid, kThreads, 0, s>>>(p, a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  tree_select_kernel<<<p.B, kThreads, 0, s>>>(p, a);
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
