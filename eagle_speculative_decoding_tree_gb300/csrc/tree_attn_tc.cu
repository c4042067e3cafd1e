// tree_attn_tc.cu -- tree attention on the tcgen05 tensor cores (bf16, head_dim 128).
//
// Same operation as tree_attn.cu (EAGLE review, terms "tree attention": each
// candidate attends only to its ancestors; lesson glossary "Tree attention"): row i
// of a request attends to the prefix keys j < seq_len and to the tree keys whose bit
// is set in its ancestor words.
//
// One CTA per (request, KV head, split, 128-row block), 320 threads, warp-specialised:
//   warp 8        TMA producer: Q once (one box per 64-dim half: the G query heads of
//                 128 / G nodes), then K and V tiles of 128 keys through rings of
//                 KST / VST stages.
//   warp 9        allocates the TMEM columns and issues tcgen05.mma from lane 0:
//                 S(t) = Q K(t)^T into buffer t & 1 (Q, K K-major, 128-byte swizzle) and
//                 O(t & 1) += P(t) V(t) (P from TMEM, V MN-major), in the order
//                 QK0 QK1 | PV0 QK2 | PV1 QK3 | ...; it zeroes V rows past the last
//                 valid key so that masked keys contribute exactly 0.
//   warps 0-3     softmax of the even tiles, warps 4-7 of the odd tiles.  Each thread
//                 owns one row (its TMEM lane) and all 128 keys of a tile, so a row's
//                 maximum needs no exchange between threads; the two warpgroups keep
//                 separate running states (m, l, O) and work on alternate tiles at the
//                 same time, so the tensor cores compute one tile's products while
//                 the other tile's softmax runs.  P = 2^((s - m) c) goes back into the
//                 tile's S columns as bf16 (precise: hi + lo, two bf16 terms, about 16
//                 significant bits; the PV product then takes one extra MMA per
//                 K-step).  O is rescaled in TMEM only when the row max grows by more
//                 than 2^8.  The two states merge in the epilogue.
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512).
//
// Splits: each CTA covers a contiguous range of key tiles (the tree tile counts as
// one) and keeps unnormalised fp32 partials (O, m, l).  One split writes the output
// directly.  When the whole grid fits on the SMs at once the launch is cooperative:
// every split stores its partial rows (TMA) and counts itself into its group
// (request, KV head, row block); once the group is complete each CTA merges a slice
// of the group's rows from L2.  Otherwise the shared combine kernel merges them; then
// (batched requests) a request's keys are cut into pieces of a fixed number of tiles,
// the requests are taken longest first, and the grid puts the row blocks of one key
// range next to each other so that they share its K/V tiles through L2.
//
// The launch is programmatic: barrier setup, TMEM allocation and descriptor prefetch
// overlap the tail of the preceding kernel; nothing is read from global memory before
// griddepcontrol.wait.
//
// Every wait is bounded; a timeout ORs a bit into the error word at the start of the
// workspace (it stays set until the caller clears it) and the roles stop, so the
// kernel ends instead of hanging.  The group counters return to zero by the end of
// every launch, so a zero-filled workspace stays valid across calls.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "sm100.cuh"

namespace eagle {
namespace {

using namespace sm100;

constexpr int KT = 128;                   // keys per tile
constexpr int HALF = 16384;               // one 64-dim half of a 128-row tile (bytes)
constexpr int TILE = 2 * HALF;            // one K or V tile
constexpr int NTHREADS = 320;
constexpr int SM_Q = 0;                   // the 128-row M-tile, 32 KB
constexpr int KST = 3;                    // K ring stages
constexpr int VST = 3;                    // V ring stages
constexpr int SM_K = TILE;
constexpr int SM_V = SM_K + KST * TILE;
constexpr int SMEM_BYTES = SM_V + VST * TILE + 1024;
static_assert(KST * TILE >= 4 * HALF, "the fp32 partial staging area reuses the K stages");
// TMEM columns: S / P of tile t in buffer t & 1, then the two O accumulators
__device__ __forceinline__ uint32_t col_s(int j) { return static_cast<uint32_t>(j) * 128u; }
__device__ __forceinline__ uint32_t col_o(int j) { return 256u + static_cast<uint32_t>(j) * 128u; }
constexpr float kRescaleLog2 = 8.f;       // lazy rescale threshold (log2 units)

enum : int { ERR_Q = 1, ERR_KFULL = 2, ERR_KEMPTY = 4, ERR_VFULL = 8, ERR_VEMPTY = 16, ERR_S = 32, ERR_P = 64, ERR_O = 128,
             ERR_GROUP = 256 };

struct TcArgs {
  const int32_t* seq_len;
  const int32_t* n_nodes;  // [B] tree rows per request (NULL: all R)
  const uint64_t* anc_mask;
  void* out;
  float* lse;
  float* part_o;   // [B*Hkv][splits][rows_pad][128] fp32
  float* part_ml;  // [B*Hkv][splits][rows_pad][2]
  int* err;
  int B, R, Hq, Hkv, G, P, W, splits, rows_pad, out_f32;
  int coop;        // 1: the splits of a group merge their partials in this kernel
  int tps;         // > 0: split s takes tile units [s tps, (s + 1) tps) of its request
                   //      (splits past a request's last unit do nothing); 0: even splits
  int lpt;         // 1: the request index of the grid is a rank in decreasing sequence length
  // Training-time-test attention (causal = 1): "request" b is TTT step j, "node" t is
  // sequence position t (R = P = S); the keys are the trunk K/V [Hkv][S][128] shared by
  // every step, row t sees keys t' <= t, and step j's rows then take j more keys, their
  // own predecessors (i, t), 1 <= i <= j, from the branch K/V [k][Hkv][S][128], folded
  // into the same softmax in the epilogue (one split, no partials).
  int causal;
  const uint16_t* qg;  // Q [k][S][Hq][128] (the branch dot products)
  const uint16_t* kb;
  const uint16_t* vb;
  int* cnt;        // coop: [2][n_groups] published / finished splits per (request, KV head, row block)
  int n_groups;
  int group_need;  // splits a group waits for (splits; one more under the failure test hook)
  unsigned long long group_limit_ns;
  float scale, scale_log2;
};

struct Tmaps {
  CUtensorMap q;   // [B*R][Hq][128] bf16, box {64, G, 128/G}
  CUtensorMap kc;  // [B*Hkv*P][128], box {64, 128}
  CUtensorMap vc;
  CUtensorMap tk;  // [B*Hkv*R][128], box {64, 128}
  CUtensorMap tv;
  CUtensorMap po;  // partial O [B*Hkv*splits*rows_pad][128] fp32, box {32, 128}
};

struct TileInfo {
  int n_pt, t_begin, n_tiles, L, Rb;
};

__device__ __forceinline__ int clamp_len(const TcArgs& a, int L) { return L < 0 ? 0 : (L > a.P ? a.P : L); }

// Tree rows of request b (n_nodes[b] clamped to [0, R]; all R rows without n_nodes).
__device__ __forceinline__ int rows_of(const TcArgs& a, int b) {
  if (!a.n_nodes) return a.R;
  const int n = a.n_nodes[b];
  return n < 0 ? 0 : (n > a.R ? a.R : n);
}

__device__ __forceinline__ TileInfo tile_info(const TcArgs& a, int b, int split, int rb) {
  TileInfo ti;
  if (a.causal) {  // keys 0 .. (last position of this CTA's rows), one split, no tree tile
    const int per = 128 / a.G;
    const int L = min(a.R, (rb + 1) * per);
    ti.t_begin = 0;
    ti.n_pt = ti.n_tiles = (L + KT - 1) / KT;
    ti.L = L;
    ti.Rb = a.R;
    return ti;
  }
  const int L = clamp_len(a, a.seq_len[b]);
  // units of work: the prefix tiles, then the tree tile; split s takes units
  // [U s / S, U (s + 1) / S) (or [s tps, (s + 1) tps) when tps > 0), so only the last
  // split that has units holds the tree tile
  const int n_pref = (L + KT - 1) / KT;
  const int U = n_pref + 1;
  int u0, u1;
  if (a.tps > 0) {
    u0 = min(U, split * a.tps);
    u1 = min(U, u0 + a.tps);
  } else {
    u0 = static_cast<int>(static_cast<long long>(U) * split / a.splits);
    u1 = static_cast<int>(static_cast<long long>(U) * (split + 1) / a.splits);
  }
  ti.t_begin = u0;
  ti.n_pt = max(0, min(u1, n_pref) - u0);
  ti.n_tiles = u1 - u0;
  ti.L = L;
  ti.Rb = rows_of(a, b);
  return ti;
}

// The request of rank r when the requests are ordered by decreasing sequence length
// (ties: lower index first).  Warp-collective; every lane returns the same value.
__device__ int request_of_rank(const TcArgs& a, int r) {
  const int lane = threadIdx.x & 31;
  int res = 0;
  for (int j0 = 0; j0 < a.B; j0 += 32) {
    const int j = j0 + lane;
    const int Lj = j < a.B ? clamp_len(a, a.seq_len[j]) : -1;
    int rank = 0;
    for (int i0 = 0; i0 < a.B; i0 += 32) {
      const int own = (i0 + lane < a.B) ? clamp_len(a, a.seq_len[i0 + lane]) : -1;
      for (int k = 0; k < 32; ++k) {
        const int i = i0 + k;
        const int Li = __shfl_sync(0xffffffffu, own, k);
        rank += (i < a.B && (Li > Lj || (Li == Lj && i < j))) ? 1 : 0;
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, j < a.B && rank == r);
    if (m) res = j0 + __ffs(m) - 1;
  }
  return res;
}

// One 128-key K or V tile (rows y .. y + 127 of the tensor map, both 64-dim halves)
// into a ring stage, completing on `bar`.
__device__ __forceinline__ void load_kv_tile(const CUtensorMap& m, uint8_t* dst, int y, uint64_t* bar,
                                             uint64_t policy) {
  tma_load_2d_hint(dst, &m, 0, y, bar, policy);
  tma_load_2d_hint(dst + HALF, &m, 64, y, bar, policy);
}

// Valid keys of tile t (prefix keys before L; tree rows before the request's row count).
__device__ __forceinline__ int tile_valid(const TileInfo& ti, int t) {
  if (t < ti.n_pt) return min(KT, ti.L - (ti.t_begin + t) * KT);
  return ti.Rb;
}

// Merge of one output row from the group's fp32 split partials, by a half-warp (16
// lanes, `hl` = lane within the half; every shuffle stays inside the half): lane s
// holds split s's (m, l) (splits beyond 16 in further rounds), M = max m_s,
// w_s = 2^((m_s - M) c), L = sum w_s l_s, O = sum w_s O_s / L.  Lane hl owns columns
// 8 hl .. 8 hl + 7.  The partial rows of up to kMergeBatch splits are requested before
// any is used (split indices past the last are clamped; their weight is 0), so a row
// costs about one L2 round trip.  grow < 0: nothing to write (the loads stay in bounds).
constexpr int kMergeBatch = 10;

__device__ __forceinline__ void load_part8(const TcArgs& a, size_t prow, int hl, float4 (&w)[2]) {
  const float4* src = reinterpret_cast<const float4*>(a.part_o + prow * 128) + 2 * hl;
  w[0] = __ldcg(src);
  w[1] = __ldcg(src + 1);
}

__device__ __forceinline__ void merge_row_hw(const TcArgs& a, int bh, int h, int b, int grow, int hl, float sl2) {
  const unsigned full = 0xffffffffu;
  const size_t base = static_cast<size_t>(bh) * a.splits * a.rows_pad + max(grow, 0);
  const size_t sstride = a.rows_pad;
  float4 v[kMergeBatch][2];
#pragma unroll
  for (int u = 0; u < kMergeBatch; ++u) load_part8(a, base + min(u, a.splits - 1) * sstride, hl, v[u]);
  float2 ml[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int sp = hl + 16 * k;
    ml[k] = sp < a.splits ? __ldcg(reinterpret_cast<const float2*>(a.part_ml + (base + sp * sstride) * 2))
                          : make_float2(-INFINITY, 0.f);
  }
  float M = fmaxf(fmaxf(ml[0].x, ml[1].x), fmaxf(ml[2].x, ml[3].x));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(full, M, o, 16));
  float w4[4], L = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    w4[k] = (ml[k].x == -INFINITY) ? 0.f : ex2((ml[k].x - M) * sl2);
    L += ml[k].y * w4[k];
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) L += __shfl_xor_sync(full, L, o, 16);
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  auto add8 = [&](float ws, const float4 (&x)[2]) {
    acc[0] = fmaf(ws, x[0].x, acc[0]);
    acc[1] = fmaf(ws, x[0].y, acc[1]);
    acc[2] = fmaf(ws, x[0].z, acc[2]);
    acc[3] = fmaf(ws, x[0].w, acc[3]);
    acc[4] = fmaf(ws, x[1].x, acc[4]);
    acc[5] = fmaf(ws, x[1].y, acc[5]);
    acc[6] = fmaf(ws, x[1].z, acc[6]);
    acc[7] = fmaf(ws, x[1].w, acc[7]);
  };
#pragma unroll
  for (int u = 0; u < kMergeBatch; ++u) {
    const float ws = __shfl_sync(full, w4[0], u, 16);  // 0 for u >= splits
    if (u < a.splits) add8(ws, v[u]);
  }
  for (int sp0 = kMergeBatch; sp0 < a.splits; sp0 += kMergeBatch) {  // further batches of splits
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) load_part8(a, base + min(sp0 + u, a.splits - 1) * sstride, hl, v[u]);
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const int sp = sp0 + u;
      const int k = (sp >> 4) & 3;
      const float ws = __shfl_sync(full, k == 0 ? w4[0] : (k == 1 ? w4[1] : (k == 2 ? w4[2] : w4[3])), sp & 15, 16);
      if (sp < a.splits) add8(ws, v[u]);
    }
  }
  if (grow < 0) return;
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int node = grow / a.G, hq = h * a.G + grow % a.G;
  const size_t orow = (static_cast<size_t>(b * a.R + node) * a.Hq + hq) * 128 + 8 * hl;
  if (a.out_f32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow);
    dst[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    dst[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
  } else {
    uint32_t wo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __nv_bfloat162 u2 = __floats2bfloat162_rn(acc[2 * k] * inv, acc[2 * k + 1] * inv);
      wo[k] = *reinterpret_cast<uint32_t*>(&u2);
    }
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + orow) = make_uint4(wo[0], wo[1], wo[2], wo[3]);
  }
  if (a.lse && hl == 0) a.lse[static_cast<size_t>(b * a.R + node) * a.Hq + hq] = a.scale * M + logf(L);
}

// Counts this split into its group and waits (at most limit_ns, then ERR_GROUP) until
// `n` splits of the group have counted.  Only valid when the whole grid is resident
// (cooperative launch).
__device__ __forceinline__ bool group_arrive_wait(int* cnt, int n, int* err, unsigned long long limit_ns) {
  __threadfence();
  atomicAdd(cnt, 1);
  if (ld_acquire_gpu(cnt) >= n) return true;
  const uint64_t t0 = global_ns();
  while (ld_acquire_gpu(cnt) < n) {
    if (global_ns() - t0 > limit_ns) {
      atomicOr(err, ERR_GROUP);
      return false;
    }
    __nanosleep(100);
  }
  return true;
}

// Bits 0..n-1 set (n clamped to [0, 32]).
__device__ __forceinline__ uint32_t low_bits(int n) {
  return n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : (1u << n) - 1u);
}

// Scores of keys whose bit is clear become -inf.
__device__ __forceinline__ void mask_keys(uint32_t (&r)[32], uint32_t bits) {
#pragma unroll
  for (int j = 0; j < 32; ++j) r[j] = ((bits >> j) & 1u) ? r[j] : 0xff800000u;
}

// Maximum of 64 floats with three-input max instructions, as a shallow tree.
__device__ __forceinline__ float max64(const uint32_t (&a)[32], const uint32_t (&b)[32]) {
  float m[22];
#pragma unroll
  for (int i = 0; i < 10; ++i)
    m[i] = max3(__uint_as_float(a[3 * i]), __uint_as_float(a[3 * i + 1]), __uint_as_float(a[3 * i + 2]));
  m[10] = max3(__uint_as_float(a[30]), __uint_as_float(a[31]), __uint_as_float(b[0]));
#pragma unroll
  for (int i = 0; i < 10; ++i)
    m[11 + i] = max3(__uint_as_float(b[3 * i + 1]), __uint_as_float(b[3 * i + 2]), __uint_as_float(b[3 * i + 3]));
  m[21] = fmaxf(__uint_as_float(b[31]), m[0]);
  float n[7];
#pragma unroll
  for (int i = 0; i < 7; ++i) n[i] = max3(m[3 * i + 1], m[3 * i + 2], m[3 * i + 3]);
  return max3(max3(n[0], n[1], n[2]), max3(n[3], n[4], n[5]), n[6]);
}

// S (TMEM columns scol) = Q K^T over the 8 K-steps of 16 head dims.
__device__ __forceinline__ void issue_qk(uint32_t tb, const uint8_t* sQ, const uint8_t* sK, uint32_t scol) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, KT, 0, 0);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t off = (ks >> 2) * HALF + (ks & 3) * 32;
    mma_ss(tb + scol, smem_desc_sw128(smem_u32(sQ) + off, 16, 1024), smem_desc_sw128(smem_u32(sK) + off, 16, 1024),
           idesc, ks > 0);
  }
}

// O (TMEM columns ocol) += P V over the 8 K-steps of 16 keys; the P of keys
// 64 h + 16 k .. sits in columns scol + 64 h + 8 k .. (the precise low parts 32 columns
// further on).
template <bool PRECISE>
__device__ __forceinline__ void issue_pv(uint32_t tb, const uint8_t* sV, uint32_t scol, uint32_t ocol, bool first) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint64_t bd = smem_desc_sw128(smem_u32(sV) + ks * 2048, HALF, 1024);
    const uint32_t acol = scol + (ks >> 2) * 64 + (ks & 3) * 8;
    mma_ts(tb + ocol, tb + acol, bd, idesc, (first && ks == 0) ? 0u : 1u);
    if constexpr (PRECISE) mma_ts(tb + ocol, tb + acol + 32, bd, idesc, 1u);
  }
}

// P of 32 keys held in registers (raw scores, masked keys -inf) -> TMEM columns
// `col` .. (bf16 pairs; the precise low parts 32 columns further on), 16 keys per
// store.  Returns the fp32 row sum of the 32 values.
template <bool PRECISE>
__device__ __forceinline__ float emit_p32(const uint32_t (&r)[32], uint32_t col, uint64_t sl2x2, uint64_t nmux2) {
  float sum = 0.f;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    uint32_t hi[8], lo[8];
    uint64_t acc2 = 0ull;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int k = 16 * g + 2 * j;
      float x0, x1;
      f32x2_split(fma_f32x2(f32x2(r[k], r[k + 1]), sl2x2, nmux2), x0, x1);
      const float p0 = ex2(x0), p1 = ex2(x1);
      __nv_bfloat162 u = __floats2bfloat162_rn(p0, p1);
      hi[j] = *reinterpret_cast<uint32_t*>(&u);
      if constexpr (PRECISE) {
        const float h0 = __uint_as_float(hi[j] << 16), h1 = __uint_as_float(hi[j] & 0xffff0000u);
        __nv_bfloat162 w = __floats2bfloat162_rn(p0 - h0, p1 - h1);
        lo[j] = *reinterpret_cast<uint32_t*>(&w);
      }
      // the row sum adds the fp32 p: hi + lo differs from p by at most 2^-17 p
      acc2 = add_f32x2(acc2, f32x2(__float_as_uint(p0), __float_as_uint(p1)));
    }
    tmem_st8(col + 8 * g, hi);
    if constexpr (PRECISE) tmem_st8(col + 32 + 8 * g, lo);
    float a0, a1;
    f32x2_split(acc2, a0, a1);
    sum += a0 + a1;
  }
  return sum;
}

template <bool PRECISE, bool CAUSAL>
__global__ void __launch_bounds__(NTHREADS, 1)
    tree_attn_tc_kernel(const __grid_constant__ Tmaps tm, const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_q, k_full[KST], k_empty[KST], v_full[VST], v_empty[VST], s_full[2], p_full[2], o_full;
  __shared__ uint32_t tmem_base;
  __shared__ int s_go;                        // group merge: every split published in time
  // [tile parity][row] running max and sum, exchanged in the epilogue (the Q area: every
  // QK has completed by then)
  float (*s_m)[128] = reinterpret_cast<float (*)[128]>(smem + SM_Q);
  float (*s_l)[128] = reinterpret_cast<float (*)[128]>(smem + SM_Q + 1024);

  // grid: cooperative (splits, B Hkv, row blocks); otherwise (row blocks, splits, B Hkv),
  // so that the row blocks of one key range, which read the same K/V tiles, are
  // dispatched next to each other and share them through L2
  const int split = a.coop ? blockIdx.x : blockIdx.y;
  const int rb = a.coop ? blockIdx.z : blockIdx.x;
  const int ybh = a.coop ? blockIdx.y : blockIdx.z;
  const int h = ybh % a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // prologue: nothing read from global memory before griddep_wait below
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&tm.q);
    prefetch_tmap(&tm.kc);
    prefetch_tmap(&tm.vc);
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar_q, 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 128);
    }
    mbar_init(&o_full, 1);
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  int issued_k[KST], issued_v[VST];  // producer: loads issued into each stage
  for (int s = 0; s < KST; ++s) issued_k[s] = 0;
  for (int s = 0; s < VST; ++s) issued_v[s] = 0;
  // the inputs (and the workspace counters) belong to the preceding kernel in the
  // stream until it completes
  griddep_wait();
  griddep_launch_dependents();
  // the request: ybh / Hkv, or (lpt) the request of that rank by decreasing length, so
  // that the longest requests' CTAs are dispatched first
  const int b = a.lpt ? request_of_rank(a, ybh / a.Hkv) : ybh / a.Hkv;
  const int bh = b * a.Hkv + h;
  uint8_t* sQ = smem + SM_Q;
  auto load_q = [&]() {
    mbar_arrive_expect_tx(&bar_q, TILE);
    const int node0 = (rb * 128) / a.G;
    for (int hh = 0; hh < 2; ++hh) tma_load_3d(sQ + hh * HALF, &tm.q, 64 * hh, h * a.G, b * a.R + node0, &bar_q);
  };
  // Q does not depend on the sequence length: with even splits its load goes out before
  // seq_len is read; with fixed-size splits only a CTA that has tiles loads it.  The MMA
  // warp waits for every Q load, so no copy is in flight at exit.
  if (a.tps == 0 && warp == 8 && lane == 0) load_q();
  const TileInfo ti = tile_info(a, b, split, rb);
  const bool q_loaded = a.tps == 0 || ti.n_tiles > 0;
  if (a.tps > 0 && q_loaded && warp == 8 && lane == 0) load_q();
  const uint32_t tb = tmem_base;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && ti.n_tiles > 0) {
      const uint64_t policy = policy_evict_first();
      for (int t = 0; t < ti.n_tiles; ++t) {
        const int s = t % KST, use = t / KST, sv = t % VST, usev = t / VST;
        const bool tree = t >= ti.n_pt;
        const int y = tree ? bh * a.R : (CAUSAL ? h : bh) * a.P + (ti.t_begin + t) * KT;
        if (use > 0 && !wait_parity(&k_empty[s], (use - 1) & 1, a.err, ERR_KEMPTY)) break;
        mbar_arrive_expect_tx(&k_full[s], TILE);
        load_kv_tile(tree ? tm.tk : tm.kc, smem + SM_K + s * TILE, y, &k_full[s], policy);
        ++issued_k[s];
        if (usev > 0 && !wait_parity(&v_empty[sv], (usev - 1) & 1, a.err, ERR_VEMPTY)) break;
        mbar_arrive_expect_tx(&v_full[sv], TILE);
        load_kv_tile(tree ? tm.tv : tm.vc, smem + SM_V + sv * TILE, y, &v_full[sv], policy);
        ++issued_v[sv];
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // S of tile t goes to TMEM buffer t & 1 and its PV into O(t & 1):
    // QK(0) QK(1) | PV(0) QK(2) | PV(1) QK(3) | ...
    bool ok = true;
    if (lane == 0 && q_loaded) ok = wait_parity(&bar_q, 0, a.err, ERR_Q);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0 && ti.n_tiles > 0;
    auto qk = [&](int t) {  // lane 0; K stage t % KST, S buffer t & 1
      const int s = t % KST;
      if (!wait_parity(&k_full[s], (t / KST) & 1, a.err, ERR_KFULL)) return false;
      tc_fence_after();
      issue_qk(tb, sQ, smem + SM_K + s * TILE, col_s(t & 1));
      mma_commit(&s_full[t & 1]);
      mma_commit(&k_empty[s]);
      return true;
    };
    if (ok && lane == 0) ok = qk(0) && (ti.n_tiles < 2 || qk(1));
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    for (int t = 0; t < ti.n_tiles && ok; ++t) {
      const int j = t & 1, sv = t % VST;
      // V of tile t: wait, then zero the rows past the last valid key
      ok = wait_parity(&v_full[sv], (t / VST) & 1, a.err, ERR_VFULL);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      const int nv = tile_valid(ti, t);
      if (nv < KT) {
        uint8_t* vt = smem + SM_V + sv * TILE;
        for (int idx = lane; idx < (KT - nv) * 16; idx += 32) {
          const int row = nv + (idx >> 4), part = idx & 15;
          *reinterpret_cast<uint4*>(vt + (part >> 3) * HALF + row * 128 + (part & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) {
        ok = wait_parity(&p_full[j], (t >> 1) & 1, a.err, ERR_P);
        if (ok) {
          tc_fence_after();
          issue_pv<PRECISE>(tb, smem + SM_V + sv * TILE, col_s(j), col_o(j), t < 2);
          mma_commit(&v_empty[sv]);
          if (t + 2 < ti.n_tiles) ok = qk(t + 2);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0 && ti.n_tiles > 0) mma_commit(&o_full);
  } else {
    // ------------------------------------------------------------ softmax, warps 0-7
    // Warpgroup j = warp >> 2 takes the tiles t with t & 1 == j; thread = TMEM lane =
    // row r_local of the M-tile, all 128 keys of the tile.
    const int wg = warp >> 2;
    const int qd = warp & 3;
    const int r_local = qd * 32 + lane;
    const uint32_t lb = tb + (static_cast<uint32_t>(qd * 32) << 16);
    const float sl2 = a.scale_log2;
    const int row = rb * 128 + r_local;
    const bool vrow = row < ti.Rb * a.G;
    const int node = vrow ? row / a.G : 0;
    const int hq = h * a.G + (vrow ? row % a.G : 0);
    uint32_t tw[4] = {0u, 0u, 0u, 0u};  // the row's ancestor words over the tree keys
    if (vrow && !CAUSAL) {
      const uint64_t* mrow = a.anc_mask + (static_cast<size_t>(b) * a.R + node) * a.W;
      const uint64_t w0 = mrow[0], w1 = a.W > 1 ? mrow[1] : 0ull;
      tw[0] = static_cast<uint32_t>(w0) & low_bits(ti.Rb);
      tw[1] = static_cast<uint32_t>(w0 >> 32) & low_bits(ti.Rb - 32);
      tw[2] = static_cast<uint32_t>(w1) & low_bits(ti.Rb - 64);
      tw[3] = static_cast<uint32_t>(w1 >> 32) & low_bits(ti.Rb - 96);
    }
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    const uint64_t sl2x2 = f32x2(__float_as_uint(sl2), __float_as_uint(sl2));
    for (int t = wg; t < ti.n_tiles && ok; t += 2) {
      if (!__all_sync(0xffffffffu, wait_parity(&s_full[wg], (t >> 1) & 1, a.err, ERR_S))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool tree = t >= ti.n_pt;
      const int nv = tile_valid(ti, t);
      uint32_t km[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        km[i] = !vrow ? 0u
                      : (CAUSAL ? low_bits(min(nv, node + 1 - (ti.t_begin + t) * KT) - 32 * i)
                                  : (tree ? tw[i] : low_bits(nv - 32 * i)));
      const bool full = __all_sync(0xffffffffu, (km[0] & km[1] & km[2] & km[3]) == 0xffffffffu);
      const uint32_t sc = lb + col_s(wg);
      // keys 64..127 stay in registers from the max to the exponentials; keys 0..63
      // are read again after their max is known
      uint32_t s0[32], s1[32], s2[32], s3[32];
      tmem_ld32(sc, s0);
      tmem_ld32(sc + 32, s1);
      tmem_ld32(sc + 64, s2);
      tmem_ld32(sc + 96, s3);
      tmem_ld_wait();
      if (!full) {
        mask_keys(s0, km[0]);
        mask_keys(s1, km[1]);
        mask_keys(s2, km[2]);
        mask_keys(s3, km[3]);
      }
      const float mx = fmaxf(max64(s0, s1), max64(s2, s3));
      const float m_new = fmaxf(m_ref, mx);
      // lazy rescale: move the row's reference max only when it grew by > 2^8.  O(wg)
      // holds this warpgroup's earlier tiles; their PV finished before S of this tile
      // did (in-order tensor pipe, one commit covers every earlier MMA).  tcgen05.ld/st
      // are warp-collective, so the whole warp touches O when any of its rows must.
      const bool move = m_new != -INFINITY && (m_ref == -INFINITY || (m_new - m_ref) * sl2 > kRescaleLog2);
      const bool scale_o = move && m_ref != -INFINITY;
      const float alpha = scale_o ? ex2((m_ref - m_new) * sl2) : 1.f;
      if (__any_sync(0xffffffffu, scale_o)) {
        l *= alpha;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(lb + col_o(wg) + 32 * c, o);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tmem_st32(lb + col_o(wg) + 32 * c, o);
        }
        tmem_st_wait();
      }
      if (move) m_ref = m_new;
      const float mu = (m_ref == -INFINITY) ? 0.f : m_ref * sl2;
      const uint64_t nmux2 = f32x2(__float_as_uint(-mu), __float_as_uint(-mu));
      // P of keys 64 h + 32 c .. + 31 goes to columns 64 h + 16 c .. + 15 (low parts
      // 32 columns further on); keys 64..127 first, whose S columns are already read
      float ls = emit_p32<PRECISE>(s2, sc + 64, sl2x2, nmux2);
      ls += emit_p32<PRECISE>(s3, sc + 80, sl2x2, nmux2);
      tmem_ld32(sc, s0);
      tmem_ld32(sc + 32, s1);
      tmem_ld_wait();
      if (!full) {
        mask_keys(s0, km[0]);
        mask_keys(s1, km[1]);
      }
      ls += emit_p32<PRECISE>(s0, sc, sl2x2, nmux2);
      ls += emit_p32<PRECISE>(s1, sc + 16, sl2x2, nmux2);
      l += ls;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[wg]);
    }
    // ---- epilogue: the two warpgroups' states merge; warpgroup j writes dims
    // [64 j, 64 j + 64) of its row to the output (one split) or the partials
    const bool have = ti.n_tiles > 0;
    const bool done = have && ok ? __all_sync(0xffffffffu, wait_parity(&o_full, 0, a.err, ERR_O)) : false;
    tc_fence_after();
    s_m[wg][r_local] = m_ref;
    s_l[wg][r_local] = l;
    const bool all_done = bar_and(1, 256, done) && have;
    const float mA = s_m[0][r_local], mB = s_m[1][r_local];
    const float M = fmaxf(mA, mB);
    const float aA = mA == -INFINITY ? 0.f : ex2((mA - M) * sl2);
    const float aB = mB == -INFINITY ? 0.f : ex2((mB - M) * sl2);
    const float L = aA * s_l[0][r_local] + aB * s_l[1][r_local];
    const bool two = ti.n_tiles > 1;  // O(1) holds tiles only when there are two or more
    float o[64];
    if (all_done) {
      uint32_t x[32], y[32];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        tmem_ld32(lb + col_o(0) + 64 * wg + 32 * c, x);
        if (two) tmem_ld32(lb + col_o(1) + 64 * wg + 32 * c, y);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 32; ++k)
          o[32 * c + k] = two ? fmaf(aA, __uint_as_float(x[k]), aB * __uint_as_float(y[k])) : aA * __uint_as_float(x[k]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 64; ++k) o[k] = 0.f;
    }
    float M_out = M, L_out = L;
    if (CAUSAL && b > 0) {
      // step b's own predecessors at this position, (i, node) for i = 1..b: one more
      // key each, folded into the row's softmax (streaming: new max, rescale, add).  The
      // two warpgroups each hold 64 of the 128 dims: partial dot products meet in shared
      // memory (the Q area, unused by now)
      float* s_dot = reinterpret_cast<float*>(smem + SM_Q + 2048);  // [2][128]
      const uint16_t* qrow = a.qg + (static_cast<size_t>(b * a.R + node) * a.Hq + hq) * 128 + 64 * wg;
      for (int i = 1; i <= b; ++i) {
        const size_t kvrow = ((static_cast<size_t>(i) * a.Hkv + h) * a.P + node) * 128 + 64 * wg;
        float part = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 u = *reinterpret_cast<const uint4*>(a.kb + kvrow + 8 * k);
          const uint4 qq = *reinterpret_cast<const uint4*>(qrow + 8 * k);
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
          const uint32_t q4[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            part = fmaf(__uint_as_float(q4[e] << 16), __uint_as_float(w4[e] << 16), part);
            part = fmaf(__uint_as_float(q4[e] & 0xffff0000u), __uint_as_float(w4[e] & 0xffff0000u), part);
          }
        }
        s_dot[wg * 128 + r_local] = part;
        bar_sync(1, 256);
        const float sc = s_dot[r_local] + s_dot[128 + r_local];  // the same sum in both halves
        bar_sync(1, 256);
        const float m_new = fmaxf(M_out, sc);
        const float a_old = M_out == -INFINITY ? 0.f : ex2((M_out - m_new) * sl2);
        const float a_new = ex2((sc - m_new) * sl2);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 u = *reinterpret_cast<const uint4*>(a.vb + kvrow + 8 * k);
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            o[8 * k + 2 * e] = fmaf(o[8 * k + 2 * e], a_old, a_new * __uint_as_float(w4[e] << 16));
            o[8 * k + 2 * e + 1] = fmaf(o[8 * k + 2 * e + 1], a_old, a_new * __uint_as_float(w4[e] & 0xffff0000u));
          }
        }
        L_out = L_out * a_old + a_new;
        M_out = m_new;
      }
    }
    const size_t prow = (static_cast<size_t>(bh) * a.splits + split) * a.rows_pad + rb * 128 + r_local;
    if (a.splits == 1) {
      if (vrow && all_done) {
        const float inv = L_out > 0.f ? 1.f / L_out : 0.f;
        const size_t orow = (static_cast<size_t>(b * a.R + node) * a.Hq + hq) * 128 + 64 * wg;
        if (a.out_f32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow);
#pragma unroll
          for (int k = 0; k < 16; ++k)
            dst[k] = make_float4(o[4 * k] * inv, o[4 * k + 1] * inv, o[4 * k + 2] * inv, o[4 * k + 3] * inv);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + orow);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              __nv_bfloat162 u = __floats2bfloat162_rn(o[8 * k + 2 * e] * inv, o[8 * k + 2 * e + 1] * inv);
              w[e] = *reinterpret_cast<uint32_t*>(&u);
            }
            dst[k] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        if (a.lse && wg == 0)
          a.lse[static_cast<size_t>(b * a.R + node) * a.Hq + hq] = a.scale * M_out + logf(L_out);
      }
    } else if (all_done) {
      // partial O of the M-tile (128 rows, contiguous in the workspace) staged in the
      // free K stages as four 128-byte-swizzled slices of 32 fp32 columns, then stored
      // with one TMA store per slice.  Row r's 16-byte chunk q sits at chunk q ^ (r & 7),
      // so each quarter-warp store covers all 32 banks.
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint8_t* dst = smem + SM_K + (2 * wg + c) * HALF + r_local * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(dst + ((q ^ (r_local & 7)) << 4)) =
              make_float4(o[32 * c + 4 * q], o[32 * c + 4 * q + 1], o[32 * c + 4 * q + 2], o[32 * c + 4 * q + 3]);
      }
      fence_proxy_async_smem();
      bar_sync(1, 256);
      if (threadIdx.x == 0) {
        const int y = (bh * a.splits + split) * a.rows_pad + rb * 128;
        for (int c = 0; c < 4; ++c) tma_store_2d(&tm.po, smem + SM_K + c * HALF, 32 * c, y);
        bulk_commit();
        if (a.coop)
          bulk_wait0();  // other CTAs of this launch read these rows
        else
          bulk_wait_read0();  // the combine kernel reads them once this grid has completed
      }
      if (wg == 0 && vrow) *reinterpret_cast<float2*>(a.part_ml + prow * 2) = make_float2(M, L);
    } else if (!(a.tps > 0 && ti.n_tiles == 0) && vrow) {
      // a split with no tiles (or one that timed out): zeros and weight 0; a split past
      // its request's last unit (fixed-size splits) writes nothing
      float4* dst = reinterpret_cast<float4*>(a.part_o + prow * 128 + 64 * wg);
#pragma unroll
      for (int k = 0; k < 16; ++k) dst[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (wg == 0) *reinterpret_cast<float2*>(a.part_ml + prow * 2) = make_float2(-INFINITY, 0.f);
    }
  }
  if (a.coop) {
    // the group's merge: publish this split's partials (every thread's writes fenced,
    // then one count), wait until every split of this (request, KV head, row block)
    // has counted, then merge rows [split n / S, (split + 1) n / S) of the block from
    // the partials in L2, a half-warp per row over all ten warps
    fence_proxy_async_global();
    __threadfence();
    __syncthreads();
    const int grp = bh * gridDim.z + rb;
    if (threadIdx.x == 0) {
      s_go = group_arrive_wait(a.cnt + grp, a.group_need, a.err, a.group_limit_ns) ? 1 : 0;
      // past the wait: the last split of the group to get here returns both counters
      // to zero for the next call
      int* fin = a.cnt + a.n_groups + grp;
      if (atomicAdd(fin, 1) == a.splits - 1) {
        atomicExch(a.cnt + grp, 0);
        atomicExch(fin, 0);
      }
    }
    __syncthreads();
    if (s_go) {
      const int n = max(0, min(128, ti.Rb * a.G - rb * 128));
      const int lo = split * n / a.splits;
      const int hi = (split + 1) * n / a.splits;
      // both halves of a warp loop together (shuffles are warp-collective), the spare
      // half on a row of its own block with no output
      for (int s0 = lo + 2 * warp; s0 < hi; s0 += 2 * (NTHREADS / 32)) {
        const int lr = s0 + (lane >> 4);
        const int grow = lr < hi ? rb * 128 + lr : -1;
        merge_row_hw(a, bh, h, b, grow, lane & 15, a.scale_log2);
      }
    }
  }
  // no copy of this CTA's may still be landing when it exits: the producer waits (at
  // most 2 s each) for the last load it issued into every stage; on the normal path
  // the MMA warp has already consumed them all
  if (warp == 8 && lane == 0) {
    for (int s = 0; s < KST; ++s)
      if (issued_k[s] > 0) (void)wait_parity(&k_full[s], (issued_k[s] - 1) & 1, a.err, ERR_KFULL);
    for (int s = 0; s < VST; ++s)
      if (issued_v[s] > 0) (void)wait_parity(&v_full[s], (issued_v[s] - 1) & 1, a.err, ERR_VFULL);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Tensor map of `rank` dims (innermost first), 128-byte swizzle, zero fill.
bool make_tmap(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int rank, const cuuint64_t* dims,
               const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// One-time per-device kernel attribute: the dynamic shared memory.
template <bool PRECISE, bool CAUSAL>
cudaError_t configure_tc() {
  static unsigned long long configured = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && (__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & (1ull << dev))) return cudaSuccess;
  e = cudaFuncSetAttribute(tree_attn_tc_kernel<PRECISE, CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (dev < 64) __atomic_fetch_or(&configured, 1ull << dev, __ATOMIC_RELEASE);
  return cudaSuccess;
}

// Cooperative launch when the CTAs of a split group wait on one another (a.coop):
// the driver then guarantees that the whole grid is resident at once, or fails the
// launch.
template <bool PRECISE, bool CAUSAL = false>
cudaError_t launch_tc(const Tmaps& tm, const TcArgs& a, dim3 grid, cudaStream_t s) {
  cudaError_t e = configure_tc<PRECISE, CAUSAL>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  // programmatic: the prologue (barriers, TMEM, descriptor prefetch) overlaps the
  // tail of the preceding kernel; the kernel waits for it before reading anything
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n++].val.programmaticStreamSerializationAllowed = 1;
  if (a.coop) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n++].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  e = cudaLaunchKernelEx(&cfg, tree_attn_tc_kernel<PRECISE, CAUSAL>, tm, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tree_attn_tc(const AttnPlan& p, const void* q, const void* k_cache, const void* v_cache,
                                const void* tree_k, const void* tree_v, const int32_t* seq_len,
                                const int32_t* n_nodes, const uint64_t* anc_mask, void* out, float* lse, void* ws,
                                cudaStream_t s) {
  Tmaps tm;
  const cuuint64_t D = 128;
  {
    const cuuint64_t dims[3] = {D, static_cast<cuuint64_t>(p.Hq), static_cast<cuuint64_t>(p.B) * p.R};
    const cuuint64_t strides[2] = {D * 2, static_cast<cuuint64_t>(p.Hq) * D * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(p.G), static_cast<cuuint32_t>(128 / p.G)};
    if (!make_tmap(&tm.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {D, static_cast<cuuint64_t>(p.B) * p.Hkv * p.P};
    const cuuint64_t strides[1] = {D * 2};
    const cuuint32_t box[2] = {64, 128};
    if (!make_tmap(&tm.kc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k_cache, 2, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_tmap(&tm.vc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v_cache, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {D, static_cast<cuuint64_t>(p.B) * p.Hkv * p.R};
    const cuuint64_t strides[1] = {D * 2};
    const cuuint32_t box[2] = {64, 128};
    if (!make_tmap(&tm.tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, tree_k, 2, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_tmap(&tm.tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, tree_v, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  uint8_t* w = static_cast<uint8_t*>(ws);
  memset(&tm.po, 0, sizeof(tm.po));
  if (p.splits > 1) {
    const cuuint64_t dims[2] = {D, static_cast<cuuint64_t>(p.B) * p.Hkv * p.splits * p.rows_pad};
    const cuuint64_t strides[1] = {D * 4};
    const cuuint32_t box[2] = {32u, 128};
    if (!make_tmap(&tm.po, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, w + p.off_o, 2, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  TcArgs a;
  a.seq_len = seq_len;
  a.n_nodes = n_nodes;
  a.anc_mask = anc_mask;
  a.out = out;
  a.lse = lse;
  const bool partials = p.splits > 1;
  a.part_o = partials ? reinterpret_cast<float*>(w + p.off_o) : nullptr;
  a.part_ml = partials ? reinterpret_cast<float*>(w + p.off_ml) : nullptr;
  a.err = reinterpret_cast<int*>(w + p.off_err);
  a.B = p.B;
  a.R = p.R;
  a.Hq = p.Hq;
  a.Hkv = p.Hkv;
  a.G = p.G;
  a.P = p.P;
  a.W = p.W;
  a.splits = p.splits;
  a.rows_pad = p.rows_pad;
  a.coop = p.coop ? 1 : 0;
  a.tps = p.tps;
  a.lpt = p.lpt ? 1 : 0;
  a.causal = 0;
  a.qg = a.kb = a.vb = nullptr;
  a.cnt = p.coop ? reinterpret_cast<int*>(w + p.off_cnt) : nullptr;
  a.n_groups = p.B * p.Hkv * p.row_blocks;
  // the failure test hook: the group waits for one split that does not exist and gives
  // up after 1 ms
  a.group_need = p.splits + (p.fault_test ? 1 : 0);
  a.group_limit_ns = p.fault_test ? 1000000ull : 2000000000ull;
  a.out_f32 = p.out_dtype == EAGLE_F32;
  a.scale = p.scale;
  a.scale_log2 = p.scale * kLog2e;
  cudaError_t e;
  const dim3 grid = p.coop ? dim3(p.splits, p.B * p.Hkv, p.row_blocks) : dim3(p.row_blocks, p.splits, p.B * p.Hkv);
  e = p.precise ? launch_tc<true>(tm, a, grid, s) : launch_tc<false>(tm, a, grid, s);
  if (e != cudaSuccess || !partials || p.coop) return e;
  return launch_tree_attn_combine(p, seq_len, n_nodes, out, lse, static_cast<const float*>(a.part_o), a.part_ml, s,
                                  true);
}

cudaError_t launch_ttt_attn_tc(int steps, int S, int Hq, int Hkv, float scale, bool out_f32, const void* q,
                               const void* k_trunk, const void* v_trunk, const void* k_branch, const void* v_branch,
                               void* out, float* lse, void* ws, cudaStream_t s) {
  const int G = Hq / Hkv;
  Tmaps tm;
  const cuuint64_t D = 128;
  {
    const cuuint64_t dims[3] = {D, static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(steps) * S};
    const cuuint64_t strides[2] = {D * 2, static_cast<cuuint64_t>(Hq) * D * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(128 / G)};
    if (!make_tmap(&tm.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {D, static_cast<cuuint64_t>(Hkv) * S};
    const cuuint64_t strides[1] = {D * 2};
    const cuuint32_t box[2] = {64, 128};
    if (!make_tmap(&tm.kc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k_trunk, 2, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_tmap(&tm.vc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v_trunk, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  tm.tk = tm.kc;  // no tree tile in this mode
  tm.tv = tm.vc;
  memset(&tm.po, 0, sizeof(tm.po));
  TcArgs a;
  memset(&a, 0, sizeof(a));
  a.out = out;
  a.lse = lse;
  a.err = static_cast<int*>(ws);
  a.B = steps;
  a.R = S;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = G;
  a.P = S;
  a.W = 1;
  a.splits = 1;
  const int row_blocks = (S * G + 127) / 128;
  a.rows_pad = row_blocks * 128;
  a.out_f32 = out_f32 ? 1 : 0;
  a.group_need = 1;
  a.group_limit_ns = 2000000000ull;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.causal = 1;
  a.qg = static_cast<const uint16_t*>(q);
  a.kb = static_cast<const uint16_t*>(k_branch);
  a.vb = static_cast<const uint16_t*>(v_branch);
  return launch_tc<true, true>(tm, a, dim3(row_blocks, 1, steps * Hkv), s);
}

}  // namespace eagle
