// tree_attn_tc.cu -- tree attention on the tcgen05 tensor cores (bf16, head_dim 128).
//
// Same operation as tree_attn.cu (EAGLE review, terms "tree attention": each
// candidate attends only to its ancestors; lesson glossary "Tree attention"): row i
// of a request attends to the prefix keys j < seq_len and to the tree keys whose bit
// is set in its ancestor words.
//
// One CTA per (request, KV head, split, 128-row block), 320 threads, warp-specialised:
//   warp 8        TMA producer: Q once (one box per 64-dim half: the G query heads of
//                 128 / G nodes), then K and V tiles of 128 keys through two-stage rings.
//   warp 9        allocates the TMEM columns and issues tcgen05.mma from lane 0:
//                 S = Q K^T (Q, K K-major, 128-byte swizzle) into buffer t & 1, and
//                 O += P V (P from TMEM, V MN-major), in the order QK0 QK1 | PV0 QK2 |
//                 PV1 QK3 | ..., so the next-but-one S is computed while the softmax works
//                 on this one; the warp zeroes V rows past the last valid key so that
//                 masked keys contribute exactly 0.
//   warps 0-7     online softmax: warp w takes TMEM lane quarter w & 3 (32 rows) and key
//                 half w >> 2; the halves of a row agree on its max through shared memory.
//                 P = 2^((s - m) c) goes back into the half's own S columns as packed bf16
//                 (the PV A operand).  O is rescaled in TMEM only when the row max grows
//                 by more than 2^8, after the previous PV has finished.
// TMEM columns: S0 [0,128) S1 [128,256) O [256,384).
//
// Splits: each CTA covers a contiguous range of key tiles (the tree tile counts as
// one) and keeps unnormalised partials (O, m, l).  One split writes the output
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
constexpr int KST = 2;                    // K ring stages
constexpr int VST = 2;                    // V ring stages
constexpr int SM_K = TILE;
constexpr int SM_V = SM_K + KST * TILE;
constexpr int SMEM_BYTES = SM_V + VST * TILE + 1024;
static_assert(KST >= 2, "the partial staging area reuses two K stages");
// TMEM columns: S / P of tile t in buffer t & 1, then the O accumulator
__device__ __forceinline__ uint32_t col_s(int j) { return static_cast<uint32_t>(j) * 128u; }
constexpr uint32_t COL_O = 256u;
constexpr float kRescaleLog2 = 8.f;       // lazy rescale threshold (log2 units)

enum : int { ERR_Q = 1, ERR_KFULL = 2, ERR_KEMPTY = 4, ERR_VFULL = 8, ERR_VEMPTY = 16, ERR_S = 32, ERR_P = 64, ERR_O = 128,
             ERR_GROUP = 256 };

struct TcArgs {
  const int32_t* seq_len;
  const uint64_t* anc_mask;
  void* out;
  float* lse;
  void* part_o;    // [B*Hkv][splits][rows_pad][128], bf16 when part_bf16 else fp32
  int part_bf16;
  float* part_ml;  // [B*Hkv][splits][rows_pad][2]
  int* err;
  int B, R, Hq, Hkv, G, P, W, splits, rows_pad, rows_per_cta, n_mt, out_f32;
  int coop;        // 1: the splits of a group merge their partials in this kernel
  int tps;         // > 0: split s takes tile units [s tps, (s + 1) tps) of its request
                   //      (splits past a request's last unit do nothing); 0: even splits
  int lpt;         // 1: the request index of the grid is a rank in decreasing sequence length
  int* cnt;        // coop: [2][n_groups] published / finished splits per (request, KV head, row block)
  int n_groups;
  float scale, scale_log2;
};

struct Tmaps {
  CUtensorMap q;   // [B*R][Hq][128] bf16, box {64, G, 128/G}
  CUtensorMap kc;  // [B*Hkv*P][128], box {64, 128}
  CUtensorMap vc;
  CUtensorMap tk;  // [B*Hkv*R][128], box {64, 128}
  CUtensorMap tv;
  CUtensorMap po;  // partial O [B*Hkv*splits*rows_pad][128]: fp32 box {32, 128} or bf16 box {64, 128}
};

struct TileInfo {
  int n_pt, t_begin, n_tiles, L;
};

__device__ __forceinline__ int clamp_len(const TcArgs& a, int L) { return L < 0 ? 0 : (L > a.P ? a.P : L); }

__device__ __forceinline__ TileInfo tile_info(const TcArgs& a, int b, int split) {
  TileInfo ti;
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

// Valid keys of tile t (prefix keys before L; tree rows before R).
__device__ __forceinline__ int tile_valid(const TcArgs& a, const TileInfo& ti, int t) {
  if (t < ti.n_pt) return min(KT, ti.L - (ti.t_begin + t) * KT);
  return a.R;
}

// Merge of one output row from the group's split partials, by a half-warp (16 lanes,
// `hl` = lane within the half; every shuffle stays inside the half): lane s holds
// split s's (m, l) (splits beyond 16 in further rounds), M = max m_s,
// w_s = 2^((m_s - M) c), L = sum w_s l_s, O = sum w_s O_s / L.  Lane hl owns columns
// 8 hl .. 8 hl + 7.  The partial rows of up to kMergeBatch splits are requested before
// any is used (split indices past the last are clamped; their weight is 0), so a row
// costs about one L2 round trip.  grow < 0: nothing to write (the loads stay in bounds).
constexpr int kMergeBatch = 16;

__device__ __forceinline__ void load_part8(const TcArgs& a, size_t prow, int hl, bool bf16, uint4 (&w)[2]) {
  if (bf16) {
    w[0] = __ldcg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.part_o) + prow * 128) + hl);
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const float*>(a.part_o) + prow * 128) + 2 * hl;
    w[0] = __ldcg(src);
    w[1] = __ldcg(src + 1);
  }
}

__device__ __forceinline__ void part8_f32(const uint4 (&w)[2], bool bf16, float (&x)[8]) {
  if (bf16) {
    const uint32_t u[4] = {w[0].x, w[0].y, w[0].z, w[0].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = __uint_as_float(u[k] << 16);
      x[2 * k + 1] = __uint_as_float(u[k] & 0xffff0000u);
    }
  } else {
    x[0] = __uint_as_float(w[0].x);
    x[1] = __uint_as_float(w[0].y);
    x[2] = __uint_as_float(w[0].z);
    x[3] = __uint_as_float(w[0].w);
    x[4] = __uint_as_float(w[1].x);
    x[5] = __uint_as_float(w[1].y);
    x[6] = __uint_as_float(w[1].z);
    x[7] = __uint_as_float(w[1].w);
  }
}

template <bool BF16>
__device__ __forceinline__ void merge_row_hw(const TcArgs& a, int bh, int h, int b, int grow, int hl, float sl2) {
  const unsigned full = 0xffffffffu;
  const size_t base = static_cast<size_t>(bh) * a.splits * a.rows_pad + max(grow, 0);
  const size_t sstride = a.rows_pad;
  constexpr int NB = BF16 ? kMergeBatch : kMergeBatch / 2;  // fp32 rows take two words per lane
  uint4 v[NB][2];
#pragma unroll
  for (int u = 0; u < NB; ++u) load_part8(a, base + min(u, a.splits - 1) * sstride, hl, BF16, v[u]);
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
#pragma unroll
  for (int u = 0; u < NB; ++u) {
    const float ws = __shfl_sync(full, w4[0], u, 16);  // 0 for u >= splits
    float x[8];
    part8_f32(v[u], BF16, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = fmaf(ws, x[e], acc[e]);
  }
  for (int sp = NB; sp < a.splits; ++sp) {  // more splits than one batch
    const int k = sp >> 4;
    const float ws = __shfl_sync(full, k == 0 ? w4[0] : (k == 1 ? w4[1] : (k == 2 ? w4[2] : w4[3])), sp & 15, 16);
    uint4 t[2];
    load_part8(a, base + sp * sstride, hl, BF16, t);
    float x[8];
    part8_f32(t, BF16, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = fmaf(ws, x[e], acc[e]);
  }
  if (grow < 0) return;
  const float inv = 1.f / L;
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

// Counts this split into its group and waits (at most 2 s, then ERR_GROUP) until all
// `n` splits of the group have counted.  Only valid when the whole grid is resident
// (cooperative launch).
__device__ __forceinline__ bool group_arrive_wait(int* cnt, int n, int* err) {
  __threadfence();
  atomicAdd(cnt, 1);
  if (ld_acquire_gpu(cnt) >= n) return true;
  const uint64_t t0 = global_ns();
  while (ld_acquire_gpu(cnt) < n) {
    if (global_ns() - t0 > 2000000000ull) {
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

// O += P V over the 8 K-steps of 16 keys; the P of keys 64 h + 16 k .. sits in columns
// scol + 64 h + 8 k .. (the precise low parts 32 columns further on).
template <bool PRECISE>
__device__ __forceinline__ void issue_pv(uint32_t tb, const uint8_t* sV, uint32_t scol, bool first) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint64_t bd = smem_desc_sw128(smem_u32(sV) + ks * 2048, HALF, 1024);
    const uint32_t acol = scol + (ks >> 2) * 64 + (ks & 3) * 8;
    mma_ts(tb + COL_O, tb + acol, bd, idesc, (first && ks == 0) ? 0u : 1u);
    if constexpr (PRECISE) mma_ts(tb + COL_O, tb + acol + 32, bd, idesc, 1u);
  }
}

template <bool PRECISE>
__global__ void __launch_bounds__(NTHREADS, 1)
    tree_attn_tc_kernel(const __grid_constant__ Tmaps tm, const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_q, k_full[KST], k_empty[KST], v_full[VST], v_empty[VST], s_full[2], p_full[2], o_done, o_full;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;
  __shared__ float s_red[2][2][2][128];  // [tile parity][M-tile][key half][row] half-row maxima
  __shared__ float s_l[2][2][128];        // [M-tile][key half][row] half-row sums
  __shared__ int s_go;                    // group merge: every split published in time

  // grid: cooperative (splits, B Hkv, row blocks); otherwise (row blocks, splits, B Hkv),
  // so that the row blocks of one key range, which read the same K/V tiles, are
  // dispatched next to each other and share them through L2
  const int split = a.coop ? blockIdx.x : blockIdx.y;
  const int rb = a.coop ? blockIdx.z : blockIdx.x;
  const int ybh = a.coop ? blockIdx.y : blockIdx.z;
  const int h = ybh % a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_mt = a.n_mt;

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
      mbar_init(&p_full[s], 256);
    }
    mbar_init(&o_done, 1);
    mbar_init(&o_full, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
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
    mbar_arrive_expect_tx(&bar_q, n_mt * TILE);
    for (int i = 0; i < n_mt; ++i) {
      const int node0 = (rb * a.rows_per_cta + i * 128) / a.G;
      for (int hh = 0; hh < 2; ++hh)
        tma_load_3d(sQ + i * TILE + hh * HALF, &tm.q, 64 * hh, h * a.G, b * a.R + node0, &bar_q);
    }
  };
  // Q does not depend on the sequence length: with even splits its load goes out before
  // seq_len is read; with fixed-size splits only a CTA that has tiles loads it.  The MMA
  // warp waits for every Q load, so no copy is in flight at exit.
  if (a.tps == 0 && warp == 8 && lane == 0) load_q();
  const TileInfo ti = tile_info(a, b, split);
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
        const CUtensorMap* mk = tree ? &tm.tk : &tm.kc;
        const CUtensorMap* mv = tree ? &tm.tv : &tm.vc;
        const int y = tree ? bh * a.R : bh * a.P + (ti.t_begin + t) * KT;
        if (use > 0 && !wait_parity(&k_empty[s], (use - 1) & 1, a.err, ERR_KEMPTY)) break;
        mbar_arrive_expect_tx(&k_full[s], TILE);
        tma_load_2d_hint(smem + SM_K + s * TILE, mk, 0, y, &k_full[s], policy);
        tma_load_2d_hint(smem + SM_K + s * TILE + HALF, mk, 64, y, &k_full[s], policy);
        if (usev > 0 && !wait_parity(&v_empty[sv], (usev - 1) & 1, a.err, ERR_VEMPTY)) break;
        mbar_arrive_expect_tx(&v_full[sv], TILE);
        tma_load_2d_hint(smem + SM_V + sv * TILE, mv, 0, y, &v_full[sv], policy);
        tma_load_2d_hint(smem + SM_V + sv * TILE + HALF, mv, 64, y, &v_full[sv], policy);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // S of tile t goes to TMEM buffer t & 1: QK(0) QK(1) | PV(0) QK(2) | PV(1) QK(3) | ...
    // so the tensor cores compute the next-but-one S while the softmax works on this one.
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
      const int s = t & 1, sv = t % VST;
      // V of tile t: wait, then zero the rows past the last valid key
      ok = wait_parity(&v_full[sv], (t / VST) & 1, a.err, ERR_VFULL);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      const int nv = tile_valid(a, ti, t);
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
        ok = wait_parity(&p_full[s], (t >> 1) & 1, a.err, ERR_P);
        if (ok) {
          tc_fence_after();
          issue_pv<PRECISE>(tb, smem + SM_V + sv * TILE, col_s(s), t == 0);
          mma_commit(&v_empty[sv]);
          mma_commit(&o_done);
          if (t + 2 < ti.n_tiles) ok = qk(t + 2);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0 && ti.n_tiles > 0) mma_commit(&o_full);
  } else {
    // ------------------------------------------------------------ softmax, warps 0-7
    // All eight warps work on one M-tile at a time: warp w reads TMEM lane quarter
    // w & 3 (32 rows) and key half w >> 2 (keys / S columns [64 hf, 64 hf + 64)).  The
    // two halves of a row agree on its max through shared memory; each half reads its
    // S once, keeps it in registers across the exchange and writes its P into its own
    // S columns.
    const int qd = warp & 3;
    const int hf = warp >> 2;
    const int r_local = qd * 32 + lane;      // row within an M-tile = TMEM lane
    const uint32_t lb = tb + (static_cast<uint32_t>(qd * 32) << 16);
    const float sl2 = a.scale_log2;
    bool vrow[2];
    int node[2], hq[2];
    uint32_t tw[2][2];                       // this half's ancestor words (keys >= R cleared)
    float m_ref[2], l[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int row = rb * a.rows_per_cta + i * 128 + r_local;
      vrow[i] = i < n_mt && row < a.R * a.G;
      node[i] = vrow[i] ? row / a.G : 0;
      hq[i] = h * a.G + (vrow[i] ? row % a.G : 0);
      tw[i][0] = tw[i][1] = 0u;
      if (vrow[i]) {
        const uint64_t* mrow = a.anc_mask + (static_cast<size_t>(b) * a.R + node[i]) * a.W;
        const uint64_t mw = (hf == 0) ? mrow[0] : (a.W > 1 ? mrow[1] : 0ull);
        tw[i][0] = static_cast<uint32_t>(mw) & low_bits(a.R - 64 * hf);
        tw[i][1] = static_cast<uint32_t>(mw >> 32) & low_bits(a.R - 64 * hf - 32);
      }
      m_ref[i] = -INFINITY;
      l[i] = 0.f;
    }
    bool ok = true;
    for (int t = 0; t < ti.n_tiles && ok; ++t) {
      const bool tree = t >= ti.n_pt;
      const int nv = tile_valid(a, ti, t);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (i >= n_mt) break;
        const bool got = __all_sync(0xffffffffu, wait_parity(&s_full[t & 1], (t >> 1) & 1, a.err, ERR_S));
        tc_fence_after();
        // the max of this half's 64 scores over the kept keys
        const uint32_t k0 = !vrow[i] ? 0u : (tree ? tw[i][0] : low_bits(nv - 64 * hf));
        const uint32_t k1 = !vrow[i] ? 0u : (tree ? tw[i][1] : low_bits(nv - 64 * hf - 32));
        const bool full = __all_sync(0xffffffffu, (k0 & k1) == 0xffffffffu);
        // S of this half-row stays in registers from the max to the exponentials
        float mx = -INFINITY;
        uint32_t s0[32], s1[32];
        if (got) {
          tmem_ld32(lb + col_s(t & 1) + 64 * hf, s0);
          tmem_ld32(lb + col_s(t & 1) + 64 * hf + 32, s1);
          tmem_ld_wait();
          if (!full) {
            mask_keys(s0, k0);
            mask_keys(s1, k1);
          }
          mx = max64(s0, s1);
        }
        s_red[t & 1][i][hf][r_local] = mx;
        if (!bar_and(1, 256, got)) {  // every softmax warp leaves together on a timeout
          ok = false;
          break;
        }
        const float m_new = fmaxf(m_ref[i], fmaxf(mx, s_red[t & 1][i][hf ^ 1][r_local]));
        // lazy rescale: move the row's reference max only when it grew by > 2^8; O
        // holds earlier tiles only when m_ref is already finite.  Both halves of a row
        // decide alike; each rescales its own 64 O columns.  tcgen05.ld/st are
        // warp-collective, so the whole warp touches O when any of its rows must.
        const bool move = m_new != -INFINITY && (m_ref[i] == -INFINITY || (m_new - m_ref[i]) * sl2 > kRescaleLog2);
        const bool scale_o = move && m_ref[i] != -INFINITY;
        const float alpha = scale_o ? ex2((m_ref[i] - m_new) * sl2) : 1.f;
        if (__any_sync(0xffffffffu, scale_o)) {
          // O must hold every earlier tile: wait for PV(t - 1) (PV(t - 2) finished
          // before S of tile t did).  A timeout only records ERR_O: leaving the loop here
          // would desert the named barriers the other softmax warps wait on.
          __syncwarp();
          (void)wait_parity(&o_done, (t - 1) & 1, a.err, ERR_O);
          __syncwarp();
          tc_fence_after();
          l[i] *= alpha;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            tmem_ld32(lb + COL_O + 64 * hf + 32 * c, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tmem_st32(lb + COL_O + 64 * hf + 32 * c, o);
          }
          tmem_st_wait();
        }
        if (move) m_ref[i] = m_new;
        const float mu = (m_ref[i] == -INFINITY) ? 0.f : m_ref[i] * sl2;
        // P = 2^(s c - m c) from the S held in registers, as bf16 pairs (masked keys hold
        // -inf and give exactly 0): keys 64 hf + 32 c .. + 31 go to columns
        // 64 hf + 16 c .. + 15; the precise path puts the low parts 32 columns further
        // on.  l sums the fp32 p (the precise path: hi + lo).
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
        uint64_t ls2[2] = {0ull, 0ull};  // standard path: packed row-sum accumulators
        const uint64_t sl2x2 = f32x2(__float_as_uint(sl2), __float_as_uint(sl2));
        const uint64_t nmux2 = f32x2(__float_as_uint(-mu), __float_as_uint(-mu));
        auto emit = [&](const uint32_t (&r)[32], int c) {
          uint32_t hi[16];
          if constexpr (!PRECISE) {
            // two keys per packed instruction: x = s c - m c, then 2^x on the MUFU
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float x0, x1;
              f32x2_split(fma_f32x2(f32x2(r[2 * j], r[2 * j + 1]), sl2x2, nmux2), x0, x1);
              const float p0 = ex2(x0), p1 = ex2(x1);
              __nv_bfloat162 u = __floats2bfloat162_rn(p0, p1);
              hi[j] = *reinterpret_cast<uint32_t*>(&u);
              ls2[j & 1] = add_f32x2(ls2[j & 1], f32x2(__float_as_uint(p0), __float_as_uint(p1)));
            }
            tmem_st16(lb + col_s(t & 1) + 64 * hf + 16 * c, hi);
          } else {
            // P = hi + lo, both bf16; the low parts go 32 columns after the high ones
            uint32_t lo[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float p0 = ex2(fmaf(__uint_as_float(r[2 * j]), sl2, -mu));
              const float p1 = ex2(fmaf(__uint_as_float(r[2 * j + 1]), sl2, -mu));
              __nv_bfloat162 u = __floats2bfloat162_rn(p0, p1);
              hi[j] = *reinterpret_cast<uint32_t*>(&u);
              const float h0 = __uint_as_float(hi[j] << 16), h1 = __uint_as_float(hi[j] & 0xffff0000u);
              __nv_bfloat162 w = __floats2bfloat162_rn(p0 - h0, p1 - h1);
              lo[j] = *reinterpret_cast<uint32_t*>(&w);
              ls[j & 3] += (h0 + __uint_as_float(lo[j] << 16)) + (h1 + __uint_as_float(lo[j] & 0xffff0000u));
            }
            tmem_st16(lb + col_s(t & 1) + 64 * hf + 16 * c, hi);
            tmem_st16(lb + col_s(t & 1) + 64 * hf + 32 + 16 * c, lo);
          }
        };
        emit(s0, 0);
        emit(s1, 1);
        if constexpr (!PRECISE) {
          float a0, a1, b0, b1;
          f32x2_split(ls2[0], a0, a1);
          f32x2_split(ls2[1], b0, b1);
          l[i] += (a0 + a1) + (b0 + b1);
        } else {
          l[i] += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[t & 1]);
      }
    }
    // ---- epilogue: O from TMEM to the output (one split) or the partials
    const bool have = ok && ti.n_tiles > 0;
    const bool done = have ? __all_sync(0xffffffffu, wait_parity(&o_full, 0, a.err, ERR_O)) : false;
    tc_fence_after();
#pragma unroll
    for (int i = 0; i < 2; ++i) s_l[i][hf][r_local] = l[i];
    const bool all_done = bar_and(2, 256, done);
    float l_tot[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) l_tot[i] = l[i] + s_l[i][hf ^ 1][r_local];
    if (a.splits > 1 && all_done) {
      // partial O of each M-tile (128 rows, contiguous in the workspace) is staged in
      // the free K/V stages as 128-byte-swizzled column slices (fp32: four slices of
      // 32 columns; bf16: two of 64), then stored with one TMA store per slice.  Row
      // r's 16-byte chunk j sits at chunk j ^ (r & 7), so each quarter-warp store
      // covers all 32 banks.
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (i >= n_mt) break;
        uint8_t* so = smem + SM_K + i * 4 * HALF;
        if (a.part_bf16) {
          uint32_t o0[32], o1[32];
          tmem_ld32(lb + COL_O + 64 * hf, o0);
          tmem_ld32(lb + COL_O + 64 * hf + 32, o1);
          tmem_ld_wait();
          uint8_t* dst = so + hf * HALF + r_local * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t* src = (j < 4) ? o0 : o1;
              const int k = 8 * (j & 3) + 2 * e;
              __nv_bfloat162 u = __floats2bfloat162_rn(__uint_as_float(src[k]), __uint_as_float(src[k + 1]));
              w[e] = *reinterpret_cast<uint32_t*>(&u);
            }
            *reinterpret_cast<uint4*>(dst + ((j ^ (r_local & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * hf + cc;
            uint32_t o[32];
            tmem_ld32(lb + COL_O + 32 * c, o);
            tmem_ld_wait();
            uint8_t* dst = so + c * HALF + r_local * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(dst + ((j ^ (r_local & 7)) << 4)) =
                  make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
          }
        }
      }
      fence_proxy_async_smem();
      bar_sync(2, 256);
      if (threadIdx.x == 0) {
        for (int i = 0; i < n_mt; ++i) {
          const int y = (bh * a.splits + split) * a.rows_pad + rb * a.rows_per_cta + i * 128;
          const int slices = a.part_bf16 ? 2 : 4;
          for (int c = 0; c < slices; ++c)
            tma_store_2d(&tm.po, smem + SM_K + i * 4 * HALF + c * HALF, (a.part_bf16 ? 64 : 32) * c, y);
        }
        bulk_commit();
        if (a.coop)
          bulk_wait0();  // other CTAs read these rows
        else
          bulk_wait_read0();
      }
      if (hf == 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (!vrow[i]) continue;
          const size_t prow = (static_cast<size_t>(bh) * a.splits + split) * a.rows_pad + rb * a.rows_per_cta + i * 128 + r_local;
          *reinterpret_cast<float2*>(a.part_ml + prow * 2) = make_float2(m_ref[i], l_tot[i]);
        }
      }
    } else if (!(a.tps > 0 && ti.n_tiles == 0)) {  // a split past its request's last unit writes nothing
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (i >= n_mt) break;
        const float inv = (a.splits == 1 && l_tot[i] > 0.f) ? 1.f / l_tot[i] : 1.f;
        const size_t prow = (static_cast<size_t>(bh) * a.splits + split) * a.rows_pad + rb * a.rows_per_cta + i * 128 + r_local;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * hf + cc;
          uint32_t o[32];
          if (all_done) {
            tmem_ld32(lb + COL_O + 32 * c, o);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = 0u;
          }
          if (!vrow[i]) continue;
          if (a.splits == 1) {
            const size_t orow = (static_cast<size_t>(b * a.R + node[i]) * a.Hq + hq[i]) * 128 + 32 * c;
            if (a.out_f32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                dst[j] = make_float4(__uint_as_float(o[4 * j]) * inv, __uint_as_float(o[4 * j + 1]) * inv,
                                     __uint_as_float(o[4 * j + 2]) * inv, __uint_as_float(o[4 * j + 3]) * inv);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + orow);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  __nv_bfloat162 u = __floats2bfloat162_rn(__uint_as_float(o[8 * j + 2 * e]) * inv,
                                                           __uint_as_float(o[8 * j + 2 * e + 1]) * inv);
                  w[e] = *reinterpret_cast<uint32_t*>(&u);
                }
                dst[j] = make_uint4(w[0], w[1], w[2], w[3]);
              }
            }
          } else if (a.part_bf16) {  // a timed-out split: zeros (its weight is 0 too)
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.part_o) + prow * 128 + 32 * c);
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = make_uint4(0u, 0u, 0u, 0u);
          } else {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.part_o) + prow * 128 + 32 * c);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(__uint_as_float(o[4 * j]), __uint_as_float(o[4 * j + 1]),
                                   __uint_as_float(o[4 * j + 2]), __uint_as_float(o[4 * j + 3]));
          }
        }
        if (vrow[i] && hf == 0) {
          if (a.splits == 1) {
            if (a.lse) a.lse[static_cast<size_t>(b * a.R + node[i]) * a.Hq + hq[i]] = a.scale * m_ref[i] + logf(l_tot[i]);
          } else {
            *reinterpret_cast<float2*>(a.part_ml + prow * 2) =
                make_float2(all_done ? m_ref[i] : -INFINITY, all_done ? l_tot[i] : 0.f);
          }
        }
      }
    }
    if (a.coop) {
      // the group's merge: publish this split's partials (all writes fenced, then one
      // release-ordered count), wait until every split of this (request, KV head, row
      // block) has counted, then merge rows [split n / S, (split + 1) n / S) of the
      // block from the partials in L2, a warp per row: M = max m_s,
      // w_s = 2^((m_s - M) c), O = sum w_s O_s / sum w_s l_s
      fence_proxy_async_global();
      __threadfence();
      bar_sync(2, 256);
      const int grp = bh * gridDim.z + rb;
      if (threadIdx.x == 0) {
        s_go = group_arrive_wait(a.cnt + grp, a.splits, a.err) ? 1 : 0;
        // past the wait: the last split of the group to get here returns both counters
        // to zero for the next call
        int* done = a.cnt + a.n_groups + grp;
        if (atomicAdd(done, 1) == a.splits - 1) {
          atomicExch(a.cnt + grp, 0);
          atomicExch(done, 0);
        }
      }
      bar_sync(2, 256);
      if (s_go) {
        const int n = min(a.rows_per_cta, a.R * a.G - rb * a.rows_per_cta);
        const int hi = (split + 1) * n / a.splits;
        // a half-warp per row; both halves of a warp loop together (shuffles are
        // warp-collective), the spare half on a row of its own block with no output
        const int lo = split * n / a.splits;
        for (int s0 = lo + 2 * warp; s0 < hi; s0 += 16) {
          const int lr = s0 + (lane >> 4);
          const int grow = lr < hi ? rb * a.rows_per_cta + lr : -1;
          if (a.part_bf16)
            merge_row_hw<true>(a, bh, h, b, grow < 0 ? -1 : grow, lane & 15, sl2);
          else
            merge_row_hw<false>(a, bh, h, b, grow < 0 ? -1 : grow, lane & 15, sl2);
        }
      }
    }
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
template <bool PRECISE>
cudaError_t configure_tc() {
  static unsigned long long configured = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && (__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & (1ull << dev))) return cudaSuccess;
  e = cudaFuncSetAttribute(tree_attn_tc_kernel<PRECISE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (dev < 64) __atomic_fetch_or(&configured, 1ull << dev, __ATOMIC_RELEASE);
  return cudaSuccess;
}

// Cooperative launch when the CTAs of a split group wait on one another (a.coop):
// the driver then guarantees that the whole grid is resident at once, or fails the
// launch.
template <bool PRECISE>
cudaError_t launch_tc(const Tmaps& tm, const TcArgs& a, dim3 grid, cudaStream_t s) {
  cudaError_t e = configure_tc<PRECISE>();
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
  e = cudaLaunchKernelEx(&cfg, tree_attn_tc_kernel<PRECISE>, tm, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tree_attn_tc(const AttnPlan& p, const void* q, const void* k_cache, const void* v_cache,
                                const void* tree_k, const void* tree_v, const int32_t* seq_len,
                                const uint64_t* anc_mask, void* out, float* lse, void* ws, cudaStream_t s) {
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
    const cuuint64_t strides[1] = {D * (p.part_bf16 ? 2 : 4)};
    const cuuint32_t box[2] = {p.part_bf16 ? 64u : 32u, 128};
    if (!make_tmap(&tm.po, p.part_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, w + p.off_o,
                   2, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  TcArgs a;
  a.seq_len = seq_len;
  a.anc_mask = anc_mask;
  a.out = out;
  a.lse = lse;
  const bool partials = p.splits > 1;
  a.part_o = partials ? static_cast<void*>(w + p.off_o) : nullptr;
  a.part_bf16 = p.part_bf16 ? 1 : 0;
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
  a.rows_per_cta = p.rows_per_cta;
  a.n_mt = p.rows_per_cta / 128;
  a.coop = p.coop ? 1 : 0;
  a.tps = p.tps;
  a.lpt = p.lpt ? 1 : 0;
  a.cnt = p.coop ? reinterpret_cast<int*>(w + p.off_cnt) : nullptr;
  a.n_groups = p.B * p.Hkv * p.row_blocks;
  a.out_f32 = p.out_dtype == EAGLE_F32;
  a.scale = p.scale;
  a.scale_log2 = p.scale * kLog2e;
  cudaError_t e;
  const dim3 grid = p.coop ? dim3(p.splits, p.B * p.Hkv, p.row_blocks) : dim3(p.row_blocks, p.splits, p.B * p.Hkv);
  e = p.precise ? launch_tc<true>(tm, a, grid, s) : launch_tc<false>(tm, a, grid, s);
  if (e != cudaSuccess || !partials || p.coop) return e;
  return launch_tree_attn_combine(p, seq_len, out, lse, static_cast<const float*>(a.part_o), a.part_ml, s);
}

}  // namespace eagle
