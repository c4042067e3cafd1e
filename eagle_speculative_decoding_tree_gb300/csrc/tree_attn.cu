// tree_attn.cu -- tree attention over the prefix KV cache plus the draft tree's own K/V.
//
// Row i of a request attends to the prefix keys j < seq_len and to the tree keys on
// its root..i path ("each candidate attends only to its ancestors": EAGLE review,
// terms "tree attention"; lesson glossary "Tree attention": flash attention with a
// tree mask).  The ancestor set of a row is one or two 64-bit words held in
// registers and applied only on the tree tiles.
//
// bf16 path: split-KV flash decoding.  A CTA owns (request, KV head, split, row
// block); its rows are (tree node, query head in the GQA group) pairs, so all G
// query heads that share a KV head read each K/V tile once.  K/V tiles of 64 keys
// stream through a 3-stage cp.async ring in XOR-swizzled shared memory; QK^T and PV
// run on mma.sync m16n8k16 bf16 with fp32 accumulators; online softmax in the exp2
// domain with quad shuffles.  Splits write unnormalised partials (O, m, l) that
// tree_attn_combine merges with the log-sum-exp rule.
//
// fp32 path: a plain SIMT kernel, one warp per (request, node, query head).
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace eagle {
namespace {

constexpr int BN = 64;      // keys per tile
constexpr int STAGES = 3;   // cp.async ring depth

struct AttnArgs {
  const uint16_t* q;
  const uint16_t* kc;
  const uint16_t* vc;
  const uint16_t* tk;
  const uint16_t* tv;
  const int32_t* seq_len;
  const int32_t* n_nodes;  // [B] tree rows per request (NULL: all R)
  const uint64_t* anc_mask;
  void* out;       // [B][R][Hq][D], bf16 or fp32 (out_f32)
  float* lse;
  float* part_o;   // [B*Hkv][splits][rows_pad][D]
  float* part_ml;  // [B*Hkv][splits][rows_pad][2]
  int B, R, Hq, Hkv, G, P, W, splits, rows_pad;
  int tps;         // > 0: fixed-size splits of tps 128-key units (tcgen05 partials)
  int out_f32;     // 1: write fp32 output rows
  float scale, scale_log2;
};

// Store two adjacent output elements (bf16 pair or fp32 pair).
__device__ __forceinline__ void store_out2(const AttnArgs& a, size_t idx, float v0, float v1);

// Tree rows of request b: n_nodes[b] clamped to [0, R], or R without n_nodes.
__device__ __forceinline__ int request_rows(const int32_t* n_nodes, int b, int R) {
  if (!n_nodes) return R;
  const int n = n_nodes[b];
  return n < 0 ? 0 : (n > R ? R : n);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // n == 0: no bytes read, destination zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t ld_u32(const uint16_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

__device__ __forceinline__ void store_out2(const AttnArgs& a, size_t idx, float v0, float v1) {
  if (a.out_f32)
    *reinterpret_cast<float2*>(static_cast<float*>(a.out) + idx) = make_float2(v0, v1);
  else
    *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.out) + idx) = pack_bf16x2(v0, v1);
}

// Offset of 16-byte chunk `ch` of tile row `row` in a [BN][D] bf16 tile, XOR swizzled
// so that the 8 rows an ldmatrix phase reads fall in 8 different bank groups.
template <int D>
__device__ __forceinline__ uint32_t tile_off(int row, int ch) {
  return static_cast<uint32_t>(row * (D * 2) + ((ch ^ (row & 7)) << 4));
}

// PRECISE: P enters the PV product as two bf16 terms (hi + lo), about 16 significant
// bits instead of 8, for sharply peaked rows where bf16 rounding of P matters.
template <int D, int NW, bool PRECISE>
__global__ void __launch_bounds__(NW * 32, (NW == 4) ? 2 : 1) tree_attn_mma_kernel(const AttnArgs a) {
  constexpr int BM = NW * 16;
  constexpr int CH = D / 8;                  // 16-byte chunks per row
  constexpr int TILE = BN * D * 2;           // bytes of one K (or V) tile
  constexpr int KS = D / 16;                 // k-steps of QK^T
  extern __shared__ __align__(128) uint8_t smem[];

  const int rb = blockIdx.x, split = blockIdx.y, bh = blockIdx.z;
  const int b = bh / a.Hkv, h = bh % a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;

  int L = a.seq_len[b];
  L = L < 0 ? 0 : (L > a.P ? a.P : L);
  const int n_pref = (L + BN - 1) / BN;
  const int t_begin = static_cast<int>(static_cast<long long>(n_pref) * split / a.splits);
  const int t_end = static_cast<int>(static_cast<long long>(n_pref) * (split + 1) / a.splits);
  const int n_pt = t_end - t_begin;
  const int Rb = request_rows(a.n_nodes, b, a.R);
  const int n_tt = (split == a.splits - 1) ? (Rb + BN - 1) / BN : 0;
  const int n_tiles = n_pt + n_tt;

  // ---- the two rows this thread's accumulators cover (rows of nodes >= Rb are idle)
  const int RG = Rb * a.G;
  int node[2], head[2];
  bool valid[2];
  uint64_t mw[2][2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = rb * BM + warp * 16 + g + 8 * i;
    valid[i] = r < RG;
    node[i] = valid[i] ? r / a.G : 0;
    head[i] = h * a.G + (valid[i] ? r % a.G : 0);
    mw[i][0] = valid[i] ? a.anc_mask[(static_cast<size_t>(b) * a.R + node[i]) * a.W] : 0ull;
    mw[i][1] = (valid[i] && a.W > 1) ? a.anc_mask[(static_cast<size_t>(b) * a.R + node[i]) * a.W + 1] : 0ull;
  }

  // ---- Q fragments (A operand of QK^T), straight from global memory
  uint32_t qa[KS][4];
  {
    const uint16_t* q0 = a.q + (static_cast<size_t>(b * a.R + node[0]) * a.Hq + head[0]) * D;
    const uint16_t* q1 = a.q + (static_cast<size_t>(b * a.R + node[1]) * a.Hq + head[1]) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][0] = valid[0] ? ld_u32(q0 + ks * 16 + tig * 2) : 0u;
      qa[ks][1] = valid[1] ? ld_u32(q1 + ks * 16 + tig * 2) : 0u;
      qa[ks][2] = valid[0] ? ld_u32(q0 + ks * 16 + 8 + tig * 2) : 0u;
      qa[ks][3] = valid[1] ? ld_u32(q1 + ks * 16 + 8 + tig * 2) : 0u;
    }
  }

  const size_t kv_head = static_cast<size_t>(b) * a.Hkv + h;
  auto load_tile = [&](int t, int stage) {
    const uint16_t* kb;
    const uint16_t* vb;
    int start, nvalid;
    if (t < n_pt) {
      start = (t_begin + t) * BN;
      kb = a.kc + kv_head * a.P * D;
      vb = a.vc + kv_head * a.P * D;
      nvalid = L - start;
    } else {
      start = (t - n_pt) * BN;
      kb = a.tk + kv_head * a.R * D;
      vb = a.tv + kv_head * a.R * D;
      nvalid = Rb - start;
    }
    const uint32_t sk = smem_addr(smem + stage * 2 * TILE);
    for (int c = threadIdx.x; c < BN * CH; c += NW * 32) {
      const int row = c / CH, ch = c % CH;
      const bool ok = row < nvalid;
      const size_t off = ok ? (static_cast<size_t>(start + row) * D + ch * 8) : 0;
      const uint32_t o = tile_off<D>(row, ch);
      cp_async16(sk + o, kb + off, ok);
      cp_async16(sk + TILE + o, vb + off, ok);
    }
  };

  float o[D / 8][4];
#pragma unroll
  for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY};
  float l_r[2] = {0.f, 0.f};
  const float sl2 = a.scale_log2;

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < n_tiles) load_tile(s, s);
    cp_async_commit();
  }

  for (int t = 0; t < n_tiles; ++t) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    if (t + STAGES - 1 < n_tiles) load_tile(t + STAGES - 1, (t + STAGES - 1) % STAGES);
    cp_async_commit();

    const uint8_t* sK = smem + (t % STAGES) * 2 * TILE;
    const uint32_t aK = smem_addr(sK), aV = aK + TILE;

    // ---- S = Q K^T for 16 rows x 64 keys per warp
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
    const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int key = np * 16 + (mi >> 1) * 8 + rr;
        const int ch = ks * 2 + (mi & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(aK + tile_off<D>(key, ch), b0, b1, b2, b3);
        mma16816(s[2 * np], qa[ks], b0, b1);
        mma16816(s[2 * np + 1], qa[ks], b2, b3);
      }
    }

    // ---- mask: prefix tiles cut at seq_len, tree tiles by the ancestor words
    const bool is_tree = t >= n_pt;
    const int start = is_tree ? (t - n_pt) * BN : (t_begin + t) * BN;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = e >> 1;
        const int key = start + j * 8 + tig * 2 + (e & 1);
        bool ok;
        if (is_tree) {
          const uint64_t w = (key < 64) ? mw[i][0] : mw[i][1];
          ok = key < Rb && ((w >> (key & 63)) & 1ull);
        } else {
          ok = key < L;
        }
        if (!ok) s[j][e] = -INFINITY;
      }
    }

    // ---- online softmax (exp2 domain)
    float mu[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fmaxf(s[j][2 * i], s[j][2 * i + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_r[i], mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = exp2f((m_r[i] - m_use) * sl2);
      m_r[i] = m_new;
      l_r[i] *= alpha;
#pragma unroll
      for (int j = 0; j < D / 8; ++j) {
        o[j][2 * i] *= alpha;
        o[j][2 * i + 1] *= alpha;
      }
      mu[i] = m_use * sl2;
    }

    // ---- P (bf16, A operand of PV).  l accumulates exactly what PV multiplies:
    // the rounded values, or (PRECISE) hi + lo, which is p to ~16 bits.
    uint32_t pa[4][4];
    uint32_t pl[PRECISE ? 4 : 1][4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int j = 2 * kk + hf;
        const float p0 = exp2f(fmaf(s[j][0], sl2, -mu[0])), p1 = exp2f(fmaf(s[j][1], sl2, -mu[0]));
        const float p2 = exp2f(fmaf(s[j][2], sl2, -mu[1])), p3 = exp2f(fmaf(s[j][3], sl2, -mu[1]));
        const uint32_t u0 = pack_bf16x2(p0, p1);
        const uint32_t u1 = pack_bf16x2(p2, p3);
        pa[kk][2 * hf] = u0;
        pa[kk][2 * hf + 1] = u1;
        if constexpr (PRECISE) {
          const uint32_t v0 = pack_bf16x2(p0 - bf16_lo(u0), p1 - bf16_hi(u0));
          const uint32_t v1 = pack_bf16x2(p2 - bf16_lo(u1), p3 - bf16_hi(u1));
          pl[kk][2 * hf] = v0;
          pl[kk][2 * hf + 1] = v1;
          l_r[0] += (bf16_lo(u0) + bf16_lo(v0)) + (bf16_hi(u0) + bf16_hi(v0));
          l_r[1] += (bf16_lo(u1) + bf16_lo(v1)) + (bf16_hi(u1) + bf16_hi(v1));
        } else {
          l_r[0] += bf16_lo(u0) + bf16_hi(u0);
          l_r[1] += bf16_lo(u1) + bf16_hi(u1);
        }
      }
    }

    // ---- O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        const int key = kk * 16 + (mi & 1) * 8 + rr;
        const int ch = dp * 2 + (mi >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(aV + tile_off<D>(key, ch), b0, b1, b2, b3);
        mma16816(o[2 * dp], pa[kk], b0, b1);
        mma16816(o[2 * dp + 1], pa[kk], b2, b3);
        if constexpr (PRECISE) {
          mma16816(o[2 * dp], pl[kk], b0, b1);
          mma16816(o[2 * dp + 1], pl[kk], b2, b3);
        }
      }
    }
  }
  cp_async_wait<0>();

#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l_r[i] += __shfl_xor_sync(0xffffffffu, l_r[i], 1);
    l_r[i] += __shfl_xor_sync(0xffffffffu, l_r[i], 2);
  }

  if (a.splits == 1) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (!valid[i]) continue;
      const float inv = 1.f / l_r[i];
      const size_t orow = (static_cast<size_t>(b * a.R + node[i]) * a.Hq + head[i]) * D;
#pragma unroll
      for (int j = 0; j < D / 8; ++j) store_out2(a, orow + j * 8 + tig * 2, o[j][2 * i] * inv, o[j][2 * i + 1] * inv);
      if (a.lse && tig == 0)
        a.lse[static_cast<size_t>(b * a.R + node[i]) * a.Hq + head[i]] = a.scale * m_r[i] + logf(l_r[i]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = rb * BM + warp * 16 + g + 8 * i;
      if (r >= RG) continue;
      const size_t prow = (static_cast<size_t>(bh) * a.splits + split) * a.rows_pad + r;
      float* po = a.part_o + prow * D;
#pragma unroll
      for (int j = 0; j < D / 8; ++j)
        *reinterpret_cast<float2*>(po + j * 8 + tig * 2) = make_float2(o[j][2 * i], o[j][2 * i + 1]);
      if (tig == 0) *reinterpret_cast<float2*>(a.part_ml + prow * 2) = make_float2(m_r[i], l_r[i]);
    }
  }
}

// Merge split partials: M = max m_s, L = sum l_s 2^((m_s - M) c), O = sum O_s 2^((m_s - M) c) / L.
// One warp per row: lane s holds split s's (m, l) (splits <= 64, two per lane) and
// the weights travel by shuffle.  The partial rows of up to 32 splits are requested
// before any of them is used, so a row costs about one memory latency.
template <int D>
__global__ void __launch_bounds__(128) tree_attn_combine_kernel(const AttnArgs a) {
  constexpr int PER = D / 32;
  constexpr int BATCH = 16;
  // a programmatic launch: the partials belong to the preceding kernel until it ends
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 4 + warp;
  const int bh = blockIdx.y;
  const int b = bh / a.Hkv, h = bh % a.Hkv;
  if (r >= request_rows(a.n_nodes, b, a.R) * a.G) return;
  const int nd = r / a.G, hq = h * a.G + r % a.G;
  const size_t base = static_cast<size_t>(bh) * a.splits * a.rows_pad + r;
  const size_t sstride = static_cast<size_t>(a.rows_pad) * D;
  const float* po0 = a.part_o + base * D + lane * PER;
  // splits that hold units of this request (fixed-size splits: ceil(U / tps) of them,
  // U = its 128-key prefix tiles + the tree tile); the rest wrote nothing
  int n_act = a.splits;
  if (a.tps > 0) {
    int L = a.seq_len[b];
    L = L < 0 ? 0 : (L > a.P ? a.P : L);
    const int U = (L + 127) / 128 + 1;
    n_act = min(a.splits, (U + a.tps - 1) / a.tps);
  }
  float2 ml[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int s = lane + 32 * k;
    ml[k] = s < n_act ? *reinterpret_cast<const float2*>(a.part_ml + (base + static_cast<size_t>(s) * a.rows_pad) * 2)
                      : make_float2(-INFINITY, 0.f);
  }
  float v[BATCH][PER];
#pragma unroll
  for (int u = 0; u < BATCH; ++u) {
    if (u < n_act) {
      const float* po = po0 + static_cast<size_t>(u) * sstride;
      if constexpr (PER == 4) {
        const float4 t = *reinterpret_cast<const float4*>(po);
        v[u][0] = t.x;
        v[u][1] = t.y;
        v[u][2] = t.z;
        v[u][3] = t.w;
      } else {
        const float2 t = *reinterpret_cast<const float2*>(po);
        v[u][0] = t.x;
        v[u][1] = t.y;
      }
    } else {
#pragma unroll
      for (int e = 0; e < PER; ++e) v[u][e] = 0.f;
    }
  }
  const float M = warp_max(fmaxf(ml[0].x, ml[1].x));
  float w2[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) w2[k] = (ml[k].x == -INFINITY) ? 0.f : exp2f((ml[k].x - M) * a.scale_log2);
  const float Ls = warp_sum(ml[0].y * w2[0] + ml[1].y * w2[1]);
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
#pragma unroll
  for (int u = 0; u < BATCH; ++u) {
    const float w = __shfl_sync(0xffffffffu, w2[0], u);
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, v[u][e], acc[e]);
  }
  for (int s0 = BATCH; s0 < n_act; s0 += 8) {  // splits beyond the first batch: eight at a time
    float x[8][PER], wv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int s = s0 + u;
      // split s's weight sits in lane s & 31 of w2[s >> 5]
      const float w_lo = __shfl_sync(0xffffffffu, w2[0], s & 31);
      const float w_hi = __shfl_sync(0xffffffffu, w2[1], s & 31);
      wv[u] = (s >> 5) ? w_hi : w_lo;
      const bool in = s < n_act;
      const float* po = po0 + static_cast<size_t>(in ? s : 0) * sstride;
#pragma unroll
      for (int e = 0; e < PER; ++e) x[u][e] = in ? po[e] : 0.f;
      if (!in) wv[u] = 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] = fmaf(wv[u], x[u][e], acc[e]);
  }
  const float inv = 1.f / Ls;
  const size_t orow = (static_cast<size_t>(b * a.R + nd) * a.Hq + hq) * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; e += 2) store_out2(a, orow + e, acc[e] * inv, acc[e + 1] * inv);
  if (a.lse && lane == 0) a.lse[static_cast<size_t>(b * a.R + nd) * a.Hq + hq] = a.scale * M + logf(Ls);
}

// fp32 path: one warp per (request, node, query head); keys one at a time.
template <int D>
__global__ void __launch_bounds__(128) tree_attn_f32_kernel(const float* __restrict__ q, const float* __restrict__ kc,
                                                            const float* __restrict__ vc, const float* __restrict__ tk,
                                                            const float* __restrict__ tv, const int32_t* seq_len,
                                                            const int32_t* n_nodes, const uint64_t* anc_mask,
                                                            float* out, float* lse, int B,
                                                            int R, int Hq, int Hkv, int P, int W, float scale) {
  constexpr int PER = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long id = static_cast<long long>(blockIdx.x) * 4 + warp;
  if (id >= static_cast<long long>(B) * R * Hq) return;
  const int hq = static_cast<int>(id % Hq);
  const int i = static_cast<int>((id / Hq) % R);
  const int b = static_cast<int>(id / (static_cast<long long>(Hq) * R));
  const int G = Hq / Hkv, h = hq / G;
  const int Rb = request_rows(n_nodes, b, R);
  if (i >= Rb) return;  // rows past the request's tree are not computed
  int L = seq_len[b];
  L = L < 0 ? 0 : (L > P ? P : L);
  float qv[PER], ov[PER];
  const float* qrow = q + (static_cast<size_t>(b * R + i) * Hq + hq) * D;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    qv[e] = qrow[lane * PER + e];
    ov[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  auto visit = [&](const float* krow, const float* vrow) {
    float d = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) d = fmaf(qv[e], krow[lane * PER + e], d);
    d = warp_sum(d) * scale;
    const float mn = fmaxf(m, d);
    const float corr = expf(m - mn);
    const float p = expf(d - mn);
    l = l * corr + p;
#pragma unroll
    for (int e = 0; e < PER; ++e) ov[e] = ov[e] * corr + p * vrow[lane * PER + e];
    m = mn;
  };
  const size_t kvh = static_cast<size_t>(b) * Hkv + h;
  for (int j = 0; j < L; ++j) visit(kc + (kvh * P + j) * D, vc + (kvh * P + j) * D);
  for (int t = 0; t < Rb; ++t) {
    const uint64_t w = anc_mask[(static_cast<size_t>(b) * R + i) * W + (t >> 6)];
    if ((w >> (t & 63)) & 1ull) visit(tk + (kvh * R + t) * D, tv + (kvh * R + t) * D);
  }
  float* orow = out + (static_cast<size_t>(b * R + i) * Hq + hq) * D;
#pragma unroll
  for (int e = 0; e < PER; ++e) orow[lane * PER + e] = ov[e] / l;
  if (lse && lane == 0) lse[static_cast<size_t>(b * R + i) * Hq + hq] = m + logf(l);
}

template <int D, int NW, bool PRECISE>
cudaError_t launch_mma(const AttnPlan& p, const AttnArgs& args, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(STAGES) * 2 * BN * D * 2;
  auto kern = tree_attn_mma_kernel<D, NW, PRECISE>;
  // opt in to > 48 KB of dynamic shared memory once per device (not a stream operation)
  static unsigned long long configured = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & (1ull << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&configured, 1ull << dev, __ATOMIC_RELEASE);
  } else if (dev >= 64) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  dim3 grid(p.row_blocks, p.splits, p.B * p.Hkv);
  kern<<<grid, NW * 32, smem, s>>>(args);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.splits == 1) return e;
  dim3 cgrid((p.R * p.G + 3) / 4, p.B * p.Hkv);
  tree_attn_combine_kernel<D><<<cgrid, 128, 0, s>>>(args);
  return cudaGetLastError();
}

}  // namespace

void plan_tree_attn(const eagle_attn_desc* d, int num_sms, AttnPlan* p) {
  p->B = d->batch;
  p->R = d->rows;
  p->Hq = d->n_q_heads;
  p->Hkv = d->n_kv_heads;
  p->G = d->n_q_heads / d->n_kv_heads;
  p->D = d->head_dim;
  p->P = d->max_seq;
  p->dtype = d->dtype;
  p->W = (d->rows + 63) / 64;
  p->scale = d->scale;
  p->out_dtype = d->out_dtype;
  p->precise = d->precision == EAGLE_ATTN_PRECISE;
  p->fault_test = d->fault_test == 1;
  p->off_err = p->off_cnt = p->off_o = p->off_ml = p->total = 0;
  p->tc = false;
  p->coop = false;
  p->tps = 0;
  p->lpt = false;
  const int RG = p->R * p->G;
  if (p->dtype == EAGLE_F32) {
    p->rows_per_cta = 4;
    p->row_blocks = 1;
    p->splits = 1;
    p->rows_pad = RG;
    return;
  }
  // tcgen05 kernel: bf16, D = 128, M-tiles of 128 rows that hold whole nodes.
  p->tc = d->engine == EAGLE_ENGINE_AUTO && p->D == 128 && (128 % p->G) == 0;
  int key_tile, slots_per_sm;
  if (p->tc) {
    p->rows_per_cta = 128;  // one M-tile: TMEM holds two S buffers and two O accumulators
    key_tile = 128;
    slots_per_sm = 1;  // one CTA per SM: it holds all 512 TMEM columns
  } else {
    const int nw = (RG <= 64) ? 4 : 8;
    p->rows_per_cta = nw * 16;
    key_tile = BN;
    slots_per_sm = (nw == 4) ? 2 : 1;
  }
  p->row_blocks = (RG + p->rows_per_cta - 1) / p->rows_per_cta;
  p->rows_pad = p->row_blocks * p->rows_per_cta;
  const int max_tiles = (p->P + key_tile - 1) / key_tile;
  const int base = std::max(1, p->B * p->Hkv * p->row_blocks);
  int splits = d->num_splits;
  if (splits <= 0) splits = num_sms * slots_per_sm / base;
  if (splits > max_tiles) splits = max_tiles;
  if (splits > 64) splits = 64;
  if (splits < 1) splits = 1;
  // tcgen05 with splits: when the whole grid fits on the SMs at once (one CTA per SM)
  // the kernel merges the partials itself (cooperative launch); else the combine
  // kernel does.
  p->coop = p->tc && splits > 1 && static_cast<long long>(base) * splits <= num_sms;
  if (p->tc && !p->coop && d->num_splits <= 0) {
    // more groups than a cooperative grid holds (batched, ragged requests): each
    // request's key range is cut into fixed pieces of T 128-key units (the tree tile
    // counts as one), so a long request spreads over several CTAs and a short one
    // takes few; T = 32 while the groups alone fill under two waves of SMs, else 64,
    // and larger when a request would need more than 64 pieces.  Up to 64 requests,
    // the longest are dispatched first (each CTA ranks the lengths: B^2 / 32 steps).
    const int units = max_tiles + 1;
    int T = (base < 2 * num_sms) ? 32 : 64;
    if ((units + T - 1) / T > 64) T = (units + 63) / 64;
    const int s2 = (units + T - 1) / T;
    if (s2 > 1) {
      splits = s2;
      p->tps = T;
    }
    p->lpt = p->B > 1 && p->B <= 64;
  }
  p->splits = splits;
  size_t off = p->tc ? 256 : 0;  // tcgen05: error word first
  if (p->coop) {
    p->off_cnt = off;
    off += (static_cast<size_t>(base) * 8 + 255) / 256 * 256;  // published / finished counts
  }
  if (splits > 1) {
    const size_t rows = static_cast<size_t>(p->B) * p->Hkv * splits * p->rows_pad;
    p->off_o = off;
    off += ((rows * p->D * 4) + 255) / 256 * 256;  // fp32 partial O
    p->off_ml = off;
    off += rows * 2 * 4;
  }
  p->total = off;
}

cudaError_t launch_tree_attn_combine(const AttnPlan& p, const int32_t* seq_len, const int32_t* n_nodes, void* out,
                                     float* lse, const float* part_o, const float* part_ml, cudaStream_t s, bool pdl) {
  AttnArgs a{};
  a.seq_len = seq_len;
  a.n_nodes = n_nodes;
  a.tps = p.tps;
  a.out = out;
  a.lse = lse;
  a.part_o = const_cast<float*>(part_o);
  a.part_ml = const_cast<float*>(part_ml);
  a.B = p.B;
  a.R = p.R;
  a.Hq = p.Hq;
  a.Hkv = p.Hkv;
  a.G = p.G;
  a.P = p.P;
  a.W = p.W;
  a.splits = p.splits;
  a.rows_pad = p.rows_pad;
  a.out_f32 = p.out_dtype == EAGLE_F32;
  a.scale = p.scale;
  a.scale_log2 = p.scale * kLog2e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.R * p.G + 3) / 4, p.B * p.Hkv);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = p.D == 64 ? cudaLaunchKernelEx(&cfg, tree_attn_combine_kernel<64>, a)
                            : cudaLaunchKernelEx(&cfg, tree_attn_combine_kernel<128>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_tree_attn(const AttnPlan& p, const void* q, const void* k_cache, const void* v_cache,
                             const void* tree_k, const void* tree_v, const int32_t* seq_len, const int32_t* n_nodes,
                             const uint64_t* anc_mask, void* out, float* lse, void* ws, cudaStream_t s) {
  if (p.tc)
    return launch_tree_attn_tc(p, q, k_cache, v_cache, tree_k, tree_v, seq_len, n_nodes, anc_mask, out, lse, ws, s);
  if (p.dtype == EAGLE_F32) {
    const long long rows = static_cast<long long>(p.B) * p.R * p.Hq;
    const int grid = static_cast<int>((rows + 3) / 4);
    if (p.D == 64)
      tree_attn_f32_kernel<64><<<grid, 128, 0, s>>>(
          static_cast<const float*>(q), static_cast<const float*>(k_cache), static_cast<const float*>(v_cache),
          static_cast<const float*>(tree_k), static_cast<const float*>(tree_v), seq_len, n_nodes, anc_mask,
          static_cast<float*>(out), lse, p.B, p.R, p.Hq, p.Hkv, p.P, p.W, p.scale);
    else
      tree_attn_f32_kernel<128><<<grid, 128, 0, s>>>(
          static_cast<const float*>(q), static_cast<const float*>(k_cache), static_cast<const float*>(v_cache),
          static_cast<const float*>(tree_k), static_cast<const float*>(tree_v), seq_len, n_nodes, anc_mask,
          static_cast<float*>(out), lse, p.B, p.R, p.Hq, p.Hkv, p.P, p.W, p.scale);
    return cudaGetLastError();
  }
  AttnArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.kc = static_cast<const uint16_t*>(k_cache);
  a.vc = static_cast<const uint16_t*>(v_cache);
  a.tk = static_cast<const uint16_t*>(tree_k);
  a.tv = static_cast<const uint16_t*>(tree_v);
  a.seq_len = seq_len;
  a.n_nodes = n_nodes;
  a.anc_mask = anc_mask;
  a.out = out;
  a.out_f32 = p.out_dtype == EAGLE_F32;
  a.lse = lse;
  a.part_o = p.splits > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + p.off_o) : nullptr;
  a.part_ml = p.splits > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + p.off_ml) : nullptr;
  a.B = p.B;
  a.R = p.R;
  a.Hq = p.Hq;
  a.Hkv = p.Hkv;
  a.G = p.G;
  a.P = p.P;
  a.W = p.W;
  a.splits = p.splits;
  a.rows_pad = p.rows_pad;
  a.tps = 0;
  a.scale = p.scale;
  a.scale_log2 = p.scale * kLog2e;
  const int nw = p.rows_per_cta / 16;
  if (p.precise) {
    if (p.D == 64) return nw == 4 ? launch_mma<64, 4, true>(p, a, s) : launch_mma<64, 8, true>(p, a, s);
    return nw == 4 ? launch_mma<128, 4, true>(p, a, s) : launch_mma<128, 8, true>(p, a, s);
  }
  if (p.D == 64) return nw == 4 ? launch_mma<64, 4, false>(p, a, s) : launch_mma<64, 8, false>(p, a, s);
  return nw == 4 ? launch_mma<128, 4, false>(p, a, s) : launch_mma<128, 8, false>(p, a, s);
}

}  // namespace eagle
