// lmhead_stats.cu -- what acceptance needs from the target model's distribution at every
// tree node, computed from the hidden states and the LM head without writing the logits.
//
// The verify pass's frozen LM head gives the distribution at each node (EAGLE review,
// "GPU / system data path", steps 3 and 6); the multi-round test reads the target
// probability of each child's token, and the bonus draw reads the distribution (section
// 3.3 / Algorithm 1).  For hidden rows H [M][h] (M <= 128) and the head W [V][h], both
// bf16, logits x = H W^T with fp32 accumulation; per row and per tile of 128 vocabulary
// entries this kernel writes the max logit, its index (lowest on ties) and
// sum exp((x - max) / T) as a float-float pair, and each tree node's token logit under
// its parent's row.  Nothing of the [M][V] logits leaves the SM.
//
// One persistent CTA per SM walks vocabulary tiles t = blockIdx.x, blockIdx.x + gridDim.x,
// ...; 192 threads, warp-specialised:
//   warp 4     TMA producer: per 64 hidden dims, the H slice [128 rows][64] and the W slice
//              [128 vocabulary rows][64] (128-byte swizzle) into a ring of stages.
//   warp 5     allocates 256 TMEM columns and issues tcgen05.mma from lane 0:
//              D(t & 1) = H W(t)^T over h / 16 K-steps, two accumulators so that a tile's
//              epilogue overlaps the next tile's products.
//   warps 0-3  epilogue: thread r = TMEM lane r = hidden row r reads its 128 logits of the
//              tile, forms the tile record, and picks out the children's token logits.
// The kernel is bound by the head's bytes (V h 2 bytes, read once); the tensor pipe
// is about a third busy at M <= 128.
//
// Every wait is bounded (2 s); a timeout ORs EAGLE_STATUS_TIMEOUT into the status word
// and the roles stop.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <limits.h>

#include "common.cuh"
#include "launch.h"
#include "sm100.cuh"

namespace eagle {
namespace {

using namespace sm100;

constexpr int NT = 128;                 // vocabulary entries per tile (MMA N)
constexpr int KS = 64;                  // hidden dims per ring stage
constexpr int SLICE = 128 * KS * 2;     // one 128-row x 64-dim bf16 slice: 16 KB
constexpr int STAGE = 2 * SLICE;        // H slice + W slice
constexpr int NSTAGE = 6;
constexpr int SMEM_BYTES = NSTAGE * STAGE + 1024;
constexpr int NTHREADS = 192;

struct LmArgs {
  const int32_t* tokens;  // [M] tree tokens (row b R + i), nullable
  const int32_t* parent;  // [M]
  eagle_vocab_record* rec;  // [M][n_tiles]
  float* child;           // [M] nullable
  uint32_t* status;
  int M, h, V, R, n_tiles;
  int h_bytes;  // bytes of one H slice: its box has M rows rounded up to 8
  float invT;
  TreeChunkRecord* trec;  // tree-build records (nullable): one per (row, CTA)
  int F, f_max;
};

struct LmMaps {
  CUtensorMap H;  // [M][h] bf16, box {64, 128}
  CUtensorMap W;  // [V][h] bf16, box {64, 128}
};

__device__ __forceinline__ bool lm_wait(uint64_t* bar, uint32_t parity, uint32_t* status) {
  if (wait_parity(bar, parity, nullptr, 0)) return true;
  atomicOr(status, EAGLE_STATUS_TIMEOUT);
  return false;
}

template <bool TREC>
__global__ void __launch_bounds__(NTHREADS, 1) lmhead_stats_kernel(const __grid_constant__ LmMaps tm,
                                                                  const LmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[NSTAGE], empty[NSTAGE], d_full[2], d_empty[2];
  __shared__ uint32_t tmem_base;
  __shared__ int s_tok[128], s_par[128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ksteps = a.h / KS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(&d_full[j], 1);
      mbar_init(&d_empty[j], 128);
    }
    fence_barrier_init();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tmap(&tm.H);
    prefetch_tmap(&tm.W);
  }
  if (warp == 5) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  for (int i = threadIdx.x; i < 128; i += NTHREADS) {
    s_tok[i] = (a.tokens && i < a.M) ? a.tokens[i] : -1;
    s_par[i] = (a.tokens && i < a.M) ? a.parent[i] : -1;
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base;
  int n_my = 0;  // tiles of this CTA
  for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x) ++n_my;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t once = policy_evict_first();  // each W slice is read once
      int it = 0;  // ring use counter over all (tile, k) slices
      bool ok = true;
      for (int j = 0; j < n_my && ok; ++j) {
        const int t = blockIdx.x + j * gridDim.x;
        for (int k = 0; k < ksteps; ++k, ++it) {
          const int s = it % NSTAGE, use = it / NSTAGE;
          if (use > 0 && !lm_wait(&empty[s], (use - 1) & 1, a.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], a.h_bytes + SLICE);
          tma_load_2d(smem + s * STAGE, &tm.H, k * KS, 0, &full[s]);
          tma_load_2d_hint(smem + s * STAGE + SLICE, &tm.W, k * KS, t * NT, &full[s], once);
        }
      }
      // drain: no copy of this CTA's may still be landing when it exits
      const int issued = it;
      for (int s = 0; s < NSTAGE && issued > 0; ++s) {
        const int n_s = issued > s ? (issued - 1 - s) / NSTAGE + 1 : 0;
        if (n_s > 0) (void)wait_parity(&full[s], (n_s - 1) & 1, nullptr, 0);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, NT, 0, 0);
      int it = 0;
      bool ok = true;
      for (int j = 0; j < n_my && ok; ++j) {
        const int buf = j & 1;
        if (j >= 2 && !lm_wait(&d_empty[buf], ((j >> 1) - 1) & 1, a.status)) break;
        tc_fence_after();
        for (int k = 0; k < ksteps; ++k, ++it) {
          const int s = it % NSTAGE;
          if (!lm_wait(&full[s], (it / NSTAGE) & 1, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * STAGE), sb = sa + SLICE;
#pragma unroll
          for (int kk = 0; kk < KS / 16; ++kk)
            mma_ss(tb + buf * NT, smem_desc_sw128(sa + kk * 32, 16, 1024), smem_desc_sw128(sb + kk * 32, 16, 1024),
                   idesc, (k > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&empty[s]);
        }
        if (ok) mma_commit(&d_full[buf]);
      }
    }
  } else if constexpr (TREC) {
    // ------------------------------------------------------------ epilogue, tree records
    // this row's running max, float-float sum exp(x - max) and best 16 (value desc, id
    // asc) over the CTA's tiles, 32 columns at a time; tiles and columns come in
    // increasing vocabulary order, so an equal value never displaces a lower id
    const int r = warp * 32 + lane;  // hidden row = TMEM lane
    const uint32_t lb = tb + (static_cast<uint32_t>(warp * 32) << 16);
    float run_m = -INFINITY;
    ff run_s = ff_make(0.f);
    float tv[16];
    int ti[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      tv[q] = -INFINITY;
      ti[q] = INT_MAX;
    }
    for (int j = 0; j < n_my; ++j) {
      const int t = blockIdx.x + j * gridDim.x;
      const int buf = j & 1;
      const bool got = __all_sync(0xffffffffu, lm_wait(&d_full[buf], (j >> 1) & 1, a.status));
      if (!got) break;
      tc_fence_after();
      // the whole accumulator first, so that the MMA may reuse it while this tile is
      // folded in
      float x[NT];
#pragma unroll
      for (int c = 0; c < NT / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(lb + buf * NT + 32 * c, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) x[32 * c + e] = __uint_as_float(v[e]);
      }
      tc_fence_before();
      mbar_arrive(&d_empty[buf]);
      if (r >= a.M) continue;
      const int base = t * NT;
      const int nv = min(NT, a.V - base);
#pragma unroll
      for (int c = 0; c < NT / 32; ++c) {
        const int lim = nv - 32 * c;  // valid columns of this slice
        float cm = -INFINITY;
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (e < lim) cm = fmaxf(cm, x[32 * c + e]);
        if (cm == -INFINITY) continue;
        if (cm > run_m) {
          run_s = (run_m == -INFINITY) ? ff_make(0.f) : ff_mul(run_s, expf(run_m - cm));
          run_m = cm;
        }
        CSum acc;
        uint32_t cand = 0u;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          if (e < lim) {
            acc.add(expf(x[32 * c + e] - run_m));
            cand |= (x[32 * c + e] > tv[15]) ? (1u << e) : 0u;
          }
        }
        run_s = ff_add(run_s, csum_ff(acc));
        while (cand) {  // rare after the first tiles: insert into the sorted list
          const int e = __ffs(cand) - 1;
          cand &= cand - 1u;
          float val = 0.f;
#pragma unroll
          for (int q = 0; q < 32; ++q) val = (q == e) ? x[32 * c + q] : val;
          if (!(val > tv[15])) continue;  // the list has moved on since the mask
          const int id = base + 32 * c + e;
#pragma unroll
          for (int q = 15; q > 0; --q) {
            const bool sh = val > tv[q - 1];
            const bool at = !sh && val > tv[q];
            tv[q] = sh ? tv[q - 1] : (at ? val : tv[q]);
            ti[q] = sh ? ti[q - 1] : (at ? id : ti[q]);
          }
          if (val > tv[0]) {
            tv[0] = val;
            ti[0] = id;
          }
        }
      }
    }
    if (r < a.M) {
      const int b = r / a.F, f = r % a.F;
      TreeChunkRecord* o = a.trec + (static_cast<size_t>(b) * a.f_max + f) * gridDim.x + blockIdx.x;
      float4* ov = reinterpret_cast<float4*>(o->tv);
      int4* oi = reinterpret_cast<int4*>(o->ti);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        ov[q] = make_float4(tv[4 * q], tv[4 * q + 1], tv[4 * q + 2], tv[4 * q + 3]);
        oi[q] = make_int4(ti[4 * q], ti[4 * q + 1], ti[4 * q + 2], ti[4 * q + 3]);
      }
      *reinterpret_cast<float4*>(&o->s1_hi) = make_float4(run_s.hi, run_s.lo, run_s.hi, run_s.lo);
      o->m = run_m;
    }
  } else {
    // ------------------------------------------------------------ epilogue, warps 0-3
    const int r = warp * 32 + lane;  // hidden row = TMEM lane
    const uint32_t lb = tb + (static_cast<uint32_t>(warp * 32) << 16);
    const int R = a.R;
    const int node = R > 0 ? r % R : 0, req = R > 0 ? r / R : 0;
    for (int j = 0; j < n_my; ++j) {
      const int t = blockIdx.x + j * gridDim.x;
      const int buf = j & 1;
      const bool got = __all_sync(0xffffffffu, lm_wait(&d_full[buf], (j >> 1) & 1, a.status));
      if (!got) break;
      tc_fence_after();
      float x[NT];
#pragma unroll
      for (int c = 0; c < NT / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(lb + buf * NT + 32 * c, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) x[32 * c + e] = __uint_as_float(v[e]);
      }
      tc_fence_before();
      mbar_arrive(&d_empty[buf]);
      if (r >= a.M) continue;
      const int base = t * NT;
      const int nv = min(NT, a.V - base);
      // max and argmax (lowest index on ties), then the compensated sum
      float m = -INFINITY;
      int am = INT_MAX;
#pragma unroll
      for (int e = 0; e < NT; ++e) {
        if (e < nv && x[e] > m) {
          m = x[e];
          am = base + e;
        }
      }
      CSum acc;
#pragma unroll
      for (int e = 0; e < NT; ++e)
        if (e < nv) acc.add(expf((x[e] - m) * a.invT));
      const ff s = csum_ff(acc);
      eagle_vocab_record out;
      out.max = m;
      out.argmax = am;
      out.sum_hi = s.hi;
      out.sum_lo = s.lo;
      a.rec[static_cast<size_t>(r) * a.n_tiles + t] = out;
      // the children of this row's node whose token falls in the tile: the logit of that
      // token under this row is what their acceptance test reads
      if (a.child) {
        for (int i = 0; i < R; ++i) {
          const int row_i = req * R + i;
          const int d = s_tok[row_i] - base;
          if (i > 0 && s_par[row_i] == node && d >= 0 && d < nv) {
            float val = 0.f;
#pragma unroll
            for (int e = 0; e < NT; ++e) val = (e == d) ? x[e] : val;
            a.child[row_i] = val;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tb, 256);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 lm_encode_fn() {
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

// box_rows: the H slices cover only the M rows (rounded up to 8): a box that is mostly
// out of bounds slowed the loads; the accumulator rows past them are never read.
bool lm_tmap(CUtensorMap* m, const void* base, int rows, int h, int box_rows = 128) {
  auto fn = lm_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(h), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(h) * 2};
  const cuuint32_t box[2] = {KS, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int lmhead_tiles(int vocab) { return (vocab + NT - 1) / NT; }

cudaError_t launch_lmhead_stats(int M, int h, int V, int R, float temperature, const void* hidden, const void* weight,
                                const int32_t* tokens, const int32_t* parent, eagle_vocab_record* rec, float* child,
                                uint32_t* status, int num_sms, cudaStream_t s) {
  LmMaps tm;
  const int hrows = (M + 7) / 8 * 8;
  if (!lm_tmap(&tm.H, hidden, M, h, hrows) || !lm_tmap(&tm.W, weight, V, h)) return cudaErrorInvalidValue;
  LmArgs a;
  a.tokens = tokens;
  a.parent = parent;
  a.rec = rec;
  a.child = child;
  a.status = status;
  a.M = M;
  a.h = h;
  a.V = V;
  a.R = R;
  a.n_tiles = lmhead_tiles(V);
  a.h_bytes = hrows * KS * 2;
  a.invT = 1.f / (temperature > 0.f ? temperature : 1.f);
  a.trec = nullptr;
  a.F = 1;
  a.f_max = 1;
  static unsigned long long configured = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & (1ull << dev))) {
    e = cudaFuncSetAttribute(lmhead_stats_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 64) __atomic_fetch_or(&configured, 1ull << dev, __ATOMIC_RELEASE);
  }
  const int grid = a.n_tiles < num_sms ? a.n_tiles : num_sms;
  lmhead_stats_kernel<false><<<grid, NTHREADS, SMEM_BYTES, s>>>(tm, a);
  return cudaGetLastError();
}

cudaError_t launch_lmhead_tree_records(int M, int h, int V, int F, int f_max, int n_rec, const void* hidden,
                                       const void* weight, TreeChunkRecord* trec, uint32_t* status, cudaStream_t s) {
  LmMaps tm;
  const int hrows = (M + 7) / 8 * 8;
  if (!lm_tmap(&tm.H, hidden, M, h, hrows) || !lm_tmap(&tm.W, weight, V, h)) return cudaErrorInvalidValue;
  LmArgs a;
  a.tokens = nullptr;
  a.parent = nullptr;
  a.rec = nullptr;
  a.child = nullptr;
  a.status = status;
  a.M = M;
  a.h = h;
  a.V = V;
  a.R = 0;
  a.n_tiles = lmhead_tiles(V);
  a.h_bytes = hrows * KS * 2;
  a.invT = 1.f;  // the tree ranks at T = 1
  a.trec = trec;
  a.F = F;
  a.f_max = f_max;
  static unsigned long long configured = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & (1ull << dev))) {
    e = cudaFuncSetAttribute(lmhead_stats_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 64) __atomic_fetch_or(&configured, 1ull << dev, __ATOMIC_RELEASE);
  }
  lmhead_stats_kernel<true><<<n_rec, NTHREADS, SMEM_BYTES, s>>>(tm, a);
  return cudaGetLastError();
}

}  // namespace eagle
