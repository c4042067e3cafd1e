// kv_commit.cu -- compact the accepted path into the contiguous KV cache.
//
// For every layer, request and KV head, path node m's K/V row (m = 0 is the root,
// whose K/V the verify pass computed) goes to cache row seq_len + m, and the
// logical length becomes seq_len + n_acc + 1; rejected rows are simply never
// copied (EAGLE review, section 3.3 and data path step 7: accepted tokens and
// their features are appended; lesson "KV cache rollback" and step 4).  Feature
// rows follow the same path.  The emitted correction / bonus token becomes the
// next root; its K/V comes from the next verify pass.
//
// Kernels
//   kv_commit_copy_kernel      one CTA per (request, path position m, layer): 16-byte
//                              vector copies of the K and V rows of every KV head.
//   kv_commit_finalize_kernel  one thread per request: commit positions, seq_len
//                              update, cache-full check.  A separate launch so the
//                              copies read the old seq_len.
#include "common.cuh"
#include "launch.h"

namespace eagle {
namespace {

__device__ __forceinline__ bool commit_ok(const eagle_commit_desc& d, const int32_t* n_acc, const int32_t* seq_len,
                                          int b) {
  const int na = n_acc[b];
  const int L = seq_len[b];
  return na >= 0 && na <= d.max_depth && L >= 0 && L + na + 1 <= d.max_seq;
}

__global__ void __launch_bounds__(128) kv_commit_copy_kernel(const eagle_commit_desc d, const CommitArgs a,
                                                             const int32_t* n_acc, const int32_t* path,
                                                             const int32_t* seq_len, void* feat_cache,
                                                             const void* tree_feat) {
  const int b = blockIdx.x, m = blockIdx.y, l = blockIdx.z;
  if (!commit_ok(d, n_acc, seq_len, b) || m > n_acc[b]) return;
  const int node = path[static_cast<size_t>(b) * (d.max_depth + 1) + m];
  if (node < 0 || node >= d.rows) return;  // flagged by the finalize kernel
  const int dst_row = seq_len[b] + m;
  const int esz = d.dtype == EAGLE_F32 ? 4 : 2;
  const int vec_per_row = d.head_dim * esz / 16;
  const int total = d.n_kv_heads * vec_per_row;
  const uint4* tk = static_cast<const uint4*>(a.tree_k[l]);
  const uint4* tv = static_cast<const uint4*>(a.tree_v[l]);
  uint4* kc = static_cast<uint4*>(a.k_cache[l]);
  uint4* vc = static_cast<uint4*>(a.v_cache[l]);
  for (int i = threadIdx.x; i < total; i += blockDim.x) {
    const int h = i / vec_per_row, c = i % vec_per_row;
    const size_t src = ((static_cast<size_t>(b) * d.n_kv_heads + h) * d.rows + node) * vec_per_row + c;
    const size_t dst = ((static_cast<size_t>(b) * d.n_kv_heads + h) * d.max_seq + dst_row) * vec_per_row + c;
    kc[dst] = tk[src];
    vc[dst] = tv[src];
  }
  if (l == 0 && d.feat_dim > 0 && feat_cache && tree_feat) {
    const int fsz = d.feat_dtype == EAGLE_F32 ? 4 : 2;
    const size_t row_bytes = static_cast<size_t>(d.feat_dim) * fsz;
    const uint8_t* src = static_cast<const uint8_t*>(tree_feat) + (static_cast<size_t>(b) * d.rows + node) * row_bytes;
    uint8_t* dst = static_cast<uint8_t*>(feat_cache) + (static_cast<size_t>(b) * d.max_seq + dst_row) * row_bytes;
    if (row_bytes % 16 == 0) {
      for (size_t i = threadIdx.x; i < row_bytes / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(src)[i];
    } else {
      for (size_t i = threadIdx.x; i < row_bytes; i += blockDim.x) dst[i] = src[i];
    }
  }
}

__global__ void kv_commit_finalize_kernel(const eagle_commit_desc d, const int32_t* n_acc, const int32_t* path,
                                          int32_t* seq_len, int32_t* commit_pos, uint32_t* status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= d.batch) return;
  const int maxp = d.max_depth + 1;
  const int na = n_acc[b];
  const int L = seq_len[b];
  unsigned st = 0;
  const bool ok = commit_ok(d, n_acc, seq_len, b);
  if (!ok) st |= EAGLE_STATUS_CACHE_FULL;
  for (int m = 0; m < maxp; ++m) {
    const bool on = ok && m <= na;
    if (on) {
      const int node = path[static_cast<size_t>(b) * maxp + m];
      if (node < 0 || node >= d.rows) st |= EAGLE_STATUS_BAD_TREE;
    }
    if (commit_pos) commit_pos[static_cast<size_t>(b) * maxp + m] = on ? L + m : -1;
  }
  if (ok) seq_len[b] = L + na + 1;
  if (st && status) atomicOr(status, st);
}

}  // namespace

cudaError_t launch_kv_commit(const eagle_commit_desc* d, const CommitArgs& a, const int32_t* n_acc,
                             const int32_t* path, int32_t* seq_len, int32_t* commit_pos, void* feat_cache,
                             const void* tree_feat, uint32_t* status, cudaStream_t s) {
  dim3 grid(d->batch, d->max_depth + 1, d->layers);
  kv_commit_copy_kernel<<<grid, 128, 0, s>>>(*d, a, n_acc, path, seq_len, feat_cache, tree_feat);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kv_commit_finalize_kernel<<<(d->batch + 127) / 128, 128, 0, s>>>(*d, n_acc, path, seq_len, commit_pos, status);
  return cudaGetLastError();
}

}  // namespace eagle
