// common.cuh -- device helpers shared by the libeagle kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/eagle.h"

namespace eagle {

constexpr float kNearTieEps = 1e-5f;
constexpr int kMaxRows = 128;     // tree rows incl. root
constexpr int kMaxTopK = 16;      // children per frontier node
constexpr int kMaxDepth = 16;     // draft levels
constexpr int kMaxPool = 2048;    // dynamic-tree candidate pool per request
constexpr int kVocabChunk = 4096; // elements of a logit row per CTA in the vocabulary passes
constexpr int kMaxVocabTiles = 512;  // vocabulary <= 512 * 4096 = 2M tokens
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }

// One element of a logit / activation row as float (bf16 widened exactly).
__device__ __forceinline__ float load_elem(const void* base, size_t i, int dtype) {
  if (dtype == EAGLE_F32) return __ldg(reinterpret_cast<const float*>(base) + i);
  return bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(base) + i));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Neumaier-compensated fp32 accumulation (Neumaier 1974): a running sum and the
// rounding error it has dropped, so a thread's partial sum is exact to ~1 ulp.
struct CSum {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float t = s + x;
    c += (fabsf(s) >= fabsf(x)) ? ((s - t) + x) : ((x - t) + s);
    s = t;
  }
  __device__ __forceinline__ void scale(float f) {
    s *= f;
    c *= f;
  }
  __device__ __forceinline__ double total() const { return static_cast<double>(s) + static_cast<double>(c); }
};

// (value desc, index asc) order: true if (va, ia) comes before (vb, ib).
__device__ __forceinline__ bool before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}
__device__ __forceinline__ bool before(double va, int ia, double vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Merge an online-softmax pair (m, s): s is a sum of exp((x - m) * c).
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2, float c) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  if (m2 > m) {
    s = s * exp2f((m - m2) * c) + s2;
    m = m2;
  } else {
    s = s + s2 * exp2f((m2 - m) * c);
  }
}

}  // namespace eagle
