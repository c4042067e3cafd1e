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
constexpr int kMaxTreeChunks = 128; // tree build: vocabulary <= 128 * 4096 = 524288 tokens
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
};

// ------------------------------------------------------------------ float-float
// A value held as an unevaluated sum hi + lo of two floats (|lo| <= ulp(hi) / 2), about
// 48 significant bits, computed with error-free transformations (Knuth's TwoSum, and
// a product whose rounding error an fma recovers) on the fp32 pipe.  Used instead of
// double where sums must stay far below 1e-7 of the total: this GPU's fp64 pipe is
// narrow, while these operations are a handful of fp32 instructions.
struct ff {
  float hi, lo;
};

__device__ __forceinline__ ff ff_make(float a) { return ff{a, 0.f}; }

// a + b exactly as s + e (any magnitudes).
__device__ __forceinline__ ff two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  const float e = (a - (s - bb)) + (b - bb);
  return ff{s, e};
}

// a + b exactly as s + e, given |a| >= |b| (or a == 0).
__device__ __forceinline__ ff fast_two_sum(float a, float b) {
  const float s = a + b;
  return ff{s, b - (s - a)};
}

__device__ __forceinline__ ff ff_add(ff a, ff b) {
  const ff s = two_sum(a.hi, b.hi);
  return fast_two_sum(s.hi, s.lo + (a.lo + b.lo));
}

__device__ __forceinline__ ff ff_add(ff a, float b) {
  const ff s = two_sum(a.hi, b);
  return fast_two_sum(s.hi, s.lo + a.lo);
}

__device__ __forceinline__ ff ff_neg(ff a) { return ff{-a.hi, -a.lo}; }
__device__ __forceinline__ ff ff_sub(ff a, ff b) { return ff_add(a, ff_neg(b)); }

// a * b for a float b.
__device__ __forceinline__ ff ff_mul(ff a, float b) {
  const float p = a.hi * b;
  float e = fmaf(a.hi, b, -p);
  e = fmaf(a.lo, b, e);
  return fast_two_sum(p, e);
}

// a * b for float-float a and b (the hi products' rounding error recovered by fma).
__device__ __forceinline__ ff ff_mul(ff a, ff b) {
  const float p = a.hi * b.hi;
  float e = fmaf(a.hi, b.hi, -p);
  e = fmaf(a.hi, b.lo, e);
  e = fmaf(a.lo, b.hi, e);
  return fast_two_sum(p, e);
}

// a / b for b != 0: a first quotient q1 = a.hi / b.hi, then the remainder a - q1 b
// divided again; about 44 significant bits.
__device__ __forceinline__ ff ff_div(ff a, ff b) {
  const float q1 = a.hi / b.hi;
  const ff r = ff_add(a, ff_neg(ff_mul(b, q1)));
  return fast_two_sum(q1, r.hi / b.hi);
}

__device__ __forceinline__ bool ff_gt(ff a, ff b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }
__device__ __forceinline__ float ff_float(ff a) { return a.hi + a.lo; }

__device__ __forceinline__ ff ff_shfl_xor(ff v, int o) {
  return ff{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ ff warp_sum_ff(ff v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = ff_add(v, ff_shfl_xor(v, o));
  return v;
}

// A compensated fp32 sum as a float-float value.
__device__ __forceinline__ ff csum_ff(const CSum& a) { return two_sum(a.s, a.c); }

// (value desc, index asc) order: true if (va, ia) comes before (vb, ib).
__device__ __forceinline__ bool before(float va, int ia, float vb, int ib) {
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
