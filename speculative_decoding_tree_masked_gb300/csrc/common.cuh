// Shared device helpers of the tree-verification kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "treeverify.h"

namespace tv {

constexpr int kMaxNodes = TV_MAX_NODES;
constexpr int kMaskWords = kMaxNodes / 32;

// First device-side error wins; the caller clears the word.
__device__ __forceinline__ void report(int32_t* dev_status, int32_t code) {
  if (dev_status != nullptr) atomicCAS(dev_status, 0, code);
}

// Checked build (-DTV_CHECKED=1): guard(ok, st) records TV_ERR_BOUNDS when
// an index test fails and returns false, so that the caller skips the
// access.  In a normal build it is the constant true and the test vanishes.
#ifndef TV_CHECKED
#define TV_CHECKED 0
#endif
__device__ __forceinline__ bool guard(bool ok, int32_t* dev_status) {
  if (!TV_CHECKED) return true;
  if (!ok) report(dev_status, TV_ERR_BOUNDS);
  return ok;
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_f32(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_f32(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Ancestor bitmask of tree node i (itself included), following parent
// pointers held in shared memory.  Every step must go to a strictly smaller
// index, so the walk ends within i + 1 steps; a parent outside [-1, u) makes
// the function return false (the bits gathered so far are kept).
__device__ __forceinline__ bool ancestor_bits(const int32_t* parent, int i,
                                              uint32_t (&bits)[kMaskWords]) {
#pragma unroll
  for (int w = 0; w < kMaskWords; ++w) bits[w] = 0u;
  int u = i;
  while (u >= 0) {
#pragma unroll
    for (int w = 0; w < kMaskWords; ++w)
      bits[w] |= ((u >> 5) == w) ? (1u << (u & 31)) : 0u;
    const int p = parent[u];
    if (p < -1 || p >= u) return false;
    u = p;
  }
  return true;
}

__device__ __forceinline__ bool mask_bit(const uint32_t (&bits)[kMaskWords], int t) {
  uint32_t w = bits[0];
#pragma unroll
  for (int k = 1; k < kMaskWords; ++k) w = ((t >> 5) == k) ? bits[k] : w;
  return (w >> (t & 31)) & 1u;
}

}  // namespace tv
