// Split-KV planning and the combine step of tree-masked attention.
//
// Flash-decoding: the key range [0, P + N) of every (KV head, row tile) is cut
// into `splits` chunks processed by different CTAs; each writes an unnormalised
// partial output with its row maximum and row sum, and the combine kernel
// merges them with log-sum-exp weights:
//   O = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s,   M = max_s m_s.
// (m in log2 units: scores are pre-multiplied by scale * log2(e).)
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace tv {

namespace {
constexpr int kSimtRows = 16;     // rows per CTA of the fp32 kernel
constexpr int kSimtKeys = 32;     // key tile of the fp32 kernel
constexpr int kSimtCtasPerSm = 4;
constexpr int kTcRowsPerTile = 128;
constexpr int kTcKeys = 128;      // key block of the tensor-core kernel
constexpr int kTcCtasPerSm = 1;

int cached_sm[64];
}  // namespace

// The bf16 tensor-core kernel is switched in once it is built.
constexpr bool kTensorCorePath = true;

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached_sm[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached_sm[dev] = v;
  }
  return cached_sm[dev];
}

bool use_tensor_cores(int32_t dtype) { return dtype == TV_BF16 && kTensorCorePath; }

SplitPlan plan_attention(int32_t n, int32_t hq, int32_t hkv, int32_t d, int32_t dtype,
                         int32_t prefix, int sm_count) {
  SplitPlan p{};
  const bool tc = use_tensor_cores(dtype);
  const int group = hq / hkv;
  const int rows = group * n;
  const int key_block = tc ? kTcKeys : kSimtKeys;
  if (tc) {
    // two 128-row tiles per CTA when the group holds more than one tile
    const int tiles = (rows + kTcRowsPerTile - 1) / kTcRowsPerTile;
    p.row_tiles = tiles <= 1 ? 1 : (tiles + 1) / 2;
  } else {
    p.row_tiles = (rows + kSimtRows - 1) / kSimtRows;
  }
  const int64_t keys = (int64_t)prefix + n;
  const int64_t kblocks = (keys + key_block - 1) / key_block;
  const int units = hkv * p.row_tiles;
  const int target = std::max(1, sm_count) * (tc ? kTcCtasPerSm : kSimtCtasPerSm);
  // the tensor-core kernel runs one CTA per SM: stay within one wave
  int64_t s = tc ? std::max(1, target / units)
                 : std::max<int64_t>(1, (target + units - 1) / units);
  s = std::min<int64_t>(s, kblocks);
  const int64_t per = (kblocks + s - 1) / s;  // key blocks per split
  p.keys_per_split = (int32_t)(per * key_block);
  p.splits = (int32_t)((kblocks + per - 1) / per);
  const size_t rows_all = (size_t)n * hq;
  p.ws_bytes = ((size_t)p.splits * rows_all * (size_t)(d + 2) * sizeof(float) + 255) & ~size_t(255);
  return p;
}

template <typename T, int D>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ ws, int splits,
                                                      int rows, T* __restrict__ out) {
  constexpr int C = D / 32;  // consecutive columns per lane
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* acc = ws;
  const float* mrow = ws + (size_t)splits * rows * D;
  const float* lrow = mrow + (size_t)splits * rows;
  float M = -INFINITY;
#pragma unroll 4
  for (int s = 0; s < splits; ++s) M = fmaxf(M, mrow[(size_t)s * rows + row]);
  float L = 0.f;
  float o[C];
#pragma unroll
  for (int c = 0; c < C; ++c) o[c] = 0.f;
#pragma unroll 4
  for (int s = 0; s < splits; ++s) {
    const float ms = mrow[(size_t)s * rows + row];
    const float w = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
    L += w * lrow[(size_t)s * rows + row];
    const float* a = acc + ((size_t)s * rows + row) * D + lane * C;
    if constexpr (C == 4) {
      const float4 x = *reinterpret_cast<const float4*>(a);
      o[0] += w * x.x; o[1] += w * x.y; o[2] += w * x.z; o[3] += w * x.w;
    } else {
#pragma unroll
      for (int c = 0; c < C; ++c) o[c] += w * a[c];
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  T* dst = out + (size_t)row * D + lane * C;
#pragma unroll
  for (int c = 0; c < C; ++c) store_f32(dst + c, o[c] * inv);
}

cudaError_t launch_combine(const AttnProblem& p, const SplitPlan& plan, const float* ws,
                           cudaStream_t s) {
  const int rows = p.n * p.hq;
  const dim3 grid((rows + 7) / 8), block(256);
  if (p.dtype == TV_BF16) {
    auto* out = static_cast<__nv_bfloat16*>(p.out);
    if (p.d == 128) combine_kernel<__nv_bfloat16, 128><<<grid, block, 0, s>>>(ws, plan.splits, rows, out);
    else combine_kernel<__nv_bfloat16, 64><<<grid, block, 0, s>>>(ws, plan.splits, rows, out);
  } else {
    auto* out = static_cast<float*>(p.out);
    if (p.d == 128) combine_kernel<float, 128><<<grid, block, 0, s>>>(ws, plan.splits, rows, out);
    else combine_kernel<float, 64><<<grid, block, 0, s>>>(ws, plan.splits, rows, out);
  }
  return cudaGetLastError();
}

}  // namespace tv
