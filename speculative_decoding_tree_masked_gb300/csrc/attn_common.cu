// Split-KV planning and the combine step of tree-masked attention.
//
// Flash-decoding: the key range [0, P + N) of every (KV head, row tile) is cut
// into `splits` chunks processed by different CTAs; each writes its
// normalised partial output O_s and the log2 of its softmax denominator
// lse_s, and the combine kernel merges them with log-sum-exp weights:
//   O = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M),   M = max_s lse_s.
// (log2 units: scores are pre-multiplied by scale * log2(e).)
#include <algorithm>
#include <cmath>
#include <vector>

#include <cuda_bf16.h>

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

std::atomic<int> cached_sm[64];  // per device (host threads may race here)
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
    // Two 128-row tiles per CTA (sharing every K/V block) when a KV head has
    // three tiles or more; with one or two, one tile per CTA (its scores
    // double-buffered) and twice the row groups: two tiles in one CTA would
    // leave a head a single row group, split into so many key ranges that
    // each CTA gets about two key blocks (measured: 24% slower at P = 4K,
    // N = 32, G = 8; at N = 64 two tiles per CTA are 1-10% faster).
    const int tiles = (rows + kTcRowsPerTile - 1) / kTcRowsPerTile;
    p.tiles_per_cta = tiles >= 3 ? 2 : 1;
    p.row_tiles = (tiles + p.tiles_per_cta - 1) / p.tiles_per_cta;
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
  const size_t o_elem = tc ? 2 : 4;  // bf16 partials for bf16, fp32 for fp32
  p.ws_bytes = (partial_o_offset(p.splits, rows_all) + (size_t)p.splits * rows_all * d * o_elem +
                255) & ~size_t(255);
  return p;
}

// Several bf16 requests in one tensor-core launch.  Each request keeps the
// single-request row tiling; its key splits are proportional to its key
// blocks, kblocks_b * SMs / W with W the batch's (units x key blocks), so
// that every CTA gets about the same number of blocks and the batch fills
// about one wave.  The workspace gives request b room for its largest
// possible split count, max(1, SMs / units_b), whatever the prefix lengths,
// so its layout depends only on the node counts.
void plan_attention_batched(int batch, const int32_t* n, const int32_t* prefix, int32_t hq,
                            int32_t hkv, int32_t d, int sm_count, SplitPlan* plans,
                            size_t* ws_offset, size_t* ws_total) {
  const int sms = std::max(1, sm_count);
  int64_t total_units = 0, work = 0;
  std::vector<int64_t> units(batch), kblocks(batch);
  for (int b = 0; b < batch; ++b) {
    const int rows = (hq / hkv) * n[b];
    const int tiles = (rows + kTcRowsPerTile - 1) / kTcRowsPerTile;
    plans[b] = SplitPlan{};
    plans[b].tiles_per_cta = tiles <= 1 ? 1 : 2;
    plans[b].row_tiles = tiles <= 1 ? 1 : (tiles + 1) / 2;
    units[b] = (int64_t)hkv * plans[b].row_tiles;
    kblocks[b] = prefix ? ((int64_t)prefix[b] + n[b] + kTcKeys - 1) / kTcKeys : 1;
    total_units += units[b];
    work += units[b] * kblocks[b];
  }
  size_t off = 0;
  for (int b = 0; b < batch; ++b) {
    int64_t s = 1;
    if (prefix && total_units < sms) s = std::max<int64_t>(1, kblocks[b] * sms / work);
    s = std::min<int64_t>(s, kblocks[b]);
    const int64_t per = (kblocks[b] + s - 1) / s;
    plans[b].keys_per_split = (int32_t)(per * kTcKeys);
    plans[b].splits = (int32_t)((kblocks[b] + per - 1) / per);
    const int64_t s_max = std::max<int64_t>(1, sms / units[b]);
    const size_t rows_all = (size_t)n[b] * hq;
    const size_t bytes = (partial_o_offset((int)s_max, rows_all) +
                          (size_t)s_max * rows_all * d * 2 + 255) & ~size_t(255);
    plans[b].ws_bytes = bytes;
    if (ws_offset) ws_offset[b] = off;
    off += bytes;
  }
  if (ws_total) *ws_total = off;
}

__device__ __forceinline__ void load_partial(const float* p, float (&o)[4]) {
  const float4 x = *reinterpret_cast<const float4*>(p);
  o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w;
}
__device__ __forceinline__ void load_partial(const float* p, float (&o)[2]) {
  const float2 x = *reinterpret_cast<const float2*>(p);
  o[0] = x.x; o[1] = x.y;
}
// A bf16 value is the top half of the float32 with the same bits.
__device__ __forceinline__ void load_partial(const __nv_bfloat16* p, float (&o)[4]) {
  const uint2 x = *reinterpret_cast<const uint2*>(p);
  o[0] = __uint_as_float(x.x << 16); o[1] = __uint_as_float(x.x & 0xffff0000u);
  o[2] = __uint_as_float(x.y << 16); o[3] = __uint_as_float(x.y & 0xffff0000u);
}
__device__ __forceinline__ void load_partial(const __nv_bfloat16* p, float (&o)[2]) {
  const uint32_t x = *reinterpret_cast<const uint32_t*>(p);
  o[0] = __uint_as_float(x << 16); o[1] = __uint_as_float(x & 0xffff0000u);
}

// One warp per output row: O = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M).
// The merge is latency-bound, so every load of a row is issued before any is
// used: with the split count S known at compile time a warp keeps all S
// partial loads in flight at once; otherwise (SMAX > 0) lane s holds split
// s's log-sum-exp, the maximum and the sum come from warp shuffles, and the
// partial loads of up to SMAX splits are issued together with it (one round
// trip in all); beyond 32 splits the loop takes one split at a time.
template <typename PT, typename T, int D, int S, int SMAX>
__global__ void __launch_bounds__(256) combine_kernel(const uint8_t* __restrict__ ws, int splits,
                                                      int rows, T* __restrict__ out) {
  constexpr int C = D / 32;  // consecutive columns per lane
  // launched under programmatic serialization: wait for the attention
  // kernel that writes the partials; only then let the next layer's
  // attention kernel start its setup (it waits for this grid to finish
  // before it reads or writes memory)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* lse = reinterpret_cast<const float*>(ws);
  const PT* po = reinterpret_cast<const PT*>(ws + partial_o_offset(splits, rows));
  float W = 0.f;
  float o[C];
#pragma unroll
  for (int c = 0; c < C; ++c) o[c] = 0.f;
  if constexpr (S > 0) {
    float ls[S], x[S][C];
#pragma unroll
    for (int s = 0; s < S; ++s) {
      ls[s] = __ldg(lse + (size_t)s * rows + row);
      load_partial(po + ((size_t)s * rows + row) * D + lane * C, x[s]);
    }
    float M = ls[0];
#pragma unroll
    for (int s = 1; s < S; ++s) M = fmaxf(M, ls[s]);
#pragma unroll
    for (int s = 0; s < S; ++s) {
      const float w = (ls[s] == -INFINITY) ? 0.f : exp2f(ls[s] - M);
      W += w;
#pragma unroll
      for (int c = 0; c < C; ++c) o[c] = fmaf(w, x[s][c], o[c]);
    }
  } else if constexpr (SMAX > 0) {
    // bf16 partials stay packed (two to a register) until they are used
    static_assert(sizeof(PT) == 2 && C % 2 == 0, "packed loads take bf16 partials");
    constexpr int P2 = C / 2;  // 32-bit words per lane and split
    const float ls = lane < splits ? __ldg(lse + (size_t)lane * rows + row) : -INFINITY;
    uint32_t raw[SMAX][P2];
#pragma unroll
    for (int s = 0; s < SMAX; ++s) {
      const uint32_t* src =
          reinterpret_cast<const uint32_t*>(po + ((size_t)s * rows + row) * D + lane * C);
      if (s < splits) {
        if constexpr (P2 == 2) {
          const uint2 v = __ldg(reinterpret_cast<const uint2*>(src));
          raw[s][0] = v.x;
          raw[s][1] = v.y;
        } else {
#pragma unroll
          for (int k = 0; k < P2; ++k) raw[s][k] = __ldg(src + k);
        }
      } else {
#pragma unroll
        for (int k = 0; k < P2; ++k) raw[s][k] = 0u;
      }
    }
    float M = ls;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float w_mine = (ls == -INFINITY) ? 0.f : exp2f(ls - M);
    W = w_mine;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
#pragma unroll
    for (int s = 0; s < SMAX; ++s) {
      const float w = __shfl_sync(0xffffffffu, w_mine, s);  // 0 for s >= splits
#pragma unroll
      for (int k = 0; k < P2; ++k) {
        // a bf16 value is the top half of the float32 with the same bits
        o[2 * k] = fmaf(w, __uint_as_float(raw[s][k] << 16), o[2 * k]);
        o[2 * k + 1] = fmaf(w, __uint_as_float(raw[s][k] & 0xffff0000u), o[2 * k + 1]);
      }
    }
  } else {
    float M = -INFINITY;
#pragma unroll 4
    for (int s = 0; s < splits; ++s) M = fmaxf(M, lse[(size_t)s * rows + row]);
#pragma unroll 4
    for (int s = 0; s < splits; ++s) {
      const float ls = lse[(size_t)s * rows + row];
      const float w = (ls == -INFINITY) ? 0.f : exp2f(ls - M);
      W += w;
      float x[C];
      load_partial(po + ((size_t)s * rows + row) * D + lane * C, x);
#pragma unroll
      for (int c = 0; c < C; ++c) o[c] = fmaf(w, x[c], o[c]);
    }
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  T* dst = out + (size_t)row * D + lane * C;
#pragma unroll
  for (int c = 0; c < C; ++c) store_f32(dst + c, o[c] * inv);
}

// The combine is launched under programmatic serialization and waits for
// the attention grid before reading.  A grid of at most one CTA per SM is
// released early: the attention kernel signals once its products are done,
// and the combine's CTAs wait, one beside each attention CTA, which hides
// its launch.  A larger grid is released only as the attention CTAs exit
// (their implicit signal): its CTAs would crowd the attention's SMs while
// waiting, but it still starts without waiting for the attention grid's
// completion and flush (0.7-3% faster than a plain launch, measured).
bool combine_launches_early(int rows) {
  const int sms = device_sm_count();
  return sms > 0 && (rows + 7) / 8 <= sms;
}

template <typename PT, typename T, int D, int S, int SMAX = 0>
cudaError_t launch_combine_s(const uint8_t* w, int splits, int rows, T* out, cudaStream_t s) {
  const dim3 grid((rows + 7) / 8);
  return launch_pdl(combine_kernel<PT, T, D, S, SMAX>, grid, dim3(256), 0, s, w, splits, rows,
                    out);
}

template <typename PT, typename T, int D>
cudaError_t launch_combine_d(const uint8_t* w, int splits, int rows, T* out, cudaStream_t s) {
  switch (splits) {
#define TV_COMBINE_CASE(n) \
  case n: return launch_combine_s<PT, T, D, n>(w, splits, rows, out, s);
    TV_COMBINE_CASE(2) TV_COMBINE_CASE(3) TV_COMBINE_CASE(4) TV_COMBINE_CASE(5)
    TV_COMBINE_CASE(6) TV_COMBINE_CASE(7) TV_COMBINE_CASE(8) TV_COMBINE_CASE(9)
    TV_COMBINE_CASE(10) TV_COMBINE_CASE(11) TV_COMBINE_CASE(12)
#undef TV_COMBINE_CASE
    default:
      if (splits <= 16) return launch_combine_s<PT, T, D, 0, 16>(w, splits, rows, out, s);
      if (splits <= 32) return launch_combine_s<PT, T, D, 0, 32>(w, splits, rows, out, s);
      return launch_combine_s<PT, T, D, 0>(w, splits, rows, out, s);
  }
}

cudaError_t launch_combine(const AttnProblem& p, const SplitPlan& plan, const float* ws,
                           cudaStream_t s) {
  const int rows = p.n * p.hq;
  const auto* w = reinterpret_cast<const uint8_t*>(ws);
  if (p.dtype == TV_BF16) {
    auto* out = static_cast<__nv_bfloat16*>(p.out);
    return p.d == 128
               ? launch_combine_d<__nv_bfloat16, __nv_bfloat16, 128>(w, plan.splits, rows, out, s)
               : launch_combine_d<__nv_bfloat16, __nv_bfloat16, 64>(w, plan.splits, rows, out, s);
  }
  // the fp32 path is not latency-critical: one loop kernel
  auto* out = static_cast<float*>(p.out);
  return p.d == 128 ? launch_combine_s<float, float, 128, 0>(w, plan.splits, rows, out, s)
                    : launch_combine_s<float, float, 64, 0>(w, plan.splits, rows, out, s);
}

}  // namespace tv
