// Sampling verification: the target's token at every tree node drawn from
// softmax(z / T) by inversion with one Philox4x64-10 uniform per node, then
// the greedy walk over the drawn tokens (walk_kernel in accept.cu).
//
// This library's reading of sampling for deterministically grown trees (the
// SwiftSpec review page verifies greedily and is silent on sampling): every
// emitted token is the target's own draw at its context, so verification
// stays lossless.
//
// One 8-CTA thread-block cluster per tree node.  Each CTA streams an eighth
// of the node's logits once (float4 loads when aligned), keeping a running
// maximum and a running sum of exp((z - max) / T) that is rescaled whenever
// the maximum grows; the CTAs combine their (max, sum) pairs through
// distributed shared memory.  The uniform u picks the target mass u * S; the
// CTA whose eighth holds that point finds the warp chunk holding it (chunk
// sums and their prefix), and that warp walks its chunk 32 logits at a time
// with a warp scan to find the token.
#include <cooperative_groups.h>

#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace tv {

namespace {

constexpr int kSampleCluster = 8;
constexpr int kSampleThreads = 256;
constexpr int kSampleWarps = kSampleThreads / 32;

// Philox4x64-10 (Salmon, Moraes, Dror and Shaw, SC 2011): the published
// multipliers and Weyl key increments; returns the first output word.
__device__ __forceinline__ uint64_t philox4x64_10_x0(uint64_t x0, uint64_t x1, uint64_t x2,
                                                     uint64_t x3, uint64_t k0, uint64_t k1) {
  constexpr uint64_t kM0 = 0xD2E7470EE14C6C93ull, kM1 = 0xCA5A826395121157ull;
  constexpr uint64_t kW0 = 0x9E3779B97F4A7C15ull, kW1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t hi0 = __umul64hi(kM0, x0), lo0 = kM0 * x0;
    const uint64_t hi1 = __umul64hi(kM1, x2), lo1 = kM1 * x2;
    const uint64_t y0 = hi1 ^ x1 ^ k0, y2 = hi0 ^ x3 ^ k1;
    x0 = y0;
    x1 = lo1;
    x2 = y2;
    x3 = lo0;
    k0 += kW0;
    k1 += kW1;
  }
  return x0;
}

// (m, s) with s = sum exp((z - m) * inv_t): merge another pair into it.
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2, float inv_t) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) { m = m2; s = s2; return; }
  if (m2 > m) {
    s = s * expf((m - m2) * inv_t) + s2;
    m = m2;
  } else {
    s += s2 * expf((m2 - m) * inv_t);
  }
}

__device__ __forceinline__ void add_logit(float& m, float& s, float z, float inv_t) {
  if (z == -INFINITY) return;
  if (z > m) {
    s = (m == -INFINITY ? 0.f : s * expf((m - z) * inv_t)) + 1.f;
    m = z;
  } else {
    s += expf((z - m) * inv_t);
  }
}

__global__ void __cluster_dims__(kSampleCluster, 1, 1) __launch_bounds__(kSampleThreads)
sample_kernel(const float* __restrict__ logits, int vocab, float inv_t, uint64_t seed,
              uint64_t offset, int32_t* __restrict__ sampled) {
  __shared__ float w_m[kSampleWarps], w_s[kSampleWarps];
  __shared__ float cta_m;    // this CTA's maximum, read by the cluster
  __shared__ double cta_s;   // its sum of exp((z - M) / T) at the row maximum M
  __shared__ double wsum[kSampleWarps];
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk = ((vocab + kSampleCluster * 4 - 1) / (kSampleCluster * 4)) * 4;
  const int beg = min(vocab, rank * chunk);
  const int end = min(vocab, beg + chunk);
  const float* base = logits + (size_t)row * vocab;

  // one pass: running (max, sum) per thread
  float m = -INFINITY, s = 0.f;
  const bool vec = ((vocab & 3) == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
  if (vec) {
    // four float4 loads per thread in flight before any is used; logits are
    // read through L2 (kept: the scan below reads one eighth again)
    const float4* b4 = reinterpret_cast<const float4*>(base);
    const int e4 = end / 4;
    for (int i40 = beg / 4 + tid; i40 < e4; i40 += 4 * kSampleThreads) {
      float4 x[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i4 = i40 + q * kSampleThreads;
        x[q] = i4 < e4 ? __ldcg(b4 + i4)
                       : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        add_logit(m, s, x[q].x, inv_t);
        add_logit(m, s, x[q].y, inv_t);
        add_logit(m, s, x[q].z, inv_t);
        add_logit(m, s, x[q].w, inv_t);
      }
    }
  } else {
    for (int i = beg + tid; i < end; i += kSampleThreads) add_logit(m, s, __ldcs(base + i), inv_t);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    merge_ms(m, s, m2, s2, inv_t);
  }
  if (lane == 0) { w_m[warp] = m; w_s[warp] = s; }
  __syncthreads();
  if (tid == 0) {
    for (int k = 1; k < kSampleWarps; ++k) merge_ms(m, s, w_m[k], w_s[k], inv_t);
    cta_m = m;
  }
  cluster.sync();
  // the row maximum, then this CTA's mass at it
  float M = -INFINITY;
#pragma unroll
  for (int r = 0; r < kSampleCluster; ++r) M = fmaxf(M, *cluster.map_shared_rank(&cta_m, r));
  if (tid == 0)
    cta_s = (m == -INFINITY || M == -INFINITY) ? 0.0 : (double)s * (double)expf((m - M) * inv_t);
  cluster.sync();
  double S = 0.0, P = 0.0, mass[kSampleCluster];
#pragma unroll
  for (int r = 0; r < kSampleCluster; ++r) {
    mass[r] = *cluster.map_shared_rank(&cta_s, r);
    S += mass[r];
  }
  const uint64_t x0 = philox4x64_10_x0((uint64_t)row, offset, 0ull, 0ull, seed, 0ull);
  const double u = ((double)(x0 >> 11) + 0.5) * (1.0 / 9007199254740992.0);  // 2^-53
  const double t = u * S;
  // the CTA whose eighth holds mass t (the last one with mass if rounding
  // puts t past the end)
  int owner = -1, last = -1;
#pragma unroll
  for (int r = 0; r < kSampleCluster; ++r) {
    if (mass[r] > 0.0) last = r;
    if (owner < 0 && mass[r] > 0.0 && P + mass[r] > t) owner = r;
    if (owner < 0) P += mass[r];
  }
  if (last < 0) {  // every logit is -inf: nothing can be drawn
    if (rank == 0 && tid == 0) sampled[row] = -1;
  } else if (owner < 0) {
    owner = last;
    P = 0.0;
    for (int r = 0; r < last; ++r) P += mass[r];
  }
  if (last >= 0 && rank == owner) {
    // The eighth in eight contiguous warp chunks (multiples of 32 logits):
    // each warp sums its chunk with coalesced loads, the chunk holding mass
    // t is found from the prefix over the warps, and that warp walks it 32
    // logits at a time with a warp scan.
    const int len = end - beg;
    const int wlen = ((len + kSampleWarps * 32 - 1) / (kSampleWarps * 32)) * 32;
    const int wb = beg + warp * wlen, we = min(end, wb + wlen);
    auto e_of = [&](float z) { return z == -INFINITY ? 0.f : expf((z - M) * inv_t); };
    float part = 0.f;
    for (int v0 = wb; v0 < we; v0 += 32 * 8) {
      float z[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int v = v0 + 32 * q + lane;
        z[q] = v < we ? __ldcg(base + v) : -INFINITY;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) part += e_of(z[q]);
    }
    double csum = part;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) csum += __shfl_xor_sync(0xffffffffu, csum, o);
    if (lane == 0) wsum[warp] = csum;
    __syncthreads();
    const double tr = t - P;  // target mass inside this eighth
    int pw = -1, lw = -1;
    double before = 0.0, before_pw = 0.0, before_lw = 0.0;
    for (int k = 0; k < kSampleWarps; ++k) {
      if (wsum[k] > 0.0) { lw = k; before_lw = before; }
      if (pw < 0 && wsum[k] > 0.0 && before + wsum[k] > tr) { pw = k; before_pw = before; }
      before += wsum[k];
    }
    if (pw < 0) { pw = lw; before_pw = before_lw; }  // rounding past the end
    if (warp == pw) {
      // eight steps of 32 logits are loaded before they are walked
      double c = before_pw;
      int tok = -1, lastp = -1;
      for (int v00 = wb; v00 < we && tok < 0; v00 += 32 * 8) {
        float e8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int v = v00 + 32 * q + lane;
          e8[q] = v < we ? __ldcg(base + v) : -INFINITY;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int v0 = v00 + 32 * q;
          if (tok >= 0 || v0 >= we) break;
          const float e = e_of(e8[q]);
          float incl = e;  // a scan of 32 terms in float32 on a double base
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          const uint32_t cross = __ballot_sync(0xffffffffu, e > 0.f && c + (double)incl > tr);
          const uint32_t pos = __ballot_sync(0xffffffffu, e > 0.f);
          if (pos) lastp = v0 + 31 - __clz(pos);
          if (cross) tok = v0 + __ffs(cross) - 1;
          c += (double)__shfl_sync(0xffffffffu, incl, 31);
        }
      }
      // rounding past the chunk's mass: its last token with positive mass
      if (lane == 0) sampled[row] = tok >= 0 ? tok : lastp;
    }
  }
  cluster.sync();  // no CTA leaves while the others may still read its shared memory
}

}  // namespace

cudaError_t launch_accept_sampled(const float* logits, int32_t vocab, const int32_t* token,
                                  const int32_t* parent, int32_t n, int32_t prefix,
                                  float temperature, uint64_t seed, uint64_t offset,
                                  int32_t* sampled, int32_t* m, int32_t* path,
                                  int32_t* out_tokens, int32_t* new_pos, int32_t* new_parent,
                                  int32_t* n_survivors, int32_t* dev_status, cudaStream_t s) {
  sample_kernel<<<dim3(kSampleCluster, n), kSampleThreads, 0, s>>>(logits, vocab,
                                                                   1.0f / temperature, seed,
                                                                   offset, sampled);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_walk(token, parent, sampled, n, vocab, prefix, m, path, out_tokens, new_pos,
                     new_parent, n_survivors, dev_status, s);
}

}  // namespace tv
