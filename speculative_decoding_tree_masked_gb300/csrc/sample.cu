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
// of the node's logits once; each of its warps owns a contiguous run of that
// eighth (lanes reading it coalesced, eight float4 loads in flight) and
// keeps running (max, sum of exp((z - max) / T)) pairs, rescaled whenever
// the maximum grows.  The CTAs combine their pairs through distributed
// shared memory into the row maximum M and every warp's mass at M.  The
// uniform u picks the target mass u * S: the CTA, then the warp whose run
// holds it follow from those masses (one thread per CTA decides, in double:
// double arithmetic is slow on this GPU); that warp re-reads its run as 32
// contiguous per-lane pieces, sums each piece, finds the piece holding the
// target with one warp scan (in double), and that lane walks its piece to
// the token.
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

// Exponentials in base 2: with c = log2(e) / T, exp((z - m) / T) is
// 2^((z - m) c), one hardware ex2 (relative error near 2^-22, far below what
// the draws can resolve).
__device__ __forceinline__ float exp2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (m, s) with s = sum 2^((z - m) c): merge another pair into it.
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2, float c) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) { m = m2; s = s2; return; }
  if (m2 > m) {
    s = s * exp2_fast((m - m2) * c) + s2;
    m = m2;
  } else {
    s += s2 * exp2_fast((m2 - m) * c);
  }
}

// Draw parameters of a packed batch: rows [off[b], off[b + 1]) are request
// b's nodes; its node i draws at temperature 1 / inv_t[b] with key
// (seed[b], 0) and counter (i, offset[b], 0, 0).
struct SampleJobs {
  int32_t off[kMaxBatch + 1];
  int32_t batch;
  float inv_t[kMaxBatch];
  uint64_t seed[kMaxBatch];
  uint64_t offset[kMaxBatch];
};

// Split cluster barrier around the kernel's work: every thread arrives
// (relaxed, without waiting) as it starts and waits before its CTA first
// stores into another CTA's shared memory, so that every CTA of the cluster
// has started by then; the wait returns at once in practice.
__device__ __forceinline__ void cluster_arrive_at_start() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_all_started() {
  asm volatile("barrier.cluster.wait;" ::: "memory");
}

__global__ void __cluster_dims__(kSampleCluster, 1, 1) __launch_bounds__(kSampleThreads)
sample_kernel(const float* __restrict__ logits, int vocab, const __grid_constant__ SampleJobs jobs,
              int32_t* __restrict__ sampled) {
  __shared__ float w_m[kSampleWarps], w_s[kSampleWarps];
  __shared__ double w_mass[kSampleWarps];  // each warp's run's mass at the row maximum
  __shared__ float all_m[kSampleCluster];  // every CTA's maximum (each CTA writes its own
  __shared__ double all_s[kSampleCluster]; // entry in every CTA) and mass at the row maximum
  __shared__ float cta_m_row;              // the row maximum
  __shared__ int sel_owner, sel_warp;      // the drawing CTA and warp (-1: none)
  // launched under programmatic serialization: the walk may be scheduled
  // now; this grid waits for the kernel before it before reading anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ double sel_rem;               // the target mass left inside that warp's run
  cg::cluster_group cluster = cg::this_cluster();
  cluster_arrive_at_start();
  const int row = blockIdx.y;
  int job = 0;  // the request owning this row
  while (job + 1 < jobs.batch && row >= jobs.off[job + 1]) ++job;
  const float c = jobs.inv_t[job] * 1.4426950408889634f;  // log2(e) / T
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk = ((vocab + kSampleCluster * 4 - 1) / (kSampleCluster * 4)) * 4;
  const int beg = min(vocab, rank * chunk);
  const int end = min(vocab, beg + chunk);
  const float* base = logits + (size_t)row * vocab;
  // warp w's run [wb, we) of this CTA's eighth (a multiple of 4 long)
  const int wlen = ((end - beg + kSampleWarps * 4 - 1) / (kSampleWarps * 4)) * 4;
  auto run_begin = [&](int w) { return min(end, beg + w * wlen); };
  auto run_end = [&](int w) { return min(end, beg + (w + 1) * wlen); };
  const int wb = run_begin(warp), we = run_end(warp);

  // one pass: a running (max, sum) pair per lane, updated once per batch of
  // 32 loaded logits (the batch's maximum first, then 32 independent
  // exponentials), so that no lane branches on a new maximum
  float mm = -INFINITY, ss = 0.f;
  auto add_batch = [&](const float (&z)[32]) {
    float bm = z[0];
#pragma unroll
    for (int q = 1; q < 32; ++q) bm = fmaxf(bm, z[q]);
    if (bm == -INFINITY) return;
    const float mn = fmaxf(mm, bm);
    float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 32; ++q) part[q & 3] += exp2_fast((z[q] - mn) * c);  // 2^-inf = 0
    ss = (mm == -INFINITY ? 0.f : ss * exp2_fast((mm - mn) * c)) +
         ((part[0] + part[1]) + (part[2] + part[3]));
    mm = mn;
  };
  const bool vec = ((vocab & 3) == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
  if (vec) {
    const float4* b4 = reinterpret_cast<const float4*>(base);
    const int e4 = we / 4;
    for (int i40 = wb / 4 + lane; i40 < e4; i40 += 8 * 32) {
      float z[32];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i4 = i40 + q * 32;
        const float4 x = i4 < e4 ? __ldcg(b4 + i4)
                                 : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        z[4 * q] = x.x;
        z[4 * q + 1] = x.y;
        z[4 * q + 2] = x.z;
        z[4 * q + 3] = x.w;
      }
      add_batch(z);
    }
  } else {
    for (int i0 = wb + lane; i0 < we; i0 += 32 * 32) {
      float z[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int i = i0 + q * 32;
        z[q] = i < we ? __ldcs(base + i) : -INFINITY;
      }
      add_batch(z);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, mm, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, ss, o);
    merge_ms(mm, ss, m2, s2, c);
  }
  if (lane == 0) { w_m[warp] = mm; w_s[warp] = ss; }
  __syncthreads();
  cluster_wait_all_started();
  if (tid == 0) {
    float cm = -INFINITY;
    for (int k = 0; k < kSampleWarps; ++k) cm = fmaxf(cm, w_m[k]);
    // this CTA's maximum into every CTA's all_m (the barrier's release and
    // acquire publish the stores): afterwards each reads only its own copy
#pragma unroll
    for (int r = 0; r < kSampleCluster; ++r) *cluster.map_shared_rank(&all_m[rank], r) = cm;
  }
  cluster.sync();
  // the row maximum, then every warp's mass and this CTA's mass at it
  if (tid == 0) {
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < kSampleCluster; ++r) M = fmaxf(M, all_m[r]);
    double total = 0.0;
    for (int k2 = 0; k2 < kSampleWarps; ++k2) {
      const double wm = (w_m[k2] == -INFINITY || M == -INFINITY)
                            ? 0.0 : (double)w_s[k2] * (double)exp2_fast((w_m[k2] - M) * c);
      w_mass[k2] = wm;
      total += wm;
    }
#pragma unroll
    for (int r = 0; r < kSampleCluster; ++r) *cluster.map_shared_rank(&all_s[rank], r) = total;
    cta_m_row = M;
  }
  cluster.sync();
  // One thread per CTA draws: the CTA whose eighth holds the target mass
  // u * S (the last one with mass if rounding puts it past the end), then,
  // in that CTA, the warp whose run holds it.  Doubles are slow on this GPU,
  // so no other thread touches them here.
  if (tid == 0) {
    double S = 0.0, P = 0.0, mass[kSampleCluster];
#pragma unroll
    for (int r = 0; r < kSampleCluster; ++r) {
      mass[r] = all_s[r];
      S += mass[r];
    }
    const uint64_t x0 = philox4x64_10_x0((uint64_t)(row - jobs.off[job]), jobs.offset[job], 0ull,
                                         0ull, jobs.seed[job], 0ull);
    const double u = ((double)(x0 >> 11) + 0.5) * (1.0 / 9007199254740992.0);  // 2^-53
    const double t = u * S;
    int owner = -1, last = -1;
    double p_last = 0.0;
#pragma unroll
    for (int r = 0; r < kSampleCluster; ++r) {
      if (mass[r] > 0.0) { last = r; p_last = P; }
      if (owner < 0 && mass[r] > 0.0 && P + mass[r] > t) owner = r;
      if (owner < 0) P += mass[r];
    }
    if (owner < 0) { owner = last; P = p_last; }
    sel_owner = owner;
    sel_warp = -1;
    if (owner == rank) {
      const double tr = t - P;
      int pw = -1, lw = -1;
      double before = 0.0, before_pw = 0.0, before_lw = 0.0;
      for (int k2 = 0; k2 < kSampleWarps; ++k2) {
        if (w_mass[k2] > 0.0) { lw = k2; before_lw = before; }
        if (pw < 0 && w_mass[k2] > 0.0 && before + w_mass[k2] > tr) { pw = k2; before_pw = before; }
        before += w_mass[k2];
      }
      if (pw < 0) { pw = lw; before_pw = before_lw; }  // rounding past the end
      sel_warp = pw;
      sel_rem = tr - before_pw;
    }
    if (last < 0 && rank == 0) sampled[row] = -1;  // every logit is -inf: nothing is drawn
  }
  __syncthreads();
  if (sel_owner != rank || warp != sel_warp) return;
  const float M = cta_m_row;
  // 32 contiguous pieces of the run, one per lane
  auto e_of = [&](float z) { return z == -INFINITY ? 0.f : exp2_fast((z - M) * c); };
  const int rb = run_begin(warp), re = run_end(warp);
  const int plen = (re - rb + 31) / 32;
  const int pb = min(re, rb + lane * plen), pe = min(re, pb + plen);
  // (L1-cached loads: the walk below reads the same piece again)
  constexpr int kBatch = 16;
  float ls = 0.f;
  for (int v0 = pb; v0 < pe; v0 += kBatch) {
    float z[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) z[q] = v0 + q < pe ? __ldg(base + v0 + q) : -INFINITY;
#pragma unroll
    for (int q = 0; q < kBatch; ++q) ls += e_of(z[q]);
  }
  double incl = ls;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const double rem = sel_rem;  // target mass inside the run
  const uint32_t cross = __ballot_sync(0xffffffffu, ls > 0.f && incl > rem);
  const uint32_t pos = __ballot_sync(0xffffffffu, ls > 0.f);
  if (pos == 0u) {  // nothing left in the run after rounding
    if (lane == 0) sampled[row] = -1;
    return;
  }
  // the crossing lane, or the last lane with mass if rounding left none; it
  // walks its piece in float, relative to the piece's start
  const int wl = cross ? __ffs(cross) - 1 : 31 - __clz(pos);
  if (lane == wl) {
    const float target = (float)(rem - (incl - (double)ls));
    float acc = 0.f;
    int tok = -1, lastp = -1;
    for (int v0 = pb; v0 < pe && tok < 0; v0 += kBatch) {
      float z[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) z[q] = v0 + q < pe ? __ldg(base + v0 + q) : -INFINITY;
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const float e = e_of(z[q]);
        if (tok < 0 && e > 0.f) {
          lastp = v0 + q;
          acc += e;
          if (acc > target) tok = v0 + q;
        }
      }
    }
    sampled[row] = tok >= 0 ? tok : lastp;
  }
}

}  // namespace

cudaError_t launch_accept_sampled(const float* logits, int32_t vocab, const int32_t* token,
                                  const int32_t* parent, int32_t n, int32_t prefix,
                                  float temperature, uint64_t seed, uint64_t offset,
                                  int32_t* sampled, int32_t* m, int32_t* path,
                                  int32_t* out_tokens, int32_t* new_pos, int32_t* new_parent,
                                  int32_t* n_survivors, int32_t* dev_status, cudaStream_t s) {
  const int32_t off[2] = {0, n};
  return launch_accept_sampled_batched(logits, vocab, token, parent, 1, off, &prefix,
                                       &temperature, &seed, &offset, sampled, m, path, out_tokens,
                                       new_pos, new_parent, n_survivors, dev_status, s);
}

cudaError_t launch_accept_sampled_batched(const float* logits, int32_t vocab,
                                          const int32_t* token, const int32_t* parent,
                                          int32_t batch, const int32_t* node_offset,
                                          const int32_t* prefix, const float* temperature,
                                          const uint64_t* seed, const uint64_t* offset,
                                          int32_t* sampled, int32_t* m, int32_t* path,
                                          int32_t* out_tokens, int32_t* new_pos,
                                          int32_t* new_parent, int32_t* n_survivors,
                                          int32_t* dev_status, cudaStream_t s) {
  SampleJobs jobs{};
  jobs.batch = batch;
  for (int b = 0; b < batch; ++b) {
    jobs.off[b] = node_offset[b];
    jobs.inv_t[b] = 1.0f / temperature[b];
    jobs.seed[b] = seed[b];
    jobs.offset[b] = offset[b];
  }
  jobs.off[batch] = node_offset[batch];
  cudaError_t e = launch_pdl(sample_kernel, dim3(kSampleCluster, node_offset[batch]),
                             dim3(kSampleThreads), 0, s, logits, vocab, jobs, sampled);
  if (e != cudaSuccess) return e;
  return launch_walk_batched(token, parent, sampled, batch, node_offset, vocab, prefix, m, path,
                             out_tokens, new_pos, new_parent, n_survivors, dev_status, s);
}

}  // namespace tv
