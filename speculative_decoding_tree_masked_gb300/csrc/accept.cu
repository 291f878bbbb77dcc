// Greedy acceptance of the draft tree (target argmax, tree walk, re-root map).
//
// argmax: one 8-CTA thread-block cluster per tree node scans the node's
// logits row (each CTA one eighth, float4 loads when rows are 16-byte
// aligned) and the partial winners meet in CTA 0 through distributed shared
// memory.  walk: one warp walks the tree with ballots (lane k holds nodes
// k, k+32, k+64, k+96) and builds the re-root map with ballot/popc ranks.
// Several requests are verified at once by packing their node arrays: the
// argmax runs over all packed rows and one warp walks each request.
#include <cooperative_groups.h>

#include <climits>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace tv {

namespace {

constexpr int kArgmaxCluster = 8;
constexpr int kArgmaxThreads = 256;
constexpr int kArgmaxLoads = 8;  // float4 loads in flight per thread

// True if (a, ia) comes before (b, ib) in NumPy argmax order: a NaN beats any
// number, larger values beat smaller ones, and ties go to the lower index.
// ib == INT_MAX stands for "no candidate yet".
__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
  if (ib == INT_MAX) return ia != INT_MAX;
  if (ia == INT_MAX) return false;
  const bool an = isnan(a), bn = isnan(b);
  if (an || bn) return an && bn ? ia < ib : an;
  return a > b || (a == b && ia < ib);
}

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

__global__ void __cluster_dims__(kArgmaxCluster, 1, 1) __launch_bounds__(kArgmaxThreads)
argmax_kernel(const float* __restrict__ logits, int vocab, int32_t* __restrict__ am) {
  __shared__ float s_val[kArgmaxThreads / 32];
  __shared__ int s_idx[kArgmaxThreads / 32];
  __shared__ float c_val[kArgmaxCluster];  // CTA 0's: every CTA's winner
  __shared__ int c_idx[kArgmaxCluster];
  // launched under programmatic serialization: the walk that follows may be
  // scheduled now (it waits for this grid); this grid waits for the kernel
  // before it (which may write the logits) before reading anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  cg::cluster_group cluster = cg::this_cluster();
  cluster_arrive_at_start();
  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.y;
  const int tid = threadIdx.x;
  const int chunk = ((vocab + kArgmaxCluster * 4 - 1) / (kArgmaxCluster * 4)) * 4;
  const int beg = rank * chunk;
  const int end = min(vocab, beg + chunk);
  const float* base = logits + (size_t)row * vocab;

  float bv = 0.f;
  int bi = INT_MAX;
  const bool vec = ((vocab & 3) == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
  if (vec) {
    // eight float4 loads per thread in flight; a batch's maximum comes from a
    // comparison tree and its first occurrence (the lowest index: indices
    // grow along the batch) from one scan, unless the batch holds a NaN,
    // which takes the element-wise order
    const float4* b4 = reinterpret_cast<const float4*>(base);
    const int e4 = end / 4;
    constexpr int kZ = 4 * kArgmaxLoads;
    for (int i40 = beg / 4 + tid; i40 < e4; i40 += kArgmaxLoads * kArgmaxThreads) {
      float z[kZ];
#pragma unroll
      for (int q = 0; q < kArgmaxLoads; ++q) {
        const int i4 = i40 + q * kArgmaxThreads;
        const float4 x = i4 < e4 ? __ldcs(b4 + i4)
                                 : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        z[4 * q] = x.x;
        z[4 * q + 1] = x.y;
        z[4 * q + 2] = x.z;
        z[4 * q + 3] = x.w;
      }
      auto index_of = [&](int k) { return (i40 + (k >> 2) * kArgmaxThreads) * 4 + (k & 3); };
      bool nan = false;
      float bm = -INFINITY;
#pragma unroll
      for (int k = 0; k < kZ; ++k) {
        nan |= isnan(z[k]);
        bm = fmaxf(bm, z[k]);
      }
      if (nan) {
#pragma unroll
        for (int k = 0; k < kZ; ++k)
          if (i40 + (k >> 2) * kArgmaxThreads < e4 && better(z[k], index_of(k), bv, bi)) {
            bv = z[k];
            bi = index_of(k);
          }
      } else {
        int first = kZ;
#pragma unroll
        for (int k = kZ - 1; k >= 0; --k)
          if (z[k] == bm) first = k;
        if (first < kZ && i40 + (first >> 2) * kArgmaxThreads < e4 &&
            better(bm, index_of(first), bv, bi)) {
          bv = bm;
          bi = index_of(first);
        }
      }
    }
  } else {
    for (int i = beg + tid; i < end; i += kArgmaxThreads) {
      const float x = __ldcs(base + i);
      if (better(x, i, bv, bi)) { bv = x; bi = i; }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
  }
  if ((tid & 31) == 0) { s_val[tid >> 5] = bv; s_idx[tid >> 5] = bi; }
  __syncthreads();
  cluster_wait_all_started();
  if (tid == 0) {
    for (int w = 1; w < kArgmaxThreads / 32; ++w)
      if (better(s_val[w], s_idx[w], bv, bi)) { bv = s_val[w]; bi = s_idx[w]; }
    // each CTA stores its winner into CTA 0's shared memory; the cluster
    // barrier's release and acquire make the stores visible to CTA 0, and no
    // CTA reads another's shared memory after it, so one barrier suffices
    *cluster.map_shared_rank(&c_val[rank], 0) = bv;
    *cluster.map_shared_rank(&c_idx[rank], 0) = bi;
  }
  cluster.sync();
  if (rank == 0 && tid == 0) {
    for (int r = 1; r < kArgmaxCluster; ++r)
      if (better(c_val[r], c_idx[r], bv, bi)) { bv = c_val[r]; bi = c_idx[r]; }
    am[row] = bi == INT_MAX ? 0 : bi;
  }
}

// Request b of a packed batch owns nodes [off[b], off[b + 1]) of every
// per-node array; its m and n_survivors are entry b, its out_tokens start at
// off[b] + b (n_b + 1 entries each).
struct WalkJobs {
  int32_t off[kMaxBatch + 1];
  int32_t prefix[kMaxBatch];
};

__global__ void __launch_bounds__(32)
walk_kernel(const __grid_constant__ WalkJobs jobs, const int32_t* __restrict__ token_all,
            const int32_t* __restrict__ parent_all, const int32_t* __restrict__ am_all,
            int vocab, int32_t* m_out, int32_t* path, int32_t* out_tokens, int32_t* new_pos,
            int32_t* new_parent, int32_t* n_surv, int32_t* dev_status) {
  __shared__ int32_t par[kMaxNodes], tok[kMaxNodes], amv[kMaxNodes], rank_of[kMaxNodes];
  __shared__ int32_t plist[kMaxNodes];
  // launched under programmatic serialization after the argmax (or the
  // sampling): wait for it; a compaction launched after this kernel may be
  // scheduled now and waits for it in turn
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x;
  const int b = blockIdx.x;
  const int o = jobs.off[b];
  const int n = jobs.off[b + 1] - o;
  const int prefix = jobs.prefix[b];
  const int32_t* token = token_all + o;
  const int32_t* parent = parent_all + o;
  const int32_t* am = am_all + o;
  m_out += b;
  n_surv += b;
  path += o;
  out_tokens += o + b;
  new_pos += o;
  new_parent += o;
  bool ok = true;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = lane + 32 * k;
    if (i < n) {
      const int p = parent[i], t = token[i], a = am[i];
      par[i] = p;
      tok[i] = t;
      amv[i] = a;
      ok &= (i == 0) ? (p == -1) : (p >= -1 && p < i);
      ok &= (t >= 0 && t < vocab);
    }
  }
  const bool bad = __any_sync(0xffffffffu, !ok);
  if (bad) {
    if (lane == 0) {
      report(dev_status, TV_ERR_INVALID_TREE);
      *m_out = 0;
      *n_surv = 0;
    }
    for (int i = lane; i < n; i += 32) {
      path[i] = -1;
      new_pos[i] = -1;
      new_parent[i] = -1;
    }
    for (int i = lane; i <= n; i += 32) out_tokens[i] = -1;
    return;
  }
  __syncwarp();

  // greedy walk from the root
  uint32_t onpath[4] = {0u, 0u, 0u, 0u};
  int u = 0, len = 1;
  onpath[0] = 1u;
  if (lane == 0) plist[0] = 0;
  for (int step = 0; step < n; ++step) {
    const int want = amv[u];
    int next = -1;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = lane + 32 * k;
      const bool match = i < n && par[i] == u && tok[i] == want;
      const uint32_t b = __ballot_sync(0xffffffffu, match);
      if (next < 0 && b != 0u) next = 32 * k + __ffs(b) - 1;
    }
    if (next < 0) break;
    u = next;
    onpath[u >> 5] |= 1u << (u & 31);
    if (lane == 0) plist[len] = u;
    ++len;
  }
  const int am_last = u;
  const int m = len - 1;

  // strict descendants of the last accepted node, then ranks in node order
  uint32_t keep[4];
  int base = 0;
  int my_rank[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = lane + 32 * k;
    bool kp = false;
    if (i < n) {
      kp = (onpath[k] >> lane) & 1u;
      if (!kp && i > am_last) {
        int x = par[i];
        while (x > am_last) x = par[x];  // indices fall strictly along the walk
        kp = (x == am_last);
      }
    }
    keep[k] = __ballot_sync(0xffffffffu, kp);
    my_rank[k] = kp ? base + __popc(keep[k] & ((1u << lane) - 1u)) : -1;
    base += __popc(keep[k]);
  }
  const int r = base - (m + 1);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = lane + 32 * k;
    if (i < n) rank_of[i] = my_rank[k];
  }
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = lane + 32 * k;
    if (i >= n) continue;
    const int rk = my_rank[k];
    new_pos[i] = rk >= 0 ? prefix + rk : -1;
    if (rk > m) {
      const int pp = par[i];
      if (guard(rk - (m + 1) < n && pp >= 0 && pp < n, dev_status))
        new_parent[rk - (m + 1)] = (pp == am_last) ? -1 : rank_of[pp] - (m + 1);
    }
    if (i >= r) new_parent[i] = -1;
    path[i] = i <= m ? plist[i] : -1;
  }
  for (int i = lane; i <= n; i += 32) {
    if (i < m && !guard(plist[i + 1] >= 0 && plist[i + 1] < n, dev_status)) continue;
    out_tokens[i] = i < m ? tok[plist[i + 1]] : (i == m ? amv[am_last] : -1);
  }
  if (lane == 0) {
    *m_out = m;
    *n_surv = r;
  }
}

}  // namespace

cudaError_t launch_accept(const float* logits, int32_t vocab, const int32_t* token,
                          const int32_t* parent, int32_t n, int32_t prefix, int32_t* am,
                          int32_t* m, int32_t* path, int32_t* out_tokens, int32_t* new_pos,
                          int32_t* new_parent, int32_t* n_survivors, int32_t* dev_status,
                          cudaStream_t s) {
  const int32_t off[2] = {0, n};
  return launch_accept_batched(logits, vocab, token, parent, 1, off, &prefix, am, m, path,
                               out_tokens, new_pos, new_parent, n_survivors, dev_status, s);
}

cudaError_t launch_accept_batched(const float* logits, int32_t vocab, const int32_t* token,
                                  const int32_t* parent, int32_t batch,
                                  const int32_t* node_offset, const int32_t* prefix,
                                  int32_t* am, int32_t* m, int32_t* path, int32_t* out_tokens,
                                  int32_t* new_pos, int32_t* new_parent, int32_t* n_survivors,
                                  int32_t* dev_status, cudaStream_t s) {
  cudaError_t e = launch_pdl(argmax_kernel, dim3(kArgmaxCluster, node_offset[batch]),
                             dim3(kArgmaxThreads), 0, s, logits, vocab, am);
  if (e != cudaSuccess) return e;
  return launch_walk_batched(token, parent, am, batch, node_offset, vocab, prefix, m, path,
                             out_tokens, new_pos, new_parent, n_survivors, dev_status, s);
}

cudaError_t launch_walk(const int32_t* token, const int32_t* parent, const int32_t* am,
                        int32_t n, int32_t vocab, int32_t prefix, int32_t* m, int32_t* path,
                        int32_t* out_tokens, int32_t* new_pos, int32_t* new_parent,
                        int32_t* n_survivors, int32_t* dev_status, cudaStream_t s) {
  const int32_t off[2] = {0, n};
  return launch_walk_batched(token, parent, am, 1, off, vocab, &prefix, m, path, out_tokens,
                             new_pos, new_parent, n_survivors, dev_status, s);
}

cudaError_t launch_walk_batched(const int32_t* token, const int32_t* parent, const int32_t* am,
                                int32_t batch, const int32_t* node_offset, int32_t vocab,
                                const int32_t* prefix, int32_t* m, int32_t* path,
                                int32_t* out_tokens, int32_t* new_pos, int32_t* new_parent,
                                int32_t* n_survivors, int32_t* dev_status, cudaStream_t s) {
  WalkJobs jobs{};
  for (int b = 0; b < batch; ++b) {
    jobs.off[b] = node_offset[b];
    jobs.prefix[b] = prefix[b];
  }
  jobs.off[batch] = node_offset[batch];
  return launch_pdl(walk_kernel, dim3(batch), dim3(32), 0, s, jobs, token, parent, am, vocab, m,
                    path, out_tokens, new_pos, new_parent, n_survivors, dev_status);
}

}  // namespace tv
