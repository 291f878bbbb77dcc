// The draft side of tree speculation: maximum-likelihood tree expansion and
// draft-side re-rooting.
//
// Expansion (SwiftSpec review page, "Assumptions & free parameters": a path
// scores the sum of the log-softmax probabilities along it, and the leaves to
// add are the best-scoring ones).  The candidates are the children (f, v) of
// the frontier nodes, scored cum[frontier[f]] + (z_f[v] - lse_f); the w best
// become new leaves, best first, equal scores going to the lower frontier
// position and then the lower token id.
//
//   chunk kernel  grid (chunks, F): one CTA holds a slice of one logits row
//                 in registers, reduces its maximum and its sum of
//                 exp(z - max), and extracts the slice's w largest logits
//                 (ties to the lower token id): each warp takes its own w
//                 best, then one warp the best of those.  Within a row the score order
//                 is the logit order, so the row's best w are among the
//                 slices' best w.
//   merge kernel  one cluster of up to 8 CTAs (one per 8 rows): a warp per
//                 row turns the row's slice records into its log-sum-exp
//                 and its w best candidates; CTA 0 gathers every row's list
//                 through distributed shared memory and one warp picks the
//                 w best of all rows by score.
//
// Re-rooting (review page, "What carries the argument": the draft tree
// re-roots at the last verified token and keeps the still-useful subtree):
// one warp finds the child b of the last accepted node that carries the bonus
// token and ranks b's subtree with ballots; the path and the subtree move to
// the rows after the prefix (tv_kv_compact applies the map to the cache).
#include <algorithm>
#include <climits>
#include <cmath>

#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace tv {

namespace cg = cooperative_groups;

namespace {

constexpr int kChunkThreads = 256;
constexpr int kChunkWarps = kChunkThreads / 32;
// logits per thread: 8 (slices of up to 2048 logits) unless the vocabulary
// needs longer slices, then 32 (up to 8192)
constexpr int kShortSlice = kChunkThreads * 8;
constexpr int kMaxChunkLen = kChunkThreads * 32;
constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMergeCluster = 8;  // merge CTAs at most (a portable cluster)
constexpr int kRowCands = 1024;  // slice candidates of one row: chunks * w

// A candidate is (value, key): key >= 0 identifies it (a token id, or a
// frontier position and a token), key < 0 is "none".  Order: larger value
// first, then the lower key.
__device__ __forceinline__ bool before(float z, int i, float y, int j) {
  // written without branches: the selection loops below run it in long
  // unrolled chains where a branch per compare would dominate
  const bool better = (z > y) | ((z == y) & (i < j));
  return (i >= 0) & ((j < 0) | better);
}

// Best live entry of N register-held candidates by a pairwise tree (depth
// log2 N rather than a dependent chain of N compares); q is its slot.
template <int N>
__device__ __forceinline__ void tree_best(const float (&v)[N], const int (&key)[N], uint32_t live,
                                          float& bv, int& bk, int& bq) {
  float tv[N];
  int tk[N], tq[N];
#pragma unroll
  for (int q = 0; q < N; ++q) {
    const bool on = (live >> q) & 1u;
    tv[q] = v[q];
    tk[q] = on ? key[q] : -1;
    tq[q] = q;
  }
#pragma unroll
  for (int step = 1; step < N; step <<= 1)
#pragma unroll
    for (int q = 0; q + step < N; q += 2 * step) {
      const bool b = before(tv[q + step], tk[q + step], tv[q], tk[q]);
      tv[q] = b ? tv[q + step] : tv[q];
      tk[q] = b ? tk[q + step] : tk[q];
      tq[q] = b ? tq[q + step] : tq[q];
    }
  bv = tv[0];
  bk = tk[0];
  bq = tq[0];
}

// Order-preserving map of a float to an unsigned integer (larger float,
// larger integer); 0 is below every float and marks "no candidate".
__device__ __forceinline__ uint32_t ordered_bits(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float from_ordered_bits(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// The warp's best candidate under before(): the largest value by a hardware
// warp reduction, then the lowest key among the lanes that hold it.
__device__ __forceinline__ void warp_best(float& v, int& k) {
  const uint32_t o = k >= 0 ? ordered_bits(v) : 0u;
  const uint32_t best = __reduce_max_sync(0xffffffffu, o);
  const uint32_t kk = (k >= 0 && o == best) ? (uint32_t)k : 0xffffffffu;
  const uint32_t bk = __reduce_min_sync(0xffffffffu, kk);
  k = best == 0u ? -1 : (int)bk;
  v = best == 0u ? 0.f : from_ordered_bits(best);
}

// One warp takes the r best of N candidates per lane (keys distinct),
// writing them best first to out_v / out_k (lane 0).
template <int N>
__device__ __forceinline__ void warp_take(const float (&v)[N], const int (&key)[N], int r,
                                          float* out_v, int* out_k) {
  const int lane = threadIdx.x & 31;
  uint32_t live = N == 32 ? 0xffffffffu : ((1u << N) - 1u);
  float bv;
  int bk, bq;
  tree_best<N>(v, key, live, bv, bk, bq);
  for (int t = 0; t < r; ++t) {
    float wv = bv;
    int wk = bk;
    warp_best(wv, wk);
    if (lane == 0) { out_v[t] = wv; out_k[t] = wk; }
    if (wk >= 0 && wk == bk) {  // this lane held the winner
      live &= ~(1u << bq);
      tree_best<N>(v, key, live, bv, bk, bq);
    }
  }
}

// Sorts 8 register-held candidates best first under before() with Knuth's
// optimal 19-comparator network (empty slots, key < 0, end up last).
__device__ __forceinline__ void sort8(float (&v)[8], int (&k)[8]) {
  constexpr int kNet[19][2] = {{0, 2}, {1, 3}, {4, 6}, {5, 7}, {0, 4}, {1, 5}, {2, 6},
                               {3, 7}, {0, 1}, {2, 3}, {4, 5}, {6, 7}, {2, 4}, {3, 5},
                               {1, 4}, {3, 6}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
  for (int c = 0; c < 19; ++c) {
    const int a = kNet[c][0], b = kNet[c][1];
    const bool swap = before(v[b], k[b], v[a], k[a]);
    const float va = v[a], vb = v[b];
    const int ka = k[a], kb = k[b];
    v[a] = swap ? vb : va;
    v[b] = swap ? va : vb;
    k[a] = swap ? kb : ka;
    k[b] = swap ? ka : kb;
  }
}

// warp_take for 8 candidates per lane: each lane sorts its 8 once, so a round
// is one warp reduction over the lanes' heads and a register shift in the
// winning lane (instead of re-scanning its candidates).
__device__ __forceinline__ void warp_take8(float (&v)[8], int (&key)[8], int r, float* out_v,
                                           int* out_k) {
  const int lane = threadIdx.x & 31;
  sort8(v, key);
  for (int t = 0; t < r; ++t) {
    float wv = v[0];
    int wk = key[0];
    warp_best(wv, wk);
    if (lane == 0) { out_v[t] = wv; out_k[t] = wk; }
    const bool pop = wk >= 0 && wk == key[0];  // this lane held the winner
#pragma unroll
    for (int q = 0; q < 7; ++q) {
      v[q] = pop ? v[q + 1] : v[q];
      key[q] = pop ? key[q + 1] : key[q];
    }
    key[7] = pop ? -1 : key[7];
  }
}

// One warp merges nl <= 128 lists held in shared memory, each sorted best
// first: list l is (vals, keys)[l * stride + 0 .. len), a key < 0 ending it
// early (keys distinct).  The r best go to out_v / out_k (lane 0 writes).
// Lane L follows the heads of lists L, L + 32, L + 64 and L + 96 and holds
// each list's next entry as well, so a round costs a depth-2 comparison tree,
// a warp reduction and a register select in the winning lane; the refill of
// that list's next entry from shared memory is not waited for until the list
// wins again.
__device__ __forceinline__ void warp_kmerge(const float* vals, const int* keys, int nl, int len,
                                            int stride, int r, float* out_v, int* out_k) {
  const int lane = threadIdx.x & 31;
  int head[4];
  float hv[4], nv[4];
  int hk[4], nk[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int l = lane + 32 * q;
    const bool on = l < nl && len > 0, on2 = l < nl && len > 1;
    hv[q] = on ? vals[l * stride] : 0.f;
    hk[q] = on ? keys[l * stride] : -1;
    nv[q] = on2 ? vals[l * stride + 1] : 0.f;
    nk[q] = on2 ? keys[l * stride + 1] : -1;
    head[q] = 1;
  }
  for (int t = 0; t < r; ++t) {
    const bool b1 = before(hv[1], hk[1], hv[0], hk[0]);
    const bool b3 = before(hv[3], hk[3], hv[2], hk[2]);
    const float v01 = b1 ? hv[1] : hv[0], v23 = b3 ? hv[3] : hv[2];
    const int k01 = b1 ? hk[1] : hk[0], k23 = b3 ? hk[3] : hk[2];
    const bool b = before(v23, k23, v01, k01);
    const float bv = b ? v23 : v01;
    const int bk = b ? k23 : k01;
    const int bq = b ? (b3 ? 3 : 2) : (b1 ? 1 : 0);
    float wv = bv;
    int wk = bk;
    warp_best(wv, wk);
    if (lane == 0) { out_v[t] = wv; out_k[t] = wk; }
    const bool won = wk >= 0 && wk == bk;  // this lane's list bq held the winner
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const bool pop = won && bq == q;
      hv[q] = pop ? nv[q] : hv[q];
      hk[q] = pop ? nk[q] : hk[q];
      if (pop) {
        ++head[q];
        const int l = lane + 32 * q;
        const bool on = head[q] < len;
        nv[q] = on ? vals[l * stride + head[q]] : 0.f;
        nk[q] = on ? keys[l * stride + head[q]] : -1;
      }
    }
  }
}

// Workspace record of one (row, slice): max, sum of exp(z - max), then w
// candidates (logit, token); token -1 marks an empty slot.
__host__ __device__ inline size_t record_words(int w) { return 2 + 2 * (size_t)w; }

// One slice of one row.  Thread t holds the slice's float4 groups t, t + 256,
// ... in registers (kPerThread logits).  Each warp takes its own w best
// logits, then warp 0 merges the warps' sorted lists into the slice's w best.
template <int kPerThread>
__global__ void __launch_bounds__(kChunkThreads)
expand_chunk_kernel(const float* __restrict__ logits, int vocab, int chunk_len, int w,
                    float* __restrict__ ws) {
  __shared__ float s_v[kChunkWarps * TV_MAX_EXPAND_WIDTH];
  __shared__ int s_k[kChunkWarps * TV_MAX_EXPAND_WIDTH];
  __shared__ float s_red[kChunkWarps];
  __shared__ float s_out_v[TV_MAX_EXPAND_WIDTH];
  __shared__ int s_out_k[TV_MAX_EXPAND_WIDTH];
  // launched under programmatic serialization: the merge may be scheduled
  // now (it waits for this grid); this grid waits for the kernel before it
  // (which may write the logits) before reading anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int f = blockIdx.y, c = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int beg = c * chunk_len;
  const int len = min(chunk_len, vocab - beg);
  const float* row = logits + (size_t)f * vocab + beg;
  const bool vec = ((vocab & 3) == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);

  float z[kPerThread];
  int key[kPerThread];
  // every whole float4 group is requested before any is used; groups that
  // the slice end cuts (or rows that are not 16-byte aligned) follow with
  // scalar loads
  float4 x4[kPerThread / 4];
#pragma unroll
  for (int j = 0; j < kPerThread / 4; ++j) {
    const int i0 = 4 * (tid + kChunkThreads * j);
    const bool whole = vec && i0 + 3 < len;
    x4[j] = whole ? __ldcs(reinterpret_cast<const float4*>(row + i0))
                  : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  }
#pragma unroll
  for (int j = 0; j < kPerThread / 4; ++j) {
    const int i0 = 4 * (tid + kChunkThreads * j);
    z[4 * j] = x4[j].x; z[4 * j + 1] = x4[j].y; z[4 * j + 2] = x4[j].z; z[4 * j + 3] = x4[j].w;
    if (!(vec && i0 + 3 < len)) {
#pragma unroll
      for (int e = 0; e < 4; ++e) z[4 * j + e] = i0 + e < len ? __ldcs(row + i0 + e) : -INFINITY;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) key[4 * j + e] = i0 + e < len ? beg + i0 + e : -1;
  }

  // slice maximum and sum of exp(z - max)
  float mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) mx = fmaxf(mx, z[k]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) s_red[warp] = mx;
  __syncthreads();
  mx = s_red[0];
#pragma unroll
  for (int k = 1; k < kChunkWarps; ++k) mx = fmaxf(mx, s_red[k]);
  float sum = 0.f;
  if (mx != -INFINITY)
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) sum += __expf(z[k] - mx);  // padding is -inf: 0
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  __syncthreads();
  if (lane == 0) s_red[warp] = sum;

  // each warp's w best, then the slice's w best of those
  if constexpr (kPerThread == 8)
    warp_take8(z, key, w, s_v + warp * w, s_k + warp * w);
  else
    warp_take<kPerThread>(z, key, w, s_v + warp * w, s_k + warp * w);
  __syncthreads();
  if (warp == 0) {
    float* rec = ws + ((size_t)f * gridDim.x + c) * record_words(w);
    int* rec_i = reinterpret_cast<int*>(rec);
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < kChunkWarps; ++k) t += s_red[k];
    if (lane == 0) {
      rec[0] = mx;
      rec[1] = t;
    }
    // the slice's w best of the warps' sorted lists, straight to the record
    float* out_v = rec + 2;
    warp_kmerge(s_v, s_k, kChunkWarps, w, w, w, s_out_v, s_out_k);
    __syncwarp();
    for (int k = lane; k < w; k += 32) {
      out_v[2 * k] = s_out_k[k] >= 0 ? s_out_v[k] : -INFINITY;
      rec_i[3 + 2 * k] = s_out_k[k];
    }
  }
}

// A grid of ncta <= 8 CTAs launched as one cluster.  Warp f % 8 of CTA
// (f / 8) % ncta stages row f's slice lists (each sorted best first) in
// shared memory, reduces the row's log-sum-exp and merges the lists into the
// row's w best (the score order within a row is the logit order), then
// scores them, keyed (f << 20) | token.  CTA 0 copies the other CTAs' row
// lists and frontier nodes into its own arrays (between two cluster
// barriers, so that no CTA exits while its shared memory is read) and its
// warp 0 merges the rows' lists by (score, frontier position, token).
constexpr size_t kMergeSmem = (size_t)(kMergeThreads / 32) * kRowCands * 8;

__global__ void __launch_bounds__(kMergeThreads)
expand_merge_kernel(const float* __restrict__ ws, int nf, int chunks, int w,
                    const int32_t* __restrict__ frontier, const float* __restrict__ cum,
                    int n_nodes, int32_t* new_parent, int32_t* new_token, float* new_score,
                    int32_t* dev_status) {
  extern __shared__ float merge_smem[];  // per warp: kRowCands logits, kRowCands tokens
  __shared__ float s_sc[kRowCands];      // rows' winners (nf * w <= 1024): score, key
  __shared__ int s_key[kRowCands];
  __shared__ float o_s[TV_MAX_EXPAND_WIDTH];
  __shared__ int o_k[TV_MAX_EXPAND_WIDTH];
  __shared__ int s_front[kRowCands];     // each row's frontier node (nf <= 1024)
  __shared__ int s_bad;
  // launched under programmatic serialization after the slice kernel
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t rw = record_words(w);
  // o / w as a multiply-high by ceil(2^32 / w): exact for o < 2^16 and
  // 2 <= w <= 64 (here o < kRowCands), and free of the long dependent chain
  // of an integer division.  For w = 1 that multiplier, 2^32, does not fit
  // in 32 bits: the quotient is o itself.
  const uint32_t w_recip =
      w > 1 ? (uint32_t)((0x100000000ull + (uint64_t)w - 1) / (uint64_t)w) : 0u;
  float* zl = merge_smem + (size_t)warp * 2 * kRowCands;
  int* tl = reinterpret_cast<int*>(zl + kRowCands);
  if (tid == 0) s_bad = 0;
  __syncthreads();
  const int ncta = (int)gridDim.x, cta = (int)blockIdx.x;
  for (int f = cta * kMergeWarps + warp; f < nf; f += ncta * kMergeWarps) {
    const float* rows = ws + (size_t)f * chunks * rw;
    const int total = chunks * w;
    // Every global read of the row is requested before any is waited for,
    // so that the row costs about two L2 round trips rather than five: the
    // frontier node first (its path score is a dependent load), then the
    // slice maxima and sums (rows of up to 128 slices; longer ones take a
    // second pass below) and the slice candidates.
    const int u = frontier[f];
    const bool u_ok = u >= 0 && u < n_nodes;
    const bool one_pass = chunks <= 128;
    float rm1[4], rs1[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int cc = lane + 32 * q;
      const bool on = one_pass && cc < chunks;
      rm1[q] = on ? rows[(size_t)cc * rw] : -INFINITY;
      rs1[q] = on ? rows[(size_t)cc * rw + 1] : 0.f;
    }
    float base = 0.f;
    // staged 32 loads per lane at a time (all of them when chunks * w <= 1024),
    // all issued before any is stored
    for (int o0 = 0; o0 < total; o0 += 32 * 32) {
      float zv[32];
      int tv[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int o = min(o0 + lane + 32 * q, total - 1);
        const int cc = w > 1 ? (int)__umulhi((uint32_t)o, w_recip) : o, k = o - cc * w;
        const float* rec = rows + (size_t)cc * rw;
        zv[q] = rec[2 + 2 * k];
        tv[q] = reinterpret_cast<const int*>(rec)[3 + 2 * k];
      }
      if (o0 == 0 && u_ok) base = cum[u];
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int o = o0 + lane + 32 * q;
        if (o < total) {
          zl[o] = zv[q];
          tl[o] = tv[q];
        }
      }
    }
    // log-sum-exp: M = max m_c, S = sum s_c e^(m_c - M), four slice records
    // per lane at a time
    float m = one_pass ? fmaxf(fmaxf(rm1[0], rm1[1]), fmaxf(rm1[2], rm1[3])) : -INFINITY;
    for (int c0 = 0; !one_pass && c0 < chunks; c0 += 128) {
      float rm[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int cc = c0 + lane + 32 * q;
        rm[q] = cc < chunks ? rows[(size_t)cc * rw] : -INFINITY;
      }
      m = fmaxf(m, fmaxf(fmaxf(rm[0], rm[1]), fmaxf(rm[2], rm[3])));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float sum = 0.f;
    if (m != -INFINITY) {
      if (one_pass) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (rm1[q] != -INFINITY) sum += rs1[q] * __expf(rm1[q] - m);
      }
      for (int c0 = 0; !one_pass && c0 < chunks; c0 += 128) {
        float rm[4], rs[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int cc = c0 + lane + 32 * q;
          rm[q] = cc < chunks ? rows[(size_t)cc * rw] : -INFINITY;
          rs[q] = cc < chunks ? rows[(size_t)cc * rw + 1] : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (rm[q] != -INFINITY) sum += rs[q] * __expf(rm[q] - m);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float lse = m + __logf(sum);
    if (lane == 0) {
      s_front[f] = u;
      if (!u_ok) s_bad = 1;
    }
    __syncwarp();
    warp_kmerge(zl, tl, chunks, w, w, w, s_sc + f * w, s_key + f * w);
    __syncwarp();
    for (int k = lane; k < w; k += 32) {
      // a row whose logits are all -inf has no children
      const int tok = s_key[f * w + k];
      const bool ok = tok >= 0 && lse > -INFINITY;
      s_key[f * w + k] = ok ? ((f << 20) | tok) : -1;
      s_sc[f * w + k] = ok ? base + (s_sc[f * w + k] - lse) : -INFINITY;
    }
    __syncwarp();
  }
  __syncthreads();
  if (ncta > 1) {
    // the grid is one cluster: CTA 0 gathers the other CTAs' row lists, row
    // f being held by CTA (f / 8) mod ncta, then merges every row
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (cta == 0) {
      for (int o = tid; o < nf * w; o += kMergeThreads) {
        const int r = (o / w / kMergeWarps) % ncta;
        if (r != 0) {
          s_sc[o] = *cluster.map_shared_rank(&s_sc[o], r);
          s_key[o] = *cluster.map_shared_rank(&s_key[o], r);
        }
      }
      for (int f = tid; f < nf; f += kMergeThreads) {
        const int r = (f / kMergeWarps) % ncta;
        if (r != 0) s_front[f] = *cluster.map_shared_rank(&s_front[f], r);
      }
      if (tid == 0)
        for (int r = 1; r < ncta; ++r)
          if (*cluster.map_shared_rank(&s_bad, r)) s_bad = 1;
    }
    cluster.sync();  // every CTA's shared memory stays until CTA 0 has read it
    if (cta != 0) return;
    __syncthreads();
  }
  if (s_bad) {
    if (tid == 0) report(dev_status, TV_ERR_INVALID_ARG);
    for (int k = tid; k < w; k += kMergeThreads) {
      new_parent[k] = -1;
      new_token[k] = -1;
      new_score[k] = -INFINITY;
    }
    return;
  }
  if (warp == 0) {
    warp_kmerge(s_sc, s_key, nf, w, w, w, o_s, o_k);
    __syncwarp();
    for (int k = lane; k < w; k += 32) {
      const int kk = o_k[k];
      new_parent[k] = kk >= 0 ? s_front[kk >> 20] : -1;
      new_token[k] = kk >= 0 ? (kk & 0xfffff) : -1;
      new_score[k] = kk >= 0 ? o_s[k] : -INFINITY;
    }
  }
}

__global__ void __launch_bounds__(32)
draft_reroot_kernel(const int32_t* __restrict__ parent, const int32_t* __restrict__ token,
                    const float* __restrict__ cum, int n, const int32_t* __restrict__ path,
                    const int32_t* __restrict__ m_in, const int32_t* __restrict__ out_tokens,
                    int prefix, int32_t* new_pos, int32_t* new_parent, int32_t* new_token,
                    float* new_cum, int32_t* n_surv, int32_t* dev_status) {
  __shared__ int32_t par[kMaxNodes], tok[kMaxNodes], rank_of[kMaxNodes];
  // launched under programmatic serialization after the walk whose path,
  // m and out_tokens it reads
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x;
  const int m = *m_in;
  bool ok = m >= 0 && m < n;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = lane + 32 * k;
    if (i < n) {
      const int p = parent[i];
      par[i] = p;
      tok[i] = token[i];
      ok &= (i == 0) ? (p == -1) : (p >= -1 && p < i);
    }
  }
  ok = !__any_sync(0xffffffffu, !ok);
  __syncwarp();
  // the accepted path must be a root-to-node chain of this tree
  if (ok) {
    bool pok = true;
    for (int k = lane; k <= m; k += 32) {
      const int a = path[k];
      const int want_parent = k == 0 ? -1 : path[k - 1];
      pok &= a >= 0 && a < n && (k == 0 ? a == 0 : par[a] == want_parent);
    }
    ok = !__any_sync(0xffffffffu, !pok);
  }
  if (!ok) {
    if (lane == 0) {
      report(dev_status, TV_ERR_INVALID_TREE);
      *n_surv = 0;
    }
    for (int i = lane; i < n; i += 32) {
      new_pos[i] = -1;
      new_parent[i] = -1;
      new_token[i] = -1;
      new_cum[i] = 0.f;
    }
    return;
  }
  const int am_last = path[m];
  const int bonus = out_tokens[m];
  // the new root: the lowest-indexed child of a_m carrying the bonus token
  int b = -1;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = lane + 32 * k;
    const uint32_t hit = __ballot_sync(0xffffffffu, i < n && par[i] == am_last && tok[i] == bonus);
    if (b < 0 && hit != 0u) b = 32 * k + __ffs(hit) - 1;
  }
  // b's subtree (b and its descendants) in node order, ranked by ballots
  int my_rank[4];
  int base = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = lane + 32 * k;
    bool s = false;
    if (b >= 0 && i < n && i >= b) {
      int x = i;
      while (x > b) x = par[x];  // indices fall strictly along the walk
      s = (x == b);
    }
    const uint32_t bal = __ballot_sync(0xffffffffu, s);
    my_rank[k] = s ? base + __popc(bal & ((1u << lane) - 1u)) : -1;
    base += __popc(bal);
  }
  const int r = base;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = lane + 32 * k;
    if (i < n) rank_of[i] = my_rank[k];
  }
  __syncwarp();
  const float cum_b = b >= 0 ? cum[b] : 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = lane + 32 * k;
    if (i >= n) continue;
    const int rk = my_rank[k];
    int pos = -1;
    if (rk >= 0) {
      pos = prefix + m + 1 + rk;
      new_parent[rk] = i == b ? -1 : rank_of[par[i]];
      new_token[rk] = tok[i];
      new_cum[rk] = cum[i] - cum_b;
    }
    new_pos[i] = pos;
  }
  __syncwarp();
  // the path rows (a node on the path is never in b's subtree)
  for (int k = lane; k <= m; k += 32) new_pos[path[k]] = prefix + k;
  for (int i = r + lane; i < n; i += 32) {
    new_parent[i] = -1;
    new_token[i] = -1;
    new_cum[i] = 0.f;
  }
  if (lane == 0) *n_surv = r;
}

}  // namespace

ExpandPlan plan_expand(int32_t n_frontier, int32_t vocab, int32_t w) {
  ExpandPlan pl{};
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      sms = v;
  }
  // About four slices per SM in all, each of at least 1024 logits where the
  // vocabulary allows.  Short slices (up to 2048 logits, 8 per thread) are
  // used when the merge can take their candidates (at most kRowCands slice
  // candidates per row), else long ones (up to 8192); the argument limit
  // ceil(vocab / 8192) * w <= TV_MAX_EXPAND_CANDIDATES keeps the long case
  // within bounds.
  const int cap_len = ((vocab + kShortSlice - 1) / kShortSlice) * w <= kRowCands ? kShortSlice
                                                                             : kMaxChunkLen;
  const int lo = (vocab + cap_len - 1) / cap_len;
  const int hi = std::max(lo, std::min((vocab + 1023) / 1024, kRowCands / w));
  const int chunks = std::min(hi, std::max(lo, (4 * sms + n_frontier - 1) / n_frontier));
  int len = (vocab + chunks - 1) / chunks;
  len = (len + 3) & ~3;
  pl.chunk_len = len;
  pl.chunks = (vocab + len - 1) / len;
  pl.ws_bytes = (size_t)n_frontier * pl.chunks * record_words(w) * 4;
  return pl;
}

cudaError_t launch_expand(const float* logits, int32_t vocab, int32_t n_frontier,
                          const int32_t* frontier, const float* cum, int32_t n_nodes, int32_t w,
                          int32_t* new_parent, int32_t* new_token, float* new_score, void* ws,
                          int32_t* dev_status, cudaStream_t s) {
  const ExpandPlan pl = plan_expand(n_frontier, vocab, w);
  const dim3 grid(pl.chunks, n_frontier);
  float* wsf = static_cast<float*>(ws);
  cudaError_t e = pl.chunk_len <= kShortSlice
                      ? launch_pdl(expand_chunk_kernel<8>, grid, dim3(kChunkThreads), 0, s,
                                   logits, vocab, pl.chunk_len, w, wsf)
                      : launch_pdl(expand_chunk_kernel<32>, grid, dim3(kChunkThreads), 0, s,
                                   logits, vocab, pl.chunk_len, w, wsf);
  if (e != cudaSuccess) return e;
  static std::atomic<bool> attr_set[64];  // per device (host threads may race here)
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(expand_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kMergeSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  // one CTA per 8 rows up to a cluster of kMergeCluster, launched as one
  // cluster under programmatic serialization
  const int ncta = std::min(kMergeCluster, (n_frontier + kMergeWarps - 1) / kMergeWarps);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ncta);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = kMergeSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = ncta;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = ncta > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, expand_merge_kernel, static_cast<const float*>(ws), n_frontier,
                            pl.chunks, w, frontier, cum, n_nodes, new_parent, new_token,
                            new_score, dev_status);
}

cudaError_t launch_draft_reroot(const int32_t* parent, const int32_t* token, const float* cum,
                                int32_t n, const int32_t* path, const int32_t* m,
                                const int32_t* out_tokens, int32_t prefix, int32_t* new_pos,
                                int32_t* new_parent, int32_t* new_token, float* new_cum,
                                int32_t* n_survivors, int32_t* dev_status, cudaStream_t s) {
  return launch_pdl(draft_reroot_kernel, dim3(1), dim3(32), 0, s, parent, token, cum, n, path, m,
                    out_tokens, prefix, new_pos, new_parent, new_token, new_cum, n_survivors,
                    dev_status);
}

}  // namespace tv
