// Tree-masked attention on the FMA pipes (fp32 storage, and the first
// correctness path of the bf16 kernel).
//
// Grid (split, row tile, KV head).  A CTA takes 16 rows of one KV head's
// query group (row r = node * G + j is query head g * G + j of tree node
// r / G), stages 32-key tiles of K and V of its key range in shared memory as
// fp32, and runs the online softmax per row with one warp per row (lane =
// key for the scores, lane = column for the output).  The ancestor mask of a
// row's node is built in the prologue as per-node bitmask words and applied to
// keys at or past the prefix: key P + t is visible iff bit t is set.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace tv {

namespace {

constexpr int kRows = 16;
constexpr int kKeys = 32;
constexpr int kWarps = 4;
constexpr int kRowsPerWarp = kRows / kWarps;

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
attn_simt_kernel(const AttnProblem p, const int keys_per_split, float* __restrict__ ws,
                 const int splits) {
  constexpr int C = D / 32;
  __shared__ float ks[kKeys][D + 1];
  __shared__ float vs[kKeys][D];
  __shared__ float qs[kRows][D];
  __shared__ int32_t par[kMaxNodes];
  __shared__ uint32_t anc[kRows][kMaskWords];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, g = blockIdx.z;
  const int G = p.hq / p.hkv;
  const int rows_total = G * p.n;
  const int r0 = blockIdx.y * kRows;
  const T* q = static_cast<const T*>(p.q);
  const T* kc = static_cast<const T*>(p.k) + (size_t)g * p.cap * D;
  const T* vc = static_cast<const T*>(p.v) + (size_t)g * p.cap * D;

  for (int i = tid; i < p.n; i += blockDim.x) par[i] = p.parent[i];
  __syncthreads();
  if (tid < kRows) {
    uint32_t bits[kMaskWords];
    const int r = r0 + tid;
    bool ok = true;
    if (r < rows_total) ok = ancestor_bits(par, r / G, bits);
    else {
#pragma unroll
      for (int w = 0; w < kMaskWords; ++w) bits[w] = 0u;
    }
    if (!ok) report(p.dev_status, TV_ERR_INVALID_TREE);
#pragma unroll
    for (int w = 0; w < kMaskWords; ++w) anc[tid][w] = bits[w];
  }
  for (int idx = tid; idx < kRows * D; idx += blockDim.x) {
    const int rr = idx / D, c = idx % D, r = r0 + rr;
    float x = 0.f;
    if (r < rows_total) {
      const int node = r / G, j = r % G;
      x = to_f32(q[((size_t)node * p.hq + (size_t)g * G + j) * D + c]) * p.scale_log2;
    }
    qs[rr][c] = x;
  }

  const int keys = p.prefix + p.n;
  const int kbeg = split * keys_per_split;
  const int kend = min(keys, kbeg + keys_per_split);

  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][C];
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    m[rr] = -INFINITY;
    l[rr] = 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c) acc[rr][c] = 0.f;
  }

  for (int kt = kbeg; kt < kend; kt += kKeys) {
    __syncthreads();
    for (int idx = tid; idx < kKeys * D; idx += blockDim.x) {
      const int j = idx / D, c = idx % D, key = kt + j;
      float kx = 0.f, vx = 0.f;
      if (key < kend) {
        kx = to_f32(kc[(size_t)key * D + c]);
        vx = to_f32(vc[(size_t)key * D + c]);
      }
      ks[j][c] = kx;
      vs[j][c] = vx;
    }
    __syncthreads();
    const int key = kt + lane;
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      const int row = warp * kRowsPerWarp + rr;
      float s = -INFINITY;
      if (key < kend) {
        float dot = 0.f;
#pragma unroll 8
        for (int c = 0; c < D; ++c) dot = fmaf(qs[row][c], ks[lane][c], dot);
        bool visible = true;
        if (key >= p.prefix) {
          const int t = key - p.prefix;
          uint32_t bits[kMaskWords];
#pragma unroll
          for (int w = 0; w < kMaskWords; ++w) bits[w] = anc[row][w];
          visible = t < p.n && mask_bit(bits, t);
        }
        s = visible ? dot : -INFINITY;
      }
      float tmax = s;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      const float m_new = fmaxf(m[rr], tmax);
      if (m_new == -INFINITY) continue;  // nothing visible to this row yet
      const float alpha = exp2f(m[rr] - m_new);
      const float pj = exp2f(s - m_new);
      float psum = pj;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      l[rr] = l[rr] * alpha + psum;
#pragma unroll
      for (int c = 0; c < C; ++c) acc[rr][c] *= alpha;
      for (int j = 0; j < kKeys; ++j) {
        const float pb = __shfl_sync(0xffffffffu, pj, j);
#pragma unroll
        for (int c = 0; c < C; ++c) acc[rr][c] = fmaf(pb, vs[j][lane + 32 * c], acc[rr][c]);
      }
      m[rr] = m_new;
    }
  }

  const int rows_all = p.n * p.hq;
  float* wlse = ws;
  float* wo = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) +
                                       partial_o_offset(splits, rows_all));
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int r = r0 + warp * kRowsPerWarp + rr;
    if (r >= rows_total) continue;
    const int node = r / G, j = r % G;
    const size_t prow = (size_t)split * rows_all + (size_t)node * p.hq + (size_t)g * G + j;
    const float inv = l[rr] > 0.f ? 1.f / l[rr] : 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c) wo[prow * D + lane + 32 * c] = acc[rr][c] * inv;
    if (lane == 0) wlse[prow] = l[rr] > 0.f ? m[rr] + log2f(l[rr]) : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_attn_simt(const AttnProblem& p, const SplitPlan& plan, float* ws,
                             cudaStream_t s) {
  const dim3 grid(plan.splits, plan.row_tiles, p.hkv), block(kWarps * 32);
  if (p.dtype == TV_BF16) {
    if (p.d == 128)
      attn_simt_kernel<__nv_bfloat16, 128><<<grid, block, 0, s>>>(p, plan.keys_per_split, ws, plan.splits);
    else
      attn_simt_kernel<__nv_bfloat16, 64><<<grid, block, 0, s>>>(p, plan.keys_per_split, ws, plan.splits);
  } else {
    if (p.d == 128)
      attn_simt_kernel<float, 128><<<grid, block, 0, s>>>(p, plan.keys_per_split, ws, plan.splits);
    else
      attn_simt_kernel<float, 64><<<grid, block, 0, s>>>(p, plan.keys_per_split, ws, plan.splits);
  }
  return cudaGetLastError();
}

}  // namespace tv
