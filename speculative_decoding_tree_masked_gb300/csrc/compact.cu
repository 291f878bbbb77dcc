// In-place KV compaction after a verification.
//
// One CTA per (layer, KV head, K or V) slab.  new_pos is read into shared
// memory and checked (each entry -1 or a row in [P, P + i], destinations
// distinct); then every row that moves is read into shared memory, the CTA
// synchronises, and the rows are written to their destinations.  Reading all
// sources before writing any destination makes the in-place gather safe even
// though destinations overlap sources.  Rows move as 16-byte vectors.
//
// A paged cache (a pool [pages][hkv][page_size][d] per layer) maps logical
// row r to row r % page_size of page page_table[r / page_size]; a move whose
// source or destination page is outside the pool is skipped and reported.
// Several requests compact in one launch: grid.y indexes the request, each
// with its own caches (or page table), prefix, tree size and new_pos.
#include "common.cuh"
#include "internal.h"

namespace tv {

namespace {

constexpr int kCompactThreads = 256;

// One request's compaction.
struct CompactJob {
  char* k;                    // layer 0 of the K cache (or K page pool)
  char* v;
  long long layer_stride;     // bytes from one layer to the next
  long long cap;              // rows per head of a contiguous cache
  const int32_t* new_pos;     // [n]
  const int32_t* page_table;  // null: contiguous [hkv][cap][row] per layer
  int prefix;
  int n;
};

template <int MAXB>
struct CompactJobs {
  CompactJob job[MAXB];
};

template <int MAXB>
__global__ void __launch_bounds__(kCompactThreads)
compact_kernel(const __grid_constant__ CompactJobs<MAXB> jobs, int hkv, int row_bytes,
               int page_size, int num_pages, int32_t* dev_status) {
  extern __shared__ uint4 buf[];
  __shared__ int src_row[kMaxNodes], dst_row[kMaxNodes];
  __shared__ uint32_t used[kMaskWords];
  __shared__ int count;
  // launched under programmatic serialization after the walk that writes
  // new_pos: wait for it (and for every earlier kernel) before any access
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const CompactJob& job = jobs.job[blockIdx.y];
  const int prefix = job.prefix, n = job.n;
  const int32_t* __restrict__ new_pos = job.new_pos;
  const int32_t* __restrict__ page_table = job.page_table;
  const int tid = threadIdx.x;
  const int slab = blockIdx.x;
  const int which = slab & 1;
  const int g = (slab >> 1) % hkv;
  const int layer = (slab >> 1) / hkv;
  char* lbase = (which ? job.v : job.k) + (size_t)layer * job.layer_stride;
  char* base = lbase + (size_t)g * job.cap * row_bytes;
  // byte offset of logical row r, or -1 when its page is outside the pool
  auto row_at = [&](int r) -> long long {
    if (page_table == nullptr) return (long long)(base - lbase) + (long long)r * row_bytes;
    const int page = __ldg(page_table + r / page_size);
    if (page < 0 || page >= num_pages) return -1;
    return (((long long)page * hkv + g) * page_size + r % page_size) * row_bytes;
  };

  if (tid == 0) count = 0;
  if (tid < kMaskWords) used[tid] = 0u;
  __syncthreads();
  if (tid < n) {
    const int pos = new_pos[tid];
    if (pos != -1) {
      const bool in_range = pos >= prefix && pos <= prefix + tid;
      bool fresh = false;
      if (in_range) {
        const int t = pos - prefix;
        const uint32_t bit = 1u << (t & 31);
        fresh = (atomicOr(&used[t >> 5], bit) & bit) == 0u;
      }
      if (!in_range || !fresh) {
        if (slab == 0) report(dev_status, TV_ERR_INVALID_ARG);
      } else if (pos != prefix + tid) {
        if (row_at(prefix + tid) < 0 || row_at(pos) < 0) {
          if (slab == 0) report(dev_status, TV_ERR_INVALID_ARG);
        } else {
          const int k = atomicAdd(&count, 1);
          src_row[k] = prefix + tid;
          dst_row[k] = pos;
        }
      }
    }
  }
  __syncthreads();
  const int moves = count;
  const int chunks = row_bytes >> 4;
  // checked build: a moving row stays inside the tree's rows [P, P + n) of
  // its head (contiguous caches), and the staging buffer holds n rows
  auto row_ok = [&](int r) {
    return guard(r >= prefix && r < prefix + n && r < job.cap && moves <= n, dev_status);
  };
  for (int e = tid; e < moves * chunks; e += kCompactThreads) {
    const int r = e / chunks, c = e - r * chunks;
    if (page_table == nullptr && !row_ok(src_row[r])) continue;
    buf[e] = reinterpret_cast<const uint4*>(lbase + row_at(src_row[r]))[c];
  }
  __syncthreads();
  for (int e = tid; e < moves * chunks; e += kCompactThreads) {
    const int r = e / chunks, c = e - r * chunks;
    if (page_table == nullptr && !row_ok(dst_row[r])) continue;
    reinterpret_cast<uint4*>(lbase + row_at(dst_row[r]))[c] = buf[e];
  }
}

__global__ void __launch_bounds__(kMaxNodes)
tree_mask_kernel(const int32_t* __restrict__ parent, int n, uint32_t* __restrict__ words,
                 int32_t* dev_status) {
  __shared__ int32_t par[kMaxNodes];
  const int i = threadIdx.x;
  if (i < n) par[i] = parent[i];
  __syncthreads();
  if (i >= n) return;
  uint32_t bits[kMaskWords];
  if (!ancestor_bits(par, i, bits)) report(dev_status, TV_ERR_INVALID_TREE);
  const int nw = (n + 31) / 32;
  for (int w = 0; w < nw; ++w) {
    uint32_t x = bits[0];
#pragma unroll
    for (int k = 1; k < kMaskWords; ++k) x = (w == k) ? bits[k] : x;
    words[(size_t)i * nw + w] = x;
  }
}

template <int MAXB>
cudaError_t launch_jobs(const CompactJobs<MAXB>& jobs, int batch, int32_t layers, int32_t hkv,
                        int32_t row_bytes, int32_t max_n, int32_t page_size, int32_t num_pages,
                        int32_t* dev_status, cudaStream_t s) {
  static std::atomic<bool> attr_set[64];  // per device (host threads may race here)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(compact_kernel<MAXB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMaxNodes * 512);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const size_t smem = (size_t)max_n * row_bytes;
  const dim3 grid((unsigned)layers * (unsigned)hkv * 2u, (unsigned)batch);
  return launch_pdl(compact_kernel<MAXB>, grid, dim3(kCompactThreads), smem, s, jobs, hkv,
                    row_bytes, page_size, num_pages, dev_status);
}

}  // namespace

cudaError_t launch_compact(void* k, void* v, int32_t layers, int64_t layer_stride_bytes,
                           int32_t hkv, int64_t cap, int32_t row_bytes, int32_t prefix,
                           int32_t n, const int32_t* new_pos, int32_t* dev_status,
                           cudaStream_t s, const int32_t* page_table, int32_t page_size,
                           int32_t num_pages) {
  CompactJobs<1> jobs{};
  jobs.job[0] = CompactJob{static_cast<char*>(k), static_cast<char*>(v), layer_stride_bytes,
                           cap, new_pos, page_table, prefix, n};
  return launch_jobs(jobs, 1, layers, hkv, row_bytes, n, page_size, num_pages, dev_status, s);
}

cudaError_t launch_compact_batched(int32_t batch, void* const* k, void* const* v,
                                   const int64_t* layer_stride_bytes, const int64_t* cap,
                                   const int32_t* const* page_table, const int32_t* prefix,
                                   const int32_t* n, const int32_t* const* new_pos,
                                   int32_t layers, int32_t hkv, int32_t row_bytes,
                                   int32_t page_size, int32_t num_pages, int32_t* dev_status,
                                   cudaStream_t s) {
  CompactJobs<kMaxBatch> jobs{};
  int max_n = 0;
  for (int b = 0; b < batch; ++b) {
    jobs.job[b] = CompactJob{static_cast<char*>(k[b]), static_cast<char*>(v[b]),
                             layer_stride_bytes[b], cap ? cap[b] : 0, new_pos[b],
                             page_table ? page_table[b] : nullptr, prefix[b], n[b]};
    max_n = n[b] > max_n ? n[b] : max_n;
  }
  return launch_jobs(jobs, batch, layers, hkv, row_bytes, max_n, page_size, num_pages,
                     dev_status, s);
}

cudaError_t launch_tree_mask(const int32_t* parent, int32_t n, uint32_t* words,
                             int32_t* dev_status, cudaStream_t s) {
  tree_mask_kernel<<<1, kMaxNodes, 0, s>>>(parent, n, words, dev_status);
  return cudaGetLastError();
}

}  // namespace tv
