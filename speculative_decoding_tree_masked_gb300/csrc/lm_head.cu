// The target's LM head fused with the argmax.
//
// For the tree nodes' final hidden states H [n][d] and the LM-head weights
// W [V][d] (bf16, rows contiguous) the kernel writes am[i] = argmax_v H[i].W[v]
// (ties to the lowest v) without ever storing the n x V logits: greedy
// verification needs only the target's argmax at every node (SwiftSpec review
// page, "What carries the argument": the emitted tokens are the target's), so
// the logits never leave the chip.
//
// One CTA per SM streams its share of the weight rows once, in tiles of 224
// rows: the whole tiles are dealt round-robin, so that the CTAs read
// neighbouring rows at the same time, and the rows after the last whole
// round are cut into 16-row units dealt in equal runs, so every SM moves the
// same bytes of W to within 16 rows.  With n small next to V the kernel is
// bound by the HBM reads of W.
//
// The products run on the tcgen05 tensor cores:
//   A = H rows       M = 128 nodes per node chunk (TMA zero-fills rows past n)
//   B = W tile       up to 224 weight rows (the MMA's N)
//   D = TMEM         [128 node lanes][224 vocab columns] fp32 per node chunk
// over K steps of 64 columns of d, one 128-byte-swizzled TMA box per operand
// and stage.  A tile's epilogue thread owns one node lane and scans the
// tile's columns in vocabulary order, keeping the first maximum.  (Measured
// on the W stream alone: 224-row boxes beat 256-row ones by 1.5%, partly by
// fitting a sixth stage; dealing tiles round-robin instead of contiguous
// runs per CTA gained 0.7%.)
//
// Warp roles (192 threads):
//   warp 0      TMA producer: H and W boxes into a ring of stages
//   warp 1      TMEM allocator and MMA issuer (one thread)
//   warps 2-5   epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31
//
// Across CTAs: each CTA stores one 64-bit key per node,
//   (order-preserving bits of its largest logit) << 32 | (2^32 - 1 - id),
// so that the largest key is the largest logit with the lowest id.  The last
// CTA to finish (a counter in the workspace) takes the maximum key of every
// node over the CTAs and writes am and the maximum logit.
//
// Every wait is bounded; on expiry the kernel records TV_ERR_TIMEOUT, the
// other roles stop at their next wait, and the CTA waits (bounded) for its
// copies and products in flight before it frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace tv {

namespace {

constexpr int kLmThreads = 192;
constexpr int kTileRows = 224;            // weight rows per tile (MMA N)
constexpr int kUnitRows = 16;             // rows of the work split and of a tail box
constexpr int kNodeRows = 128;            // nodes per chunk (MMA M, TMEM lanes)
constexpr int kWSlot = kTileRows * 128;   // one stage of W: 224 rows x 64 bf16
constexpr int kTailBox = kUnitRows * 128;
constexpr long long kLmWaitCycles = 4000000000LL;
constexpr uint32_t kLmSleepNs = 20000;

constexpr int kMaxStages = 8;
constexpr int kARead = kNodeRows * 128;   // bytes an MMA reads from an H slot (128 rows)
// Dynamic shared memory: 1024 bytes of alignment slack, then the W slots,
// the H slots, the barriers and a few words.  An H slot holds only the rows
// of the H box (a small tree needs a small slot), so that more stages and
// bytes of W fit in flight; but the MMA reads 128 rows (kARead bytes) from
// the slot's start, so the H region is padded to keep the last slot's read
// inside it.  Rows past the box belong to neighbouring slots or the pad:
// they only reach TMEM lanes of nodes >= n, which nothing reads.
constexpr int kSmemLimit = 232448;   // 227 KB, the most a CTA may have
constexpr int kBarBytes = 8 * (2 * kMaxStages + 3) + 16;

struct LmShape {
  int stages;
  int hslot;      // bytes of one node chunk of H per stage (1024-aligned)
  int smem;       // dynamic shared memory of a CTA
};

// Bytes of the H region: S * nc slots and the pad after the last one.
__host__ __device__ constexpr int h_region(int stages, int nc, int hslot) {
  return (stages * nc - 1) * hslot + kARead;
}

LmShape lm_shape(int nc, int hbox_rows) {
  LmShape sh;
  sh.hslot = ((hbox_rows * 128) + 1023) & ~1023;
  const int stage = kWSlot + nc * sh.hslot;
  const int fixed = 1024 + kBarBytes + (kARead - sh.hslot);
  sh.stages = std::min(kMaxStages, (kSmemLimit - fixed) / stage);
  sh.smem = 1024 + sh.stages * kWSlot + h_region(sh.stages, nc, sh.hslot) + kBarBytes;
  return sh;
}

struct LmArgs {
  CUtensorMap hmap;     // H [n][d], boxes of 64 columns x hbox_rows rows
  CUtensorMap wmap;     // W [V][d], boxes of 64 columns x kTileRows rows
  CUtensorMap tmap;     // W [V][d], boxes of 64 columns x 16 rows (tile tails)
  int32_t n, d, vocab, hbox_rows, stages, hslot;
  int32_t* am;
  float* max_logit;
  unsigned long long* keys;   // [n][gridDim.x]
  unsigned int* counter;
  int32_t* dev_status;
};

__device__ __forceinline__ bool lm_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                        int32_t* dev_status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait_sleep(bar, parity, kLmSleepNs)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kLmWaitCycles) {
      *abort_flag = 1;
      report(dev_status, TV_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// A wait that ignores the abort flag, for copies or products still in
// flight when a CTA gives up; bounded all the same.
__device__ __forceinline__ void lm_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait_sleep(bar, parity, kLmSleepNs))
    if (clock64() - t0 > kLmWaitCycles) return;
}

__device__ __forceinline__ uint32_t ordered_bits(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float from_ordered_bits(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

template <int NC>
__global__ void __launch_bounds__(kLmThreads, 1)
lm_head_argmax_kernel(const __grid_constant__ LmArgs a) {
  constexpr uint32_t kTmemCols = NC * 256;
  const int S = a.stages;
  // W slot s at sW + s * kWSlot, H slot (s, c) at sH + (s * NC + c) * hslot
  const uint32_t sW = 0, sH = S * kWSlot, sBar = sH + h_region(S, NC, a.hslot);
  const uint32_t sMisc = sBar + 8 * (2 * S + 3);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t base = ptx::smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, b = blockIdx.x;

  // Whole tiles are dealt round-robin (this CTA's tile t starts at row
  // (t G + b) kTileRows, so the CTAs read neighbouring rows at the same
  // time); the rows past the last whole round are cut into 16-row units,
  // dealt in equal runs: one last, partial tile per CTA.
  const int rounds = a.vocab / (G * kTileRows);
  const int tail0 = rounds * G * kTileRows;
  const int tunits = (a.vocab - tail0 + kUnitRows - 1) / kUnitRows;
  const int tu0 = (int)((long long)tunits * b / G), tu1 = (int)((long long)tunits * (b + 1) / G);
  const int tr0 = tail0 + tu0 * kUnitRows, tr1 = min(a.vocab, tail0 + tu1 * kUnitRows);
  const int ntiles = rounds + (tr1 > tr0 ? 1 : 0);
  auto tile_row0 = [&](int t) { return t < rounds ? (t * G + b) * kTileRows : tr0; };
  auto tile_rows = [&](int t) { return t < rounds ? kTileRows : tr1 - tr0; };
  const int nk = (a.d + 63) / 64;

  const uint32_t bar0 = base + sBar;
  auto full = [&](int s) { return bar0 + 8 * s; };            // stage s has landed
  auto empty = [&](int s) { return bar0 + 8 * (S + s); };     // stage s has been read
  const uint32_t acc_full = bar0 + 8 * (2 * S);               // a tile's products are done
  const uint32_t acc_empty = bar0 + 8 * (2 * S + 1);          // its epilogue has read TMEM
  const uint32_t done = bar0 + 8 * (2 * S + 2);               // every product is done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + sMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + sMisc + 4);
  volatile int* is_last = reinterpret_cast<volatile int*>(sm + sMisc + 8);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(full(s), 1);
      ptx::mbar_init(empty(s), 1);
    }
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(acc_empty, 4);
    ptx::mbar_init(done, 1);
    *abort_flag = 0;
    *is_last = 0;
    ptx::fence_mbar_init();
    ptx::tma_prefetch_desc(&a.hmap);
    if (a.vocab >= kTileRows) ptx::tma_prefetch_desc(&a.wmap);
    ptx::tma_prefetch_desc(&a.tmap);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t hbytes = NC * a.hbox_rows * 128;
      int it = 0, s = 0;
      uint32_t ph = 0;  // phase of the ring's current pass
      bool ok = true;
      for (int t = 0; ok && t < ntiles; ++t) {
        const int row0 = tile_row0(t);
        const int rows = tile_rows(t);
        const bool whole = rows == kTileRows;
        const int nbox = whole ? 1 : (rows + kUnitRows - 1) / kUnitRows;
        const uint32_t bytes = hbytes + (whole ? kWSlot : nbox * kTailBox);
        for (int k = 0; k < nk; ++k) {
          if (it >= S && !(ok = lm_wait(empty(s), ph ^ 1u, abort_flag, a.dev_status))) break;
          ptx::mbar_arrive_expect_tx(full(s), bytes);
#pragma unroll
          for (int c = 0; c < NC; ++c)
            ptx::tma_load_2d(base + sH + (s * NC + c) * a.hslot, &a.hmap, full(s), k * 64,
                             c * kNodeRows);
          const uint32_t wdst = base + sW + s * kWSlot;
          if (whole) {
            ptx::tma_load_2d(wdst, &a.wmap, full(s), k * 64, row0);
          } else {
            for (int x = 0; x < nbox; ++x)
              ptx::tma_load_2d(wdst + x * kTailBox, &a.tmap, full(s), k * 64,
                               row0 + x * kUnitRows);
          }
          ++it;
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        // the last (up to S) stages issued may still be landing: each sits on
        // its own slot, whose barrier has seen no later phase
        for (int j = max(0, it - S); j < it; ++j) lm_drain(full(j % S), (j / S) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint64_t hdesc = ptx::smem_desc_sw128(base + sH, 16, 1024);
      const uint64_t wdesc = ptx::smem_desc_sw128(base + sW, 16, 1024);
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = 0; ok && t < ntiles; ++t) {
        const int rows = tile_rows(t);
        const uint32_t idesc = ptx::idesc_bf16(kNodeRows, (rows + 15) & ~15, false);
        if (t > 0 && !(ok = lm_wait(acc_empty, (t - 1) & 1, abort_flag, a.dev_status))) break;
        ptx::tc_fence_after();
        for (int k = 0; k < nk; ++k) {
          if (!(ok = lm_wait(full(s), ph, abort_flag, a.dev_status))) break;
          ptx::tc_fence_after();
#pragma unroll
          for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::mma_ss(tmem + c * 256, hdesc + (((s * NC + c) * a.hslot + kk * 32) >> 4),
                          wdesc + ((s * kWSlot + kk * 32) >> 4), idesc,
                          (k > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_commit(empty(s));
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (ok) ptx::mma_commit(acc_full);
      }
      // products still running finish before the tensor memory is freed
      ptx::mma_commit(done);
      lm_drain(done, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    float bv[NC];
    int bi[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      bv[c] = -INFINITY;
      bi[c] = -1;
    }
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int row0 = tile_row0(t);
      const int rows = tile_rows(t);
      if (!(ok = lm_wait(acc_full, t & 1, abort_flag, a.dev_status))) break;
      ptx::tc_fence_after();
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        for (int cb = 0; cb < rows; cb += 32) {
          uint32_t r[32];
          ptx::tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + c * 256 + cb, r);
          ptx::tmem_wait_ld(r);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float x = __uint_as_float(r[j]);
            if (cb + j < rows && x > bv[c]) {
              bv[c] = x;
              bi[c] = row0 + cb + j;
            }
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(acc_empty);
    }
    if (ok) {
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const int node = c * kNodeRows + 32 * q + lane;
        if (node < a.n)
          a.keys[(size_t)node * G + b] =
              bi[c] < 0 ? 0ull
                        : ((unsigned long long)ordered_bits(bv[c]) << 32) |
                              (unsigned long long)(0xFFFFFFFFu - (uint32_t)bi[c]);
      }
      __threadfence();
    }
  }

  // the last CTA to finish reduces the keys of every node over the CTAs
  __syncthreads();
  if (tid == 0 && !*abort_flag) {
    const unsigned int prev = atomicAdd(a.counter, 1u);
    *is_last = prev == (unsigned int)(G - 1);
  }
  __syncthreads();
  if (*is_last) {
    __threadfence();
    for (int node = warp; node < a.n; node += kLmThreads / 32) {
      unsigned long long k = 0ull;
      for (int c = lane; c < G; c += 32) k = max(k, __ldcg(a.keys + (size_t)node * G + c));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) k = max(k, __shfl_xor_sync(0xffffffffu, k, o));
      if (lane == 0) {
        a.am[node] = k == 0ull ? -1 : (int32_t)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
        if (a.max_logit != nullptr)
          a.max_logit[node] = k == 0ull ? -INFINITY : from_ordered_bits((uint32_t)(k >> 32));
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

int lm_grid(int32_t vocab, int sm_count) {
  const long long units = ((long long)vocab + kUnitRows - 1) / kUnitRows;
  return (int)std::max(1LL, std::min<long long>(sm_count, units));
}

bool make_rows_map(CUtensorMap* map, const void* base, int d, long long rows, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NC>
cudaError_t launch_nc(const LmArgs& args, int grid, int smem, cudaStream_t s) {
  static std::atomic<bool> attr_set[64];  // per device (host threads may race here)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(lm_head_argmax_kernel<NC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemLimit);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  lm_head_argmax_kernel<NC><<<grid, kLmThreads, smem, s>>>(args);
  return cudaGetLastError();
}

size_t keys_bytes(int32_t n, int grid) {
  return (((size_t)n * grid * sizeof(unsigned long long)) + 255) & ~size_t(255);
}

}  // namespace

size_t lm_head_workspace_bytes(int32_t n, int32_t vocab, int sm_count) {
  return keys_bytes(n, lm_grid(vocab, sm_count)) + 256;
}

cudaError_t launch_lm_head_argmax(const void* hidden, const void* weight, int32_t n,
                                  int32_t d_model, int32_t vocab, int32_t* am, float* max_logit,
                                  void* ws, int32_t* dev_status, cudaStream_t s) {
  const int grid = lm_grid(vocab, device_sm_count());
  LmArgs args;
  memset(&args, 0, sizeof(args));
  const int nc = n > kNodeRows ? 2 : 1;
  args.hbox_rows = nc == 1 ? ((n + 7) & ~7) : kNodeRows;
  const LmShape sh = lm_shape(nc, args.hbox_rows);
  args.stages = sh.stages;
  args.hslot = sh.hslot;
  if (!make_rows_map(&args.hmap, hidden, d_model, n, args.hbox_rows) ||
      !make_rows_map(&args.tmap, weight, d_model, vocab, kUnitRows))
    return cudaErrorInvalidValue;
  // whole tiles exist only when the vocabulary holds a round of them
  if (vocab >= kTileRows && !make_rows_map(&args.wmap, weight, d_model, vocab, kTileRows))
    return cudaErrorInvalidValue;
  args.n = n;
  args.d = d_model;
  args.vocab = vocab;
  args.am = am;
  args.max_logit = max_logit;
  args.keys = reinterpret_cast<unsigned long long*>(ws);
  args.counter = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + keys_bytes(n, grid));
  args.dev_status = dev_status;
  cudaError_t e = cudaMemsetAsync(args.counter, 0, sizeof(unsigned int), s);
  if (e != cudaSuccess) return e;
  return nc == 1 ? launch_nc<1>(args, grid, sh.smem, s) : launch_nc<2>(args, grid, sh.smem, s);
}

}  // namespace tv
