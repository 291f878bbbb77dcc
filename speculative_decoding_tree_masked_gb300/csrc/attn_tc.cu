// Tree-masked attention on the tcgen05 tensor cores (bf16 in, fp32 accumulate).
//
// Split-KV flash-decoding.  A CTA owns one KV head g, up to two tiles of 128
// query rows of g's group (row r = node * G + j is query head g * G + j of
// tree node r / G), and one key range [kbeg, kend) of that head's prefix+tree
// keys.  All rows of the group share every K/V block, so each block is
// fetched once per CTA and multiplied against up to 256 rows.
//
// Warp roles (320 threads; every warp helps to load Q first):
//   warp 0      TMA producer: K and V blocks of 128 keys into a 2-stage ring
//   warp 1      TMEM allocator and MMA issuer (one thread)
//   warps 2-5   softmax of row tile 0, warps 6-9 of tile 1: one thread per
//               query row; a warp reaches the TMEM lanes 32 * (warp % 4) ..
//               + 31, which are its rows, so a row's maximum and sum never
//               leave its thread
//
// Tensor memory (512 columns x 128 lanes of 32 bit):
//   S_t  columns [128 t, 128 t + 128)   scores of tile t, fp32; the softmax
//        overwrites its first 64 columns with P (bf16 pairs), the A operand
//        of the PV product
//   O_t  columns [256 + D t, 256 + D t + D)   output accumulator of tile t
//
// Per key block j the MMA thread issues, for each tile t in turn,
//   PV_t(j)     O_t += P_t . V        (A from TMEM, V from shared memory)
//   QK_t(j+1)   S_t  = Q_t . K^T      (both from shared memory)
// so that while the softmax warps of one tile work, the tensor core runs the
// other tile's products (ping-pong).  MMAs issued by one thread complete in
// order, so S_t(j+1) being complete implies PV_t(j) is complete: the softmax
// may then rescale O_t in place before releasing P_t(j+1).
//
// A CTA with a single row tile (G * N <= 128 rows per KV head) uses the
// second tile's score columns as a second score buffer instead: QK^T(j + 2)
// is issued right after PV(j), so the tensor core computes the next block's
// scores while the softmax works on the current one, and a rescale of O
// waits for the previous PV on its own barrier.
//
// Online softmax with a lazily moved maximum: the running maximum m used for
// exponentiation is only raised when a block's maximum exceeds it by more
// than 2^8 in probability, which bounds every P value by 256 and keeps the
// result exact up to rounding while O is rarely rescaled.
//
// Masking: keys below the prefix length are visible to every row; tree key
// P + t is visible to the rows of node i iff t is i or an ancestor of i (the
// row's ancestor bitmask, built in the prologue from the parent array);
// keys at or past kend (the split end, or P + N) are hidden.  Hidden scores
// become -inf before the row maximum, so hidden K/V contents cannot change a
// single output bit.  The K/V tensor maps end at row P + N, so TMA zero-fills
// any part of a block past the tree.
//
// Every wait is bounded (about two seconds); on expiry the kernel records
// TV_ERR_TIMEOUT and the other roles stop at their next wait.  Before the CTA
// frees its tensor memory and exits, the producer waits for the copies it
// requested and the MMA thread for the MMAs it issued, so nothing it started
// is still writing its shared or tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace tv {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  // looked up once; the initialisation of a function-local static is
  // thread-safe
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

namespace {

constexpr int kBM = 128;         // rows per tile (TMEM lanes)
constexpr int kBN = 128;         // keys per block
constexpr int kTiles = 2;        // row tiles per CTA
constexpr int kStages = 2;       // K/V ring depth
static_assert(kStages == 2, "single-tile CTAs read K slot b's release from score buffer b");
constexpr int kThreads = 320;
constexpr int kSoftmaxWarp0 = 2;
constexpr int kWarpsPerTile = 4;  // softmax warps of one row tile
constexpr int kPageRows = 64;     // rows of one paged K/V box (half a key block)
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr long long kWaitCycles = 4000000000LL;
constexpr uint32_t kSleepHintNs = 20000;  // longest single hardware sleep of a wait

struct TcParams {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  float* ws;  // lse [splits][rows], then bf16 partials (see internal.h)
  const int32_t* parent;
  int32_t* dev_status;
  int32_t n, hq, hkv, prefix, keys, keys_per_split, splits, rows_per_head;
  int32_t q_tma;  // 1: Q tiles arrive by TMA (G divides 128), 0: threads gather them
  int32_t signal_combine;  // 1: a combine launched early follows this kernel
  int32_t tiles_per_cta;  // 128-row tiles of one row group (1 or 2)
  float scale_log2;
  // paged K/V (null: one contiguous cache per KV head): logical key row r
  // is row r % page_size of page page_table[r / page_size] of the pool
  const int32_t* page_table;
  int32_t page_size, num_pages;
};

// Kernel argument: up to MAXB requests, each with its tensor maps (K, V, Q,
// output) and parameters.  With MAXB == 1 the grid is (splits, row groups,
// KV heads); with several requests the grid is one-dimensional and cta[]
// names each CTA's (request, KV head, row group, split).
constexpr int kMaxBatchCtas = 2048;

__host__ __device__ constexpr uint32_t pack_cta(int b, int g, int rg, int split) {
  return ((uint32_t)b << 28) | ((uint32_t)g << 20) | ((uint32_t)rg << 12) | (uint32_t)split;
}

template <int MAXB>
struct TcBatch {
  CUtensorMap kmap[MAXB], vmap[MAXB], qmap[MAXB], omap[MAXB];
  TcParams req[MAXB];
  uint32_t cta[MAXB == 1 ? 1 : kMaxBatchCtas];
};

template <int D, bool PAGED>
struct Layout {
  static constexpr uint32_t kQTile = kBM * D * 2;   // bytes of one Q tile
  static constexpr uint32_t kKV = kBN * D * 2;      // bytes of one K (or V) block
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kTiles * kQTile;
  static constexpr uint32_t kV = kK + kStages * kKV;
  static constexpr uint32_t kPar = kV + kStages * kKV;
  static constexpr uint32_t kPtab = kPar + kMaxNodes * 4;   // the CTA's page-table slice
  static constexpr uint32_t kBar = kPtab + (PAGED ? kMaxPageSlots * 4 : 0);
  static constexpr uint32_t kNumBars = 3 * kTiles + 4 * kStages + kTiles + 2;
  static constexpr uint32_t kMisc = kBar + kNumBars * 8;
  static constexpr uint32_t kBytes = kMisc + 16;
  static constexpr uint32_t kAlloc = kBytes + 1024;  // slack to align the base to 1024
};

struct Bars {
  uint32_t base;
  __device__ uint32_t s_full(int t) const { return base + 8 * t; }
  __device__ uint32_t p_full(int t) const { return base + 8 * (kTiles + t); }
  __device__ uint32_t o_final(int t) const { return base + 8 * (2 * kTiles + t); }
  __device__ uint32_t k_full(int s) const { return base + 8 * (3 * kTiles + s); }
  __device__ uint32_t v_full(int s) const { return base + 8 * (3 * kTiles + kStages + s); }
  // two tiles: K slot 0 may be refilled once block 0's QK^T are done (later
  // K slots are released with the V slots)
  __device__ uint32_t k_empty(int s) const { return base + 8 * (3 * kTiles + 2 * kStages + s); }
  // V slot s may be refilled: the last PV reading it is done (with two
  // tiles, K slot s + 1 too; with one tile, also the softmax's sign that
  // PV(j) is complete)
  __device__ uint32_t v_empty(int s) const { return base + 8 * (3 * kTiles + 3 * kStages + s); }
  // every softmax thread of tile t has staged its output row
  __device__ uint32_t epi(int t) const { return base + 8 * (3 * kTiles + 4 * kStages + t); }
  // the Q tiles have landed (TMA path)
  __device__ uint32_t q_full() const { return base + 8 * (4 * kTiles + 4 * kStages); }
  // after an abort: every MMA the issuing thread has started is complete
  __device__ uint32_t drain() const { return base + 8 * (4 * kTiles + 4 * kStages + 1); }
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int32_t* dev_status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait_sleep(bar, parity, kSleepHintNs)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1;
      report(dev_status, TV_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// A wait on the teardown path after an abort: for this thread's own copies
// or MMAs, which complete by themselves; bounded all the same.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int32_t* dev_status) {
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait_sleep(bar, parity, kSleepHintNs)) {
    if (clock64() - t0 > kWaitCycles) {
      report(dev_status, TV_ERR_TIMEOUT);
      return;
    }
  }
}

__device__ __forceinline__ uint32_t pick(const uint32_t (&a)[kMaskWords], int i) {
  uint32_t w = 0u;
#pragma unroll
  for (int k = 0; k < kMaskWords; ++k) w = (i == k) ? a[k] : w;
  return w;
}

// Visibility of the 32 keys [base, base + 32) to a row whose node has the
// ancestor bitmask `anc`: bit i set iff key base + i is visible.
__device__ __forceinline__ uint32_t visible32(const uint32_t (&anc)[kMaskWords], int prefix,
                                              int kend, int base) {
  const int np = prefix - base;  // prefix keys in the window
  uint32_t vis = np >= 32 ? 0xffffffffu : (np > 0 ? (1u << np) - 1u : 0u);
  const int lo = base - prefix;  // tree index of the window's first key
  if (lo > -32 && lo < 32 * kMaskWords) {
    if (lo < 0) {
      vis |= anc[0] << (-lo);
    } else {
      const int wi = lo >> 5, sh = lo & 31;
      const uint32_t a = pick(anc, wi), b = pick(anc, wi + 1);
      vis |= sh ? __funnelshift_r(a, b, sh) : a;
    }
  }
  const int ne = kend - base;  // keys before the end in the window
  if (ne <= 0) return 0u;
  if (ne < 32) vis &= (1u << ne) - 1u;
  return vis;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int D, int MAXB, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ TcBatch<MAXB> batch) {
  using L = Layout<D, PAGED>;
  int b = 0, split, g, rgroup;
  if (MAXB == 1) {
    split = blockIdx.x;
    rgroup = blockIdx.y;
    g = blockIdx.z;
  } else {
    const uint32_t e = batch.cta[blockIdx.x];
    b = (int)(e >> 28);
    g = (int)((e >> 20) & 0xffu);
    rgroup = (int)((e >> 12) & 0xffu);
    split = (int)(e & 0xfffu);
  }
  const TcParams& p = batch.req[b];
  const CUtensorMap* kmap = &batch.kmap[b];
  const CUtensorMap* vmap = &batch.vmap[b];
  const CUtensorMap* qmap = &batch.qmap[b];
  const CUtensorMap* omap = &batch.omap[b];
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.hq / p.hkv;
  const int row0 = rgroup * (p.tiles_per_cta * kBM);
  const int ntiles = min(p.tiles_per_cta, (p.rows_per_head - row0 + kBM - 1) / kBM);
  const int kbeg = split * p.keys_per_split;
  const int kend = min(p.keys, kbeg + p.keys_per_split);
  const int nb = (kend - kbeg + kBN - 1) / kBN;
  // With a single row tile the second tile's score columns are free: the
  // scores are double-buffered, so that QK^T of block j + 1 runs while the
  // softmax works on block j.
  const bool db = ntiles == 1;

  const Bars bars{base + L::kBar};
  int32_t* par = reinterpret_cast<int32_t*>(sm + L::kPar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 4);

  if (tid == 0) {
    for (int t = 0; t < kTiles; ++t) {
      ptx::mbar_init(bars.s_full(t), 1);
      ptx::mbar_init(bars.p_full(t), kWarpsPerTile);
      ptx::mbar_init(bars.o_final(t), 1);
    }
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bars.k_full(s), 1);
      ptx::mbar_init(bars.v_full(s), 1);
      ptx::mbar_init(bars.k_empty(s), 1);
      ptx::mbar_init(bars.v_empty(s), 1);
    }
    for (int t = 0; t < kTiles; ++t) {
      ptx::mbar_init(bars.epi(t), kWarpsPerTile);
    }
    ptx::mbar_init(bars.q_full(), 1);
    ptx::mbar_init(bars.drain(), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  // Paged K/V: a key block is two 64-row boxes, each from its own page.  A
  // box past the last key is moved back onto the last 64-row piece that
  // holds keys (its keys are hidden either way), so every page looked up is
  // one the table maps.  The CTA's slice of the table is staged in shared
  // memory; the first block, requested before that, reads the table itself.
  constexpr bool paged = PAGED;
  constexpr int kHalves = kBN / kPageRows;
  const int last64 = ((p.keys - 1) / kPageRows) * kPageRows;
  const int pfirst = paged ? kbeg / p.page_size : 0;
  int32_t* ptab = reinterpret_cast<int32_t*>(sm + L::kPtab);
  auto load_block = [&](const CUtensorMap* map, uint32_t dst, uint32_t bar, int j,
                        bool table_in_global) {
    if constexpr (!paged) {
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        ptx::tma_load_3d(dst + c * (kBN * 128), map, bar, c * 64, kbeg + j * kBN, g);
    } else {
      // both pages are looked up before either copy is issued, so that the
      // table reads overlap
      int page[kHalves], off[kHalves];
#pragma unroll
      for (int h = 0; h < kHalves; ++h) {
        const int row = min(kbeg + j * kBN + h * kPageRows, last64);
        const int slot = row / p.page_size;
        page[h] = table_in_global ? __ldg(p.page_table + slot) : ptab[slot - pfirst];
        off[h] = row - slot * p.page_size;
      }
#pragma unroll
      for (int h = 0; h < kHalves; ++h)
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          ptx::tma_load_4d(dst + c * (kBN * 128) + h * (kPageRows * 128), map, bar, c * 64,
                           off[h], g, page[h]);
    }
  };
  // The producer thread (tid 0) starts streaming K/V at once: the first
  // kStages blocks need no free slot and do not depend on Q.  It counts what
  // it has requested, so that after an abort it can wait for its own copies
  // to land before the CTA exits.
  int k_last = -1, v_last = -1;  // last K and V block requested
  bool q_requested = false;
  // With two tiles, K(j + 1) lands on V(j)'s barrier, armed for both copies
  // (one wait per block for the MMA thread), except K(2), which waits for
  // block 0's products and so keeps its own barrier: no armed phase may wait
  // on anything but copies already requested.
  const bool kv_pair = !db;
  auto paired_k = [&](int j) { return kv_pair && j >= 1 && j != kStages; };
  auto load_k = [&](int j) {
    const int s = j % kStages;
    if (paired_k(j)) {
      load_block(kmap, base + L::kK + s * L::kKV, bars.v_full((j - 1) % kStages), j, j == 0);
    } else {
      ptx::mbar_arrive_expect_tx(bars.k_full(s), L::kKV);
      load_block(kmap, base + L::kK + s * L::kKV, bars.k_full(s), j, j == 0);
    }
    k_last = j;
  };
  auto load_v = [&](int j) {
    const int s = j % kStages;
    const bool pair = j + 1 < nb && paired_k(j + 1);
    ptx::mbar_arrive_expect_tx(bars.v_full(s), pair ? 2 * L::kKV : L::kKV);
    load_block(vmap, base + L::kV + s * L::kKV, bars.v_full(s), j, false);
    v_last = j;
  };
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  if constexpr (!PAGED) {
    // While an earlier kernel on the stream may still run, warm L2 with the
    // boxes this CTA loads first (its Q tiles, K and V of its first block,
    // K of its second).  A prefetch returns nothing to the CTA and L2 is
    // where every write lands, so it cannot make a later load see stale
    // data; it only moves the first loads' DRAM latency off the critical
    // path.  (Warming more blocks ahead, or the whole key range, measured
    // slower: the extra requests delay the first loads.)
    if (tid == 0 && nb > 0) {
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        ptx::tma_prefetch_l2_3d(kmap, c * 64, kbeg, g);
        ptx::tma_prefetch_l2_3d(vmap, c * 64, kbeg, g);
        if (nb > 1) ptx::tma_prefetch_l2_3d(kmap, c * 64, kbeg + kBN, g);
        if (p.q_tma)
          for (int t = 0; t < ntiles; ++t)
            ptx::tma_prefetch_l2_3d(qmap, c * 64, g * G, (row0 + t * kBM) / G);
      }
    }
  }
  // Everything above reads nothing an earlier kernel may write.  The kernel
  // is launched under programmatic stream serialization, so it may start
  // while the previous kernel (the last layer's combine, say) finishes; it
  // waits for that grid here, before its first global read or write.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0 && p.q_tma) {
    // A tile's 128 rows are 128/G consecutive nodes x the G query heads of
    // KV head g: one box per 64-column chunk over Q seen as [N][Hq][d], in
    // the 128-byte-swizzled K-major layout; nodes past the tree read as zero.
    ptx::mbar_arrive_expect_tx(bars.q_full(), ntiles * L::kQTile);
    q_requested = true;
    for (int t = 0; t < ntiles; ++t)
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        ptx::tma_load_3d(base + L::kQ + t * L::kQTile + c * (kBM * 128), qmap, bars.q_full(),
                         c * 64, g * G, (row0 + t * kBM) / G);
  }
  if (tid == 0 && nb > 0) load_k(0);  // V_0 follows once K_0 has landed
  for (int i = tid; i < p.n; i += kThreads) par[i] = p.parent[i];
  if (PAGED && nb > 0) {
    // the pages of rows [kbeg, the last row a box of this CTA starts at]
    const int plast = min(kbeg + (nb - 1) * kBN + kPageRows, last64) / p.page_size;
    for (int i = tid; i <= plast - pfirst; i += kThreads) {
      const int page = p.page_table[pfirst + i];
      if (page < 0 || page >= p.num_pages) report(p.dev_status, TV_ERR_INVALID_ARG);
      ptab[i] = page;
    }
  }
  if (!p.q_tma) {
    // Q tiles into shared memory in the K-major 128-byte-swizzled layout:
    // 64-element column chunks of [128 rows][128 B], the 16-byte piece c of
    // row r stored at piece position c ^ (r % 8).  All loads of a thread are
    // issued before its stores so that their latencies overlap.
    constexpr int kPieces = D / 8;
    constexpr int kTotal = kTiles * kBM * kPieces;
    constexpr int kPer = (kTotal + kThreads - 1) / kThreads;
    uint4 v[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = tid + i * kThreads;
      v[i] = make_uint4(0u, 0u, 0u, 0u);
      if (e < kTotal) {
        const int t = e / (kBM * kPieces);
        const int rem = e - t * (kBM * kPieces);
        const int r = rem / kPieces, c = rem - r * kPieces;
        const int grow = row0 + t * kBM + r;
        if (t < ntiles && grow < p.rows_per_head &&
            guard(grow / G < p.n && g * G + (grow % G) < p.hq, p.dev_status)) {
          const int node = grow / G, j = grow - node * G;
          v[i] = __ldg(reinterpret_cast<const uint4*>(
                           p.q + ((size_t)node * p.hq + (size_t)g * G + j) * D) + c);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = tid + i * kThreads;
      if (e < kTotal) {
        const int t = e / (kBM * kPieces);
        const int rem = e - t * (kBM * kPieces);
        const int r = rem / kPieces, c = rem - r * kPieces;
        const uint32_t off = L::kQ + t * L::kQTile + (c >> 3) * (kBM * 128) + r * 128 +
                             (((c & 7) ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(sm + off) = v[i];
      }
    }
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // V_0 and block 1 are requested once K_0 has landed, so that the first
      // QK^T of every CTA is fed ahead of everything else.  After that a
      // slot is refilled once the last product reading it is done: with two
      // tiles, block j's single release frees V slot j % 2 and K slot
      // (j + 1) % 2, for V(j + 2) and K(j + 3), which land on one barrier;
      // keys run about half a block ahead of values.
      if (db) {
        // double-buffered scores: QK^T runs a block ahead of PV, so keys are
        // requested a block ahead of values (K_0, K_1, V_0, K_2, V_1, ...)
        bool ok = nb > 0 && wait_bar(bars.k_full(0), 0, abort_flag, p.dev_status);
        if (ok && nb > 1) load_k(1);
        if (ok) load_v(0);
        for (int j = 1; ok && j < nb; ++j) {
          if (j + 1 < nb) {
            const int s = (j + 1) % kStages, u = (j + 1) / kStages;
            // K slot s is free once QK^T(j - 1) is done, which completes
            // score buffer s (slot and buffer indices coincide)
            if (j + 1 >= kStages)
              ok = wait_bar(bars.s_full(s), (u - 1) & 1, abort_flag, p.dev_status);
            if (!ok) break;
            load_k(j + 1);
          }
          const int s = j % kStages, u = j / kStages;
          if (j >= kStages) ok = wait_bar(bars.v_empty(s), (u - 1) & 1, abort_flag, p.dev_status);
          if (!ok) break;
          load_v(j);
        }
      } else if (nb > 0 && wait_bar(bars.k_full(0), 0, abort_flag, p.dev_status)) {
        load_v(0);
      }
      for (int j = 1; !db && j < nb; ++j) {
        const int s = j % kStages, u = j / kStages;
        // K(2) waits for the first QK^T products; a later K(j) was released
        // together with V(j - 1), whose wait has passed
        bool ready = j != kStages ? true
                                  : wait_bar(bars.k_empty(s), (u - 1) & 1, abort_flag, p.dev_status);
        if (!ready) break;
        load_k(j);
        if (j >= kStages &&
            !wait_bar(bars.v_empty(s), (u - 1) & 1, abort_flag, p.dev_status))
          break;
        load_v(j);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescQK = ptx::idesc_bf16(kBM, kBN, false);
      constexpr uint32_t kIdescPV = ptx::idesc_bf16(kBM, D, true);
      // Descriptors are built once; a K step only moves the start address
      // (the low field, in 16-byte units), so each MMA issues in a couple of
      // instructions.
      const uint64_t q_desc = ptx::smem_desc_sw128(base + L::kQ, 16, 1024);
      const uint64_t k_desc = ptx::smem_desc_sw128(base + L::kK, 16, 1024);
      // V block, MN-major: 8-key groups 1024 B apart (SBO), the two 64-column
      // halves of d kBN * 128 B apart (LBO)
      const uint64_t v_desc = ptx::smem_desc_sw128(base + L::kV, kBN * 128, 1024);
      // S buffer b (TMEM columns [128 b, 128 b + 128)) = Q tile t . K slot s
      auto issue_qk_to = [&](int t, int b, int s) {
        const uint64_t qd = q_desc + ((t * L::kQTile) >> 4);
        const uint64_t kd = k_desc + ((s * L::kKV) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qo = ((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4;
          const uint32_t ko = ((kk >> 2) * (kBN * 128) + (kk & 3) * 32) >> 4;
          ptx::mma_ss(tmem + b * kBN, qd + qo, kd + ko, kIdescQK, kk > 0 ? 1u : 0u);
        }
      };
      // O_t (+)= P in S buffer b . V slot s
      auto issue_pv_from = [&](int b, int t, int s, bool acc) {
        const uint64_t vd = v_desc + ((s * L::kKV) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          ptx::mma_ts(tmem + 2 * kBN + t * D, tmem + b * kBN + kk * 8, vd + ((kk * 2048) >> 4),
                      kIdescPV, (acc || kk > 0) ? 1u : 0u);
      };
      auto issue_qk = [&](int t, int s) { issue_qk_to(t, t, s); };
      auto issue_pv = [&](int t, int s, bool acc) { issue_pv_from(t, t, s, acc); };
      bool ok = nb > 0 && wait_bar(bars.k_full(0), 0, abort_flag, p.dev_status);
      if (ok && p.q_tma) ok = wait_bar(bars.q_full(), 0, abort_flag, p.dev_status);
      if (db) {
        // one tile, scores in two buffers: QK^T(j + 2) is issued right after
        // PV(j) has freed buffer j % 2; MMAs from one thread run in order, so
        // PV(j) reads P before QK^T overwrites it.  Two commits per block:
        // the V slot release (also the softmax's sign that PV(j) is done) and
        // the scores of block j + 2 (also the release of K slot j % 2).
        if (ok) {
          ptx::tc_fence_after();
          issue_qk_to(0, 0, 0);
          ptx::mma_commit(bars.s_full(0));
        }
        if (ok && nb > 1) {
          ok = wait_bar(bars.k_full(1), 0, abort_flag, p.dev_status);
          if (ok) {
            ptx::tc_fence_after();
            issue_qk_to(0, 1, 1);
            ptx::mma_commit(bars.s_full(1));
          }
        }
        for (int j = 0; ok && j < nb; ++j) {
          const int b = j & 1;
          const int s = j % kStages, u = j / kStages;
          ok = wait_bar(bars.v_full(s), u & 1, abort_flag, p.dev_status);
          if (ok) ok = wait_bar(bars.p_full(b), (j >> 1) & 1, abort_flag, p.dev_status);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_pv_from(b, 0, s, j > 0);
          ptx::mma_commit(bars.v_empty(s));
          if (j + 2 < nb) {
            const int s2 = (j + 2) % kStages, u2 = (j + 2) / kStages;
            ok = wait_bar(bars.k_full(s2), u2 & 1, abort_flag, p.dev_status);
            if (!ok) break;
            ptx::tc_fence_after();
            issue_qk_to(0, b, s2);
            ptx::mma_commit(bars.s_full(b));
          }
          if (j + 1 == nb) ptx::mma_commit(bars.o_final(0));
        }
        ok = false;  // the two-tile loop below is not for this CTA
      }
      if (ok) {
        ptx::tc_fence_after();
        for (int t = 0; t < ntiles; ++t) {
          issue_qk(t, 0);
          ptx::mma_commit(bars.s_full(t));
        }
        ptx::mma_commit(bars.k_empty(0));
      }
      // The tensor pipe queues only a few MMAs and every barrier operation
      // of this thread costs tens of cycles, so none sits between a tile's
      // PV and QK^T: V of this block and K of the next (one barrier, but for
      // K(2)) are waited for at the top of the block (in this compute-bound
      // path they have landed), the products of a tile then issue back to
      // back, and one commit per block releases both slots.  (Each barrier
      // operation taken out of the product stream measured 1-2% at N >= 64.)
      for (int j = 0; ok && j < nb; ++j) {
        const int s = j % kStages, u = j / kStages;
        const bool more = j + 1 < nb;
        const int s2 = (j + 1) % kStages, u2 = (j + 1) / kStages;
        ok = wait_bar(bars.v_full(s), u & 1, abort_flag, p.dev_status);
        if (ok && more && j + 1 == kStages)  // K(2) has its own barrier
          ok = wait_bar(bars.k_full(s2), u2 & 1, abort_flag, p.dev_status);
        for (int t = 0; t < ntiles && ok; ++t) {
          ok = wait_bar(bars.p_full(t), j & 1, abort_flag, p.dev_status);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_pv(t, s, j > 0);
          if (more) {
            issue_qk(t, s2);
            ptx::mma_commit(bars.s_full(t));
          } else {
            ptx::mma_commit(bars.o_final(t));
          }
        }
        // V slot s and K slot s2 are both free once this block's products
        // are done: one release for both (the producer reads it as v_empty)
        if (ok) ptx::mma_commit(bars.v_empty(s));
      }
    }
  } else if (warp >= kSoftmaxWarp0) {
    // ------------------------------------------------------------ softmax
    // One thread per query row: warp w of tile t reaches the TMEM lanes
    // 32 (w % 4) .. + 31, so the row maximum and sum stay in the thread.
    // Each block's 128 scores are read from TMEM in one load and one wait
    // (128 registers; no spills): fewer TMEM instructions per block, which
    // measured 2-6% faster than two passes of two 64-column loads, with
    // bit-identical output.
    const int sw = warp - kSoftmaxWarp0;
    const int t = sw >> 2;
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;
    const int grow = row0 + t * kBM + r;
    if (t < ntiles) {
      const bool row_ok = grow < p.rows_per_head;
      uint32_t anc[kMaskWords];
#pragma unroll
      for (int w = 0; w < kMaskWords; ++w) anc[w] = 0u;
      if (row_ok && !ancestor_bits(par, grow / G, anc)) report(p.dev_status, TV_ERR_INVALID_TREE);
      const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
      const uint32_t t_o = tmem + lane_base + 2 * kBN + t * D;
      const float c = p.scale_log2;
      const float rescale_raw = kRescaleLog2 / c;
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < nb; ++j) {
        // the score buffer of this block and the phase of its barriers
        const int b = db ? (j & 1) : t;
        const uint32_t ph = db ? ((j >> 1) & 1) : (j & 1);
        const uint32_t t_s = tmem + lane_base + b * kBN;
        ok = wait_bar(bars.s_full(b), ph, abort_flag, p.dev_status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        ptx::tc_fence_after();
        const int kb0 = kbeg + j * kBN;
        const bool edge = kb0 + kBN > min(p.prefix, kend);
        // the block's 128 scores in one TMEM load
        uint32_t sv[kBN];
        ptx::tmem_ld128(t_s, sv);
        ptx::tmem_wait_ld(sv);
        float* sc = reinterpret_cast<float*>(sv);
        if (edge) {
#pragma unroll
          for (int q = 0; q < kBN / 32; ++q) {
            const uint32_t vis = visible32(anc, p.prefix, kend, kb0 + 32 * q);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (!((vis >> i) & 1u)) sc[q * 32 + i] = -INFINITY;
          }
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
        for (int i = 0; i < kBN; ++i) mx[i & 7] = fmaxf(mx[i & 7], sc[i]);
        const float mb = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        const float m_new = fmaxf(m_used, mb);
        const bool raise = m_new > m_used + rescale_raw;
        float alpha = 1.f;
        if (raise) {
          alpha = ptx::ex2((m_used - m_new) * c);
          m_used = m_new;
        }
        const float mc = (m_used == -INFINITY) ? 0.f : m_used * c;
        float sum0 = 0.f, sum1 = 0.f;
        // P (bf16 pairs) overwrites the first 64 columns of S, all of which
        // this thread has read
#pragma unroll
        for (int q = 0; q < kBN / 32; ++q) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a = ptx::ex2(fmaf(sc[q * 32 + 2 * i], c, -mc));
            const float b = ptx::ex2(fmaf(sc[q * 32 + 2 * i + 1], c, -mc));
            sum0 += a;
            sum1 += b;
            pk[i] = pack_bf16x2(a, b);
          }
          ptx::tmem_st16(t_s + q * 16, pk);
        }
        l = l * alpha + (sum0 + sum1);
        if (j > 0 && __any_sync(0xffffffffu, raise)) {
          // O_t must hold the sum through block j-1.  With one buffer per
          // tile, S_t(j) complete implies PV_t(j-1) complete (see above);
          // with double-buffered scores PV(j-1) may still run: wait for it
          // (its V slot's release).  PV_t(j) waits for this thread's P_full
          // arrival.
          if (db && !wait_bar(bars.v_empty((j - 1) % kStages), ((j - 1) / kStages) & 1, abort_flag,
                              p.dev_status))
            ok = false;
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          ptx::tc_fence_after();
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t v[32];
            ptx::tmem_ld32(t_o + q * 32, v);
            ptx::tmem_wait_ld(v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            ptx::tmem_st32(t_o + q * 32, v);
          }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars.p_full(b));
      }
      // epilogue: O_t is final once the last PV has completed
      if (ok) ok = wait_bar(bars.o_final(t), 0, abort_flag, p.dev_status);
      // every product of the CTA is done once its last tile's O is final:
      // the combine, launched behind this kernel under programmatic
      // serialization, may be scheduled now (it waits for this grid before
      // reading)
      if (p.signal_combine && t == ntiles - 1 && (sw & 3) == 0 && lane == 0)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
      // Stage this thread's normalised row as 16-bit values in shared memory
      // (the Q tiles are free: every MMA has completed), then copy the tile
      // out.  With one split the result is the final bf16 output; otherwise
      // it is the split's bf16 partial plus its log-sum-exp (bf16 keeps
      // float32's exponent range, so any finite V gives a finite partial).
      constexpr int kChunks = D / 8;
      const bool to_out = p.splits == 1;
      const size_t rows_all = (size_t)p.n * p.hq;
      const int R = t * kBM + r;
      if (__all_sync(0xffffffffu, ok)) {
        ptx::tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint8_t* srow = sm + L::kQ + (size_t)R * (D * 2);
        // the whole row in one TMEM load and one wait
        uint32_t v[D];
        if constexpr (D == 128) {
          ptx::tmem_ld128(t_o, v);
        } else {
          ptx::tmem_ld64(t_o, v);
        }
        ptx::tmem_wait_ld(v);
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float a = __uint_as_float(v[32 * q + 8 * cc + 2 * e]) * inv;
              const float b = __uint_as_float(v[32 * q + 8 * cc + 2 * e + 1]) * inv;
              w[e] = pack_bf16x2(a, b);
            }
            const int k = q * 4 + cc;  // 16-byte chunk of the row
            if (p.q_tma) {
              // the TMA store's layout: 64-column chunks of [128 rows][128 B],
              // 16-byte piece c of row r at piece position c ^ (r % 8)
              const uint32_t off = L::kQ + t * L::kQTile + (k >> 3) * (kBM * 128) + r * 128 +
                                   (((k & 7) ^ (r & 7)) << 4);
              *reinterpret_cast<uint4*>(sm + off) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
              // row R's chunk k at chunk position (k + R) % kChunks spreads a
              // warp's stores over all banks
              *reinterpret_cast<uint4*>(srow + ((k + R) % kChunks) * 16) =
                  make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
        if (p.q_tma) ptx::fence_proxy_async_smem();
        if (!to_out && row_ok &&
            guard(split < p.splits && (size_t)(grow / G) * p.hq + (size_t)g * G + grow % G <
                                          rows_all, p.dev_status)) {
          const int node = grow / G, jj = grow - node * G;
          const size_t prow = (size_t)node * p.hq + (size_t)g * G + jj;
          p.ws[(size_t)split * rows_all + prow] =
              l > 0.f ? m_used * c + __log2f(l) : -INFINITY;
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars.epi(t));
      if (p.q_tma) {
        // one thread of the tile writes it with tensor-map stores: a box of
        // 64 columns x G heads x 128/G nodes per chunk, nodes past the tree
        // clipped by the map
        if ((sw & 3) == 0 && lane == 0 &&
            wait_bar(bars.epi(t), 0, abort_flag, p.dev_status)) {
#pragma unroll
          for (int cc = 0; cc < D / 64; ++cc)
            ptx::tma_store_4d(omap, base + L::kQ + t * L::kQTile + cc * (kBM * 128), cc * 64,
                              g * G, (row0 + t * kBM) / G, to_out ? 0 : split);
          ptx::bulk_commit_group();
          ptx::bulk_wait_group_read0();
        }
      } else if (wait_bar(bars.epi(t), 0, abort_flag, p.dev_status)) {
        uint8_t* dst_base = to_out ? reinterpret_cast<uint8_t*>(p.out)
                                   : reinterpret_cast<uint8_t*>(p.ws) +
                                         partial_o_offset(p.splits, rows_all) +
                                         (size_t)split * rows_all * D * 2;
        const int k0 = (sw & 3) * 32 + lane;  // 0..127 within the tile
#pragma unroll 4
        for (int idx = k0; idx < kBM * kChunks; idx += kBM) {
          const int rl = idx / kChunks, ch = idx - rl * kChunks;
          const int Rr = t * kBM + rl;
          const int gr = row0 + Rr;
          if (gr < p.rows_per_head &&
              guard((size_t)(gr / G) * p.hq + (size_t)g * G + gr % G < rows_all, p.dev_status)) {
            const int node = gr / G, jj = gr - node * G;
            const size_t prow = (size_t)node * p.hq + (size_t)g * G + jj;
            const uint4 v = *reinterpret_cast<const uint4*>(sm + L::kQ + (size_t)Rr * (D * 2) +
                                                            ((ch + Rr) % kChunks) * 16);
            *reinterpret_cast<uint4*>(dst_base + prow * (D * 2) + ch * 16) = v;
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // A wait ran out and the roles stopped early.  No CTA exits with its own
    // copies or MMAs in flight: the producer waits for every K, V and Q copy
    // it requested to land in shared memory, the MMA thread for every MMA it
    // issued (one commit covers them all), and only then is TMEM freed.
    if (tid == 0) {
      for (int s = 0; s < kStages; ++s) {
        // the last block requested into slot s is the newest phase there
        // (with two tiles K(0) and K(2) use k_full(0); every other K(j)
        // completes within V(j - 1)'s phase, awaited below)
        const int jk = k_last - ((k_last - s) % kStages + kStages) % kStages;
        const int jk_own = !kv_pair ? jk : (s == 0 ? (k_last >= kStages ? kStages : 0) : -1);
        if (k_last >= 0 && jk_own >= 0)
          drain_wait(bars.k_full(s), (jk_own / kStages) & 1, p.dev_status);
        const int jv = v_last - ((v_last - s) % kStages + kStages) % kStages;
        if (v_last >= 0 && jv >= 0) drain_wait(bars.v_full(s), (jv / kStages) & 1, p.dev_status);
      }
      if (q_requested) drain_wait(bars.q_full(), 0, p.dev_status);
    }
    if (warp == 1 && lane == 0) {
      ptx::mma_commit(bars.drain());
      drain_wait(bars.drain(), 0, p.dev_status);
    }
    ptx::tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}


// 3-D map over one layer's cache [hkv][cap][d] that ends at row `rows`
// (= P + N): boxes of 64 columns x 128 rows x 1 head, 128-byte swizzle,
// rows past the end read as zero.
bool make_kv_map(CUtensorMap* map, const void* base, int d, int rows, int64_t cap, int hkv) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)hkv};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)cap * d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)kBN, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map over a page pool [pages][hkv][page_size][d] (bf16): boxes of 64
// columns x 64 rows of one page and KV head, 128-byte swizzle.
bool make_paged_kv_map(CUtensorMap* map, const void* base, int d, int page_size, int hkv,
                       int num_pages) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)page_size, (cuuint64_t)hkv,
                              (cuuint64_t)num_pages};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)page_size * d * 2,
                                 (cuuint64_t)hkv * page_size * d * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)kPageRows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over Q [n][hq][d] (bf16): boxes of 64 columns x G heads x 128/G
// nodes (one 128-row tile of a KV head's query group), 128-byte swizzle,
// nodes past the tree read as zero.
// 4-D map over an output-shaped array [layers][n][hq][d] of bf16 values
// (the split partials, or the output with one layer): boxes of 64 columns x
// G heads x 128/G nodes x 1, no swizzle change from the Q tiles.
bool make_o_map(CUtensorMap* map, void* base, int d, int n, int hq, int group, int layers) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)hq, (cuuint64_t)n, (cuuint64_t)layers};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)hq * d * 2,
                                 (cuuint64_t)n * hq * d * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)group, (cuuint32_t)(kBM / group), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base,
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_q_map(CUtensorMap* map, const void* base, int d, int n, int hq, int group) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)hq, (cuuint64_t)n};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)hq * d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)(kBM / group)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int MAXB, bool PAGED>
cudaError_t set_smem_attr() {
  static std::atomic<bool> attr_set[64];  // per device (host threads may race here)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(attn_tc_kernel<D, MAXB, PAGED>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Layout<D, PAGED>::kAlloc);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  return cudaSuccess;
}

// Launches the attention kernel with programmatic stream serialization: it
// may begin its setup before the previous kernel on the stream has finished
// (that kernel must signal griddepcontrol.launch_dependents, as the combine
// does) and waits for it with griddepcontrol.wait before touching memory.
template <typename Arg>
cudaError_t launch_early(void (*kernel)(Arg), dim3 grid, uint32_t smem, cudaStream_t s,
                         const Arg& arg) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, arg);
}

// The tensor maps and parameters of one request under its split plan.
template <int D>
bool fill_request(const AttnProblem& p, const SplitPlan& plan, float* ws, CUtensorMap* kmap,
                  CUtensorMap* vmap, CUtensorMap* qmap, CUtensorMap* omap, TcParams* tp) {
  const int rows = p.prefix + p.n;
  if (p.page_table != nullptr) {
    if (!make_paged_kv_map(kmap, p.k, D, p.page_size, p.hkv, p.num_pages) ||
        !make_paged_kv_map(vmap, p.v, D, p.page_size, p.hkv, p.num_pages))
      return false;
  } else if (!make_kv_map(kmap, p.k, D, rows, p.cap, p.hkv) ||
             !make_kv_map(vmap, p.v, D, rows, p.cap, p.hkv)) {
    return false;
  }
  const int group = p.hq / p.hkv;
  const bool q_tma = (kBM % group) == 0;
  if (q_tma && !make_q_map(qmap, p.q, D, p.n, p.hq, group)) return false;
  if (!q_tma) memset(qmap, 0, sizeof(*qmap));
  if (q_tma) {
    const bool to_out = plan.splits == 1;
    void* obase = to_out ? p.out
                         : static_cast<void*>(reinterpret_cast<uint8_t*>(ws) +
                                              partial_o_offset(plan.splits, (size_t)p.n * p.hq));
    if (!make_o_map(omap, obase, D, p.n, p.hq, group, to_out ? 1 : plan.splits))
      return false;
  } else {
    memset(omap, 0, sizeof(*omap));
  }
  *tp = TcParams{};
  tp->q = static_cast<const __nv_bfloat16*>(p.q);
  tp->out = static_cast<__nv_bfloat16*>(p.out);
  tp->ws = ws;
  tp->parent = p.parent;
  tp->dev_status = p.dev_status;
  tp->n = p.n;
  tp->hq = p.hq;
  tp->hkv = p.hkv;
  tp->prefix = p.prefix;
  tp->keys = rows;
  tp->keys_per_split = plan.keys_per_split;
  tp->signal_combine = plan.splits > 1 && combine_launches_early(p.n * p.hq) ? 1 : 0;
  tp->tiles_per_cta = plan.tiles_per_cta;
  tp->splits = plan.splits;
  tp->rows_per_head = (p.hq / p.hkv) * p.n;
  tp->scale_log2 = p.scale_log2;
  tp->q_tma = q_tma ? 1 : 0;
  tp->page_table = p.page_table;
  tp->page_size = p.page_size;
  tp->num_pages = p.num_pages;
  return true;
}

template <int D, bool PAGED>
cudaError_t launch_d(const AttnProblem& p, const SplitPlan& plan, float* ws, cudaStream_t s) {
  cudaError_t e = set_smem_attr<D, 1, PAGED>();
  if (e != cudaSuccess) return e;
  TcBatch<1> batch;
  memset(&batch, 0, sizeof(batch));
  if (!fill_request<D>(p, plan, ws, &batch.kmap[0], &batch.vmap[0], &batch.qmap[0],
                       &batch.omap[0], &batch.req[0]))
    return cudaErrorInvalidValue;
  const dim3 grid(plan.splits, plan.row_tiles, p.hkv);
  return launch_early(attn_tc_kernel<D, 1, PAGED>, grid, Layout<D, PAGED>::kAlloc, s, batch);
}

template <int D, bool PAGED>
cudaError_t launch_batched_d(const AttnProblem* probs, const SplitPlan* plans, int batch_n,
                             float* const* ws, cudaStream_t s) {
  cudaError_t e = set_smem_attr<D, kMaxBatch, PAGED>();
  if (e != cudaSuccess) return e;
  // about 13 KB: built on the heap, passed by value to the launch
  auto* batch = new TcBatch<kMaxBatch>;
  memset(batch, 0, sizeof(*batch));
  int ctas = 0;
  bool ok = batch_n <= kMaxBatch;
  for (int b = 0; ok && b < batch_n; ++b) {
    ok = (probs[b].page_table != nullptr) == PAGED;  // one launch is all paged or none
    ok = ok && fill_request<D>(probs[b], plans[b], ws[b], &batch->kmap[b], &batch->vmap[b],
                         &batch->qmap[b], &batch->omap[b], &batch->req[b]);
    for (int g = 0; ok && g < probs[b].hkv; ++g)
      for (int rg = 0; ok && rg < plans[b].row_tiles; ++rg)
        for (int sp = 0; ok && sp < plans[b].splits; ++sp) {
          ok = ctas < kMaxBatchCtas && g < 256 && rg < 256 && sp < 4096;
          if (ok) batch->cta[ctas++] = pack_cta(b, g, rg, sp);
        }
  }
  cudaError_t le = cudaSuccess;
  if (ok)
    le = launch_early(attn_tc_kernel<D, kMaxBatch, PAGED>, dim3(ctas), Layout<D, PAGED>::kAlloc, s,
                      *batch);
  delete batch;
  if (!ok) return cudaErrorInvalidValue;
  return le;
}

}  // namespace

cudaError_t launch_attn_tc(const AttnProblem& p, const SplitPlan& plan, float* ws,
                           cudaStream_t s) {
  if (p.page_table != nullptr)
    return p.d == 128 ? launch_d<128, true>(p, plan, ws, s) : launch_d<64, true>(p, plan, ws, s);
  return p.d == 128 ? launch_d<128, false>(p, plan, ws, s) : launch_d<64, false>(p, plan, ws, s);
}

cudaError_t launch_attn_tc_batched(const AttnProblem* probs, const SplitPlan* plans,
                                   int batch_n, float* const* ws, cudaStream_t s) {
  if (batch_n < 1) return cudaErrorInvalidValue;
  if (probs[0].page_table != nullptr)
    return probs[0].d == 128 ? launch_batched_d<128, true>(probs, plans, batch_n, ws, s)
                             : launch_batched_d<64, true>(probs, plans, batch_n, ws, s);
  return probs[0].d == 128 ? launch_batched_d<128, false>(probs, plans, batch_n, ws, s)
                           : launch_batched_d<64, false>(probs, plans, batch_n, ws, s);
}

}  // namespace tv
