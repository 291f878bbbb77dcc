// Launchers behind the C ABI (host side).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "treeverify.h"

namespace tv {

// Launches `kernel` with programmatic stream serialization: its CTAs may be
// scheduled once the previous kernel on the stream signals
// griddepcontrol.launch_dependents (or finishes), so the kernel must execute
// griddepcontrol.wait before it reads or writes any memory that kernel
// touches.  The launch gap of a short kernel then overlaps its predecessor.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// The driver's tensor-map encoder (null when the driver does not offer it).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();

struct AttnProblem {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  const int32_t* parent;
  int32_t* dev_status;
  int64_t cap;
  int32_t prefix;
  int32_t n;
  int32_t hq;
  int32_t hkv;
  int32_t d;
  int32_t dtype;
  float scale_log2;  // softmax scale * log2(e)
  // paged K/V (bf16 only): k and v are page pools [num_pages][hkv][page_size][d]
  // and logical key row r lives in page page_table[r / page_size]; null for
  // contiguous caches [hkv][cap][d]
  const int32_t* page_table = nullptr;
  int32_t page_size = 0;
  int32_t num_pages = 0;
};

// Most page-table entries one CTA of the tensor-core kernel stages.
constexpr int kMaxPageSlots = 1024;

// Split-KV plan: key range [0, P + N) cut into `splits` chunks of
// `keys_per_split` keys (a multiple of the kernel's key block).
struct SplitPlan {
  int32_t row_tiles;       // row groups per KV head (CTAs along the rows)
  int32_t tiles_per_cta;   // 128-row tiles per row group (tensor-core kernel: 1 or 2)
  int32_t splits;
  int32_t keys_per_split;
  size_t ws_bytes;         // partial O + row max + row sum
};

int device_sm_count();

// bf16 runs on the tcgen05 kernel, fp32 on the FMA kernel.
bool use_tensor_cores(int32_t dtype);

SplitPlan plan_attention(int32_t n, int32_t hq, int32_t hkv, int32_t d, int32_t dtype,
                         int32_t prefix, int sm_count);

// Partials inside the workspace, for R = n * hq rows (row n_i * hq + h):
//   lse [splits][R]  fp32: log2 of the split's softmax denominator, in the
//                    log2-scaled score units (-inf when the split holds no
//                    key the row may see)
//   o   [splits][R][d]  the split's normalised output: fp32 for fp32
//                    attention, bf16 for bf16 attention (float32's exponent
//                    range, so a finite V never overflows a partial); starts
//                    at byte partial_o_offset(splits, R)
__host__ __device__ inline size_t partial_o_offset(int splits, size_t rows) {
  return ((size_t)splits * rows * sizeof(float) + 255) & ~size_t(255);
}
cudaError_t launch_attn_simt(const AttnProblem& p, const SplitPlan& plan, float* ws,
                             cudaStream_t s);
cudaError_t launch_attn_tc(const AttnProblem& p, const SplitPlan& plan, float* ws,
                           cudaStream_t s);
void plan_attention_batched(int batch, const int32_t* n, const int32_t* prefix, int32_t hq,
                            int32_t hkv, int32_t d, int sm_count, SplitPlan* plans,
                            size_t* ws_offset, size_t* ws_total);

// Several requests in one launch of the tensor-core kernel (bf16): request b
// under plans[b] with its partials at ws[b].
constexpr int kMaxBatch = TV_MAX_BATCH;
cudaError_t launch_attn_tc_batched(const AttnProblem* probs, const SplitPlan* plans,
                                   int batch_n, float* const* ws, cudaStream_t s);
cudaError_t launch_combine(const AttnProblem& p, const SplitPlan& plan, const float* ws,
                           cudaStream_t s);
// Whether the combine of an attention with this many output rows (N * Hq)
// is launched under programmatic serialization right behind the kernel.
bool combine_launches_early(int rows);

cudaError_t launch_tree_mask(const int32_t* parent, int32_t n, uint32_t* words,
                             int32_t* dev_status, cudaStream_t s);

cudaError_t launch_accept(const float* logits, int32_t vocab, const int32_t* token,
                          const int32_t* parent, int32_t n, int32_t prefix, int32_t* am,
                          int32_t* m, int32_t* path, int32_t* out_tokens, int32_t* new_pos,
                          int32_t* new_parent, int32_t* n_survivors, int32_t* dev_status,
                          cudaStream_t s);

// Several requests with packed node arrays: request b owns nodes
// [node_offset[b], node_offset[b + 1]) (host array of batch + 1 entries) and
// has prefix length prefix[b] (host); m and n_survivors hold one entry per
// request and request b's out_tokens start at node_offset[b] + b.
cudaError_t launch_accept_batched(const float* logits, int32_t vocab, const int32_t* token,
                                  const int32_t* parent, int32_t batch,
                                  const int32_t* node_offset, const int32_t* prefix,
                                  int32_t* am, int32_t* m, int32_t* path, int32_t* out_tokens,
                                  int32_t* new_pos, int32_t* new_parent, int32_t* n_survivors,
                                  int32_t* dev_status, cudaStream_t s);
cudaError_t launch_walk_batched(const int32_t* token, const int32_t* parent, const int32_t* am,
                                int32_t batch, const int32_t* node_offset, int32_t vocab,
                                const int32_t* prefix, int32_t* m, int32_t* path,
                                int32_t* out_tokens, int32_t* new_pos, int32_t* new_parent,
                                int32_t* n_survivors, int32_t* dev_status, cudaStream_t s);

// Maximum-likelihood expansion: slices of each frontier logits row.
struct ExpandPlan {
  int chunks;      // slices per row
  int chunk_len;   // logits per slice (a multiple of 4)
  size_t ws_bytes; // workspace: one record per (row, slice)
};
ExpandPlan plan_expand(int32_t n_frontier, int32_t vocab, int32_t w);
cudaError_t launch_expand(const float* logits, int32_t vocab, int32_t n_frontier,
                          const int32_t* frontier, const float* cum, int32_t n_nodes, int32_t w,
                          int32_t* new_parent, int32_t* new_token, float* new_score, void* ws,
                          int32_t* dev_status, cudaStream_t s);
cudaError_t launch_draft_reroot(const int32_t* parent, const int32_t* token, const float* cum,
                                int32_t n, const int32_t* path, const int32_t* m,
                                const int32_t* out_tokens, int32_t prefix, int32_t* new_pos,
                                int32_t* new_parent, int32_t* new_token, float* new_cum,
                                int32_t* n_survivors, int32_t* dev_status, cudaStream_t s);
// The greedy walk and re-root map from per-node target tokens am (the
// argmax, or the sampled tokens).
cudaError_t launch_walk(const int32_t* token, const int32_t* parent, const int32_t* am,
                        int32_t n, int32_t vocab, int32_t prefix, int32_t* m, int32_t* path,
                        int32_t* out_tokens, int32_t* new_pos, int32_t* new_parent,
                        int32_t* n_survivors, int32_t* dev_status, cudaStream_t s);
cudaError_t launch_accept_sampled(const float* logits, int32_t vocab, const int32_t* token,
                                  const int32_t* parent, int32_t n, int32_t prefix,
                                  float temperature, uint64_t seed, uint64_t offset,
                                  int32_t* sampled, int32_t* m, int32_t* path,
                                  int32_t* out_tokens, int32_t* new_pos, int32_t* new_parent,
                                  int32_t* n_survivors, int32_t* dev_status, cudaStream_t s);
// Sampling verification over packed requests (host arrays of batch entries:
// temperature, seed, offset, prefix; node_offset of batch + 1).
cudaError_t launch_accept_sampled_batched(const float* logits, int32_t vocab,
                                          const int32_t* token, const int32_t* parent,
                                          int32_t batch, const int32_t* node_offset,
                                          const int32_t* prefix, const float* temperature,
                                          const uint64_t* seed, const uint64_t* offset,
                                          int32_t* sampled, int32_t* m, int32_t* path,
                                          int32_t* out_tokens, int32_t* new_pos,
                                          int32_t* new_parent, int32_t* n_survivors,
                                          int32_t* dev_status, cudaStream_t s);
// Contiguous caches [hkv][cap][row] per layer, or (page_table given) page
// pools [num_pages][hkv][page_size][row] per layer.
cudaError_t launch_compact(void* k, void* v, int32_t layers, int64_t layer_stride_bytes,
                           int32_t hkv, int64_t cap, int32_t row_bytes, int32_t prefix,
                           int32_t n, const int32_t* new_pos, int32_t* dev_status,
                           cudaStream_t s, const int32_t* page_table = nullptr,
                           int32_t page_size = 0, int32_t num_pages = 0);

// Several requests in one launch: request b's caches k[b], v[b] (layer l at
// l * layer_stride_bytes[b]), contiguous with cap[b] rows per head, or paged
// through page_table[b] (cap may then be null).  All arrays are host arrays.
cudaError_t launch_compact_batched(int32_t batch, void* const* k, void* const* v,
                                   const int64_t* layer_stride_bytes, const int64_t* cap,
                                   const int32_t* const* page_table, const int32_t* prefix,
                                   const int32_t* n, const int32_t* const* new_pos,
                                   int32_t layers, int32_t hkv, int32_t row_bytes,
                                   int32_t page_size, int32_t num_pages, int32_t* dev_status,
                                   cudaStream_t s);

// The target's LM head fused with the argmax (bf16 hidden states and weights).
size_t lm_head_workspace_bytes(int32_t n, int32_t vocab, int sm_count);
cudaError_t launch_lm_head_argmax(const void* hidden, const void* weight, int32_t n,
                                  int32_t d_model, int32_t vocab, int32_t* am, float* max_logit,
                                  void* ws, int32_t* dev_status, cudaStream_t s);

}  // namespace tv
