// The C ABI: argument checks on the host, then the kernel launches.
#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "treeverify.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_size(int32_t dtype) {
  switch (dtype) {
    case TV_F32: return 4;
    case TV_BF16: return 2;
    default: return 0;
  }
}

tv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? TV_OK : TV_ERR_CUDA; }

// Shapes the attention kernels implement.
tv_status check_attn_shape(int32_t n, int32_t hq, int32_t hkv, int32_t d, int32_t dtype) {
  if (n < 1 || n > TV_MAX_NODES || hq < 1 || hkv < 1) return TV_ERR_INVALID_ARG;
  if (hq % hkv != 0) return TV_ERR_INVALID_ARG;
  if (elem_size(dtype) == 0) return TV_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return TV_ERR_UNSUPPORTED;
  if ((int64_t)n * hq > (int64_t)1 << 24) return TV_ERR_UNSUPPORTED;
  return TV_OK;
}

// Page pools [num_pages][hkv][page_size][d] of bf16: pages of whole 64-row
// boxes, coordinates within int32.
tv_status check_paging(int32_t num_pages, int32_t page_size, int32_t hkv, int32_t d) {
  if (num_pages < 1 || page_size < 64 || page_size % 64 != 0) return TV_ERR_INVALID_ARG;
  if ((int64_t)num_pages * hkv * page_size * d > ((int64_t)1 << 40)) return TV_ERR_UNSUPPORTED;
  return TV_OK;
}

tv::AttnProblem attn_problem(const void* q, const void* k, const void* v, int64_t cap,
                             int32_t prefix_len, int32_t n_nodes, const int32_t* parent,
                             void* out, int32_t hq, int32_t hkv, int32_t d, int32_t dtype,
                             float scale, int32_t* dev_status) {
  tv::AttnProblem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.parent = parent;
  p.dev_status = dev_status;
  p.cap = cap;
  p.prefix = prefix_len;
  p.n = n_nodes;
  p.hq = hq;
  p.hkv = hkv;
  p.d = d;
  p.dtype = dtype;
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt((float)d);
  p.scale_log2 = sc * 1.4426950408889634f;  // log2(e)
  return p;
}

// Packed per-request node ranges of the batched acceptance: node_offset[0]
// is 0 and every request holds 1 to TV_MAX_NODES nodes.
tv_status check_packed(int32_t batch, const int32_t* node_offset, const int32_t* prefix_len) {
  if (batch < 1 || batch > TV_MAX_BATCH || !node_offset || !prefix_len) return TV_ERR_INVALID_ARG;
  if (node_offset[0] != 0) return TV_ERR_INVALID_ARG;
  for (int b = 0; b < batch; ++b) {
    const int64_t n = (int64_t)node_offset[b + 1] - node_offset[b];
    if (n < 1 || n > TV_MAX_NODES || prefix_len[b] < 0) return TV_ERR_INVALID_ARG;
    if ((int64_t)prefix_len[b] + n > INT32_MAX) return TV_ERR_INVALID_ARG;
  }
  return TV_OK;
}

// Checks shared by the batched compactions: every request's tree size,
// prefix and new_pos.
tv_status check_compact_requests(int32_t batch, const int32_t* prefix_len,
                                 const int32_t* n_nodes, const int32_t* const* new_pos) {
  if (batch < 1 || batch > TV_MAX_BATCH || !prefix_len || !n_nodes || !new_pos)
    return TV_ERR_INVALID_ARG;
  for (int b = 0; b < batch; ++b) {
    if (!new_pos[b] || prefix_len[b] < 0) return TV_ERR_INVALID_ARG;
    if (n_nodes[b] < 1 || n_nodes[b] > TV_MAX_NODES) return TV_ERR_INVALID_ARG;
    if ((int64_t)prefix_len[b] + n_nodes[b] > INT32_MAX / 2) return TV_ERR_UNSUPPORTED;
  }
  return TV_OK;
}

// The attention kernel, then the merge of its split partials.
tv_status run_attention(const tv::AttnProblem& p, const tv::SplitPlan& plan, void* workspace,
                        tv_stream_t stream) {
  auto s = reinterpret_cast<cudaStream_t>(stream);
  float* ws = static_cast<float*>(workspace);
  const bool tc = tv::use_tensor_cores(p.dtype);
  cudaError_t e = tc ? tv::launch_attn_tc(p, plan, ws, s) : tv::launch_attn_simt(p, plan, ws, s);
  if (e != cudaSuccess) return TV_ERR_CUDA;
  if (tc && plan.splits == 1) return TV_OK;  // the kernel wrote the normalised output
  return from_cuda(tv::launch_combine(p, plan, ws, s));
}

}  // namespace

extern "C" {

const char* tv_status_string(int32_t status) {
  switch (status) {
    case TV_OK: return "ok";
    case TV_ERR_INVALID_ARG: return "invalid argument";
    case TV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case TV_ERR_CAPACITY: return "capacity too small";
    case TV_ERR_CUDA: return "CUDA error";
    case TV_ERR_INVALID_TREE: return "invalid draft tree";
    case TV_ERR_TIMEOUT: return "device wait timed out";
    case TV_ERR_BOUNDS: return "device bounds check failed";
    default: return "unknown status";
  }
}

int32_t tv_version(void) { return 101; }

int32_t tv_checked_build(void) { return TV_CHECKED ? 1 : 0; }

tv_status tv_tree_mask(const int32_t* parent, int32_t n_nodes, uint32_t* mask_words,
                       int32_t* dev_status, tv_stream_t stream) {
  if (parent == nullptr || mask_words == nullptr) return TV_ERR_INVALID_ARG;
  if (n_nodes < 1 || n_nodes > TV_MAX_NODES) return TV_ERR_INVALID_ARG;
  return from_cuda(tv::launch_tree_mask(parent, n_nodes, mask_words, dev_status,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int32_t tv_attn_uses_tensor_cores(int32_t dtype) {
  if (elem_size(dtype) == 0) return -1;
  return tv::use_tensor_cores(dtype) ? 1 : 0;
}

size_t tv_attn_workspace_size(int32_t n_nodes, int32_t hq, int32_t hkv, int32_t d,
                              int32_t dtype, int32_t max_prefix) {
  if (check_attn_shape(n_nodes, hq, hkv, d, dtype) != TV_OK || max_prefix < 0) return 0;
  int sms = tv::device_sm_count();
  if (sms <= 0) sms = 256;  // no device visible: an upper bound
  return tv::plan_attention(n_nodes, hq, hkv, d, dtype, max_prefix, sms).ws_bytes;
}

tv_status tv_attn_plan(int32_t n_nodes, int32_t hq, int32_t hkv, int32_t d, int32_t dtype,
                       int32_t prefix_len, int32_t sm_count, int32_t* row_groups,
                       int32_t* splits, int32_t* keys_per_split, size_t* ws_bytes) {
  const tv_status st = check_attn_shape(n_nodes, hq, hkv, d, dtype);
  if (st != TV_OK) return st;
  if (prefix_len < 0 || sm_count < 0 || !row_groups || !splits || !keys_per_split || !ws_bytes)
    return TV_ERR_INVALID_ARG;
  const int sms = sm_count > 0 ? sm_count : tv::device_sm_count();
  if (sms <= 0) return TV_ERR_CUDA;
  const tv::SplitPlan plan = tv::plan_attention(n_nodes, hq, hkv, d, dtype, prefix_len, sms);
  *row_groups = plan.row_tiles;
  *splits = plan.splits;
  *keys_per_split = plan.keys_per_split;
  *ws_bytes = plan.ws_bytes;
  return TV_OK;
}

tv_status tv_tree_attn_verify(const void* q, const void* k_cache, const void* v_cache,
                              int64_t cap, int32_t prefix_len, int32_t n_nodes,
                              const int32_t* parent, void* out, int32_t hq, int32_t hkv,
                              int32_t d, int32_t dtype, float scale, void* workspace,
                              size_t ws_bytes, int32_t* dev_status, tv_stream_t stream) {
  tv_status st = check_attn_shape(n_nodes, hq, hkv, d, dtype);
  if (st != TV_OK) return st;
  if (!q || !k_cache || !v_cache || !parent || !out || !workspace) return TV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned16(workspace))
    return TV_ERR_INVALID_ARG;
  if (prefix_len < 0 || cap < 1 || !(scale >= 0.f) || std::isinf(scale)) return TV_ERR_INVALID_ARG;
  if ((int64_t)prefix_len + n_nodes > cap) return TV_ERR_CAPACITY;
  if ((int64_t)prefix_len + n_nodes > INT32_MAX / 2) return TV_ERR_UNSUPPORTED;
  const int sms = tv::device_sm_count();
  if (sms <= 0) return TV_ERR_CUDA;
  const tv::SplitPlan plan = tv::plan_attention(n_nodes, hq, hkv, d, dtype, prefix_len, sms);
  if (ws_bytes < plan.ws_bytes) return TV_ERR_CAPACITY;

  const tv::AttnProblem p = attn_problem(q, k_cache, v_cache, cap, prefix_len, n_nodes, parent,
                                         out, hq, hkv, d, dtype, scale, dev_status);

  return run_attention(p, plan, workspace, stream);
}

tv_status tv_tree_attn_verify_paged(const void* q, const void* k_pool, const void* v_pool,
                                    int32_t num_pages, int32_t page_size,
                                    const int32_t* page_table, int32_t prefix_len,
                                    int32_t n_nodes, const int32_t* parent, void* out, int32_t hq,
                                    int32_t hkv, int32_t d, int32_t dtype, float scale,
                                    void* workspace, size_t ws_bytes, int32_t* dev_status,
                                    tv_stream_t stream) {
  tv_status st = check_attn_shape(n_nodes, hq, hkv, d, dtype);
  if (st != TV_OK) return st;
  if (!q || !k_pool || !v_pool || !page_table || !parent || !out || !workspace)
    return TV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) ||
      !aligned16(workspace))
    return TV_ERR_INVALID_ARG;
  if (prefix_len < 0 || !(scale >= 0.f) || std::isinf(scale)) return TV_ERR_INVALID_ARG;
  st = check_paging(num_pages, page_size, hkv, d);
  if (st != TV_OK) return st;
  if (dtype != TV_BF16) return TV_ERR_UNSUPPORTED;
  if ((int64_t)prefix_len + n_nodes > INT32_MAX / 2) return TV_ERR_UNSUPPORTED;
  const int sms = tv::device_sm_count();
  if (sms <= 0) return TV_ERR_CUDA;
  const tv::SplitPlan plan = tv::plan_attention(n_nodes, hq, hkv, d, dtype, prefix_len, sms);
  if (ws_bytes < plan.ws_bytes) return TV_ERR_CAPACITY;
  if (plan.keys_per_split / page_size + 2 > tv::kMaxPageSlots) return TV_ERR_UNSUPPORTED;
  tv::AttnProblem p = attn_problem(q, k_pool, v_pool, 0, prefix_len, n_nodes, parent, out, hq, hkv,
                                   d, dtype, scale, dev_status);
  p.page_table = page_table;
  p.page_size = page_size;
  p.num_pages = num_pages;
  return run_attention(p, plan, workspace, stream);
}

size_t tv_attn_batched_workspace_size(int32_t batch, const int32_t* n_nodes, int32_t hq,
                                      int32_t hkv, int32_t d, int32_t dtype) {
  if (batch < 1 || batch > TV_MAX_BATCH || !n_nodes || dtype != TV_BF16) return 0;
  for (int b = 0; b < batch; ++b)
    if (check_attn_shape(n_nodes[b], hq, hkv, d, dtype) != TV_OK) return 0;
  int sms = tv::device_sm_count();
  if (sms <= 0) sms = 256;  // no device visible: an upper bound
  tv::SplitPlan plans[TV_MAX_BATCH];
  size_t total = 0;
  tv::plan_attention_batched(batch, n_nodes, nullptr, hq, hkv, d, sms, plans, nullptr, &total);
  return total;
}

tv_status tv_tree_attn_verify_batched(int32_t batch, const void* const* q,
                                      const void* const* k_cache, const void* const* v_cache,
                                      const int64_t* cap, const int32_t* prefix_len,
                                      const int32_t* n_nodes, const int32_t* const* parent,
                                      void* const* out, int32_t hq, int32_t hkv, int32_t d,
                                      int32_t dtype, float scale, void* workspace,
                                      size_t ws_bytes, int32_t* dev_status, tv_stream_t stream) {
  if (batch < 1 || batch > TV_MAX_BATCH) return TV_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !cap || !prefix_len || !n_nodes || !parent || !out ||
      !workspace)
    return TV_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return TV_ERR_INVALID_ARG;
  if (!(scale >= 0.f) || std::isinf(scale)) return TV_ERR_INVALID_ARG;
  for (int b = 0; b < batch; ++b) {
    const tv_status st = check_attn_shape(n_nodes[b], hq, hkv, d, dtype);
    if (st != TV_OK) return st;
    if (!q[b] || !k_cache[b] || !v_cache[b] || !parent[b] || !out[b]) return TV_ERR_INVALID_ARG;
    if (!aligned16(q[b]) || !aligned16(k_cache[b]) || !aligned16(v_cache[b]) ||
        !aligned16(out[b]))
      return TV_ERR_INVALID_ARG;
    if (prefix_len[b] < 0 || cap[b] < 1) return TV_ERR_INVALID_ARG;
    if ((int64_t)prefix_len[b] + n_nodes[b] > cap[b]) return TV_ERR_CAPACITY;
    if ((int64_t)prefix_len[b] + n_nodes[b] > INT32_MAX / 2) return TV_ERR_UNSUPPORTED;
  }
  if (dtype != TV_BF16) return TV_ERR_UNSUPPORTED;
  const int sms = tv::device_sm_count();
  if (sms <= 0) return TV_ERR_CUDA;
  tv::SplitPlan plans[TV_MAX_BATCH];
  size_t offs[TV_MAX_BATCH], total = 0;
  tv::plan_attention_batched(batch, n_nodes, prefix_len, hq, hkv, d, sms, plans, offs, &total);
  if (ws_bytes < total) return TV_ERR_CAPACITY;
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt((float)d);
  tv::AttnProblem probs[TV_MAX_BATCH];
  float* ws[TV_MAX_BATCH];
  for (int b = 0; b < batch; ++b) {
    tv::AttnProblem& p = probs[b];
    p = tv::AttnProblem{};
    p.q = q[b];
    p.k = k_cache[b];
    p.v = v_cache[b];
    p.out = out[b];
    p.parent = parent[b];
    p.dev_status = dev_status;
    p.cap = cap[b];
    p.prefix = prefix_len[b];
    p.n = n_nodes[b];
    p.hq = hq;
    p.hkv = hkv;
    p.d = d;
    p.dtype = dtype;
    p.scale_log2 = sc * 1.4426950408889634f;  // log2(e)
    ws[b] = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + offs[b]);
  }
  auto s = reinterpret_cast<cudaStream_t>(stream);
  if (tv::launch_attn_tc_batched(probs, plans, batch, ws, s) != cudaSuccess) return TV_ERR_CUDA;
  for (int b = 0; b < batch; ++b)
    if (plans[b].splits > 1) {
      const tv_status st = from_cuda(tv::launch_combine(probs[b], plans[b], ws[b], s));
      if (st != TV_OK) return st;
    }
  return TV_OK;
}

tv_status tv_tree_attn_verify_batched_paged(
    int32_t batch, const void* const* q, const void* k_pool, const void* v_pool,
    int32_t num_pages, int32_t page_size, const int32_t* const* page_table,
    const int32_t* prefix_len, const int32_t* n_nodes, const int32_t* const* parent,
    void* const* out, int32_t hq, int32_t hkv, int32_t d, int32_t dtype, float scale,
    void* workspace, size_t ws_bytes, int32_t* dev_status, tv_stream_t stream) {
  if (batch < 1 || batch > TV_MAX_BATCH) return TV_ERR_INVALID_ARG;
  if (!q || !k_pool || !v_pool || !page_table || !prefix_len || !n_nodes || !parent || !out ||
      !workspace)
    return TV_ERR_INVALID_ARG;
  if (!aligned16(workspace) || !aligned16(k_pool) || !aligned16(v_pool)) return TV_ERR_INVALID_ARG;
  if (!(scale >= 0.f) || std::isinf(scale)) return TV_ERR_INVALID_ARG;
  tv_status st = check_paging(num_pages, page_size, hkv, d);
  if (st != TV_OK) return st;
  for (int b = 0; b < batch; ++b) {
    st = check_attn_shape(n_nodes[b], hq, hkv, d, dtype);
    if (st != TV_OK) return st;
    if (!q[b] || !page_table[b] || !parent[b] || !out[b]) return TV_ERR_INVALID_ARG;
    if (!aligned16(q[b]) || !aligned16(out[b])) return TV_ERR_INVALID_ARG;
    if (prefix_len[b] < 0) return TV_ERR_INVALID_ARG;
    if ((int64_t)prefix_len[b] + n_nodes[b] > INT32_MAX / 2) return TV_ERR_UNSUPPORTED;
  }
  if (dtype != TV_BF16) return TV_ERR_UNSUPPORTED;
  const int sms = tv::device_sm_count();
  if (sms <= 0) return TV_ERR_CUDA;
  tv::SplitPlan plans[TV_MAX_BATCH];
  size_t offs[TV_MAX_BATCH], total = 0;
  tv::plan_attention_batched(batch, n_nodes, prefix_len, hq, hkv, d, sms, plans, offs, &total);
  if (ws_bytes < total) return TV_ERR_CAPACITY;
  tv::AttnProblem probs[TV_MAX_BATCH];
  float* ws[TV_MAX_BATCH];
  for (int b = 0; b < batch; ++b) {
    if (plans[b].keys_per_split / page_size + 2 > tv::kMaxPageSlots) return TV_ERR_UNSUPPORTED;
    probs[b] = attn_problem(q[b], k_pool, v_pool, 0, prefix_len[b], n_nodes[b], parent[b], out[b],
                            hq, hkv, d, dtype, scale, dev_status);
    probs[b].page_table = page_table[b];
    probs[b].page_size = page_size;
    probs[b].num_pages = num_pages;
    ws[b] = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + offs[b]);
  }
  auto s = reinterpret_cast<cudaStream_t>(stream);
  if (tv::launch_attn_tc_batched(probs, plans, batch, ws, s) != cudaSuccess) return TV_ERR_CUDA;
  for (int b = 0; b < batch; ++b)
    if (plans[b].splits > 1) {
      st = from_cuda(tv::launch_combine(probs[b], plans[b], ws[b], s));
      if (st != TV_OK) return st;
    }
  return TV_OK;
}

tv_status tv_kv_compact_paged(void* k_pool, void* v_pool, int32_t n_layers,
                              int64_t layer_stride_elems, int32_t num_pages, int32_t hkv,
                              int32_t page_size, int32_t d, int32_t dtype,
                              const int32_t* page_table, int32_t prefix_len, int32_t n_nodes,
                              const int32_t* new_pos, int32_t* dev_status, tv_stream_t stream) {
  const int es = elem_size(dtype);
  if (!k_pool || !v_pool || !page_table || !new_pos || es == 0) return TV_ERR_INVALID_ARG;
  if (n_layers < 1 || hkv < 1 || d < 1 || prefix_len < 0) return TV_ERR_INVALID_ARG;
  if (num_pages < 1 || page_size < 1) return TV_ERR_INVALID_ARG;
  if (n_nodes < 1 || n_nodes > TV_MAX_NODES) return TV_ERR_INVALID_ARG;
  const int64_t row_bytes = (int64_t)d * es;
  if (row_bytes % 16 != 0 || row_bytes > 512) return TV_ERR_UNSUPPORTED;
  if (!aligned16(k_pool) || !aligned16(v_pool)) return TV_ERR_INVALID_ARG;
  if (layer_stride_elems < (int64_t)num_pages * hkv * page_size * d) return TV_ERR_INVALID_ARG;
  if ((int64_t)n_layers * hkv * 2 > INT32_MAX) return TV_ERR_UNSUPPORTED;
  if ((int64_t)prefix_len + n_nodes > INT32_MAX / 2) return TV_ERR_UNSUPPORTED;
  return from_cuda(tv::launch_compact(k_pool, v_pool, n_layers, layer_stride_elems * es, hkv,
                                      page_size, (int32_t)row_bytes, prefix_len, n_nodes, new_pos,
                                      dev_status, reinterpret_cast<cudaStream_t>(stream),
                                      page_table, page_size, num_pages));
}

tv_status tv_tree_accept(const float* logits, int32_t vocab, const int32_t* token,
                         const int32_t* parent, int32_t n_nodes, int32_t prefix_len,
                         int32_t* am, int32_t* m, int32_t* path, int32_t* out_tokens,
                         int32_t* new_pos, int32_t* new_parent, int32_t* n_survivors,
                         int32_t* dev_status, tv_stream_t stream) {
  if (!logits || !token || !parent || !am || !m || !path || !out_tokens || !new_pos ||
      !new_parent || !n_survivors)
    return TV_ERR_INVALID_ARG;
  if (vocab < 1 || n_nodes < 1 || n_nodes > TV_MAX_NODES || prefix_len < 0)
    return TV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) != 0) return TV_ERR_INVALID_ARG;
  if ((int64_t)prefix_len + n_nodes > INT32_MAX) return TV_ERR_INVALID_ARG;
  return from_cuda(tv::launch_accept(logits, vocab, token, parent, n_nodes, prefix_len, am, m,
                                     path, out_tokens, new_pos, new_parent, n_survivors,
                                     dev_status, reinterpret_cast<cudaStream_t>(stream)));
}

tv_status tv_tree_accept_batched(int32_t batch, const int32_t* node_offset,
                                 const int32_t* prefix_len, const float* logits, int32_t vocab,
                                 const int32_t* token, const int32_t* parent, int32_t* am,
                                 int32_t* m, int32_t* path, int32_t* out_tokens,
                                 int32_t* new_pos, int32_t* new_parent, int32_t* n_survivors,
                                 int32_t* dev_status, tv_stream_t stream) {
  if (!logits || !token || !parent || !am || !m || !path || !out_tokens || !new_pos ||
      !new_parent || !n_survivors || vocab < 1)
    return TV_ERR_INVALID_ARG;
  const tv_status st = check_packed(batch, node_offset, prefix_len);
  if (st != TV_OK) return st;
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) != 0) return TV_ERR_INVALID_ARG;
  return from_cuda(tv::launch_accept_batched(logits, vocab, token, parent, batch, node_offset,
                                             prefix_len, am, m, path, out_tokens, new_pos,
                                             new_parent, n_survivors, dev_status,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

tv_status tv_tree_accept_tokens_batched(int32_t batch, const int32_t* node_offset,
                                        const int32_t* prefix_len, const int32_t* target_token,
                                        int32_t vocab, const int32_t* token,
                                        const int32_t* parent, int32_t* m, int32_t* path,
                                        int32_t* out_tokens, int32_t* new_pos,
                                        int32_t* new_parent, int32_t* n_survivors,
                                        int32_t* dev_status, tv_stream_t stream) {
  if (!target_token || !token || !parent || !m || !path || !out_tokens || !new_pos ||
      !new_parent || !n_survivors || vocab < 1)
    return TV_ERR_INVALID_ARG;
  const tv_status st = check_packed(batch, node_offset, prefix_len);
  if (st != TV_OK) return st;
  return from_cuda(tv::launch_walk_batched(token, parent, target_token, batch, node_offset,
                                           vocab, prefix_len, m, path, out_tokens, new_pos,
                                           new_parent, n_survivors, dev_status,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

tv_status tv_tree_accept_sampled_batched(int32_t batch, const int32_t* node_offset,
                                         const int32_t* prefix_len, const float* logits,
                                         int32_t vocab, const int32_t* token,
                                         const int32_t* parent, const float* temperature,
                                         const uint64_t* seed, const uint64_t* offset,
                                         int32_t* sampled, int32_t* m, int32_t* path,
                                         int32_t* out_tokens, int32_t* new_pos,
                                         int32_t* new_parent, int32_t* n_survivors,
                                         int32_t* dev_status, tv_stream_t stream) {
  if (!logits || !token || !parent || !temperature || !seed || !offset || !sampled || !m ||
      !path || !out_tokens || !new_pos || !new_parent || !n_survivors || vocab < 1)
    return TV_ERR_INVALID_ARG;
  const tv_status st = check_packed(batch, node_offset, prefix_len);
  if (st != TV_OK) return st;
  for (int b = 0; b < batch; ++b)
    if (!(temperature[b] > 0.f) || std::isinf(temperature[b])) return TV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) != 0) return TV_ERR_INVALID_ARG;
  return from_cuda(tv::launch_accept_sampled_batched(
      logits, vocab, token, parent, batch, node_offset, prefix_len, temperature, seed, offset,
      sampled, m, path, out_tokens, new_pos, new_parent, n_survivors, dev_status,
      reinterpret_cast<cudaStream_t>(stream)));
}

tv_status tv_kv_compact_batched(int32_t batch, void* const* k_cache, void* const* v_cache,
                                const int64_t* layer_stride_elems, const int64_t* cap,
                                const int32_t* prefix_len, const int32_t* n_nodes,
                                const int32_t* const* new_pos, int32_t n_layers, int32_t hkv,
                                int32_t d, int32_t dtype, int32_t* dev_status,
                                tv_stream_t stream) {
  const int es = elem_size(dtype);
  if (!k_cache || !v_cache || !layer_stride_elems || !cap || es == 0) return TV_ERR_INVALID_ARG;
  if (n_layers < 1 || hkv < 1 || d < 1) return TV_ERR_INVALID_ARG;
  tv_status st = check_compact_requests(batch, prefix_len, n_nodes, new_pos);
  if (st != TV_OK) return st;
  const int64_t row_bytes = (int64_t)d * es;
  if (row_bytes % 16 != 0 || row_bytes > 512) return TV_ERR_UNSUPPORTED;
  if ((int64_t)n_layers * hkv * 2 > INT32_MAX) return TV_ERR_UNSUPPORTED;
  int64_t stride_bytes[TV_MAX_BATCH];
  for (int b = 0; b < batch; ++b) {
    if (!k_cache[b] || !v_cache[b] || !aligned16(k_cache[b]) || !aligned16(v_cache[b]))
      return TV_ERR_INVALID_ARG;
    if (cap[b] < 1) return TV_ERR_INVALID_ARG;
    if ((int64_t)prefix_len[b] + n_nodes[b] > cap[b]) return TV_ERR_CAPACITY;
    if (layer_stride_elems[b] < (int64_t)hkv * cap[b] * d) return TV_ERR_INVALID_ARG;
    stride_bytes[b] = layer_stride_elems[b] * es;
  }
  return from_cuda(tv::launch_compact_batched(batch, k_cache, v_cache, stride_bytes, cap,
                                              nullptr, prefix_len, n_nodes, new_pos, n_layers,
                                              hkv, (int32_t)row_bytes, 0, 0, dev_status,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

tv_status tv_kv_compact_batched_paged(int32_t batch, void* k_pool, void* v_pool,
                                      int32_t n_layers, int64_t layer_stride_elems,
                                      int32_t num_pages, int32_t hkv, int32_t page_size,
                                      int32_t d, int32_t dtype, const int32_t* const* page_table,
                                      const int32_t* prefix_len, const int32_t* n_nodes,
                                      const int32_t* const* new_pos, int32_t* dev_status,
                                      tv_stream_t stream) {
  const int es = elem_size(dtype);
  if (!k_pool || !v_pool || !page_table || es == 0) return TV_ERR_INVALID_ARG;
  if (n_layers < 1 || hkv < 1 || d < 1 || num_pages < 1 || page_size < 1)
    return TV_ERR_INVALID_ARG;
  tv_status st = check_compact_requests(batch, prefix_len, n_nodes, new_pos);
  if (st != TV_OK) return st;
  const int64_t row_bytes = (int64_t)d * es;
  if (row_bytes % 16 != 0 || row_bytes > 512) return TV_ERR_UNSUPPORTED;
  if (!aligned16(k_pool) || !aligned16(v_pool)) return TV_ERR_INVALID_ARG;
  if (layer_stride_elems < (int64_t)num_pages * hkv * page_size * d) return TV_ERR_INVALID_ARG;
  if ((int64_t)n_layers * hkv * 2 > INT32_MAX) return TV_ERR_UNSUPPORTED;
  void* ks[TV_MAX_BATCH];
  void* vs[TV_MAX_BATCH];
  int64_t stride_bytes[TV_MAX_BATCH];
  for (int b = 0; b < batch; ++b) {
    if (!page_table[b]) return TV_ERR_INVALID_ARG;
    ks[b] = k_pool;
    vs[b] = v_pool;
    stride_bytes[b] = layer_stride_elems * es;
  }
  return from_cuda(tv::launch_compact_batched(batch, ks, vs, stride_bytes, nullptr, page_table,
                                              prefix_len, n_nodes, new_pos, n_layers, hkv,
                                              (int32_t)row_bytes, page_size, num_pages,
                                              dev_status, reinterpret_cast<cudaStream_t>(stream)));
}

tv_status tv_tree_accept_tokens(const int32_t* target_token, int32_t vocab, const int32_t* token,
                                const int32_t* parent, int32_t n_nodes, int32_t prefix_len,
                                int32_t* m, int32_t* path, int32_t* out_tokens, int32_t* new_pos,
                                int32_t* new_parent, int32_t* n_survivors, int32_t* dev_status,
                                tv_stream_t stream) {
  if (!target_token || !token || !parent || !m || !path || !out_tokens || !new_pos ||
      !new_parent || !n_survivors)
    return TV_ERR_INVALID_ARG;
  if (vocab < 1 || n_nodes < 1 || n_nodes > TV_MAX_NODES || prefix_len < 0)
    return TV_ERR_INVALID_ARG;
  if ((int64_t)prefix_len + n_nodes > INT32_MAX) return TV_ERR_INVALID_ARG;
  return from_cuda(tv::launch_walk(token, parent, target_token, n_nodes, vocab, prefix_len, m,
                                   path, out_tokens, new_pos, new_parent, n_survivors,
                                   dev_status, reinterpret_cast<cudaStream_t>(stream)));
}

tv_status tv_tree_accept_sampled(const float* logits, int32_t vocab, const int32_t* token,
                                 const int32_t* parent, int32_t n_nodes, int32_t prefix_len,
                                 float temperature, uint64_t seed, uint64_t offset,
                                 int32_t* sampled, int32_t* m, int32_t* path, int32_t* out_tokens,
                                 int32_t* new_pos, int32_t* new_parent, int32_t* n_survivors,
                                 int32_t* dev_status, tv_stream_t stream) {
  if (!logits || !token || !parent || !sampled || !m || !path || !out_tokens || !new_pos ||
      !new_parent || !n_survivors)
    return TV_ERR_INVALID_ARG;
  if (vocab < 1 || n_nodes < 1 || n_nodes > TV_MAX_NODES || prefix_len < 0)
    return TV_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || std::isinf(temperature)) return TV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) != 0) return TV_ERR_INVALID_ARG;
  if ((int64_t)prefix_len + n_nodes > INT32_MAX) return TV_ERR_INVALID_ARG;
  return from_cuda(tv::launch_accept_sampled(logits, vocab, token, parent, n_nodes, prefix_len,
                                             temperature, seed, offset, sampled, m, path,
                                             out_tokens, new_pos, new_parent, n_survivors,
                                             dev_status, reinterpret_cast<cudaStream_t>(stream)));
}

tv_status tv_kv_compact(void* k_cache, void* v_cache, int32_t n_layers,
                        int64_t layer_stride_elems, int32_t hkv, int64_t cap, int32_t d,
                        int32_t dtype, int32_t prefix_len, int32_t n_nodes,
                        const int32_t* new_pos, int32_t* dev_status, tv_stream_t stream) {
  const int es = elem_size(dtype);
  if (!k_cache || !v_cache || !new_pos || es == 0) return TV_ERR_INVALID_ARG;
  if (n_layers < 1 || hkv < 1 || cap < 1 || d < 1 || prefix_len < 0) return TV_ERR_INVALID_ARG;
  if (n_nodes < 1 || n_nodes > TV_MAX_NODES) return TV_ERR_INVALID_ARG;
  const int64_t row_bytes = (int64_t)d * es;
  if (row_bytes % 16 != 0 || row_bytes > 512) return TV_ERR_UNSUPPORTED;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return TV_ERR_INVALID_ARG;
  if ((int64_t)prefix_len + n_nodes > cap) return TV_ERR_CAPACITY;
  if (layer_stride_elems < (int64_t)hkv * cap * d) return TV_ERR_INVALID_ARG;
  if ((int64_t)n_layers * hkv * 2 > INT32_MAX) return TV_ERR_UNSUPPORTED;
  return from_cuda(tv::launch_compact(k_cache, v_cache, n_layers, layer_stride_elems * es, hkv,
                                      cap, (int32_t)row_bytes, prefix_len, n_nodes, new_pos,
                                      dev_status, reinterpret_cast<cudaStream_t>(stream)));
}

static bool expand_args_ok(int32_t n_frontier, int32_t vocab, int32_t w) {
  if (vocab < 1 || vocab > TV_MAX_VOCAB) return false;
  if (n_frontier < 1 || n_frontier > TV_MAX_NODES) return false;
  if (w < 1 || w > TV_MAX_EXPAND_WIDTH) return false;
  if ((int64_t)n_frontier * w > TV_MAX_EXPAND_CANDIDATES) return false;
  if ((int64_t)((vocab + 8191) / 8192) * w > TV_MAX_EXPAND_CANDIDATES) return false;
  return (int64_t)w <= (int64_t)n_frontier * vocab;
}

size_t tv_expand_workspace_size(int32_t n_frontier, int32_t vocab, int32_t w) {
  if (!expand_args_ok(n_frontier, vocab, w)) return 0;
  return tv::plan_expand(n_frontier, vocab, w).ws_bytes;
}

tv_status tv_tree_expand(const float* logits, int32_t vocab, int32_t n_frontier,
                         const int32_t* frontier, const float* cum, int32_t n_nodes, int32_t w,
                         int32_t* new_parent, int32_t* new_token, float* new_score,
                         void* workspace, size_t ws_bytes, int32_t* dev_status,
                         tv_stream_t stream) {
  if (!logits || !frontier || !cum || !new_parent || !new_token || !new_score || !workspace)
    return TV_ERR_INVALID_ARG;
  if (!expand_args_ok(n_frontier, vocab, w) || n_nodes < 1) return TV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(workspace) & 3u) != 0)
    return TV_ERR_INVALID_ARG;
  if (ws_bytes < tv::plan_expand(n_frontier, vocab, w).ws_bytes) return TV_ERR_CAPACITY;
  return from_cuda(tv::launch_expand(logits, vocab, n_frontier, frontier, cum, n_nodes, w,
                                     new_parent, new_token, new_score, workspace, dev_status,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

tv_status tv_draft_reroot(const int32_t* parent, const int32_t* token, const float* cum,
                          int32_t n_nodes, const int32_t* path, const int32_t* m,
                          const int32_t* out_tokens, int32_t prefix_len, int32_t* new_pos,
                          int32_t* new_parent, int32_t* new_token, float* new_cum,
                          int32_t* n_survivors, int32_t* dev_status, tv_stream_t stream) {
  if (!parent || !token || !cum || !path || !m || !out_tokens || !new_pos || !new_parent ||
      !new_token || !new_cum || !n_survivors)
    return TV_ERR_INVALID_ARG;
  if (n_nodes < 1 || n_nodes > TV_MAX_NODES || prefix_len < 0) return TV_ERR_INVALID_ARG;
  if ((int64_t)prefix_len + n_nodes > INT32_MAX) return TV_ERR_INVALID_ARG;
  return from_cuda(tv::launch_draft_reroot(parent, token, cum, n_nodes, path, m, out_tokens,
                                           prefix_len, new_pos, new_parent, new_token, new_cum,
                                           n_survivors, dev_status,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

size_t tv_lm_head_workspace_size(int32_t n_nodes, int32_t vocab) {
  if (n_nodes < 1 || n_nodes > TV_MAX_LM_NODES || vocab < 1) return 0;
  return tv::lm_head_workspace_bytes(n_nodes, vocab, tv::device_sm_count());
}

tv_status tv_lm_head_argmax(const void* hidden, const void* weight, int32_t n_nodes,
                            int32_t d_model, int32_t vocab, int32_t* am, float* max_logit,
                            void* workspace, size_t ws_bytes, int32_t* dev_status,
                            tv_stream_t stream) {
  if (!hidden || !weight || !am || !workspace) return TV_ERR_INVALID_ARG;
  if (n_nodes < 1 || n_nodes > TV_MAX_LM_NODES || vocab < 1) return TV_ERR_INVALID_ARG;
  if (d_model < 8 || d_model % 8 != 0) return TV_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(weight) || !aligned16(workspace)) return TV_ERR_INVALID_ARG;
  if (ws_bytes < tv::lm_head_workspace_bytes(n_nodes, vocab, tv::device_sm_count()))
    return TV_ERR_CAPACITY;
  return from_cuda(tv::launch_lm_head_argmax(hidden, weight, n_nodes, d_model, vocab, am,
                                             max_logit, workspace, dev_status,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
