/*
 * treeverify.h -- C ABI of the tree-masked speculative verification library.
 *
 * The library implements, on one NVIDIA GB300 (sm_103a) GPU, the target-side
 * verification step of tree-based speculative decoding as the SwiftSpec
 * review page (pith.science, paper 2506.11309) describes it:
 *
 *   - "What carries the argument": the KV cache holds the verified tokens
 *     contiguously as a prefix, with the draft-tree tokens right after it; the
 *     target checks the tree with a mask attention kernel; after verification
 *     the tree re-roots at the last verified token and the cache is
 *     reorganised so that only the still-useful subtree stays.
 *   - "Core claim": verified tokens are moved into the prefix and the
 *     surviving tree states are laid out contiguously after it.
 *   - "Referee Report", major comment 3: the paper does not describe the
 *     target-side cache management; this library's reading of it (greedy
 *     acceptance from the target's argmax, survivors = strict descendants of
 *     the last accepted node) is stated with each call below.
 *
 * Conventions shared by every call:
 *   - Every pointer named "device" is CUDA device memory owned by the caller.
 *     The library allocates nothing (the caller passes the workspace) and keeps
 *     no state between calls other than per-device caches (the SM count, the
 *     kernels' shared-memory limits once set, the address of the static
 *     scratch array) and the driver's tensor-map entry point; host threads
 *     may call it concurrently.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and never synchronises the host.
 *   - Problems visible on the host are returned at once, before anything is
 *     launched: TV_ERR_INVALID_ARG (null or misaligned pointer, bad size),
 *     TV_ERR_UNSUPPORTED (a shape the kernels do not implement),
 *     TV_ERR_CAPACITY (the cache cannot hold prefix + tree, or the workspace is
 *     too small).  A failed launch returns TV_ERR_CUDA.
 *   - Problems only visible on the device (an invalid parent array, a token id
 *     outside the vocabulary, a bad new_pos entry) never trap: the kernel
 *     stores the code into *dev_status if *dev_status is still 0 (the first
 *     error wins; the caller clears it), skips the offending work and leaves
 *     the outputs unspecified.  dev_status may be NULL.
 *   - A draft tree is given by parent[N] (device int32) in node order: node 0
 *     is a root, and for every i, -1 <= parent[i] < i (-1 marks a root; the
 *     attention accepts forests, acceptance walks from node 0).  1 <= N <= 128.
 */
#ifndef TREEVERIFY_H
#define TREEVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define TV_API __attribute__((visibility("default")))
#else
#define TV_API
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st* tv_stream_t;

typedef enum {
  TV_OK = 0,
  TV_ERR_INVALID_ARG = 1,
  TV_ERR_UNSUPPORTED = 2,
  TV_ERR_CAPACITY = 3,
  TV_ERR_CUDA = 4,
  TV_ERR_INVALID_TREE = 5,
  TV_ERR_TIMEOUT = 6,
  TV_ERR_BOUNDS = 7  /* a device bounds check failed (checked builds only) */
} tv_status;

typedef enum {
  TV_F32 = 0,  /* IEEE binary32 */
  TV_BF16 = 1  /* bfloat16 */
} tv_dtype;

#define TV_MAX_NODES 128

/* Human-readable name of a status code (static string, never NULL). */
TV_API const char* tv_status_string(int32_t status);

/* Library version as 10000*major + 100*minor + patch. */
TV_API int32_t tv_version(void);

/*
 * 1 if this library is a checked build, 0 otherwise.  A checked build
 * (compiled with -DTV_CHECKED=1) tests, in device code, the index ranges of
 * the accesses that depend on device data or on the launch arithmetic (tree
 * arrays, compaction rows, partial and output rows) before making them; a
 * failed test stores TV_ERR_BOUNDS into dev_status (when it is still 0) and
 * skips that access.  Nothing traps.  It stands in for a memory checker
 * where none can run.  Normal builds compile the tests away.
 */
TV_API int32_t tv_checked_build(void);

/*
 * tv_tree_mask -- the ancestor mask of a draft tree as per-node bitmasks.
 *
 * Passage: SwiftSpec review page, "What carries the argument" (the target's
 * mask attention over the draft tree).  Each tree node sees itself and its
 * ancestors.
 *
 *   parent      device int32 [n_nodes], tree in node order (see above)
 *   n_nodes     1..128
 *   mask_words  device uint32 [n_nodes][ceil(n_nodes/32)], written: bit
 *               (j % 32) of word j / 32 of row i is set iff node j is node i
 *               or an ancestor of node i
 *   dev_status  device int32 or NULL; TV_ERR_INVALID_TREE on a bad parent
 *
 * The attention call below builds the same mask itself; this entry point
 * exposes it for callers and tests.
 */
TV_API tv_status tv_tree_mask(const int32_t* parent, int32_t n_nodes, uint32_t* mask_words,
                       int32_t* dev_status, tv_stream_t stream);

/*
 * tv_attn_workspace_size -- bytes of device workspace tv_tree_attn_verify
 * needs for any prefix_len <= max_prefix with these shapes on the current
 * device (it reads the current device's SM count).  Returns 0 for shapes
 * the attention does not support.
 */
TV_API size_t tv_attn_workspace_size(int32_t n_nodes, int32_t hq, int32_t hkv, int32_t d,
                              int32_t dtype, int32_t max_prefix);

/*
 * tv_attn_uses_tensor_cores -- 1 if tv_tree_attn_verify runs dtype on the
 * tcgen05 tensor-core kernel, 0 if on the fp32 FMA kernel, -1 for an unknown
 * dtype.  Informative only; both give the results documented below.
 */
TV_API int32_t tv_attn_uses_tensor_cores(int32_t dtype);

/*
 * tv_attn_plan -- the split plan tv_tree_attn_verify uses for this shape on
 * a GPU with sm_count SMs (0: the current device's).  Host only: it
 * launches nothing and, given sm_count > 0, makes no CUDA call.
 *
 *   row_groups      CTAs per KV head along the query rows (each CTA holds up
 *                   to two 128-row tiles on the tensor-core path)
 *   splits          key splits; the CTAs of one layer are
 *                   hkv * row_groups * splits, and a combine launch follows
 *                   when splits > 1
 *   keys_per_split  keys of every split but the last (a multiple of the key
 *                   block), the last holding the rest of [0, P + N)
 *   ws_bytes        workspace bytes (tv_attn_workspace_size gives the same
 *                   on the current device)
 * Errors: those of tv_attn_workspace_size's shape checks, TV_ERR_INVALID_ARG
 * for a negative prefix or sm_count or a null output, TV_ERR_CUDA when
 * sm_count is 0 and no device answers.
 */
TV_API tv_status tv_attn_plan(int32_t n_nodes, int32_t hq, int32_t hkv, int32_t d, int32_t dtype,
                              int32_t prefix_len, int32_t sm_count, int32_t* row_groups,
                              int32_t* splits, int32_t* keys_per_split, size_t* ws_bytes);

/*
 * tv_tree_attn_verify -- one layer of tree-masked grouped-query attention of
 * the draft tree against the prefix KV cache plus the tree's own KV.
 *
 * Passage: SwiftSpec review page, "What carries the argument" (prefix then
 * tree tokens in the cache; mask attention kernel on the target) and
 * "Referee Report", summary (Section 3.3, masked attention).
 *
 * For tree node i and query head h, with G = hq / hkv and KV head g = h / G:
 *   out[i][h] = softmax(q[i][h] . K^T * scale) . V
 * over the cache rows [0, prefix_len) of KV head g plus the rows
 * prefix_len + j for every j that is i or an ancestor of i.
 *
 *   q          device [n_nodes][hq][d] of dtype
 *   k_cache    device [hkv][cap][d] of dtype: rows [0, prefix_len) are the
 *   v_cache    verified prefix, row prefix_len + j holds tree node j; rows at
 *              or past prefix_len + n_nodes are never read
 *   cap        rows per KV head, >= prefix_len + n_nodes
 *   prefix_len P >= 0
 *   n_nodes    N, 1..128
 *   parent     device int32 [N], see the conventions above
 *   out        device [n_nodes][hq][d] of dtype, written
 *   hq, hkv    query and KV heads, hq % hkv == 0
 *   d          head dimension: 64 or 128
 *   dtype      TV_BF16 (tensor cores, fp32 accumulation) or TV_F32 (fp32 FMA)
 *   scale      softmax scale; 0 means 1/sqrt(d)
 *   workspace  device scratch of ws_bytes >= tv_attn_workspace_size(...)
 *              bytes; its contents on entry do not matter
 *   dev_status device int32 or NULL; TV_ERR_INVALID_TREE on a bad parent
 *
 * All device pointers must be 16-byte aligned.  Rows of one KV head are
 * d elements apart and heads cap * d elements apart.
 *
 * The bf16 kernel is launched with programmatic stream serialization: it may
 * begin its setup before the previous kernel on the stream has finished (if
 * that kernel allows it, as this library's split merge does), and it waits
 * for that kernel to complete before it reads or writes any memory, so
 * stream order holds for every buffer.
 */
TV_API tv_status tv_tree_attn_verify(const void* q, const void* k_cache, const void* v_cache,
                              int64_t cap, int32_t prefix_len, int32_t n_nodes,
                              const int32_t* parent, void* out, int32_t hq, int32_t hkv,
                              int32_t d, int32_t dtype, float scale, void* workspace,
                              size_t ws_bytes, int32_t* dev_status, tv_stream_t stream);

/*
 * tv_tree_attn_verify_static -- tv_tree_attn_verify without a caller-passed
 * workspace, for callers that cannot allocate device memory: code running
 * inside a serving framework whose caching allocator owns all of the GPU's
 * memory and forbids outside allocations, plug-ins that are only handed their
 * input and output buffers, and latency-critical loops in which cudaMalloc or
 * cudaFree would synchronise the device.  The paper has no counterpart; this
 * is a convenience of this library.
 *
 * The split partials go to one scratch array of TV_STATIC_SCRATCH_BYTES
 * (16 MiB) that the library defines in device memory; every GPU that loads
 * the library holds it until the process exits.  The call allocates nothing
 * and calls no allocating routine.  Arguments, layouts and results are those
 * of tv_tree_attn_verify (minus workspace and ws_bytes).
 *
 *   - CUDA loads a library's device code and data lazily by default, so the
 *     16 MiB are reserved on a device at the first call there, not when the
 *     library is loaded.  Make that first call early: before a framework's
 *     caching allocator has taken the GPU's free memory (else the first call
 *     fails with TV_ERR_CUDA), and before any stream capture.
 *   - Every call made outside a stream capture looks the array's device
 *     address up again on the current device (a lookup, no allocation), so a
 *     device reset or a new primary context between calls is harmless.  A
 *     call made while its stream is being captured reuses the address the
 *     last uncaptured call on that device found, and fails with TV_ERR_CUDA
 *     if there was none.
 *   - A problem that needs more scratch than the array holds is rejected with
 *     TV_ERR_CAPACITY before anything is launched (tv_attn_workspace_size
 *     gives the bytes a problem needs).
 *   - Every call shares the one array and it keeps the last call's contents;
 *     nothing in it needs to start at zero, but two calls that overlap on the
 *     GPU (different streams, or different host threads) race on it.
 */
#define TV_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

TV_API tv_status tv_tree_attn_verify_static(const void* q, const void* k_cache,
                                            const void* v_cache, int64_t cap, int32_t prefix_len,
                                            int32_t n_nodes, const int32_t* parent, void* out,
                                            int32_t hq, int32_t hkv, int32_t d, int32_t dtype,
                                            float scale, int32_t* dev_status, tv_stream_t stream);

/*
 * Batched tree attention: up to TV_MAX_BATCH requests (independent
 * sequences, each with its own prefix length, tree and caches) in one launch
 * of the tensor-core kernel.  The pages verify a single request; batching is
 * the serving form of the same operation, and every request's output is
 * exactly what tv_tree_attn_verify gives for it (up to rounding: the split
 * plans differ).
 */
#define TV_MAX_BATCH 16

/* Bytes of workspace tv_tree_attn_verify_batched needs for these node counts
 * (any prefix lengths) on the current device; 0 for arguments it rejects
 * (bf16 only). */
TV_API size_t tv_attn_batched_workspace_size(int32_t batch, const int32_t* n_nodes, int32_t hq,
                                             int32_t hkv, int32_t d, int32_t dtype);

/*
 * tv_tree_attn_verify_batched -- tv_tree_attn_verify for `batch` requests at
 * once.  The per-request arguments are HOST arrays of `batch` entries:
 *   q, k_cache, v_cache, out, parent   device pointers, as tv_tree_attn_verify
 *   cap, prefix_len, n_nodes           sizes, as tv_tree_attn_verify
 * hq, hkv, d, scale and dtype are shared; dtype must be TV_BF16 (other types
 * return TV_ERR_UNSUPPORTED).  workspace: device memory of at least
 * tv_attn_batched_workspace_size bytes, 16-byte aligned, contents on entry
 * irrelevant.  Every check of tv_tree_attn_verify applies to every request
 * and is made before anything is launched.  The key splits of the requests
 * are sized in proportion to their key counts so that one launch keeps the
 * GPU busy; requests with several splits are merged by one extra launch each.
 */
TV_API tv_status tv_tree_attn_verify_batched(int32_t batch, const void* const* q,
                                             const void* const* k_cache,
                                             const void* const* v_cache, const int64_t* cap,
                                             const int32_t* prefix_len, const int32_t* n_nodes,
                                             const int32_t* const* parent, void* const* out,
                                             int32_t hq, int32_t hkv, int32_t d, int32_t dtype,
                                             float scale, void* workspace, size_t ws_bytes,
                                             int32_t* dev_status, tv_stream_t stream);

/*
 * Paged K/V caches.  A page pool holds fixed-size pages of key rows,
 * [num_pages][hkv][page_size][d] (bf16); a request's logical key row r
 * (rows [0, P) its prefix, row P + j tree node j, as in tv_tree_attn_verify)
 * is row r % page_size of page page_table[r / page_size].  Many requests
 * share one pool and each has its own table, so prefixes need no contiguous
 * room and whole pages can be shared or recycled.  Passage: the same as
 * tv_tree_attn_verify; paging is the serving form of its cache layout (the
 * review page verifies one request).
 *
 * Contract for every paged call:
 *   page_size     a multiple of 64 (a key block is two 64-row boxes)
 *   num_pages     >= 1; pools 16-byte aligned
 *   page_table    device int32 [ceil((P + N) / page_size)]: the pages of rows
 *                 [0, P + N) in order; an entry outside [0, num_pages) is
 *                 reported as TV_ERR_INVALID_ARG in dev_status (attention
 *                 then reads zeros for it; compaction skips the rows)
 *   rows of those pages past P + N must hold finite values (they are read,
 *   weighted by exactly zero, so a NaN or an infinity there would leak in)
 * The attention takes the workspace of tv_attn_workspace_size (the same
 * plan) and returns TV_ERR_UNSUPPORTED when one CTA's key range spans more
 * than 1022 pages (very long prefixes with small pages).
 */

/* tv_tree_attn_verify over a page pool (bf16 only; other arguments as for
 * tv_tree_attn_verify, less cap). */
TV_API tv_status tv_tree_attn_verify_paged(const void* q, const void* k_pool, const void* v_pool,
                                           int32_t num_pages, int32_t page_size,
                                           const int32_t* page_table, int32_t prefix_len,
                                           int32_t n_nodes, const int32_t* parent, void* out,
                                           int32_t hq, int32_t hkv, int32_t d, int32_t dtype,
                                           float scale, void* workspace, size_t ws_bytes,
                                           int32_t* dev_status, tv_stream_t stream);

/* tv_tree_attn_verify_batched over one shared page pool: page_table[b] is
 * request b's table (host array of device pointers); the workspace is that
 * of tv_attn_batched_workspace_size. */
TV_API tv_status tv_tree_attn_verify_batched_paged(
    int32_t batch, const void* const* q, const void* k_pool, const void* v_pool,
    int32_t num_pages, int32_t page_size, const int32_t* const* page_table,
    const int32_t* prefix_len, const int32_t* n_nodes, const int32_t* const* parent,
    void* const* out, int32_t hq, int32_t hkv, int32_t d, int32_t dtype, float scale,
    void* workspace, size_t ws_bytes, int32_t* dev_status, tv_stream_t stream);

/* tv_kv_compact over page pools: every layer's pool is
 * [num_pages][hkv][page_size][d] (layer l at l * layer_stride_elems); the
 * accepted path and the survivors move between logical rows, each mapped
 * through page_table (the request's table, shared by all layers).  Any
 * page_size >= 1 is accepted here.  Other arguments as for tv_kv_compact. */
TV_API tv_status tv_kv_compact_paged(void* k_pool, void* v_pool, int32_t n_layers,
                                     int64_t layer_stride_elems, int32_t num_pages, int32_t hkv,
                                     int32_t page_size, int32_t d, int32_t dtype,
                                     const int32_t* page_table, int32_t prefix_len,
                                     int32_t n_nodes, const int32_t* new_pos,
                                     int32_t* dev_status, tv_stream_t stream);

/*
 * tv_tree_accept -- greedy acceptance of the draft tree and the re-root map.
 *
 * Passage: SwiftSpec review page, "What carries the argument" (the tree
 * re-roots at the last verified token; only the still-useful subtree stays)
 * and "Core claim" (verified tokens move into the prefix, surviving tree
 * states follow contiguously).  Greedy matching and the survivor rule are
 * this library's reading of the undescribed target side ("Referee Report",
 * major comment 3).
 *
 *   logits     device float32 [n_nodes][vocab]: the target's logits at each
 *              tree node
 *   vocab      >= 1
 *   token      device int32 [n_nodes]: draft token of each node, in [0, vocab)
 *   parent     device int32 [n_nodes]: the tree (node 0 is the root)
 *   prefix_len P, the prefix length before this step
 * Outputs (device int32, written):
 *   am         [n_nodes]   am[i] = argmax_v logits[i][v]; ties go to the
 *                          lowest v, a NaN counts as the largest value
 *   m          [1]         number of accepted draft tokens
 *   path       [n_nodes]   a_0 = 0, a_1..a_m: from the root, step to the
 *                          lowest-indexed child c of the current node u with
 *                          token[c] == am[u]; stop when there is none.
 *                          Entries past m are -1
 *   out_tokens [n_nodes+1] token[a_1..a_m] then the bonus token am[a_m];
 *                          entries past m are -1
 *   new_pos    [n_nodes]   cache row each node's KV moves to (old node
 *                          order): keep = a_0..a_m followed by the strict
 *                          descendants of a_m in node order; node keep[k]
 *                          moves to row P + k; dropped nodes get -1
 *   new_parent [n_nodes]   parent array of the surviving subtree in its new
 *                          node order (survivor k = keep[m + 1 + k]): the
 *                          parent's new index, or -1 when the parent is a_m;
 *                          entries k >= r are -1
 *   n_survivors [1]        r, the number of surviving tree nodes; the next
 *                          prefix length is P + m + 1
 *   dev_status device int32 or NULL; TV_ERR_INVALID_TREE on a bad parent or
 *              token id
 */
TV_API tv_status tv_tree_accept(const float* logits, int32_t vocab, const int32_t* token,
                         const int32_t* parent, int32_t n_nodes, int32_t prefix_len,
                         int32_t* am, int32_t* m, int32_t* path, int32_t* out_tokens,
                         int32_t* new_pos, int32_t* new_parent, int32_t* n_survivors,
                         int32_t* dev_status, tv_stream_t stream);

/*
 * tv_tree_accept_tokens -- tv_tree_accept without the argmax pass: the
 * target's token at every node is given (am of tv_lm_head_argmax, which
 * never writes the logits).  Same passage and outputs as tv_tree_accept,
 * less am.
 *
 *   target_token  device int32 [n_nodes]: the target's token at each node
 *                 (a value outside [0, vocab) matches no draft token; it is
 *                 still emitted as the bonus token when the walk stops there)
 *   vocab, token, parent, n_nodes, prefix_len, outputs, dev_status: as for
 *                 tv_tree_accept
 */
TV_API tv_status tv_tree_accept_tokens(const int32_t* target_token, int32_t vocab,
                                       const int32_t* token, const int32_t* parent,
                                       int32_t n_nodes, int32_t prefix_len, int32_t* m,
                                       int32_t* path, int32_t* out_tokens, int32_t* new_pos,
                                       int32_t* new_parent, int32_t* n_survivors,
                                       int32_t* dev_status, tv_stream_t stream);

/*
 * tv_tree_accept_sampled -- sampling (stochastic) verification of the draft
 * tree at temperature T, with the outputs of tv_tree_accept.
 *
 * The SwiftSpec review page verifies greedily ("What carries the argument":
 * the verified tokens are the target's) and is silent on sampling; this is
 * the library's reading for trees grown deterministically by
 * maximum-likelihood expansion ("Assumptions & free parameters").  At every
 * node i the target's token is drawn from p_i = softmax(logits[i] / T) by
 * inversion: the smallest v with p_i[0] + ... + p_i[v] > u_i, where u_i is
 * the uniform (x0 >> 11 + 1/2) / 2^53 from the first word x0 of
 * Philox4x64-10 (Salmon et al., SC 2011) with key (seed, 0) and counter
 * (i, offset, 0, 0).  The walk is tv_tree_accept's with the drawn tokens in
 * place of the argmax, so every emitted token is the target's own draw at its
 * context (the step is lossless).  The draws are made in float32 with double
 * sums: a u within about 1e-6 of a cumulative-probability boundary may fall
 * on either side of it.
 *
 *   temperature  T > 0 and finite (0 is the greedy tv_tree_accept)
 *   seed, offset the generator's key and the counter's second word; use a
 *                new offset for every verification step
 *   sampled      device int32 [n_nodes], written: the drawn token per node
 *                (-1 for a node whose logits are all -inf)
 * Other arguments and outputs: as tv_tree_accept (logits finite or -inf).
 */
TV_API tv_status tv_tree_accept_sampled(const float* logits, int32_t vocab, const int32_t* token,
                                        const int32_t* parent, int32_t n_nodes,
                                        int32_t prefix_len, float temperature, uint64_t seed,
                                        uint64_t offset, int32_t* sampled, int32_t* m,
                                        int32_t* path, int32_t* out_tokens, int32_t* new_pos,
                                        int32_t* new_parent, int32_t* n_survivors,
                                        int32_t* dev_status, tv_stream_t stream);

/*
 * tv_kv_compact -- in-place reorganisation of the K and V caches of every
 * layer after a verification.
 *
 * Passage: SwiftSpec review page, "What carries the argument" and "Core
 * claim" (accepted tokens join the prefix; surviving tree entries are
 * reorganised contiguously after it).
 *
 * For every layer l < n_layers, KV head g < hkv and both caches, the row of
 * tree node i (row prefix_len + i) is copied to row new_pos[i] for every i
 * with new_pos[i] >= 0.  new_pos is read on the device (it is normally the
 * output of tv_tree_accept), so no host synchronisation is needed.  Rows
 * below prefix_len are never touched, no row outside
 * [prefix_len, prefix_len + n_nodes) is written, and rows of the tree region
 * that no node moves to keep whatever they held.
 *
 *   k_cache, v_cache   device base of layer 0, [n_layers][hkv][cap][d]
 *                      with layer l at element offset l * layer_stride_elems
 *   layer_stride_elems >= hkv * cap * d
 *   cap                rows per head, >= prefix_len + n_nodes
 *   d                  row length in elements; d * sizeof(dtype) must be a
 *                      multiple of 16 bytes, at most 512 bytes
 *   new_pos            device int32 [n_nodes]: -1 or a row in
 *                      [prefix_len, prefix_len + i] for node i, distinct;
 *                      any other entry is skipped and reported as
 *                      TV_ERR_INVALID_ARG in dev_status
 */
TV_API tv_status tv_kv_compact(void* k_cache, void* v_cache, int32_t n_layers,
                        int64_t layer_stride_elems, int32_t hkv, int64_t cap, int32_t d,
                        int32_t dtype, int32_t prefix_len, int32_t n_nodes,
                        const int32_t* new_pos, int32_t* dev_status, tv_stream_t stream);

/*
 * Batched acceptance and compaction: the rest of a verification step for up
 * to TV_MAX_BATCH requests at once, beside tv_tree_attn_verify_batched.
 * Same passages as tv_tree_accept and tv_kv_compact; every request's results
 * are exactly (bit for bit) what the single-request calls give for it.
 *
 * Packed node arrays.  node_offset is a HOST int32 array of batch + 1
 * entries, node_offset[0] = 0: request b owns entries
 * [node_offset[b], node_offset[b + 1]) of every per-node device array
 * (logits rows, token, parent, am, path, new_pos, new_parent), with 1 to
 * TV_MAX_NODES nodes, and its parent entries are indices within the request
 * (node 0 is its root).  m and n_survivors hold one entry per request;
 * request b's n_b + 1 out_tokens start at entry node_offset[b] + b.
 * prefix_len is a HOST int32 array of batch entries.  A tree or token error
 * in one request is reported in dev_status and leaves that request's
 * outputs as tv_tree_accept leaves them; the other requests are unaffected.
 */

/* tv_tree_accept over packed requests: logits device float32
 * [node_offset[batch]][vocab], one argmax pass over all rows, then one walk
 * per request.  Host-side errors as tv_tree_accept, plus TV_ERR_INVALID_ARG
 * for batch outside [1, TV_MAX_BATCH] or a bad node_offset. */
TV_API tv_status tv_tree_accept_batched(int32_t batch, const int32_t* node_offset,
                                        const int32_t* prefix_len, const float* logits,
                                        int32_t vocab, const int32_t* token,
                                        const int32_t* parent, int32_t* am, int32_t* m,
                                        int32_t* path, int32_t* out_tokens, int32_t* new_pos,
                                        int32_t* new_parent, int32_t* n_survivors,
                                        int32_t* dev_status, tv_stream_t stream);

/* tv_tree_accept_tokens over packed requests (target_token packed like
 * token). */
TV_API tv_status tv_tree_accept_tokens_batched(int32_t batch, const int32_t* node_offset,
                                               const int32_t* prefix_len,
                                               const int32_t* target_token, int32_t vocab,
                                               const int32_t* token, const int32_t* parent,
                                               int32_t* m, int32_t* path, int32_t* out_tokens,
                                               int32_t* new_pos, int32_t* new_parent,
                                               int32_t* n_survivors, int32_t* dev_status,
                                               tv_stream_t stream);

/* tv_tree_accept_sampled over packed requests: temperature (float), seed
 * and offset (uint64) are HOST arrays of `batch` entries, one sampling
 * setting per request; node i of request b draws with the counter of its
 * index within the request, (i, offset[b], 0, 0), under key (seed[b], 0),
 * so every request's draws equal those of tv_tree_accept_sampled with its
 * own setting.  sampled is packed like token.  Host-side errors as
 * tv_tree_accept_sampled and tv_tree_accept_batched. */
TV_API tv_status tv_tree_accept_sampled_batched(int32_t batch, const int32_t* node_offset,
                                                const int32_t* prefix_len, const float* logits,
                                                int32_t vocab, const int32_t* token,
                                                const int32_t* parent, const float* temperature,
                                                const uint64_t* seed, const uint64_t* offset,
                                                int32_t* sampled, int32_t* m, int32_t* path,
                                                int32_t* out_tokens, int32_t* new_pos,
                                                int32_t* new_parent, int32_t* n_survivors,
                                                int32_t* dev_status, tv_stream_t stream);

/*
 * tv_kv_compact for `batch` requests in one launch.  HOST arrays of `batch`
 * entries:
 *   k_cache, v_cache     device bases of layer 0 of request b's caches,
 *                        [n_layers][hkv][cap[b]][d] with layer l at element
 *                        offset l * layer_stride_elems[b]
 *   layer_stride_elems   >= hkv * cap[b] * d
 *   cap, prefix_len, n_nodes   as tv_kv_compact, per request
 *   new_pos              device pointers, request b's new_pos [n_nodes[b]]
 *                        (for packed acceptance outputs: new_pos +
 *                        node_offset[b])
 * n_layers, hkv, d and dtype are shared.  The rows
 * [prefix_len[b], prefix_len[b] + n_nodes[b]) of different requests must not
 * overlap in memory (they are moved concurrently).  Every check of
 * tv_kv_compact applies to every request and is made before the launch.
 */
TV_API tv_status tv_kv_compact_batched(int32_t batch, void* const* k_cache,
                                       void* const* v_cache, const int64_t* layer_stride_elems,
                                       const int64_t* cap, const int32_t* prefix_len,
                                       const int32_t* n_nodes, const int32_t* const* new_pos,
                                       int32_t n_layers, int32_t hkv, int32_t d, int32_t dtype,
                                       int32_t* dev_status, tv_stream_t stream);

/* tv_kv_compact_paged for `batch` requests sharing one page pool per layer:
 * page_table, prefix_len, n_nodes and new_pos are HOST arrays of `batch`
 * entries (page_table[b] and new_pos[b] device pointers).  No page may hold
 * tree rows [prefix_len[b], prefix_len[b] + n_nodes[b]) of one request and
 * any row of another; prefix pages may be shared, since compaction never
 * writes below prefix_len. */
TV_API tv_status tv_kv_compact_batched_paged(int32_t batch, void* k_pool, void* v_pool,
                                             int32_t n_layers, int64_t layer_stride_elems,
                                             int32_t num_pages, int32_t hkv, int32_t page_size,
                                             int32_t d, int32_t dtype,
                                             const int32_t* const* page_table,
                                             const int32_t* prefix_len, const int32_t* n_nodes,
                                             const int32_t* const* new_pos, int32_t* dev_status,
                                             tv_stream_t stream);

/*
 * The draft side.  These two calls serve the draft model that proposes the
 * trees; they are not part of the target's verification step.
 */

#define TV_MAX_EXPAND_WIDTH 64          /* w, new leaves per expansion */
#define TV_MAX_EXPAND_CANDIDATES 1024   /* n_frontier * w, and ceil(vocab / 8192) * w */
#define TV_MAX_VOCAB 524288

/* Bytes of workspace tv_tree_expand needs; 0 for arguments it rejects. */
TV_API size_t tv_expand_workspace_size(int32_t n_frontier, int32_t vocab, int32_t w);

/*
 * tv_tree_expand -- one maximum-likelihood expansion of the draft tree.
 *
 * Passage: SwiftSpec review page, "Assumptions & free parameters" (the
 * domain assumption on maximum-likelihood tree expansion: a path scores the
 * sum of the log-softmax probabilities along it, and the leaves to expand
 * are chosen by that score; Algorithm 1 and Section 3.1 of the paper) and
 * "Core claim".  The page gives the rule in prose; this library reads it as:
 * every child (f, v) of a frontier node scores
 *     cum[frontier[f]] + log_softmax(logits[f])[v]
 * and the w best become new leaves, best first, equal scores going to the
 * lower frontier position f and then to the lower token id v.
 *
 *   logits      device float32 [n_frontier][vocab]: the draft's logits at
 *               each frontier node; finite or -inf (NaN is not supported).
 *               A -inf logit's child scores -inf; a row that is -inf
 *               throughout has no children
 *   vocab       1 .. TV_MAX_VOCAB
 *   n_frontier  1 .. TV_MAX_NODES
 *   frontier    device int32 [n_frontier]: tree node of each logits row,
 *               in [0, n_nodes)
 *   cum         device float32 [n_nodes]: cumulative log-probability of
 *               every tree node (0 at the root)
 *   w           1 .. TV_MAX_EXPAND_WIDTH and at most n_frontier * vocab;
 *               n_frontier * w and ceil(vocab / 8192) * w at most
 *               TV_MAX_EXPAND_CANDIDATES (w = 64 allows a 131072-token
 *               vocabulary, w = 16 the largest)
 * Outputs (device, written; pass parent + N, token + N, cum + N to append
 * the new leaves to a tree of N nodes):
 *   new_parent  int32 [w]   tree node of each new leaf's parent
 *   new_token   int32 [w]   its token
 *   new_score   float32 [w] its cumulative log-probability (its score)
 * workspace: device memory of at least tv_expand_workspace_size bytes; its
 * contents on entry do not matter.  dev_status: device int32 or NULL;
 * TV_ERR_INVALID_ARG when a frontier entry is out of range (the outputs are
 * then -1 / -inf).  Scores are computed in float32, so candidates whose
 * scores differ by less than float32 rounding may come out in either order.
 */
TV_API tv_status tv_tree_expand(const float* logits, int32_t vocab, int32_t n_frontier,
                                const int32_t* frontier, const float* cum, int32_t n_nodes,
                                int32_t w, int32_t* new_parent, int32_t* new_token,
                                float* new_score, void* workspace, size_t ws_bytes,
                                int32_t* dev_status, tv_stream_t stream);

/*
 * tv_draft_reroot -- the draft tree's re-root map after a verification.
 *
 * Passage: SwiftSpec review page, "What carries the argument" (after each
 * verification the draft tree re-roots at the last verified token and the
 * cache keeps only the still-useful subtree) and "Core claim".  The draft
 * keeps expanding while the target verifies, so its tree extends the tree
 * that was verified (the first nodes are the same).  This library reads the
 * survivor rule as: the new root is the child b of the last accepted node
 * a_m that carries the bonus token (the lowest-indexed one if several), and
 * the survivors are b and its descendants, in node order; without such a
 * child nothing survives.
 *
 *   parent, token  device int32 [n_nodes]: the draft tree (node 0 the root)
 *   cum            device float32 [n_nodes]: cumulative log-probabilities
 *   n_nodes        1 .. TV_MAX_NODES
 *   path, m, out_tokens  device: the outputs of tv_tree_accept for the
 *                  verified tree (path a_0..a_m, the bonus token out_tokens[m])
 *   prefix_len     P, the prefix length before the verification
 * Outputs (device, written):
 *   new_pos      int32 [n_nodes]  cache row of each node's KV (old order):
 *                a_k moves to row P + k, survivor k to row P + m + 1 + k,
 *                others -1 (feed it to tv_kv_compact for the draft's cache)
 *   new_parent   int32 [n_nodes]  parents of the survivors in their new order
 *                (-1 for the new root b and for entries k >= r)
 *   new_token    int32 [n_nodes]  their tokens (-1 for k >= r)
 *   new_cum      float32 [n_nodes] their cumulative log-probabilities minus
 *                that of b, so the new root has 0 (0 for k >= r)
 *   n_survivors  int32 [1]        r
 *   dev_status   device int32 or NULL; TV_ERR_INVALID_TREE on a bad parent,
 *                m or path (outputs then -1 / 0, r = 0)
 */
TV_API tv_status tv_draft_reroot(const int32_t* parent, const int32_t* token, const float* cum,
                                 int32_t n_nodes, const int32_t* path, const int32_t* m,
                                 const int32_t* out_tokens, int32_t prefix_len,
                                 int32_t* new_pos, int32_t* new_parent, int32_t* new_token,
                                 float* new_cum, int32_t* n_survivors, int32_t* dev_status,
                                 tv_stream_t stream);

/*
 * The target's LM head fused with the argmax.
 */

#define TV_MAX_LM_NODES 256

/* Bytes of workspace tv_lm_head_argmax needs on the current device; 0 for
 * arguments it rejects. */
TV_API size_t tv_lm_head_workspace_size(int32_t n_nodes, int32_t vocab);

/*
 * tv_lm_head_argmax -- the target's greedy token at every tree node, straight
 * from the final hidden states.
 *
 * Passage: SwiftSpec review page, "What carries the argument" (the verified
 * tokens are the target's greedy choices at the tree nodes); the logits the
 * greedy walk compares are the LM head's, z_i = W h_i.  This call computes
 *     am[i] = argmax_v  sum_k hidden[i][k] * weight[v][k]
 * (ties to the lowest v) on the tensor cores with fp32 accumulation, and
 * never writes the n_nodes x vocab logits to memory.  am feeds the greedy
 * walk in place of tv_tree_accept's own argmax pass.
 *
 *   hidden     device bf16 [n_nodes][d_model], rows contiguous, 16-byte
 *              aligned: the final (normalised) hidden state of each node
 *   weight     device bf16 [vocab][d_model], rows contiguous, 16-byte
 *              aligned: the LM head (the layout of a linear layer's weight)
 *   n_nodes    1 .. TV_MAX_LM_NODES
 *   d_model    a multiple of 8, at least 8
 *   vocab      >= 1
 * Outputs (device, written):
 *   am         int32 [n_nodes]    the argmax token of each node
 *   max_logit  float32 [n_nodes]  its fp32 logit; may be NULL
 * workspace: device memory of at least tv_lm_head_workspace_size bytes,
 * 16-byte aligned; its contents on entry do not matter.  dev_status: device
 * int32 or NULL; TV_ERR_TIMEOUT if a device wait ran out (outputs are then
 * unspecified).  Logits are rounded float32 sums, so tokens whose exact
 * logits differ by less than that rounding may be chosen either way; a node
 * whose logits are all NaN or -inf gets -1.
 */
TV_API tv_status tv_lm_head_argmax(const void* hidden, const void* weight, int32_t n_nodes,
                                   int32_t d_model, int32_t vocab, int32_t* am, float* max_logit,
                                   void* workspace, size_t ws_bytes, int32_t* dev_status,
                                   tv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TREEVERIFY_H */
