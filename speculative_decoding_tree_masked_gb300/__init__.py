"""Tree-masked speculative verification on one GB300 GPU.

A thin Python binding over the C ABI of libtreeverify.so (include/treeverify.h):
the functions below only check tensor shapes, take device pointers and the
current CUDA stream from PyTorch and call the library; every step of the
computation runs in the library's CUDA kernels.

    tree_mask(parent)                                  ancestor bitmasks
    tree_attn_verify(q, k_cache, v_cache, P, parent)   one layer of tree attention
    tree_accept(logits, token, parent, P)              argmax, greedy walk, re-root map
    kv_compact(k_caches, v_caches, P, N, new_pos)      in-place cache reorganisation

The step follows the SwiftSpec review page (pith.science, paper 2506.11309),
"What carries the argument" and "Core claim".
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib

TV_OK, TV_ERR_INVALID_ARG, TV_ERR_UNSUPPORTED, TV_ERR_CAPACITY, TV_ERR_CUDA, \
    TV_ERR_INVALID_TREE, TV_ERR_TIMEOUT, TV_ERR_BOUNDS = range(8)
TV_F32, TV_BF16 = 0, 1
MAX_NODES = 128

_DTYPES = {torch.float32: TV_F32, torch.bfloat16: TV_BF16}


class TreeVerifyError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        name = _lib.load().tv_status_string(status).decode()
        super().__init__(f"{what}: {name} (status {status})")


def lib() -> ctypes.CDLL:
    return _lib.load()


def _check(status: int, what: str) -> None:
    if status != TV_OK:
        raise TreeVerifyError(status, what)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _need_cuda(*ts: torch.Tensor) -> None:
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return _DTYPES[t.dtype]


def tree_mask(parent: torch.Tensor, out: Optional[torch.Tensor] = None,
              status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Ancestor bitmask words [N][ceil(N/32)] (uint32 stored as int32)."""
    _need_cuda(parent)
    n = parent.numel()
    if out is None:
        out = torch.empty((n, (n + 31) // 32), dtype=torch.int32, device=parent.device)
    _check(lib().tv_tree_mask(_ptr(parent), n, _ptr(out), _ptr(status),
                              _stream(stream, parent.device)), "tv_tree_mask")
    return out


def attn_workspace_size(n_nodes: int, hq: int, hkv: int, d: int, dtype: torch.dtype,
                        max_prefix: int) -> int:
    return int(lib().tv_attn_workspace_size(n_nodes, hq, hkv, d, _DTYPES[dtype], max_prefix))


def attn_plan(n_nodes: int, hq: int, hkv: int, d: int, dtype: torch.dtype, prefix_len: int,
              sm_count: int = 0) -> dict:
    """The split plan of tree_attn_verify for this shape on a GPU with
    sm_count SMs (0: the current device's): row_groups, splits,
    keys_per_split and ws_bytes."""
    rg, sp, kps = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    ws = ctypes.c_size_t()
    _check(lib().tv_attn_plan(n_nodes, hq, hkv, d, _DTYPES[dtype], prefix_len, sm_count,
                              ctypes.byref(rg), ctypes.byref(sp), ctypes.byref(kps),
                              ctypes.byref(ws)), "tv_attn_plan")
    return {"row_groups": rg.value, "splits": sp.value, "keys_per_split": kps.value,
            "ws_bytes": ws.value}


def attn_workspace(n_nodes: int, hq: int, hkv: int, d: int, dtype: torch.dtype, max_prefix: int,
                   device) -> torch.Tensor:
    """A workspace tensor large enough for every prefix up to max_prefix."""
    nbytes = attn_workspace_size(n_nodes, hq, hkv, d, dtype, max_prefix)
    # 0 means the library does not take this shape; a token buffer lets the
    # call itself report why
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def tree_attn_verify(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     prefix_len: int, parent: torch.Tensor, out: Optional[torch.Tensor] = None,
                     scale: float = 0.0, workspace: Optional[torch.Tensor] = None,
                     status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One layer of tree-masked GQA attention.

    q [N][Hq][d]; k_cache, v_cache [Hkv][cap][d] (rows [0, P) prefix, row P+j
    tree node j); parent int32 [N].  Returns out [N][Hq][d] in q's dtype."""
    _need_cuda(q, k_cache, v_cache, parent)
    n, hq, d = q.shape
    hkv, cap, dk = k_cache.shape
    if v_cache.shape != k_cache.shape or dk != d or parent.numel() != n:
        raise ValueError("shape mismatch")
    if k_cache.dtype != q.dtype or v_cache.dtype != q.dtype or parent.dtype != torch.int32:
        raise ValueError("dtype mismatch")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = attn_workspace(n, hq, hkv, d, q.dtype, prefix_len, q.device)
    _check(lib().tv_tree_attn_verify(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), cap, prefix_len, n, _ptr(parent), _ptr(out), hq,
        hkv, d, _dtype_code(q), float(scale), _ptr(workspace), workspace.numel() *
        workspace.element_size(), _ptr(status), _stream(stream, q.device)), "tv_tree_attn_verify")
    return out


def tree_attn_verify_static(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            prefix_len: int, parent: torch.Tensor, out: torch.Tensor,
                            scale: float = 0.0, status: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    """tree_attn_verify for callers that cannot allocate device memory: no
    workspace is passed or allocated (the library's fixed 16 MiB device
    scratch array holds the split partials) and `out` must be given.

    CUDA loads the array lazily, so its 16 MiB are reserved on a device at
    the first call there: make that call before a framework's caching
    allocator takes the GPU's free memory, and before any stream capture.
    Calls that overlap on the GPU share the scratch array and race."""
    _need_cuda(q, k_cache, v_cache, parent, out)
    n, hq, d = q.shape
    hkv, cap, dk = k_cache.shape
    if v_cache.shape != k_cache.shape or dk != d or parent.numel() != n or out.shape != q.shape:
        raise ValueError("shape mismatch")
    if k_cache.dtype != q.dtype or v_cache.dtype != q.dtype or out.dtype != q.dtype or \
            parent.dtype != torch.int32:
        raise ValueError("dtype mismatch")
    _check(lib().tv_tree_attn_verify_static(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), cap, prefix_len, n, _ptr(parent), _ptr(out), hq,
        hkv, d, _dtype_code(q), float(scale), _ptr(status), _stream(stream, q.device)),
        "tv_tree_attn_verify_static")
    return out


def _host_array(ctype, values):
    return (ctype * len(values))(*values)


def attn_batched_workspace_size(n_nodes, hq: int, hkv: int, d: int, dtype: torch.dtype) -> int:
    ns = _host_array(ctypes.c_int32, [int(x) for x in n_nodes])
    return int(lib().tv_attn_batched_workspace_size(len(ns), ctypes.cast(ns, ctypes.c_void_p),
                                                    hq, hkv, d, _DTYPES[dtype]))


def tree_attn_verify_batched(qs, k_caches, v_caches, prefix_lens, parents, outs=None,
                             scale: float = 0.0, workspace: Optional[torch.Tensor] = None,
                             status: Optional[torch.Tensor] = None, stream=None) -> list:
    """Tree attention for several requests in one launch (bf16).  Lists of
    per-request tensors: q [N_b][Hq][d], caches [Hkv][cap_b][d], parent int32
    [N_b]; prefix_lens a list of ints.  Returns the list of outputs."""
    batch = len(qs)
    if not (len(k_caches) == len(v_caches) == len(prefix_lens) == len(parents) == batch):
        raise ValueError("per-request lists differ in length")
    _need_cuda(*qs, *k_caches, *v_caches, *parents)
    hq, d = qs[0].shape[1], qs[0].shape[2]
    hkv = k_caches[0].shape[0]
    for q, k, v, par in zip(qs, k_caches, v_caches, parents):
        if q.shape[1:] != (hq, d) or k.shape[0] != hkv or k.shape[2] != d or \
                v.shape != k.shape or par.numel() != q.shape[0]:
            raise ValueError("shape mismatch")
        if q.dtype != qs[0].dtype or k.dtype != q.dtype or v.dtype != q.dtype or \
                par.dtype != torch.int32:
            raise ValueError("dtype mismatch")
    if outs is None:
        outs = [torch.empty_like(q) for q in qs]
    ns = [q.shape[0] for q in qs]
    if workspace is None:
        nbytes = attn_batched_workspace_size(ns, hq, hkv, d, qs[0].dtype)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=qs[0].device)
    vp = lambda ts: _host_array(ctypes.c_void_p, [_ptr(t) for t in ts])
    arrs = [vp(qs), vp(k_caches), vp(v_caches),
            _host_array(ctypes.c_int64, [k.shape[1] for k in k_caches]),
            _host_array(ctypes.c_int32, [int(x) for x in prefix_lens]),
            _host_array(ctypes.c_int32, ns), vp(parents), vp(outs)]
    cp = [ctypes.cast(a, ctypes.c_void_p) for a in arrs]
    _check(lib().tv_tree_attn_verify_batched(
        batch, cp[0], cp[1], cp[2], cp[3], cp[4], cp[5], cp[6], cp[7], hq, hkv, d,
        _dtype_code(qs[0]), float(scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream, qs[0].device)), "tv_tree_attn_verify_batched")
    return outs


def _check_pool(k_pool: torch.Tensor, v_pool: torch.Tensor):
    if k_pool.dim() != 4 or v_pool.shape != k_pool.shape or v_pool.dtype != k_pool.dtype:
        raise ValueError("pools must be [num_pages][Hkv][page_size][d] and alike")
    if not k_pool.is_contiguous() or not v_pool.is_contiguous():
        raise ValueError("pools must be contiguous")
    return k_pool.shape


def tree_attn_verify_paged(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                           page_table: torch.Tensor, prefix_len: int, parent: torch.Tensor,
                           out: Optional[torch.Tensor] = None, scale: float = 0.0,
                           workspace: Optional[torch.Tensor] = None,
                           status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Tree attention over a paged K/V cache (bf16): pools [num_pages][Hkv]
    [page_size][d], page_table int32 [ceil((P + N) / page_size)] naming the
    page of each run of page_size logical rows.  Otherwise as
    tree_attn_verify."""
    _need_cuda(q, k_pool, v_pool, page_table, parent)
    num_pages, hkv, page_size, d = _check_pool(k_pool, v_pool)
    n, hq, dq = q.shape
    if dq != d or parent.numel() != n or page_table.dtype != torch.int32:
        raise ValueError("shape mismatch")
    if k_pool.dtype != q.dtype or parent.dtype != torch.int32:
        raise ValueError("dtype mismatch")
    if page_table.numel() * page_size < prefix_len + n:
        raise ValueError("page table shorter than prefix + tree")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = attn_workspace(n, hq, hkv, d, q.dtype, prefix_len, q.device)
    _check(lib().tv_tree_attn_verify_paged(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), num_pages, page_size, _ptr(page_table), prefix_len,
        n, _ptr(parent), _ptr(out), hq, hkv, d, _dtype_code(q), float(scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream, q.device)),
        "tv_tree_attn_verify_paged")
    return out


def tree_attn_verify_batched_paged(qs, k_pool: torch.Tensor, v_pool: torch.Tensor, page_tables,
                                   prefix_lens, parents, outs=None, scale: float = 0.0,
                                   workspace: Optional[torch.Tensor] = None,
                                   status: Optional[torch.Tensor] = None, stream=None) -> list:
    """tree_attn_verify_batched over one shared page pool: request b has its
    own page table page_tables[b] (int32)."""
    batch = len(qs)
    if not (len(page_tables) == len(prefix_lens) == len(parents) == batch):
        raise ValueError("per-request lists differ in length")
    _need_cuda(k_pool, v_pool, *qs, *page_tables, *parents)
    num_pages, hkv, page_size, d = _check_pool(k_pool, v_pool)
    hq = qs[0].shape[1]
    for q, tab, par, p in zip(qs, page_tables, parents, prefix_lens):
        if q.shape[1:] != (hq, d) or par.numel() != q.shape[0] or tab.dtype != torch.int32 or \
                par.dtype != torch.int32 or q.dtype != k_pool.dtype:
            raise ValueError("shape or dtype mismatch")
        if tab.numel() * page_size < int(p) + q.shape[0]:
            raise ValueError("page table shorter than prefix + tree")
    if outs is None:
        outs = [torch.empty_like(q) for q in qs]
    ns = [q.shape[0] for q in qs]
    if workspace is None:
        nbytes = attn_batched_workspace_size(ns, hq, hkv, d, qs[0].dtype)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=qs[0].device)
    vp = lambda ts: _host_array(ctypes.c_void_p, [_ptr(t) for t in ts])
    arrs = [vp(qs), vp(page_tables), _host_array(ctypes.c_int32, [int(x) for x in prefix_lens]),
            _host_array(ctypes.c_int32, ns), vp(parents), vp(outs)]
    cp = [ctypes.cast(a, ctypes.c_void_p) for a in arrs]
    _check(lib().tv_tree_attn_verify_batched_paged(
        batch, cp[0], _ptr(k_pool), _ptr(v_pool), num_pages, page_size, cp[1], cp[2], cp[3],
        cp[4], cp[5], hq, hkv, d, _dtype_code(qs[0]), float(scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream, qs[0].device)), "tv_tree_attn_verify_batched_paged")
    return outs


def kv_compact_paged(k_pools: torch.Tensor, v_pools: torch.Tensor, page_table: torch.Tensor,
                     prefix_len: int, n_nodes: int, new_pos: torch.Tensor,
                     status: Optional[torch.Tensor] = None, stream=None) -> None:
    """In-place compaction of paged caches: pools [L][num_pages][Hkv]
    [page_size][d] (or one layer without L); logical rows map through
    page_table."""
    _need_cuda(k_pools, v_pools, page_table, new_pos)
    if k_pools.shape != v_pools.shape or k_pools.dtype != v_pools.dtype:
        raise ValueError("k and v pools differ")
    shape = k_pools.shape if k_pools.dim() == 5 else (1,) + tuple(k_pools.shape)
    layers, num_pages, hkv, page_size, d = shape
    if new_pos.dtype != torch.int32 or new_pos.numel() != n_nodes or \
            page_table.dtype != torch.int32:
        raise ValueError("new_pos and page_table must be int32")
    _check(lib().tv_kv_compact_paged(
        _ptr(k_pools), _ptr(v_pools), layers, num_pages * hkv * page_size * d, num_pages, hkv,
        page_size, d, _dtype_code(k_pools), _ptr(page_table), prefix_len, n_nodes, _ptr(new_pos),
        _ptr(status), _stream(stream, k_pools.device)), "tv_kv_compact_paged")


def tree_accept(logits: torch.Tensor, token: torch.Tensor, parent: torch.Tensor, prefix_len: int,
                outs: Optional[dict] = None, status: Optional[torch.Tensor] = None,
                stream=None) -> dict:
    """Greedy acceptance and the re-root map; all results stay on the device.

    Returns a dict of int32 tensors: am [N], m [1], path [N], out_tokens [N+1],
    new_pos [N], new_parent [N], n_survivors [1]."""
    _need_cuda(logits, token, parent)
    n, vocab = logits.shape
    if logits.dtype != torch.float32 or token.dtype != torch.int32 or parent.dtype != torch.int32:
        raise ValueError("dtype mismatch")
    if token.numel() != n or parent.numel() != n:
        raise ValueError("shape mismatch")
    if outs is None:
        dev = logits.device
        outs = {k: torch.empty(sz, dtype=torch.int32, device=dev) for k, sz in (
            ("am", n), ("m", 1), ("path", n), ("out_tokens", n + 1), ("new_pos", n),
            ("new_parent", n), ("n_survivors", 1))}
    _check(lib().tv_tree_accept(
        _ptr(logits), vocab, _ptr(token), _ptr(parent), n, prefix_len, _ptr(outs["am"]),
        _ptr(outs["m"]), _ptr(outs["path"]), _ptr(outs["out_tokens"]), _ptr(outs["new_pos"]),
        _ptr(outs["new_parent"]), _ptr(outs["n_survivors"]), _ptr(status),
        _stream(stream, logits.device)), "tv_tree_accept")
    return outs


def tree_accept_tokens(target_token: torch.Tensor, vocab: int, token: torch.Tensor,
                       parent: torch.Tensor, prefix_len: int, outs: Optional[dict] = None,
                       status: Optional[torch.Tensor] = None, stream=None) -> dict:
    """tree_accept with the target's token at every node given (the "am" of
    lm_head_argmax) instead of logits.  Returns the dict of tree_accept
    without "am"."""
    _need_cuda(target_token, token, parent)
    n = parent.numel()
    if target_token.dtype != torch.int32 or token.dtype != torch.int32 or \
            parent.dtype != torch.int32:
        raise ValueError("dtype mismatch")
    if token.numel() != n or target_token.numel() != n:
        raise ValueError("shape mismatch")
    if outs is None:
        dev = parent.device
        outs = {k: torch.empty(sz, dtype=torch.int32, device=dev) for k, sz in (
            ("m", 1), ("path", n), ("out_tokens", n + 1), ("new_pos", n), ("new_parent", n),
            ("n_survivors", 1))}
    _check(lib().tv_tree_accept_tokens(
        _ptr(target_token), vocab, _ptr(token), _ptr(parent), n, prefix_len, _ptr(outs["m"]),
        _ptr(outs["path"]), _ptr(outs["out_tokens"]), _ptr(outs["new_pos"]),
        _ptr(outs["new_parent"]), _ptr(outs["n_survivors"]), _ptr(status),
        _stream(stream, parent.device)), "tv_tree_accept_tokens")
    return outs


def tree_accept_sampled(logits: torch.Tensor, token: torch.Tensor, parent: torch.Tensor,
                        prefix_len: int, temperature: float, seed: int, offset: int,
                        outs: Optional[dict] = None, status: Optional[torch.Tensor] = None,
                        stream=None) -> dict:
    """Sampling verification at temperature T: the target's token at every
    node drawn from softmax(logits / T) with a counter-based generator keyed
    by (seed, offset), then the walk of tree_accept over the drawn tokens.
    Returns the dict of tree_accept with "sampled" [N] in place of "am"."""
    _need_cuda(logits, token, parent)
    n, vocab = logits.shape
    if logits.dtype != torch.float32 or token.dtype != torch.int32 or parent.dtype != torch.int32:
        raise ValueError("dtype mismatch")
    if token.numel() != n or parent.numel() != n:
        raise ValueError("shape mismatch")
    if outs is None:
        dev = logits.device
        outs = {k: torch.empty(sz, dtype=torch.int32, device=dev) for k, sz in (
            ("sampled", n), ("m", 1), ("path", n), ("out_tokens", n + 1), ("new_pos", n),
            ("new_parent", n), ("n_survivors", 1))}
    _check(lib().tv_tree_accept_sampled(
        _ptr(logits), vocab, _ptr(token), _ptr(parent), n, prefix_len, float(temperature),
        int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), _ptr(outs["sampled"]),
        _ptr(outs["m"]), _ptr(outs["path"]), _ptr(outs["out_tokens"]), _ptr(outs["new_pos"]),
        _ptr(outs["new_parent"]), _ptr(outs["n_survivors"]), _ptr(status),
        _stream(stream, logits.device)), "tv_tree_accept_sampled")
    return outs


def kv_compact(k_cache: torch.Tensor, v_cache: torch.Tensor, prefix_len: int, n_nodes: int,
               new_pos: torch.Tensor, status: Optional[torch.Tensor] = None,
               stream=None) -> None:
    """In-place compaction of K and V caches shaped [L][Hkv][cap][d] (or
    [Hkv][cap][d] for one layer): row P+i moves to new_pos[i] for kept i."""
    _need_cuda(k_cache, v_cache, new_pos)
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise ValueError("k and v caches differ")
    shape = k_cache.shape if k_cache.dim() == 4 else (1,) + tuple(k_cache.shape)
    layers, hkv, cap, d = shape
    if new_pos.dtype != torch.int32 or new_pos.numel() != n_nodes:
        raise ValueError("new_pos must be int32 [n_nodes]")
    _check(lib().tv_kv_compact(
        _ptr(k_cache), _ptr(v_cache), layers, hkv * cap * d, hkv, cap, d, _dtype_code(k_cache),
        prefix_len, n_nodes, _ptr(new_pos), _ptr(status), _stream(stream, k_cache.device)),
        "tv_kv_compact")


# ------------------------------------------------- batched acceptance, compaction

def node_offsets(n_nodes) -> list:
    """The packed layout's offsets: [0, n_0, n_0 + n_1, ...]."""
    off = [0]
    for n in n_nodes:
        off.append(off[-1] + int(n))
    return off


def _packed_outs(names, n_nodes, device) -> dict:
    off = node_offsets(n_nodes)
    total, batch = off[-1], len(n_nodes)
    sizes = {"am": total, "sampled": total, "m": batch, "path": total,
             "out_tokens": total + batch, "new_pos": total, "new_parent": total,
             "n_survivors": batch}
    return {k: torch.empty(sizes[k], dtype=torch.int32, device=device) for k in names}


def _check_packed(n_nodes, prefix_lens, *per_node):
    if len(n_nodes) != len(prefix_lens):
        raise ValueError("n_nodes and prefix_lens differ in length")
    total = sum(int(n) for n in n_nodes)
    for t in per_node:
        if t.dtype != torch.int32 or t.numel() != total:
            raise ValueError("packed per-node arrays must be int32 [sum(n_nodes)]")
    return node_offsets(n_nodes)


def tree_accept_batched(logits: torch.Tensor, token: torch.Tensor, parent: torch.Tensor,
                        n_nodes, prefix_lens, outs: Optional[dict] = None,
                        status: Optional[torch.Tensor] = None, stream=None) -> dict:
    """Greedy acceptance of several requests over packed node arrays: request
    b owns rows off[b] .. off[b + 1] - 1 of logits [total][V], token [total]
    and parent [total] (its parent entries index its own nodes), where off =
    node_offsets(n_nodes).  Returns a dict of packed int32 tensors: am [total],
    m [B], path [total], out_tokens [total + B] (request b's n_b + 1 entries
    from off[b] + b), new_pos [total], new_parent [total], n_survivors [B];
    batched_request(outs, b) gives request b's part in tree_accept's form."""
    _need_cuda(logits, token, parent)
    total, vocab = logits.shape
    off = _check_packed(n_nodes, prefix_lens, token, parent)
    if logits.dtype != torch.float32 or off[-1] != total:
        raise ValueError("logits must be float32 [sum(n_nodes)][V]")
    if outs is None:
        outs = _packed_outs(("am", "m", "path", "out_tokens", "new_pos", "new_parent",
                             "n_survivors"), n_nodes, logits.device)
    offs = _host_array(ctypes.c_int32, off)
    pre = _host_array(ctypes.c_int32, [int(x) for x in prefix_lens])
    _check(lib().tv_tree_accept_batched(
        len(n_nodes), ctypes.cast(offs, ctypes.c_void_p), ctypes.cast(pre, ctypes.c_void_p),
        _ptr(logits), vocab, _ptr(token), _ptr(parent), _ptr(outs["am"]), _ptr(outs["m"]),
        _ptr(outs["path"]), _ptr(outs["out_tokens"]), _ptr(outs["new_pos"]),
        _ptr(outs["new_parent"]), _ptr(outs["n_survivors"]), _ptr(status),
        _stream(stream, logits.device)), "tv_tree_accept_batched")
    outs["node_offset"] = off
    return outs


def tree_accept_tokens_batched(target_token: torch.Tensor, vocab: int, token: torch.Tensor,
                               parent: torch.Tensor, n_nodes, prefix_lens,
                               outs: Optional[dict] = None,
                               status: Optional[torch.Tensor] = None, stream=None) -> dict:
    """tree_accept_batched with the target's token at every packed node given
    instead of logits.  Returns its dict without "am"."""
    _need_cuda(target_token, token, parent)
    off = _check_packed(n_nodes, prefix_lens, target_token, token, parent)
    if outs is None:
        outs = _packed_outs(("m", "path", "out_tokens", "new_pos", "new_parent",
                             "n_survivors"), n_nodes, parent.device)
    offs = _host_array(ctypes.c_int32, off)
    pre = _host_array(ctypes.c_int32, [int(x) for x in prefix_lens])
    _check(lib().tv_tree_accept_tokens_batched(
        len(n_nodes), ctypes.cast(offs, ctypes.c_void_p), ctypes.cast(pre, ctypes.c_void_p),
        _ptr(target_token), vocab, _ptr(token), _ptr(parent), _ptr(outs["m"]),
        _ptr(outs["path"]), _ptr(outs["out_tokens"]), _ptr(outs["new_pos"]),
        _ptr(outs["new_parent"]), _ptr(outs["n_survivors"]), _ptr(status),
        _stream(stream, parent.device)), "tv_tree_accept_tokens_batched")
    outs["node_offset"] = off
    return outs


def tree_accept_sampled_batched(logits: torch.Tensor, token: torch.Tensor, parent: torch.Tensor,
                                n_nodes, prefix_lens, temperatures, seeds, offsets,
                                outs: Optional[dict] = None,
                                status: Optional[torch.Tensor] = None, stream=None) -> dict:
    """tree_accept_sampled over packed requests (the layout of
    tree_accept_batched), each with its own temperature, seed and offset.
    Returns tree_accept_batched's dict with "sampled" [total] in place of
    "am"."""
    _need_cuda(logits, token, parent)
    total, vocab = logits.shape
    off = _check_packed(n_nodes, prefix_lens, token, parent)
    if logits.dtype != torch.float32 or off[-1] != total:
        raise ValueError("logits must be float32 [sum(n_nodes)][V]")
    batch = len(n_nodes)
    if not (len(temperatures) == len(seeds) == len(offsets) == batch):
        raise ValueError("one temperature, seed and offset per request")
    if outs is None:
        outs = _packed_outs(("sampled", "m", "path", "out_tokens", "new_pos", "new_parent",
                             "n_survivors"), n_nodes, logits.device)
    mask = 2**64 - 1
    arrs = [_host_array(ctypes.c_int32, off),
            _host_array(ctypes.c_int32, [int(x) for x in prefix_lens]),
            _host_array(ctypes.c_float, [float(t) for t in temperatures]),
            _host_array(ctypes.c_uint64, [int(x) & mask for x in seeds]),
            _host_array(ctypes.c_uint64, [int(x) & mask for x in offsets])]
    cp = [ctypes.cast(a, ctypes.c_void_p) for a in arrs]
    _check(lib().tv_tree_accept_sampled_batched(
        batch, cp[0], cp[1], _ptr(logits), vocab, _ptr(token), _ptr(parent), cp[2], cp[3],
        cp[4], _ptr(outs["sampled"]), _ptr(outs["m"]), _ptr(outs["path"]),
        _ptr(outs["out_tokens"]), _ptr(outs["new_pos"]), _ptr(outs["new_parent"]),
        _ptr(outs["n_survivors"]), _ptr(status), _stream(stream, logits.device)),
        "tv_tree_accept_sampled_batched")
    outs["node_offset"] = off
    return outs


def batched_request(outs: dict, b: int) -> dict:
    """Request b's results from a packed batched-acceptance dict, as views
    shaped like tree_accept's."""
    off = outs["node_offset"]
    lo, hi = off[b], off[b + 1]
    r = {k: outs[k][lo:hi] for k in ("am", "sampled", "path", "new_pos", "new_parent")
         if k in outs}
    r["out_tokens"] = outs["out_tokens"][lo + b:hi + b + 1]
    r["m"] = outs["m"][b:b + 1]
    r["n_survivors"] = outs["n_survivors"][b:b + 1]
    return r


def _per_request_new_pos(new_pos, n_nodes) -> list:
    """A packed int32 tensor (sliced at node_offsets) or a list of tensors."""
    if isinstance(new_pos, torch.Tensor):
        off = node_offsets(n_nodes)
        if new_pos.numel() != off[-1]:
            raise ValueError("packed new_pos must hold sum(n_nodes) entries")
        new_pos = [new_pos[off[b]:off[b + 1]] for b in range(len(n_nodes))]
    if len(new_pos) != len(n_nodes):
        raise ValueError("one new_pos per request")
    for t, n in zip(new_pos, n_nodes):
        if t.dtype != torch.int32 or t.numel() != int(n):
            raise ValueError("new_pos must be int32 [n_nodes]")
    return list(new_pos)


def kv_compact_batched(k_caches, v_caches, prefix_lens, n_nodes, new_pos,
                       status: Optional[torch.Tensor] = None, stream=None) -> None:
    """kv_compact for several requests in one launch: lists of per-request
    caches [L][Hkv][cap_b][d] (or [Hkv][cap_b][d]), prefix lengths and tree
    sizes; new_pos packed (the new_pos of tree_accept_batched) or a list."""
    batch = len(k_caches)
    if not (len(v_caches) == len(prefix_lens) == len(n_nodes) == batch):
        raise ValueError("per-request lists differ in length")
    new_pos = _per_request_new_pos(new_pos, n_nodes)
    _need_cuda(*k_caches, *v_caches, *new_pos)
    shapes = []
    for k, v in zip(k_caches, v_caches):
        if k.shape != v.shape or k.dtype != v.dtype or k.dtype != k_caches[0].dtype:
            raise ValueError("k and v caches differ")
        if not k.is_contiguous() or not v.is_contiguous():
            raise ValueError("caches must be contiguous")
        shapes.append(k.shape if k.dim() == 4 else (1,) + tuple(k.shape))
    layers, hkv, _, d = shapes[0]
    if any(s[0] != layers or s[1] != hkv or s[3] != d for s in shapes):
        raise ValueError("layers, heads and d must agree")
    vp = lambda ts: _host_array(ctypes.c_void_p, [_ptr(t) for t in ts])
    arrs = [vp(k_caches), vp(v_caches),
            _host_array(ctypes.c_int64, [hkv * s[2] * d for s in shapes]),
            _host_array(ctypes.c_int64, [s[2] for s in shapes]),
            _host_array(ctypes.c_int32, [int(x) for x in prefix_lens]),
            _host_array(ctypes.c_int32, [int(x) for x in n_nodes]), vp(new_pos)]
    cp = [ctypes.cast(a, ctypes.c_void_p) for a in arrs]
    _check(lib().tv_kv_compact_batched(
        batch, cp[0], cp[1], cp[2], cp[3], cp[4], cp[5], cp[6], layers, hkv, d,
        _dtype_code(k_caches[0]), _ptr(status), _stream(stream, k_caches[0].device)),
        "tv_kv_compact_batched")


def kv_compact_batched_paged(k_pools: torch.Tensor, v_pools: torch.Tensor, page_tables,
                             prefix_lens, n_nodes, new_pos,
                             status: Optional[torch.Tensor] = None, stream=None) -> None:
    """kv_compact_paged for several requests sharing one pool per layer
    ([L][num_pages][Hkv][page_size][d], or without L): one page table per
    request; new_pos packed or a list."""
    batch = len(page_tables)
    if not (len(prefix_lens) == len(n_nodes) == batch):
        raise ValueError("per-request lists differ in length")
    new_pos = _per_request_new_pos(new_pos, n_nodes)
    _need_cuda(k_pools, v_pools, *page_tables, *new_pos)
    if k_pools.shape != v_pools.shape or k_pools.dtype != v_pools.dtype:
        raise ValueError("k and v pools differ")
    if not k_pools.is_contiguous() or not v_pools.is_contiguous():
        raise ValueError("pools must be contiguous")
    shape = k_pools.shape if k_pools.dim() == 5 else (1,) + tuple(k_pools.shape)
    layers, num_pages, hkv, page_size, d = shape
    if any(t.dtype != torch.int32 for t in page_tables):
        raise ValueError("page tables must be int32")
    vp = lambda ts: _host_array(ctypes.c_void_p, [_ptr(t) for t in ts])
    arrs = [vp(page_tables), _host_array(ctypes.c_int32, [int(x) for x in prefix_lens]),
            _host_array(ctypes.c_int32, [int(x) for x in n_nodes]), vp(new_pos)]
    cp = [ctypes.cast(a, ctypes.c_void_p) for a in arrs]
    _check(lib().tv_kv_compact_batched_paged(
        batch, _ptr(k_pools), _ptr(v_pools), layers, num_pages * hkv * page_size * d, num_pages,
        hkv, page_size, d, _dtype_code(k_pools), cp[0], cp[1], cp[2], cp[3], _ptr(status),
        _stream(stream, k_pools.device)), "tv_kv_compact_batched_paged")


# ---------------------------------------------------------------- draft side

def expand_workspace(n_frontier: int, vocab: int, w: int, device) -> torch.Tensor:
    """Workspace of tree_expand for these sizes (raises on sizes it rejects)."""
    nbytes = int(lib().tv_expand_workspace_size(n_frontier, vocab, w))
    if nbytes == 0:
        raise TreeVerifyError(TV_ERR_INVALID_ARG, "tv_expand_workspace_size")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def tree_expand(logits: torch.Tensor, frontier: torch.Tensor, cum: torch.Tensor, w: int,
                outs: Optional[dict] = None, workspace: Optional[torch.Tensor] = None,
                status: Optional[torch.Tensor] = None, stream=None) -> dict:
    """One maximum-likelihood expansion: the w best children of the frontier
    nodes by cumulative log-probability.  logits float32 [F][V] (row f for
    tree node frontier[f]), frontier int32 [F], cum float32 [N] (every tree
    node's cumulative log-probability).  Returns (or fills) a dict of device
    tensors parent int32 [w], token int32 [w], score float32 [w]."""
    _need_cuda(logits, frontier, cum)
    nf, vocab = logits.shape
    if logits.dtype != torch.float32 or cum.dtype != torch.float32 or \
            frontier.dtype != torch.int32:
        raise ValueError("dtype mismatch")
    if frontier.numel() != nf or not logits.is_contiguous():
        raise ValueError("shape mismatch")
    if outs is None:
        dev = logits.device
        outs = {"parent": torch.empty(w, dtype=torch.int32, device=dev),
                "token": torch.empty(w, dtype=torch.int32, device=dev),
                "score": torch.empty(w, dtype=torch.float32, device=dev)}
    if workspace is None:
        workspace = expand_workspace(nf, vocab, w, logits.device)
    _check(lib().tv_tree_expand(
        _ptr(logits), vocab, nf, _ptr(frontier), _ptr(cum), cum.numel(), w, _ptr(outs["parent"]),
        _ptr(outs["token"]), _ptr(outs["score"]), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream, logits.device)), "tv_tree_expand")
    return outs


def lm_head_workspace(n_nodes: int, vocab: int, device) -> torch.Tensor:
    """A workspace for lm_head_argmax (bytes, 16-byte aligned)."""
    nbytes = int(lib().tv_lm_head_workspace_size(n_nodes, vocab))
    if nbytes == 0:
        raise TreeVerifyError(TV_ERR_INVALID_ARG, "tv_lm_head_workspace_size")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def lm_head_argmax(hidden: torch.Tensor, weight: torch.Tensor, outs: Optional[dict] = None,
                   workspace: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None, stream=None) -> dict:
    """The target's greedy token at every tree node from its final hidden
    state: am[i] = argmax_v hidden[i] . weight[v] (lowest v on ties), the
    logits never written out.  hidden bf16 [N][d_model], weight bf16
    [V][d_model] (both contiguous).  Returns (or fills) a dict of device
    tensors am int32 [N] and max_logit float32 [N]."""
    _need_cuda(hidden, weight)
    if hidden.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
        raise ValueError("hidden and weight must be bfloat16")
    if hidden.dim() != 2 or weight.dim() != 2 or hidden.shape[1] != weight.shape[1]:
        raise ValueError("shape mismatch")
    if not hidden.is_contiguous() or not weight.is_contiguous():
        raise ValueError("hidden and weight must be contiguous")
    n, d = hidden.shape
    vocab = weight.shape[0]
    if outs is None:
        dev = hidden.device
        outs = {"am": torch.empty(n, dtype=torch.int32, device=dev),
                "max_logit": torch.empty(n, dtype=torch.float32, device=dev)}
    if workspace is None:
        workspace = lm_head_workspace(n, vocab, hidden.device)
    _check(lib().tv_lm_head_argmax(
        _ptr(hidden), _ptr(weight), n, d, vocab, _ptr(outs["am"]), _ptr(outs.get("max_logit")),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream, hidden.device)), "tv_lm_head_argmax")
    return outs


def draft_reroot(parent: torch.Tensor, token: torch.Tensor, cum: torch.Tensor, accepted: dict,
                 prefix_len: int, outs: Optional[dict] = None,
                 status: Optional[torch.Tensor] = None, stream=None) -> dict:
    """The draft tree's re-root map after a verification.  parent, token
    int32 [N] and cum float32 [N] describe the draft tree; `accepted` is the
    dict tree_accept returned for the verified tree (its path, m and
    out_tokens are read on the device).  Returns a dict of device tensors
    new_pos, new_parent, new_token (int32 [N]), new_cum (float32 [N]) and
    n_survivors (int32 [1]); new_pos feeds kv_compact for the draft's cache."""
    _need_cuda(parent, token, cum)
    n = parent.numel()
    if parent.dtype != torch.int32 or token.dtype != torch.int32 or cum.dtype != torch.float32:
        raise ValueError("dtype mismatch")
    if token.numel() != n or cum.numel() != n:
        raise ValueError("shape mismatch")
    if outs is None:
        dev = parent.device
        outs = {"new_pos": torch.empty(n, dtype=torch.int32, device=dev),
                "new_parent": torch.empty(n, dtype=torch.int32, device=dev),
                "new_token": torch.empty(n, dtype=torch.int32, device=dev),
                "new_cum": torch.empty(n, dtype=torch.float32, device=dev),
                "n_survivors": torch.empty(1, dtype=torch.int32, device=dev)}
    _check(lib().tv_draft_reroot(
        _ptr(parent), _ptr(token), _ptr(cum), n, _ptr(accepted["path"]), _ptr(accepted["m"]),
        _ptr(accepted["out_tokens"]), prefix_len, _ptr(outs["new_pos"]), _ptr(outs["new_parent"]),
        _ptr(outs["new_token"]), _ptr(outs["new_cum"]), _ptr(outs["n_survivors"]), _ptr(status),
        _stream(stream, parent.device)), "tv_draft_reroot")
    return outs
