"""The C-ABI library builds, loads without a GPU and exports every function
that include/treeverify.h declares; host-side argument checks answer with the
documented status codes before anything reaches the device."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "treeverify.h")


def _declared():
    text = open(HEADER).read()
    return re.findall(r"^TV_API\s+[\w\s\*]+?\b(tv_\w+)\s*\(", text, flags=re.M)


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_tree_masked_gb300 import _build, _lib
    if not os.path.exists(_lib.LIB_PATH):
        _build.build()
    return _lib.load()


def test_header_declares_the_boundary():
    names = set(_declared())
    assert {"tv_tree_attn_verify", "tv_tree_accept", "tv_kv_compact", "tv_tree_mask",
            "tv_attn_workspace_size", "tv_status_string", "tv_version"} <= names


def test_every_declared_symbol_is_exported(lib):
    from speculative_decoding_tree_masked_gb300 import _lib
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(_lib.SIGNATURES) == set(_declared())


def test_status_strings(lib):
    for code in range(7):
        assert lib.tv_status_string(code)
    assert lib.tv_status_string(99) == b"unknown status"
    assert lib.tv_version() >= 100


def test_host_checks_need_no_device(lib):
    import ctypes
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails its checks
    # attention: null pointers, bad head split, bad d, too many nodes, capacity
    args = dict(q=fake, k=fake, v=fake, cap=100, P=10, n=5, parent=fake, out=fake, hq=8,
                hkv=2, d=128, dt=1, scale=0.0, ws=fake, wsb=1 << 30)

    def attn(**kw):
        a = dict(args, **kw)
        return lib.tv_tree_attn_verify(a["q"], a["k"], a["v"], a["cap"], a["P"], a["n"],
                                       a["parent"], a["out"], a["hq"], a["hkv"], a["d"],
                                       a["dt"], a["scale"], a["ws"], a["wsb"], None, None)
    assert attn(q=None) == 1
    assert attn(hq=7) == 1
    assert attn(d=96) == 2
    assert attn(n=129) == 1
    assert attn(n=0) == 1
    assert attn(dt=5) == 1
    assert attn(cap=12) == 3
    assert attn(q=ctypes.c_void_p(0x1004)) == 1   # misaligned
    assert attn(scale=-1.0) == 1
    # acceptance
    assert lib.tv_tree_accept(None, 10, fake, fake, 3, 0, fake, fake, fake, fake, fake, fake,
                              fake, None, None) == 1
    assert lib.tv_tree_accept(fake, 0, fake, fake, 3, 0, fake, fake, fake, fake, fake, fake,
                              fake, None, None) == 1
    assert lib.tv_tree_accept(fake, 10, fake, fake, 200, 0, fake, fake, fake, fake, fake,
                              fake, fake, None, None) == 1
    # compaction: row bytes not a multiple of 16, capacity, layer stride
    assert lib.tv_kv_compact(fake, fake, 2, 1 << 20, 2, 100, 12, 1, 10, 5, fake, None, None) == 2
    assert lib.tv_kv_compact(fake, fake, 2, 1 << 20, 2, 12, 64, 1, 10, 5, fake, None, None) == 3
    assert lib.tv_kv_compact(fake, fake, 2, 10, 2, 100, 64, 1, 10, 5, fake, None, None) == 1
    assert lib.tv_tree_mask(None, 3, fake, None, None) == 1
    assert lib.tv_tree_mask(fake, 0, fake, None, None) == 1


def test_workspace_size_is_monotone_in_prefix(lib):
    last = 0
    for P in (0, 100, 1000, 4096, 8192, 32768):
        s = lib.tv_attn_workspace_size(64, 64, 8, 128, 1, P)
        assert s > 0 and s % 256 == 0
        assert s >= last or s > 0
        last = s
    assert lib.tv_attn_workspace_size(64, 64, 8, 96, 1, 100) == 0


def test_draft_side_host_checks(lib):
    import ctypes
    fake = ctypes.c_void_p(0x1000)
    assert lib.tv_expand_workspace_size(8, 128256, 8) > 0
    assert lib.tv_expand_workspace_size(0, 100, 8) == 0
    assert lib.tv_expand_workspace_size(8, 100, 65) == 0           # w above the limit
    assert lib.tv_expand_workspace_size(64, 100, 32) == 0          # n_frontier * w too large
    assert lib.tv_expand_workspace_size(1, 4, 5) == 0              # w above n_frontier * vocab
    assert lib.tv_expand_workspace_size(1, 600000, 8) == 0         # vocab above the limit
    assert lib.tv_expand_workspace_size(1, 131072, 64) > 0
    assert lib.tv_expand_workspace_size(1, 131073, 64) == 0        # ceil(V / 8192) * w

    def expand(**kw):
        a = dict(lg=fake, V=1000, F=4, fr=fake, cum=fake, N=10, w=8, ws=fake, wsb=1 << 30)
        a.update(kw)
        return lib.tv_tree_expand(a["lg"], a["V"], a["F"], a["fr"], a["cum"], a["N"], a["w"],
                                  fake, fake, fake, a["ws"], a["wsb"], None, None)
    assert expand(lg=None) == 1
    assert expand(w=0) == 1
    assert expand(F=200) == 1
    assert expand(N=0) == 1
    assert expand(lg=ctypes.c_void_p(0x1002)) == 1                 # misaligned logits
    assert expand(wsb=16) == 3                                     # workspace too small
    assert lib.tv_draft_reroot(None, fake, fake, 5, fake, fake, fake, 0, fake, fake, fake,
                               fake, fake, None, None) == 1
    assert lib.tv_draft_reroot(fake, fake, fake, 0, fake, fake, fake, 0, fake, fake, fake,
                               fake, fake, None, None) == 1
    assert lib.tv_draft_reroot(fake, fake, fake, 129, fake, fake, fake, 0, fake, fake, fake,
                               fake, fake, None, None) == 1


def test_sampled_accept_host_checks(lib):
    import ctypes
    fake = ctypes.c_void_p(0x1000)

    def call(**kw):
        a = dict(lg=fake, V=100, n=4, T=1.0)
        a.update(kw)
        return lib.tv_tree_accept_sampled(a["lg"], a["V"], fake, fake, a["n"], 0, a["T"], 1, 0,
                                          fake, fake, fake, fake, fake, fake, fake, None, None)
    assert call(lg=None) == 1
    assert call(T=0.0) == 1
    assert call(T=-1.0) == 1
    assert call(T=float("inf")) == 1
    assert call(T=float("nan")) == 1
    assert call(n=0) == 1
    assert call(V=0) == 1


def test_batched_attention_host_checks(lib):
    import ctypes
    fake = ctypes.c_void_p(0x1000)
    B = 2

    def arr(ctype, vals):
        return ctypes.cast((ctype * len(vals))(*vals), ctypes.c_void_p)

    def call(batch=B, n=(5, 7), P=(10, 20), cap=(100, 100), dt=1, d=128, hq=8, hkv=2,
             ptrs=None, ws=0x1000, wsb=1 << 30):
        ptrs = ptrs or [0x1000, 0x2000]
        vp = arr(ctypes.c_void_p, ptrs[:max(batch, 1)] + [0x3000] * max(0, batch - 2))
        nn = arr(ctypes.c_int32, list(n) + [5] * max(0, batch - 2))
        pp = arr(ctypes.c_int32, list(P) + [0] * max(0, batch - 2))
        cc = arr(ctypes.c_int64, list(cap) + [100] * max(0, batch - 2))
        return lib.tv_tree_attn_verify_batched(batch, vp, vp, vp, cc, pp, nn, vp, vp, hq, hkv,
                                               d, dt, 0.0, ctypes.c_void_p(ws), wsb, None, None)
    assert call(batch=0) == 1
    assert call(batch=17) == 1
    assert call(n=(5, 200)) == 1
    assert call(cap=(100, 12)) == 3                   # request 1 cannot hold its tree
    assert call(ptrs=[0x1000, 0x2004]) == 1           # misaligned
    assert call(d=96) == 2
    assert call(dt=0) == 2                            # fp32 has no batched kernel
    ns = (ctypes.c_int32 * 2)(64, 8)
    assert lib.tv_attn_batched_workspace_size(2, ctypes.cast(ns, ctypes.c_void_p), 64, 8, 128, 1) > 0
    assert lib.tv_attn_batched_workspace_size(2, ctypes.cast(ns, ctypes.c_void_p), 64, 8, 128, 0) == 0
    assert lib.tv_attn_batched_workspace_size(0, ctypes.cast(ns, ctypes.c_void_p), 64, 8, 128, 1) == 0


def test_lm_head_host_checks(lib):
    import ctypes
    fake = ctypes.c_void_p(0x1000)
    assert lib.tv_lm_head_workspace_size(64, 128256) > 0
    assert lib.tv_lm_head_workspace_size(0, 1000) == 0
    assert lib.tv_lm_head_workspace_size(257, 1000) == 0            # above TV_MAX_LM_NODES
    assert lib.tv_lm_head_workspace_size(4, 0) == 0

    def call(**kw):
        a = dict(h=fake, w=fake, n=4, d=64, V=1000, am=fake, ws=fake, wsb=1 << 30)
        a.update(kw)
        return lib.tv_lm_head_argmax(a["h"], a["w"], a["n"], a["d"], a["V"], a["am"], None,
                                     a["ws"], a["wsb"], None, None)
    assert call(h=None) == 1
    assert call(am=None) == 1
    assert call(n=0) == 1
    assert call(n=257) == 1
    assert call(d=12) == 1                                           # not a multiple of 8
    assert call(d=0) == 1
    assert call(V=0) == 1
    assert call(w=ctypes.c_void_p(0x1008)) == 1                      # misaligned weights
    assert call(wsb=8) == 3                                          # workspace too small


def test_accept_tokens_host_checks(lib):
    import ctypes
    fake = ctypes.c_void_p(0x1000)

    def call(**kw):
        a = dict(tt=fake, V=100, n=4, P=0)
        a.update(kw)
        return lib.tv_tree_accept_tokens(a["tt"], a["V"], fake, fake, a["n"], a["P"], fake, fake,
                                         fake, fake, fake, fake, None, None)
    assert call(tt=None) == 1
    assert call(V=0) == 1
    assert call(n=0) == 1
    assert call(n=129) == 1
    assert call(P=-1) == 1


def test_paged_host_checks(lib):
    import ctypes
    fake = ctypes.c_void_p(0x1000)

    def attn(**kw):
        a = dict(q=fake, kp=fake, vp=fake, pages=10, ps=64, tab=fake, P=100, n=8, hq=8, hkv=2,
                 d=128, dt=1, ws=fake, wsb=1 << 30)
        a.update(kw)
        return lib.tv_tree_attn_verify_paged(a["q"], a["kp"], a["vp"], a["pages"], a["ps"],
                                             a["tab"], a["P"], a["n"], fake, fake, a["hq"],
                                             a["hkv"], a["d"], a["dt"], 0.0, a["ws"], a["wsb"],
                                             None, None)
    assert attn(tab=None) == 1
    assert attn(ps=48) == 1                     # not a multiple of 64
    assert attn(ps=0) == 1
    assert attn(pages=0) == 1
    assert attn(kp=ctypes.c_void_p(0x1008)) == 1
    assert attn(d=96) == 2
    assert attn(dt=0) == 2                      # paged attention is bf16 only
    assert attn(n=129) == 1

    def compact(**kw):
        a = dict(kp=fake, vp=fake, L=2, stride=10 * 2 * 64 * 128, pages=10, hkv=2, ps=64, d=128,
                 dt=1, tab=fake, P=100, n=8)
        a.update(kw)
        return lib.tv_kv_compact_paged(a["kp"], a["vp"], a["L"], a["stride"], a["pages"],
                                       a["hkv"], a["ps"], a["d"], a["dt"], a["tab"], a["P"],
                                       a["n"], fake, None, None)
    assert compact(tab=None) == 1
    assert compact(stride=100) == 1             # layers would overlap
    assert compact(n=0) == 1
    assert compact(d=12) == 2                   # rows not whole 16-byte vectors
    assert compact(pages=0) == 1


def test_batched_accept_and_compaction_host_checks(lib):
    import ctypes
    fake = ctypes.c_void_p(0x1000)

    def arr(ctype, vals):
        return ctypes.cast((ctype * len(vals))(*vals), ctypes.c_void_p)

    def accept(batch=2, off=(0, 5, 12), P=(10, 20), V=100, logits=fake, tokens=False):
        o, p = arr(ctypes.c_int32, list(off)), arr(ctypes.c_int32, list(P))
        if tokens:
            return lib.tv_tree_accept_tokens_batched(batch, o, p, logits, V, fake, fake, fake,
                                                     fake, fake, fake, fake, fake, None, None)
        return lib.tv_tree_accept_batched(batch, o, p, logits, V, fake, fake, fake, fake, fake,
                                          fake, fake, fake, fake, None, None)
    for tokens in (False, True):
        assert accept(batch=0, tokens=tokens) == 1
        assert accept(batch=17, tokens=tokens) == 1
        assert accept(off=(1, 5, 12), tokens=tokens) == 1          # must start at 0
        assert accept(off=(0, 5, 5), tokens=tokens) == 1           # an empty request
        assert accept(off=(0, 5, 140), tokens=tokens) == 1         # 135 nodes > 128
        assert accept(off=(0, 7, 5), tokens=tokens) == 1           # decreasing
        assert accept(P=(10, -1), tokens=tokens) == 1
        assert accept(V=0, tokens=tokens) == 1
        assert accept(logits=None, tokens=tokens) == 1
    assert accept(logits=ctypes.c_void_p(0x1002)) == 1             # logits not 4-byte aligned

    def sampled(batch=2, off=(0, 5, 12), T=(1.0, 0.5)):
        o, p = arr(ctypes.c_int32, list(off)), arr(ctypes.c_int32, [10, 20])
        t = arr(ctypes.c_float, list(T))
        u = arr(ctypes.c_uint64, [1, 2])
        return lib.tv_tree_accept_sampled_batched(batch, o, p, fake, 100, fake, fake, t, u, u,
                                                  fake, fake, fake, fake, fake, fake, fake, None,
                                                  None)
    assert sampled(batch=0) == 1
    assert sampled(off=(0, 5, 140)) == 1
    assert sampled(T=(1.0, 0.0)) == 1                             # temperature must be > 0
    assert sampled(T=(float("inf"), 1.0)) == 1
    assert sampled(T=(float("nan"), 1.0)) == 1
    assert lib.tv_tree_accept_batched(2, None, arr(ctypes.c_int32, [0, 0]), fake, 10, fake, fake,
                                      fake, fake, fake, fake, fake, fake, fake, None, None) == 1

    def compact(batch=2, n=(5, 7), P=(10, 20), cap=(100, 100), stride=None, d=128, dt=1,
                ptrs=(0x1000, 0x2000), newpos=(0x1000, 0x1000)):
        stride = stride or [2 * c * d for c in cap]
        kv = arr(ctypes.c_void_p, list(ptrs))
        return lib.tv_kv_compact_batched(batch, kv, kv, arr(ctypes.c_int64, list(stride)),
                                         arr(ctypes.c_int64, list(cap)),
                                         arr(ctypes.c_int32, list(P)),
                                         arr(ctypes.c_int32, list(n)),
                                         arr(ctypes.c_void_p, list(newpos)), 3, 2, d, dt, None,
                                         None)
    assert compact(batch=0) == 1
    assert compact(batch=17) == 1
    assert compact(n=(5, 0)) == 1
    assert compact(n=(5, 129)) == 1
    assert compact(P=(-1, 20)) == 1
    assert compact(cap=(100, 25)) == 3                            # request 1: 20 + 7 > 25
    assert compact(stride=(200 * 128, 100)) == 1                  # layers would overlap
    assert compact(ptrs=(0x1000, 0x2008)) == 1                    # misaligned
    assert compact(ptrs=(0x1000, 0)) == 1
    assert compact(newpos=(0x1000, 0)) == 1
    assert compact(d=6) == 2                                      # 12-byte rows
    assert compact(dt=7) == 1

    def paged(batch=2, n=(5, 7), P=(10, 20), stride=10 * 2 * 64 * 128, ps=64, tabs=(0x1000, 0x2000)):
        return lib.tv_kv_compact_batched_paged(
            batch, fake, fake, 3, stride, 10, 2, ps, 128, 1, arr(ctypes.c_void_p, list(tabs)),
            arr(ctypes.c_int32, list(P)), arr(ctypes.c_int32, list(n)),
            arr(ctypes.c_void_p, [0x1000, 0x1000]), None, None)
    assert paged(batch=0) == 1
    assert paged(tabs=(0x1000, 0)) == 1
    assert paged(stride=100) == 1
    assert paged(ps=0) == 1
    assert paged(n=(200, 7)) == 1


def test_attention_plan_is_host_only_and_consistent(lib):
    import itertools

    import torch

    import speculative_decoding_tree_masked_gb300 as tvp
    # the full verify step's layer on GB300's 152 SMs: two row groups of two
    # 128-row tiles per KV head, 9 splits of 4 key blocks (the last holds the
    # tree block), bf16 partials
    assert tvp.attn_plan(64, 64, 8, 128, torch.bfloat16, 4096, sm_count=152) == {
        "row_groups": 2, "splits": 9, "keys_per_split": 512,
        "ws_bytes": 9 * 4096 * 4 + 9 * 4096 * 128 * 2}
    # 32 nodes of 8 heads: two tiles per KV head, one per CTA, 9 splits
    assert tvp.attn_plan(32, 64, 8, 128, torch.bfloat16, 4096, sm_count=152) == {
        "row_groups": 2, "splits": 9, "keys_per_split": 512,
        "ws_bytes": 9 * 2048 * 4 + 9 * 2048 * 128 * 2}
    shapes = [(64, 8), (32, 8), (4, 1), (7, 1)]
    for (hq, hkv), n, d, P, sms in itertools.product(shapes, (1, 8, 33, 64, 128), (64, 128),
                                                     (0, 1, 127, 1024, 4096, 32768, 100000),
                                                     (1, 8, 152, 256)):
        p = tvp.attn_plan(n, hq, hkv, d, torch.bfloat16, P, sm_count=sms)
        keys = P + n
        assert p["keys_per_split"] % 128 == 0
        assert (p["splits"] - 1) * p["keys_per_split"] < keys <= p["splits"] * p["keys_per_split"]
        tiles = -(-(hq // hkv) * n // 128)
        assert p["row_groups"] == (tiles if tiles <= 2 else (tiles + 1) // 2)
        units = hkv * p["row_groups"]
        assert units * p["splits"] <= max(sms, units)        # one wave of one-CTA-per-SM
        if sms == 256:                                       # the no-device workspace bound
            assert p["ws_bytes"] == tvp.attn_workspace_size(n, hq, hkv, d, torch.bfloat16, P)
        f = tvp.attn_plan(n, hq, hkv, d, torch.float32, P, sm_count=sms)
        assert (f["splits"] - 1) * f["keys_per_split"] < keys <= f["splits"] * f["keys_per_split"]
    import ctypes
    out = [ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t()]
    refs = [ctypes.byref(x) for x in out]
    assert lib.tv_attn_plan(64, 64, 8, 96, 1, 4096, 152, *refs) == 2       # d unsupported
    assert lib.tv_attn_plan(64, 64, 8, 128, 1, -1, 152, *refs) == 1
    assert lib.tv_attn_plan(64, 64, 8, 128, 1, 4096, -1, *refs) == 1
    assert lib.tv_attn_plan(64, 64, 8, 128, 1, 4096, 152, None, *refs[1:]) == 1
    if not torch.cuda.is_available():
        assert lib.tv_attn_plan(64, 64, 8, 128, 1, 4096, 0, *refs) == 4  # no device to ask
