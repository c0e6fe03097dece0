"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every entry point include/qsa.h declares, validates
configurations and arguments on the host, and the oracle and the product
never import each other."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qsa.h")


@pytest.fixture(scope="module")
def Q():
    from indexer_selected_sparse_gb300 import build
    if not os.path.exists(build.LIB):
        build.build_library()
    from indexer_selected_sparse_gb300 import qsa
    return qsa


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|int|size_t|unsigned\s+long\s+long)\s*(qsa_\w+)\s*\(",
                                 text, re.M)))


def test_every_declared_symbol_is_exported(Q):
    names = declared_functions()
    assert len(names) >= 9
    lib = ctypes.CDLL(Q.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in qsa.h but not exported"
    assert set(names) == set(Q.EXPORTED)


def test_config_check(Q):
    ok = Q.Config(4, 2048, 64, 128, 32, 4)
    assert Q.qsa_config_check(ok) == Q.QSA_OK
    assert Q.qsa_config_check(Q.Config(4, 256, 4, 64, 8, 1)) == Q.QSA_OK
    bad = [Q.Config(3, 2048, 64, 128, 32, 4),     # ratio not a power of two
           Q.Config(4, 2050, 64, 128, 32, 4),     # budget not a multiple of ratio
           Q.Config(4, 8196, 64, 128, 32, 4),     # K > 2048
           Q.Config(4, 2048, 65, 128, 32, 4),     # too many index heads
           Q.Config(4, 2048, 64, 96, 32, 4),      # d_I
           Q.Config(4, 2048, 64, 128, 32, 3),     # Hkv
           Q.Config(4, 2048, 64, 128, 64, 4),     # group of 16
           Q.Config(4, 2048, 64, 128, 32, 4, head_dim=64),
           Q.Config(4, 2048, 64, 128, 32, 4, page_size=32)]
    for c in bad:
        assert Q.qsa_config_check(c) == Q.QSA_ERR_UNSUPPORTED, c


def test_workspace_bytes(Q):
    c = Q.Config(4, 2048, 64, 128, 32, 4)
    a = Q.qsa_workspace_bytes(c, 32, 8200)
    b = Q.qsa_workspace_bytes(c, 64, 8200)
    assert a > 32 * 8200 * 4 and b > a
    assert Q.qsa_workspace_bytes(Q.Config(3, 2048, 64, 128, 32, 4), 32, 8200) == 0


def test_strerror(Q):
    assert Q.qsa_strerror(0) == "ok"
    assert "ingested" in Q.qsa_strerror(Q.QSA_ERR_DESYNC)
    assert "page" in Q.qsa_strerror(Q.QSA_ERR_CAPACITY)
    assert Q.qsa_strerror(1234) == "unknown status"


def test_null_arguments_rejected_on_host(Q):
    cfg = Q.Config(4, 2048, 64, 128, 32, 4).c()
    lib = Q.LIB
    assert lib.qsa_append(ctypes.byref(cfg), None, None, None, None, None, None, None) == Q.QSA_ERR_INVALID_ARG
    assert lib.qsa_decode(ctypes.byref(cfg), None, None, None, None, None, None, None, None, None, None,
                          None, None, 0, None, None) == Q.QSA_ERR_INVALID_ARG
    rows = Q.qsa_rows(2, 1, None, None, None, 0)
    assert lib.qsa_index_score(ctypes.byref(cfg), ctypes.byref(rows), None, None, None, None, 0, None,
                               None) == Q.QSA_ERR_INVALID_ARG
    assert lib.qsa_rewind(ctypes.byref(cfg), 1, None, None, None, None, None) == Q.QSA_ERR_INVALID_ARG
    # misaligned pointers are rejected before any launch
    cache = Q.qsa_cache(16, 1, 4, 4, 16, 16, 16, 16, 16)
    rows = Q.qsa_rows(1, 1, 16, 16, None, 0)
    assert lib.qsa_append(ctypes.byref(cfg), ctypes.byref(rows), ctypes.byref(cache), 18, 16, 16, 16,
                          None) == Q.QSA_ERR_INVALID_ARG
    # select reads score rows with 16-byte loads: misaligned base or odd stride
    assert lib.qsa_topk_select(ctypes.byref(cfg), ctypes.byref(rows), 20, 1024, 16, 16, 16,
                               None) == Q.QSA_ERR_INVALID_ARG
    assert lib.qsa_topk_select(ctypes.byref(cfg), ctypes.byref(rows), 16, 1022, 16, 16, 16,
                               None) == Q.QSA_ERR_INVALID_ARG
    # too many rows for one launch grid
    rows = Q.qsa_rows(70000, 1, 16, 16, None, 0)
    assert lib.qsa_append(ctypes.byref(cfg), ctypes.byref(rows), ctypes.byref(cache), 16, 16, 16, 16,
                          16) == Q.QSA_ERR_INVALID_ARG


def test_host_capacity_check(Q):
    import numpy as np
    cfg = Q.Config(4, 256, 4, 64, 8, 1).c()
    cache = Q.qsa_cache(16, 1, 4, 4, 16, 16, 16, 16, 16)      # 4 pages x 64 = 256 tokens
    pos = (ctypes.c_int32 * 1)(250)
    rows = Q.qsa_rows(1, 7, 16, 16, ctypes.cast(pos, ctypes.c_void_p), 0)
    assert Q.LIB.qsa_append(ctypes.byref(cfg), ctypes.byref(rows), ctypes.byref(cache), 16, 16, 16, 16,
                            16) == Q.QSA_ERR_CAPACITY


def test_missing_library_fails_loudly(Q, monkeypatch):
    monkeypatch.setattr(Q, "_LIB_PATH", "/nonexistent/libqsa.so")
    with pytest.raises(RuntimeError, match="not built"):
        Q._load()


def test_oracle_and_product_do_not_import_each_other():
    pkg = os.path.join(ROOT, "indexer_selected_sparse_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle", text, re.M), f
                assert "qsa_oracle" not in text, f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith(".py"):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert "indexer_selected_sparse_gb300" not in text, f


def test_pre_indexer_arguments_checked_on_host(Q):
    import torch
    cfg = Q.Config(ratio=4, budget=2048, n_idx_heads=64, idx_dim=128, n_q_heads=32, n_kv_heads=4,
                   head_dim=128, page_size=64)
    rows = Q.Rows(torch.zeros(1, dtype=torch.int32), torch.zeros(1, dtype=torch.int32), 1)
    g = torch.zeros(128)
    q = torch.zeros(1, 64, 128, dtype=torch.bfloat16)
    cases = [(Q.PreIndexer(g, g, 1e-6, 1e4, 32), Q.QSA_ERR_UNSUPPORTED),   # rotary dims not 0 / 64 / d_I
             (Q.PreIndexer(g, g, -1.0, 1e4, 64), Q.QSA_ERR_INVALID_ARG),   # negative epsilon
             (Q.PreIndexer(g, g, 1e-6, 0.0, 64), Q.QSA_ERR_INVALID_ARG)]   # RoPE base must be positive
    for pre, code in cases:
        rc = Q.LIB.qsa_pre_index_q(ctypes.byref(cfg.c()), ctypes.byref(pre.c()), ctypes.byref(rows.c()),
                                   q.data_ptr(), q.data_ptr() + 2, None)
        assert rc == code, (rc, code)
    rc = Q.LIB.qsa_pre_index_q(ctypes.byref(cfg.c()), None, ctypes.byref(rows.c()), q.data_ptr(),
                               q.data_ptr() + 2, None)
    assert rc == Q.QSA_ERR_INVALID_ARG
    assert Q.qsa_workspace_bytes_pre(cfg, 32, 8192) > Q.qsa_workspace_bytes(cfg, 32, 8192)


def test_index_format_checked_and_page_bytes(Q):
    mx = Q.QSA_INDEX_MXFP8
    assert Q.qsa_config_check(Q.Config(4, 2048, 64, 128, 32, 4, index_format=mx)) == Q.QSA_OK
    assert Q.qsa_config_check(Q.Config(8, 1024, 16, 64, 8, 1, index_format=mx)) == Q.QSA_OK
    # 4 blocks per page (ratio 16): the MXFP8 plane is not supported there
    assert Q.qsa_config_check(Q.Config(16, 2048, 64, 128, 32, 4, index_format=mx)) == Q.QSA_ERR_UNSUPPORTED
    assert Q.qsa_config_check(Q.Config(4, 2048, 64, 128, 32, 4, index_format=3)) == Q.QSA_ERR_UNSUPPORTED
    m4 = Q.QSA_INDEX_MXFP4
    assert Q.qsa_config_check(Q.Config(4, 2048, 64, 128, 32, 4, index_format=m4)) == Q.QSA_OK
    assert Q.qsa_config_check(Q.Config(16, 2048, 64, 128, 32, 4, index_format=m4)) == Q.QSA_ERR_UNSUPPORTED
    assert Q.qsa_idxblk_page_bytes(Q.Config(4, 2048, 64, 128, 32, 4, index_format=m4)) == 16 * (64 + 4)
    assert Q.qsa_idxblk_page_bytes(Q.Config(8, 1024, 16, 64, 8, 1, index_format=m4)) == 8 * (32 + 2)
    # page bytes: bf16 bpp * d_I * 2; MXFP8 bpp * (d_I + d_I / 32)
    assert Q.qsa_idxblk_page_bytes(Q.Config(4, 2048, 64, 128, 32, 4)) == 16 * 128 * 2
    assert Q.qsa_idxblk_page_bytes(Q.Config(4, 2048, 64, 128, 32, 4, index_format=mx)) == 16 * 132
    assert Q.qsa_idxblk_page_bytes(Q.Config(8, 1024, 16, 64, 8, 1, index_format=mx)) == 8 * 66
    assert Q.qsa_idxblk_page_bytes(Q.Config(3, 2048, 64, 128, 32, 4)) == 0
    # the MXFP8 step rounds its queries inside the scorer: no extra workspace
    bf = Q.qsa_workspace_bytes(Q.Config(4, 2048, 64, 128, 32, 4), 32, 8200)
    m8 = Q.qsa_workspace_bytes(Q.Config(4, 2048, 64, 128, 32, 4, index_format=mx), 32, 8200)
    assert m8 == bf
    cfg = Q.ctypes.byref(Q.Config(4, 2048, 64, 128, 32, 4).c())
    assert Q.LIB.qsa_quantize_index_q(cfg, 0, None, None, None) == Q.QSA_OK      # nothing to do
    assert Q.LIB.qsa_quantize_index_q(cfg, 3, None, None, None) == Q.QSA_ERR_INVALID_ARG
    assert Q.LIB.qsa_quantize_index_q(cfg, -1, None, None, None) == Q.QSA_ERR_INVALID_ARG


def test_local_window_checked_and_sizes_grow(Q):
    base = Q.Config(4, 2048, 64, 128, 32, 4)
    win = Q.Config(4, 2048, 64, 128, 32, 4, local_window=128)
    assert Q.qsa_config_check(win) == Q.QSA_OK
    assert Q.qsa_config_check(Q.Config(4, 2048, 64, 128, 32, 4, local_window=-1)) == Q.QSA_ERR_UNSUPPORTED
    assert Q.qsa_config_check(Q.Config(4, 2048, 64, 128, 32, 4, local_window=16385)) == Q.QSA_ERR_UNSUPPORTED
    # the split plan covers budget + W + ratio - 1 tokens
    assert Q.qsa_max_attend_tokens(win) >= 2048 + 128 + 3
    assert Q.qsa_max_attend_tokens(base) >= 2048 + 3
    assert Q.qsa_max_attend_tokens(win) > Q.qsa_max_attend_tokens(base)
    assert Q.qsa_workspace_bytes(win, 32, 8200) > Q.qsa_workspace_bytes(base, 32, 8200)


def test_attention_options_checked_on_host(Q):
    cfg = Q.Config(4, 2048, 64, 128, 32, 4)
    c = ctypes.byref(cfg.c())
    lib = Q.LIB
    cache = Q.qsa_cache(16, 1, 4, 4, 16, 16, 16, 16, 16)      # 4 pages of 64 tokens, fake aligned pointers
    rows = Q.qsa_rows(1, 1, 16, 16, None, 0)

    def opts(eps=1e-6, theta=1e4, rot=64, gate=None):
        return Q.qsa_attn_options(16, 16, eps, theta, rot, gate)

    def decode(o, ws_bytes=1 << 30):
        return lib.qsa_decode_ex(c, None, ctypes.byref(o), ctypes.byref(rows), ctypes.byref(cache), 16, 16, 16,
                                 16, 16, 16, None, None, 16, 16, ws_bytes, 16, None)

    cases = [(opts(eps=-1.0), Q.QSA_ERR_INVALID_ARG),          # epsilon below zero
             (opts(eps=float("nan")), Q.QSA_ERR_INVALID_ARG),
             (opts(theta=0.0), Q.QSA_ERR_INVALID_ARG),         # RoPE base must be positive
             (opts(rot=32), Q.QSA_ERR_UNSUPPORTED),            # rotary dims 0, 64 or D
             (opts(gate=18), Q.QSA_ERR_INVALID_ARG)]           # the gate is read with 16-byte loads
    for o, code in cases:
        assert lib.qsa_append_ex(c, None, ctypes.byref(o), ctypes.byref(rows), ctypes.byref(cache), 16, 16, 16,
                                 16, None) == code
        assert decode(o) == code
    # the step's prepared main queries live in the workspace: the plain size is refused before any launch
    plain = Q.qsa_workspace_bytes(cfg, 1, 64)
    ex = Q.qsa_workspace_bytes_ex(cfg, 1, 64)
    assert ex >= plain + 32 * 128 * 2
    assert decode(opts(), plain) == Q.QSA_ERR_WORKSPACE
    # without a query norm (gate and key options only) the bar is the plain size: one byte less is refused
    # (a size that passes would go on to launch kernels, which these fake pointers must never reach)
    assert decode(Q.qsa_attn_options(None, 16, 1e-6, 1e4, 64, 16), plain - 1) == Q.QSA_ERR_WORKSPACE


def test_mrope_arguments_checked_on_host(Q):
    cfg = Q.Config(4, 2048, 64, 128, 32, 4)
    c = ctypes.byref(cfg.c())
    lib = Q.LIB
    # rows at 250 + 7 > 256 tokens: a call that passes every MRoPE check stops at the host capacity
    # check (QSA_ERR_CAPACITY), so none of these fake pointers ever reaches a kernel
    pos = (ctypes.c_int32 * 1)(250)
    over = ctypes.cast(pos, ctypes.c_void_p)
    rows = Q.qsa_rows(1, 7, 16, 16, over, 0, None)
    rows_mis = Q.qsa_rows(1, 7, 16, 16, over, 0, 18)            # triples not 4-byte aligned
    no_pool = Q.qsa_cache(16, 1, 4, 4, 16, 16, 16, 16, 16)       # 4 pages x 64 tokens
    pool = Q.qsa_cache(16, 1, 4, 4, 16, 16, 16, 16, 16, 16)      # with a block-position pool

    def pre(sec, rot=64):
        return Q.qsa_pre_indexer(16, 16, 1e-6, 1e4, rot, Q._SEC3(*sec))

    def append(p, r, cache):
        return lib.qsa_append_pre(c, ctypes.byref(p), ctypes.byref(r), ctypes.byref(cache), 16, 16, 16, 16, None)

    # a section is three non-negative pair counts adding up to rotary_dim / 2
    for sec, rot in (((11, 11, 11), 64), ((-1, 17, 16), 64), ((11, 11, 10), 0), ((22, 22, 20), 64)):
        assert append(pre(sec, rot), rows, pool) == Q.QSA_ERR_INVALID_ARG, sec
    # keys pooled at stored triples need the cache's block-position pool; triples are int32-aligned
    assert append(pre((11, 11, 10)), rows, no_pool) == Q.QSA_ERR_INVALID_ARG
    assert append(pre((11, 11, 10)), rows_mis, pool) == Q.QSA_ERR_INVALID_ARG
    assert append(pre((11, 11, 10)), rows, pool) == Q.QSA_ERR_CAPACITY          # every MRoPE check passed
    assert append(pre((0, 0, 0)), rows, no_pool) == Q.QSA_ERR_CAPACITY          # plain RoPE needs no pool
    assert append(pre((32, 0, 0), 64), rows, pool) == Q.QSA_ERR_CAPACITY       # temporal only is a section

    # attention options: the same section rule; keys turn at their own row's triple, no pool needed
    def attn(sec):
        return Q.qsa_attn_options(16, 16, 1e-6, 1e4, 64, None, Q._SEC3(*sec))

    def append_ex(a, r, cache):
        return lib.qsa_append_ex(c, None, ctypes.byref(a), ctypes.byref(r), ctypes.byref(cache), 16, 16, 16, 16,
                                 None)
    assert append_ex(attn((11, 11, 11)), rows, no_pool) == Q.QSA_ERR_INVALID_ARG
    assert append_ex(attn((11, 11, 10)), rows_mis, no_pool) == Q.QSA_ERR_INVALID_ARG
    assert append_ex(attn((11, 11, 10)), rows, no_pool) == Q.QSA_ERR_CAPACITY


def test_wait_limit_hook_clamps_and_restores(Q):
    """The failure-path test hook (no GPU needed): 0 restores 1 s, values clamp to
    [1 us, 10 s], and each call returns the previous limit."""
    first = Q.qsa_set_wait_limit_ns(0)
    assert Q.qsa_set_wait_limit_ns(5) == 1_000_000_000
    assert Q.qsa_set_wait_limit_ns(20_000_000_000) == 1_000        # 5 ns clamped up to 1 us
    assert Q.qsa_set_wait_limit_ns(0) == 10_000_000_000            # clamped down to 10 s
    assert Q.qsa_set_wait_limit_ns(first) == 1_000_000_000
    Q.qsa_set_wait_limit_ns(0)


def test_stage_in_arguments_checked_on_host(Q):
    """qsa_stage_in refuses null or misaligned pointers and sizes that are not a
    multiple of 16 before touching CUDA; a zero-byte copy is a no-op."""
    buf = ctypes.create_string_buffer(256)
    a16 = (ctypes.addressof(buf) + 15) // 16 * 16
    lib = Q.LIB
    assert lib.qsa_stage_in(None, a16, 16, None) == Q.QSA_ERR_INVALID_ARG
    assert lib.qsa_stage_in(a16, None, 16, None) == Q.QSA_ERR_INVALID_ARG
    assert lib.qsa_stage_in(a16 + 4, a16, 16, None) == Q.QSA_ERR_INVALID_ARG
    assert lib.qsa_stage_in(a16, a16 + 8, 16, None) == Q.QSA_ERR_INVALID_ARG
    assert lib.qsa_stage_in(a16, a16, 24, None) == Q.QSA_ERR_INVALID_ARG
    assert lib.qsa_stage_in(a16, a16, 0, None) == Q.QSA_OK
