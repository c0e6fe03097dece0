"""qsa_stage_in: a step's inputs copied from host memory by a kernel in the
stream's programmatic chain. The copy is byte-exact, a pageable source is
refused before any launch where the device cannot reach it (and copied where it
can), and a decode step fed through it equals the same step fed from device
tensors bit for bit."""
import math

import pytest
import torch

from indexer_selected_sparse_gb300 import synth as S

pytestmark = pytest.mark.gpu

Q = pytest.importorskip("indexer_selected_sparse_gb300.qsa")


def test_stage_in_copies_bytes_exactly():
    g = torch.Generator().manual_seed(7)
    for n in (16, 4096 + 48, 868352 + 16):
        src = torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g).pin_memory()
        dst = torch.full((n,), 0xA5, dtype=torch.uint8, device="cuda")
        Q.qsa_stage_in(dst, src)
        torch.cuda.synchronize()
        assert torch.equal(dst.cpu(), src), n


def test_stage_in_pageable_source_refused_or_copied():
    # pageable host memory: refused where the device cannot reach it; on systems
    # whose GPU reads pageable host memory (a coherent CPU-GPU link) it is copied
    src = torch.arange(64, dtype=torch.uint8)
    dst = torch.zeros(64, dtype=torch.uint8, device="cuda")
    rc = Q.LIB.qsa_stage_in(dst.data_ptr(), src.data_ptr(), 64, None)
    torch.cuda.synchronize()  # a refusal launches nothing and leaves no error
    assert rc in (Q.QSA_OK, Q.QSA_ERR_INVALID_ARG)
    if rc == Q.QSA_OK:
        assert torch.equal(dst.cpu(), src)


def packed(tensors, device, pin=False):
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(total, dtype=torch.uint8, device=device, pin_memory=pin)
    views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, tensors)]
    return buf, views


def test_decode_step_fed_through_stage_in_matches():
    dev = torch.device("cuda", 0)
    wl = S.workload(2)
    sh = wl.shapes
    cfg = Q.Config.of(sh)
    B, start = 4, 9000
    max_pages = math.ceil((start + 64) / sh.page_size)
    cache = Q.PagedCache(cfg, S.page_table(wl.seed, B, max_pages, False), B * max_pages, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for s in range(B):
        for a in range(0, start, 8192):
            m = min(8192, start - a)
            k, v, ix = S.token_rows(sh, wl.seed, s, torch.arange(a, a + m), device=dev)
            Q.qsa_append(cfg, Q.Rows(torch.tensor([s], device=dev), torch.tensor([a], device=dev, dtype=torch.int32),
                                     m), cache, k, v, ix, status)
    ids = torch.arange(B, dtype=torch.int32, device=dev)
    pos0 = torch.full((B,), start, dtype=torch.int32, device=dev)
    rows_in = [S.token_rows(sh, wl.seed, s, torch.tensor([start]), device=dev) for s in range(B)]
    qs = [S.query_rows(sh, wl.seed, s, torch.tensor([start]), device=dev) for s in range(B)]
    cat = lambda xs: torch.cat(xs).contiguous()
    ins = [cat([r[0] for r in rows_in]), cat([r[1] for r in rows_in]), cat([r[2] for r in rows_in]),
           cat([x[1] for x in qs]), cat([x[2] for x in qs]), cat([x[0] for x in qs])]  # k v ix q_idx w q
    ws = Q.workspace(cfg, B, cache.max_blocks, device=dev)
    one = torch.ones(B, dtype=torch.int32, device=dev)

    def step(k, v, ix, qi, w, q):
        out = torch.empty(B, sh.n_q_heads, sh.head_dim, dtype=torch.bfloat16, device=dev)
        sel = torch.empty(B, cfg.topk, dtype=torch.int32, device=dev)
        nsel = torch.empty(B, dtype=torch.int32, device=dev)
        Q.qsa_decode(cfg, Q.Rows(ids, pos0, 1), cache, k, v, ix, qi, w, q, out, ws, status,
                     sel_out=sel, n_sel_out=nsel)
        return out, sel, nsel

    out_a, sel_a, nsel_a = step(*ins)
    Q.qsa_rewind(cfg, ids, one, cache.ingested, status)
    hbuf, hviews = packed(ins, "cpu", pin=True)
    for hv, t in zip(hviews, ins):
        hv.copy_(t.cpu())
    dbuf, dviews = packed(ins, dev)
    dbuf.zero_()
    Q.qsa_stage_in(dbuf, hbuf)
    out_b, sel_b, nsel_b = step(*dviews)
    torch.cuda.synchronize()
    assert status.item() == 0, Q.qsa_strerror(status.item())
    assert torch.equal(sel_a, sel_b) and torch.equal(nsel_a, nsel_b)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
