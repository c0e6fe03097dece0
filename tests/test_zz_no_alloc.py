"""qsa_gather_attn_static: the gather-attention entry point for callers that
cannot allocate device memory (it keeps its split scratch in a fixed array
inside the library). Checked through the C ABI against qsa_gather_attn with a
caller workspace, on two calls in a row with different inputs, so that
anything the first call leaves in the shared array would show in the second.

This file is collected last on purpose: it must pass both alone in a fresh
process and after every other test."""
import numpy as np
import pytest
import torch

from indexer_selected_sparse_gb300 import synth as S
from tests.gpu_harness import SEL_TOL_MAXABS, SEL_TOL_RELL2, GpuState, bits

pytestmark = pytest.mark.gpu


def close(a, b):
    x = a.float().cpu().numpy().astype(np.float64)
    y = b.float().cpu().numpy().astype(np.float64)
    maxabs = np.abs(x - y).max()
    rel = np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-30)
    return maxabs <= SEL_TOL_MAXABS and rel <= SEL_TOL_RELL2, (maxabs, rel)


def test_static_scratch_matches_workspace_entry_twice():
    sh = S.SHAPES_MAIN
    wl = S.Workload("no-alloc", 11, sh, [5000, 9000, 2050, 40000, 700, 33000], 1)
    g = GpuState(wl, extra_tokens=16)
    g.append_prefix()
    Q = g.Q
    pos0 = list(wl.prefixes)
    for call in range(2):
        res = g.decode(pos0, 1)              # appends the step's tokens, gives q / sel / n_sel
        g.check_status()
        rows = g.rows(pos0, 1)
        q, sel, nsel = res["inputs"]["q"], res["sel"], res["n_sel"]
        ref = torch.empty_like(res["out"])
        Q.qsa_gather_attn(g.cfg, rows, g.cache, q, sel, nsel, ref, g.ws, g.status)
        got = torch.full_like(res["out"], float("nan"))
        Q.qsa_gather_attn_static(g.cfg, rows, g.cache, q, sel, nsel, got, g.status)
        torch.cuda.synchronize()
        g.check_status()
        ok, err = close(got, ref)
        assert ok, f"call {call}: static-scratch output differs from the workspace entry: {err}"
        pos0 = [p + 1 for p in pos0]


def test_static_scratch_rejects_too_many_rows():
    sh = S.SHAPES_MAIN
    Q = pytest.importorskip("indexer_selected_sparse_gb300.qsa")
    cfg = Q.Config.of(sh)
    n_split = -(-(sh.budget + sh.ratio - 1) // 112)      # fixed 112-slot splits of the widest row
    per_row = n_split * sh.n_q_heads * (128 + 2) * 4      # its split partials (m, l, acc)
    too_many = Q.QSA_STATIC_SCRATCH_BYTES // per_row + 1
    ids = torch.arange(too_many, dtype=torch.int32, device="cuda")
    rows = Q.Rows(ids, torch.zeros_like(ids), 1)
    cache = Q.PagedCache(cfg, torch.zeros(too_many, 1, dtype=torch.int32), 1)
    q = torch.zeros(too_many, sh.n_q_heads, 128, dtype=torch.bfloat16, device="cuda")
    sel = torch.zeros(too_many, cfg.topk, dtype=torch.int32, device="cuda")
    nsel = torch.zeros(too_many, dtype=torch.int32, device="cuda")
    with pytest.raises(Q.QsaError) as e:
        Q.qsa_gather_attn_static(cfg, rows, cache, q, sel, nsel, torch.empty_like(q))
    assert e.value.code == Q.QSA_ERR_WORKSPACE
