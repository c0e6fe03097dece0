"""qsa_gather_attn_static: the gather-attention entry point for callers that
cannot allocate device memory (it keeps its split scratch in a fixed array
inside the library). Checked through the C ABI against qsa_gather_attn with a
caller workspace, bit for bit, on two calls in a row with different inputs, so
that anything the first call leaves in the shared array would show in the
second; the first call's outputs are also compared with the CPU oracle.

This file is collected last on purpose: it must pass both alone in a fresh
process and after every other test."""
import numpy as np
import pytest
import torch

from indexer_selected_sparse_gb300 import synth as S
from tests.gpu_harness import GpuState, OracleSeq, bits, compare_row

pytestmark = pytest.mark.gpu


def test_static_scratch_matches_workspace_entry_twice():
    sh = S.SHAPES_MAIN
    wl = S.Workload("no-alloc", 11, sh, [5000, 9000, 2050, 40000, 700, 33000], 1)
    g = GpuState(wl, extra_tokens=16)
    g.append_prefix()
    Q = g.Q
    pos0 = list(wl.prefixes)
    oracles = {s: OracleSeq(wl, s, pos0[i] + 1) for i, s in enumerate(g.slots)}
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
        # the same kernel over the same inputs: equal bit for bit
        assert np.array_equal(bits(got), bits(ref)), f"call {call}: static-scratch output differs"
        if call == 0:
            sel_h, nsel_h, out_h = sel.cpu().numpy(), nsel.cpu().numpy(), bits(got)
            for i, s in enumerate(g.slots):
                compare_row(out_h[i], sel_h[i], int(nsel_h[i]), oracles[s].row(pos0[i]), g.cfg.topk)
        pos0 = [p + 1 for p in pos0]


def test_static_scratch_rejects_too_many_rows():
    """The largest accepted row count, found by bisection on the library's own
    answer: that many rows run, one more returns QSA_ERR_WORKSPACE (before any
    launch). At Hq = 32 and budget 2048 the header documents 106 rows."""
    sh = S.SHAPES_MAIN
    Q = pytest.importorskip("indexer_selected_sparse_gb300.qsa")
    cfg = Q.Config.of(sh)
    hi_rows = 4096
    ids = torch.arange(hi_rows, dtype=torch.int32, device="cuda")
    cache = Q.PagedCache(cfg, torch.zeros(hi_rows, 1, dtype=torch.int32), 1)
    q = torch.zeros(hi_rows, sh.n_q_heads, 128, dtype=torch.bfloat16, device="cuda")
    sel = torch.zeros(hi_rows, cfg.topk, dtype=torch.int32, device="cuda")
    nsel = torch.zeros(hi_rows, dtype=torch.int32, device="cuda")   # rows at position 0: one token each
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def accepted(n):
        rows = Q.Rows(ids[:n], torch.zeros(n, dtype=torch.int32, device="cuda"), 1)
        try:
            Q.qsa_gather_attn_static(cfg, rows, cache, q[:n], sel[:n], nsel[:n], out[:n], status)
        except Q.QsaError as e:
            assert e.code == Q.QSA_ERR_WORKSPACE
            return False
        return True

    assert accepted(1) and not accepted(hi_rows)
    lo, hi = 1, hi_rows                        # accepted(lo), not accepted(hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if accepted(mid):
            lo = mid
        else:
            hi = mid
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert lo == 106, f"the fixed array holds {lo} rows, not the documented 106"
    # a row at position 0 attends to its own token only: the output is that token's V (zeros here)
    assert not torch.isnan(out[:lo].float()).any()
