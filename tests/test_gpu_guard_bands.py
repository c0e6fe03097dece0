"""Guard bands: every buffer the path writes sits between two bands of
poisoned bytes, and after appends, fused decode and verify steps, the separate
stages and a rewind, every band must still hold its poison. An out-of-range
write anywhere (a pool, the workspace, an output, the status word, the
positions) shows up as a changed band. This stands in for a memory checker,
which this pool does not offer. The bands are 4 KiB, a multiple of 256 bytes,
so every buffer keeps the alignment its allocation would have."""
import math

import numpy as np
import pytest
import torch

from indexer_selected_sparse_gb300 import synth as S
from tests.gpu_harness import GpuState

pytestmark = pytest.mark.gpu

BAND = 4096
POISON = 0xA5


class Guarded:
    """Buffers carved from larger allocations, a poisoned band on each side."""

    def __init__(self, device):
        self.device = device
        self.raw = {}

    def make(self, name, shape, dtype, init=None):
        n = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((BAND + n + BAND,), POISON, dtype=torch.uint8, device=self.device)
        inner = raw[BAND:BAND + n].view(dtype).view(shape)
        if init is not None:
            inner.copy_(init)
        self.raw[name] = raw
        return inner

    def check(self, when):
        torch.cuda.synchronize()
        for name, raw in self.raw.items():
            for side, band in (("before", raw[:BAND]), ("after", raw[-BAND:])):
                bad = (band != POISON).nonzero()
                assert bad.numel() == 0, f"{when}: {int(bad.numel())} bytes {side} {name} changed"


def guarded_state(wl, index_format=0, local_window=0):
    g = GpuState(wl, extra_tokens=8, index_format=index_format, local_window=local_window)
    G = Guarded(g.device)
    for name in ("k_pool", "v_pool", "idxraw_pool", "idxblk_pool", "ingested"):
        t = getattr(g.cache, name)
        setattr(g.cache, name, G.make(name, t.shape, t.dtype, t))
    g.status = G.make("status", (1,), torch.int32, torch.zeros(1, dtype=torch.int32))
    return g, G


def guarded_step(g, G, pos0, R, tag):
    """One fused step with every output, the workspace and the positions guarded."""
    Q = g.Q
    n = len(g.slots) * R
    inp = g.step_inputs(pos0, R)
    pos = G.make(f"pos0_{tag}", (len(g.slots),), torch.int32, torch.tensor(pos0, dtype=torch.int32))
    rows = Q.Rows(torch.tensor(g.slots, dtype=torch.int32, device=g.device), pos, R, advance=True)
    out = G.make(f"out_{tag}", (n, g.sh.n_q_heads, g.sh.head_dim), torch.bfloat16)
    sel = G.make(f"sel_{tag}", (n, g.cfg.topk), torch.int32)
    nsel = G.make(f"nsel_{tag}", (n,), torch.int32)
    nbytes = Q.qsa_workspace_bytes(g.cfg, n, g.cache.max_blocks)
    ws = G.make(f"ws_{tag}", (nbytes,), torch.uint8)
    Q.qsa_decode(g.cfg, rows, g.cache, inp["k"], inp["v"], inp["idx"], inp["q_idx"], inp["w"], inp["q"],
                 out, ws, g.status, sel_out=sel, n_sel_out=nsel)
    G.check(f"fused step {tag}")
    g.check_status()
    assert pos.cpu().tolist() == [p + R for p in pos0]   # advanced in place, inside its bands
    return inp


CASES = {
    # ratio, budget, H_I, d_I, Hq, Hkv, prefixes, index format, window
    "bf16_r4": (4, 256, 16, 128, 16, 2, [3000, 130, 4097], 0, 0),
    "mxfp8_r4": (4, 256, 16, 128, 16, 2, [3000, 257], 1, 0),
    "mxfp4_r8_dI64": (8, 256, 16, 64, 8, 1, [2000, 4097], 2, 0),
    "window_r4": (4, 256, 16, 128, 16, 2, [3000, 300], 0, 96),
}


@pytest.mark.parametrize("name", list(CASES))
def test_bands_survive_every_entry_point(name):
    r, b, hi, di, hq, hkv, pre, fmt, W = CASES[name]
    sh = S.Shapes(r, b, hi, di, hq, hkv, 128, 64)
    wl = S.Workload("guard", 23, sh, pre, 3, contiguous_pages=False)
    g, G = guarded_state(wl, fmt, W)
    g.append_prefix(chunk=1000)
    G.check("prefix appends")
    # decode (R = 1) then verify (R = 3), with device-side position advance
    guarded_step(g, G, list(pre), 1, "decode")
    guarded_step(g, G, [p + 1 for p in pre], 3, "verify")
    # the separate stages, into guarded buffers, for the verify step's last row (already ingested)
    Q = g.Q
    last = [p + 3 for p in pre]
    rows = Q.Rows(torch.tensor(g.slots, dtype=torch.int32, device=g.device),
                  torch.tensor(last, dtype=torch.int32, device=g.device), 1)
    inp = g.step_inputs(last, 1)
    n = len(g.slots)
    ld = (g.cache.max_blocks + 3) // 4 * 4
    scores = G.make("scores", (n, ld), torch.float32)
    sel = G.make("sel", (n, g.cfg.topk), torch.int32)
    nsel = G.make("nsel", (n,), torch.int32)
    out = G.make("out", (n, sh.n_q_heads, sh.head_dim), torch.bfloat16)
    ws = G.make("ws", (Q.qsa_workspace_bytes(g.cfg, n, g.cache.max_blocks),), torch.uint8)
    Q.qsa_index_score(g.cfg, rows, g.cache, inp["q_idx"], inp["w"], scores, ld, g.status)
    Q.qsa_topk_select(g.cfg, rows, scores, ld, sel, nsel, g.status)
    Q.qsa_gather_attn(g.cfg, rows, g.cache, inp["q"], sel, nsel, out, ws, g.status)
    G.check("separate stages")
    g.check_status()
    # rewind the verify rows
    Q.qsa_rewind(g.cfg, torch.tensor(g.slots, dtype=torch.int32, device=g.device),
                 torch.full((n,), 3, dtype=torch.int32, device=g.device), g.cache.ingested, g.status)
    G.check("rewind")
    g.check_status()
    ing = g.cache.ingested.cpu().numpy()
    assert np.array_equal(ing[g.slots], np.array(pre) + 1)
