"""GPU parity of the always-kept local window (local_window = W: every row also
attends to its last W visible tokens, a union with the top-k set) against the
CPU oracle on the same seeded inputs. Selections are unchanged by the window
and must match bit-exactly; outputs within the bf16 gates. Covers windows that
cut a selected block (W not a multiple of the ratio), windows past the whole
prefix (dense), verify rows, the batch-32 x 32k shape, and a reused selection."""
import numpy as np
import pytest
import torch

from indexer_selected_sparse_gb300 import synth as S
from oracle import qsa_oracle as O
from tests.gpu_harness import GpuState, OracleSeq, bits, compare_row
from tests.test_gpu_reuse import close, reuse_step

pytestmark = pytest.mark.gpu


def small_wl(ratio, budget, h_i, d_i, hq, hkv, prefixes, R=1, seed=13):
    sh = S.Shapes(ratio, budget, h_i, d_i, hq, hkv, 128, 64)
    return S.Workload("window", seed, sh, list(prefixes), R, contiguous_pages=False)


CASES = {
    # ratio, budget, H_I, d_I, Hq, Hkv, prefixes, R, window
    "r4_B256_W128": (4, 256, 16, 128, 16, 2, [300, 4000, 9001, 130, 259, 260], 1, 128),
    "r4_B256_W10_cuts_blocks": (4, 256, 16, 128, 16, 2, [2000, 5001, 5002, 5003], 1, 10),
    "r8_B512_W4096_dense": (8, 512, 8, 64, 8, 1, [3000, 4095, 600], 1, 4096),
    "r4_B128_verify_W64": (4, 128, 64, 128, 32, 4, [2000, 7000], 3, 64),
    "r2_B64_W1": (2, 64, 4, 64, 8, 1, [500, 777], 2, 1),
}


@pytest.mark.parametrize("name", list(CASES))
def test_window_every_row(name):
    r, b, hi, di, hq, hkv, pre, R, W = CASES[name]
    wl = small_wl(r, b, hi, di, hq, hkv, pre, R)
    g = GpuState(wl, extra_tokens=8, local_window=W)
    g.append_prefix(chunk=3000)
    pos0 = list(wl.prefixes)
    res = g.decode(pos0, R)
    g.check_status()
    sel = res["sel"].cpu().numpy(); nsel = res["n_sel"].cpu().numpy(); out = bits(res["out"])
    for i, s in enumerate(g.slots):
        orc = OracleSeq(wl, s, pos0[i] + R)
        for j in range(R):
            row = i * R + j
            ref = orc.row(pos0[i] + j, window=W)
            compare_row(out[row], sel[row], int(nsel[row]), ref, g.cfg.topk)


def test_window_batch32_prefix32k_sampled_rows():
    wl = S.workload(2)
    g = GpuState(wl, extra_tokens=8, local_window=128)
    g.append_prefix()
    sampled = [0, 11, 31]
    oracles = {s: OracleSeq(wl, s, wl.prefixes[0] + 2) for s in sampled}
    pos0 = list(wl.prefixes)
    for step in range(2):
        res = g.decode(pos0, 1)
        g.check_status()
        sel = res["sel"].cpu().numpy(); nsel = res["n_sel"].cpu().numpy(); out = bits(res["out"])
        for s in sampled:
            ref = oracles[s].row(pos0[s], window=128)
            assert len(ref["tokens"]) > 2049          # the window added tokens the top-k left out
            compare_row(out[s], sel[s], int(nsel[s]), ref, g.cfg.topk)
        pos0 = [p + 1 for p in pos0]


def test_window_with_a_reused_selection():
    wl = S.workload(2)
    g = GpuState(wl, slots=[2, 19], local_window=96)
    g.wl = S.Workload(wl.name, wl.seed, wl.shapes, [wl.prefixes[0]] * 2, 1)
    g.append_prefix()
    p = wl.prefixes[0]
    res0 = g.decode([p] * 2, 1)
    g.check_status()
    sel0, nsel0 = res0["sel"].clone(), res0["n_sel"].clone()
    oracles = {s: OracleSeq(wl, s, p + 4) for s in g.slots}
    for d in (1, 3):
        if d == 3:
            reuse_step(g, [p + 2] * 2, sel0, nsel0, [p] * 2)   # step 2, not checked
            g.check_status()
        out, _ = reuse_step(g, [p + d] * 2, sel0, nsel0, [p] * 2)
        g.check_status()
        for i, s in enumerate(g.slots):
            orc = oracles[s]
            q, _, _ = S.query_rows(wl.shapes, wl.seed, s, torch.tensor([p + d]))
            sel = sel0[i, : int(nsel0[i])].cpu().numpy().astype(np.int64)
            orc.fill_kv(O.token_set(sel, (p + 1) // wl.shapes.ratio, p + d + 1, wl.shapes.ratio, 96))
            ref = O.attend_row_reused(orc.st, p + d, sel, p, bits(q[0]), window=96)
            close(bits(out[i]), ref)
