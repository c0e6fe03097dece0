"""The index-score kernel's bounded waits, made to run out ("Atlas Flash-Next
defect investigations", Report A, Defect 4: an error reaches the caller, it is
never laundered into success).

With the wait limit shortened to 1 us (qsa_set_wait_limit_ns), the scorer's
first waits (keys still on their way from HBM) expire: the CTAs record
QSA_ERR_TIMEOUT in the status word, let their own copies and tensor-core work
land (a bounded 2 ms), free their tensor memory and return. Nothing faults and
nothing hangs: the next step on the same stream, with the default limit, runs
normally and matches the oracle on every row."""
import numpy as np
import pytest
import torch

from indexer_selected_sparse_gb300 import synth as S
from tests.gpu_harness import GpuState, OracleSeq, bits, compare_row

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_the_next_step_is_sound():
    wl0 = S.workload(2)
    sh = wl0.shapes
    wl = S.Workload(wl0.name, wl0.seed, sh, [32768] * 4, 1)
    g = GpuState(wl, extra_tokens=16)
    g.append_prefix()
    Q = g.Q
    pos0 = list(wl.prefixes)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=g.device)
    flush.fill_(1)                      # the keys come from HBM, not L2
    torch.cuda.synchronize()
    prev = Q.qsa_set_wait_limit_ns(1000)
    try:
        g.decode(pos0, 1)
        torch.cuda.synchronize()
    finally:
        Q.qsa_set_wait_limit_ns(0)
    assert prev == 1_000_000_000
    assert int(g.status.item()) == Q.QSA_ERR_TIMEOUT
    # the step still appended its tokens and committed the counters
    pos0 = [p + 1 for p in pos0]
    assert g.cache.ingested.cpu().tolist() == pos0
    g.status.zero_()
    res = g.decode(pos0, 1)
    g.check_status()
    sel, nsel, out = res["sel"].cpu().numpy(), res["n_sel"].cpu().numpy(), bits(res["out"])
    for i, s in enumerate(g.slots):
        orc = OracleSeq(wl, s, pos0[i] + 1)
        compare_row(out[i], sel[i], int(nsel[i]), orc.row(pos0[i]), g.cfg.topk)
