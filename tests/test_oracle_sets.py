"""CPU check of the every-row selection helper the full-size GPU parity tests
use: its selections (sequences regenerated in spawned workers, index side only)
equal the oracle's attend_row selections of the same rows, built in this
process with K/V, for decode rows, verify rows and rows after a rewind whose
re-appended tokens were drawn with a new epoch."""
import numpy as np
import torch

from indexer_selected_sparse_gb300 import synth as S
from oracle import qsa_oracle as O
from tests.oracle_sets import assert_every_row, oracle_selections


def _oracle_rows(wl, seq, n_tokens, epoch_from, positions):
    sh = wl.shapes
    pos = np.arange(n_tokens)
    ep = np.zeros(n_tokens, np.int64)
    for p, e in epoch_from:
        ep[pos >= p] = e
    k = np.empty((n_tokens, sh.n_kv_heads, sh.head_dim), np.uint16)
    v = np.empty_like(k)
    ix = np.empty((n_tokens, sh.idx_dim), np.uint16)
    b = lambda t: t.contiguous().view(torch.int16).numpy().astype(np.uint16)
    for e in np.unique(ep):
        m = np.nonzero(ep == e)[0]
        kk, vv, ii = S.token_rows(sh, wl.seed, seq, torch.from_numpy(pos[m]), epoch=int(e))
        k[m], v[m], ix[m] = b(kk), b(vv), b(ii)
    st = O.SeqState(sh.ratio, sh.n_kv_heads, sh.head_dim, sh.idx_dim, n_tokens)
    st.append(0, k, v, ix)
    sel, nsel = [], []
    for p in positions:
        e = int(ep[p]) if p < n_tokens else 0
        q, qi, w = S.query_rows(sh, wl.seed, seq, torch.tensor([p]), epoch=e)
        ref = O.attend_row(st, p, b(qi[0]), w[0].numpy(), b(q[0]), sh.topk)
        sel.append(O.padded_selection(ref["sel"], sh.topk))
        nsel.append(len(ref["sel"]))
    return np.stack(sel), np.array(nsel)


def test_every_row_helper_equals_attend_row():
    sh = S.Shapes(4, 64, 4, 64, 4, 1, 128, 64)          # K = 16, inert bound 67
    wl = S.Workload("small", 11, sh, [300, 66, 67], 3)
    cases = [(0, 303, [(0, 0)], [300, 301, 302]),        # verify rows, selection active
             (1, 69, [(0, 0)], [66, 67, 68]),            # across the inert bound
             (2, 90, [(0, 0), (80, 1)], [80, 85, 89])]   # rows drawn after a rewind (epoch 1)
    want = oracle_selections(wl, cases)
    rows, sels, nsels, n = {}, [], [], 0
    for seq, n_tok, ef, pos in cases:
        s, c = _oracle_rows(wl, seq, n_tok, ef, pos)
        sels.append(s)
        nsels.append(c)
        rows[seq] = list(range(n, n + len(pos)))
        n += len(pos)
    assert assert_every_row(np.concatenate(sels), np.concatenate(nsels), rows, want) == 9
    # the dense row (66 + 1 visible tokens, 16 blocks) selects all, the next ones K
    assert want[1][1].tolist() == [16, 16, 16]
    # a planted difference is caught
    bad = np.concatenate(sels).copy()
    bad[4, 3] += 1
    try:
        assert_every_row(bad, np.concatenate(nsels), rows, want)
    except AssertionError:
        pass
    else:
        raise AssertionError("a wrong selection passed")
