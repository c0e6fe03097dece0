"""The oracle's selected block set for every query row of a full-size workload.

Scores of the workloads' inputs are exact (integer index keys and queries,
power-of-two head weights), so the oracle's selection of each row is the one
correct set, and every row of a GPU step can be checked against it, not only
sampled ones. Only the index side is needed: each sequence's raw index keys are
regenerated from the seeded generator on the host, pooled by the oracle's
SeqState, scored by block_scores and ranked by select_blocks, one row at a
time. Nothing here reads GPU data.

Sequences are spread over a process pool started with `spawn` (a pool forked
after the parent has touched the GPU can hang), a few hundred rows per job.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

_POOL: Optional[ProcessPoolExecutor] = None
ROWS_PER_JOB = 512


def _pool() -> ProcessPoolExecutor:
    global _POOL
    if _POOL is None:
        n = max(1, min(16, os.cpu_count() or 1))
        _POOL = ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))
    return _POOL


def _epochs(epoch_from: Sequence[Tuple[int, int]], positions: np.ndarray) -> np.ndarray:
    out = np.zeros(len(positions), np.int64)
    for p, e in epoch_from:
        out[positions >= p] = e
    return out


def _job(args):
    """One sequence, some of its rows: padded selections [n, K] and n_sel [n]."""
    import torch

    from indexer_selected_sparse_gb300 import synth as S
    from oracle import qsa_oracle as O

    torch.set_num_threads(1)
    wl, seq, n_tokens, epoch_from, positions, index_format = args
    sh = wl.shapes
    irange = wl.extra.get("int_range", (-8, 8))
    pos_all = np.arange(n_tokens, dtype=np.int64)
    ep = _epochs(epoch_from, pos_all)
    raw = np.empty((n_tokens, sh.idx_dim), np.uint16)
    for e in np.unique(ep):
        idx = np.nonzero(ep == e)[0]
        _, _, ix = S.token_rows(S.Shapes(sh.ratio, sh.budget, 1, sh.idx_dim, 1, 1, 8, sh.page_size), wl.seed, seq,
                                torch.from_numpy(pos_all[idx]), epoch=int(e), int_range=irange)
        raw[idx] = ix.contiguous().view(torch.int16).numpy().astype(np.uint16)
    st = O.SeqState(sh.ratio, 1, 8, sh.idx_dim, n_tokens)
    z = np.zeros((n_tokens, 1, 8), np.uint16)
    st.append(0, z, z, raw)
    score_fn = {"bf16": O.block_scores, "mxfp8": O.block_scores_mxfp8, "mxfp4": O.block_scores_mxfp4}[index_format]
    positions = np.asarray(positions, np.int64)
    sel = np.empty((len(positions), sh.topk), np.int64)
    nsel = np.empty(len(positions), np.int64)
    for r, p in enumerate(positions):
        e = int(_epochs(epoch_from, np.array([p]))[0])
        _, qi, w = S.query_rows(sh, wl.seed, seq, torch.tensor([int(p)]), epoch=e, int_range=irange)
        n_blk = (int(p) + 1) // sh.ratio
        if n_blk > sh.topk:
            qb = qi[0].contiguous().view(torch.int16).numpy().astype(np.uint16)
            s = O.select_blocks(score_fn(qb, w[0].numpy(), st.idx_blk[:n_blk]), sh.topk)
        else:
            s = O.select_blocks(np.zeros(n_blk), sh.topk)
        sel[r] = O.padded_selection(s, sh.topk)
        nsel[r] = len(s)
    return sel, nsel


def oracle_selections(wl, requests: List[Tuple[int, int, Sequence[Tuple[int, int]], Sequence[int]]],
                      index_format: str = "bf16") -> Dict[int, Tuple[np.ndarray, np.ndarray]]:
    """requests: (seq, n_tokens, epoch_from, positions) per sequence, where the
    sequence holds tokens 0..n_tokens-1 (epoch_from as in the harness's History:
    positions >= p were drawn with epoch e) and `positions` are the query rows.
    Returns {seq: (sel [n, K] ascending, -1 padded; n_sel [n])} in the order of
    `positions`."""
    jobs, keys = [], []
    for seq, n_tokens, epoch_from, positions in requests:
        positions = list(positions)
        for a in range(0, len(positions), ROWS_PER_JOB):
            jobs.append((wl, seq, n_tokens, list(epoch_from), positions[a:a + ROWS_PER_JOB], index_format))
            keys.append(seq)
    results = list(_pool().map(_job, jobs))
    out: Dict[int, Tuple[list, list]] = {}
    for seq, (s, n) in zip(keys, results):
        a, b = out.setdefault(seq, ([], []))
        a.append(s)
        b.append(n)
    return {seq: (np.concatenate(a), np.concatenate(b)) for seq, (a, b) in out.items()}


def assert_every_row(sel_gpu: np.ndarray, nsel_gpu: np.ndarray, row_of: Dict[int, Sequence[int]],
                     want: Dict[int, Tuple[np.ndarray, np.ndarray]]) -> int:
    """Compare the GPU's selection of every listed row (row_of: seq -> the GPU
    rows of its positions, in request order) with the oracle's, bit for bit.
    Returns the number of rows checked."""
    n = 0
    for seq, rows in row_of.items():
        ws, wn = want[seq]
        rows = np.asarray(rows, np.int64)
        got_n = nsel_gpu[rows].astype(np.int64)
        bad = np.nonzero(got_n != wn)[0]
        assert len(bad) == 0, f"seq {seq}: n_sel differs at rows {rows[bad][:8].tolist()}"
        got = sel_gpu[rows].astype(np.int64)
        bad = np.nonzero((got != ws).any(axis=1))[0]
        assert len(bad) == 0, (f"seq {seq}: selected block set differs from the oracle at "
                               f"{len(bad)} rows, first {rows[bad][:8].tolist()}")
        n += len(rows)
    return n


class StepLog:
    """The selections of every row of a series of steps, for one comparison
    with the oracle's at the end: per sequence, its rows in step order."""

    def __init__(self):
        self.sel, self.nsel = [], []
        self.rows = {}     # seq -> GPU rows in the concatenation
        self.pos = {}      # seq -> positions of those rows
        self.n = 0

    def add(self, res, seqs, pos0, R):
        self.sel.append(res["sel"].cpu().numpy())
        self.nsel.append(res["n_sel"].cpu().numpy())
        for i, s in enumerate(seqs):
            for j in range(R):
                self.rows.setdefault(s, []).append(self.n + i * R + j)
                self.pos.setdefault(s, []).append(pos0[i] + j)
        self.n += len(seqs) * R

    def check(self, wl, hist=None, index_format="bf16"):
        """Every logged row against the oracle (hist: seq -> History of the
        epochs its tokens were drawn with; index_format: the plane the keys are
        scored in). Returns the number of rows."""
        req = [(s, max(p) + 1, (hist[s].epoch_from if hist else [(0, 0)]), p) for s, p in self.pos.items()]
        want = oracle_selections(wl, req, index_format)
        return assert_every_row(np.concatenate(self.sel), np.concatenate(self.nsel), self.rows, want)
