"""Test plumbing shared by the GPU parity tests: builds a workload's paged GPU
state through the library's own append, runs steps through the C ABI, and
builds the CPU oracle's logical state for sampled sequences from the same
seeded generator (never from GPU data)."""
from __future__ import annotations

import math
from typing import Dict, List, Optional

import numpy as np
import torch

from indexer_selected_sparse_gb300 import synth as S
from oracle import qsa_oracle as O

SEL_TOL_MAXABS = 2e-2
SEL_TOL_RELL2 = 1e-3


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns (host numpy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().astype(np.uint16)


def bf16_value(b: np.ndarray) -> np.ndarray:
    return O.bf16_bits_to_f64(b)


def block_pool_index(bpp: int, d_idx: int) -> np.ndarray:
    """[bpp, d_idx] element offsets of a block-pool page in the library's tiled
    page layout (tiles of min(bpp, 8) rows x 8 values, row-group major, then
    8-value chunk, row-major inside a tile), as the C ABI header documents."""
    g = min(bpp, 8)
    rr = np.arange(bpp)[:, None]
    d = np.arange(d_idx)[None, :]
    return ((rr // g) * (d_idx // 8) + d // 8) * (8 * g) + (rr % g) * 8 + d % 8


def e4m3_values() -> np.ndarray:
    """Value of every E4M3 byte (256 entries), from the bit definition: sign |
    4-bit exponent (bias 7) | 3-bit mantissa; exponent field 0 is subnormal
    (m/8 * 2^-6); 0x7F / 0xFF are NaN."""
    v = np.empty(256)
    for code in range(256):
        e, m = (code >> 3) & 15, code & 7
        mag = m / 8 * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        if e == 15 and m == 7:
            mag = np.nan
        v[code] = -mag if code & 0x80 else mag
    return v


def mxfp8_page_index(bpp: int, d_idx: int):
    """Byte offsets of a block-pool page in the MXFP8 format the C ABI header
    documents: elements [bpp, d_idx] in 8-block x 16-byte core matrices, then
    scales [bpp, d_idx / 32]."""
    rr = np.arange(bpp)[:, None]
    d = np.arange(d_idx)[None, :]
    el = ((rr // 8) * (d_idx // 16) + d // 16) * 128 + (rr % 8) * 16 + d % 16
    c = np.arange(d_idx // 32)[None, :]
    sc = bpp * d_idx + rr * (d_idx // 32) + c
    return el, sc


class History:
    """Per-sequence record of which epoch wrote each position (positions
    re-appended after a rewind carry fresh random rows)."""

    def __init__(self):
        self.epoch_from: List[tuple] = []   # (first_pos, epoch): positions >= first_pos use epoch

    def set(self, first_pos: int, epoch: int):
        self.epoch_from = [(p, e) for (p, e) in self.epoch_from if p < first_pos]
        self.epoch_from.append((first_pos, epoch))

    def epochs(self, positions: np.ndarray) -> np.ndarray:
        out = np.zeros(len(positions), np.int64)
        for p, e in self.epoch_from:
            out[positions >= p] = e
        return out


def gen_token_rows(sh, seed, seq, positions, epochs, device, int_range=(-8, 8)):
    """K, V, idx rows for positions with per-position epochs."""
    positions = np.asarray(positions, np.int64)
    epochs = np.asarray(epochs, np.int64)
    ks, vs, iis, order = [], [], [], []
    for e in np.unique(epochs):
        sel = np.nonzero(epochs == e)[0]
        k, v, i = S.token_rows(sh, seed, seq, torch.from_numpy(positions[sel]), epoch=int(e), device=device,
                               int_range=int_range)
        ks.append(k); vs.append(v); iis.append(i); order.append(sel)
    order = np.concatenate(order)
    inv = torch.from_numpy(np.argsort(order, kind="stable")).to(device)
    return torch.cat(ks)[inv], torch.cat(vs)[inv], torch.cat(iis)[inv]


class GpuState:
    """A workload's cache on the GPU, filled through qsa_append."""

    def __init__(self, wl: S.Workload, extra_tokens: int = 64, contiguous: Optional[bool] = None,
                 page_seed: Optional[int] = None, device: str = "cuda", slots: Optional[List[int]] = None,
                 index_format: int = 0, local_window: int = 0, mrope: bool = False):
        from indexer_selected_sparse_gb300 import qsa as Q
        self.Q = Q
        self.wl = wl
        self.sh = wl.shapes
        self.irange = wl.extra.get("int_range", (-8, 8))
        self.cfg = Q.Config.of(self.sh, index_format, local_window)
        self.device = device
        P = self.sh.page_size
        need = max(wl.prefixes) + wl.rows_per_seq + extra_tokens
        self.max_pages = math.ceil(need / P)
        self.slots = list(range(wl.n_seq)) if slots is None else list(slots)
        n_slots = max(self.slots) + 1
        contiguous = wl.contiguous_pages if contiguous is None else contiguous
        pt = S.page_table(wl.seed if page_seed is None else page_seed, n_slots, self.max_pages, contiguous)
        self.cache = Q.PagedCache(self.cfg, pt, n_slots * self.max_pages, device=device, mrope=mrope)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.hist: Dict[int, History] = {s: History() for s in self.slots}
        for s in self.slots:
            self.hist[s].set(0, 0)
        self.ws = Q.workspace(self.cfg, max(wl.n_rows, 1), self.cache.max_blocks, device=device)

    def seq_of(self, i: int) -> int:
        return self.slots[i]

    def append_prefix(self, chunk: int = 8192):
        Q = self.Q
        for i, s in enumerate(self.slots):
            n = self.wl.prefixes[i]
            start = 0
            while start < n:
                m = min(chunk, n - start)
                pos = np.arange(start, start + m)
                k, v, ix = gen_token_rows(self.sh, self.wl.seed, s, pos, self.hist[s].epochs(pos), self.device, self.irange)
                rows = Q.Rows(torch.tensor([s], device=self.device), torch.tensor([start], device=self.device), m)
                Q.qsa_append(self.cfg, rows, self.cache, k, v, ix, self.status)
                start += m
        torch.cuda.synchronize()
        self.check_status()

    def check_status(self, expect: int = 0):
        st = int(self.status.item())
        assert st == expect, f"device status {st} ({self.Q.qsa_strerror(st)}), expected {expect}"

    def step_inputs(self, pos0: List[int], R: int, seqs: Optional[List[int]] = None):
        """Append rows and query rows of a step, sequence-major, on the device."""
        seqs = self.slots if seqs is None else seqs
        ks, vs, iis, qs, qis, ws = [], [], [], [], [], []
        for s, p in zip(seqs, pos0):
            pos = np.arange(p, p + R)
            ep = self.hist[s].epochs(pos)
            k, v, ix = gen_token_rows(self.sh, self.wl.seed, s, pos, ep, self.device, self.irange)
            assert ep.min() == ep.max(), "a step's rows share one epoch"
            q, qi, w = S.query_rows(self.sh, self.wl.seed, s, torch.from_numpy(pos), epoch=int(ep.max()),
                                    device=self.device, int_range=self.irange)
            ks.append(k); vs.append(v); iis.append(ix); qs.append(q); qis.append(qi); ws.append(w)
        cat = lambda xs: torch.cat(xs).contiguous()
        return dict(k=cat(ks), v=cat(vs), idx=cat(iis), q=cat(qs), q_idx=cat(qis), w=cat(ws))

    def rows(self, pos0: List[int], R: int, seqs: Optional[List[int]] = None, host_pos: bool = True):
        seqs = self.slots if seqs is None else seqs
        p = torch.tensor(pos0, dtype=torch.int32)
        return self.Q.Rows(torch.tensor(seqs, dtype=torch.int32, device=self.device), p.to(self.device), R,
                           pos0_host=p if host_pos else None)

    def decode(self, pos0: List[int], R: int, seqs: Optional[List[int]] = None, inputs=None):
        Q = self.Q
        seqs = self.slots if seqs is None else seqs
        inp = inputs or self.step_inputs(pos0, R, seqs)
        rows = self.rows(pos0, R, seqs)
        n = len(seqs) * R
        out = torch.empty(n, self.sh.n_q_heads, self.sh.head_dim, dtype=torch.bfloat16, device=self.device)
        sel = torch.empty(n, self.cfg.topk, dtype=torch.int32, device=self.device)
        nsel = torch.empty(n, dtype=torch.int32, device=self.device)
        ws = self.ws if n <= self.wl.n_rows else Q.workspace(self.cfg, n, self.cache.max_blocks, self.device)
        Q.qsa_decode(self.cfg, rows, self.cache, inp["k"], inp["v"], inp["idx"], inp["q_idx"], inp["w"],
                     inp["q"], out, ws, self.status, sel_out=sel, n_sel_out=nsel)
        torch.cuda.synchronize()
        return dict(out=out, sel=sel, n_sel=nsel, inputs=inp)

    def rewind(self, n_drop: List[int], seqs: Optional[List[int]] = None, new_epoch: int = 1):
        Q = self.Q
        seqs = self.slots if seqs is None else seqs
        ing = self.cache.ingested.cpu()
        Q.qsa_rewind(self.cfg, torch.tensor(seqs, dtype=torch.int32, device=self.device),
                     torch.tensor(n_drop, dtype=torch.int32, device=self.device), self.cache.ingested,
                     self.status)
        torch.cuda.synchronize()
        for s, n in zip(seqs, n_drop):
            if n > 0:
                self.hist[s].set(int(ing[s]) - n, new_epoch)

    # pools read back through the page table (test-side decoding)
    def logical_blocks(self, s: int, n_blk: int) -> np.ndarray:
        sh = self.sh
        bpp = sh.page_size // sh.ratio
        pt = self.cache.page_table[s].cpu().numpy()
        b = np.arange(n_blk)
        pages = pt[b // bpp]
        blk = self.cache.idxblk_pool.view(torch.int16).cpu().numpy().astype(np.uint16)
        return blk[pages[:, None], block_pool_index(bpp, sh.idx_dim)[b % bpp]]

    def logical_blocks_mxfp8(self, s: int, n_blk: int):
        """The MXFP8 plane's blocks 0..n_blk-1 of sequence s: E4M3 element values
        [n_blk, d_I] and scale exponents [n_blk, d_I / 32]."""
        sh = self.sh
        bpp = sh.page_size // sh.ratio
        pt = self.cache.page_table[s].cpu().numpy()
        b = np.arange(n_blk)
        pages = pt[b // bpp]
        plane = self.cache.idxblk_pool.cpu().numpy()
        el, sc = mxfp8_page_index(bpp, sh.idx_dim)
        elems = e4m3_values()[plane[pages[:, None], el[b % bpp]]]
        exps = plane[pages[:, None], sc[b % bpp]].astype(np.int64) - 127
        return elems, exps

    def logical_blocks_mxfp4(self, s: int, n_blk: int):
        """The MXFP4 plane's blocks 0..n_blk-1 of sequence s: E2M1 element values
        [n_blk, d_I] (decoded from the nibbles: sign | 2-bit exponent, bias 1 |
        1-bit mantissa) and scale exponents [n_blk, d_I / 32]."""
        sh = self.sh
        bpp = sh.page_size // sh.ratio
        d = sh.idx_dim
        pt = self.cache.page_table[s].cpu().numpy()
        b = np.arange(n_blk)
        pages = pt[b // bpp]
        plane = self.cache.idxblk_pool.cpu().numpy()
        rr = (b % bpp)[:, None]
        dd = np.arange(d)[None, :]
        byte = ((rr // 8) * (d // 32) + dd // 32) * 128 + (rr % 8) * 16 + (dd % 32) // 2
        raw = plane[pages[:, None], byte]
        nib = np.where(dd % 2 == 0, raw & 15, raw >> 4).astype(np.int64)
        e, m = (nib >> 1) & 3, nib & 1
        mag = np.where(e == 0, 0.5 * m, (1 + m / 2) * np.exp2(e - 1))
        elems = np.where(nib & 8, -mag, mag)
        sc = bpp * d // 2 + rr * (d // 32) + np.arange(d // 32)[None, :]
        exps = plane[pages[:, None], sc].astype(np.int64) - 127
        return elems, exps

    def logical_rows(self, pool: torch.Tensor, s: int, positions: np.ndarray) -> np.ndarray:
        P = self.sh.page_size
        pt = self.cache.page_table[s].cpu().numpy()
        arr = pool.view(torch.int16)
        pages = torch.from_numpy(pt[positions // P]).long().to(arr.device)
        offs = torch.from_numpy(positions % P).long().to(arr.device)
        return arr[pages, offs].cpu().numpy().astype(np.uint16)


class OracleSeq:
    """The oracle's logical state of one sequence, built from the generator.

    K/V rows are generated only for the tokens a row attends to (filled in
    before the oracle attends); the index keys are generated for every
    position, so pooling and scoring see the whole sequence."""

    def __init__(self, wl: S.Workload, seq: int, n_tokens: int, hist: Optional[History] = None,
                 lazy_kv: bool = True):
        self.wl, self.sh, self.seq = wl, wl.shapes, seq
        self.irange = wl.extra.get("int_range", (-8, 8))
        self.hist = hist or History()
        if not self.hist.epoch_from:
            self.hist.set(0, 0)
        sh = self.sh
        self.st = O.SeqState(sh.ratio, sh.n_kv_heads, sh.head_dim, sh.idx_dim, n_tokens)
        pos = np.arange(n_tokens)
        self.lazy = lazy_kv
        self.filled = np.zeros(n_tokens, bool)
        ep = self.hist.epochs(pos)
        _, _, ix = gen_token_rows(sh, wl.seed, seq, pos, ep, "cpu", self.irange)
        z = np.zeros((n_tokens, sh.n_kv_heads, sh.head_dim), np.uint16)
        if lazy_kv:
            self.st.append(0, z, z, bits(ix))
        else:
            k, v, _ = gen_token_rows(sh, wl.seed, seq, pos, ep, "cpu", self.irange)
            self.st.append(0, bits(k), bits(v), bits(ix))
            self.filled[:] = True

    def fill_kv(self, tokens: np.ndarray):
        need = np.asarray(sorted(set(int(t) for t in tokens if not self.filled[t])), np.int64)
        if len(need) == 0:
            return
        k, v, _ = gen_token_rows(self.sh, self.wl.seed, self.seq, need, self.hist.epochs(need), "cpu", self.irange)
        self.st.K[need] = bits(k)
        self.st.V[need] = bits(v)
        self.filled[need] = True

    def row(self, pos: int, index_format: str = "bf16", window: int = 0):
        """Oracle result for the query row at `pos` (uses that row's q inputs)."""
        sh = self.sh
        ep = int(self.hist.epochs(np.array([pos]))[0])
        q, qi, w = S.query_rows(sh, self.wl.seed, self.seq, torch.tensor([pos]), epoch=ep, int_range=self.irange)
        visible = pos + 1
        n_blk = visible // sh.ratio
        if n_blk > sh.topk:
            score_fn = {"bf16": O.block_scores, "mxfp8": O.block_scores_mxfp8,
                        "mxfp4": O.block_scores_mxfp4}[index_format]
            sc = score_fn(bits(qi[0]), w[0].numpy(), self.st.idx_blk[:n_blk])
            sel = O.select_blocks(sc, sh.topk)
        else:
            sel = np.arange(n_blk)
        self.fill_kv(O.token_set(sel, n_blk, visible, sh.ratio, window))
        return O.attend_row(self.st, pos, bits(qi[0]), w[0].numpy(), bits(q[0]), sh.topk, index_format, window)


def compare_row(gpu_out_bits: np.ndarray, gpu_sel: np.ndarray, gpu_nsel: int, ref: Dict, topk: int):
    """Selected set bit-exact; output within max-abs 2e-2 and rel-L2 1e-3 of
    the bf16-rounded oracle."""
    want_sel = O.padded_selection(ref["sel"], topk)
    assert gpu_nsel == len(ref["sel"]), f"n_sel {gpu_nsel} != {len(ref['sel'])}"
    assert np.array_equal(gpu_sel.astype(np.int64), want_sel), "selected block set differs"
    got = bf16_value(gpu_out_bits)
    want = bf16_value(ref["out_bf16"])
    err = np.abs(got - want)
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    assert err.max() <= SEL_TOL_MAXABS, f"max-abs {err.max()}"
    assert rel <= SEL_TOL_RELL2, f"rel-L2 {rel}"
    return float(err.max()), float(rel)
