"""GPU parity of the pre-indexer (Gemma RMSNorm + NeoX RoPE of the index
queries and of every compressed key) against the CPU oracle.

The GPU forms the RoPE angles in double, reduced exactly to [-pi, pi], and
runs their sine / cosine, the norm and the rotation in fp32, then rounds to
bf16; the oracle computes in fp64 and rounds once. Stage results must agree to
one bf16 ulp, almost all bit for bit. Scores of pre-indexed keys are real
numbers, so a selected set may differ from the oracle's only by swapping
blocks whose oracle scores sit within the change that one bf16 ulp of every
key and query element allows around the K-th largest; the output is then
checked against the oracle's attention over the GPU's own token set."""
import math

import numpy as np
import pytest
import torch

from indexer_selected_sparse_gb300 import synth as S
from oracle import qsa_oracle as O
from tests.gpu_harness import SEL_TOL_MAXABS, SEL_TOL_RELL2, GpuState, bf16_value, bits, gen_token_rows

pytestmark = pytest.mark.gpu

EPS, THETA, ROT = 1e-6, 10000.0, 64


def gains(seed, d_idx, stream):
    u = S.uniform01(seed, stream, torch.arange(d_idx, dtype=torch.int64)).to(torch.float64)
    return (0.4 * (u - 0.5)).to(torch.float32)   # gains in [-0.2, 0.2)


def make_pre(Q, d_idx, device, seed=5):
    gq, gk = gains(seed, d_idx, 101), gains(seed, d_idx, 102)
    gpu = Q.PreIndexer(gq.to(device), gk.to(device), EPS, THETA, ROT)
    orc = O.PreIndexer(gq.double().numpy(), gk.double().numpy(), EPS, THETA, ROT)
    return gpu, orc


def ulp_check(got_bits, want_bits, min_exact=0.99):
    """At most one bf16 ulp apart everywhere; at least min_exact bit-identical."""
    g = np.asarray(got_bits, np.uint16).astype(np.int64).ravel()
    w = np.asarray(want_bits, np.uint16).astype(np.int64).ravel()
    # order-preserving integer map of bf16 bit patterns: adjacent values differ by 1
    key = lambda b: np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + b)
    d = np.abs(key(g) - key(w))
    assert d.max() <= 1, f"{int((d > 1).sum())} values more than one ulp apart (max {d.max()})"
    exact = float((d == 0).mean())
    assert exact >= min_exact, f"only {exact:.4f} bit-identical"
    return exact


@pytest.mark.parametrize("wl_id,n_seq,prefix", [(1, 1, 3000), (2, 2, 4100)])
def test_pre_indexed_keys_and_queries_match_the_oracle(wl_id, n_seq, prefix):
    wl0 = S.workload(wl_id)
    sh = wl0.shapes
    wl = S.Workload(wl0.name, wl0.seed, sh, [prefix] * n_seq, 1, contiguous_pages=wl0.contiguous_pages)
    g = GpuState(wl)
    Q = g.Q
    pre, opre = make_pre(Q, sh.idx_dim, g.device)
    for s in g.slots:     # fill every sequence through the pre-indexed append
        k, v, ix = gen_token_rows(sh, wl.seed, s, np.arange(prefix), np.zeros(prefix, np.int64), g.device)
        Q.qsa_append_pre(g.cfg, pre, Q.Rows(torch.tensor([s], device=g.device),
                                            torch.tensor([0], dtype=torch.int32, device=g.device), prefix),
                         g.cache, k, v, ix, g.status)
    torch.cuda.synchronize()
    g.check_status()
    exact = []
    for s in g.slots:
        _, _, ix = gen_token_rows(sh, wl.seed, s, np.arange(prefix), np.zeros(prefix, np.int64), "cpu")
        st = O.SeqState(sh.ratio, 1, 8, sh.idx_dim, prefix, pre=opre)
        z = np.zeros((prefix, 1, 8), np.uint16)
        st.append(0, z, z, bits(ix))
        nb = prefix // sh.ratio
        exact.append(ulp_check(g.logical_blocks(s, nb), st.idx_blk[:nb]))
    # queries of a step of 3 rows per sequence at the end of the prefix
    R = 3
    pos = [prefix - R] * n_seq
    rows = Q.Rows(torch.tensor(g.slots, dtype=torch.int32, device=g.device),
                  torch.tensor(pos, dtype=torch.int32, device=g.device), R)
    qi = torch.cat([S.query_rows(sh, wl.seed, s, torch.arange(p, p + R), device=g.device)[1]
                    for s, p in zip(g.slots, pos)]).contiguous()
    q_out = torch.empty_like(qi)
    Q.qsa_pre_index_q(g.cfg, pre, rows, qi, q_out)
    torch.cuda.synchronize()
    got = bits(q_out)
    qc = bits(qi)
    want = np.stack([O.pre_index_query(qc[r], pos[r // R] + r % R, opre) for r in range(n_seq * R)])
    exact.append(ulp_check(got, want))
    print("bit-identical fractions:", exact)


def score_error_bound(q_bits, w, blk_bits):
    """Largest change of each block's score when every element of the query
    heads and of the compressed keys moves by up to one bf16 ulp (relative
    2^-8 each; the stage tests above assert that much agreement): |d(q.k)| <=
    (2^-8 + 2^-8 + 2^-16) sum_d |q_d k_d|, times w_h through the ReLU (which is
    1-Lipschitz), plus fp32 accumulation (2^-20 of the same sum)."""
    q = np.abs(O.bf16_bits_to_f64(q_bits))
    k = np.abs(O.bf16_bits_to_f64(blk_bits))
    mag = np.asarray(w, np.float64) @ (q @ k.T)
    return (2.0 ** -7 + 2.0 ** -16 + 2.0 ** -20) * mag


def test_fused_decode_pre_against_the_oracle():
    """16 rows (4 sequences x 4 causal verify rows at the end of a 32k prefix)
    through qsa_decode_pre. A row's set equals the oracle's, or differs only by
    blocks whose oracle score lies within the 1-ulp score bound of the K-th
    score; either way the output must match the oracle's attention over the
    GPU's own (then valid) token set within the a4 gates."""
    wl0 = S.workload(2)
    sh = wl0.shapes
    R = 4
    p = 32768 - R
    slots = [0, 7, 20, 31]
    wl = S.Workload(wl0.name, wl0.seed, sh, [p] * len(slots), R)
    g = GpuState(wl, slots=slots)
    g.wl = wl
    Q = g.Q
    pre, opre = make_pre(Q, sh.idx_dim, g.device)
    for i, s in enumerate(slots):
        a = 0
        while a < p:
            m = min(8192, p - a)
            k, v, ix = gen_token_rows(sh, wl.seed, s, np.arange(a, a + m), np.zeros(m, np.int64), g.device)
            Q.qsa_append_pre(g.cfg, pre, Q.Rows(torch.tensor([s], device=g.device),
                                                torch.tensor([a], dtype=torch.int32, device=g.device), m),
                             g.cache, k, v, ix, g.status)
            a += m
    torch.cuda.synchronize()
    g.check_status()
    inp = g.step_inputs([p] * len(slots), R)
    rows = g.rows([p] * len(slots), R)
    n = len(slots) * R
    out = torch.empty(n, sh.n_q_heads, sh.head_dim, dtype=torch.bfloat16, device=g.device)
    sel = torch.empty(n, g.cfg.topk, dtype=torch.int32, device=g.device)
    nsel = torch.empty(n, dtype=torch.int32, device=g.device)
    ws = Q.workspace_pre(g.cfg, n, g.cache.max_blocks, device=g.device)
    Q.qsa_decode_pre(g.cfg, pre, rows, g.cache, inp["k"], inp["v"], inp["idx"], inp["q_idx"], inp["w"], inp["q"],
                     out, ws, g.status, sel_out=sel, n_sel_out=nsel)
    torch.cuda.synchronize()
    g.check_status()
    K = g.cfg.topk
    sel_h, nsel_h, out_h = sel.cpu().numpy(), nsel.cpu().numpy(), bits(out)
    same = checked = 0
    for i, s in enumerate(slots):
        n_tok = p + R
        _, _, ix = gen_token_rows(sh, wl.seed, s, np.arange(n_tok), np.zeros(n_tok, np.int64), "cpu")
        st = O.SeqState(sh.ratio, sh.n_kv_heads, sh.head_dim, sh.idx_dim, n_tok, pre=opre)
        z = np.zeros((n_tok, sh.n_kv_heads, sh.head_dim), np.uint16)
        st.append(0, z, z, bits(ix))             # K/V filled below for the tokens attended
        q, qi, w = S.query_rows(sh, wl.seed, s, torch.arange(p, p + R))
        for j in range(R):
            row = i * R + j
            pos = p + j
            visible = pos + 1
            n_blk = visible // sh.ratio
            qpre = O.pre_index_query(bits(qi[j]), pos, opre)
            sc = O.block_scores(qpre, w[j].numpy(), st.idx_blk[:n_blk])
            want_sel = O.select_blocks(sc, K)
            assert int(nsel_h[row]) == len(want_sel)
            got_sel = sel_h[row, : int(nsel_h[row])].astype(np.int64)
            assert np.all(np.diff(got_sel) > 0) and got_sel.min() >= 0 and got_sel.max() < n_blk
            if np.array_equal(got_sel, want_sel):
                same += 1
            else:
                # only blocks whose score sits within the 1-ulp bound of the K-th may swap
                bound = score_error_bound(qpre, w[j].numpy(), st.idx_blk[:n_blk])
                kb = int(np.lexsort((np.arange(n_blk), -sc))[K - 1])
                diff = np.setxor1d(got_sel, want_sel)
                assert np.all(np.abs(sc[diff] - sc[kb]) <= bound[diff] + bound[kb]), \
                    "a selected set differs beyond near-ties"
            # the output against the oracle's attention over the GPU's own token set
            toks = O.token_set(got_sel, n_blk, visible, sh.ratio)
            kk, vv, _ = gen_token_rows(sh, wl.seed, s, toks, np.zeros(len(toks), np.int64), "cpu")
            ref = O.f64_to_bf16_bits(O.gqa_attention(bits(q[j]), bits(kk), bits(vv)))
            got = bf16_value(out_h[row])
            want = bf16_value(ref)
            err = np.abs(got - want).max()
            rel = np.linalg.norm(got - want) / np.linalg.norm(want)
            assert err <= SEL_TOL_MAXABS and rel <= SEL_TOL_RELL2, (row, err, rel)
            checked += 1
    assert checked == n
    assert same >= n // 2, f"only {same} of {n} rows selected exactly the oracle's blocks"
