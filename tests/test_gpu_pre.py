"""GPU parity of the pre-indexer (Gemma RMSNorm + NeoX RoPE of the index
queries and of every compressed key) against the CPU oracle.

The GPU forms the RoPE angles in double, reduced exactly to [-pi, pi], and
runs their sine / cosine, the norm and the rotation in fp32, then rounds to
bf16; the oracle computes in fp64 and rounds once. Stage results must agree to
one bf16 ulp, almost all bit for bit. Scores of pre-indexed keys are real
numbers, so a selected set may differ from the oracle's only by swapping
blocks whose oracle scores sit within a relative 1e-4 of the K-th largest."""
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


def test_fused_decode_pre_against_the_oracle():
    wl0 = S.workload(2)
    sh = wl0.shapes
    p = 32768
    slots = [0, 7, 20]
    wl = S.Workload(wl0.name, wl0.seed, sh, [p] * 3, 1)
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
    inp = g.step_inputs([p] * 3, 1)
    rows = g.rows([p] * 3, 1)
    n = 3
    out = torch.empty(n, sh.n_q_heads, sh.head_dim, dtype=torch.bfloat16, device=g.device)
    sel = torch.empty(n, g.cfg.topk, dtype=torch.int32, device=g.device)
    nsel = torch.empty(n, dtype=torch.int32, device=g.device)
    ws = Q.workspace_pre(g.cfg, n, g.cache.max_blocks, device=g.device)
    Q.qsa_decode_pre(g.cfg, pre, rows, g.cache, inp["k"], inp["v"], inp["idx"], inp["q_idx"], inp["w"], inp["q"],
                     out, ws, g.status, sel_out=sel, n_sel_out=nsel)
    torch.cuda.synchronize()
    g.check_status()
    K = g.cfg.topk
    same = 0
    for i, s in enumerate(slots):
        pos = np.arange(p + 1)
        kk, vv, ix = gen_token_rows(sh, wl.seed, s, pos, np.zeros(p + 1, np.int64), "cpu")
        st = O.SeqState(sh.ratio, sh.n_kv_heads, sh.head_dim, sh.idx_dim, p + 1, pre=opre)
        st.append(0, bits(kk), bits(vv), bits(ix))
        q, qi, w = S.query_rows(sh, wl.seed, s, torch.tensor([p]))
        qpre = O.pre_index_query(bits(qi[0]), p, opre)
        ref = O.attend_row(st, p, qpre, w[0].numpy(), bits(q[0]), K)
        got_sel = sel[i, : int(nsel[i])].cpu().numpy().astype(np.int64)
        assert int(nsel[i]) == len(ref["sel"])
        if np.array_equal(got_sel, ref["sel"]):
            same += 1
            got = bf16_value(bits(out[i]))
            want = bf16_value(ref["out_bf16"])
            err = np.abs(got - want).max()
            rel = np.linalg.norm(got - want) / np.linalg.norm(want)
            assert err <= SEL_TOL_MAXABS and rel <= SEL_TOL_RELL2, (err, rel)
        else:
            # only near-ties at the K-th score may swap
            sc = ref["scores"]
            kth = np.sort(sc)[::-1][K - 1]
            band = 1e-4 * abs(kth)
            diff = np.setxor1d(got_sel, ref["sel"])
            assert np.all(np.abs(sc[diff] - kth) <= band), "a selected set differs beyond near-ties"
    assert same >= 2, f"only {same} of 3 rows selected exactly the oracle's blocks"
