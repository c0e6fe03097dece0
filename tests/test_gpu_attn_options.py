"""GPU parity of the main-attention options (qsa_attn_options: GemmaRMSNorm +
NeoX RoPE of the q and k heads, sigmoid output gate) against the CPU oracle.

Keys prepared by the append kernel agree with the oracle's to one bf16 ulp or
2^-16 absolute, whichever is larger (fp32 norm and rotation against fp64, one
rounding each side: where the rotation nearly cancels, the result is small and
fp32's absolute error of about 1e-7 on terms of order 1 can span a few ulps of
it), and at least 99% bit for bit. The index path is untouched by these
options, so selected block sets stay bit-exact; outputs within the bf16 gates
of the plain path."""
import numpy as np
import pytest
import torch

from indexer_selected_sparse_gb300 import synth as S
from oracle import qsa_oracle as O
from tests.gpu_harness import GpuState, OracleSeq, bits, compare_row, gen_token_rows


def close_keys(got_bits, want_bits, abs_tol=2.0 ** -16, min_exact=0.99):
    g = O.bf16_bits_to_f64(np.asarray(got_bits, np.uint16).ravel())
    w = O.bf16_bits_to_f64(np.asarray(want_bits, np.uint16).ravel())
    _, e = np.frexp(np.where(w != 0, np.abs(w), 1.0))
    ulp = np.ldexp(1.0, np.maximum(e - 1, -126) - 7)
    d = np.abs(g - w)
    bad = d > np.maximum(ulp, abs_tol)
    assert not bad.any(), f"{int(bad.sum())} values beyond one ulp and {abs_tol} (max {d[bad].max()})"
    exact = float((d == 0).mean())
    assert exact >= min_exact, f"only {exact:.4f} bit-identical"
    return exact


pytestmark = pytest.mark.gpu

EPS, THETA, ROT = 1e-6, 1e4, 64


def gains(seed, n, stream):
    u = S.uniform01(seed, stream, torch.arange(n, dtype=torch.int64)).to(torch.float64)
    return (0.4 * (u - 0.5)).to(torch.float32)


def options(Q, device, with_q=True, with_k=True, gate=None, seed=9):
    gq, gk = gains(seed, 128, 201), gains(seed, 128, 202)
    gpu = Q.AttnOptions(gq.to(device) if with_q else None, gk.to(device) if with_k else None, EPS, THETA, ROT, gate)
    orc = O.AttnOptions(gq.double().numpy() if with_q else None, gk.double().numpy() if with_k else None,
                        EPS, THETA, ROT)
    return gpu, orc


def gate_rows(n, hq, seed=3):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(n, hq, 128, generator=g) * 2).to(torch.bfloat16)


def small_wl(prefixes, R=1, seed=17):
    sh = S.Shapes(4, 256, 16, 128, 16, 2, 128, 64)
    return S.Workload("attn-options", seed, sh, list(prefixes), R, contiguous_pages=False)


def fill_ex(g, att, n_tokens):
    Q = g.Q
    for i, s in enumerate(g.slots):
        a = 0
        while a < n_tokens[i]:
            m = min(4096, n_tokens[i] - a)
            k, v, ix = gen_token_rows(g.sh, g.wl.seed, s, np.arange(a, a + m), np.zeros(m, np.int64), g.device)
            Q.qsa_append_ex(g.cfg, None, att, Q.Rows(torch.tensor([s], device=g.device),
                                                     torch.tensor([a], dtype=torch.int32, device=g.device), m),
                            g.cache, k, v, ix, g.status)
            a += m
    torch.cuda.synchronize()
    g.check_status()


def oracle_state(g, s, n_tokens, oatt):
    sh = g.sh
    pos = np.arange(n_tokens)
    k, v, ix = gen_token_rows(sh, g.wl.seed, s, pos, np.zeros(n_tokens, np.int64), "cpu")
    st = O.SeqState(sh.ratio, sh.n_kv_heads, sh.head_dim, sh.idx_dim, n_tokens, attn=oatt)
    st.append(0, bits(k), bits(v), bits(ix))
    return st


def test_keys_prepared_on_append_match_the_oracle():
    wl = small_wl([3000, 130])
    g = GpuState(wl)
    att, oatt = options(g.Q, g.device, with_q=False)
    fill_ex(g, att, wl.prefixes)
    for i, s in enumerate(g.slots):
        n = wl.prefixes[i]
        st = oracle_state(g, s, n, oatt)
        got = g.logical_rows(g.cache.k_pool, s, np.arange(n))
        close_keys(got, st.K[:n])
        # V rows are stored as given
        assert np.array_equal(g.logical_rows(g.cache.v_pool, s, np.arange(n)), st.V[:n])


def test_gate_only_every_row():
    wl = small_wl([300, 4000, 9001], R=2)
    g = GpuState(wl, extra_tokens=8)
    g.append_prefix()
    Q = g.Q
    pos0 = list(wl.prefixes)
    n = len(pos0) * 2
    gate = gate_rows(n, 16).to(g.device)
    att, _ = options(Q, g.device, with_q=False, with_k=False, gate=gate)
    inp = g.step_inputs(pos0, 2)
    out = torch.empty(n, 16, 128, dtype=torch.bfloat16, device=g.device)
    sel = torch.empty(n, g.cfg.topk, dtype=torch.int32, device=g.device)
    nsel = torch.empty(n, dtype=torch.int32, device=g.device)
    ws = Q.workspace_ex(g.cfg, n, g.cache.max_blocks, device=g.device)
    Q.qsa_decode_ex(g.cfg, None, att, g.rows(pos0, 2), g.cache, inp["k"], inp["v"], inp["idx"], inp["q_idx"],
                    inp["w"], inp["q"], out, ws, g.status, sel_out=sel, n_sel_out=nsel)
    torch.cuda.synchronize()
    g.check_status()
    gb = bits(gate)
    for i, s in enumerate(g.slots):
        orc = OracleSeq(wl, s, pos0[i] + 2)
        for j in range(2):
            row = i * 2 + j
            ref_plain = orc.row(pos0[i] + j)
            qq, qi, w = S.query_rows(wl.shapes, wl.seed, s, torch.tensor([pos0[i] + j]))
            ref = O.attend_row(orc.st, pos0[i] + j, bits(qi[0]), w[0].numpy(), bits(qq[0]), g.cfg.topk,
                               gate_bits=gb[row])
            assert np.array_equal(ref["sel"], ref_plain["sel"])
            compare_row(bits(out[row]), sel[row].cpu().numpy(), int(nsel[row]), ref, g.cfg.topk)


def test_qk_norm_rope_and_gate_fused_step():
    wl = small_wl([2500, 6001, 255])
    g = GpuState(wl, extra_tokens=8)
    Q = g.Q
    n = len(wl.prefixes)
    gate = gate_rows(n, 16, seed=5).to(g.device)
    att, oatt = options(Q, g.device, gate=gate)
    fill_ex(g, att, wl.prefixes)
    pos0 = list(wl.prefixes)
    inp = g.step_inputs(pos0, 1)
    out = torch.empty(n, 16, 128, dtype=torch.bfloat16, device=g.device)
    sel = torch.empty(n, g.cfg.topk, dtype=torch.int32, device=g.device)
    nsel = torch.empty(n, dtype=torch.int32, device=g.device)
    ws = Q.workspace_ex(g.cfg, n, g.cache.max_blocks, device=g.device)
    Q.qsa_decode_ex(g.cfg, None, att, g.rows(pos0, 1), g.cache, inp["k"], inp["v"], inp["idx"], inp["q_idx"],
                    inp["w"], inp["q"], out, ws, g.status, sel_out=sel, n_sel_out=nsel)
    torch.cuda.synchronize()
    g.check_status()
    gb = bits(gate)
    for i, s in enumerate(g.slots):
        p = pos0[i]
        st = oracle_state(g, s, p + 1, oatt)
        qq, qi, w = S.query_rows(wl.shapes, wl.seed, s, torch.tensor([p]))
        ref = O.attend_row(st, p, bits(qi[0]), w[0].numpy(), bits(qq[0]), g.cfg.topk, attn=oatt, gate_bits=gb[i])
        compare_row(bits(out[i]), sel[i].cpu().numpy(), int(nsel[i]), ref, g.cfg.topk)
