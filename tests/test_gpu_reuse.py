"""GPU parity for attention with a reused selection (MTP draft steps reusing
the step-0 selection; shared indexer layers reusing a full layer's top-k),
against the CPU oracle's attend_row_reused on the same seeded inputs."""
import numpy as np
import pytest
import torch

from indexer_selected_sparse_gb300 import synth as S
from oracle import qsa_oracle as O
from tests.gpu_harness import SEL_TOL_MAXABS, SEL_TOL_RELL2, GpuState, OracleSeq, bf16_value, bits

pytestmark = pytest.mark.gpu


def close(got_bits, ref):
    got = bf16_value(got_bits)
    want = bf16_value(ref["out_bf16"])
    err = np.abs(got - want).max()
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    assert err <= SEL_TOL_MAXABS and rel <= SEL_TOL_RELL2, (err, rel)


def reuse_step(g: GpuState, pos, sel, nsel, sel_pos, fused=True):
    """One decode step per sequence at `pos` with the selection reused from sel_pos."""
    Q = g.Q
    inp = g.step_inputs(pos, 1)
    rows = g.rows(pos, 1)
    n = len(pos)
    out = torch.empty(n, g.sh.n_q_heads, g.sh.head_dim, dtype=torch.bfloat16, device=g.device)
    sp = torch.tensor(sel_pos, dtype=torch.int32, device=g.device)
    if fused:
        Q.qsa_decode_reuse(g.cfg, rows, g.cache, inp["k"], inp["v"], inp["idx"], inp["q"], sel, nsel, sp, out,
                           g.ws, g.status)
    else:
        Q.qsa_gather_attn_reuse(g.cfg, rows, g.cache, inp["q"], sel, nsel, sp, out, g.ws, g.status)
    torch.cuda.synchronize()
    return out, inp


def test_draft_steps_reuse_the_step0_selection():
    # steady-decode shapes, four sequences: step 0 selects (prefix 32768 -> 8192
    # blocks, tail {32768}); draft steps 1..4 reuse it, and step 3 completes
    # block 8192, whose tokens must stay visible through the reused tail
    wl = S.workload(2)
    g = GpuState(wl, slots=[0, 5, 17, 31])
    g.wl = S.Workload(wl.name, wl.seed, wl.shapes, [wl.prefixes[0]] * 4, 1)
    g.append_prefix()
    p = wl.prefixes[0]
    res0 = g.decode([p] * 4, 1)
    g.check_status()
    sel0 = res0["sel"].clone()
    nsel0 = res0["n_sel"].clone()
    oracles = {s: OracleSeq(wl, s, p + 5) for s in g.slots}
    for i, s in enumerate(g.slots):
        ref0 = oracles[s].row(p)
        assert np.array_equal(sel0[i].cpu().numpy().astype(np.int64), O.padded_selection(ref0["sel"], g.cfg.topk))
    for d in range(1, 5):
        out, _ = reuse_step(g, [p + d] * 4, sel0, nsel0, [p] * 4)
        g.check_status()
        assert g.cache.ingested[g.slots].cpu().tolist() == [p + d + 1] * 4
        for i, s in enumerate(g.slots):
            orc = oracles[s]
            ep = int(orc.hist.epochs(np.array([p + d]))[0])
            q, _, _ = S.query_rows(wl.shapes, wl.seed, s, torch.tensor([p + d]), epoch=ep)
            sel = sel0[i, : int(nsel0[i])].cpu().numpy().astype(np.int64)
            orc.fill_kv(O.token_set(sel, (p + 1) // wl.shapes.ratio, p + d + 1, wl.shapes.ratio))
            ref = O.attend_row_reused(orc.st, p + d, sel, p, bits(q[0]))
            if d >= 3:
                assert (p + 1) // 4 * 4 in ref["tokens"] and p + d in ref["tokens"]
            close(bits(out[i]), ref)


def test_shared_layer_reuse_at_the_same_position_is_bitwise_the_decode():
    wl = S.workload(2)
    g = GpuState(wl, slots=[3, 9])
    g.wl = S.Workload(wl.name, wl.seed, wl.shapes, [wl.prefixes[0]] * 2, 1)
    g.append_prefix()
    p = wl.prefixes[0]
    res = g.decode([p] * 2, 1)
    g.check_status()
    # the "shared layer": same position, same q, the full layer's selection
    n = 2
    out = torch.empty(n, wl.shapes.n_q_heads, wl.shapes.head_dim, dtype=torch.bfloat16, device=g.device)
    rows = g.rows([p] * 2, 1)
    g.Q.qsa_gather_attn_reuse(g.cfg, rows, g.cache, res["inputs"]["q"], res["sel"], res["n_sel"],
                              torch.tensor([p, p], dtype=torch.int32, device=g.device), out, g.ws, g.status)
    torch.cuda.synchronize()
    g.check_status()
    assert np.array_equal(bits(out), bits(res["out"]))


def test_reused_dense_selection_stays_dense_past_the_inert_bound():
    # tiny shapes (budget 256, inert bound 259): a row at V0 = 259 selects every
    # block; reused at V = 259..265 it must equal dense attention over V tokens
    wl = S.workload(1)
    sh = wl.shapes
    p = sh.inert_bound - 1
    g = GpuState(S.Workload(wl.name, wl.seed, sh, [p], 1, contiguous_pages=True))
    g.append_prefix()
    res0 = g.decode([p], 1)
    g.check_status()
    assert int(res0["n_sel"][0]) == sh.inert_bound // sh.ratio
    orc = OracleSeq(g.wl, 0, p + 8, lazy_kv=False)
    for d in range(1, 7):
        out, _ = reuse_step(g, [p + d], res0["sel"], res0["n_sel"], [p])
        g.check_status()
        ep = int(orc.hist.epochs(np.array([p + d]))[0])
        q, _, _ = S.query_rows(sh, wl.seed, 0, torch.tensor([p + d]), epoch=ep)
        V = p + d + 1
        dense = O.dense_attention(bits(q[0]), orc.st.K[:V], orc.st.V[:V], sh.n_kv_heads)
        close(bits(out[0]), {"out_bf16": O.f64_to_bf16_bits(dense)})


def test_reuse_errors_are_reported_on_the_device():
    wl = S.workload(1)
    sh = wl.shapes
    g = GpuState(wl, extra_tokens=256)
    g.append_prefix()
    p = wl.prefixes[0]
    res0 = g.decode([p], 1)
    g.check_status()
    max_tok = g.Q.qsa_max_attend_tokens(g.cfg)
    assert max_tok == -(-sh.inert_bound // 112) * 112
    # a selection "from the future"
    out, _ = reuse_step(g, [p + 1], res0["sel"], res0["n_sel"], [p + 2], fused=False)
    g.check_status(g.Q.QSA_ERR_REUSE)
    g.status.zero_()
    # a selection so old that its token set no longer fits the split plan:
    # 64 blocks x 4 + tail from block 750's boundary to the row
    far = p + (max_tok - sh.topk * sh.ratio) + 8
    n_fill = far - (p + 1)
    pos = np.arange(p + 1, p + 1 + n_fill)
    k, v, ix = S.token_rows(sh, wl.seed, 0, torch.from_numpy(pos), device=g.device)
    g.Q.qsa_append(g.cfg, g.Q.Rows(torch.tensor([0], device=g.device),
                                   torch.tensor([p + 1], dtype=torch.int32, device=g.device), n_fill),
                   g.cache, k, v, ix, g.status)
    torch.cuda.synchronize()
    g.check_status()
    out, _ = reuse_step(g, [far], res0["sel"], res0["n_sel"], [p])
    g.check_status(g.Q.QSA_ERR_REUSE)
