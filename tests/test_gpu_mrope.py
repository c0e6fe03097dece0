"""GPU parity of interleaved MRoPE (position triples) against the CPU oracle.

A multimodal sequence carries a (t, h, w) triple per token (text (p, p, p),
then an image grid at one temporal step, then text again). Through the
pre-indexer, each compressed key turns at its block's first token's triple,
kept beside the page for blocks that a later append completes. Index queries
and, with the attention options, the main q and k heads turn at their own
row's triple. Values agree with the fp64 oracle to one bf16 ulp and almost all
bit for bit. Text triples reproduce the plain RoPE path bit for bit on the GPU
itself."""
import numpy as np
import pytest
import torch

from indexer_selected_sparse_gb300 import synth as S
from oracle import qsa_oracle as O
from tests.gpu_harness import GpuState, bits, compare_row, gen_token_rows
from tests.test_gpu_attn_options import close_keys, gains as attn_gains, gate_rows
from tests.test_gpu_pre import EPS, ROT, THETA, gains, ulp_check

pytestmark = pytest.mark.gpu

SECTION = (11, 11, 10)   # the pages' sections over 64 rotary dimensions


def pre_pair(Q, d_idx, device, section, seed=5):
    gq, gk = gains(seed, d_idx, 101), gains(seed, d_idx, 102)
    gpu = Q.PreIndexer(gq.to(device), gk.to(device), EPS, THETA, ROT, mrope_section=section)
    orc = O.PreIndexer(gq.double().numpy(), gk.double().numpy(), EPS, THETA, ROT, mrope_section=section)
    return gpu, orc


def triples(n, img_start, gh, gw):
    return S.mrope_positions(n, img_start, gh, gw)


def fill_pre(g, pre, s, n, mpos, chunks, data_seq=None):
    """Append tokens 0..n-1 of slot s through the pre-indexer in the given chunk sizes
    (sizes that cut blocks, so some blocks complete in a later call). The token rows are
    those of sequence `data_seq` (default s), so several slots can hold the same data."""
    Q = g.Q
    src = s if data_seq is None else data_seq
    a = 0
    for m in chunks:
        m = min(m, n - a)
        if m <= 0:
            break
        k, v, ix = gen_token_rows(g.sh, g.wl.seed, src, np.arange(a, a + m), np.zeros(m, np.int64), g.device)
        Q.qsa_append_pre(g.cfg, pre, Q.Rows(torch.tensor([s], device=g.device),
                                            torch.tensor([a], dtype=torch.int32, device=g.device), m,
                                            mrope_pos=None if mpos is None else mpos[a:a + m].to(g.device)),
                         g.cache, k, v, ix, g.status)
        a += m
    assert a == n


def oracle_blocks(g, s, n, opre, mpos):
    _, _, ix = gen_token_rows(g.sh, g.wl.seed, s, np.arange(n), np.zeros(n, np.int64), "cpu")
    st = O.SeqState(g.sh.ratio, 1, 8, g.sh.idx_dim, n, pre=opre)
    z = np.zeros((n, 1, 8), np.uint16)
    st.append(0, z, z, bits(ix), mpos=None if mpos is None else mpos.numpy())
    return st.idx_blk[: n // g.sh.ratio]


@pytest.mark.parametrize("wl_id", [1, 2])
def test_keys_and_queries_turn_at_their_triples(wl_id):
    wl0 = S.workload(wl_id)
    sh = wl0.shapes
    n = 3001
    wl = S.Workload(wl0.name, wl0.seed, sh, [n], 1, contiguous_pages=wl0.contiguous_pages)
    g = GpuState(wl, mrope=True)
    Q = g.Q
    pre, opre = pre_pair(Q, sh.idx_dim, g.device, SECTION)
    mpos = triples(n, 1000, 24, 40)   # image tokens 1000 .. 1959
    s = g.slots[0]
    # block 375 (tokens 1500 .. 1503) starts in the 4th call and completes in the 5th: its first
    # token's triple (1000, 1012, 1020) is read back from beside the page
    fill_pre(g, pre, s, n, mpos, [999, 2, 1, 501, 1498])
    torch.cuda.synchronize()
    g.check_status()
    nb = n // sh.ratio
    want = oracle_blocks(g, s, n, opre, mpos)
    got = g.logical_blocks(s, nb)
    ulp_check(got, want)
    # the image changed the keys: plain RoPE at the sequence positions gives others
    _, plain = pre_pair(Q, sh.idx_dim, g.device, None)
    assert not np.array_equal(want, oracle_blocks(g, s, n, plain, None))
    # index queries of 3 rows inside the image, each at its own triple
    R = 3
    p0 = 1500
    rows = Q.Rows(torch.tensor([s], dtype=torch.int32, device=g.device),
                  torch.tensor([p0], dtype=torch.int32, device=g.device), R,
                  mrope_pos=mpos[p0:p0 + R].to(g.device))
    qi = S.query_rows(sh, wl.seed, s, torch.arange(p0, p0 + R), device=g.device)[1].contiguous()
    q_out = torch.empty_like(qi)
    Q.qsa_pre_index_q(g.cfg, pre, rows, qi, q_out)
    torch.cuda.synchronize()
    qc = bits(qi)
    want_q = np.stack([O.pre_index_query(qc[r], tuple(mpos[p0 + r].tolist()), opre) for r in range(R)])
    ulp_check(bits(q_out), want_q)


def test_text_triples_are_the_plain_path_bit_for_bit():
    wl0 = S.workload(1)
    sh = wl0.shapes
    n = 2003
    wl = S.Workload(wl0.name, wl0.seed, sh, [n, n, n], 1, contiguous_pages=wl0.contiguous_pages)
    g = GpuState(wl, mrope=True)
    Q = g.Q
    pre_m, _ = pre_pair(Q, sh.idx_dim, g.device, SECTION)
    pre_p, _ = pre_pair(Q, sh.idx_dim, g.device, None)
    text = triples(n, n, 1, 1)        # no image: (p, p, p) throughout
    a, b, c = g.slots
    # the same token rows in all three slots
    fill_pre(g, pre_p, a, n, None, [700, 700, 700], data_seq=a)        # plain RoPE
    fill_pre(g, pre_m, b, n, None, [701, 699, 700], data_seq=a)        # MRoPE section, text rows (no triples)
    fill_pre(g, pre_m, c, n, text, [333, 1000, 777], data_seq=a)       # MRoPE section, explicit (p, p, p)
    torch.cuda.synchronize()
    g.check_status()
    nb = n // sh.ratio
    ref = g.logical_blocks(a, nb)
    assert np.array_equal(g.logical_blocks(b, nb), ref)
    assert np.array_equal(g.logical_blocks(c, nb), ref)


def test_attention_heads_turn_at_their_triples_in_the_fused_step():
    sh = S.Shapes(4, 256, 16, 128, 16, 2, 128, 64)
    n = 2500
    wl = S.Workload("mrope-attn", 17, sh, [n], 1, contiguous_pages=False)
    g = GpuState(wl, extra_tokens=8, mrope=True)
    Q = g.Q
    gq, gk = attn_gains(9, 128, 201), attn_gains(9, 128, 202)
    gate = gate_rows(1, 16, seed=5).to(g.device)
    att = Q.AttnOptions(gq.to(g.device), gk.to(g.device), EPS, THETA, ROT, gate, mrope_section=SECTION)
    oatt = O.AttnOptions(gq.double().numpy(), gk.double().numpy(), EPS, THETA, ROT, mrope_section=SECTION)
    mpos = triples(n + 1, 600, 30, 50)        # image tokens 600 .. 2099
    s = g.slots[0]
    a = 0
    for m in (1234, n - 1234):
        k, v, ix = gen_token_rows(sh, wl.seed, s, np.arange(a, a + m), np.zeros(m, np.int64), g.device)
        Q.qsa_append_ex(g.cfg, None, att, Q.Rows(torch.tensor([s], device=g.device),
                                                 torch.tensor([a], dtype=torch.int32, device=g.device), m,
                                                 mrope_pos=mpos[a:a + m].to(g.device)),
                        g.cache, k, v, ix, g.status)
        a += m
    torch.cuda.synchronize()
    g.check_status()
    # the stored keys: each head normed and turned at its own token's triple
    kk, vv, ix = gen_token_rows(sh, wl.seed, s, np.arange(n + 1), np.zeros(n + 1, np.int64), "cpu")
    st = O.SeqState(sh.ratio, sh.n_kv_heads, sh.head_dim, sh.idx_dim, n + 1, attn=oatt)
    st.append(0, bits(kk)[:n], bits(vv)[:n], bits(ix)[:n], mpos=mpos[:n].numpy())
    close_keys(g.logical_rows(g.cache.k_pool, s, np.arange(n)), st.K[:n])
    # one fused decode row at position n (a text token after the image)
    inp = g.step_inputs([n], 1)
    rows = Q.Rows(torch.tensor([s], dtype=torch.int32, device=g.device),
                  torch.tensor([n], dtype=torch.int32, device=g.device), 1, mrope_pos=mpos[n:n + 1].to(g.device))
    out = torch.empty(1, 16, 128, dtype=torch.bfloat16, device=g.device)
    sel = torch.empty(1, g.cfg.topk, dtype=torch.int32, device=g.device)
    nsel = torch.empty(1, dtype=torch.int32, device=g.device)
    ws = Q.workspace_ex(g.cfg, 1, g.cache.max_blocks, device=g.device)
    Q.qsa_decode_ex(g.cfg, None, att, rows, g.cache, inp["k"], inp["v"], inp["idx"], inp["q_idx"], inp["w"],
                    inp["q"], out, ws, g.status, sel_out=sel, n_sel_out=nsel)
    torch.cuda.synchronize()
    g.check_status()
    st.append(n, bits(kk)[n:], bits(vv)[n:], bits(ix)[n:], mpos=mpos[n:].numpy())
    qq, qi, w = S.query_rows(sh, wl.seed, s, torch.tensor([n]))
    ref = O.attend_row(st, n, bits(qi[0]), w[0].numpy(), bits(qq[0]), g.cfg.topk, attn=oatt,
                       gate_bits=bits(gate)[0], q_mpos=tuple(mpos[n].tolist()))
    compare_row(bits(out[0]), sel[0].cpu().numpy(), int(nsel[0]), ref, g.cfg.topk)
