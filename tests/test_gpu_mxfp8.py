"""GPU parity of the MXFP8 index plane (index_format QSA_INDEX_MXFP8) against
the CPU oracle.

* The plane: every compressed key's E4M3 elements and E8M0 scales, decoded from
  the stored bytes with the format's bit definition, equal the oracle's MXFP8
  quantisation of its bf16 compressed key (values compared, so the sign of a
  zero element is not).
* The query round trip: bit-exact bf16, including nearest-even ties, the
  subnormal range, saturation at 448 and all-zero blocks.
* Scores: bit-exact against the oracle's MXFP8 score (the synthetic integer
  inputs keep every sum of products exact in fp32).
* The scorer's own query rounding, on real-valued queries that do round (both
  MX formats): scores of unrounded queries equal, bit for bit, those of the
  same queries rounded first by qsa_quantize_index_q, whose output equals the
  oracle's rounding.
* Fused steps (decode, verify, ragged prefixes, d_I 64 and 8 blocks per page):
  selected sets bit-exact against the oracle scoring with the same
  quantisation; outputs within the bf16 gates."""
import numpy as np
import pytest
import torch

from indexer_selected_sparse_gb300 import synth as S
from oracle import qsa_oracle as O
from tests.gpu_harness import GpuState, OracleSeq, bits, compare_row, gen_token_rows
from tests.oracle_sets import StepLog

pytestmark = pytest.mark.gpu

MX = 1  # QSA_INDEX_MXFP8


def small_wl(ratio, budget, h_i, d_i, hq, hkv, prefixes, R=1, seed=11):
    sh = S.Shapes(ratio, budget, h_i, d_i, hq, hkv, 128, 64)
    return S.Workload("mxfp8", seed, sh, list(prefixes), R, contiguous_pages=False)


def oracle_blocks(g, s, n_tokens):
    sh = g.sh
    _, _, ix = gen_token_rows(sh, g.wl.seed, s, np.arange(n_tokens), g.hist[s].epochs(np.arange(n_tokens)),
                              "cpu", g.irange)
    st = O.SeqState(sh.ratio, 1, 8, sh.idx_dim, n_tokens)
    z = np.zeros((n_tokens, 1, 8), np.uint16)
    st.append(0, z, z, bits(ix))
    return st.idx_blk[: n_tokens // sh.ratio]


def check_plane(g, s, n_tokens):
    want_bits = oracle_blocks(g, s, n_tokens)
    n_blk = len(want_bits)
    el, ex = g.logical_blocks_mxfp8(s, n_blk)
    want_el, want_ex = O.mxfp8_quantize(O.bf16_bits_to_f64(want_bits))
    assert np.array_equal(ex, want_ex), "scale bytes differ"
    assert np.array_equal(el, want_el), "E4M3 elements differ"


PLANES = {
    # ratio, budget, H_I, d_I, Hq, Hkv, prefixes
    "r4_dI64": (4, 256, 4, 64, 8, 1, [3000, 1]),
    "r4_dI128": (4, 2048, 64, 128, 32, 4, [9001, 64, 130]),
    "r8_dI128_bpp8": (8, 1024, 16, 128, 16, 2, [5003]),
}


@pytest.mark.parametrize("name", list(PLANES))
def test_plane_bytes_match_the_oracle(name):
    r, b, hi, di, hq, hkv, pre = PLANES[name]
    g = GpuState(small_wl(r, b, hi, di, hq, hkv, pre), index_format=MX)
    g.append_prefix(chunk=1000)
    for i, s in enumerate(g.slots):
        check_plane(g, s, pre[i])


def test_query_round_trip_bit_exact():
    from indexer_selected_sparse_gb300 import qsa as Q
    sh = S.workload(2).shapes
    cfg = Q.Config.of(sh, MX)
    rng = np.random.default_rng(71)
    n = 9
    x = rng.standard_normal((n, sh.n_idx_heads, sh.idx_dim))
    x *= np.repeat(10.0 ** rng.uniform(-30, 30, (n, sh.n_idx_heads, sh.idx_dim // 32)), 32, axis=-1)
    x[0, 0] = 0.0                                   # an all-zero head
    x[0, 1, :32] = 0.0
    x[0, 1, 5] = -3.0e-38                           # a block whose amax is near fp32's smallest normal
    # one block with amax in [256, 512), scale 1: nearest-even ties, subnormals, saturation
    ties = np.zeros(32)
    ties[:9] = [1.0625, 1.1875, -2.0 ** -10, 3 * 2.0 ** -10, 456.0, 464.0, -300.0, 2.0 ** -9, 0.4375]
    x[1, 0, :32] = ties
    q = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    want = O.f64_to_bf16_bits(O.mxfp8_round_bits(bits(q)))
    qd = q.cuda()
    out = torch.empty_like(qd)
    Q.qsa_quantize_index_q(cfg, qd, out)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), want)
    # in place
    Q.qsa_quantize_index_q(cfg, qd, qd)
    torch.cuda.synchronize()
    assert np.array_equal(bits(qd), want)
    # the hand-worked block (scale 1): 1.0625 -> 1, 1.1875 -> 1.25 (ties to even),
    # 2^-10 -> 0, 3*2^-10 -> 2^-8 (subnormal quantum 2^-9), 456 and 464 -> 448,
    # -300 -> -288 (quantum 32 in [256, 512): 9.375 -> 9), 2^-9 and 0.4375 stay
    got = O.bf16_bits_to_f64(bits(out)[1, 0, :9])
    assert got.tolist() == [1.0, 1.25, 0.0, 2.0 ** -8, 448.0, 448.0, -288.0, 2.0 ** -9, 0.4375]


def test_scores_bit_exact():
    wl = small_wl(4, 256, 64, 128, 32, 4, [3000, 9000, 20001], R=2)
    g = GpuState(wl, index_format=MX)
    g.append_prefix()
    Q = g.Q
    pos0 = list(wl.prefixes)
    res = g.decode(pos0, 2)
    g.check_status()
    inp = res["inputs"]
    q_hat = torch.empty_like(inp["q_idx"])
    Q.qsa_quantize_index_q(g.cfg, inp["q_idx"], q_hat)
    rows = g.rows(pos0, 2)
    n = len(pos0) * 2
    ld = (g.cache.max_blocks + 3) // 4 * 4
    scores = torch.full((n, ld), float("nan"), dtype=torch.float32, device="cuda")
    Q.qsa_index_score(g.cfg, rows, g.cache, q_hat, inp["w"], scores, ld, g.status)
    torch.cuda.synchronize()
    g.check_status()
    for i, s in enumerate(g.slots):
        orc = OracleSeq(wl, s, pos0[i] + 2)
        for j in range(2):
            ref = orc.row(pos0[i] + j, "mxfp8")
            nb = ref["n_blk"]
            assert np.array_equal(scores[i * 2 + j, :nb].cpu().numpy().astype(np.float64), ref["scores"])
    # the scorer rounds its queries itself: unrounded queries score the same
    scores2 = torch.full((n, ld), float("nan"), dtype=torch.float32, device="cuda")
    Q.qsa_index_score(g.cfg, rows, g.cache, inp["q_idx"], inp["w"], scores2, ld, g.status)
    torch.cuda.synchronize()
    g.check_status()
    for r in range(n):
        nb = (pos0[r // 2] + r % 2 + 1) // 4
        assert torch.equal(scores2[r, :nb], scores[r, :nb])


def real_queries(n, h_i, d_i, seed=29):
    """Gaussian bf16 index queries with magnitudes spread over 2^-20 .. 2^12 per
    32-value block (so blocks land in every scale range), an all-zero block and
    a block of one tiny value: values that round in both MX formats."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, h_i, d_i, generator=g, dtype=torch.float64)
    mag = torch.pow(2.0, torch.randint(-20, 13, (n, h_i, d_i // 32), generator=g).double())
    x = x * mag.repeat_interleave(32, dim=-1)
    x[0, 0, :32] = 0.0
    x[0, 1, :32] = 0.0
    x[0, 1, 5] = -(2.0 ** -130)
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("fmt", [1, 2], ids=["mxfp8", "mxfp4"])
def test_scorer_rounds_real_valued_queries(fmt):
    wl = small_wl(4, 256, 64, 128, 32, 4, [3000, 9000, 20001], R=2)
    g = GpuState(wl, index_format=fmt)
    g.append_prefix()
    Q = g.Q
    pos0 = list(wl.prefixes)
    g.decode(pos0, 2)
    g.check_status()
    n = len(pos0) * 2
    q = real_queries(n, 64, 128).to("cuda")
    w = (torch.rand(n, 64, generator=torch.Generator().manual_seed(31)) + 0.25).to("cuda")
    q_hat = torch.empty_like(q)
    Q.qsa_quantize_index_q(g.cfg, q, q_hat)
    torch.cuda.synchronize()
    rnd = O.mxfp8_round_bits if fmt == 1 else O.mxfp4_round_bits
    want = rnd(bits(q).reshape(-1, 128))
    got = O.bf16_bits_to_f64(bits(q_hat).reshape(-1, 128))
    assert np.array_equal(got, want), "qsa_quantize_index_q differs from the oracle's rounding"
    assert not np.array_equal(got, O.bf16_bits_to_f64(bits(q).reshape(-1, 128))), "nothing rounded"
    rows = g.rows(pos0, 2)
    ld = (g.cache.max_blocks + 3) // 4 * 4
    out = []
    for qq in (q_hat, q):
        sc = torch.full((n, ld), float("nan"), dtype=torch.float32, device="cuda")
        Q.qsa_index_score(g.cfg, rows, g.cache, qq, w, sc, ld, g.status)
        torch.cuda.synchronize()
        g.check_status()
        out.append(sc)
    for r in range(n):
        nb = (pos0[r // 2] + r % 2 + 1) // 4
        assert torch.equal(out[1][r, :nb], out[0][r, :nb]), f"row {r}"
        assert torch.isfinite(out[0][r, :nb]).all()


FUSED = {
    # ratio, budget, H_I, d_I, Hq, Hkv, prefixes, R
    "decode_main": (4, 2048, 64, 128, 32, 4, [32768, 9000, 2051, 2052], 1),
    "verify_R4_groups_of_3": (4, 512, 64, 128, 32, 4, [5000, 12001], 4),
    "dI64_r8_bpp8": (8, 256, 16, 64, 8, 1, [300, 4097], 2),
}


@pytest.mark.parametrize("name", list(FUSED))
def test_fused_step_every_row(name):
    r, b, hi, di, hq, hkv, pre, R = FUSED[name]
    wl = small_wl(r, b, hi, di, hq, hkv, pre, R)
    g = GpuState(wl, extra_tokens=8, index_format=MX)
    g.append_prefix()
    pos0 = list(wl.prefixes)
    res = g.decode(pos0, R)
    g.check_status()
    sel = res["sel"].cpu().numpy(); nsel = res["n_sel"].cpu().numpy(); out = bits(res["out"])
    for i, s in enumerate(g.slots):
        orc = OracleSeq(wl, s, pos0[i] + R)
        for j in range(R):
            row = i * R + j
            compare_row(out[row], sel[row], int(nsel[row]), orc.row(pos0[i] + j, "mxfp8"), g.cfg.topk)
        check_plane(g, s, pos0[i] + R)


def test_steady_decode_batch32_prefix32k_every_row():
    """Batch 32 x 32k with the MXFP8 plane: every row's selection of two steps
    against the oracle's MXFP8 scores; outputs on sampled rows."""
    wl = S.workload(2)
    g = GpuState(wl, extra_tokens=8, index_format=MX)
    g.append_prefix()
    sampled = [0, 17, 31]
    oracles = {s: OracleSeq(wl, s, wl.prefixes[0] + 2) for s in sampled}
    pos0 = list(wl.prefixes)
    log = StepLog()
    for step in range(2):
        res = g.decode(pos0, 1)
        g.check_status()
        log.add(res, g.slots, pos0, 1)
        sel = res["sel"].cpu().numpy(); nsel = res["n_sel"].cpu().numpy(); out = bits(res["out"])
        for s in sampled:
            compare_row(out[s], sel[s], int(nsel[s]), oracles[s].row(pos0[s], "mxfp8"), g.cfg.topk)
        pos0 = [p + 1 for p in pos0]
    assert log.check(wl, index_format="mxfp8") == 2 * wl.n_seq
