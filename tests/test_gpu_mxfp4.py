"""GPU parity of the MXFP4 index plane (index_format QSA_INDEX_MXFP4: E2M1
elements, one E8M0 scale per 32 values) against the CPU oracle: stored planes
(element values decoded from the nibbles, scale bytes), the query round trip,
bit-exact scores (the synthetic integer inputs keep every sum exact), and
selections of fused steps bit-exact against the oracle scoring in the same
format, outputs within the bf16 gates."""
import numpy as np
import pytest
import torch

from indexer_selected_sparse_gb300 import synth as S
from oracle import qsa_oracle as O
from tests.gpu_harness import GpuState, OracleSeq, bits, compare_row
from tests.oracle_sets import StepLog
from tests.test_gpu_mxfp8 import oracle_blocks, small_wl

pytestmark = pytest.mark.gpu

MX4 = 2  # QSA_INDEX_MXFP4


def check_plane4(g, s, n_tokens):
    want_bits = oracle_blocks(g, s, n_tokens)
    el, ex = g.logical_blocks_mxfp4(s, len(want_bits))
    want_el, want_ex = O.mxfp4_quantize(O.bf16_bits_to_f64(want_bits))
    assert np.array_equal(ex, want_ex), "scale bytes differ"
    assert np.array_equal(el, want_el), "E2M1 elements differ"


PLANES = {
    "r4_dI64": (4, 256, 4, 64, 8, 1, [3000, 1]),
    "r4_dI128": (4, 2048, 64, 128, 32, 4, [9001, 130]),
    "r8_dI128_bpp8": (8, 1024, 16, 128, 16, 2, [5003]),
}


@pytest.mark.parametrize("name", list(PLANES))
def test_plane_bytes_match_the_oracle(name):
    r, b, hi, di, hq, hkv, pre = PLANES[name]
    g = GpuState(small_wl(r, b, hi, di, hq, hkv, pre), index_format=MX4)
    g.append_prefix(chunk=1000)
    for i, s in enumerate(g.slots):
        check_plane4(g, s, pre[i])


def test_query_round_trip_bit_exact():
    from indexer_selected_sparse_gb300 import qsa as Q
    sh = S.workload(2).shapes
    cfg = Q.Config.of(sh, MX4)
    rng = np.random.default_rng(97)
    x = rng.standard_normal((5, sh.n_idx_heads, sh.idx_dim))
    x *= np.repeat(10.0 ** rng.uniform(-20, 20, (5, sh.n_idx_heads, sh.idx_dim // 32)), 32, axis=-1)
    x[0, 0] = 0.0
    ties = np.zeros(32)
    ties[:8] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.9]   # scale 1 (amax 7.9): ties to even, clamp
    x[1, 0, :32] = ties
    q = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    want = O.f64_to_bf16_bits(O.mxfp4_round_bits(bits(q)))
    qd = q.cuda()
    out = torch.empty_like(qd)
    Q.qsa_quantize_index_q(cfg, qd, out)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), want)
    got = O.bf16_bits_to_f64(bits(out)[1, 0, :8])
    assert got.tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0]


def test_scores_bit_exact_queries_rounded_in_the_kernel():
    wl = small_wl(4, 256, 64, 128, 32, 4, [3000, 9000], R=2)
    g = GpuState(wl, index_format=MX4)
    g.append_prefix()
    Q = g.Q
    pos0 = list(wl.prefixes)
    res = g.decode(pos0, 2)
    g.check_status()
    inp = res["inputs"]
    rows = g.rows(pos0, 2)
    n = len(pos0) * 2
    ld = (g.cache.max_blocks + 3) // 4 * 4
    scores = torch.full((n, ld), float("nan"), dtype=torch.float32, device="cuda")
    Q.qsa_index_score(g.cfg, rows, g.cache, inp["q_idx"], inp["w"], scores, ld, g.status)
    torch.cuda.synchronize()
    g.check_status()
    for i, s in enumerate(g.slots):
        orc = OracleSeq(wl, s, pos0[i] + 2)
        for j in range(2):
            ref = orc.row(pos0[i] + j, "mxfp4")
            nb = ref["n_blk"]
            assert np.array_equal(scores[i * 2 + j, :nb].cpu().numpy().astype(np.float64), ref["scores"])


FUSED = {
    "decode_main": (4, 2048, 64, 128, 32, 4, [32768, 2051, 2052], 1),
    "verify_R4": (4, 512, 64, 128, 32, 4, [5000, 12001], 4),
    "dI64_r8_bpp8": (8, 256, 16, 64, 8, 1, [300, 4097], 2),
}


@pytest.mark.parametrize("name", list(FUSED))
def test_fused_step_every_row(name):
    r, b, hi, di, hq, hkv, pre, R = FUSED[name]
    wl = small_wl(r, b, hi, di, hq, hkv, pre, R)
    g = GpuState(wl, extra_tokens=8, index_format=MX4)
    g.append_prefix()
    pos0 = list(wl.prefixes)
    res = g.decode(pos0, R)
    g.check_status()
    sel = res["sel"].cpu().numpy(); nsel = res["n_sel"].cpu().numpy(); out = bits(res["out"])
    for i, s in enumerate(g.slots):
        orc = OracleSeq(wl, s, pos0[i] + R)
        for j in range(R):
            row = i * R + j
            compare_row(out[row], sel[row], int(nsel[row]), orc.row(pos0[i] + j, "mxfp4"), g.cfg.topk)
        check_plane4(g, s, pos0[i] + R)


def test_steady_decode_batch32_prefix32k_every_row():
    """Batch 32 x 32k with the MXFP4 plane: every row's selection of two steps
    against the oracle's MXFP4 scores; outputs on sampled rows."""
    wl = S.workload(2)
    g = GpuState(wl, extra_tokens=8, index_format=MX4)
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
            compare_row(out[s], sel[s], int(nsel[s]), oracles[s].row(pos0[s], "mxfp4"), g.cfg.topk)
        pos0 = [p + 1 for p in pos0]
    assert log.check(wl, index_format="mxfp4") == 2 * wl.n_seq
