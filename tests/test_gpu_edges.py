"""GPU edge cases: shape variants against the oracle on every row (dense,
boundary, zero-block and sparse rows; verify form), tie-heavy scores, the
device error channel (desync, capacity, rewind, bad page), invariants
(page permutation, ablation, head permutation, w scaling), the standalone
stages against the fused step, and CUDA-graph capture of the fused step."""
import numpy as np
import pytest
import torch

from indexer_selected_sparse_gb300 import synth as S
from oracle import qsa_oracle as O
from tests.gpu_harness import GpuState, OracleSeq, bits, compare_row

pytestmark = pytest.mark.gpu


def small_wl(ratio, budget, h_i, d_i, hq, hkv, prefixes, R=1, seed=7, contiguous=False,
             int_range=(-8, 8)):
    sh = S.Shapes(ratio, budget, h_i, d_i, hq, hkv, 128, 64)
    return S.Workload("edge", seed, sh, list(prefixes), R, contiguous_pages=contiguous,
                      extra={"int_range": int_range})


def run_and_check_all_rows(wl, extra=8):
    g = GpuState(wl, extra_tokens=extra)
    g.append_prefix(chunk=3000)
    pos0 = list(wl.prefixes)
    R = wl.rows_per_seq
    res = g.decode(pos0, R)
    g.check_status()
    assert g.cache.ingested.cpu().tolist() == [p + R for p in pos0]
    sel = res["sel"].cpu().numpy(); nsel = res["n_sel"].cpu().numpy(); out = bits(res["out"])
    for i, s in enumerate(g.slots):
        orc = OracleSeq(wl, s, pos0[i] + R, lazy_kv=False)
        for j in range(R):
            row = i * R + j
            compare_row(out[row], sel[row], int(nsel[row]), orc.row(pos0[i] + j), g.cfg.topk)
    return g, res


SHAPES = {
    # ratio, budget, H_I, d_I, Hq, Hkv, prefixes (V = prefix + 1), R
    "r4_B32_tiny": (4, 32, 4, 64, 8, 1, [0, 1, 2, 3, 30, 33, 34, 35, 36, 200, 1000], 1),
    "r2_B64_mha1": (2, 64, 1, 64, 1, 1, [5, 62, 64, 65, 66, 700], 1),
    "r8_B256_gqa3": (8, 256, 33, 128, 12, 4, [100, 262, 263, 264, 3000], 1),
    "r16_B512_hkv2": (16, 512, 8, 64, 8, 2, [526, 527, 528, 5000], 1),
    "r4_B128_verify": (4, 128, 64, 128, 32, 4, [120, 129, 130, 131, 2000], 3),
    "r4_B8192_topk2048": (4, 8192, 16, 128, 16, 2, [8190, 8192, 20000], 1),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_shape_variants_every_row(name):
    r, b, hi, di, hq, hkv, pre, R = SHAPES[name]
    run_and_check_all_rows(small_wl(r, b, hi, di, hq, hkv, pre, R))


def test_tie_heavy_scores():
    # index q and k in {-1, 0, 1}: many equal scores, ties go to the lower block
    wl = small_wl(4, 64, 2, 64, 8, 1, [300, 1000, 4000], R=2, int_range=(-1, 1))
    run_and_check_all_rows(wl)


def test_desync_is_reported_and_nothing_written():
    wl = small_wl(4, 32, 4, 64, 8, 1, [100, 200])
    g = GpuState(wl)
    g.append_prefix()
    before_k = g.cache.k_pool.clone()
    before_ing = g.cache.ingested.clone()
    bad = [101, 200]                          # sequence 0 is one ahead of its counter
    inp = g.step_inputs(bad, 1)
    rows = g.rows(bad, 1, host_pos=False)
    out = torch.empty(2, 8, 128, dtype=torch.bfloat16, device="cuda")
    g.Q.qsa_append(g.cfg, rows, g.cache, inp["k"], inp["v"], inp["idx"], g.status)
    torch.cuda.synchronize()
    g.check_status(g.Q.QSA_ERR_DESYNC)
    ing = g.cache.ingested.cpu().tolist()
    assert ing[0] == 100 and ing[1] == 201    # the healthy sequence still advanced
    # the desynced sequence wrote nothing: only sequence 1's page changed
    pt = g.cache.page_table.cpu()
    diff = (g.cache.k_pool != before_k).any(dim=3).any(dim=2).any(dim=1).nonzero().flatten().tolist()
    assert diff == [int(pt[1][200 // 64])]


def test_capacity_host_and_device():
    wl = small_wl(4, 32, 4, 64, 8, 1, [100])
    g = GpuState(wl, extra_tokens=0)          # capacity = ceil(101 / 64) * 64 = 128
    g.append_prefix()
    cap = g.cache.capacity
    assert cap == 128
    inp = g.step_inputs([100], 29)
    with pytest.raises(g.Q.QsaError) as e:     # host copy of pos0 given: rejected before any launch
        g.Q.qsa_append(g.cfg, g.rows([100], 29), g.cache, inp["k"], inp["v"], inp["idx"], g.status)
    assert e.value.code == g.Q.QSA_ERR_CAPACITY and "capacity 128" in str(e.value)
    g.Q.qsa_append(g.cfg, g.rows([100], 29, host_pos=False), g.cache, inp["k"], inp["v"], inp["idx"], g.status)
    torch.cuda.synchronize()
    g.check_status(g.Q.QSA_ERR_CAPACITY)
    assert g.cache.ingested.cpu().tolist() == [100]
    g.status.zero_()
    inp = g.step_inputs([100], 28)             # exactly fills the capacity: fine
    g.Q.qsa_append(g.cfg, g.rows([100], 28), g.cache, inp["k"], inp["v"], inp["idx"], g.status)
    torch.cuda.synchronize()
    g.check_status()
    assert g.cache.ingested.cpu().tolist() == [128]


def test_rewind_errors_and_zero():
    wl = small_wl(4, 32, 4, 64, 8, 1, [10, 20])
    g = GpuState(wl)
    g.append_prefix()
    Q = g.Q
    ids = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    Q.qsa_rewind(g.cfg, ids, torch.tensor([11, 3], dtype=torch.int32, device="cuda"), g.cache.ingested, g.status)
    torch.cuda.synchronize()
    g.check_status(Q.QSA_ERR_REWIND)
    assert g.cache.ingested.cpu().tolist() == [10, 17]
    g.status.zero_()
    Q.qsa_rewind(g.cfg, ids, torch.tensor([10, 0], dtype=torch.int32, device="cuda"), g.cache.ingested, g.status)
    torch.cuda.synchronize()
    g.check_status()
    assert g.cache.ingested.cpu().tolist() == [0, 17]


def test_bad_page_id_is_reported():
    wl = small_wl(4, 32, 4, 64, 8, 1, [100])
    g = GpuState(wl)
    g.append_prefix()
    g.cache.page_table[0, 1] = g.cache.num_pages + 5   # points outside the pool
    res = g.decode([100], 1)
    g.check_status(g.Q.QSA_ERR_PAGE)


def test_page_permutation_invariance():
    wl = small_wl(4, 128, 16, 128, 16, 2, [700, 1500, 2600], R=2)
    a = GpuState(wl, contiguous=True)
    b = GpuState(wl, contiguous=False, page_seed=99)
    a.append_prefix(); b.append_prefix()
    ra = a.decode(list(wl.prefixes), 2)
    rb = b.decode(list(wl.prefixes), 2)
    a.check_status(); b.check_status()
    assert np.array_equal(bits(ra["out"]), bits(rb["out"]))
    assert torch.equal(ra["sel"], rb["sel"]) and torch.equal(ra["n_sel"], rb["n_sel"])


def stage_run(g, pos0, R, inp):
    """The standalone stages on an already-appended step."""
    Q = g.Q
    rows = g.rows(pos0, R)
    n = len(pos0) * R
    ld = (g.cache.max_blocks + 3) // 4 * 4
    scores = torch.full((n, ld), float("nan"), dtype=torch.float32, device="cuda")
    Q.qsa_index_score(g.cfg, rows, g.cache, inp["q_idx"], inp["w"], scores, ld, g.status)
    sel = torch.empty(n, g.cfg.topk, dtype=torch.int32, device="cuda")
    nsel = torch.empty(n, dtype=torch.int32, device="cuda")
    Q.qsa_topk_select(g.cfg, rows, scores, ld, sel, nsel, g.status)
    out = torch.empty(n, g.sh.n_q_heads, 128, dtype=torch.bfloat16, device="cuda")
    Q.qsa_gather_attn(g.cfg, rows, g.cache, inp["q"], sel, nsel, out, g.ws, g.status)
    torch.cuda.synchronize()
    return scores, sel, nsel, out


def test_stages_equal_fused_and_scores_exact():
    wl = small_wl(4, 256, 64, 128, 32, 4, [3000, 9000], R=1)
    g = GpuState(wl)
    g.append_prefix()
    pos0 = list(wl.prefixes)
    res = g.decode(pos0, 1)
    g.check_status()
    scores, sel, nsel, out = stage_run(g, pos0, 1, res["inputs"])
    g.check_status()
    assert torch.equal(sel, res["sel"]) and torch.equal(nsel, res["n_sel"])
    assert np.array_equal(bits(out), bits(res["out"]))
    for i, s in enumerate(g.slots):
        orc = OracleSeq(wl, s, pos0[i] + 1)
        ref = orc.row(pos0[i])
        n_blk = ref["n_blk"]
        assert np.array_equal(scores[i, :n_blk].cpu().numpy().astype(np.float64), ref["scores"])


def test_scores_head_permutation_and_w_scaling():
    wl = small_wl(4, 256, 64, 128, 32, 4, [5000], R=1)
    g = GpuState(wl)
    g.append_prefix()
    res = g.decode([5000], 1)
    inp = res["inputs"]
    s0, sel0, _, _ = stage_run(g, [5000], 1, inp)
    perm = torch.randperm(64, generator=torch.Generator().manual_seed(3)).cuda()
    inp2 = dict(inp, q_idx=inp["q_idx"][:, perm].contiguous(), w=inp["w"][:, perm].contiguous())
    s1, sel1, _, _ = stage_run(g, [5000], 1, inp2)
    n = 5001 // 4
    assert torch.equal(s0[:, :n], s1[:, :n]) and torch.equal(sel0, sel1)
    inp3 = dict(inp, w=(inp["w"] * 2).contiguous())
    s2, sel2, _, _ = stage_run(g, [5000], 1, inp3)
    assert torch.equal(s2[:, :n], 2 * s0[:, :n]) and torch.equal(sel2, sel0)


def test_ablation_of_unselected_tokens():
    wl = small_wl(4, 128, 16, 128, 16, 2, [3000], R=1)
    g = GpuState(wl)
    g.append_prefix()
    res = g.decode([3000], 1)
    inp = res["inputs"]
    sel = res["sel"][0].cpu().numpy()
    n_blk = 3001 // 4
    toks = O.token_set(sel, n_blk, 3001, 4)
    unsel = np.setdiff1d(np.arange(3001), toks)
    pt = g.cache.page_table[0].cpu().numpy()
    pages = torch.from_numpy(pt[unsel // 64]).long().cuda()
    offs = torch.from_numpy(unsel % 64).long().cuda()
    noise = torch.randn(len(unsel), 2, 128, device="cuda").to(torch.bfloat16)
    g.cache.k_pool[pages, offs] = noise
    g.cache.v_pool[pages, offs] = noise
    out = torch.empty_like(res["out"])
    rows = g.rows([3000], 1)
    g.Q.qsa_gather_attn(g.cfg, rows, g.cache, inp["q"], res["sel"], res["n_sel"], out, g.ws, g.status)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), bits(res["out"]))
    t = int(toks[5])
    g.cache.v_pool[int(pt[t // 64]), t % 64] += 1.0
    g.Q.qsa_gather_attn(g.cfg, rows, g.cache, inp["q"], res["sel"], res["n_sel"], out, g.ws, g.status)
    torch.cuda.synchronize()
    assert not np.array_equal(bits(out), bits(res["out"]))


def test_fused_step_captured_in_a_cuda_graph():
    wl = small_wl(4, 256, 64, 128, 32, 4, [3000, 4100, 900, 5000], R=1)
    eager = GpuState(wl); eager.append_prefix()
    cap = GpuState(wl); cap.append_prefix()
    pos0 = list(wl.prefixes)
    ref = eager.decode(pos0, 1)
    Q = cap.Q
    inp = cap.step_inputs(pos0, 1)
    rows = cap.rows(pos0, 1, host_pos=False)
    out = torch.empty_like(ref["out"])
    sel = torch.empty_like(ref["sel"]); nsel = torch.empty_like(ref["n_sel"])
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        Q.qsa_decode(cap.cfg, rows, cap.cache, inp["k"], inp["v"], inp["idx"], inp["q_idx"], inp["w"],
                     inp["q"], out, cap.ws, cap.status, sel_out=sel, n_sel_out=nsel)
    graph.replay()
    torch.cuda.synchronize()
    cap.check_status()
    assert np.array_equal(bits(out), bits(ref["out"])) and torch.equal(sel, ref["sel"])
    # replaying at the same positions desyncs the counters: reported, not silent
    graph.replay()
    torch.cuda.synchronize()
    cap.check_status(Q.QSA_ERR_DESYNC)
