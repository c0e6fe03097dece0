"""Pins of the CPU oracle against facts that do not come from the oracle itself:
values printed on the pages, hand-worked examples, closed forms, library
routines, brute force on tiny inputs, special cases and invariants.

Pages cited: "Agentic shootout -- Atlas x Flash-Next research" (reports
"Flash-Next support: vLLM vs Atlas" (a)6, "PR 16 review ... (Claude's
review)" (a), "Flash-Next support: llama.cpp vs Atlas" (a)3) and "Atlas
Flash-Next defect investigations" (Report A Defect 1, Report P Defect 5).
"""
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import qsa_oracle as O
from tests.conftest import read_golden_table

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def bf16(vals):
    """bf16 bit patterns of values, via torch's own fp32 -> bf16 conversion."""
    t = torch.as_tensor(np.asarray(vals, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().astype(np.uint16)


def state_from_raw(raw, ratio, idx_dim, capacity=None):
    raw = np.asarray(raw, np.float32).reshape(-1, idx_dim)
    n = raw.shape[0]
    st = O.SeqState(ratio, 1, 4, idx_dim, capacity or max(n, 4))
    z = np.zeros((n, 1, 4), np.uint16)
    st.append(0, z, z, bf16(raw))
    return st


# ---------------------------------------------------------------------------
# bf16 rounding: library routine + hand cases
# ---------------------------------------------------------------------------

def test_bf16_rounding_matches_torch_on_fp32_values():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = O.f64_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_rounding_hand_cases():
    # spacing at 1.0 is 2^-7: 1 + 2^-8 is a tie -> even (1.0);
    # 1 + 3*2^-8 is a tie between 1+2^-7 (odd) and 1+2^-6 (even) -> 1+2^-6
    assert O.round_bf16(1 + 2**-8) == 1.0
    assert O.round_bf16(1 + 3 * 2**-8) == 1 + 2**-6
    assert O.round_bf16(1 + 2**-8 + 2**-30) == 1 + 2**-7     # above the tie
    assert O.round_bf16(-(1 + 2**-8)) == -1.0
    # fp64-only information must not be lost to a double rounding via fp32:
    # 1 + 2^-8 + 2^-40 rounds up in one step, but to 1.0 through fp32
    assert O.round_bf16(1 + 2**-8 + 2**-40) == 1 + 2**-7
    assert math.isinf(O.round_bf16(2.0**128 * 0.9999999))
    assert O.round_bf16(2.0**-133) == 2.0**-133               # smallest subnormal
    assert O.round_bf16(2.0**-135) == 0.0


# ---------------------------------------------------------------------------
# Pooling
# ---------------------------------------------------------------------------

def test_pool_hand_cases(golden_cases):
    c = golden_cases["pool_round"]
    raw = bf16(np.array(c["raw"]).reshape(-1, 1))
    assert O.bf16_bits_to_f64(O.pool_block(raw))[0] == c["blk"][0][0]
    raw = bf16(np.array([[1.0], [2.0], [3.0], [5.0]]))       # 11/4 exact
    assert O.bf16_bits_to_f64(O.pool_block(raw))[0] == 2.75


def test_worked_example_blocks(golden_cases):
    for name in ("select", "tie"):
        c = golden_cases[name]
        r = int(c["ratio"][0][0])
        st = state_from_raw(c["raw"], r, 2)
        assert st.n_blocks == len(c["blk"])
        got = O.bf16_bits_to_f64(st.idx_blk[: st.n_blocks])
        assert np.array_equal(got, np.array(c["blk"]))


def test_pool_of_integer_keys_is_exact():
    # ratio 4, integer keys in [-8, 8]: every mean is a multiple of 1/4 with
    # magnitude <= 8, exact in bf16, so the pooled key equals the exact mean
    rng = np.random.default_rng(3)
    raw = rng.integers(-8, 9, size=(64, 32)).astype(np.float64)
    st = state_from_raw(raw, 4, 32)
    exact = raw.reshape(16, 4, 32).mean(axis=1)
    assert np.array_equal(O.bf16_bits_to_f64(st.idx_blk[:16]), exact)


# ---------------------------------------------------------------------------
# Scores
# ---------------------------------------------------------------------------

def test_worked_example_scores_and_selection(golden_cases):
    for name in ("select", "tie"):
        c = golden_cases[name]
        r = int(c["ratio"][0][0])
        K = int(c["budget"][0][0]) // r
        st = state_from_raw(c["raw"], r, 2)
        s = O.block_scores(bf16(c["q_idx"]), np.array(c["w"][0]), st.idx_blk[: st.n_blocks])
        assert np.array_equal(s, np.array(c["scores"][0]))
        sel = O.select_blocks(s, K)
        assert sel.tolist() == [int(v) for v in c["sel"][0]]
        toks = O.token_set(sel, st.n_blocks, int(c["visible"][0][0]), r)
        assert toks.tolist() == [int(v) for v in c["tokens"][0]]


def test_score_closed_forms():
    e0 = np.zeros(8); e0[0] = 1
    k = np.array([[3, -1, 2, 0, 0, 0, 0, 5], [-4, 1, 1, 1, 1, 1, 1, 1]], np.float64)
    # one head, unit query: score = max(0, k[0])
    s = O.block_scores(bf16([e0]), [1.0], bf16(k))
    assert s.tolist() == [3.0, 0.0]
    # two heads, w = (0.5, 2): head 0 reads dim 0, head 1 reads dim 7
    e7 = np.zeros(8); e7[7] = 1
    s = O.block_scores(bf16([e0, e7]), [0.5, 2.0], bf16(k))
    assert s.tolist() == [0.5 * 3 + 2 * 5, 0.5 * 0 + 2 * 1]
    # the ReLU acts per head, before the weighted head sum: a negative head
    # cannot cancel a positive one
    s = O.block_scores(bf16([e0, -e0]), [1.0, 1.0], bf16(k))
    assert s.tolist() == [3.0, 4.0]


def test_score_invariants():
    rng = np.random.default_rng(5)
    q = rng.integers(-8, 9, size=(6, 16)).astype(np.float64)
    k = rng.integers(-8, 9, size=(40, 16)).astype(np.float64)
    w = 2.0 ** rng.integers(-2, 2, size=6)
    s = O.block_scores(bf16(q), w, bf16(k))
    perm = rng.permutation(6)
    assert np.array_equal(O.block_scores(bf16(q[perm]), w[perm], bf16(k)), s)
    assert np.array_equal(O.block_scores(bf16(q), 2 * w, bf16(k)), 2 * s)
    # w == 1 (weight-free) equals the sum of per-head ReLU dots
    s1 = O.block_scores(bf16(q), np.ones(6), bf16(k))
    brute = [sum(max(0.0, float(np.dot(q[h], k[b]))) for h in range(6)) for b in range(40)]
    assert s1.tolist() == brute


# ---------------------------------------------------------------------------
# Selection
# ---------------------------------------------------------------------------

def brute_topk(scores, K):
    idx = sorted(range(len(scores)), key=lambda b: (-scores[b], b))
    return sorted(idx[:K]) if len(scores) > K else list(range(len(scores)))


def test_selection_brute_force_with_ties():
    rng = np.random.default_rng(7)
    for trial in range(300):
        n = int(rng.integers(1, 64))
        K = int(rng.integers(1, 20))
        H = int(rng.integers(1, 5))
        q = rng.integers(-1, 2, size=(H, 4)).astype(np.float64)
        k = rng.integers(-1, 2, size=(n, 4)).astype(np.float64)
        s = O.block_scores(bf16(q), np.ones(H), bf16(k))
        assert O.select_blocks(s, K).tolist() == brute_topk(s.tolist(), K)


def test_selection_special_cases():
    K = 5
    assert O.select_blocks(np.full(12, 3.5), K).tolist() == [0, 1, 2, 3, 4]
    assert O.select_blocks(np.zeros(12), K).tolist() == [0, 1, 2, 3, 4]
    assert O.select_blocks(np.arange(12.0), K).tolist() == [7, 8, 9, 10, 11]
    assert O.select_blocks(np.arange(12.0)[::-1].copy(), K).tolist() == [0, 1, 2, 3, 4]
    assert O.select_blocks(np.arange(3.0), K).tolist() == [0, 1, 2]   # n <= K
    # all heads ReLU'd to zero -> all scores 0 -> the first K blocks
    q = -np.ones((2, 4)); k = np.ones((9, 4))
    s = O.block_scores(bf16(q), [1.0, 1.0], bf16(k))
    assert O.select_blocks(s, 3).tolist() == [0, 1, 2]


def test_raising_an_unselected_block_enters_the_set():
    rng = np.random.default_rng(11)
    s = rng.permutation(50).astype(np.float64)       # distinct scores
    K = 8
    sel = O.select_blocks(s, K)
    out = next(b for b in range(50) if b not in sel)
    weakest = min(sel, key=lambda b: s[b])
    s2 = s.copy(); s2[out] = s[sel].max() + 1
    sel2 = O.select_blocks(s2, K)
    assert out in sel2 and weakest not in sel2
    assert set(sel2) == (set(sel) - {weakest}) | {out}


# ---------------------------------------------------------------------------
# Inert bound and token set (values printed on the pages)
# ---------------------------------------------------------------------------

def test_inert_bound_from_pages():
    for budget, ratio, topk, bound, width in [[int(v) for v in row] for row in read_golden_table("inert_bound.txt")]:
        assert budget // ratio == topk
        # visible == bound: every complete block fits in the budget -> dense
        n_blk = bound // ratio
        assert n_blk <= topk
        sel = O.select_blocks(np.arange(float(n_blk)), topk)
        toks = O.token_set(sel, n_blk, bound, ratio)
        assert toks.tolist() == list(range(bound))
        # visible == bound + 1: one block too many -> selection active
        n_blk = (bound + 1) // ratio
        assert n_blk == topk + 1
        sel = O.select_blocks(np.arange(float(n_blk)), topk)
        assert len(sel) == topk and 0 not in sel
        # the widest token set is K * ratio + (ratio - 1) = the buffer width
        worst = max(len(O.token_set(np.arange(min(v // ratio, topk)), v // ratio, v, ratio))
                    for v in range(bound - 8, bound + 40))
        assert worst == width


def test_indexer_memory_from_pages():
    for tokens, d, ratio, raw_b, blk_b, total_mb in read_golden_table("indexer_memory.txt"):
        st = O.SeqState(int(ratio), 1, 4, int(d), int(tokens))
        assert st.idx_raw.nbytes == int(raw_b)
        assert st.idx_blk.nbytes == int(blk_b)
        assert round((st.idx_raw.nbytes + st.idx_blk.nbytes) / 1e6, 1) == float(total_mb)


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def test_worked_example_attention(golden_cases):
    c = golden_cases["attend"]
    q = bf16(c["q"])
    k = bf16(np.array(c["k"]).reshape(2, 1, 4))
    v = bf16(np.array(c["v"]).reshape(2, 1, 4))
    out = O.gqa_attention(q, k, v)
    assert np.allclose(out[0], c["out"][0], rtol=0, atol=1e-15)
    assert O.bf16_bits_to_f64(O.f64_to_bf16_bits(out))[0].tolist() == c["out_bf16"][0]


def test_attention_special_cases():
    rng = np.random.default_rng(13)
    D = 16
    q = bf16(rng.standard_normal((4, D)))
    # one token: the output is that token's V row of the head's group
    k = bf16(rng.standard_normal((1, 2, D))); v = bf16(rng.standard_normal((1, 2, D)))
    out = O.gqa_attention(q, k, v)
    vv = O.bf16_bits_to_f64(v)
    assert np.array_equal(out, vv[0][[0, 0, 1, 1]])
    # all V rows equal: the output is that row whatever the weights
    k = bf16(rng.standard_normal((9, 2, D)))
    row = rng.standard_normal((2, D))
    v = bf16(np.broadcast_to(row, (9, 2, D)))
    out = O.gqa_attention(q, k, v)
    assert np.allclose(out, O.bf16_bits_to_f64(v)[0][[0, 0, 1, 1]], atol=1e-14)
    # q == 0: uniform weights -> the mean of the V rows
    v = bf16(rng.standard_normal((9, 2, D)))
    out = O.gqa_attention(bf16(np.zeros((4, D))), k, v)
    vv = O.bf16_bits_to_f64(v)
    assert np.allclose(out, vv.mean(axis=0)[[0, 0, 1, 1]], atol=1e-14)


def test_attention_textbook_single_head():
    # Hq = Hkv = 1: out = sum_t softmax(q.k_t / sqrt(D))_t v_t, written out
    rng = np.random.default_rng(17)
    D, T = 8, 5
    q = rng.standard_normal(D); k = rng.standard_normal((T, D)); v = rng.standard_normal((T, D))
    qb, kb, vb = bf16([q]), bf16(k.reshape(T, 1, D)), bf16(v.reshape(T, 1, D))
    qv, kv, vv = (O.bf16_bits_to_f64(x) for x in (qb, kb, vb))
    e = [math.exp(float(np.dot(qv[0], kv[t, 0])) / math.sqrt(D)) for t in range(T)]
    want = sum(e[t] * vv[t, 0] for t in range(T)) / sum(e)
    assert np.allclose(O.gqa_attention(qb, kb, vb)[0], want, atol=1e-13)


def test_gqa_head_mapping_contiguous_groups():
    # Hq = 4, Hkv = 2: heads 0,1 -> kv 0 and heads 2,3 -> kv 1
    D = 8
    k = bf16(np.zeros((3, 2, D)))
    v = np.zeros((3, 2, D)); v[:, 0, :] = 1.0; v[:, 1, :] = -2.0
    out = O.gqa_attention(bf16(np.ones((4, D))), k, bf16(v))
    assert out[:, 0].tolist() == [1.0, 1.0, -2.0, -2.0]
    assert [O.kv_head_of(h, 32, 4) for h in (0, 7, 8, 31)] == [0, 0, 1, 3]


def make_state(rng, n, ratio=4, hkv=2, D=16, dI=8, cap=None):
    st = O.SeqState(ratio, hkv, D, dI, cap or n + 16)
    st.append(0, bf16(rng.standard_normal((n, hkv, D))), bf16(rng.standard_normal((n, hkv, D))),
              bf16(rng.integers(-8, 9, size=(n, dI))))
    return st


def test_dense_identity_at_and_below_inert_bound():
    rng = np.random.default_rng(19)
    ratio, budget = 4, 32
    bound = budget + ratio - 1
    st = make_state(rng, bound + 5, ratio)
    for V in (17, 1, 2, 3, 4, 5, bound - 1, bound):
        q = bf16(rng.standard_normal((4, 16)))
        qi = bf16(rng.integers(-8, 9, size=(3, 8))); w = np.ones(3)
        res = O.attend_row(st, V - 1, qi, w, q, budget // ratio)
        assert res["tokens"].tolist() == list(range(V))
        dense = O.dense_attention(q, st.K[:V], st.V[:V], 2)
        assert np.max(np.abs(res["out"] - dense)) <= 1e-12
    # one past the bound: selection is active and drops exactly one block
    res = O.attend_row(st, bound, qi, w, q, budget // ratio)
    assert res["n_blk"] == budget // ratio + 1 and len(res["sel"]) == budget // ratio
    assert len(res["tokens"]) == budget


def test_ablation_of_unselected_tokens():
    rng = np.random.default_rng(23)
    ratio, topk = 4, 4
    st = make_state(rng, 61, ratio)
    q = bf16(rng.standard_normal((4, 16)))
    qi = bf16(rng.integers(-8, 9, size=(3, 8))); w = np.array([1.0, 0.5, 2.0])
    res = O.attend_row(st, 60, qi, w, q, topk)
    unsel = np.setdiff1d(np.arange(61), res["tokens"])
    assert len(unsel) > 0
    st.K[unsel] = bf16(rng.standard_normal((len(unsel), 2, 16)))
    st.V[unsel] = bf16(rng.standard_normal((len(unsel), 2, 16)))
    res2 = O.attend_row(st, 60, qi, w, q, topk)
    assert np.array_equal(res2["out"], res["out"])
    t = res["tokens"][0]
    st.V[t] = bf16(rng.standard_normal((2, 16)))
    res3 = O.attend_row(st, 60, qi, w, q, topk)
    assert not np.array_equal(res3["out"], res["out"])


def test_reused_selection_at_its_own_position_is_attend_row():
    # a shared indexer layer reuses the top-k of the full layer at the same position
    rng = np.random.default_rng(29)
    ratio, topk = 4, 4
    st = make_state(rng, 61, ratio)
    for pos in (60, 41, 18):
        q = bf16(rng.standard_normal((4, 16)))
        qi = bf16(rng.integers(-8, 9, size=(3, 8))); w = np.array([1.0, 0.5, 2.0])
        ref = O.attend_row(st, pos, qi, w, q, topk)
        got = O.attend_row_reused(st, pos, ref["sel"], pos, q)
        assert np.array_equal(got["tokens"], ref["tokens"])
        assert np.array_equal(got["out_bf16"], ref["out_bf16"])


def test_reused_dense_selection_stays_exactly_dense():
    # a selection made at or below the inert bound holds every block; reused at a
    # later position (past the bound, blocks completed since) it must still
    # cover every visible token: exactly dense attention
    rng = np.random.default_rng(31)
    ratio, budget = 4, 32
    bound = budget + ratio - 1
    st = make_state(rng, bound + 12, ratio)
    qi = bf16(rng.integers(-8, 9, size=(3, 8))); w = np.ones(3)
    for sel_V in (bound, bound - 2, 9):
        sel = O.attend_row(st, sel_V - 1, qi, w, bf16(rng.standard_normal((4, 16))), budget // ratio)["sel"]
        for V in (sel_V, sel_V + 1, sel_V + 3, sel_V + 4, bound + 12):
            q = bf16(rng.standard_normal((4, 16)))
            got = O.attend_row_reused(st, V - 1, sel, sel_V - 1, q)
            assert got["tokens"].tolist() == list(range(V))
            dense = O.dense_attention(q, st.K[:V], st.V[:V], 2)
            assert np.max(np.abs(got["out"] - dense)) <= 1e-12


def test_reused_sparse_selection_token_set():
    rng = np.random.default_rng(37)
    ratio, topk = 4, 4
    st = make_state(rng, 80, ratio)
    qi = bf16(rng.integers(-8, 9, size=(3, 8))); w = np.array([1.0, 0.5, 2.0])
    q = bf16(rng.standard_normal((4, 16)))
    ref = O.attend_row(st, 60, qi, w, q, topk)       # 61 visible: 15 blocks, tail {60}
    for pos in (60, 61, 62, 63, 64, 70, 79):
        got = O.attend_row_reused(st, pos, ref["sel"], 60, q)
        body = [b * ratio + j for b in ref["sel"] for j in range(ratio)]
        assert got["tokens"].tolist() == body + list(range(60, pos + 1))
    with pytest.raises(ValueError):
        O.attend_row_reused(st, 59, ref["sel"], 60, q)       # selection from the future
    with pytest.raises(O.DesyncError):
        O.attend_row_reused(st, 80, ref["sel"], 60, q)       # row not ingested


# ---------------------------------------------------------------------------
# Pre-indexer: Gemma RMSNorm and NeoX RoPE
# ---------------------------------------------------------------------------

def test_gemma_rmsnorm_closed_forms():
    g0 = np.zeros(4)
    assert np.allclose(O.gemma_rmsnorm(np.full(4, 3.0), g0, 0.0), 1.0, atol=1e-15)
    assert np.allclose(O.gemma_rmsnorm(np.full(4, -0.5), g0, 0.0), -1.0, atol=1e-15)
    # [3, 4]: mean square 12.5, rms 5 / sqrt(2); gain 1 + gamma
    got = O.gemma_rmsnorm(np.array([3.0, 4.0]), np.array([0.0, 1.0]), 0.0)
    assert np.allclose(got, [3 * math.sqrt(2) / 5, 2 * 4 * math.sqrt(2) / 5], atol=1e-15)
    rng = np.random.default_rng(41)
    x = rng.standard_normal((5, 16)); g = rng.standard_normal(16) * 0.1
    assert np.allclose(O.gemma_rmsnorm(7.5 * x, g, 0.0), O.gemma_rmsnorm(x, g, 0.0), atol=1e-13)
    y = O.gemma_rmsnorm(x, np.zeros(16), 0.0)
    assert np.allclose(np.mean(y * y, axis=-1), 1.0, atol=1e-13)   # unit RMS before the gain
    assert np.all(O.gemma_rmsnorm(np.zeros(8), np.zeros(8), 1e-6) == 0.0)


def test_rope_neox_closed_forms():
    x = np.array([1.0, 0.0, 0.0, 1.0])
    # rotary 4, base 1: both pairs turn by the position; a quarter turn maps
    # (x0, x2) = (1, 0) -> (0, 1) and (x1, x3) = (0, 1) -> (-1, 0)
    assert np.allclose(O.rope_neox(x, math.pi / 2, 4, 1.0), [0.0, -1.0, 1.0, 0.0], atol=1e-15)
    rng = np.random.default_rng(43)
    v = rng.standard_normal(128)
    assert np.array_equal(O.rope_neox(v, 0, 64, 1e4), v)                 # position 0: identity
    assert np.array_equal(O.rope_neox(v, 123, 64, 1e4)[64:], v[64:])     # dims past rotary untouched
    # pair i of a 64-dim rotary at base 1e4 turns by pos * 1e4^(-i/32): pair 16 at pos 100 -> 1 rad
    e = np.zeros(128); e[16] = 1.0
    r = O.rope_neox(e, 100, 64, 1e4)
    assert abs(r[16] - math.cos(1.0)) < 1e-12 and abs(r[48] - math.sin(1.0)) < 1e-12
    assert np.count_nonzero(np.abs(r) > 1e-15) == 2
    # rotations: pair norms kept, composition adds angles, dot products see only the offset
    a, b = 37, 1291
    ra = O.rope_neox(v, a, 64, 1e4)
    assert np.allclose(ra[:32] ** 2 + ra[32:64] ** 2, v[:32] ** 2 + v[32:64] ** 2, atol=1e-12)
    assert np.allclose(O.rope_neox(ra, b, 64, 1e4), O.rope_neox(v, a + b, 64, 1e4), atol=1e-9)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    d1 = O.rope_neox(q, 5000, 64, 1e4)[:64] @ O.rope_neox(k, 4000, 64, 1e4)[:64]
    d2 = O.rope_neox(q, 1000, 64, 1e4)[:64] @ k[:64]
    assert abs(d1 - d2) < 1e-9


def test_pre_indexed_blocks_norm_then_rope_at_the_first_position():
    # raw keys constant over each block: the mean is that key; the compressed key
    # must be RoPE(GemmaRMSNorm(key)) at the block's first position b * ratio
    rng = np.random.default_rng(47)
    dI, ratio = 128, 4
    pre = O.PreIndexer(rng.standard_normal(dI) * 0.2, rng.standard_normal(dI) * 0.2, 1e-6, 1e4, 64)
    st = O.SeqState(ratio, 1, 16, dI, 64, pre=pre)
    keys = rng.integers(-8, 9, size=(5, dI)).astype(np.float64)
    raw = np.repeat(keys, ratio, axis=0)
    z = np.zeros((5 * ratio, 1, 16), np.uint16)
    st.append(0, z, z, O.f64_to_bf16_bits(raw))
    for b in range(5):
        want = O.f64_to_bf16_bits(O.rope_neox(O.gemma_rmsnorm(keys[b], pre.gamma_k, 1e-6), b * ratio, 64, 1e4))
        assert np.array_equal(st.idx_blk[b], want), b
    # queries: per-head norm, then RoPE at the row's position
    qh = rng.integers(-8, 9, size=(3, dI)).astype(np.float64)
    got = O.pre_index_query(O.f64_to_bf16_bits(qh), 77, pre)
    want = O.f64_to_bf16_bits(O.rope_neox(O.gemma_rmsnorm(qh, pre.gamma_q, 1e-6), 77, 64, 1e4))
    assert np.array_equal(got, want)
    # a block's score sees only the offset between the row and the block start
    qn = O.gemma_rmsnorm(qh[0], pre.gamma_q, 1e-6)
    kn = O.gemma_rmsnorm(keys[2], pre.gamma_k, 1e-6)
    s1 = O.rope_neox(qn, 77, 64, 1e4) @ O.rope_neox(kn, 8, 64, 1e4)
    s2 = O.rope_neox(qn, 77 + 4000, 64, 1e4) @ O.rope_neox(kn, 8 + 4000, 64, 1e4)
    assert abs(s1 - s2) < 1e-9


# Interleaved MRoPE: a position is a (t, h, w) triple; NeoX pair i turns by h
# when i % 3 == 1 below 3 x the height section, by w when i % 3 == 2 below
# 3 x the width section, and by t otherwise


def pairs_moved_by_each_axis(section, rotary_dim=64, theta=1e4):
    """For each coordinate of the position triple, the NeoX pairs it turns,
    found by rotating unit vectors and moving one coordinate at a time."""
    moved = {0: [], 1: [], 2: []}
    for i in range(rotary_dim // 2):
        e = np.zeros(rotary_dim); e[i] = 1.0
        still = O.rope_neox(e, (0, 0, 0), rotary_dim, theta, section)
        for ax in range(3):
            p = [0, 0, 0]; p[ax] = 7
            if not np.allclose(O.rope_neox(e, tuple(p), rotary_dim, theta, section), still, atol=1e-12):
                moved[ax].append(i)
    return moved


def test_mrope_pairs_follow_the_interleave_and_its_section_bounds():
    # the pages' sections [11, 11, 10] over 64 rotary dims: t, h, w in turn to the end
    m = pairs_moved_by_each_axis((11, 11, 10))
    assert m[0] == [0, 3, 6, 9, 12, 15, 18, 21, 24, 27, 30]
    assert m[1] == [1, 4, 7, 10, 13, 16, 19, 22, 25, 28, 31]
    assert m[2] == [2, 5, 8, 11, 14, 17, 20, 23, 26, 29]
    # sections [16, 8, 8]: the height and width bounds end the interleave at pair 24
    m = pairs_moved_by_each_axis((16, 8, 8))
    assert m[0] == [0, 3, 6, 9, 12, 15, 18, 21] + list(range(24, 32))
    assert m[1] == [1, 4, 7, 10, 13, 16, 19, 22]
    assert m[2] == [2, 5, 8, 11, 14, 17, 20, 23]
    # every pair turns with exactly one axis, as many pairs per axis as its section
    for sec in ((11, 11, 10), (16, 8, 8), (12, 10, 10), (32, 0, 0)):
        m = pairs_moved_by_each_axis(sec)
        assert sorted(m[0] + m[1] + m[2]) == list(range(32))
        assert [len(m[a]) for a in range(3)] == list(sec)
    with pytest.raises(ValueError):
        O.PreIndexer(np.zeros(128), np.zeros(128), 1e-6, 1e4, 64, mrope_section=(11, 11, 11))


def test_mrope_is_plain_rope_for_text_and_sees_only_per_axis_offsets():
    rng = np.random.default_rng(53)
    sec = (11, 11, 10)
    v = rng.standard_normal(128)
    for p in (0, 5, 4097, 32768):   # a text token (t = h = w = p) turns as plain RoPE at p, bit for bit
        assert np.array_equal(O.rope_neox(v, (p, p, p), 64, 1e4, sec), O.rope_neox(v, p, 64, 1e4))
        assert np.array_equal(O.rope_neox(v, p, 64, 1e4, sec), O.rope_neox(v, p, 64, 1e4))
    P1, P2 = (40, 3, 17), (900, 12, 5)
    r1 = O.rope_neox(v, P1, 64, 1e4, sec)
    assert np.allclose(r1[:32] ** 2 + r1[32:64] ** 2, v[:32] ** 2 + v[32:64] ** 2, atol=1e-12)
    both = tuple(a + b for a, b in zip(P1, P2))
    assert np.allclose(O.rope_neox(r1, P2, 64, 1e4, sec), O.rope_neox(v, both, 64, 1e4, sec), atol=1e-9)
    assert np.array_equal(O.rope_neox(v, P1, 64, 1e4, sec)[64:], v[64:])
    q, k = rng.standard_normal(128), rng.standard_normal(128)

    def dot(pq, pk):
        return O.rope_neox(q, pq, 64, 1e4, sec)[:64] @ O.rope_neox(k, pk, 64, 1e4, sec)[:64]
    d1 = dot((5000, 40, 60), (4000, 30, 70))
    assert abs(d1 - dot((1000, 10, 0), (0, 0, 10))) < 1e-9      # the same offsets on every axis
    assert abs(d1 - dot((5000, 41, 60), (4000, 30, 70))) > 1e-6  # one row further down: another score


def test_mrope_blocks_rope_at_their_first_tokens_triple():
    rng = np.random.default_rng(59)
    dI, ratio, sec = 128, 4, (11, 11, 10)
    pre = O.PreIndexer(rng.standard_normal(dI) * 0.2, rng.standard_normal(dI) * 0.2, 1e-6, 1e4, 64,
                       mrope_section=sec)
    # an image run (t fixed, (h, w) walking a 4-wide grid), then text
    mpos = np.array([(10, 10 + i // 4, 10 + i % 4) for i in range(12)] + [(14 + i, 14 + i, 14 + i) for i in range(8)])
    keys = rng.integers(-8, 9, size=(5, dI)).astype(np.float64)
    raw = O.f64_to_bf16_bits(np.repeat(keys, ratio, axis=0))
    z = np.zeros((5 * ratio, 1, 16), np.uint16)
    st = O.SeqState(ratio, 1, 16, dI, 64, pre=pre)
    st.append(0, z, z, raw, mpos=mpos)
    for b in range(5):
        kn = O.gemma_rmsnorm(keys[b], pre.gamma_k, 1e-6)
        assert np.array_equal(st.idx_blk[b], O.f64_to_bf16_bits(O.rope_neox(kn, tuple(mpos[b * ratio]), 64, 1e4, sec)))
    # block 1 spans (10, 11, 10) .. (10, 11, 13): its last token's triple gives another key
    kn = O.gemma_rmsnorm(keys[1], pre.gamma_k, 1e-6)
    assert not np.array_equal(st.idx_blk[1], O.f64_to_bf16_bits(O.rope_neox(kn, tuple(mpos[7]), 64, 1e4, sec)))
    # a block completed by a later append uses the triple stored with its first token
    st2 = O.SeqState(ratio, 1, 16, dI, 64, pre=pre)
    st2.append(0, z[:6], z[:6], raw[:6], mpos=mpos[:6])
    st2.append(6, z[6:], z[6:], raw[6:], mpos=mpos[6:])
    assert np.array_equal(st2.idx_blk[:5], st.idx_blk[:5])
    # text positions (the default) reduce to the plain pre-indexer
    plain = O.PreIndexer(pre.gamma_q, pre.gamma_k, 1e-6, 1e4, 64)
    a, b_ = O.SeqState(ratio, 1, 16, dI, 64, pre=pre), O.SeqState(ratio, 1, 16, dI, 64, pre=plain)
    a.append(0, z, z, raw); b_.append(0, z, z, raw)
    assert np.array_equal(a.idx_blk[:5], b_.idx_blk[:5])


def test_mrope_attention_heads_at_their_own_triples():
    rng = np.random.default_rng(61)
    sec, D, n = (11, 11, 10), 128, 9
    att = O.AttnOptions(rng.standard_normal(D) * 0.1, rng.standard_normal(D) * 0.1, 1e-6, 1e4, 64, mrope_section=sec)
    mpos = np.array([(3, 3 + i % 3, 3 + i // 3) for i in range(n)])
    k, v = bf16(rng.standard_normal((n, 2, D))), bf16(rng.standard_normal((n, 2, D)))
    st = O.SeqState(4, 2, D, 8, 16, attn=att)
    st.append(0, k, v, np.zeros((n, 8), np.uint16), mpos=mpos)
    for t in range(n):
        assert np.array_equal(st.K[t], O.prep_heads(k[t], tuple(mpos[t]), att.gamma_k, 1e-6, 64, 1e4, sec))
    # the row's query heads turn at the row's own triple
    q = bf16(rng.standard_normal((4, D)))
    qp = (6, 5, 4)
    got = O.attend_row(st, n - 1, np.zeros((1, 8), np.uint16), np.ones(1), q, 4, attn=att, q_mpos=qp)
    q_prep = O.prep_heads(q, qp, att.gamma_q, 1e-6, 64, 1e4, sec)
    ref = O.attend_row(st, n - 1, np.zeros((1, 8), np.uint16), np.ones(1), q_prep, 4)
    assert np.array_equal(got["out"], ref["out"])
    other = O.attend_row(st, n - 1, np.zeros((1, 8), np.uint16), np.ones(1), q, 4, attn=att, q_mpos=(6, 5, 5))
    assert not np.array_equal(got["out"], other["out"])


# ---------------------------------------------------------------------------
# State: append / rewind / chunking / counters
# ---------------------------------------------------------------------------

def rows(rng, n, hkv=2, D=16, dI=8):
    return (bf16(rng.standard_normal((n, hkv, D))), bf16(rng.standard_normal((n, hkv, D))),
            bf16(rng.integers(-8, 9, size=(n, dI))))


def same_state(a, b):
    n = a.ingested
    return (a.ingested == b.ingested and np.array_equal(a.K[:n], b.K[:n])
            and np.array_equal(a.V[:n], b.V[:n]) and np.array_equal(a.idx_raw[:n], b.idx_raw[:n])
            and np.array_equal(a.idx_blk[: a.n_blocks], b.idx_blk[: b.n_blocks]))


def test_chunked_and_token_by_token_append_agree():
    rng = np.random.default_rng(29)
    k, v, i = rows(rng, 37)
    one = O.SeqState(4, 2, 16, 8, 64); one.append(0, k, v, i)
    chunks = O.SeqState(4, 2, 16, 8, 64)
    for a, b in ((0, 5), (5, 6), (6, 20), (20, 37)):
        chunks.append(a, k[a:b], v[a:b], i[a:b])
    tok = O.SeqState(4, 2, 16, 8, 64)
    for t in range(37):
        tok.append(t, k[t:t + 1], v[t:t + 1], i[t:t + 1])
    assert same_state(one, chunks) and same_state(one, tok)
    assert one.n_blocks == 9


def test_rewind_then_reappend_equals_never_drafting():
    rng = np.random.default_rng(31)
    k, v, i = rows(rng, 30)
    dk, dv, di = rows(rng, 3)
    ref = O.SeqState(4, 2, 16, 8, 64); ref.append(0, k, v, i)
    st = O.SeqState(4, 2, 16, 8, 64); st.append(0, k[:27], v[:27], i[:27])
    st.append(27, dk, dv, di)          # three draft tokens complete block 6 (tokens 24..27)
    st.rewind(3)
    assert st.ingested == 27 and st.n_blocks == 6
    st.append(27, k[27:], v[27:], i[27:])
    assert same_state(st, ref)
    # the re-completed block 6 was pooled from the new raw rows
    assert np.array_equal(st.idx_blk[6], O.pool_block(i[24:28]))
    assert not np.array_equal(O.pool_block(np.concatenate([i[24:27], di[:1]])), st.idx_blk[6])


def test_counter_discipline():
    rng = np.random.default_rng(37)
    k, v, i = rows(rng, 8)
    st = O.SeqState(4, 2, 16, 8, 10)
    st.append(0, k[:4], v[:4], i[:4])
    assert st.ingested == 4
    with pytest.raises(O.DesyncError):
        st.append(5, k[4:5], v[4:5], i[4:5])       # pos != ingested
    with pytest.raises(O.DesyncError):
        st.append(3, k[4:5], v[4:5], i[4:5])
    with pytest.raises(O.CapacityError):
        st.append(4, np.concatenate([k, k[:1]]), np.concatenate([v, v[:1]]), np.concatenate([i, i[:1]]))
    with pytest.raises(ValueError):
        st.rewind(5)
    st.rewind(4)
    assert st.ingested == 0 and st.n_blocks == 0


def test_verify_rows_are_causal():
    # three rows appended together; row j sees pos0 + j + 1 tokens
    rng = np.random.default_rng(41)
    st = make_state(rng, 38, 4)                     # 38 tokens already cached
    k, v, i = rows(rng, 3)
    st.append(38, k, v, i)
    q = bf16(rng.standard_normal((4, 16)))
    qi = bf16(rng.integers(-8, 9, size=(3, 8))); w = np.ones(3)
    for j in range(3):
        res = O.attend_row(st, 38 + j, qi, w, q, 4)
        assert res["tokens"].max() == 38 + j
        assert res["n_blk"] == (38 + j + 1) // 4


# ---------------------------------------------------------------------------
# MXFP8 index plane. The format is the OCP Microscaling (MX v1.0) MXFP8: E4M3
# elements, one E8M0 scale per 32 values. The pins decode E4M3 from its bit
# definition, compare rounding with brute force and with torch's float8_e4m3fn
# cast, and check the scale rule on hand-worked blocks.
# ---------------------------------------------------------------------------


def e4m3_table():
    """Every finite non-negative E4M3 value, in code order 0x00 .. 0x7E, decoded
    from the bit fields: sign | 4-bit exponent (bias 7) | 3-bit mantissa;
    exponent field 0 is subnormal (m/8 * 2^-6); 0x7F is NaN."""
    vals = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        vals.append(m / 8 * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals)


def test_e4m3_grid_from_the_format_definition():
    t = e4m3_table()
    assert np.all(np.diff(t) > 0)                       # codes are ordered by magnitude
    assert t[-1] == 448.0 and t[1] == 2.0 ** -9
    assert O.E4M3_MAX == 448.0
    # every grid point, either sign, is a fixed point of the rounding
    assert np.array_equal(O.e4m3_round(t), t)
    assert np.array_equal(O.e4m3_round(-t[1:]), -t[1:])
    # and nothing between two adjacent grid points is on the grid
    mids = (t[1:] + t[:-1]) / 2
    assert not np.any(O.e4m3_round(mids) == mids)


def test_e4m3_rounding_is_nearest_even_by_brute_force():
    t = e4m3_table()
    rng = np.random.default_rng(53)
    mags = np.exp2(rng.uniform(-12, 9.6, 4000))         # past 448 too
    mids = (t[1:] + t[:-1]) / 2                         # exact halfway points
    v = np.concatenate([mags, -mags, mids, -mids, [0.0, 448.0, 460.0, 464.0, 1e6]])
    got = O.e4m3_round(v)
    a = np.minimum(np.abs(v), 448.0)
    d = np.abs(a[:, None] - t[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # ties: the code with an even mantissa (even code index)
    idx = np.where(cand.sum(axis=1) > 1, np.argmax(cand & (np.arange(len(t)) % 2 == 0)[None, :], axis=1),
                   np.argmax(cand, axis=1))
    want = np.copysign(t[idx], v)
    assert np.array_equal(np.abs(got), np.abs(want))
    assert np.all((got == 0) | (np.sign(got) == np.sign(v)))


def test_e4m3_rounding_matches_torch_float8():
    rng = np.random.default_rng(59)
    v = np.concatenate([rng.standard_normal(3000) * 40, np.exp2(rng.uniform(-11, 8.8, 3000))])
    v = O.bf16_bits_to_f64(bf16(v))                     # bf16 values (exact in fp32)
    v = v[np.abs(v) <= 448.0]
    lib = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(O.e4m3_round(v), lib)


def test_mxfp8_scale_rule_on_hand_worked_blocks():
    # amax 3 -> floor(log2 3) = 1 -> scale 2^(1-8) = 2^-7: 3*128 = 384 and
    # -1.5*128 = -192 are on the grid; 0.1*128 = 12.8 lies in [8, 16) where the
    # quantum is 1, so it becomes 13, i.e. 13/128 = 0.1015625
    x = np.zeros(32); x[:3] = [3.0, -1.5, 0.1]
    el, ex = O.mxfp8_quantize(x)
    assert ex.tolist() == [-7]
    assert el[:3].tolist() == [384.0, -192.0, 13.0] and not el[3:].any()
    assert O.mxfp8_dequantize(el, ex)[:3].tolist() == [3.0, -1.5, 0.1015625]
    # amax a power of two lands on 256; amax 1.99 -> 509.4 past 448 is clamped
    y = np.zeros(32); y[0] = 4.0; y[1] = 1.0
    el, ex = O.mxfp8_quantize(y)
    assert ex.tolist() == [-6] and el[0] == 256.0 and el[1] == 64.0
    z = np.zeros(32); z[5] = -1.99
    el, ex = O.mxfp8_quantize(z)
    assert ex.tolist() == [-8] and el[5] == -448.0
    assert O.mxfp8_dequantize(el, ex)[5] == -1.75
    # an all-zero block takes the smallest scale, 2^-127
    el, ex = O.mxfp8_quantize(np.zeros(32))
    assert ex.tolist() == [-127] and not el.any()


def test_mxfp8_scales_are_per_32_value_block():
    rng = np.random.default_rng(61)
    x = rng.standard_normal((5, 128)) * np.array([1e-3, 1.0, 50.0, 3e3])[None, :].repeat(32, axis=1)
    el, ex = O.mxfp8_quantize(x)
    assert ex.shape == (5, 4)
    for c in range(4):
        blk = x[:, 32 * c:32 * (c + 1)]
        amax = np.abs(blk).max(axis=1)
        ratio = amax / np.exp2(ex[:, c])
        assert np.all((ratio >= 256) & (ratio < 512))   # amax / scale in [256, 512)
        e1, x1 = O.mxfp8_quantize(blk)
        assert np.array_equal(e1, el[:, 32 * c:32 * (c + 1)]) and np.array_equal(x1[:, 0], ex[:, c])
    # error: at most half an E4M3 quantum of the element's binade (unclamped), and idempotent
    back = O.mxfp8_dequantize(el, ex)
    scaled = np.abs(x) / np.repeat(np.exp2(ex), 32, axis=1)
    lead = np.maximum(np.floor(np.log2(np.maximum(scaled, 2.0 ** -30))), -6)
    half_q = np.exp2(lead - 4) * np.repeat(np.exp2(ex), 32, axis=1)
    ok = scaled <= 448
    assert np.all(np.abs(back - x)[ok] <= half_q[ok])
    el2, ex2 = O.mxfp8_quantize(back)
    assert np.array_equal(O.mxfp8_dequantize(el2, ex2), back)


def test_mxfp8_scores_hand_worked_and_identity_on_small_integers():
    # one 32-value block, one head, w = 1: q = (3, 0.1, 0, ...) -> (3, 0.1015625, ...)
    # (first hand-worked block above); k = (1, 1, 0, ...) is on its grid (amax 1 ->
    # scale 2^-8, 256 and 256). Score = 3 + 0.1015625.
    q = np.zeros((1, 32)); q[0, :2] = [3.0, 0.1]
    k = np.zeros((1, 32)); k[0, :2] = [1.0, 1.0]
    s = O.block_scores_mxfp8(bf16(q), np.ones(1), bf16(k))
    assert s.tolist() == [3.1015625]
    # the synthetic recipe's integer queries in [-8, 8] are exact in MXFP8, so
    # with keys of small integers the MXFP8 score is the bf16 score
    rng = np.random.default_rng(67)
    qi = bf16(rng.integers(-8, 9, size=(6, 64)))
    kb = bf16(rng.integers(-8, 9, size=(20, 64)))
    w = rng.standard_normal(6)
    assert np.array_equal(O.block_scores_mxfp8(qi, w, kb), O.block_scores(qi, w, kb))


# ---------------------------------------------------------------------------
# Always-kept local window ("Flash-Next support: llama.cpp vs Atlas", (d)
# adoption plan, phase 2, item 6: the last 128 tokens are kept, a union with
# the top-k set).
# ---------------------------------------------------------------------------


def test_local_window_is_the_union_with_the_last_tokens():
    rng = np.random.default_rng(73)
    for _ in range(300):
        r = int(rng.choice([2, 4, 8]))
        V = int(rng.integers(1, 400))
        n_blk = V // r
        k = int(rng.integers(0, n_blk + 1))
        sel = np.sort(rng.choice(n_blk, size=k, replace=False)) if k else np.zeros(0, np.int64)
        W = int(rng.integers(0, 300))
        got = O.token_set(sel, n_blk, V, r, W)
        # brute force over positions: selected block, the tail, or among the last W
        want = [t for t in range(V) if (t // r in set(sel.tolist()) and t < n_blk * r) or t >= n_blk * r
                or (W > 0 and t >= V - W)]
        assert got.tolist() == want
    # window 0 is the plain token set; a window covering everything is dense
    sel = np.array([1, 5, 9])
    assert np.array_equal(O.token_set(sel, 12, 50, 4, 0), O.token_set(sel, 12, 50, 4))
    assert O.token_set(sel, 12, 50, 4, 50).tolist() == list(range(50))


def test_local_window_hand_worked_row():
    # V = 5000 visible, ratio 4 (1250 complete blocks), window 128: the run starts
    # at 4872 = block 1218. Selected blocks 3 and 1217 lie before it (8 tokens),
    # block 1218 starts exactly at the run, block 1240 lies inside it: 8 + 128 tokens.
    toks = O.token_set(np.array([3, 1217, 1218, 1240]), 1250, 5000, 4, 128)
    assert toks.tolist() == [12, 13, 14, 15, 4868, 4869, 4870, 4871] + list(range(4872, 5000))
    # a run start inside a selected block keeps that block's earlier tokens: V = 5001
    # puts it at 4873 (inside block 1218): tokens 4872 plus the run 4873..5000
    toks = O.token_set(np.array([1218]), 1250, 5001, 4, 128)
    assert toks.tolist() == [4872] + list(range(4873, 5001))


def test_attend_row_with_window_at_and_below_the_bound_is_dense():
    rng = np.random.default_rng(79)
    st = make_state(rng, 40, 4)                     # 40 tokens, K = 4 blocks
    q = bf16(rng.standard_normal((4, 16)))
    qi = bf16(rng.integers(-8, 9, size=(8,)))[None].repeat(1, 0).reshape(1, 8); w = np.ones(1)
    # below the bound (n_blk <= K) the window changes nothing: dense
    res0 = O.attend_row(st, 14, qi, w, q, 4)
    res1 = O.attend_row(st, 14, qi, w, q, 4, window=8)
    assert np.array_equal(res0["tokens"], np.arange(15)) and np.array_equal(res1["tokens"], np.arange(15))
    # past the bound the window adds the recent tokens the selection left out
    res = O.attend_row(st, 39, qi, w, q, 4, window=12)
    assert set(range(28, 40)) <= set(res["tokens"].tolist())
    assert set(O.token_set(res["sel"], 10, 40, 4).tolist()) <= set(res["tokens"].tolist())


# ---------------------------------------------------------------------------
# Main-attention options ("Flash-Next support: vLLM vs Atlas", (a) item 6,
# Dataflow bullet: sigmoid output gate, GemmaRMSNorm q/k heads, QK-norm + RoPE).
# ---------------------------------------------------------------------------


def test_attention_qk_norm_rope_and_gate_hand_worked():
    # D = 4, one head, gains 0, eps 0, rotary 4: a head [1, 0, 0, 0] normalises to
    # [2, 0, 0, 0] (rms 1/2) and at position p becomes [2 cos p, 0, 2 sin p, 0]
    # (pair (0, 2) turns by p, pair (1, 3) is zero). Keys at 0 and 1, the row at 1:
    # q.k0 = 4 cos 1, q.k1 = 4; logits (scale 1/2) 2 cos 1 and 2; V0 = [1, 0, 1, 1],
    # V1 = [0, 1, 1, -1], so out = [w0, 1 - w0, 1, 2 w0 - 1] with
    # w0 = 1 / (1 + exp(2 - 2 cos 1)).
    a = O.AttnOptions(np.zeros(4), np.zeros(4), eps=0.0, theta=1e4, rotary_dim=4)
    st = O.SeqState(2, 1, 4, 8, 8, attn=a)
    k = bf16([[[1, 0, 0, 0]], [[1, 0, 0, 0]]])
    v = bf16([[[1, 0, 1, 1]], [[0, 1, 1, -1]]])
    st.append(0, k, v, bf16(np.zeros((2, 8))))
    q = bf16([[1, 0, 0, 0]])
    res = O.attend_row(st, 1, bf16(np.zeros((1, 8))), np.ones(1), q, 4, attn=a)
    w0 = 1.0 / (1.0 + math.exp(2.0 - 2.0 * math.cos(1.0)))
    assert np.allclose(res["out"][0], [w0, 1 - w0, 1, 2 * w0 - 1], atol=1e-2)
    assert abs(res["out"][0][0] - 0.285) < 1e-2
    # the stored keys are the prepared ones: k0 = [2, 0, 0, 0], k1 = [2 cos 1, 0, 2 sin 1, 0]
    kk = O.bf16_bits_to_f64(st.K[:2, 0])
    assert np.allclose(kk[0], [2, 0, 0, 0]) and np.allclose(kk[1], [2 * math.cos(1), 0, 2 * math.sin(1), 0], atol=1e-2)
    # gate: sigmoid(ln 3) = 3/4, sigmoid(0) = 1/2, sigmoid(-ln 3) = 1/4, sigmoid(30) = 1 - 1e-13
    g = bf16([[math.log(3), 0.0, -math.log(3), 30.0]])
    gl = O.bf16_bits_to_f64(g)[0]
    gated = O.attend_row(st, 1, bf16(np.zeros((1, 8))), np.ones(1), q, 4, attn=a, gate_bits=g)
    assert np.allclose(gated["out"][0] / res["out"][0],
                       [1 / (1 + math.exp(-gl[0])), 0.5, 1 / (1 + math.exp(-gl[2])), 1.0], atol=1e-12)
    assert abs(1 / (1 + math.exp(-gl[0])) - 0.75) < 2e-3 and abs(1 / (1 + math.exp(-gl[2])) - 0.25) < 2e-3
    # without options the path is unchanged
    st0 = O.SeqState(2, 1, 4, 8, 8)
    st0.append(0, k, v, bf16(np.zeros((2, 8))))
    plain = O.attend_row(st0, 1, bf16(np.zeros((1, 8))), np.ones(1), q, 4)
    assert np.allclose(plain["out"][0], [0.5, 0.5, 1, 0])


def test_sigmoid_closed_forms():
    assert O.sigmoid(0.0) == 0.5
    assert abs(O.sigmoid(math.log(3)) - 0.75) < 1e-15 and abs(O.sigmoid(-math.log(3)) - 0.25) < 1e-15
    x = np.linspace(-20, 20, 81)
    assert np.allclose(O.sigmoid(x) + O.sigmoid(-x), 1.0, atol=1e-15)


# MXFP4 (OCP MX v1.0: E2M1 elements, one E8M0 scale per 32 values)


def e2m1_table():
    """The 8 non-negative E2M1 values in code order 0..7 from the bit fields:
    2-bit exponent (bias 1) | 1-bit mantissa; exponent 0 is subnormal (m * 0.5)."""
    return np.array([(m * 0.5) if e == 0 else (1 + m / 2) * 2.0 ** (e - 1) for e in range(4) for m in range(2)])


def test_e2m1_grid_and_nearest_even_rounding():
    t = e2m1_table()
    assert t.tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert np.array_equal(O.e2m1_round(t), t) and np.array_equal(O.e2m1_round(-t), -t)
    mids = (t[1:] + t[:-1]) / 2
    assert not np.any(O.e2m1_round(mids) == mids)
    rng = np.random.default_rng(83)
    v = np.concatenate([rng.uniform(-8, 8, 5000), mids, -mids])
    got = O.e2m1_round(v)
    a = np.minimum(np.abs(v), 6.0)
    d = np.abs(a[:, None] - t[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    idx = np.where(cand.sum(axis=1) > 1, np.argmax(cand & (np.arange(8) % 2 == 0)[None, :], axis=1),
                   np.argmax(cand, axis=1))
    assert np.array_equal(np.abs(got), t[idx])


def test_mxfp4_scale_rule_on_a_hand_worked_block():
    # amax 3 -> floor(log2 3) - 2 = -1 -> scale 1/2: 3 -> 6, -1.5 -> -3, 0.1 -> 0.2
    # (below the 0.25 midpoint: 0), 0.7 -> 1.4 (nearer 1.5 than 1)
    x = np.zeros(32); x[:4] = [3.0, -1.5, 0.1, 0.7]
    el, ex = O.mxfp4_quantize(x)
    assert ex.tolist() == [-1] and el[:4].tolist() == [6.0, -3.0, 0.0, 1.5]
    assert O.mxfp8_dequantize(el, ex)[:4].tolist() == [3.0, -1.5, 0.0, 0.75]
    # amax / scale in [4, 8): values past 6 clamp (amax 7.9 at scale 1 -> 6)
    y = np.zeros(32); y[0] = 7.9
    el, ex = O.mxfp4_quantize(y)
    assert ex.tolist() == [0] and el[0] == 6.0
    rng = np.random.default_rng(89)
    z = rng.standard_normal((4, 64)) * 10
    el, ex = O.mxfp4_quantize(z)
    amax = np.abs(z.reshape(4, 2, 32)).max(axis=-1)
    assert np.all((amax / np.exp2(ex) >= 4) & (amax / np.exp2(ex) < 8))
    # idempotent
    back = O.mxfp8_dequantize(el, ex)
    assert np.array_equal(O.mxfp8_dequantize(*O.mxfp4_quantize(back)), back)


def test_mxfp4_scores_hand_worked():
    # q = (3, 0.7, 0, ...) -> (3, 0.75); k = (1, 1, 0, ...) exact (scale 2^-2, 4 and 4)
    q = np.zeros((1, 32)); q[0, :2] = [3.0, 0.7]
    k = np.zeros((1, 32)); k[0, :2] = [1.0, 1.0]
    assert O.block_scores_mxfp4(bf16(q), np.ones(1), bf16(k)).tolist() == [3.75]
