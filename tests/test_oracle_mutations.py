"""Planted mistakes: each test plants one plausible bug in the oracle (on the
CPU, by monkeypatching) and checks that at least one pin then fails. A pin
suite that still passes with the bug would not be able to tell it apart."""
import math

import numpy as np
import pytest

from oracle import qsa_oracle as O
from tests import test_oracle_pins as P
from tests.conftest import read_golden_cases


def _cases():
    return read_golden_cases("worked_example.txt")


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def no_relu(q_idx_bits, w, blk_bits):
    q = O.bf16_bits_to_f64(q_idx_bits); k = O.bf16_bits_to_f64(blk_bits)
    return np.asarray(w, np.float64) @ (q @ k.T)


def relu_outside(q_idx_bits, w, blk_bits):
    q = O.bf16_bits_to_f64(q_idx_bits); k = O.bf16_bits_to_f64(blk_bits)
    return np.maximum(np.asarray(w, np.float64) @ (q @ k.T), 0.0)


def tie_to_higher(scores, topk):
    s = np.asarray(scores, np.float64); n = len(s)
    if n <= topk:
        return np.arange(n)
    order = np.lexsort((-np.arange(n), -s))
    return np.sort(order[:topk])


def rank_order(scores, topk):
    s = np.asarray(scores, np.float64); n = len(s)
    if n <= topk:
        return np.arange(n)
    return np.lexsort((np.arange(n), -s))[:topk]


def no_tail(sel, n_blk, visible, ratio):
    sel = np.asarray(sel, np.int64)
    return (sel[:, None] * ratio + np.arange(ratio)[None, :]).reshape(-1)


def kv_head_modulo(h, hq, hkv):
    return h % hkv


def pool_sum(raw_bits):
    return O.f64_to_bf16_bits(O.bf16_bits_to_f64(raw_bits).sum(axis=0))


def truncating_bf16(x):
    x = np.asarray(x, np.float64)
    return (x.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def attention_scale_1_over_d(q_bits, k_bits, v_bits):
    q = O.bf16_bits_to_f64(q_bits); k = O.bf16_bits_to_f64(k_bits); v = O.bf16_bits_to_f64(v_bits)
    hq, d = q.shape; hkv = k.shape[1]
    out = np.empty((hq, d))
    for h in range(hq):
        g = O.kv_head_of(h, hq, hkv)
        s = (k[:, g, :] @ q[h]) / d
        p = np.exp(s - s.max())
        out[h] = (p @ v[:, g, :]) / p.sum()
    return out


def visible_excludes_own_token(state, pos, q_idx_bits, w, q_bits, topk):
    r = state.ratio
    visible = pos
    n_blk = visible // r
    scores = O.block_scores(q_idx_bits, w, state.idx_blk[:n_blk]) if n_blk > topk else None
    sel = O.select_blocks(scores if scores is not None else np.zeros(n_blk), topk)
    toks = O.token_set(sel, n_blk, visible, r)
    out = O.gqa_attention(q_bits, state.K[toks], state.V[toks])
    return {"n_blk": n_blk, "scores": scores, "sel": sel, "tokens": toks, "out": out,
            "out_bf16": O.f64_to_bf16_bits(out)}


def reuse_tail_from_current_blocks(state, pos, sel, sel_pos, q_bits):
    # bug: the tail starts at the row's own block boundary, so the tokens of
    # blocks completed since the selection was made are dropped
    r = state.ratio
    visible = pos + 1
    toks = O.token_set(np.asarray(sel, np.int64), visible // r, visible, r)
    out = O.gqa_attention(q_bits, state.K[toks], state.V[toks])
    return {"n_blk_sel": visible // r, "sel": sel, "tokens": toks, "out": out,
            "out_bf16": O.f64_to_bf16_bits(out)}


def pool_pre_rope_then_norm(raw_bits, first_pos, pre):
    # bug: RoPE before the norm (the per-dimension gain lands on rotated values)
    raw = O.bf16_bits_to_f64(raw_bits)
    k = O.rope_neox(raw.mean(axis=0), first_pos, pre.rotary_dim, pre.theta)
    return O.f64_to_bf16_bits(O.gemma_rmsnorm(k, pre.gamma_k, pre.eps))


def pool_pre_at_last_position(raw_bits, first_pos, pre):
    # bug: RoPE at the block's last token instead of its first
    raw = O.bf16_bits_to_f64(raw_bits)
    k = O.gemma_rmsnorm(raw.mean(axis=0), pre.gamma_k, pre.eps)
    return O.f64_to_bf16_bits(O.rope_neox(k, first_pos + raw.shape[0] - 1, pre.rotary_dim, pre.theta))


def norm_without_unit_offset(x, gamma, eps):
    # bug: scales by gamma instead of 1 + gamma
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(gamma, np.float64)


class StickyRewind(O.SeqState):
    def rewind(self, n_drop):
        if n_drop < 0 or n_drop > self.ingested:
            raise ValueError("bad rewind")
        # bug: forgets to move the counter


def e4m3_truncating(v):
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), O.E4M3_MAX)
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    q = np.ldexp(1.0, np.maximum(e - 1, -6) - 3)
    return np.copysign(np.floor(a / q) * q, v)


def e4m3_wrong_subnormal_quantum(v):
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), O.E4M3_MAX)
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    q = np.ldexp(1.0, np.maximum(e - 1, -7) - 3)
    return np.copysign(np.minimum(np.rint(a / q) * q, O.E4M3_MAX), v)


def mxfp8_emax_7(x):
    x = np.asarray(x, np.float64)
    b = x.reshape(x.shape[:-1] + (-1, 32))
    amax = np.abs(b).max(axis=-1)
    _, e = np.frexp(np.where(amax > 0, amax, 1.0))
    exp = np.where(amax > 0, e - 1 - 7, -127).astype(np.int64)
    return O.e4m3_round(b / np.ldexp(1.0, exp)[..., None]).reshape(x.shape), exp


def mxfp8_one_scale_per_vector(x):
    x = np.asarray(x, np.float64)
    amax = np.abs(x).max(axis=-1, keepdims=True)
    _, e = np.frexp(np.where(amax > 0, amax, 1.0))
    exp = np.where(amax > 0, e - 1 - 8, -127).astype(np.int64)
    n = x.shape[-1] // 32
    return O.e4m3_round(x / np.ldexp(1.0, exp)), np.repeat(exp, n, axis=-1)


def mxfp8_scores_keys_only(q_idx_bits, w, blk_bits):
    q = O.bf16_bits_to_f64(q_idx_bits)
    k = O.mxfp8_round_bits(blk_bits)
    return np.asarray(w, np.float64) @ np.maximum(q @ k.T, 0.0)


def _token_set_with(run_start_fn, name):
    def ts(sel, n_blk, visible, ratio, window=0):
        sel = np.asarray(sel, np.int64)
        body = (sel[:, None] * ratio + np.arange(ratio)[None, :]).reshape(-1)
        rs = run_start_fn(n_blk * ratio, visible, window, ratio) if window > 0 else n_blk * ratio
        return np.concatenate([body[body < rs], np.arange(rs, visible, dtype=np.int64)])
    ts.__name__ = name
    return ts


window_block_aligned = _token_set_with(lambda t0, V, W, r: min(t0, max(0, (V - W) // r * r)), "window_block_aligned")
window_off_by_one = _token_set_with(lambda t0, V, W, r: min(t0, max(0, V - W + 1)), "window_off_by_one")
window_drops_tail = _token_set_with(lambda t0, V, W, r: max(0, V - W), "window_drops_tail")


class KeysRopedAtZero(O.SeqState):
    def append(self, pos, k_bits, v_bits, idx_bits):
        if self.attn is not None and self.attn.gamma_k is not None:
            a = self.attn
            k_bits = np.asarray(k_bits, np.uint16)
            k_bits = np.stack([O.prep_heads(k_bits[t], 0, a.gamma_k, a.eps, a.rotary_dim, a.theta)
                               for t in range(len(k_bits))])
            saved, self.attn = self.attn, None
            try:
                super().append(pos, k_bits, v_bits, idx_bits)
            finally:
                self.attn = saved
        else:
            super().append(pos, k_bits, v_bits, idx_bits)


def sigmoid_of_minus(x):
    x = np.asarray(x, np.float64)
    return 1.0 / (1.0 + np.exp(x))


def mxfp4_emax_3(x):
    x = np.asarray(x, np.float64)
    b = x.reshape(x.shape[:-1] + (-1, 32))
    amax = np.abs(b).max(axis=-1)
    _, e = np.frexp(np.where(amax > 0, amax, 1.0))
    exp = np.where(amax > 0, e - 1 - 3, -127).astype(np.int64)
    return O.e2m1_round(b / np.ldexp(1.0, exp)[..., None]).reshape(x.shape), exp


def e2m1_ties_up(v):
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), 6.0)
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    q = np.ldexp(1.0, np.maximum(e - 1, 0) - 1)
    return np.copysign(np.minimum(np.floor(a / q + 0.5) * q, 6.0), v)


def mrope_h_w_swapped(rotary_dim, section):
    i = np.arange(rotary_dim // 2)
    ax = np.zeros(rotary_dim // 2, np.int64)
    ax[(i % 3 == 2) & (i < 3 * section[1])] = 1
    ax[(i % 3 == 1) & (i < 3 * section[2])] = 2
    return ax


def mrope_bounds_not_tripled(rotary_dim, section):
    i = np.arange(rotary_dim // 2)
    ax = np.zeros(rotary_dim // 2, np.int64)
    ax[(i % 3 == 1) & (i < section[1])] = 1
    ax[(i % 3 == 2) & (i < section[2])] = 2
    return ax


def mrope_temporal_only(pos, rotary_dim, section):
    p = pos if section is None else np.broadcast_to(np.asarray(pos, np.float64), (3,))[0]
    return np.full(rotary_dim // 2, float(p))


class MropeBlocksAtLastToken(O.SeqState):
    def block_rope_pos(self, b):
        return self.rope_pos((b + 1) * self.ratio - 1, self.pre.mrope_section)


def _rope_with(pairs, freq_exp, sin_sign, name):
    def rope(x, pos, rotary_dim, theta, section=None):
        x = np.array(x, np.float64)
        if rotary_dim == 0:
            return x
        half = rotary_dim // 2
        i = np.arange(half, dtype=np.float64)
        ang = O.pair_positions(pos, rotary_dim, section) * theta ** (-freq_exp * i / rotary_dim)
        c, sn = np.cos(ang), sin_sign * np.sin(ang)
        a_idx, b_idx = pairs(half)
        x1, x2 = x[..., a_idx].copy(), x[..., b_idx].copy()
        x[..., a_idx] = x1 * c - x2 * sn
        x[..., b_idx] = x2 * c + x1 * sn
        return x
    rope.__name__ = name
    return rope


_neox = lambda h: (np.arange(h), np.arange(h) + h)
_gptj = lambda h: (2 * np.arange(h), 2 * np.arange(h) + 1)
rope_sine_flipped = _rope_with(_neox, 2.0, -1.0, "rope_sine_flipped")
rope_gptj_pairs = _rope_with(_gptj, 2.0, 1.0, "rope_gptj_pairs")
rope_freq_exponent_halved = _rope_with(_neox, 1.0, 1.0, "rope_freq_exponent_halved")


def bf16_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    m, e = np.frexp(np.where(np.isfinite(a) & (a > 0), a, 1.0))
    quantum = np.ldexp(1.0, np.maximum(e - 1, -126) - 7)
    r = np.where(a > 0, np.floor(a / quantum + 0.5) * quantum, 0.0)
    r = np.where(r >= 2.0 ** 128, np.inf, r)
    out = np.copysign(np.where(np.isfinite(a), r, np.inf), x)
    bits = (out.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    return np.where(np.isnan(x), np.uint16(0x7FC0), bits).astype(np.uint16)


def select_one_short(scores, topk):
    s = np.asarray(scores, np.float64); n = s.shape[0]
    if n <= topk:
        return np.arange(n, dtype=np.int64)
    return np.sort(np.lexsort((np.arange(n), -s))[:topk - 1])


def e4m3_unclamped(v):
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    quantum = np.ldexp(1.0, np.maximum(e - 1, -6) - 3)
    return np.copysign(np.where(a > 0, np.rint(a / quantum) * quantum, 0.0), v)


def scores_ignore_weights(q_idx_bits, w, blk_bits):
    q = O.bf16_bits_to_f64(q_idx_bits); k = O.bf16_bits_to_f64(blk_bits)
    return np.ones(len(np.asarray(w))) @ np.maximum(q @ k.T, 0.0)


MUTATIONS = [
    ("block_scores", no_relu, [P.test_score_closed_forms]),
    ("block_scores", relu_outside, [P.test_score_closed_forms]),
    ("select_blocks", tie_to_higher, [P.test_selection_special_cases]),
    ("select_blocks", rank_order, [P.test_worked_example_scores_and_selection]),
    ("token_set", no_tail, [P.test_inert_bound_from_pages]),
    ("kv_head_of", kv_head_modulo, [P.test_gqa_head_mapping_contiguous_groups]),
    ("pool_block", pool_sum, [P.test_worked_example_blocks]),
    ("f64_to_bf16_bits", truncating_bf16, [P.test_bf16_rounding_hand_cases]),
    ("gqa_attention", attention_scale_1_over_d, [P.test_worked_example_attention]),
    ("attend_row", visible_excludes_own_token, [P.test_dense_identity_at_and_below_inert_bound]),
    ("SeqState", StickyRewind, [P.test_counter_discipline]),
    ("attend_row_reused", reuse_tail_from_current_blocks, [P.test_reused_dense_selection_stays_exactly_dense]),
    ("pool_block_pre", pool_pre_rope_then_norm, [P.test_pre_indexed_blocks_norm_then_rope_at_the_first_position]),
    ("pool_block_pre", pool_pre_at_last_position, [P.test_pre_indexed_blocks_norm_then_rope_at_the_first_position]),
    ("gemma_rmsnorm", norm_without_unit_offset, [P.test_gemma_rmsnorm_closed_forms]),
    ("e4m3_round", e4m3_truncating, [P.test_e4m3_rounding_is_nearest_even_by_brute_force]),
    ("e4m3_round", e4m3_wrong_subnormal_quantum, [P.test_e4m3_grid_from_the_format_definition]),
    ("mxfp8_quantize", mxfp8_emax_7, [P.test_mxfp8_scale_rule_on_hand_worked_blocks]),
    ("mxfp8_quantize", mxfp8_one_scale_per_vector, [P.test_mxfp8_scales_are_per_32_value_block]),
    ("block_scores_mxfp8", mxfp8_scores_keys_only, [P.test_mxfp8_scores_hand_worked_and_identity_on_small_integers]),
    ("token_set", window_block_aligned, [P.test_local_window_is_the_union_with_the_last_tokens]),
    ("token_set", window_off_by_one, [P.test_local_window_is_the_union_with_the_last_tokens]),
    ("token_set", window_drops_tail, [P.test_local_window_is_the_union_with_the_last_tokens]),
    ("SeqState", KeysRopedAtZero, [P.test_attention_qk_norm_rope_and_gate_hand_worked]),
    ("mxfp4_quantize", mxfp4_emax_3, [P.test_mxfp4_scale_rule_on_a_hand_worked_block]),
    ("e2m1_round", e2m1_ties_up, [P.test_e2m1_grid_and_nearest_even_rounding]),
    ("mrope_axes", mrope_h_w_swapped, [P.test_mrope_pairs_follow_the_interleave_and_its_section_bounds]),
    ("mrope_axes", mrope_bounds_not_tripled, [P.test_mrope_pairs_follow_the_interleave_and_its_section_bounds]),
    ("pair_positions", mrope_temporal_only, [P.test_mrope_pairs_follow_the_interleave_and_its_section_bounds,
                                             P.test_mrope_is_plain_rope_for_text_and_sees_only_per_axis_offsets]),
    ("SeqState", MropeBlocksAtLastToken, [P.test_mrope_blocks_rope_at_their_first_tokens_triple]),
    ("rope_neox", rope_sine_flipped, [P.test_rope_neox_closed_forms]),
    ("rope_neox", rope_gptj_pairs, [P.test_rope_neox_closed_forms]),
    ("rope_neox", rope_freq_exponent_halved, [P.test_rope_neox_closed_forms]),
    ("f64_to_bf16_bits", bf16_ties_away, [P.test_bf16_rounding_hand_cases,
                                          P.test_bf16_rounding_matches_torch_on_fp32_values]),
    ("select_blocks", select_one_short, [P.test_selection_brute_force_with_ties]),
    ("e4m3_round", e4m3_unclamped, [P.test_e4m3_rounding_is_nearest_even_by_brute_force,
                                    P.test_e4m3_rounding_matches_torch_float8]),
    ("block_scores", scores_ignore_weights, [P.test_score_invariants, P.test_score_closed_forms]),
    ("sigmoid", sigmoid_of_minus, [P.test_sigmoid_closed_forms, P.test_attention_qk_norm_rope_and_gate_hand_worked]),
]


@pytest.mark.parametrize("name,bug,pins", MUTATIONS, ids=[f"{m[0]}:{m[1].__name__}" for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, bug, pins):
    monkeypatch.setattr(O, name, bug)
    args = {P.test_worked_example_blocks: (_cases(),),
            P.test_worked_example_scores_and_selection: (_cases(),),
            P.test_worked_example_attention: (_cases(),)}
    caught = []
    for pin in pins:
        try:
            pin(*args.get(pin, ()))
            caught.append(False)
        except AssertionError:
            caught.append(True)
    assert any(caught), f"no pin caught the planted mistake in {name}"
