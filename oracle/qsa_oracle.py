"""CPU fp64 oracle for indexer-selected (QSA-style) block-sparse attention.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module: only
the tests, the smoke check and the benchmark's CPU-baseline leg may call it. It
shares no code with the CUDA library (no kernels, headers, tables or helpers);
the two meet only in the seeded inputs they both consume.

It is the plain definition of the method, written for readability, not speed:
logical per-sequence token arrays (no paging), numpy fp64 arithmetic, a library
matmul and a library sort as the only building blocks.

Sources (web pages, cited by title and section):
  [VA6]   "Agentic shootout -- Atlas x Flash-Next research", report
          "Flash-Next support: vLLM vs Atlas", section (a) item 6 "QSA sparse
          attention + indexer": one compressed key per complete group of
          `compress_ratio` tokens (mean-pool), weight-free scoring of the query
          against the compressed keys, block top-k with budget/ratio groups,
          expansion of the selected groups back to token indices
          (budget + ratio - 1 wide, -1 padded), sparse paged GQA attention.
  [PR16]  same page, "PR 16 review: qwen4exp serving in Atlas (Claude's
          review)", section (a), QSA bullet: 4-token mean-pooled blocks,
          relu-score, top-512 + tail, inert at <= 2051 visible tokens.
  [LC3]   same page, "Flash-Next support: llama.cpp vs Atlas", section (a)
          item 3: blocks cut the position line; the incomplete tail block is
          always visible; incomplete blocks are not scored.
  [INV1]  "Atlas Flash-Next defect investigations", Report A, Defect 1,
          proposed fix: rewind sets ingested -= dropped, pooled =
          ingested / ratio; decode at pos requires pos == ingested.
  The score formula sum_h w_h * ReLU(q_h . k_b) is the relu-score of [PR16];
  w == 1 is the weight-free case of [VA6].

Readings taken where the pages are silent (each is also listed in the design
notes): the row's own token is visible (V = pos + 1); a block completed by the
row's own token competes in the top-K (it is not force-kept); ties go to the
lower block index; output indices ascending, -1 padded; GQA head h uses KV head
floor(h * Hkv / Hq); softmax scale 1/sqrt(D); the final output is rounded to
bf16 (round to nearest even).

Every function is pinned by tests that do not re-derive it (closed forms,
brute force on tiny inputs, special cases, invariants, hand-worked examples).
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Tuple

import numpy as np

# ---------------------------------------------------------------------------
# bf16 <-> fp64
# ---------------------------------------------------------------------------


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 values to bf16 (8 significant bits), nearest-even, directly
    from fp64 (no intermediate fp32 rounding). Overflow goes to +-inf, NaN to
    the canonical quiet NaN, and values below 2^-126 use the subnormal quantum
    2^-133."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    out = np.empty(x.shape, dtype=np.float64)
    finite = np.isfinite(a)
    m, e = np.frexp(np.where(finite & (a > 0), a, 1.0))   # a = m * 2^e, m in [0.5, 1)
    lead = np.maximum(e - 1, -126)                         # exponent of the leading bit
    quantum = np.ldexp(1.0, lead - 7)
    r = np.rint(a / quantum) * quantum                    # rint: half to even
    r = np.where(a > 0, r, 0.0)
    r = np.where(r >= 2.0 ** 128, np.inf, r)
    out[...] = np.where(finite, r, np.inf)
    out = np.copysign(out, x)
    bits = (out.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    bits = np.where(np.isnan(x), np.uint16(0x7FC0), bits)
    return bits.astype(np.uint16)


def round_bf16(x) -> np.ndarray:
    """Value of x after rounding to bf16."""
    return bf16_bits_to_f64(f64_to_bf16_bits(x))


# ---------------------------------------------------------------------------
# Per-sequence indexer state (append / pool / rewind)
# ---------------------------------------------------------------------------


class DesyncError(RuntimeError):
    """An append at a position other than the number of ingested tokens."""


class CapacityError(RuntimeError):
    """An append beyond the sequence's capacity."""


def pool_block(raw_bits) -> np.ndarray:
    """Compressed key of one block: the mean of its `ratio` raw index keys,
    rounded to bf16 ([VA6] mean-pool; [PR16] "4-token mean-pooled blocks")."""
    raw = bf16_bits_to_f64(raw_bits)
    return f64_to_bf16_bits(raw.mean(axis=0))


# ---------------------------------------------------------------------------
# Pre-indexer ("Agentic shootout", "Flash-Next support: vLLM vs Atlas", (a)
# item 6: the indexer normalises its q/k heads with Gemma RMSNorm and applies
# the same RoPE as main attention; a compressed key is mean-pool, then Gemma
# RMSNorm, then RoPE at the group's first position. The report on the fused
# pre-indexer kernel adds: RMSNorm scales by weight + 1 with fp32 accumulation,
# NeoX RoPE, head_dim 128 with rotary 64.)
# ---------------------------------------------------------------------------


class PreIndexer:
    """Parameters of the pre-indexer. The pages leave epsilon and the RoPE base
    open: both are inputs. gamma_q / gamma_k: per-dimension gains (the norm
    multiplies by 1 + gamma). rotary_dim: leading dimensions rotated (NeoX:
    dimension i pairs with i + rotary_dim / 2); 0 disables RoPE."""

    def __init__(self, gamma_q, gamma_k, eps: float, theta: float, rotary_dim: int, mrope_section=None):
        self.gamma_q = np.asarray(gamma_q, np.float64)
        self.gamma_k = np.asarray(gamma_k, np.float64)
        self.eps = float(eps)
        self.theta = float(theta)
        self.rotary_dim = int(rotary_dim)
        self.mrope_section = check_mrope_section(mrope_section, self.rotary_dim)


def gemma_rmsnorm(x, gamma, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * (1 + gamma), over the last axis, fp64."""
    x = np.asarray(x, np.float64)
    rms = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x / rms * (1.0 + np.asarray(gamma, np.float64))


# Interleaved MRoPE ("Agentic shootout", "Flash-Next support: vLLM vs Atlas",
# (a) item 6: the indexer's RoPE is main attention's, interleaved MRoPE
# included; the report on the fused pre-indexer kernel: temporal, height and
# width rotary pairs interleave, a pair's axis chosen by its index modulo 3,
# with bounds for the height and width sections; the notes on a dense sibling
# model: mrope_section = [11, 11, 10] over 64 rotary dimensions). Reading: a
# token's position is a triple (t, h, w); NeoX pair i turns by the height
# position when i % 3 == 1 and i < 3 * section_h, by the width position when
# i % 3 == 2 and i < 3 * section_w, and by the temporal one otherwise. The
# sections add up to rotary_dim / 2. A text token has t = h = w = its position.


def check_mrope_section(section, rotary_dim: int):
    """(t, h, w) section sizes in rotary pairs, or None (plain RoPE)."""
    if section is None:
        return None
    sec = tuple(int(v) for v in section)
    if len(sec) != 3 or min(sec) < 0 or sum(sec) != rotary_dim // 2:
        raise ValueError(f"mrope section {section} must be 3 counts adding up to {rotary_dim // 2}")
    return sec


def mrope_axes(rotary_dim: int, section) -> np.ndarray:
    """Axis of each NeoX pair i < rotary_dim / 2: 0 temporal, 1 height, 2 width."""
    i = np.arange(rotary_dim // 2)
    ax = np.zeros(rotary_dim // 2, np.int64)
    ax[(i % 3 == 1) & (i < 3 * section[1])] = 1
    ax[(i % 3 == 2) & (i < 3 * section[2])] = 2
    return ax


def pair_positions(pos, rotary_dim: int, section) -> np.ndarray:
    """The position each NeoX pair turns by: pos for plain RoPE (section None);
    with MRoPE, pos is a (t, h, w) triple (an integer stands for (p, p, p))."""
    half = rotary_dim // 2
    if section is None:
        return np.full(half, float(pos))
    trip = np.broadcast_to(np.asarray(pos, np.float64), (3,))
    return trip[mrope_axes(rotary_dim, section)]


def rope_neox(x, pos, rotary_dim: int, theta: float, section=None) -> np.ndarray:
    """NeoX rotary embedding at position pos over the last axis: for
    i < rotary_dim/2 the pair (x_i, x_{i+rotary_dim/2}) is rotated by the angle
    p_i * theta^(-2i/rotary_dim), p_i = pos (or, with an MRoPE section, the
    coordinate of the triple pos that pair i takes); dimensions >= rotary_dim
    are unchanged."""
    x = np.array(x, np.float64)
    if rotary_dim == 0:
        return x
    half = rotary_dim // 2
    i = np.arange(half, dtype=np.float64)
    ang = pair_positions(pos, rotary_dim, section) * theta ** (-2.0 * i / rotary_dim)
    c, s = np.cos(ang), np.sin(ang)
    x1 = x[..., :half].copy()
    x2 = x[..., half:rotary_dim].copy()
    x[..., :half] = x1 * c - x2 * s
    x[..., half:rotary_dim] = x2 * c + x1 * s
    return x


def pre_index_query(q_bits, pos, pre: PreIndexer) -> np.ndarray:
    """Index query heads [H_I, d_I] of the row at pos (a (t, h, w) triple with
    MRoPE): Gemma RMSNorm per head, then RoPE at the row's position; bf16 bits."""
    q = bf16_bits_to_f64(q_bits)
    return f64_to_bf16_bits(rope_neox(gemma_rmsnorm(q, pre.gamma_q, pre.eps), pos, pre.rotary_dim, pre.theta,
                                      pre.mrope_section))


def pool_block_pre(raw_bits, first_pos, pre: PreIndexer) -> np.ndarray:
    """Compressed key of the block whose first token is at first_pos (that
    token's (t, h, w) triple with MRoPE): the mean of its raw index keys, then
    Gemma RMSNorm, then RoPE at first_pos; bf16."""
    raw = bf16_bits_to_f64(raw_bits)
    k = gemma_rmsnorm(raw.mean(axis=0), pre.gamma_k, pre.eps)
    return f64_to_bf16_bits(rope_neox(k, first_pos, pre.rotary_dim, pre.theta, pre.mrope_section))


# ---------------------------------------------------------------------------
# Main-attention options ("Agentic shootout", "Flash-Next support: vLLM vs
# Atlas", (a) item 6, Dataflow bullet: the attention is GQA with a sigmoid
# output gate, always on, and GemmaRMSNorm on the q and k heads; a fused
# QK-norm + RoPE + gate path). The pages leave the gate's granularity, epsilon
# and the RoPE base open. Readings: the gate is elementwise (one value per query
# head and dimension), o' = o * sigmoid(g), applied before the output's bf16
# rounding; each q and k head is Gemma-RMSNormed over D, then NeoX-roped at its
# token's position (the same two functions as the pre-indexer), the key when it
# is appended to the cache.
# ---------------------------------------------------------------------------


class AttnOptions:
    """gamma_q, gamma_k: per-dimension gains [D] of the q and k head norms (None:
    that side is not normed or roped); eps, theta, rotary_dim as in PreIndexer."""

    def __init__(self, gamma_q=None, gamma_k=None, eps: float = 1e-6, theta: float = 1e4,
                 rotary_dim: int = 64, mrope_section=None):
        self.gamma_q = None if gamma_q is None else np.asarray(gamma_q, np.float64)
        self.gamma_k = None if gamma_k is None else np.asarray(gamma_k, np.float64)
        self.eps = float(eps)
        self.theta = float(theta)
        self.rotary_dim = int(rotary_dim)
        self.mrope_section = check_mrope_section(mrope_section, self.rotary_dim)


def prep_heads(x_bits, pos, gamma, eps: float, rotary_dim: int, theta: float, section=None) -> np.ndarray:
    """Heads [H, D] of the token at pos (a (t, h, w) triple with an MRoPE
    section): Gemma RMSNorm per head, then RoPE at pos; bf16 bits."""
    x = bf16_bits_to_f64(x_bits)
    return f64_to_bf16_bits(rope_neox(gemma_rmsnorm(x, gamma, eps), pos, rotary_dim, theta, section))


def sigmoid(x) -> np.ndarray:
    """1 / (1 + exp(-x)), fp64."""
    x = np.asarray(x, np.float64)
    return 1.0 / (1.0 + np.exp(-x))


# ---------------------------------------------------------------------------
# MXFP8 index plane ("Agentic shootout", "Flash-Next support: vLLM vs Atlas",
# the report whose (a) item 3 is "QSA sparse attention + n-gram indexer",
# Scores bullet: with an MXFP8 indexer cache both the index queries and the
# cached index keys are MXFP8-quantised before scoring; "ATOM Model Support
# Guide", "Model architecture details", DeepSeek-V4.1, Cache bullet: an fp8
# index plane, values and E8M0 scales held in two planes).
#
# The pages name the format but do not restate it; MXFP8 is the OCP
# Microscaling format (MX specification v1.0): a block of 32 consecutive values
# shares one scale 2^e stored as an E8M0 byte (e + 127), and each value is an FP8
# E4M3 element (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; the
# all-ones pattern is NaN, so the largest finite magnitude is 448). The scale
# is 2^(floor(log2(amax)) - 8), 8 being the exponent of E4M3's largest binade,
# so amax / scale lies in [256, 512); elements are value / scale rounded to
# nearest-even on the E4M3 grid, magnitudes past 448 clamped to 448.
# ---------------------------------------------------------------------------

MX_BLOCK = 32
E4M3_MAX = 448.0
E4M3_EMAX = 8          # exponent of the largest E4M3 binade
E8M0_MIN_EXP = -127    # smallest scale exponent an E8M0 byte holds (byte 0)


def e4m3_round(v) -> np.ndarray:
    """Round fp64 values to the E4M3 grid, nearest-even, magnitudes clamped to
    448. Normal binades [2^E, 2^(E+1)) for E = -6 .. 8 hold 8 values each
    (quantum 2^(E-3)); below 2^-6 the subnormal quantum is 2^-9."""
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    _, e = np.frexp(np.where(a > 0, a, 1.0))          # a = m * 2^e, m in [0.5, 1)
    lead = np.maximum(e - 1, -6)                        # exponent of the leading bit
    quantum = np.ldexp(1.0, lead - 3)
    r = np.rint(a / quantum) * quantum                  # rint: half to even
    r = np.minimum(np.where(a > 0, r, 0.0), E4M3_MAX)
    return np.copysign(r, v)


def mxfp8_quantize(x) -> Tuple[np.ndarray, np.ndarray]:
    """MXFP8 blocks of the last axis (a multiple of 32): returns the E4M3
    element values [..., n] and the scale exponents [..., n / 32] (ints). A
    block whose largest magnitude is 0 (or below 2^-126) takes the smallest
    scale, 2^-127."""
    x = np.asarray(x, np.float64)
    n = x.shape[-1]
    assert n % MX_BLOCK == 0, "MXFP8 blocks need a multiple of 32 values"
    blocks = x.reshape(x.shape[:-1] + (n // MX_BLOCK, MX_BLOCK))
    amax = np.abs(blocks).max(axis=-1)
    _, e = np.frexp(np.where(amax > 0, amax, 1.0))
    exp = np.where(amax >= 2.0 ** -126, (e - 1) - E4M3_EMAX, E8M0_MIN_EXP)
    exp = np.maximum(exp, E8M0_MIN_EXP).astype(np.int64)
    elems = e4m3_round(blocks / np.ldexp(1.0, exp)[..., None])
    return elems.reshape(x.shape), exp


def mxfp8_dequantize(elems, exps) -> np.ndarray:
    """Values of MXFP8 blocks: element times 2^(its block's exponent)."""
    elems = np.asarray(elems, np.float64)
    n = elems.shape[-1]
    scale = np.repeat(np.ldexp(1.0, np.asarray(exps)), MX_BLOCK, axis=-1)
    assert scale.shape[-1] == n
    return elems * scale


# MXFP4 ("ATOM Model Support Guide", "Model architecture details",
# DeepSeek-V4.1, Cache bullet: an fp4 index plane of E2M1 values with E8M0
# scales, the two kept in separate planes). OCP MX v1.0 MXFP4: blocks of 32
# values share an E8M0 scale 2^(floor(log2 amax) - 2) (2: the exponent of E2M1's
# top binade), each value an E2M1 element (sign, 2 exponent bits with bias 1,
# 1 mantissa bit: 0, 0.5, 1, 1.5, 2, 3, 4, 6), value / scale rounded
# nearest-even on that grid and clamped to 6.

E2M1_MAX = 6.0
E2M1_EMAX = 2


def e2m1_round(v) -> np.ndarray:
    """Round fp64 values to the E2M1 grid, nearest-even, magnitudes clamped to 6.
    Binades [2^E, 2^(E+1)) for E = 0 .. 2 hold 2 values each (quantum 2^(E-1));
    below 1 the subnormal quantum is 0.5."""
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), E2M1_MAX)
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    lead = np.maximum(e - 1, 0)
    quantum = np.ldexp(1.0, lead - 1)
    r = np.minimum(np.where(a > 0, np.rint(a / quantum) * quantum, 0.0), E2M1_MAX)
    return np.copysign(r, v)


def mxfp4_quantize(x) -> Tuple[np.ndarray, np.ndarray]:
    """MXFP4 blocks of the last axis (a multiple of 32): E2M1 element values and
    scale exponents, as mxfp8_quantize with E2M1's top binade 2."""
    x = np.asarray(x, np.float64)
    n = x.shape[-1]
    assert n % MX_BLOCK == 0, "MXFP4 blocks need a multiple of 32 values"
    blocks = x.reshape(x.shape[:-1] + (n // MX_BLOCK, MX_BLOCK))
    amax = np.abs(blocks).max(axis=-1)
    _, e = np.frexp(np.where(amax > 0, amax, 1.0))
    exp = np.where(amax >= 2.0 ** -126, (e - 1) - E2M1_EMAX, E8M0_MIN_EXP)
    exp = np.maximum(exp, E8M0_MIN_EXP).astype(np.int64)
    elems = e2m1_round(blocks / np.ldexp(1.0, exp)[..., None])
    return elems.reshape(x.shape), exp


def mxfp4_round_bits(bits) -> np.ndarray:
    """bf16 vectors (last axis) through MXFP4 and back (exact in bf16), fp64."""
    return mxfp8_dequantize(*mxfp4_quantize(bf16_bits_to_f64(bits)))


def block_scores_mxfp4(q_idx_bits, w, blk_bits) -> np.ndarray:
    """block_scores with an MXFP4 index plane: query heads and compressed keys
    MXFP4-quantised along d_I (the reading: both operands in the plane's
    arithmetic), then the same fp64 sum."""
    q = mxfp4_round_bits(q_idx_bits)
    k = mxfp4_round_bits(blk_bits)
    return np.asarray(w, np.float64) @ np.maximum(q @ k.T, 0.0)


def mxfp8_round_bits(bits) -> np.ndarray:
    """bf16 vectors (last axis) through MXFP8 and back: the values the scores
    see, as fp64 (every such value is exact in bf16)."""
    return mxfp8_dequantize(*mxfp8_quantize(bf16_bits_to_f64(bits)))


class SeqState:
    """Logical token arrays of one sequence: K, V, raw index keys (bf16 bits),
    the compressed key of every complete block, and the ingested counter.

    Block b covers logical positions [b*ratio, (b+1)*ratio) ([LC3]: blocks cut
    the position line). A block is complete once all of its tokens have been
    ingested; only complete blocks have compressed keys.
    """

    def __init__(self, ratio: int, n_kv_heads: int, head_dim: int, idx_dim: int,
                 capacity: int, pre: "PreIndexer" = None, attn: "AttnOptions" = None):
        self.ratio = ratio
        self.pre = pre  # compressed keys through the pre-indexer when given
        self.attn = attn  # key heads normed and roped as they are appended, when given
        self.capacity = capacity
        self.K = np.zeros((capacity, n_kv_heads, head_dim), np.uint16)
        self.V = np.zeros((capacity, n_kv_heads, head_dim), np.uint16)
        self.idx_raw = np.zeros((capacity, idx_dim), np.uint16)
        self.idx_blk = np.zeros((capacity // ratio, idx_dim), np.uint16)
        self.mpos = np.zeros((capacity, 3), np.int64)  # (t, h, w) of every token (MRoPE)
        self.ingested = 0

    def rope_pos(self, p: int, section):
        """The position token p turns by: its (t, h, w) triple with MRoPE, else p."""
        return tuple(self.mpos[p]) if section is not None else p

    def block_rope_pos(self, b: int):
        """A compressed key turns at its block's first token ([VA6]: RoPE at the
        group's first position)."""
        return self.rope_pos(b * self.ratio, self.pre.mrope_section)

    @property
    def n_blocks(self) -> int:
        """pooled = ingested / ratio ([INV1])."""
        return self.ingested // self.ratio

    def append(self, pos: int, k_bits, v_bits, idx_bits, mpos=None) -> None:
        """Ingest n new tokens at positions pos..pos+n-1.

        Requires pos == ingested ([INV1]: decode at pos requires
        pos == ingested). Every block completed by the new tokens is pooled
        from the raw keys it holds now. mpos [n, 3]: the tokens' (t, h, w)
        MRoPE positions (default: (p, p, p), a text token's)."""
        k_bits = np.asarray(k_bits, np.uint16)
        n = k_bits.shape[0]
        if pos != self.ingested:
            raise DesyncError(f"append at pos {pos} but {self.ingested} tokens ingested")
        if pos + n > self.capacity:
            raise CapacityError(f"append of {n} at pos {pos} exceeds capacity {self.capacity}")
        p = np.arange(pos, pos + n, dtype=np.int64)
        self.mpos[pos:pos + n] = np.stack([p, p, p], axis=1) if mpos is None else np.asarray(mpos, np.int64)
        if self.attn is not None and self.attn.gamma_k is not None:
            a = self.attn
            k_bits = np.stack([prep_heads(k_bits[t], self.rope_pos(pos + t, a.mrope_section), a.gamma_k, a.eps,
                                          a.rotary_dim, a.theta, a.mrope_section)
                               for t in range(n)]) if n else k_bits
        self.K[pos:pos + n] = k_bits
        self.V[pos:pos + n] = np.asarray(v_bits, np.uint16)
        self.idx_raw[pos:pos + n] = np.asarray(idx_bits, np.uint16)
        r = self.ratio
        first_done = pos // r            # first block that may complete now
        last_done = (pos + n) // r       # blocks [first_done, last_done) are complete
        for b in range(first_done, last_done):
            if self.pre is None:
                self.idx_blk[b] = pool_block(self.idx_raw[b * r:(b + 1) * r])
            else:
                self.idx_blk[b] = pool_block_pre(self.idx_raw[b * r:(b + 1) * r], self.block_rope_pos(b), self.pre)
        self.ingested = pos + n

    def rewind(self, n_drop: int) -> None:
        """Drop the last n_drop tokens ([INV1]: ingested -= dropped,
        pooled = ingested / ratio). Rows past the new end are dead; a block
        that becomes incomplete is re-pooled from its new raw rows when it is
        completed again."""
        if n_drop < 0 or n_drop > self.ingested:
            raise ValueError(f"rewind of {n_drop} with {self.ingested} ingested")
        self.ingested -= n_drop


# ---------------------------------------------------------------------------
# One query row: score, select, expand, attend
# ---------------------------------------------------------------------------


def block_scores(q_idx_bits, w, blk_bits) -> np.ndarray:
    """s_b = sum_h w_h * max(0, q_h . k_b) for every complete block b, fp64.

    q_idx_bits [H_I, d_I] bf16 bits, w [H_I] float, blk_bits [n_blk, d_I]."""
    q = bf16_bits_to_f64(q_idx_bits)
    k = bf16_bits_to_f64(blk_bits)
    dots = q @ k.T                              # [H_I, n_blk]
    return np.asarray(w, np.float64) @ np.maximum(dots, 0.0)


def block_scores_mxfp8(q_idx_bits, w, blk_bits) -> np.ndarray:
    """block_scores with an MXFP8 index plane: every query head and every
    compressed key (bf16) is MXFP8-quantised along d_I, and the score is the
    same fp64 sum over the quantised values."""
    q = mxfp8_round_bits(q_idx_bits)
    k = mxfp8_round_bits(blk_bits)
    dots = q @ k.T
    return np.asarray(w, np.float64) @ np.maximum(dots, 0.0)


def select_blocks(scores, topk: int) -> np.ndarray:
    """Top-K blocks by (score descending, block index ascending), returned in
    ascending block order. With n_blk <= K every block is selected, which makes
    a visible prefix of at most budget + ratio - 1 tokens exactly dense
    ([PR16]: inert at <= 2051 visible tokens for budget 2048, ratio 4)."""
    s = np.asarray(scores, np.float64)
    n = s.shape[0]
    if n <= topk:
        return np.arange(n, dtype=np.int64)
    order = np.lexsort((np.arange(n), -s))     # last key is primary
    return np.sort(order[:topk])


def token_set(sel, n_blk: int, visible: int, ratio: int, window: int = 0) -> np.ndarray:
    """Selected blocks expanded to token positions, plus the tail
    [n_blk*ratio, visible) of the incomplete block ([VA6] expansion; [LC3]
    tail always visible). Ascending.

    window > 0 also keeps the last `window` visible tokens ("Agentic shootout",
    "Flash-Next support: llama.cpp vs Atlas", (d) adoption plan, phase 2, item 6
    "Sparse attention gather": the last 128 tokens are always kept, a union with
    the top-k set; the same report's (a) hparams bullet names llama.cpp's
    indexer_local_blocks). Reading: the selection is
    made as without the window; the token set is its union with
    [visible - window, visible) and the tail, i.e. the selected tokens before
    run_start = min(visible - window, n_blk*ratio) followed by the run
    [run_start, visible)."""
    sel = np.asarray(sel, np.int64)
    body = (sel[:, None] * ratio + np.arange(ratio)[None, :]).reshape(-1)
    run_start = n_blk * ratio
    if window > 0:
        run_start = min(run_start, max(0, visible - window))
    body = body[body < run_start]
    tail = np.arange(run_start, visible, dtype=np.int64)
    return np.concatenate([body, tail])


def kv_head_of(h: int, n_q_heads: int, n_kv_heads: int) -> int:
    """GQA: contiguous groups of Hq/Hkv query heads share one KV head."""
    return (h * n_kv_heads) // n_q_heads


def gqa_attention(q_bits, k_bits, v_bits) -> np.ndarray:
    """Softmax attention of each query head over the given token rows, fp64.

    q_bits [Hq, D]; k_bits, v_bits [T, Hkv, D]. Scale 1/sqrt(D), max
    subtracted before exponentiation. Returns [Hq, D] float64 (unrounded)."""
    q = bf16_bits_to_f64(q_bits)
    k = bf16_bits_to_f64(k_bits)
    v = bf16_bits_to_f64(v_bits)
    hq, d = q.shape
    hkv = k.shape[1]
    out = np.empty((hq, d), np.float64)
    for h in range(hq):
        g = kv_head_of(h, hq, hkv)
        s = (k[:, g, :] @ q[h]) / math.sqrt(d)
        p = np.exp(s - s.max())
        out[h] = (p @ v[:, g, :]) / p.sum()
    return out


def attend_row(state: SeqState, pos: int, q_idx_bits, w, q_bits, topk: int,
               index_format: str = "bf16", window: int = 0, attn: "AttnOptions" = None,
               gate_bits=None, q_mpos=None) -> Dict:
    """The whole path for one query row at logical position pos.

    The row's token is already ingested, so V = pos + 1 tokens are visible and
    n_blk = V // ratio blocks are complete. index_format "mxfp8" scores with
    the MXFP8 index plane (block_scores_mxfp8); window keeps the last `window`
    tokens as well (token_set). attn (with gamma_q) norms and ropes the query
    heads at pos (at the triple q_mpos with an MRoPE section; default
    (pos, pos, pos)); gate_bits [Hq, D] gates the output: o * sigmoid(g)."""
    r = state.ratio
    visible = pos + 1
    if visible > state.ingested:
        raise DesyncError(f"row at pos {pos} but only {state.ingested} ingested")
    n_blk = visible // r
    if n_blk > topk:
        score_fn = {"bf16": block_scores, "mxfp8": block_scores_mxfp8, "mxfp4": block_scores_mxfp4}[index_format]
        scores = score_fn(q_idx_bits, w, state.idx_blk[:n_blk])
    else:
        scores = None                        # everything is selected; no scoring needed
    sel = select_blocks(scores if scores is not None else np.zeros(n_blk), topk)
    toks = token_set(sel, n_blk, visible, r, window)
    if attn is not None and attn.gamma_q is not None:
        qp = pos if q_mpos is None else tuple(q_mpos)
        q_bits = prep_heads(q_bits, qp, attn.gamma_q, attn.eps, attn.rotary_dim, attn.theta, attn.mrope_section)
    out = gqa_attention(q_bits, state.K[toks], state.V[toks])
    if gate_bits is not None:
        out = out * sigmoid(bf16_bits_to_f64(gate_bits))
    return {"n_blk": n_blk, "scores": scores, "sel": sel, "tokens": toks,
            "out": out, "out_bf16": f64_to_bf16_bits(out)}


def attend_row_reused(state: SeqState, pos: int, sel, sel_pos: int, q_bits, window: int = 0) -> Dict:
    """Attention of the row at logical position pos with a block selection made
    earlier, by the row at sel_pos <= pos ("Flash-Next support: vLLM vs Atlas",
    (a) item 6, MTP: later draft steps reuse the step-0 selection while the side
    caches keep updating; "Flash-Next support: llama.cpp vs Atlas", (a) item 3:
    a shared indexer layer reuses the previous full layer's top-k).

    Reading (the pages give no token-set rule for reuse): the token set is the
    reused blocks plus every token from the selection's complete-block boundary
    up to the row, sel x ratio  U  [((sel_pos + 1) // ratio) * ratio, pos + 1);
    the tail stays always visible, including blocks completed since the
    selection was made. With sel_pos == pos this is attend_row's token set."""
    r = state.ratio
    visible = pos + 1
    if visible > state.ingested:
        raise DesyncError(f"row at pos {pos} but only {state.ingested} ingested")
    if not 0 <= sel_pos <= pos:
        raise ValueError(f"selection position {sel_pos} is not in [0, {pos}]")
    n_blk_sel = (sel_pos + 1) // r
    sel = np.asarray(sel, np.int64)
    if sel.size and (sel.min() < 0 or sel.max() >= n_blk_sel):
        raise ValueError("reused selection names a block that was not complete at sel_pos")
    toks = token_set(sel, n_blk_sel, visible, r, window)
    out = gqa_attention(q_bits, state.K[toks], state.V[toks])
    return {"n_blk_sel": n_blk_sel, "sel": sel, "tokens": toks, "out": out,
            "out_bf16": f64_to_bf16_bits(out)}


def padded_selection(sel, topk: int) -> np.ndarray:
    """Selection as a fixed-width row: ascending ids, -1 padded to K."""
    row = np.full(topk, -1, np.int64)
    row[: len(sel)] = sel
    return row


# ---------------------------------------------------------------------------
# Independent dense attention (used only to pin the sparse path below the
# inert bound)
# ---------------------------------------------------------------------------


def dense_attention(q_bits, k_bits, v_bits, n_kv_heads: int) -> np.ndarray:
    """Plain causal-prefix attention over ALL given tokens, coded separately
    from gqa_attention: per head, weights = exp(s - logsumexp(s))."""
    from scipy.special import logsumexp

    q = bf16_bits_to_f64(q_bits)
    k = bf16_bits_to_f64(k_bits)
    v = bf16_bits_to_f64(v_bits)
    hq, d = q.shape
    group = hq // n_kv_heads
    out = np.zeros((hq, d))
    for g in range(n_kv_heads):
        for j in range(group):
            h = g * group + j
            logits = np.einsum("td,d->t", k[:, g, :], q[h]) * (d ** -0.5)
            wts = np.exp(logits - logsumexp(logits))
            out[h] = np.einsum("t,td->d", wts, v[:, g, :])
    return out


# ---------------------------------------------------------------------------
# A batch of rows in the library's layout: n_seq sequences, R rows each,
# row j of sequence i at position pos0[i] + j, appended before attending.
# ---------------------------------------------------------------------------


def step(states: List[SeqState], pos0: List[int], k_new, v_new, idx_new,
         q_idx, w, q, topk: int, rows_per_seq: int, index_format: str = "bf16", window: int = 0) -> List[Dict]:
    """Append each sequence's R new tokens, then run every row.

    k_new/v_new [n_seq*R, Hkv, D], idx_new [n_seq*R, d_I], q_idx
    [n_seq*R, H_I, d_I], w [n_seq*R, H_I], q [n_seq*R, Hq, D] (bf16 bits
    except w). Returns one result dict per row, sequence-major."""
    R = rows_per_seq
    for i, st in enumerate(states):
        sl = slice(i * R, (i + 1) * R)
        st.append(pos0[i], k_new[sl], v_new[sl], idx_new[sl])
    out = []
    for i, st in enumerate(states):
        for j in range(R):
            row = i * R + j
            out.append(attend_row(st, pos0[i] + j, q_idx[row], w[row], q[row], topk, index_format, window))
    return out
