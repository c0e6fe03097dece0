"""Seeded synthetic inputs for the indexer-selected sparse attention workloads.

This module is shared by the GPU path's tests/benchmark and by the CPU oracle's
tests. It holds no arithmetic of the method itself: only a counter-based random
number generator, the value distributions of the workloads, and the workload
recipes (shapes, seeds, prefix lengths).

Generator
---------
Every value is a pure function of (seed, stream, epoch, sequence slot, token
position, element index), so any token row of any sequence can be regenerated
on its own, on the host or on the device, bit for bit:

    base  = H(H(H(H(seed * 0x9E3779B9 + stream) ^ epoch) ^ seq) ^ pos)
    draw  = H(base ^ (j * 0x9E3779B9 mod 2^32))         j = element draw index

H is Chris Wellons' "lowbias32" integer hash (hash-prospector, 2018):
x ^= x>>16; x *= 0x7feb352d; x ^= x>>15; x *= 0x846ca68b; x ^= x>>16 (mod 2^32).
It is evaluated with int64 torch tensors holding values in [0, 2^32), with the
32-bit multiply split into 16-bit halves so no intermediate leaves int64 range.
The same code therefore runs on CPU and CUDA tensors with identical results.

Distributions (per the workload recipes):
  * "normal"  : Irwin-Hall sum of the 12 bytes of 3 draws, (S - 1530) / 256,
                mean 0, variance 65535/65536 ~ 1, support [-5.98, 5.98]; the
                exact fp32 value is rounded to bf16 (round-to-nearest-even).
  * "int"     : uniform integer in [-8, 8] (draw mod 17 - 8), exact in bf16.
  * "pow2w"   : head weight 2^(k-2), k uniform in {0,1,2,3}: {0.25,0.5,1,2}.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

_M32 = 0xFFFFFFFF
_GOLD = 0x9E3779B9

# Stream identifiers: one independent random stream per input tensor kind.
STREAM_K = 1
STREAM_V = 2
STREAM_IDX_K = 3
STREAM_Q = 4
STREAM_Q_IDX = 5
STREAM_W = 6
STREAM_PAGES = 7
STREAM_PREFIX = 8
STREAM_REJECT = 9
STREAM_SCORES = 10


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    lo = c & 0xFFFF
    hi = c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & _M32


def hash32(x: torch.Tensor) -> torch.Tensor:
    """lowbias32 on an int64 tensor whose values lie in [0, 2^32)."""
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _as_i64(v, device) -> torch.Tensor:
    if isinstance(v, torch.Tensor):
        return v.to(device=device, dtype=torch.int64)
    return torch.as_tensor(v, dtype=torch.int64, device=device)


def token_base(seed: int, stream: int, epoch, seq, pos, device="cpu") -> torch.Tensor:
    """Per-token base key; seq/pos/epoch broadcast against each other."""
    s0 = (seed * _GOLD + stream) & _M32
    h = hash32(torch.tensor(s0, dtype=torch.int64, device=device))
    h = hash32(h ^ (_as_i64(epoch, device) & _M32))
    h = hash32(h ^ (_as_i64(seq, device) & _M32))
    h = hash32(h ^ (_as_i64(pos, device) & _M32))
    return h


def draws(base: torch.Tensor, n: int) -> torch.Tensor:
    """n draws per base key: shape base.shape + (n,)."""
    j = torch.arange(n, dtype=torch.int64, device=base.device)
    return hash32(base.unsqueeze(-1) ^ _mul32(j, _GOLD))


def normal_bf16(base: torch.Tensor, n: int) -> torch.Tensor:
    """n approximately-N(0,1) bf16 values per base key (Irwin-Hall, 12 bytes)."""
    d = draws(base, 3 * n).reshape(*base.shape, n, 3)
    s = ((d & 0xFF) + ((d >> 8) & 0xFF) + ((d >> 16) & 0xFF) + ((d >> 24) & 0xFF)).sum(-1)
    return ((s - 1530).to(torch.float32) * (1.0 / 256.0)).to(torch.bfloat16)


def int_bf16(base: torch.Tensor, n: int, lo: int = -8, hi: int = 8) -> torch.Tensor:
    """n uniform integers in [lo, hi] per base key, stored as bf16 (exact)."""
    d = draws(base, n)
    return ((d % (hi - lo + 1)) + lo).to(torch.float32).to(torch.bfloat16)


def pow2_weights(base: torch.Tensor, n: int) -> torch.Tensor:
    """n head weights in {0.25, 0.5, 1, 2} per base key (fp32)."""
    d = draws(base, n)
    return torch.pow(2.0, ((d & 3) - 2).to(torch.float32))


def uniform01(seed: int, stream: int, idx) -> torch.Tensor:
    """Uniform doubles in [0, 1) from one draw per index (host use)."""
    b = token_base(seed, stream, 0, 0, idx)
    return b.to(torch.float64) / 4294967296.0


# ---------------------------------------------------------------------------
# Per-token inputs of one sequence slot
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Shapes:
    ratio: int
    budget: int
    n_idx_heads: int
    idx_dim: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int = 64

    @property
    def topk(self) -> int:
        return self.budget // self.ratio

    @property
    def inert_bound(self) -> int:
        return self.budget + self.ratio - 1


def token_rows(sh: Shapes, seed: int, seq: int, positions, epoch=0, device="cpu", int_range=(-8, 8)):
    """K, V, raw index key rows for the given token positions of one sequence.

    Returns (k [n, Hkv, D] bf16, v [n, Hkv, D] bf16, idx_k [n, d_I] bf16).
    Index keys are integers uniform in int_range (inclusive).
    """
    pos = _as_i64(positions, device)
    n = pos.numel()
    kb = token_base(seed, STREAM_K, epoch, seq, pos, device)
    vb = token_base(seed, STREAM_V, epoch, seq, pos, device)
    ib = token_base(seed, STREAM_IDX_K, epoch, seq, pos, device)
    k = normal_bf16(kb, sh.n_kv_heads * sh.head_dim).reshape(n, sh.n_kv_heads, sh.head_dim)
    v = normal_bf16(vb, sh.n_kv_heads * sh.head_dim).reshape(n, sh.n_kv_heads, sh.head_dim)
    ik = int_bf16(ib, sh.idx_dim, *int_range).reshape(n, sh.idx_dim)
    return k, v, ik


def query_rows(sh: Shapes, seed: int, seq: int, positions, epoch=0, device="cpu", int_range=(-8, 8)):
    """Query-side inputs of the rows at the given positions of one sequence.

    Returns (q [n, Hq, D] bf16, q_idx [n, H_I, d_I] bf16, w [n, H_I] fp32).
    """
    pos = _as_i64(positions, device)
    n = pos.numel()
    qb = token_base(seed, STREAM_Q, epoch, seq, pos, device)
    ib = token_base(seed, STREAM_Q_IDX, epoch, seq, pos, device)
    wb = token_base(seed, STREAM_W, epoch, seq, pos, device)
    q = normal_bf16(qb, sh.n_q_heads * sh.head_dim).reshape(n, sh.n_q_heads, sh.head_dim)
    qi = int_bf16(ib, sh.n_idx_heads * sh.idx_dim, *int_range).reshape(n, sh.n_idx_heads, sh.idx_dim)
    w = pow2_weights(wb, sh.n_idx_heads).reshape(n, sh.n_idx_heads)
    return q, qi, w


def page_permutation(seed: int, n_pages: int) -> torch.Tensor:
    """A seeded random permutation of the global page pool (int32, host)."""
    keys = token_base(seed, STREAM_PAGES, 0, 0, torch.arange(n_pages, dtype=torch.int64))
    # ties (astronomically rare) are broken by page index via the stable sort
    return torch.sort(keys, stable=True).indices.to(torch.int32)


def page_table(seed: int, n_slots: int, max_pages: int, contiguous: bool) -> torch.Tensor:
    """[n_slots, max_pages] int32 page table over a pool of n_slots*max_pages pages."""
    n = n_slots * max_pages
    perm = torch.arange(n, dtype=torch.int32) if contiguous else page_permutation(seed, n)
    return perm.reshape(n_slots, max_pages).contiguous()


# ---------------------------------------------------------------------------
# Workload recipes
# ---------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    seed: int
    shapes: Shapes
    prefixes: List[int]             # tokens cached before the step, per sequence
    rows_per_seq: int               # appended tokens (= query rows) per sequence
    contiguous_pages: bool = False
    form: str = "decode"            # decode | verify | prefill
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def n_seq(self) -> int:
        return len(self.prefixes)

    @property
    def n_rows(self) -> int:
        return self.n_seq * self.rows_per_seq


SHAPES_TINY = Shapes(ratio=4, budget=256, n_idx_heads=4, idx_dim=64,
                     n_q_heads=8, n_kv_heads=1, head_dim=128, page_size=64)
SHAPES_MAIN = Shapes(ratio=4, budget=2048, n_idx_heads=64, idx_dim=128,
                     n_q_heads=32, n_kv_heads=4, head_dim=128, page_size=64)


def ragged_prefixes(seed: int, n: int = 64, lo: int = 512, hi: int = 131072) -> List[int]:
    """Log-uniform prefix lengths in [lo, hi], with the inert-bound boundary
    (2050, 2051, 2052) and three dense prefixes (< 2050) forced in."""
    u = uniform01(seed, STREAM_PREFIX, torch.arange(n, dtype=torch.int64)).tolist()
    out = [int(round(lo * math.exp(x * math.log(hi / lo)))) for x in u]
    forced = [2050, 2051, 2052, 600, 1300, 2049]
    out[: len(forced)] = forced
    return [min(max(p, lo), hi) for p in out]


def workload(i: int) -> Workload:
    """The five workloads (1-based), each seeded with seed = i - 1."""
    if i == 1:
        return Workload("tiny-decode b1 prefix3000 r4 B256 HI4xdI64 Hq8/Hkv1", 0, SHAPES_TINY,
                        [3000], 1, contiguous_pages=True, form="decode")
    if i == 2:
        return Workload("steady-decode b32 prefix32768 r4 B2048 HI64xdI128 Hq32/Hkv4", 1,
                        SHAPES_MAIN, [32768] * 32, 1, form="decode")
    if i == 3:
        return Workload("ragged-decode b64 prefix loguniform[512,131072] r4 B2048", 2,
                        SHAPES_MAIN, ragged_prefixes(2), 1, form="decode")
    if i == 4:
        return Workload("verify-rewind b16 prefix65536 R3 r4 B2048", 3, SHAPES_MAIN,
                        [65536] * 16, 3, form="verify", extra={"decode_after": 4})
    if i == 5:
        return Workload("chunked-prefill b1 prefix24576 chunk8193 r4 B2048", 4, SHAPES_MAIN,
                        [24576], 8193, form="prefill")
    raise ValueError(f"no workload {i}")


SCORE_KINDS = ("spread", "nonneg", "cluster", "few_values", "signed_zero", "relu_sum", "infinite")


def select_scores(seed: int, n_rows: int, n: int, kind: str) -> torch.Tensor:
    """Synthetic block-score rows [n_rows, n] (fp32) for exercising top-K
    selection on its own, each kind a score distribution a row can have:
      spread       signed, uniform in [-4, 4)
      nonneg       exponential(1) with about 1 in 32 exactly zero (a weighted
                   ReLU sum with non-negative weights)
      cluster      1 + u * 2^-10 (a narrow cluster) with one huge and one tiny
                   outlier per row, so the row's key range is wide while most
                   keys share their high bits
      few_values   one of {-1, -0.0, +0.0, 0.5, 1}: heavy ties
      signed_zero  +0.0 or -0.0 except about 1 in 64 positive values
      relu_sum     about N(270, 70^2), clipped at 0: the shape of a row of
                   sum_h w_h ReLU(q_h . k) over 64 heads with the decode
                   workload's bf16 inputs (Irwin-Hall of 12 uniforms)
      infinite     spread, with about 1 in 16 values +inf and 1 in 64 -inf
                   (a row whose range is not finite; ties at +inf)"""
    rows = torch.arange(n_rows, dtype=torch.int64)[:, None]
    cols = torch.arange(n, dtype=torch.int64)[None, :]
    b = token_base(seed, STREAM_SCORES, 0, rows, cols)
    u = b.to(torch.float64) / 4294967296.0
    if kind == "spread":
        x = u * 8.0 - 4.0
    elif kind == "nonneg":
        x = -torch.log1p(-u)
        x = torch.where((b & 31) == 0, torch.zeros_like(x), x)
    elif kind == "cluster":
        x = 1.0 + u * 2.0 ** -10
        x[:, 7 % n] = 1e30
        x[:, 11 % n] = -1e30
    elif kind == "few_values":
        vals = torch.tensor([-1.0, -0.0, 0.0, 0.5, 1.0], dtype=torch.float64)
        x = vals[b % 5]
    elif kind == "signed_zero":
        x = torch.where((b & 1) == 0, torch.zeros_like(u), -torch.zeros_like(u))
        x = torch.where(((b >> 1) & 63) == 0, 1.0 + u, x)
    elif kind == "relu_sum":
        u12 = draws(b, 12).to(torch.float64) / 4294967296.0
        x = torch.clamp(270.0 + 70.0 * (u12.sum(-1) - 6.0), min=0.0)
    elif kind == "infinite":
        x = u * 8.0 - 4.0
        x = torch.where((b >> 8) % 16 == 0, torch.full_like(x, float("inf")), x)
        x = torch.where((b >> 12) % 64 == 1, torch.full_like(x, float("-inf")), x)
    else:
        raise ValueError(f"unknown score kind {kind}")
    return x.to(torch.float32)


def reject_counts(seed: int, n_seq: int, max_reject: int = 2) -> List[int]:
    """Per-sequence number of rejected verify rows, uniform in {0..max_reject}."""
    b = token_base(seed, STREAM_REJECT, 0, 0, torch.arange(n_seq, dtype=torch.int64))
    return (b % (max_reject + 1)).tolist()


def mrope_positions(n: int, img_start: int, grid_h: int, grid_w: int) -> torch.Tensor:
    """(t, h, w) positions [n, 3] int32 of a multimodal sequence: text tokens
    (p, p, p) before img_start; then an image of grid_h x grid_w patches in
    row-major order at one temporal step (t = img_start, h = img_start + row,
    w = img_start + column); then text again, its positions continuing from
    img_start + max(grid_h, grid_w)."""
    p = torch.arange(n, dtype=torch.int64)
    out = torch.stack([p, p, p], dim=1)
    n_img = grid_h * grid_w
    k = torch.arange(n_img, dtype=torch.int64)
    img = slice(img_start, min(n, img_start + n_img))
    m = img.stop - img.start
    if m > 0:
        out[img, 0] = img_start
        out[img, 1] = img_start + k[:m] // grid_w
        out[img, 2] = img_start + k[:m] % grid_w
    after = img_start + n_img
    if after < n:
        q = torch.arange(after, n, dtype=torch.int64) - after + img_start + max(grid_h, grid_w)
        out[after:] = torch.stack([q, q, q], dim=1)
    return out.to(torch.int32)
