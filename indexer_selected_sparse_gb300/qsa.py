"""Thin ctypes binding over libqsa (include/qsa.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. PyTorch provides device memory and the current stream. Importing this
module loads the library and fails loudly if it has not been built; there is
no fallback implementation.

The functions keep the C names (qsa_append, qsa_rewind, qsa_index_score,
qsa_topk_select, qsa_gather_attn, qsa_decode, qsa_config_check,
qsa_workspace_bytes, qsa_strerror). A non-zero return raises QsaError.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libqsa.so")

QSA_OK = 0
QSA_ERR_INVALID_ARG = 1
QSA_ERR_UNSUPPORTED = 2
QSA_ERR_CAPACITY = 3
QSA_ERR_WORKSPACE = 4
QSA_ERR_CUDA = 5
QSA_ERR_CUDA_FATAL = 6
QSA_ERR_DESYNC = 7
QSA_ERR_PAGE = 8
QSA_ERR_REWIND = 9
QSA_ERR_TIMEOUT = 10
QSA_ERR_REUSE = 11

QSA_INDEX_BF16 = 0
QSA_INDEX_MXFP8 = 1
QSA_INDEX_MXFP4 = 2

EXPORTED = ("qsa_strerror", "qsa_config_check", "qsa_workspace_bytes", "qsa_append",
            "qsa_rewind", "qsa_index_score", "qsa_topk_select", "qsa_gather_attn", "qsa_decode",
            "qsa_gather_attn_static", "qsa_max_attend_tokens", "qsa_gather_attn_reuse",
            "qsa_decode_reuse", "qsa_append_pre", "qsa_pre_index_q", "qsa_workspace_bytes_pre",
            "qsa_decode_pre", "qsa_idxblk_page_bytes", "qsa_quantize_index_q", "qsa_append_ex",
            "qsa_workspace_bytes_ex", "qsa_decode_ex", "qsa_set_wait_limit_ns", "qsa_stage_in")
QSA_STATIC_SCRATCH_BYTES = 32 << 20


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"libqsa is not built ({_LIB_PATH} missing): run "
            "`python -c 'import __graft_entry__ as g; g.build()'` first")
    return ctypes.CDLL(_LIB_PATH)


LIB = _load()
LIB_PATH = _LIB_PATH


class qsa_config(ctypes.Structure):
    _fields_ = [("ratio", ctypes.c_int), ("budget", ctypes.c_int), ("n_idx_heads", ctypes.c_int),
                ("idx_dim", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("page_size", ctypes.c_int), ("index_format", ctypes.c_int),
                ("local_window", ctypes.c_int)]


_SEC3 = ctypes.c_int * 3


class qsa_pre_indexer(ctypes.Structure):
    _fields_ = [("gamma_q", ctypes.c_void_p), ("gamma_k", ctypes.c_void_p), ("eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("rotary_dim", ctypes.c_int), ("mrope_section", _SEC3)]


class qsa_attn_options(ctypes.Structure):
    _fields_ = [("gamma_q", ctypes.c_void_p), ("gamma_k", ctypes.c_void_p), ("eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("rotary_dim", ctypes.c_int), ("gate", ctypes.c_void_p),
                ("mrope_section", _SEC3)]


class qsa_rows(ctypes.Structure):
    _fields_ = [("n_seq", ctypes.c_int), ("rows_per_seq", ctypes.c_int),
                ("seq_ids", ctypes.c_void_p), ("pos0", ctypes.c_void_p),
                ("pos0_host", ctypes.c_void_p), ("advance", ctypes.c_int), ("mrope_pos", ctypes.c_void_p)]


class qsa_cache(ctypes.Structure):
    _fields_ = [("page_table", ctypes.c_void_p), ("n_slots", ctypes.c_int),
                ("max_pages", ctypes.c_int), ("num_pages", ctypes.c_int),
                ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("idxraw_pool", ctypes.c_void_p), ("idxblk_pool", ctypes.c_void_p),
                ("ingested", ctypes.c_void_p), ("blkpos_pool", ctypes.c_void_p)]


def _section(sec) -> "_SEC3":
    return _SEC3(*(0, 0, 0) if sec is None else tuple(int(v) for v in sec))


_P = ctypes.c_void_p
_I = ctypes.c_int
_CFG = ctypes.POINTER(qsa_config)
_ROWS = ctypes.POINTER(qsa_rows)
_CACHE = ctypes.POINTER(qsa_cache)

LIB.qsa_strerror.restype = ctypes.c_char_p
LIB.qsa_strerror.argtypes = [_I]
LIB.qsa_config_check.restype = _I
LIB.qsa_config_check.argtypes = [_CFG]
LIB.qsa_workspace_bytes.restype = ctypes.c_size_t
LIB.qsa_workspace_bytes.argtypes = [_CFG, _I, _I]
LIB.qsa_append.restype = _I
LIB.qsa_append.argtypes = [_CFG, _ROWS, _CACHE, _P, _P, _P, _P, _P]
LIB.qsa_rewind.restype = _I
LIB.qsa_rewind.argtypes = [_CFG, _I, _P, _P, _P, _P, _P]
LIB.qsa_index_score.restype = _I
LIB.qsa_index_score.argtypes = [_CFG, _ROWS, _CACHE, _P, _P, _P, _I, _P, _P]
LIB.qsa_topk_select.restype = _I
LIB.qsa_topk_select.argtypes = [_CFG, _ROWS, _P, _I, _P, _P, _P, _P]
LIB.qsa_gather_attn.restype = _I
LIB.qsa_gather_attn.argtypes = [_CFG, _ROWS, _CACHE, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]
LIB.qsa_gather_attn_static.restype = _I
LIB.qsa_gather_attn_static.argtypes = [_CFG, _ROWS, _CACHE, _P, _P, _P, _P, _P, _P]
LIB.qsa_set_wait_limit_ns.restype = ctypes.c_ulonglong
LIB.qsa_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
LIB.qsa_stage_in.restype = _I
LIB.qsa_stage_in.argtypes = [_P, _P, ctypes.c_size_t, _P]
LIB.qsa_max_attend_tokens.restype = _I
LIB.qsa_max_attend_tokens.argtypes = [_CFG]
LIB.qsa_gather_attn_reuse.restype = _I
LIB.qsa_gather_attn_reuse.argtypes = [_CFG, _ROWS, _CACHE, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]
LIB.qsa_decode_reuse.restype = _I
LIB.qsa_decode_reuse.argtypes = [_CFG, _ROWS, _CACHE, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                 _P, _P]
_PRE = ctypes.POINTER(qsa_pre_indexer)
LIB.qsa_append_pre.restype = _I
LIB.qsa_append_pre.argtypes = [_CFG, _PRE, _ROWS, _CACHE, _P, _P, _P, _P, _P]
LIB.qsa_pre_index_q.restype = _I
LIB.qsa_pre_index_q.argtypes = [_CFG, _PRE, _ROWS, _P, _P, _P]
LIB.qsa_workspace_bytes_pre.restype = ctypes.c_size_t
LIB.qsa_workspace_bytes_pre.argtypes = [_CFG, _I, _I]
LIB.qsa_idxblk_page_bytes.restype = ctypes.c_size_t
LIB.qsa_idxblk_page_bytes.argtypes = [_CFG]
LIB.qsa_quantize_index_q.restype = _I
LIB.qsa_quantize_index_q.argtypes = [_CFG, _I, _P, _P, _P]
_ATT = ctypes.POINTER(qsa_attn_options)
LIB.qsa_append_ex.restype = _I
LIB.qsa_append_ex.argtypes = [_CFG, _PRE, _ATT, _ROWS, _CACHE, _P, _P, _P, _P, _P]
LIB.qsa_workspace_bytes_ex.restype = ctypes.c_size_t
LIB.qsa_workspace_bytes_ex.argtypes = [_CFG, _I, _I]
LIB.qsa_decode_ex.restype = _I
LIB.qsa_decode_ex.argtypes = [_CFG, _PRE, _ATT, _ROWS, _CACHE, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                              ctypes.c_size_t, _P, _P]
LIB.qsa_decode_pre.restype = _I
LIB.qsa_decode_pre.argtypes = [_CFG, _PRE, _ROWS, _CACHE, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                               ctypes.c_size_t, _P, _P]
LIB.qsa_decode.restype = _I
LIB.qsa_decode.argtypes = [_CFG, _ROWS, _CACHE, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                           ctypes.c_size_t, _P, _P]


class QsaError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = code
        msg = f"{where}: {qsa_strerror(code)} (status {code})"
        super().__init__(msg + (f"; {detail}" if detail else ""))


def qsa_strerror(code: int) -> str:
    return LIB.qsa_strerror(int(code)).decode()


def _check(rc: int, where: str, detail: str = "") -> None:
    if rc != QSA_OK:
        raise QsaError(rc, where, detail)


def _ptr(t: Optional[torch.Tensor], dtype=None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libqsa must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ---------------------------------------------------------------------------
# Marshalling helpers
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Config:
    ratio: int
    budget: int
    n_idx_heads: int
    idx_dim: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int = 128
    page_size: int = 64
    index_format: int = QSA_INDEX_BF16
    local_window: int = 0

    def c(self) -> qsa_config:
        return qsa_config(self.ratio, self.budget, self.n_idx_heads, self.idx_dim,
                          self.n_q_heads, self.n_kv_heads, self.head_dim, self.page_size,
                          self.index_format, self.local_window)

    @property
    def topk(self) -> int:
        return self.budget // self.ratio

    @classmethod
    def of(cls, shapes, index_format: int = QSA_INDEX_BF16, local_window: int = 0) -> "Config":
        return cls(shapes.ratio, shapes.budget, shapes.n_idx_heads, shapes.idx_dim,
                   shapes.n_q_heads, shapes.n_kv_heads, shapes.head_dim, shapes.page_size, index_format,
                   local_window)


class PagedCache:
    """Device pools of a paged indexer + KV cache, allocated with torch.

    page_table: [n_slots, max_pages] int32 (host or device; copied to device)."""

    def __init__(self, cfg: Config, page_table: torch.Tensor, num_pages: int, device="cuda",
                 mrope: bool = False):
        self.cfg = cfg
        P = cfg.page_size
        self.page_table = page_table.to(device=device, dtype=torch.int32).contiguous()
        self.n_slots, self.max_pages = self.page_table.shape
        self.num_pages = num_pages
        self.k_pool = torch.zeros(num_pages, P, cfg.n_kv_heads, cfg.head_dim, dtype=torch.bfloat16, device=device)
        self.v_pool = torch.zeros_like(self.k_pool)
        self.idxraw_pool = torch.zeros(num_pages, P, cfg.idx_dim, dtype=torch.bfloat16, device=device)
        # block keys: P/ratio rows of idx_dim per page, stored tiled (see qsa.h); with the
        # MXFP8 / MXFP4 index formats a byte plane of qsa_idxblk_page_bytes() per page
        if cfg.index_format in (QSA_INDEX_MXFP8, QSA_INDEX_MXFP4):
            self.idxblk_pool = torch.zeros(num_pages, qsa_idxblk_page_bytes(cfg), dtype=torch.uint8, device=device)
        else:
            self.idxblk_pool = torch.zeros(num_pages, (P // cfg.ratio) * cfg.idx_dim, dtype=torch.bfloat16,
                                           device=device)
        self.ingested = torch.zeros(self.n_slots, dtype=torch.int32, device=device)
        # mrope: the (t, h, w) of each block's first token, for a pre-indexer with an MRoPE section
        self.blkpos_pool = (torch.zeros(num_pages, P // cfg.ratio, 4, dtype=torch.int32, device=device)
                            if mrope else None)

    @property
    def capacity(self) -> int:
        return self.max_pages * self.cfg.page_size

    @property
    def max_blocks(self) -> int:
        return self.capacity // self.cfg.ratio

    def c(self) -> qsa_cache:
        return qsa_cache(_ptr(self.page_table), self.n_slots, self.max_pages, self.num_pages,
                         _ptr(self.k_pool), _ptr(self.v_pool), _ptr(self.idxraw_pool),
                         _ptr(self.idxblk_pool), _ptr(self.ingested),
                         None if self.blkpos_pool is None else _ptr(self.blkpos_pool))


class Rows:
    """Row layout of a step: n_seq sequences x R rows, sequence-major."""

    def __init__(self, seq_ids: torch.Tensor, pos0: torch.Tensor, rows_per_seq: int,
                 pos0_host: Optional[torch.Tensor] = None, advance: bool = False,
                 mrope_pos: Optional[torch.Tensor] = None):
        self.seq_ids = seq_ids.to(torch.int32).contiguous()
        # [n_seq * R, 3] device int32: each row's (t, h, w) for MRoPE (None: text rows)
        self.mrope_pos = None if mrope_pos is None else mrope_pos.to(torch.int32).contiguous()
        self.pos0 = pos0 if (pos0.dtype == torch.int32 and pos0.is_contiguous()) else pos0.to(torch.int32).contiguous()
        self.R = rows_per_seq
        self.pos0_host = None if pos0_host is None else pos0_host.to(torch.int32).cpu().contiguous()
        self.advance = bool(advance)

    @property
    def n_seq(self) -> int:
        return self.seq_ids.numel()

    @property
    def n_rows(self) -> int:
        return self.n_seq * self.R

    def c(self) -> qsa_rows:
        return qsa_rows(self.n_seq, self.R, _ptr(self.seq_ids), _ptr(self.pos0),
                        None if self.pos0_host is None else _ptr(self.pos0_host), int(self.advance),
                        None if self.mrope_pos is None else _ptr(self.mrope_pos))


# ---------------------------------------------------------------------------
# Entry points (same names as the C ABI)
# ---------------------------------------------------------------------------

def qsa_config_check(cfg: Config) -> int:
    return LIB.qsa_config_check(ctypes.byref(cfg.c()))


def qsa_workspace_bytes(cfg: Config, max_rows: int, max_blocks_per_row: int) -> int:
    return LIB.qsa_workspace_bytes(ctypes.byref(cfg.c()), max_rows, max_blocks_per_row)


def qsa_append(cfg: Config, rows: Rows, cache: PagedCache, k_new, v_new, idx_k_new, status,
               stream=None) -> None:
    rc = LIB.qsa_append(ctypes.byref(cfg.c()), ctypes.byref(rows.c()), ctypes.byref(cache.c()),
                        _ptr(k_new, torch.bfloat16), _ptr(v_new, torch.bfloat16),
                        _ptr(idx_k_new, torch.bfloat16), _ptr(status, torch.int32), _stream(stream))
    _check(rc, "qsa_append", f"capacity {cache.capacity} tokens per sequence" if rc == QSA_ERR_CAPACITY else "")


def qsa_rewind(cfg: Config, seq_ids, n_drop, ingested, status, stream=None) -> None:
    rc = LIB.qsa_rewind(ctypes.byref(cfg.c()), seq_ids.numel(), _ptr(seq_ids, torch.int32),
                        _ptr(n_drop, torch.int32), _ptr(ingested, torch.int32),
                        _ptr(status, torch.int32), _stream(stream))
    _check(rc, "qsa_rewind")


def qsa_index_score(cfg: Config, rows: Rows, cache: PagedCache, q_idx, w, scores, ld_scores: int,
                    status=None, stream=None) -> None:
    rc = LIB.qsa_index_score(ctypes.byref(cfg.c()), ctypes.byref(rows.c()), ctypes.byref(cache.c()),
                             _ptr(q_idx, torch.bfloat16), _ptr(w, torch.float32),
                             _ptr(scores, torch.float32), ld_scores, _ptr(status, torch.int32),
                             _stream(stream))
    _check(rc, "qsa_index_score")


def qsa_topk_select(cfg: Config, rows: Rows, scores, ld_scores: int, sel, n_sel, status=None,
                    stream=None) -> None:
    rc = LIB.qsa_topk_select(ctypes.byref(cfg.c()), ctypes.byref(rows.c()),
                             _ptr(scores, torch.float32), ld_scores, _ptr(sel, torch.int32),
                             _ptr(n_sel, torch.int32), _ptr(status, torch.int32), _stream(stream))
    _check(rc, "qsa_topk_select")


def qsa_gather_attn(cfg: Config, rows: Rows, cache: PagedCache, q, sel, n_sel, out, ws,
                    status=None, stream=None) -> None:
    rc = LIB.qsa_gather_attn(ctypes.byref(cfg.c()), ctypes.byref(rows.c()), ctypes.byref(cache.c()),
                             _ptr(q, torch.bfloat16), _ptr(sel, torch.int32), _ptr(n_sel, torch.int32),
                             _ptr(out, torch.bfloat16), _ptr(ws), ws.numel() * ws.element_size(),
                             _ptr(status, torch.int32), _stream(stream))
    _check(rc, "qsa_gather_attn")


def qsa_set_wait_limit_ns(ns: int) -> int:
    """Test hook: the index-score kernel's wait limit in ns (0 = default 1 s);
    returns the previous limit."""
    return int(LIB.qsa_set_wait_limit_ns(ctypes.c_ulonglong(ns)))


def qsa_stage_in(dst: torch.Tensor, src: torch.Tensor, stream=None) -> None:
    """Copy the bytes of pinned host tensor `src` into device tensor `dst` (same
    byte size, a multiple of 16) with a kernel in the stream's programmatic
    chain (see include/qsa.h)."""
    if not src.is_pinned() or dst.device.type != "cuda":
        raise ValueError("qsa_stage_in copies a pinned host tensor into a device tensor")
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("qsa_stage_in: source and destination sizes differ")
    _check(LIB.qsa_stage_in(_ptr(dst), _ptr(src), nbytes, _stream(stream)), "qsa_stage_in")


def qsa_gather_attn_static(cfg: Config, rows: Rows, cache: PagedCache, q, sel, n_sel, out,
                           status=None, stream=None) -> None:
    """qsa_gather_attn for callers that cannot pass a workspace: the split
    partials live in a fixed array inside the library (shared by every call on
    the device; calls must not overlap on the GPU). Allocates nothing."""
    rc = LIB.qsa_gather_attn_static(ctypes.byref(cfg.c()), ctypes.byref(rows.c()), ctypes.byref(cache.c()),
                                    _ptr(q, torch.bfloat16), _ptr(sel, torch.int32), _ptr(n_sel, torch.int32),
                                    _ptr(out, torch.bfloat16), _ptr(status, torch.int32), _stream(stream))
    _check(rc, "qsa_gather_attn_static")


def qsa_decode(cfg: Config, rows: Rows, cache: PagedCache, k_new, v_new, idx_k_new, q_idx, w, q,
               out, ws, status, sel_out=None, n_sel_out=None, stream=None) -> None:
    rc = LIB.qsa_decode(ctypes.byref(cfg.c()), ctypes.byref(rows.c()), ctypes.byref(cache.c()),
                        _ptr(k_new, torch.bfloat16), _ptr(v_new, torch.bfloat16),
                        _ptr(idx_k_new, torch.bfloat16), _ptr(q_idx, torch.bfloat16),
                        _ptr(w, torch.float32), _ptr(q, torch.bfloat16),
                        _ptr(sel_out, torch.int32), _ptr(n_sel_out, torch.int32),
                        _ptr(out, torch.bfloat16), _ptr(ws), ws.numel() * ws.element_size(),
                        _ptr(status, torch.int32), _stream(stream))
    _check(rc, "qsa_decode", f"capacity {cache.capacity} tokens per sequence" if rc == QSA_ERR_CAPACITY else "")


def qsa_max_attend_tokens(cfg: Config) -> int:
    return LIB.qsa_max_attend_tokens(ctypes.byref(cfg.c()))


def qsa_gather_attn_reuse(cfg: Config, rows: Rows, cache: PagedCache, q, sel, n_sel, sel_pos, out, ws,
                          status=None, stream=None) -> None:
    """Gather attention with a selection made earlier by the row at sel_pos
    (MTP draft steps, shared indexer layers): reused blocks plus every token
    from that position's block boundary to the row."""
    rc = LIB.qsa_gather_attn_reuse(ctypes.byref(cfg.c()), ctypes.byref(rows.c()), ctypes.byref(cache.c()),
                                   _ptr(q, torch.bfloat16), _ptr(sel, torch.int32), _ptr(n_sel, torch.int32),
                                   _ptr(sel_pos, torch.int32), _ptr(out, torch.bfloat16), _ptr(ws),
                                   ws.numel() * ws.element_size(), _ptr(status, torch.int32), _stream(stream))
    _check(rc, "qsa_gather_attn_reuse")


def qsa_decode_reuse(cfg: Config, rows: Rows, cache: PagedCache, k_new, v_new, idx_k_new, q, sel, n_sel,
                     sel_pos, out, ws, status, stream=None) -> None:
    """The fused step with a reused selection: append (side caches keep
    updating), then attention over the reused token set; no scoring or
    selection."""
    rc = LIB.qsa_decode_reuse(ctypes.byref(cfg.c()), ctypes.byref(rows.c()), ctypes.byref(cache.c()),
                              _ptr(k_new, torch.bfloat16), _ptr(v_new, torch.bfloat16),
                              _ptr(idx_k_new, torch.bfloat16), _ptr(q, torch.bfloat16),
                              _ptr(sel, torch.int32), _ptr(n_sel, torch.int32), _ptr(sel_pos, torch.int32),
                              _ptr(out, torch.bfloat16), _ptr(ws), ws.numel() * ws.element_size(),
                              _ptr(status, torch.int32), _stream(stream))
    _check(rc, "qsa_decode_reuse", f"capacity {cache.capacity} tokens per sequence" if rc == QSA_ERR_CAPACITY else "")


class PreIndexer:
    """Pre-indexer parameters: per-dimension norm gains (device fp32 [d_I]; the
    norm multiplies by 1 + gain), epsilon, RoPE base and rotary dims."""

    def __init__(self, gamma_q: torch.Tensor, gamma_k: torch.Tensor, eps: float, rope_theta: float,
                 rotary_dim: int, mrope_section=None):
        self.gamma_q = gamma_q.to(torch.float32).contiguous()
        self.gamma_k = gamma_k.to(torch.float32).contiguous()
        self.eps, self.rope_theta, self.rotary_dim = float(eps), float(rope_theta), int(rotary_dim)
        self.mrope_section = mrope_section  # (t, h, w) pairs, or None: plain RoPE

    def c(self) -> qsa_pre_indexer:
        return qsa_pre_indexer(_ptr(self.gamma_q), _ptr(self.gamma_k), self.eps, self.rope_theta,
                               self.rotary_dim, _section(self.mrope_section))


def qsa_append_pre(cfg: Config, pre: PreIndexer, rows: Rows, cache: PagedCache, k_new, v_new, idx_k_new,
                   status, stream=None) -> None:
    rc = LIB.qsa_append_pre(ctypes.byref(cfg.c()), ctypes.byref(pre.c()), ctypes.byref(rows.c()),
                            ctypes.byref(cache.c()), _ptr(k_new, torch.bfloat16), _ptr(v_new, torch.bfloat16),
                            _ptr(idx_k_new, torch.bfloat16), _ptr(status, torch.int32), _stream(stream))
    _check(rc, "qsa_append_pre", f"capacity {cache.capacity} tokens per sequence" if rc == QSA_ERR_CAPACITY else "")


def qsa_pre_index_q(cfg: Config, pre: PreIndexer, rows: Rows, q_idx, q_out, stream=None) -> None:
    rc = LIB.qsa_pre_index_q(ctypes.byref(cfg.c()), ctypes.byref(pre.c()), ctypes.byref(rows.c()),
                             _ptr(q_idx, torch.bfloat16), _ptr(q_out, torch.bfloat16), _stream(stream))
    _check(rc, "qsa_pre_index_q")


class AttnOptions:
    """Main-attention options (qsa_attn_options): optional q / k norm gains
    (device fp32 [D]; the norm multiplies by 1 + gain), eps, RoPE base, rotary
    dims, and an optional sigmoid output gate (device bf16 [rows, Hq, D])."""

    def __init__(self, gamma_q=None, gamma_k=None, eps: float = 1e-6, rope_theta: float = 1e4,
                 rotary_dim: int = 64, gate=None, mrope_section=None):
        self.gamma_q = None if gamma_q is None else gamma_q.to(torch.float32).contiguous()
        self.gamma_k = None if gamma_k is None else gamma_k.to(torch.float32).contiguous()
        self.eps, self.rope_theta, self.rotary_dim = float(eps), float(rope_theta), int(rotary_dim)
        self.gate = gate
        self.mrope_section = mrope_section  # (t, h, w) pairs, or None: plain RoPE

    def c(self) -> qsa_attn_options:
        return qsa_attn_options(_ptr(self.gamma_q), _ptr(self.gamma_k), self.eps, self.rope_theta,
                                self.rotary_dim, _ptr(self.gate, torch.bfloat16), _section(self.mrope_section))


def _ref(x):
    return None if x is None else ctypes.byref(x.c())


def qsa_append_ex(cfg: Config, pre, attn, rows: Rows, cache: PagedCache, k_new, v_new, idx_k_new, status,
                  stream=None) -> None:
    rc = LIB.qsa_append_ex(ctypes.byref(cfg.c()), _ref(pre), _ref(attn), ctypes.byref(rows.c()),
                           ctypes.byref(cache.c()), _ptr(k_new, torch.bfloat16), _ptr(v_new, torch.bfloat16),
                           _ptr(idx_k_new, torch.bfloat16), _ptr(status, torch.int32), _stream(stream))
    _check(rc, "qsa_append_ex", f"capacity {cache.capacity} tokens per sequence" if rc == QSA_ERR_CAPACITY else "")


def qsa_workspace_bytes_ex(cfg: Config, max_rows: int, max_blocks_per_row: int) -> int:
    return LIB.qsa_workspace_bytes_ex(ctypes.byref(cfg.c()), max_rows, max_blocks_per_row)


def workspace_ex(cfg: Config, max_rows: int, max_blocks_per_row: int, device="cuda") -> torch.Tensor:
    """A device workspace of qsa_workspace_bytes_ex() bytes (uint8)."""
    n = qsa_workspace_bytes_ex(cfg, max_rows, max_blocks_per_row)
    if n == 0:
        raise QsaError(QSA_ERR_UNSUPPORTED, "qsa_workspace_bytes_ex")
    return torch.empty(n, dtype=torch.uint8, device=device)


def qsa_decode_ex(cfg: Config, pre, attn, rows: Rows, cache: PagedCache, k_new, v_new, idx_k_new, q_idx, w, q,
                  out, ws, status, sel_out=None, n_sel_out=None, stream=None) -> None:
    rc = LIB.qsa_decode_ex(ctypes.byref(cfg.c()), _ref(pre), _ref(attn), ctypes.byref(rows.c()),
                           ctypes.byref(cache.c()), _ptr(k_new, torch.bfloat16), _ptr(v_new, torch.bfloat16),
                           _ptr(idx_k_new, torch.bfloat16), _ptr(q_idx, torch.bfloat16), _ptr(w, torch.float32),
                           _ptr(q, torch.bfloat16), _ptr(sel_out, torch.int32), _ptr(n_sel_out, torch.int32),
                           _ptr(out, torch.bfloat16), _ptr(ws), ws.numel() * ws.element_size(),
                           _ptr(status, torch.int32), _stream(stream))
    _check(rc, "qsa_decode_ex", f"capacity {cache.capacity} tokens per sequence" if rc == QSA_ERR_CAPACITY else "")


def qsa_idxblk_page_bytes(cfg: Config) -> int:
    """Bytes of one block-pool page for the configuration's index format (0: invalid)."""
    return LIB.qsa_idxblk_page_bytes(ctypes.byref(cfg.c()))


def qsa_quantize_index_q(cfg: Config, q_idx, q_out, stream=None) -> None:
    """MX round trip of index query heads [rows, H_I, d_I] (bf16 in and out): MXFP4 for an
    MXFP4 configuration, else MXFP8."""
    n_rows = q_idx.numel() // (cfg.n_idx_heads * cfg.idx_dim)
    if q_out.numel() != q_idx.numel():
        raise ValueError("q_out must match q_idx")
    rc = LIB.qsa_quantize_index_q(ctypes.byref(cfg.c()), n_rows, _ptr(q_idx, torch.bfloat16),
                                  _ptr(q_out, torch.bfloat16), _stream(stream))
    _check(rc, "qsa_quantize_index_q")


def qsa_workspace_bytes_pre(cfg: Config, max_rows: int, max_blocks_per_row: int) -> int:
    return LIB.qsa_workspace_bytes_pre(ctypes.byref(cfg.c()), max_rows, max_blocks_per_row)


def workspace_pre(cfg: Config, max_rows: int, max_blocks_per_row: int, device="cuda") -> torch.Tensor:
    """A device workspace of qsa_workspace_bytes_pre() bytes (uint8)."""
    n = qsa_workspace_bytes_pre(cfg, max_rows, max_blocks_per_row)
    if n == 0:
        raise QsaError(QSA_ERR_UNSUPPORTED, "qsa_workspace_bytes_pre")
    return torch.empty(n, dtype=torch.uint8, device=device)


def qsa_decode_pre(cfg: Config, pre: PreIndexer, rows: Rows, cache: PagedCache, k_new, v_new, idx_k_new, q_idx,
                   w, q, out, ws, status, sel_out=None, n_sel_out=None, stream=None) -> None:
    rc = LIB.qsa_decode_pre(ctypes.byref(cfg.c()), ctypes.byref(pre.c()), ctypes.byref(rows.c()),
                            ctypes.byref(cache.c()), _ptr(k_new, torch.bfloat16), _ptr(v_new, torch.bfloat16),
                            _ptr(idx_k_new, torch.bfloat16), _ptr(q_idx, torch.bfloat16), _ptr(w, torch.float32),
                            _ptr(q, torch.bfloat16), _ptr(sel_out, torch.int32), _ptr(n_sel_out, torch.int32),
                            _ptr(out, torch.bfloat16), _ptr(ws), ws.numel() * ws.element_size(),
                            _ptr(status, torch.int32), _stream(stream))
    _check(rc, "qsa_decode_pre", f"capacity {cache.capacity} tokens per sequence" if rc == QSA_ERR_CAPACITY else "")


def workspace(cfg: Config, max_rows: int, max_blocks_per_row: int, device="cuda") -> torch.Tensor:
    """A device workspace of qsa_workspace_bytes() bytes (uint8)."""
    n = qsa_workspace_bytes(cfg, max_rows, max_blocks_per_row)
    if n == 0:
        raise QsaError(QSA_ERR_UNSUPPORTED, "qsa_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)
