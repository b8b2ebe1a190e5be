"""CPU oracle for the sparse MXFP4 attention decode step (ctypes binding of smx_oracle.c).

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package. The CUDA library never does,
and this package imports nothing from it.

All array arguments are NumPy arrays; outputs are returned as new arrays. The arithmetic
lives in ``smx_oracle.c`` (fp64, explicit format tables); this file only marshals arguments.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "smx_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

KV_MXFP4 = 0
KV_E4M3_ROWSCALE = 1
KV_NVFP4 = 2
MXFP4_PAGE_BYTES = 8704
E4M3RS_PAGE_BYTES = 16896
NVFP4_PAGE_BYTES = 9216


def compile_library(src: str, out: str, quiet: bool = False) -> None:
    """gcc, -O2, no fast-math, no FMA contraction (so x86-64 and aarch64 give the same bits)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=quiet)


def build(force: bool = False) -> str:
    """Compile smx_oracle.c into oracle/_build/liboracle.so."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    hdr = os.path.join(_HERE, "smx_oracle.h")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC), os.path.getmtime(hdr))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    compile_library(_SRC, tmp)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Q", ctypes.c_int32), ("Hq", ctypes.c_int32),
                ("Hkv", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("n_pool_pages", ctypes.c_int64), ("topk", ctypes.c_int32),
                ("num_splits", ctypes.c_int32), ("kv_format", ctypes.c_int32),
                ("pages_per_block", ctypes.c_int32), ("idx_format", ctypes.c_int32),
                ("nv_scale_k", ctypes.c_float), ("nv_scale_v", ctypes.c_float),
                ("nv_scale_idx", ctypes.c_float)]


@dataclass
class Shape:
    B: int
    Q: int
    Hq: int
    Hkv: int
    max_pages: int
    n_pool_pages: int
    topk: int
    num_splits: int
    kv_format: int = KV_MXFP4
    pages_per_block: int = 1
    idx_format: int = KV_MXFP4
    nv_scale_k: float = 1.0
    nv_scale_v: float = 1.0
    nv_scale_idx: float = 1.0

    def c(self) -> _Shape:
        return _Shape(self.B, self.Q, self.Hq, self.Hkv, self.max_pages, self.n_pool_pages,
                      self.topk, self.num_splits, self.kv_format, self.pages_per_block,
                      self.idx_format, self.nv_scale_k, self.nv_scale_v, self.nv_scale_idx)

    @property
    def kv_page_bytes(self) -> int:
        return {KV_E4M3_ROWSCALE: E4M3RS_PAGE_BYTES, KV_NVFP4: NVFP4_PAGE_BYTES}.get(self.kv_format, MXFP4_PAGE_BYTES)

    @property
    def idx_page_bytes(self) -> int:
        return NVFP4_PAGE_BYTES if self.idx_format == KV_NVFP4 else MXFP4_PAGE_BYTES


def shape_of(w, num_splits=None) -> Shape:
    """Oracle shape of a workload object (anything with B, Q, Hq, Hkv, max_pages, ...)."""
    return Shape(w.B, w.Q, w.Hq, w.Hkv, w.max_pages, w.n_pool_pages, w.topk,
                 w.num_splits if num_splits is None else num_splits, w.kv_format,
                 getattr(w, "pages_per_block", 1), getattr(w, "idx_format", KV_MXFP4),
                 getattr(w, "nv_scale_k", 1.0), getattr(w, "nv_scale_v", 1.0),
                 getattr(w, "nv_scale_idx", 1.0))


def lib():
    """The oracle library, built on first use. SMX_ORACLE_LIB names a prebuilt copy to load
    instead (the pins' own test runs them against copies with planted mistakes)."""
    global _lib
    if _lib is None:
        path = os.environ.get("SMX_ORACLE_LIB") or build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        S = ctypes.POINTER(_Shape)
        sigs = {
            "orc_e2m1_value": (ctypes.c_double, [ctypes.c_int]),
            "orc_e8m0_value": (ctypes.c_double, [ctypes.c_int]),
            "orc_e4m3_value": (ctypes.c_double, [ctypes.c_int]),
            "orc_bf16_value": (ctypes.c_double, [ctypes.c_uint16]),
            "orc_e2m1_encode": (ctypes.c_uint8, [ctypes.c_double]),
            "orc_e4m3_encode": (ctypes.c_uint8, [ctypes.c_double]),
            "orc_mxfp4_quant_row": (None, [P, P, P]),
            "orc_e4m3rs_quant_row": (None, [P, P, P]),
            "orc_nvfp4_quant_row": (None, [P, ctypes.c_float, P, P]),
            "orc_nvfp4_load_row": (None, [P, ctypes.c_int, ctypes.c_float, P]),
            "orc_pack_q_one": (ctypes.c_uint8, [ctypes.c_float]),
            "orc_pack_q_e4m3": (None, [P, P, ctypes.c_int64]),
            "orc_mxfp4_load_row": (None, [P, ctypes.c_int, P]),
            "orc_e4m3rs_load_row": (None, [P, ctypes.c_int, P]),
            "orc_kv_insert": (None, [S, P, P, P, P, P, P, P, P]),
            "orc_kv_fill": (None, [S, P, P, P, ctypes.c_int64, P, P, P, P, P]),
            "orc_index_scores": (None, [S, P, P, P, P, P]),
            "orc_topk": (None, [S, P, P, P, P]),
            "orc_sparse_attn_split": (None, [S, P, P, P, P, P, P, P, P, P, P]),
            "orc_sparse_attn_merge": (None, [S, P, P, P, P]),
            "orc_decode_step": (None, [S] + [P] * 19),
            "orc_decode_step_reuse": (None, [S] + [P] * 15),
            "orc_set_threads": (None, [ctypes.c_int]),
            "orc_max_threads": (ctypes.c_int, []),
        }
        for name, (res, args) in sigs.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def max_threads() -> int:
    return int(lib().orc_max_threads())


# ---- element formats -------------------------------------------------------------------
def e2m1_value(nibble: int) -> float:
    return lib().orc_e2m1_value(int(nibble))


def e8m0_value(byte: int) -> float:
    return lib().orc_e8m0_value(int(byte))


def e4m3_value(byte: int) -> float:
    return lib().orc_e4m3_value(int(byte))


def bf16_value(bits: int) -> float:
    return lib().orc_bf16_value(int(bits))


def e2m1_encode(v: float) -> int:
    return int(lib().orc_e2m1_encode(float(v)))


def e4m3_encode(v: float) -> int:
    return int(lib().orc_e4m3_encode(float(v)))


# ---- quantisers ------------------------------------------------------------------------
def mxfp4_quant_row(x):
    x = _c(x, np.float32).reshape(128)
    nib = np.zeros(64, np.uint8)
    sc = np.zeros(4, np.uint8)
    lib().orc_mxfp4_quant_row(_p(x), _p(nib), _p(sc))
    return nib, sc


def e4m3rs_quant_row(x):
    x = _c(x, np.float32).reshape(128)
    codes = np.zeros(128, np.uint8)
    s = np.zeros(1, np.float32)
    lib().orc_e4m3rs_quant_row(_p(x), _p(codes), _p(s))
    return codes, s[0]


def nvfp4_quant_row(x, g: float):
    """One row to NVFP4 with the per-tensor decode scale g: (64 nibble bytes, 8 E4M3 scale bytes)."""
    x = _c(x, np.float32).reshape(128)
    nib = np.zeros(64, np.uint8)
    sc = np.zeros(8, np.uint8)
    lib().orc_nvfp4_quant_row(_p(x), float(g), _p(nib), _p(sc))
    return nib, sc


def nvfp4_load_row(page, slot: int, g: float):
    page = _c(page, np.uint8).reshape(-1)
    assert page.size >= NVFP4_PAGE_BYTES
    out = np.zeros(128, np.float64)
    lib().orc_nvfp4_load_row(_p(page), int(slot), float(g), _p(out))
    return out


def pack_q_e4m3(q):
    q = _c(q, np.float32)
    out = np.zeros(q.shape, np.uint8)
    lib().orc_pack_q_e4m3(_p(q), _p(out), q.size)
    return out


def mxfp4_load_row(page, slot: int):
    page = _c(page, np.uint8).reshape(-1)
    assert page.size >= MXFP4_PAGE_BYTES
    out = np.zeros(128, np.float64)
    lib().orc_mxfp4_load_row(_p(page), int(slot), _p(out))
    return out


def e4m3rs_load_row(page, slot: int):
    page = _c(page, np.uint8).reshape(-1)
    assert page.size >= E4M3RS_PAGE_BYTES
    out = np.zeros(128, np.float64)
    lib().orc_e4m3rs_load_row(_p(page), int(slot), _p(out))
    return out


# ---- the step's parts --------------------------------------------------------------------
def kv_insert(sh: Shape, k_new, v_new, kidx_new, page_table, ctx_len, k_pool, v_pool, idx_pool):
    """In place on the three pools (uint8 arrays, C-contiguous)."""
    k_new, v_new, kidx_new = (_c(a, np.float32) for a in (k_new, v_new, kidx_new))
    page_table, ctx_len = _c(page_table, np.int32), _c(ctx_len, np.int32)
    cs = sh.c()
    lib().orc_kv_insert(ctypes.byref(cs), _p(k_new), _p(v_new), _p(kidx_new), _p(page_table),
                        _p(ctx_len), _p(k_pool), _p(v_pool), _p(idx_pool))


def kv_fill(sh: Shape, k, v, kidx, page_table, n_fill, k_pool, v_pool, idx_pool):
    """Quantise positions [0, n_fill[b]) from dense k, v [B][T][Hkv][128], kidx [B][T][128]."""
    k, v, kidx = (_c(a, np.float32) for a in (k, v, kidx))
    T = kidx.shape[1]
    page_table, n_fill = _c(page_table, np.int32), _c(n_fill, np.int32)
    cs = sh.c()
    lib().orc_kv_fill(ctypes.byref(cs), _p(k), _p(v), _p(kidx), T, _p(page_table), _p(n_fill),
                      _p(k_pool), _p(v_pool), _p(idx_pool))


def index_scores(sh: Shape, qidx_bf16, idx_pool, page_table, ctx_len):
    qidx_bf16 = _c(qidx_bf16, np.uint16)
    page_table, ctx_len = _c(page_table, np.int32), _c(ctx_len, np.int32)
    out = np.zeros((sh.B, sh.max_pages), np.float64)
    cs = sh.c()
    lib().orc_index_scores(ctypes.byref(cs), _p(qidx_bf16), _p(idx_pool), _p(page_table),
                           _p(ctx_len), _p(out))
    return out


def topk(sh: Shape, scores, ctx_len):
    scores = _c(scores, np.float64)
    ctx_len = _c(ctx_len, np.int32)
    pages = np.zeros((sh.B, sh.topk), np.int32)
    count = np.zeros(sh.B, np.int32)
    cs = sh.c()
    lib().orc_topk(ctypes.byref(cs), _p(scores), _p(ctx_len), _p(pages), _p(count))
    return pages, count


def sparse_attn_split(sh: Shape, q, k_pool, v_pool, page_table, ctx_len, topk_pages, topk_count):
    """q: uint8 e4m3 bytes (MXFP4 K/V) or uint16 bf16 bits (e4m3 row-scale K/V),
    [B][Q][Hq][128]. Returns (part_o [B][S][Q][Hq][128], part_m, part_l [B][S][Q][Hq])."""
    q = _c(q, np.uint16 if sh.kv_format == KV_E4M3_ROWSCALE else np.uint8)
    page_table, ctx_len = _c(page_table, np.int32), _c(ctx_len, np.int32)
    topk_pages, topk_count = _c(topk_pages, np.int32), _c(topk_count, np.int32)
    S = sh.num_splits
    po = np.zeros((sh.B, S, sh.Q, sh.Hq, 128), np.float64)
    pm = np.zeros((sh.B, S, sh.Q, sh.Hq), np.float64)
    pl = np.zeros((sh.B, S, sh.Q, sh.Hq), np.float64)
    cs = sh.c()
    lib().orc_sparse_attn_split(ctypes.byref(cs), _p(q), _p(k_pool), _p(v_pool), _p(page_table),
                                _p(ctx_len), _p(topk_pages), _p(topk_count), _p(po), _p(pm), _p(pl))
    return po, pm, pl


def sparse_attn_merge(sh: Shape, part_o, part_m, part_l):
    part_o, part_m, part_l = (_c(a, np.float64) for a in (part_o, part_m, part_l))
    out = np.zeros((sh.B, sh.Q, sh.Hq, 128), np.float64)
    cs = sh.c()
    lib().orc_sparse_attn_merge(ctypes.byref(cs), _p(part_o), _p(part_m), _p(part_l), _p(out))
    return out


def decode_step(sh: Shape, *, q_f32=None, q_bf16=None, qidx_bf16, k_new, v_new, kidx_new,
                page_table, ctx_len, k_pool, v_pool, idx_pool, want_partials=False):
    """The whole step; the pools are updated in place. Returns a dict with scores, topk_pages,
    topk_count, q_e4m3 (MXFP4 K/V only), out and, if asked, the partials."""
    q_f32 = None if q_f32 is None else _c(q_f32, np.float32)
    q_bf16 = None if q_bf16 is None else _c(q_bf16, np.uint16)
    qidx_bf16 = _c(qidx_bf16, np.uint16)
    k_new, v_new, kidx_new = (_c(a, np.float32) for a in (k_new, v_new, kidx_new))
    page_table, ctx_len = _c(page_table, np.int32), _c(ctx_len, np.int32)
    if sh.kv_format == KV_E4M3_ROWSCALE:
        assert q_bf16 is not None
    else:
        assert q_f32 is not None
    B, Q, Hq, S = sh.B, sh.Q, sh.Hq, sh.num_splits
    scores = np.zeros((B, sh.max_pages), np.float64)
    pages = np.zeros((B, sh.topk), np.int32)
    count = np.zeros(B, np.int32)
    q8 = np.zeros((B, Q, Hq, 128), np.uint8)
    out = np.zeros((B, Q, Hq, 128), np.float64)
    po = pm = pl = None
    if want_partials:
        po = np.zeros((B, S, Q, Hq, 128), np.float64)
        pm = np.zeros((B, S, Q, Hq), np.float64)
        pl = np.zeros((B, S, Q, Hq), np.float64)
    cs = sh.c()
    lib().orc_decode_step(ctypes.byref(cs), _p(q_f32), _p(q_bf16), _p(qidx_bf16), _p(k_new),
                          _p(v_new), _p(kidx_new), _p(page_table), _p(ctx_len), _p(k_pool),
                          _p(v_pool), _p(idx_pool), _p(scores), _p(pages), _p(count), _p(q8),
                          _p(po), _p(pm), _p(pl), _p(out))
    res = dict(scores=scores, topk_pages=pages, topk_count=count, out=out)
    if sh.kv_format != KV_E4M3_ROWSCALE:
        res["q_e4m3"] = q8
    if want_partials:
        res.update(part_o=po, part_m=pm, part_l=pl)
    return res



def decode_step_reuse(sh: Shape, *, q_f32=None, q_bf16=None, k_new, v_new, page_table, ctx_len,
                      k_pool, v_pool, topk_pages, topk_count, want_partials=False):
    """The step of a layer reusing an earlier layer's selection: K/V insert (the K and V pools
    updated in place; no index cache), q packing, split over (topk_pages, topk_count) as given,
    merge. Returns a dict with q_e4m3 (MXFP4 K/V only), out and, if asked, the partials."""
    q_f32 = None if q_f32 is None else _c(q_f32, np.float32)
    q_bf16 = None if q_bf16 is None else _c(q_bf16, np.uint16)
    k_new, v_new = (_c(a, np.float32) for a in (k_new, v_new))
    page_table, ctx_len = _c(page_table, np.int32), _c(ctx_len, np.int32)
    topk_pages, topk_count = _c(topk_pages, np.int32), _c(topk_count, np.int32)
    if sh.kv_format == KV_E4M3_ROWSCALE:
        assert q_bf16 is not None
    else:
        assert q_f32 is not None
    B, Q, Hq, S = sh.B, sh.Q, sh.Hq, sh.num_splits
    q8 = np.zeros((B, Q, Hq, 128), np.uint8)
    out = np.zeros((B, Q, Hq, 128), np.float64)
    po = pm = pl = None
    if want_partials:
        po = np.zeros((B, S, Q, Hq, 128), np.float64)
        pm = np.zeros((B, S, Q, Hq), np.float64)
        pl = np.zeros((B, S, Q, Hq), np.float64)
    cs = sh.c()
    lib().orc_decode_step_reuse(ctypes.byref(cs), _p(q_f32), _p(q_bf16), _p(k_new), _p(v_new),
                                _p(page_table), _p(ctx_len), _p(k_pool), _p(v_pool), _p(topk_pages),
                                _p(topk_count), _p(q8), _p(po), _p(pm), _p(pl), _p(out))
    res = dict(out=out)
    if sh.kv_format != KV_E4M3_ROWSCALE:
        res["q_e4m3"] = q8
    if want_partials:
        res.update(part_o=po, part_m=pm, part_l=pl)
    return res
