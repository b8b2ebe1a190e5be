"""ctypes binding of libsmx (include/smx.h), one Python function per C entry point.

Argument marshalling only: every step of the decode path runs in the CUDA kernels of
libsmx.so. Tensors must be CUDA tensors (torch is used for device memory and streams); outputs
that are not passed in are allocated with torch. Every call enqueues on the current torch
stream unless `stream` (a torch.cuda.Stream) is given. A non-zero status raises SmxError, and so
does a buffer smaller than the shape needs (checked here, before the call: the C ABI sees only
pointers).
There is no CPU fallback: if libsmx.so is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsmx.so")

KV_MXFP4 = 0
KV_E4M3_ROWSCALE = 1
KV_NVFP4 = 2   # E2M1 + an E4M3 scale per 16 elements + the pool's fp32 scale (K/V and index pools)
MXFP4_PAGE_BYTES = 8704
E4M3RS_PAGE_BYTES = 16896
NVFP4_PAGE_BYTES = 9216
DEV_BAD_PAGE_ID, DEV_BAD_CTX, DEV_BAD_TOPK, DEV_TIMEOUT = 1, 2, 4, 8
SMX_ERR_WORKSPACE = -4

# every symbol include/smx.h declares
SYMBOLS = ("smx_workspace_bytes", "smx_kv_insert_mxfp4", "smx_kv_insert", "smx_kv_prefill", "smx_pack_q_e4m3",
           "smx_index_score", "smx_index_score_topk", "smx_sparse_attn_split", "smx_sparse_attn_merge",
           "smx_decode_step", "smx_status_string", "smx_decode_step_launches",
           "smx_suggest_num_splits", "smx_decode_step_noalloc", "smx_decode_step_tensor_cores",
           "smx_decode_step_reuse", "smx_set_wait_limit_ns")


class SmxError(RuntimeError):
    pass


class _CShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Q", ctypes.c_int32), ("Hq", ctypes.c_int32),
                ("Hkv", ctypes.c_int32), ("D", ctypes.c_int32), ("Di", ctypes.c_int32),
                ("page_tokens", ctypes.c_int32), ("max_pages_per_row", ctypes.c_int32),
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
    max_pages_per_row: int
    n_pool_pages: int
    topk: int
    num_splits: int
    kv_format: int = KV_MXFP4
    D: int = 128
    Di: int = 128
    page_tokens: int = 128
    pages_per_block: int = 1
    idx_format: int = KV_MXFP4
    nv_scale_k: float = 0.0    # NVFP4 per-tensor decode scales (> 0 where that pool is NVFP4)
    nv_scale_v: float = 0.0
    nv_scale_idx: float = 0.0

    @classmethod
    def of(cls, w, num_splits=None) -> "Shape":
        """Shape of a workload object (B, Q, Hq, Hkv, max_pages, n_pool_pages, topk, ...)."""
        return cls(w.B, w.Q, w.Hq, w.Hkv, w.max_pages, w.n_pool_pages, w.topk,
                   w.num_splits if num_splits is None else num_splits, w.kv_format,
                   pages_per_block=getattr(w, "pages_per_block", 1),
                   idx_format=getattr(w, "idx_format", KV_MXFP4), nv_scale_k=getattr(w, "nv_scale_k", 0.0),
                   nv_scale_v=getattr(w, "nv_scale_v", 0.0), nv_scale_idx=getattr(w, "nv_scale_idx", 0.0))

    def c(self) -> _CShape:
        return _CShape(self.B, self.Q, self.Hq, self.Hkv, self.D, self.Di, self.page_tokens,
                       self.max_pages_per_row, self.n_pool_pages, self.topk, self.num_splits,
                       self.kv_format, self.pages_per_block, self.idx_format, self.nv_scale_k,
                       self.nv_scale_v, self.nv_scale_idx)

    @property
    def kv_page_bytes(self) -> int:
        return {KV_E4M3_ROWSCALE: E4M3RS_PAGE_BYTES, KV_NVFP4: NVFP4_PAGE_BYTES}.get(self.kv_format, MXFP4_PAGE_BYTES)

    @property
    def idx_page_bytes(self) -> int:
        return NVFP4_PAGE_BYTES if self.idx_format == KV_NVFP4 else MXFP4_PAGE_BYTES


_lib = None


def lib() -> ctypes.CDLL:
    """Load libsmx.so (built by __graft_entry__.build() or python -m ...build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise SmxError(f"libsmx.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, S, I64, ST = ctypes.c_void_p, ctypes.POINTER(_CShape), ctypes.c_int64, ctypes.c_void_p
        sigs = {
            "smx_workspace_bytes": (ctypes.c_size_t, [S]),
            "smx_kv_insert_mxfp4": (ctypes.c_int, [S] + [P] * 9 + [ST]),
            "smx_kv_insert": (ctypes.c_int, [S] + [P] * 9 + [ST]),
            "smx_kv_prefill": (ctypes.c_int, [S, P, P, P, I64] + [P] * 6 + [ST]),
            "smx_pack_q_e4m3": (ctypes.c_int, [P, P, I64, ST]),
            "smx_index_score": (ctypes.c_int, [S] + [P] * 6 + [ST]),
            "smx_index_score_topk": (ctypes.c_int, [S] + [P] * 8 + [ST]),
            "smx_sparse_attn_split": (ctypes.c_int, [S] + [P] * 11 + [ST]),
            "smx_sparse_attn_merge": (ctypes.c_int, [S, P, P, P, P, ST]),
            "smx_decode_step": (ctypes.c_int, [S] + [P] * 15 + [ctypes.c_size_t, P, ST]),
            "smx_decode_step_reuse": (ctypes.c_int, [S] + [P] * 12 + [ctypes.c_size_t, P, ST]),
            "smx_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "smx_decode_step_launches": (ctypes.c_int, [S]),
            "smx_suggest_num_splits": (ctypes.c_int, [S]),
            "smx_decode_step_tensor_cores": (ctypes.c_int, [S]),
            "smx_decode_step_noalloc": (ctypes.c_int, [S] + [P] * 15 + [ST]),
            "smx_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
        }
        for name, (res, args) in sigs.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise SmxError(f"{what}: {lib().smx_status_string(rc).decode()} ({rc})")


def _p(t):
    # a plain int: the entry points declare their pointer arguments c_void_p
    if t is None:
        return None
    if not t.is_cuda:
        raise SmxError("libsmx takes CUDA tensors only")
    if not t.is_contiguous():
        raise SmxError("libsmx takes contiguous tensors only")
    return t.data_ptr()


def _st(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(*ts):
    for t in ts:
        if t is not None:
            return t.device
    return torch.device("cuda")


def _need(what, **bufs):
    """Refuse a buffer smaller than the shape needs before anything is enqueued: the C ABI takes
    plain pointers and cannot see sizes. bufs: name -> (tensor or None, bytes the shape needs)."""
    for name, (t, nbytes) in bufs.items():
        if t is None:
            continue
        have = t.numel() * t.element_size()
        if have < nbytes:
            raise SmxError(f"{what}: {name} holds {have} bytes, the shape needs {nbytes}")


def _step_bufs(shape, q_f32, q_bf16, k_new, v_new, page_table, ctx_len, k_pool, v_pool, dev_status):
    """Sizes of the arguments every form of the step shares."""
    B, Q, Hq, Hkv = shape.B, shape.Q, shape.Hq, shape.Hkv
    return dict(q_f32=(q_f32, B * Q * Hq * 128 * 4), q_bf16=(q_bf16, B * Q * Hq * 128 * 2),
                k_new=(k_new, B * Q * Hkv * 128 * 4), v_new=(v_new, B * Q * Hkv * 128 * 4),
                page_table=(page_table, B * shape.max_pages_per_row * 4), ctx_len=(ctx_len, B * 4),
                k_pool=(k_pool, shape.n_pool_pages * Hkv * shape.kv_page_bytes),
                v_pool=(v_pool, shape.n_pool_pages * Hkv * shape.kv_page_bytes), dev_status=(dev_status, 4))


def workspace_bytes(shape: Shape) -> int:
    cs = shape.c()
    return int(lib().smx_workspace_bytes(ctypes.byref(cs)))


def decode_step_launches(shape: Shape) -> int:
    cs = shape.c()
    return int(lib().smx_decode_step_launches(ctypes.byref(cs)))


def decode_step_tensor_cores(shape: Shape) -> bool:
    """Whether the fused step runs its attention on tcgen05 (128-row tiles) for `shape` here."""
    cs = shape.c()
    rc = int(lib().smx_decode_step_tensor_cores(ctypes.byref(cs)))
    if rc < 0:
        raise SmxError(f"smx_decode_step_tensor_cores: {lib().smx_status_string(rc).decode()} ({rc})")
    return rc == 1


def suggest_num_splits(shape: Shape) -> int:
    """Partition count for `shape` on the current device (one wave of split CTAs, equal pages)."""
    cs = shape.c()
    n = int(lib().smx_suggest_num_splits(ctypes.byref(cs)))
    if n < 1:
        raise SmxError("smx_suggest_num_splits: invalid shape or CUDA query failed")
    return n


def kv_insert(shape, k_new, v_new, kidx_new, page_table, ctx_len, k_pool, v_pool, idx_pool,
              dev_status=None, stream=None):
    B, Q = shape.B, shape.Q
    _need("smx_kv_insert_mxfp4", **_step_bufs(shape, None, None, k_new, v_new, page_table, ctx_len, k_pool, v_pool,
                                        dev_status),
          kidx_new=(kidx_new, B * Q * 128 * 4), idx_pool=(idx_pool, shape.n_pool_pages * shape.idx_page_bytes))
    cs = shape.c()
    _check(lib().smx_kv_insert_mxfp4(ctypes.byref(cs), _p(k_new), _p(v_new), _p(kidx_new), _p(page_table),
                                     _p(ctx_len), _p(k_pool), _p(v_pool), _p(idx_pool), _p(dev_status),
                                     _st(stream)), "smx_kv_insert_mxfp4")


def kv_prefill(shape, k, v, kidx, page_table, n_fill, k_pool, v_pool, idx_pool, dev_status=None,
               stream=None):
    T = kidx.shape[1]
    B, Hkv = shape.B, shape.Hkv
    _need("smx_kv_prefill", k=(k, B * T * Hkv * 128 * 4), v=(v, B * T * Hkv * 128 * 4), kidx=(kidx, B * T * 128 * 4),
          **_step_bufs(shape, None, None, None, None, page_table, None, k_pool, v_pool, dev_status),
          n_fill=(n_fill, B * 4), idx_pool=(idx_pool, shape.n_pool_pages * shape.idx_page_bytes))
    cs = shape.c()
    _check(lib().smx_kv_prefill(ctypes.byref(cs), _p(k), _p(v), _p(kidx), T, _p(page_table),
                                _p(n_fill), _p(k_pool), _p(v_pool), _p(idx_pool), _p(dev_status),
                                _st(stream)), "smx_kv_prefill")


def pack_q_e4m3(q, out=None, stream=None):
    if out is None:
        out = torch.empty(q.shape, dtype=torch.uint8, device=q.device)
    _need("smx_pack_q_e4m3", out=(out, q.numel()))
    _check(lib().smx_pack_q_e4m3(_p(q), _p(out), q.numel(), _st(stream)), "smx_pack_q_e4m3")
    return out


def _index_bufs(shape, qidx_bf16, idx_pool, page_table, ctx_len, page_scores, dev_status):
    B = shape.B
    return dict(qidx_bf16=(qidx_bf16, B * shape.Q * 128 * 2), idx_pool=(idx_pool, shape.n_pool_pages * shape.idx_page_bytes),
                page_table=(page_table, B * shape.max_pages_per_row * 4), ctx_len=(ctx_len, B * 4),
                page_scores=(page_scores, B * shape.max_pages_per_row * 4), dev_status=(dev_status, 4))


def index_score(shape, qidx_bf16, idx_pool, page_table, ctx_len, page_scores=None, dev_status=None,
                stream=None):
    if page_scores is None:
        page_scores = torch.empty((shape.B, shape.max_pages_per_row), dtype=torch.float32,
                                  device=idx_pool.device)
    _need("smx_index_score", **_index_bufs(shape, qidx_bf16, idx_pool, page_table, ctx_len, page_scores, dev_status))
    cs = shape.c()
    _check(lib().smx_index_score(ctypes.byref(cs), _p(qidx_bf16), _p(idx_pool), _p(page_table),
                                 _p(ctx_len), _p(page_scores), _p(dev_status), _st(stream)),
           "smx_index_score")
    return page_scores


def index_score_topk(shape, qidx_bf16, idx_pool, page_table, ctx_len, page_scores=None,
                     topk_pages=None, topk_count=None, dev_status=None, stream=None):
    dev = _dev(idx_pool)
    if page_scores is None:
        page_scores = torch.empty((shape.B, shape.max_pages_per_row), dtype=torch.float32, device=dev)
    if topk_pages is None:
        topk_pages = torch.empty((shape.B, shape.topk), dtype=torch.int32, device=dev)
    if topk_count is None:
        topk_count = torch.empty((shape.B,), dtype=torch.int32, device=dev)
    _need("smx_index_score_topk", **_index_bufs(shape, qidx_bf16, idx_pool, page_table, ctx_len, page_scores,
                                                dev_status),
          topk_pages=(topk_pages, shape.B * shape.topk * 4), topk_count=(topk_count, shape.B * 4))
    cs = shape.c()
    _check(lib().smx_index_score_topk(ctypes.byref(cs), _p(qidx_bf16), _p(idx_pool), _p(page_table),
                                      _p(ctx_len), _p(page_scores), _p(topk_pages), _p(topk_count),
                                      _p(dev_status), _st(stream)), "smx_index_score_topk")
    return page_scores, topk_pages, topk_count


def sparse_attn_split(shape, q, k_pool, v_pool, page_table, ctx_len, topk_pages, topk_count,
                      part_o=None, part_m=None, part_l=None, dev_status=None, stream=None):
    dev = _dev(k_pool)
    rows = (shape.B, shape.num_splits, shape.Q, shape.Hq)
    if part_o is None:
        part_o = torch.empty(rows + (128,), dtype=torch.float32, device=dev)
    if part_m is None:
        part_m = torch.empty(rows, dtype=torch.float32, device=dev)
    if part_l is None:
        part_l = torch.empty(rows, dtype=torch.float32, device=dev)
    n_rows = shape.B * shape.num_splits * shape.Q * shape.Hq
    q_bytes = shape.B * shape.Q * shape.Hq * 128 * (2 if shape.kv_format == KV_E4M3_ROWSCALE else 1)
    _need("smx_sparse_attn_split", q=(q, q_bytes),
          **_step_bufs(shape, None, None, None, None, page_table, ctx_len, k_pool, v_pool, dev_status),
          topk_pages=(topk_pages, shape.B * shape.topk * 4), topk_count=(topk_count, shape.B * 4),
          part_o=(part_o, n_rows * 128 * 4), part_m=(part_m, n_rows * 4), part_l=(part_l, n_rows * 4))
    cs = shape.c()
    _check(lib().smx_sparse_attn_split(ctypes.byref(cs), _p(q), _p(k_pool), _p(v_pool), _p(page_table),
                                       _p(ctx_len), _p(topk_pages), _p(topk_count), _p(part_o),
                                       _p(part_m), _p(part_l), _p(dev_status), _st(stream)),
           "smx_sparse_attn_split")
    return part_o, part_m, part_l


def sparse_attn_merge(shape, part_o, part_m, part_l, out=None, stream=None):
    if out is None:
        out = torch.empty((shape.B, shape.Q, shape.Hq, 128), dtype=torch.float32, device=part_o.device)
    n_rows = shape.B * shape.num_splits * shape.Q * shape.Hq
    _need("smx_sparse_attn_merge", part_o=(part_o, n_rows * 128 * 4), part_m=(part_m, n_rows * 4),
          part_l=(part_l, n_rows * 4), out=(out, shape.B * shape.Q * shape.Hq * 128 * 4))
    cs = shape.c()
    _check(lib().smx_sparse_attn_merge(ctypes.byref(cs), _p(part_o), _p(part_m), _p(part_l), _p(out),
                                       _st(stream)), "smx_sparse_attn_merge")
    return out


def set_wait_limit_ns(ns: int) -> int:
    """Bound of the fused steps' waits for other CTAs (0 = the default); returns the previous one."""
    return int(lib().smx_set_wait_limit_ns(int(ns)))


def alloc_workspace(shape, device=None) -> torch.Tensor:
    """Zeroed workspace for decode_step (its per-row counters must start at zero)."""
    return torch.zeros(max(256, workspace_bytes(shape)), dtype=torch.uint8, device=device or "cuda")


def _full_step_bufs(shape, q_f32, q_bf16, qidx_bf16, k_new, v_new, kidx_new, page_table, ctx_len, k_pool, v_pool,
                    idx_pool, topk_pages, topk_count, out, dev_status):
    B, Q = shape.B, shape.Q
    return dict(**_step_bufs(shape, q_f32, q_bf16, k_new, v_new, page_table, ctx_len, k_pool, v_pool, dev_status),
                qidx_bf16=(qidx_bf16, B * Q * 128 * 2), kidx_new=(kidx_new, B * Q * 128 * 4),
                idx_pool=(idx_pool, shape.n_pool_pages * shape.idx_page_bytes),
                topk_pages=(topk_pages, B * shape.topk * 4), topk_count=(topk_count, B * 4),
                out=(out, B * Q * shape.Hq * 128 * 4))


def decode_step(shape, *, q_f32=None, q_bf16=None, qidx_bf16, k_new, v_new, kidx_new, page_table,
                ctx_len, k_pool, v_pool, idx_pool, topk_pages=None, topk_count=None, out=None,
                workspace=None, dev_status=None, stream=None):
    dev = _dev(k_pool)
    if topk_pages is None:
        topk_pages = torch.empty((shape.B, shape.topk), dtype=torch.int32, device=dev)
    if topk_count is None:
        topk_count = torch.empty((shape.B,), dtype=torch.int32, device=dev)
    if out is None:
        out = torch.empty((shape.B, shape.Q, shape.Hq, 128), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(shape, dev)
    _need("smx_decode_step", **_full_step_bufs(shape, q_f32, q_bf16, qidx_bf16, k_new, v_new, kidx_new, page_table,
                                               ctx_len, k_pool, v_pool, idx_pool, topk_pages, topk_count, out,
                                               dev_status))
    cs = shape.c()
    _check(lib().smx_decode_step(ctypes.byref(cs), _p(q_f32), _p(q_bf16), _p(qidx_bf16), _p(k_new),
                                 _p(v_new), _p(kidx_new), _p(page_table), _p(ctx_len), _p(k_pool),
                                 _p(v_pool), _p(idx_pool), _p(topk_pages), _p(topk_count), _p(out),
                                 _p(workspace), workspace.numel(), _p(dev_status), _st(stream)),
           "smx_decode_step")
    return out, topk_pages, topk_count


def decode_step_reuse(shape, *, q_f32=None, q_bf16=None, k_new, v_new, page_table, ctx_len, k_pool, v_pool,
                      topk_pages, topk_count, out=None, workspace=None, dev_status=None, stream=None):
    """The step of a layer reusing an earlier layer's selection (topk_pages [B][topk] and
    topk_count [B] int32, inputs): K/V insert, q packing, split and merge."""
    dev = _dev(k_pool)
    if out is None:
        out = torch.empty((shape.B, shape.Q, shape.Hq, 128), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(shape, dev)
    _need("smx_decode_step_reuse", **_step_bufs(shape, q_f32, q_bf16, k_new, v_new, page_table, ctx_len, k_pool,
                                                v_pool, dev_status),
          topk_pages=(topk_pages, shape.B * shape.topk * 4), topk_count=(topk_count, shape.B * 4),
          out=(out, shape.B * shape.Q * shape.Hq * 128 * 4))
    cs = shape.c()
    _check(lib().smx_decode_step_reuse(ctypes.byref(cs), _p(q_f32), _p(q_bf16), _p(k_new), _p(v_new),
                                       _p(page_table), _p(ctx_len), _p(k_pool), _p(v_pool), _p(topk_pages),
                                       _p(topk_count), _p(out), _p(workspace), workspace.numel(), _p(dev_status),
                                       _st(stream)),
           "smx_decode_step_reuse")
    return out


NOALLOC_SCRATCH_BYTES = 16 << 20


def decode_step_noalloc(shape, *, q_f32=None, q_bf16=None, qidx_bf16, k_new, v_new, kidx_new, page_table,
                        ctx_len, k_pool, v_pool, idx_pool, topk_pages, topk_count, out, dev_status=None,
                        stream=None):
    """smx_decode_step_noalloc: the whole step in the library's static device scratch. Every
    output buffer is the caller's; the call allocates nothing (first call per device: before any
    stream capture). Calls that overlap on one device race on the shared scratch."""
    if workspace_bytes(shape) > NOALLOC_SCRATCH_BYTES:
        _check(SMX_ERR_WORKSPACE, "smx_decode_step_noalloc")
    _need("smx_decode_step_noalloc", **_full_step_bufs(shape, q_f32, q_bf16, qidx_bf16, k_new, v_new, kidx_new,
                                                       page_table, ctx_len, k_pool, v_pool, idx_pool, topk_pages,
                                                       topk_count, out, dev_status))
    cs = shape.c()
    _check(lib().smx_decode_step_noalloc(ctypes.byref(cs), _p(q_f32), _p(q_bf16), _p(qidx_bf16), _p(k_new),
                                         _p(v_new), _p(kidx_new), _p(page_table), _p(ctx_len), _p(k_pool),
                                         _p(v_pool), _p(idx_pool), _p(topk_pages), _p(topk_count), _p(out),
                                         _p(dev_status), _st(stream)),
           "smx_decode_step_noalloc")
    return out, topk_pages, topk_count
