"""Host-side checks of the C ABI (no GPU needed): the library builds for sm_103a, loads, exports
every symbol include/smx.h declares, and refuses bad shapes and pointers before any launch."""
import ctypes
import re
import os
import subprocess

import pytest

from sparse_attention_decode_mxfp4_gb300 import build as smx_build
from sparse_attention_decode_mxfp4_gb300 import ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    smx_build.build()
    return ops.lib()


def declared_symbols():
    hdr = open(os.path.join(ROOT, "include", "smx.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"\b(smx_\w+)\s*\(", hdr)))


def test_exports_every_declared_symbol(L):
    decl = declared_symbols()
    assert set(decl) == set(ops.SYMBOLS)
    nm = subprocess.run(["nm", "-D", "--defined-only", ops.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (smx_\w+)", nm))
    for name in decl:
        assert name in exported, name
        assert getattr(L, name) is not None


def good_shape(**kw):
    s = ops.Shape(B=2, Q=8, Hq=16, Hkv=1, max_pages_per_row=16, n_pool_pages=32, topk=4, num_splits=2)
    for k, v in kw.items():
        setattr(s, k, v)
    return s


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), -1), (dict(Q=0), -1), (dict(Hq=0), -1), (dict(Hkv=0), -1), (dict(Hq=12, Hkv=5), -1),
    (dict(topk=0), -1), (dict(num_splits=0), -1), (dict(n_pool_pages=0), -1),
    (dict(max_pages_per_row=0), -1),
    (dict(D=64), -2), (dict(Di=256), -2), (dict(page_tokens=64), -2), (dict(Q=17), -2),
    (dict(kv_format=7), -2), (dict(idx_format=1), -2), (dict(idx_format=3), -2),
    # NVFP4 pools need a finite positive per-tensor scale, and one page per selected block
    (dict(kv_format=2), -1), (dict(kv_format=2, nv_scale_k=0.5), -1),
    (dict(kv_format=2, nv_scale_k=0.5, nv_scale_v=float("nan")), -1),
    (dict(kv_format=2, nv_scale_k=0.5, nv_scale_v=float("inf")), -1), (dict(idx_format=2), -1),
    (dict(idx_format=2, nv_scale_idx=-1.0), -1),
    (dict(kv_format=2, nv_scale_k=0.5, nv_scale_v=0.5, pages_per_block=2), -2),
    (dict(topk=5000), -2), (dict(pages_per_block=3), -2),
    (dict(pages_per_block=4, topk=2000), -2),
])
def test_bad_shapes_are_refused(L, kw, code):
    s = good_shape(**kw)
    cs = s.c()
    fake = ctypes.c_void_p(1 << 20)     # never dereferenced: the check fails first
    assert L.smx_workspace_bytes(ctypes.byref(cs)) == 0
    rc = L.smx_index_score_topk(ctypes.byref(cs), fake, fake, fake, fake, fake, fake, fake, None, None)
    assert rc == code
    rc = L.smx_sparse_attn_merge(ctypes.byref(cs), fake, fake, fake, fake, None)
    assert rc == code
    rc = L.smx_decode_step_reuse(ctypes.byref(cs), *([fake] * 12), 1 << 30, None, None)
    assert rc == code


@pytest.mark.parametrize("kw,launches", [
    (dict(kv_format=2, nv_scale_k=0.5, nv_scale_v=0.25), 6),
    (dict(idx_format=2, nv_scale_idx=0.125), 6),
    (dict(kv_format=2, idx_format=2, nv_scale_k=0.5, nv_scale_v=0.25, nv_scale_idx=0.125), 6),
    (dict(kv_format=1, idx_format=2, nv_scale_idx=0.125), 5),
    (dict(), 1),
])
def test_nvfp4_shapes_are_taken(L, kw, launches):
    # a step with an NVFP4 pool runs the standalone kernels in sequence (no q packing with FP8-KV)
    cs = good_shape(**kw).c()
    assert L.smx_workspace_bytes(ctypes.byref(cs)) > 0
    assert L.smx_decode_step_launches(ctypes.byref(cs)) == launches
    assert L.smx_decode_step_tensor_cores(ctypes.byref(cs)) == (0 if launches > 1 else L.smx_decode_step_tensor_cores(ctypes.byref(cs)))


def test_null_and_misaligned_pointers_are_refused(L):
    cs = good_shape().c()
    a = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 4)
    for insert in (L.smx_kv_insert_mxfp4, L.smx_kv_insert):   # the call and its shorter alias
        assert insert(ctypes.byref(cs), None, a, a, a, a, a, a, a, None, None) == -1
        assert insert(ctypes.byref(cs), mis, a, a, a, a, a, a, a, None, None) == -1
    assert L.smx_pack_q_e4m3(a, a, 0, None) == -1
    assert L.smx_pack_q_e4m3(mis, a, 16, None) == -1
    ws = L.smx_workspace_bytes(ctypes.byref(cs))
    assert ws > 0 and ws % 256 == 0
    args = [a] * 14
    # workspace too small / missing
    assert L.smx_decode_step(ctypes.byref(cs), *args, a, ws - 256, None, None) == -4
    assert L.smx_decode_step(ctypes.byref(cs), *args, None, ws, None, None) == -4
    # MXFP4 K/V needs q_f32
    args2 = [None] + [a] * 13
    assert L.smx_decode_step(ctypes.byref(cs), *args2, a, ws, None, None) == -1


def test_reuse_step_refuses_null_misaligned_and_workspace(L):
    cs = good_shape().c()
    a = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 4)
    ws = L.smx_workspace_bytes(ctypes.byref(cs))
    # q_f32, q_bf16, k_new, v_new, page_table, ctx_len, k_pool, v_pool, topk_pages, topk_count, out
    ok = [a] * 11
    assert L.smx_decode_step_reuse(ctypes.byref(cs), *ok, a, ws - 256, None, None) == -4
    assert L.smx_decode_step_reuse(ctypes.byref(cs), *ok, None, ws, None, None) == -4
    for i in (0, 2, 3, 4, 5, 6, 7, 8, 9, 10):   # q_f32 (MXFP4 K/V) and every other required pointer
        args = list(ok)
        args[i] = None
        assert L.smx_decode_step_reuse(ctypes.byref(cs), *args, a, ws, None, None) == -1, i
    for i in (0, 2, 3, 6, 7):   # 16-byte aligned: q_f32, k_new, v_new, k_pool, v_pool
        args = list(ok)
        args[i] = mis
        assert L.smx_decode_step_reuse(ctypes.byref(cs), *args, a, ws, None, None) == -1, i
    # q_bf16 may be NULL with MXFP4 K/V (q_f32 is the one used)
    args = list(ok)
    args[1] = None
    assert L.smx_decode_step_reuse(ctypes.byref(cs), *args, a, ws - 256, None, None) == -4


def test_standalone_topk_and_split_refuse_blocks_of_pages(L):
    cs = good_shape(pages_per_block=2).c()
    fake = ctypes.c_void_p(1 << 20)
    assert L.smx_index_score_topk(ctypes.byref(cs), fake, fake, fake, fake, fake, fake, fake, None, None) == -2
    assert L.smx_sparse_attn_split(ctypes.byref(cs), *([fake] * 10), None, None) == -2
    assert L.smx_workspace_bytes(ctypes.byref(cs)) > 0   # the fused steps take it


def test_status_strings(L):
    for rc in (0, -1, -2, -3, -4, -99):
        assert L.smx_status_string(rc)
    assert L.smx_decode_step_launches(ctypes.byref(good_shape().c())) >= 1


def test_split_suggestion_refuses_bad_shapes(L):
    bad = good_shape(Hq=12, Hkv=5)   # Hq not a multiple of Hkv
    assert L.smx_suggest_num_splits(ctypes.byref(bad.c())) == 0
    assert L.smx_suggest_num_splits(None) == 0
    assert L.smx_decode_step_tensor_cores(ctypes.byref(bad.c())) < 0
