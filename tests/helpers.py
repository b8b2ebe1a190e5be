"""Test helpers: pools built by the oracle from the seeded workloads, and dense references
built from library routines (torch float64 softmax / scaled_dot_product_attention)."""
import numpy as np
import torch

import oracle
from sparse_attention_decode_mxfp4_gb300 import workloads as wl


def oracle_pools(w, data, include_new=True):
    """History rows [0, ctx-Q) quantised by the oracle; new-token slots (include_new), tails
    and unused pages poisoned."""
    k_pool, v_pool, idx_pool = wl.empty_pools(w)
    oracle.kv_fill(oracle.shape_of(w), data["k"], data["v"], data["kidx"], data["page_table"],
                   data["n_hist"], k_pool, v_pool, idx_pool)
    wl.poison_pools(w, data, k_pool, v_pool, idx_pool, include_new=include_new)
    return k_pool, v_pool, idx_pool


def oracle_step(w, data, pools, num_splits=None, want_partials=False):
    """The oracle's whole step on copies of the pools; returns (result dict, new pools)."""
    k_pool, v_pool, idx_pool = (p.copy() for p in pools)
    sh = oracle.shape_of(w, num_splits)
    res = oracle.decode_step(sh, q_f32=data["q"], q_bf16=data["q_bf16"],
                             qidx_bf16=data["qidx_bf16"], k_new=data["k_new"],
                             v_new=data["v_new"], kidx_new=data["kidx_new"],
                             page_table=data["page_table"], ctx_len=data["ctx_len"],
                             k_pool=k_pool, v_pool=v_pool, idx_pool=idx_pool,
                             want_partials=want_partials)
    return res, (k_pool, v_pool, idx_pool)


def load_kv_row(w, pool, phys, kvh, slot, pool_is_k=True):
    page = pool.reshape(w.n_pool_pages, w.Hkv, w.kv_page_bytes)[phys, kvh]
    if w.kv_format == wl.KV_E4M3_ROWSCALE:
        return oracle.e4m3rs_load_row(page, slot)
    if w.kv_format == wl.KV_NVFP4:
        g = w.nv_scale_k if pool_is_k else w.nv_scale_v
        return oracle.nvfp4_load_row(page, slot, g)
    return oracle.mxfp4_load_row(page, slot)


def q_values(w, data, res):
    """The q the attention uses, as float64: decoded e4m3 bytes, or bf16 for FP8-KV."""
    if w.kv_format == wl.KV_E4M3_ROWSCALE:
        return wl.bf16_bits_to_f32(data["q_bf16"]).astype(np.float64)
    return torch.from_numpy(res["q_e4m3"]).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def dense_selected_attention(w, data, q, k_pool, v_pool, topk_pages, topk_count):
    """Textbook softmax attention (torch float64) over exactly the selected tokens of each
    query: j in a selected page, j < ctx_len, j <= pos_t."""
    out = np.zeros((w.B, w.Q, w.Hq, 128))
    G = w.Hq // w.Hkv
    for b in range(w.B):
        ctx = int(data["ctx_len"][b])
        pages = [int(p) for p in topk_pages[b, :topk_count[b]]]
        for kvh in range(w.Hkv):
            toks, K, V = [], [], []
            for p in pages:
                phys = int(data["page_table"][b, p])
                for slot in range(128):
                    j = p * 128 + slot
                    if j < ctx:
                        toks.append(j)
                        K.append(load_kv_row(w, k_pool, phys, kvh, slot))
                        V.append(load_kv_row(w, v_pool, phys, kvh, slot, pool_is_k=False))
            if not toks:
                continue
            toks = torch.tensor(toks)
            K = torch.tensor(np.array(K))
            V = torch.tensor(np.array(V))
            for t in range(w.Q):
                pos = ctx - w.Q + t
                keep = toks <= pos
                if not bool(keep.any()):
                    continue
                for hh in range(G):
                    h = kvh * G + hh
                    qv = torch.tensor(q[b, t, h])
                    z = (K[keep] @ qv) / np.sqrt(128.0)
                    p = torch.softmax(z, dim=0)
                    out[b, t, h] = (p @ V[keep]).numpy()
    return out
