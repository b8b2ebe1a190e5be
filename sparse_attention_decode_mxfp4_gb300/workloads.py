"""Seeded synthetic workloads for the sparse MXFP4 decode step.

This module only draws inputs: fp32 rows from N(0, 1), the structure of each workload
(ragged context lengths, rows scaled x50, index-K pages shifted by +3, a random physical
page permutation) and the poison bytes written into slots a step must never read. It holds
none of the method's arithmetic (no quantisation, scoring, selection or attention), so both
the CUDA path and the CPU oracle can take their inputs from it.

Recipe (per workload, numpy PCG64 ``default_rng(seed)``; draws in this order):
  1. sweep cases only: per-row context fractions U(0.5, 1.0); ctx = max(Q, floor(f * max_ctx));
  2. for each row b: index-K [T][128], K [T][Hkv][128], V [T][Hkv][128] as standard normal
     float32 (T = the longest context of the workload, tokens beyond a row's context unused);
  3. q [B][Q][Hq][128], then q_idx [B][Q][128], standard normal float32;
  4. rows scaled x50 (FP8-KV workload): three independent masks (index-K, K, V), each row
     chosen with probability 0.01;
  5. index-K page shift (long-context workload): per row round(0.05 * n_pages) distinct pages
     get +3.0 on every element of index-K;
  6. the page table: a random permutation of the physical page ids, row-major;
  7. poison bytes for tail slots (random nibble bytes; scales 0xFF / NaN; NVFP4 scales 0x7F /
     NaN).
q_idx and, for the FP8-KV workload, q are rounded to bf16 (round to nearest even).
NVFP4 variants (K/V and index pages NVFP4) draw the same inputs; their per-tensor decode scales
are fixed calibration inputs of the workload (NV_SCALE: with N(0, 1) rows a 16-element block's
largest |x| of about 1 to 4 maps to E4M3 block scales of about 10 to 40, rows scaled x50 to
about 500 before saturation at 448), not something this module computes.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

PAGE = 128
D = 128
KV_MXFP4 = 0
KV_E4M3_ROWSCALE = 1
KV_NVFP4 = 2
MXFP4_PAGE_BYTES = 8704
E4M3RS_PAGE_BYTES = 16896
NVFP4_PAGE_BYTES = 9216
NV_SCALE = 0.0173   # per-tensor NVFP4 decode scale of the synthetic K, V and index pools


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Q: int
    Hq: int
    Hkv: int
    max_ctx: int
    topk: int
    num_splits: int
    kv_format: int = KV_MXFP4
    seed: int = 0
    ctx_lens: tuple = ()            # per row; empty -> drawn (ragged) or max_ctx
    ragged: bool = False            # draw per-row lengths from U(0.5, 1.0) x max_ctx
    big_row_frac: float = 0.0
    big_row_factor: float = 50.0
    shift_page_frac: float = 0.0
    shift_value: float = 3.0
    pages_per_block: int = 1        # pages per selected block of the sparse table
    idx_format: int = KV_MXFP4      # index pool: MXFP4 or NVFP4
    nv_scale_k: float = NV_SCALE    # NVFP4 per-tensor decode scales (used by NVFP4 pools only)
    nv_scale_v: float = NV_SCALE
    nv_scale_idx: float = NV_SCALE

    @property
    def max_pages(self) -> int:
        return (self.max_ctx + PAGE - 1) // PAGE

    @property
    def n_pool_pages(self) -> int:
        return self.B * self.max_pages

    @property
    def kv_page_bytes(self) -> int:
        return {KV_E4M3_ROWSCALE: E4M3RS_PAGE_BYTES, KV_NVFP4: NVFP4_PAGE_BYTES}.get(self.kv_format, MXFP4_PAGE_BYTES)

    @property
    def idx_page_bytes(self) -> int:
        return NVFP4_PAGE_BYTES if self.idx_format == KV_NVFP4 else MXFP4_PAGE_BYTES

    def describe(self) -> dict:
        names = {KV_MXFP4: "mxfp4", KV_E4M3_ROWSCALE: "e4m3_rowscale", KV_NVFP4: "nvfp4"}
        d = dict(workload=self.name, B=self.B, Q=self.Q, Hq=self.Hq, Hkv=self.Hkv,
                 max_ctx=self.max_ctx, topk=self.topk, kv=names[self.kv_format], seed=self.seed)
        if self.idx_format != KV_MXFP4:
            d["index"] = names[self.idx_format]
        return d


def config(n: int) -> Workload:
    """The fixed workloads (1 = tiny, 2 = fixed 7-draft verify, 3 = FP8 KV, 4 = long) and, as 5, the
    largest case of the sweep (B 4, Q 8, 16 heads, contexts up to 262144 tokens, top-k 128)."""
    if n == 5:
        return sweep_cases()[-1]
    if n == 1:
        return Workload("tiny_b1_q1_h8_ctx1024_k4", B=1, Q=1, Hq=8, Hkv=1, max_ctx=1024,
                        topk=4, num_splits=2, seed=1001)
    if n == 2:
        return Workload("verify_b4_q8_h16_ctx16384_k16", B=4, Q=8, Hq=16, Hkv=1,
                        max_ctx=16384, topk=16, num_splits=4, seed=1002)
    if n == 3:
        return Workload("fp8kv_b4_q8_h16_ctx65536_k32", B=4, Q=8, Hq=16, Hkv=1,
                        max_ctx=65536, topk=32, num_splits=8, kv_format=KV_E4M3_ROWSCALE,
                        seed=1003, big_row_frac=0.01)
    if n == 4:
        # 1919 full pages + 75 tokens; the 53 tail slots of the last page are poisoned.
        return Workload("long_b2_q8_h16_ctx245707_k64", B=2, Q=8, Hq=16, Hkv=1,
                        max_ctx=245760, topk=64, num_splits=16, seed=1004,
                        ctx_lens=(245707, 245707), shift_page_frac=0.05)
    raise ValueError(f"no workload {n}")


SWEEP_B = (1, 2, 4)
SWEEP_Q = (1, 4, 8)
SWEEP_CTX = (4096, 32768, 131072, 262144)
SWEEP_K = (8, 32, 128)
SWEEP_HQ = (8, 16)


def nvfp4_variant(w: Workload) -> Workload:
    """The same workload with NVFP4 K/V and index pages (E2M1 + E4M3 scale per 16 + the
    per-tensor scales NV_SCALE)."""
    return replace(w, name="nvfp4_" + w.name, kv_format=KV_NVFP4, idx_format=KV_NVFP4)


def sweep_cases() -> list:
    """216 cases: B x Q x max ctx x k x Hq with ragged per-row lengths. S = k + 3 (more
    partitions than selected pages: empty partitions) whenever k = 8 and Hq = 16, which
    happens for every (B, Q, ctx); otherwise S = min(k, 8)."""
    cases = []
    i = 0
    for B in SWEEP_B:
        for Q in SWEEP_Q:
            for ctx in SWEEP_CTX:
                for k in SWEEP_K:
                    for Hq in SWEEP_HQ:
                        S = k + 3 if (k == 8 and Hq == 16) else min(k, 8)
                        cases.append(Workload(f"sweep{i:03d}_b{B}_q{Q}_ctx{ctx}_k{k}_h{Hq}",
                                              B=B, Q=Q, Hq=Hq, Hkv=1, max_ctx=ctx, topk=k,
                                              num_splits=S, seed=5000 + i, ragged=True))
                        i += 1
    return cases


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the 16-bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[np.isnan(x)] = 0x7FC0
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def context_lengths(w: Workload, rng: np.random.Generator) -> np.ndarray:
    if w.ctx_lens:
        return np.asarray(w.ctx_lens, np.int32)
    if w.ragged:
        f = rng.uniform(0.5, 1.0, size=w.B)
        return np.maximum(w.Q, np.floor(f * w.max_ctx).astype(np.int64)).astype(np.int32)
    return np.full(w.B, w.max_ctx, np.int32)


def generate(w: Workload) -> dict:
    """All fp32/bf16 inputs of one workload (see the module docstring for the recipe)."""
    rng = np.random.default_rng(w.seed)
    ctx = context_lengths(w, rng)
    T = int(ctx.max())
    B, Q, Hq, Hkv = w.B, w.Q, w.Hq, w.Hkv
    kidx = np.empty((B, T, D), np.float32)
    k = np.empty((B, T, Hkv, D), np.float32)
    v = np.empty((B, T, Hkv, D), np.float32)
    for b in range(B):
        kidx[b] = rng.standard_normal((T, D), dtype=np.float32)
        k[b] = rng.standard_normal((T, Hkv, D), dtype=np.float32)
        v[b] = rng.standard_normal((T, Hkv, D), dtype=np.float32)
    q = rng.standard_normal((B, Q, Hq, D), dtype=np.float32)
    qidx = rng.standard_normal((B, Q, D), dtype=np.float32)
    if w.big_row_frac > 0:
        for arr in (kidx, k, v):
            m = rng.random((B, T)) < w.big_row_frac
            arr[m] *= np.float32(w.big_row_factor)
    shifted = []
    if w.shift_page_frac > 0:
        for b in range(B):
            n_pages = (int(ctx[b]) + PAGE - 1) // PAGE
            n_shift = int(round(w.shift_page_frac * n_pages))
            pages = np.sort(rng.choice(n_pages, size=n_shift, replace=False))
            for p in pages:
                kidx[b, p * PAGE:(p + 1) * PAGE] += np.float32(w.shift_value)
            shifted.append(pages)
    perm = rng.permutation(w.n_pool_pages).astype(np.int32)
    page_table = perm[: B * w.max_pages].reshape(B, w.max_pages).copy()
    poison_seed = int(rng.integers(0, 2**31 - 1))

    rows = np.arange(Q)[None, :] + (ctx[:, None] - Q)          # [B][Q] new positions
    bidx = np.arange(B)[:, None]
    return dict(
        ctx_len=ctx, page_table=page_table, T=T,
        kidx=kidx, k=k, v=v,
        q=q, q_bf16=f32_to_bf16_bits(q), qidx_bf16=f32_to_bf16_bits(qidx),
        k_new=np.ascontiguousarray(k[bidx, rows]),             # [B][Q][Hkv][128]
        v_new=np.ascontiguousarray(v[bidx, rows]),
        kidx_new=np.ascontiguousarray(kidx[bidx, rows]),       # [B][Q][128]
        n_hist=(ctx - Q).astype(np.int32),
        shifted_pages=shifted, poison_seed=poison_seed,
    )


# ---- poison: bytes written into slots the step must never read ---------------------------
def poison_slots(w: Workload, data: dict, include_new: bool = True):
    """(physical page, first slot) pairs to poison: every slot at or beyond the row's context
    (tail of the last page and whole unused pages) and, with include_new, the slots of the Q
    new tokens (a step must write them before reading)."""
    out = []
    ctx, pt = data["ctx_len"], data["page_table"]
    for b in range(w.B):
        c = int(ctx[b])
        first = c - w.Q if include_new else c
        for p in range(w.max_pages):
            lo = max(0, first - p * PAGE)
            if lo < PAGE:
                out.append((int(pt[b, p]), lo))
    return out


def poison_pools(w: Workload, data: dict, k_pool: np.ndarray, v_pool: np.ndarray,
                 idx_pool: np.ndarray, include_new: bool = True) -> None:
    """Fill the poison slots in place (NumPy uint8 pools, [n_pool][Hkv][page] for K/V and
    [n_pool][8704] for the index). MXFP4 slots get random nibble bytes and scale byte 0xFF
    (NaN); e4m3 row-scale slots get codes 0x7F (NaN) and a NaN fp32 scale."""
    rng = np.random.default_rng(data["poison_seed"])
    nan_f32 = np.frombuffer(np.array([np.nan], np.float32).tobytes(), np.uint8)
    idx = idx_pool.reshape(w.n_pool_pages, w.idx_page_bytes)
    kk = k_pool.reshape(w.n_pool_pages, w.Hkv, w.kv_page_bytes)
    vv = v_pool.reshape(w.n_pool_pages, w.Hkv, w.kv_page_bytes)
    for phys, lo in poison_slots(w, data, include_new):
        n = PAGE - lo
        idx[phys, lo * 64:PAGE * 64] = rng.integers(0, 256, n * 64, dtype=np.uint8)
        if w.idx_format == KV_NVFP4:
            idx[phys, 8192 + lo * 8:8192 + PAGE * 8] = 0x7F
        else:
            idx[phys, 8192 + lo * 4:8192 + PAGE * 4] = 0xFF
        for pool in (kk, vv):
            if w.kv_format == KV_E4M3_ROWSCALE:
                pool[phys, :, lo * 128:PAGE * 128] = 0x7F
                pool[phys, :, 16384 + lo * 4:16384 + PAGE * 4] = np.tile(nan_f32, n)
            else:
                pool[phys, :, lo * 64:PAGE * 64] = rng.integers(0, 256, (w.Hkv, n * 64),
                                                                dtype=np.uint8)
                if w.kv_format == KV_NVFP4:
                    pool[phys, :, 8192 + lo * 8:8192 + PAGE * 8] = 0x7F
                else:
                    pool[phys, :, 8192 + lo * 4:8192 + PAGE * 4] = 0xFF


def empty_pools(w: Workload):
    return (np.zeros((w.n_pool_pages, w.Hkv, w.kv_page_bytes), np.uint8),
            np.zeros((w.n_pool_pages, w.Hkv, w.kv_page_bytes), np.uint8),
            np.zeros((w.n_pool_pages, w.idx_page_bytes), np.uint8))


def shrink(w: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (used for small parity cases)."""
    return replace(w, **kw)
