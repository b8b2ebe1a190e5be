"""The fused step's packed q, byte for byte against the oracle's q packing.

On the tensor-core path the scanning CTAs pack every q row of their row (e4m3 by the q packing
rule: NaN -> 0x7F, clamp to +-448, round to nearest even, the input's sign) into one 16 KB tile
image per attention unit, in the operand layout the QK MMA reads (128 rows of 128 bytes, 16-byte
chunks swizzled within 8-row atoms). The images are the workspace's last B x Hkv x ceil(M / 128)
x 16384 bytes. This test reads them after a step and compares every written row with
orc_pack_q_e4m3 of the same q row, bit for bit, including the special values the rule names.
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_decode_mxfp4_gb300 import ops
from sparse_attention_decode_mxfp4_gb300 import workloads as wl
from tests import gpu_common as C
from tests import helpers as H

pytestmark = pytest.mark.gpu

IMG = 128 * 128


def _chunk_offset(i, c):
    return (i >> 3) * 1024 + (i & 7) * 128 + (((c ^ i) & 7) << 4)


def _plant_specials(q, rng):
    """Overwrite a few q entries with the values the packing rule singles out."""
    specials = np.array([np.nan, np.inf, -np.inf, 448.0, -448.0, 449.0, 464.0, 1e30, -1e30, 0.0, -0.0,
                         2.0 ** -9, -(2.0 ** -9), 2.0 ** -10, 2.0 ** -7 * 1.0625, 0.1015625, 240.0, 232.0,
                         1.5e-45], dtype=np.float32)
    flat = q.reshape(-1)
    idx = rng.choice(flat.size, size=4 * specials.size, replace=False)
    flat[idx] = np.tile(specials, 4)
    return q


CASES = [
    dict(name="img_tc", B=8, Q=8, Hq=16, Hkv=1, max_ctx=3000, topk=12, num_splits=12, seed=77, ragged=True),
    dict(name="img_gqa", B=4, Q=8, Hq=32, Hkv=2, max_ctx=3000, topk=8, num_splits=12, seed=78, ragged=True),
    dict(name="img_partial", B=3, Q=5, Hq=16, Hkv=1, max_ctx=3000, topk=8, num_splits=12, seed=79, ragged=True),
    dict(name="img_two_groups", B=20, Q=16, Hq=16, Hkv=1, max_ctx=6000, topk=32, num_splits=4, seed=80, ragged=True),
]


@pytest.mark.parametrize("kw", CASES, ids=[c["name"] for c in CASES])
def test_fused_step_packed_q_is_bit_exact(kw):
    w = wl.Workload(**kw)
    shape = ops.Shape.of(w)
    if not ops.decode_step_tensor_cores(shape):
        pytest.skip("this shape runs the mma.sync attention on this device")
    data = wl.generate(w)
    data["q"] = _plant_specials(np.array(data["q"], dtype=np.float32, copy=True), np.random.default_rng(kw["seed"]))
    pools = H.oracle_pools(w, data)
    G, M = w.Hq // w.Hkv, (w.Hq // w.Hkv) * w.Q
    n_rg = (M + 127) // 128
    img_bytes = w.B * w.Hkv * n_rg * IMG
    start = ops.workspace_bytes(shape) - img_bytes
    assert start > 0
    ws = ops.alloc_workspace(shape, torch.device("cuda"))   # zeroed: the counters start at zero
    ws[start:start + img_bytes].fill_(0xA5)                  # image rows the step does not write keep this
    C.gpu_step(w, data, pools, workspace=ws)
    imgs = ws.cpu().numpy().view(np.uint8)[start:start + img_bytes]
    want = oracle.pack_q_e4m3(data["q"]).reshape(w.B, w.Q, w.Hq, 128)
    bad = 0
    for b in range(w.B):
        for kvh in range(w.Hkv):
            for rg in range(n_rg):
                img = imgs[((b * w.Hkv + kvh) * n_rg + rg) * IMG:][:IMG]
                for i in range(min(128, M - rg * 128)):
                    m = rg * 128 + i
                    got = np.concatenate([img[_chunk_offset(i, c):][:16] for c in range(8)])
                    ref = want[b, m // G, kvh * G + m % G]
                    bad += int(not np.array_equal(got, ref))
    assert bad == 0, f"{bad} packed q rows differ from the oracle's"
