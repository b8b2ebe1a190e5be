"""Why the attention keeps each softmax weight as a bf16 high part plus a bf16 low part. The pages
hold the weights in bf16 for the PV product, but the oracle is fp64 and the output bound is
max|err| <= 2e-3 + 1e-2 |ref|. A model of the kernels' arithmetic on a seeded case shows the two
outcomes. The case has context == Q, so each query row sees 1 to 8 tokens and its mass sits on a
few of them. The model uses fp32 scores, weights 2^(z - m) with the exact running maximum, and
wide sums. bf16 weights alone miss the bound. The high-plus-low pair (about 16 significant bits)
meets it with room. Host only: the weights and the oracle's decoded K, V and q."""
import numpy as np
import torch

from sparse_attention_decode_mxfp4_gb300 import workloads as wl
from tests import helpers as H

LOG2E = 1.4426950408889634


def bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def worst_ratio(weights):
    """max err/tol over every output element, for a weight model weights(e) -> (numerator weights,
    denominator weights)."""
    w = wl.Workload("ctx_eq_q", B=8, Q=8, Hq=16, Hkv=1, max_ctx=8, ctx_lens=(8,) * 8, topk=2, num_splits=1,
                    seed=5151, ragged=False)
    data = wl.generate(w)
    res, (kp, vp, _) = H.oracle_step(w, data, H.oracle_pools(w, data))
    q = H.q_values(w, data, res)                                   # [B][Q][Hq][128]
    worst = 0.0
    for b in range(w.B):
        ctx = int(data["ctx_len"][b])
        phys = int(data["page_table"][b][0])
        K = np.array([H.load_kv_row(w, kp, phys, 0, j) for j in range(ctx)])
        V = np.array([H.load_kv_row(w, vp, phys, 0, j, pool_is_k=False) for j in range(ctx)])
        for t in range(w.Q):
            n = ctx - w.Q + t + 1                                   # tokens 0 .. pos_t
            z = (q[b, t] @ K[:n].T).astype(np.float32).astype(np.float64) * (LOG2E / np.sqrt(128.0))
            e = np.exp2(z - z.max(axis=1, keepdims=True))           # [Hq][n], the largest is exactly 1
            num, den = weights(e)
            out = (num @ V[:n]) / den.sum(axis=1, keepdims=True)
            ref = res["out"][b, t]
            worst = max(worst, float(np.max(np.abs(out - ref) / (2e-3 + 1e-2 * np.abs(ref)))))
    return worst


def test_bf16_weights_alone_miss_the_bound():
    # tensor-core form (the sum l through the same bf16 weights) and mma.sync form (l in fp32)
    assert max(worst_ratio(lambda e: (bf16(e), bf16(e))), worst_ratio(lambda e: (bf16(e), e))) > 1.0


def test_high_plus_low_weights_meet_the_bound():
    def hi_lo(e):
        hi = bf16(e)
        p = hi + bf16(e - hi)
        return p, p
    assert worst_ratio(hi_lo) < 0.5
