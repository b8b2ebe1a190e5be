"""The fused step's bounded waits for other CTAs give up cleanly ([vLLM-60528] "Merge Danger": a
persistent kernel that waits for CTAs which never arrive holds a shared GPU). With the test-only
bound set to 1 ns, a row's attention units stop waiting for its page scores and the merges stop
waiting for their partitions: the call must come back within a second with SMX_DEV_TIMEOUT in the
device status and a finite output, and the next step on the same workspace, with the default
bound, must match the oracle (the counters were left at zero)."""
import time

import numpy as np
import pytest
import torch

from sparse_attention_decode_mxfp4_gb300 import ops
from sparse_attention_decode_mxfp4_gb300 import workloads as wl
from tests import gpu_common as C
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from sparse_attention_decode_mxfp4_gb300 import build
    build.build()
    ops.lib()


@pytest.mark.parametrize("n", [2, 4])
def test_wait_gives_up_then_next_step_is_sound(n):
    w = wl.config(n)
    data = wl.generate(w)
    pools = H.oracle_pools(w, data)
    shape = ops.Shape.of(w)
    ws = ops.alloc_workspace(shape)
    default = ops.set_wait_limit_ns(0)
    ops.set_wait_limit_ns(1)
    seen = 0
    try:
        for _ in range(5):
            g = C.gpu_inputs(w, data, pools)
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            t0 = time.perf_counter()
            out, _, _ = ops.decode_step(shape, q_f32=g["q_f32"], qidx_bf16=g["qidx_bf16"], k_new=g["k_new"],
                                        v_new=g["v_new"], kidx_new=g["kidx_new"], page_table=g["page_table"],
                                        ctx_len=g["ctx_len"], k_pool=g["k_pool"], v_pool=g["v_pool"],
                                        idx_pool=g["idx_pool"], workspace=ws, dev_status=status)
            torch.cuda.synchronize()
            assert time.perf_counter() - t0 < 1.0
            assert bool(torch.isfinite(out).all())
            st = int(status.item())
            assert st & ~ops.DEV_TIMEOUT == 0, st
            seen |= st
    finally:
        ops.set_wait_limit_ns(0)
    assert seen & ops.DEV_TIMEOUT, "no wait ran out with a 1 ns bound"
    assert ops.set_wait_limit_ns(0) == default
    C.full_step_parity(w, data=data, workspace=ws)
