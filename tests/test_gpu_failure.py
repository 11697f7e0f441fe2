"""Failure detection on the GPU without a fault: a kernel whose bounded wait
runs out (a barrier phase nothing completes) reports DEVICE_TIMEOUT through
the plan's error word, drains, frees its tensor memory and exits; the CUDA
context and the plan stay usable."""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_plan_recovers():
    from realtime_transformer_gb300.ffn import FFNPlan
    from realtime_transformer_gb300._native import FrtError
    plan = FFNPlan(256, 1024, "geglu_tanh", 64, 1)
    with pytest.raises(FrtError) as err:
        plan.debug_stall()
    assert err.value.name == "FRT_ERR_DEVICE_TIMEOUT"
    plan.device_status()  # the flag was cleared by the report
    # the same kernels still compute exactly afterwards
    rng = np.random.default_rng(3)
    e = rng.integers(5, 9, (2, 40, 64))
    m = rng.integers(0, 8, (2, 40, 64))
    sgn = rng.integers(0, 2, (2, 40, 64))
    codes = ((sgn << 7) | (e << 3) | m).astype(np.uint8)
    A = codes[0]
    B = np.concatenate([codes[1]] * 4 + [codes[1][:8]], axis=0)[:128]
    dev = torch.device("cuda")
    C = plan.gemm(torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev), alpha=1.0, path=1, splits=1)
    torch.cuda.synchronize()
    plan.device_status()
    assert np.array_equal(C.cpu().numpy(), oracle.gemm_e4m3(A, B))
    plan.close()


@pytest.mark.parametrize("M", [8, 300], ids=["weight_streaming", "tiled"])
def test_nvfp4_bounded_wait_gives_up_and_plan_recovers(M):
    """The NVFP4 GEMM (with its scale warps and per-stage scale barriers)
    gives up the same way, and the plan then computes the same bits."""
    from realtime_transformer_gb300.nvfp4 import FP4Plan
    from realtime_transformer_gb300._native import FrtError
    wl = synthetic.WORKLOADS["tiny"].with_(M=M, d=512, ff=1024)
    lw = synthetic.layer_weights(wl, 0, device=torch.device("cuda"))
    r, h = synthetic.inputs(wl, device=torch.device("cuda"))
    plan = FP4Plan(wl.d, wl.ff, wl.act, wl.M, 1)
    try:
        plan.load_weights(0, lw["w_norm"], lw["w_gate"], lw["w_up"], lw["w_down"])
        plan.set_scales([[0.002, 0.01, 0.01, 0.004]])
        before = plan.forward(r, h)
        torch.cuda.synchronize()
        with pytest.raises(FrtError) as err:
            plan.debug_stall(M)
        assert err.value.name == "FRT_ERR_DEVICE_TIMEOUT"
        plan.device_status()  # the flag was cleared by the report
        after = plan.forward(r, h)
        torch.cuda.synchronize()
        plan.device_status()
        assert torch.equal(before, after)
    finally:
        plan.close()
