"""Failure detection on the GPU without a fault: every grouped-GEMM pipeline
wait is bounded. The self-test entry point starves one CTA of operands (a
flag that nothing sets), the wait gives up, the device error word says so,
and the context keeps working for the next call."""

import numpy as np
import pytest
import torch

from workloads import generate, get_config

pytestmark = pytest.mark.gpu


def test_starved_pipeline_wait_times_out_and_context_survives():
    from demand_side_expert_gb300 import RecalibratedExpertBackward, lrm

    dev = torch.device("cuda:0")
    ws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    lrm.lrm_selftest_wait_timeout(ws, ws.numel())
    code = lrm.lrm_get_device_error(ws, ws.numel())
    assert code & lrm.LRM_DEVERR_TIMEOUT

    # the context still runs the real path correctly afterwards
    cfg = get_config("qwen3-30b-a3b-t4k", T=256, D=128, H=64, E=8, K=2)
    inp = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in generate(cfg).items()}
    pipe = RecalibratedExpertBackward(cfg.T, cfg.D, cfg.H, cfg.E, cfg.K, cfg.dtype, dev)
    pipe.dispatch(inp["topk_idx"])
    ab = pipe.to_dispatch_order(inp["ab_pair"])
    phi = pipe.to_dispatch_order(inp["phi_pair"])
    pipe.step(inp["topk_idx"], inp["alpha"], inp["x"], inp["g"], ab, phi, inp["w_gate"],
              inp["w_up"], inp["w_down"], rate=(1, 2))
    torch.cuda.synchronize()
    assert pipe.device_error() == 0
    assert np.isfinite(pipe.dw_gate.cpu().numpy()).all()
    assert float(pipe.dw_gate.abs().sum()) > 0
