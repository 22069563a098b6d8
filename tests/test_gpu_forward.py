"""Parity of the forward expert pass (token gather, gate/up products with the
SwiGLU epilogue, down products, weighted combine) with the oracle (GPU).

Sizes span several 128 x 256 tiles per expert with ragged tails: H = 192
(the second gate/up tile holds 64 valid columns), D = 320 (the second down
tile likewise), groups of about 256 rows, dead and single-row experts, T = 0,
and the benchmark's full layer on sampled rows.
"""

import numpy as np
import pytest
import torch

import oracle
from workloads import generate, get_config

from parity_util import numpy_inputs, to_np
from test_gpu_parity import full_parity

pytestmark = pytest.mark.gpu

# relative L2 error per row against the FP64 chain. A row of y or out has been
# rounded twice on the way (phi, then y), each rounding at most 2^-9 relative
# in BF16, so about 2e-3 per row: the same tolerance holds for every output.
BF16_ROW_TOL = 2e-2
F32_ROW_TOL = 1e-5


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    from demand_side_expert_gb300 import lrm  # noqa: F401  (liblrm.so must load)
    return torch.device("cuda:0")


def _pipe(cfg, dev):
    from demand_side_expert_gb300 import RecalibratedExpertBackward
    return RecalibratedExpertBackward(cfg.T, cfg.D, cfg.H, cfg.E, cfg.K, cfg.dtype, dev)


def _to(inp, dev):
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()}


def check_rows(got, ref, tol, name):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, name
    err = np.linalg.norm(got - ref, axis=1)
    lim = tol * np.linalg.norm(ref, axis=1) + 1e-6 * tol * max(np.abs(ref).max(), 1e-30)
    bad = np.nonzero(err > lim)[0]
    assert bad.size == 0, (f"{name}: {bad.size} rows off, first {bad[:5]}, worst rel "
                           f"{float((err / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)).max()):.3e}")


def forward_parity(cfg, dev, seed=None):
    inp_cpu = generate(cfg, device="cpu", seed=seed)
    inp = _to(inp_cpu, dev)
    pipe = _pipe(cfg, dev)
    pipe.forward(inp["topk_idx"], inp["alpha"], inp["x"], inp["w_gate"], inp["w_up"],
                 inp["w_down"])
    torch.cuda.synchronize()
    assert pipe.device_error() == 0
    nin = numpy_inputs(inp_cpu)
    f = oracle.moe_forward(nin["topk_idx"], nin["alpha"], nin["x"], nin["w_gate"], nin["w_up"],
                           nin["w_down"], cfg.E)
    N = cfg.N
    assert np.array_equal(to_np(pipe.perm)[:N], f["perm"])
    assert np.array_equal(to_np(pipe.off), f["off"])
    assert np.array_equal(to_np(pipe.x_disp)[:N].astype(np.float64), f["x_disp"])  # a copy
    # the GPU's later products read its own rounded intermediates: compare each
    # product with the oracle applied to the GPU's inputs of that product, and
    # the chain as a whole with the oracle's FP64 forward
    tol = BF16_ROW_TOL if cfg.dtype == "bf16" else F32_ROW_TOL
    check_rows(to_np(pipe.ab)[:N], f["ab"], tol, "ab")
    check_rows(to_np(pipe.phi)[:N], f["phi"], tol, "phi")
    _, _, y_own = oracle.expert_fwd(f["off"], nin["w_gate"], nin["w_up"], nin["w_down"],
                                    f["x_disp"])
    check_rows(to_np(pipe.y)[:N], y_own, tol, "y")
    y_from_gpu_phi = np.zeros_like(y_own)
    for e in range(cfg.E):
        lo, hi = int(f["off"][e]), int(f["off"][e + 1])
        y_from_gpu_phi[lo:hi] = to_np(pipe.phi)[lo:hi].astype(np.float64) @ nin["w_down"][e]
    check_rows(to_np(pipe.y)[:N], y_from_gpu_phi, tol, "y (GPU phi)")
    out_from_gpu_y = oracle.combine(to_np(pipe.y)[:N], nin["alpha"], f["inv"], cfg.K)
    check_rows(to_np(pipe.out)[:cfg.T], out_from_gpu_y, 1e-5, "out (GPU y)")
    check_rows(to_np(pipe.out)[:cfg.T], f["out"], tol, "out")
    return pipe, inp_cpu


def test_forward_tiny_fp32(dev):
    forward_parity(get_config("tiny"), dev)


def test_forward_fp32_wider(dev):
    forward_parity(get_config("tiny", T=200, D=48, H=40, E=6, K=3), dev)


def test_forward_bf16_ragged_tiles(dev):
    forward_parity(get_config("qwen3-30b-a3b-t4k", T=1024, D=320, H=192, E=12, K=3), dev)


def test_forward_bf16_wide_layer_many_experts(dev):
    forward_parity(get_config("glm45-106b-a12b-t16k", T=768, D=512, H=320, E=24, K=4), dev)


def test_forward_stress_edge_groups(dev):
    cfg = get_config("stress-e256", T=2048, D=256, H=128)
    pipe, inp = forward_parity(cfg, dev)
    counts = to_np(pipe.counts)
    assert (counts == 0).sum() >= 16 and (counts == 1).sum() >= 1


def test_forward_empty_layer(dev):
    cfg = get_config("qwen3-30b-a3b-t4k", T=0, D=128, H=64, E=4, K=2)
    pipe = _pipe(cfg, dev)
    z = torch.zeros(0, 2, dtype=torch.int32, device=dev)
    w = torch.zeros(4, 128, 64, dtype=torch.bfloat16, device=dev)
    wd = torch.zeros(4, 64, 128, dtype=torch.bfloat16, device=dev)
    pipe.forward(z, torch.zeros(0, 2, device=dev),
                 torch.zeros(0, 128, dtype=torch.bfloat16, device=dev), w, w, wd)
    torch.cuda.synchronize()
    assert pipe.device_error() == 0


def test_forward_split_calls_match_one_call(dev):
    cfg = get_config("qwen3-30b-a3b-t4k", T=512, D=256, H=192, E=8, K=4)
    inp = _to(generate(cfg, device="cpu"), dev)
    pipe = _pipe(cfg, dev)
    pipe.forward(inp["topk_idx"], inp["alpha"], inp["x"], inp["w_gate"], inp["w_up"],
                 inp["w_down"])
    ref = {k: getattr(pipe, k).clone() for k in ("x_disp", "ab", "phi", "y", "out")}
    for k in ref:
        getattr(pipe, k).fill_(float("nan"))
    pipe.gather_tokens(inp["x"])
    pipe.fc1_fwd(inp["w_gate"], inp["w_up"])
    pipe.fc2_fwd(inp["w_down"])
    pipe.combine(inp["alpha"])
    torch.cuda.synchronize()
    for k, v in ref.items():
        assert torch.equal(getattr(pipe, k), v), k


def test_forward_saved_state_drives_the_backward(dev):
    """The forward's [a | b] and phi, taken as the saved state, through the
    whole recalibrated backward against the oracle."""
    cfg = get_config("qwen3-30b-a3b-t4k", T=1024, D=320, H=192, E=12, K=3)
    inp_cpu = generate(cfg, device="cpu")
    inp = _to(inp_cpu, dev)
    pipe = _pipe(cfg, dev)
    pipe.forward(inp["topk_idx"], inp["alpha"], inp["x"], inp["w_gate"], inp["w_up"],
                 inp["w_down"])
    torch.cuda.synchronize()
    inv = pipe.inv[:cfg.N].long()
    inp_cpu["ab_pair"] = pipe.ab[inv].cpu()    # back to pair order
    inp_cpu["phi_pair"] = pipe.phi[inv].cpu()
    full_parity(cfg, dev, (1, 2), inp_cpu=inp_cpu)


def test_full_size_forward_qwen3_t4k(dev):
    """The benchmark's layer in the launch configuration it times; sampled
    dispatch rows and tokens computed one by one by the oracle."""
    cfg = get_config("qwen3-30b-a3b-t4k")
    inp = generate(cfg, device=dev)
    pipe = _pipe(cfg, dev)
    pipe.forward(inp["topk_idx"], inp["alpha"], inp["x"], inp["w_gate"], inp["w_up"],
                 inp["w_down"])
    torch.cuda.synchronize()
    assert pipe.device_error() == 0
    topk = to_np(inp["topk_idx"])
    perm, inv, counts, off = oracle.dispatch_permute(topk, cfg.E)
    assert np.array_equal(to_np(pipe.perm)[:cfg.N], perm)
    rng = np.random.default_rng(0)
    P = np.sort(rng.choice(cfg.N, size=512, replace=False))
    x = to_np(inp["x"])
    # the sampled rows of each expert as one small group through that expert
    ex = np.searchsorted(off, P, side="right") - 1
    for e in np.unique(ex):
        sel = P[ex == e]
        w = [to_np(inp[k][e:e + 1]) for k in ("w_gate", "w_up", "w_down")]
        ab, phi, y = oracle.expert_fwd(np.array([0, sel.size]), *w, x[perm[sel] // cfg.K])
        idx = torch.as_tensor(sel, device=dev)
        check_rows(to_np(pipe.ab[idx]), ab, BF16_ROW_TOL, f"ab of expert {e}")
        check_rows(to_np(pipe.phi[idx]), phi, BF16_ROW_TOL, f"phi of expert {e}")
        check_rows(to_np(pipe.y[idx]), y, BF16_ROW_TOL, f"y of expert {e}")
    # combine on sampled tokens from the GPU's own y rows
    y_all = pipe.y
    for t in rng.choice(cfg.T, size=64, replace=False):
        rows = [int(inv[t * cfg.K + k]) for k in range(cfg.K)]
        want = sum(float(inp["alpha"][t, k]) * to_np(y_all[r]).astype(np.float64)
                   for k, r in enumerate(rows))
        check_rows(to_np(pipe.out[int(t)])[None], want[None], 1e-5, f"out[{t}]")
