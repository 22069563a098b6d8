"""Element-by-element parity of the CUDA path with the CPU oracle (GPU).

Sizes here span several 128 x 256 tiles per expert with ragged tails in
every dimension (rows per group, K blocks of the weight-gradient products,
N tiles), plus the degenerate cases: empty and single-row experts, a group
holding every token, zero and full retention, capped quotas, T = 0, bad
expert ids and oversize quotas (flagged on the device, never trapped).
"""

import numpy as np
import pytest
import torch

import oracle
from workloads import generate, get_config

from parity_util import (check_backward, check_compaction, check_dispatch, check_scores,
                         check_selection, check_set_agreement, numpy_inputs, rel_fro, run_gpu,
                         to_np)

pytestmark = pytest.mark.gpu


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


def full_parity(cfg, dev, rate, cap=0, quota=None, seed=None, metric=0, rseed=0,
                inp_cpu=None, gathered=False):
    """Every step of the path against the oracle on one seeded layer; `metric`
    and `rseed` pick the selection criterion and the random criterion's seed;
    `inp_cpu` replaces the generated layer."""
    if inp_cpu is None:
        inp_cpu = generate(cfg, device="cpu", seed=seed)
    inp = _to(inp_cpu, dev)
    pipe = _pipe(cfg, dev)
    q_t = None if quota is None else torch.as_tensor(quota, dtype=torch.int32, device=dev)
    if gathered:  # rows the gathered products must not need
        for k in ("x_c", "ab_c", "phi_c"):
            getattr(pipe, k).fill_(float("nan"))
    run_gpu(pipe, inp, rate, cap, q_t, metric, rseed, gathered)
    assert pipe.device_error() == 0
    nin = numpy_inputs(inp_cpu)
    perm, inv, counts, off = check_dispatch(pipe, nin["topk_idx"], cfg.E)
    ab = oracle.lrm_oracle.permute_rows(nin["ab_pair"], perm)
    phi = oracle.lrm_oracle.permute_rows(nin["phi_pair"], perm)
    assert np.array_equal(to_np(pipe.quota),
                          oracle.quota_from_rate(counts, rate[0], rate[1], cap)
                          if quota is None else np.asarray(quota))
    qv = to_np(pipe.quota).astype(np.int64)
    ref_score = oracle.score_variant(metric, nin["g"], phi, nin["alpha"], perm, cfg.K, rseed)
    N = cfg.N
    if metric == oracle.METRIC_RANDOM:  # integer arithmetic: bit-exact
        assert np.array_equal(to_np(pipe.score)[:N].astype(np.float64), ref_score)
    else:
        check_scores(to_np(pipe.score)[:N], ref_score)
    keep, sel_off, sel_pos = check_selection(pipe, perm, off, qv)
    check_set_agreement(keep, ref_score, off, qv)
    c = check_compaction(pipe, nin, perm, sel_off, sel_pos, ab, phi, cfg.K, cfg.dtype,
                         copies=not gathered)
    errs = check_backward(pipe, nin, c, sel_off, inv, cfg.T, cfg.K, cfg.dtype)
    return pipe, errs


# ---------------------------------------------------------------------------
def test_tiny_fp32_layer(dev):
    full_parity(get_config("tiny"), dev, (1, 2))


@pytest.mark.parametrize("rate", [(1, 2), (3, 5), (1, 4)])
def test_bf16_ragged_tiles(dev, rate):
    # H=192: G1 N tile and G2 M tile ragged; 2H=384 ragged in G3; m_e ~ 160
    # rows: several row tiles and a K tail that is not a multiple of 16
    cfg = get_config("qwen3-30b-a3b-t4k", T=1024, D=320, H=192, E=12, K=3)
    full_parity(cfg, dev, rate)


@pytest.mark.parametrize("rate", [(1, 2), (1, 1)])
@pytest.mark.parametrize("gathered", [False, True])
def test_fc1_dgrad_on_wide_tiles(dev, rate, gathered):
    # 2H = 2048 spans 32 K blocks: FC1 dgrad runs on 256 x 512 tiles. D = 640
    # ends in a tile whose first accumulator is partly outside D and whose
    # second lies wholly outside it (its copies and MMAs are skipped); the
    # smaller experts' tiles leave the odd CTA of a pair without rows.
    cfg = get_config("glm45-106b-a12b-t16k", T=1024, D=640, H=1024, E=12, K=3)
    full_parity(cfg, dev, rate, gathered=gathered)


@pytest.mark.parametrize("over,rate", [
    # 2H = 2176: 34 K blocks, 17 from each of W_gate and W_up; D = 576: the
    # second tile's first accumulator holds 64 valid columns and its second none
    ({"T": 700, "D": 576, "H": 1088, "E": 5, "K": 2}, (2, 3)),
    # D = 832: two tiles across D, the second one's second accumulator holds
    # 64 valid columns; K = 4 slots, groups of 42 to 286 retained rows
    ({"T": 900, "D": 832, "H": 1024, "E": 9, "K": 4}, (1, 3)),
])
def test_fc1_dgrad_on_wide_tiles_ragged(dev, over, rate):
    full_parity(get_config("glm45-106b-a12b-t16k", **over), dev, rate)


def test_bf16_wide_layer_many_experts(dev):
    cfg = get_config("glm45-106b-a12b-t16k", T=768, D=512, H=320, E=24, K=4)
    full_parity(cfg, dev, (3, 4))


def test_fp32_wider_layer(dev):
    cfg = get_config("tiny", T=200, D=48, H=40, E=6, K=3)
    full_parity(cfg, dev, (3, 5))


def test_stress_edge_groups(dev):
    # dead experts, single-row experts, near-full experts and a capped quota
    cfg = get_config("stress-e256", T=2048, D=256, H=128)
    inp = generate(cfg, device="cpu")
    counts = np.bincount(inp["topk_idx"].reshape(-1).numpy(), minlength=cfg.E)
    assert (counts == 0).sum() >= 16 and (counts == 1).sum() >= 1
    cap = 100  # below the hot experts' ceil(n/2)
    full_parity(cfg, dev, (1, 2), cap=cap)


def test_explicit_quotas_and_extremes(dev):
    cfg = get_config("qwen3-30b-a3b-t4k", T=300, D=128, H=64, E=10, K=2)
    inp = generate(cfg, device="cpu")
    counts = np.bincount(inp["topk_idx"].reshape(-1).numpy(), minlength=cfg.E)
    quota = counts.copy()
    quota[0] = 0                 # nothing kept
    quota[1] = min(1, counts[1])  # one row
    quota[2] = counts[2]         # everything kept
    quota[3:] = counts[3:] // 3
    full_parity(cfg, dev, (1, 1), quota=quota.astype(np.int32))


@pytest.mark.parametrize("over", [
    dict(T=256, D=128, H=1664, E=8, K=4),   # phi rows longer than the up-front kernels hold
    dict(T=128, D=128, H=128, E=16, K=10),  # more than 8 routed experts per token
])
def test_bf16_score_generic_kernel(dev, over):
    """BF16 shapes outside the up-front score kernel's instantiations take the
    generic kernel; the whole path still matches the oracle."""
    full_parity(get_config("qwen3-30b-a3b-t4k", **over), dev, (1, 2))


@pytest.mark.parametrize("over,rate", [
    (dict(T=300, D=128, H=64, E=6, K=1), (1, 2)),   # top-1 routing
    (dict(T=200, D=128, H=64, E=1, K=1), (3, 5)),   # one expert holding every token
    (dict(T=1, D=128, H=64, E=8, K=2), (1, 1)),     # a single token
    (dict(T=1, D=128, H=64, E=8, K=2), (1, 2)),     # a single token, half its pairs
])
def test_degenerate_routings(dev, over, rate):
    full_parity(get_config("qwen3-30b-a3b-t4k", **over), dev, rate)


@pytest.mark.parametrize("over,rate", [
    (dict(T=300, D=128, H=64, E=6, K=1), (1, 2)),
    (dict(T=200, D=128, H=64, E=1, K=1), (3, 5)),
])
def test_degenerate_routings_gathered(dev, over, rate):
    full_parity(get_config("qwen3-30b-a3b-t4k", **over), dev, rate, gathered=True)


def test_zero_retention(dev):
    cfg = get_config("qwen3-30b-a3b-t4k", T=256, D=128, H=64, E=8, K=2)
    pipe, _ = full_parity(cfg, dev, (0, 1))
    assert pipe.retained_rows == 0
    assert float(pipe.dw_down.abs().max()) == 0.0 and float(pipe.dx.abs().max()) == 0.0


def test_empty_layer(dev):
    cfg = get_config("qwen3-30b-a3b-t4k", T=0, D=128, H=64, E=4, K=2)
    from workloads.configs import LayerConfig  # noqa: F401
    pipe = _pipe(cfg, dev)
    z = torch.zeros(0, 2, dtype=torch.int32, device=dev)
    pipe.dispatch(z)
    pipe.quota_from_rate(1, 2)
    pipe.score_select_compact(torch.zeros(0, 2, device=dev),
                              torch.zeros(0, 128, dtype=torch.bfloat16, device=dev),
                              torch.zeros(0, 128, dtype=torch.bfloat16, device=dev),
                              torch.zeros(1, 128, dtype=torch.bfloat16, device=dev),
                              torch.zeros(1, 64, dtype=torch.bfloat16, device=dev))
    w = torch.zeros(4, 128, 64, dtype=torch.bfloat16, device=dev)
    pipe.expert_bwd(w, w, torch.zeros(4, 64, 128, dtype=torch.bfloat16, device=dev))
    torch.cuda.synchronize()
    assert pipe.device_error() == 0
    assert to_np(pipe.off).tolist() == [0] * 5
    assert to_np(pipe.sel_off).tolist() == [0] * 5
    assert float(pipe.dw_gate.abs().max()) == 0.0


def test_full_retention_bitwise_equals_uncompacted_run(dev):
    cfg = get_config("qwen3-30b-a3b-t4k", T=640, D=256, H=128, E=8, K=2)
    inp = _to(generate(cfg, device="cpu"), dev)
    pipe = _pipe(cfg, dev)
    ab, phi = run_gpu(pipe, inp, (1, 1))
    N = cfg.N
    perm = pipe.perm[:N].long()
    assert torch.equal(pipe.sel_pos[:N].long(), torch.arange(N, device=dev))
    assert torch.equal(pipe.row_of_pos[:N].long(), torch.arange(N, device=dev))
    assert torch.equal(pipe.ab_c[:N], ab) and torch.equal(pipe.phi_c[:N], phi)
    # the unpruned backward run directly on the uncompacted dispatch-order rows
    dy = (inp["alpha"].reshape(-1)[perm][:, None] * inp["g"][perm // cfg.K].float()).to(
        torch.bfloat16)
    xs = inp["x"][perm // cfg.K].contiguous()
    assert torch.equal(pipe.dy_c[:N], dy) and torch.equal(pipe.x_c[:N], xs)
    outs = {k: getattr(pipe, k).clone() for k in ("dw_gate", "dw_up", "dw_down", "dx")}
    from demand_side_expert_gb300 import lrm
    ident = torch.arange(N, dtype=torch.int32, device=dev)
    dab = torch.empty_like(pipe.dab_c)
    dxc = torch.empty_like(pipe.dx_c)
    res = {k: torch.empty_like(v) for k, v in outs.items()}
    lrm.lrm_expert_bwd_grouped(pipe.shape, pipe.off, inp["w_gate"], inp["w_up"],
                               inp["w_down"], dy, xs, ab, phi, pipe.inv, ident, dab, dxc,
                               res["dw_gate"], res["dw_up"], res["dw_down"], res["dx"],
                               pipe.ws, pipe.ws_bytes)
    torch.cuda.synchronize()
    for k in outs:
        assert torch.equal(outs[k], res[k]), k


@pytest.mark.parametrize("name,over,gathered", [
    ("qwen3-30b-a3b-t4k", {"T": 512, "D": 256, "H": 128, "E": 8, "K": 4}, False),
    # wide FC1 dgrad tiles, the weight-gradient tile queue and the gather warps
    ("glm45-106b-a12b-t16k", {"T": 1024, "D": 640, "H": 1024, "E": 12, "K": 3}, True),
])
def test_deterministic_repeats(dev, name, over, gathered):
    cfg = get_config(name, **over)
    inp = _to(generate(cfg, device="cpu"), dev)
    pipe = _pipe(cfg, dev)
    first = None
    for _ in range(3):
        run_gpu(pipe, inp, (3, 5), gathered=gathered)
        cur = [getattr(pipe, k).clone() for k in ("score", "sel_pos", "dw_gate", "dw_up",
                                                   "dw_down", "dx")]
        if first is None:
            first = cur
        else:
            for a, b in zip(first, cur):
                assert torch.equal(a, b)


@pytest.mark.parametrize("T", [16384, 16385, 131073])
def test_dispatch_either_side_of_the_single_launch_limit(dev, T):
    """2^17 routed pairs take the one-cluster launch, 2^17 + 8 and 2^20 + 8 the three launches;
    all are the oracle's stable counting sort, bit for bit."""
    cfg = get_config("qwen3-30b-a3b-t4k", T=T, D=64, H=64)
    inp = generate(cfg, device="cpu")
    pipe = _pipe(cfg, dev)
    pipe.dispatch(inp["topk_idx"].to(dev))
    torch.cuda.synchronize()
    assert pipe.device_error() == 0
    check_dispatch(pipe, inp["topk_idx"].numpy(), cfg.E)


def test_weight_gradient_queue_flags_a_bad_header_and_rewinds(dev):
    """The weight-gradient products take their tiles from a queue in the
    workspace header that every launch leaves at zero. A queue that does not
    start at zero (a header never cleared) skips tiles: the launch flags
    LRM_DEVERR_QUEUE and rewinds the queue, and the next step is exact again."""
    from demand_side_expert_gb300 import lrm
    cfg = get_config("qwen3-30b-a3b-t4k", T=512, D=256, H=128, E=8, K=4)
    inp = _to(generate(cfg, device="cpu"), dev)
    pipe = _pipe(cfg, dev)
    words = pipe.ws.view(torch.int32)
    run_gpu(pipe, inp, (1, 2), gathered=True)
    assert pipe.device_error() == 0
    assert words[4:8].tolist() == [0, 0, 0, 0]
    ref = [getattr(pipe, k).clone() for k in ("dw_gate", "dw_up", "dw_down", "dx")]
    words[4] = 3  # the queue would start past three tiles
    run_gpu(pipe, inp, (1, 2), gathered=True)
    assert pipe.device_error() & lrm.LRM_DEVERR_QUEUE
    assert words[4:8].tolist() == [0, 0, 0, 0]
    pipe.clear_device_error()
    run_gpu(pipe, inp, (1, 2), gathered=True)
    assert pipe.device_error() == 0
    for k, r in zip(("dw_gate", "dw_up", "dw_down", "dx"), ref):
        assert torch.equal(getattr(pipe, k), r), k


def test_bad_expert_ids_and_quotas_are_flagged(dev):
    from demand_side_expert_gb300 import lrm
    cfg = get_config("qwen3-30b-a3b-t4k", T=64, D=128, H=64, E=8, K=2)
    inp = _to(generate(cfg, device="cpu"), dev)
    pipe = _pipe(cfg, dev)
    bad = inp["topk_idx"].clone()
    bad[3, 1] = 99
    bad[5, 0] = -4
    pipe.dispatch(bad)
    assert pipe.device_error() & lrm.LRM_DEVERR_EXPERT_ID
    clamped = bad.clamp(0, cfg.E - 1).cpu().numpy()
    check_dispatch(pipe, clamped, cfg.E)
    pipe.clear_device_error()
    pipe.dispatch(inp["topk_idx"])
    quota = pipe.counts.clone()
    quota[2] += 5
    quota[4] = -1
    ab = pipe.to_dispatch_order(inp["ab_pair"])
    phi = pipe.to_dispatch_order(inp["phi_pair"])
    pipe.quota.copy_(quota)
    pipe.score_select_compact(inp["alpha"], inp["x"], inp["g"], ab, phi)
    assert pipe.device_error() & lrm.LRM_DEVERR_QUOTA
    q = to_np(pipe.quota).astype(np.int64)
    n = to_np(pipe.counts).astype(np.int64)
    assert np.array_equal(np.diff(to_np(pipe.sel_off)), np.clip(q, 0, n))


# ---------------------------------------------------------------------------
# full-size layers, in the launch configuration the benchmark times
# ---------------------------------------------------------------------------
def _f64(t) -> np.ndarray:
    return to_np(t).astype(np.float64)


def _oracle_rows(perm, sel_pos, lo, hi, alpha, x, g, ab, phi, K):
    """The oracle's compaction of the retained rows lo..hi-1 (one stretch of
    the compacted buffers), from the layer's own inputs."""
    return oracle.compact(perm, np.array([0, hi - lo]), sel_pos[lo:hi], alpha, x, g, ab, phi, K)


def _full_size(name, rate, cap=0, sample_experts=5, sample_tokens=64, seed=None,
               gathered=True, chunk=8192, every=False):
    """A full-size layer in the launch configuration bench.py times (by
    default the gathered backward). The oracle builds every operand from the
    layer's inputs itself: its own dispatch-order layout of the saved state,
    its own score of every pair and its own compacted rows; nothing the GPU
    produced is fed back into it except the selection indices, which are
    first shown equal to the oracle selector's.

    Checked: dispatch, quotas, selection, tok_c and row_of_pos exhaustively;
    every score (1e-5 relative) and set agreement of the selection with the
    FP64 scores outside the 1e-5 band; every retained gradient row dy_c
    within one rounding of alpha*g (and, with the compacted backward, every
    copied row of x_c, ab_c and phi_c bit for bit); weight gradients and the
    data-gradient rows of sampled experts and dx of sampled tokens within
    2e-2 relative Frobenius error. With ``every``, the weight gradients and
    data-gradient rows of every expert (exact zeros for experts with no
    retained row) and dx of every token, the latter summed by the oracle's
    own scatter from its own rows."""
    cfg = get_config(name)
    dev = torch.device("cuda:0")
    inp = generate(cfg, device=dev, seed=seed)
    pipe = _pipe(cfg, dev)
    run_gpu(pipe, inp, rate, cap, gathered=gathered)
    assert pipe.device_error() == 0
    K, N = cfg.K, cfg.N
    alpha, x, g = _f64(inp["alpha"]), _f64(inp["x"]), _f64(inp["g"])
    perm, inv, counts, off = check_dispatch(pipe, to_np(inp["topk_idx"]), cfg.E)
    qv = oracle.quota_from_rate(counts, rate[0], rate[1], cap)
    assert np.array_equal(to_np(pipe.quota), qv)
    # the saved state in the oracle's own dispatch order
    phi = oracle.lrm_oracle.permute_rows(_f64(inp["phi_pair"]), perm)
    ab = oracle.lrm_oracle.permute_rows(_f64(inp["ab_pair"]), perm)
    ref_score = oracle.score(g, phi, alpha, perm, K)
    check_scores(to_np(pipe.score)[:N], ref_score)
    keep, sel_off, sel_pos = check_selection(pipe, perm, off, qv)
    check_set_agreement(keep, ref_score, off, qv)
    M = int(sel_off[-1])
    # every retained row, the oracle's compaction taken a stretch at a time
    rop = np.full(N, -1, dtype=np.int64)
    for lo in range(0, M, chunk):
        hi = min(M, lo + chunk)
        c = _oracle_rows(perm, sel_pos, lo, hi, alpha, x, g, ab, phi, K)
        assert np.array_equal(to_np(pipe.tok_c[lo:hi]), c["tok_c"]), (name, lo)
        kept = c["row_of_pos"] >= 0
        rop[kept] = lo + c["row_of_pos"][kept]
        dy = _f64(pipe.dy_c[lo:hi])
        assert np.all(np.abs(dy - c["dy_c"]) <= 2.0 ** -8 * np.abs(c["dy_c"]) + 1e-30), \
            (name, "dy_c", lo)
        if not gathered:  # pure copies: bitwise
            for k in ("x_c", "ab_c", "phi_c"):
                assert np.array_equal(_f64(getattr(pipe, k)[lo:hi]), c[k]), (name, k, lo)
    assert np.array_equal(to_np(pipe.row_of_pos)[:N], rop)
    # weight gradients and data-gradient rows of sampled experts (largest,
    # smallest non-empty, random), from the oracle's own compacted rows
    rng = np.random.default_rng(0)
    m = np.diff(sel_off)
    nonempty = np.nonzero(m)[0]
    if every:
        picks = set(range(cfg.E))
        dxc_all = np.zeros((M, cfg.D))
    else:
        picks = {int(np.argmax(m)), int(nonempty[np.argmin(m[nonempty])])}
        picks |= set(int(e) for e in rng.choice(nonempty, size=min(sample_experts, nonempty.size),
                                                replace=False))
    wcache = {}

    def weights(e):
        if e not in wcache:
            wcache[e] = tuple(_f64(inp[k][e:e + 1]) for k in ("w_gate", "w_up", "w_down"))
        return wcache[e]

    for e in sorted(picks):
        lo, hi = int(sel_off[e]), int(sel_off[e + 1])
        if hi == lo:  # no retained row: the weight gradients are exactly zero
            for k in ("dw_gate", "dw_up", "dw_down"):
                assert not getattr(pipe, k)[e].any(), (name, e, k)
            continue
        c = _oracle_rows(perm, sel_pos, lo, hi, alpha, x, g, ab, phi, K)
        b = oracle.expert_bwd(np.array([0, hi - lo]), *weights(e), c["dy_c"], c["x_c"],
                              c["ab_c"], c["phi_c"])
        for k in ("dw_gate", "dw_up", "dw_down"):
            err = rel_fro(to_np(getattr(pipe, k)[e]), b[k][0])
            assert err <= 2e-2, (name, e, k, err)
        for k in ("dab_c", "dx_c"):
            err = rel_fro(to_np(getattr(pipe, k)[lo:hi]), b[k])
            assert err <= 2e-2, (name, e, k, err)
        if every:
            dxc_all[lo:hi] = b["dx_c"]
    if every:  # dx of every token from the oracle's rows and its own scatter
        want = oracle.dx_gather(dxc_all, inv, rop, cfg.T, K)
        got = _f64(pipe.dx[:cfg.T])
        err = np.linalg.norm(got - want, axis=1)
        lim = 2e-2 * np.maximum(np.linalg.norm(want, axis=1), 1e-12)
        assert (err <= lim).all(), (name, "dx", int((err > lim).sum()))
        assert rel_fro(got, want) <= 2e-2
        return pipe
    # dx on sampled tokens: the oracle's rows of the token's kept slots, summed
    for t in rng.choice(cfg.T, size=min(sample_tokens, cfg.T), replace=False):
        want = np.zeros(cfg.D)
        for k in range(K):
            j = int(rop[inv[t * K + k]])
            if j < 0:
                continue
            e = int(np.searchsorted(sel_off, j, side="right") - 1)
            c = _oracle_rows(perm, sel_pos, j, j + 1, alpha, x, g, ab, phi, K)
            _, dxc = oracle.expert_bwd_rows(np.array([0]), np.array([0, 1]), *weights(e),
                                            c["dy_c"], c["ab_c"])
            want += dxc[0]
        got = to_np(pipe.dx[int(t)])
        assert np.linalg.norm(got - want) <= 2e-2 * max(np.linalg.norm(want), 1e-12), (name, t)
    return pipe


def test_full_size_qwen3_t4k(dev):
    _full_size("qwen3-30b-a3b-t4k", (3, 5), every=True)


def test_full_size_qwen3_t4k_compacted(dev):
    _full_size("qwen3-30b-a3b-t4k", (3, 5), gathered=False, every=True)


def test_full_size_qwen3_t32k(dev):
    pipe = _full_size("qwen3-30b-a3b-t32k", (1, 2), every=True)
    counts = to_np(pipe.counts)
    assert counts.max() > 10 * counts.mean()


@pytest.mark.parametrize("rate", [(1, 4), (1, 2), (1, 1)])
def test_full_size_glm45_sweep(dev, rate):
    # every expert and token where the FP64 oracle takes seconds (rho <= 1/2),
    # sampled ones at rho = 1
    pipe = _full_size("glm45-106b-a12b-t16k", rate, every=rate != (1, 1))
    if rate == (1, 1):
        N = pipe.N
        assert torch.equal(pipe.sel_pos[:N].long(), torch.arange(N, device=dev))


def test_full_size_stress(dev):
    cfg = get_config("stress-e256")
    pipe = _full_size("stress-e256", (1, 2), cap=cfg.cap, every=True)
    q = to_np(pipe.quota)
    assert q.max() == cfg.cap


def test_split_substeps_match_one_call(dev):
    cfg = get_config("qwen3-30b-a3b-t4k", T=512, D=256, H=192, E=8, K=4)
    inp = _to(generate(cfg, device="cpu"), dev)
    pipe = _pipe(cfg, dev)
    run_gpu(pipe, inp, (1, 2))
    ref = {k: getattr(pipe, k).clone() for k in ("dab_c", "dx_c", "dw_gate", "dw_up",
                                                  "dw_down", "dx")}
    for k in ref:
        getattr(pipe, k).fill_(float("nan"))
    pipe.fc2_dgrad(inp["w_down"])
    pipe.fc2_wgrad()
    pipe.fc1_wgrad()
    pipe.fc1_dgrad(inp["w_gate"], inp["w_up"])
    pipe.scatter_dx()
    torch.cuda.synchronize()
    M = pipe.retained_rows
    for k, v in ref.items():
        got = getattr(pipe, k)
        if k in ("dab_c", "dx_c"):
            got, v = got[:M], v[:M]
        assert torch.equal(got, v), k


# ---------------------------------------------------------------------------
# the alternative selection criteria of the ablation (LRMoE Sec. 4.7)
# ---------------------------------------------------------------------------
CRITERIA = [oracle.METRIC_GRAD_SQ, oracle.METRIC_GRAD_ABS, oracle.METRIC_RANDOM]


@pytest.mark.parametrize("metric", CRITERIA)
def test_alternative_criteria_whole_path(dev, metric):
    cfg = get_config("qwen3-30b-a3b-t4k", T=1024, D=320, H=192, E=12, K=3)
    full_parity(cfg, dev, (1, 2), metric=metric, rseed=12345)


@pytest.mark.parametrize("metric", CRITERIA)
def test_alternative_criteria_fp32(dev, metric):
    full_parity(get_config("tiny", T=200, D=48, H=40, E=6, K=3), dev, (3, 5), metric=metric,
                rseed=2**64 - 1)


@pytest.mark.parametrize("metric", CRITERIA)
def test_full_size_alternative_criteria(dev, metric):
    """Every score and the whole selection at the benchmark's layer size."""
    cfg = get_config("qwen3-30b-a3b-t4k")
    inp = generate(cfg, device=dev)
    pipe = _pipe(cfg, dev)
    run_gpu(pipe, inp, (3, 5), metric=metric, seed=7)
    assert pipe.device_error() == 0
    topk = to_np(inp["topk_idx"])
    perm, inv, counts, off = check_dispatch(pipe, topk, cfg.E)
    qv = oracle.quota_from_rate(counts, 3, 5)
    ref = oracle.score_variant(metric, to_np(inp["g"]), None, None, perm, cfg.K, 7)
    got = to_np(pipe.score)[:cfg.N]
    if metric == oracle.METRIC_RANDOM:
        assert np.array_equal(got.astype(np.float64), ref)
    else:
        check_scores(got, ref)
    keep, _, _ = check_selection(pipe, perm, off, qv)
    check_set_agreement(keep, ref, off, qv)


def test_random_criterion_depends_on_seed_only(dev):
    cfg = get_config("qwen3-30b-a3b-t4k", T=512, D=128, H=64, E=8, K=2)
    inp = _to(generate(cfg, device="cpu"), dev)
    pipe = _pipe(cfg, dev)
    picks = []
    for seed in (1, 2, 1):
        run_gpu(pipe, inp, (1, 2), metric=oracle.METRIC_RANDOM, seed=seed)
        picks.append(pipe.keep[:cfg.N].clone())
    assert torch.equal(picks[0], picks[2]) and not torch.equal(picks[0], picks[1])


# ---------------------------------------------------------------------------
# retained-only recompute of [a | b] (RelayMoE Sec. 3.3)
# ---------------------------------------------------------------------------
def recompute_parity(cfg, dev, rate, cap=0):
    inp_cpu = generate(cfg, device="cpu")
    inp = _to(inp_cpu, dev)
    pipe = _pipe(cfg, dev)
    pipe.dispatch(inp["topk_idx"])
    phi = pipe.to_dispatch_order(inp["phi_pair"])
    pipe.ab_c.fill_(float("nan"))  # every retained row must be rebuilt
    pipe.step(inp["topk_idx"], inp["alpha"], inp["x"], inp["g"], None, phi, inp["w_gate"],
              inp["w_up"], inp["w_down"], rate=rate, cap=cap)
    torch.cuda.synchronize()
    assert pipe.device_error() == 0
    nin = numpy_inputs(inp_cpu)
    perm, inv, counts, off = check_dispatch(pipe, nin["topk_idx"], cfg.E)
    qv = oracle.quota_from_rate(counts, rate[0], rate[1], cap)
    keep, sel_off, sel_pos = check_selection(pipe, perm, off, qv)
    M = int(sel_off[-1])
    ab = oracle.lrm_oracle.permute_rows(nin["ab_pair"], perm)
    phi_np = oracle.lrm_oracle.permute_rows(nin["phi_pair"], perm)
    c = oracle.compact(perm, sel_off, sel_pos, nin["alpha"], nin["x"], nin["g"], ab, phi_np,
                       cfg.K)
    for name in ("x_c", "phi_c"):
        assert np.array_equal(to_np(getattr(pipe, name))[:M], c[name]), name
    c["ab_c"] = oracle.recompute_ab(sel_off, nin["w_gate"], nin["w_up"], c["x_c"])
    got = to_np(pipe.ab_c)[:M].astype(np.float64)
    err = np.linalg.norm(got - c["ab_c"], axis=1)
    assert np.all(err <= 2e-2 * np.linalg.norm(c["ab_c"], axis=1) + 1e-12), "ab_c rows"
    c["dy_c"] = to_np(pipe.dy_c)[:M].astype(np.float64)
    return check_backward(pipe, nin, c, sel_off, inv, cfg.T, cfg.K, cfg.dtype)


@pytest.mark.parametrize("rate", [(1, 2), (1, 1)])
def test_recompute_bf16_ragged_tiles(dev, rate):
    recompute_parity(get_config("qwen3-30b-a3b-t4k", T=1024, D=320, H=192, E=12, K=3), dev,
                     rate)


def test_recompute_fp32(dev):
    recompute_parity(get_config("tiny", T=200, D=48, H=40, E=6, K=3), dev, (3, 5))


def test_recompute_stress_edge_groups(dev):
    recompute_parity(get_config("stress-e256", T=2048, D=256, H=128), dev, (1, 2), cap=100)


def test_recompute_zero_retention(dev):
    cfg = get_config("qwen3-30b-a3b-t4k", T=256, D=128, H=64, E=8, K=2)
    recompute_parity(cfg, dev, (0, 1))


# ---------------------------------------------------------------------------
# products reading x, [a | b] and phi rows in place (TMA gather4)
# ---------------------------------------------------------------------------
def gathered_equals_compacted(cfg, dev, rate, cap=0, inp=None):
    """The gathered backward gives the compacted backward's results bit for
    bit: the same tiles and reduction order, only the operand source differs."""
    if inp is None:
        inp = _to(generate(cfg, device="cpu"), dev)
    pipe = _pipe(cfg, dev)
    run_gpu(pipe, inp, rate, cap)
    keys = ("dy_c", "tok_c", "row_of_pos", "dab_c", "dx_c", "dw_gate", "dw_up", "dw_down", "dx")
    ref = {k: getattr(pipe, k).clone() for k in keys}
    M = pipe.retained_rows
    for k in ("x_c", "ab_c", "phi_c", "dab_c", "dx_c", "dw_gate", "dw_up", "dw_down", "dx"):
        getattr(pipe, k).fill_(float("nan"))
    run_gpu(pipe, inp, rate, cap, gathered=True)
    assert pipe.device_error() == 0
    for k, v in ref.items():
        got = getattr(pipe, k)
        if k in ("dy_c", "tok_c", "dab_c", "dx_c"):
            got, v = got[:M], v[:M]
        assert torch.equal(got, v), k
    assert bool(torch.isnan(pipe.x_c[:max(M, 1)]).all())  # never written
    return pipe


@pytest.mark.parametrize("rate", [(1, 2), (3, 5), (1, 1)])
def test_gathered_bf16_ragged_tiles_vs_oracle(dev, rate):
    cfg = get_config("qwen3-30b-a3b-t4k", T=1024, D=320, H=192, E=12, K=3)
    full_parity(cfg, dev, rate, gathered=True)


def test_gathered_fp32_vs_oracle(dev):
    full_parity(get_config("tiny", T=200, D=48, H=40, E=6, K=3), dev, (3, 5), gathered=True)


def test_gathered_stress_vs_oracle(dev):
    full_parity(get_config("stress-e256", T=2048, D=256, H=128), dev, (1, 2), cap=100,
                gathered=True)


@pytest.mark.parametrize("rate", [(1, 2), (0, 1), (1, 1)])
def test_gathered_equals_compacted_bitwise(dev, rate):
    gathered_equals_compacted(
        get_config("glm45-106b-a12b-t16k", T=768, D=512, H=320, E=24, K=4), dev, rate)


def test_gathered_equals_compacted_full_size(dev):
    cfg = get_config("qwen3-30b-a3b-t4k")
    gathered_equals_compacted(cfg, dev, (3, 5), inp=generate(cfg, device=dev))


def test_gathered_equals_compacted_full_size_three_stage_ring(dev):
    # 256 experts leave shared memory for a 3-stage operand ring only
    cfg = get_config("stress-e256")
    gathered_equals_compacted(cfg, dev, (1, 2), cap=cfg.cap, inp=generate(cfg, device=dev))


def test_gathered_equals_compacted_fp32(dev):
    gathered_equals_compacted(get_config("tiny"), dev, (1, 2))


# ---------------------------------------------------------------------------
# launches that overlap their predecessor (programmatic dependent launch)
# ---------------------------------------------------------------------------
def test_back_to_back_steps_without_sync_match_synchronized_steps(dev):
    """Two layers' steps issued back to back on one stream (every kernel may be
    scheduled while the previous one drains) give the results of steps run
    one at a time; then the second layer's outputs are checked."""
    cfg = get_config("qwen3-30b-a3b-t4k", T=1024, D=320, H=192, E=12, K=3)
    a = _to(generate(cfg, device="cpu", seed=5), dev)
    b = _to(generate(cfg, device="cpu", seed=6), dev)
    keys = ("perm", "score", "keep", "sel_pos", "dy_c", "dab_c", "dx_c", "dw_gate", "dw_up",
            "dw_down", "dx")

    def run(pipe, inp, gathered):
        pipe.dispatch(inp["topk_idx"])
        abd = pipe.to_dispatch_order(inp["ab_pair"])
        phid = pipe.to_dispatch_order(inp["phi_pair"])
        pipe.step(inp["topk_idx"], inp["alpha"], inp["x"], inp["g"], abd, phid, inp["w_gate"],
                  inp["w_up"], inp["w_down"], rate=(1, 2), gathered=gathered)

    for gathered in (False, True):
        ref = _pipe(cfg, dev)
        run(ref, b, gathered)
        torch.cuda.synchronize()
        want = {k: getattr(ref, k).clone() for k in keys}
        pipe = _pipe(cfg, dev)
        for _ in range(3):  # a, b, a, b, a, b with no synchronization in between
            run(pipe, a, gathered)
            run(pipe, b, gathered)
        torch.cuda.synchronize()
        assert pipe.device_error() == 0
        M = pipe.retained_rows
        for k, v in want.items():
            got = getattr(pipe, k)
            if k in ("dy_c", "dab_c", "dx_c", "sel_pos"):
                got, v = got[:M], v[:M]
            assert torch.equal(got, v), (gathered, k)


def test_padding_rows_after_the_retained_rows_are_zero(dev):
    """The weight-gradient products read 64 rows past the last group as
    padding; the compaction (dy_c) and the FC2 dgrad product (dab_c) write
    them as zeros."""
    cfg = get_config("qwen3-30b-a3b-t4k", T=512, D=256, H=128, E=8, K=2)
    inp = _to(generate(cfg, device="cpu"), dev)
    pipe = _pipe(cfg, dev)
    pipe.dy_c.fill_(float("nan"))
    pipe.dab_c.fill_(float("nan"))
    run_gpu(pipe, inp, (1, 2))
    M, N = pipe.retained_rows, cfg.N
    hi = min(M + 64, N)
    assert hi > M
    assert bool((pipe.dy_c[M:hi] == 0).all()) and bool((pipe.dab_c[M:hi] == 0).all())


def test_select_rate_equals_quota_then_select(dev):
    """The one-launch quota rule + selection gives the two-launch result."""
    cfg = get_config("stress-e256", T=2048, D=256, H=128)
    inp = _to(generate(cfg, device="cpu"), dev)
    for rate, cap in (((1, 2), 100), ((3, 5), 0), ((1, 1), 0), ((0, 1), 0)):
        a, b = _pipe(cfg, dev), _pipe(cfg, dev)
        for pipe in (a, b):
            pipe.dispatch(inp["topk_idx"])
            phi = pipe.to_dispatch_order(inp["phi_pair"])
            pipe.score_pairs(inp["alpha"], inp["g"], phi)
        a.quota_from_rate(rate[0], rate[1], cap)
        a.select()
        b.select_rate(rate[0], rate[1], cap)
        torch.cuda.synchronize()
        assert a.device_error() == 0 and b.device_error() == 0
        N = cfg.N
        M = a.retained_rows
        for k in ("quota", "sel_off"):
            assert torch.equal(getattr(a, k), getattr(b, k)), (rate, k)
        assert torch.equal(a.keep[:N], b.keep[:N]) and torch.equal(a.sel_pos[:M], b.sel_pos[:M])


def test_selection_of_segments_beyond_the_shared_memory_key_stage(dev):
    """The selection stages up to 40,960 keys of a segment in shared memory;
    a larger segment is counted, copied to candidates and kept straight from
    global memory. One expert here holds more than 40,960 pairs; three
    criteria give it scores with many top bytes (LRM), few (squared gradient
    norm) and uniform ones (random). Bit-exact against the oracle's selector
    run on the GPU's scores, with the quotas the exact integer ceiling."""
    cfg = get_config("qwen3-30b-a3b-t4k", T=65536, D=64, H=64, E=4, K=2)
    inp = generate(cfg, device="cpu")
    d = _to(inp, dev)
    pipe = _pipe(cfg, dev)
    pipe.dispatch(d["topk_idx"])
    phi = pipe.to_dispatch_order(d["phi_pair"])
    torch.cuda.synchronize()
    perm, _, _, off = check_dispatch(pipe, inp["topk_idx"].numpy(), cfg.E)
    assert np.diff(off).max() > 40960
    for metric, rate in ((0, (1, 2)), (1, (3, 5)), (3, (1, 2)), (0, (1, 4))):
        pipe.score_pairs(d["alpha"], d["g"], phi, metric=metric, seed=11)
        pipe.select_rate(rate[0], rate[1], 0)
        torch.cuda.synchronize()
        assert pipe.device_error() == 0
        quota = oracle.quota_from_rate(np.diff(off), rate[0], rate[1])
        assert np.array_equal(to_np(pipe.quota), quota), (metric, rate)
        check_selection(pipe, perm, off, quota)
