"""Host orchestration of the recalibrated expert backward on one GPU.

``RecalibratedExpertBackward`` owns the device buffers of one layer shape
(allocated once through PyTorch, reused every step) and issues the C-ABI
calls of liblrm in order on one CUDA stream:

  lrm_dispatch_permute -> lrm_quota_from_rate -> lrm_score ->
  lrm_select_quota -> lrm_compact -> lrm_expert_bwd_grouped

and, for the forward expert pass that produces the saved state,
lrm_dispatch_permute -> lrm_expert_fwd_grouped.

Every step of the path runs in liblrm's kernels; this class only allocates
and passes pointers.
"""

from __future__ import annotations

import torch

from . import lrm

_TORCH_DTYPE = {lrm.LRM_F32: torch.float32, lrm.LRM_BF16: torch.bfloat16}


def dtype_code(name: str) -> int:
    return {"f32": lrm.LRM_F32, "bf16": lrm.LRM_BF16}[name]


class RecalibratedExpertBackward:
    """Buffers + call sequence for one (T, D, H, E, K, dtype) layer shape."""

    def __init__(self, T: int, D: int, H: int, E: int, K: int, dtype: str = "bf16",
                 device: str | torch.device = "cuda"):
        self.T, self.D, self.H, self.E, self.K = T, D, H, E, K
        self.N = T * K
        self.dtype_code = dtype_code(dtype)
        self.tdtype = _TORCH_DTYPE[self.dtype_code]
        self.shape = lrm.make_shape(T, D, H, E, K, self.dtype_code)
        dev = torch.device(device)
        self.device = dev
        i32, f32, dt = torch.int32, torch.float32, self.tdtype
        rows = max(self.N, 1)

        def empty(*shape, dtype):
            return torch.empty(*shape, dtype=dtype, device=dev)

        self.ws_bytes = lrm.lrm_workspace_bytes(self.shape)
        if self.ws_bytes == 0:
            raise lrm.LrmError("lrm_workspace_bytes", lrm.LRM_ERR_INVALID_ARG)
        self.ws = empty(self.ws_bytes, dtype=torch.uint8)
        self.perm, self.inv = empty(rows, dtype=i32), empty(rows, dtype=i32)
        self.counts, self.off = empty(E, dtype=i32), empty(E + 1, dtype=i32)
        self.quota = empty(E, dtype=i32)
        self.score = empty(rows, dtype=f32)
        self.keep = empty(rows, dtype=torch.uint8)
        self.sel_off, self.sel_pos = empty(E + 1, dtype=i32), empty(rows, dtype=i32)
        self.dy_c, self.x_c = empty(rows, D, dtype=dt), empty(rows, D, dtype=dt)
        self.ab_c, self.phi_c = empty(rows, 2 * H, dtype=dt), empty(rows, H, dtype=dt)
        self.tok_c, self.row_of_pos = empty(rows, dtype=i32), empty(rows, dtype=i32)
        self.dab_c, self.dx_c = empty(rows, 2 * H, dtype=dt), empty(rows, D, dtype=f32)
        self.dw_gate, self.dw_up = empty(E, D, H, dtype=f32), empty(E, D, H, dtype=f32)
        self.dw_down = empty(E, H, D, dtype=f32)
        self.dx = empty(max(T, 1), D, dtype=f32)
        lrm.lrm_clear_device_error(self.ws, self.ws_bytes)

    # -- forward side -------------------------------------------------------
    def dispatch(self, topk_idx, stream=None):
        lrm.lrm_dispatch_permute(self.shape, topk_idx, self.perm, self.inv, self.counts,
                                 self.off, self.ws, self.ws_bytes, stream)

    def _forward_buffers(self):
        """Forward outputs, allocated on the first forward call only."""
        if getattr(self, "x_disp", None) is None:
            rows, dt, dev = max(self.N, 1), self.tdtype, self.device
            self.x_disp = torch.empty(rows, self.D, dtype=dt, device=dev)
            self.ab = torch.empty(rows, 2 * self.H, dtype=dt, device=dev)
            self.phi = torch.empty(rows, self.H, dtype=dt, device=dev)
            self.y = torch.empty(rows, self.D, dtype=dt, device=dev)
            self.out = torch.empty(max(self.T, 1), self.D, dtype=torch.float32, device=dev)

    def forward(self, topk_idx, alpha, x, w_gate, w_up, w_down, stream=None):
        """Forward expert pass: dispatch, gather, gate/up + SwiGLU, down,
        combine. Leaves the saved state in ``ab`` / ``phi`` (dispatch order)
        and the layer output in ``out`` (float32 [T, D])."""
        self._forward_buffers()
        self.dispatch(topk_idx, stream)
        lrm.lrm_expert_fwd_grouped(self.shape, self.perm, self.inv, self.off, alpha, x, w_gate,
                                   w_up, w_down, self.x_disp, self.ab, self.phi, self.y,
                                   self.out, self.ws, self.ws_bytes, stream)

    def gather_tokens(self, x, stream=None):
        self._forward_buffers()
        lrm.lrm_gather_tokens(self.shape, self.perm, x, self.x_disp, self.ws, self.ws_bytes,
                              stream)

    def fc1_fwd(self, w_gate, w_up, stream=None):
        lrm.lrm_expert_fc1_fwd(self.shape, self.off, self.x_disp, w_gate, w_up, self.ab,
                               self.phi, self.ws, self.ws_bytes, stream)

    def fc2_fwd(self, w_down, stream=None):
        lrm.lrm_expert_fc2_fwd(self.shape, self.off, self.phi, w_down, self.y, self.ws,
                               self.ws_bytes, stream)

    def combine(self, alpha, stream=None):
        lrm.lrm_combine(self.shape, self.y, alpha, self.inv, self.out, self.ws, self.ws_bytes,
                        stream)

    def to_dispatch_order(self, rows_by_pair: torch.Tensor, stream=None) -> torch.Tensor:
        """Lay per-pair rows out in dispatch order with the current perm."""
        out = torch.empty_like(rows_by_pair)
        row_bytes = rows_by_pair[0].numel() * rows_by_pair.element_size()
        lrm.lrm_permute_rows(self.perm, self.N, rows_by_pair, out, row_bytes, stream)
        return out

    # -- backward -----------------------------------------------------------
    def quota_from_rate(self, num: int, den: int, cap: int = 0, stream=None):
        lrm.lrm_quota_from_rate(self.counts, self.E, num, den, cap, self.quota, stream)

    def score_pairs(self, alpha, g, phi, stream=None, metric: int = 0, seed: int = 0):
        """LRM scores (metric 0) or one of the ablation criteria (lrm.LRM_METRIC_*)."""
        if metric == lrm.LRM_METRIC_LRM:
            lrm.lrm_score(self.shape, g, phi, alpha, self.inv, self.score, self.ws,
                          self.ws_bytes, stream)
        else:
            lrm.lrm_score_variant(self.shape, metric, seed, g, phi, alpha, self.inv, self.score,
                                  self.ws, self.ws_bytes, stream)

    def select_rate(self, num: int, den: int, cap: int = 0, stream=None):
        """Quotas from the rate and the selection in one launch."""
        lrm.lrm_select_rate(self.shape, self.score, self.off, num, den, cap, self.quota,
                            self.keep, self.sel_off, self.sel_pos, self.ws, self.ws_bytes, stream)

    def select(self, stream=None):
        lrm.lrm_select_quota(self.shape, self.score, self.off, self.quota, self.keep,
                             self.sel_off, self.sel_pos, self.ws, self.ws_bytes, stream)

    def compact(self, alpha, x, g, ab, phi, stream=None, gathered: bool = False):
        """Gather the retained rows; ab=None copies no [a | b] (recompute);
        gathered=True writes only the gradient rows (the products then read
        x, ab and phi in place)."""
        x_c = None if gathered else self.x_c
        ab_c = None if (gathered or ab is None) else self.ab_c
        phi_c = None if gathered else self.phi_c
        lrm.lrm_compact(self.shape, self.perm, self.keep, self.sel_off, self.sel_pos, alpha, x,
                        g, ab, phi, self.dy_c, x_c, ab_c, phi_c, self.tok_c, self.row_of_pos,
                        self.ws, self.ws_bytes, stream)

    def fc1_recompute(self, w_gate, w_up, stream=None):
        """[a | b] of the retained rows rebuilt from x_c (no saved [a | b])."""
        lrm.lrm_expert_fc1_recompute(self.shape, self.sel_off, self.x_c, w_gate, w_up,
                                     self.ab_c, self.ws, self.ws_bytes, stream)

    def score_select_compact(self, alpha, x, g, ab, phi, stream=None, metric: int = 0,
                             seed: int = 0, gathered: bool = False):
        self.score_pairs(alpha, g, phi, stream, metric, seed)
        self.select(stream)
        self.compact(alpha, x, g, ab, phi, stream, gathered)

    def expert_bwd_gathered(self, x, ab, phi, w_gate, w_up, w_down, parts: int | None = None,
                            stream=None):
        """The expert backward reading x, ab and phi rows in place (after a
        gathered compaction); `parts` selects sub-steps (lrm.LRM_BWD_*)."""
        lrm.lrm_expert_bwd_gathered(
            self.shape, lrm.LRM_BWD_ALL if parts is None else parts, self.sel_off, self.sel_pos,
            self.tok_c, w_gate, w_up, w_down, self.dy_c, x, ab, phi, self.inv, self.row_of_pos,
            self.dab_c, self.dx_c, self.dw_gate, self.dw_up, self.dw_down, self.dx, self.ws,
            self.ws_bytes, stream)

    def expert_bwd(self, w_gate, w_up, w_down, stream=None):
        lrm.lrm_expert_bwd_grouped(
            self.shape, self.sel_off, w_gate, w_up, w_down, self.dy_c, self.x_c, self.ab_c,
            self.phi_c, self.inv, self.row_of_pos, self.dab_c, self.dx_c, self.dw_gate,
            self.dw_up, self.dw_down, self.dx, self.ws, self.ws_bytes, stream)

    # the same backward as five separate calls (one kernel each), so that a
    # caller can time or overlap the sub-steps
    def fc2_dgrad(self, w_down, stream=None):
        lrm.lrm_expert_fc2_dgrad(self.shape, self.sel_off, w_down, self.dy_c, self.ab_c,
                                 self.dab_c, self.ws, self.ws_bytes, stream)

    def fc2_wgrad(self, stream=None):
        lrm.lrm_expert_fc2_wgrad(self.shape, self.sel_off, self.phi_c, self.dy_c, self.dw_down,
                                 self.ws, self.ws_bytes, stream)

    def fc1_wgrad(self, stream=None):
        lrm.lrm_expert_fc1_wgrad(self.shape, self.sel_off, self.x_c, self.dab_c, self.dw_gate,
                                 self.dw_up, self.ws, self.ws_bytes, stream)

    def fc1_dgrad(self, w_gate, w_up, stream=None):
        lrm.lrm_expert_fc1_dgrad(self.shape, self.sel_off, w_gate, w_up, self.dab_c, self.dx_c,
                                 self.ws, self.ws_bytes, stream)

    def scatter_dx(self, stream=None):
        lrm.lrm_scatter_dx(self.shape, self.dx_c, self.inv, self.row_of_pos, self.dx, self.ws,
                           self.ws_bytes, stream)

    def step(self, topk_idx, alpha, x, g, ab, phi, w_gate, w_up, w_down, rate=(1, 1),
             cap: int = 0, quota: torch.Tensor | None = None, stream=None, metric: int = 0,
             seed: int = 0, gathered: bool = False):
        """One pass of the whole path. ab / phi are in dispatch order; `metric`
        picks the selection criterion (LRM by default). ab=None recomputes
        [a | b] of the retained rows instead of reading saved state;
        gathered=True lets the products read x, ab and phi rows in place."""
        if gathered and ab is None:
            raise ValueError("the gathered backward reads saved [a | b]")
        self.dispatch(topk_idx, stream)
        self.score_pairs(alpha, g, phi, stream, metric, seed)
        if quota is None:
            self.select_rate(rate[0], rate[1], cap, stream)
        else:
            self.quota.copy_(quota)
            self.select(stream)
        self.compact(alpha, x, g, ab, phi, stream, gathered)
        if gathered:
            self.expert_bwd_gathered(x, ab, phi, w_gate, w_up, w_down, stream=stream)
            return
        if ab is None:
            self.fc1_recompute(w_gate, w_up, stream)
        self.expert_bwd(w_gate, w_up, w_down, stream)

    def device_error(self, stream=None) -> int:
        return lrm.lrm_get_device_error(self.ws, self.ws_bytes, stream)

    def clear_device_error(self, stream=None):
        lrm.lrm_clear_device_error(self.ws, self.ws_bytes, stream)

    @property
    def retained_rows(self) -> int:
        return int(self.sel_off[self.E].item())
