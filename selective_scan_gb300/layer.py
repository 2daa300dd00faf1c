"""The Mamba2 layer around the recurrent path: in_proj (split into z, xBC, dt by the
GEMM's epilogue) -> causal conv + SiLU -> selective scan -> gated RMSNorm -> out_proj,
the order of the layer the page "Granite Mamba2 Inference Optimization" ports (gllm
PR #85, "Ops": the model splits in_proj into z, xBC and dt). Every step runs in
libmamba2's kernels; this module orders the calls and allocates the intermediates with
torch.
"""
from __future__ import annotations

import torch

from . import (causal_conv1d, decode_step, gated_rmsnorm, in_proj, out_proj, ssd_scan,
               ssd_scan_workspace_bytes)
from .padded import Mamba2Weights


class Mamba2Layer:
    """Weights of one layer: ``w_in`` [d_inner + conv_dim + heads, d_model] and ``w_out``
    [d_model, d_inner] bf16, plus the path's parameters (``Mamba2Weights``)."""

    def __init__(self, w_in: torch.Tensor, w_out: torch.Tensor, weights: Mamba2Weights, dims):
        self.w_in, self.w_out, self.w, self.dims = w_in, w_out, weights, dims
        self.d_model = int(w_in.shape[1])

    def _split(self, rows, dev, act):
        d = self.dims
        return (torch.empty((rows, d.d_inner), dtype=act, device=dev),
                torch.empty((rows, d.conv_dim), dtype=act, device=dev),
                torch.empty((rows, d.heads), dtype=act, device=dev))

    def prefill(self, hidden, conv_pool, ssm_pool, cu_seqlens, slots, fresh, stream=None) -> torch.Tensor:
        """hidden [rows, d_model] (packed runs) -> [rows, d_model]; the pools are updated at the slots."""
        rows, dev, act, w = hidden.shape[0], hidden.device, hidden.dtype, self.w
        z, x, dt = self._split(rows, dev, act)
        in_proj(z, x, dt, hidden, self.w_in, self.dims, stream=stream)
        xbc = torch.empty_like(x)
        causal_conv1d(xbc, x, w.conv_w, w.conv_b, conv_pool, cu_seqlens, slots, fresh, stream=stream)
        y = torch.empty_like(z)
        need = ssd_scan_workspace_bytes(self.dims, rows, cu_seqlens, slots, fresh)
        ws = torch.empty(need, dtype=torch.uint8, device=dev) if need else None
        ssd_scan(y, xbc, dt, w.A_log, w.dt_bias, w.D, ssm_pool, self.dims, cu_seqlens, slots, fresh, workspace=ws,
                 stream=stream)
        g = torch.empty_like(z)
        gated_rmsnorm(g, y, z, w.norm_w, w.norm_groups, w.eps, stream=stream)
        out = torch.empty((rows, self.d_model), dtype=act, device=dev)
        out_proj(out, g, self.w_out, stream=stream)
        return out

    def decode(self, hidden, conv_pool, ssm_pool, slots, fresh=None, stream=None) -> torch.Tensor:
        """One token per sequence: hidden [n, d_model] -> [n, d_model]."""
        n, dev, act, w = hidden.shape[0], hidden.device, hidden.dtype, self.w
        z, x, dt = self._split(n, dev, act)
        in_proj(z, x, dt, hidden, self.w_in, self.dims, stream=stream)
        g = torch.empty_like(z)
        decode_step(g, x, z, dt, w.conv_w, w.conv_b, w.A_log, w.dt_bias, w.D, w.norm_w, w.norm_groups, w.eps,
                    conv_pool, ssm_pool, self.dims, slots, fresh if fresh is not None else [0] * n, stream=stream)
        out = torch.empty((n, self.d_model), dtype=act, device=dev)
        out_proj(out, g, self.w_out, stream=stream)
        return out
