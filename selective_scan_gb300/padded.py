"""Padded batches and an HF-style cache view over the state pools.

The page "Granite Mamba2 Inference Optimization" asks for a layer whose forward takes
``(hidden_states, cache=None, attention_mask=None)``, serves variable-length padded
batches, and returns a cache that exposes ``conv_state``, ``ssm_state``,
``has_previous_state`` and decode-position semantics. This module gives the recurrent
path that interface. The path's own inputs (xBC, z, dt, each ``[batch, seqlen, ...]``)
take the place of the hidden states; the projections around the path are not part of
it. A padding position is not a token: each row's tokens (mask != 0) must be one
contiguous span, left- or right-padded. The tokens are packed into a RecurrentBatch
(``mamba2_padded_spans``, ``mamba2_pack_rows``), the three prefill ops run on the
packed rows, and the output is scattered back with zeros at padding
(``mamba2_unpack_rows``). With left padding from an empty cache this is the same as
zeroing the padded inputs and conv outputs and running every row whole: zero inputs
keep a zero state at zero. Every step runs in libmamba2's kernels; this module only
orders the calls and allocates the packed buffers with torch.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import (causal_conv1d, decode_step, gated_rmsnorm, pack_rows, padded_spans, ssd_scan,
               ssd_scan_workspace_bytes, unpack_rows)


@dataclass
class Mamba2Weights:
    """The path's parameters (device tensors): conv taps and bias, A_log, dt_bias, D, norm weight."""
    conv_w: torch.Tensor
    conv_b: torch.Tensor
    A_log: torch.Tensor
    dt_bias: torch.Tensor
    D: torch.Tensor
    norm_w: torch.Tensor
    norm_groups: int = 1
    eps: float = 1e-5


class Mamba2Cache:
    """HF-style view of one batch's recurrent state, held in slots of the pools.

    ``conv_state`` is ``[batch, conv_dim, kernel - 1]`` (channels first, oldest input
    first), ``ssm_state`` is ``[batch, heads, headdim, d_state]`` fp32; both are
    gathered from the pools at the batch's slots. ``has_previous_state`` turns true
    after the first forward; ``seqlen_offset[b]`` counts the tokens sequence b has
    seen, which is the position of its next token.
    """

    def __init__(self, conv_pool: torch.Tensor, ssm_pool: torch.Tensor, slots):
        self.conv_pool, self.ssm_pool = conv_pool, ssm_pool
        self.slots = [int(s) for s in slots]
        self.has_previous_state = False
        self.seqlen_offset = [0] * len(self.slots)

    def _idx(self):
        return torch.tensor(self.slots, dtype=torch.long, device=self.ssm_pool.device)

    @property
    def conv_state(self) -> torch.Tensor:
        return self.conv_pool[self._idx()].transpose(1, 2)

    @property
    def ssm_state(self) -> torch.Tensor:
        return self.ssm_pool[self._idx()]


def forward(xBC, z, dt, weights: Mamba2Weights, dims, cache: Mamba2Cache,
            attention_mask: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Prefill (or a multi-token continuation) of a padded batch; returns ``[batch, seqlen, d_inner]``.

    ``xBC`` ``[batch, seqlen, conv_dim]``, ``z`` ``[batch, seqlen, d_inner]``, ``dt``
    ``[batch, seqlen, heads]`` are device tensors; ``attention_mask`` ``[batch, seqlen]``
    is on the host (None: every position is a token). A sequence starts from zero state
    on the cache's first forward and resumes its slot afterwards.
    """
    batch, seqlen = int(xBC.shape[0]), int(xBC.shape[1])
    if len(cache.slots) != batch:
        raise ValueError(f"cache holds {len(cache.slots)} sequences, the batch {batch}")
    if attention_mask is None:
        attention_mask = torch.ones((batch, seqlen), dtype=torch.uint8)
    cu, first = padded_spans(attention_mask.cpu())
    rows = cu[-1]
    dev, act = xBC.device, xBC.dtype
    fresh = [0 if cache.has_previous_state else 1] * batch
    x_p = torch.empty((rows, xBC.shape[2]), dtype=act, device=dev)
    z_p = torch.empty((rows, z.shape[2]), dtype=act, device=dev)
    dt_p = torch.empty((rows, dt.shape[2]), dtype=act, device=dev)
    for dst, src in ((x_p, xBC), (z_p, z), (dt_p, dt)):
        pack_rows(dst, src.contiguous(), cu, first, stream=stream)
    w = weights
    xbc_p = torch.empty_like(x_p)
    causal_conv1d(xbc_p, x_p, w.conv_w, w.conv_b, cache.conv_pool, cu, cache.slots, fresh, stream=stream)
    y_p = torch.empty_like(z_p)
    ws_bytes = ssd_scan_workspace_bytes(dims, rows, cu, cache.slots, fresh)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev) if ws_bytes else None
    ssd_scan(y_p, xbc_p, dt_p, w.A_log, w.dt_bias, w.D, cache.ssm_pool, dims, cu, cache.slots, fresh,
             workspace=ws, stream=stream)
    out_p = torch.empty_like(z_p)
    gated_rmsnorm(out_p, y_p, z_p, w.norm_w, w.norm_groups, w.eps, stream=stream)
    out = torch.empty((batch, seqlen, z.shape[2]), dtype=act, device=dev)
    unpack_rows(out, out_p, cu, first, stream=stream)
    cache.has_previous_state = True
    cache.seqlen_offset = [o + cu[b + 1] - cu[b] for b, o in enumerate(cache.seqlen_offset)]
    return out


def decode(xBC, z, dt, weights: Mamba2Weights, dims, cache: Mamba2Cache, stream=None) -> torch.Tensor:
    """One token per sequence (``[batch, conv_dim]`` etc., or with a length-1 middle axis);
    returns ``[batch, d_inner]`` and advances every sequence's position by one."""
    if xBC.dim() == 3:
        xBC, z, dt = xBC[:, 0], z[:, 0], dt[:, 0]
    batch = int(xBC.shape[0])
    fresh = [0 if cache.has_previous_state else 1] * batch
    w = weights
    out = torch.empty((batch, z.shape[1]), dtype=z.dtype, device=z.device)
    decode_step(out, xBC.contiguous(), z.contiguous(), dt.contiguous(), w.conv_w, w.conv_b, w.A_log, w.dt_bias,
                w.D, w.norm_w, w.norm_groups, w.eps, cache.conv_pool, cache.ssm_pool, dims, cache.slots, fresh,
                stream=stream)
    cache.has_previous_state = True
    cache.seqlen_offset = [o + 1 for o in cache.seqlen_offset]
    return out

