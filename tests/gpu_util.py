"""Helpers for the GPU parity tests: run the CUDA path (through the C ABI) and
the oracle on the same seeded inputs."""
from __future__ import annotations

import pytest
import torch

import oracle
import selective_scan_gb300 as ss


def device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ss.library()  # raises if the library is not built
    return torch.device("cuda:0")


def gpu_conv(wl, dev, conv_state=None):
    p, b = wl.params, wl.batch
    x = wl.xBC.to(dev)
    conv = (wl.conv_state if conv_state is None else conv_state).to(dev)
    xbc = torch.empty_like(x)
    ss.causal_conv1d(xbc, x, p.conv_w.to(dev), p.conv_b.to(dev), conv, b.cu_seqlens, b.slots, b.fresh)
    return xbc, conv


def gpu_scan(wl, dev, xbc, ssm_state=None, cu=None, slots=None, fresh=None, dt=None):
    p, b, d = wl.params, wl.batch, wl.dims
    xbc = xbc.to(dev)
    ssm = (wl.ssm_state if ssm_state is None else ssm_state).to(dev)
    y = torch.empty((xbc.shape[0], d.d_inner), dtype=xbc.dtype, device=dev)
    ss.ssd_scan(y, xbc, (wl.dt if dt is None else dt).to(dev), p.A_log.to(dev), p.dt_bias.to(dev),
                p.D.to(dev), ssm, d, b.cu_seqlens if cu is None else cu, b.slots if slots is None else slots,
                b.fresh if fresh is None else fresh)
    return y, ssm


def gpu_norm(wl, dev, y, z=None):
    p = wl.params
    y = y.to(dev)
    out = torch.empty_like(y)
    ss.gated_rmsnorm(out, y, (wl.z if z is None else z).to(dev), p.norm_w.to(dev), p.norm_groups, p.eps)
    return out


def oracle_prefill(wl):
    p, b, d = wl.params, wl.batch, wl.dims
    conv, ssm = wl.conv_state.clone(), wl.ssm_state.clone()
    xbc, xbc64 = oracle.causal_conv1d(wl.xBC, p.conv_w, p.conv_b, conv, b.cu_seqlens, b.slots, b.fresh)
    y, y64 = oracle.ssd_scan(xbc, wl.dt, p.A_log, p.dt_bias, p.D, ssm, d.tuple4(), b.cu_seqlens, b.slots,
                             b.fresh)
    out, out64 = oracle.gated_rmsnorm(y, wl.z, p.norm_w, p.norm_groups, p.eps)
    return dict(xbc=xbc, xbc64=xbc64, y=y, y64=y64, out=out, out64=out64, conv=conv, ssm=ssm)


def slot_rel_l2(got_pool, ref_pool, slots):
    """Relative L2 of the named slots of a device pool against the oracle's CPU
    pool, gathered on each side and reduced in double on the device."""
    idx = torch.tensor(list(slots), dtype=torch.long)
    dev = got_pool.device
    g = got_pool[idx.to(dev)].double()
    r = ref_pool[idx].to(dev).double()
    den = torch.linalg.vector_norm(r).item()
    num = torch.linalg.vector_norm(g - r).item()
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / den
