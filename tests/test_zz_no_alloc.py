"""The scan entry point that allocates nothing, through the C ABI.

mamba2_ssd_scan_static_scratch serves callers that cannot allocate device
memory when they call the scan (a server whose allocator has given all device
memory to its pools, a plugin host that exposes only input and output buffers,
a latency-critical loop that cannot afford an allocation's synchronisation):
it uses a fixed scratch array inside the library instead of a caller-provided
workspace. These tests check that it gives the workspace entry point's results
on two calls in a row (different batches, so stale scratch contents from the
first call cannot pass for the second), and that a batch needing more scratch
than the array holds is rejected before anything runs.

This file sorts last so that a run that stops at the first failure has run
every other test before it.
"""
import ctypes

import pytest
import torch

import selective_scan_gb300 as ss
import workloads as W
from tests.gpu_util import device, gpu_conv
from tests.util import STATE_PREFILL_REL_L2, assert_bits_equal, check_act, rel_l2

pytestmark = pytest.mark.gpu

MAX_SCRATCH = 32 << 20  # MAMBA2_STATIC_SCAN_SCRATCH_BYTES


def _static_fn():
    lib = ss.library()
    fn = lib.mamba2_ssd_scan_static_scratch
    p, i32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [p, p, p, p, p, p, p, i32, i32, ctypes.POINTER(ss.Dims), ctypes.c_int,
                   ctypes.POINTER(ss.RecurrentBatch), p]
    fn.restype = ctypes.c_int
    return fn


def _run_static(fn, y, xbc, dt, params, ssm, dims, batch):
    d = ss.Dims(dims.heads, dims.headdim, dims.d_state, dims.ngroups, dims.conv_kernel)
    stream = torch.cuda.current_stream().cuda_stream
    return fn(y.data_ptr(), xbc.data_ptr(), dt.data_ptr(), params[0].data_ptr(), params[1].data_ptr(),
              params[2].data_ptr(), ssm.data_ptr(), ssm.shape[0], xbc.shape[0], ctypes.byref(d), ss.BF16,
              batch.ref(), stream)


def _compare_once(fn, wl, dev):
    p, b, d = wl.params, wl.batch, wl.dims
    batch = ss.Batch(b.cu_seqlens, b.slots, b.fresh)
    need = ss.ssd_scan_workspace_bytes(d, b.rows, batch=batch)
    # the dt' region alone is rows x heads floats; anything beyond it is the
    # segments' states and decays, which only a segmented batch has
    dtp_bytes = b.rows * d.heads * 4
    assert dtp_bytes < need <= MAX_SCRATCH, (
        f"workload should be segmented (scratch beyond the {dtp_bytes}-byte dt' region) and fit the array "
        f"({need} bytes)")
    xbc, _ = gpu_conv(wl, dev)
    dt = wl.dt.to(dev)
    prm = [p.A_log.to(dev), p.dt_bias.to(dev), p.D.to(dev)]
    # the workspace entry point
    ssm_ref = wl.ssm_state.to(dev)
    y_ref = torch.empty((b.rows, d.d_inner), dtype=torch.bfloat16, device=dev)
    ss.ssd_scan(y_ref, xbc, dt, *prm, ssm_ref, d, batch=batch)
    # the static-scratch entry point
    ssm = wl.ssm_state.to(dev)
    y = torch.full((b.rows, d.d_inner), float("nan"), dtype=torch.bfloat16, device=dev)
    st = _run_static(fn, y, xbc, dt, prm, ssm, d, batch)
    assert st == ss.OK, ss.status_string(st)
    torch.cuda.synchronize()
    check_act(y.cpu(), y_ref.cpu().double(), "static-scratch scan output")
    idx = torch.tensor(b.slots)
    assert rel_l2(ssm.cpu()[idx], ssm_ref.cpu()[idx]) <= STATE_PREFILL_REL_L2
    others = [i for i in range(ssm.shape[0]) if i not in set(b.slots)]
    if others:
        o = torch.tensor(others)
        assert_bits_equal(ssm.cpu()[o], wl.ssm_state[o], "slots outside the batch")


def test_static_scratch_matches_workspace_entry_twice():
    dev = device()
    fn = _static_fn()
    _compare_once(fn, W.prefill_130m(), dev)  # first call on this device: address look-up
    _compare_once(fn, W.varlen_130m(), dev)   # second call: the scratch holds the first call's contents


def test_static_scratch_rejects_oversized_batch():
    dev = device()
    fn = _static_fn()
    d = W.DIMS_48H
    # 199 one-chunk runs and one 65536-token run: many segments' worth of state
    lengths = [64] * 199 + [65536]
    total = sum(lengths)
    xbc = torch.zeros((total, d.conv_dim), dtype=torch.bfloat16, device=dev)
    dt = torch.zeros((total, d.heads), dtype=torch.bfloat16, device=dev)
    prm = [torch.zeros(d.heads, device=dev) for _ in range(3)]
    ssm = torch.zeros((200, d.heads, d.headdim, d.d_state), device=dev)
    y = torch.full((total, d.d_inner), 7.0, dtype=torch.bfloat16, device=dev)
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    batch = ss.Batch(cu, list(range(200)), [1] * 200)
    assert ss.ssd_scan_workspace_bytes(d, total, batch=batch) > MAX_SCRATCH
    st = _run_static(fn, y, xbc, dt, prm, ssm, d, batch)
    assert st == ss.ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert (y.cpu() == 7.0).all() and (ssm.cpu() == 0).all()
