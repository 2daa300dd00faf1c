"""The projections around the path (gllm PR #85 "feat(backend): Mamba2 ops, with CPU
reference implementations", "Ops": the model splits in_proj into z, xBC and dt) and the
layer chain in_proj -> conv -> scan -> norm -> out_proj.

Oracle pins: with one-hot weight rows the product picks input columns exactly, which
fixes the weight's orientation (output features x input features) and the split order
z | xBC | dt. GPU: the tcgen05 GEMMs against the oracle's double product (each output
within 2e-2 + a bf16 half-ulp of it), with ragged rows, a K that is not a multiple of
the 64-wide k-block, and sampled rows of the 65 536-token layer.
"""
import ctypes

import pytest
import torch

import oracle
import selective_scan_gb300 as ss
import workloads as W
from tests.util import STATE_PREFILL_REL_L2, check_act

FAKE = [0x10000 * (i + 1) for i in range(6)]


def _one_hot(rows, cols, g):
    pick = torch.randint(0, cols, (rows,), generator=g)
    w = torch.zeros((rows, cols))
    w[torch.arange(rows), pick] = 1.0
    return w, pick


def test_oracle_in_proj_one_hot_split():
    g = torch.Generator("cpu").manual_seed(51)
    dims, d_model = (4, 16, 16, 2), 24
    H, P, N, G = dims
    d_inner, conv_dim = H * P, H * P + 2 * G * N
    w, pick = _one_hot(d_inner + conv_dim + H, d_model, g)
    hidden = torch.randn((5, d_model), generator=g)
    z, x, dt = oracle.in_proj(hidden, w, dims)
    full = hidden.double()[:, pick]
    assert torch.equal(z, full[:, :d_inner])
    assert torch.equal(x, full[:, d_inner:d_inner + conv_dim])
    assert torch.equal(dt, full[:, d_inner + conv_dim:])


def test_oracle_out_proj_one_hot():
    g = torch.Generator("cpu").manual_seed(52)
    w, pick = _one_hot(12, 40, g)
    x = torch.randn((3, 40), generator=g)
    assert torch.equal(oracle.out_proj(x, w), x.double()[:, pick])
    # and a closed form: all-ones weights sum each row
    assert torch.allclose(oracle.out_proj(x, torch.ones((2, 40))), x.double().sum(1, keepdim=True).expand(3, 2))


def test_projection_host_rejections(product_lib):
    lib = product_lib
    d = ss.Dims(24, 64, 128, 1, 4)
    call_in = lambda act=ss.BF16, d_model=768, rows=4, z=FAKE[0]: lib.mamba2_in_proj(
        z, FAKE[1], FAKE[2], FAKE[3], FAKE[4], rows, d_model, ctypes.byref(d), act, None)
    assert call_in(act=ss.F32) == ss.ERR_NOT_IMPLEMENTED
    assert call_in(d_model=100) == ss.ERR_NOT_IMPLEMENTED
    assert call_in(d_model=0) == ss.ERR_INVALID_ARGUMENT
    assert call_in(z=None) == ss.ERR_INVALID_ARGUMENT
    assert call_in(z=FAKE[0] + 8) == ss.ERR_INVALID_ARGUMENT
    assert call_in(rows=-1) == ss.ERR_INVALID_ARGUMENT
    assert call_in(rows=0) == ss.OK
    d_odd = ss.Dims(4, 16, 16, 2, 4)  # 4 heads: dt rows of 8 bytes, no 16-byte stores
    assert lib.mamba2_in_proj(*FAKE[:5], 4, 64, ctypes.byref(d_odd), ss.BF16, None) == ss.ERR_NOT_IMPLEMENTED
    call_out = lambda act=ss.BF16, d_inner=1536, d_model=768, out=FAKE[0]: lib.mamba2_out_proj(
        out, FAKE[1], FAKE[2], 4, d_inner, d_model, act, None)
    assert call_out(act=ss.F32) == ss.ERR_NOT_IMPLEMENTED
    assert call_out(d_inner=1540) == ss.ERR_NOT_IMPLEMENTED
    assert call_out(out=None) == ss.ERR_INVALID_ARGUMENT


# ---------------------------------------------------------------- GPU

def _gpu_in_proj(hidden, w_in, dims, dev):
    rows = hidden.shape[0]
    z = torch.empty((rows, dims.d_inner), dtype=torch.bfloat16, device=dev)
    x = torch.empty((rows, dims.conv_dim), dtype=torch.bfloat16, device=dev)
    dt = torch.empty((rows, dims.heads), dtype=torch.bfloat16, device=dev)
    ss.in_proj(z, x, dt, hidden.to(dev), w_in.to(dev), dims)
    torch.cuda.synchronize()
    return z.cpu(), x.cpu(), dt.cpu()


@pytest.mark.gpu
@pytest.mark.parametrize("dims,d_model,rows", [
    (W.DIMS_130M, 768, 300),   # 3 row tiles (44-row tail), 14 column tiles (24-column tail)
    (W.DIMS_130M, 200, 129),   # K = 200: the last k-block is 8 wide, zero-filled past it
    (W.DIMS_48H, 1536, 1),
])
def test_in_proj_matches_oracle(dims, d_model, rows):
    from tests.gpu_util import device
    dev = device()
    g = torch.Generator("cpu").manual_seed(53)
    w_in, _ = W.draw_proj(g, dims, d_model)
    hidden = torch.randn((rows, d_model), generator=g).to(torch.bfloat16)
    z, x, dt = _gpu_in_proj(hidden, w_in, dims, dev)
    rz, rx, rdt = oracle.in_proj(hidden, w_in, dims.tuple4())
    check_act(z, rz, "in_proj z")
    check_act(x, rx, "in_proj xBC")
    check_act(dt, rdt, "in_proj dt")


@pytest.mark.gpu
@pytest.mark.parametrize("d_inner,d_model,rows", [(1536, 768, 300), (3072, 200, 257), (64, 1536, 5)])
def test_out_proj_matches_oracle(d_inner, d_model, rows):
    from tests.gpu_util import device
    dev = device()
    g = torch.Generator("cpu").manual_seed(54)
    w_out = (torch.randn((d_model, d_inner), generator=g) * d_inner ** -0.5).to(torch.bfloat16)
    x = torch.randn((rows, d_inner), generator=g).to(torch.bfloat16)
    out = torch.empty((rows, d_model), dtype=torch.bfloat16, device=dev)
    ss.out_proj(out, x.to(dev), w_out.to(dev))
    torch.cuda.synchronize()
    check_act(out.cpu(), oracle.out_proj(x, w_out), "out_proj")


@pytest.mark.gpu
def test_in_proj_65536_rows_sampled():
    """The 48-head layer's in_proj over 65 536 rows (d_model 1536), 64 sampled rows
    against the oracle."""
    from tests.gpu_util import device
    dev = device()
    dims, d_model, rows = W.DIMS_48H, 1536, 65536
    g = torch.Generator("cpu").manual_seed(55)
    w_in, _ = W.draw_proj(g, dims, d_model)
    hidden = torch.randn((rows, d_model), generator=g).to(torch.bfloat16)
    z, x, dt = _gpu_in_proj(hidden, w_in, dims, dev)
    pick = torch.randperm(rows, generator=g)[:64]
    pick[0], pick[1] = 0, rows - 1
    rz, rx, rdt = oracle.in_proj(hidden[pick], w_in, dims.tuple4())
    check_act(z[pick], rz, "z (sampled rows)")
    check_act(x[pick], rx, "xBC (sampled rows)")
    check_act(dt[pick], rdt, "dt (sampled rows)")


@pytest.mark.gpu
def test_layer_chain_matches_oracle():
    """hidden -> in_proj -> conv -> scan -> norm -> out_proj, three packed runs (one
    resuming), then a decode step: each GEMM against the oracle on the GPU chain's own
    input, the whole chain against the oracle's chain in aggregate."""
    from selective_scan_gb300 import layer, padded
    from tests.gpu_util import device, slot_rel_l2
    from tests.util import rel_l2
    dev = device()
    dims, d_model = W.DIMS_130M, 768
    H, P, N, G = dims.tuple4()
    wl = W.make_prefill("layer", 56, dims, [300, 77, 500], torch.bfloat16, 8, [1, 0, 1])
    p, b = wl.params, wl.batch
    g = torch.Generator("cpu").manual_seed(57)
    w_in, w_out = W.draw_proj(g, dims, d_model)
    hidden = torch.randn((b.rows, d_model), generator=g).to(torch.bfloat16)
    wts = padded.Mamba2Weights(*[t.to(dev) for t in (p.conv_w, p.conv_b, p.A_log, p.dt_bias, p.D, p.norm_w)],
                               p.norm_groups, p.eps)
    L = layer.Mamba2Layer(w_in.to(dev), w_out.to(dev), wts, dims)
    conv_g, ssm_g = wl.conv_state.to(dev), wl.ssm_state.to(dev)
    out = L.prefill(hidden.to(dev), conv_g, ssm_g, b.cu_seqlens, b.slots, b.fresh)
    torch.cuda.synchronize()
    # the oracle's chain
    z64, x64, dt64 = oracle.in_proj(hidden, w_in, (H, P, N, G))
    z, x, dt = (t.to(torch.bfloat16) for t in (z64, x64, dt64))
    conv_o, ssm_o = wl.conv_state.clone(), wl.ssm_state.clone()
    xbc, _ = oracle.causal_conv1d(x.contiguous(), p.conv_w, p.conv_b, conv_o, b.cu_seqlens, b.slots, b.fresh)
    y, _ = oracle.ssd_scan(xbc, dt.contiguous(), p.A_log, p.dt_bias, p.D, ssm_o, (H, P, N, G), b.cu_seqlens,
                           b.slots, b.fresh)
    gn, _ = oracle.gated_rmsnorm(y, z.contiguous(), p.norm_w, p.norm_groups, p.eps)
    out64 = oracle.out_proj(gn, w_out)
    assert rel_l2(out.cpu(), out64) <= 1e-2, rel_l2(out.cpu(), out64)
    assert slot_rel_l2(ssm_g, ssm_o, b.slots) <= STATE_PREFILL_REL_L2
    # a decode step through the layer
    h1 = torch.randn((3, d_model), generator=g).to(torch.bfloat16)
    o1 = L.decode(h1.to(dev), conv_g, ssm_g, b.slots)
    z1, x1, dt1 = (t.to(torch.bfloat16) for t in oracle.in_proj(h1, w_in, (H, P, N, G)))
    g1, _ = oracle.decode_step(x1.contiguous(), z1.contiguous(), dt1.contiguous(), p.conv_w, p.conv_b, p.A_log,
                               p.dt_bias, p.D, p.norm_w, p.norm_groups, p.eps, conv_o, ssm_o, (H, P, N, G),
                               b.slots, [0] * 3)
    torch.cuda.synchronize()
    assert rel_l2(o1.cpu(), oracle.out_proj(g1, w_out)) <= 1e-2
