"""Pins for the CPU oracle: values and properties fixed by the pages and by
mathematics, independent of the oracle's own code.

Sources:
  gllm PR #85 "feat(backend): Mamba2 ops, with CPU reference implementations",
    sections "Ops", "CPU reference" and "Testing";
  InfiniLM PR #575 "feat(mamba2): integrate model loading and recurrent
    inference", section "Motivation" (state bytes per request).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.util import assert_bits_equal, bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(v) for v in line.split()])
    return np.array(rows)


def _silu(v):
    return v / (1.0 + math.exp(-v))


# ---------------------------------------------------------------------------
# T1: hand-worked conv pre-activations (section "Testing")
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kernel", [3, 4])
def test_conv_hand_worked(kernel):
    g = _golden("conv_hand_worked.txt")
    inputs, pre = g[:, 1], g[:, 2]
    T = len(inputs)
    x = torch.tensor(inputs, dtype=torch.float32).view(T, 1)
    taps = [1.0, 2.0, 3.0] if kernel == 3 else [0.0, 1.0, 2.0, 3.0]
    w = torch.tensor([taps], dtype=torch.float32)
    b = torch.tensor([0.5], dtype=torch.float32)
    state = torch.full((1, kernel - 1, 1), float("nan"))  # fresh: must not be read
    out, out64 = oracle.causal_conv1d(x, w, b, state, [0, T], [0], [1])
    want = np.array([_silu(v) for v in pre])
    np.testing.assert_allclose(out64[:, 0].numpy(), want, rtol=1e-15, atol=0)
    np.testing.assert_array_equal(out[:, 0].numpy(), want.astype(np.float32))
    # afterwards the slot holds the last kernel-1 inputs, oldest first
    np.testing.assert_array_equal(state[0, :, 0].numpy(), inputs[-(kernel - 1):].astype(np.float32))


def test_conv_hand_worked_rejects_flipped_taps():
    """The pin discriminates: reversed taps give different pre-activations."""
    g = _golden("conv_hand_worked.txt")
    x = torch.tensor(g[:, 1], dtype=torch.float32).view(-1, 1)
    w = torch.tensor([[3.0, 2.0, 1.0]])
    state = torch.zeros((1, 2, 1))
    _, out64 = oracle.causal_conv1d(x, w, torch.tensor([0.5]), state, [0, 5], [0], [1])
    assert abs(out64[0, 0].item() - _silu(3.5)) > 1.0


# ---------------------------------------------------------------------------
# T2: hand-worked scan (section "Testing")
# ---------------------------------------------------------------------------

def _tiny_scan_inputs(rows):
    xbc = torch.tensor([[r[1], r[2], r[3]] for r in rows], dtype=torch.float32)
    return xbc


def test_scan_hand_worked():
    g = _golden("scan_hand_worked.txt")
    xbc = _tiny_scan_inputs(g)
    T = xbc.shape[0]
    dt = torch.full((T, 1), math.log(math.e - 1.0), dtype=torch.float32)
    A_log = torch.zeros(1)
    dt_bias = torch.zeros(1)
    D = torch.tensor([0.5])
    state = torch.full((1, 1, 1, 1), float("nan"))
    y, y64 = oracle.ssd_scan(xbc, dt, A_log, dt_bias, D, state, (1, 1, 1, 1), [0, T], [0], [1])
    np.testing.assert_allclose(y64[:, 0].numpy(), g[:, 4], rtol=2e-7, atol=0)
    assert abs(g[1, 4] - (2.0 / math.e + 2.5)) < 1e-15
    # final state h = 2/e + 2 (fp32)
    np.testing.assert_allclose(state.item(), 2.0 / math.e + 2.0, rtol=1e-6)


# ---------------------------------------------------------------------------
# closed forms: conv = correlation (library routine), scan = dual quadratic form
# ---------------------------------------------------------------------------

def test_conv_matches_numpy_correlate():
    rng = np.random.default_rng(7)
    C, K, T = 5, 4, 37
    x = rng.standard_normal((T, C)).astype(np.float32)
    w = rng.standard_normal((C, K)).astype(np.float32)
    b = rng.standard_normal(C).astype(np.float32)
    hist = rng.standard_normal((K - 1, C)).astype(np.float32)
    state = torch.from_numpy(hist.copy()).view(1, K - 1, C)
    _, out64 = oracle.causal_conv1d(torch.from_numpy(x), torch.from_numpy(w), torch.from_numpy(b),
                                    state, [0, T], [0], [0])
    for c in range(C):
        u = np.concatenate([hist[:, c], x[:, c]]).astype(np.float64)
        pre = np.correlate(u, w[c].astype(np.float64), mode="valid") + float(b[c])
        want = pre / (1.0 + np.exp(-pre))
        np.testing.assert_allclose(out64[:, c].numpy(), want, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(state[0].numpy(), x[-(K - 1):])


def _dual_form(xbc, dt, A_log, dt_bias, D, h0, H, P, N, G):
    """y and the final state from the dual (attention-like) closed form:
    y_t = sum_{j<=t} (C_t . B_j) exp(s_t - s_j) dt'_j x_j + exp(s_t) C_t . h0 + D x_t
    with s the inclusive cumulative sum of -exp(A_log) dt'."""
    xbc = xbc.astype(np.float64)
    T = xbc.shape[0]
    y = np.zeros((T, H * P))
    hT = np.zeros((H, P, N))
    for h in range(H):
        g = h // (H // G)
        x = xbc[:, h * P:(h + 1) * P]
        B = xbc[:, H * P + g * N: H * P + (g + 1) * N]
        C = xbc[:, H * P + G * N + g * N: H * P + G * N + (g + 1) * N]
        dtp = np.logaddexp(0.0, dt[:, h].astype(np.float64) + float(dt_bias[h]))
        s = np.cumsum(-math.exp(float(A_log[h])) * dtp)
        L = np.tril(np.exp(s[:, None] - s[None, :]))
        M = (C @ B.T) * L * dtp[None, :]
        y[:, h * P:(h + 1) * P] = M @ x + np.exp(s)[:, None] * (C @ h0[h].T) + float(D[h]) * x
        w = np.exp(s[-1] - s) * dtp
        hT[h] = (x * w[:, None]).T @ B + math.exp(s[-1]) * h0[h]
    return y, hT


def test_scan_matches_dual_form():
    rng = np.random.default_rng(11)
    H, P, N, G, T = 4, 3, 5, 2, 50
    xbc = rng.standard_normal((T, H * P + 2 * G * N)).astype(np.float32)
    dt = rng.standard_normal((T, H)).astype(np.float32)
    A_log = np.log(rng.uniform(1, 16, H)).astype(np.float32)
    yb = rng.uniform(1e-3, 0.1, H)
    dt_bias = (yb + np.log(-np.expm1(-yb))).astype(np.float32)
    D = (1 + 0.1 * rng.standard_normal(H)).astype(np.float32)
    h0 = (0.1 * rng.standard_normal((H, P, N))).astype(np.float32)
    state = torch.from_numpy(h0.copy()).view(1, H, P, N)
    _, y64 = oracle.ssd_scan(torch.from_numpy(xbc), torch.from_numpy(dt), torch.from_numpy(A_log),
                             torch.from_numpy(dt_bias), torch.from_numpy(D), state,
                             (H, P, N, G), [0, T], [0], [0])
    y_ref, h_ref = _dual_form(xbc, dt, A_log, dt_bias, D, h0.astype(np.float64), H, P, N, G)
    # the oracle rounds its state to fp32 after every token: errors of a few fp32 ulps
    np.testing.assert_allclose(y64.numpy(), y_ref, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(state[0].numpy(), h_ref, rtol=1e-5, atol=1e-6)


# ---------------------------------------------------------------------------
# gated norm closed forms (section "Ops": gate before the norm, RMS per group)
# ---------------------------------------------------------------------------

def test_gated_norm_closed_form():
    # silu(50) == 50 in double, so v = 50 * x and out = x / rms(x).
    x = torch.tensor([[1.0, 2.0]])
    z = torch.tensor([[50.0, 50.0]])
    w = torch.ones(2)
    _, o64 = oracle.gated_rmsnorm(x, z, w, 1, 0.0)
    np.testing.assert_allclose(o64[0].numpy(), np.array([1.0, 2.0]) / math.sqrt(2.5), rtol=1e-15)
    # gate on z, not x: silu(z) at z = ln 3 is (3/4) ln 3; two channels with different z
    z2 = torch.tensor([[math.log(3.0), 50.0]], dtype=torch.float32)
    _, o64 = oracle.gated_rmsnorm(x, z2, w, 1, 0.0)
    v = np.array([1.0 * _silu(float(z2[0, 0])), 2.0 * 50.0])
    np.testing.assert_allclose(o64[0].numpy(), v / math.sqrt((v ** 2).mean()), rtol=1e-14)


def test_gated_norm_eps_weight_and_groups():
    # eps inside the square root; weight multiplies after the norm; groups independent
    x = torch.tensor([[0.5, -1.5, 3.0, 4.0]])
    z = torch.full((1, 4), 50.0)
    w = torch.tensor([2.0, 3.0, 0.5, -1.0])
    eps = 1.0
    _, o64 = oracle.gated_rmsnorm(x, z, w, 2, eps)
    v = 50.0 * x[0].double().numpy()
    g0 = v[:2] / math.sqrt((v[:2] ** 2).mean() + eps)
    g1 = v[2:] / math.sqrt((v[2:] ** 2).mean() + eps)
    np.testing.assert_allclose(o64[0].numpy(), np.concatenate([g0, g1]) * w.double().numpy(), rtol=1e-14)


def test_gated_norm_unit_rms_invariant():
    rng = np.random.default_rng(3)
    x = torch.from_numpy(rng.standard_normal((6, 32)).astype(np.float32))
    z = torch.from_numpy(rng.standard_normal((6, 32)).astype(np.float32))
    eps = 1e-5
    _, o64 = oracle.gated_rmsnorm(x, z, torch.ones(32), 4, eps)
    v = x.double() * torch.nn.functional.silu(z.double())
    for gi in range(4):
        sl = slice(gi * 8, (gi + 1) * 8)
        ms = (v[:, sl] ** 2).mean(dim=1)
        np.testing.assert_allclose((o64[:, sl] ** 2).mean(dim=1).numpy(), (ms / (ms + eps)).numpy(), rtol=1e-10)


# ---------------------------------------------------------------------------
# T3/T4: split == whole, bit-exact; resume from a saved state (sections
# "CPU reference" and "Testing")
# ---------------------------------------------------------------------------

def _tiny_wl(T=37, seed=5):
    return W.make_prefill("t", seed, W.DIMS_TINY, [T], torch.float32, 2, [1], slots=[1], norm_groups=2)


@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16])
def test_split_equals_whole_bit_exact(act):
    wl = W.make_prefill("t", 9, W.DIMS_TINY, [41], act, 2, [1], slots=[1], norm_groups=2)
    p, dims = wl.params, wl.dims
    T = wl.batch.rows
    conv_w, ssm_w = wl.conv_state.clone(), wl.ssm_state.clone()
    xbc_w, _ = oracle.causal_conv1d(wl.xBC, p.conv_w, p.conv_b, conv_w, [0, T], [1], [1])
    y_w, _ = oracle.ssd_scan(xbc_w, wl.dt, p.A_log, p.dt_bias, p.D, ssm_w, dims.tuple4(), [0, T], [1], [1])
    # pieces: one token (shorter than the conv history), two tokens, then the rest
    cuts = [0, 1, 3, 20, T]
    conv_s, ssm_s = wl.conv_state.clone(), wl.ssm_state.clone()
    xs, ys = [], []
    for i in range(len(cuts) - 1):
        a, b = cuts[i], cuts[i + 1]
        fr = [1 if i == 0 else 0]
        xb, _ = oracle.causal_conv1d(wl.xBC[a:b].contiguous(), p.conv_w, p.conv_b, conv_s, [0, b - a], [1], fr)
        y, _ = oracle.ssd_scan(xb, wl.dt[a:b].contiguous(), p.A_log, p.dt_bias, p.D, ssm_s, dims.tuple4(),
                               [0, b - a], [1], fr)
        xs.append(xb)
        ys.append(y)
    assert_bits_equal(torch.cat(xs), xbc_w, "conv output")
    assert_bits_equal(conv_s, conv_w, "conv state")
    assert_bits_equal(torch.cat(ys), y_w, "scan output")
    assert_bits_equal(ssm_s, ssm_w, "ssm state")


def test_resume_from_saved_state():
    wl = _tiny_wl(T=30)
    p, dims = wl.params, wl.dims
    xbc, _ = oracle.causal_conv1d(wl.xBC, p.conv_w, p.conv_b, wl.conv_state.clone(), [0, 30], [1], [1])
    st = wl.ssm_state.clone()
    y_all, _ = oracle.ssd_scan(xbc, wl.dt, p.A_log, p.dt_bias, p.D, st, dims.tuple4(), [0, 30], [1], [1])
    st1 = wl.ssm_state.clone()
    oracle.ssd_scan(xbc[:12].contiguous(), wl.dt[:12].contiguous(), p.A_log, p.dt_bias, p.D, st1,
                    dims.tuple4(), [0, 12], [1], [1])
    saved = st1[1].clone()
    # a different pool and slot, seeded with the saved state
    pool = torch.zeros((3,) + tuple(st1.shape[1:]))
    pool[2] = saved
    y_rest, _ = oracle.ssd_scan(xbc[12:].contiguous(), wl.dt[12:].contiguous(), p.A_log, p.dt_bias, p.D,
                                pool, dims.tuple4(), [0, 18], [2], [0])
    assert_bits_equal(y_rest, y_all[12:], "resumed output")
    assert_bits_equal(pool[2], st[1], "resumed final state")


# ---------------------------------------------------------------------------
# T5/T6: slot routing (section "Testing")
# ---------------------------------------------------------------------------

def test_swapped_slots_match_solo_runs():
    dims = W.DIMS_TINY
    g = torch.Generator().manual_seed(21)
    La, Lb = 9, 14
    xA, _, dtA = W.draw_tokens(g, La, dims, torch.float32)
    xB, _, dtB = W.draw_tokens(g, Lb, dims, torch.float32)
    p = W.draw_params(g, dims, 2)
    conv0, ssm0 = W.empty_pools(2, dims, torch.float32)
    # B resumes from slot 0; A is fresh on slot 1 (its slot holds the NaN sentinel)
    conv0[0] = torch.randn(conv0.shape[1:], generator=g)
    ssm0[0] = 0.1 * torch.randn(ssm0.shape[1:], generator=g)
    # batched: A on slot 1 (fresh), B on slot 0 (resume)
    conv_b, ssm_b = conv0.clone(), ssm0.clone()
    x = torch.cat([xA, xB])
    dt = torch.cat([dtA, dtB])
    cu = [0, La, La + Lb]
    xbc, _ = oracle.causal_conv1d(x, p.conv_w, p.conv_b, conv_b, cu, [1, 0], [1, 0])
    y, _ = oracle.ssd_scan(xbc, dt, p.A_log, p.dt_bias, p.D, ssm_b, dims.tuple4(), cu, [1, 0], [1, 0])
    # solo runs, each on its own pool
    cA, sA = conv0.clone(), ssm0.clone()
    xa, _ = oracle.causal_conv1d(xA, p.conv_w, p.conv_b, cA, [0, La], [1], [1])
    ya, _ = oracle.ssd_scan(xa, dtA, p.A_log, p.dt_bias, p.D, sA, dims.tuple4(), [0, La], [1], [1])
    cB, sB = conv0.clone(), ssm0.clone()
    xb, _ = oracle.causal_conv1d(xB, p.conv_w, p.conv_b, cB, [0, Lb], [0], [0])
    yb, _ = oracle.ssd_scan(xb, dtB, p.A_log, p.dt_bias, p.D, sB, dims.tuple4(), [0, Lb], [0], [0])
    assert_bits_equal(y, torch.cat([ya, yb]), "batched vs solo outputs")
    assert_bits_equal(conv_b[1], cA[1], "slot 1 conv")
    assert_bits_equal(conv_b[0], cB[0], "slot 0 conv")
    assert_bits_equal(ssm_b[1], sA[1], "slot 1 ssm")
    assert_bits_equal(ssm_b[0], sB[0], "slot 0 ssm")


def test_fresh_ignores_dirty_slot():
    wl = _tiny_wl(T=16)
    p, dims = wl.params, wl.dims
    dirty_c, dirty_s = wl.conv_state.clone(), wl.ssm_state.clone()
    dirty_c[1].fill_(float("nan"))
    dirty_s[1].fill_(float("nan"))
    xa, _ = oracle.causal_conv1d(wl.xBC, p.conv_w, p.conv_b, dirty_c, [0, 16], [1], [1])
    ya, _ = oracle.ssd_scan(xa, wl.dt, p.A_log, p.dt_bias, p.D, dirty_s, dims.tuple4(), [0, 16], [1], [1])
    assert torch.isfinite(ya).all() and torch.isfinite(dirty_s[1]).all() and torch.isfinite(dirty_c[1]).all()
    zero_c, zero_s = wl.conv_state.clone(), wl.ssm_state.clone()
    zero_c[1].zero_()
    zero_s[1].zero_()
    xb, _ = oracle.causal_conv1d(wl.xBC, p.conv_w, p.conv_b, zero_c, [0, 16], [1], [0])
    yb, _ = oracle.ssd_scan(xb, wl.dt, p.A_log, p.dt_bias, p.D, zero_s, dims.tuple4(), [0, 16], [1], [0])
    assert_bits_equal(ya, yb, "fresh vs zero-slot output")
    assert_bits_equal(dirty_s[1], zero_s[1], "fresh vs zero-slot state")


# ---------------------------------------------------------------------------
# T7: head -> group mapping (section "Testing")
# ---------------------------------------------------------------------------

def test_head_group_mapping_zeroed_group():
    wl = W.tiny()
    p, dims = wl.params, wl.dims
    H, P, N, G = dims.tuple4()
    xbc, _ = oracle.causal_conv1d(wl.xBC, p.conv_w, p.conv_b, wl.conv_state.clone(), [0, 64], [0], [1])
    y0, _ = oracle.ssd_scan(xbc, wl.dt, p.A_log, p.dt_bias, p.D, wl.ssm_state.clone(), dims.tuple4(),
                            [0, 64], [0], [1])
    z = xbc.clone()
    z[:, H * P + 1 * N: H * P + 2 * N] = 0.0  # B of group 1
    z[:, H * P + G * N + 1 * N: H * P + G * N + 2 * N] = 0.0  # C of group 1
    y1, _ = oracle.ssd_scan(z, wl.dt, p.A_log, p.dt_bias, p.D, wl.ssm_state.clone(), dims.tuple4(),
                            [0, 64], [0], [1])
    assert_bits_equal(y1[:, :2 * P], y0[:, :2 * P], "heads 0,1 untouched")
    for h in (2, 3):
        dx = (p.D[h].double() * xbc[:, h * P:(h + 1) * P].double()).float()
        assert_bits_equal(y1[:, h * P:(h + 1) * P], dx, f"head {h} = D*x")
    assert not torch.equal(y0[:, 2 * P:], y1[:, 2 * P:])


# ---------------------------------------------------------------------------
# T8: malformed batches rejected, nothing written (section "Ops")
# ---------------------------------------------------------------------------

BAD_BATCHES = [
    ("slot out of range", [0, 3, 7], [0, 2], oracle.ERR_SLOT_OUT_OF_RANGE),
    ("negative slot", [0, 3, 7], [-1, 0], oracle.ERR_SLOT_OUT_OF_RANGE),
    ("shared slot", [0, 3, 7], [1, 1], oracle.ERR_SLOT_SHARED),
    ("runs short of rows", [0, 3, 6], [0, 1], oracle.ERR_RUNS_DONT_COVER_ROWS),
    ("runs past rows", [0, 3, 8], [0, 1], oracle.ERR_RUNS_DONT_COVER_ROWS),
    ("non-monotone", [0, 5, 4], [0, 1], oracle.ERR_RUNS_DONT_COVER_ROWS),
    ("first boundary not 0", [1, 3, 7], [0, 1], oracle.ERR_RUNS_DONT_COVER_ROWS),
]


@pytest.mark.parametrize("name,cu,slots,status", BAD_BATCHES, ids=[b[0] for b in BAD_BATCHES])
def test_malformed_batches_rejected(name, cu, slots, status):
    dims = W.DIMS_TINY
    g = torch.Generator().manual_seed(1)
    x, _, dt = W.draw_tokens(g, 7, dims, torch.float32)
    p = W.draw_params(g, dims, 2)
    conv, ssm = W.empty_pools(2, dims, torch.float32)
    c0, s0 = conv.clone(), ssm.clone()
    assert oracle.validate_batch(cu, slots, 2, 7) == status
    with pytest.raises(oracle.OracleError) as e:
        oracle.causal_conv1d(x, p.conv_w, p.conv_b, conv, cu, slots, [0, 0])
    assert e.value.status == status
    with pytest.raises(oracle.OracleError) as e:
        oracle.ssd_scan(x, dt, p.A_log, p.dt_bias, p.D, ssm, dims.tuple4(), cu, slots, [0, 0])
    assert e.value.status == status
    assert_bits_equal(conv, c0, "conv pool untouched")
    assert_bits_equal(ssm, s0, "ssm pool untouched")


# ---------------------------------------------------------------------------
# T9: state bytes per request (InfiniLM PR #575, section "Motivation")
# ---------------------------------------------------------------------------

def test_state_size_130m():
    (layers, H, P, N, G, K, mib), = _golden("state_size_130m.txt")
    per_layer = oracle.state_bytes_per_layer(int(H), int(P), int(N), int(G), int(K), oracle.BF16)
    total = int(layers) * per_layer
    assert total == 24 * (24 * 64 * 128 * 4 + 1792 * 3 * 2)
    assert round(total / 2 ** 20, 2) == mib
    # the page's figure discriminates the readings: fp32 history or K columns miss it
    assert round(int(layers) * oracle.state_bytes_per_layer(24, 64, 128, 1, 5, oracle.BF16) / 2 ** 20, 2) != mib
    assert round(int(layers) * oracle.state_bytes_per_layer(24, 64, 128, 1, 4, oracle.F32) / 2 ** 20, 2) != mib


# ---------------------------------------------------------------------------
# decode step = the three ops on one token; decode steps = prefill token by token
# ---------------------------------------------------------------------------

def test_decode_steps_equal_prefill():
    dims = W.DIMS_TINY
    g = torch.Generator().manual_seed(13)
    steps, n = 5, 3
    x, z, dt = W.draw_tokens(g, steps * n, dims, torch.bfloat16)
    x, z, dt = x.view(steps, n, -1), z.view(steps, n, -1), dt.view(steps, n, -1)
    p = W.draw_params(g, dims, 2)
    conv, ssm = W.empty_pools(4, dims, torch.bfloat16)
    slots, fresh = [3, 0, 2], [0, 1, 0]
    W.fill_resumed_slots(g, conv, ssm, slots, fresh, torch.bfloat16)
    # decode
    cd, sd = conv.clone(), ssm.clone()
    outs, outs64 = [], []
    for t in range(steps):
        fr = fresh if t == 0 else [0, 0, 0]
        o_t, o64_t = oracle.decode_step(x[t].contiguous(), z[t].contiguous(), dt[t].contiguous(), p.conv_w,
                                        p.conv_b, p.A_log, p.dt_bias, p.D, p.norm_w, 2, p.eps, cd, sd,
                                        dims.tuple4(), slots, fr)
        outs.append(o_t)
        outs64.append(o64_t)
    # prefill of the same tokens, packed per sequence
    xs = torch.cat([x[:, i] for i in range(n)])
    zs = torch.cat([z[:, i] for i in range(n)])
    dts = torch.cat([dt[:, i] for i in range(n)])
    cu = [0, steps, 2 * steps, 3 * steps]
    cp, sp = conv.clone(), ssm.clone()
    xb, _ = oracle.causal_conv1d(xs, p.conv_w, p.conv_b, cp, cu, slots, fresh)
    y, _ = oracle.ssd_scan(xb, dts, p.A_log, p.dt_bias, p.D, sp, dims.tuple4(), cu, slots, fresh)
    o, o64 = oracle.gated_rmsnorm(y, zs, p.norm_w, 2, p.eps)
    dec = torch.stack(outs)  # [steps, n, d_inner]
    pre = torch.stack([o[i * steps:(i + 1) * steps] for i in range(n)], dim=1)
    assert_bits_equal(dec, pre, "decode outputs vs prefill")
    # the unrounded outputs too: the decode step hands back the norm's own values
    pre64 = torch.stack([o64[i * steps:(i + 1) * steps] for i in range(n)], dim=1)
    assert_bits_equal(torch.stack(outs64), pre64, "decode unrounded outputs vs prefill")
    assert_bits_equal(torch.stack(outs64).to(torch.bfloat16), dec, "decode output is its unrounded value rounded")
    assert_bits_equal(cd, cp, "conv pool")
    assert_bits_equal(sd, sp, "ssm pool")


def test_unnamed_slots_untouched():
    wl = W.make_prefill("v", 3, W.DIMS_TINY, [5, 9, 4], torch.bfloat16, 8, [1, 0, 1], norm_groups=2)
    p, dims, b = wl.params, wl.dims, wl.batch
    conv, ssm = wl.conv_state.clone(), wl.ssm_state.clone()
    xb, _ = oracle.causal_conv1d(wl.xBC, p.conv_w, p.conv_b, conv, b.cu_seqlens, b.slots, b.fresh)
    oracle.ssd_scan(xb, wl.dt, p.A_log, p.dt_bias, p.D, ssm, dims.tuple4(), b.cu_seqlens, b.slots, b.fresh)
    others = [s for s in range(8) if s not in b.slots]
    assert_bits_equal(conv[others], wl.conv_state[others], "unnamed conv slots")
    assert_bits_equal(ssm[others], wl.ssm_state[others], "unnamed ssm slots")
    assert torch.isfinite(ssm[b.slots]).all()
