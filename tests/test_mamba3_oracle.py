"""Pins of the Mamba-3 SISO forward oracle (page "Mamba-3 SISO Long-Ragged
Multi-Chunk Joint States Full VJP", the reference's forward steps 1-7), on CPU.

What pins what:
- With no rotation (angles 0), p = 1 (trap large: the shifted weight vanishes) and
  no biases, the operator is the Mamba2 selective scan with C = q, B = k, x = v,
  log-decay adt and weight dt; the Mamba2 oracle (itself pinned to the gllm
  page's worked values) must agree. This fixes the decayed QK recurrence, y after
  the update, the head-wise D skip, the GQA expansion and the z * sigmoid(z) gate.
- Two tokens with one rotary pair, worked by hand with 2x2 rotation matrices: the
  rotation's direction, the cumulative angle (current token included), the pair
  (0, 1) and the unrotated columns, and that q and k share the angle.
- The final angle is the cumulative sum mod 2 pi.
- p = 0 (trap very negative): every token's weight is the next token's dt, so the
  operator must equal the "previous token" recurrence g_t = exp(adt_t)(g_{t-1} +
  dt_t k^_{t-1} v_{t-1}), y_t = q^_t . g_t + d v_t, computed here by brute force:
  this fixes the shift's direction, the zero after the last token, and that the
  correction removes exactly the current token's share of the shifted weight.
  (The page names the correction without its form; this repository's reading is
  the one tested, so that part's parity is pinned to the reading, not the page.)
- Packed sequences are independent (state, angle and shift reset at boundaries),
  and an empty sequence has zero final states.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W

BF = torch.bfloat16


def _small(seed, lengths, H=2, P=3, N=8, R=2):
    return W.mamba3_batch(seed=seed, lengths=lengths, heads=H, headdim=P, d_state=N, rot_dim=R)


def _silu64(z):
    z = z.double()
    return z / (1.0 + torch.exp(-z))


def test_reduces_to_mamba2_scan():
    # fp32 Mamba2 activations hold the bf16 values exactly
    b = _small(1, [37, 0, 20], H=3, P=4, N=8, R=2)
    T, H, P, N = b.rows, b.heads, b.headdim, b.d_state
    g = torch.Generator().manual_seed(11)
    dt_in = torch.randn((T, H), generator=g)
    A_log = torch.log(torch.rand(H, generator=g) * 15 + 1)
    dtp = torch.nn.functional.softplus(dt_in.double())          # dt' of the Mamba2 scan (dt_bias 0)
    b.dt = dtp.float()
    b.adt = (-torch.exp(A_log.double()) * dtp).float()
    b.angles = torch.zeros_like(b.angles)
    b.trap = torch.full_like(b.trap, 40.0)                      # p = sigmoid(40) = 1 in double
    b.q_bias.zero_()
    b.k_bias.zero_()
    out, fa, fs, fk, fv, out64 = oracle.mamba3_siso_forward(*b.tensors(), b.cu_seqlens)
    # the Mamba2 oracle on xbc = [v | B = k | C = q] (one group), fp32 activations
    xbc = torch.cat([b.v.reshape(T, H * P), b.k, b.q], dim=1).float().contiguous()
    ssm = torch.zeros((3, H, P, N))
    _, y64 = oracle.ssd_scan(xbc, dt_in.contiguous(), A_log.contiguous(), torch.zeros(H), b.d.contiguous(), ssm,
                             (H, P, N, 1), b.cu_seqlens, [0, 1, 2], [1, 1, 1])
    ref = y64.reshape(T, H, P) * _silu64(b.z)
    assert torch.allclose(out64, ref, rtol=1e-5, atol=1e-9), (out64 - ref).abs().max()
    # final SSM state: the Mamba2 oracle's slot (state rounded to fp32 each token)
    assert torch.allclose(fs, ssm, rtol=1e-5, atol=1e-7)
    assert (fs[1] == 0).all() and (fk[1] == 0).all() and (fv[1].float() == 0).all() and (fa[1].float() == 0).all()


def _rot(x01, phi):
    c, s = math.cos(phi), math.sin(phi)
    return np.array([c * x01[0] - s * x01[1], s * x01[0] + c * x01[1]])


def test_two_tokens_one_rotary_pair_by_hand():
    b = _small(2, [2], H=1, P=1, N=4, R=1)
    b.q = torch.tensor([[1.0, 2.0, 0.5, -1.0], [0.25, -1.5, 2.0, 1.0]], dtype=BF)
    b.k = torch.tensor([[-0.5, 1.0, 1.5, 0.75], [2.0, 0.5, -1.0, 0.25]], dtype=BF)
    b.v = torch.tensor([[[3.0]], [[-2.0]]], dtype=BF)
    b.z = torch.tensor([[[1.5]], [[-0.75]]], dtype=BF)
    b.dt = torch.tensor([[0.5], [0.25]])
    b.adt = torch.tensor([[-0.3], [-0.7]])
    b.trap = torch.full((2, 1), 40.0, dtype=BF)
    b.angles = torch.tensor([[0.75], [-1.25]], dtype=BF)
    b.q_bias.zero_()
    b.k_bias.zero_()
    b.d = torch.tensor([0.5])
    out, fa, fs, fk, fv, out64 = oracle.mamba3_siso_forward(*b.tensors(), b.cu_seqlens)
    q, k = b.q.double().numpy(), b.k.double().numpy()
    th = [math.tanh(0.75) * math.pi, math.tanh(-1.25) * math.pi]
    phi0 = (th[0] * 0.5) % (2 * math.pi)
    phi1 = (th[0] * 0.5 + th[1] * 0.25) % (2 * math.pi)
    qh = [np.concatenate([_rot(q[0, :2], phi0), q[0, 2:]]), np.concatenate([_rot(q[1, :2], phi1), q[1, 2:]])]
    kh = [np.concatenate([_rot(k[0, :2], phi0), k[0, 2:]]), np.concatenate([_rot(k[1, :2], phi1), k[1, 2:]])]
    v = [3.0, -2.0]
    a1 = float(b.adt[1, 0])  # -0.7 as stored (fp32)
    # p = 1: each token's weight is its own dt; no shifted part, no correction
    y0 = 0.5 * float(qh[0] @ kh[0]) * v[0] + 0.5 * v[0]
    y1 = math.exp(a1) * 0.5 * float(qh[1] @ kh[0]) * v[0] + 0.25 * float(qh[1] @ kh[1]) * v[1] + 0.5 * v[1]
    gate = lambda zz: zz / (1.0 + math.exp(-zz))  # noqa: E731
    assert out64[0, 0, 0].item() == pytest.approx(y0 * gate(1.5), rel=1e-12)
    assert out64[1, 0, 0].item() == pytest.approx(y1 * gate(-0.75), rel=1e-12)
    # a rotation keeps q . k at equal angles
    assert float(qh[0] @ kh[0]) == pytest.approx(float(q[0] @ k[0]), rel=1e-12)
    # final states: the angle, the state, the last rotated k, the last v
    assert fa[0, 0, 0].item() == pytest.approx(phi1, abs=2 ** -7 * phi1)
    h = math.exp(a1) * 0.5 * np.outer([v[0]], kh[0]) + 0.25 * np.outer([v[1]], kh[1])
    assert np.allclose(fs[0, 0].double().numpy(), h, rtol=1e-6)
    assert np.allclose(fk[0, 0].double().numpy(), kh[1], rtol=1e-6)
    assert fv[0, 0, 0].item() == -2.0


def test_final_angle_is_taken_mod_2pi():
    b = _small(3, [3], H=1, P=1, N=2, R=1)
    b.angles = torch.full((3, 1), 20.0, dtype=BF)  # tanh(20) = 1 in double: theta = pi
    b.dt = torch.ones((3, 1))
    _, fa, _, _, _, _ = oracle.mamba3_siso_forward(*b.tensors(), b.cu_seqlens)
    assert fa[0, 0, 0].item() == pytest.approx(math.pi, rel=2 ** -8)  # 3 pi mod 2 pi


def _rotate_np(x, phi, R):
    y = x.copy()
    for i in range(R):
        c, s = math.cos(phi[i]), math.sin(phi[i])
        y[2 * i] = c * x[2 * i] - s * x[2 * i + 1]
        y[2 * i + 1] = s * x[2 * i] + c * x[2 * i + 1]
    return y


def test_p_zero_is_the_previous_token_rule():
    b = _small(4, [9, 5], H=2, P=3, N=6, R=2)
    b.trap = torch.full_like(b.trap, -40.0)  # p = 0: every weight is the next token's dt
    out, fa, fs, fk, fv, out64 = oracle.mamba3_siso_forward(*b.tensors(), b.cu_seqlens)
    H, P, N, R = b.heads, b.headdim, b.d_state, b.rot_dim
    q, k, v, z = (t.double().numpy() for t in (b.q, b.k, b.v, b.z))
    adt, dt, ang = b.adt.double().numpy(), b.dt.double().numpy(), b.angles.double().numpy()
    qb, kb, d = b.q_bias.double().numpy(), b.k_bias.double().numpy(), b.d.double().numpy()
    for s in range(2):
        r0, r1 = b.cu_seqlens[s], b.cu_seqlens[s + 1]
        for h in range(H):
            cum = np.zeros(R)
            g = np.zeros((P, N))
            prev = None  # (k^, v) of the previous token
            for t in range(r0, r1):
                cum += np.tanh(ang[t]) * math.pi * dt[t, h]
                phi = np.mod(cum, 2 * math.pi)
                qh = _rotate_np(q[t] + qb[h], phi, R)
                kh = _rotate_np(k[t] + kb[h], phi, R)
                g = math.exp(adt[t, h]) * (g + (dt[t, h] * np.outer(prev[1], prev[0]) if prev else 0.0))
                y = g @ qh + d[h] * v[t, h]
                ref = y * z[t, h] / (1.0 + np.exp(-z[t, h]))
                assert np.allclose(out64[t, h].numpy(), ref, rtol=1e-9, atol=1e-12), (s, h, t)
                prev = (kh, v[t, h])
            assert np.allclose(fs[s, h].double().numpy(), g, rtol=1e-6, atol=1e-7)


def test_packed_sequences_are_independent():
    b = _small(6, [13, 7, 21])
    whole = oracle.mamba3_siso_forward(*b.tensors(), b.cu_seqlens)
    for s in range(3):
        r0, r1 = b.cu_seqlens[s], b.cu_seqlens[s + 1]
        part = [t[r0:r1].contiguous() if t.dim() >= 1 and t.shape[0] == b.rows else t for t in b.tensors()]
        one = oracle.mamba3_siso_forward(*part, [0, r1 - r0])
        assert torch.equal(one[5], whole[5][r0:r1])
        for a, w in zip(one[1:5], whole[1:5]):
            assert torch.equal(a[0].view(torch.int16) if a.dtype == BF else a[0],
                               w[s].view(torch.int16) if w.dtype == BF else w[s])


def test_rejects_malformed_batches():
    b = _small(7, [4, 4])
    with pytest.raises(oracle.OracleError):
        oracle.mamba3_siso_forward(*b.tensors(), [0, 5, 4])
    bad = _small(7, [4], N=2, R=2)  # 2 R > N
    with pytest.raises(oracle.OracleError):
        oracle.mamba3_siso_forward(*bad.tensors(), bad.cu_seqlens)
