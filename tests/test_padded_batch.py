"""Padded batches: attention mask -> RecurrentBatch, token gather and scatter, and the
padded forward with its HF-style cache view (page "Granite Mamba2 Inference
Optimization": the layer serves variable-length padded batches and returns a cache
exposing conv_state, ssm_state, has_previous_state and decode positions).

Reading: a padding position is not a token, and a row's tokens are one contiguous span.
Pins of the oracle's index maps: hand-worked spans, round-trip invariants, and the
equivalence with the masking form of padding (for left padding from an empty cache,
zeroing the padding's inputs and conv outputs and running each row whole gives
bit-identical outputs and states, because zero inputs keep a zero state at zero).
"""
import ctypes

import pytest
import torch

import oracle
import selective_scan_gb300 as ss
import workloads as W
from tests.util import STATE_PREFILL_REL_L2, assert_bits_equal, check_act

FAKE = [0x10000 * (i + 1) for i in range(4)]


def _plus_zero(t):
    """t with -0 replaced by +0 (NaN and every other value keep their bits)."""
    return torch.where(t == 0, torch.zeros_like(t), t)


# ---------------------------------------------------------------- oracle pins

def test_oracle_spans_hand_worked():
    mask = torch.tensor([[0, 0, 1, 1, 1], [1, 1, 1, 0, 0], [0, 0, 0, 0, 0], [1, 1, 1, 1, 1]])
    st, cu, first = oracle.padded_spans(mask)
    assert st == oracle.OK
    assert cu == [0, 3, 6, 6, 11] and first == [2, 0, 0, 0]
    for holes in ([[0, 1, 0, 1]], [[1, 0, 1]], [[1, 1, 1], [1, 0, 1]]):
        assert oracle.padded_spans(torch.tensor(holes))[0] == oracle.ERR_INVALID_ARGUMENT


def test_oracle_pack_unpack_round_trip():
    g = torch.Generator("cpu").manual_seed(41)
    lengths, seqlen = [7, 0, 3, 9], 9
    mask = torch.zeros((4, seqlen), dtype=torch.uint8)
    for b, L in enumerate(lengths):
        start = int(torch.randint(0, seqlen - L + 1, (1,), generator=g))
        mask[b, start:start + L] = 1
    x = torch.randn((4, seqlen, 5), generator=g)
    st, cu, first = oracle.padded_spans(mask)
    assert st == oracle.OK and cu[-1] == sum(lengths)
    packed = oracle.pack_rows(x, cu, first)
    assert packed.shape == (sum(lengths), 5)
    assert torch.equal(oracle.unpack_rows(packed, cu, first, seqlen), x * mask[:, :, None])
    assert torch.equal(oracle.pack_rows(oracle.unpack_rows(packed, cu, first, seqlen), cu, first), packed)


@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16])
def test_left_padding_is_zero_masking(act):
    dims = W.DIMS_TINY
    H, P, N, G = dims.tuple4()
    lengths, seqlen = [24, 13, 2], 24  # 2 < kernel - 1: the history keeps zeros
    xBC, z, dt, mask, p, conv0, ssm0, slots = W.padded_batch(42, lengths, seqlen, ["left"] * 3, dims, act,
                                                             norm_groups=2)
    # packed form
    st, cu, first = oracle.padded_spans(mask)
    conv_a, ssm_a = conv0.clone(), ssm0.clone()
    fresh = [1] * 3
    xbc, _ = oracle.causal_conv1d(oracle.pack_rows(xBC, cu, first), p.conv_w, p.conv_b, conv_a, cu, slots, fresh)
    y, _ = oracle.ssd_scan(xbc, oracle.pack_rows(dt, cu, first), p.A_log, p.dt_bias, p.D, ssm_a, (H, P, N, G), cu,
                           slots, fresh)
    out, _ = oracle.gated_rmsnorm(y, oracle.pack_rows(z, cu, first), p.norm_w, p.norm_groups, p.eps)
    out_a = oracle.unpack_rows(out, cu, first, seqlen)
    # masking form: each row whole, padding's inputs, dt and conv outputs zeroed
    conv_b, ssm_b = conv0.clone(), ssm0.clone()
    for b in range(3):
        m = mask[b].to(act)[:, None]
        row_cu = [0, seqlen]
        xb, _ = oracle.causal_conv1d((xBC[b] * m).contiguous(), p.conv_w, p.conv_b, conv_b, row_cu, [slots[b]], [1])
        xb = (xb * m).contiguous()
        yb, _ = oracle.ssd_scan(xb, (dt[b] * m).contiguous(), p.A_log, p.dt_bias, p.D, ssm_b, (H, P, N, G), row_cu,
                                [slots[b]], [1])
        ob, _ = oracle.gated_rmsnorm(yb, z[b].contiguous(), p.norm_w, p.norm_groups, p.eps)
        tok = mask[b] != 0
        assert_bits_equal(ob[tok], out_a[b][tok], f"row {b} output at its tokens")
        assert (ob[~tok] == 0).all() and (out_a[b][~tok] == 0).all()  # padding: zero (either sign)
    assert_bits_equal(ssm_b, ssm_a, "ssm pool")
    # a history shorter than kernel - 1 keeps the masked padding's zeros, -0 where a negative
    # input was masked: equal up to the sign of zero
    assert_bits_equal(_plus_zero(conv_b), _plus_zero(conv_a), "conv pool")


# ---------------------------------------------------------------- host ABI

def test_spans_match_oracle(product_lib):
    g = torch.Generator("cpu").manual_seed(43)
    for trial in range(40):
        batch, seqlen = int(torch.randint(1, 9, (1,), generator=g)), int(torch.randint(0, 12, (1,), generator=g))
        mask = torch.zeros((batch, seqlen), dtype=torch.uint8)
        for b in range(batch):
            L = int(torch.randint(0, seqlen + 1, (1,), generator=g))
            s0 = int(torch.randint(0, seqlen - L + 1, (1,), generator=g))
            mask[b, s0:s0 + L] = 1
        if trial % 4 == 3 and seqlen >= 3:  # a hole
            mask[0] = 0
            mask[0, 0] = mask[0, seqlen - 1] = 1
        st, cu, first = oracle.padded_spans(mask)
        if st == oracle.OK:
            assert ss.padded_spans(mask) == (cu, first)
        else:
            with pytest.raises(ss.Mamba2Error) as e:
                ss.padded_spans(mask)
            assert e.value.status == ss.ERR_INVALID_ARGUMENT


def test_pack_host_rejections(product_lib):
    lib = product_lib

    def call(fn, cu, first, batch=2, seqlen=4, width=16, dst=FAKE[0], src=FAKE[1]):
        c = (ctypes.c_int32 * len(cu))(*cu)
        f = (ctypes.c_int32 * max(len(first), 1))(*first)
        return fn(dst, src, batch, seqlen, width, c, f, None)

    for fn in (lib.mamba2_pack_rows, lib.mamba2_unpack_rows):
        assert call(fn, [0, 3, 5], [1, 3]) == ss.ERR_INVALID_ARGUMENT  # span 3..5 past row end 4
        assert call(fn, [1, 3, 5], [0, 0]) == ss.ERR_INVALID_ARGUMENT  # cu does not start at 0
        assert call(fn, [0, 3, 2], [0, 0]) == ss.ERR_INVALID_ARGUMENT  # decreasing
        assert call(fn, [0, 3, 5], [-1, 0]) == ss.ERR_INVALID_ARGUMENT
        assert call(fn, [0, 3, 5], [0, 0], width=0) == ss.ERR_INVALID_ARGUMENT
        assert call(fn, [0, 3, 5], [0, 0], dst=None) == ss.ERR_INVALID_ARGUMENT
        assert call(fn, [0, 3, 5], [0, 0], batch=-1) == ss.ERR_INVALID_ARGUMENT
        assert call(fn, [0, 0, 0], [0, 0], seqlen=0) == ss.OK  # nothing to move: no launch


# ---------------------------------------------------------------- GPU

@pytest.mark.gpu
@pytest.mark.parametrize("dtype,width", [(torch.bfloat16, 128), (torch.bfloat16, 3), (torch.float32, 5),
                                         (torch.uint8, 7)])
def test_pack_unpack_match_oracle(dtype, width):
    from tests.gpu_util import device
    dev = device()
    g = torch.Generator("cpu").manual_seed(44)
    lengths, seqlen = [37, 0, 12, 37, 5], 37
    mask = torch.zeros((5, seqlen), dtype=torch.uint8)
    for b, L in enumerate(lengths):
        s0 = 0 if b % 2 else seqlen - L
        mask[b, s0:s0 + L] = 1
    x = (torch.randn((5, seqlen, width), generator=g) * 50).to(dtype)
    cu, first = ss.padded_spans(mask)
    packed = torch.full((cu[-1], width), 7, dtype=dtype, device=dev)
    ss.pack_rows(packed, x.to(dev), cu, first)
    back = torch.full((5, seqlen, width), 9, dtype=dtype, device=dev)
    ss.unpack_rows(back, packed, cu, first)
    torch.cuda.synchronize()
    assert_bits_equal(packed.cpu(), oracle.pack_rows(x, cu, first), "packed rows")
    assert_bits_equal(back.cpu(), oracle.unpack_rows(oracle.pack_rows(x, cu, first), cu, first, seqlen),
                      "unpacked rows")


@pytest.mark.gpu
def test_padded_forward_and_cache_view():
    """The padded forward equals the packed ops on the same tokens bit for bit (the
    adapter only routes rows), with zeros at padding; the packed chain is within the
    chained tolerances of the oracle (each op's own parity is tested elsewhere)."""
    from selective_scan_gb300 import padded
    from tests.gpu_util import device, slot_rel_l2
    from tests.util import rel_l2
    dev = device()
    dims = W.DIMS_130M
    H, P, N, G = dims.tuple4()
    lengths, seqlen = [300, 171, 0, 45], 300
    sides = ["left", "right", "left", "right"]
    xBC, z, dt, mask, p, conv0, ssm0, slots = W.padded_batch(45, lengths, seqlen, sides, dims, torch.bfloat16,
                                                             num_slots=7)
    wts = [t.to(dev) for t in (p.conv_w, p.conv_b, p.A_log, p.dt_bias, p.D, p.norm_w)]
    w = padded.Mamba2Weights(*wts, p.norm_groups, p.eps)
    cache = padded.Mamba2Cache(conv0.to(dev), ssm0.to(dev), slots)
    assert not cache.has_previous_state
    out = padded.forward(xBC.to(dev), z.to(dev), dt.to(dev), w, dims, cache, attention_mask=mask)
    # the same tokens through the packed ops (rows gathered by the oracle's index map)
    st, cu, first = oracle.padded_spans(mask)
    fresh = [1] * 4
    xp, zp, dtp = (oracle.pack_rows(t, cu, first).to(dev) for t in (xBC, z, dt))
    conv_k, ssm_k = conv0.to(dev), ssm0.to(dev)
    xbc_k = torch.empty_like(xp)
    ss.causal_conv1d(xbc_k, xp, wts[0], wts[1], conv_k, cu, slots, fresh)
    y_k = torch.empty_like(zp)
    ss.ssd_scan(y_k, xbc_k, dtp, wts[2], wts[3], wts[4], ssm_k, dims, cu, slots, fresh)
    out_k = torch.empty_like(zp)
    ss.gated_rmsnorm(out_k, y_k, zp, wts[5], p.norm_groups, p.eps)
    torch.cuda.synchronize()
    got = out.cpu()
    assert_bits_equal(oracle.pack_rows(got, cu, first), out_k.cpu(), "padded forward vs packed ops")
    assert (got[mask == 0] == 0).all(), "padding positions must be zero"
    assert_bits_equal(cache.conv_pool.cpu(), conv_k.cpu(), "conv pool")
    assert_bits_equal(cache.ssm_pool.cpu(), ssm_k.cpu(), "ssm pool")
    # the chain against the oracle's chain
    conv_o, ssm_o = conv0.clone(), ssm0.clone()
    xbc, _ = oracle.causal_conv1d(xp.cpu(), p.conv_w, p.conv_b, conv_o, cu, slots, fresh)
    y, _ = oracle.ssd_scan(xbc, dtp.cpu(), p.A_log, p.dt_bias, p.D, ssm_o, (H, P, N, G), cu, slots, fresh)
    _, out64 = oracle.gated_rmsnorm(y, zp.cpu(), p.norm_w, p.norm_groups, p.eps)
    assert rel_l2(out_k.cpu(), out64) <= 1e-2
    assert_bits_equal(conv_k.cpu(), conv_o, "conv pool vs oracle")
    assert slot_rel_l2(ssm_k, ssm_o, slots) <= STATE_PREFILL_REL_L2
    # the HF-style view
    assert cache.has_previous_state and cache.seqlen_offset == lengths
    assert cache.conv_state.shape == (4, dims.conv_dim, dims.conv_kernel - 1)
    assert_bits_equal(cache.conv_state.cpu(), conv_o[torch.tensor(slots)].transpose(1, 2), "conv_state view")
    assert cache.ssm_state.shape == (4, H, P, N)
    assert_bits_equal(cache.ssm_state.cpu(), ssm_k.cpu()[torch.tensor(slots)], "ssm_state view")
    # two decode steps resume every slot (the empty sequence from its zeroed slot)
    g = torch.Generator("cpu").manual_seed(46)
    for step in range(2):
        dx, dz, ddt = (t.to(dev) for t in W.draw_tokens(g, 4, dims, torch.bfloat16))
        o = padded.decode(dx, dz, ddt, w, dims, cache)
        o_k = torch.empty_like(o)
        ss.decode_step(o_k, dx, dz, ddt, *wts, p.norm_groups, p.eps, conv_k, ssm_k, dims, slots, [0] * 4)
        oo, _ = oracle.decode_step(dx.cpu(), dz.cpu(), ddt.cpu(), p.conv_w, p.conv_b, p.A_log, p.dt_bias, p.D,
                                   p.norm_w, p.norm_groups, p.eps, conv_o, ssm_o, (H, P, N, G), slots, [0] * 4)
        torch.cuda.synchronize()
        assert_bits_equal(o.cpu(), o_k.cpu(), f"decode step {step} vs the plain decode call")
        assert rel_l2(o.cpu(), oo) <= 1e-2
        assert slot_rel_l2(cache.ssm_pool, ssm_o, slots) <= STATE_PREFILL_REL_L2
    assert cache.seqlen_offset == [L + 2 for L in lengths]
