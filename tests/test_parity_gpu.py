"""GPU parity: the CUDA path (through the C ABI) against the oracle on the same
seeded inputs, per op and chained, on the five named workloads and on small
multi-chunk, ragged and degenerate batches.

Acceptance (the target's tolerances): conv histories, slot routing and
rejections bit-exact; activation outputs within 2e-2 absolute plus a bf16
half-ulp relative of the oracle's unrounded value and 1e-2 relative L2; fp32
SSM state within 1e-3 relative L2 after chunked prefill and 1e-5 after decode.
Semantics: gllm PR #85 "feat(backend): Mamba2 ops, with CPU reference
implementations", sections "Ops", "CPU reference" and "Testing".
"""
import pytest
import torch

import oracle
import selective_scan_gb300 as ss
import workloads as W
from tests.gpu_util import device, gpu_conv, gpu_norm, gpu_scan, oracle_prefill, slot_rel_l2
from tests.util import (STATE_DECODE_REL_L2, STATE_PREFILL_REL_L2, assert_bits_equal, check_act, rel_l2)

pytestmark = pytest.mark.gpu


def _untouched(pool_after, pool_before, slots, what):
    others = [i for i in range(pool_before.shape[0]) if i not in set(slots)]
    if others:
        idx = torch.tensor(others, dtype=torch.long)
        assert_bits_equal(pool_after.cpu()[idx], pool_before[idx], f"{what}: slots outside the batch")


def _prefill_parity(wl):
    dev = device()
    ref = oracle_prefill(wl)
    b = wl.batch
    # conv (per op)
    xbc, conv = gpu_conv(wl, dev)
    torch.cuda.synchronize()
    check_act(xbc.cpu(), ref["xbc64"], "conv output")
    assert_bits_equal(conv.cpu(), ref["conv"], "conv state pool")
    # scan fed the oracle's conv output (per op)
    y, ssm = gpu_scan(wl, dev, ref["xbc"])
    torch.cuda.synchronize()
    check_act(y.cpu(), ref["y64"], "scan output")
    rl = slot_rel_l2(ssm, ref["ssm"], b.slots)
    assert rl <= STATE_PREFILL_REL_L2, f"ssm state rel L2 {rl:.3g}"
    _untouched(ssm, wl.ssm_state, b.slots, "ssm pool")
    assert torch.isfinite(ssm.cpu()[torch.tensor(b.slots)]).all()
    # norm fed the oracle's y (per op)
    out = gpu_norm(wl, dev, ref["y"])
    torch.cuda.synchronize()
    check_act(out.cpu(), ref["out64"], "norm output")
    # chained: conv -> scan -> norm entirely on the GPU. Each op is checked
    # against the oracle on the very input it received in the chain (the conv
    # output and y are rounding points, where the two implementations may land
    # one bf16 step apart); the chain as a whole is checked in aggregate.
    p = wl.params
    y2, ssm2 = gpu_scan(wl, dev, xbc)
    out2 = gpu_norm(wl, dev, y2)
    torch.cuda.synchronize()
    xbc_c, y2_c = xbc.cpu(), y2.cpu()
    ssm_o = wl.ssm_state.clone()
    _, y2_64 = oracle.ssd_scan(xbc_c, wl.dt, p.A_log, p.dt_bias, p.D, ssm_o, wl.dims.tuple4(),
                               b.cu_seqlens, b.slots, b.fresh)
    check_act(y2_c, y2_64, "chained scan output")
    _, out2_64 = oracle.gated_rmsnorm(y2_c, wl.z, p.norm_w, p.norm_groups, p.eps)
    check_act(out2.cpu(), out2_64, "chained norm output")
    rl2 = slot_rel_l2(ssm2, ssm_o, b.slots)
    assert rl2 <= STATE_PREFILL_REL_L2, f"chained ssm state rel L2 {rl2:.3g}"
    rl3 = slot_rel_l2(ssm2, ref["ssm"], b.slots)
    assert rl3 <= STATE_PREFILL_REL_L2, f"chain vs oracle chain: ssm state rel L2 {rl3:.3g}"
    assert rel_l2(out2.cpu(), ref["out64"]) <= 1e-2, "chain vs oracle chain: output rel L2"
    return ref, dict(xbc=xbc, y=y2, out=out2, ssm=ssm2, conv=conv)


def test_tiny_fp32():
    """4 heads x 16, d_state 16, 2 groups, fp32, 64 tokens (token-serial kernel)."""
    _prefill_parity(W.tiny())


def test_tiny_dims_bf16_ragged_multichunk():
    """The chunked kernel at 16x16 tiles: many chunks, ragged tails, a run of
    one token, a zero-length fresh run and a zero-length resumed run."""
    lengths = [1, 63, 64, 65, 130, 300, 0, 0, 517]
    fresh = [1, 0, 1, 0, 1, 0, 1, 0, 0]
    wl = W.make_prefill("tiny-bf16", 17, W.DIMS_TINY, lengths, torch.bfloat16, 16, fresh, norm_groups=2)
    _prefill_parity(wl)


def test_prefill_130m_2048():
    _prefill_parity(W.prefill_130m())


def test_varlen_130m():
    _prefill_parity(W.varlen_130m())


def test_130m_short_runs_unsegmented():
    """Many short runs (one chunk or less each): every sequence is one segment."""
    lengths = [5, 64, 17, 33, 1, 60, 64, 2]
    wl = W.make_prefill("short", 23, W.DIMS_130M, lengths, torch.bfloat16, 12, [i % 2 for i in range(8)])
    _prefill_parity(wl)


@pytest.mark.parametrize("H,G", [(8, 2), (6, 2), (5, 1)])
def test_state_pass_head_pairs(H, G):
    """Runs long enough to be cut into segments, so the state pass runs: with 8
    heads in 2 groups its CTAs take heads in pairs that never cross a group; with
    6 heads in 2 groups or 5 in 1 (an odd number of heads per group) one head each.
    A resumed sequence seeds the first piece from its slot."""
    d = W.Dims(H, 64, 128, G, 4)
    wl = W.make_prefill(f"pairs-{H}x{G}", 71, d, [2600, 1700, 90], torch.bfloat16, 6, [0, 1, 0])
    _prefill_parity(wl)


def test_many_heads_dt_prime_by_head_tiles():
    """800 heads (above the 768 whose dt' rows fit one CTA's shared memory): the
    scan's dt' pre-pass runs as 32 x 32 tiles instead of 64-row blocks."""
    d = W.Dims(800, 64, 128, 2, 4)
    wl = W.make_prefill("heads-800", 83, d, [300, 129], torch.bfloat16, 3, [1, 0])
    _prefill_parity(wl)


def test_scan_fp16_range_fallback():
    """Inputs whose Y = M . X operands leave the fp16 range: a token whose C and
    B rows are large and aligned (an M entry near 1.5e5, in every head's
    segment, since the heads share one group) and one x entry of 7e4 in one head.
    The CTAs that meet them recompute their segment's y token by token; y and
    the state still match the oracle, and no wait times out."""
    dev = device()
    wl = W.make_prefill("range", 61, W.DIMS_130M, [700, 1300], torch.bfloat16, 6, [1, 0])
    H, P, N, G = wl.dims.tuple4()
    ref = oracle_prefill(wl)
    xbc = ref["xbc"].clone()
    dt = wl.dt.clone()
    t_m = 300                                   # sequence 0: C_t . B_t = 900 * 128, dt' about 1.3
    xbc[t_m, H * P:H * P + N] = 30.0
    xbc[t_m, H * P + G * N:H * P + G * N + N] = 30.0
    dt[t_m, :] = 5.0
    t_x, h_x = 700 + 900, 5                     # sequence 1, head 5: one x of 7e4
    xbc[t_x, h_x * P + 7] = 7.0e4
    p, b = wl.params, wl.batch
    lib = ss.library()
    before = lib.mamba2_device_timeouts()
    y, ssm = gpu_scan(wl, dev, xbc, dt=dt)
    torch.cuda.synchronize()
    ssm_o = wl.ssm_state.clone()
    _, y64 = oracle.ssd_scan(xbc, dt, p.A_log, p.dt_bias, p.D, ssm_o, (H, P, N, G), b.cu_seqlens, b.slots, b.fresh)
    assert y64.abs().max().item() > 1e5, "the planted values should make some y large"
    check_act(y.cpu(), y64, "scan output with fp16-range fallback")
    rl = slot_rel_l2(ssm, ssm_o, b.slots)
    assert rl <= STATE_PREFILL_REL_L2, f"ssm state rel L2 {rl:.3g}"
    _untouched(ssm, wl.ssm_state, b.slots, "ssm pool")
    assert lib.mamba2_device_timeouts() == before


def test_head_group_mapping_gpu():
    """Zeroing group 1's B and C leaves heads 2, 3 with D*x exactly and heads 0, 1 unchanged."""
    dev = device()
    wl = W.make_prefill("t7", 0, W.DIMS_TINY, [200], torch.bfloat16, 1, [1], slots=[0], norm_groups=2)
    H, P, N, G = wl.dims.tuple4()
    ref = oracle_prefill(wl)
    xbc = ref["xbc"]
    z = xbc.clone()
    z[:, H * P + N: H * P + 2 * N] = 0
    z[:, H * P + G * N + N: H * P + G * N + 2 * N] = 0
    y0, _ = gpu_scan(wl, dev, xbc)
    y1, _ = gpu_scan(wl, dev, z)
    y0, y1 = y0.cpu(), y1.cpu()
    assert_bits_equal(y1[:, :2 * P], y0[:, :2 * P], "heads 0,1 untouched")
    for h in (2, 3):
        dx = (wl.params.D[h].double() * xbc[:, h * P:(h + 1) * P].double()).float().to(torch.bfloat16)
        assert_bits_equal(y1[:, h * P:(h + 1) * P], dx, f"head {h} = D*x")


def test_split_equals_whole_gpu():
    """One run vs the same run cut into calls (a one-token first call, then
    pieces with ragged chunk tails); conv bit-exact, state to 1e-6."""
    dev = device()
    wl = W.make_prefill("split", 31, W.DIMS_130M, [700], torch.bfloat16, 2, [1], slots=[1])
    p = wl.params
    xbc_w, conv_w = gpu_conv(wl, dev)
    y_w, ssm_w = gpu_scan(wl, dev, xbc_w)
    conv_s, ssm_s = wl.conv_state.to(dev), wl.ssm_state.to(dev)
    cuts = [0, 1, 3, 130, 450, 700]
    xs, ys = [], []
    for i in range(len(cuts) - 1):
        a, b = cuts[i], cuts[i + 1]
        fr = [1 if i == 0 else 0]
        x = wl.xBC[a:b].contiguous().to(dev)
        xb = torch.empty_like(x)
        ss.causal_conv1d(xb, x, p.conv_w.to(dev), p.conv_b.to(dev), conv_s, [0, b - a], [1], fr)
        y = torch.empty((b - a, wl.dims.d_inner), dtype=x.dtype, device=dev)
        ss.ssd_scan(y, xb, wl.dt[a:b].contiguous().to(dev), p.A_log.to(dev), p.dt_bias.to(dev), p.D.to(dev),
                    ssm_s, wl.dims, [0, b - a], [1], fr)
        xs.append(xb)
        ys.append(y)
    torch.cuda.synchronize()
    assert_bits_equal(torch.cat(xs).cpu(), xbc_w.cpu(), "conv output split vs whole")
    assert_bits_equal(conv_s.cpu(), conv_w.cpu(), "conv state split vs whole")
    # the cuts are not chunk-aligned, so the chunking differs: operand precision ~2^-17
    assert rel_l2(ssm_s.cpu()[1], ssm_w.cpu()[1]) <= 1e-5
    assert rel_l2(torch.cat(ys).cpu(), y_w.cpu()) <= 1e-3


def test_swapped_slots_and_dirty_fresh_slot_gpu():
    """Two sequences on swapped slots (one fresh on a NaN-poisoned slot, one
    resuming) match their solo runs; nothing reads the dirty slot."""
    dev = device()
    d = W.DIMS_130M
    g = torch.Generator().manual_seed(41)
    La, Lb = 150, 333
    xA, zA, dtA = W.draw_tokens(g, La, d, torch.bfloat16)
    xB, zB, dtB = W.draw_tokens(g, Lb, d, torch.bfloat16)
    params = W.draw_params(g, d, 1)
    conv0, ssm0 = W.empty_pools(3, d, torch.bfloat16)  # slot 2 stays sentinel; slot 1 dirty for A
    W.fill_resumed_slots(g, conv0, ssm0, [0], [0], torch.bfloat16)

    def run(x, dt, cu, slots, fresh):
        wl = W.Workload("t", d, torch.bfloat16, params, W.Batch(cu, slots, fresh), x, x[:, :d.d_inner], dt,
                        conv0.clone(), ssm0.clone())
        xbc, conv = gpu_conv(wl, dev)
        y, ssm = gpu_scan(wl, dev, xbc)
        torch.cuda.synchronize()
        return xbc.cpu(), y.cpu(), conv.cpu(), ssm.cpu()

    xb, yb, cb, sb = run(torch.cat([xA, xB]), torch.cat([dtA, dtB]), [0, La, La + Lb], [1, 0], [1, 0])
    xa1, ya1, ca1, sa1 = run(xA, dtA, [0, La], [1], [1])
    xb1, yb1, cb1, sb1 = run(xB, dtB, [0, Lb], [0], [0])
    assert torch.isfinite(yb).all() and torch.isfinite(sb[1]).all()
    assert_bits_equal(xb, torch.cat([xa1, xb1]), "conv outputs batched vs solo")
    assert_bits_equal(cb[1], ca1[1], "slot 1 conv")
    assert_bits_equal(cb[0], cb1[0], "slot 0 conv")
    assert_bits_equal(cb[2], conv0[2], "slot 2 conv untouched")
    assert_bits_equal(sb[2], ssm0[2], "slot 2 ssm untouched")
    assert rel_l2(sb[1], sa1[1]) <= 1e-6 and rel_l2(sb[0], sb1[0]) <= 1e-6
    assert rel_l2(yb, torch.cat([ya1, yb1])) <= 1e-3
    # fresh on a dirty slot == resume from an all-zero slot
    z0 = ssm0.clone()
    z0[1].zero_()
    c0 = conv0.clone()
    c0[1].zero_()
    wl = W.Workload("t", d, torch.bfloat16, params, W.Batch([0, La], [1], [0]), xA, xA[:, :d.d_inner], dtA,
                    c0, z0)
    xz, cz = gpu_conv(wl, dev)
    yz, sz = gpu_scan(wl, dev, xz)
    torch.cuda.synchronize()
    assert_bits_equal(xz.cpu(), xa1, "fresh vs zero-slot conv output")
    assert_bits_equal(yz.cpu(), ya1, "fresh vs zero-slot scan output")
    assert_bits_equal(sz.cpu()[1], sa1[1], "fresh vs zero-slot state")


BAD = [
    ("slot out of range", [0, 30, 70], [0, 5], ss.ERR_SLOT_OUT_OF_RANGE),
    ("shared slot", [0, 30, 70], [2, 2], ss.ERR_SLOT_SHARED),
    ("runs short", [0, 30, 69], [0, 1], ss.ERR_RUNS_DONT_COVER_ROWS),
]


@pytest.mark.parametrize("name,cu,slots,status", BAD, ids=[b[0] for b in BAD])
def test_rejection_leaves_buffers_untouched_gpu(name, cu, slots, status):
    dev = device()
    wl = W.make_prefill("rej", 5, W.DIMS_TINY, [30, 40], torch.bfloat16, 4, [0, 0], slots=[0, 1],
                        norm_groups=2)
    p = wl.params
    x = wl.xBC.to(dev)
    conv, ssm = wl.conv_state.to(dev), wl.ssm_state.to(dev)
    dst = torch.full_like(x, 7.0)
    y = torch.full((70, wl.dims.d_inner), 3.0, dtype=torch.bfloat16, device=dev)
    st = ss.causal_conv1d(dst, x, p.conv_w.to(dev), p.conv_b.to(dev), conv, cu, slots, [0, 0], check=False)
    assert st == status
    st = ss.ssd_scan(y, x, wl.dt.to(dev), p.A_log.to(dev), p.dt_bias.to(dev), p.D.to(dev), ssm, wl.dims, cu,
                     slots, [0, 0], check=False)
    assert st == status
    torch.cuda.synchronize()
    assert_bits_equal(conv.cpu(), wl.conv_state, "conv pool")
    assert_bits_equal(ssm.cpu(), wl.ssm_state, "ssm pool")
    assert (dst.cpu() == 7.0).all() and (y.cpu() == 3.0).all()


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------

def _decode_parity(wl, steps, dev):
    p, d, b = wl.params, wl.dims, wl.batch
    conv_g, ssm_g = wl.conv_state.to(dev), wl.ssm_state.to(dev)
    conv_o, ssm_o = wl.conv_state.clone(), wl.ssm_state.clone()
    args = [t.to(dev) for t in (p.conv_w, p.conv_b, p.A_log, p.dt_bias, p.D, p.norm_w)]
    n = b.num_seqs
    worst = 0.0
    for t in range(steps):
        fr = b.fresh if t == 0 else [0] * n
        x, z, dt = wl.dec_xBC[t].contiguous(), wl.dec_z[t].contiguous(), wl.dec_dt[t].contiguous()
        out_g = torch.empty((n, d.d_inner), dtype=x.dtype, device=dev)
        ss.decode_step(out_g, x.to(dev), z.to(dev), dt.to(dev), *args, p.norm_groups, p.eps, conv_g, ssm_g, d,
                       b.slots, fr)
        _, out64 = oracle.decode_step(x, z, dt, p.conv_w, p.conv_b, p.A_log, p.dt_bias, p.D, p.norm_w,
                                      p.norm_groups, p.eps, conv_o, ssm_o, d.tuple4(), b.slots, fr)
        torch.cuda.synchronize()
        # every step: the output against the oracle's unrounded double, the conv
        # pool bit for bit, the named slots' SSM state by relative L2
        check_act(out_g.cpu(), out64, f"decode out step {t}")
        assert_bits_equal(conv_g.cpu(), conv_o, f"conv pool after step {t}")
        rl = slot_rel_l2(ssm_g, ssm_o, b.slots)
        worst = max(worst, rl)
        assert rl <= STATE_DECODE_REL_L2, f"step {t}: ssm rel L2 {rl:.3g}"
    _untouched(ssm_g, wl.ssm_state, b.slots, "ssm pool")
    return worst


def test_decode_small_batches():
    dev = device()
    # tiny dims (2 groups, norm groups 2), a fresh sequence among resumed ones
    wl = W.decode_batch(seed=7, num_seqs=5, steps=6, num_slots=9, dims=W.DIMS_TINY)
    wl.params.norm_groups = 2
    wl.batch.fresh[2] = 1
    _decode_parity(wl, 6, dev)


def test_decode_batch_256x128():
    """256 sequences x 128 steps against a 512-slot pool, state carried."""
    dev = device()
    wl = W.decode_batch()
    _decode_parity(wl, 128, dev)


# ---------------------------------------------------------------------------
# long prefill with continuation: 65536 tokens, 48 heads
# ---------------------------------------------------------------------------

def test_long_prefill_65536_split_and_decode():
    dev = device()
    wl = W.long_prefill()
    p, d = wl.params, wl.dims
    T = wl.batch.rows
    # GPU: whole call
    xbc, conv = gpu_conv(wl, dev)
    y, ssm = gpu_scan(wl, dev, xbc)
    out = gpu_norm(wl, dev, y)
    # GPU: 4 resumed calls of 16384
    conv_s, ssm_s = wl.conv_state.to(dev), wl.ssm_state.to(dev)
    xs, ys = [], []
    L = T // 4
    for i in range(4):
        a, b = i * L, (i + 1) * L
        x = wl.xBC[a:b].contiguous().to(dev)
        xb = torch.empty_like(x)
        ss.causal_conv1d(xb, x, p.conv_w.to(dev), p.conv_b.to(dev), conv_s, [0, L], [0], [1 if i == 0 else 0])
        yy = torch.empty((L, d.d_inner), dtype=x.dtype, device=dev)
        ss.ssd_scan(yy, xb, wl.dt[a:b].contiguous().to(dev), p.A_log.to(dev), p.dt_bias.to(dev), p.D.to(dev),
                    ssm_s, d, [0, L], [0], [1 if i == 0 else 0])
        xs.append(xb.cpu())
        ys.append(yy.cpu())
    torch.cuda.synchronize()
    assert_bits_equal(torch.cat(xs), xbc.cpu(), "conv split vs whole")
    assert_bits_equal(conv_s.cpu(), conv.cpu(), "conv state split vs whole")
    assert rel_l2(ssm_s.cpu(), ssm.cpu()) <= 1e-6, "state split vs whole"
    check_act(torch.cat(ys), y.cpu().double(), "y split vs whole", rel_ulp=2.0 ** -7)

    # oracle conv over the whole run
    conv_o = wl.conv_state.clone()
    xbc_o, xbc64 = oracle.causal_conv1d(wl.xBC, p.conv_w, p.conv_b, conv_o, [0, T], [0], [1])
    check_act(xbc.cpu(), xbc64, "conv output")
    assert_bits_equal(conv.cpu(), conv_o, "conv state")
    del xbc64

    # oracle scan over all 48 heads; GPU scan fed the oracle's conv output
    y_g, ssm_g = gpu_scan(wl, dev, xbc_o)
    torch.cuda.synchronize()
    ssm_o = wl.ssm_state.clone()
    _, y64 = oracle.ssd_scan(xbc_o, wl.dt, p.A_log, p.dt_bias, p.D, ssm_o, d.tuple4(), [0, T], [0], [1])
    check_act(y_g.cpu(), y64, "scan output (every head)")
    del y64
    rl = rel_l2(ssm_g.cpu()[0], ssm_o[0])
    assert rl <= STATE_PREFILL_REL_L2, f"state rel L2 (every head) {rl:.3g}"

    # norm per op on the GPU's own y
    _, out64 = oracle.gated_rmsnorm(y.cpu(), wl.z, p.norm_w, p.norm_groups, p.eps)
    check_act(out.cpu(), out64, "norm output")
    del out64

    # 64 decode steps continuing from the prefill's end state
    cont = W.Workload("tail", d, wl.act, p, W.Batch([0, 1], [0], [0]), wl.xBC[:0], wl.z[:0], wl.dt[:0],
                      conv.cpu(), ssm.cpu(), wl.dec_xBC, wl.dec_z, wl.dec_dt)
    _decode_parity(cont, wl.dec_xBC.shape[0], dev)


def _host_pieces(cu, slots, fresh, piece_rows, min_tail=512):
    """The piece rule of mamba2_prefill_host, restated: pieces of piece_rows rows,
    the last piece_rows or fewer rows halved while the remainder keeps at least
    2 * min_tail rows; a run cut at a piece edge continues in the next piece
    (fresh only in its first part); a zero-length run goes to the piece holding
    its start row."""
    rows = cu[-1]
    cuts, r = [0], 0
    while rows - r > piece_rows:
        r += piece_rows
        cuts.append(r)
    left = rows - r
    while left >= 2 * min_tail:
        r += left // 2
        cuts.append(r)
        left -= left // 2
    if rows > 0:
        cuts.append(rows)
    n_pieces = 1 if rows == 0 else len(cuts) - 1
    out = []
    for k in range(n_pieces):
        r0, r1 = cuts[k], (cuts[k + 1] if rows > 0 else 0)
        pc, ps, pf = [0], [], []
        for i in range(len(slots)):
            a, b = cu[i], cu[i + 1]
            inside = (r0 <= a < r1 or (a == rows and k == n_pieces - 1)) if a == b else (a < r1 and b > r0)
            if inside:
                pc.append(min(b, r1) - r0)
                ps.append(slots[i])
                pf.append(1 if fresh[i] and max(a, r0) == a else 0)
        out.append((r0, r1, pc, ps, pf))
    return out


HOST_CASES = [
    # pieces of 200 rows cutting runs mid-way, zero-length runs at piece starts; oracle-checked
    ("small", [1, 63, 0, 300, 65, 0, 517, 130, 0], [1, 0, 1, 0, 1, 0, 0, 1, 1], 200, True),
    # 5 900 rows in pieces of 2 048: the last 1 804 rows are halved into 902 + 902
    ("tail", [3000, 1, 0, 2899], [1, 0, 1, 0], 2048, False),
    # 6 000 rows in pieces of 4 096: the last 1 904 rows are halved into 952 + 952
    ("tail-halved", [700, 5300], [0, 1], 4096, False),
    # fp32 activations at the tiny shape (4 heads x 16, d_state 16, 2 groups): the other
    # scan kernel through the same pieces; oracle-checked
    ("tiny-f32", [5, 130, 0, 64, 301], [1, 0, 1, 1, 0], 100, True),
]


@pytest.mark.gpu
@pytest.mark.parametrize("name,lengths,fresh,P,with_oracle", HOST_CASES, ids=[c[0] for c in HOST_CASES])
def test_prefill_host_streamed(name, lengths, fresh, P, with_oracle):
    """mamba2_prefill_host from pinned host memory: bit-identical to the device ops
    called once per piece (so the copies, buffers and ordering lose nothing), and,
    on the small case, against the oracle over the whole batch: conv state
    bit-exact, the chained output and the SSM state by relative L2."""
    dev = torch.device("cuda:0")
    tiny = name.startswith("tiny")
    wl = W.make_prefill("host-" + name, 41, W.DIMS_TINY if tiny else W.DIMS_130M, lengths,
                        torch.float32 if tiny else torch.bfloat16, 12, fresh, **({"norm_groups": 2} if tiny else {}))
    p, b, d = wl.params, wl.batch, wl.dims
    act = wl.act
    w = [t.to(dev) for t in (p.conv_w, p.conv_b, p.A_log, p.dt_bias, p.D, p.norm_w)]
    hx, hz, hdt = wl.xBC.pin_memory(), wl.z.pin_memory(), wl.dt.pin_memory()
    hout = torch.full((b.rows, d.d_inner), float("nan"), dtype=act).pin_memory()
    conv_h, ssm_h = wl.conv_state.to(dev), wl.ssm_state.to(dev)
    ss.prefill_host(hout, hx, hz, hdt, *w[:5], w[5], p.norm_groups, p.eps, conv_h, ssm_h, d, b.cu_seqlens,
                    b.slots, b.fresh, piece_rows=P)
    torch.cuda.synchronize()

    conv_r, ssm_r = wl.conv_state.to(dev), wl.ssm_state.to(dev)
    out_r = torch.empty((b.rows, d.d_inner), dtype=act, device=dev)
    pieces = _host_pieces(b.cu_seqlens, b.slots, b.fresh, P)
    assert len(pieces) > 2
    for r0, r1, pc, ps, pf in pieces:
        x = wl.xBC[r0:r1].to(dev)
        xbc = torch.empty_like(x)
        ss.causal_conv1d(xbc, x, w[0], w[1], conv_r, pc, ps, pf)
        y = torch.empty((r1 - r0, d.d_inner), dtype=act, device=dev)
        ss.ssd_scan(y, xbc, wl.dt[r0:r1].to(dev), w[2], w[3], w[4], ssm_r, d, pc, ps, pf)
        ss.gated_rmsnorm(out_r[r0:r1], y, wl.z[r0:r1].to(dev), w[5], p.norm_groups, p.eps)
    torch.cuda.synchronize()
    assert_bits_equal(hout, out_r.cpu(), "streamed output vs per-piece device calls")
    assert_bits_equal(conv_h.cpu(), conv_r.cpu(), "conv pool")
    assert_bits_equal(ssm_h.cpu(), ssm_r.cpu(), "ssm pool")
    if name == "tail-halved":
        assert [r1 - r0 for r0, r1, *_ in pieces] == [4096, 952, 952]
    if not with_oracle:
        return

    conv_o, ssm_o = wl.conv_state.clone(), wl.ssm_state.clone()
    xbc_o, _ = oracle.causal_conv1d(wl.xBC, p.conv_w, p.conv_b, conv_o, b.cu_seqlens, b.slots, b.fresh)
    y_o, _ = oracle.ssd_scan(xbc_o, wl.dt, p.A_log, p.dt_bias, p.D, ssm_o, d.tuple4(), b.cu_seqlens, b.slots,
                             b.fresh)
    _, out64 = oracle.gated_rmsnorm(y_o, wl.z, p.norm_w, p.norm_groups, p.eps)
    assert_bits_equal(conv_h.cpu(), conv_o, "conv pool vs oracle")
    assert rel_l2(hout.double(), out64) <= 1e-2
    idx = torch.tensor(b.slots)
    assert rel_l2(ssm_h.cpu()[idx], ssm_o[idx]) <= 1e-3


NORM_SHAPES = [
    # rows, dim, groups, act: an odd row count (the last CTA holds one row), several groups,
    # groups wider than the vectors a thread keeps in registers, and a group too wide for
    # its weights to be staged in shared memory
    (7, 3072, 1, torch.bfloat16),
    (33, 1536, 4, torch.bfloat16),
    (5, 8192, 1, torch.bfloat16),
    (3, 16384, 1, torch.bfloat16),
    (9, 2048, 2, torch.float32),
]


@pytest.mark.gpu
@pytest.mark.parametrize("rows,dim,groups,act", NORM_SHAPES,
                         ids=[f"{r}x{d}g{g}{'bf16' if a == torch.bfloat16 else 'f32'}" for r, d, g, a in NORM_SHAPES])
def test_gated_rmsnorm_shapes(rows, dim, groups, act):
    """GatedRMSNorm alone on seeded N(0,1) inputs and weights N(1, 0.1^2) against the
    oracle, element by element, across the kernel's row pairing and its three weight
    and width paths."""
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(rows * 1000 + dim + groups)
    x = torch.randn((rows, dim), generator=g).to(act)
    z = torch.randn((rows, dim), generator=g).to(act)
    w = 1.0 + 0.1 * torch.randn(dim, generator=g)
    out = torch.empty((rows, dim), dtype=act, device=dev)
    ss.gated_rmsnorm(out, x.to(dev), z.to(dev), w.to(dev), groups, 1e-5)
    torch.cuda.synchronize()
    _, out64 = oracle.gated_rmsnorm(x, z, w, groups, 1e-5)
    check_act(out.cpu(), out64, f"norm {rows}x{dim} groups {groups}")


@pytest.mark.gpu
def test_prefill_host_all_runs_empty():
    """A streamed host prefill whose runs are all empty (no rows at all): fresh slots
    end with zero conv history and zero state, resumed slots and the others are left
    untouched, and the output buffer is not written."""
    dev = torch.device("cuda:0")
    wl = W.make_prefill("host-empty", 43, W.DIMS_130M, [0, 0, 0], torch.bfloat16, 6, [1, 0, 1])
    p, b, d = wl.params, wl.batch, wl.dims
    w = [t.to(dev) for t in (p.conv_w, p.conv_b, p.A_log, p.dt_bias, p.D, p.norm_w)]
    conv0, ssm0 = wl.conv_state.clone(), wl.ssm_state.clone()
    conv_h, ssm_h = conv0.to(dev), ssm0.to(dev)
    empty = torch.empty((0, d.conv_dim), dtype=torch.bfloat16).pin_memory()
    hz = torch.empty((0, d.d_inner), dtype=torch.bfloat16).pin_memory()
    hdt = torch.empty((0, d.heads), dtype=torch.bfloat16).pin_memory()
    hout = torch.empty((0, d.d_inner), dtype=torch.bfloat16).pin_memory()
    ss.prefill_host(hout, empty, hz, hdt, *w[:5], w[5], p.norm_groups, p.eps, conv_h, ssm_h, d, b.cu_seqlens,
                    b.slots, b.fresh, piece_rows=256)
    torch.cuda.synchronize()
    conv_g, ssm_g = conv_h.cpu(), ssm_h.cpu()
    for i, s in enumerate(b.slots):
        if b.fresh[i]:
            assert not conv_g[s].float().abs().any() and not ssm_g[s].abs().any(), f"fresh slot {s} not zeroed"
        else:
            assert_bits_equal(conv_g[s], conv0[s], f"resumed slot {s} conv")
            assert_bits_equal(ssm_g[s], ssm0[s], f"resumed slot {s} ssm")
    others = [s for s in range(conv0.shape[0]) if s not in set(b.slots)]
    assert_bits_equal(conv_g[others], conv0[others], "other conv slots")
    assert_bits_equal(ssm_g[others], ssm0[others], "other ssm slots")
