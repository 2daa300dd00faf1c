"""GPU parity of the Mamba-3 SISO forward (page "Mamba-3 SISO Long-Ragged
Multi-Chunk Joint States Full VJP", forward steps 1-7) against the oracle, through
the C ABI (include/mamba3.h).

Acceptance: out within the activation tolerance of tests/util.py (2e-2 absolute
plus 2^-8 relative of the oracle's unrounded double, rel-L2 <= 1e-2); the fp32
final state within the prefill state tolerance (rel-L2 <= 1e-3); the final rotated
k elementwise within 1e-3 absolute + 1e-3 relative (fp32 rotation of the same
inputs; the angle is summed in fp32 on the GPU); the final angle, a bf16 value on
the circle, within the activation tolerance after wrapping the difference into
(-pi, pi] (the two sides may put a value near 2 pi k on either side of the cut);
the final v bit for bit (a copy).
"""
import math

import pytest
import torch

import oracle
import selective_scan_gb300 as ss
import workloads as W
from tests.gpu_util import device
from tests.util import STATE_PREFILL_REL_L2, assert_bits_equal, check_act, rel_l2

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


def run_gpu(b, dev):
    n = len(b.cu_seqlens) - 1
    H, P, N, R = b.heads, b.headdim, b.d_state, b.rot_dim
    ins = [t.to(dev).contiguous() for t in b.tensors()]
    if R == 0:
        ins[8] = torch.empty((b.rows, 0), dtype=BF, device=dev)
    out = torch.full((b.rows, H, P), float("nan"), dtype=BF, device=dev)
    fa = torch.full((n, H, R), float("nan"), dtype=BF, device=dev)
    fs = torch.full((n, H, P, N), float("nan"), dtype=torch.float32, device=dev)
    fk = torch.full((n, H, N), float("nan"), dtype=torch.float32, device=dev)
    fv = torch.full((n, H, P), float("nan"), dtype=BF, device=dev)
    ss.mamba3_siso_varlen_forward(out, fa, fs, fk, fv, *ins, b.cu_seqlens)
    torch.cuda.synchronize()
    return [t.cpu() for t in (out, fa, fs, fk, fv)]


def compare(b, got, what):
    ro, ra, rs, rk, rv, r64 = oracle.mamba3_siso_forward(*b.tensors(), b.cu_seqlens)
    out, fa, fs, fk, fv = got
    check_act(out, r64, f"{what} out")
    if b.rot_dim > 0:
        d = (fa.double() - ra.double() + math.pi) % (2 * math.pi) - math.pi
        check_act(ra.double() + d, ra.double(), f"{what} final angle")
    assert rel_l2(fs, rs) <= STATE_PREFILL_REL_L2, f"{what} final ssm rel L2 {rel_l2(fs, rs):.3g}"
    assert torch.allclose(fk.double(), rk.double(), rtol=1e-3, atol=1e-3), f"{what} final k"
    assert_bits_equal(fv, rv, f"{what} final v")
    assert ss.library().mamba2_device_timeouts() == 0, f"{what}: a tensor-core wait timed out"


@pytest.mark.parametrize("seed", [5, 6, 7])
def test_frozen_shapes(seed):
    """32 heads, Q/K width 128, V width 64, 32 angles, 3-5 sequences of 3-15
    chunks of 64, lengths not multiples of 64."""
    dev = device()
    b = W.mamba3_batch(seed=seed)
    compare(b, run_gpu(b, dev), f"seed {seed}")


@pytest.mark.parametrize("heads", [5, 8])
def test_ragged_edges(heads):
    """An empty sequence, one token, a whole 128-token chunk, one past it, and a
    long one, packed together. With 8 heads the per-token scalars come by TMA
    (rows of 16-byte multiples), with 5 by strided loads."""
    dev = device()
    b = W.mamba3_batch(seed=11, lengths=[0, 1, 128, 129, 700, 255], heads=heads)
    compare(b, run_gpu(b, dev), f"ragged, {heads} heads")


@pytest.mark.parametrize("R,heads", [(0, 3), (1, 3), (6, 3), (34, 3), (40, 3), (64, 3), (0, 8), (34, 8), (64, 8)])
def test_rotary_widths(R, heads):
    """Rotary widths from none to every pair (above 32 each thread's second pair turns
    too); with 8 heads the per-token scalars come by TMA, with 3 by strided loads."""
    dev = device()
    b = W.mamba3_batch(seed=12, lengths=[300, 97], heads=heads, rot_dim=R)
    compare(b, run_gpu(b, dev), f"rot_dim {R}, {heads} heads")


def test_all_sequences_empty():
    """Sequences but no rows: the kernel still runs every (sequence, head) item and
    writes zero final states (NaN-poisoned before), issuing no copy."""
    dev = device()
    b = W.mamba3_batch(seed=17, lengths=[0, 0, 0], heads=8)
    assert b.rows == 0
    out, fa, fs, fk, fv = run_gpu(b, dev)
    for t, name in ((fa, "final angle"), (fs, "final ssm"), (fk, "final k"), (fv, "final v")):
        assert torch.equal(t.float(), torch.zeros_like(t.float())), f"{name} not zero"
    assert out.numel() == 0
    assert ss.library().mamba2_device_timeouts() == 0


def test_more_items_than_sms():
    """More (sequence, head) items than SMs: CTAs take a second item."""
    dev = device()
    g = torch.Generator().manual_seed(3)
    lengths = [int(x) for x in torch.randint(1, 300, (200,), generator=g)]
    b = W.mamba3_batch(seed=13, lengths=lengths, heads=2)
    compare(b, run_gpu(b, dev), "200 sequences")


def test_fp16_range_fallback():
    """v beyond the fp16 range of the tensor-core operands (the output scales with
    v, so the problem stays well conditioned): the CTA recomputes its item token by
    token in fp32."""
    dev = device()
    b = W.mamba3_batch(seed=14, lengths=[150, 40], heads=2)
    b.v = (b.v.float() * 1e5).to(BF)
    compare(b, run_gpu(b, dev), "fp16 range")


def test_rejects_bad_batches_before_launch():
    dev = device()
    b = W.mamba3_batch(seed=15, lengths=[10, 10], heads=2)
    n = 2
    ins = [t.to(dev).contiguous() for t in b.tensors()]
    outs = [torch.empty((b.rows, 2, 64), dtype=BF, device=dev), torch.empty((n, 2, 32), dtype=BF, device=dev),
            torch.empty((n, 2, 64, 128), device=dev), torch.empty((n, 2, 128), device=dev),
            torch.empty((n, 2, 64), dtype=BF, device=dev)]
    st = ss.mamba3_siso_varlen_forward(*outs, *ins, [0, 12, 21], check=False)
    assert st == ss.ERR_RUNS_DONT_COVER_ROWS
    st = ss.mamba3_siso_varlen_forward(*outs, *ins, [0, 12, 10], check=False)
    assert st == ss.ERR_RUNS_DONT_COVER_ROWS


@pytest.mark.parametrize("heads", [1, 8])
def test_long_sequence_many_chunks(heads):
    """A 4 000-token sequence (32 chunks of 128: the angle carry and the state cross
    31 chunk boundaries) and a run of one-token sequences beside it; the last rows
    of the batch end inside the final chunk's boxes (read as zero past the tensor)."""
    dev = device()
    b = W.mamba3_batch(seed=16, lengths=[4000, 1, 1, 3, 130], heads=heads)
    compare(b, run_gpu(b, dev), f"4000 tokens, {heads} heads")
