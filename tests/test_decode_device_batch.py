"""GPU tests of mamba2_decode_step_device, the decode step whose batch (slots,
fresh flags, count) lives in device memory and is checked on the device.

- Against the host-batch decode step (itself checked against the oracle in
  test_parity_gpu.py): bit-identical outputs and pools for the same batch.
- The device check applies the host check's rules in its order (gllm PR #85
  "feat(backend): Mamba2 ops, with CPU reference implementations", section
  "Ops": a slot out of range or shared by two sequences is rejected); a
  rejected step leaves every buffer but the status word bit-unchanged.
- One captured CUDA graph replayed with a new batch each step (InfiniLM PR #575
  "feat(mamba2): integrate model loading and recurrent inference", "Summary":
  indexed recurrent Decode replayed through Decode graphs), every replayed step
  also checked against the oracle's decode step on the same batch: output at
  the activation tolerance against the oracle's unrounded values, conv pool bit
  for bit, the named slots' SSM state by relative L2, and the rejected replay
  rejected by the oracle with the same status.
"""
import pytest
import torch

import oracle
import selective_scan_gb300 as ss
import workloads as W
from tests.gpu_util import device, slot_rel_l2
from tests.util import STATE_DECODE_REL_L2, assert_bits_equal, check_act

pytestmark = pytest.mark.gpu


class _Layer:
    """Weights, pools and static device buffers of one decode layer."""

    def __init__(self, dev, seed, num_slots, capacity, dims=W.DIMS_48H, norm_groups=1, filled=None):
        g = torch.Generator("cpu").manual_seed(seed)
        act = torch.bfloat16
        self.dims, self.capacity, self.num_slots = dims, capacity, num_slots
        self.p = W.draw_params(g, dims, norm_groups)
        conv, ssm = W.empty_pools(num_slots, dims, act)
        filled = list(range(num_slots)) if filled is None else filled  # the rest keep the NaN sentinel
        W.fill_resumed_slots(g, conv, ssm, filled, [0] * len(filled), act)
        self.conv, self.ssm = conv.to(dev), ssm.to(dev)
        self.w = [t.to(dev) for t in (self.p.conv_w, self.p.conv_b, self.p.A_log, self.p.dt_bias, self.p.D,
                                      self.p.norm_w)]
        self.gen = g
        self.x = torch.zeros((capacity, dims.conv_dim), dtype=act, device=dev)
        self.z = torch.zeros((capacity, dims.d_inner), dtype=act, device=dev)
        self.dt = torch.zeros((capacity, dims.heads), dtype=act, device=dev)
        self.out = torch.full((capacity, dims.d_inner), 5.0, dtype=act, device=dev)
        self.slots = torch.zeros(capacity, dtype=torch.int32, device=dev)
        self.fresh = torch.zeros(capacity, dtype=torch.uint8, device=dev)
        self.n = torch.zeros(1, dtype=torch.int32, device=dev)
        self.status = torch.full((1,), -1, dtype=torch.int32, device=dev)

    def draw_step(self, n):
        """Inputs of n sequences, n distinct slots (some fresh), into the static buffers."""
        x, z, dt = W.draw_tokens(self.gen, n, self.dims, torch.bfloat16)
        slots = torch.randperm(self.num_slots, generator=self.gen)[:n].tolist()
        fresh = (torch.rand(n, generator=self.gen) < 0.25).to(torch.uint8).tolist()
        self.set_batch(slots, fresh, n)
        self.x[:n].copy_(x)
        self.z[:n].copy_(z)
        self.dt[:n].copy_(dt)
        return slots, fresh

    def set_batch(self, slots, fresh, n):
        k = len(slots)
        self.slots[:k].copy_(torch.tensor(slots, dtype=torch.int32))
        self.fresh[:k].copy_(torch.tensor(fresh, dtype=torch.uint8))
        self.n.fill_(n)

    def device_step(self, check=True):
        return ss.decode_step_device(self.out, self.x, self.z, self.dt, *self.w, self.p.norm_groups, self.p.eps,
                                     self.conv, self.ssm, self.dims, self.slots, self.fresh, self.n, self.status,
                                     check=check)

    def host_step(self, conv, ssm, slots, fresh):
        n = len(slots)
        out = torch.empty((n, self.dims.d_inner), dtype=torch.bfloat16, device=self.x.device)
        ss.decode_step(out, self.x[:n], self.z[:n], self.dt[:n], *self.w, self.p.norm_groups, self.p.eps,
                       conv, ssm, self.dims, slots, fresh)
        return out


def _same_step(L, n):
    """One step through both paths on equal pools: bit-identical results."""
    conv_h, ssm_h = L.conv.clone(), L.ssm.clone()
    slots, fresh = L.draw_step(n)
    L.out.fill_(5.0)
    out_h = L.host_step(conv_h, ssm_h, slots, fresh)
    L.device_step()
    torch.cuda.synchronize()
    assert int(L.status.item()) == ss.OK
    assert_bits_equal(L.out[:n].cpu(), out_h.cpu(), f"decode output, n={n}")
    assert (L.out[n:].cpu() == 5.0).all(), "rows past the device count were written"
    assert_bits_equal(L.conv.cpu(), conv_h.cpu(), "conv pool")
    assert_bits_equal(L.ssm.cpu(), ssm_h.cpu(), "ssm pool")


def test_device_batch_matches_host_batch():
    dev = device()
    # capacity = n: the same CTAs per sequence as the host call (6 at 40 sequences)
    L = _Layer(dev, seed=31, num_slots=96, capacity=40)
    for _ in range(3):
        _same_step(L, 40)
    # a small batch (16 CTAs per sequence) and fewer sequences than the capacity
    S = _Layer(dev, seed=32, num_slots=12, capacity=4)
    for n in (4, 3, 1, 4):
        _same_step(S, n)
    # tiny dims: two B/C groups, two norm groups
    T = _Layer(dev, seed=33, num_slots=9, capacity=5, dims=W.DIMS_TINY, norm_groups=2)
    for n in (5, 2):
        _same_step(T, n)


@pytest.mark.parametrize("slots,n,status", [
    ([3, 96], 2, ss.ERR_SLOT_OUT_OF_RANGE),
    ([-1, 4], 2, ss.ERR_SLOT_OUT_OF_RANGE),
    ([7, 8, 7], 3, ss.ERR_SLOT_SHARED),
    ([0, 0], 1, ss.OK),                       # only the first n slots form the batch
    ([1, 2], 9, ss.ERR_INVALID_ARGUMENT),     # count above the capacity
    ([1, 2], -1, ss.ERR_INVALID_ARGUMENT),
    ([96, 5, 5], 3, ss.ERR_SLOT_OUT_OF_RANGE),  # range is checked before sharing
])
def test_device_batch_rejections(slots, n, status):
    dev = device()
    L = _Layer(dev, seed=34, num_slots=96, capacity=8)
    L.draw_step(3)
    L.set_batch(slots, [0] * len(slots), n)
    conv0, ssm0 = L.conv.clone(), L.ssm.clone()
    L.out.fill_(5.0)
    assert L.device_step() == ss.OK  # the host checks pass; the device check decides
    torch.cuda.synchronize()
    assert int(L.status.item()) == status
    if status != ss.OK:
        assert (L.out.cpu() == 5.0).all()
        assert_bits_equal(L.conv.cpu(), conv0.cpu(), "conv pool after a rejected step")
        assert_bits_equal(L.ssm.cpu(), ssm0.cpu(), "ssm pool after a rejected step")
        # the same status word then takes a valid step
        _same_step(L, 8)


def test_device_batch_pairwise_duplicate_check():
    """A pool too large for the check's bitmap (over 262 144 slots): pairwise check."""
    dev = device()
    L = _Layer(dev, seed=35, num_slots=270_000, capacity=6, dims=W.DIMS_TINY, norm_groups=2,
               filled=[269_999, 5, 131_072, 77])
    L.draw_step(6)
    L.set_batch([269_999, 5, 131_072, 5], [0, 0, 0, 0], 4)
    ssm_row = L.ssm[5].clone()
    L.device_step()
    torch.cuda.synchronize()
    assert int(L.status.item()) == ss.ERR_SLOT_SHARED
    assert_bits_equal(L.ssm[5].cpu(), ssm_row.cpu(), "slot 5 after a rejected step")
    conv_h, ssm_h = L.conv.clone(), L.ssm.clone()
    slots, fresh = [269_999, 5, 131_072, 77], [0, 1, 0, 0]
    L.set_batch(slots, fresh, 4)
    out_h = L.host_step(conv_h, ssm_h, slots, fresh)
    L.device_step()
    torch.cuda.synchronize()
    assert int(L.status.item()) == ss.OK
    assert_bits_equal(L.out[:4].cpu(), out_h.cpu(), "decode output")
    idx = torch.tensor(slots)
    assert_bits_equal(L.ssm[idx].cpu(), ssm_h[idx].cpu(), "ssm slots")
    assert_bits_equal(L.conv[idx].cpu(), conv_h[idx].cpu(), "conv slots")


def test_device_batch_graph_replay():
    """One captured graph, replayed with a new batch, count and inputs every step."""
    dev = device()
    L = _Layer(dev, seed=36, num_slots=64, capacity=24)
    L.draw_step(24)
    L.device_step()  # outside the capture: kernel attributes are set here
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        L.device_step()
    conv_h, ssm_h = L.conv.clone(), L.ssm.clone()
    conv_o, ssm_o = L.conv.cpu(), L.ssm.cpu()  # the oracle's pools, carried through the replays
    p = L.p
    for step, n in enumerate((24, 17, 10, 24, 13)):  # >= 10 sequences: one cluster shape on both paths
        slots, fresh = L.draw_step(n)
        x, z, dt = (t[:n].cpu().contiguous() for t in (L.x, L.z, L.dt))
        if step == 3:  # a rejected replay in the middle leaves everything as it was
            bad = slots[:2] + [slots[0]]
            L.set_batch(bad, [0, 0, 0], 3)
            L.out.fill_(5.0)
            graph.replay()
            torch.cuda.synchronize()
            assert int(L.status.item()) == ss.ERR_SLOT_SHARED
            assert (L.out.cpu() == 5.0).all()
            assert_bits_equal(L.ssm.cpu(), ssm_h.cpu(), "ssm pool after a rejected replay")
            with pytest.raises(oracle.OracleError) as rej:
                oracle.decode_step(x[:3].contiguous(), z[:3].contiguous(), dt[:3].contiguous(), p.conv_w,
                                   p.conv_b, p.A_log, p.dt_bias, p.D, p.norm_w, p.norm_groups, p.eps, conv_o,
                                   ssm_o, L.dims.tuple4(), bad, [0, 0, 0])
            assert rej.value.status == oracle.ERR_SLOT_SHARED
            L.set_batch(slots, fresh, n)
        out_h = L.host_step(conv_h, ssm_h, slots, fresh)
        graph.replay()
        _, out64 = oracle.decode_step(x, z, dt, p.conv_w, p.conv_b, p.A_log, p.dt_bias, p.D, p.norm_w,
                                      p.norm_groups, p.eps, conv_o, ssm_o, L.dims.tuple4(), slots, fresh)
        torch.cuda.synchronize()
        assert int(L.status.item()) == ss.OK, step
        assert_bits_equal(L.out[:n].cpu(), out_h.cpu(), f"graph step {step} output")
        assert_bits_equal(L.conv.cpu(), conv_h.cpu(), f"graph step {step} conv pool")
        assert_bits_equal(L.ssm.cpu(), ssm_h.cpu(), f"graph step {step} ssm pool")
        # the replayed step against the oracle on the same batch
        check_act(L.out[:n].cpu(), out64, f"graph step {step} output vs oracle")
        assert_bits_equal(L.conv.cpu(), conv_o, f"graph step {step} conv pool vs oracle")
        rl = slot_rel_l2(L.ssm, ssm_o, slots)
        assert rl <= STATE_DECODE_REL_L2, f"graph step {step}: ssm rel L2 {rl:.3g}"
