"""Failure detection without a GPU fault: the bounded mbarrier wait that every
tensor-core kernel uses gives up on a barrier that nothing arrives at, raises the
CTA's abort flag and returns a status the host reads; the context then still
computes correct results. (Host-side failure detection, the batch checks before any
launch, is tested in test_abi_host.py and the rejection tests.)"""
import pytest
import torch

import oracle
import selective_scan_gb300 as ss
import workloads as W
from tests.util import check_act


def test_selftest_host_rejections(product_lib):
    assert product_lib.mamba2_selftest_bounded_wait(None, None) == ss.ERR_INVALID_ARGUMENT
    assert product_lib.mamba2_selftest_bounded_wait(0x10002, None) == ss.ERR_INVALID_ARGUMENT


@pytest.mark.gpu
def test_bounded_wait_gives_up_and_context_survives():
    from tests.gpu_util import device, gpu_conv
    dev = device()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    assert ss.library().mamba2_selftest_bounded_wait(status.data_ptr(), stream) == ss.OK
    torch.cuda.synchronize()
    assert int(status.item()) == 2, "the wait must give up with the abort flag raised"
    # the context still runs the path: a small prefill's conv against the oracle
    wl = W.tiny()
    p, b = wl.params, wl.batch
    xbc, _ = gpu_conv(wl, dev)
    torch.cuda.synchronize()
    _, xbc64 = oracle.causal_conv1d(wl.xBC, p.conv_w, p.conv_b, wl.conv_state.clone(), b.cu_seqlens, b.slots,
                                    b.fresh)
    check_act(xbc.cpu(), xbc64, "conv after the self-test")
