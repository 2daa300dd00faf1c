"""Comparison helpers shared by the tests (no method arithmetic here)."""
from __future__ import annotations

import torch

# Floating-point acceptance for activation outputs (y of the scan, the gated
# norm output, the conv output): each element within 2e-2 absolute plus one
# bf16 half-ulp (2^-8) relative of the oracle's unrounded double, and the
# relative L2 error over the tensor at most 1e-2.
ABS_TOL = 2e-2
REL_ULP = 2.0 ** -8
REL_L2 = 1e-2
# fp32 SSM state: relative L2 after chunked prefill / after decode.
STATE_PREFILL_REL_L2 = 1e-3
STATE_DECODE_REL_L2 = 1e-5


def rel_l2(got: torch.Tensor, ref: torch.Tensor) -> float:
    g = got.double().flatten()
    r = ref.double().flatten()
    den = torch.linalg.vector_norm(r).item()
    num = torch.linalg.vector_norm(g - r).item()
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / den


def check_act(got: torch.Tensor, ref64: torch.Tensor, what: str = "",
              abs_tol: float = ABS_TOL, rel_ulp: float = REL_ULP, rel_l2_tol: float = REL_L2):
    """Elementwise |g - r| <= abs_tol + rel_ulp*|r| and rel-L2 <= rel_l2_tol."""
    g = got.double().cpu()
    r = ref64.double().cpu()
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert torch.isfinite(g).all(), f"{what}: non-finite output"
    err = (g - r).abs()
    bound = abs_tol + rel_ulp * r.abs()
    bad = err > bound
    if bad.any():
        idx = bad.nonzero()[0].tolist()
        raise AssertionError(
            f"{what}: {int(bad.sum())} elements out of tolerance; first at {idx}: "
            f"got {g[tuple(idx)].item()} ref {r[tuple(idx)].item()} (max abs err {err.max().item():.3g})")
    rl = rel_l2(g, r)
    assert rl <= rel_l2_tol, f"{what}: rel L2 {rl:.3g} > {rel_l2_tol}"
    return err.max().item(), rl


def bits(t: torch.Tensor) -> torch.Tensor:
    """Raw bit pattern (for bit-exact comparisons that see NaN payloads)."""
    t = t.contiguous()
    if t.element_size() == 4:
        return t.view(torch.int32)
    if t.element_size() == 2:
        return t.view(torch.int16)
    if t.element_size() == 1:
        return t.view(torch.uint8)
    return t.view(torch.int64)


def assert_bits_equal(a: torch.Tensor, b: torch.Tensor, what: str = ""):
    a, b = bits(a.cpu()), bits(b.cpu())
    if not torch.equal(a, b):
        diff = (a != b).nonzero()
        raise AssertionError(f"{what}: {diff.shape[0]} elements differ bitwise; first at {diff[0].tolist()}")

