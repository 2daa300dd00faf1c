"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/*.h declares, and rejects malformed
RecurrentBatches before touching any device pointer, with the same status the
oracle returns (gllm PR #85 "feat(backend): Mamba2 ops, with CPU reference
implementations", section "Ops": out-of-range slot, shared slot, runs that do
not cover the rows)."""
import ctypes
import os
import re

import pytest

import oracle
import selective_scan_gb300 as ss
import workloads as W

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include")


def declared_functions():
    names = set()
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, h)).read(), flags=re.S)
            names.update(re.findall(r"\b(mamba[23]_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(product_lib):
    names = declared_functions()
    for op in ("mamba2_causal_conv1d", "mamba2_ssd_scan", "mamba2_gated_rmsnorm", "mamba2_decode_step",
               "mamba3_siso_varlen_forward"):
        assert op in names
    missing = [n for n in names if not hasattr(product_lib, n)]
    assert not missing, missing


def test_status_strings(product_lib):
    for code in range(8):
        s = ss.status_string(code)
        assert s.startswith("MAMBA2_")
    assert ss.status_string(ss.ERR_SLOT_SHARED) == "MAMBA2_ERR_SLOT_SHARED"


def test_state_bytes_match_oracle_and_page(product_lib):
    d = W.Dims(24, 64, 128, 1, 4)
    per_layer = ss.state_bytes_per_layer(d, ss.BF16)
    assert per_layer == oracle.state_bytes_per_layer(24, 64, 128, 1, 4, oracle.BF16)
    assert round(24 * per_layer / 2 ** 20, 2) == 18.25
    assert ss.state_bytes_per_layer(W.Dims(0, 64, 128, 1, 4)) == -1


# fake, 16-byte aligned device addresses: a rejected call must never touch them
FAKE = [0x10000 * (i + 1) for i in range(16)]

BAD = [
    ("slot out of range", [0, 3, 7], [0, 5], ss.ERR_SLOT_OUT_OF_RANGE),
    ("negative slot", [0, 3, 7], [-1, 0], ss.ERR_SLOT_OUT_OF_RANGE),
    ("shared slot", [0, 3, 7], [2, 2], ss.ERR_SLOT_SHARED),
    ("runs short", [0, 3, 6], [0, 1], ss.ERR_RUNS_DONT_COVER_ROWS),
    ("runs long", [0, 3, 9], [0, 1], ss.ERR_RUNS_DONT_COVER_ROWS),
    ("non-monotone", [0, 5, 4], [0, 1], ss.ERR_RUNS_DONT_COVER_ROWS),
    ("nonzero start", [2, 3, 7], [0, 1], ss.ERR_RUNS_DONT_COVER_ROWS),
    ("range before shared", [0, 3, 7], [9, 9], ss.ERR_SLOT_OUT_OF_RANGE),
]


@pytest.mark.parametrize("name,cu,slots,status", BAD, ids=[b[0] for b in BAD])
def test_rejections_match_oracle(product_lib, name, cu, slots, status):
    num_slots, rows = 4, 7
    assert oracle.validate_batch(cu, slots, num_slots, rows) == status
    lib = product_lib
    b = ss._Batch(cu, slots, [0] * len(slots))
    st = lib.mamba2_causal_conv1d(FAKE[0], FAKE[1], FAKE[2], FAKE[3], FAKE[4], num_slots, rows, 128, 4,
                                  ss.BF16, b.ref(), None)
    assert st == status
    d = ss.Dims(4, 16, 16, 2, 4)
    st = lib.mamba2_ssd_scan(FAKE[0], FAKE[1], FAKE[2], FAKE[3], FAKE[4], FAKE[5], FAKE[6], num_slots, rows,
                             ctypes.byref(d), ss.BF16, b.ref(), None, 0, None)
    assert st == status


def test_decode_rejections(product_lib):
    lib = product_lib
    d = ss.Dims(4, 16, 16, 2, 4)

    def call(slots, cu=None, num_slots=4):
        b = ss._Batch(cu, slots, [0] * len(slots))
        return lib.mamba2_decode_step(*FAKE[:10], 2, 1e-5, FAKE[10], FAKE[11], num_slots, ctypes.byref(d),
                                      ss.BF16, b.ref(), None)

    assert call([0, 4]) == ss.ERR_SLOT_OUT_OF_RANGE
    assert call([1, 1]) == ss.ERR_SLOT_SHARED
    assert call([0, 1], cu=[0, 1, 3]) == ss.ERR_RUNS_DONT_COVER_ROWS  # 3 rows != 2 sequences
    assert call([0, 1], cu=[0, 2, 2]) == ss.ERR_INVALID_ARGUMENT  # a run of 2 tokens


def test_argument_checks(product_lib):
    lib = product_lib
    b = ss._Batch([0, 4], [0], [1])
    # conv_dim * 2 bytes not a multiple of 16
    assert lib.mamba2_causal_conv1d(FAKE[0], FAKE[1], FAKE[2], FAKE[3], FAKE[4], 1, 4, 100, 4, ss.BF16,
                                    b.ref(), None) == ss.ERR_NOT_IMPLEMENTED
    # misaligned activation pointer
    assert lib.mamba2_causal_conv1d(FAKE[0], FAKE[1] + 2, FAKE[2], FAKE[3], FAKE[4], 1, 4, 128, 4, ss.BF16,
                                    b.ref(), None) == ss.ERR_INVALID_ARGUMENT
    # dst aliasing x
    assert lib.mamba2_causal_conv1d(FAKE[1], FAKE[1], FAKE[2], FAKE[3], FAKE[4], 1, 4, 128, 4, ss.BF16,
                                    b.ref(), None) == ss.ERR_INVALID_ARGUMENT
    # heads not a multiple of ngroups
    d = ss.Dims(3, 16, 16, 2, 4)
    assert lib.mamba2_ssd_scan(*FAKE[:7], 1, 4, ctypes.byref(d), ss.BF16, b.ref(), None, 0,
                               None) == ss.ERR_INVALID_ARGUMENT
    # too many sequences for one call
    n = ss.MAX_SEQS + 1
    big = ss._Batch(list(range(n + 1)), list(range(n)), [1] * n)
    assert lib.mamba2_causal_conv1d(FAKE[0], FAKE[1], FAKE[2], FAKE[3], FAKE[4], n, n, 128, 4, ss.BF16,
                                    big.ref(), None) == ss.ERR_INVALID_ARGUMENT
    # norm: groups must divide dim
    assert lib.mamba2_gated_rmsnorm(FAKE[0], FAKE[1], FAKE[2], FAKE[3], 2, 64, 3, 1e-5, ss.BF16,
                                    None) == ss.ERR_INVALID_ARGUMENT


def _prefill_host(lib, cu, slots, piece_rows=64, ws=None, ws_bytes=1 << 30, num_slots=4, fresh=None):
    d = ss.Dims(4, 16, 16, 2, 4)
    b = ss._Batch(cu, slots, fresh if fresh is not None else [0] * len(slots))
    return lib.mamba2_prefill_host(*FAKE[:10], 2, 1e-5, FAKE[10], FAKE[11], num_slots, ctypes.byref(d), ss.BF16,
                                   b.ref(), piece_rows, FAKE[12] if ws is None else ws, ws_bytes, None)


def test_prefill_host_rejections(product_lib):
    """The streamed host prefill applies the ops' batch checks to the whole batch,
    then its own (piece size, workspace), all before anything is enqueued."""
    lib = product_lib
    assert _prefill_host(lib, [0, 3, 7], [0, 4]) == ss.ERR_SLOT_OUT_OF_RANGE
    assert _prefill_host(lib, [0, 3, 7], [2, 2]) == ss.ERR_SLOT_SHARED
    assert _prefill_host(lib, [0, 5, 4], [0, 1]) == ss.ERR_RUNS_DONT_COVER_ROWS
    assert _prefill_host(lib, [2, 3, 7], [0, 1]) == ss.ERR_RUNS_DONT_COVER_ROWS
    assert _prefill_host(lib, [0, 3, 7], [0, 1], piece_rows=0) == ss.ERR_INVALID_ARGUMENT
    d = ss.Dims(4, 16, 16, 2, 4)
    b = ss._Batch([0, 3, 7], [0, 1], [1, 0])
    need = lib.mamba2_prefill_host_workspace_bytes(ctypes.byref(d), ss.BF16, b.ref(), 64)
    assert need > 0
    assert _prefill_host(lib, [0, 3, 7], [0, 1], ws_bytes=need - 1) == ss.ERR_WORKSPACE_TOO_SMALL
    assert _prefill_host(lib, [0, 3, 7], [0, 1], ws=FAKE[12] + 16, ws_bytes=need) == ss.ERR_INVALID_ARGUMENT
    assert lib.mamba2_prefill_host_workspace_bytes(ctypes.byref(d), ss.BF16, b.ref(), 0) == 0


def test_prefill_host_workspace_grows_with_piece(product_lib):
    """Piece buffers scale with the piece size (capped at the call's rows)."""
    lib = product_lib
    d = ss.Dims(24, 64, 128, 1, 4)
    b = ss._Batch([0, 5000], [0], [1])
    sizes = [lib.mamba2_prefill_host_workspace_bytes(ctypes.byref(d), ss.BF16, b.ref(), p)
             for p in (256, 1024, 5000, 100000)]
    assert sizes[0] < sizes[1] < sizes[2] == sizes[3]
    conv_dim, d_inner = 24 * 64 + 2 * 128, 24 * 64
    per_row = 2 * (conv_dim + 2 * d_inner + 24) * 2 + (conv_dim + d_inner) * 2  # double-buffered in/out, xbc, y
    assert sizes[2] >= 5000 * per_row


def test_decode_device_batch_host_rejections(product_lib):
    """mamba2_decode_step_device: the host-side checks (nothing enqueued) reject a
    capacity outside [1, MAMBA2_MAX_SEQS], null or misaligned batch pointers and bad
    scalars; the batch itself is checked on the device (GPU tests)."""
    lib = product_lib
    d = ss.Dims(4, 16, 16, 2, 4)

    def call(capacity=4, slots=FAKE[12], fresh=FAKE[13], n=FAKE[14], status=FAKE[15], groups=2, eps=1e-5,
             num_slots=8, dst=FAKE[0]):
        return lib.mamba2_decode_step_device(dst, *FAKE[1:10], groups, eps, FAKE[10], FAKE[11], num_slots,
                                             ctypes.byref(d), ss.BF16, slots, fresh, n, capacity, status, None)

    assert call(capacity=0) == ss.ERR_INVALID_ARGUMENT
    assert call(capacity=ss.MAX_SEQS + 1) == ss.ERR_INVALID_ARGUMENT
    for kw in ({"slots": None}, {"fresh": None}, {"n": None}, {"status": None}, {"dst": None}):
        assert call(**kw) == ss.ERR_INVALID_ARGUMENT, kw
    for kw in ({"slots": FAKE[12] + 2}, {"n": FAKE[14] + 1}, {"status": FAKE[15] + 2}, {"dst": FAKE[0] + 4}):
        assert call(**kw) == ss.ERR_INVALID_ARGUMENT, kw
    assert call(groups=0) == ss.ERR_INVALID_ARGUMENT
    assert call(eps=-1.0) == ss.ERR_INVALID_ARGUMENT
    assert call(num_slots=-1) == ss.ERR_INVALID_ARGUMENT


def _m3_call(lib, cu, rows=20, heads=2, headdim=64, d_state=128, rot_dim=32, ptrs=None):
    p = ptrs if ptrs is not None else FAKE
    arr = (ctypes.c_int32 * len(cu))(*cu)
    return lib.mamba3_siso_varlen_forward(*p[:16], arr, len(cu) - 1, rows, heads, headdim, d_state, rot_dim, None)


def test_mamba3_rejects_before_touching_memory(product_lib):
    """Mamba-3 SISO forward: malformed calls return their status on the host (the fake
    device pointers are never dereferenced)."""
    lib = product_lib
    assert _m3_call(lib, [0, 12, 21]) == ss.ERR_RUNS_DONT_COVER_ROWS
    assert _m3_call(lib, [0, 12, 10, 20]) == ss.ERR_RUNS_DONT_COVER_ROWS
    assert _m3_call(lib, [1, 12, 20]) == ss.ERR_RUNS_DONT_COVER_ROWS
    assert _m3_call(lib, [0, 12, 20], rot_dim=65) == ss.ERR_INVALID_ARGUMENT   # 2 R > N
    assert _m3_call(lib, [0, 12, 20], heads=0) == ss.ERR_INVALID_ARGUMENT
    assert _m3_call(lib, [0, 12, 20], headdim=32) == ss.ERR_NOT_IMPLEMENTED
    assert _m3_call(lib, [0, 12, 20], d_state=64, rot_dim=16) == ss.ERR_NOT_IMPLEMENTED
    misaligned = list(FAKE)
    misaligned[5] += 2   # q
    assert _m3_call(lib, [0, 12, 20], ptrs=misaligned) == ss.ERR_INVALID_ARGUMENT
    nulls = list(FAKE)
    nulls[2] = None      # final_ssm
    assert _m3_call(lib, [0, 12, 20], ptrs=nulls) == ss.ERR_INVALID_ARGUMENT
    # an empty batch is a no-op
    assert lib.mamba3_siso_varlen_forward(*([None] * 16), None, 0, 0, 2, 64, 128, 32, None) == ss.OK
