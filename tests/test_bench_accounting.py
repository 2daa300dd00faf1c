"""The algorithmic byte and FLOP counts bench.py divides by its timings (the
roofline numerators), against the same counts worked out by hand from the ops'
interface tensors (gllm PR #85 "feat(backend): Mamba2 ops, with CPU reference
implementations", "Ops": what each op reads and writes).

Per token of a bf16 prefill: the conv reads and writes conv_dim channels; the scan
reads xbc (conv_dim) and dt (heads) and writes y (d_inner); the norm reads y and z
and writes the output (d_inner each). Per sequence of a decode step: the fp32 SSM
state and the kernel-1 rows of conv history are read and written once; the token's
xBC, z and dt are read and the output written.
"""
import bench
import workloads as W


def test_prefill_bytes_per_token():
    # 48 heads x 64, d_state 128, 1 group: conv_dim 3328, d_inner 3072
    d = W.DIMS_48H
    assert bench.conv_bytes(1, d) == 2 * 3328 * 2 == 13_312
    assert bench.scan_bytes(1, d, state_rw=0) == (3328 + 48 + 3072) * 2 == 12_896
    assert bench.norm_bytes(1, d) == 3 * 3072 * 2 == 18_432
    assert 13_312 + 12_896 + 18_432 == 44_640
    # the 130m shape (24 heads): conv_dim 1792, d_inner 1536
    d = W.DIMS_130M
    per_tok = bench.conv_bytes(1, d) + bench.scan_bytes(1, d, state_rw=0) + bench.norm_bytes(1, d)
    assert per_tok == 2 * 1792 * 2 + (1792 + 24 + 1536) * 2 + 3 * 1536 * 2 == 23_088


def test_scan_state_bytes_and_flops():
    d = W.DIMS_48H
    # one sequence's fp32 state, written once at the end of the call
    assert bench.scan_bytes(0, d) == 48 * 64 * 128 * 4 == 1_572_864
    # the chunked algorithm per token: per head 2 (Q P + 2 P N), per group 2 Q N
    assert bench.scan_flops(1, d, Q=64) == 48 * 2 * (64 * 64 + 2 * 64 * 128) + 2 * 64 * 128 == 1_982_464
    assert bench.scan_flops(1, d, Q=128) == 48 * 2 * (128 * 64 + 2 * 64 * 128) + 2 * 128 * 128 == 2_392_064


def test_decode_bytes_per_sequence():
    d = W.DIMS_48H
    ssm = 2 * 48 * 64 * 128 * 4          # state read and written
    conv = 2 * 3 * 3328 * 2              # history read and written
    io = 3328 * 2 + 3072 * 2 + 48 * 2 + 3072 * 2  # xBC, z, dt in; output out
    assert (ssm, conv, io) == (3_145_728, 39_936, 19_040)
    assert bench.decode_bytes_per_seq(d) == ssm + conv + io == 3_204_704
    # 256 sequences a step: 820.4 MB
    assert bench.decode_bytes_per_seq(d) * 256 == 820_404_224


def test_prefill_call_bytes_with_states():
    # the 130m-shaped prefill: one fresh sequence of 2 048 tokens; its history
    # (3 rows of 1 792 bf16 channels) and fp32 state (24 x 64 x 128) are written once
    wl = W.prefill_130m()
    assert bench.prefill_call_bytes(wl) == 2048 * 23_088 + 3 * 1792 * 2 + 24 * 64 * 128 * 4 == 48_081_408
    # the varlen batch: 8 sequences, 4 of them resuming (their history and state are
    # also read), 16 407 tokens with seed 2
    wl = W.varlen_130m()
    assert wl.batch.rows == 16_407 and sum(1 for f in wl.batch.fresh if not f) == 4
    per_seq = 3 * 1792 * 2 + 24 * 64 * 128 * 4
    assert bench.prefill_call_bytes(wl) == 16_407 * 23_088 + (8 + 4) * per_seq


def test_mamba3_bytes_frozen_batch():
    # Mamba-3 SISO forward, seed-5 frozen batch: 5 sequences, 3 109 tokens, 32 heads x 64,
    # Q/K width 128, 32 angles. Inputs: q, k [T,128] bf16; v, z [T,32,64] bf16; adt, dt
    # [T,32] f32; trap [T,32] bf16; angles [T,32] bf16; biases [32,128] f32; d [32] f32.
    # Outputs: out [T,32,64] bf16; per (sequence, head) angle 32 bf16, state 64x128 f32,
    # k 128 f32, v 64 bf16.
    b = W.mamba3_batch(seed=5)
    assert b.rows == 3109 and len(b.cu_seqlens) == 6
    reads = 2 * 3109 * 128 * 2 + 2 * 3109 * 32 * 64 * 2 + 3109 * 32 * (4 + 4 + 2) + 3109 * 32 * 2 + 2 * 32 * 128 * 4 + 32 * 4
    writes = 3109 * 32 * 64 * 2 + 5 * 32 * (32 * 2 + 64 * 128 * 4 + 128 * 4 + 64 * 2)
    assert (reads, writes) == (28_287_488, 18_089_984)
    assert bench.mamba3_bytes(b) == 46_377_472


def test_prefill_fused_bytes():
    """The fused minimum at the 65 536-token shape: 19 040 bytes a token (xBC 6 656,
    z 6 144, dt 96, output 6 144) plus one fresh sequence's conv history and SSM
    state written once."""
    wl = W.long_prefill(tokens=65536, decode_steps=1)
    assert bench.prefill_fused_bytes(wl) == 65536 * 19_040 + 3 * 3328 * 2 + 48 * 64 * 128 * 4
