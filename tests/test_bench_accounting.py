"""The algorithmic work the benchmark divides by (CPU): bytes and flops of one decode call,
checked against hand-counted values for the cache layout (per packed C4 token: 256 B of latent
codes, 32 B of k_R codes, 16 B of latent metadata; 256 B of k_R metadata per page; 1152 B per
BF16 token)."""
import math

import bench
import workloads


def test_c4r4_one_sequence_by_hand():
    w = workloads.Workload("acct", 1, 16, 8192, 4, 128)
    protected = 4 + 128
    packed = 8192 - protected
    pages = math.ceil((8192 - 128) / 128)  # pages holding packed tokens: 0 .. 62
    want = packed * (256 + 32 + 16) + pages * 256 + protected * 1152 + 16 * 1152 + 16 * 513 * 4
    assert want == 2_669_696
    assert bench.decode_bytes(w, [8192], 16) == want


def test_c2r4_and_short_sequences():
    w = workloads.Workload("acct2", 3, 16, 1000, 2, 64)
    per_tok = 128 + 32 + 16
    # T = 100: every token protected; T = 0: nothing but the query/output rows
    t1000 = (1000 - 132) * per_tok + math.ceil((1000 - 128) / 64) * 256 + 132 * 1152
    t100 = 100 * 1152
    rows = 3 * (16 * 1152 + 16 * 513 * 4)
    assert bench.decode_bytes(w, [1000, 100, 0], 16) == t1000 + t100 + rows


def test_bf16_bytes_and_flops():
    assert bench.bf16_decode_bytes([1000, 24], 16) == 1024 * 1152 + 2 * 16 * 1152 + 2 * 16 * 513 * 4
    assert bench.decode_flops([1000, 24], 64) == 1024 * 64 * 2 * (576 + 512)
