"""Byte accounting of the oracle against the numbers the pages print.

Golden table: tests/golden/llama3_8b_kv_bytes.txt ("KV-Cache Quantization: I Ran the
Experiments So You Don't Have To", "Component 1", table under Figure 3).
"""
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "llama3_8b_kv_bytes.txt")


def _rows():
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            yield [float(x) for x in line.split()]


def test_llama3_8b_table(oracle_lib):
    rows = list(_rows())
    assert len(rows) == 4
    for ctx, *gb in rows:
        for bits, want in zip((16, 8, 4, 2), gb):
            got = oracle.kv_bytes_plain(32, 8, 128, bits, ctx, 1) / 1e9
            assert round(got, 2) == want, (ctx, bits, got, want)


def test_llama3_8b_prose_figures(oracle_lib):
    assert oracle.kv_bytes_plain(32, 8, 128, 16, 1, 1) == 128 * 1024          # 128 KiB per token
    assert round(oracle.kv_bytes_plain(32, 8, 128, 16, 32768, 64) / 1e9) == 275
    assert round(oracle.kv_bytes_plain(32, 8, 128, 4, 32768, 64) / 1e9) == 69


def test_seq_bytes_metadata_is_one_bit_per_element(oracle_lib):
    """fp16 scale + zero per 32 elements add 32/32 = 1 bit per element: 3 bits per
    element at 2-bit (96 B per token and kv head at D = 128), 5 bits at 4-bit (160 B)."""
    for bits, per_token in ((2, 96), (4, 160)):
        cfg = oracle.Cfg(bits=bits, num_q_heads=32, num_kv_heads=8, head_dim=128)
        ring = 2 * (128 + 32) * 128 * 2
        for cap in (0, 32, 4096, 32768):
            assert oracle.seq_bytes(cfg, cap) == 8 * (cap * per_token + ring)
        assert per_token * 8 == (bits + 1) * 2 * 128
