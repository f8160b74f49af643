"""Byte accounting against the figures printed in Table 14 and §5.5."""
import os

import pytest

from oracle.accounting import (bf16_row_bytes, decode_bytes, int4_row_bytes,
                               proxy_buffer_bytes, vl_overhead, window_overhead)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "table14_memory.txt")


def _rows():
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def test_row_sizes():
    assert int4_row_bytes() == 80 and int4_row_bytes(with_meta=False) == 64
    assert bf16_row_bytes() == 256


@pytest.mark.parametrize("row", [r for r in _rows() if r[0] != "proxy_buffer_bytes"])
def test_table14_percentages(row):
    name, prefix, pct = row[0], int(row[1]), float(row[2])
    if name == "vl_tokens":
        got = 100 * vl_overhead(0.05)
    else:  # window and staging buffer both hold W = 128 BF16 rows
        got = 100 * window_overhead(prefix, 128)
    assert abs(got - pct) < 0.1, (name, got, pct)


def test_proxy_buffer_size():
    row = [r for r in _rows() if r[0] == "proxy_buffer_bytes"][0]
    assert proxy_buffer_bytes(int(row[1]), int(row[2])) == int(row[3])


def test_decode_bytes_llama_32k():
    # 8 KV heads, 31008 4-bit rows, 1632 vertical-line rows, 128 tail rows
    b = decode_bytes(1, 32, 8, 128, 31008, 1632, 128)
    assert b == 8 * (31008 * 160 + 1760 * 512) + 2 * 32 * 128 * 2
    assert abs(b / 1e6 - 46.9) < 0.1
