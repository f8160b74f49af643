"""The decode kernel's register-level reading of the quantised tile format,
emulated on the CPU for 4- and 8-bit codes.

mma.m16n8k16 fragments (PTX ISA, f16 A/B, f32 C), lane = 4 g + t:
  A a0 (row g, cols 2t, 2t+1)  a1 (row g+8, cols 2t, 2t+1)
    a2 (row g, cols 2t+8, 2t+9) a3 (row g+8, cols 2t+8, 2t+9)
  B b0 (rows 2t, 2t+1, col g)   b1 (rows 2t+8, 2t+9, col g)
  C c0, c1 (row g, cols 2t, 2t+1)  c2, c3 (row g+8, cols 2t, 2t+1)
Tiles are packed by ``pack_qblocks`` (the documented format); each lane's A
registers are formed from its code words exactly as the kernel does (masks,
shift, byte permute: the 16-bit halves hold c or 16 c as integers), its B
registers from the query / probabilities in the kernel's element order, and
the emulated products must equal plain dot products of the codes."""
import numpy as np
import pytest

from hybrid_precision_quantized_gb300 import pack_qblocks
from hybrid_precision_quantized_gb300 import _lib as L


def halves(x):
    return np.array([x & 0xFFFF, x >> 16], dtype=np.int64)


def byte_perm_odd(w):
    """__byte_perm(w, 0, 0x4341): bytes 1 and 3 of w into the low bytes of the halves."""
    return ((w >> 8) & 0xFF) | (((w >> 24) & 0xFF) << 16)


def words(region, lane, n):
    return [int.from_bytes(region[512 * (u // 4) + 16 * lane + 4 * (u % 4):][:4].tobytes(), "little")
            for u in range(n)]


def mma(acc, a, b):
    """acc[g][t][ci] += A B for one m16n8k16 step; a[lane] = (a0, a1, a2, a3)
    halves, b[lane] = (b0, b1) halves."""
    A = np.zeros((16, 16))
    Bm = np.zeros((16, 8))
    for lane in range(32):
        g, t = lane // 4, lane % 4
        a0, a1, a2, a3 = a[lane]
        A[g, 2 * t:2 * t + 2] = a0
        A[g + 8, 2 * t:2 * t + 2] = a1
        A[g, 2 * t + 8:2 * t + 10] = a2
        A[g + 8, 2 * t + 8:2 * t + 10] = a3
        b0, b1 = b[lane]
        Bm[2 * t:2 * t + 2, g] = b0
        Bm[2 * t + 8:2 * t + 10, g] = b1
    D = A @ Bm
    for lane in range(32):
        g, t = lane // 4, lane % 4
        acc[lane] += np.array([D[g, 2 * t], D[g, 2 * t + 1], D[g + 8, 2 * t], D[g + 8, 2 * t + 1]])


@pytest.mark.parametrize("bk", [4, 8])
def test_key_products_per_group(bk):
    """S = q . c per token, head and group of 32 (the kernel's C[q])."""
    rng = np.random.default_rng(bk)
    kc = rng.integers(0, 1 << bk, (64, 128), dtype=np.uint8)
    z = np.zeros((64, 4), np.float16)
    tile = pack_qblocks(kc, kc, z, z, z, z, bits_k=bk, bits_v=4).reshape(-1)[:L.qtile_bytes(bk, 4)]
    q = rng.integers(-8, 8, (8, 128))          # 8 heads
    region = tile[:256 * bk]
    C = [np.zeros((32, 4)) for _ in range(4)]
    for ks in range(8):
        a, b = [], []
        for lane in range(32):
            g, t = lane // 4, lane % 4
            if bk == 4:
                w = words(region, lane, 8)[ks]
                w8 = w >> 8
                a.append((halves(w & 0x000F000F), halves(w & 0x00F000F0), halves(w8 & 0x000F000F),
                          halves(w8 & 0x00F000F0)))
                e = 8 * (t + 4 * (ks // 2)) + 4 * (ks % 2)
            else:
                ws = words(region, lane, 16)
                w0, w1 = ws[2 * ks], ws[2 * ks + 1]
                a.append((halves(w0 & 0x00FF00FF), halves(w1 & 0x00FF00FF), halves(byte_perm_odd(w0)),
                          halves(byte_perm_odd(w1))))
                e = 16 * ks + 4 * t
            b.append((q[g, e:e + 2], q[g, e + 2:e + 4]))
        mma(C[ks // 2], a, b)
    for grp in range(4):
        want = kc[:16, 32 * grp:32 * grp + 32].astype(np.int64) @ q[:, 32 * grp:32 * grp + 32].T  # tokens x heads
        for lane in range(32):
            g, t = lane // 4, lane % 4
            hi = 16 if bk == 4 else 1           # 4-bit tokens g+8 arrive as 16 c
            got = C[grp][lane]
            assert got[0] == want[g, 2 * t] and got[1] == want[g, 2 * t + 1]
            assert got[2] == hi * want[g + 8, 2 * t] and got[3] == hi * want[g + 8, 2 * t + 1]


@pytest.mark.parametrize("bv", [4, 8])
def test_value_products_and_output_order(bv):
    """O[d][head] = sum over the 16 tokens of c[token][d] p[token][head], with
    the B operand in the kernel's (transposed probability) order and the
    epilogue's element order per m-tile."""
    rng = np.random.default_rng(10 + bv)
    vc = rng.integers(0, 1 << bv, (64, 128), dtype=np.uint8)
    z = np.zeros((64, 4), np.float16)
    tile = pack_qblocks(vc, vc, z, z, z, z, bits_k=4, bits_v=bv).reshape(-1)[:L.qtile_bytes(4, bv)]
    p = rng.integers(0, 5, (16, 8))            # tokens x heads
    region = tile[1024:1024 + 256 * bv]
    want = vc[:16].astype(np.int64).T @ p       # dims x heads
    for mt in range(8):
        acc = np.zeros((32, 4))
        a, b = [], []
        for lane in range(32):
            g, t = lane // 4, lane % 4
            if bv == 4:
                x = words(region, lane, 8)[mt]
                x8 = x >> 8
                a.append((halves(x & 0x000F000F), halves(x & 0x00F000F0), halves(x8 & 0x000F000F),
                          halves(x8 & 0x00F000F0)))
            else:
                ws = words(region, lane, 16)
                x0, x1 = ws[2 * mt], ws[2 * mt + 1]
                a.append((halves(x0 & 0x00FF00FF), halves(x1 & 0x00FF00FF), halves(byte_perm_odd(x0)),
                          halves(byte_perm_odd(x1))))
            b.append((p[2 * t:2 * t + 2, g], p[2 * t + 8:2 * t + 10, g]))
        mma(acc, a, b)
        for lane in range(32):
            g, t = lane // 4, lane % 4
            for ci in range(4):
                d = 32 * (mt // 2) + 4 * g + 2 * (mt % 2) + (ci >> 1)   # the same output order
                f = 16 if (bv == 4 and ci >= 2) else 1                     # 4-bit high nibbles
                assert acc[lane][ci] == f * want[d, 2 * t + (ci & 1)], (mt, lane, ci)
