"""Pins of the oracle's number formats (MXFP4 main KV, FP8 SWA / indexer keys).

Independent anchors: hand-worked vectors (tests/golden/*.txt, each citing the
page that names the format), the E2M1 / E4M3 value tables of the OCP
definitions, torch's own float8_e4m3fn conversion (a separate library
routine), exhaustive round trips and scaling invariances.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _lines(name):
    with open(os.path.join(GOLD, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


# ---------------------------------------------------------------- E2M1
def test_e2m1_value_table():
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]          # OCP FP4 E2M1 grid
    for c in range(8):
        assert oracle.e2m1_value(c) == mags[c]
        assert oracle.e2m1_value(c | 8) == -mags[c]
    assert np.signbit(oracle.e2m1_value(8))


def test_e2m1_saturates_far_beyond_the_grid():
    for v in (6.5, 1e3, 1e30, 6.7e35, 3e38):
        assert oracle.e2m1_encode(v) == 7 and oracle.e2m1_encode(-v) == 15


def test_e2m1_roundtrip_all_codes():
    for c in range(16):
        assert oracle.e2m1_encode(oracle.e2m1_value(c)) == c


def test_e2m1_nearest_and_ties():
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    rng = np.random.default_rng(1)
    for v in rng.uniform(0, 8, 4000):
        c = oracle.e2m1_encode(float(v))
        d = np.abs(grid - v)
        assert d[c] == d.min()
    # midpoints go to the even-mantissa neighbour
    for mid, want in [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6)]:
        assert oracle.e2m1_encode(mid) == want
        assert oracle.e2m1_encode(-mid) == want | 8
    assert oracle.e2m1_encode(7.99) == 7 and oracle.e2m1_encode(100.0) == 7


# ---------------------------------------------------------------- MXFP4
def test_mx_exponent_definition():
    # X = floor(log2 amax) - 2 (E2M1's largest exponent is 2)
    assert oracle.mx_exponent(1.0) == -2
    assert oracle.mx_exponent(6.0) == 0
    assert oracle.mx_exponent(7.99) == 0
    assert oracle.mx_exponent(8.0) == 1
    assert oracle.mx_exponent(0.3) == -4
    assert oracle.mx_exponent(2.0 ** -120) == -122
    assert oracle.mx_exponent(1e-40) == -127        # clamped at the E8M0 floor
    assert oracle.mx_exponent(0.0) == 0


def test_mxfp4_golden_vectors():
    for ln in _lines("mxfp4_vectors.txt"):
        sb, vals, codes = [p.split() for p in ln.split("|")]
        x = np.zeros((1, 512), np.float32)
        x[0, :32] = np.array([float(v) for v in vals], np.float32)
        c, s = oracle.quant_mxfp4(x)
        assert s[0, 0] == int(sb[0])
        want = [int(h, 16) for h in codes]
        got = [(c[0, i // 2] >> (4 * (i & 1))) & 15 for i in range(32)]
        assert got == want


def test_mxfp4_layout_and_roundtrip():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((64, 512)).astype(np.float32) * np.float32(3.0)
    c, s = oracle.quant_mxfp4(x)
    assert c.shape == (64, 256) and s.shape == (64, 16)
    deq = oracle.dequant_mxfp4(c, s)
    # element 2i sits in the low nibble of byte i
    for r in range(4):
        for d in (0, 1, 2, 3, 100, 511):
            code = (c[r, d // 2] >> (4 * (d & 1))) & 15
            X = int(s[r, d // 32]) - 127
            assert deq[r, d] == oracle.e2m1_value(code) * 2.0 ** X
    # nearest representable under the block scale, saturating beyond 6*2^X
    for r in range(64):
        for b in range(16):
            X = int(s[r, b]) - 127
            blk = x[r, b * 32:(b + 1) * 32].astype(np.float64)
            grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6]) * 2.0 ** X
            for v, q in zip(blk, deq[r, b * 32:(b + 1) * 32]):
                target = min(abs(v), 6 * 2.0 ** X)
                assert abs(abs(q) - target) == np.abs(grid - target).min()
                assert q == 0 or np.sign(q) == np.sign(v)
    # quantise(dequantise(q)) == q
    c2, s2 = oracle.quant_mxfp4(deq.astype(np.float32))
    assert np.array_equal(c, c2) and np.array_equal(s, s2)


def test_mxfp4_power_of_two_scaling():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((16, 512)).astype(np.float32)
    c0, s0 = oracle.quant_mxfp4(x)
    for k in (-5, 3, 20):
        c, s = oracle.quant_mxfp4(x * np.float32(2.0 ** k))
        assert np.array_equal(c, c0)
        assert np.array_equal(s.astype(int), s0.astype(int) + k)


# ---------------------------------------------------------------- E4M3
def test_e4m3_golden_vectors():
    for ln in _lines("fp8_vectors.txt"):
        v, h = ln.split()
        assert oracle.e4m3_encode(float(v)) == int(h, 16), ln


def test_e4m3_decode_exhaustive():
    vals = [oracle.e4m3_value(c) for c in range(127)]
    assert vals[0] == 0.0 and vals[126] == 448.0
    assert all(a < b for a, b in zip(vals, vals[1:]))
    assert np.isnan(oracle.e4m3_value(0x7F)) and np.isnan(oracle.e4m3_value(0xFF))
    for c in list(range(127)) + list(range(128, 255)):
        assert oracle.e4m3_encode(oracle.e4m3_value(c)) == c
    # matches torch's reading of every code
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert t[c] == oracle.e4m3_value(c)


def test_e4m3_encode_matches_torch():
    rng = np.random.default_rng(11)
    # random magnitudes across the whole range, plus exact midpoints and their neighbours
    a = np.concatenate([
        rng.uniform(-464, 464, 20000),
        np.exp2(rng.uniform(-14, 8.8, 20000)) * rng.choice([-1, 1], 20000),
    ]).astype(np.float32)
    vals = np.array([oracle.e4m3_value(c) for c in range(127)])
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    a = np.concatenate([a, near, -near, [0.0, -0.0]]).astype(np.float32)
    a = a[np.abs(a) <= 464]        # torch's cast is non-saturating above 464
    want = torch.from_numpy(a).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in a], np.uint8)
    bad = np.nonzero(want != got)[0]
    assert bad.size == 0, (a[bad[:5]], want[bad[:5]], got[bad[:5]])


def test_quant_fp8_rows():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((32, 128)).astype(np.float32)
    c, s = oracle.quant_fp8(x)
    amax = np.abs(x).max(axis=1)
    assert np.array_equal(s, (amax / np.float32(448.0)).astype(np.float32))
    # the largest-magnitude element lands on +-448
    j = np.abs(x).argmax(axis=1)
    for r in range(32):
        assert c[r, j[r]] & 0x7F == 0x7E
    # zero row: scale 1, codes zero
    c0, s0 = oracle.quant_fp8(np.zeros((1, 512), np.float32))
    assert s0[0] == 1.0 and not c0.any()
    # power-of-two rescaling leaves the codes alone and scales s exactly
    c2, s2 = oracle.quant_fp8(x * np.float32(8.0))
    assert np.array_equal(c, c2) and np.array_equal(s2, s * np.float32(8.0))
    # dequantised error within half an E4M3 step of x / s: 2^-4 relative in the
    # normal range, 2^-10 * s (half the subnormal step) below it
    deq = oracle.dequant_fp8(c, s)
    bound = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * s[:, None]) * (1 + 1e-6)
    assert (np.abs(deq - x) <= bound).all()


# ---------------------------------------------------------------- FP4, 16-element blocks, E4M3 scale
# The block size and scale type the pages give for the FP4 cache
# ("DeepSeek-V4.1-Flash 架构详解" §4; "How DeepSeek V4.1 Flash beats 1.6T models"):
# 16 elements share one E4M3 scale.
def _brute_fp4_e4m3_block(vals):
    """Independent reference: nearest-value searches over the full E4M3 and
    E2M1 grids (torch for the fp32 divisions), ties to the even code."""
    e4 = np.array([oracle.e4m3_value(c) for c in range(127)])          # positive finite codes
    amax = np.float32(np.max(np.abs(vals)))
    q = float((torch.tensor(amax) / torch.tensor(6.0, dtype=torch.float32)).item())
    d = np.abs(e4 - q)
    best = np.flatnonzero(d == d.min())
    sb = int(best[0] if best.size == 1 else best[best % 2 == 0][0]) if q <= e4[-1] else 126
    sv = np.float32(e4[sb])
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    codes = []
    for v in vals:
        if sv == 0:
            codes.append(8 if np.signbit(v) else 0)
            continue
        y = float((torch.tensor(np.float32(v)) / torch.tensor(sv)).item())
        dd = np.abs(grid - min(abs(y), 6.0))
        cand = np.flatnonzero(dd == dd.min())
        c = int(cand[0] if cand.size == 1 else cand[cand % 2 == 0][0])
        codes.append(c | (8 if np.signbit(y) else 0))
    return sb, codes


def test_fp4_e4m3_hand_values():
    x = np.zeros((1, 512), np.float32)
    x[0, :16] = 1.0                          # s = e4m3(1/6) = 0.171875 (code 0x23), 1/s = 5.82 -> 6
    blk = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -6.0, 0.0, -0.0, 3.0, 4.0, 1.5, 0.5, 2.0]
    x[0, 16:32] = blk                        # amax 6 -> s = 1: the E2M1 ties land on even codes
    x[0, 32:48] = 6.2                        # s = e4m3(1.0333) = 1.0: 6.2 saturates to 6
    x[0, 48:64] = -0.0                       # amax 0: scale 0, sign bits only
    x[0, 64:80] = 2.0 ** -16                 # amax / 6 rounds to 0 in E4M3: scale 0
    codes, scales = oracle.quant_fp4_e4m3(x)
    assert scales.shape == (1, 32) and codes.shape == (1, 256)
    assert scales[0, 0] == 0x23 and oracle.e4m3_value(0x23) == 0.171875
    assert all(codes[0, i] == 0x77 for i in range(8))
    assert scales[0, 1] == 0x38                                         # 1.0
    want = [7, 0, 2, 2, 4, 4, 6, 6, 15, 0, 8, 5, 6, 3, 1, 4]
    got = [(codes[0, 8 + i // 2] >> (4 * (i % 2))) & 15 for i in range(16)]
    assert got == want
    assert scales[0, 2] == 0x38 and all(codes[0, 16 + i] == 0x77 for i in range(8))
    assert scales[0, 3] == 0 and all(codes[0, 24 + i] == 0x88 for i in range(8))
    assert scales[0, 4] == 0 and all(codes[0, 32 + i] == 0x00 for i in range(8))
    deq = oracle.dequant_fp4_e4m3(codes, scales)[0]
    assert np.all(deq[:16] == 6 * 0.171875)
    assert np.array_equal(deq[16:32], [6, 0, 1, 1, 2, 2, 4, 4, -6, 0, 0, 3, 4, 1.5, 0.5, 2])


def test_fp4_e4m3_matches_brute_force():
    rng = np.random.default_rng(17)
    x = rng.standard_normal((6, 512)).astype(np.float32)
    x[1] *= np.float32(1e-3)
    x[2] *= np.float32(3e3)                                              # scales near the top of E4M3
    x[3, ::7] = 0.0
    x[4] = np.round(x[4] * 4) / 4                                        # many exact grid points and ties
    x[5, :40] = np.float32(3e38)                                         # quotients far beyond 6: saturate
    x[5, 3] = np.float32(-1.7e38)
    codes, scales = oracle.quant_fp4_e4m3(x)
    for r in range(x.shape[0]):
        for b in range(32):
            sb, cs = _brute_fp4_e4m3_block(x[r, 16 * b:16 * b + 16])
            assert scales[r, b] == sb, (r, b)
            got = [(codes[r, 8 * b + i // 2] >> (4 * (i % 2))) & 15 for i in range(16)]
            assert got == cs, (r, b)


def test_fp4_e4m3_products_exact_in_bf16():
    """Every (element code, scale code) product is a bf16 value: the attention
    can dequantise this format exactly with one bf16 multiply."""
    for sb in range(127):
        s = oracle.e4m3_value(sb)
        for c in range(16):
            v = oracle.e2m1_value(c) * s
            assert float(torch.tensor(v, dtype=torch.float64).to(torch.bfloat16).double()) == v


def test_fp4_e4m3_bytes_per_entry():
    # 512 E2M1 codes (256 B) + 32 E4M3 scales = 288 B per entry (MXFP4: 256 + 16 = 272 B)
    x = np.ones((3, 512), np.float32)
    c4, s4 = oracle.quant_fp4_e4m3(x)
    cm, sm = oracle.quant_mxfp4(x)
    assert c4.nbytes // 3 + s4.nbytes // 3 == 288
    assert cm.nbytes // 3 + sm.nbytes // 3 == 272
