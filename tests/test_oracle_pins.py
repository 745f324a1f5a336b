"""Pins for the CPU oracle: tie it to things other than itself.

Each ``check_*`` takes an oracle library handle, so the same pins also run
against copies of the oracle with a planted mistake (test_oracle_mutants.py)
to show that a plausible slip anywhere in the oracle fails at least one pin.

Independent sources used here:
  * the E2M1 magnitude list {0, .5, 1, 1.5, 2, 3, 4, 6} of the FP4 E2M1 format;
  * PyTorch's float8_e4m3fn decode (all 256 bytes) and fp32 -> e4m3 cast;
  * brute-force nearest-value searches (Python, exact rational comparisons);
  * the hand-worked block in tests/golden/hand_block.txt;
  * exact rational (fractions.Fraction) dot products on tiny inputs;
  * closed forms (one-hot activations, all-ones activations, zero tensors).
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E2M1_MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


# ---------------------------------------------------------------------------
# Independent references
# ---------------------------------------------------------------------------

def e2m1_ref(code: int) -> float:
    mag = E2M1_MAG[code & 7]
    return -mag if code & 8 else mag


def e4m3_torch_table() -> np.ndarray:
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def e4m3_brute(q: float) -> int:
    """Nearest finite non-negative E4M3 byte to q >= 0, ties to the even byte,
    values beyond the largest finite saturate (fp32 input, exact comparison)."""
    table = e4m3_torch_table()
    qf = Fraction(float(np.float32(q)))
    best, best_d = None, None
    for b in range(0x7F):  # 0x00..0x7E, all finite non-negative
        d = abs(Fraction(float(table[b])) - qf)
        if best is None or d < best_d or (d == best_d and b % 2 == 0):
            best, best_d = b, d
    return best


def e2m1_brute(v: float) -> int:
    """Nearest E2M1 code to fp32 v, ties to the even code, |v| > 6 -> 6, sign kept."""
    vf = float(np.float32(v))
    if math.isinf(vf):
        return 7 | (8 if vf < 0 else 0)
    a = Fraction(abs(vf))
    best, best_d = None, None
    for c in range(8):
        d = abs(Fraction(E2M1_MAG[c]) - a)
        if best is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    return best | (8 if math.copysign(1.0, vf) < 0 else 0)


def f32(v) -> np.float32:
    return np.float32(v)


def quantize_ref(w: np.ndarray):
    """The recipe re-derived with numpy fp32 ops and brute-force rounding."""
    w = np.asarray(w, np.float32)
    M, K = w.shape
    amax = f32(np.max(np.abs(w))) if w.size else f32(0)
    ts = f32(amax / f32(2688.0))
    table = e4m3_torch_table()
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros((M, K // 16), np.uint8)
    for m in range(M):
        for b in range(K // 16):
            blk = w[m, 16 * b:16 * b + 16]
            bamax = f32(np.max(np.abs(blk)))
            sb = 0
            if ts > 0:
                sb = e4m3_brute(f32(f32(bamax / f32(6.0)) / ts))
            scales[m, b] = sb
            d = f32(f32(table[sb]) * ts)
            c = [0 if d == 0 else e2m1_brute(f32(v / d)) for v in blk]
            for j in range(8):
                codes[m, 8 * b + j] = c[2 * j] | (c[2 * j + 1] << 4)
    return codes, scales, ts


def dequant_ref(codes, scales, ts) -> list[list[Fraction]]:
    table = e4m3_torch_table()
    M, K2 = codes.shape
    out = []
    for m in range(M):
        row = []
        for k in range(2 * K2):
            byte = int(codes[m, k // 2])
            c = (byte >> 4) if k & 1 else (byte & 0xF)
            row.append(Fraction(e2m1_ref(c)) * Fraction(float(table[scales[m, k // 16]]))
                       * Fraction(float(ts)))
        out.append(row)
    return out


def bf16_round(a) -> np.ndarray:
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_value(bits) -> float:
    return float(np.array([int(bits) << 16], np.uint32).view(np.float32)[0])


def read_golden_block():
    vals = {}
    with open(os.path.join(GOLDEN, "hand_block.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            vals[k] = v
    w = np.array([float(t) for t in vals["w"].split()], np.float32)
    codes = [int(t, 16) for t in vals["codes"].split()]
    return w, int(vals["scale_byte"], 16), codes


# ---------------------------------------------------------------------------
# Pins (each raises AssertionError on a mismatch)
# ---------------------------------------------------------------------------

def check_e2m1_table(lib):
    for c in range(16):
        got = oracle.e2m1_value(c, lib=lib)
        exp = e2m1_ref(c)
        assert got == exp and math.copysign(1, got) == math.copysign(1, exp), (c, got, exp)


def check_e4m3_table(lib):
    table = e4m3_torch_table()
    for b in range(256):
        got = oracle.e4m3_value(b, lib=lib)
        if np.isnan(table[b]):
            assert math.isnan(got), b
        else:
            assert got == table[b], (hex(b), got, table[b])
    # spot values of the format
    assert oracle.e4m3_value(0x01, lib=lib) == 2.0 ** -9
    assert oracle.e4m3_value(0x08, lib=lib) == 2.0 ** -6
    assert oracle.e4m3_value(0x38, lib=lib) == 1.0
    assert oracle.e4m3_value(0x7E, lib=lib) == 448.0


def e4m3_probe_values():
    table = e4m3_torch_table()
    pos = sorted(set(float(table[b]) for b in range(0x7F)))
    vals = []
    for a, b in zip(pos, pos[1:]):
        mid = np.float32((a + b) / 2)  # exact in fp32 for this range
        vals += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(1e9)), np.float32(a)]
    vals += [np.float32(v) for v in (448.0, 450.0, 463.99, 464.0, 500.0, 1e6, 3e38, 2.0 ** -10, 2.0 ** -11, 1e-30, 0.0)]
    rng = np.random.default_rng(7)
    vals += list((rng.standard_normal(400) ** 2 * 30).astype(np.float32))
    vals += list(np.exp(rng.uniform(-9, 6.2, 400)).astype(np.float32))
    return vals


def check_e4m3_encode(lib):
    for q in e4m3_probe_values():
        assert oracle.e4m3_encode(q, lib=lib) == e4m3_brute(q), (repr(q),)


def check_e4m3_encode_vs_torch(lib):
    vals = [v for v in e4m3_probe_values() if v < 464.0]
    t = torch.tensor(np.array(vals, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(v, lib=lib) for v in vals], np.uint8)
    assert np.array_equal(got, t)


def e2m1_probe_values():
    grid = E2M1_MAG
    vals = []
    for a, b in zip(grid, grid[1:]):
        mid = np.float32((a + b) / 2)
        vals += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(9)), np.float32(a)]
    vals += [np.float32(v) for v in (6.0, 6.5, 7.0, 100.0, 3e38, np.inf)]
    vals = vals + [np.float32(-v) for v in vals]
    rng = np.random.default_rng(11)
    vals += list(rng.uniform(-8, 8, 800).astype(np.float32))
    vals += [np.float32(-0.0), np.float32(-0.2), np.float32(-1e-30)]
    return vals


def check_e2m1_encode(lib):
    for v in e2m1_probe_values():
        assert oracle.e2m1_encode(v, lib=lib) == e2m1_brute(v), (repr(v),)


def check_hand_block(lib):
    w, sb_exp, codes_exp = read_golden_block()
    codes, scales, ts = oracle.quantize(w.reshape(1, 16), lib=lib)
    assert ts == f32(f32(0.6) / f32(2688.0))
    assert scales[0, 0] == sb_exp
    got = []
    for byte in codes[0]:
        got += [int(byte) & 0xF, int(byte) >> 4]
    assert got == codes_exp, (got, codes_exp)
    # all-ones activation: closed form ts * 448 * sum of decoded codes
    x = bf16_round(np.ones((1, 16), np.float32))
    y, A = oracle.gemv(x, codes, scales, ts, lib=lib)
    exact = float(ts) * 448.0 * sum(e2m1_ref(c) for c in codes_exp)
    assert abs(y[0, 0] - exact) <= 1e-12 * abs(exact)
    assert abs(A[0, 0] - float(ts) * 448.0 * sum(abs(e2m1_ref(c)) for c in codes_exp)) <= 1e-12


def check_quantize_random(lib):
    rng = np.random.default_rng(3)
    for (M, K, scale) in [(3, 48, 0.02), (2, 32, 1.0), (4, 16, 1e-3)]:
        w = (rng.standard_normal((M, K)) * scale).astype(np.float32)
        # heavy-tailed elements give large and subnormal block scales
        w[rng.random((M, K)) < 0.05] *= 40.0
        w[0, :16] *= 1e-4  # a block far below the tensor max
        c, s, ts = oracle.quantize(w, lib=lib)
        rc, rs, rts = quantize_ref(w)
        assert ts == rts
        assert np.array_equal(s, rs), (s, rs)
        assert np.array_equal(c, rc)


def check_quantize_special(lib):
    # all-zero tensor: ts 0, scale bytes 0, codes 0
    c, s, ts = oracle.quantize(np.zeros((2, 32), np.float32), lib=lib)
    assert ts == 0 and not c.any() and not s.any()
    # a zero block inside a non-zero tensor, and signed tiny values
    w = np.zeros((1, 32), np.float32)
    w[0, 16:] = np.linspace(-1, 1, 16, dtype=np.float32)
    w[0, 17] = -1e-3  # rounds to magnitude 0 -> keeps its sign (0x8)
    c, s, ts = oracle.quantize(w, lib=lib)
    assert s[0, 0] == 0 and not c[0, :8].any()
    assert (int(c[0, 8]) >> 4) == 0x8
    rc, rs, rts = quantize_ref(w)
    assert np.array_equal(c, rc) and np.array_equal(s, rs)


def check_gemv_exact_small(lib):
    rng = np.random.default_rng(5)
    M, K, N = 5, 48, 3  # non-square, several tokens, 3 blocks per row
    w = (rng.standard_normal((M, K)) * 0.02).astype(np.float32)
    codes, scales, ts = oracle.quantize(w, lib=lib)
    xb = bf16_round(rng.standard_normal((N, K)).astype(np.float32) * np.array([[1.0], [8.0], [0.5]], np.float32))
    y, A = oracle.gemv(xb, codes, scales, ts, lib=lib)
    wq = dequant_ref(codes, scales, ts)
    for n in range(N):
        for m in range(M):
            terms = [wq[m][k] * Fraction(bf16_value(xb[n, k])) for k in range(K)]
            exact = sum(terms, Fraction(0))
            aexact = sum((abs(t) for t in terms), Fraction(0))
            assert abs(Fraction(y[n, m]) - exact) <= Fraction(1, 10 ** 12) * aexact + Fraction(1, 10 ** 300)
            assert abs(Fraction(A[n, m]) - aexact) <= Fraction(1, 10 ** 12) * aexact + Fraction(1, 10 ** 300)
    # subsets of rows / tokens agree with the full product, in the order asked
    ys, As = oracle.gemv(xb, codes, scales, ts, rows=[4, 0], tokens=[2], lib=lib)
    assert ys[0, 0] == y[2, 4] and ys[0, 1] == y[2, 0] and As[0, 0] == A[2, 4]


def check_gemv_one_hot(lib):
    rng = np.random.default_rng(9)
    M, K = 4, 64
    w = (rng.standard_normal((M, K)) * 0.02).astype(np.float32)
    codes, scales, ts = oracle.quantize(w, lib=lib)
    wq = dequant_ref(codes, scales, ts)
    for k in (0, 1, 17, 63):
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        y, _ = oracle.gemv(bf16_round(x), codes, scales, ts, lib=lib)
        for m in range(M):
            assert y[0, m] == float(wq[m][k]), (k, m)


def check_swiglu(lib):
    rng = np.random.default_rng(13)
    M, K, N = 3, 32, 2
    gw = (rng.standard_normal((M, K)) * 0.3).astype(np.float32)
    uw = (rng.standard_normal((M, K)) * 0.3).astype(np.float32)
    g = oracle.quantize(gw, lib=lib)
    u = oracle.quantize(uw, lib=lib)
    xb = bf16_round(rng.standard_normal((N, K)).astype(np.float32))
    h, gr, ur, Ag, Au = oracle.swiglu(xb, g, u, lib=lib)
    gq, uq = dequant_ref(*g), dequant_ref(*u)
    for n in range(N):
        for m in range(M):
            ge = float(sum((gq[m][k] * Fraction(bf16_value(xb[n, k])) for k in range(K)), Fraction(0)))
            ue = float(sum((uq[m][k] * Fraction(bf16_value(xb[n, k])) for k in range(K)), Fraction(0)))
            he = ge / (1.0 + math.exp(-ge)) * ue
            assert abs(gr[n, m] - ge) <= 1e-12 * Ag[n, m] + 1e-300
            assert abs(ur[n, m] - ue) <= 1e-12 * Au[n, m] + 1e-300
            assert abs(h[n, m] - he) <= 1e-12 * abs(he) + 1e-300
    # limits of SiLU: g = 0 gives 0
    zero = (np.zeros((M, K // 2), np.uint8), np.zeros((M, K // 16), np.uint8), np.float32(0))
    h0, *_ = oracle.swiglu(xb, zero, u, lib=lib)
    assert not h0.any()


def rounding_order_matrix():
    """A matrix whose block scales depend on doing (bamax / 6) / ts in that
    order (rather than bamax / (6 * ts)) and whose codes depend on dividing by
    d (rather than multiplying by a rounded 1/d).  Found by a seeded search;
    the expected values come from quantize_ref, not from the oracle."""
    rng = np.random.default_rng(21)
    amax = np.float32(0.0731)
    ts = f32(amax / f32(2688.0))
    table = e4m3_torch_table()
    mids = [(table[b] + table[b + 1]) / 2 for b in (0x02, 0x09, 0x21, 0x33, 0x38, 0x45, 0x5A, 0x6C)]
    bam = np.concatenate([
        (np.float32(mq * 6.0 * float(ts)) + np.arange(-400, 401, dtype=np.float32)
         * np.spacing(np.float32(mq * 6.0 * float(ts)))).astype(np.float32)
        for mq in mids])
    q1 = ((bam / f32(6.0)).astype(np.float32) / ts).astype(np.float32)
    q2 = (bam / f32(f32(6.0) * ts)).astype(np.float32)
    b1 = torch.tensor(q1).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    b2 = torch.tensor(q2).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    pick = list(bam[b1 != b2][:6])
    assert len(pick) >= 2, "search found no order-sensitive block amax"
    rows = [np.full(16, amax / 4, np.float32)]
    rows[0][5] = amax
    for b in pick:
        r = (rng.uniform(-1, 1, 16) * float(b)).astype(np.float32)
        r[7] = b
        rows.append(r)
    # elements whose w/d and w*(1/d) land on opposite sides of an E2M1 midpoint
    extra = []
    for sb in (0x30, 0x31, 0x35, 0x3B, 0x46, 0x52, 0x5D, 0x66):
        d = f32(f32(e4m3_torch_table()[sb]) * ts)
        inv = f32(f32(1.0) / d)
        for mid in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0):
            cand = (np.float32(mid) * d + np.arange(-64, 65, dtype=np.float32) * np.spacing(np.float32(mid) * d)).astype(np.float32)
            dv = (cand / d).astype(np.float32)
            mv = (cand * inv).astype(np.float32)
            diff = np.nonzero((dv < mid) != (mv < mid))[0]
            if len(diff):
                extra.append((sb, cand[diff[0]]))
    return np.stack(rows), extra


def check_quantize_rounding_order(lib):
    w, extra = rounding_order_matrix()
    c, s, ts = oracle.quantize(w, lib=lib)
    rc, rs, rts = quantize_ref(w)
    assert ts == rts and np.array_equal(s, rs) and np.array_equal(c, rc)
    # division by d: build blocks whose scale byte is sb and that hold the element
    assert extra, "search found no element sensitive to 1/d rounding"
    ts0 = f32(f32(0.0731) / f32(2688.0))
    rows = []
    for sb, v in extra[:12]:
        target = f32(e4m3_torch_table()[sb])
        # block amax chosen so that the block scale rounds to sb exactly
        bam = f32(target * f32(6.0) * ts0)
        r = np.zeros(16, np.float32)
        r[0] = bam
        r[1] = v
        rows.append(r)
    amax_row = np.zeros(16, np.float32)
    amax_row[0] = np.float32(0.0731)
    w2 = np.stack([amax_row] + rows)
    c2, s2, t2 = oracle.quantize(w2, lib=lib)
    rc2, rs2, rt2 = quantize_ref(w2)
    assert t2 == rt2 and np.array_equal(s2, rs2) and np.array_equal(c2, rc2)


ALL_CHECKS = [check_e2m1_table, check_e4m3_table, check_e4m3_encode, check_e4m3_encode_vs_torch,
              check_e2m1_encode, check_hand_block, check_quantize_random, check_quantize_special,
              check_gemv_exact_small, check_gemv_one_hot, check_swiglu,
              check_quantize_rounding_order]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(None)


def test_oracle_rejects_bad_input():
    with pytest.raises(ValueError):
        oracle.quantize(np.zeros((2, 24), np.float32))
    w = np.zeros((1, 16), np.float32)
    w[0, 3] = np.nan
    with pytest.raises(ValueError):
        oracle.quantize(w)


# ---------------------------------------------------------------------------
# Ingest: bf16 quantiser and the blocked scale layout
# ---------------------------------------------------------------------------

def test_quantize_bf16_matches_torch_decode_and_recipe():
    """bf16 bits are decoded by PyTorch (independent of the oracle) and the
    values re-quantised by the numpy re-derivation of the recipe."""
    rng = np.random.default_rng(21)
    for M, K in [(3, 48), (17, 160)]:
        w = (rng.standard_normal((M, K)) * rng.uniform(0.01, 3.0, (M, 1))).astype(np.float32)
        bits = torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        vals = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
        c, s, ts = oracle.quantize_bf16(bits)
        rc, rs, rts = quantize_ref(vals)
        assert ts == rts and np.array_equal(s, rs) and np.array_equal(c, rc)


def test_quantize_bf16_hand_values():
    """Hand-decoded bf16 patterns: 0x3F00 = 0.5, 0xBE80 = -0.25, 0x3E00 = 0.125,
    0x0000 = 0.  With amax 0.5: ts = 0.5/2688, block scale 448 (0x7E), d = 448 ts
    = 0.5/6, so w/d = 6, -3, 1.5, 0 -> codes 7, D, 3, 0."""
    bits = np.array([[0x3F00, 0xBE80, 0x3E00, 0x0000] * 4], np.uint16)
    c, s, ts = oracle.quantize_bf16(bits)
    assert ts == f32(f32(0.5) / f32(2688.0))
    assert s[0, 0] == 0x7E
    assert list(c[0]) == [0xD7, 0x03] * 4


def test_blocked_scale_positions_hand_worked():
    """M = 130, K = 128: S = 8 scale columns -> 2 x 2 blocks of 512 bytes.
    (r, c) -> block (r // 128) * 2 + c // 4, byte (r % 32) * 16 + (r % 128 // 32) * 4 + c % 4:
      (0, 0) -> 0;  (1, 0) -> 16;  (32, 0) -> 4;  (33, 3) -> 23;  (0, 4) -> 512;
      (127, 7) -> 512 + 31 * 16 + 3 * 4 + 3 = 1023;  (129, 5) -> 1536 + 16 + 1 = 1553."""
    assert oracle.blocked_scale_bytes(130, 128) == 2048
    cases = {(0, 0): 0, (1, 0): 16, (32, 0): 4, (33, 3): 23, (0, 4): 512, (127, 7): 1023, (129, 5): 1553}
    for (r, c), pos in cases.items():
        s = np.zeros((130, 8), np.uint8)
        s[r, c] = 0x5A
        b = oracle.interleave_scales(s)
        assert b.shape == (2048,)
        assert np.flatnonzero(b).tolist() == [pos], ((r, c), np.flatnonzero(b))


def test_blocked_scale_layout_is_a_bijection_with_zero_padding():
    # 64 rows x 4 columns = 256 distinct bytes, one block, rows 64..127 padding
    s = np.arange(256, dtype=np.uint32).reshape(64, 4).astype(np.uint8)
    b = oracle.interleave_scales(s)
    assert b.shape == (512,)
    live = np.zeros(512, bool)
    for r in range(64):
        live[(r % 32) * 16 + (r // 32) * 4: (r % 32) * 16 + (r // 32) * 4 + 4] = True
    assert sorted(b[live].tolist()) == list(range(256))
    assert not b[~live].any()


@pytest.mark.parametrize("M,K", [(1, 16), (128, 64), (130, 80), (257, 1040), (5, 16 * 9)])
def test_blocked_scale_round_trip(M, K):
    rng = np.random.default_rng(M * 1000 + K)
    s = rng.integers(0, 256, (M, K // 16), dtype=np.uint8)
    b = oracle.interleave_scales(s)
    assert b.size == oracle.blocked_scale_bytes(M, K)
    assert np.array_equal(oracle.deinterleave_scales(b, M, K), s)
    # padding is ignored on the way back
    junk = b.copy()
    pad = oracle.interleave_scales(np.full_like(s, 1)) == 0
    junk[pad] = 0xEE
    assert np.array_equal(oracle.deinterleave_scales(junk, M, K), s)


# ---------------------------------------------------------------------------
# FP6 E2M3 block-scaled variant
# ---------------------------------------------------------------------------

# The 32 E2M3 magnitudes listed by their spacing: [0, 2) in steps of 1/8,
# [2, 4) in steps of 1/4, [4, 7.5] in steps of 1/2.
E2M3_MAG = [m / 8 for m in range(16)] + [2 + m / 4 for m in range(8)] + [4 + m / 2 for m in range(8)]


def e2m3_ref(code: int) -> float:
    mag = E2M3_MAG[code & 31]
    return -mag if code & 32 else mag


def e2m3_brute(v: float) -> int:
    """Nearest E2M3 code to fp32 v, ties to the even code, saturating at 7.5, sign kept."""
    vf = float(np.float32(v))
    a = Fraction(abs(vf))
    best, best_d = None, None
    for c in range(32):
        d = abs(Fraction(E2M3_MAG[c]) - a)
        if best is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    return best | (32 if math.copysign(1.0, vf) < 0 else 0)


def floor_log2_f32(a: np.float32) -> int:
    """floor(log2(a)) of a positive fp32 from its bit pattern."""
    bits = int(np.array([a], np.float32).view(np.uint32)[0])
    e = bits >> 23
    if e:
        return e - 127
    return bits.bit_length() - 1 - 149  # subnormal: value = bits * 2^-149


def pack6_ref(codes_row) -> np.ndarray:
    """Little-endian 6-bit stream built as a bit string."""
    s = "".join(format(int(c), "06b")[::-1] for c in codes_row)  # LSB first
    return np.array([int(s[i:i + 8][::-1], 2) for i in range(0, len(s), 8)], np.uint8)


def fp6_quantize_ref(w: np.ndarray):
    w = np.asarray(w, np.float32)
    M, K = w.shape
    codes = np.zeros((M, K // 8 * 6), np.uint8)
    scales = np.zeros((M, K // 128), np.uint8)
    for m in range(M):
        row = []
        for b in range(K // 128):
            blk = w[m, 128 * b:128 * b + 128]
            amax = np.float32(np.max(np.abs(blk)))
            shared = max(floor_log2_f32(amax) - 2, -127) if amax > 0 else -127
            scales[m, b] = shared + 127
            X = np.float32(2.0 ** shared)
            row += [e2m3_brute(np.float32(v / X)) for v in blk]
        codes[m] = pack6_ref(row)
    return codes, scales


def unpack6_ref(codes_row, K):
    s = "".join(format(int(b), "08b")[::-1] for b in codes_row)
    return [int(s[6 * k:6 * k + 6][::-1], 2) for k in range(K)]


def read_fp6_golden():
    vals = {}
    with open(os.path.join(GOLDEN, "fp6_hand_block.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = (t.strip() for t in line.split("=", 1))
                vals[k] = v
    w = np.zeros(128, np.float32)
    given = [float(t) for t in vals["w"].split()]
    w[:len(given)] = given
    return (w, int(vals["scale_byte"], 16), [int(t, 16) for t in vals["codes"].split()],
            [int(t, 16) for t in vals["first_bytes"].split()])


def check_fp6_e2m3_table(lib):
    for c in range(64):
        got = oracle.e2m3_value(c, lib=lib)
        exp = e2m3_ref(c)
        assert got == exp and math.copysign(1, got) == math.copysign(1, exp), (c, got, exp)
    assert oracle.e2m3_value(0x1F, lib=lib) == 7.5 and oracle.e2m3_value(0x01, lib=lib) == 0.125


def check_fp6_e2m3_encode(lib):
    vals = []
    for a, b in zip(E2M3_MAG, E2M3_MAG[1:]):
        mid = np.float32((a + b) / 2)
        vals += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(9)), np.float32(a)]
    vals += [np.float32(v) for v in (7.5, 7.7, 7.75, 7.8, 7.99, 100.0, 1e-40)]
    vals = vals + [np.float32(-v) for v in vals]
    rng = np.random.default_rng(17)
    vals += list(rng.uniform(-8, 8, 600).astype(np.float32)) + [np.float32(-0.0), np.float32(-0.03)]
    for v in vals:
        assert oracle.e2m3_encode(v, lib=lib) == e2m3_brute(v), (repr(v),)


def check_fp6_hand_block(lib):
    w, sb, codes_exp, first = read_fp6_golden()
    codes, scales = oracle.fp6_quantize(w.reshape(1, 128), lib=lib)
    assert scales[0, 0] == sb
    got = unpack6_ref(codes[0], 128)
    assert got[:len(codes_exp)] == codes_exp, (got[:12], codes_exp)
    assert not any(got[len(codes_exp):])
    assert list(codes[0, :3]) == first
    # one-hot activation at k = 4 reads back 7.5 * 2^-1
    x = np.zeros((1, 128), np.uint16)
    x[0, 4] = 0x3F80  # bf16 1.0
    y, A = oracle.fp6_gemv(x, codes, scales, lib=lib)
    assert y[0, 0] == 3.75 and A[0, 0] == 3.75


def check_fp6_quantize_random(lib):
    rng = np.random.default_rng(23)
    w = (rng.standard_normal((5, 256)) * np.array([[0.02], [1.0], [300.0], [1e-20], [1e-39]])).astype(np.float32)
    w[0, 7] = np.float32(-0.0)
    w = np.concatenate([w, np.zeros((1, 256), np.float32)])
    w[5, 130] = np.float32(2.0 ** -120)   # block 1 of row 5: amax a power of two
    w[5, 131] = np.float32(-(2.0 ** -120) * 0.75)
    c, s = oracle.fp6_quantize(w, lib=lib)
    rc, rs = fp6_quantize_ref(w)
    assert np.array_equal(s, rs), (s, rs)
    assert np.array_equal(c, rc)
    assert s[5, 0] == 0 and s[5, 1] == 127 - 122 and s[4, 0] == 0  # zero block; 2^-120; clamped


def check_fp6_gemv_exact_small(lib):
    rng = np.random.default_rng(29)
    w = (rng.standard_normal((3, 256)) * 0.05).astype(np.float32)
    c, s = fp6_quantize_ref(w)  # expected bytes from the independent re-derivation
    x = bf16_round(rng.standard_normal((2, 256)))
    y, A = oracle.fp6_gemv(x, c, s, lib=lib)
    for m in range(3):
        codes = unpack6_ref(c[m], 256)
        wq = [Fraction(e2m3_ref(codes[k])) * Fraction(2) ** (int(s[m, k // 128]) - 127) for k in range(256)]
        for n in range(2):
            xs = [Fraction(bf16_value(b)) for b in x[n]]
            exact = sum(a * b for a, b in zip(wq, xs))
            aexact = sum(abs(a * b) for a, b in zip(wq, xs))
            assert abs(Fraction(y[n, m]) - exact) <= Fraction(1, 10 ** 12) * aexact
            assert abs(Fraction(A[n, m]) - aexact) <= Fraction(1, 10 ** 12) * aexact


def check_fp6_swiglu(lib):
    """h = silu(g) * u for FP6 weights against exact rational g and u (codes
    from the independent re-derivation), plus the g = 0 limit of SiLU."""
    rng = np.random.default_rng(31)
    K = 256
    gw = (rng.standard_normal((3, K)) * 0.3).astype(np.float32)
    uw = (rng.standard_normal((3, K)) * 0.3).astype(np.float32)
    gc, gs = fp6_quantize_ref(gw)
    uc, us = fp6_quantize_ref(uw)
    x = bf16_round(rng.standard_normal((2, K)))
    h, gr, ur, Ag, Au = oracle.fp6_swiglu(x, (gc, gs), (uc, us), lib=lib)

    def wq(c, sc, m):
        codes = unpack6_ref(c[m], K)
        return [Fraction(e2m3_ref(codes[k])) * Fraction(2) ** (int(sc[m, k // 128]) - 127) for k in range(K)]

    for m in range(3):
        gq, uq = wq(gc, gs, m), wq(uc, us, m)
        for n in range(2):
            xs = [Fraction(bf16_value(b)) for b in x[n]]
            ge = float(sum(a * b for a, b in zip(gq, xs)))
            ue = float(sum(a * b for a, b in zip(uq, xs)))
            he = ge / (1.0 + math.exp(-ge)) * ue
            assert abs(gr[n, m] - ge) <= 1e-12 * Ag[n, m] + 1e-300
            assert abs(ur[n, m] - ue) <= 1e-12 * Au[n, m] + 1e-300
            assert abs(h[n, m] - he) <= 1e-12 * (abs(he) + Ag[n, m] * abs(ue) + Au[n, m] * abs(ge)) + 1e-300
    # an all-zero gate (codes 0, smallest scale) makes every h zero
    h0, *_ = oracle.fp6_swiglu(x, (np.zeros_like(gc), np.zeros_like(gs)), (uc, us), lib=lib)
    assert not h0.any()


ALL_CHECKS += [check_fp6_e2m3_table, check_fp6_e2m3_encode, check_fp6_hand_block,
               check_fp6_quantize_random, check_fp6_gemv_exact_small, check_fp6_swiglu]


# ---------------------------------------------------------------------------
# W4A4: activations quantised to NVFP4 as well
# ---------------------------------------------------------------------------

def check_w4a4_exact_small(lib):
    """Activation bytes from the independent recipe; products from exact rationals."""
    rng = np.random.default_rng(37)
    N, M, K = 3, 4, 48
    xb = bf16_round(rng.standard_normal((N, K)).astype(np.float32) * np.array([[1.0], [8.0], [0.25]], np.float32))
    xf = (xb.astype(np.uint32) << np.uint32(16)).view(np.float32)
    xq = oracle.quantize_activations(xb, lib=lib)
    rxq = quantize_ref(xf)
    assert xq[2] == rxq[2] and np.array_equal(xq[1], rxq[1]) and np.array_equal(xq[0], rxq[0])
    w = (rng.standard_normal((M, K)) * 0.02).astype(np.float32)
    wq = quantize_ref(w)
    y, A = oracle.w4a4_gemm(rxq, wq, lib=lib)
    xd, wd = dequant_ref(*rxq), dequant_ref(*wq)
    for n in range(N):
        for m in range(M):
            terms = [xd[n][k] * wd[m][k] for k in range(K)]
            exact = sum(terms, Fraction(0))
            aexact = sum((abs(t) for t in terms), Fraction(0))
            assert abs(Fraction(y[n, m]) - exact) <= Fraction(1, 10 ** 12) * aexact + Fraction(1, 10 ** 300)
            assert abs(Fraction(A[n, m]) - aexact) <= Fraction(1, 10 ** 12) * aexact + Fraction(1, 10 ** 300)
    # row / token subsets, in the order asked
    ys, As = oracle.w4a4_gemm(rxq, wq, rows=[3, 1], tokens=[2, 0], lib=lib)
    assert ys[0, 0] == y[2, 3] and ys[1, 1] == y[0, 1] and As[1, 0] == A[0, 3]


def check_w4a4_equals_w4a16_on_exact_activations(lib):
    """With an activation tensor scale of 1 the decoded activations
    e2m1 * e4m3 have at most 6 significant bits, so they are exact bf16
    values; the W4A4 product must then equal the W4A16 product of those bf16
    activations bit for bit (same exact terms, same k order)."""
    rng = np.random.default_rng(41)
    N, M, K = 3, 5, 64
    xc = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    xs = rng.integers(0x08, 0x7F, (N, K // 16), dtype=np.uint8)  # normal, finite E4M3 bytes
    xd = np.array([[float(v) for v in row] for row in dequant_ref(xc, xs, np.float32(1.0))], np.float64)
    xb = bf16_round(xd.astype(np.float32))
    assert np.array_equal((xb.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64), xd)
    w = (rng.standard_normal((M, K)) * 0.02).astype(np.float32)
    wq = quantize_ref(w)
    y4, A4 = oracle.w4a4_gemm((xc, xs, np.float32(1.0)), wq, lib=lib)
    y16, A16 = oracle.gemv(xb, *wq, lib=lib)
    assert np.array_equal(y4, y16) and np.array_equal(A4, A16)


def check_w4a4_operand_symmetry_and_zero(lib):
    """The definition is symmetric in its two NVFP4 operands; zero activations
    give a zero tensor scale and a zero product."""
    rng = np.random.default_rng(43)
    K = 32
    a = quantize_ref((rng.standard_normal((3, K)) * 0.5).astype(np.float32))
    b = quantize_ref((rng.standard_normal((5, K)) * 0.02).astype(np.float32))
    yab, Aab = oracle.w4a4_gemm(a, b, lib=lib)
    yba, Aba = oracle.w4a4_gemm(b, a, lib=lib)
    assert np.array_equal(yab, yba.T) and np.array_equal(Aab, Aba.T)
    z = oracle.quantize_activations(np.zeros((2, K), np.uint16), lib=lib)
    assert z[2] == 0 and not z[0].any() and not z[1].any()
    yz, Az = oracle.w4a4_gemm(z, b, lib=lib)
    assert not yz.any() and not Az.any()


ALL_CHECKS += [check_w4a4_exact_small, check_w4a4_equals_w4a16_on_exact_activations,
               check_w4a4_operand_symmetry_and_zero]


# (test_oracle_pin above runs every entry of ALL_CHECKS, these included)


def test_fp6_pack_and_dequantize_helpers():
    codes = [1, 2, 3, 4, 63, 0, 32, 31]
    packed = pack6_ref(codes)
    assert list(packed[:3]) == [0x81, 0x30, 0x10]  # 1 | 2<<6 | 3<<12 | 4<<18 = 0x103081
    assert unpack6_ref(packed, 8) == codes
    w = np.random.default_rng(31).standard_normal((2, 128)).astype(np.float32)
    c, s = oracle.fp6_quantize(w)
    d = oracle.fp6_dequantize(c, s)
    for m in range(2):
        cc = unpack6_ref(c[m], 128)
        assert all(d[m, k] == e2m3_ref(cc[k]) * 2.0 ** (int(s[m, 0]) - 127) for k in range(128))
    with pytest.raises(ValueError):
        oracle.fp6_quantize(np.zeros((1, 64), np.float32))


def test_dequantize_pinned_by_hand_block_and_closed_form():
    """oracle.dequantize against the hand-worked block (its printed E2M1 values
    times the decoded scale 448 and the tensor scale), against the E2M1 list and
    PyTorch's E4M3 decode on a two-block row (each block its own scale byte,
    both nibble orders), and against a one-hot product of the C oracle."""
    ts = float(np.float32(np.float32(0.6) / np.float32(2688.0)))
    codes_hex = "7 D 3 1 0 F 5 A 3 4 E 1 7 8 5 C".split()
    values = [6, -3, 1.5, 0.5, 0, -6, 3, -1, 1.5, 2, -4, 0.5, 6, -0.0, 3, -2]
    c = [int(h, 16) for h in codes_hex]
    packed = np.array([[c[2 * j] | (c[2 * j + 1] << 4) for j in range(8)]], np.uint8)
    d = oracle.dequantize(packed, np.array([[0x7E]], np.uint8), ts)
    assert d.shape == (1, 16)
    assert [float(v) for v in d[0]] == [v * 448.0 * ts for v in values]
    assert math.copysign(1.0, d[0, 13]) == -1.0  # code 8 is -0
    # two blocks with different scale bytes; every code in both nibble positions
    e4 = e4m3_torch_table()
    row = np.zeros((1, 16), np.uint8)
    for j in range(16):
        row[0, j] = (j & 15) | (((15 - j) & 15) << 4)
    sc = np.array([[0x31, 0x5B]], np.uint8)
    d2 = oracle.dequantize(row, sc, 1.0)
    for k in range(32):
        byte = int(row[0, k // 2])
        code = byte & 15 if k % 2 == 0 else byte >> 4
        assert d2[0, k] == e2m1_ref(code) * float(e4[sc[0, k // 16]])
    # the C oracle's product with a one-hot activation reads the same weight
    w = np.random.default_rng(5).standard_normal((3, 64)).astype(np.float32) * 0.02
    qc, qs, qts = oracle.quantize(w)
    dq = oracle.dequantize(qc, qs, qts)
    for k in (0, 17, 63):
        x = np.zeros((1, 64), np.uint16)
        x[0, k] = 0x3F80  # bf16 1.0
        y, _ = oracle.gemv(x, qc, qs, qts)
        assert np.array_equal(y[0], dq[:, k])
