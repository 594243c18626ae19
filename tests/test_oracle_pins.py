"""Pins for the CPU oracle: values fixed by mathematics or by hand, not by the oracle.

Each test ties one oracle routine to something independent of it: IEEE
binary16 encodings (numpy), closed forms, hand-derived blocks in
tests/golden/, exact rational arithmetic on tiny shapes, round-trip bounds,
special blocks and symmetry.  A dropped term, wrong sign, wrong nibble order,
transposed operand or misplaced epsilon fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_blocks.json")


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ---------------------------------------------------------------- helpers
def unpack_q4(Wq, K):
    """Independent vectorised unpack: codes [O][K] in 0..15 and scales [O][K/32]."""
    O = Wq.shape[0]
    blk = Wq.reshape(O, K // 32, 18)
    d = blk[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    qs = blk[:, :, 2:]
    lo = (qs & 0x0F).astype(np.int64)
    hi = (qs >> 4).astype(np.int64)
    codes = np.concatenate([lo, hi], axis=2).reshape(O, K)
    return codes, d


def unpack_q8(xq, K):
    N = xq.shape[0]
    blk = xq.reshape(N, K // 32, 34)
    d = blk[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    q = blk[:, :, 2:].view(np.int8).astype(np.int64).reshape(N, K)
    return q, d


def ulp32(v):
    return float(np.spacing(np.float32(abs(v))))


# ---------------------------------------------------------------- fp16
def test_f16_to_f32_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([orc.f16_to_f32(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_f16_matches_ieee(orc):
    rng = np.random.default_rng(7)
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9,
            2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 3 * 2.0 ** -26, 2.0 ** -14,
            2.0 ** -14 - 2.0 ** -25, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 0.1, 1 / 127]
    vals += list(rng.standard_normal(3000) * 10.0 ** rng.integers(-9, 6, 3000))
    # exact ties in the normal and subnormal ranges
    m = rng.integers(1024, 2048, 500)
    e = rng.integers(-14, 15, 500)
    vals += list((m + 0.5) * 2.0 ** (e - 10))
    vals += list((rng.integers(0, 1024, 200) + 0.5) * 2.0 ** -24)
    v32 = np.array(vals, dtype=np.float32)
    ref = v32.astype(np.float16).view(np.uint16)
    got = np.array([orc.f32_to_f16(float(v)) for v in v32], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- Q4_0
def test_q4_golden_block(orc):
    g = golden()["q4_weights"]
    w = np.array(g["w"], dtype=np.float32).reshape(1, 32)
    out = orc.quantize_q4_0(w)
    assert list(out[0]) == g["bytes"]
    codes, d = unpack_q4(out, 32)
    assert list(codes[0]) == g["q"]
    assert out[0, :2].view(np.uint16)[0] == g["d_bits"]


def test_q4_invariants_random(orc):
    rng = np.random.default_rng(11)
    O, K = 64, 256
    w = (rng.standard_normal((O, K)) * 0.02).astype(np.float32)
    w[3, 32:64] = 0.0                                  # an all-zero block
    w[5, 0:32] = 0.01                                  # ties on the max magnitude
    w[5, 7] = -0.01
    Wq = orc.quantize_q4_0(w)
    codes, d16 = unpack_q4(Wq, K)
    blocks = w.reshape(O, K // 32, 32).astype(np.float64)
    cb = codes.reshape(O, K // 32, 32)
    # all-zero block: d = 0, every code 8
    assert d16[3, 1] == 0.0 and np.all(cb[3, 1] == 8)
    # ties: the first element of largest magnitude sets the sign of d (w=+0.01 first -> d<0)
    assert d16[5, 0] < 0 and cb[5, 0, 0] == 0 and cb[5, 0, 7] == 15
    for o in range(O):
        for b in range(K // 32):
            v = blocks[o, b]
            if not np.any(v):
                continue
            i = int(np.argmax(np.abs(v)))               # first on ties
            m = v[i]
            d = np.float32(np.float32(m) / np.float32(-8.0))
            # the extreme element maps to code 0 and d has the opposite sign of m
            assert cb[o, b, i] == 0
            assert np.sign(d16[o, b]) == -np.sign(m)
            assert d16[o, b] == float(np.float16(d))
            # round trip with the fp32 scale: within d/2 (+ fp32 slop) unless clamped at 15
            err = np.abs(v - float(d) * (cb[o, b] - 8))
            clamped = cb[o, b] == 15
            assert np.all(err[~clamped] <= abs(float(d)) * (0.5 + 2 ** -17))
            assert np.all(err[clamped] <= abs(float(d)) * (1.0 + 2 ** -17))


# ---------------------------------------------------------------- RMS statistic
@pytest.mark.parametrize("K", [32, 256, 2048, 4096, 14336])
def test_rms_scale_vs_fp64(orc, K):
    rng = np.random.default_rng(K)
    for scale in (1.0, 1e-3, 30.0):
        x = (rng.standard_normal(K) * scale).astype(np.float32)
        eps = 1e-6
        ref = 1.0 / math.sqrt(float(np.mean(x.astype(np.float64) ** 2)) + eps)
        got = orc.rms_scale(x, eps)
        bound = (K / 256 + 12) * 2.0 ** -24
        assert abs(got - ref) <= bound * ref, (scale, got, ref)


def test_rms_eps_inside_sqrt(orc):
    g = golden()["norm_eps_position"]
    x = np.full(g["K"], g["x_value"], dtype=np.float32)
    s = orc.rms_scale(x, g["eps"])
    assert abs(s - g["s"]) <= 2e-6 * g["s"]
    # the other placement would be far away
    assert abs(s - 1.0 / (math.sqrt(1e-6) + 1e-6)) > 100


# ---------------------------------------------------------------- Q8_0
def test_q8_golden_plain(orc):
    g = golden()["q8_plain"]
    xq = orc.quantize_q8_0(np.array(g["x"], dtype=np.float32), None)
    q, d = unpack_q8(xq, 32)
    assert xq[0, :2].view(np.uint16)[0] == g["d_bits"]
    assert list(q[0]) == g["q"]


@pytest.mark.parametrize("case", ["norm_constant", "norm_eps_position"])
def test_q8_golden_norm(orc, case):
    g = golden()[case]
    K = g["K"]
    x = np.full((1, K), g["x_value"], dtype=np.float32)
    xq = orc.quantize_q8_0(x, np.ones(K, np.float32), g["eps"])
    q, d = unpack_q8(xq, K)
    assert np.all(q == g["q_value"])
    assert np.all(xq.reshape(1, K // 32, 34)[:, :, :2].copy().view(np.uint16) == g["d_bits"])


def test_q8_roundtrip_bound_plain(orc):
    rng = np.random.default_rng(3)
    N, K = 4, 1024
    x = rng.standard_normal((N, K)).astype(np.float32)
    x[1, 64:96] = 0.0
    x[2, :] *= 20.0
    xq = orc.quantize_q8_0(x, None)
    q, d16 = unpack_q8(xq, K)
    xb = x.reshape(N, K // 32, 32).astype(np.float64)
    qb = q.reshape(N, K // 32, 32)
    amax = np.abs(xb).max(axis=2)
    d32 = (amax.astype(np.float32) / np.float32(127.0)).astype(np.float64)
    # stored scale is the fp16 rounding of amax/127
    assert np.array_equal(d16, d32.astype(np.float16).astype(np.float64))
    # zero block
    assert np.all(qb[1, 2] == 0) and d16[1, 2] == 0.0
    # the extreme element reaches |q| = 127, nothing exceeds it
    nz = amax > 0
    assert np.all(np.abs(qb).max(axis=2)[nz] == 127)
    # round trip |x - d q| <= d/2 with the fp32 scale (plus division rounding)
    err = np.abs(xb - d32[:, :, None] * qb)
    assert np.all(err <= d32[:, :, None] * (0.5 + 2 ** -16))


def test_q8_norm_scale_equivariance(orc):
    rng = np.random.default_rng(5)
    N, K = 3, 4096
    x = rng.standard_normal((N, K)).astype(np.float32)
    gam = rng.uniform(0.5, 1.5, K).astype(np.float32)
    a = orc.quantize_q8_0(x, gam, 1e-6)
    b = orc.quantize_q8_0(x, gam * np.float32(2.0), 1e-6)
    qa, da = unpack_q8(a, K)
    qb, db = unpack_q8(b, K)
    assert np.array_equal(qa, qb)
    assert np.array_equal(db, 2.0 * da)


def test_q8_norm_matches_definition(orc):
    """Quantized codes agree with the fp64 definition up to the rounding of v/d."""
    rng = np.random.default_rng(9)
    N, K = 2, 4096
    x = rng.standard_normal((N, K)).astype(np.float32)
    x[0, rng.choice(K, 40, replace=False)] *= 20.0
    gam = rng.uniform(0.5, 1.5, K).astype(np.float32)
    xq = orc.quantize_q8_0(x, gam, 1e-6)
    q, d16 = unpack_q8(xq, K)
    x64 = x.astype(np.float64)
    s = 1.0 / np.sqrt(np.mean(x64 ** 2, axis=1, keepdims=True) + 1e-6)
    v = (x64 * s * gam).reshape(N, K // 32, 32)
    d = np.abs(v).max(axis=2) / 127.0
    ideal = v / d[:, :, None]
    qb = q.reshape(N, K // 32, 32)
    assert np.all(np.abs(qb - ideal) <= 0.5 + 1e-4)
    assert np.allclose(d16, d, rtol=2 ** -11, atol=0)


# ---------------------------------------------------------------- block sums / product
def test_golden_dot(orc):
    g = golden()
    W = orc.quantize_q4_0(np.array(g["q4_weights"]["w"], dtype=np.float32).reshape(1, 32))
    xq = orc.quantize_q8_0(np.array(g["q8_plain"]["x"], dtype=np.float32), None)
    assert int(orc.block_sums(W, xq, 32)[0, 0, 0]) == g["dot"]["isum"]
    y32, y64, S = orc.matvec(W, xq, 32)
    assert y64[0, 0] == g["dot"]["y"] and y32[0, 0] == g["dot"]["y"]
    assert S[0, 0] == 3.0


def random_problem(rng, O, K, N):
    import oracle
    w = (rng.standard_normal((O, K)) * 0.02).astype(np.float32)
    x = rng.standard_normal((N, K)).astype(np.float32)
    gam = rng.uniform(0.5, 1.5, K).astype(np.float32)
    return oracle.quantize_q4_0(w), oracle.quantize_q8_0(x, gam, 1e-6)


@pytest.mark.parametrize("O,K,N", [(1, 32, 1), (7, 64, 2), (16, 256, 3), (33, 256, 8)])
def test_block_sums_brute_force(orc, O, K, N):
    rng = np.random.default_rng(O * 1000 + K + N)
    Wq, xq = random_problem(rng, O, K, N)
    codes, _ = unpack_q4(Wq, K)
    q, _ = unpack_q8(xq, K)
    ref = np.einsum("obj,nbj->nob", (codes - 8).reshape(O, K // 32, 32),
                    q.reshape(N, K // 32, 32))
    got = orc.block_sums(Wq, xq, K)
    assert got.dtype == np.int32
    assert np.array_equal(got.astype(np.int64), ref)


@pytest.mark.parametrize("O,K,N", [(3, 32, 1), (5, 64, 2), (4, 256, 2)])
def test_matvec_exact_rational(orc, O, K, N):
    rng = np.random.default_rng(100 + O + K + N)
    Wq, xq = random_problem(rng, O, K, N)
    codes, dw = unpack_q4(Wq, K)
    q, dx = unpack_q8(xq, K)
    y32, y64, S = orc.matvec(Wq, xq, K)
    for n in range(N):
        for o in range(O):
            exact = Fraction(0)
            mag = Fraction(0)
            for b in range(K // 32):
                fw = Fraction(float(dw[o, b]))
                fx = Fraction(float(dx[n, b]))
                isum = sum(int(codes[o, b * 32 + j] - 8) * int(q[n, b * 32 + j]) for j in range(32))
                exact += fw * fx * isum
                mag += abs(fw * fx * isum)
            assert abs(Fraction(float(y64[n, o])) - exact) <= Fraction(2.0 ** -50) * mag
            assert abs(float(y32[n, o]) - float(exact)) <= ulp32(float(exact))
            assert float(S[n, o]) == pytest.approx(float(mag), rel=1e-15)


def test_matvec_vs_numpy_dequant(orc):
    rng = np.random.default_rng(21)
    O, K, N = 48, 512, 3
    Wq, xq = random_problem(rng, O, K, N)
    codes, dw = unpack_q4(Wq, K)
    q, dx = unpack_q8(xq, K)
    Wf = (codes - 8).astype(np.float64) * np.repeat(dw, 32, axis=1)
    Xf = q.astype(np.float64) * np.repeat(dx, 32, axis=1)
    ref = Xf @ Wf.T                                   # [N][O]
    y32, y64, S = orc.matvec(Wq, xq, K)
    assert np.all(np.abs(y64 - ref) <= 1e-12 * S)
    # row subset and threading give the same numbers
    rows = np.array([0, 5, 47, 6], dtype=np.int64)
    a32, a64, aS = orc.matvec(Wq, xq, K, rows=rows, threads=3)
    assert np.array_equal(a64, y64[:, rows]) and np.array_equal(aS, S[:, rows])


def test_special_blocks(orc):
    """All-zero codes contribute -8 d_w sum(q_x); all-8 contribute 0; all-15 contribute 7 d_w sum(q_x)."""
    import oracle
    rng = np.random.default_rng(4)
    K = 64
    xq = oracle.quantize_q8_0(rng.standard_normal((1, K)).astype(np.float32), None)
    q, dx = unpack_q8(xq, K)
    W = np.zeros((3, K // 32 * 18), dtype=np.uint8)
    d_bits = np.float16(0.5).view(np.uint16)
    for r, byte in enumerate((0x00, 0x88, 0xFF)):
        for b in range(K // 32):
            W[r, b * 18:b * 18 + 2] = np.array([d_bits], dtype=np.uint16).view(np.uint8)
            W[r, b * 18 + 2:b * 18 + 18] = byte
    y32, y64, S = orc.matvec(W, xq, K)
    sums = q.reshape(K // 32, 32).sum(axis=1)
    expect = [sum(-8 * 0.5 * dx[0, b] * sums[b] for b in range(K // 32)), 0.0,
              sum(7 * 0.5 * dx[0, b] * sums[b] for b in range(K // 32))]
    assert np.allclose(y64[0], expect, rtol=0, atol=1e-12)
    isum = orc.block_sums(W, xq, K)
    assert np.array_equal(isum[0, 0], -8 * sums) and np.all(isum[0, 1] == 0)
    assert np.array_equal(isum[0, 2], 7 * sums)


def test_selection_and_permutation(orc):
    import oracle
    rng = np.random.default_rng(8)
    O, K = 6, 256
    Wq, xq = random_problem(rng, O, K, 1)
    nb = K // 32
    isum = orc.block_sums(Wq, xq, K)
    _, dw = unpack_q4(Wq, K)
    _, dx = unpack_q8(xq, K)
    # selection: keep one block per row, neutralise the others with code 8
    sel = Wq.copy().reshape(O, nb, 18)
    keep = rng.integers(0, nb, O)
    for o in range(O):
        for b in range(nb):
            if b != keep[o]:
                sel[o, b, 2:] = 0x88
    y32, y64, S = orc.matvec(sel.reshape(O, -1), xq, K)
    for o in range(O):
        b = keep[o]
        assert y64[0, o] == dw[o, b] * dx[0, b] * isum[0, o, b]
    # permutation of K-blocks applied to both operands
    perm = rng.permutation(nb)
    Wp = Wq.reshape(O, nb, 18)[:, perm].reshape(O, -1)
    xp = xq.reshape(1, nb, 34)[:, perm].reshape(1, -1)
    a = orc.matvec(Wq, xq, K)
    b = orc.matvec(Wp, xp, K)
    assert np.all(np.abs(a[1] - b[1]) <= 1e-12 * a[2])
    assert np.array_equal(orc.block_sums(Wp, xp, K)[0], isum[0][:, perm])


# ---- RMS_NORM + MUL + ADD -> Q8_0 (the fusion pattern counted in the Metal
# fusion-table refactor's CI notes): v = (x*s)*gamma + a, one fp32 add after
# the two products; the RMS statistic is over x alone.

def _half_away(r):
    from fractions import Fraction
    r = Fraction(r)
    f = r.numerator // r.denominator
    return f + 1 if (r - f) * 2 >= 1 and r > 0 else (f if r >= 0 else (f + 1 if (r - f) * 2 > 1 else f))


def test_q8_add_closed_form(orc):
    """x = 2 (constant), gamma = 1, eps = 0: x*s = 1 exactly, so v_j = 1 + a_j.
    With a_j = (j - 8)/8, v_j = j/8, amax = 31/8 and q_j = round(127 j / 31)
    (never a tie: 31 is odd)."""
    from fractions import Fraction
    K = 32
    x = np.full((1, K), 2.0, np.float32)
    a = ((np.arange(K) - 8) / 8).astype(np.float32)
    q = orc.quantize_q8_0(x, np.ones(K, np.float32), 0.0, add=a)[0]
    d = np.float32(np.float32(3.875) / np.float32(127.0))
    assert q[:2].view(np.uint16)[0] == np.float16(d).view(np.uint16)
    want = [_half_away(Fraction(127 * j, 31)) for j in range(K)]
    assert list(q[2:].view(np.int8)) == want


def test_q8_add_after_mul(orc):
    """gamma = 2, a = 1: v = 1*2 + 1 = 3 everywhere (adding before the MUL would give 4)."""
    K = 64
    x = np.full((1, K), 2.0, np.float32)
    q = orc.quantize_q8_0(x, np.full(K, 2.0, np.float32), 0.0, add=np.ones(K, np.float32))[0]
    for b in range(K // 32):
        blk = q[b * 34:(b + 1) * 34]
        assert blk[:2].view(np.uint16)[0] == np.float16(np.float32(3.0) / np.float32(127.0)).view(np.uint16)
        assert np.all(blk[2:].view(np.int8) == 127)


def test_q8_add_norm_over_x_only(orc):
    """Large addends leave the statistic alone: x = 2 gives x*s = 1 whatever a is."""
    from fractions import Fraction
    K = 32
    x = np.full((1, K), 2.0, np.float32)
    a = (64.0 * (np.arange(K) - 16)).astype(np.float32)            # v_j = 1 + 64 (j - 16), exact
    q = orc.quantize_q8_0(x, np.ones(K, np.float32), 0.0, add=a)[0]
    v = [1 + 64 * (j - 16) for j in range(K)]
    amax = max(abs(t) for t in v)                                  # 1023 at j = 0
    assert q[:2].view(np.uint16)[0] == np.float16(np.float32(amax) / np.float32(127.0)).view(np.uint16)
    want = [_half_away(Fraction(127 * t, amax)) for t in v]
    assert list(q[2:].view(np.int8)) == want


def test_q8_add_zero_is_identity(orc):
    rng = np.random.default_rng(11)
    N, K = 3, 512
    x = rng.standard_normal((N, K)).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(K)).astype(np.float32)
    base = orc.quantize_q8_0(x, g, 1e-6)
    assert np.array_equal(orc.quantize_q8_0(x, g, 1e-6, add=np.zeros(K, np.float32)), base)
    assert np.array_equal(orc.quantize_q8_0(x, g, 1e-6, add=np.zeros((N, K), np.float32)), base)


def test_q8_add_plain_is_sum_then_quantize(orc):
    """Without gamma the ADD reduces to quantizing the fp32 sum x + a."""
    rng = np.random.default_rng(12)
    N, K = 2, 256
    x = rng.standard_normal((N, K)).astype(np.float32)
    a = rng.standard_normal((N, K)).astype(np.float32)
    assert np.array_equal(orc.quantize_q8_0(x, None, add=a), orc.quantize_q8_0(x + a, None))


def test_q8_add_rows_and_broadcast(orc):
    """Row n uses its own addend row; a broadcast addend equals the same row repeated."""
    rng = np.random.default_rng(13)
    N, K = 3, 256
    x = rng.standard_normal((N, K)).astype(np.float32)
    g = rng.standard_normal(K).astype(np.float32)
    a = rng.standard_normal((N, K)).astype(np.float32)
    rows = orc.quantize_q8_0(x, g, 1e-6, add=a)
    for n in range(N):
        assert np.array_equal(rows[n], orc.quantize_q8_0(x[n], g, 1e-6, add=a[n])[0])
    assert np.array_equal(orc.quantize_q8_0(x, g, 1e-6, add=a[1]),
                          orc.quantize_q8_0(x, g, 1e-6, add=np.tile(a[1], (N, 1))))


# ---------------------------------------------------------------- Q4_0 segment layout
SEG_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q4_0_seg_layout.json")


def seg_golden():
    with open(SEG_GOLDEN) as f:
        return json.load(f)


def test_seg_row_bytes_golden(orc):
    g = seg_golden()["row_bytes"]
    assert [orc.q4_0_seg_row_bytes(K) for K in g["K"]] == g["bytes"]


def test_seg_layout_golden_spots(orc):
    g = seg_golden()["one_row"]
    K = g["K"]
    nb = K // 32
    row = np.zeros(nb * 18, dtype=np.uint8)
    for b in range(nb):                      # the fixture's input rule
        row[b * 18] = b
        row[b * 18 + 1] = 0x10
        for j in range(16):
            row[b * 18 + 2 + j] = (5 * b + 3 * j + 1) % 256
    out = orc.repack_q4_0_seg(row[None, :], K)[0]
    assert out.shape[0] == 1408
    for sp in g["spots"]:
        at, want = sp["at"], sp["bytes"]
        assert list(out[at:at + len(want)]) == want, sp["derivation"]


@pytest.mark.parametrize("K", [256, 2304, 4096, 4352])
def test_seg_layout_moves_every_byte_once(orc, K):
    """Every block's 16 nibble bytes appear once, intact and in block order
    within the row's nibble areas; every block's scale appears once among the
    scale words; the remaining halves are zero."""
    rng = np.random.default_rng(K)
    O, nb = 3, K // 32
    Wq = rng.integers(0, 256, size=(O, nb * 18), dtype=np.uint8)
    Wq.reshape(O, nb, 18)[:, :, 1] = rng.integers(1, 0x7B, size=(O, nb), dtype=np.uint8)  # non-zero finite scales
    out = orc.repack_q4_0_seg(Wq, K)
    assert out.shape == (O, orc.q4_0_seg_row_bytes(K))
    for o in range(O):
        nib, scales = [], []
        pos = 0
        left = nb
        while left > 0:
            r = min(64, left)
            nib.append(out[o, pos:pos + 16 * r].reshape(r, 16))
            w = out[o, pos + 16 * r:pos + 16 * r + 128].copy().view(np.uint16).reshape(32, 2)
            scales.append(w)
            pos += 16 * r + 128
            left -= r
        assert pos == out.shape[1]
        got_nib = np.concatenate(nib)
        assert np.array_equal(got_nib, Wq[o].reshape(nb, 18)[:, 2:])
        want_sc = Wq[o].reshape(nb, 18)[:, :2].copy().view(np.uint16)[:, 0]
        halves = np.concatenate([s.reshape(-1) for s in scales])
        nz = halves[halves != 0]
        assert sorted(nz.tolist()) == sorted(want_sc.tolist())
        assert np.count_nonzero(halves) == nb


# ---------------------------------------------------------------- Q8_0 weights
def _q8_block(codes, d_bits):
    blk = np.zeros(34, dtype=np.uint8)
    blk[0] = d_bits & 0xFF
    blk[1] = d_bits >> 8
    blk[2:] = np.array(codes, dtype=np.int8).view(np.uint8)
    return blk


@pytest.mark.parametrize("case", ["q8w_dot", "q8w_extreme"])
def test_q8w_golden(orc, case):
    g = golden()[case]
    W = _q8_block(g["w_codes"], g["w_d_bits"])[None, :]
    x = _q8_block(g["x_codes"], g["x_d_bits"])[None, :]
    assert orc.block_sums(W, x, 32, wtype="q8_0")[0, 0, 0] == g["isum"]
    y32, y64, S = orc.matvec(W, x, 32, wtype="q8_0")
    assert y64[0, 0] == g["y"] and y32[0, 0] == np.float32(g["y"])
    assert S[0, 0] == abs(g["y"])


@pytest.mark.parametrize("O,K,N", [(3, 64, 2), (2, 96, 1)])
def test_q8w_exact_rational(orc, O, K, N):
    """Brute force in exact rationals from the block definition (independent unpack)."""
    rng = np.random.default_rng(O * K + N)
    W = orc.quantize_q8_0(rng.standard_normal((O, K)).astype(np.float32), None)
    x = orc.quantize_q8_0(rng.standard_normal((N, K)).astype(np.float32), None)
    qw, dw = unpack_q8(W, K)
    qx, dx = unpack_q8(x, K)
    isum = orc.block_sums(W, x, K, wtype="q8_0")
    _, y64, S = orc.matvec(W, x, K, wtype="q8_0")
    for n in range(N):
        for o in range(O):
            exact = Fraction(0)
            mag = Fraction(0)
            for b in range(K // 32):
                s = sum(int(qw[o, 32 * b + j]) * int(qx[n, 32 * b + j]) for j in range(32))
                assert isum[n, o, b] == s
                term = Fraction(float(dw[o, b])) * Fraction(float(dx[n, b])) * s
                exact += term
                mag += abs(term)
            assert abs(Fraction(float(y64[n, o])) - exact) <= Fraction(1, 10 ** 12) * (mag + 1)
            assert abs(float(S[n, o]) - float(mag)) <= 1e-12 * float(mag) + 1e-300


# ---------------------------------------------------------------- Q4_K weights
def _q4k_golden_block(g):
    """The hand-derived super-block: header bytes as written in the golden
    file, codes by its rule and nibble placement."""
    blk = np.zeros(144, dtype=np.uint8)
    blk[0], blk[1] = g["d_bits"] & 0xFF, g["d_bits"] >> 8
    blk[2], blk[3] = g["dmin_bits"] & 0xFF, g["dmin_bits"] >> 8
    blk[4:16] = g["scales_bytes"]
    for j in range(8):
        for i in range(32):
            q = (i + 3 * j) % 16
            b = 16 + 32 * (j // 2) + i
            blk[b] |= np.uint8(q if j % 2 == 0 else q << 4)
    return blk


def _ones_q8(nblocks, d_bits):
    x = np.zeros((1, nblocks * 34), dtype=np.uint8)
    for b in range(nblocks):
        x[0, 34 * b] = d_bits & 0xFF
        x[0, 34 * b + 1] = d_bits >> 8
        x[0, 34 * b + 2:34 * b + 34] = 1
    return x


def test_q4k_golden(orc):
    g = golden()["q4k_superblock"]
    blk = _q4k_golden_block(g)
    for k, v in g["spot_bytes"].items():
        assert int(blk[int(k)]) == v
    deq = orc.dequantize_q4_k(blk[None, :], 256)[0]
    for k, v in g["spot_values"].items():
        assert deq[int(k)] == v
    for j in range(8):
        for i in range(32):
            assert deq[32 * j + i] == 0.5 * g["sc"][j] * ((i + 3 * j) % 16) - 0.25 * g["m"][j], (j, i)
    x = _ones_q8(8, g["x_d_bits"])
    isum = orc.block_sums(blk[None, :], x, 256, wtype="q4_k")
    assert np.all(isum == g["isum_each"])
    y32, y64, S = orc.matvec(blk[None, :], x, 256, wtype="q4_k")
    assert y64[0, 0] == g["y"] and y32[0, 0] == np.float32(g["y"]) and S[0, 0] == g["S"]


def test_q4k_quantizer_special_blocks(orc):
    w = np.zeros((3, 256), dtype=np.float32)
    w[1, :] = 0.75                                     # one positive constant
    w[2, :] = np.tile((np.arange(32) % 16) * 0.25 - 1.0, 8)   # codes 0..15 on an exact grid
    Wq = orc.quantize_q4_k(w)
    deq = orc.dequantize_q4_k(Wq, 256)
    assert np.all(Wq[0] == 0) and np.all(deq[0] == 0.0)       # zero block: everything zero
    assert np.all(np.abs(deq[1] - 0.75) <= 0.75 * 2.0 ** -8)   # within the fp16 scale's rounding
    nib = Wq[2, 16:]
    codes = np.concatenate([np.stack([nib[32 * p:32 * p + 32] & 15, nib[32 * p:32 * p + 32] >> 4]).reshape(-1)
                            for p in range(4)])
    assert np.array_equal(codes, np.tile(np.arange(32) % 16, 8))
    assert np.max(np.abs(deq[2] - w[2])) <= 4e-3


def test_q4k_quantizer_roundtrip_random(orc):
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((24, 1024)) * 0.02).astype(np.float32)
    Wq = orc.quantize_q4_k(w)
    deq = orc.dequantize_q4_k(Wq, 1024)
    err = np.abs(deq - w).reshape(24, 32, 32).max(axis=2)
    rng_ = (w.reshape(24, 32, 32).max(axis=2) - np.minimum(w.reshape(24, 32, 32).min(axis=2), 0))
    assert np.all(err <= 0.75 * rng_ / 15 + 1e-7)      # within three quarters of a code step


def test_q4k_matvec_vs_numpy_dequant(orc):
    rng = np.random.default_rng(12)
    K = 512
    W = orc.quantize_q4_k((rng.standard_normal((5, K)) * 0.02).astype(np.float32))
    x = orc.quantize_q8_0(rng.standard_normal((2, K)).astype(np.float32), None)
    qx = x.reshape(2, K // 32, 34)
    dx = qx[:, :, :2].copy().view(np.float16).astype(np.float64)[:, :, 0]
    xv = (qx[:, :, 2:].view(np.int8).astype(np.float64) * dx[:, :, None]).reshape(2, K)
    ref = xv @ orc.dequantize_q4_k(W, K).T
    _, y64, S = orc.matvec(W, x, K, wtype="q4_k")
    assert np.all(np.abs(y64 - ref) <= 1e-12 * (S + 1e-30))


# ---------------------------------------------------------------- Q5_K weights
def _q5k_golden_block(g):
    """The hand-derived Q5_K super-block: header bytes from the golden file,
    codes by its rule, low four bits placed as the Q4_K codes from byte 48,
    top bits in qh (bit j of byte 16 + i for element i of sub-block j)."""
    blk = np.zeros(176, dtype=np.uint8)
    blk[0], blk[1] = g["d_bits"] & 0xFF, g["d_bits"] >> 8
    blk[2], blk[3] = g["dmin_bits"] & 0xFF, g["dmin_bits"] >> 8
    blk[4:16] = g["scales_bytes"]
    for j in range(8):
        for i in range(32):
            q = (i + 3 * j) % 32
            b = 48 + 32 * (j // 2) + i
            blk[b] |= np.uint8((q & 15) if j % 2 == 0 else (q & 15) << 4)
            blk[16 + i] |= np.uint8((q >> 4) << j)
    return blk


def _q5k_codes(Wrow):
    """Codes of one Q5_K super-block by the documented placement (Python)."""
    qh, low = Wrow[16:48], Wrow[48:176]
    out = np.zeros(256, dtype=np.int64)
    for j in range(8):
        for i in range(32):
            byte = int(low[32 * (j // 2) + i])
            lo = byte & 15 if j % 2 == 0 else byte >> 4
            out[32 * j + i] = lo + 16 * ((int(qh[i]) >> j) & 1)
    return out


def test_q5k_golden(orc):
    g = golden()["q5k_superblock"]
    blk = _q5k_golden_block(g)
    for k, v in g["spot_bytes"].items():
        assert int(blk[int(k)]) == v, k
    deq = orc.dequantize_q5_k(blk[None, :], 256)[0]
    for k, v in g["spot_values"].items():
        assert deq[int(k)] == v, k
    for j in range(8):
        for i in range(32):
            assert deq[32 * j + i] == 0.5 * g["sc"][j] * ((i + 3 * j) % 32) - 0.25 * g["m"][j], (j, i)
    x = _ones_q8(8, g["x_d_bits"])
    isum = orc.block_sums(blk[None, :], x, 256, wtype="q5_k")
    assert np.all(isum == g["isum_each"])
    y32, y64, S = orc.matvec(blk[None, :], x, 256, wtype="q5_k")
    assert y64[0, 0] == g["y"] and y32[0, 0] == np.float32(g["y"]) and S[0, 0] == g["S"]


def test_q5k_quantizer_special_blocks(orc):
    w = np.zeros((3, 256), dtype=np.float32)
    w[1, :] = 0.75                                     # one positive constant
    w[2, :] = np.tile(np.arange(32) * 0.25 - 1.0, 8)  # codes 0..31 on an exact grid
    Wq = orc.quantize_q5_k(w)
    deq = orc.dequantize_q5_k(Wq, 256)
    assert np.all(Wq[0] == 0) and np.all(deq[0] == 0.0)       # zero block: everything zero
    assert np.all(np.abs(deq[1] - 0.75) <= 0.75 * 2.0 ** -8)   # within the fp16 scale's rounding
    assert np.array_equal(_q5k_codes(Wq[2]), np.tile(np.arange(32), 8))
    assert np.max(np.abs(deq[2] - w[2])) <= 4e-3


def test_q5k_quantizer_roundtrip_random(orc):
    rng = np.random.default_rng(13)
    w = (rng.standard_normal((24, 1024)) * 0.02).astype(np.float32)
    Wq = orc.quantize_q5_k(w)
    deq = orc.dequantize_q5_k(Wq, 1024)
    err = np.abs(deq - w).reshape(24, 32, 32).max(axis=2)
    rng_ = (w.reshape(24, 32, 32).max(axis=2) - np.minimum(w.reshape(24, 32, 32).min(axis=2), 0))
    assert np.all(err <= 0.75 * rng_ / 31 + 1e-7)      # within three quarters of a code step
    # the codes the bytes hold are the ones the dequantizer used
    for r in range(3):
        codes = _q5k_codes(Wq[r, :176])
        assert codes.max() <= 31 and codes.min() >= 0


def test_q5k_matvec_vs_numpy_dequant(orc):
    rng = np.random.default_rng(14)
    K = 512
    W = orc.quantize_q5_k((rng.standard_normal((5, K)) * 0.02).astype(np.float32))
    x = orc.quantize_q8_0(rng.standard_normal((2, K)).astype(np.float32), None)
    qx = x.reshape(2, K // 32, 34)
    dx = qx[:, :, :2].copy().view(np.float16).astype(np.float64)[:, :, 0]
    xv = (qx[:, :, 2:].view(np.int8).astype(np.float64) * dx[:, :, None]).reshape(2, K)
    ref = xv @ orc.dequantize_q5_k(W, K).T
    _, y64, S = orc.matvec(W, x, K, wtype="q5_k")
    assert np.all(np.abs(y64 - ref) <= 1e-12 * (S + 1e-30))
    # exact block sums against a Python restatement of the code placement
    isum = orc.block_sums(W, x, K, wtype="q5_k")
    qxi = qx[:, :, 2:].view(np.int8).astype(np.int64)
    for o in range(5):
        codes = np.concatenate([_q5k_codes(W[o, 176 * s:176 * (s + 1)]) for s in range(K // 256)])
        ref_sums = (codes.reshape(K // 32, 32)[None] * qxi).sum(axis=2)
        assert np.array_equal(isum[:, o, :], ref_sums)
