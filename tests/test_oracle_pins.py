"""Pins for the CPU oracle: each check ties an oracle function to something
other than itself -- hand-worked examples from the format definition, brute
force over the code table, closed forms, and library routines (torch's
float8_e4m3fn / bfloat16 casts, torch's silu) on the cases where they coincide
with the definition.  No GPU.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers --

def _bf16(x):
    return synth.to_bf16_bits(np.asarray(x, dtype=np.float32))


def _f32_from_bf16(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _code_values():
    """Brute-force side: value of each code from sign/exponent/mantissa fields."""
    vals = {}
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue
        v = Fraction(m, 512) if e == 0 else Fraction(8 + m, 8) * Fraction(2) ** (e - 7)
        vals[c] = -v if s else v
    return vals


_POS = sorted((v, c) for c, v in _code_values().items() if c < 128)
_POS_VALS = np.array([float(v) for v, _ in _POS])
_POS_CODES = np.array([c for _, c in _POS], dtype=np.int64)


def nearest_code(x: np.ndarray) -> np.ndarray:
    """Brute force: nearest finite e4m3 value, ties to the even code, |x| beyond
    the finite range (nearest would be 480) saturating to 448."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    idx = np.searchsorted(_POS_VALS, a)            # first value >= a
    hi = np.clip(idx, 0, len(_POS_VALS) - 1)
    lo = np.clip(idx - 1, 0, len(_POS_VALS) - 1)
    dlo = np.abs(a - _POS_VALS[lo])
    dhi = np.abs(_POS_VALS[hi] - a)
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi,
                    np.where(_POS_CODES[lo] % 2 == 0, lo, hi)))
    code = _POS_CODES[pick]
    # above 448 the nearest representable neighbour in the infinitely extended
    # format is 480 (odd code): 464 is the tie (-> 448), everything else saturates
    code = np.where(a >= 448.0, 0x7E, code)
    sign = np.signbit(x).astype(np.int64) << 7
    return (code | sign).astype(np.uint8)


def _read_codec_golden():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_codec_worked.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = line.split()
            rows.append((float.fromhex(parts[0]), int(parts[1], 16), " ".join(parts[2:])))
    return rows


def _read_group_golden():
    ex, cur = [], None
    with open(os.path.join(GOLDEN, "group_quant_worked.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            key, *rest = line.split()
            if key == "example":
                cur = {"name": rest[0], "x": {}, "fill": 0.0, "q": {}, "qfill": 0}
                ex.append(cur)
            elif key == "x":
                for tok in rest:
                    i, v = tok.split(":")
                    cur["x"][int(i)] = float.fromhex(v)
            elif key == "fill":
                cur["fill"] = float.fromhex(rest[0])
            elif key == "s":
                cur["s"] = float.fromhex(rest[0])
            elif key == "q":
                for tok in rest:
                    i, v = tok.split(":")
                    cur["q"][int(i)] = int(v, 16)
            elif key == "qfill":
                cur["qfill"] = int(rest[0], 16)
    return ex


# ------------------------------------------------------------------ codec --

@pytest.mark.parametrize("value,code,note", _read_codec_golden())
def test_codec_worked_examples(oracle, value, code, note):
    assert oracle.e4m3_encode(value) == code, note


def test_decode_all_codes_vs_torch(oracle):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode_table()
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    # and against the field definition
    vals = _code_values()
    for c, v in vals.items():
        assert got[c] == float(v)


def _codec_probe_set(rng):
    # every e4m3 value, every midpoint between neighbours, and +-1,2 fp32 ulps around them
    v = _POS_VALS.astype(np.float32)
    mids = ((_POS_VALS[1:] + _POS_VALS[:-1]) / 2).astype(np.float32)
    base = np.concatenate([v, mids, np.float32([448, 464, 480, 1e6, 3.4e38, 1e-30, 1e-45])])
    around = [base]
    for k in (1, 2):
        around.append(np.nextafter(base, np.float32(np.inf)))
        around.append(np.nextafter(base, np.float32(0)))
        base = np.concatenate([around[-1], around[-2]])
    pts = np.concatenate(around)
    # random magnitudes over the whole fp32 exponent range
    bits = rng.integers(0, 0x7F800000, size=400_000, dtype=np.uint32)
    pts = np.concatenate([pts, bits.view(np.float32),
                          rng.uniform(0, 512, 200_000).astype(np.float32),
                          rng.uniform(0, 0.02, 200_000).astype(np.float32)])
    return np.concatenate([pts, -pts]).astype(np.float32)


def test_encode_bruteforce(oracle):
    rng = np.random.default_rng(11)
    x = _codec_probe_set(rng)
    assert np.array_equal(oracle.e4m3_encode_array(x), nearest_code(x))


def test_encode_dense_sweep(oracle):
    """Every fp32 pattern in [2^-11, 2^9) with a stride of 3 (about 56M values),
    checked against the brute-force nearest code."""
    lo = np.float32(2.0 ** -11).view(np.uint32)
    hi = np.float32(2.0 ** 9).view(np.uint32)
    step = 1 << 22
    for start in range(int(lo), int(hi), step):
        n = min(step, int(hi) - start)
        got = oracle.e4m3_encode_bits(start, n)[::3]
        x = np.arange(start, start + n, dtype=np.uint32)[::3].view(np.float32)
        ref = nearest_code(x)
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, (x[bad[:5]], got[bad[:5]], ref[bad[:5]])


def test_encode_vs_torch_nonsaturating(oracle):
    """torch's float8_e4m3fn cast rounds to nearest even and returns NaN above the
    finite range instead of saturating; the two agree for |x| <= 464."""
    rng = np.random.default_rng(12)
    x = _codec_probe_set(rng)
    x = x[np.abs(x) <= 464.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode_array(x), ref)


# ------------------------------------------------------------------- bf16 --

def test_bf16_rounding_vs_torch(oracle):
    rng = np.random.default_rng(13)
    bits = rng.integers(0, 0xFFFFFFFF, size=300_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    # ties: values exactly halfway between bf16 neighbours
    ties = ((rng.integers(0, 1 << 16, 50_000).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties)]
    x = np.concatenate([x, ties, np.float32([0.0, -0.0, 1e-40, -1e-40, 3.3e38])])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f32_to_bf16_bits(x), ref)


def test_f64_to_bf16_single_rounding(oracle):
    # 1 + 2^-8 + 2^-40: just above the midpoint between 1.0 and 1 + 2^-7;
    # rounding through fp32 first would land on the tie and go to 1.0.
    assert oracle.f64_to_bf16_bits(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert oracle.f64_to_bf16_bits(1.0 + 2.0 ** -8) == 0x3F80           # tie -> even
    assert oracle.f64_to_bf16_bits(1.0 + 3 * 2.0 ** -8) == 0x3F82       # tie -> even
    assert oracle.f64_to_bf16_bits(-2.0 ** -133) == 0x8001               # smallest subnormal
    assert oracle.f64_to_bf16_bits(2.0 ** 128) == 0x7F80


# --------------------------------------------------------- group quant --

@pytest.mark.parametrize("ex", _read_group_golden(), ids=lambda e: e["name"])
def test_group_quant_worked(oracle, ex):
    x = np.full(128, ex["fill"], dtype=np.float32)
    for i, v in ex["x"].items():
        x[i] = v
    xb = _bf16(x)[None, :]
    assert np.array_equal(_f32_from_bf16(xb)[0], x), "example values must be exact bf16"
    q, s = oracle.quant_group(xb)
    assert s.shape == (1, 1)
    assert s[0, 0] == np.float32(ex["s"]), (s[0, 0], ex["s"])
    exp_q = np.full(128, ex["qfill"], dtype=np.uint8)
    for i, c in ex["q"].items():
        exp_q[i] = c
    # unlisted entries that are zero in x quantise to 0x00
    for i in range(128):
        if i not in ex["q"] and x[i] == 0.0:
            exp_q[i] = 0x80 if np.signbit(x[i]) and ex["s"] != 0 else 0x00
    assert np.array_equal(q[0], exp_q), np.nonzero(q[0] != exp_q)


def _random_groups(rng, M, K, p=0.01, factor=20.0):
    x = rng.standard_normal((M, K)).astype(np.float32)
    mask = rng.random((M, K)) < p
    x[mask] *= factor
    return _bf16(x)


def test_group_quant_bruteforce(oracle):
    rng = np.random.default_rng(21)
    M, K = 7, 640
    xb = _random_groups(rng, M, K)
    xb[2, 128:256] = 0                                   # a zero group
    xb[3, 256:384] = _bf16(np.full(128, 1e-38, np.float32))  # tiny amax -> subnormal scale
    q, s = oracle.quant_group(xb)
    x = _f32_from_bf16(xb)
    for m in range(M):
        for g in range(K // 128):
            grp = x[m, 128 * g:128 * (g + 1)]
            amax = np.float32(np.abs(grp).max())
            s_ref = amax / np.float32(448.0)              # one IEEE fp32 division (numpy)
            assert s[m, g] == s_ref
            if amax == 0:
                assert not q[m, 128 * g:128 * (g + 1)].any()
                continue
            t = grp / s_ref                               # numpy fp32 division
            assert np.array_equal(q[m, 128 * g:128 * (g + 1)], nearest_code(t))


def test_group_quant_one_scale_per_row(oracle):
    """group = K gives the one-scale-per-row reading: s[m] = max|x[m]| / 448."""
    rng = np.random.default_rng(22)
    xb = _random_groups(rng, 5, 512)
    q, s = oracle.quant_group(xb, group=512)
    x = _f32_from_bf16(xb)
    assert s.shape == (5, 1)
    assert np.array_equal(s[:, 0], np.abs(x).max(axis=1).astype(np.float32) / np.float32(448))
    assert np.array_equal(q, nearest_code(x / s))


def test_weight_block_quant(oracle):
    rng = np.random.default_rng(23)
    N, K = 384, 256                       # 3 x 2 blocks, distinct amax per block
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    for nb in range(3):
        for kb in range(2):
            w[128 * nb + 5, 128 * kb + 7] = 0.5 + nb + 10 * kb   # block's max, unique per block
    q, s = oracle.quant_block128(w)
    assert s.shape == (3, 2)
    for nb in range(3):
        for kb in range(2):
            blk = w[128 * nb:128 * (nb + 1), 128 * kb:128 * (kb + 1)]
            s_ref = np.float32(0.5 + nb + 10 * kb) / np.float32(448)
            assert s[nb, kb] == s_ref
            assert np.array_equal(q[128 * nb:128 * (nb + 1), 128 * kb:128 * (kb + 1)],
                                  nearest_code(blk / s_ref))


# ------------------------------------------------------------------ GEMM --

def test_gemm_w8a8_closed_form(oracle):
    """x[m][k] = 448 * 2^a_m, w[n][k] = 448 * 2^(b_{n/128} + c_{k/128}): every
    code is 0x7E and every scale a power of two, so
    y[m][n] = 128 * 448^2 * sum_kb 2^(a_m + b_nb + c_kb) exactly."""
    M, N, K = 3, 384, 512
    a = np.array([0, -3, 2])
    b = np.array([1, -2, 0])
    c = np.array([0, 1, -1, 3])
    sign = np.array([1, -1, 1])
    x = (448.0 * sign[:, None] * 2.0 ** a[:, None] * np.ones((M, K))).astype(np.float32)
    w = np.empty((N, K), dtype=np.float32)
    for nb in range(3):
        for kb in range(4):
            w[128 * nb:128 * (nb + 1), 128 * kb:128 * (kb + 1)] = 448.0 * 2.0 ** (b[nb] + c[kb])
    xq, xs = oracle.quant_group(_bf16(x))
    wq, ws = oracle.quant_block128(w)
    assert (wq == 0x7E).all() and set(np.unique(xq)) <= {0x7E, 0xFE}
    acc, y = oracle.gemm_w8a8(xq, xs, wq, ws)
    for m in range(M):
        for n in range(N):
            exact = sign[m] * 128 * 448 ** 2 * sum(2.0 ** (a[m] + b[n // 128] + c[kb]) for kb in range(4))
            assert acc[m, n] == exact
    assert np.array_equal(y, torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def _exact_w8a8(aq, a_s, w, ws):
    vals = _code_values()
    M, K = aq.shape
    N = w.shape[0]
    out = np.empty((M, N), dtype=object)
    absum = np.empty((M, N), dtype=object)
    for m in range(M):
        for n in range(N):
            tot, ab = Fraction(0), Fraction(0)
            for kb in range(K // 128):
                p = sum(vals[int(aq[m, k])] * vals[int(w[n, k])] for k in range(128 * kb, 128 * kb + 128))
                pa = sum(abs(vals[int(aq[m, k])] * vals[int(w[n, k])]) for k in range(128 * kb, 128 * kb + 128))
                sc = Fraction(float(a_s[m, kb])) * Fraction(float(ws[n // 128, kb]))
                tot += p * sc
                ab += pa * abs(sc)
            out[m, n], absum[m, n] = tot, ab
    return out, absum


def _finite_codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint16).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x7E
    return c


def test_gemm_w8a8_bruteforce_exact(oracle):
    """Tiny asymmetric shapes with random codes and scales: the oracle's fp32
    result is within the fp32 summation bound of the exact rational value."""
    rng = np.random.default_rng(31)
    M, N, K = 3, 256, 384
    aq = _finite_codes(rng, (M, K))
    wq = _finite_codes(rng, (N, K))
    a_s = rng.uniform(0.001, 0.1, (M, K // 128)).astype(np.float32)
    ws = rng.uniform(1e-5, 1e-3, (N // 128, K // 128)).astype(np.float32)
    acc, _ = oracle.gemm_w8a8(aq, a_s, wq, ws)
    exact, absum = _exact_w8a8(aq, a_s, wq, ws)
    u = Fraction(1, 1 << 24)
    gamma = (128 + 2 + K // 128) * u
    for m in range(M):
        for n in range(N):
            assert abs(Fraction(float(acc[m, n])) - exact[m, n]) <= gamma * absum[m, n] * Fraction(101, 100)
    # rows subset returns the same values in the requested order
    acc2, _ = oracle.gemm_w8a8(aq, a_s, wq, ws, rows=np.array([2, 0]))
    assert np.array_equal(acc2, acc[[2, 0]])


def test_gemm_w8bf16_closed_form(oracle):
    """x = 2^a_m (bf16), w = 448 * 2^b per 128x128 block: codes 0x7E, scales 2^b,
    y[m][n] = 448 * sum_kb 128 * 2^(a_m + b_{nb,kb})."""
    M, N, K = 2, 256, 384
    a = np.array([0, -1])
    b = np.array([[0, 1, 2], [-1, 0, 3]])
    x = (2.0 ** a[:, None] * np.ones((M, K))).astype(np.float32)
    w = np.empty((N, K), dtype=np.float32)
    for nb in range(2):
        for kb in range(3):
            w[128 * nb:128 * (nb + 1), 128 * kb:128 * (kb + 1)] = 448.0 * 2.0 ** b[nb, kb]
    wq, ws = oracle.quant_block128(w)
    acc, _ = oracle.gemm_w8bf16(_bf16(x), wq, ws)
    for m in range(M):
        for n in range(N):
            assert acc[m, n] == 448 * 128 * sum(2.0 ** (a[m] + b[n // 128, kb]) for kb in range(3))


def test_gemm_w8bf16_bruteforce_exact(oracle):
    rng = np.random.default_rng(32)
    M, N, K = 2, 256, 256
    xb = _random_groups(rng, M, K)
    wq = _finite_codes(rng, (N, K))
    ws = rng.uniform(1e-5, 1e-3, (N // 128, K // 128)).astype(np.float32)
    acc, _ = oracle.gemm_w8bf16(xb, wq, ws)
    vals = _code_values()
    x = _f32_from_bf16(xb)
    u = Fraction(1, 1 << 24)
    for m in range(M):
        for n in range(N):
            tot, ab = Fraction(0), Fraction(0)
            for kb in range(K // 128):
                terms = [Fraction(float(x[m, k])) * vals[int(wq[n, k])] for k in range(128 * kb, 128 * kb + 128)]
                sc = Fraction(float(ws[n // 128, kb]))
                tot += sum(terms) * sc
                ab += sum(abs(t) for t in terms) * sc
            assert abs(Fraction(float(acc[m, n])) - tot) <= (131 + K // 128) * u * ab * Fraction(101, 100)


def test_gemm_weight_only_all_codes_one_hot(oracle):
    """One-hot activations pick single weight codes: y = bf16(value(code) * ws)."""
    K, N = 128, 256
    wq = np.arange(N * K, dtype=np.int64).reshape(N, K) % 256
    wq = wq.astype(np.uint8)
    wq[(wq & 0x7F) == 0x7F] = 0
    ws = np.array([[1.0], [0.25]], dtype=np.float32)
    x = np.zeros((4, K), np.float32)
    for m, k in enumerate((0, 1, 77, 127)):
        x[m, k] = 1.0
    acc, _ = oracle.gemm_w8bf16(_bf16(x), wq, ws)
    tab = oracle.e4m3_decode_table()
    for m, k in enumerate((0, 1, 77, 127)):
        assert np.array_equal(acc[m], (tab[wq[:, k]] * np.repeat(ws[:, 0], 128)).astype(np.float32))


# ------------------------------------------------------------------- exp --

def _exp_sweep_points():
    """Every 397th fp32 pattern of [-104, ln(FLT_MAX)) plus every bf16 value there."""
    hi = np.float32(88.72).view(np.uint32)
    lo = np.float32(-104.0).view(np.uint32)
    pos = np.arange(0, hi + 1, 397, dtype=np.uint32)
    neg = np.arange(0x80000000, lo + 1, 397, dtype=np.uint32)
    b = np.arange(0, 1 << 16, dtype=np.uint32) << 16
    bx = b.view(np.float32)
    bx = b[np.isfinite(bx) & (bx >= -104.0) & (bx <= 88.72)]
    return np.concatenate([pos, neg, bx]).view(np.float32)


def test_expf_dense_sweep(oracle):
    """The oracle's exp (Cody-Waite reduction, degree-7 Taylor polynomial, one
    final scaling) against float64 exp: below 1 ulp everywhere on the sweep
    (subnormal results included, where the ulp is 2^-149), and correctly
    rounded at >= 99 % of the points.  A dropped polynomial term, a wrong
    reduction constant or a sign error breaks one of the two."""
    x = _exp_sweep_points()
    y = oracle.expf(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(np.abs(ref.astype(np.float32))).astype(np.float64)
    err = np.abs(y - ref) / ulp
    assert err.max() < 1.0, (float(err.max()), float(x[np.argmax(err)]))
    assert np.mean(y == ref.astype(np.float32)) >= 0.99


def test_expf_special_values(oracle):
    """exp(+-0) = 1 exactly; e^x for x above ln(FLT_MAX) (88.7228...) by more than
    one part in 1e7 overflows to +inf (the true value then rounds to inf); below
    -104 (e^-104 < 2^-150, half the smallest subnormal) it is +0; powers of two
    k*ln2 land within an ulp of 2^k."""
    assert oracle.expf(np.float32([0.0, -0.0])).tolist() == [1.0, 1.0]
    over = np.float32([88.7229, 88.75, 88.8, 88.81, 100.0, 1e30])
    assert np.all(np.isinf(oracle.expf(over)) & (oracle.expf(over) > 0))
    under = np.float32([-104.01, -150.0, -1e30])
    got = oracle.expf(under)
    assert np.all(got == 0.0) and not np.any(np.signbit(got))
    k = np.arange(-120, 120)
    x = (k * np.log(2.0)).astype(np.float32)
    ref = np.exp(x.astype(np.float64))
    assert np.all(np.abs(oracle.expf(x) - ref) <= np.spacing(ref.astype(np.float32)))


# ---------------------------------------------------------------- SwiGLU --

def _near_bf16(h_bits, ref64):
    """h (bf16 bits) is the bf16 rounding of an fp32 evaluation of ref64:
    within half a bf16 ulp of ref64 plus the fp32 evaluation error (four fp32
    ulps: exp below one, then the add, the divide and the multiply).  Where
    |ref64| is past the largest bf16 (3.3895e38 plus half an ulp), h is the
    infinity of its sign."""
    h = _f32_from_bf16(h_bits).astype(np.float64)
    a = np.abs(ref64)
    over = a >= float.fromhex("0x1.ff0000p+127")
    a32 = np.where(over, 1.0, a).astype(np.float32)
    ulp32 = np.spacing(a32).astype(np.float64)
    ulp16 = ulp32 * 65536.0
    with np.errstate(invalid="ignore"):
        near = np.abs(h - ref64) <= 0.5 * ulp16 + 4.0 * ulp32 + 1e-45
    return np.where(over, np.isinf(h) & (np.signbit(h) == np.signbit(ref64)), near)


def test_swiglu_special_cases(oracle):
    """u == 1: h = bf16(silu(g)); u == 2: h = bf16(2 silu(g)) (a swapped
    interleave would give silu(2) * g instead).  silu from torch in float64:
    h equals its bf16 rounding except within the fp32 evaluation error of a
    rounding boundary, where it is one of the two neighbours."""
    rng = np.random.default_rng(41)
    M, I = 3, 256
    g = _f32_from_bf16(_bf16(rng.standard_normal((M, I)) * 4))
    for uval in (1.0, 2.0):
        gu = np.empty((M, 2 * I), dtype=np.float32)
        for j in range(I // 128):
            gu[:, 256 * j:256 * j + 128] = g[:, 128 * j:128 * (j + 1)]
            gu[:, 256 * j + 128:256 * (j + 1)] = uval
        h = oracle.swiglu_interleaved(_bf16(gu))
        ref64 = torch.nn.functional.silu(torch.from_numpy(g.astype(np.float64))).numpy() * uval
        ref = np.array([oracle.f64_to_bf16_bits(v) for v in ref64.ravel()], dtype=np.uint16).reshape(M, I)
        assert np.all(_near_bf16(h, ref64))
        assert np.mean(h == ref) >= 0.99


def test_swiglu_every_bf16_gate(oracle):
    """Every finite bf16 gate value g with u = 1 and u = -3: the fp32 SwiGLU
    against float64 silu(g)*u.  Products past the bf16 range give infinities of
    the right sign; below g = -88.8 the fp32 evaluation gives a signed zero."""
    b = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    g = _f32_from_bf16(b)
    b = b[np.isfinite(g)]
    g = g[np.isfinite(g)]
    for uval in (1.0, -3.0):
        gu = np.empty((1, 2 * 128 * ((g.size + 127) // 128)), dtype=np.uint16)
        n = g.size
        pad = gu.shape[1] // 2 - n
        gg = np.concatenate([b, np.zeros(pad, np.uint16)]).reshape(-1, 128)
        uu = np.full_like(gg, _bf16(np.float32([uval]))[0])
        gu[0] = np.stack([gg, uu], axis=1).reshape(-1)
        h = oracle.swiglu_interleaved(gu)[0, :n]
        with np.errstate(over="ignore"):
            ref64 = g.astype(np.float64) / (1.0 + np.exp(-g.astype(np.float64))) * uval
        # below -88.8 the fp32 exp(-g) overflows, so silu(g) is -0 (times u)
        # where float64 still gives a tiny negative number
        flushed = g < -88.8
        assert np.all(_f32_from_bf16(h[flushed]) == 0.0)
        assert np.all(np.signbit(_f32_from_bf16(h[flushed])) == (uval > 0))
        assert np.all(_near_bf16(h[~flushed], ref64[~flushed]))


def test_gate_up_swiglu_down_wiring(oracle):
    """The fused MLP equals the chain of pinned pieces, with the gate/up
    interleave read through a numpy view ([M][I/128][gate|up][128])."""
    rng = np.random.default_rng(42)
    M, H, I, Hout = 3, 256, 256, 384
    xb = _random_groups(rng, M, H)
    w_gu, s_gu = oracle.quant_block128((rng.standard_normal((2 * I, H)) * 0.02).astype(np.float32))
    w_dn, s_dn = oracle.quant_block128((rng.standard_normal((Hout, I)) * 0.02).astype(np.float32))
    for weight_only in (False, True):
        r = oracle.gate_up_swiglu_down(xb, w_gu, s_gu, w_dn, s_dn, weight_only=weight_only)
        if weight_only:
            _, gu = oracle.gemm_w8bf16(xb, w_gu, s_gu)
        else:
            xq, xs = oracle.quant_group(xb)
            _, gu = oracle.gemm_w8a8(xq, xs, w_gu, s_gu)
        assert np.array_equal(r["gu"], gu)
        v = _f32_from_bf16(gu).reshape(M, I // 128, 2, 128)
        g, u = v[:, :, 0, :].reshape(M, I), v[:, :, 1, :].reshape(M, I)
        h64 = torch.nn.functional.silu(torch.from_numpy(g.astype(np.float64))).numpy() * u
        assert np.all(_near_bf16(r["h"], h64))
        h = r["h"]
        if weight_only:
            _, y = oracle.gemm_w8bf16(h, w_dn, s_dn)
        else:
            hq, hs = oracle.quant_group(h)
            assert np.array_equal(r["hq"], hq) and np.array_equal(r["hs"], hs)
            _, y = oracle.gemm_w8a8(hq, hs, w_dn, s_dn)
        assert np.array_equal(r["y"], y)


# ------------------------------------------------------------- tolerance --

def test_tolerance_helper(oracle):
    ref = np.array([1.0, -2.0, 100.0])
    ok, worst = oracle.tolerance_ok(ref * (1 + 7e-3), ref)
    assert ok and worst < 1.0
    ok, _ = oracle.tolerance_ok(ref + np.array([0.0, 0.0, 1.0 + 0.1]), ref)
    assert not ok
