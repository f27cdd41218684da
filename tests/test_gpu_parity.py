"""GPU parity: every entry point of libr9q, called through the C ABI binding,
against the CPU oracle on the same seeded inputs.

  * e4m3 conversion, group-128 quant and weight block quant: bit-exact;
  * GEMM outputs: |gpu - ref| <= 8e-3 |ref| + 1e-3 max|ref| per element, ref =
    the oracle's fp32 accumulator on the same (bit-identical) quantised operands;
  * fused vs unfused quant: identical bytes, scales and outputs;
  * fused expert MLP vs the separate-launch chain: identical h, hq, hs, y.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _helpers import (activations_bf16, assert_close, bf16_to_dev, bits_of, dev, f32_of_bits,
                      quantised_weights)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def r9q():
    import __graft_entry__
    __graft_entry__.build()
    import block_scaled_fp8_x128_gb300 as lib
    return lib


# ------------------------------------------------------------------ codec --

def test_codec_dense_range(r9q):
    """Every fp32 pattern with |x| in [2^-12, 2^10), both signs, plus samples of
    all other finite patterns: GPU cvt.rn.satfinite == oracle codec."""
    lo = int(np.float32(2.0 ** -12).view(np.uint32))
    hi = int(np.float32(2.0 ** 10).view(np.uint32))
    step = 1 << 24
    for sign in (0, 0x80000000):
        for start in range(lo, hi, step):
            n = min(step, hi - start)
            ref = oracle.e4m3_encode_bits(start | sign, n)
            pat = np.arange(start, start + n, dtype=np.uint32) | np.uint32(sign)
            q = r9q.r9q_e4m3_from_f32(torch.from_numpy(pat.view(np.float32)).to(dev()))
            got = q.cpu().numpy()
            bad = np.nonzero(got != ref)[0]
            assert bad.size == 0, [(hex((start | sign) + int(i)), got[i], ref[i]) for i in bad[:5]]


def test_codec_sampled_all_patterns(r9q):
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 32, size=4_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    x = np.concatenate([x, np.float32([0.0, -0.0, 448, 464, -464, 480, 1e38, -1e38, 1e-45])])
    got = r9q.r9q_e4m3_from_f32(torch.from_numpy(x).to(dev())).cpu().numpy()
    assert np.array_equal(got, oracle.e4m3_encode_array(x))
    # tail handling (n not a multiple of 4)
    got7 = r9q.r9q_e4m3_from_f32(torch.from_numpy(x[:7].copy()).to(dev())).cpu().numpy()
    assert np.array_equal(got7, oracle.e4m3_encode_array(x[:7]))


# ---------------------------------------------------------- group quant --

@pytest.mark.parametrize("M,K,p,factor,seed", [
    (1, 1024, 0.01, 20.0, 0),        # c0 activations
    (16, 4096, 0.005, 50.0, 2),      # c2 activations
    (3, 384, 0.0, 1.0, 7),           # ragged M, few groups
    (255, 4096, 0.0, 1.0, 4),        # c4 M=255
])
def test_quant_group128_bit_exact(r9q, M, K, p, factor, seed):
    xb = activations_bf16(seed, M, K, p, factor)
    if M >= 3:
        xb[0, 128:256] = 0                                         # zero group
        xb[1, 0:128] = synth.to_bf16_bits(np.full(128, 1e-38, np.float32))  # subnormal scale
        xb[2, 0] = synth.to_bf16_bits(np.float32([448.0]))[0]      # amax exactly 448 ...
        xb[2, 1:128] = synth.to_bf16_bits(np.float32(np.linspace(-3, 3, 127)))
        xb[2, 5] = 0x8000                                          # ... with a -0.0 inside
    xq, xs = r9q.r9q_quant_group128(bf16_to_dev(xb))
    torch.cuda.synchronize()
    oq, os_ = oracle.quant_group(xb)
    assert np.array_equal(xs.cpu().numpy(), os_)
    assert np.array_equal(xq.cpu().numpy(), oq)


def _every_value_groups(seed=77):
    """Groups [amax, x...]: every finite bf16 magnitude x, both signs, against
    600 group maxima (random bf16 values plus subnormal, tiny and huge ones);
    rows of K = 1024."""
    rng = np.random.default_rng(seed)
    all_pos = np.arange(0, 0x7F80, dtype=np.uint16)                    # finite non-negative bf16
    amaxes = np.concatenate([rng.integers(0x0001, 0x7F80, 590).astype(np.uint16),
                             np.uint16([0x0001, 0x0040, 0x0080, 0x0100, 0x0C00, 0x3F80, 0x43E0, 0x7F7F,
                                        0x7F00, 0x0200])])
    xs_all = f32_of_bits(all_pos)
    groups = []
    for a in amaxes:
        av = f32_of_bits(np.uint16([a]))[0]
        cand = all_pos[xs_all <= av]
        cand = cand[rng.permutation(cand.size)[:4064]]                  # up to 32 groups per amax
        cand = cand | (rng.integers(0, 2, cand.size).astype(np.uint16) << 15)   # random signs
        pad = (-cand.size) % 127
        cand = np.concatenate([cand, np.zeros(pad, np.uint16)]).reshape(-1, 127)
        groups.append(np.concatenate([np.full((cand.shape[0], 1), a, np.uint16), cand], axis=1))
    flat = np.concatenate(groups)
    flat = np.concatenate([flat, np.zeros(((-flat.shape[0]) % 8, 128), np.uint16)])
    return flat.reshape(-1, 1024)


def test_quant_quotient_every_bf16_value(r9q):
    """The quantiser's division-free quotient against the oracle's fp32 division."""
    xb = _every_value_groups()
    xq, xs = r9q.r9q_quant_group128(bf16_to_dev(xb))
    torch.cuda.synchronize()
    oq, os_ = oracle.quant_group(xb)
    assert np.array_equal(xs.cpu().numpy(), os_)
    bad = np.nonzero(xq.cpu().numpy() != oq)
    assert bad[0].size == 0, (bad[0][:5], bad[1][:5])


@pytest.mark.parametrize("rows", [48, None])        # 48: decode kernel's A-load quant; all: prefill kernel
def test_fused_quant_every_bf16_value(r9q, rows):
    """The GEMMs' fused activation quant (decode A-load and the prefill
    kernel's quant phase) on the same groups: codes and scales bit-exact."""
    xb = _every_value_groups()
    if rows is not None:
        xb = xb[:rows]
    M, K = xb.shape
    wq, ws = quantised_weights(r9q, 5, 256, K, check_oracle=False)
    aq = torch.empty((M, K), dtype=torch.uint8, device=dev())
    a_s = torch.empty((M, K // 128), dtype=torch.float32, device=dev())
    r9q.r9q_gemm_fp8_block_qa(bf16_to_dev(xb), wq, ws, aq=aq, as_=a_s)
    torch.cuda.synchronize()
    oq, os_ = oracle.quant_group(xb)
    assert np.array_equal(a_s.cpu().numpy(), os_)
    bad = np.nonzero(aq.cpu().numpy() != oq)
    assert bad[0].size == 0, (bad[0][:5], bad[1][:5])


def test_quant_every_bf16_group_max(r9q):
    """One group per positive finite bf16 maximum (32,639 groups): scales and
    codes bit-exact against the oracle's fp32 divisions."""
    rng = np.random.default_rng(78)
    amax = np.arange(1, 0x7F80, dtype=np.uint16)
    af = f32_of_bits(amax).astype(np.float64)
    frac = rng.uniform(-1.0, 1.0, (amax.size, 127))
    xs = synth.to_bf16_bits((frac * af[:, None]).astype(np.float32))
    xs_f = f32_of_bits(xs)
    xs = np.where(np.abs(xs_f) <= af[:, None], xs, np.uint16(0))      # keep amax the group maximum
    groups = np.concatenate([amax[:, None], xs], axis=1)
    pad = (-groups.shape[0]) % 8
    groups = np.concatenate([groups, np.zeros((pad, 128), np.uint16)])
    xb = groups.reshape(-1, 1024)
    xq, xsc = r9q.r9q_quant_group128(bf16_to_dev(xb))
    torch.cuda.synchronize()
    oq, os_ = oracle.quant_group(xb)
    assert np.array_equal(xsc.cpu().numpy(), os_)
    assert np.array_equal(xq.cpu().numpy(), oq)


def test_weight_block_quant_bit_exact(r9q):
    quantised_weights(r9q, 0, 512, 1024)
    quantised_weights(r9q, 1, 4096, 4096)
    # a block of zeros gives scale 0 and codes 0
    w = np.zeros((256, 256), np.float32)
    w[128:, :128] = synth.weights(9, 128, 128)
    wq, ws = r9q.r9q_quant_weight_block128(torch.from_numpy(w).to(dev()))
    oq, os_ = oracle.quant_block128(w)
    assert np.array_equal(wq.cpu().numpy(), oq) and np.array_equal(ws.cpu().numpy(), os_)


# ---------------------------------------------------------------- W8A8 --

def _w8a8_case(r9q, M, N, K, p, factor, seed, rows=None):
    xb = activations_bf16(seed, M, K, p, factor)
    wq, ws = quantised_weights(r9q, seed, N, K)
    x = bf16_to_dev(xb)
    aq = torch.empty((M, K), dtype=torch.uint8, device=dev())
    a_s = torch.empty((M, K // 128), dtype=torch.float32, device=dev())
    y = r9q.r9q_gemm_fp8_block_qa(x, wq, ws, aq=aq, as_=a_s)
    # unfused: separate quant pass, then the GEMM on (aq, as)
    uq, us = r9q.r9q_quant_group128(x)
    yu = r9q.r9q_gemm_fp8_block_qa(None, wq, ws, aq=uq, as_=us)
    torch.cuda.synchronize()
    oq, os_ = oracle.quant_group(xb)
    assert np.array_equal(aq.cpu().numpy(), oq), "fused A-load quant codes != oracle"
    assert np.array_equal(a_s.cpu().numpy(), os_), "fused A-load quant scales != oracle"
    assert torch.equal(aq, uq) and torch.equal(a_s, us), "fused and unfused quant operands differ"
    assert torch.equal(y.view(torch.int16), yu.view(torch.int16)), "fused and unfused outputs differ"
    acc, _ = oracle.gemm_w8a8(oq, os_, wq.cpu().numpy(), ws.cpu().numpy(), rows=rows)
    yb = bits_of(y)
    if rows is not None:
        yb = yb[rows]
    return assert_close(yb, acc, f"W8A8 M={M} N={N} K={K}")


def test_w8a8_c0(r9q):
    _w8a8_case(r9q, 1, 512, 1024, 0.01, 20.0, 0)


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_w8a8_c2(r9q, M):
    _w8a8_case(r9q, M, 12288, 4096, 0.005, 50.0, 2)


@pytest.mark.parametrize("M", [32, 64, 128, 255])
def test_w8a8_c4(r9q, M):
    _w8a8_case(r9q, M, 4096, 4096, 0.0, 1.0, 4)


def test_w8a8_c4_prefill_sampled(r9q):
    """M = 8192: the full aq/as against the oracle, and the output on one row of
    every 128-row m-tile (each m-tile is a different (CTA, persistent
    iteration) of the tensor-core kernel), the row's position in the tile
    rotating over the four 32-lane quarters of the TMEM accumulator, plus the
    first and last rows."""
    t = np.arange(8192 // 128)
    rows = 128 * t + 32 * (t % 4) + (t * 7) % 32
    rows = np.unique(np.concatenate([rows, [0, 1, 127, 128, 8190, 8191]]))
    _w8a8_case(r9q, 8192, 4096, 4096, 0.0, 1.0, 4, rows=rows)


@pytest.mark.parametrize("M,N,K", [(3, 256, 384), (5, 384, 640), (4, 256, 2048), (13, 128, 128), (17, 640, 256),
                                   (33, 256, 1152), (63, 384, 512), (65, 256, 512), (100, 128, 384),
                                   (130, 384, 5120),     # tensor-core path (split-K), two scale buffers
                                   (200, 256, 8192),     # ... one scale buffer
                                   (1000, 5120, 256)])   # persistent whole-K tiles: 160 tiles, a partial m-tile
def test_w8a8_ragged(r9q, M, N, K):
    _w8a8_case(r9q, M, N, K, 0.01, 20.0, 11)


# --------------------------------------------------------- weight-only --

def _w8bf16_case(r9q, M, N, K, seed):
    xb = activations_bf16(seed, M, K)
    wq, ws = quantised_weights(r9q, seed, N, K)
    y = r9q.r9q_gemm_fp8w_bf16a(bf16_to_dev(xb), wq, ws)
    torch.cuda.synchronize()
    acc, _ = oracle.gemm_w8bf16(xb, wq.cpu().numpy(), ws.cpu().numpy())
    return assert_close(bits_of(y), acc, f"weight-only M={M} N={N} K={K}")


def test_w8bf16_c1(r9q):
    _w8bf16_case(r9q, 16, 4096, 4096, 1)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (3, 256, 384), (9, 384, 1280), (31, 256, 256),
                                   (64, 128, 640), (70, 256, 256)])
def test_w8bf16_ragged(r9q, M, N, K):
    _w8bf16_case(r9q, M, N, K, 12)


def test_w8bf16_every_code_exact(r9q):
    """One-hot activations select single weight codes: y = bf16(value * ws) must
    be exact for every finite code, subnormals included (checks the in-register
    e4m3 -> bf16 conversion)."""
    K, N = 256, 256
    wq = ((np.arange(N, dtype=np.int64)[:, None] * 131 + np.arange(K)[None, :] * 7) % 256).astype(np.uint8)
    wq[(wq & 0x7F) == 0x7F] = 0x7E
    ws = np.array([[1.0, 2.0], [0.5, 0.25]], np.float32)
    ks = np.arange(0, K, 1)
    x = np.zeros((len(ks), K), np.float32)
    x[np.arange(len(ks)), ks] = 1.0
    xb = synth.to_bf16_bits(x)
    y = r9q.r9q_gemm_fp8w_bf16a(bf16_to_dev(xb), torch.from_numpy(wq).to(dev()), torch.from_numpy(ws).to(dev()))
    acc, yo = oracle.gemm_w8bf16(xb, wq, ws)
    assert np.array_equal(bits_of(y), yo)
    seen = set(np.unique(wq[:, ks]))
    assert len(seen) == 254        # all finite codes exercised


# ------------------------------------------------------ grouped (experts) --

def _grouped_case(r9q, counts, N, K, flags, seed):
    """One launch over len(counts) experts; each expert's rows against the
    oracle's GEMM on the same operands (W8A8: the oracle quantises the rows)."""
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    E, Mtot = len(counts), int(off[-1])
    xb = activations_bf16(seed, Mtot, K, 0.01, 20.0)
    wq = [quantised_weights(r9q, seed, N, K, tensor=10 + e, check_oracle=False) for e in range(E)]
    W = torch.stack([q for q, _ in wq])
    WS = torch.stack([s for _, s in wq])
    y = r9q.r9q_grouped_gemm_fp8(bf16_to_dev(xb), off.tolist(), W, WS, flags=flags)
    torch.cuda.synchronize()
    yb = bits_of(y)
    for e in range(E):
        r = slice(int(off[e]), int(off[e + 1]))
        if off[e + 1] == off[e]:
            continue
        we, se = wq[e][0].cpu().numpy(), wq[e][1].cpu().numpy()
        if flags & r9q.R9Q_GROUPED_WEIGHT_ONLY:
            acc, gu = oracle.gemm_w8bf16(xb[r], we, se)
        else:
            oq, os_ = oracle.quant_group(xb[r])
            acc, gu = oracle.gemm_w8a8(oq, os_, we, se)
        if flags & r9q.R9Q_GROUPED_SWIGLU:
            assert_close(yb[r], f32_of_bits(oracle.swiglu_interleaved(gu)), f"expert {e} h")
        else:
            assert_close(yb[r], acc, f"expert {e} y")
    if flags & r9q.R9Q_GROUPED_SWIGLU:
        # the same launch without the epilogue gives the GPU's own bf16 gate/up
        # values; h must be the oracle's SwiGLU of exactly those, bit for bit
        gu_gpu = r9q.r9q_grouped_gemm_fp8(bf16_to_dev(xb), off.tolist(), W, WS,
                                          flags=flags & ~r9q.R9Q_GROUPED_SWIGLU)
        torch.cuda.synchronize()
        assert np.array_equal(yb, oracle.swiglu_interleaved(bits_of(gu_gpu))), "h != oracle SwiGLU of the GPU's g, u"
    return y


@pytest.mark.parametrize("flags", [0, 1])           # W8A8 with fused quant; weight-only
@pytest.mark.parametrize("counts", [[3, 0, 1, 16, 5], [70, 3], [0, 0, 2]])
def test_grouped_gemm(r9q, flags, counts):
    _grouped_case(r9q, counts, 384, 512, flags, 21)


@pytest.mark.parametrize("flags", [2, 3])           # SwiGLU epilogue: W8A8; weight-only
def test_grouped_gemm_swiglu(r9q, flags):
    _grouped_case(r9q, [2, 7, 0, 1], 512, 384, flags, 22)


def test_grouped_gemm_many_experts(r9q):
    rng = np.random.default_rng(23)
    counts = rng.integers(0, 3, 128).tolist()
    _grouped_case(r9q, counts, 128, 256, 0, 23)


def test_grouped_gemm_no_tokens_is_noop(r9q):
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=dev())
    w = torch.zeros((2, 128, 256), dtype=torch.uint8, device=dev())
    ws = torch.ones((2, 1, 2), dtype=torch.float32, device=dev())
    y = r9q.r9q_grouped_gemm_fp8(x, [0, 0, 0], w, ws)
    assert y.shape == (0, 128)


# ----------------------------------------------------------- expert MLP --

@pytest.mark.parametrize("weight_only", [False, True])
@pytest.mark.parametrize("M,H,I,Ho", [(8, 4096, 1536, 4096), (3, 256, 384, 640), (20, 512, 256, 384),
                                      (48, 512, 256, 384)])
def test_mlp_fused_vs_unfused_and_oracle(r9q, weight_only, M, H, I, Ho):
    seed = 3
    xb = activations_bf16(seed, M, H)
    wgu, sgu = quantised_weights(r9q, seed, 2 * I, H, tensor=1)
    wdn, sdn = quantised_weights(r9q, seed, Ho, I, tensor=2)
    x = bf16_to_dev(xb)
    flags = r9q.R9Q_MLP_WEIGHT_ONLY if weight_only else 0
    outs = {}
    for unfused in (False, True):
        h = torch.empty((M, I), dtype=torch.bfloat16, device=dev())
        hq = None if weight_only else torch.empty((M, I), dtype=torch.uint8, device=dev())
        hs = None if weight_only else torch.empty((M, I // 128), dtype=torch.float32, device=dev())
        y = r9q.r9q_gate_up_swiglu_down(x, wgu, sgu, wdn, sdn, h=h, hq=hq, hs=hs,
                                        flags=flags | (r9q.R9Q_MLP_UNFUSED if unfused else 0))
        outs[unfused] = (y, h, hq, hs)
    torch.cuda.synchronize()
    (y0, h0, hq0, hs0), (y1, h1, hq1, hs1) = outs[False], outs[True]
    assert torch.equal(h0.view(torch.int16), h1.view(torch.int16)), "fused h != separate-launch h"
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16)), "fused y != separate-launch y"
    if not weight_only:
        assert torch.equal(hq0, hq1) and torch.equal(hs0, hs1), "fused hq/hs != separate-launch hq/hs"
    ref = oracle.gate_up_swiglu_down(xb, wgu.cpu().numpy(), sgu.cpu().numpy(), wdn.cpu().numpy(),
                                     sdn.cpu().numpy(), weight_only=weight_only)
    hb = bits_of(h0)
    assert_close(hb, f32_of_bits(ref["h"]), "h")
    assert_close(bits_of(y0), f32_of_bits(ref["y"]), "y")
    # The GPU's own bf16 gate/up values (the gate_up GEMM without its
    # epilogue: a one-expert grouped launch runs the MLP's stream kernel with
    # the same plan), within the GEMM bound of the oracle's accumulators ...
    gu_gpu = bits_of(r9q.r9q_grouped_gemm_fp8(x, [0, M], wgu[None], sgu[None],
                                              flags=r9q.R9Q_GROUPED_WEIGHT_ONLY if weight_only else 0))
    if weight_only:
        gacc, _ = oracle.gemm_w8bf16(xb, wgu.cpu().numpy(), sgu.cpu().numpy())
    else:
        xq, xs = oracle.quant_group(xb)
        gacc, _ = oracle.gemm_w8a8(xq, xs, wgu.cpu().numpy(), sgu.cpu().numpy())
    assert_close(gu_gpu, gacc, "gate_up")
    # ... and h is the oracle's fp32 SwiGLU of exactly those values, bit for bit
    h_ref = oracle.swiglu_interleaved(gu_gpu)
    assert np.array_equal(hb, h_ref), f"h: {int((hb != h_ref).sum())} elements differ from the oracle SwiGLU"
    if not weight_only:
        # the down GEMM's fp8 operand: the oracle's row quant of that h, bit for bit
        oq, os_ = oracle.quant_group(h_ref)
        assert np.array_equal(hq0.cpu().numpy(), oq) and np.array_equal(hs0.cpu().numpy(), os_)
        # and y against the oracle's down GEMM on those operands
        acc, _ = oracle.gemm_w8a8(oq, os_, wdn.cpu().numpy(), sdn.cpu().numpy())
        assert_close(bits_of(y0), acc, "y from the GPU's hq")
    else:
        acc, _ = oracle.gemm_w8bf16(hb, wdn.cpu().numpy(), sdn.cpu().numpy())
        assert_close(bits_of(y0), acc, "y from the GPU's h")


def test_swiglu_every_bf16_gate_bit_exact(r9q):
    """The SwiGLU pass (the library's own exp, fp32 steps) against the oracle,
    bit for bit, for every finite bf16 gate value against four up rows:
    u = 1, u = -3, random normal values and random finite bf16 patterns."""
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    g = b[np.isfinite(f32_of_bits(b))]
    I = g.size                                     # 65280 = 510 * 128
    rng = np.random.default_rng(31)
    u = np.stack([np.full(I, synth.to_bf16_bits(np.float32([1.0]))[0], np.uint16),
                  np.full(I, synth.to_bf16_bits(np.float32([-3.0]))[0], np.uint16),
                  synth.to_bf16_bits((rng.standard_normal(I) * 10).astype(np.float32)),
                  rng.permutation(g)])
    M = u.shape[0]
    gu = np.empty((M, 2 * I), np.uint16)
    v = gu.reshape(M, I // 128, 2, 128)
    v[:, :, 0, :] = g.reshape(I // 128, 128)[None]
    v[:, :, 1, :] = u.reshape(M, I // 128, 128)
    h = r9q.r9q_swiglu_interleaved(bf16_to_dev(gu))
    torch.cuda.synchronize()
    ref = oracle.swiglu_interleaved(gu)
    got = bits_of(h)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, [(hex(int(g[j])), hex(int(u[i, j])), hex(int(got[i, j])), hex(int(ref[i, j])))
                           for i, j in bad[:5]]


def test_mlp_without_optional_outputs(r9q):
    M, H, I, Ho = 8, 256, 256, 256
    xb = activations_bf16(5, M, H)
    wgu, sgu = quantised_weights(r9q, 5, 2 * I, H, tensor=1, check_oracle=False)
    wdn, sdn = quantised_weights(r9q, 5, Ho, I, tensor=2, check_oracle=False)
    x = bf16_to_dev(xb)
    h = torch.empty((M, I), dtype=torch.bfloat16, device=dev())
    y_ref = r9q.r9q_gate_up_swiglu_down(x, wgu, sgu, wdn, sdn, h=h)
    y = r9q.r9q_gate_up_swiglu_down(x, wgu, sgu, wdn, sdn)             # h in the workspace
    y_u = r9q.r9q_gate_up_swiglu_down(x, wgu, sgu, wdn, sdn, flags=r9q.R9Q_MLP_UNFUSED)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    assert torch.equal(y_u.view(torch.int16), y_ref.view(torch.int16))


# ----------------------------------------------------------- determinism --

def test_repeat_calls_bit_identical(r9q):
    M, N, K = 16, 4096, 4096
    xb = activations_bf16(2, M, K, 0.005, 50.0)
    wq, ws = quantised_weights(r9q, 2, N, K, check_oracle=False)
    x = bf16_to_dev(xb)
    first = r9q.r9q_gemm_fp8_block_qa(x, wq, ws).clone()
    first_w = r9q.r9q_gemm_fp8w_bf16a(x, wq, ws).clone()
    for _ in range(50):
        assert torch.equal(r9q.r9q_gemm_fp8_block_qa(x, wq, ws).view(torch.int16), first.view(torch.int16))
        assert torch.equal(r9q.r9q_gemm_fp8w_bf16a(x, wq, ws).view(torch.int16), first_w.view(torch.int16))
    assert r9q.r9q_last_device_error() == 0


def test_graph_replay_alternating_shapes(r9q):
    """Captured calls with different M replayed many times give the eager results."""
    N, K = 1024, 2048
    wq, ws = quantised_weights(r9q, 8, N, K, check_oracle=False)
    xs = [bf16_to_dev(activations_bf16(8, M, K, tensor=M)) for M in (1, 16, 3, 8)]
    eager = [r9q.r9q_gemm_fp8_block_qa(x, wq, ws).clone() for x in xs]
    outs = [torch.empty_like(e) for e in eager]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for x, o in zip(xs, outs):
            r9q.r9q_gemm_fp8_block_qa(x, wq, ws, y=o)
    for _ in range(300):
        g.replay()
    torch.cuda.synchronize()
    for e, o in zip(eager, outs):
        assert torch.equal(e.view(torch.int16), o.view(torch.int16))


def test_tensor_core_calls_share_one_workspace_in_a_graph(r9q):
    """W8A8 calls on the tensor-core path (split-K and persistent tiles, fused and
    unfused quant) share one zeroed workspace: each call returns the counter
    header to zero, so captured calls replayed many times match the eager ones."""
    N, K = 1024, 2048
    wq, ws = quantised_weights(r9q, 9, N, K, check_oracle=False)
    shapes = (64, 300, 2600, 40)          # split-K 8, split-K 8, persistent (84 tiles), split-K 8
    xs = [bf16_to_dev(activations_bf16(9, M, K, tensor=M)) for M in shapes]
    need = max(r9q.r9q_workspace_bytes(r9q.R9Q_OP_GEMM_W8A8, M, N, K) for M in shapes)
    wsp = torch.zeros(need, dtype=torch.uint8, device=dev())
    eager = [r9q.r9q_gemm_fp8_block_qa(x, wq, ws, workspace=wsp).clone() for x in xs]
    uq, us = r9q.r9q_quant_group128(xs[1])
    eager_unfused = r9q.r9q_gemm_fp8_block_qa(None, wq, ws, aq=uq, as_=us, workspace=wsp).clone()
    assert torch.equal(eager_unfused.view(torch.int16), eager[1].view(torch.int16))
    outs = [torch.empty_like(e) for e in eager]
    out_u = torch.empty_like(eager_unfused)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for x, o in zip(xs, outs):
            r9q.r9q_gemm_fp8_block_qa(x, wq, ws, y=o, workspace=wsp)
        r9q.r9q_gemm_fp8_block_qa(None, wq, ws, aq=uq, as_=us, y=out_u, workspace=wsp)
    for _ in range(50):
        g.replay()
    torch.cuda.synchronize()
    assert r9q.r9q_last_device_error() == 0
    for e, o in zip(eager, outs):
        assert torch.equal(e.view(torch.int16), o.view(torch.int16))
    assert torch.equal(eager_unfused.view(torch.int16), out_u.view(torch.int16))
    assert torch.count_nonzero(wsp[:64 * 1024]) == 0, "counter header not returned to zero"
    # the first shape against the oracle
    xb = activations_bf16(9, shapes[0], K, tensor=shapes[0])
    oq, os_ = oracle.quant_group(xb)
    acc, _ = oracle.gemm_w8a8(oq, os_, wq.cpu().numpy(), ws.cpu().numpy())
    assert_close(bits_of(outs[0]), acc, "W8A8 M=64 from a graph replay")


def test_device_error_word_clear(r9q):
    assert r9q.r9q_last_device_error() == 0


def test_selftest_without_waits_records_nothing(r9q):
    assert r9q.r9q_last_device_error() == 0
    r9q.r9q_selftest_wait_timeout(0)
    assert r9q.r9q_last_device_error() == 0


@pytest.mark.parametrize("which", [1, 2, 4, 8])
def test_bounded_wait_runs_out_and_context_survives(r9q, which):
    """A wait on an mbarrier / counter that nothing completes gives up within
    its bound, the host reads R9Q_ERR_TIMEOUT (once), and the next GEMM on the
    same context is correct."""
    import time
    assert r9q.r9q_last_device_error() == 0
    t0 = time.perf_counter()
    r9q.r9q_selftest_wait_timeout(which)
    assert r9q.r9q_last_device_error() == r9q.R9Q_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 30.0
    assert r9q.r9q_last_device_error() == 0
    _w8a8_case(r9q, 5, 384, 640, 0.01, 20.0, 11)
    assert r9q.r9q_last_device_error() == 0


def test_pdl_dependent_chain_matches_serialised(r9q):
    """With programmatic launch on, a GEMM whose activations are the previous
    GEMM's output must still see that output: a 6-deep chain, PDL on vs off."""
    K = 1024
    ws_list = [quantised_weights(r9q, 20 + i, K, K, check_oracle=False) for i in range(6)]
    x = bf16_to_dev(activations_bf16(21, 16, K))
    outs = {}
    for pdl in (False, True):
        prev = r9q.r9q_set_pdl(pdl)
        try:
            h = x
            for i, (wq, ws) in enumerate(ws_list):
                if i % 2:
                    h = r9q.r9q_gemm_fp8w_bf16a(h, wq, ws)
                else:
                    h = r9q.r9q_gemm_fp8_block_qa(h, wq, ws)
            torch.cuda.synchronize()
            outs[pdl] = h.clone()
        finally:
            r9q.r9q_set_pdl(prev)
    assert torch.equal(outs[False].view(torch.int16), outs[True].view(torch.int16))
    assert r9q.r9q_last_device_error() == 0


# ------------------------------------------------- decode layer, chained --

def test_decode_layer_chain_graph_pdl_vs_oracle(r9q):
    """A decode layer's GEMM sequence (QKV projection N=12288, output
    projection 4096x4096, then the fused expert MLP on the projection's
    output; attention between them is out of scope) captured in one CUDA graph
    with programmatic dependent launch on, replayed, and compared with the
    oracle end to end: every GEMM output within the output bound of the
    oracle on the same operands, the MLP's fp8 operand hq/hs bit-exact, and
    the whole replay bit-identical to the same launches serialised (PDL off,
    no graph)."""
    M, H, I = 8, 4096, 1536
    xb = activations_bf16(50, M, H, 0.01, 20.0)
    wqkv, sqkv = quantised_weights(r9q, 51, 3 * H, H, check_oracle=False)
    wo, so = quantised_weights(r9q, 52, H, H, check_oracle=False)
    wgu, sgu = quantised_weights(r9q, 53, 2 * I, H, tensor=1, check_oracle=False)
    wdn, sdn = quantised_weights(r9q, 53, H, I, tensor=2, check_oracle=False)
    x = bf16_to_dev(xb)

    def bufs():
        return {"qkv": torch.empty((M, 3 * H), dtype=torch.bfloat16, device=dev()),
                "o": torch.empty((M, H), dtype=torch.bfloat16, device=dev()),
                "h": torch.empty((M, I), dtype=torch.bfloat16, device=dev()),
                "hq": torch.empty((M, I), dtype=torch.uint8, device=dev()),
                "hs": torch.empty((M, I // 128), dtype=torch.float32, device=dev()),
                "y": torch.empty((M, H), dtype=torch.bfloat16, device=dev())}

    def layer(b):
        r9q.r9q_gemm_fp8_block_qa(x, wqkv, sqkv, y=b["qkv"])
        r9q.r9q_gemm_fp8_block_qa(x, wo, so, y=b["o"])
        r9q.r9q_gate_up_swiglu_down(b["o"], wgu, sgu, wdn, sdn, y=b["y"], h=b["h"], hq=b["hq"], hs=b["hs"])

    serial = bufs()
    prev = r9q.r9q_set_pdl(False)
    layer(serial)
    torch.cuda.synchronize()
    chained = bufs()
    s = torch.cuda.Stream()
    r9q.r9q_set_pdl(True)
    try:
        with torch.cuda.stream(s):
            layer(chained)                    # warm-up outside the capture
        torch.cuda.synchronize()
        for t in chained.values():
            t.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            layer(chained)
        g.replay()
        g.replay()
        torch.cuda.synchronize()
    finally:
        r9q.r9q_set_pdl(prev)
    for k in serial:
        a, b = serial[k], chained[k]
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"{k}: graph + PDL differs from serialised"
    # end to end against the oracle
    xq, xs = oracle.quant_group(xb)
    acc_qkv, _ = oracle.gemm_w8a8(xq, xs, wqkv.cpu().numpy(), sqkv.cpu().numpy())
    assert_close(bits_of(chained["qkv"]), acc_qkv, "qkv")
    acc_o, _ = oracle.gemm_w8a8(xq, xs, wo.cpu().numpy(), so.cpu().numpy())
    o_bits = bits_of(chained["o"])
    assert_close(o_bits, acc_o, "o")
    ref = oracle.gate_up_swiglu_down(o_bits, wgu.cpu().numpy(), sgu.cpu().numpy(), wdn.cpu().numpy(),
                                     sdn.cpu().numpy())
    assert_close(bits_of(chained["y"]), f32_of_bits(ref["y"]), "y")
    h_ref = oracle.swiglu_interleaved(bits_of(r9q.r9q_grouped_gemm_fp8(chained["o"], [0, M], wgu[None], sgu[None])))
    assert np.array_equal(bits_of(chained["h"]), h_ref), "h != oracle SwiGLU of the GPU's g, u"
    oq, os_ = oracle.quant_group(h_ref)
    assert np.array_equal(chained["hq"].cpu().numpy(), oq) and np.array_equal(chained["hs"].cpu().numpy(), os_)
    assert r9q.r9q_last_device_error() == 0
