"""Pins for the CPU oracle, against things other than the oracle itself.

Each test ties one part of the oracle to a fact the pages or plain mathematics
fix: library routines for the special cases that reduce to them (numpy's
float16 conversion, numpy's little-endian unpackbits plus a dense fp64 matmul),
closed forms (all bits set, all bits clear, one bit set), invariants (a whole
row flipped negates that output exactly; the XOR patch is its own inverse),
the footprint figures printed on the pages, and brute force over every 16-bit
pattern.  A plausible slip in the oracle (bit order, sign polarity, scale
index, a dropped group, a double rounding) fails at least one of them.
"""
import json
import os

import numpy as np
import pytest
import torch

from bit_weight_gemv_sign_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")


# ---------------------------------------------------------------- decoding

def test_half_decode_all_patterns(orc):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)        # library conversion
    got = np.array([orc.half_to_double(int(p)) for p in pats])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    assert np.array_equal(np.signbit(got[~np.isnan(got)]), np.signbit(ref[~np.isnan(ref)]))


def test_bf16_decode_all_patterns(orc):
    pats = np.arange(65536, dtype=np.int64).astype(np.uint16)
    ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([orc.bf16_to_double(int(p)) for p in pats])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


# ---------------------------------------------------------------- rounding

def _edge_doubles(rng, n):
    mags = np.exp2(rng.uniform(-30, 20, size=n))
    sgn = np.where(rng.integers(0, 2, size=n) == 1, 1.0, -1.0)
    return mags * sgn


def test_double_to_half_matches_numpy(orc):
    rng = np.random.default_rng(1)
    vals = list(_edge_doubles(rng, 4000))
    # exact ties between neighbouring fp16 values (normal and subnormal),
    # the overflow boundary and signed zeros
    grid = np.arange(0, 0x7c00, 97, dtype=np.uint16).view(np.float16).astype(np.float64)
    vals += list((grid[:-1] + grid[1:]) / 2)
    sub = np.arange(0, 1024, dtype=np.uint16).view(np.float16).astype(np.float64)
    vals += list((sub[:-1] + sub[1:]) / 2)
    vals += [65504.0, 65519.99, 65520.0, 70000.0, 0.0, -0.0, 2.0 ** -25, 2.0 ** -26, -2.0 ** -25 * 3]
    vals = np.array(vals, dtype=np.float64)
    ref = vals.astype(np.float16).view(np.uint16)          # numpy: direct RNE
    got = np.array([orc.double_to_half(v) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def _bf16_grid():
    """Every finite non-negative bf16 value, plus IEEE's virtual next grid
    point 2^128 standing for +inf (pattern 0x7f80, even), so that overflow
    follows the same nearest/ties-to-even rule."""
    pats = np.arange(0, 0x7f80, dtype=np.int64)  # +0 .. max finite
    vals = torch.from_numpy(pats.astype(np.uint16).view(np.int16)).view(torch.bfloat16)
    vals = vals.to(torch.float64).numpy()
    return np.append(pats, 0x7f80), np.append(vals, 2.0 ** 128)


def test_double_to_bf16_is_nearest_even(orc):
    pats, grid = _bf16_grid()
    rng = np.random.default_rng(2)
    vals = list(np.abs(_edge_doubles(rng, 3000)))
    vals += list((grid[:-2:37] + grid[1:-1:37]) / 2)         # exact ties
    vals += [0.0, 2.0 ** -140, 1e-45, 3.0e38, 3.4e38, 2.0 ** 128 - 2.0 ** 119,
             2.0 ** 128 - 2.0 ** 119 - 2.0 ** 90]
    for v in vals:
        got = orc.double_to_bf16(v)
        i = np.searchsorted(grid, v)
        cands = [j for j in (i - 1, i) if 0 <= j < len(grid)]
        dist = [abs(grid[j] - v) for j in cands]
        best = min(dist)
        near = [cands[t] for t in range(len(cands)) if dist[t] == best]
        if len(near) > 1:
            near = [j for j in near if pats[j] % 2 == 0]
        exp = int(pats[near[0]])
        assert got == exp, (v, hex(got), hex(exp))
        neg = orc.double_to_bf16(-v)
        assert neg == (exp | 0x8000)


# ---------------------------------------------------------------- GEMV

def _dense(bits, scales, x, N, K):
    """Independent route: numpy's little-endian unpackbits, dequantise to a
    dense fp64 matrix, then a library matmul."""
    b = np.unpackbits(bits.reshape(N, K // 8), axis=1, bitorder="little")
    sgn = np.where(b == 1, 1.0, -1.0)
    s = scales.reshape(N, K // 128).view(np.float16).astype(np.float64)
    W = sgn * np.repeat(s, 128, axis=1)
    X = torch.from_numpy(x.reshape(-1, K).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    return X @ W.T, W, X


def _bound(W, X):
    return np.abs(X) @ np.abs(W).T


@pytest.mark.parametrize("N,K,B", [(1, 128, 1), (3, 128, 2), (5, 256, 3), (8, 256, 1), (7, 384, 2)])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gemv_brute_force_matches_dense(orc, N, K, B, seed):
    g = synth.rng(100 + seed)
    bits = synth.sign_bits(N, K, g)
    scales = synth.group_scales(N, K, g, offset=1e-3)
    x = synth.activations(B, K, g)
    y = orc.gemv(bits, scales, x, B, N, K)
    ref, W, X = _dense(bits, scales, x, N, K)
    tol = 1e-12 * _bound(W, X) + 1e-300
    assert np.all(np.abs(y - ref) <= tol)
    # third route: torch fp64 matmul on the same dense matrix
    ref2 = (torch.from_numpy(X) @ torch.from_numpy(W).T).numpy()
    assert np.all(np.abs(y - ref2) <= tol)


def test_gemv_scales_are_per_row_and_group(orc):
    """Distinct scale per (row, group): a transposed or shifted scale index
    changes the result."""
    N, K, B = 3, 384, 1
    bits = np.full((N, K // 8), 0xFF, dtype=np.uint8)
    svals = np.array([[1, 2, 4], [8, 16, 32], [64, 128, 256]], dtype=np.float16)
    x = synth.to_bf16_bits(np.concatenate([np.full(128, 1.0), np.full(128, 3.0),
                                           np.full(128, 5.0)]).astype(np.float32)[None])
    y = orc.gemv(bits, svals.view(np.uint16), x, B, N, K)
    want = np.array([[128 * (1 * 1 + 2 * 3 + 4 * 5), 128 * (8 + 16 * 3 + 32 * 5),
                      128 * (64 + 128 * 3 + 256 * 5)]], dtype=np.float64)
    assert np.array_equal(y, want)


def test_closed_form_all_bits_set_and_clear(orc):
    N, K, B = 6, 512, 2
    g = synth.rng(7)
    scales = synth.group_scales(N, K, g)
    x = synth.activations(B, K, g)
    ones = np.full((N, K // 8), 0xFF, dtype=np.uint8)
    zeros = np.zeros((N, K // 8), dtype=np.uint8)
    y1 = orc.gemv(ones, scales, x, B, N, K)
    y0 = orc.gemv(zeros, scales, x, B, N, K)
    s = scales.view(np.float16).astype(np.float64)
    X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    gs = X.reshape(B, K // 128, 128).sum(axis=2)            # sum_k x_k per group
    closed = gs @ s.T                                        # sum_g s_g * sum_k x_k
    bound = np.abs(X).reshape(B, K // 128, 128).sum(axis=2) @ s.T
    assert np.all(np.abs(y1 - closed) <= 1e-12 * bound)
    assert np.array_equal(y0, -y1)                           # exact negation


def test_closed_form_single_bit(orc):
    N, K, B = 1, 256, 1
    g = synth.rng(8)
    scales = synth.group_scales(N, K, g, offset=1e-3)
    x = synth.activations(B, K, g)
    s = scales.view(np.float16).astype(np.float64)[0]
    X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()[0]
    base = -(s[0] * X[:128].sum() + s[1] * X[128:].sum())
    for k in (0, 1, 7, 8, 127, 128, 200, 255):
        bits = np.zeros((1, K // 8), dtype=np.uint8)
        bits[0, k // 8] = 1 << (k % 8)
        y = orc.gemv(bits, scales, x, B, N, K)[0, 0]
        want = base + 2 * s[k // 128] * X[k]
        assert abs(y - want) <= 1e-12 * (np.abs(X[:128]).sum() * s[0] + np.abs(X[128:]).sum() * s[1])


def test_row_flip_negates_exactly(orc):
    N, K, B = 9, 1024, 2
    bits, scales = synth.matrix(N, K, 11)
    x = synth.x_for(B, K, 11)
    y = orc.gemv(bits, scales, x, B, N, K)
    for r in (0, 4, 8):
        fl = bits.copy()
        fl[r] ^= 0xFF
        yf = orc.gemv(fl, scales, x, B, N, K)
        assert np.array_equal(yf[:, r], -y[:, r])
        others = [i for i in range(N) if i != r]
        assert np.array_equal(yf[:, others], y[:, others])


def test_gemv_select_and_threads_agree(orc):
    N, K, B = 37, 1024, 2
    bits, scales = synth.matrix(N, K, 12)
    x = synth.x_for(B, K, 12)
    y = orc.gemv(bits, scales, x, B, N, K)
    rows = [0, 5, 36, 5]
    ys = orc.gemv_select(bits, scales, x, B, N, K, rows)
    assert np.array_equal(ys, y[:, rows])
    yt = orc.gemv_threads(bits, scales, x, B, N, K, 4)
    assert np.array_equal(yt, y)


# ---------------------------------------------------------------- SwiGLU pair

def _silu_np(g):
    """silu(g) = g * sigmoid(g), the sigmoid from scipy's expit (a library
    routine, not the oracle's g / (1 + exp(-g)))."""
    from scipy.special import expit
    return g * expit(g)


@pytest.mark.parametrize("N2,K,B,seed", [(2, 128, 1, 0), (6, 256, 2, 1), (10, 384, 3, 2)])
def test_swiglu_matches_dense_and_library_silu(orc, N2, K, B, seed):
    """Gate rows 2n, up rows 2n+1: dense fp64 matmul, then the library
    sigmoid.  Tolerance: the GEMV rounding (1e-12 of sum |s x|) carried
    through h = silu(g) u with |silu'| <= 1.1, plus the product's rounding."""
    g = synth.rng(300 + seed)
    bits = synth.sign_bits(N2, K, g)
    scales = synth.group_scales(N2, K, g, offset=1e-3)
    x = synth.activations(B, K, g)
    h = orc.gemv_swiglu(bits, scales, x, B, N2, K)
    y, W, X = _dense(bits, scales, x, N2, K)
    bd = _bound(W, X)
    gate, up = y[:, 0::2], y[:, 1::2]
    want = _silu_np(gate) * up
    tol = 1e-12 * (1.1 * bd[:, 0::2] * np.abs(up) + np.abs(gate) * bd[:, 1::2]) + 1e-14 * np.abs(want) + 1e-300
    assert h.shape == (B, N2 // 2)
    assert np.all(np.abs(h - want) <= tol)
    # the pair is not symmetric: gate and up swapped gives another result
    assert not np.allclose(h, _silu_np(up) * gate, rtol=1e-6, atol=0)


def test_swiglu_zero_gate_or_zero_up_gives_zero(orc):
    """silu(0) = 0 and u = 0 each force h = 0 exactly; the other outputs are
    untouched by zeroing one pair's scales."""
    N2, K, B = 8, 256, 2
    bits, scales = synth.matrix(N2, K, 31, scale_offset=1e-3)
    x = synth.x_for(B, K, 31)
    h = orc.gemv_swiglu(bits, scales, x, B, N2, K)
    s0 = scales.reshape(N2, K // 128).copy()
    s0[2] = 0          # gate of output 1
    s0[7] = 0          # up of output 3
    hz = orc.gemv_swiglu(bits, s0, x, B, N2, K)
    assert np.all(hz[:, [1, 3]] == 0.0)
    assert np.array_equal(hz[:, [0, 2]], h[:, [0, 2]])


def test_swiglu_closed_form_saturation(orc):
    """All bits set and one scale value per row: g = s_g * sum x and
    u = s_u * sum x in closed form; a large positive gate passes through
    (silu(g) = g up to e^-g), a large negative one closes (h ~ g e^g u)."""
    N2, K, B = 4, 128, 1
    bits = np.full((N2, K // 8), 0xFF, dtype=np.uint8)
    x = synth.to_bf16_bits(np.full((B, K), 0.25))      # sum x = 32 exactly
    sv = np.array([1.25, 0.5, -1.25, 0.5], dtype=np.float16)   # g = +-40, u = 16
    scales = sv.view(np.uint16).reshape(N2, 1)
    h = orc.gemv_swiglu(bits, scales, x, B, N2, K)
    assert abs(h[0, 0] - 40.0 * 16.0) <= 640.0 * 1e-15 + 640.0 * np.exp(-40.0)
    want_neg = -40.0 * np.exp(-40.0) / (1.0 + np.exp(-40.0)) * 16.0
    assert abs(h[0, 1] - want_neg) <= 1e-12 * abs(want_neg)


def test_swiglu_select_matches_full(orc):
    N2, K, B = 14, 384, 2
    bits, scales = synth.matrix(N2, K, 33, scale_offset=1e-3)
    x = synth.x_for(B, K, 33)
    h = orc.gemv_swiglu(bits, scales, x, B, N2, K)
    units = [6, 0, 3, 3]
    hs = orc.gemv_swiglu_select(bits, scales, x, B, N2, K, units)
    assert np.array_equal(hs, h[:, units])
    with pytest.raises(orc.OracleError) as e:
        orc.gemv_swiglu_select(bits, scales, x, B, N2, K, [7])
    assert e.value.status == orc.ERANGE


def test_swiglu_rejects_odd_row_count(orc):
    bits = np.zeros((3, 16), dtype=np.uint8)
    scales = np.zeros((3, 1), dtype=np.uint16)
    x = np.zeros((1, 128), dtype=np.uint16)
    with pytest.raises(orc.OracleError) as e:
        orc.gemv_swiglu(bits, scales, x, 1, 3, 128)
    assert e.value.status == orc.ESHAPE


def test_gemv_rejects_bad_shapes(orc):
    bits = np.zeros((2, 24), dtype=np.uint8)
    scales = np.zeros((2, 2), dtype=np.uint16)
    x = np.zeros((1, 192), dtype=np.uint16)
    with pytest.raises(orc.OracleError) as e:
        orc.gemv(bits, scales, x, 1, 2, 192)
    assert e.value.status == orc.ESHAPE


# ---------------------------------------------------------------- XOR patch

def test_xor_patch_flips_listed_rows_only(orc):
    N, K = 16, 1024
    bits, _ = synth.matrix(N, K, 13)
    rows = [3, 9, 15]
    p = orc.xor_patch(bits, N, K, rows)
    ub = np.unpackbits(bits, axis=1, bitorder="little")
    up = np.unpackbits(p, axis=1, bitorder="little")
    for r in range(N):
        if r in rows:
            assert np.array_equal(up[r], 1 - ub[r])           # every bit complemented
        else:
            assert np.array_equal(up[r], ub[r])


def test_xor_patch_is_self_inverse_and_duplicates_cancel(orc):
    N, K = 32, 512
    bits, _ = synth.matrix(N, K, 14)
    rows = synth.distinct_rows(N, 8, 0)
    once = orc.xor_patch(bits, N, K, rows)
    twice = orc.xor_patch(once, N, K, rows)
    assert np.array_equal(twice, bits)
    assert not np.array_equal(once, bits)
    dup = orc.xor_patch(bits, N, K, [5, 5, 7])
    assert np.array_equal(dup, orc.xor_patch(bits, N, K, [7]))


def test_xor_patch_range_checked_before_any_change(orc):
    N, K = 8, 256
    bits, _ = synth.matrix(N, K, 15)
    for bad in ([1, 8], [-1], [0, 2, 100]):
        assert orc.xor_patch_status(bits, N, K, bad) == orc.ERANGE
    with pytest.raises(orc.OracleError):
        orc.xor_patch(bits, N, K, [8])


def test_xor_patch_negates_gemv_rows(orc):
    N, K, B = 12, 1024, 1
    bits, scales = synth.matrix(N, K, 16)
    x = synth.x_for(B, K, 16)
    rows = [2, 7]
    y = orc.gemv(bits, scales, x, B, N, K)
    yp = orc.gemv(orc.xor_patch(bits, N, K, rows), scales, x, B, N, K)
    assert np.array_equal(yp[:, rows], -y[:, rows])
    keep = [i for i in range(N) if i not in rows]
    assert np.array_equal(yp[:, keep], y[:, keep])


# ---------------------------------------------------------------- packing

def test_pack_round_trip(orc):
    """Dequantise (bits, s) with s > 0, pack again: identical bits and scales
    (the mean of 128 equal magnitudes is exact)."""
    N, K = 6, 512
    bits, scales = synth.matrix(N, K, 17, scale_offset=1e-3)
    _, W, _ = _dense(bits, scales, np.zeros((1, K), dtype=np.uint16), N, K)
    for dtype, arr in ((orc.F32, W.astype(np.float32)),
                       (orc.F16, W.astype(np.float16).view(np.uint16)),
                       (orc.BF16, None)):
        if dtype == orc.BF16:
            continue  # fp16 scales are not all exactly representable in bf16
        st, b2, s2 = orc.pack(arr, dtype, N, K)
        assert st == orc.OK
        assert np.array_equal(b2, bits)
        assert np.array_equal(s2, scales)


def test_pack_bits_are_sign_test_little_endian(orc):
    N, K = 4, 256
    w = synth.fp_weights(N, K, 18)
    w[0, :5] = [0.0, -0.0, 1e-30, -1e-30, 3.0]
    st, b, _ = orc.pack(w, orc.F32, N, K)
    assert st == orc.OK
    want = np.packbits(~(w < 0), axis=1, bitorder="little")   # library packing
    assert np.array_equal(b, want)
    assert np.unpackbits(b[:1, :1], bitorder="little")[:5].tolist() == [1, 1, 1, 0, 1]


def test_pack_scale_is_fp16_of_mean_abs(orc):
    N, K = 5, 384
    w = synth.fp_weights(N, K, 19)
    st, _, s = orc.pack(w, orc.F32, N, K)
    assert st == orc.OK
    mean = np.abs(w.astype(np.float64)).reshape(N, K // 128, 128).mean(axis=2)
    assert np.array_equal(s, mean.astype(np.float16).view(np.uint16))
    # all-equal magnitudes: the scale is that magnitude exactly
    w2 = np.full((1, 128), -0.375, dtype=np.float32)
    st, b2, s2 = orc.pack(w2, orc.F32, 1, 128)
    assert st == orc.OK and s2[0, 0] == np.float16(0.375).view(np.uint16) and not b2.any()


def test_pack_scale_minimises_squared_error(orc):
    """mean|w| minimises sum (w - s*sign(w))^2 over s (least squares); no
    perturbation of the unrounded mean does better."""
    w = synth.fp_weights(1, 128, 20).astype(np.float64)[0]
    sg = np.where(w < 0, -1.0, 1.0)
    m = np.abs(w).sum() / 128
    err = lambda s: ((w - s * sg) ** 2).sum()
    for d in (1e-2, 1e-4, 1e-6):
        assert err(m) <= err(m * (1 + d)) and err(m) <= err(m * (1 - d))


def test_pack_flags_nan_and_overflow(orc):
    w = synth.fp_weights(2, 128, 21)
    w[1, 3] = np.nan
    st, _, _ = orc.pack(w, orc.F32, 2, 128)
    assert st == orc.ENAN
    w = np.full((1, 128), 70000.0, dtype=np.float32)
    st, _, _ = orc.pack(w, orc.F32, 1, 128)
    assert st == orc.ERANGE
    w = np.full((1, 128), 65504.0, dtype=np.float32)
    st, _, s = orc.pack(w, orc.F32, 1, 128)
    assert st == orc.OK and s[0, 0] == 0x7bff


def test_pack_accepts_bf16_and_fp16_inputs(orc):
    N, K = 3, 256
    w32 = synth.fp_weights(N, K, 22)
    wb = synth.to_bf16_bits(w32)
    wh = w32.astype(np.float16)
    st, bb, sb = orc.pack(wb, orc.BF16, N, K)
    assert st == orc.OK
    wb64 = torch.from_numpy(wb.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(sb, np.abs(wb64).reshape(N, 2, 128).mean(axis=2).astype(np.float16).view(np.uint16))
    assert np.array_equal(bb, np.packbits(~(wb64 < 0), axis=1, bitorder="little"))
    st, bh, sh = orc.pack(wh.view(np.uint16), orc.F16, N, K)
    assert st == orc.OK
    assert np.array_equal(bh, np.packbits(~(wh < 0), axis=1, bitorder="little"))


# ---------------------------------------------------------------- footprint

def test_footprint_is_1_125_bits_per_weight(orc):
    fig = json.load(open(GOLDEN))
    beff = fig["b_eff_binary_bits_per_weight"]["value"]
    for N, K in ((1, 128), (256, 1024), (12288, 4096), (4096, 12288), (17408, 5120)):
        assert orc.footprint_bytes(N, K) * 8 == beff * N * K
        assert orc.footprint_bytes(N, K) == N * K // 8 + 2 * N * (K // 128)
    assert round(16 / beff, fig["compression_binary_vs_fp16"]["printed_digits"]) == \
        fig["compression_binary_vs_fp16"]["value"]
    hn = fig["hn_group_framing"]
    assert 1 + hn["scale_bits"] / hn["group_size"] == hn["bits_per_weight"]


def test_footprint_8b_class_matches_printed_size(orc):
    """The 8B-class decoder shapes plus the embedding (151936 x 4096, also
    1-bit) give about 8.2 B parameters in about 1.15 GB."""
    fig = json.load(open(GOLDEN))
    mats = synth.sweep_8b()
    params = sum(m.N * m.K for m in mats) + 151936 * 4096
    nbytes = sum(orc.footprint_bytes(m.N, m.K) for m in mats) + orc.footprint_bytes(151936, 4096)
    assert round(params / 1e9, 1) == fig["bonsai_8b_parameters"]["value"] / 1e9
    assert round(nbytes / 1e9, 2) == fig["bonsai_8b_gigabytes"]["value"]
    assert nbytes == 1_151_778_816
    swept = sum(orc.footprint_bytes(m.N, m.K) for m in mats)
    assert swept == 1_064_263_680


def test_footprint_27b_matches_printed_size(orc):
    fig = json.load(open(GOLDEN))
    sp = fig["bonsai_27b_parameter_split"]
    total = sp["language_model"] + sp["vision_tower"] + sp["embedding_and_lm_head"]
    gb = total * fig["b_eff_binary_bits_per_weight"]["value"] / 8 / 1e9
    assert round(gb, 1) == fig["bonsai_27b_binary_gigabytes"]["value"]
    assert round(total * 2 / 1e9) == pytest.approx(fig["bonsai_27b_fp16_gigabytes"]["value"], abs=2)
    swept = sum(orc.footprint_bytes(m.N, m.K) for m in synth.sweep_27b())
    assert swept == 2_972_712_960


def test_patch_list_size_is_kilobyte_scale():
    """100 (layer u16, projection u8, row u32) entries are 700 bytes of
    payload: the same order as the 840 B - 1.1 KB patches on the page."""
    fig = json.load(open(GOLDEN))["bankai_patch_bytes"]
    entries = synth.patch_entries_27b(100, 0)
    assert len(set(entries)) == 100
    payload = len(entries) * (2 + 1 + 4)
    assert fig["min"] / 2 <= payload <= fig["max"]


# ---------------------------------------------------------------- ternary

def _np_planes(t):
    """Independent encoding route: numpy's little-endian packbits of the two
    threshold masks a = (t >= 0), b = (t > 0)."""
    a = np.packbits((t >= 0).astype(np.uint8), axis=1, bitorder="little")
    b = np.packbits((t > 0).astype(np.uint8), axis=1, bitorder="little")
    return a, b


def _dense_ternary(t, scales, x, N, K):
    s = scales.reshape(N, K // 128).view(np.float16).astype(np.float64)
    W = t.astype(np.float64) * np.repeat(s, 128, axis=1)
    X = torch.from_numpy(x.reshape(-1, K).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    return X @ W.T, W, X


def test_ternary_planes_match_numpy(orc):
    N, K = 6, 384
    t = synth.ternary_codes(N, K, synth.rng(700))
    a, b = orc.ternary_planes(t, N, K)
    na, nb = _np_planes(t)
    assert np.array_equal(a, na) and np.array_equal(b, nb)
    # decoding the planes with numpy gives the codes back
    ua = np.unpackbits(a, axis=1, bitorder="little").astype(np.int64) * 2 - 1
    ub = np.unpackbits(b, axis=1, bitorder="little").astype(np.int64) * 2 - 1
    assert np.array_equal((ua + ub) // 2, t.astype(np.int64))


@pytest.mark.parametrize("bad", [2, -2, 127, -128])
def test_ternary_planes_reject_other_codes(orc, bad):
    import oracle
    N, K = 2, 128
    t = np.zeros((N, K), dtype=np.int8)
    t[1, 77] = bad
    with pytest.raises(oracle.OracleError) as e:
        orc.ternary_planes(t, N, K)
    assert e.value.status == 3


@pytest.mark.parametrize("N,K,B", [(1, 128, 1), (3, 128, 2), (5, 256, 3), (7, 384, 2)])
@pytest.mark.parametrize("seed", [0, 1])
def test_ternary_brute_force_matches_dense(orc, N, K, B, seed):
    """The product through the planes equals a dense fp64 matmul of the codes
    times the group scales (the ternary weight definition), with planes made
    by numpy, not by the oracle."""
    g = synth.rng(710 + seed)
    t = synth.ternary_codes(N, K, g)
    scales = synth.group_scales(N, K, g, offset=1e-3)
    x = synth.activations(B, K, g)
    a, b = _np_planes(t)
    y = orc.gemv_ternary(a, b, scales, x, B, N, K)
    ref, W, X = _dense_ternary(t, scales, x, N, K)
    tol = 1e-12 * (np.abs(X) @ np.abs(W).T) + 1e-300
    assert np.all(np.abs(y - ref) <= tol)


def test_ternary_without_zeros_is_the_binary_product(orc):
    """a == b means every code is +-1: the ternary layer is then the binary
    layer with those bits (same summation order, so bit-identical)."""
    N, K, B = 9, 512, 3
    bits, scales = synth.matrix(N, K, 720)
    x = synth.x_for(B, K, 720)
    assert np.array_equal(orc.gemv_ternary(bits, bits, scales, x, B, N, K),
                          orc.gemv(bits, scales, x, B, N, K))


def test_ternary_all_zero_codes_give_exact_zero(orc):
    N, K, B = 4, 256, 2
    a, _, scales = synth.ternary_matrix(N, K, 721)
    x = synth.x_for(B, K, 721)
    y = orc.gemv_ternary(a, ~a, scales, x, B, N, K)
    assert np.all(y == 0.0)


def test_ternary_single_code_closed_form(orc):
    """One +1 and one -1 in an otherwise zero row: y = s_g1 x_k1 - s_g2 x_k2."""
    N, K = 2, 384
    t = np.zeros((N, K), dtype=np.int8)
    t[1, 5] = 1
    t[1, 300] = -1
    scales = np.array([0x3C00, 0x3C00, 0x3C00, 0x4000, 0x3800, 0x4400], dtype=np.uint16)  # 1,1,1 / 2,0.5,4
    x = synth.activations(1, K, synth.rng(722))
    xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy().reshape(K)
    a, b = _np_planes(t)
    y = orc.gemv_ternary(a, b, scales, x, 1, N, K)
    assert y[0, 0] == 0.0
    assert y[0, 1] == 2.0 * xv[5] - 4.0 * xv[300]


def test_ternary_flipping_both_planes_negates_exactly(orc):
    """XOR of a row in both planes maps +1 <-> -1 and keeps 0 (1,0 <-> 0,1):
    that output row is negated exactly, the others are unchanged."""
    N, K, B = 6, 256, 2
    a, b, scales = synth.ternary_matrix(N, K, 723)
    x = synth.x_for(B, K, 723)
    y0 = orc.gemv_ternary(a, b, scales, x, B, N, K)
    rows = [1, 4]
    a1, b1 = orc.xor_patch(a, N, K, rows), orc.xor_patch(b, N, K, rows)
    y1 = orc.gemv_ternary(a1, b1, scales, x, B, N, K)
    for n in range(N):
        assert np.array_equal(y1[:, n], -y0[:, n] if n in rows else y0[:, n])


def test_ternary_select_matches_full(orc):
    N, K, B = 10, 256, 3
    a, b, scales = synth.ternary_matrix(N, K, 724)
    x = synth.x_for(B, K, 724)
    full = orc.gemv_ternary(a, b, scales, x, B, N, K)
    rows = [9, 0, 3, 3]
    assert np.array_equal(orc.gemv_ternary_select(a, b, scales, x, B, N, K, rows), full[:, rows])


@pytest.mark.parametrize("N2,K,B,seed", [(2, 128, 1, 0), (8, 256, 2, 1), (12, 384, 3, 2)])
def test_ternary_swiglu_matches_dense_and_library_silu(orc, N2, K, B, seed):
    """Ternary gate/up pairs: a dense fp64 matmul of the codes (planes built by
    numpy), then scipy's sigmoid; the tolerance as for the binary pair."""
    g = synth.rng(500 + seed)
    t = synth.ternary_codes(N2, K, g)
    scales = synth.group_scales(N2, K, g, offset=1e-3)
    x = synth.activations(B, K, g)
    a, b = _np_planes(t)
    h = orc.gemv_ternary_swiglu(a, b, scales, x, B, N2, K)
    y, W, X = _dense_ternary(t, scales, x, N2, K)
    bd = _bound(W, X)
    gate, up = y[:, 0::2], y[:, 1::2]
    want = _silu_np(gate) * up
    tol = 1e-12 * (1.1 * bd[:, 0::2] * np.abs(up) + np.abs(gate) * bd[:, 1::2]) + 1e-14 * np.abs(want) + 1e-300
    assert np.all(np.abs(h - want) <= tol)


def test_ternary_swiglu_without_zeros_is_the_binary_pair(orc):
    """Planes a = b (no zero codes) are the binary matrix: the ternary pair
    equals the binary pair bit for bit; zero codes in a gate or an up row
    give exactly 0."""
    N2, K, B = 10, 256, 2
    bits, scales = synth.matrix(N2, K, 41, scale_offset=1e-3)
    x = synth.x_for(B, K, 41)
    assert np.array_equal(orc.gemv_ternary_swiglu(bits, bits, scales, x, B, N2, K),
                          orc.gemv_swiglu(bits, scales, x, B, N2, K))
    a, b = bits.copy(), bits.copy()
    b[4] = ~a[4]          # row 4 (gate of unit 2): all codes 0
    b[7] = ~a[7]          # row 7 (up of unit 3): all codes 0
    h = orc.gemv_ternary_swiglu(a, b, scales, x, B, N2, K)
    assert np.all(h[:, [2, 3]] == 0.0)


def test_ternary_rejects_bad_shapes(orc):
    import oracle
    a, b, scales = synth.ternary_matrix(2, 128, 725)
    x = synth.x_for(1, 128, 725)
    for B, N, K in [(1, 2, 100), (0, 2, 128), (1, 0, 128)]:
        with pytest.raises(oracle.OracleError):
            orc.gemv_ternary(a, b, scales, x, B, N, K)
    with pytest.raises(oracle.OracleError):
        orc.gemv_ternary_select(a, b, scales, x, 1, 2, 128, [2])


def test_ternary_footprint_and_printed_sizes(orc):
    """2-bit slots with one fp16 scale per 128 inputs are 2.125 bits/weight;
    the pages' ideal ternary cost log2(3) + 16/128 prints as 1.71 bits and
    9.4x against fp16; over the 27B parameter split it gives the printed
    5.9 GB, and the 2-bit slots give 7.37 GB, the pages' 'about 7.2 GB'."""
    fig = json.load(open(GOLDEN))
    N, K = 5120, 17408
    assert orc.ternary_footprint_bytes(N, K) * 8 == 2.125 * N * K
    assert orc.ternary_footprint_bytes(N, K) == 2 * orc.footprint_bytes(N, K) - 2 * N * (K // 128)
    ideal = np.log2(3.0) + 16.0 / 128.0
    assert round(ideal, 2) == fig["b_eff_ternary_bits_per_weight"]["value"]
    assert round(16.0 / fig["b_eff_ternary_bits_per_weight"]["value"], 1) == fig["compression_ternary_vs_fp16"]["value"]
    sp = fig["bonsai_27b_parameter_split"]
    total = sp["language_model"] + sp["vision_tower"] + sp["embedding_and_lm_head"]
    assert round(total * fig["b_eff_ternary_bits_per_weight"]["value"] / 8 / 1e9, 1) == \
        fig["bonsai_27b_ternary_gigabytes"]["value"]
    slot_bpw = orc.ternary_footprint_bytes(128, 128) * 8 / (128 * 128)
    deployed = total * slot_bpw / 8 / 1e9
    assert deployed == pytest.approx(fig["bonsai_27b_ternary_deployed_gigabytes"]["value"], rel=0.03)


# ---------------------------------------------------------------- ternary, five codes per byte

def _np_t5(t):
    """Independent packing route: numpy dot products of (t + 1) with the
    powers of three, per group: 25 five-code bytes, then one three-code byte."""
    N, K = t.shape
    d = (t.astype(np.int64) + 1).reshape(N, K // 128, 128)
    five = d[:, :, :125].reshape(N, K // 128, 25, 5) @ np.array([1, 3, 9, 27, 81])
    three = d[:, :, 125:] @ np.array([1, 3, 9])
    return np.concatenate([five, three[:, :, None]], axis=2).reshape(N, -1).astype(np.uint8)


def test_t5_pack_matches_numpy(orc):
    N, K = 5, 384
    t = synth.ternary_codes(N, K, synth.rng(900))
    p = orc.t5_pack(t, N, K)
    assert p.shape == (N, 3 * 26)
    assert np.array_equal(p, _np_t5(t))
    assert np.array_equal(orc.t5_unpack(p, N, K), t)


def test_t5_every_byte_value_decodes_to_its_base3_digits(orc):
    """Brute force over all 243 five-code bytes and all 27 three-code bytes,
    against Python's own base-3 digits."""
    N, K = 243, 128
    p = np.empty((N, 26), dtype=np.uint8)
    p[:, :25] = 121                     # five codes 0 (digit 1)
    p[:, 25] = 13                       # three codes 0
    p[:, 7] = np.arange(243)
    p[:27, 25] = np.arange(27)
    t = orc.t5_unpack(p, N, K)
    for v in range(243):
        digits = [int(c) for c in np.base_repr(v, 3).zfill(5)[::-1]]
        assert list(t[v, 35:40]) == [d - 1 for d in digits]
        assert not np.any(np.delete(t[v], list(range(35, 40)) + ([125, 126, 127] if v < 27 else [])))
    for v in range(27):
        digits = [int(c) for c in np.base_repr(v, 3).zfill(3)[::-1]]
        assert list(t[v, 125:128]) == [d - 1 for d in digits]


def test_t5_rejects_out_of_range(orc):
    import oracle
    N, K = 2, 256
    t = np.zeros((N, K), dtype=np.int8)
    t[1, 200] = 3
    with pytest.raises(oracle.OracleError):
        orc.t5_pack(t, N, K)
    p = orc.t5_pack(np.zeros((N, K), dtype=np.int8), N, K)
    x = synth.x_for(1, K, 901)
    scales = synth.group_scales(N, K, synth.rng(901))
    for pos, val in ((3, 243), (25, 27), (51, 27)):
        q = p.copy()
        q[1, pos] = val
        with pytest.raises(oracle.OracleError):
            orc.t5_unpack(q, N, K)
        with pytest.raises(oracle.OracleError):
            orc.gemv_t5(q, scales, x, 1, N, K)
    q = p.copy()
    q[1, 24] = 242                      # largest valid five-code byte
    q[1, 25] = 26                       # largest valid three-code byte
    orc.t5_unpack(q, N, K)


@pytest.mark.parametrize("N,K,B", [(1, 128, 1), (4, 256, 2), (7, 384, 3)])
def test_t5_gemv_matches_dense_and_planes(orc, N, K, B):
    g = synth.rng(910 + N)
    t = synth.ternary_codes(N, K, g)
    scales = synth.group_scales(N, K, g, offset=1e-3)
    x = synth.activations(B, K, g)
    y = orc.gemv_t5(_np_t5(t), scales, x, B, N, K)
    ref, W, X = _dense_ternary(t, scales, x, N, K)
    assert np.all(np.abs(y - ref) <= 1e-12 * (np.abs(X) @ np.abs(W).T) + 1e-300)
    a, b = _np_planes(t)
    assert np.array_equal(y, orc.gemv_ternary(a, b, scales, x, B, N, K))


def test_t5_footprint_between_ideal_and_slots(orc):
    """26 bytes per 128 codes plus the fp16 scale are 1.75 bits/weight: over
    the 27B parameter split that is 6.07 GB, between the pages' ideal 5.9 GB
    and their 2-bit-slot 'about 7.2 GB'; 8/5 bits per code is above log2(3)."""
    fig = json.load(open(GOLDEN))
    N, K = 5120, 17408
    assert orc.t5_footprint_bytes(N, K) * 8 == 1.75 * N * K
    assert 8 / 5 >= np.log2(3.0)
    sp = fig["bonsai_27b_parameter_split"]
    total = sp["language_model"] + sp["vision_tower"] + sp["embedding_and_lm_head"]
    gb = total * 1.75 / 8 / 1e9
    assert fig["bonsai_27b_ternary_gigabytes"]["value"] < gb < fig["bonsai_27b_ternary_deployed_gigabytes"]["value"]
    assert orc.t5_footprint_bytes(N, K) < orc.ternary_footprint_bytes(N, K)


# ---------------------------------------------------------------- g128x layout
# A storage format of the library (not from the pages).  What pins the
# oracle's conversion is that it is a permutation of the 128 bits of each
# group, acting on each group alone: then every bit keeps its value and a
# whole-row XOR commutes with it.  That the library's kernels read the
# permuted bits as the same inputs is checked on the GPU (a grouped product
# over converted bits equals the canonical one bit for bit).

def test_g128x_is_a_permutation_of_each_group(orc):
    K = 128
    eye = np.zeros((128, K // 8), dtype=np.uint8)
    for k in range(128):
        eye[k, k // 8] = 1 << (k % 8)
    out = orc.g128x_repack(eye, 128, K)
    ones = np.unpackbits(out, axis=1, bitorder="little")
    assert np.all(ones.sum(axis=1) == 1)                  # one bit in, one bit out
    pos = ones.argmax(axis=1)
    assert sorted(pos.tolist()) == list(range(128))       # all 128 positions used once
    assert np.array_equal(orc.g128x_unpack(out, 128, K), eye)


def test_g128x_inverse_complement_and_groupwise(orc):
    N, K = 5, 1024
    bits = synth.sign_bits(N, K, synth.rng(930))
    r = orc.g128x_repack(bits, N, K)
    assert np.array_equal(orc.g128x_unpack(r, N, K), bits)
    assert not np.array_equal(r, bits)
    # bit counts are kept per group, and complementing (a whole-row XOR)
    # commutes with the conversion
    cnt = lambda a: np.unpackbits(a.reshape(N, K // 128, 16), axis=2).sum(axis=2)
    assert np.array_equal(cnt(r), cnt(bits))
    assert np.array_equal(orc.g128x_repack(bits ^ 0xFF, N, K), r ^ 0xFF)
    # each group is converted on its own: changing one group changes only it
    b2 = bits.copy()
    b2[2, 16 * 3: 16 * 4] ^= 0x5A
    d = orc.g128x_repack(b2, N, K) != r
    assert d[2, 16 * 3: 16 * 4].any() and d.sum() == d[2, 16 * 3: 16 * 4].sum()
    # the same permutation in every group and row
    assert np.array_equal(orc.g128x_repack(bits[:, :16], N, 128), r[:, :16])


def test_g128x_leaves_the_last_word_and_keeps_fields_together(orc):
    """The layout's purpose, on the unit vectors: inputs 96..127 keep their
    positions, each field of six inputs 6f..6f+5 (f < 12) lands in one byte
    (bits 1..6, in order), and the 24 inputs 72..95 fill bits 0 and 7 of
    bytes 0..11."""
    K = 128
    pos = []
    for k in range(128):
        e = np.zeros((1, 16), dtype=np.uint8)
        e[0, k // 8] = 1 << (k % 8)
        pos.append(int(np.unpackbits(orc.g128x_repack(e, 1, K), bitorder="little").argmax()))
    assert pos[96:] == list(range(96, 128))
    for f in range(12):
        assert [pos[6 * f + i] for i in range(6)] == [8 * f + 1 + i for i in range(6)]
    assert sorted(pos[72:96]) == sorted([8 * b for b in range(12)] + [8 * b + 7 for b in range(12)])
