"""The SwiGLU epilogue of the grouped launch: a problem whose rows are
interleaved (gate, up) pairs writes h = silu(gate) * up instead of the two
products (the Bonsai 27B page, section "Bonsai 27B의 표현 방식": the base
model's MLP is SwiGLU).  Against the CPU oracle on mixed plans (SwiGLU and
plain problems in one launch; one and several K chunks; ragged pair counts),
batch rows 1 .. 6, fp32 and bf16 output; the full 8B-class sweep with fused
gate/up matrices on sampled outputs of every matrix."""
import numpy as np
import pytest
import torch

import bit_weight_gemv_sign_b300 as b1
from bit_weight_gemv_sign_b300 import synth
from bit_weight_gemv_sign_b300.sweep import Sweep
from tests.helpers import (abs_bound, assert_gemv_close, assert_swiglu_close, carried_bound, dev_bf16, dev_u8,
                           dev_u16, swiglu_h_tol)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    b1.load()


# (N, K, SwiGLU): N is the interleaved row count of a SwiGLU problem
SHAPES = [(2000, 4096, True), (300, 4096, False), (64, 1024, True), (2050, 5120, True),
          (300, 12288, True), (2, 2048, True), (4096, 1024, False), (24576, 4096, True)]


def _problems(B, seed, ydt, shapes=SHAPES):
    host, probs = [], []
    for i, (N, K, sw) in enumerate(shapes):
        bits, scales = synth.matrix(N, K, seed + i)
        x = synth.x_for(B, K, seed + i)
        out = N // 2 if sw else N
        y = torch.empty((B, out), dtype=torch.bfloat16 if ydt == b1.BF16 else torch.float32, device="cuda")
        host.append((bits, scales, x))
        xd = dev_bf16(x).view(B, K) if B > 1 else dev_bf16(x).view(K)
        probs.append((dev_u8(bits), dev_u16(scales), xd, y, b1.EPI_SWIGLU if sw else b1.EPI_NONE))
    return host, probs


def _check(orc, shapes, host, probs, B, what):
    for (N, K, sw), (bits, scales, x), pr in zip(shapes, host, probs):
        y = pr[3]
        bound = abs_bound(scales, x, K)
        if not sw:
            assert_gemv_close(y, orc.gemv(bits, scales, x, B, N, K), bound, f"{what} plain N={N} K={K}")
            continue
        yo = orc.gemv(bits, scales, x, B, N, K)
        h = orc.gemv_swiglu(bits, scales, x, B, N, K)
        assert_swiglu_close(y, h, yo[:, 0::2], yo[:, 1::2], bound[:, 0::2], bound[:, 1::2],
                            f"{what} SwiGLU N={N} K={K}")


@pytest.mark.parametrize("B", [1, 2, 3, 5, 6])
@pytest.mark.parametrize("ydt", [b1.F32, b1.BF16])
def test_swiglu_grouped_matches_oracle(orc, B, ydt):
    shapes = SHAPES if B <= 2 else SHAPES[:-1]
    host, probs = _problems(B, 9400 + 10 * B + ydt, ydt, shapes)
    plan = b1.GroupPlan(probs, B=B)
    plan.run()
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    _check(orc, shapes, host, probs, B, f"grouped B={B} y={ydt}")
    first = [p[3].clone() for p in probs]
    plan.run(flags=b1.FLAG_PDL)
    torch.cuda.synchronize()
    for a, p in zip(first, probs):
        assert torch.equal(a, p[3])


def test_swiglu_pairs_the_plain_products():
    """The fused epilogue acts on the very accumulators the plain launch
    writes: h agrees with silu(g) * u formed by torch in fp32 from the plain
    fp32 results to a few ulps, pair by pair, in the interleaved order."""
    shapes = [(2000, 4096, True), (300, 12288, True), (2050, 5120, True)]
    for B in (1, 4):
        host, probs = _problems(B, 9500 + B, b1.F32, shapes)
        plain = [(p[0], p[1], p[2], torch.empty((B, s[0]), dtype=torch.float32, device="cuda"))
                 for p, s in zip(probs, shapes)]
        b1.GroupPlan(probs, B=B).run()
        b1.GroupPlan(plain, B=B).run()
        torch.cuda.synchronize()
        for p, q in zip(probs, plain):
            g, u = q[3][:, 0::2], q[3][:, 1::2]
            want = torch.nn.functional.silu(g) * u
            tol = 8 * 2.0 ** -24 * (g.abs() * u.abs()) + 1e-30
            assert torch.all((p[3] - want).abs() <= tol)


def test_swiglu_rejects_odd_rows_and_unknown_epilogue():
    host, probs = _problems(1, 9600, b1.F32, [(64, 1024, True)])
    bits, scales, x, _, _ = probs[0]
    odd = (bits[:63], scales[:63], x, torch.empty(31, device="cuda"), b1.EPI_SWIGLU)
    with pytest.raises(b1.Bit1Error) as e:
        b1.GroupPlan([odd])
    assert e.value.status == b1.ESHAPE
    bad = (bits, scales, x, torch.empty(64, device="cuda"), 2)
    with pytest.raises(b1.Bit1Error) as e:
        b1.GroupPlan([bad])
    assert e.value.status == b1.ESHAPE


def _sample(n, count, seed):
    r = np.random.default_rng(seed).choice(n, min(count, n), replace=False)
    return np.unique(np.concatenate([r, [0, n - 1]])).astype(np.int64)


def test_fused_mlp_sweep_8b_sampled_parity(orc):
    """The 8B-class sweep with every layer's gate and up in one interleaved
    24576 x 4096 matrix ending in SwiGLU: one grouped launch, bf16 output,
    sampled outputs of all 217 matrices against the oracle."""
    sw = Sweep(synth.sweep_8b_fused_mlp(), seed0=800, batch=1, y_dtype=b1.BF16).fill()
    plan = sw.group_plan()
    plan.run()
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    for i, m in enumerate(sw.mats):
        hb, hs, hx = sw.host_matrix(i)
        units = _sample(m.out, 8, 4000 + i)
        got = sw.y_of(i)[:, torch.from_numpy(units).cuda()]
        if not m.swiglu:
            ref = orc.gemv_select(hb, hs, hx, 1, m.N, m.K, units)
            assert_gemv_close(got, ref, abs_bound(hs[units], hx, m.K), f"fused sweep {m.name}")
            continue
        h = orc.gemv_swiglu_select(hb, hs, hx, 1, m.N, m.K, units)
        gu = orc.gemv_select(hb, hs, hx, 1, m.N, m.K, np.stack([2 * units, 2 * units + 1], 1).ravel())
        bd = abs_bound(hs.reshape(m.N, -1)[np.stack([2 * units, 2 * units + 1], 1).ravel()], hx, m.K)
        assert_swiglu_close(got, h, gu[:, 0::2], gu[:, 1::2], bd[:, 0::2], bd[:, 1::2],
                            f"fused sweep {m.name}")


# ---------------------------------------------------------------- single call (bit1_gemv_ex)

# (N, K): interleaved row counts; ragged pair counts against the CTA split,
# one K word per lane up to the largest table kernel K, and beyond it
EX_SHAPES = [(2, 1024), (514, 2048), (2000, 4096), (24576, 4096), (8190, 5120), (4096, 12288),
             (300, 13312), (600, 16384)]


@pytest.mark.parametrize("N,K", EX_SHAPES)
@pytest.mark.parametrize("variant", [b1.AUTO, b1.LUT, b1.STREAM])
def test_gemv_ex_swiglu_matches_oracle(orc, N, K, variant):
    if variant == b1.LUT and K > 13312:
        pytest.skip("the nibble-table kernel holds K <= 13312")
    bits, scales = synth.matrix(N, K, 9700 + N % 97 + K // 1024)
    x = synth.x_for(1, K, 9700 + K // 1024)
    db, ds, dx = dev_u8(bits), dev_u16(scales), dev_bf16(x).view(1, K)
    for ydt in (b1.F32, b1.BF16):
        h = b1.bit1_gemv_ex(db, ds, dx, y_dtype=ydt, variant=variant, flags=b1.FLAG_SWIGLU)
        torch.cuda.synchronize()
        assert h.shape == (1, N // 2)
        yo = orc.gemv(bits, scales, x, 1, N, K)
        ho = orc.gemv_swiglu(bits, scales, x, 1, N, K)
        bd = abs_bound(scales, x, K)
        assert_swiglu_close(h, ho, yo[:, 0::2], yo[:, 1::2], bd[:, 0::2], bd[:, 1::2],
                            f"gemv_ex SwiGLU N={N} K={K} variant={variant} y={ydt}")


def test_gemv_ex_swiglu_equals_grouped_epilogue():
    """The single call on the grouped kernel (STREAM) and a one-problem grouped
    plan run the same code: bit-identical h."""
    N, K = 2050, 5120
    bits, scales = synth.matrix(N, K, 9800)
    x = synth.x_for(1, K, 9800)
    db, ds, dx = dev_u8(bits), dev_u16(scales), dev_bf16(x).view(1, K)
    h1 = b1.bit1_gemv_ex(db, ds, dx, variant=b1.STREAM, flags=b1.FLAG_SWIGLU)
    h2 = torch.empty((1, N // 2), device="cuda")
    b1.GroupPlan([(db, ds, dx.view(K), h2, b1.EPI_SWIGLU)]).run()
    torch.cuda.synchronize()
    assert torch.equal(h1, h2)


def test_gemv_ex_swiglu_feeds_the_down_projection(orc):
    """gate/up -> h (bf16) -> down with no kernel in between, under PDL.  The
    oracle runs the same chain on its own h (rounded to bf16 by torch); the
    down tolerance adds what the GPU's h may differ from it by (the SwiGLU
    tolerance plus both bf16 roundings), carried through |W_down|."""
    H, D = 2048, 1024          # hidden units, model width
    gb, gs = synth.matrix(2 * H, D, 9900)
    x = synth.x_for(1, D, 9900)
    db2, ds2 = synth.matrix(D, H, 9901)
    h = b1.bit1_gemv_ex(dev_u8(gb), dev_u16(gs), dev_bf16(x).view(1, D), y_dtype=b1.BF16,
                        flags=b1.FLAG_SWIGLU | b1.FLAG_PDL)
    y = b1.bit1_gemv_ex(dev_u8(db2), dev_u16(ds2), h, flags=b1.FLAG_PDL)
    torch.cuda.synchronize()
    ho = orc.gemv_swiglu(gb, gs, x, 1, 2 * H, D)
    yo = orc.gemv(gb, gs, x, 1, 2 * H, D)
    bd = abs_bound(gs, x, D)
    assert_swiglu_close(h, ho, yo[:, 0::2], yo[:, 1::2], bd[:, 0::2], bd[:, 1::2], "gate/up")
    hx = synth.to_bf16_bits(ho.astype(np.float32))                 # the oracle's h as bf16
    ref = orc.gemv(db2, ds2, hx, 1, D, H)
    dh = swiglu_h_tol(yo[:, 0::2], yo[:, 1::2], bd[:, 0::2], bd[:, 1::2], ho)
    got = y.float().cpu().numpy().astype(np.float64)
    tol = 1e-3 * abs_bound(ds2, hx, H) + 1e-6 + carried_bound(ds2, dh, H)
    assert np.all(np.abs(got - ref) <= tol)


def test_fused_decode_chain_layer(orc):
    """One layer of the fused 8B-class decode chain through the sweep's
    dependent launches (graph + PDL): q|k|v and o against the oracle, the
    gate|up h against the oracle's SwiGLU, and down -- which reads the GPU's
    h -- against the oracle's down of its own h, with the h tolerance carried
    through |W_down|."""
    from bit_weight_gemv_sign_b300.synth import decode_chain_8b_fused
    mats = decode_chain_8b_fused()[:4]
    sw = Sweep(mats, seed0=1200, batch=1, y_dtype=b1.BF16, feed_swiglu=True).fill()
    sw.capture(pdl=True)
    with torch.cuda.stream(sw.stream):
        sw.replay()
    sw.stream.synchronize()
    host = [sw.host_matrix(i) for i in range(4)]
    for i in (0, 1):
        m, (hb, hs, hx) = mats[i], host[i]
        assert_gemv_close(sw.y_of(i), orc.gemv(hb, hs, hx, 1, m.N, m.K), abs_bound(hs, hx, m.K), m.name)
    m, (gb, gs, gx) = mats[2], host[2]
    yo = orc.gemv(gb, gs, gx, 1, m.N, m.K)
    ho = orc.gemv_swiglu(gb, gs, gx, 1, m.N, m.K)
    bd = abs_bound(gs, gx, m.K)
    assert_swiglu_close(sw.y_of(2), ho, yo[:, 0::2], yo[:, 1::2], bd[:, 0::2], bd[:, 1::2], m.name)
    m, (db_, ds_, _) = mats[3], host[3]
    hx = synth.to_bf16_bits(ho.astype(np.float32))
    ref = orc.gemv(db_, ds_, hx, 1, m.N, m.K)
    dh = swiglu_h_tol(yo[:, 0::2], yo[:, 1::2], bd[:, 0::2], bd[:, 1::2], ho)
    tol = 1e-3 * abs_bound(ds_, hx, m.K) + 1e-6 + carried_bound(ds_, dh, m.K) + 2.0 ** -8 * np.abs(ref)
    got = sw.y_of(3).float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= tol), m.name
    with pytest.raises(ValueError):
        sw.group_plan()


# (N, K) on the 6-bit cluster kernel at 2-8 rows: ragged row blocks, a short N
# whose K is split over warps, several K chunks
T6_SHAPES = [(1000, 2048), (64, 4096), (2050, 5120), (4096, 12288)]


@pytest.mark.parametrize("N,K", T6_SHAPES)
@pytest.mark.parametrize("B", [2, 3, 5, 8])
def test_gemv_ex_swiglu_six_bit_kernel(orc, N, K, B):
    """The cluster kernel's rank-order reduction splits the rows by pairs, so
    one thread sums a gate and its up row: against the oracle, AUTO (which
    picks this kernel at 2-8 rows) and the explicit variant, fp32 and bf16."""
    bits, scales = synth.matrix(N, K, 9930 + B + N % 7)
    x = synth.x_for(B, K, 9930 + B)
    db, ds, dx = dev_u8(bits), dev_u16(scales), dev_bf16(x).view(B, K)
    yo = orc.gemv(bits, scales, x, B, N, K)
    ho = orc.gemv_swiglu(bits, scales, x, B, N, K)
    bd = abs_bound(scales, x, K)
    for variant in (b1.AUTO, b1.LUT6):
        for ydt in (b1.F32, b1.BF16):
            h = b1.bit1_gemv_ex(db, ds, dx, y_dtype=ydt, variant=variant, flags=b1.FLAG_SWIGLU)
            torch.cuda.synchronize()
            assert h.shape == (B, N // 2)
            assert_swiglu_close(h, ho, yo[:, 0::2], yo[:, 1::2], bd[:, 0::2], bd[:, 1::2],
                                f"t6 SwiGLU N={N} K={K} B={B} v={variant} y={ydt}")
    assert b1.bit1_device_wait_timeouts() == 0


# (N, K, B) on the tensor cores: ragged row tiles, K split over a cluster
# (few row tiles, long K), batch padding, and batch > 64 (several chunks)
TC_SHAPES = [(2, 1024, 16), (300, 1024, 16), (1000, 2048, 20), (2048, 4096, 16), (64, 17408, 16),
             (4100, 2048, 48), (2048, 1024, 100)]


@pytest.mark.parametrize("N,K,B", TC_SHAPES)
def test_gemv_ex_swiglu_tensor_cores(orc, N, K, B):
    bits, scales = synth.matrix(N, K, 9960 + B)
    x = synth.x_for(B, K, 9960 + B)
    db, ds, dx = dev_u8(bits), dev_u16(scales), dev_bf16(x).view(B, K)
    yo = orc.gemv(bits, scales, x, B, N, K)
    ho = orc.gemv_swiglu(bits, scales, x, B, N, K)
    bd = abs_bound(scales, x, K)
    full = b1.bit1_gemv_workspace_bytes(B, N, K)
    sizes = [full] + ([b1.bit1_gemv_workspace_bytes(64, N, K)] if B > 64 else [])
    for ws_bytes in sizes:
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        for ydt in (b1.F32, b1.BF16):
            for variant in (b1.TC, b1.AUTO):
                h = b1.bit1_gemv_ex(db, ds, dx, y_dtype=ydt, workspace=ws, variant=variant,
                                    flags=b1.FLAG_SWIGLU | b1.FLAG_PDL)
                torch.cuda.synchronize()
                assert h.shape == (B, N // 2)
                assert_swiglu_close(h, ho, yo[:, 0::2], yo[:, 1::2], bd[:, 0::2], bd[:, 1::2],
                                    f"tc SwiGLU N={N} K={K} B={B} ws={ws_bytes} y={ydt} v={variant}")
    h2 = b1.bit1_gemv_tc_noalloc(db, ds, dx, flags=b1.FLAG_SWIGLU)
    torch.cuda.synchronize()
    assert_swiglu_close(h2, ho, yo[:, 0::2], yo[:, 1::2], bd[:, 0::2], bd[:, 1::2], f"tc noalloc SwiGLU N={N}")
    assert b1.bit1_device_wait_timeouts() == 0


@pytest.mark.parametrize("B", [64, 256])
def test_gemv_ex_swiglu_tensor_cores_mlp_gate_up(orc, B):
    """The 8B MLP's gate/up pair as one interleaved 24576 x 4096 matrix at a
    decode batch (64: split K) and a prompt batch (256: 128-row chunks):
    sampled hidden units of every batch row against the oracle."""
    N, K = 24576, 4096
    bits, scales = synth.matrix(N, K, 9990 + B)
    x = synth.x_for(B, K, 9990 + B)
    ws = torch.empty(b1.bit1_gemv_workspace_bytes(B, N, K), dtype=torch.uint8, device="cuda")
    h = b1.bit1_gemv_ex(dev_u8(bits), dev_u16(scales), dev_bf16(x).view(B, K), y_dtype=b1.BF16, workspace=ws,
                        flags=b1.FLAG_SWIGLU)
    torch.cuda.synchronize()
    units = _sample(N // 2, 24, 9990 + B)
    pairs = np.stack([2 * units, 2 * units + 1], 1).ravel()
    ho = orc.gemv_swiglu_select(bits, scales, x, B, N, K, units)
    gu = orc.gemv_select(bits, scales, x, B, N, K, pairs)
    bd = abs_bound(scales[pairs], x, K)
    assert_swiglu_close(h[:, torch.from_numpy(units).cuda()], ho, gu[:, 0::2], gu[:, 1::2], bd[:, 0::2],
                        bd[:, 1::2], f"tc SwiGLU gate/up B={B}")
    assert b1.bit1_device_wait_timeouts() == 0


def test_gemv_ex_swiglu_rejections():
    N, K = 64, 1024
    bits, scales = synth.matrix(N, K, 9950)
    x = synth.x_for(4, K, 9950)
    db, ds = dev_u8(bits), dev_u16(scales)
    dx1 = dev_bf16(x[:1]).view(1, K)
    dx4 = dev_bf16(x).view(4, K)
    cases = [
        (dict(x=dx1, N=63, y=torch.empty((1, 31), device="cuda")), b1.ESHAPE),        # odd rows
        (dict(x=dx1, variant=b1.SIMPLE), b1.ESHAPE),
        (dict(x=dx4, variant=b1.LUT), b1.ESHAPE),                                      # batch 1 only
    ]
    for kw, st in cases:
        with pytest.raises(b1.Bit1Error) as e:
            b1.bit1_gemv_ex(db, ds, flags=b1.FLAG_SWIGLU, **kw)
        assert e.value.status == st, kw
    with pytest.raises(b1.Bit1Error) as e:
        b1.bit1_gemv_ex(db, ds, dx1, flags=8)
    assert e.value.status == b1.EINVAL


# ---------------------------------------------------------------- ternary (2-bit slots)

@pytest.mark.parametrize("B,N,K,variant", [(1, 2000, 4096, b1.AUTO), (1, 514, 2048, b1.LUT6), (3, 1000, 2048, b1.AUTO),
                                           (16, 1024, 4096, b1.AUTO), (20, 300, 1024, b1.TC)])
def test_gemv_ternary_swiglu_matches_oracle(orc, B, N, K, variant):
    """Ternary gate/up pairs: both binary passes run plain (any variant), the
    combine forms the two means and h; against the ternary oracle pair."""
    a, b, scales = synth.ternary_matrix(N, K, 9970 + B)
    x = synth.x_for(B, K, 9970 + B)
    da, db_, ds, dx = dev_u8(a), dev_u8(b), dev_u16(scales), dev_bf16(x).view(B, K)
    yo = orc.gemv_ternary(a, b, scales, x, B, N, K)
    ho = orc.gemv_ternary_swiglu(a, b, scales, x, B, N, K)
    bd = abs_bound(scales, x, K)
    for ydt in (b1.F32, b1.BF16):
        h = b1.bit1_gemv_ternary(da, db_, ds, dx, y_dtype=ydt, variant=variant, flags=b1.FLAG_SWIGLU)
        torch.cuda.synchronize()
        assert h.shape == (B, N // 2)
        assert_swiglu_close(h, ho, yo[:, 0::2], yo[:, 1::2], bd[:, 0::2], bd[:, 1::2],
                            f"ternary SwiGLU B={B} N={N} K={K} v={variant} y={ydt}")
    assert b1.bit1_device_wait_timeouts() == 0
