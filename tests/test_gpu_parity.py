"""GPU parity: the CUDA kernels (through the C ABI) against the CPU oracle on
the same seeded inputs.  Bit-exact for packing and the XOR patch; within
1e-3 * sum_k |s x_k| + 1e-6 (plus bf16 output rounding) for the GEMV."""
import numpy as np
import pytest
import torch

import bit_weight_gemv_sign_b300 as b1
from bit_weight_gemv_sign_b300 import synth
from tests.helpers import (abs_bound, assert_gemv_close, dev_bf16, dev_u8, dev_u16, host_u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    b1.load()


def _problem(N, K, B, seed, offset=0.0):
    bits, scales = synth.matrix(N, K, seed, scale_offset=offset)
    x = synth.x_for(B, K, seed)
    return bits, scales, x


def _run(bits, scales, x, N, K, B, variant, y_dtype=b1.F32, flags=0):
    y = b1.bit1_gemv_ex(dev_u8(bits), dev_u16(scales), dev_bf16(x).view(B, K), y_dtype=y_dtype,
                        variant=variant, flags=flags, N=N, K=K)
    torch.cuda.synchronize()
    return y


# ---------------------------------------------------------------- GEMV

SHAPES_B1 = [(1, 1024), (7, 1024), (256, 1024), (149, 2048), (300, 3072), (1025, 4096),
             (37, 5120), (64, 6144), (33, 7168), (513, 12288), (40, 13312),
             (151, 3072), (4097, 4096), (32, 4096), (33, 12288), (5000, 12288)]


@pytest.mark.parametrize("N,K", SHAPES_B1)
@pytest.mark.parametrize("variant", [b1.LUT6, b1.LUT, b1.SIMPLE, b1.AUTO])
def test_gemv_b1_matches_oracle(orc, N, K, variant):
    if variant == b1.LUT6 and b1.bit1_gemv_launches(1, N, K, b1.LUT6) == 0:
        pytest.skip("shape outside the 6-bit table kernel's limits")
    bits, scales, x = _problem(N, K, 1, 1000 + N + K)
    ref = orc.gemv(bits, scales, x, 1, N, K)
    y = _run(bits, scales, x, N, K, 1, variant)
    assert_gemv_close(y, ref, abs_bound(scales, x, K), f"variant {variant} N={N} K={K}")


@pytest.mark.parametrize("N,K,B", [(5, 128, 1), (33, 384, 2), (70, 1152, 3), (129, 2048, 5),
                                   (64, 4096, 8), (17, 640, 4)])
def test_gemv_simple_any_shape(orc, N, K, B):
    bits, scales, x = _problem(N, K, B, 2000 + N + K + B)
    ref = orc.gemv(bits, scales, x, B, N, K)
    y = _run(bits, scales, x, N, K, B, b1.SIMPLE)
    assert_gemv_close(y, ref, abs_bound(scales, x, K), f"simple N={N} K={K} B={B}")
    y = _run(bits, scales, x, N, K, B, b1.AUTO)
    assert_gemv_close(y, ref, abs_bound(scales, x, K), f"auto N={N} K={K} B={B}")


@pytest.mark.parametrize("variant", [b1.LUT6, b1.LUT, b1.SIMPLE])
def test_gemv_bf16_output(orc, variant):
    N, K = 777, 4096
    bits, scales, x = _problem(N, K, 1, 3001)
    ref = orc.gemv(bits, scales, x, 1, N, K)
    y = _run(bits, scales, x, N, K, 1, variant, y_dtype=b1.BF16)
    assert y.dtype == torch.bfloat16
    assert_gemv_close(y, ref, abs_bound(scales, x, K), "bf16 out")


@pytest.mark.parametrize("variant", [b1.LUT6, b1.LUT, b1.SIMPLE])
def test_gemv_row_flip_negates_exactly(variant):
    """Flipping all bits of a row negates its output bit for bit: the kernels
    sum +-x symmetrically (the table entries of complementary nibbles are exact
    negatives)."""
    N, K = 300, 4096
    bits, scales, x = _problem(N, K, 1, 3002)
    y0 = _run(bits, scales, x, N, K, 1, variant).cpu()
    fl = bits.copy()
    rows = [0, 17, 299]
    fl[rows] ^= 0xFF
    y1 = _run(fl, scales, x, N, K, 1, variant).cpu()
    assert torch.equal(y1[0, rows], -y0[0, rows])
    keep = [i for i in range(N) if i not in rows]
    assert torch.equal(y1[0, keep], y0[0, keep])


def test_gemv_special_values(orc):
    """Subnormal fp16 scales are used exactly; zero scales and zero
    activations give exact zeros."""
    N, K = 64, 2048
    bits, scales, x = _problem(N, K, 1, 3003)
    scales = scales.copy()
    scales[0, :] = 0x0001          # smallest fp16 subnormal
    scales[1, :] = 0x03FF          # largest subnormal
    scales[2, :] = 0x0000
    x = x.copy()
    x[0, :128] = 0                 # a whole group of zero activations
    ref = orc.gemv(bits, scales, x, 1, N, K)
    for v in (b1.LUT6, b1.LUT, b1.SIMPLE):
        y = _run(bits, scales, x, N, K, 1, v)
        assert_gemv_close(y, ref, abs_bound(scales, x, K), f"special {v}")
        assert float(y[0, 2]) == 0.0


@pytest.mark.parametrize("variant", [b1.LUT6, b1.LUT])
def test_gemv_pdl_flag_same_result(orc, variant):
    N, K = 999, 4096
    bits, scales, x = _problem(N, K, 1, 3004)
    a = _run(bits, scales, x, N, K, 1, variant)
    b = _run(bits, scales, x, N, K, 1, variant, flags=b1.FLAG_PDL)
    assert torch.equal(a, b)
    assert b1.bit1_device_wait_timeouts() == 0


def test_gemv_lut6_extreme_activation_ranges(orc):
    """Groups whose activations are tiny, huge or mixed in magnitude: the
    per-group power-of-two prescale keeps the fp16 table entries in range."""
    N, K = 96, 4096
    bits, scales, x = _problem(N, K, 1, 3005)
    xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float().numpy()
    xf[0, 0:128] *= 2.0 ** -100
    xf[0, 128:256] *= 2.0 ** 60
    xf[0, 256:384] *= np.where(np.arange(128) % 2 == 0, 2.0 ** 20, 2.0 ** -20)
    xf[0, 384:512] = 0.0
    xf[0, 512:640] = 65504.0 * 4
    x2 = synth.to_bf16_bits(xf)
    ref = orc.gemv(bits, scales, x2, 1, N, K)
    for v in (b1.LUT6, b1.SIMPLE):
        y = _run(bits, scales, x2, N, K, 1, v)
        assert_gemv_close(y, ref, abs_bound(scales, x2, K), f"extreme ranges {v}")


@pytest.mark.parametrize("m", synth.PROJ_8B, ids=[m.name for m in synth.PROJ_8B])
def test_gemv_8b_projections_full(orc, m):
    """The 8B-class projection shapes at full size, every output checked, in
    the launch configuration the benchmark times (AUTO, PDL)."""
    bits, scales, x = _problem(m.N, m.K, 1, 4000 + m.N + m.K)
    ref = orc.gemv_threads(bits, scales, x, 1, m.N, m.K, 8)
    y = _run(bits, scales, x, m.N, m.K, 1, b1.AUTO, flags=b1.FLAG_PDL)
    assert_gemv_close(y, ref, abs_bound(scales, x, m.K), m.name)


def test_tiny_config_with_patch(orc):
    """256 x 1024, scales |N(0,0.02)| + 1e-3; GEMV, then an 8-row XOR patch
    applied (GEMV against the patched oracle), then removed (bit-identical)."""
    m = synth.TINY
    bits, scales, x = _problem(m.N, m.K, 1, 0, offset=1e-3)
    dbits = dev_u8(bits)
    ds, dx = dev_u16(scales), dev_bf16(x).view(1, m.K)
    y = b1.bit1_gemv(dbits, ds, dx)
    assert_gemv_close(y, orc.gemv(bits, scales, x, 1, m.N, m.K), abs_bound(scales, x, m.K), "tiny")
    rows = synth.distinct_rows(m.N, 8, 0)
    b1.bit1_xor_patch(dbits, rows)
    patched = orc.xor_patch(bits, m.N, m.K, rows)
    assert np.array_equal(dbits.cpu().numpy(), patched)
    y = b1.bit1_gemv(dbits, ds, dx)
    assert_gemv_close(y, orc.gemv(patched, scales, x, 1, m.N, m.K), abs_bound(scales, x, m.K), "tiny patched")
    b1.bit1_xor_patch(dbits, rows)
    assert np.array_equal(dbits.cpu().numpy(), bits)


# ---------------------------------------------------------------- XOR patch

def test_xor_patch_bit_exact(orc):
    N, K = 1000, 4096
    bits, _ = synth.matrix(N, K, 5001)
    d = dev_u8(bits)
    rows = [3, 999, 0, 500, 3, 3, 77]          # 3 listed three times: flips once
    b1.bit1_xor_patch(d, rows)
    assert np.array_equal(d.cpu().numpy(), orc.xor_patch(bits, N, K, rows))
    b1.bit1_xor_patch(d, rows)
    assert np.array_equal(d.cpu().numpy(), bits)


def test_xor_patch_many_rows_and_range_error(orc):
    N, K = 4096, 1024
    bits, _ = synth.matrix(N, K, 5002)
    d = dev_u8(bits)
    rows = synth.distinct_rows(N, 2500, 1)      # more than one launch's worth
    b1.bit1_xor_patch(d, rows)
    assert np.array_equal(d.cpu().numpy(), orc.xor_patch(bits, N, K, rows))
    before = d.clone()
    with pytest.raises(b1.Bit1Error) as e:
        b1.bit1_xor_patch(d, [1, 2, N])
    assert e.value.status == b1.ERANGE
    torch.cuda.synchronize()
    assert torch.equal(d, before)
    b1.bit1_xor_patch(d, [])                    # empty patch is a no-op
    assert torch.equal(d, before)


# ---------------------------------------------------------------- pack

@pytest.mark.parametrize("N,K", [(1, 128), (37, 384), (256, 1024), (100, 4096)])
@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
def test_pack_bit_exact(orc, N, K, dt):
    w32 = synth.fp_weights(N, K, 6000 + N + K)
    w32[0, :4] = [0.0, -0.0, 1e-30, -1e-30]
    if dt == "f32":
        host, code, dev = w32, orc.F32, torch.from_numpy(w32).cuda()
    elif dt == "bf16":
        host = synth.to_bf16_bits(w32)
        code, dev = orc.BF16, dev_bf16(host).view(N, K)
    else:
        host = w32.astype(np.float16).view(np.uint16)
        code, dev = orc.F16, dev_u16(host).view(torch.float16).view(N, K)
    st, rbits, rscales = orc.pack(host, code, N, K)
    assert st == orc.OK
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    bits, scales = b1.bit1_pack(dev, flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    assert np.array_equal(bits.cpu().numpy(), rbits)
    assert np.array_equal(host_u16(scales), rscales)


def test_pack_flags_nan_and_range(orc):
    w = synth.fp_weights(4, 256, 6100)
    w[2, 7] = np.nan
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    b1.bit1_pack(torch.from_numpy(w).cuda(), flags=flags)
    torch.cuda.synchronize()
    assert b1.bit1_pack_flags_status(int(flags.item())) == b1.ENAN
    assert orc.pack(w, orc.F32, 4, 256)[0] == orc.ENAN
    w = np.full((2, 128), 7e4, dtype=np.float32)
    b1.bit1_pack(torch.from_numpy(w).cuda(), flags=flags)
    torch.cuda.synchronize()
    assert b1.bit1_pack_flags_status(int(flags.item())) == b1.ERANGE
    assert orc.pack(w, orc.F32, 2, 128)[0] == orc.ERANGE


def test_pack_then_gemv_round_trip(orc):
    """Pack on the GPU, run the GEMV on the packed result, compare with the
    oracle's GEMV on the oracle's own packing (identical bits/scales)."""
    N, K = 512, 4096
    w = synth.fp_weights(N, K, 6200)
    bits, scales = b1.bit1_pack(torch.from_numpy(w).cuda())
    x = synth.x_for(1, K, 6200)
    y = b1.bit1_gemv(bits, scales, dev_bf16(x).view(1, K))
    st, rb, rs = orc.pack(w, orc.F32, N, K)
    assert_gemv_close(y, orc.gemv(rb, rs, x, 1, N, K), abs_bound(rs, x, K), "pack+gemv")


# ---------------------------------------------------------------- grouped GEMV

GROUP_SHAPES = [(33, 5120), (1, 1024), (999, 12288), (40, 2048), (4096, 4096), (7, 17408),
                (1025, 4096), (300, 3072), (64, 6144)]


def test_group_matches_stream_and_oracle(orc):
    """Many independent problems in one launch: every output bit-identical to
    the one-problem launches of the same kernel, and within tolerance of the
    oracle (mixed K, ragged N, fp32 and bf16 outputs)."""
    probs, host = [], []
    for i, (N, K) in enumerate(GROUP_SHAPES):
        bits, scales, x = _problem(N, K, 1, 7000 + i)
        yd = torch.float32 if i % 2 == 0 else torch.bfloat16
        y = torch.empty(1, N, dtype=yd, device="cuda")
        probs.append((dev_u8(bits), dev_u16(scales), dev_bf16(x).view(1, K), y))
        host.append((bits, scales, x, N, K))
    plan = b1.GroupPlan(probs)
    plan.run()
    torch.cuda.synchronize()
    for (bits, scales, x, N, K), (db, ds, dx, y) in zip(host, probs):
        ref = orc.gemv(bits, scales, x, 1, N, K)
        assert_gemv_close(y, ref, abs_bound(scales, x, K), f"group N={N} K={K}")
        y1 = b1.bit1_gemv_ex(db, ds, dx, y=torch.empty_like(y), variant=b1.STREAM)
        torch.cuda.synchronize()
        assert torch.equal(y1, y), f"group vs single N={N} K={K}"
    # a second run of the same plan gives the same bits
    before = [p[3].clone() for p in probs]
    plan.run(flags=b1.FLAG_PDL)
    torch.cuda.synchronize()
    assert all(torch.equal(a, p[3]) for a, p in zip(before, probs))
    assert b1.bit1_device_wait_timeouts() == 0


@pytest.mark.parametrize("N,K", [(1, 1024), (151936, 4096), (4096, 12288), (5120, 17408), (37, 5120)])
def test_stream_variant_matches_oracle(orc, N, K):
    bits, scales, x = _problem(N, K, 1, 7100 + N)
    ref = orc.gemv_threads(bits, scales, x, 1, N, K, 8)
    y = _run(bits, scales, x, N, K, 1, b1.STREAM)
    assert_gemv_close(y, ref, abs_bound(scales, x, K), f"stream N={N} K={K}")


def test_stream_row_flip_negates_exactly():
    N, K = 300, 12288
    bits, scales, x = _problem(N, K, 1, 7200)
    y0 = _run(bits, scales, x, N, K, 1, b1.STREAM).cpu()
    fl = bits.copy()
    fl[[5, 299]] ^= 0xFF
    y1 = _run(fl, scales, x, N, K, 1, b1.STREAM).cpu()
    assert torch.equal(y1[0, [5, 299]], -y0[0, [5, 299]])
