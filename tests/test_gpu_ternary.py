"""Ternary weights in 2-bit slots on the GPU against the CPU oracle: the
codes -> planes encoder bit-exact, the product through every kernel family
within the GEMV tolerance, the special cases the reading fixes exactly (no
zeros = the binary product, all zeros = 0), and the full-size 8B-class
ternary sweep in the benchmark's launch configuration (one grouped launch over
both planes of every matrix plus one combine) on sampled rows."""
import numpy as np
import pytest
import torch

import bit_weight_gemv_sign_b300 as b1
from bit_weight_gemv_sign_b300 import synth
from bit_weight_gemv_sign_b300.sweep import TernarySweep
from tests.helpers import abs_bound, assert_gemv_close, dev_bf16, dev_u8, dev_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    b1.load()


@pytest.mark.parametrize("N,K", [(1, 128), (37, 1152), (300, 4096)])
def test_planes_bit_exact(orc, N, K):
    t = synth.ternary_codes(N, K, synth.rng(800 + N))
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    a, b = b1.bit1_ternary_planes(torch.from_numpy(t).cuda(), flags=flags)
    torch.cuda.synchronize()
    ea, eb = orc.ternary_planes(t, N, K)
    assert np.array_equal(a.cpu().numpy(), ea) and np.array_equal(b.cpu().numpy(), eb)
    assert b1.bit1_pack_flags_status(int(flags.item())) == b1.OK


@pytest.mark.parametrize("bad", [2, -2, 100, -128])
def test_planes_flag_bad_codes(bad):
    N, K = 4, 256
    t = np.zeros((N, K), dtype=np.int8)
    t[3, 255] = bad
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    b1.bit1_ternary_planes(torch.from_numpy(t).cuda(), flags=flags)
    torch.cuda.synchronize()
    assert b1.bit1_pack_flags_status(int(flags.item())) == b1.ERANGE


CASES = [  # (variant, B, N, K)
    (b1.AUTO, 1, 1000, 4096), (b1.LUT, 1, 333, 3072), (b1.LUT6, 1, 4100, 4096), (b1.AUTO, 1, 129, 1152),
    (b1.STREAM, 1, 2049, 2048), (b1.SIMPLE, 2, 77, 384), (b1.LUT6, 5, 1000, 4096),
    (b1.AUTO, 3, 640, 1024), (b1.TC, 16, 700, 2048), (b1.TC, 64, 512, 4096),
]


@pytest.mark.parametrize("variant,B,N,K", CASES)
def test_gemv_ternary_parity(orc, variant, B, N, K):
    seed = 810 + N + B
    a, b, scales = synth.ternary_matrix(N, K, seed)
    x = synth.x_for(B, K, seed)
    ref = orc.gemv_ternary(a, b, scales, x, B, N, K)
    bound = abs_bound(scales, x, K)
    da, db, ds, dx = dev_u8(a), dev_u8(b), dev_u16(scales), dev_bf16(x).view(B, K)
    for ydt in (b1.F32, b1.BF16):
        y = b1.bit1_gemv_ternary(da, db, ds, dx, y_dtype=ydt, variant=variant)
        torch.cuda.synchronize()
        assert_gemv_close(y, ref, bound, f"ternary variant {variant} B={B} N={N} K={K} y={ydt}")
    assert b1.bit1_device_wait_timeouts() == 0


def test_codes_to_product_on_the_device(orc):
    """Codes encoded by the GPU, multiplied by the GPU, against the oracle's
    product of the codes' own planes."""
    N, K, B = 512, 2048, 1
    g = synth.rng(830)
    t = synth.ternary_codes(N, K, g)
    scales = synth.group_scales(N, K, g)
    x = synth.activations(B, K, g)
    a, b = b1.bit1_ternary_planes(torch.from_numpy(t).cuda())
    y = b1.bit1_gemv_ternary(a, b, dev_u16(scales), dev_bf16(x).view(B, K))
    torch.cuda.synchronize()
    ea, eb = orc.ternary_planes(t, N, K)
    assert_gemv_close(y, orc.gemv_ternary(ea, eb, scales, x, B, N, K), abs_bound(scales, x, K), "codes->y")


@pytest.mark.parametrize("variant,B", [(b1.LUT, 1), (b1.LUT6, 1), (b1.LUT6, 4), (b1.TC, 16)])
def test_no_zeros_is_the_binary_product_bit_for_bit(variant, B):
    """a == b: both halves are the same binary product, and (y + y) / 2 == y
    in fp32, so the ternary result equals the binary kernel's bits."""
    N, K = 1024, 4096
    bits, scales = synth.matrix(N, K, 840)
    x = synth.x_for(B, K, 840)
    da, ds, dx = dev_u8(bits), dev_u16(scales), dev_bf16(x).view(B, K)
    ws = torch.empty(max(b1.bit1_gemv_ternary_workspace_bytes(B, N, K), 256), dtype=torch.uint8, device="cuda")
    yt = b1.bit1_gemv_ternary(da, da, ds, dx, workspace=ws, variant=variant)
    wsb = torch.empty(max(b1.bit1_gemv_workspace_bytes(B, N, K), 256), dtype=torch.uint8, device="cuda")
    yb = b1.bit1_gemv_ex(da, ds, dx, workspace=wsb, variant=variant)
    torch.cuda.synchronize()
    assert torch.equal(yt, yb)


def test_all_zero_codes_give_exact_zero():
    N, K, B = 256, 4096, 2
    a, _, scales = synth.ternary_matrix(N, K, 841)
    x = synth.x_for(B, K, 841)
    da = dev_u8(a)
    y = b1.bit1_gemv_ternary(da, torch.bitwise_not(da), dev_u16(scales), dev_bf16(x).view(B, K))
    torch.cuda.synchronize()
    assert torch.count_nonzero(y).item() == 0


def test_row_flipped_in_both_planes(orc):
    N, K, B = 600, 4096, 1
    a, b, scales = synth.ternary_matrix(N, K, 842)
    x = synth.x_for(B, K, 842)
    da, db = dev_u8(a), dev_u8(b)
    rows = [0, 17, 599]
    b1.bit1_xor_patch(da, rows, N=N, K=K)
    b1.bit1_xor_patch(db, rows, N=N, K=K)
    y = b1.bit1_gemv_ternary(da, db, dev_u16(scales), dev_bf16(x).view(B, K))
    torch.cuda.synchronize()
    pa, pb = orc.xor_patch(a, N, K, rows), orc.xor_patch(b, N, K, rows)
    ref = orc.gemv_ternary(pa, pb, scales, x, B, N, K)
    assert_gemv_close(y, ref, abs_bound(scales, x, K), "patched ternary")
    ref0 = orc.gemv_ternary(a, b, scales, x, B, N, K)
    assert np.array_equal(ref[:, rows], -ref0[:, rows])


def test_workspace_is_required():
    N, K = 64, 1024
    a, b, scales = synth.ternary_matrix(N, K, 843)
    x = dev_bf16(synth.x_for(1, K, 843)).view(1, K)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(b1.Bit1Error) as e:
        b1.bit1_gemv_ternary(dev_u8(a), dev_u8(b), dev_u16(scales), x, workspace=small)
    assert e.value.status == b1.EINVAL


def test_combine_ragged_lengths():
    for n in (1, 3, 4, 5, 1023, 4097):
        g = torch.Generator(device="cuda")
        g.manual_seed(n)
        ya = torch.randn(n, device="cuda", generator=g)
        yb = torch.randn(n, device="cuda", generator=g)
        y = torch.empty(n, device="cuda")
        b1.bit1_ternary_combine(ya, yb, y)
        yh = torch.empty(n, device="cuda", dtype=torch.bfloat16)
        b1.bit1_ternary_combine(ya, yb, yh)
        torch.cuda.synchronize()
        exact = (ya.double() + yb.double()) / 2
        assert torch.equal(y, ((ya + yb) * 0.5))
        assert (y.double() - exact).abs().max().item() <= 2.0 ** -24 * exact.abs().max().item() + 1e-30
        assert torch.equal(yh, y.bfloat16())


def _sample_rows(N, count, seed):
    rows = np.random.default_rng(seed).choice(N, min(count, N), replace=False)
    return np.unique(np.concatenate([rows, [0, N - 1]])).astype(np.int64)


def test_ternary_sweep_8b_grouped_sampled_parity(orc):
    """Both planes of all 253 matrices (2.1 GB of planes) in one grouped
    launch plus one combine, bf16 output: sampled rows of every matrix
    against the oracle; a second step gives the same bits."""
    sw = TernarySweep(synth.sweep_8b(), seed0=500, y_dtype=b1.BF16).fill()
    plan = sw.group_plan()
    plan.run()
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    for i in range(len(sw.mats)):
        m = sw.mats[i]
        ha, hb, hs, hx = sw.host_matrix(i)
        rows = _sample_rows(m.N, 16, 2000 + i)
        ref = orc.gemv_ternary_select(ha, hb, hs, hx, 1, m.N, m.K, rows)
        got = sw.y_of(i)[:, torch.from_numpy(rows).cuda()]
        assert_gemv_close(got, ref, abs_bound(hs[rows], hx, m.K), f"ternary sweep matrix {i} ({m.name})")
    first = sw.yt.clone()
    plan.run()
    torch.cuda.synchronize()
    assert torch.equal(first, sw.yt)


# ---------------------------------------------------------------- five codes per byte

@pytest.mark.parametrize("N,K", [(1, 128), (37, 1152), (300, 4096)])
def test_t5_pack_and_planes_bit_exact(orc, N, K):
    t = synth.ternary_codes(N, K, synth.rng(850 + N))
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = b1.bit1_t5_pack(torch.from_numpy(t).cuda(), flags=flags)
    torch.cuda.synchronize()
    assert b1.bit1_pack_flags_status(int(flags.item())) == b1.OK
    ep = orc.t5_pack(t, N, K)
    assert np.array_equal(p.cpu().numpy(), ep)
    a, b = b1.bit1_t5_to_planes(p, K, flags=flags)
    torch.cuda.synchronize()
    assert b1.bit1_pack_flags_status(int(flags.item())) == b1.OK
    ea, eb = orc.ternary_planes(orc.t5_unpack(ep, N, K), N, K)
    assert np.array_equal(a.cpu().numpy(), ea) and np.array_equal(b.cpu().numpy(), eb)


def test_t5_every_byte_value_through_the_planes(orc):
    """All 243 five-code bytes and all 27 three-code bytes, decoded by the
    device transcode, against the oracle's base-3 decoding."""
    N, K = 243, 128
    p = np.empty((N, 26), dtype=np.uint8)
    p[:, :25] = 121
    p[:, 25] = 13
    p[:, 7] = np.arange(243)
    p[:27, 25] = np.arange(27)
    a, b = b1.bit1_t5_to_planes(torch.from_numpy(p).cuda(), K)
    torch.cuda.synchronize()
    ea, eb = orc.ternary_planes(orc.t5_unpack(p, N, K), N, K)
    assert np.array_equal(a.cpu().numpy(), ea) and np.array_equal(b.cpu().numpy(), eb)


def test_t5_flags_bad_codes_and_bytes():
    N, K = 2, 256
    t = np.zeros((N, K), dtype=np.int8)
    t[1, 130] = -3
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    b1.bit1_t5_pack(torch.from_numpy(t).cuda(), flags=flags)
    torch.cuda.synchronize()
    assert b1.bit1_pack_flags_status(int(flags.item())) == b1.ERANGE
    for pos, val in ((3, 243), (25, 27), (51, 200)):
        p = np.full((N, 52), 121, dtype=np.uint8)
        p[:, 25] = p[:, 51] = 13
        p[1, pos] = val
        b1.bit1_t5_to_planes(torch.from_numpy(p).cuda(), K, flags=flags)
        torch.cuda.synchronize()
        assert b1.bit1_pack_flags_status(int(flags.item())) == b1.ERANGE, (pos, val)


@pytest.mark.parametrize("B,N,K", [(1, 1000, 4096), (3, 129, 1152), (8, 257, 2048), (11, 64, 1024)])
def test_gemv_t5_parity(orc, B, N, K):
    g = synth.rng(860 + B)
    t = synth.ternary_codes(N, K, g)
    scales = synth.group_scales(N, K, g)
    x = synth.activations(B, K, g)
    p = orc.t5_pack(t, N, K)
    ref = orc.gemv_t5(p, scales, x, B, N, K)
    bound = abs_bound(scales, x, K)
    for ydt in (b1.F32, b1.BF16):
        y = b1.bit1_gemv_t5(dev_u8(p), dev_u16(scales), dev_bf16(x).view(B, K), y_dtype=ydt, N=N)
        torch.cuda.synchronize()
        assert_gemv_close(y, ref, bound, f"t5 B={B} N={N} K={K} y={ydt}")


def test_t5_stored_then_run_on_the_slot_kernels(orc):
    """The compact packing, expanded on the device, multiplied by the 2-bit
    slot path: the same result (within tolerance) as the direct product."""
    N, K, B = 4096, 4096, 1
    g = synth.rng(870)
    t = synth.ternary_codes(N, K, g)
    scales = synth.group_scales(N, K, g)
    x = synth.activations(B, K, g)
    p = dev_u8(orc.t5_pack(t, N, K))
    a, b = b1.bit1_t5_to_planes(p, K)
    ds, dx = dev_u16(scales), dev_bf16(x).view(B, K)
    y1 = b1.bit1_gemv_ternary(a, b, ds, dx)
    y2 = b1.bit1_gemv_t5(p, ds, dx, N=N)
    torch.cuda.synchronize()
    rows = np.arange(0, N, 37)
    ea, eb = orc.ternary_planes(t, N, K)
    ref = orc.gemv_ternary_select(ea, eb, scales, x, B, N, K, rows)
    bd = abs_bound(scales[rows], x, K)
    idx = torch.from_numpy(rows).cuda()
    assert_gemv_close(y1[:, idx], ref, bd, "t5 -> planes -> slot kernels")
    assert_gemv_close(y2[:, idx], ref, bd, "t5 direct")


@pytest.mark.parametrize("N,K", [(1, 1024), (33, 4096), (1000, 5120), (300, 12288), (5000, 2048), (64, 17408)])
def test_gemv_t5_batch1_table_kernel(orc, N, K):
    """Batch 1 with K a multiple of 1024 runs the table-lookup kernel (K in one
    chunk, in several, and with a partial last chunk; ragged N): every output
    against the oracle, fp32 and bf16, and the same result as the slot
    kernels on the planes of the same codes (within the tolerance)."""
    g = synth.rng(880 + N)
    t = synth.ternary_codes(N, K, g)
    scales = synth.group_scales(N, K, g)
    x = synth.activations(1, K, g)
    p = orc.t5_pack(t, N, K)
    ref = orc.gemv_t5(p, scales, x, 1, N, K)
    bound = abs_bound(scales, x, K)
    dp, ds, dx = dev_u8(p), dev_u16(scales), dev_bf16(x).view(1, K)
    for ydt in (b1.F32, b1.BF16):
        y = b1.bit1_gemv_t5(dp, ds, dx, y_dtype=ydt, N=N)
        torch.cuda.synchronize()
        assert_gemv_close(y, ref, bound, f"t5 table kernel N={N} K={K} y={ydt}")
    a, b = b1.bit1_t5_to_planes(dp, K)
    ys = b1.bit1_gemv_ternary(a, b, ds, dx)
    y = b1.bit1_gemv_t5(dp, ds, dx, N=N)
    torch.cuda.synchronize()
    assert_gemv_close(y, ys.double().cpu().numpy(), 2 * bound, "t5 table kernel vs slot kernels")
    y2 = b1.bit1_gemv_t5(dp, ds, dx, N=N)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)                      # deterministic
    assert b1.bit1_gemv_t5_launches(1, N, K) == 1
