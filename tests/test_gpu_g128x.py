"""The g128x sign-bit layout (bit1_repack_g128x / bit1_unpack_g128x and
grouped plans built with BIT1_LAYOUT_G128X): the conversion bit for bit
against the oracle, grouped products over converted bits identical to the
canonical ones and within the oracle's tolerance, row patches applied in the
converted layout, and the full 8B-class sweep in the configuration the
benchmark times (converted bits, one grouped launch, bf16 output)."""
import numpy as np
import pytest
import torch

import bit_weight_gemv_sign_b300 as b1
from bit_weight_gemv_sign_b300 import synth
from bit_weight_gemv_sign_b300.sweep import Sweep
from tests.helpers import abs_bound, assert_gemv_close, assert_swiglu_close, dev_bf16, dev_u8, dev_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    b1.load()


@pytest.mark.parametrize("N,K", [(1, 128), (1000, 1024), (77, 5120), (300, 4096), (33, 17408)])
def test_repack_and_unpack_match_oracle(orc, N, K):
    bits = synth.sign_bits(N, K, synth.rng(7000 + N))
    want = orc.g128x_repack(bits, N, K)
    d = dev_u8(bits)
    got = b1.bit1_repack_g128x(d)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), want)
    back = b1.bit1_unpack_g128x(got)
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy(), bits)
    # in place, both ways
    b1.bit1_repack_g128x(d, out=d)
    torch.cuda.synchronize()
    assert np.array_equal(d.cpu().numpy(), want)
    b1.bit1_unpack_g128x(d, out=d)
    torch.cuda.synchronize()
    assert np.array_equal(d.cpu().numpy(), bits)


# (N, K, epilogue): ragged row counts, several K chunks, gate/up pairs
SHAPES = [(4096, 4096, b1.EPI_NONE), (1000, 1024, b1.EPI_NONE), (514, 12288, b1.EPI_NONE),
          (2050, 4096, b1.EPI_SWIGLU), (96, 5120, b1.EPI_NONE)]


def _problems(B, seed, ydt):
    host, canon, conv = [], [], []
    yt = torch.bfloat16 if ydt == b1.BF16 else torch.float32
    for i, (N, K, epi) in enumerate(SHAPES):
        bits, scales = synth.matrix(N, K, seed + i)
        x = synth.x_for(B, K, seed + i)
        host.append((bits, scales, x))
        db, ds, dx = dev_u8(bits), dev_u16(scales), dev_bf16(x).view(B, K)
        out = N // 2 if epi == b1.EPI_SWIGLU else N
        canon.append((db, ds, dx, torch.empty((B, out), dtype=yt, device="cuda"), epi))
        conv.append((b1.bit1_repack_g128x(db), ds, dx, torch.empty((B, out), dtype=yt, device="cuda"), epi))
    torch.cuda.synchronize()
    return host, canon, conv


@pytest.mark.parametrize("B", [1, 2, 5])
@pytest.mark.parametrize("ydt", [b1.F32, b1.BF16])
def test_grouped_g128x_equals_canonical_and_oracle(orc, B, ydt):
    host, canon, conv = _problems(B, 7100 + 10 * B + ydt, ydt)
    b1.GroupPlan(canon, B=B).run()
    b1.GroupPlan(conv, B=B, layout=b1.LAYOUT_G128X).run()
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    for (N, K, epi), (bits, scales, x), pc, pg in zip(SHAPES, host, canon, conv):
        # the same tables, lookups and summation order: bit for bit the same
        assert torch.equal(pc[3], pg[3]), f"N={N} K={K} B={B}"
        bound = abs_bound(scales, x, K)
        yo = orc.gemv(bits, scales, x, B, N, K)
        if epi == b1.EPI_SWIGLU:
            h = orc.gemv_swiglu(bits, scales, x, B, N, K)
            assert_swiglu_close(pg[3], h, yo[:, 0::2], yo[:, 1::2], bound[:, 0::2], bound[:, 1::2],
                                f"g128x SwiGLU N={N} B={B}")
        else:
            assert_gemv_close(pg[3], yo, bound, f"g128x N={N} K={K} B={B}")


def test_g128x_row_patch_applies_in_the_converted_layout(orc):
    N, K = 4096, 4096
    bits, scales = synth.matrix(N, K, 7200)
    x = synth.x_for(1, K, 7200)
    rows = synth.distinct_rows(N, 40, 7201)
    d = b1.bit1_repack_g128x(dev_u8(bits))
    b1.bit1_xor_patch(d, rows, N=N, K=K)
    torch.cuda.synchronize()
    patched = orc.xor_patch(bits, N, K, rows)
    # patching the converted bits = converting the patched bits
    assert np.array_equal(d.cpu().numpy(), orc.g128x_repack(patched, N, K))
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    b1.GroupPlan([(d, dev_u16(scales), dev_bf16(x).view(1, K), y)], layout=b1.LAYOUT_G128X).run()
    torch.cuda.synchronize()
    assert_gemv_close(y, orc.gemv(patched, scales, x, 1, N, K), abs_bound(scales, x, K), "patched g128x")
    b1.bit1_xor_patch(d, rows, N=N, K=K)
    b1.bit1_unpack_g128x(d, out=d)
    torch.cuda.synchronize()
    assert np.array_equal(d.cpu().numpy(), bits)        # removed and converted back: bit-identical


def test_sweep_8b_g128x_benchmarked_launch_sampled_parity(orc):
    """The benchmark's headline configuration: the 8B-class sweep's bits
    converted once to g128x, one grouped launch per step, bf16 output;
    every matrix checked on sampled rows against the oracle on the canonical
    bits, and equal bit for bit to the canonical plan's output."""
    sw = Sweep(synth.sweep_8b(), seed0=0, batch=1, y_dtype=b1.BF16).fill()
    canon = sw.group_plan()
    canon.run()
    torch.cuda.synchronize()
    y_canon = sw.y.clone()
    sw.to_g128x()
    plan = sw.group_plan()
    assert plan.layout == b1.LAYOUT_G128X
    plan.run()
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    assert torch.equal(sw.y, y_canon)
    rng = np.random.default_rng(7300)
    for i, m in enumerate(sw.mats):
        rows = np.unique(np.concatenate([rng.choice(m.N, min(16, m.N), replace=False), [0, m.N - 1]]))
        hb, hs, hx = sw.host_matrix(i)
        ref = orc.gemv_select(hb, hs, hx, 1, m.N, m.K, rows)
        got = sw.y_of(i)[:, torch.from_numpy(rows).cuda()]
        assert_gemv_close(got, ref, abs_bound(hs[rows], hx, m.K), f"g128x sweep matrix {i} ({m.name})")


def test_dependent_grouped_launches_with_pdl(orc):
    """Two grouped launches in a row with programmatic dependent launch, the
    second reading the first one's output as its activations (a decode
    step's dependence): the second kernel starts streaming its weights early
    but reads x only after the first has completed."""
    N, K = 4096, 4096
    b_a, s_a = synth.matrix(N, K, 7400)
    b_b, s_b = synth.matrix(N, K, 7401)
    da, db = b1.bit1_repack_g128x(dev_u8(b_a)), b1.bit1_repack_g128x(dev_u8(b_b))
    xa = dev_bf16(synth.x_for(1, K, 7402)).view(1, K)
    h = torch.randn((1, K), device="cuda").bfloat16()        # stale contents the second launch must not see
    yb = torch.empty((1, N), dtype=torch.float32, device="cuda")
    pa = b1.GroupPlan([(da, dev_u16(s_a), xa, h)], layout=b1.LAYOUT_G128X)
    pb = b1.GroupPlan([(db, dev_u16(s_b), h, yb)], layout=b1.LAYOUT_G128X)
    for step in range(3):
        pa.run(flags=b1.FLAG_PDL)
        pb.run(flags=b1.FLAG_PDL)
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    xh = xa.view(torch.int16).cpu().numpy().view(np.uint16).reshape(1, K)
    assert_gemv_close(h, orc.gemv(b_a, s_a, xh, 1, N, K), abs_bound(s_a, xh, K), "first launch")
    hh = h.view(torch.int16).cpu().numpy().view(np.uint16).reshape(1, K)
    assert_gemv_close(yb, orc.gemv(b_b, s_b, hh, 1, N, K), abs_bound(s_b, hh, K), "second launch on the first's output")
