"""Full-size decode sweeps in the launch configuration the benchmark times (one
grouped persistent launch per step, bf16 output), checked against the CPU
oracle on sampled rows of every matrix, and the 27B-class sweep with a
100-entry row patch: applied, verified against the oracle on the patched
weights, then removed and checked bit-identical to the original weights."""
import numpy as np
import pytest
import torch

import bit_weight_gemv_sign_b300 as b1
from bit_weight_gemv_sign_b300 import synth
from bit_weight_gemv_sign_b300.sweep import Sweep
from tests.helpers import abs_bound, assert_gemv_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    b1.load()


def _sample_rows(N, count, seed, extra=()):
    rows = np.random.default_rng(seed).choice(N, min(count, N), replace=False)
    return np.unique(np.concatenate([rows, [0, N - 1], np.asarray(extra, dtype=np.int64)])).astype(np.int64)


def _check_matrix(orc, sw, i, y, rows, bits=None, what=""):
    m = sw.mats[i]
    hb, hs, hx = sw.host_matrix(i)
    if bits is not None:
        hb = bits
    ref = orc.gemv_select(hb, hs, hx, 1, m.N, m.K, rows)
    got = y[:, torch.from_numpy(rows).cuda()]
    assert_gemv_close(got, ref, abs_bound(hs[rows], hx, m.K), f"{what} matrix {i} ({m.name})")


def test_sweep_8b_grouped_launch_sampled_parity(orc):
    sw = Sweep(synth.sweep_8b(), seed0=0, batch=1, y_dtype=b1.BF16).fill()
    plan = sw.group_plan()
    plan.run()
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    for i in range(len(sw.mats)):
        rows = _sample_rows(sw.mats[i].N, 24, 1000 + i)
        _check_matrix(orc, sw, i, sw.y_of(i), rows, what="8B sweep")
    # a second step over the same plan gives the same bits
    first = sw.y.clone()
    plan.run()
    torch.cuda.synchronize()
    assert torch.equal(first, sw.y)


def test_decode_chain_8b_launch_chain_sampled_parity(orc):
    """The benchmark's decode_chain configuration: the 253 products as
    dependent launches captured in one CUDA graph with programmatic dependent
    launch, every matrix checked on sampled rows."""
    sw = Sweep(synth.sweep_8b(), seed0=0, batch=1, y_dtype=b1.BF16).fill()
    sw.capture(pdl=True)
    with torch.cuda.stream(sw.stream):
        sw.replay()
    sw.stream.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    for i in range(len(sw.mats)):
        rows = _sample_rows(sw.mats[i].N, 16, 1500 + i)
        _check_matrix(orc, sw, i, sw.y_of(i), rows, what="8B launch chain")


def test_decode_chain_8b_fused_sampled_parity(orc):
    """The benchmark's decode_chain_fused configuration (145 dependent
    launches: q|k|v, o, gate|up with SwiGLU, down reading h, and the LM head,
    one CUDA graph with programmatic dependent launch).  Stages with their own
    input are checked on sampled outputs against the oracle.  A down
    projection reads the GPU's h, so the oracle runs it on its own h, rounded
    to bf16 by torch, and the tolerance adds what the two h may differ by,
    carried through |W_down|."""
    from tests.helpers import assert_swiglu_close, carried_bound, swiglu_h_tol
    sw = Sweep(synth.decode_chain_8b_fused(), seed0=0, batch=1, y_dtype=b1.BF16, feed_swiglu=True).fill()
    sw.capture(pdl=True)
    with torch.cuda.stream(sw.stream):
        sw.replay()
    sw.stream.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    h_oracle = {}
    for i, m in enumerate(sw.mats):
        hb, hs, hx = sw.host_matrix(i)
        if m.swiglu:
            units = _sample_rows(m.out, 16, 1700 + i)
            pairs = np.stack([2 * units, 2 * units + 1], 1).ravel()
            gu = orc.gemv_select(hb, hs, hx, 1, m.N, m.K, pairs)
            bd = abs_bound(hs[pairs], hx, m.K)
            assert_swiglu_close(sw.y_of(i)[:, torch.from_numpy(units).cuda()],
                                orc.gemv_swiglu_select(hb, hs, hx, 1, m.N, m.K, units),
                                gu[:, 0::2], gu[:, 1::2], bd[:, 0::2], bd[:, 1::2], f"fused chain {m.name}")
            if (i + 1) in sw.fed:                                  # the full h feeds the next stage
                yo = orc.gemv(hb, hs, hx, 1, m.N, m.K)
                ho = orc.gemv_swiglu(hb, hs, hx, 1, m.N, m.K)
                ball = abs_bound(hs, hx, m.K)
                h_oracle[i + 1] = (ho, swiglu_h_tol(yo[:, 0::2], yo[:, 1::2], ball[:, 0::2], ball[:, 1::2], ho))
        elif i in sw.fed:
            ho, dh = h_oracle[i]
            hx16 = synth.to_bf16_bits(ho.astype(np.float32))
            rows = _sample_rows(m.N, 16, 1700 + i)
            ref = orc.gemv_select(hb, hs, hx16, 1, m.N, m.K, rows)
            got = sw.y_of(i)[:, torch.from_numpy(rows).cuda()].float().cpu().numpy().astype(np.float64)
            tol = (1e-3 * abs_bound(hs[rows], hx16, m.K) + 1e-6 + carried_bound(hs[rows], dh, m.K)
                   + 2.0 ** -8 * np.abs(ref))
            assert np.all(np.abs(got - ref) <= tol), f"fused chain {m.name}"
        else:
            rows = _sample_rows(m.N, 16, 1700 + i)
            _check_matrix(orc, sw, i, sw.y_of(i), rows, what="fused chain")


def test_sweep_27b_patch_apply_verify_remove(orc):
    sw = Sweep(synth.sweep_27b(), seed0=0, batch=1, y_dtype=b1.BF16).fill()
    plan = sw.group_plan()
    plan.run()
    torch.cuda.synchronize()
    y_before = sw.y.clone()

    entries = synth.patch_entries_27b(100, 0)
    by_mat = sw.apply_patch(entries)
    torch.cuda.synchronize()
    patch_bytes = sum(sw.mats[i].K // 8 * len(rows) for i, rows in by_mat.items())
    assert len(entries) == 100 and patch_bytes > 0

    plan.run()
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    for i, rows in sorted(by_mat.items()):
        m = sw.mats[i]
        hb, _, _ = sw.host_matrix(i)
        patched = orc.xor_patch(hb, m.N, m.K, rows)
        # the device weights equal the oracle's patched bytes, bit for bit
        assert np.array_equal(sw.bits_of(i).cpu().numpy(), patched), f"patched bytes of matrix {i}"
        sample = _sample_rows(m.N, 16, 2000 + i, extra=rows)
        _check_matrix(orc, sw, i, sw.y_of(i), sample, bits=patched, what="27B patched")
        # a flipped row is the exact negation of its unpatched output
        r = torch.tensor(sorted(set(rows)), device="cuda")
        assert torch.equal(sw.y_of(i)[:, r], -sw.y_of(i, y_before)[:, r])
    # unpatched matrices: unchanged outputs
    for i in range(len(sw.mats)):
        if i not in by_mat:
            assert torch.equal(sw.y_of(i), sw.y_of(i, y_before)), f"matrix {i} changed"

    sw.apply_patch(entries)           # the same XOR removes the patch
    torch.cuda.synchronize()
    for i in sorted(by_mat):
        hb, _, _ = sw.host_matrix(i)
        assert np.array_equal(sw.bits_of(i).cpu().numpy(), hb), f"restore of matrix {i}"
    plan.run()
    torch.cuda.synchronize()
    assert torch.equal(sw.y, y_before)
