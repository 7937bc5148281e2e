"""Grouped launch with several batch rows per problem (the verify pass of a
speculative drafter): every problem of one launch multiplies B rows of its
own activations.  Against the CPU oracle on mixed shapes (K with one and with
several chunks, ragged N), fp32 and bf16 output, B = 2 .. 6; the full
8B-class sweep at B = 5 on sampled rows of every matrix."""
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


SHAPES = [(1000, 4096), (64, 1024), (2049, 5120), (300, 12288), (700, 17408), (1, 2048), (4096, 4096)]


def _problems(B, seed, ydt):
    host, probs = [], []
    for i, (N, K) in enumerate(SHAPES):
        bits, scales = synth.matrix(N, K, seed + i)
        x = synth.x_for(B, K, seed + i)
        y = torch.empty((B, N), dtype=torch.bfloat16 if ydt == b1.BF16 else torch.float32, device="cuda")
        host.append((bits, scales, x))
        probs.append((dev_u8(bits), dev_u16(scales), dev_bf16(x).view(B, K), y))
    return host, probs


@pytest.mark.parametrize("B", [2, 3, 5, 6])
@pytest.mark.parametrize("ydt", [b1.F32, b1.BF16])
def test_grouped_batched_matches_oracle(orc, B, ydt):
    host, probs = _problems(B, 9100 + 10 * B + ydt, ydt)
    plan = b1.GroupPlan(probs, B=B)
    plan.run()
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    for (N, K), (bits, scales, x), (_, _, _, y) in zip(SHAPES, host, probs):
        ref = orc.gemv(bits, scales, x, B, N, K)
        assert_gemv_close(y, ref, abs_bound(scales, x, K), f"grouped B={B} N={N} K={K} y={ydt}")
    first = [p[3].clone() for p in probs]
    plan.run(flags=b1.FLAG_PDL)
    torch.cuda.synchronize()
    for a, p in zip(first, probs):
        assert torch.equal(a, p[3])


def test_grouped_batch_limit():
    _, probs = _problems(1, 9200, b1.F32)
    with pytest.raises(b1.Bit1Error) as e:
        b1.GroupPlan(probs[:1], B=7)
    assert e.value.status == b1.ESHAPE


def _sample_rows(N, count, seed):
    rows = np.random.default_rng(seed).choice(N, min(count, N), replace=False)
    return np.unique(np.concatenate([rows, [0, N - 1]])).astype(np.int64)


def test_verify_sweep_8b_b5_sampled_parity(orc):
    """The benchmarked verify configuration: all 253 matrices, 5 rows each, one
    grouped launch, bf16 output."""
    sw = Sweep(synth.sweep_8b(), seed0=700, batch=5, y_dtype=b1.BF16).fill()
    plan = sw.group_plan()
    plan.run()
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    for i in range(len(sw.mats)):
        m = sw.mats[i]
        hb, hs, hx = sw.host_matrix(i)
        rows = _sample_rows(m.N, 8, 3000 + i)
        ref = orc.gemv_select(hb, hs, hx, 5, m.N, m.K, rows)
        got = sw.y_of(i)[:, torch.from_numpy(rows).cuda()]
        assert_gemv_close(got, ref, abs_bound(hs[rows], hx, m.K), f"verify sweep matrix {i} ({m.name})")


# ---------------------------------------------------------------- MMA engine
MMA_SHAPES = SHAPES + [(514, 8192)]      # the SwiGLU pair: two (B <= 8) or four (B > 8) K chunks


def _mma_problems(B, seed, ydt, swiglu_last=True):
    host, probs = [], []
    yt = torch.bfloat16 if ydt == b1.BF16 else torch.float32
    for i, (N, K) in enumerate(MMA_SHAPES):
        bits, scales = synth.matrix(N, K, seed + i)
        x = synth.x_for(B, K, seed + i)
        epi = b1.EPI_SWIGLU if (swiglu_last and i == len(MMA_SHAPES) - 1) else b1.EPI_NONE
        out = N // 2 if epi == b1.EPI_SWIGLU else N
        host.append((bits, scales, x, epi))
        probs.append((dev_u8(bits), dev_u16(scales), dev_bf16(x).view(B, K),
                      torch.full((B, out), float("nan"), dtype=yt, device="cuda"), epi))
    torch.cuda.synchronize()
    return host, probs


@pytest.mark.parametrize("B", [1, 2, 5, 8, 9, 16])
@pytest.mark.parametrize("ydt", [b1.F32, b1.BF16])
def test_grouped_mma_engine_matches_oracle(orc, B, ydt):
    """Register-sourced MMAs (bit1_group_plan_mma): one and two 8-column
    tiles, K with one and several 2048/1024-input chunks, ragged N, a SwiGLU
    pair; against the oracle, and bit-identical on a second (PDL) run."""
    host, probs = _mma_problems(B, 9300 + 10 * B + ydt, ydt)
    plan = b1.GroupPlan(probs, B=B, mma=True)
    plan.run()
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    for (N, K), (bits, scales, x, epi), pr in zip(MMA_SHAPES, host, probs):
        y = pr[3]
        bd = abs_bound(scales, x, K)
        yo = orc.gemv(bits, scales, x, B, N, K)
        if epi == b1.EPI_SWIGLU:
            h = orc.gemv_swiglu(bits, scales, x, B, N, K)
            assert_swiglu_close(y, h, yo[:, 0::2], yo[:, 1::2], bd[:, 0::2], bd[:, 1::2], f"mma SwiGLU B={B} N={N}")
        else:
            assert_gemv_close(y, yo, bd, f"mma B={B} N={N} K={K} y={ydt}")
    first = [p[3].clone() for p in probs]
    for p in probs:
        p[3].fill_(float("nan"))
    plan.run(flags=b1.FLAG_PDL)
    torch.cuda.synchronize()
    for a, p in zip(first, probs):
        assert torch.equal(a, p[3])


def test_grouped_mma_engine_limits():
    _, probs = _problems(1, 9400, b1.F32)
    with pytest.raises(b1.Bit1Error) as e:
        b1.GroupPlan(probs[:1], B=17, mma=True)
    assert e.value.status == b1.ESHAPE
    with pytest.raises(ValueError):
        b1.GroupPlan(probs[:1], B=2, mma=True, layout=b1.LAYOUT_G128X)


@pytest.mark.parametrize("B", [5, 16])
def test_verify_sweep_8b_mma_sampled_parity(orc, B):
    """The 8B-class sweep on the MMA engine, B rows per matrix, bf16 output:
    sampled rows of every matrix against the oracle."""
    sw = Sweep(synth.sweep_8b(), seed0=710 + B, batch=B, y_dtype=b1.BF16).fill()
    plan = sw.group_plan(mma=True)
    plan.run()
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    for i in range(len(sw.mats)):
        m = sw.mats[i]
        hb, hs, hx = sw.host_matrix(i)
        rows = _sample_rows(m.N, 6, 3100 + i)
        ref = orc.gemv_select(hb, hs, hx, B, m.N, m.K, rows)
        got = sw.y_of(i)[:, torch.from_numpy(rows).cuda()]
        assert_gemv_close(got, ref, abs_bound(hs[rows], hx, m.K), f"mma sweep B={B} matrix {i} ({m.name})")
