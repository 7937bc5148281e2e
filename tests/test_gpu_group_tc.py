"""Grouped launch on the tensor cores (bit1_group_plan_tc): every problem of
one plan multiplies B rows of its own activations with tcgen05 MMAs.  Against
the CPU oracle on mixed shapes (ragged N, one and several 256-row tiles, K
from 1024 to 17408, a SwiGLU gate/up pair), fp32 and bf16 output, B from 1
to 64 (padding to the MMA's N = 16, 32, 64); repeated runs are bit-identical;
the full 8B-class sweep at B = 5 and B = 16 on sampled rows of every
matrix."""
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


# (N, K, epilogue)
SHAPES = [(1000, 4096, b1.EPI_NONE), (64, 1024, b1.EPI_NONE), (513, 5120, b1.EPI_NONE),
          (300, 12288, b1.EPI_NONE), (700, 17408, b1.EPI_NONE), (1, 2048, b1.EPI_NONE),
          (514, 2048, b1.EPI_SWIGLU), (256, 1024, b1.EPI_NONE)]


def _problems(B, seed, ydt):
    host, probs = [], []
    yt = torch.bfloat16 if ydt == b1.BF16 else torch.float32
    for i, (N, K, epi) in enumerate(SHAPES):
        bits, scales = synth.matrix(N, K, seed + i)
        x = synth.x_for(B, K, seed + i)
        out = N // 2 if epi == b1.EPI_SWIGLU else N
        host.append((bits, scales, x))
        probs.append((dev_u8(bits), dev_u16(scales), dev_bf16(x).view(B, K),
                      torch.full((B, out), float("nan"), dtype=yt, device="cuda"), epi))
    torch.cuda.synchronize()
    return host, probs


def _rows(N, count, seed):
    rows = np.random.default_rng(seed).choice(N, min(count, N), replace=False)
    return np.unique(np.concatenate([rows, [0, N - 1]])).astype(np.int64)


def _check(orc, host, probs, B, what):
    for (N, K, epi), (bits, scales, x), pr in zip(SHAPES, host, probs):
        y = pr[3]
        if epi == b1.EPI_SWIGLU:
            yo = orc.gemv(bits, scales, x, B, N, K)
            h = orc.gemv_swiglu(bits, scales, x, B, N, K)
            bd = abs_bound(scales, x, K)
            assert_swiglu_close(y, h, yo[:, 0::2], yo[:, 1::2], bd[:, 0::2], bd[:, 1::2], f"{what} SwiGLU N={N}")
        elif N * K * B <= 64 * 4096 * 1000:
            assert_gemv_close(y, orc.gemv(bits, scales, x, B, N, K), abs_bound(scales, x, K), f"{what} N={N} K={K}")
        else:
            rows = _rows(N, 48, N + K)
            ref = orc.gemv_select(bits, scales, x, B, N, K, rows)
            got = y[:, torch.from_numpy(rows).cuda()]
            assert_gemv_close(got, ref, abs_bound(scales[rows], x, K), f"{what} N={N} K={K} (sampled rows)")


@pytest.mark.parametrize("B", [1, 5, 16, 17, 40, 64])
@pytest.mark.parametrize("ydt", [b1.F32, b1.BF16])
def test_grouped_tc_matches_oracle(orc, B, ydt):
    host, probs = _problems(B, 9500 + 10 * B + ydt, ydt)
    plan = b1.GroupPlan(probs, B=B, tensor_cores=True)
    plan.run()
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    _check(orc, host, probs, B, f"tc grouped B={B} y={ydt}")
    # a second run (with PDL) writes the same bits: fixed summation order
    first = [p[3].clone() for p in probs]
    for p in probs:
        p[3].fill_(float("nan"))
    plan.run(flags=b1.FLAG_PDL)
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    for a, p in zip(first, probs):
        assert torch.equal(a, p[3])


def test_grouped_tc_batch_limit_and_layout():
    _, probs = _problems(1, 9600, b1.F32)
    with pytest.raises(b1.Bit1Error) as e:
        b1.GroupPlan(probs[:1], B=65, tensor_cores=True)
    assert e.value.status == b1.ESHAPE
    with pytest.raises(ValueError):
        b1.GroupPlan(probs[:1], B=1, tensor_cores=True, layout=b1.LAYOUT_G128X)


def test_grouped_tc_and_tables_plans_interleaved(orc):
    """A tensor-core plan and a CUDA-core plan over the same problems, run
    back to back on one stream (each plan's kind picks its kernel): both
    within tolerance of the oracle."""
    B = 4
    host, probs = _problems(B, 9700, b1.F32)
    tc = b1.GroupPlan(probs, B=B, tensor_cores=True)
    probs2 = [(p[0], p[1], p[2], torch.empty_like(p[3]), p[4]) for p in probs]
    tab = b1.GroupPlan(probs2, B=B)
    for _ in range(2):
        tc.run(flags=b1.FLAG_PDL)
        tab.run(flags=b1.FLAG_PDL)
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    _check(orc, host, probs, B, "tc interleaved")
    _check(orc, host, probs2, B, "tables interleaved")


@pytest.mark.parametrize("B", [5, 16])
def test_sweep_8b_tc_grouped_sampled_parity(orc, B):
    """The benchmarked batched configurations: all 253 matrices of the
    8B-class sweep, B rows each, one tensor-core grouped plan, bf16 output;
    sampled rows of every matrix against the oracle."""
    sw = Sweep(synth.sweep_8b(), seed0=800 + B, batch=B, y_dtype=b1.BF16).fill()
    plan = sw.group_plan(tensor_cores=True)
    plan.run()
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    for i in range(len(sw.mats)):
        m = sw.mats[i]
        hb, hs, hx = sw.host_matrix(i)
        rows = _rows(m.N, 6, 4000 + i)
        got = sw.y_of(i)[:, torch.from_numpy(rows).cuda()]
        ref = orc.gemv_select(hb, hs, hx, B, m.N, m.K, rows)
        assert_gemv_close(got, ref, abs_bound(hs[rows], hx, m.K), f"tc sweep B={B} matrix {i} ({m.name})")
