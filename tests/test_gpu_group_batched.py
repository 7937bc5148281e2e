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
from tests.helpers import abs_bound, assert_gemv_close, dev_bf16, dev_u8, dev_u16

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
