"""Non-finite activations through every kernel family, against the oracle: a
+-Inf input makes every output of its batch row +-Inf (the sign of that
weight), a NaN input makes them NaN; other batch rows stay finite and within
the tolerance."""
import numpy as np
import pytest
import torch

import bit_weight_gemv_sign_b300 as b1
from bit_weight_gemv_sign_b300 import synth
from tests.helpers import abs_bound, assert_gemv_close, dev_bf16, dev_u8, dev_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    b1.load()


def _inputs(N, K, B, seed):
    bits, scales = synth.matrix(N, K, seed)
    xf = torch.from_numpy(synth.x_for(B, K, seed).view(np.int16)).view(torch.bfloat16).float().numpy().reshape(B, K)
    xf[0, 300] = np.inf
    if B > 1:
        xf[1, 1000] = -np.inf
    if B > 2:
        xf[2, 77] = np.nan
    return bits, scales, synth.to_bf16_bits(xf)


def _compare(y, ref, bound, what):
    yg = y.detach().float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    assert np.array_equal(np.isnan(yg), np.isnan(ref)), f"{what}: NaN pattern"
    inf = np.isinf(ref)
    assert np.array_equal(np.isinf(yg), inf), f"{what}: Inf pattern"
    assert np.array_equal(np.sign(yg[inf]), np.sign(ref[inf])), f"{what}: Inf signs"
    fin = np.isfinite(ref)
    rows = np.where(fin.all(axis=1))[0]
    if rows.size:
        assert_gemv_close(y[torch.from_numpy(rows).to(y.device)], ref[rows], bound[rows], what)


@pytest.mark.parametrize("variant,B", [(b1.LUT6, 1), (b1.LUT, 1), (b1.SIMPLE, 1), (b1.STREAM, 1),
                                       (b1.LUT6, 4), (b1.SIMPLE, 3), (b1.TC, 16)])
def test_non_finite_activations(orc, variant, B):
    N, K = 512, 4096
    bits, scales, x = _inputs(N, K, B, 9000 + B)
    ref = orc.gemv(bits, scales, x, B, N, K)
    assert np.isinf(ref[0]).all() and (B < 3 or np.isnan(ref[2]).all())
    ws = torch.empty(max(b1.bit1_gemv_workspace_bytes(max(B, 16), N, K), 256), dtype=torch.uint8, device="cuda")
    with np.errstate(invalid="ignore"):
        bound = abs_bound(scales, x, K)     # finite on the rows without non-finite inputs
    for ydt in (b1.F32, b1.BF16):
        y = b1.bit1_gemv_ex(dev_u8(bits), dev_u16(scales), dev_bf16(x).view(B, K), y_dtype=ydt,
                            workspace=ws, variant=variant, N=N, K=K)
        torch.cuda.synchronize()
        _compare(y, ref, bound, f"variant {variant} B={B} y_dtype={ydt}")
    assert b1.bit1_device_wait_timeouts() == 0


@pytest.mark.parametrize("engine,B", [("mma", 5), ("mma", 12), ("tc", 5), ("tc", 16)])
def test_non_finite_activations_grouped_engines(orc, engine, B):
    """The same rows through the batched grouped engines (register-sourced
    MMAs, tcgen05 plan): a non-finite input must not hide the other batch
    rows' products (each row has its own prescale), and its own row follows
    the oracle's Inf / NaN pattern."""
    N, K = 512, 4096
    bits, scales, x = _inputs(N, K, B, 9100 + B)
    ref = orc.gemv(bits, scales, x, B, N, K)
    with np.errstate(invalid="ignore"):
        bound = abs_bound(scales, x, K)
    for ydt in (b1.F32, b1.BF16):
        y = torch.empty((B, N), dtype=torch.bfloat16 if ydt == b1.BF16 else torch.float32, device="cuda")
        plan = b1.GroupPlan([(dev_u8(bits), dev_u16(scales), dev_bf16(x).view(B, K), y)], B=B,
                            mma=engine == "mma", tensor_cores=engine == "tc")
        plan.run()
        torch.cuda.synchronize()
        _compare(y, ref, bound, f"grouped {engine} B={B} y_dtype={ydt}")
    assert b1.bit1_device_wait_timeouts() == 0
