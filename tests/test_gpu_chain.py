"""The persistent dependent chain (bit1_chain_plan + bit1_gemv_chain): a decode
step's products in data order in one cooperative launch, with a grid-wide
barrier between stages.  Every row is computed with the arithmetic of the
single-launch nibble-table kernel, so the chain must reproduce, bit for bit,
the same stages run one by one with BIT1_GEMV_LUT (themselves checked against
the oracle elsewhere); the first stage of each chain is also checked against
the oracle here."""
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


def _stage_by_stage(stages):
    for bits, scales, x, y, epi in stages:
        b1.bit1_gemv_ex(bits, scales, x.view(1, -1), y=y, variant=b1.LUT,
                        flags=b1.FLAG_PDL | (b1.FLAG_SWIGLU if epi == b1.EPI_SWIGLU else 0),
                        N=bits.shape[0], K=x.numel())


@pytest.mark.parametrize("ydt", [b1.BF16, b1.F32])
def test_chain_where_every_stage_reads_the_previous_output(orc, ydt):
    """Six 2048 x 2048 stages, each reading the previous stage's y (bf16), then
    a SwiGLU stage and a stage reading its h: every output must match the
    stage-by-stage launches exactly, and stage 0 the oracle."""
    D = 2048
    stages, host = [], []
    x0 = dev_bf16(synth.x_for(1, D, 5000)).view(D)
    x = x0
    for i in range(6):
        bits, scales = synth.matrix(D, D, 5001 + i)
        host.append((bits, scales))
        y = torch.empty((1, D), dtype=torch.bfloat16, device="cuda")
        stages.append((dev_u8(bits), dev_u16(scales), x, y, b1.EPI_NONE))
        x = y.view(D)
    gb, gs = synth.matrix(2 * D, D, 5010)
    h = torch.empty((1, D), dtype=torch.bfloat16, device="cuda")
    stages.append((dev_u8(gb), dev_u16(gs), x, h, b1.EPI_SWIGLU))
    db_, ds_ = synth.matrix(1024, D, 5011)
    yl = torch.empty((1, 1024), dtype=torch.bfloat16 if ydt == b1.BF16 else torch.float32, device="cuda")
    stages.append((dev_u8(db_), dev_u16(ds_), h.view(D), yl, b1.EPI_NONE))

    plan = b1.ChainPlan(stages)
    plan.run()
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    got = [s[3].clone() for s in stages]
    ref0 = orc.gemv(host[0][0], host[0][1], synth.x_for(1, D, 5000), 1, D, D)
    assert_gemv_close(got[0], ref0, abs_bound(host[0][1], synth.x_for(1, D, 5000), D), "chain stage 0")
    for s in stages:
        s[3].zero_()
    _stage_by_stage(stages)
    torch.cuda.synchronize()
    for i, s in enumerate(stages):
        assert torch.equal(got[i], s[3]), f"stage {i}"
    plan.run()                                   # the barrier resets itself: a second launch agrees
    torch.cuda.synchronize()
    for i, s in enumerate(stages):
        assert torch.equal(got[i], s[3]), f"second launch, stage {i}"
    assert b1.bit1_device_wait_timeouts() == 0


def test_fused_8b_decode_chain_persistent_matches_launch_chain():
    """The full fused 8B-class decode chain (145 stages: q|k|v, o, gate|up with
    SwiGLU, down reading h, x 36, and the LM head) as one launch against the
    same chain as 145 launches of the nibble-table kernel: every output equal."""
    sw = Sweep(synth.decode_chain_8b_fused(), seed0=900, batch=1, y_dtype=b1.BF16, variant=b1.LUT,
               feed_swiglu=True).fill_device(9)
    sw.run_eager()
    torch.cuda.synchronize()
    ref = sw.y.clone()
    sw.y.zero_()
    plan = sw.chain_plan()
    plan.run()
    torch.cuda.synchronize()
    assert b1.bit1_device_wait_timeouts() == 0
    assert torch.equal(sw.y, ref)


def test_chain_rejects_bad_stages():
    D = 1024
    bits, scales = synth.matrix(D, D, 5100)
    db, ds = dev_u8(bits), dev_u16(scales)
    x = dev_bf16(synth.x_for(1, D, 5100)).view(D)
    y = torch.empty((1, D), device="cuda")
    with pytest.raises(b1.Bit1Error) as e:                 # x overlapping its own y
        b1.ChainPlan([(db, ds, y.view(torch.bfloat16).view(-1)[:D], y, b1.EPI_NONE)])
    assert e.value.status == b1.EINVAL
    with pytest.raises(b1.Bit1Error) as e:                 # odd row count with SwiGLU
        b1.ChainPlan([(db[:D - 1], ds[:D - 1], x, y, b1.EPI_SWIGLU)])
    assert e.value.status == b1.ESHAPE
    xl = dev_bf16(synth.x_for(1, 14336, 5101)).view(-1)    # K beyond the table kernel
    bl, sl = synth.matrix(8, 14336, 5102)
    with pytest.raises(b1.Bit1Error) as e:
        b1.ChainPlan([(dev_u8(bl), dev_u16(sl), xl, torch.empty((1, 8), device="cuda"), b1.EPI_NONE)])
    assert e.value.status == b1.ESHAPE
