"""GPU parity of the tensor-core batched kernel (BIT1_GEMV_TC, batch >= 16)
against the CPU oracle on the same seeded inputs, through the C ABI.
Tolerance: 1e-3 * sum_k |s x_k| + 1e-6 (plus bf16 output rounding)."""
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


def _problem(N, K, B, seed):
    bits, scales = synth.matrix(N, K, seed)
    x = synth.x_for(B, K, seed)
    return bits, scales, x


def _ws(B, N, K):
    n = b1.bit1_gemv_workspace_bytes(B, N, K)
    assert n > 0
    return torch.empty(n, dtype=torch.uint8, device="cuda")


def _run_tc(bits, scales, x, N, K, B, y_dtype=b1.F32, flags=0, variant=b1.TC, workspace=None):
    ws = _ws(B, N, K) if workspace is None else workspace
    y = b1.bit1_gemv_ex(dev_u8(bits), dev_u16(scales), dev_bf16(x).view(B, K), y_dtype=y_dtype,
                        workspace=ws, variant=variant, flags=flags, N=N, K=K)
    torch.cuda.synchronize()
    return y


# (N, K, B): one and several 256-row tiles, a ragged last tile, split K, batch
# padding to a multiple of 16, and batch > 64 (two launches over the weights)
TC_SHAPES = [(256, 1024, 16), (300, 1024, 16), (1000, 2048, 20), (512, 4096, 32),
             (777, 3072, 64), (129, 5120, 17), (2048, 1024, 100), (64, 17408, 16),
             (4100, 2048, 48), (1, 1024, 16)]


@pytest.mark.parametrize("N,K,B", TC_SHAPES)
def test_tc_matches_oracle(orc, N, K, B):
    bits, scales, x = _problem(N, K, B, 7000 + N + K + B)
    ref = orc.gemv(bits, scales, x, B, N, K)
    y = _run_tc(bits, scales, x, N, K, B)
    assert_gemv_close(y, ref, abs_bound(scales, x, K), f"tc N={N} K={K} B={B}")
    assert b1.bit1_device_wait_timeouts() == 0


@pytest.mark.parametrize("N,K,B", [(20000, 8192, 16), (40000, 2048, 32)])
def test_tc_long_rings_and_two_waves(orc, N, K, B):
    """Row tiles alone fill the SMs (no K split): each CTA streams all of K
    through its sign-bit ring several times over; 40000 rows need a second
    wave of CTAs.  Sampled rows against the oracle."""
    bits, scales, x = _problem(N, K, B, 7050 + N)
    y = _run_tc(bits, scales, x, N, K, B)
    rows = np.unique(np.concatenate([np.random.default_rng(N).choice(N, 384, replace=False),
                                     [0, 255, 256, N - 1]]))
    ref = orc.gemv_select(bits, scales, x, B, N, K, rows)
    assert_gemv_close(y[:, torch.from_numpy(rows).cuda()], ref, abs_bound(scales[rows], x, K),
                      f"tc N={N} K={K} B={B}")
    assert b1.bit1_device_wait_timeouts() == 0


def test_tc_bf16_output(orc):
    N, K, B = 700, 4096, 24
    bits, scales, x = _problem(N, K, B, 7101)
    ref = orc.gemv(bits, scales, x, B, N, K)
    y = _run_tc(bits, scales, x, N, K, B, y_dtype=b1.BF16)
    assert y.dtype == torch.bfloat16
    assert_gemv_close(y, ref, abs_bound(scales, x, K), "tc bf16 out")


@pytest.mark.parametrize("N,K", [(12288, 4096), (4096, 12288)])
@pytest.mark.parametrize("B", [16, 32, 64])
def test_tc_mlp_shapes_full_size(orc, N, K, B):
    """The 8B-class MLP shapes at the batch sizes of the skinny-GEMM sweep, in
    the launch configuration the benchmark times (AUTO with workspace, PDL);
    512 sampled rows (all batch rows) against the oracle, every output finite."""
    bits, scales, x = _problem(N, K, B, 7200 + N + B)
    ws = _ws(B, N, K)
    assert b1.bit1_gemv_pick(B, N, K, ws.numel()) == b1.TC
    y = _run_tc(bits, scales, x, N, K, B, flags=b1.FLAG_PDL, variant=b1.AUTO, workspace=ws)
    rows = np.random.default_rng(B).choice(N, 512, replace=False)
    rows = np.unique(np.concatenate([rows, [0, N - 1, 255, 256]]))
    ref = orc.gemv_select(bits, scales, x, B, N, K, rows)
    bound = abs_bound(scales[rows], x, K)
    assert_gemv_close(y[:, torch.from_numpy(rows).cuda()], ref, bound, f"tc full N={N} K={K} B={B}")
    assert torch.isfinite(y).all()


def test_tc_prompt_batch_512(orc):
    """A 512-row prompt batch (eight 64-row chunks, all in one launch pair):
    sampled rows of every batch row against the oracle."""
    N, K, B = 2048, 4096, 512
    bits, scales, x = _problem(N, K, B, 7250)
    y = _run_tc(bits, scales, x, N, K, B, y_dtype=b1.BF16)
    rows = np.unique(np.concatenate([np.random.default_rng(512).choice(N, 96, replace=False), [0, N - 1]]))
    ref = orc.gemv_select(bits, scales, x, B, N, K, rows)
    assert_gemv_close(y[:, torch.from_numpy(rows).cuda()], ref, abs_bound(scales[rows], x, K), "tc B=512")


def test_tc_pp512_up_gate_shape(orc):
    """The benchmarked prompt-processing configuration: the 8B up/gate shape
    12288 x 4096 at B = 512 with bit1_gemv_workspace_bytes of scratch (one
    launch pair, 128-row chunks): sampled rows of every batch row against the
    oracle."""
    N, K, B = 12288, 4096, 512
    bits, scales, x = _problem(N, K, B, 7260)
    y = _run_tc(bits, scales, x, N, K, B)
    rows = np.unique(np.concatenate([np.random.default_rng(5120).choice(N, 40, replace=False), [0, N - 1]]))
    ref = orc.gemv_select(bits, scales, x, B, N, K, rows)
    assert_gemv_close(y[:, torch.from_numpy(rows).cuda()], ref, abs_bound(scales[rows], x, K), "tc PP512")
    assert b1.bit1_device_wait_timeouts() == 0


def test_tc_row_flip_negates_exactly():
    """Negated weights flow through the same products and the same fixed
    accumulation order, so a flipped row gives the exact negation."""
    N, K, B = 600, 4096, 32
    bits, scales, x = _problem(N, K, B, 7300)
    y = _run_tc(bits, scales, x, N, K, B)
    flipped = bits.copy()
    flipped[[3, 256, 599]] ^= 0xFF
    y2 = _run_tc(flipped, scales, x, N, K, B)
    flip = torch.tensor([3, 256, 599], device="cuda")
    assert torch.equal(y2[:, flip], -y[:, flip])
    keep = torch.from_numpy(np.setdiff1d(np.arange(N), [3, 256, 599])).cuda()
    assert torch.equal(y2[:, keep], y[:, keep])


def test_tc_extreme_activation_ranges(orc):
    """Per-batch-row power-of-two prescale: rows of tiny, huge and mixed
    magnitudes stay within the tolerance."""
    N, K, B = 256, 4096, 16
    bits, scales, x = _problem(N, K, B, 7400)
    xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float().numpy().reshape(B, K)
    xf[0] *= 2.0 ** -100
    xf[1] *= 2.0 ** 100
    xf[2, ::2] *= 2.0 ** 20
    xf[2, 1::2] *= 2.0 ** -20
    xf[3] = 0.0
    xf[4, :128] *= 2.0 ** -60
    x2 = synth.to_bf16_bits(xf)
    ref = orc.gemv(bits, scales, x2, B, N, K)
    y = _run_tc(bits, scales, x2, N, K, B)
    assert_gemv_close(y, ref, abs_bound(scales, x2, K), "tc extreme ranges")
    assert float(y[3].abs().max()) == 0.0


def test_tc_subnormal_and_zero_scales(orc):
    N, K, B = 64, 2048, 16
    bits, scales, x = _problem(N, K, B, 7500)
    scales = scales.copy()
    scales[0, :] = 0x0001
    scales[1, :] = 0x03FF
    scales[2, :] = 0x0000
    ref = orc.gemv(bits, scales, x, B, N, K)
    y = _run_tc(bits, scales, x, N, K, B)
    assert_gemv_close(y, ref, abs_bound(scales, x, K), "tc special scales")
    assert float(y[:, 2].abs().max()) == 0.0


def test_tc_repeat_and_pdl_identical():
    """Two calls in a row, with and without PDL, give identical bits (the
    split-K partials are summed in a fixed order)."""
    N, K, B = 4096, 12288, 32
    bits, scales, x = _problem(N, K, B, 7600)
    a = _run_tc(bits, scales, x, N, K, B)
    b = _run_tc(bits, scales, x, N, K, B, flags=b1.FLAG_PDL)
    c = _run_tc(bits, scales, x, N, K, B)
    assert torch.equal(a, b) and torch.equal(a, c)
    assert b1.bit1_device_wait_timeouts() == 0


def test_tc_workspace_rules():
    N, K, B = 512, 2048, 16
    bits, scales, x = _problem(N, K, B, 7700)
    need = b1.bit1_gemv_workspace_bytes(B, N, K)
    assert need > 0
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(b1.Bit1Error):
        _run_tc(bits, scales, x, N, K, B, workspace=small)
    # AUTO without enough scratch picks a kernel that needs none
    assert b1.bit1_gemv_pick(B, N, K, need - 256) != b1.TC
    assert b1.bit1_gemv_pick(B, N, K, need) == b1.TC
    # K not a multiple of 1024: the tensor-core kernel refuses the shape
    assert b1.bit1_gemv_launches(B, 512, 1152, b1.TC) == 0
    # batch 1: AUTO never picks the tensor cores; batch 8 (past the measured
    # crossover) takes them when the scratch is there
    assert b1.bit1_gemv_pick(1, N, K, 1 << 30) != b1.TC
    assert b1.bit1_gemv_pick(8, N, K, 1 << 30) == b1.TC
    assert b1.bit1_gemv_pick(8, N, K, 0) != b1.TC


@pytest.mark.parametrize("B", [100, 200])
def test_tc_batch_chunks_one_launch_and_sequential(orc, B):
    """More than 64 batch rows: with bit1_gemv_workspace_bytes of scratch all
    64-row chunks run as one launch pair (grid y = chunk, a ragged last
    chunk); with only one chunk's scratch they run one pair per chunk.  Both
    against the oracle, fp32 and bf16."""
    N, K = 700, 2048
    bits, scales, x = _problem(N, K, B, 7800 + B)
    full = b1.bit1_gemv_workspace_bytes(B, N, K)
    one_chunk = b1.bit1_gemv_workspace_bytes(64, N, K)
    assert full > one_chunk
    ref = orc.gemv(bits, scales, x, B, N, K)
    bound = abs_bound(scales, x, K)
    for ws_bytes in (full, one_chunk):
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        for ydt in (b1.F32, b1.BF16):
            y = _run_tc(bits, scales, x, N, K, B, y_dtype=ydt, workspace=ws)
            assert_gemv_close(y, ref, bound, f"tc B={B} ws={ws_bytes} y={ydt}")
    assert b1.bit1_device_wait_timeouts() == 0


@pytest.mark.parametrize("N,K,B", [(12288, 4096, 256), (12288, 4096, 200), (30000, 2048, 100)])
def test_tc_wide_chunks(orc, N, K, B):
    """Shapes whose cost estimate picks 128-row chunks with one accumulator per
    half (many row tiles, B > 64; 200 rows leave a ragged last chunk, 100 rows
    a single 112-row chunk): sampled rows of every batch row against the oracle."""
    bits, scales, x = _problem(N, K, B, 7900 + B)
    for ydt in (b1.F32, b1.BF16):
        y = _run_tc(bits, scales, x, N, K, B, y_dtype=ydt)
        rows = np.unique(np.concatenate([np.random.default_rng(N + B).choice(N, 40, replace=False), [0, N - 1]]))
        ref = orc.gemv_select(bits, scales, x, B, N, K, rows)
        assert_gemv_close(y[:, torch.from_numpy(rows).cuda()], ref, abs_bound(scales[rows], x, K),
                          f"tc wide N={N} K={K} B={B} y={ydt}")
    assert b1.bit1_device_wait_timeouts() == 0
