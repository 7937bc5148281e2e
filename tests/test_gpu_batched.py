"""GPU parity of the CUDA-core batched path (BIT1_GEMV_LUT6 with B > 1: 6-bit
tables per batch row, up to 8 rows per launch) against the CPU oracle on the
same seeded inputs, through the C ABI."""
import numpy as np
import pytest
import torch

import bit_weight_gemv_sign_b300 as b1
from bit_weight_gemv_sign_b300 import synth
from tests.helpers import abs_bound, assert_gemv_close, assert_swiglu_close, dev_bf16, dev_u8, dev_u16

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


def _run(bits, scales, x, N, K, B, variant=b1.LUT6, y_dtype=b1.F32, flags=0):
    y = b1.bit1_gemv_ex(dev_u8(bits), dev_u16(scales), dev_bf16(x).view(B, K), y_dtype=y_dtype,
                        variant=variant, flags=flags, N=N, K=K)
    torch.cuda.synchronize()
    return y


# one launch (B <= 8 when the tables fit), several launches (B = 9, 16), ragged
# row blocks, long K with deep cluster splits; short N (few row blocks per
# CTA) puts several warps on one block, each on part of its groups
BATCHED = [(256, 1024, 2), (300, 2048, 3), (1000, 4096, 4), (777, 4096, 5), (4100, 4096, 8),
           (513, 12288, 6), (129, 5120, 7), (3000, 4096, 16), (64, 16384, 4), (5000, 12288, 9),
           (4096, 4096, 4), (1024, 4096, 5), (2048, 12288, 3), (1, 4096, 2), (33, 1024, 8),
           (4096, 12288, 2)]


@pytest.mark.parametrize("N,K,B", BATCHED)
def test_batched_tables_match_oracle(orc, N, K, B):
    bits, scales, x = _problem(N, K, B, 8000 + N + K + B)
    ref = orc.gemv(bits, scales, x, B, N, K)
    y = _run(bits, scales, x, N, K, B)
    assert_gemv_close(y, ref, abs_bound(scales, x, K), f"lut6 N={N} K={K} B={B}")
    assert b1.bit1_device_wait_timeouts() == 0


def test_batched_auto_bf16_and_pdl(orc):
    N, K, B = 2000, 4096, 4
    bits, scales, x = _problem(N, K, B, 8101)
    assert b1.bit1_gemv_pick(B, N, K) == b1.LUT6
    ref = orc.gemv(bits, scales, x, B, N, K)
    y = _run(bits, scales, x, N, K, B, variant=b1.AUTO, y_dtype=b1.BF16)
    assert y.dtype == torch.bfloat16
    assert_gemv_close(y, ref, abs_bound(scales, x, K), "lut6 batched bf16")
    a = _run(bits, scales, x, N, K, B)
    c = _run(bits, scales, x, N, K, B, flags=b1.FLAG_PDL)
    assert torch.equal(a, c)


def test_batched_rows_independent_of_batch_size():
    """A batch row's result does not depend on the other rows of the batch
    (tables and prescales are per batch row; the row walk is the same)."""
    N, K = 1500, 4096
    bits, scales, x = _problem(N, K, 5, 8102)
    y5 = _run(bits, scales, x, N, K, 5)
    for b in range(5):
        y1 = _run(bits, scales, x[b:b + 1], N, K, 1)
        assert torch.equal(y1[0], y5[b]), f"batch row {b}"


def test_batched_row_flip_negates_exactly():
    N, K, B = 700, 4096, 4
    bits, scales, x = _problem(N, K, B, 8103)
    y = _run(bits, scales, x, N, K, B)
    flipped = bits.copy()
    flipped[[0, 31, 32, 699]] ^= 0xFF
    y2 = _run(flipped, scales, x, N, K, B)
    rows = torch.tensor([0, 31, 32, 699], device="cuda")
    assert torch.equal(y2[:, rows], -y[:, rows])


def test_splitk_names_the_cluster_split_kernel():
    """BIT1_GEMV_SPLITK runs the cluster split-K table kernel: the same bits as
    BIT1_GEMV_LUT6, and within the tolerance of the oracle."""
    N, K, B = 300, 8192, 3
    bits, scales, x = _problem(N, K, B, 8104)
    a = _run(bits, scales, x, N, K, B, variant=b1.SPLITK)
    b = _run(bits, scales, x, N, K, B, variant=b1.LUT6)
    assert torch.equal(a, b)
    assert b1.bit1_gemv_launches(B, N, K, b1.SPLITK) == b1.bit1_gemv_launches(B, N, K, b1.LUT6)


# K = 17408 (the 27B-class down projection, 17 x 1024) has no cluster split
# for the 6-bit tables; without a workspace AUTO runs it on the grouped kernel
# (BIT1_GEMV_STREAM: up to 6 rows per launch), with one on the tensor cores.
@pytest.mark.parametrize("B", [2, 4, 8])
def test_k17408_small_batch_grouped_and_tensor_cores(orc, B):
    N, K = 5120, 17408
    bits, scales, x = _problem(N, K, B, 8200 + B)
    assert b1.bit1_gemv_pick(B, N, K) == (b1.STREAM if B < 3 else b1.MMA)
    assert b1.bit1_gemv_launches(B, N, K, b1.STREAM) == (B + 5) // 6
    # with bit1_gemv_workspace_bytes of scratch AUTO takes the tensor cores
    assert b1.bit1_gemv_launches(B, N, K, b1.AUTO) == b1.bit1_gemv_launches(B, N, K, b1.TC)
    ref = orc.gemv(bits, scales, x, B, N, K)
    bound = abs_bound(scales, x, K)
    y = _run(bits, scales, x, N, K, B, variant=b1.AUTO)
    assert_gemv_close(y, ref, bound, f"AUTO without workspace N={N} K={K} B={B}")
    yb = _run(bits, scales, x, N, K, B, variant=b1.STREAM, y_dtype=b1.BF16)
    assert_gemv_close(yb, ref, bound, f"grouped bf16 N={N} K={K} B={B}")
    ws = torch.empty(b1.bit1_gemv_workspace_bytes(B, N, K), dtype=torch.uint8, device="cuda")
    assert b1.bit1_gemv_pick(B, N, K, ws.numel()) == b1.TC
    yt = b1.bit1_gemv_ex(dev_u8(bits), dev_u16(scales), dev_bf16(x).view(B, K), workspace=ws, N=N, K=K)
    torch.cuda.synchronize()
    assert_gemv_close(yt, ref, bound, f"tensor cores N={N} K={K} B={B}")
    assert b1.bit1_device_wait_timeouts() == 0


def test_stream_rows_split_with_unaligned_output_rows(orc):
    """Seven rows as 4 + 3 over N = 513 bf16 outputs: the second launch's y
    starts 4 * 513 * 2 bytes in (not 16-byte aligned)."""
    N, K, B = 513, 4096, 7
    bits, scales, x = _problem(N, K, B, 8220)
    y = _run(bits, scales, x, N, K, B, variant=b1.STREAM, y_dtype=b1.BF16)
    assert_gemv_close(y, orc.gemv(bits, scales, x, B, N, K), abs_bound(scales, x, K), "stream 4 + 3, N = 513")


def test_stream_rows_split_over_launches():
    """Seven rows run as two grouped launches, of 4 and 3 rows: the result
    equals those two launches made separately, row for row."""
    N, K = 3000, 4096
    bits, scales, x = _problem(N, K, 7, 8210)
    assert b1.bit1_gemv_launches(7, N, K, b1.STREAM) == 2
    y7 = _run(bits, scales, x, N, K, 7, variant=b1.STREAM)
    y4 = _run(bits, scales, x[:4], N, K, 4, variant=b1.STREAM)
    y3 = _run(bits, scales, x[4:], N, K, 3, variant=b1.STREAM)
    assert torch.equal(y7[:4], y4) and torch.equal(y7[4:], y3)


# (N, K, B): one chunk and several, ragged N, one and two 8-column tiles, two launches (B > 16)
MMA1_SHAPES = [(1000, 4096, 1), (300, 12288, 3), (4096, 4096, 5), (777, 5120, 8), (129, 17408, 9),
               (2048, 2048, 16), (513, 4096, 20)]


@pytest.mark.parametrize("N,K,B", MMA1_SHAPES)
def test_single_call_mma_variant_matches_oracle(orc, N, K, B):
    """bit1_gemv_ex with BIT1_GEMV_MMA: the grouped kernel's register-MMA engine
    with the one problem, fp32 and bf16 output, against the oracle."""
    bits, scales, x = _problem(N, K, B, 8300 + B)
    assert b1.bit1_gemv_launches(B, N, K, b1.MMA) == (B + 15) // 16
    ref = orc.gemv(bits, scales, x, B, N, K)
    bound = abs_bound(scales, x, K)
    for ydt in (b1.F32, b1.BF16):
        y = _run(bits, scales, x, N, K, B, variant=b1.MMA, y_dtype=ydt)
        assert_gemv_close(y, ref, bound, f"mma variant N={N} K={K} B={B} y={ydt}")
    assert b1.bit1_device_wait_timeouts() == 0


def test_single_call_mma_variant_swiglu(orc):
    N, K, B = 1026, 4096, 6
    bits, scales, x = _problem(N, K, B, 8400)
    yo = orc.gemv(bits, scales, x, B, N, K)
    h = orc.gemv_swiglu(bits, scales, x, B, N, K)
    bd = abs_bound(scales, x, K)
    y = b1.bit1_gemv_ex(dev_u8(bits), dev_u16(scales), dev_bf16(x).view(B, K), variant=b1.MMA,
                        flags=b1.FLAG_SWIGLU, N=N, K=K)
    torch.cuda.synchronize()
    assert_swiglu_close(y, h, yo[:, 0::2], yo[:, 1::2], bd[:, 0::2], bd[:, 1::2], "mma variant SwiGLU")
