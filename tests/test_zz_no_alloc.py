"""The allocation-free tensor-core entry point (bit1_gemv_tc_noalloc) against
the workspace entry point (bit1_gemv_ex with BIT1_GEMV_TC) on the same
inputs, two calls in a row, plus its host-side size limit.  Collected last so
that it also runs after every other test in the same process."""
import ctypes

import numpy as np
import pytest
import torch

import bit_weight_gemv_sign_b300 as b1
from bit_weight_gemv_sign_b300 import synth
from tests.helpers import abs_bound, assert_gemv_close, assert_swiglu_close, dev_bf16, dev_u8, dev_u16

NOALLOC_SCRATCH_BYTES = 4 * 1024 * 1024 + 4096   # BIT1_NOALLOC_SCRATCH_BYTES in bit1.h


def test_noalloc_rejects_oversized_shapes_on_host():
    """K = 33792 at batch 64 needs more than the static scratch: rejected
    before any CUDA call (runs without a GPU)."""
    lib = b1.load()
    fake = ctypes.c_void_p(16)
    st = lib.bit1_gemv_tc_noalloc(fake, fake, fake, 64, 256, 33792, fake, b1.F32, 0, None)
    assert st == b1.ESHAPE
    # K not a multiple of 1024 is outside the tensor-core kernel
    st = lib.bit1_gemv_tc_noalloc(fake, fake, fake, 16, 256, 1152, fake, b1.F32, 0, None)
    assert st == b1.ESHAPE
    # the same K fits at batch 16: the need is 2 * 16 * K + 256 bytes
    assert 2 * 16 * 33792 + 256 <= NOALLOC_SCRATCH_BYTES


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    b1.load()
    cases = [(4096, 4096, 32, 9100), (1000, 2048, 16, 9101)]
    for N, K, B, seed in cases:
        bits, scales = synth.matrix(N, K, seed)
        d_bits, d_scales = dev_u8(bits), dev_u16(scales)
        ws = torch.empty(b1.bit1_gemv_workspace_bytes(B, N, K), dtype=torch.uint8, device="cuda")
        for call in range(2):   # two calls in a row, different activations
            x = dev_bf16(synth.x_for(B, K, seed + 17 * call)).view(B, K)
            ref = b1.bit1_gemv_ex(d_bits, d_scales, x, workspace=ws, variant=b1.TC, N=N, K=K)
            got = b1.bit1_gemv_tc_noalloc(d_bits, d_scales, x, N=N, K=K)
            torch.cuda.synchronize()
            assert torch.equal(got, ref), f"N={N} K={K} B={B} call {call}"
            assert torch.isfinite(got).all()
    assert b1.bit1_device_wait_timeouts() == 0


def _same_mode_workspace():
    """A caller workspace of exactly the static array's size: the workspace
    entry point then stages the batch the same way as the allocation-free one
    (all chunks at once when they fit, else one 64-row chunk at a time), so
    the two results must agree bit for bit."""
    return torch.empty(NOALLOC_SCRATCH_BYTES, dtype=torch.uint8, device="cuda")


@pytest.mark.gpu
@pytest.mark.parametrize("N,K,B,flags,seed", [
    # every 64-row chunk of a prompt batch staged at once: 512 x 4096 fp16
    # activations plus the prescale factors fill the array to 4,196,352 of
    # its 4,198,400 bytes
    (4096, 4096, 512, 0, 9200),
    # too large to stage at once (6.3 MB): one chunk at a time, the array
    # reused by each of the three chunks in turn
    (1024, 16384, 192, 0, 9201),
    # gate/up pairs with the SwiGLU epilogue, bf16 output
    (2048, 4096, 96, b1.FLAG_SWIGLU, 9202),
])
def test_noalloc_large_batches_and_swiglu(N, K, B, flags, seed, orc):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    b1.load()
    bits, scales = synth.matrix(N, K, seed)
    d_bits, d_scales = dev_u8(bits), dev_u16(scales)
    ws = _same_mode_workspace()
    ydt = b1.BF16 if flags & b1.FLAG_SWIGLU else b1.F32
    for call in range(2):       # two calls in a row, different activations
        xh = synth.x_for(B, K, seed + 31 * call)
        x = dev_bf16(xh).view(B, K)
        ref = b1.bit1_gemv_ex(d_bits, d_scales, x, workspace=ws, variant=b1.TC, flags=flags, y_dtype=ydt,
                              N=N, K=K)
        got = b1.bit1_gemv_tc_noalloc(d_bits, d_scales, x, flags=flags, y_dtype=ydt, N=N, K=K)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"N={N} K={K} B={B} flags={flags} call {call}"
        # and within the oracle's tolerance on three rows of the batch
        for r in (0, B // 2, B - 1):
            xr = np.ascontiguousarray(xh.reshape(B, K)[r:r + 1])
            bound = abs_bound(scales, xr, K)
            yo = orc.gemv(bits, scales, xr, 1, N, K)
            if flags & b1.FLAG_SWIGLU:
                h = orc.gemv_swiglu(bits, scales, xr, 1, N, K)
                assert_swiglu_close(got[r:r + 1], h, yo[:, 0::2], yo[:, 1::2], bound[:, 0::2], bound[:, 1::2],
                                    f"row {r} call {call}")
            else:
                assert_gemv_close(got[r:r + 1], yo, bound, f"row {r} call {call}")
    assert b1.bit1_device_wait_timeouts() == 0
