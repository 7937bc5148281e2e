"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/bit1.h declares, and rejects bad arguments on the host
before any CUDA call (so these run on a machine without a device)."""
import ctypes
import os
import re

import pytest

import bit_weight_gemv_sign_b300 as b1
from bit_weight_gemv_sign_b300 import build as b1build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bit1.h")


@pytest.fixture(scope="module")
def lib():
    b1build.build()
    return b1.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(bit1_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = _declared_functions()
    for want in ("bit1_pack", "bit1_gemv", "bit1_gemv_ex", "bit1_xor_patch",
                 "bit1_gemv_workspace_bytes", "bit1_status_str", "bit1_ternary_planes",
                 "bit1_gemv_ternary", "bit1_ternary_combine"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(b1.library_path())
    missing = [n for n in _declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_status_strings(lib):
    for s in range(6):
        assert len(b1.bit1_status_str(s)) >= 2
    assert "unknown" in b1.bit1_status_str(99)
    assert "sm_103a" in b1.bit1_version()


def test_pack_flags_mapping(lib):
    assert b1.bit1_pack_flags_status(0) == b1.OK
    assert b1.bit1_pack_flags_status(1) == b1.ENAN
    assert b1.bit1_pack_flags_status(2) == b1.ERANGE
    assert b1.bit1_pack_flags_status(3) == b1.ENAN
    assert b1.bit1_pack_flags_status(4) == b1.ERANGE      # ternary code out of range
    assert b1.bit1_pack_flags_status(8) == b1.ERANGE      # packed ternary byte out of range


FAKE = 1 << 20  # aligned non-null address: never dereferenced by the checks below


def test_gemv_rejects_bad_shapes_on_host(lib):
    f = lib.bit1_gemv_ex
    for B, N, K in ((1, 1, 100), (1, 1, 0), (0, 8, 128), (1, 0, 128), (1, 8, -128), (1, 8, 129)):
        assert f(FAKE, FAKE, FAKE, B, N, K, FAKE, b1.F32, None, 0, 0, 0, None) == b1.ESHAPE


def test_gemv_rejects_bad_pointers_and_types_on_host(lib):
    f = lib.bit1_gemv_ex
    assert f(None, FAKE, FAKE, 1, 8, 128, FAKE, b1.F32, None, 0, 0, 0, None) == b1.EINVAL
    assert f(FAKE, FAKE, FAKE, 1, 8, 128, None, b1.F32, None, 0, 0, 0, None) == b1.EINVAL
    assert f(FAKE + 2, FAKE, FAKE, 1, 8, 128, FAKE, b1.F32, None, 0, 0, 0, None) == b1.EINVAL
    assert f(FAKE, FAKE, FAKE + 8, 1, 8, 128, FAKE, b1.F32, None, 0, 0, 0, None) == b1.EINVAL
    assert f(FAKE, FAKE, FAKE, 1, 8, 128, FAKE, 7, None, 0, 0, 0, None) == b1.EINVAL
    assert f(FAKE, FAKE, FAKE, 1, 8, 128, FAKE, b1.F16, None, 0, 0, 0, None) == b1.EINVAL
    assert f(FAKE, FAKE, FAKE, 1, 8, 128, FAKE, b1.F32, None, 0, 99, 0, None) == b1.EINVAL
    assert f(FAKE, FAKE, FAKE, 1, 8, 128, FAKE, b1.F32, None, 0, 0, 0x80, None) == b1.EINVAL
    assert f(FAKE, FAKE, FAKE, 1, 8, 128, FAKE, b1.F32, None, 64, 0, 0, None) == b1.EINVAL


def test_gemv_variant_limits_on_host(lib):
    f = lib.bit1_gemv_ex
    # the table-lookup kernel takes batch 1 and K a multiple of 1024 up to its table limit
    assert f(FAKE, FAKE, FAKE, 2, 8, 1024, FAKE, b1.F32, None, 0, b1.LUT, 0, None) == b1.ESHAPE
    assert f(FAKE, FAKE, FAKE, 1, 8, 1152, FAKE, b1.F32, None, 0, b1.LUT, 0, None) == b1.ESHAPE


def test_pick_and_launch_counts(lib):
    assert b1.bit1_gemv_pick(1, 4096, 4096) == b1.LUT       # one projection: nibble tables
    assert b1.bit1_gemv_pick(1, 151936, 4096) == b1.LUT6    # very tall: 6-bit tables
    assert b1.bit1_gemv_pick(1, 4096, 12288) == b1.LUT
    assert b1.bit1_gemv_pick(1, 70000, 12288) == b1.LUT6
    assert b1.bit1_gemv_pick(1, 4096, 13312) == b1.LUT
    assert b1.bit1_gemv_pick(1, 5120, 17408) == b1.STREAM   # no table kernel splits K = 17 x 1024: the grouped one
    assert b1.bit1_gemv_pick(1, 4096, 1152) == b1.SIMPLE
    assert b1.bit1_gemv_pick(0, 4096, 4096) == 0
    assert b1.bit1_gemv_launches(1, 4096, 4096, b1.AUTO) == 1
    assert b1.bit1_gemv_launches(1, 4096, 100, b1.AUTO) == 0
    assert b1.bit1_gemv_workspace_bytes(1, 4096, 100) == 0
    # batched: the table kernel without scratch, the tensor cores from 16 rows with it
    assert b1.bit1_gemv_pick(4, 12288, 4096) == b1.LUT6
    assert b1.bit1_gemv_pick(16, 12288, 4096) == b1.MMA     # no scratch, many rows, K <= 4096: register MMAs
    assert b1.bit1_gemv_pick(12, 4096, 4096) == b1.MMA
    assert b1.bit1_gemv_pick(11, 4096, 4096) == b1.LUT6
    assert b1.bit1_gemv_pick(16, 4096, 12288) == b1.LUT6    # K = 12288: the 6-bit tables stay faster
    ws = b1.bit1_gemv_workspace_bytes(16, 12288, 4096)
    assert ws > 0 and b1.bit1_gemv_pick(16, 12288, 4096, ws) == b1.TC
    # the measured crossover with scratch: 12288x4096 from 8 rows, N <= 8192 from 4,
    # 17408x5120 (89M weights) from 5; every batch of 2+ rows where the tables
    # cannot split K
    big = 1 << 30
    assert b1.bit1_gemv_pick(6, 12288, 4096, big) == b1.LUT6
    assert b1.bit1_gemv_pick(8, 12288, 4096, big) == b1.TC
    assert b1.bit1_gemv_pick(3, 4096, 12288, big) == b1.LUT6
    assert b1.bit1_gemv_pick(4, 4096, 12288, big) == b1.TC
    assert b1.bit1_gemv_pick(4, 17408, 5120, big) == b1.LUT6
    assert b1.bit1_gemv_pick(5, 17408, 5120, big) == b1.TC
    assert b1.bit1_gemv_pick(2, 5120, 17408, big) == b1.TC
    assert b1.bit1_gemv_pick(1, 5120, 17408, big) == b1.STREAM
    # without scratch, K = 17408 at 2-8 rows: the grouped kernel, up to 6 rows a launch
    assert b1.bit1_gemv_pick(4, 5120, 17408) == b1.MMA      # no 6-bit split, no scratch: register MMAs from 3 rows
    assert b1.bit1_gemv_pick(2, 5120, 17408) == b1.STREAM
    assert b1.bit1_gemv_launches(20, 5120, 17408, b1.MMA) == 2
    assert b1.bit1_gemv_launches(6, 5120, 17408, b1.STREAM) == 1
    assert b1.bit1_gemv_launches(8, 5120, 17408, b1.STREAM) == 2
    assert b1.bit1_gemv_launches(4, 12288, 4096, b1.LUT6) == 1
    assert b1.bit1_gemv_launches(16, 12288, 4096, b1.LUT6) >= 2
    assert b1.bit1_gemv_launches(16, 12288, 4096, b1.TC) == 2


def test_pack_rejects_on_host(lib):
    f = lib.bit1_pack
    assert f(FAKE, b1.F32, 8, 100, FAKE, FAKE, None, None) == b1.ESHAPE
    assert f(None, b1.F32, 8, 128, FAKE, FAKE, None, None) == b1.EINVAL
    assert f(FAKE, 9, 8, 128, FAKE, FAKE, None, None) == b1.EINVAL
    assert f(FAKE, b1.F32, 8, 128, FAKE + 4, FAKE, None, None) == b1.EINVAL


def test_xor_patch_range_checked_on_host(lib):
    import numpy as np
    f = lib.bit1_xor_patch
    rows = np.array([0, 5, 8], dtype=np.int32)
    assert f(FAKE, 8, 128, rows.ctypes.data, 3, None) == b1.ERANGE
    rows = np.array([-1], dtype=np.int32)
    assert f(FAKE, 8, 128, rows.ctypes.data, 1, None) == b1.ERANGE
    assert f(FAKE, 8, 128, None, 0, None) == b1.OK      # empty patch: nothing to do
    assert f(FAKE, 8, 128, None, -1, None) == b1.EINVAL
    assert f(FAKE, 8, 100, None, 0, None) == b1.ESHAPE


def test_binding_fails_loudly_without_cuda_tensors(lib):
    import torch
    x = torch.zeros(1, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        b1.bit1_gemv(torch.zeros(8, 16, dtype=torch.uint8), torch.zeros(8, 1, dtype=torch.int16), x)


def test_ternary_rejects_on_host(lib):
    f = lib.bit1_ternary_planes
    assert f(FAKE, 8, 100, FAKE, FAKE, None, None) == b1.ESHAPE
    assert f(None, 8, 128, FAKE, FAKE, None, None) == b1.EINVAL
    assert f(FAKE, 8, 128, FAKE + 4, FAKE, None, None) == b1.EINVAL
    assert f(FAKE, 8, 128, FAKE, FAKE, FAKE + 2, None) == b1.EINVAL
    g = lib.bit1_gemv_ternary
    half = 256                                        # 1 x 8 fp32, rounded up to 256
    assert g(FAKE, FAKE, FAKE, FAKE, 1, 8, 100, FAKE, b1.F32, FAKE, 2 * half, 0, 0, None) == b1.ESHAPE
    assert g(FAKE, None, FAKE, FAKE, 1, 8, 128, FAKE, b1.F32, FAKE, 2 * half, 0, 0, None) == b1.EINVAL
    assert g(FAKE, FAKE, FAKE, FAKE, 1, 8, 128, FAKE, b1.F32, None, 0, 0, 0, None) == b1.EINVAL
    assert g(FAKE, FAKE, FAKE, FAKE, 1, 8, 128, FAKE, b1.F32, FAKE, 2 * half - 1, 0, 0, None) == b1.EINVAL
    assert g(FAKE, FAKE, FAKE, FAKE, 1, 8, 128, FAKE, b1.F16, FAKE, 2 * half, 0, 0, None) == b1.EINVAL
    assert g(FAKE, FAKE, FAKE, FAKE, 2, 8, 1024, FAKE, b1.F32, FAKE, 2 * half, b1.LUT, 0, None) == b1.ESHAPE
    assert g(FAKE, FAKE, FAKE, FAKE, 1, 8, 128, FAKE, b1.F32, FAKE, 2 * half, 0, 0x80, None) == b1.EINVAL
    c = lib.bit1_ternary_combine
    assert c(FAKE, FAKE, 0, FAKE, b1.F32, None) == b1.ESHAPE
    assert c(FAKE, FAKE + 4, 8, FAKE, b1.F32, None) == b1.EINVAL
    assert c(FAKE, FAKE, 8, FAKE, b1.F16, None) == b1.EINVAL


def test_ternary_workspace_and_launch_counts(lib):
    assert b1.bit1_gemv_ternary_workspace_bytes(1, 4096, 4096) == 2 * 16384
    assert b1.bit1_gemv_ternary_workspace_bytes(3, 10, 128) == 2 * 256
    ws16 = b1.bit1_gemv_ternary_workspace_bytes(16, 12288, 4096)
    assert ws16 == 2 * 16 * 12288 * 4 + b1.bit1_gemv_workspace_bytes(16, 12288, 4096)
    assert b1.bit1_gemv_ternary_workspace_bytes(1, 8, 100) == 0
    assert b1.bit1_gemv_ternary_launches(1, 4096, 4096) == 3
    assert b1.bit1_gemv_ternary_launches(16, 12288, 4096, b1.TC) == 5
    assert b1.bit1_gemv_ternary_launches(1, 8, 100) == 0


def test_t5_rejects_on_host(lib):
    assert lib.bit1_t5_pack(FAKE, 8, 100, FAKE, None, None) == b1.ESHAPE
    assert lib.bit1_t5_pack(FAKE, 8, 128, FAKE + 1, None, None) == b1.EINVAL
    assert lib.bit1_t5_to_planes(FAKE, 8, 128, FAKE, None, None, None) == b1.EINVAL
    assert lib.bit1_t5_to_planes(FAKE, 0, 128, FAKE, FAKE, None, None) == b1.ESHAPE
    g = lib.bit1_gemv_t5
    assert g(FAKE, FAKE, FAKE, 1, 8, 100, FAKE, b1.F32, None) == b1.ESHAPE
    assert g(FAKE, FAKE, None, 1, 8, 128, FAKE, b1.F32, None) == b1.EINVAL
    assert g(FAKE, FAKE, FAKE, 1, 8, 128, FAKE, b1.F16, None) == b1.EINVAL
    assert b1.bit1_gemv_t5_launches(1, 8, 128) == 1
    assert b1.bit1_gemv_t5_launches(17, 8, 128) == 3
    assert b1.bit1_gemv_t5_launches(1, 8, 100) == 0


def test_selftest_rejects_bad_pointer_on_host(lib):
    assert lib.bit1_selftest_wait_timeout(None, None) == b1.EINVAL
    assert lib.bit1_selftest_wait_timeout(FAKE + 2, None) == b1.EINVAL


def test_swiglu_flag_checked_on_host(lib):
    f = lib.bit1_gemv_ex
    S = b1.FLAG_SWIGLU
    assert f(FAKE, FAKE, FAKE, 1, 7, 1024, FAKE, b1.F32, None, 0, 0, S, None) == b1.ESHAPE     # odd rows
    assert f(FAKE, FAKE, FAKE, 1, 8, 1024, FAKE, b1.F32, None, 0, b1.SIMPLE, S, None) == b1.ESHAPE
    for v in (b1.LUT6, b1.SPLITK):                    # the 6-bit kernels' own limit: K a multiple of 1024
        assert f(FAKE, FAKE, FAKE, 2, 8, 1152, FAKE, b1.F32, None, 0, v, S, None) == b1.ESHAPE
    # the tensor cores take the flag at any batch, with their workspace
    assert f(FAKE, FAKE, FAKE, 1, 8, 1024, FAKE, b1.F32, None, 0, b1.TC, S, None) == b1.EINVAL
    assert f(FAKE, FAKE, FAKE, 2, 8, 1024, FAKE, b1.F32, None, 0, b1.TC, S, None) == b1.EINVAL
    assert f(FAKE, FAKE, FAKE, 2, 8, 1024, FAKE, b1.F32, None, 0, b1.LUT, S, None) == b1.ESHAPE  # batch 1 only
    assert f(FAKE, FAKE, FAKE, 2, 8, 1152, FAKE, b1.F32, None, 0, b1.STREAM, S, None) == b1.ESHAPE  # K % 1024
    # AUTO at 2 rows where only the warp-per-row kernel takes the shape
    assert f(FAKE, FAKE, FAKE, 2, 8, 1152, FAKE, b1.F32, None, 0, b1.AUTO, S, None) == b1.ESHAPE
    assert f(FAKE, FAKE, FAKE, 1, 8, 1152, FAKE, b1.F32, None, 0, b1.LUT, S, None) == b1.ESHAPE
    assert f(FAKE, FAKE, FAKE, 1, 8, 1024, FAKE, b1.F32, None, 0, 0, S | 4, None) == b1.EINVAL
    g = lib.bit1_gemv_ternary                     # pairs formed in the combine: only N must be even
    assert g(FAKE, FAKE, FAKE, FAKE, 1, 7, 128, FAKE, b1.F32, FAKE, 512, 0, S, None) == b1.ESHAPE
    assert g(FAKE, FAKE, FAKE, FAKE, 1, 8, 128, FAKE, b1.F32, FAKE, 512, 0, S | 4, None) == b1.EINVAL


def test_group_plan_epilogue_checked_on_host(lib):
    import numpy as np
    n = lib.bit1_group_plan_bytes(1)
    raw = np.zeros(n + 128, dtype=np.uint8)
    off = (-raw.ctypes.data) % 128
    plan = raw[off:off + n]
    for N, epi in ((63, b1.EPI_SWIGLU), (64, 2), (64, -1)):
        p = b1._Problem(FAKE, FAKE, FAKE, FAKE, N, 1024, b1.F32, epi)
        assert lib.bit1_group_plan(ctypes.byref(p), 1, plan.ctypes.data, n) == b1.ESHAPE, (N, epi)


def test_group_tc_plan_checked_on_host(lib):
    """Tensor-core grouped plans: sizes and argument checks, all before any
    CUDA call (a fake, aligned workspace address is never dereferenced)."""
    import numpy as np
    assert lib.bit1_group_tc_plan_bytes(0) == 0
    n = lib.bit1_group_tc_plan_bytes(3)
    assert n >= 3 * 256 + 128
    raw = np.zeros(n + 128, dtype=np.uint8)
    off = (-raw.ctypes.data) % 128
    plan = raw[off:off + n]
    probs = (b1._Problem * 2)(b1._Problem(FAKE, FAKE, FAKE, FAKE, 300, 4096, b1.F32, 0),
                              b1._Problem(FAKE, FAKE, FAKE, FAKE, 64, 17408, b1.BF16, b1.EPI_SWIGLU))
    # x' [Bp][K] fp16 and Bp scale factors per problem, each rounded up to 256 bytes
    for B, Bp in ((1, 16), (5, 16), (16, 16), (17, 32), (64, 64)):
        want = sum(Bp * K * 2 + (Bp * 4 + 255) // 256 * 256 for K in (4096, 17408))
        assert lib.bit1_group_tc_workspace_bytes(probs, 2, B) == want, B
    for B in (0, 65, -1):
        assert lib.bit1_group_tc_workspace_bytes(probs, 2, B) == 0
    ws = lib.bit1_group_tc_workspace_bytes(probs, 2, 16)
    call = lambda B=16, w=FAKE, wsz=ws, pl=plan.ctypes.data, nb=n, pr=probs, c=2: \
        lib.bit1_group_plan_tc(pr, c, B, w, wsz, pl, nb)
    assert call(B=0) == b1.ESHAPE and call(B=65) == b1.ESHAPE
    assert call(w=FAKE + 128) == b1.EINVAL                     # workspace not 256-byte aligned
    assert call(w=None) == b1.EINVAL
    assert call(wsz=ws - 1) == b1.EINVAL                        # workspace too small
    assert call(nb=lib.bit1_group_tc_plan_bytes(2) - 1) == b1.EINVAL   # plan buffer too small
    assert call(pl=plan.ctypes.data + 8, nb=n - 8) == b1.EINVAL  # plan not 128-byte aligned
    assert call(c=0) == b1.EINVAL
    bad = (b1._Problem * 1)(b1._Problem(FAKE, FAKE, FAKE, FAKE, 300, 1152, b1.F32, 0))   # K % 1024 != 0
    assert lib.bit1_group_tc_workspace_bytes(bad, 1, 16) == 0
    assert call(pr=bad, c=1) == b1.ESHAPE
    odd = (b1._Problem * 1)(b1._Problem(FAKE, FAKE, FAKE, FAKE, 63, 1024, b1.F32, b1.EPI_SWIGLU))
    assert call(pr=odd, c=1) == b1.ESHAPE


def test_group_plan_mma_checked_on_host(lib):
    """The MMA-engine grouped plan: B outside [1, 16] and bad problems are
    refused on the host, before any CUDA call."""
    import numpy as np
    n = lib.bit1_group_plan_bytes(1)
    raw = np.zeros(n + 128, dtype=np.uint8)
    off = (-raw.ctypes.data) % 128
    plan = raw[off:off + n]
    p = b1._Problem(FAKE, FAKE, FAKE, FAKE, 300, 4096, b1.F32, 0)
    for B in (0, 17, -3):
        assert lib.bit1_group_plan_mma(ctypes.byref(p), 1, B, plan.ctypes.data, n) == b1.ESHAPE, B
    bad = b1._Problem(FAKE, FAKE, FAKE, FAKE, 300, 1152, b1.F32, 0)       # K % 1024 != 0
    assert lib.bit1_group_plan_mma(ctypes.byref(bad), 1, 4, plan.ctypes.data, n) == b1.ESHAPE
    assert lib.bit1_group_plan_mma(ctypes.byref(p), 1, 4, plan.ctypes.data, n - 1) == b1.EINVAL
    assert lib.bit1_group_plan_mma(ctypes.byref(p), 0, 4, plan.ctypes.data, n) == b1.EINVAL


def test_sweep_feeds_swiglu_output_to_the_next_matrix():
    """Host wiring of the fused chain: the matrix after a SwiGLU matrix reads
    its h; a grouped plan over such a sweep is refused (its problems run
    concurrently); a mismatched width is refused."""
    from bit_weight_gemv_sign_b300 import synth
    from bit_weight_gemv_sign_b300.sweep import Sweep
    mats = [synth.Mat("gate_up", 256, 1024, swiglu=True), synth.Mat("down", 64, 128), synth.Mat("o", 64, 1024)]
    sw = Sweep(mats, device="cpu", feed_swiglu=True)
    assert sw.fed == {1: 0}
    assert sw.x_of(1).data_ptr() == sw.y_of(0).data_ptr() and sw.x_of(1).shape == (1, 128)
    assert sw.y_of(0).shape == (1, 128) and sw.x_of(2).data_ptr() != sw.y_of(1).data_ptr()
    with pytest.raises(ValueError):
        sw.group_plan()
    with pytest.raises(ValueError):
        Sweep([synth.Mat("gate_up", 256, 1024, swiglu=True), synth.Mat("down", 64, 256)], device="cpu",
              feed_swiglu=True)
    with pytest.raises(ValueError):
        Sweep(mats, device="cpu", feed_swiglu=True, y_dtype=b1.F32)
    assert sum(m.N * m.K for m in synth.decode_chain_8b_fused()) == sum(m.N * m.K for m in synth.sweep_8b())
    assert sum(m.N * m.K for m in synth.sweep_8b_fused_mlp()) == sum(m.N * m.K for m in synth.sweep_8b())


def test_ternary_sweep_refuses_swiglu_matrices():
    from bit_weight_gemv_sign_b300 import synth
    from bit_weight_gemv_sign_b300.sweep import TernarySweep
    with pytest.raises(ValueError):
        TernarySweep([synth.Mat("gate_up", 256, 1024, swiglu=True)], device="cpu")


def test_g128x_conversion_and_plan_layout_rejected_on_host(lib):
    f = ctypes.c_void_p(FAKE)
    assert lib.bit1_repack_g128x(f, 4, 120, f, None) == b1.ESHAPE                     # K % 128
    assert lib.bit1_repack_g128x(ctypes.c_void_p(FAKE + 8), 4, 128, f, None) == b1.EINVAL   # misaligned
    assert lib.bit1_unpack_g128x(None, 4, 128, f, None) == b1.EINVAL                  # null
    assert lib.bit1_unpack_g128x(f, 0, 128, f, None) == b1.ESHAPE                     # no rows
    assert lib.bit1_group_plan_ex(None, 1, 1, 7, None, 0) == b1.EINVAL                # layout value
