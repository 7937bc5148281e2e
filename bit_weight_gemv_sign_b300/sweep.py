"""A decode-step weight sweep: many packed 1-bit matrices resident in HBM,
each multiplied by its own activation vector, captured once into a CUDA graph
and replayed (one replay = one decode token's worth of linear layers).

The pages state that autoregressive decode reads essentially the whole weight
set for every token and that at batch 1 the time goes to memory traffic and to
kernel launch/synchronisation latency (web page "Bonsai 27B: 노트북과 폰에서
실행되는 27B급 이진 및 삼진 저비트 LLM", sections "27B 규모에서 효율은 선택이
아닌 제약" and "하이브리드 어텐션을 위한 저비트 커널").  The sweep therefore
keeps every matrix resident in one device arena and removes host launch cost
with a CUDA graph; with programmatic dependent launch each kernel starts
streaming its weights while the previous one finishes, and waits for it only
before reading its activations (the data dependence of a real decode step).
"""
from __future__ import annotations

import numpy as np
import torch

from . import synth
from . import (BF16, F32, FLAG_PDL, FLAG_SWIGLU, AUTO, EPI_NONE, EPI_SWIGLU, LAYOUT_CANONICAL, LAYOUT_G128X,
               GroupPlan, bit1_gemv_ex, bit1_gemv_launches, bit1_repack_g128x, bit1_unpack_g128x, bit1_ternary_combine,
               bit1_xor_patch)


def _align(n: int, a: int = 256) -> int:
    return (n + a - 1) // a * a


class Sweep:
    """``feed_swiglu``: the matrix after each SwiGLU matrix reads that
    matrix's output h as its x (gate/up -> down), instead of an x of its own;
    for the dependent per-matrix chain (run_eager / capture)."""

    def __init__(self, mats, seed0: int = 0, batch: int = 1, y_dtype: int = BF16,
                 device: str = "cuda", variant: int = AUTO, feed_swiglu: bool = False):
        self.mats = list(mats)
        self.fed = {}
        if feed_swiglu:
            if y_dtype != BF16:
                raise ValueError("h feeds the next product as bf16 activations")
            for i, m in enumerate(self.mats[:-1]):
                if m.swiglu:
                    if self.mats[i + 1].K != m.out:
                        raise ValueError(f"{self.mats[i + 1].name} does not take {m.name}'s h")
                    self.fed[i + 1] = i
        self.seed0 = seed0
        self.B = batch
        self.y_dtype = y_dtype
        self.variant = variant
        self.device = device
        ysz = 2 if y_dtype == BF16 else 4
        self.bits_off, self.sc_off, self.x_off, self.y_off = [], [], [], []
        nb = ns = nx = ny = 0
        for m in self.mats:
            self.bits_off.append(nb); nb += _align(m.N * m.K // 8)
            self.sc_off.append(ns); ns += _align(m.N * (m.K // 128) * 2)
            self.x_off.append(nx); nx += _align(batch * m.K * 2)
            self.y_off.append(ny); ny += _align(batch * m.out * ysz)
        self.bits = torch.empty(nb, dtype=torch.uint8, device=device)
        self.scales = torch.empty(ns // 2, dtype=torch.int16, device=device)
        self.x = torch.empty(nx // 2, dtype=torch.bfloat16, device=device)
        self.y = torch.empty(ny, dtype=torch.uint8, device=device)
        self.weight_bytes = sum(m.N * m.K // 8 + 2 * m.N * (m.K // 128) for m in self.mats)
        self.x_bytes = sum(batch * m.K * 2 for m in self.mats)
        self.graph = None
        self.stream = None

    # ---- views ---------------------------------------------------------
    def bits_of(self, i):
        m = self.mats[i]
        return self.bits[self.bits_off[i]: self.bits_off[i] + m.N * m.K // 8].view(m.N, m.K // 8)

    def scales_of(self, i):
        m = self.mats[i]
        o = self.sc_off[i] // 2
        return self.scales[o: o + m.N * (m.K // 128)].view(m.N, m.K // 128)

    def x_of(self, i, xbuf=None):
        if i in self.fed and xbuf is None:
            return self.y_of(self.fed[i])
        m = self.mats[i]
        o = self.x_off[i] // 2
        xb = self.x if xbuf is None else xbuf
        return xb[o: o + self.B * m.K].view(self.B, m.K)

    def y_of(self, i, ybuf=None):
        m = self.mats[i]
        yb = self.y if ybuf is None else ybuf
        if self.y_dtype == BF16:
            return yb[self.y_off[i]: self.y_off[i] + 2 * self.B * m.out].view(torch.bfloat16).view(self.B, m.out)
        return yb[self.y_off[i]: self.y_off[i] + 4 * self.B * m.out].view(torch.float32).view(self.B, m.out)

    # ---- data ------------------------------------------------------------
    def host_matrix(self, i):
        """The seeded host copy of matrix i (bits, scales) and its input x."""
        m = self.mats[i]
        bits, scales = synth.matrix(m.N, m.K, self.seed0 + i)
        x = synth.x_for(self.B, m.K, self.seed0 + i)
        return bits, scales, x

    def fill(self):
        """Generate every matrix on the host (seeded) and copy it to the arena."""
        for i in range(len(self.mats)):
            bits, scales, x = self.host_matrix(i)
            self.bits_of(i).copy_(torch.from_numpy(bits), non_blocking=False)
            self.scales_of(i).copy_(torch.from_numpy(scales.view(np.int16)))
            if i not in self.fed:
                self.x_of(i).copy_(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16))
        torch.cuda.synchronize()
        return self

    def fill_device(self, seed: int = 0):
        """The same distributions generated on the device from one seeded
        generator (sign bytes uniform, scales |N(0, 0.02)| in fp16, x N(0, 1) in
        bf16): for timing runs that need no host copy of the weights."""
        g = torch.Generator(device=self.device)
        g.manual_seed(seed)
        for i, m in enumerate(self.mats):
            self.bits_of(i).copy_(torch.randint(0, 256, (m.N, m.K // 8), dtype=torch.uint8,
                                                device=self.device, generator=g))
            sc = torch.randn((m.N, m.K // 128), device=self.device, generator=g).abs_().mul_(0.02)
            self.scales_of(i).copy_(sc.half().view(torch.int16))
            xr = torch.randn((self.B, m.K), device=self.device, generator=g).bfloat16()
            if i not in self.fed:
                self.x_of(i).copy_(xr)
        torch.cuda.synchronize()
        return self

    # ---- execution ---------------------------------------------------------
    def launches_per_step(self) -> int:
        return sum(bit1_gemv_launches(self.B, m.N, m.K, self.variant) for m in self.mats)

    def run_eager(self, stream=None, pdl: bool = True):
        for i, m in enumerate(self.mats):
            flags = (FLAG_PDL if pdl else 0) | (FLAG_SWIGLU if m.swiglu else 0)
            bit1_gemv_ex(self.bits_of(i), self.scales_of(i), self.x_of(i), y=self.y_of(i),
                         variant=self.variant, flags=flags, stream=stream, N=m.N, K=m.K)

    def capture(self, pdl: bool = True):
        self.stream = torch.cuda.Stream()
        self.stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(self.stream):
            self.run_eager(self.stream, pdl)       # warm-up (attributes, module load)
        self.stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            self.run_eager(self.stream, pdl)
        self.graph = g
        return self

    def replay(self):
        self.graph.replay()

    def to_g128x(self):
        """Convert every matrix's bits to the g128x layout in place (for
        grouped launches built with layout=LAYOUT_G128X; the per-matrix
        calls read the canonical layout).  Row patches apply unchanged."""
        for i in range(len(self.mats)):
            b = self.bits_of(i)
            bit1_repack_g128x(b, out=b)
        torch.cuda.synchronize()
        self.layout = LAYOUT_G128X
        return self

    def to_canonical(self):
        """The inverse of to_g128x (for the per-matrix calls)."""
        if getattr(self, "layout", LAYOUT_CANONICAL) == LAYOUT_G128X:
            for i in range(len(self.mats)):
                b = self.bits_of(i)
                bit1_unpack_g128x(b, out=b)
            torch.cuda.synchronize()
        self.layout = LAYOUT_CANONICAL
        return self

    def group_plan(self, x=None, y=None, tensor_cores: bool = False, mma: bool = False):
        """One grouped launch over every matrix of the sweep (each with its own
        input, ``batch`` rows of it): the plan is built once; run() is one
        kernel launch (two with ``tensor_cores``: the activation prep and the
        persistent tcgen05 kernel).  ``x`` and
        ``y`` replace the activation / output arenas (same layout), e.g. for a
        second I/O slot over the same resident weights."""
        if self.fed:
            raise ValueError("a grouped launch runs its problems concurrently: no x may be another's y")
        probs = [(self.bits_of(i), self.scales_of(i), self.x_of(i, x), self.y_of(i, y),
                  EPI_SWIGLU if m.swiglu else EPI_NONE) for i, m in enumerate(self.mats)]
        return GroupPlan(probs, device=self.device, B=self.B, layout=getattr(self, "layout", LAYOUT_CANONICAL),
                         tensor_cores=tensor_cores, mma=mma)

    def apply_patch(self, entries, proj_count: int = 7):
        """Apply (or, applied again, remove) a list of (layer, projection, row)
        entries: each is routed to its matrix and XOR-flipped there."""
        by_mat = {}
        for layer, proj, row in entries:
            by_mat.setdefault(layer * proj_count + proj, []).append(row)
        for i, rows in sorted(by_mat.items()):
            m = self.mats[i]
            bit1_xor_patch(self.bits_of(i), rows, N=m.N, K=m.K)
        return by_mat


class TernaryPlan:
    """A grouped launch over both sign planes of every ternary matrix (two
    problems per matrix, fp32 halves into one contiguous arena each) and one
    combine launch that forms y = (ya + yb) / 2 over the whole arena."""

    def __init__(self, sweep: "TernarySweep"):
        sw = sweep
        probs = []
        for i in range(len(sw.mats)):
            probs.append((sw.bits_of(i), sw.scales_of(i), sw.x_of(i), sw.half_of(sw.ya, i)))
            probs.append((sw.bits_b_of(i), sw.scales_of(i), sw.x_of(i), sw.half_of(sw.yb, i)))
        self.sweep = sw
        self.group = GroupPlan(probs, device=sw.device)

    def run(self, flags: int = 0, stream=None) -> None:
        self.group.run(flags=flags, stream=stream)
        sw = self.sweep
        bit1_ternary_combine(sw.ya, sw.yb, sw.yt, stream=stream)


class TernarySweep(Sweep):
    """The same decode sweep with ternary weights in 2-bit slots: two sign
    planes per matrix (t = (a + b) / 2) sharing one scale array; batch 1.
    Outputs are laid out contiguously (row offsets rounded up to 64) so that
    one combine launch serves every matrix."""

    def __init__(self, mats, seed0: int = 0, y_dtype: int = BF16, device: str = "cuda"):
        if any(m.swiglu for m in mats):
            raise ValueError("the ternary sweep combines plain products (use bit1_gemv_ternary with "
                             "FLAG_SWIGLU for a ternary gate/up pair)")
        super().__init__(mats, seed0=seed0, batch=1, y_dtype=y_dtype, device=device)
        self.bits_b = torch.empty_like(self.bits)
        self.row_off = []
        nr = 0
        for m in self.mats:
            self.row_off.append(nr)
            nr += _align(m.N, 64)
        self.rows_total = nr
        self.ya = torch.empty(nr, dtype=torch.float32, device=device)
        self.yb = torch.empty(nr, dtype=torch.float32, device=device)
        self.yt = torch.empty(nr, dtype=torch.bfloat16 if y_dtype == BF16 else torch.float32, device=device)
        self.weight_bytes = sum(2 * (m.N * m.K // 8) + 2 * m.N * (m.K // 128) for m in self.mats)

    def bits_b_of(self, i):
        m = self.mats[i]
        return self.bits_b[self.bits_off[i]: self.bits_off[i] + m.N * m.K // 8].view(m.N, m.K // 8)

    def half_of(self, arena, i):
        return arena[self.row_off[i]: self.row_off[i] + self.mats[i].N].view(1, self.mats[i].N)

    def y_of(self, i, ybuf=None):
        return self.half_of(self.yt if ybuf is None else ybuf, i)

    def host_matrix(self, i):
        """(a, b, scales, x) of ternary matrix i, seeded."""
        m = self.mats[i]
        a, b, scales = synth.ternary_matrix(m.N, m.K, self.seed0 + i)
        x = synth.x_for(1, m.K, self.seed0 + i)
        return a, b, scales, x

    def fill(self):
        for i in range(len(self.mats)):
            a, b, scales, x = self.host_matrix(i)
            self.bits_of(i).copy_(torch.from_numpy(a))
            self.bits_b_of(i).copy_(torch.from_numpy(b))
            self.scales_of(i).copy_(torch.from_numpy(scales.view(np.int16)))
            self.x_of(i).copy_(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16))
        torch.cuda.synchronize()
        return self

    def fill_device(self, seed: int = 0):
        super().fill_device(seed)
        g = torch.Generator(device=self.device)
        g.manual_seed(seed + 1)
        self.bits_b.copy_(torch.randint(0, 256, self.bits_b.shape, dtype=torch.uint8, device=self.device,
                                        generator=g))
        torch.cuda.synchronize()
        return self

    def launches_per_step(self) -> int:
        return 2

    def group_plan(self, x=None, y=None):
        if x is not None or y is not None:
            raise ValueError("a ternary sweep has one I/O slot")
        return TernaryPlan(self)
