"""Shared test plumbing: host<->device copies of the seeded inputs and the
GEMV tolerance.  No arithmetic of the method lives here."""
import numpy as np
import torch


def dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_u16(a: np.ndarray) -> torch.Tensor:
    """uint16 bit patterns -> int16 CUDA tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    return dev_u16(a).view(torch.bfloat16)


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def abs_bound(scales: np.ndarray, x: np.ndarray, K: int) -> np.ndarray:
    """sum_k |s_{n,g(k)} * x_{b,k}| as [B, N] (fp64), the scale of the stated
    GEMV tolerance 1e-3 * sum_k |s x_k| + 1e-6."""
    G = K // 128
    s = np.abs(scales.reshape(-1, G).view(np.float16).astype(np.float64))
    xv = torch.from_numpy(x.reshape(-1, K).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    gx = np.abs(xv).reshape(xv.shape[0], G, 128).sum(axis=2)
    return gx @ s.T


def assert_gemv_close(y_gpu: torch.Tensor, y_ref: np.ndarray, bound: np.ndarray, what: str = ""):
    """|y_gpu - y_oracle| <= 1e-3 * sum|s x| + 1e-6, plus the bf16 output's own
    round-to-nearest error (2^-8 |y|) when y is bf16."""
    yg = y_gpu.detach().float().cpu().numpy().astype(np.float64).reshape(y_ref.shape)
    tol = 1e-3 * bound + 1e-6
    if y_gpu.dtype == torch.bfloat16:
        tol = tol + 2.0 ** -8 * np.abs(y_ref)
    err = np.abs(yg - y_ref)
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outputs out of tolerance; first at {tuple(i)}: "
                             f"gpu {yg[tuple(i)]!r} oracle {y_ref[tuple(i)]!r} tol {tol[tuple(i)]!r}")
    return float((err / tol).max()) if err.size else 0.0


def assert_swiglu_close(h_gpu: torch.Tensor, h_ref: np.ndarray, g_ref: np.ndarray, u_ref: np.ndarray,
                        bound_g: np.ndarray, bound_u: np.ndarray, what: str = ""):
    """Tolerance of h = silu(g) u from the GEMV tolerance of g and u
    (dg <= 1e-3 * bound_g + 1e-6, likewise du): |silu'| <= 1.1 and
    |silu(g)| <= |g| give |dh| <= 1.1 dg (|u| + du) + |g| du; plus eight fp32
    ulps of h for the activation and the product, and the bf16 output's own
    rounding (2^-8 |h|) when h is bf16."""
    hg = h_gpu.detach().float().cpu().numpy().astype(np.float64).reshape(h_ref.shape)
    dg = 1e-3 * bound_g + 1e-6
    du = 1e-3 * bound_u + 1e-6
    tol = 1.1 * dg * (np.abs(u_ref) + du) + np.abs(g_ref) * du + 8 * 2.0 ** -24 * np.abs(h_ref) + 1e-30
    if h_gpu.dtype == torch.bfloat16:
        tol = tol + 2.0 ** -8 * np.abs(h_ref)
    err = np.abs(hg - h_ref)
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outputs out of tolerance; first at {tuple(i)}: "
                             f"gpu {hg[tuple(i)]!r} oracle {h_ref[tuple(i)]!r} tol {tol[tuple(i)]!r}")
    return float((err / tol).max()) if err.size else 0.0


def swiglu_h_tol(g_ref, u_ref, bound_g, bound_u, h_ref):
    """Elementwise bound on |h_gpu(bf16) - bf16(h_oracle)|: the SwiGLU
    tolerance of assert_swiglu_close plus both bf16 roundings."""
    dg = 1e-3 * bound_g + 1e-6
    du = 1e-3 * bound_u + 1e-6
    return 1.1 * dg * (np.abs(u_ref) + du) + np.abs(g_ref) * du + 2 * 2.0 ** -8 * np.abs(h_ref) + 1e-30


def carried_bound(scales: np.ndarray, dx: np.ndarray, K: int) -> np.ndarray:
    """sum_k |s_{n,g(k)}| * dx_{b,k} as [B, N]: how far an input error dx can
    move each output of the product."""
    G = K // 128
    s = np.abs(scales.reshape(-1, G).view(np.float16).astype(np.float64))
    return dx.reshape(-1, G, 128).sum(axis=2) @ s.T
