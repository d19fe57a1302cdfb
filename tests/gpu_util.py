"""Helpers shared by the GPU parity tests (not a test module)."""
from __future__ import annotations

import numpy as np
import torch


def require_gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from scaling_quantization_gemm_gb300 import build
    build.build()
    import scaling_quantization_gemm_gb300 as q
    q.lib()
    return q


def dev_bf16(x_bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns (host) -> bf16 tensor on cuda:0."""
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to("cuda").view(torch.bfloat16)


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def nan_code(c: np.ndarray, fmt: int) -> np.ndarray:
    c = c & 0x7F
    return c == 0x7F if fmt == 0 else c > 0x7C


def assert_codes_equal(got: np.ndarray, ref: np.ndarray, fmt: int, what: str = "codes") -> None:
    """Bit-exact comparison; NaN codes are compared by class (sign/payload are not pinned)."""
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    gn, rn = nan_code(got, fmt), nan_code(ref, fmt)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ"
    diff = (got != ref) & ~rn
    if diff.any():
        idx = np.argwhere(diff)[:5]
        raise AssertionError(f"{what}: {int(diff.sum())} mismatches, first at {idx.tolist()}: "
                             f"got {[hex(int(got[tuple(i)])) for i in idx]} ref {[hex(int(ref[tuple(i)])) for i in idx]}")


def assert_gemm_close(y: np.ndarray, y_ref: np.ndarray, mag: np.ndarray, out_bf16: bool, what: str = "D") -> None:
    """|y - y_ref| <= 1e-3 sum_k |a_k b_k| (+ half a bf16 ulp of y_ref for a bf16 output)."""
    import oracle
    tol = oracle.gemm_tolerance(y_ref, mag, out_bf16)
    err = np.abs(y.astype(np.float64) - y_ref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; first {i.tolist()}: "
                             f"y={[float(y[tuple(k)]) for k in i]} ref={[float(y_ref[tuple(k)]) for k in i]} "
                             f"tol={[float(tol[tuple(k)]) for k in i]}")


def bf16_out_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def sample_coords(M: int, N: int, seed: int, n_random: int = 4096, corner: int = 32):
    """Output coordinates for sampled GEMM checks: the corner corner x corner block of each of the
    four corner 128x128 tiles, plus seeded random elements."""
    rng = np.random.default_rng(seed)
    ms, ns = [], []
    for m0 in sorted({0, max(0, M - corner)}):
        for n0 in sorted({0, max(0, N - corner)}):
            mm, nn = np.meshgrid(np.arange(m0, min(M, m0 + corner)), np.arange(n0, min(N, n0 + corner)),
                                 indexing="ij")
            ms.append(mm.ravel())
            ns.append(nn.ravel())
    ms.append(rng.integers(0, M, n_random))
    ns.append(rng.integers(0, N, n_random))
    return np.concatenate(ms).astype(np.int64), np.concatenate(ns).astype(np.int64)
