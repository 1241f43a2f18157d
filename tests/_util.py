"""Helpers shared by the GPU parity tests: upload, download, comparisons.

Tolerances (stated by the target of this library, written here once):
  - integer-valued fp32 inputs: bit-exact;
  - bf16 storage: max|gpu - oracle| <= 2e-2 * RMS(oracle);
  - fp32 storage with real-valued inputs: max|gpu - oracle| <= 1e-4 * RMS(oracle).
Elementwise outputs stored in bf16 whose values are heavy-tailed (a SwiGLU
product, a norm times a gain) can sit 15-20x above their RMS, where the
storage rounding alone (half an ulp, 2^-9 of the value) exceeds 2e-2 * RMS.
For those intermediates the bound adds that rounding per element:
|gpu - oracle| <= 2e-2 * RMS(oracle) + 2^-8 * |oracle|  (assert_close_stored).
"""
import numpy as np
import torch

TOL_BF16 = 2e-2
TOL_F32 = 1e-4


def dev(a: np.ndarray, dtype=torch.bfloat16) -> torch.Tensor:
    """Upload a float32 array (bf16-representable for bf16) to cuda:0."""
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(dtype).contiguous()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def f64(a: np.ndarray) -> np.ndarray:
    return np.asarray(a, np.float64)


def i64(a: np.ndarray) -> np.ndarray:
    return np.asarray(a).astype(np.int64)


def rms(ref: np.ndarray) -> float:
    return float(np.sqrt(np.mean(np.square(ref))))


def assert_close(gpu, ref, tol, what=""):
    g = host(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    err = float(np.max(np.abs(g - ref))) if ref.size else 0.0
    r = rms(ref) if ref.size else 0.0
    assert err <= tol * r, f"{what}: max err {err:.4g} > {tol} * rms {r:.4g} (ratio {err / max(r, 1e-300):.3g})"
    return err / max(r, 1e-300)


def assert_close_stored(gpu, ref, tol=TOL_BF16, what=""):
    """Bound for bf16-stored elementwise outputs: tol * RMS plus the storage
    rounding of each element (2^-8 of its magnitude)."""
    g = host(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    bound = tol * rms(ref) + np.abs(ref) * 2.0 ** -8
    excess = np.abs(g - ref) - bound
    i = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess[i] <= 0, f"{what}: at {i} err {abs(g[i] - ref[i]):.4g} > bound {bound[i]:.4g}"


def assert_exact(gpu, ref, what=""):
    g = host(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    ref = np.asarray(ref)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    bad = np.argwhere(g != ref)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {bad[0].tolist()}: gpu {g[tuple(bad[0])]} ref {ref[tuple(bad[0])]}"


def sample_rows(T: int, n: int, seed: int = 1234) -> np.ndarray:
    """A fixed sorted sample of token rows, always including the first and last."""
    if T <= n:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    rows = rng.choice(np.arange(1, T - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, T - 1], rows]))
