"""Shared test helpers: tensor -> numpy views and the parity metrics.

Tolerances (bf16 output, fp32 LSE) against the fp64 oracle:
  out rel-L2 <= 3e-3                      (the bf16 output floor is ~1.66e-3)
  out max-abs <= 2e-2 * RMS(out_ref), counted beyond one bf16 rounding of the
      result: each element may also differ by half a bf16 ulp at its
      magnitude.  Rounding the exact result to bf16 alone already reaches
      0.02-0.04 * RMS on elements above 0.5 (measured on the b=64, h=128,
      t=4096 rows), so without that allowance no bf16 output could pass.
  |lse - lse_ref| <= 1e-3.
"""
import numpy as np
import torch

OUT_REL_L2 = 3e-3
OUT_MAX_ABS_REL_RMS = 2e-2
LSE_ABS = 1e-3


def bf16_np(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (no rounding)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f64_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def bf16_half_ulp(x):
    """Half the spacing of bfloat16 numbers at |x| (8 significant bits)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 8)


def parity_stats(out, out_ref, lse, lse_ref):
    """Error statistics of (out, lse) against the reference, over finite rows."""
    out = np.asarray(out, dtype=np.float64)
    out_ref = np.asarray(out_ref, dtype=np.float64)
    diff = out - out_ref
    rms = float(np.sqrt(np.mean(out_ref ** 2)))
    rel_l2 = float(np.linalg.norm(diff) / max(np.linalg.norm(out_ref), 1e-300))
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    slack = bf16_half_ulp(np.maximum(np.abs(out), np.abs(out_ref)))
    beyond = float(np.max(np.abs(diff) - slack)) if diff.size else 0.0
    lse = np.asarray(lse, dtype=np.float64)
    lse_ref = np.asarray(lse_ref, dtype=np.float64)
    both_inf = np.isinf(lse) & np.isinf(lse_ref) & (np.sign(lse) == np.sign(lse_ref))
    with np.errstate(invalid="ignore"):  # -inf - -inf where both rows are empty
        lse_err = np.where(both_inf, 0.0, np.abs(lse - lse_ref))
    return dict(rel_l2=rel_l2, max_abs=max_abs, max_abs_beyond_rounding=beyond, rms=rms,
                max_abs_over_rms=max_abs / rms if rms > 0 else float(max_abs > 0) * np.inf,
                lse_max_err=float(np.max(lse_err)) if lse_err.size else 0.0)


def assert_parity(out, out_ref, lse, lse_ref, what=""):
    st = parity_stats(out, out_ref, lse, lse_ref)
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    assert st["rel_l2"] <= OUT_REL_L2, f"{what}: {st}"
    assert st["max_abs_beyond_rounding"] <= OUT_MAX_ABS_REL_RMS * st["rms"], f"{what}: {st}"
    assert st["lse_max_err"] <= LSE_ABS, f"{what}: {st}"
    return st
