"""Shared test helpers: tensor -> numpy views and the parity metrics.

Tolerances (bf16 output, fp32 LSE) against the fp64 oracle:
  out rel-L2 <= 3e-3                      (the bf16 output floor is ~1.66e-3)
  out max-abs <= 2e-2 * RMS(out_ref), counted beyond one bf16 rounding of the
      result: each element may also differ by half a bf16 ulp at its
      magnitude.  Rounding the exact result to bf16 alone already reaches
      0.02-0.04 * RMS on elements above 0.5 (measured on the b=64, h=128,
      t=4096 rows), so without that allowance no bf16 output could pass.
  |lse - lse_ref| <= 1e-3.
The RMS that max-abs is relative to is that of one query token's output
(all its heads): tokens of one call have outputs of very different size
(a token over 16k keys averages to far smaller values than one over 1k, or
one dominated by a few keys), and each token's error scales with its own
output.  assert_parity_per_token applies the three bounds to every token
and rel-L2 to the whole call as well.
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


def assert_parity_per_token(out, out_ref, lse, lse_ref, what=""):
    """out [b, s_q, h, 512], lse [b, h, s_q]: every query token (b, j) meets
    all three bounds relative to its own output; the whole call meets the
    rel-L2 and LSE bounds.  Returns the worst per-token statistics."""
    out = np.asarray(out, dtype=np.float64)
    out_ref = np.asarray(out_ref, dtype=np.float64)
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    whole = parity_stats(out, out_ref, lse, lse_ref)
    assert whole["rel_l2"] <= OUT_REL_L2, f"{what} (whole call): {whole}"
    assert whole["lse_max_err"] <= LSE_ABS, f"{what} (whole call): {whole}"
    worst = dict(rel_l2=0.0, max_abs_beyond_over_rms=0.0, lse_max_err=0.0)
    b, s_q = out.shape[:2]
    for bi in range(b):
        for j in range(s_q):
            st = assert_parity(out[bi, j], out_ref[bi, j], lse[bi, :, j], lse_ref[bi, :, j],
                               f"{what} token ({bi}, {j})")
            worst["rel_l2"] = max(worst["rel_l2"], st["rel_l2"])
            worst["max_abs_beyond_over_rms"] = max(worst["max_abs_beyond_over_rms"],
                                                   st["max_abs_beyond_rounding"] / st["rms"])
            worst["lse_max_err"] = max(worst["lse_max_err"], st["lse_max_err"])
    return dict(whole=whole, worst_token=worst)
