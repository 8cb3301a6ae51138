"""Shared comparison helpers for the GPU parity tests (CUDA path vs. oracle)."""
import numpy as np
import torch

# Acceptance on bf16 outputs against the float64 oracle (element by element).
# |O - O_ref| <= 1e-2 + 2^-9 |O_ref|: the 1e-2 bound on top of the half-unit
# rounding of the bf16 output format itself (a bf16 O in [4, 8) cannot be
# nearer than 2^-6 to a value between two representable numbers; on the K*8
# workload the exactly rounded oracle result is already 0.015 away).  The mean
# abs bound gets the same allowance on average, 1e-3 + 2^-9 mean|O_ref|: for
# rows that see one or two keys (short windows) O is of unit size and rounding
# it to bf16 alone averages about 1e-3; for long rows the term is ~4e-5.
BF16_MAX_ABS = 1e-2
BF16_OUT_HALF_ULP = 2.0 ** -9
BF16_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3
# FP8: RMSE of O against the oracle run on the unquantised inputs, plus a
# relative bound so that a degenerate output (O ~ 0) cannot pass.
FP8_RMSE = 3e-2
FP8_REL_RMSE = 0.1
# Kernel fidelity: against the oracle run on the oracle's own E4M3 operands the
# only differences left are P's E4M3 rounding, f32 accumulation and the output
# rounding.
FP8_Q_REL_RMSE = 0.05
FP8_Q_LSE_MAX_ABS = 0.02


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def metrics(o_gpu, lse_gpu, O_ref, L_ref):
    o = f64(o_gpu) if isinstance(o_gpu, torch.Tensor) else o_gpu
    lse = f64(lse_gpu) if isinstance(lse_gpu, torch.Tensor) else lse_gpu
    err = np.abs(o - O_ref)
    lerr = np.abs(lse - L_ref)
    return {
        "max_abs": float(err.max()),
        "max_excess": float((err - BF16_OUT_HALF_ULP * np.abs(O_ref)).max()),
        "mean_abs": float(err.mean()),
        "mean_half_ulp": float(BF16_OUT_HALF_ULP * np.abs(O_ref).mean()),
        "rmse": float(np.sqrt((err ** 2).mean())),
        "rel_rmse": float(np.sqrt((err ** 2).mean() / max((O_ref ** 2).mean(), 1e-300))),
        "lse_max_abs": float(lerr.max()),
        "finite": bool(np.isfinite(o).all() and np.isfinite(lse).all()),
    }


def assert_bf16_parity(m, what=""):
    assert m["finite"], f"{what}: non-finite output"
    assert m["max_excess"] <= BF16_MAX_ABS, \
        f"{what}: max abs {m['max_abs']:.3e} (beyond output rounding {m['max_excess']:.3e})"
    assert m["mean_abs"] <= BF16_MEAN_ABS + m["mean_half_ulp"], \
        f"{what}: mean abs {m['mean_abs']:.3e} (output rounding allowance {m['mean_half_ulp']:.1e})"
    assert m["lse_max_abs"] <= LSE_MAX_ABS, f"{what}: lse max abs {m['lse_max_abs']:.3e}"


def assert_fp8_parity(m, what=""):
    assert m["finite"], f"{what}: non-finite output"
    assert m["rmse"] <= FP8_RMSE, f"{what}: rmse {m['rmse']:.3e}"
    assert m["rel_rmse"] <= FP8_REL_RMSE, f"{what}: relative rmse {m['rel_rmse']:.3e}"


def assert_fp8_fidelity(mq, what=""):
    """Against the oracle on the oracle's own quantised operands."""
    assert mq["finite"], f"{what}: non-finite output"
    assert mq["rel_rmse"] <= FP8_Q_REL_RMSE, f"{what}: relative rmse {mq['rel_rmse']:.3e}"
    assert mq["lse_max_abs"] <= FP8_Q_LSE_MAX_ABS, f"{what}: lse max abs {mq['lse_max_abs']:.3e}"
