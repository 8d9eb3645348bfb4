"""Plants plausible mistakes in the oracle (on the CPU, by rewriting its source
in memory) and checks that at least one pin catches each.  Nothing here runs
on a GPU; the oracle files on disk are never modified."""
import inspect
import json
import os

import numpy as np
import pytest

import oracle
from oracle import add_rmsnorm_quant as OP
from oracle import formats as FM

import test_oracle_formats as TF
import test_oracle_global_scale as TG
import test_oracle_invariants as TI
import test_oracle_rows as TR


def _mutant(module, func_name, old, new):
    src = inspect.getsource(getattr(module, func_name))
    assert old in src, f"mutation anchor not found: {old!r}"
    ns = dict(vars(module))
    exec(compile(src.replace(old, new, 1), f"<mutant {func_name}>", "exec"), ns)
    return ns[func_name]


def _golden_all():
    for spec in TR.ROWS:
        for fmt in ("nvfp4", "mxfp4"):
            TR.test_worked_row(spec, fmt)


def _pins_fail(checks):
    for check in checks:
        try:
            check()
        except (AssertionError, ValueError):
            return True
    return False


OP_MUTANTS = {
    "nibble order swapped": ("codes[:, 0::2] | (codes[:, 1::2] << np.uint8(4))",
                             "codes[:, 1::2] | (codes[:, 0::2] << np.uint8(4))"),
    "eps dropped": ("np.sqrt(ms + F32(eps))", "np.sqrt(ms)"),
    "squares of the unrounded sum": ("ss = np.sum(h.astype(np.float64) ** 2, axis=1)",
                                     "ss = np.sum((x + r).astype(np.float64) ** 2, axis=1)"),
    "scale from amax/4": ("t = amax / E2M1_MAX", "t = amax / F32(4.0)"),
    "no E4M3 clamp, scale from amax/8": ("t = np.minimum((gs * amax) / E2M1_MAX, E4M3_MAX)",
                                         "t = (gs * amax) / F32(8.0)"),
    "global scale divides": ("t = np.minimum((gs * amax) / E2M1_MAX, E4M3_MAX)",
                             "t = np.minimum((amax / gs) / E2M1_MAX, E4M3_MAX)"),
    "global scale left out of the reciprocal": ("inv = (inv * gs).astype(np.float32)",
                                                "inv = inv.astype(np.float32)"),
    "global scale applied to UE8M0": ("        t = amax / E2M1_MAX\n",
                                      "        t = (gs * amax) / E2M1_MAX\n"),
    "weight ignored": ("y = (h * w[None, :]) * rstd[:, None]", "y = h * rstd[:, None]"),
    "two roundings in y": ("y = (h * w[None, :]) * rstd[:, None]",
                           "y = (h * rstd[:, None]) * w[None, :]"),
    "mean over H-1": ("ms = (ss / H)", "ms = (ss / (H - 1))"),
    "residual not rounded": ("h = round_to_dtype(x + r, dtype)", "h = x + r"),
    "swizzle inner/outer m swapped": (
        "(m % 32) * 16\n            + ((m % 128) // 32) * 4",
        "(m % 32) * 4\n            + ((m % 128) // 32) * 16"),
}


def _golden_gs():
    for spec in TG.ROWS:
        TG.test_golden_row(spec)


@pytest.mark.parametrize("name", list(OP_MUTANTS))
def test_op_mutant_is_caught(name, monkeypatch):
    old, new = OP_MUTANTS[name]
    target = next(f for f in ("swizzled_sf_offset", "add_rmsnorm_fp4_quant", "_quantize_rows")
                  if old in inspect.getsource(getattr(OP, f)))
    mut = _mutant(OP, target, old, new)
    monkeypatch.setattr(OP, target, mut)
    if hasattr(oracle, target):
        monkeypatch.setattr(oracle, target, mut)
    checks = [
        _golden_all,
        _golden_gs,
        lambda: TR.test_residual_is_rounded_sum(),
        lambda: TR.test_constant_row_rms_closed_form(0.125, "bf16"),
        lambda: TI.test_swizzle_matches_nested_tile_shape(130, 6),
        lambda: TI.test_dequant_error_within_half_step("nvfp4", "bf16"),
        lambda: TI.test_mxfp4_scale_brackets_amax(),
        lambda: TI.test_nvfp4_scale_is_nearest_e4m3_to_amax_over_6(),
        lambda: TI.test_y_is_one_rounding_of_h_w_rstd("bf16"),
    ]
    assert _pins_fail(checks), f"no pin caught: {name}"


FORMAT_MUTANTS = {
    "E2M1 ties away from zero": ("on_tie_pick = upper if upper % 2 == 0 else i",
                                 "on_tie_pick = upper"),
    "E2M1 sign dropped": ("return (sign << np.uint8(3)) | idx", "return idx"),
    "E4M3 ties away from zero": ("n = np.rint(t / q)", "n = np.floor(t / q + 0.5)"),
    "E4M3 no subnormals": ("e = np.maximum(k - 1, -6)", "e = k - 1"),
    "UE8M0 floor instead of ceil": ("e = np.where(f == 0.5, k - 1, k)", "e = k - 1"),
    "bf16 truncation": ("rounded = (bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)",
                        "rounded = bits >> np.uint64(16)"),
}

_FORMAT_FUNC = {
    "E2M1 ties away from zero": "e2m1_index_rne",
    "E2M1 sign dropped": "e2m1_encode",
    "E4M3 ties away from zero": "e4m3_encode_rne",
    "E4M3 no subnormals": "e4m3_encode_rne",
    "UE8M0 floor instead of ceil": "ue8m0_encode_ceil",
    "bf16 truncation": "bf16_round",
}


@pytest.mark.parametrize("name", list(FORMAT_MUTANTS))
def test_format_mutant_is_caught(name, monkeypatch):
    old, new = FORMAT_MUTANTS[name]
    fname = _FORMAT_FUNC[name]
    mut = _mutant(FM, fname, old, new)
    monkeypatch.setattr(FM, fname, mut)
    if hasattr(oracle, fname):
        monkeypatch.setattr(oracle, fname, mut)
    if hasattr(OP, fname):
        monkeypatch.setattr(OP, fname, mut)
    # functions that call the mutated one through the module namespace
    for caller in ("e2m1_encode", "round_to_dtype"):
        if caller != fname:
            rebound = _mutant(FM, caller, "def ", "def ")
            monkeypatch.setattr(FM, caller, rebound)
            if hasattr(oracle, caller):
                monkeypatch.setattr(oracle, caller, rebound)
            if hasattr(OP, caller):
                monkeypatch.setattr(OP, caller, rebound)
    checks = [
        TF.test_e2m1_encode_inverts_decode,
        TF.test_e2m1_encode_matches_brute_force,
        TF.test_e2m1_ties_go_to_even,
        TF.test_e4m3_encode_matches_torch_cast,
        TF.test_ue8m0_exhaustive_and_ceiling,
        lambda: TF.test_dtype_rounding_matches_torch("bf16", __import__("torch").bfloat16),
        _golden_all,
    ]
    assert _pins_fail(checks), f"no pin caught: {name}"
