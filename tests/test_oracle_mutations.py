"""Planted slips in the oracle must be caught by its pins.

Each case edits one line of a copy of the oracle's C source (on the CPU, in a
temporary directory), builds it, and runs every pin of test_oracle_pins.py
against it: at least one pin has to fail.  This shows the pins are strong
enough that a plausible mistake in the oracle cannot pass unnoticed.
"""
import inspect

import pytest

import oracle
import test_oracle_pins as pins

MUTATIONS = {
    "scale_sign": ("yr[d] = xhat * (1.0 + sc[d]) + sh[d];", "yr[d] = xhat * (1.0 - sc[d]) + sh[d];"),
    "shift_dropped": ("yr[d] = xhat * (1.0 + sc[d]) + sh[d];", "yr[d] = xhat * (1.0 + sc[d]);"),
    "unbiased_var": ("v = v / (double)D;", "v = v / (double)(D - 1);"),
    "eps_outside_sqrt": ("*rstd_out = 1.0 / sqrt(v + eps);", "*rstd_out = 1.0 / (sqrt(v) + eps);"),
    "bwd_mean_g_dropped": ("dxr[d] = rs * (g - mean_g - xhat * mean_gx);",
                           "dxr[d] = rs * (g - xhat * mean_gx);"),
    "bwd_wrong_projection": ("dxr[d] = rs * (g - mean_g - xhat * mean_gx);",
                             "dxr[d] = rs * (g - mean_g - xhat * mean_g);"),
    "bwd_scale_not_in_g": ("const double g = dyr[d] * (1.0 + sc[d]);\n                dxr",
                           "const double g = dyr[d];\n                dxr"),
    "dscale_missing_xhat": ("ds[d] += dyr[d] * xhat;", "ds[d] += dyr[d];"),
    "dshift_wrong_operand": ("db[d] += dyr[d];", "db[d] += dyr[d] * (1.0 + sc[d]);"),
    "gate_transposed": ("r[row * D + d] + g[d] * z[row * D + d]", "z[row * D + d] + g[d] * r[row * D + d]"),
    "dgate_wrong_operand": ("dg[d] += dout[row * D + d] * z[row * D + d];",
                            "dg[d] += dout[row * D + d] * g[d];"),
    "dz_missing_gate": ("dz[row * D + d] = g[d] * dout[row * D + d];", "dz[row * D + d] = dout[row * D + d];"),
    "fused_gate_on_r": ("oracle_gate_residual(r, y, gate, offsets, nseg, D, out);",
                        "oracle_gate_residual(y, r, gate, offsets, nseg, D, out);"),
    "fused_bwd_gate_dropped": ("oracle_adaln_bwd(x, scale, dy, offsets, nseg, D, eps, dx, d_scale, d_shift);",
                               "oracle_adaln_bwd(x, scale, dout, offsets, nseg, D, eps, dx, d_scale, d_shift);"),
    "fused_dgate_on_x": ("oracle_gate_residual_bwd(dout, y, gate, offsets, nseg, D, dy, d_gate);",
                         "oracle_gate_residual_bwd(dout, x, gate, offsets, nseg, D, dy, d_gate);"),
    "rms_mean_removed": ("for (int64_t d = 0; d < D; ++d) y[row * D + d] = xr[d] * rs * (1.0 + sc[d]) + sh[d];",
                         "for (int64_t d = 0; d < D; ++d) y[row * D + d] = (xr[d] - q / (double)D) * rs * (1.0 + sc[d]) + sh[d];"),
    "rms_eps_outside": ("const double rs = 1.0 / sqrt(q / (double)D + eps);\n            rstd[row] = rs;",
                        "const double rs = 1.0 / (sqrt(q / (double)D) + eps);\n            rstd[row] = rs;"),
    "rms_bwd_projection_dropped": ("dx[row * D + d] = rs * (g - xhat * mean_gx);",
                                   "dx[row * D + d] = rs * g;"),
    "segment_row_zero": ("const double *sc = scale + k * D;\n        for (int64_t row = offsets[k]; row < offsets[k + 1]; ++row) {\n            const double *xr = x + row * D;\n            double *yr",
                         "const double *sc = scale;\n        for (int64_t row = offsets[k]; row < offsets[k + 1]; ++row) {\n            const double *xr = x + row * D;\n            double *yr"),
}

PINS = [f for n, f in inspect.getmembers(pins, inspect.isfunction)
        if n.startswith("test_") and "oracle_mod" in inspect.signature(f).parameters]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_slip_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation anchor not unique/not found: {name}"
    so = oracle.compile_variant(src.replace(old, new), str(tmp_path), "mut_" + name)
    variant = oracle.Variant(so)
    failed = []
    for pin in PINS:
        try:
            pin(variant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted slip {name}"
