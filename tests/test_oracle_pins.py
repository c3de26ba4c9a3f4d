"""Pins of the fp64 oracle against things other than itself.

Each check is fixed by the operator's definition (the DiT adaptive LayerNorm
of the "AdaptiveLoad" summary, section 2.B) or by mathematics, never by the
CUDA library: library routines that reduce to a special case (torch's
layer_norm and autograd in fp64, numpy var/sum), closed forms, invariants,
central finite differences, and exact integer arithmetic.  A plausible slip
in the oracle (a sign of scale, a dropped mean term, a transposed operand, a
wrong segment index) fails at least one of them; test_oracle_mutations.py
plants such slips on purpose and checks that.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import workloads


def _rng(seed):
    return np.random.default_rng(seed)


def _problem(seed=0, seg=(8, 8), D=16, mod_std=0.1):
    r = _rng(seed)
    rows = sum(seg)
    off = np.concatenate([[0], np.cumsum(seg)]).astype(np.int64)
    nseg = len(seg)
    P = dict(
        x=r.standard_normal((rows, D)),
        shift=mod_std * r.standard_normal((nseg, D)),
        scale=mod_std * r.standard_normal((nseg, D)),
        gate=mod_std * r.standard_normal((nseg, D)),
        r=r.standard_normal((rows, D)),
        z=r.standard_normal((rows, D)),
        dy=r.standard_normal((rows, D)),
        dout=r.standard_normal((rows, D)),
        off=off,
    )
    return P


# ----------------------------------------------------------------------------- forward

def test_fwd_equals_torch_layer_norm_with_modulation_as_affine(oracle_mod):
    """Per segment k, y is torch's fp64 layer_norm with weight 1+scale[k], bias shift[k]."""
    P = _problem(1, seg=(5, 0, 9, 3), D=24)
    for eps in (1e-6, 1e-2):
        y, mean, rstd = oracle_mod.adaln_fwd(P["x"], P["shift"], P["scale"], P["off"], eps)
        for k in range(len(P["off"]) - 1):
            a, b = P["off"][k], P["off"][k + 1]
            xt = torch.from_numpy(P["x"][a:b])
            ref = F.layer_norm(xt, (24,), weight=torch.from_numpy(1.0 + P["scale"][k]),
                               bias=torch.from_numpy(P["shift"][k]), eps=eps).numpy()
            np.testing.assert_allclose(y[a:b], ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(mean, P["x"].mean(axis=1), rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(rstd, 1.0 / np.sqrt(P["x"].var(axis=1) + eps), rtol=1e-13)


def test_fwd_unit_moments_at_eps0(oracle_mod):
    """shift=scale=0, eps=0: every output row has mean 0 and variance 1 (1e-12)."""
    P = _problem(2, seg=(7, 4), D=64)
    z = np.zeros_like(P["shift"])
    y, _, _ = oracle_mod.adaln_fwd(P["x"] * 3.0 + 5.0, z, z, P["off"], 0.0)
    assert np.max(np.abs(y.mean(axis=1))) < 1e-12
    assert np.max(np.abs(y.var(axis=1) - 1.0)) < 1e-12


def test_fwd_variance_closed_form_with_eps(oracle_mod):
    """With eps > 0 the row variance of xhat is sigma^2 / (sigma^2 + eps)."""
    P = _problem(3, seg=(6,), D=32)
    x = P["x"] * 0.01  # small variance so that eps matters
    z = np.zeros((1, 32))
    eps = 1e-6
    y, _, _ = oracle_mod.adaln_fwd(x, z, z, P["off"], eps)
    s2 = x.var(axis=1)
    np.testing.assert_allclose(y.var(axis=1), s2 / (s2 + eps), rtol=0, atol=1e-12)


def test_fwd_translation_invariance_and_shift_only(oracle_mod):
    P = _problem(4, seg=(3, 5), D=16)
    y0, _, rs0 = oracle_mod.adaln_fwd(P["x"], P["shift"], P["scale"], P["off"], 1e-6)
    y1, _, rs1 = oracle_mod.adaln_fwd(P["x"] + 7.25, P["shift"], P["scale"], P["off"], 1e-6)
    np.testing.assert_allclose(y1, y0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(rs1, rs0, rtol=1e-12)
    # scale = 0, shift = c: y = xhat + c
    c = np.full_like(P["shift"], 0.375)
    y2, _, _ = oracle_mod.adaln_fwd(P["x"], c, np.zeros_like(c), P["off"], 1e-6)
    zero = np.zeros_like(c)
    yhat, _, _ = oracle_mod.adaln_fwd(P["x"], zero, zero, P["off"], 1e-6)
    np.testing.assert_allclose(y2 - yhat, 0.375, rtol=0, atol=1e-14)


def test_fwd_segment_uses_its_own_modulation_row(oracle_mod):
    """Ragged rows: each segment equals the dense oracle on that segment alone (bitwise)."""
    P = _problem(5, seg=(4, 1, 0, 6), D=8)
    y, m, rs = oracle_mod.adaln_fwd(P["x"], P["shift"], P["scale"], P["off"], 1e-6)
    for k in range(4):
        a, b = P["off"][k], P["off"][k + 1]
        yk, mk, rk = oracle_mod.adaln_fwd(P["x"][a:b], P["shift"][k:k + 1], P["scale"][k:k + 1],
                                          [0, b - a], 1e-6)
        assert np.array_equal(yk, y[a:b]) and np.array_equal(mk, m[a:b]) and np.array_equal(rk, rs[a:b])


# ----------------------------------------------------------------------------- backward

def test_bwd_equals_torch_autograd_fp64(oracle_mod):
    """dx, d_scale, d_shift are the fp64 autograd gradients of sum(dy * y)."""
    P = _problem(6, seg=(5, 7), D=20)
    eps = 1e-6
    dx, dsc, dsh = oracle_mod.adaln_bwd(P["x"], P["scale"], P["dy"], P["off"], eps)
    for k in range(2):
        a, b = P["off"][k], P["off"][k + 1]
        xt = torch.from_numpy(P["x"][a:b].copy()).requires_grad_(True)
        w = torch.from_numpy(1.0 + P["scale"][k]).requires_grad_(True)
        bias = torch.from_numpy(P["shift"][k].copy()).requires_grad_(True)
        y = F.layer_norm(xt, (20,), weight=w, bias=bias, eps=eps)
        (y * torch.from_numpy(P["dy"][a:b])).sum().backward()
        np.testing.assert_allclose(dx[a:b], xt.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dsc[k], w.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dsh[k], bias.grad.numpy(), rtol=0, atol=1e-12)


def _loss(oracle_mod, P, eps):
    y, _, _ = oracle_mod.adaln_fwd(P["x"], P["shift"], P["scale"], P["off"], eps)
    out = oracle_mod.gate_residual(P["r"], P["z"], P["gate"], P["off"])
    return float(np.sum(P["dy"] * y) + np.sum(P["dout"] * out))


def test_bwd_central_finite_differences_2x8x16(oracle_mod):
    """B=2, N=8, D=16: all gradients agree with central differences within 1e-6."""
    P = _problem(7, seg=(8, 8), D=16)
    eps = 1e-6
    dx, dsc, dsh = oracle_mod.adaln_bwd(P["x"], P["scale"], P["dy"], P["off"], eps)
    dz, dg = oracle_mod.gate_residual_bwd(P["dout"], P["z"], P["gate"], P["off"])
    analytic = {"x": dx, "scale": dsc, "shift": dsh, "gate": dg, "z": dz, "r": P["dout"]}
    for name, grad in analytic.items():
        base = P[name]
        fd = np.empty_like(base)
        for idx in np.ndindex(base.shape):
            v = base[idx]
            h = 1e-6 * max(1.0, abs(v))
            base[idx] = v + h
            lp = _loss(oracle_mod, P, eps)
            base[idx] = v - h
            lm = _loss(oracle_mod, P, eps)
            base[idx] = v
            fd[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(fd - grad))
        assert err < 1e-6, (name, err)


def test_bwd_shift_grad_is_exact_column_sum(oracle_mod):
    P = _problem(8, seg=(33, 17), D=12)
    # integer-valued dy: every partial sum is exact in fp64, so any order gives the same bits
    dy_int = np.rint(P["dy"] * 8.0)
    _, _, dsh = oracle_mod.adaln_bwd(P["x"], P["scale"], dy_int, P["off"], 1e-6)
    assert np.array_equal(dsh[0], dy_int[:33].sum(axis=0))
    assert np.array_equal(dsh[1], dy_int[33:].sum(axis=0))
    # random dy: within 1e-12 (relative to the column's L1 mass) of the exact fsum
    _, _, dsh = oracle_mod.adaln_bwd(P["x"], P["scale"], P["dy"], P["off"], 1e-6)
    for d in range(12):
        ex = math.fsum(P["dy"][:33, d])
        assert abs(dsh[0, d] - ex) <= 1e-12 * np.abs(P["dy"][:33, d]).sum()
    # dy == 1: d_shift = N exactly
    _, _, dsh = oracle_mod.adaln_bwd(P["x"], P["scale"], np.ones_like(P["dy"]), P["off"], 1e-6)
    assert np.array_equal(dsh[0], np.full(12, 33.0)) and np.array_equal(dsh[1], np.full(12, 17.0))


def test_bwd_layernorm_invariants(oracle_mod):
    """sum_d dx = 0 per row; at eps = 0 also sum_d dx * xhat = 0."""
    P = _problem(9, seg=(10,), D=48)
    for eps in (1e-6, 0.0):
        dx, _, _ = oracle_mod.adaln_bwd(P["x"], P["scale"], P["dy"], P["off"], eps)
        g = P["dy"] * (1 + P["scale"][0])
        tol = 1e-12 * np.abs(g).sum(axis=1) * (1.0 / P["x"].std(axis=1))
        assert np.all(np.abs(dx.sum(axis=1)) <= tol)
        if eps == 0.0:
            xhat = (P["x"] - P["x"].mean(axis=1, keepdims=True)) / P["x"].std(axis=1, keepdims=True)
            assert np.all(np.abs((dx * xhat).sum(axis=1)) <= tol * 8)


def test_bwd_scale_grad_against_numpy_einsum(oracle_mod):
    P = _problem(10, seg=(9, 4), D=10)
    _, dsc, _ = oracle_mod.adaln_bwd(P["x"], P["scale"], P["dy"], P["off"], 1e-6)
    x = P["x"]
    xhat = (x - x.mean(axis=1, keepdims=True)) / np.sqrt(x.var(axis=1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(dsc[0], np.einsum("nd,nd->d", P["dy"][:9], xhat[:9]), atol=1e-12)
    np.testing.assert_allclose(dsc[1], np.einsum("nd,nd->d", P["dy"][9:], xhat[9:]), atol=1e-12)


# ----------------------------------------------------------------------------- gate

def test_gate_zero_gate_and_einsum(oracle_mod):
    P = _problem(11, seg=(6, 3), D=8)
    zero = np.zeros_like(P["gate"])
    out = oracle_mod.gate_residual(P["r"], P["z"], zero, P["off"])
    assert np.array_equal(out, P["r"])
    dz, dg = oracle_mod.gate_residual_bwd(P["dout"], P["z"], zero, P["off"])
    assert np.array_equal(dz, np.zeros_like(dz))
    np.testing.assert_allclose(dg[0], np.einsum("nd,nd->d", P["dout"][:6], P["z"][:6]), atol=1e-13)
    # gate = 1: out = r + z
    one = np.ones_like(P["gate"])
    out1 = oracle_mod.gate_residual(P["r"], P["z"], one, P["off"])
    assert np.array_equal(out1, P["r"] + P["z"])
    dz1, _ = oracle_mod.gate_residual_bwd(P["dout"], P["z"], one, P["off"])
    assert np.array_equal(dz1, P["dout"])


# ----------------------------------------------------------------------------- fused gated chain
# out = r + gate[k] * y with y the modulated LayerNorm (the chain as one node,
# section 2.B, "Simplificacion de Grafos").

def _torch_fused(P, k, eps, D):
    a, b = P["off"][k], P["off"][k + 1]
    xt = torch.from_numpy(P["x"][a:b].copy()).requires_grad_(True)
    w = torch.from_numpy(1.0 + P["scale"][k]).requires_grad_(True)
    bias = torch.from_numpy(P["shift"][k].copy()).requires_grad_(True)
    g = torch.from_numpy(P["gate"][k].copy()).requires_grad_(True)
    out = torch.from_numpy(P["r"][a:b]) + g * F.layer_norm(xt, (D,), weight=w, bias=bias, eps=eps)
    return out, (xt, w, bias, g)


def test_fused_fwd_equals_torch_and_reduces_to_parts(oracle_mod):
    """out is torch's fp64 r + gate * layer_norm(x; 1+scale, shift); gate = 0 gives r,
    gate = 1 with r = 0 gives the plain forward's y."""
    P = _problem(12, seg=(5, 0, 9), D=24)
    eps = 1e-6
    out, y, mean, rstd = oracle_mod.adaln_fwd_gated(P["x"], P["shift"], P["scale"], P["gate"],
                                                    P["r"], P["off"], eps)
    for k in range(len(P["off"]) - 1):
        a, b = P["off"][k], P["off"][k + 1]
        ref, _ = _torch_fused(P, k, eps, 24)
        np.testing.assert_allclose(out[a:b], ref.detach().numpy(), rtol=0, atol=1e-12)
    zero = np.zeros_like(P["gate"])
    out0, _, _, _ = oracle_mod.adaln_fwd_gated(P["x"], P["shift"], P["scale"], zero, P["r"],
                                               P["off"], eps)
    assert np.array_equal(out0, P["r"])
    one = np.ones_like(P["gate"])
    out1, _, _, _ = oracle_mod.adaln_fwd_gated(P["x"], P["shift"], P["scale"], one,
                                               np.zeros_like(P["r"]), P["off"], eps)
    yplain, _, _ = oracle_mod.adaln_fwd(P["x"], P["shift"], P["scale"], P["off"], eps)
    assert np.array_equal(out1, yplain)


def test_fused_bwd_equals_torch_autograd_fp64(oracle_mod):
    """dx, d_scale, d_shift, d_gate are the fp64 autograd gradients of sum(dout * out)."""
    P = _problem(13, seg=(6, 7), D=20)
    eps = 1e-6
    dx, dsc, dsh, dg = oracle_mod.adaln_bwd_gated(P["x"], P["shift"], P["scale"], P["gate"],
                                                  P["dout"], P["off"], eps)
    for k in range(2):
        a, b = P["off"][k], P["off"][k + 1]
        out, (xt, w, bias, g) = _torch_fused(P, k, eps, 20)
        (out * torch.from_numpy(P["dout"][a:b])).sum().backward()
        np.testing.assert_allclose(dx[a:b], xt.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dsc[k], w.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dsh[k], bias.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dg[k], g.grad.numpy(), rtol=0, atol=1e-12)


def test_fused_bwd_central_finite_differences_2x8x16(oracle_mod):
    """B=2, N=8, D=16: the fused backward agrees with central differences of the
    fused forward within 1e-6."""
    P = _problem(14, seg=(8, 8), D=16)
    eps = 1e-6

    def loss():
        out, _, _, _ = oracle_mod.adaln_fwd_gated(P["x"], P["shift"], P["scale"], P["gate"],
                                                  P["r"], P["off"], eps)
        return float(np.sum(P["dout"] * out))
    dx, dsc, dsh, dg = oracle_mod.adaln_bwd_gated(P["x"], P["shift"], P["scale"], P["gate"],
                                                  P["dout"], P["off"], eps)
    for name, grad in {"x": dx, "scale": dsc, "shift": dsh, "gate": dg, "r": P["dout"]}.items():
        base = P[name]
        fd = np.empty_like(base)
        for idx in np.ndindex(base.shape):
            v = base[idx]
            h = 1e-6 * max(1.0, abs(v))
            base[idx] = v + h
            lp = loss()
            base[idx] = v - h
            lm = loss()
            base[idx] = v
            fd[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(fd - grad))
        assert err < 1e-6, (name, err)


# ----------------------------------------------------------------------------- RMSNorm modulation

def test_rms_fwd_equals_torch_rms_norm(oracle_mod):
    """Per segment, y is torch's fp64 rms_norm with weight 1+scale[k], plus shift[k];
    rstd matches numpy's 1/sqrt(mean x^2 + eps)."""
    if not hasattr(F, "rms_norm"):
        pytest.skip("torch without rms_norm")
    P = _problem(15, seg=(5, 0, 9, 3), D=24)
    for eps in (1e-6, 1e-2):
        y, rstd = oracle_mod.rms_fwd(P["x"], P["shift"], P["scale"], P["off"], eps)
        for k in range(len(P["off"]) - 1):
            a, b = P["off"][k], P["off"][k + 1]
            ref = F.rms_norm(torch.from_numpy(P["x"][a:b]), (24,),
                             weight=torch.from_numpy(1.0 + P["scale"][k]), eps=eps).numpy()
            np.testing.assert_allclose(y[a:b], ref + P["shift"][k], rtol=0, atol=1e-12)
        np.testing.assert_allclose(rstd, 1.0 / np.sqrt((P["x"] ** 2).mean(axis=1) + eps),
                                   rtol=1e-13)


def test_rms_fwd_scale_invariance_at_eps0(oracle_mod):
    """With eps = 0, y(c x) = y(x) for c > 0 and rstd(c x) = rstd(x) / c; the mean is
    not removed, so y(x + c) != y(x)."""
    P = _problem(16, seg=(6, 4), D=16)
    y, r = oracle_mod.rms_fwd(P["x"], P["shift"], P["scale"], P["off"], 0.0)
    y2, r2 = oracle_mod.rms_fwd(4.0 * P["x"], P["shift"], P["scale"], P["off"], 0.0)
    np.testing.assert_allclose(y2, y, rtol=0, atol=1e-13)
    np.testing.assert_allclose(r2 * 4.0, r, rtol=1e-14)
    y3, _ = oracle_mod.rms_fwd(P["x"] + 3.0, P["shift"], P["scale"], P["off"], 0.0)
    assert np.max(np.abs(y3 - y)) > 0.1


def test_rms_bwd_equals_torch_autograd_fp64(oracle_mod):
    if not hasattr(F, "rms_norm"):
        pytest.skip("torch without rms_norm")
    P = _problem(17, seg=(5, 7), D=20)
    eps = 1e-6
    dx, dsc, dsh = oracle_mod.rms_bwd(P["x"], P["scale"], P["dy"], P["off"], eps)
    for k in range(2):
        a, b = P["off"][k], P["off"][k + 1]
        xt = torch.from_numpy(P["x"][a:b].copy()).requires_grad_(True)
        w = torch.from_numpy(1.0 + P["scale"][k]).requires_grad_(True)
        bias = torch.from_numpy(P["shift"][k].copy()).requires_grad_(True)
        y = F.rms_norm(xt, (20,), weight=w, eps=eps) + bias
        (y * torch.from_numpy(P["dy"][a:b])).sum().backward()
        np.testing.assert_allclose(dx[a:b], xt.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dsc[k], w.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dsh[k], bias.grad.numpy(), rtol=0, atol=1e-12)


def test_rms_bwd_central_finite_differences_2x8x16(oracle_mod):
    P = _problem(18, seg=(8, 8), D=16)
    eps = 1e-6

    def loss():
        y, _ = oracle_mod.rms_fwd(P["x"], P["shift"], P["scale"], P["off"], eps)
        return float(np.sum(P["dy"] * y))
    dx, dsc, dsh = oracle_mod.rms_bwd(P["x"], P["scale"], P["dy"], P["off"], eps)
    for name, grad in {"x": dx, "scale": dsc, "shift": dsh}.items():
        base = P[name]
        fd = np.empty_like(base)
        for idx in np.ndindex(base.shape):
            v = base[idx]
            h = 1e-6 * max(1.0, abs(v))
            base[idx] = v + h
            lp = loss()
            base[idx] = v - h
            lm = loss()
            base[idx] = v
            fd[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(fd - grad))
        assert err < 1e-6, (name, err)


# ----------------------------------------------------------------------------- inputs

def test_inputs_are_deterministic_and_rounded():
    s = workloads.Spec("t", "bf16", 16, 1e-6, (3, 5), outlier_frac=0.25)
    a = workloads.make_inputs(s, seed=0)
    b = workloads.make_inputs(s, seed=0)
    for k in a:
        assert torch.equal(a[k], b[k])
        assert a[k].dtype == torch.bfloat16
    assert a["x"].shape == (8, 16) and a["shift"].shape == (2, 16)
    big = (a["x"].float().abs().amax(dim=1) > 8).sum().item()
    assert big >= 1  # the two outlier rows (x20) dominate
    L = workloads.ragged_lengths(0)
    assert len(L) == 256 and min(L) >= 256 and max(L) <= 32768
    assert sum(1 for v in L if v == 256) >= 51


def test_indexed_modulation_gradients_by_finite_differences(oracle_mod):
    """Segments that share a modulation row (the indexed calls: segment k uses row
    mod_index[k] of a table).  Gathering the table rows and scattering the per-segment
    gradients back (the expected values of the indexed GPU tests) matches central
    differences of the loss with respect to the table itself."""
    P = _problem(11, seg=(4, 3, 5, 2), D=8)
    eps = 1e-6
    mod_index = np.array([1, 0, 1, 1])
    nmod = 3  # row 2 is used by no segment
    r = _rng(12)
    table = {k: 0.1 * r.standard_normal((nmod, 8)) for k in ("shift", "scale", "gate")}

    def loss():
        Q = dict(P)
        for k in table:
            Q[k] = table[k][mod_index]
        return _loss(oracle_mod, Q, eps)
    Q = dict(P)
    for k in table:
        Q[k] = table[k][mod_index]
    _, dsc, dsh = oracle_mod.adaln_bwd(Q["x"], Q["scale"], Q["dy"], Q["off"], eps)
    _, dg = oracle_mod.gate_residual_bwd(Q["dout"], Q["z"], Q["gate"], Q["off"])
    for name, per_seg in (("scale", dsc), ("shift", dsh), ("gate", dg)):
        scattered = np.zeros((nmod, 8))
        np.add.at(scattered, mod_index, per_seg)
        base = table[name]
        fd = np.empty_like(base)
        for idx in np.ndindex(base.shape):
            v = base[idx]
            h = 1e-6 * max(1.0, abs(v))
            base[idx] = v + h
            lp = loss()
            base[idx] = v - h
            lm = loss()
            base[idx] = v
            fd[idx] = (lp - lm) / (2 * h)
        assert np.max(np.abs(fd - scattered)) < 1e-6, name
        assert np.all(scattered[2] == 0.0)
