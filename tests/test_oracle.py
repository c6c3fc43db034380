"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test fixes some part of the oracle with an independent source: exact
arithmetic facts, closed forms, finite differences, torch's own fp64 autograd,
torch's fp32->bf16 conversion, or inputs (permutation weights) under which a
product reduces to a gather that can be checked element by element.  A dropped
term, a flipped sign, a transposed operand or a swapped left/gate split each
fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from bwd_gemm_epilogue_gb300 import ledger, workloads


# ----------------------------------------------------------------------------
# bf16 rounding
# ----------------------------------------------------------------------------

def test_round_bf16_hand_worked_ties():
    r = oracle.round_bf16
    assert r(1.0 + 2 ** -8) == 1.0                       # tie -> even mantissa (0)
    assert r(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6         # tie between mantissa 1 and 2 -> 2
    assert r(-(1.0 + 2 ** -8)) == -1.0
    assert r(1.0 + 2 ** -8 + 2 ** -30) == 1.0 + 2 ** -7  # just above the tie
    assert r(3.0) == 3.0
    assert r(2 ** -134) == 0.0                           # half the smallest subnormal: tie -> 0
    assert r(3 * 2 ** -134) == 2 ** -132                 # subnormal tie -> even
    assert r(3.39e38) == (2 - 2 ** -7) * 2.0 ** 127      # below the overflow midpoint
    assert math.isinf(r(3.4e38))                         # above it
    assert r(0.0) == 0.0 and math.isnan(r(float("nan")))


def test_round_bf16_matches_torch_fp32_conversion():
    g = torch.Generator().manual_seed(123)
    v = torch.randn(4000, generator=g, dtype=torch.float32)
    v = v * torch.exp2(torch.randint(-60, 60, (4000,), generator=g).float())
    want = v.to(torch.bfloat16).double().numpy()
    got = np.array([oracle.round_bf16(float(a)) for a in v.double().numpy()])
    np.testing.assert_array_equal(got, want)


# ----------------------------------------------------------------------------
# sigma, silu, silu'
# ----------------------------------------------------------------------------

def test_silu_prime_matches_central_difference():
    h = 1e-5
    for g in np.linspace(-20.0, 20.0, 401):
        fd = (oracle.silu(g + h) - oracle.silu(g - h)) / (2 * h)
        assert abs(fd - oracle.silu_prime(g)) < 1e-8, g


def test_silu_prime_three_forms_agree():
    # sigma + g*sigma*(1-sigma) = sigma*(1 + g*(1-sigma)) = sigma + silu*(1-sigma)
    for g in np.linspace(-20.0, 20.0, 81):
        s, si = oracle.sigmoid(g), oracle.silu(g)
        sp = oracle.silu_prime(g)
        assert abs(sp - (s + g * s * (1 - s))) < 1e-14
        assert abs(sp - (s + si * (1 - s))) < 1e-14


def test_sigmoid_silu_special_values():
    assert oracle.sigmoid(0.0) == 0.5
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu_prime(0.0) == 0.5
    e20 = 2.061153622438558e-09                     # e^-20
    assert abs(oracle.sigmoid(-20.0) - e20 / (1 + e20)) < 1e-22
    assert abs(oracle.sigmoid(20.0) - 1 / (1 + e20)) < 1e-16
    # silu'(20) = 1 + 19*e^-20 + O(e^-40); silu'(-20) = -19*e^-20 + O(e^-40)
    # (1 - sigma) cancels near sigma = 1: about 20 ulp of absolute slack
    assert abs(oracle.silu_prime(20.0) - (1 + 19 * e20)) < 5e-15
    assert abs(oracle.silu_prime(-20.0) - (-19 * e20)) < 1e-15
    # deep saturation: exp(-g) overflows to inf and sigma -> 0 exactly
    assert oracle.sigmoid(-800.0) == 0.0 and oracle.silu_prime(-800.0) == 0.0
    assert oracle.sigmoid(800.0) == 1.0 and oracle.silu_prime(800.0) == 1.0


# ----------------------------------------------------------------------------
# whole chain, unrounded: torch fp64 autograd and finite differences
# ----------------------------------------------------------------------------

def _rand64(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float64) * scale)


def _torch_chain(x, W1, W2, dy):
    x = x.clone().requires_grad_(True)
    W1 = W1.clone().requires_grad_(True)
    W2 = W2.clone().requires_grad_(True)
    preact = x @ W1.T
    preact.retain_grad()
    H = W1.shape[0] // 2
    left, gate = preact[:, :H], preact[:, H:]
    h = left * torch.nn.functional.silu(gate)
    y = h @ W2.T
    (y * dy).sum().backward()
    return dict(preact=preact.detach(), h=h.detach(), y=y.detach(), grad_preact=preact.grad,
                dx=x.grad, dW1=W1.grad, dW2=W2.grad)


@pytest.mark.parametrize("M,D,H,Dout", [(5, 8, 12, 6), (17, 16, 24, 40), (1, 8, 8, 8)])
def test_unrounded_chain_matches_torch_autograd(M, D, H, Dout):
    x, W1, W2, dy = (_rand64((M, D), 1), _rand64((2 * H, D), 2, D ** -0.5),
                     _rand64((Dout, H), 3, H ** -0.5), _rand64((M, Dout), 4))
    ref = _torch_chain(x, W1, W2, dy)
    preact, h, y = oracle.fwd(x, W1, W2, round_intermediates=False)
    gh, gp, h2, dx, dW1, dW2 = oracle.bwd_full(x, W1, W2, torch.from_numpy(preact), dy,
                                               round_intermediates=False)
    tol = dict(rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(preact, ref["preact"].numpy(), **tol)
    np.testing.assert_allclose(h, ref["h"].numpy(), **tol)
    np.testing.assert_allclose(h2, ref["h"].numpy(), **tol)
    np.testing.assert_allclose(y, ref["y"].numpy(), **tol)
    np.testing.assert_allclose(gh, (dy @ W2).numpy(), **tol)
    np.testing.assert_allclose(gp, ref["grad_preact"].numpy(), **tol)
    np.testing.assert_allclose(dx, ref["dx"].numpy(), **tol)
    np.testing.assert_allclose(dW1, ref["dW1"].numpy(), **tol)
    np.testing.assert_allclose(dW2, ref["dW2"].numpy(), **tol)


def test_unrounded_gradients_match_finite_differences():
    M, D, H, Dout = 4, 8, 16, 8
    x, W1, W2, dy = (_rand64((M, D), 11), _rand64((2 * H, D), 12, D ** -0.5),
                     _rand64((Dout, H), 13, H ** -0.5), _rand64((M, Dout), 14))
    xn, w1n, w2n, dyn = x.numpy(), W1.numpy(), W2.numpy(), dy.numpy()

    def loss(a, b, c):
        return float((oracle.fwd(a, b, c, round_intermediates=False)[2] * dyn).sum())

    preact, _, _ = oracle.fwd(xn, w1n, w2n, round_intermediates=False)
    _, _, _, dx, dW1, dW2 = oracle.bwd_full(xn, w1n, w2n, preact, dyn, round_intermediates=False)
    eps = 1e-6
    for which, arr, grad in (("x", xn, dx), ("W1", w1n, dW1), ("W2", w2n, dW2)):
        fd = np.empty_like(arr)
        for idx in np.ndindex(arr.shape):
            args = [xn.copy(), w1n.copy(), w2n.copy()]
            k = {"x": 0, "W1": 1, "W2": 2}[which]
            args[k][idx] += eps
            lp = loss(*args)
            args[k][idx] -= 2 * eps
            lm = loss(*args)
            fd[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8, err_msg=which)


# ----------------------------------------------------------------------------
# rounded chain: permutation weights reduce every product to a gather
# ----------------------------------------------------------------------------

def _perm_matrix(n, shift):
    P = torch.zeros(n, n, dtype=torch.float64)
    for i in range(n):
        P[i, (i + shift) % n] = 1.0
    return P


def test_rounded_chain_with_permutation_weights():
    # D = H = Dout = n.  W1 = [P_a ; P_b] makes preact[:, r] = x[:, pi(r)] exactly,
    # W2 = P_c makes y[:, o] = h[:, o + c] and grad_h[:, j] = dy[:, j - c].
    n, M = 24, 9
    a, b, c = 3, 7, 5
    g = torch.Generator().manual_seed(5)
    x = torch.randn(M, n, generator=g).mul(3).to(torch.bfloat16)
    dy = torch.randn(M, n, generator=g).to(torch.bfloat16)
    W1 = torch.cat([_perm_matrix(n, a), _perm_matrix(n, b)]).to(torch.bfloat16)
    W2 = _perm_matrix(n, c).to(torch.bfloat16)
    xd, dyd = x.double(), dy.double()
    preact, h, y = oracle.fwd(x, W1, W2)
    cols = np.arange(n)
    left_want = xd[:, (cols + a) % n].numpy()
    gate_want = xd[:, (cols + b) % n].numpy()
    np.testing.assert_array_equal(preact[:, :n], left_want)
    np.testing.assert_array_equal(preact[:, n:], gate_want)
    # h = bf16(left * bf16(silu(gate))); silu rounded by torch (fp64 -> fp32 -> bf16;
    # the product of two bf16 values is exact in fp32, so its rounding is single).
    silu_b = torch.nn.functional.silu(torch.from_numpy(gate_want)).float().to(torch.bfloat16)
    h_want = (torch.from_numpy(left_want).float() * silu_b.float()).to(torch.bfloat16).double()
    np.testing.assert_array_equal(h, h_want.numpy())
    np.testing.assert_array_equal(y, h[:, (cols + c) % n])

    pre_b = torch.from_numpy(preact).to(torch.bfloat16)
    gh, gp, h2, dx = oracle.bwd_rows(W1, W2, pre_b, dy)
    np.testing.assert_array_equal(gh, dyd[:, (cols - c) % n].numpy())
    np.testing.assert_array_equal(h2, h)
    # dx[:, d] = sum_r gp[:, r] W1[r, d] = gp[:, left row hitting d] + gp[:, gate row hitting d]
    np.testing.assert_allclose(dx, gp[:, (cols - a) % n] + gp[:, n + (cols - b) % n], rtol=0, atol=0)
    dW2c, dW1l, dW1g = oracle.bwd_cols(x, W2, pre_b, dy)
    np.testing.assert_allclose(dW1l, gp[:, :n].T @ xd.numpy(), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(dW1g, gp[:, n:].T @ xd.numpy(), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(dW2c.T, dyd.numpy().T @ h, rtol=1e-14, atol=1e-14)


def test_rounded_outputs_within_bf16_bound_of_exact():
    s, x, W1, W2, dy = workloads.make_block(workloads.Shape(40, 64, 96, 48), seed=9)
    p_r, h_r, y_r = oracle.fwd(x, W1, W2)
    p_e, h_e, y_e = oracle.fwd(x, W1, W2, round_intermediates=False)
    assert np.max(np.abs(p_r - p_e)) <= 2 ** -8 * np.max(np.abs(p_e))
    rel = np.linalg.norm(y_r - y_e) / np.linalg.norm(y_e)
    assert 0 < rel < 1e-2
    pre = torch.from_numpy(p_r).to(torch.bfloat16)
    out_r = oracle.bwd_full(x, W1, W2, pre, dy)
    out_e = oracle.bwd_full(x, W1, W2, pre, dy, round_intermediates=False)
    for a, b in zip(out_r[1:], out_e[1:]):
        assert np.linalg.norm(a - b) <= 1e-2 * np.linalg.norm(b)


def test_row_and_column_subsets_agree_with_full():
    s, x, W1, W2, dy = workloads.make_block(workloads.Shape(33, 40, 56, 24), seed=3)
    p, h, y = oracle.fwd(x, W1, W2)
    rows = [0, 7, 32, 7]
    p2, h2, y2 = oracle.fwd(x, W1, W2, rows=rows)
    np.testing.assert_array_equal(p2, p[rows]); np.testing.assert_array_equal(y2, y[rows])
    pre = torch.from_numpy(p).to(torch.bfloat16)
    gh, gp, hb, dx, dW1, dW2 = oracle.bwd_full(x, W1, W2, pre, dy)
    gh2, gp2, hb2, dx2 = oracle.bwd_rows(W1, W2, pre, dy, rows=rows)
    np.testing.assert_array_equal(gp2, gp[rows]); np.testing.assert_array_equal(dx2, dx[rows])
    cols = [55, 0, 13]
    c2, l2, g2 = oracle.bwd_cols(x, W2, pre, dy, cols=cols)
    np.testing.assert_array_equal(c2, dW2[:, cols].T)
    np.testing.assert_array_equal(l2, dW1[cols])
    np.testing.assert_array_equal(g2, dW1[[56 + c for c in cols]])


def test_tiny_workload_gate_sweep_saturates():
    s, x, W1, W2, dy = workloads.make_block("tiny")
    p, h, y = oracle.fwd(x, W1, W2, rows=[0, s.M - 1])
    assert p[0, s.H] == -20.0 and p[1, s.H] == 20.0
    assert h[0, 0] == 0.0 or abs(h[0, 0]) < 1e-6 * abs(p[0, 0]) + 1e-30
    pre = torch.from_numpy(oracle.fwd(x, W1, W2)[0]).to(torch.bfloat16)
    gh, gp, _, _ = oracle.bwd_rows(W1, W2, pre, dy, rows=[0, s.M - 1])
    # g = -20: dleft ~ grad_h * (-20 e^-20), dgate ~ grad_h * left * (-19 e^-20)
    assert abs(gp[0, 0]) <= 25 * 2.1e-9 * abs(gh[0, 0]) + 1e-30
    # g = +20: silu = 20, silu' ~ 1
    assert gp[1, 0] == oracle.round_bf16(gh[1, 0] * 20.0)


# ----------------------------------------------------------------------------
# FLOP ledger
# ----------------------------------------------------------------------------

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "printed_figures.json")))


@pytest.mark.parametrize("name", list(workloads.CONFIGS))
def test_backward_flops_are_twice_forward(name):
    s = workloads.CONFIGS[name]["shape"]
    f = ledger.gemm_flops(s.M, s.D, s.H, s.Dout)
    assert f["bwd"] == 2 * f["fwd"]
    # the per-GEMM proportions of the printed ledger (116 : 116 : 232 : 232, 696 = 2 x 348)
    g = GOLDEN["flop_ledger_gf"]
    for k in ("bwd_grad_h", "bwd_dW2", "bwd_dx", "bwd_dW1"):
        assert f[k] * g["bwd"] == g[k] * f["bwd"]
    assert g["bwd"] == 2 * g["fwd"] == g["bwd_grad_h"] + g["bwd_dW2"] + g["bwd_dx"] + g["bwd_dW1"]


def test_target_flops_and_activation_bytes():
    s = workloads.CONFIGS["target"]["shape"]
    f = ledger.gemm_flops(s.M, s.D, s.H, s.Dout)
    assert round(f["fwd"] / 1e9, 1) == 3433.0 and round(f["bwd"] / 1e9, 1) == 6866.0
    mem = GOLDEN["target_memory_mib"]
    # dropping h saves M*H bf16 after the forward
    assert round(s.M * s.H * 2 / 2 ** 20, 1) == mem["saved_by_drop_h"]
    assert round(mem["after_fwd_normal"] - mem["after_fwd_drop_h"], 1) == mem["saved_by_drop_h"]
    # what stays after the forward: preact [M,2H] + y [M,Dout] (plus allocator slack)
    assert abs((s.M * 2 * s.H + s.M * s.Dout) * 2 / 2 ** 20 - mem["after_fwd_drop_h"]) < 1.5
    st = GOLDEN["stack4_memory_mib"]
    assert round(st["after_fwd_normal"] - st["after_fwd_drop_h"], 1) == 4 * mem["saved_by_drop_h"]


# ----------------------------------------------------------------------------
# residual block y = x + MLP(x)
# ----------------------------------------------------------------------------

def test_residual_chain_matches_torch_autograd_and_finite_differences():
    M, D, H = 5, 8, 12
    x, W1, W2, dy = (_rand64((M, D), 21), _rand64((2 * H, D), 22, D ** -0.5),
                     _rand64((D, H), 23, H ** -0.5), _rand64((M, D), 24))
    ref = _torch_chain(x, W1, W2, dy)          # MLP part only; the residual adds x and passes dy
    _, _, y = oracle.fwd(x, W1, W2, round_intermediates=False, residual=True)
    np.testing.assert_allclose(y, (ref["y"] + x).numpy(), rtol=1e-11, atol=1e-12)
    preact, _, _ = oracle.fwd(x, W1, W2, round_intermediates=False)
    _, _, _, dx, dW1, dW2 = oracle.bwd_full(x, W1, W2, torch.from_numpy(preact), dy,
                                           round_intermediates=False, residual=True)
    np.testing.assert_allclose(dx, (ref["dx"] + dy).numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dW1, ref["dW1"].numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dW2, ref["dW2"].numpy(), rtol=1e-11, atol=1e-12)
    # finite differences of L = sum(dy * (x + MLP(x))) with respect to x
    xn, w1n, w2n, dyn = x.numpy(), W1.numpy(), W2.numpy(), dy.numpy()
    eps = 1e-6
    fd = np.empty_like(xn)
    for idx in np.ndindex(xn.shape):
        a = xn.copy()
        a[idx] += eps
        lp = float((oracle.fwd(a, w1n, w2n, round_intermediates=False, residual=True)[2] * dyn).sum())
        a[idx] -= 2 * eps
        lm = float((oracle.fwd(a, w1n, w2n, round_intermediates=False, residual=True)[2] * dyn).sum())
        fd[idx] = (lp - lm) / (2 * eps)
    np.testing.assert_allclose(dx, fd, rtol=1e-6, atol=1e-8)


def test_residual_with_zero_down_projection_is_the_identity():
    g = torch.Generator().manual_seed(31)
    M, D, H = 7, 16, 24
    x = torch.randn(M, D, generator=g).to(torch.bfloat16)
    dy = torch.randn(M, D, generator=g).to(torch.bfloat16)
    W1 = torch.randn(2 * H, D, generator=g).mul(D ** -0.5).to(torch.bfloat16)
    W2 = torch.zeros(D, H, dtype=torch.bfloat16)
    _, _, y = oracle.fwd(x, W1, W2, residual=True)
    np.testing.assert_array_equal(y, x.double().numpy())
    preact = torch.from_numpy(oracle.fwd(x, W1, W2)[0]).to(torch.bfloat16)
    _, gp, _, dx = oracle.bwd_rows(W1, W2, preact, dy, residual=True)
    assert not gp.any()                                   # grad_h = dy @ 0 = 0
    np.testing.assert_array_equal(dx, dy.double().numpy())


# ----------------------------------------------------------------------------
# mixture of experts: experts built from one dense block
# ----------------------------------------------------------------------------

def _expert_of(counts, t):
    # the expert owning global row t, by walking the segments one by one
    end = 0
    for e, c in enumerate(counts):
        end += c
        if t < end:
            return e
    raise IndexError(t)


def test_moe_experts_are_permuted_and_scaled_copies_of_one_block():
    # Expert e gets W1[e] = the base W1 with its hidden units permuted by pi_e (the same
    # permutation in the left and gate halves) and W2[e] = 2^e * base W2 with its columns
    # permuted by pi_e.  Hidden-unit permutations leave an MLP's output unchanged and a
    # power-of-two scale commutes with bf16 rounding, so for a token t of expert e:
    #   preact_moe[t] = preact[t] with both halves permuted by pi_e,
    #   y_moe[t] = 2^e y[t],  dx_moe[t] = 2^e dx[t]  (under dy),
    # and summing the experts' gradients back through their permutations and scales gives
    # the dense block's gradients over all tokens.  A wrong segment offset, a wrong
    # expert's weights or a transposed slice breaks one of these.
    E, D, H, Dout = 4, 24, 40, 16
    counts = [9, 0, 14, 5]
    T = sum(counts)
    g = torch.Generator().manual_seed(77)
    x = torch.randn(T, D, generator=g).to(torch.bfloat16)
    dy = torch.randn(T, Dout, generator=g).to(torch.bfloat16)
    W1 = (torch.randn(2 * H, D, generator=g) / D ** 0.5).to(torch.bfloat16)
    W2 = (torch.randn(Dout, H, generator=g) / H ** 0.5).to(torch.bfloat16)
    perms = [torch.randperm(H, generator=g) for _ in range(E)]
    W1e = torch.stack([torch.cat([W1[:H][p], W1[H:][p]]) for p in perms])
    W2e = torch.stack([W2[:, p] * 2.0 ** e for e, p in enumerate(perms)])

    p_d, h_d, y_d = oracle.fwd(x, W1, W2)
    p_m, h_m, y_m = oracle.moe_fwd(x, W1e, W2e, counts)
    pre = torch.from_numpy(p_d).to(torch.bfloat16)
    pre_m = torch.from_numpy(p_m).to(torch.bfloat16)
    _, gp_d, _, dx_d, dW1_d, dW2_d = oracle.bwd_full(x, W1, W2, pre, dy)
    _, gp_m, h2_m, dx_m, dW1_m, dW2_m = oracle.moe_bwd_full(x, W1e, W2e, pre_m, dy, counts)
    for t in range(T):
        e = _expert_of(counts, t)
        p = perms[e].numpy()
        np.testing.assert_array_equal(p_m[t, :H], p_d[t, :H][p])
        np.testing.assert_array_equal(p_m[t, H:], p_d[t, H:][p])
        np.testing.assert_array_equal(h_m[t], h_d[t][p])
        np.testing.assert_array_equal(h2_m[t], h_d[t][p])
        np.testing.assert_allclose(y_m[t], 2.0 ** e * y_d[t], rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(gp_m[t, :H], 2.0 ** e * gp_d[t, :H][p])
        np.testing.assert_allclose(dx_m[t], 2.0 ** e * dx_d[t], rtol=1e-12, atol=1e-11)
    dW1_sum = np.zeros_like(dW1_d)
    dW2_sum = np.zeros_like(dW2_d)
    for e, p in enumerate(perms):
        p = p.numpy()
        dW1_sum[p] += dW1_m[e][:H] / 2.0 ** e
        dW1_sum[H + p] += dW1_m[e][H:] / 2.0 ** e
        dW2_sum[:, p] += dW2_m[e]
    np.testing.assert_allclose(dW1_sum, dW1_d, rtol=1e-12, atol=1e-11)
    np.testing.assert_allclose(dW2_sum, dW2_d, rtol=1e-12, atol=1e-11)
    assert not dW1_m[1].any() and not dW2_m[1].any()       # the expert with no tokens


def test_moe_single_expert_is_the_dense_block_and_samples_agree():
    s = workloads.Shape(21, 16, 24, 32)
    _, x, W1, W2, dy = workloads.make_block(s, seed=78)
    p_d, _, y_d = oracle.fwd(x, W1, W2)
    p_m, _, y_m = oracle.moe_fwd(x, W1[None], W2[None], [21])
    np.testing.assert_array_equal(p_m, p_d)
    np.testing.assert_array_equal(y_m, y_d)
    # sampled rows / columns against the full computation, with three experts
    counts = [8, 0, 13]
    W1e = torch.stack([W1, W1.flip(0), -W1])
    W2e = torch.stack([W2, W2.flip(1), W2 * 0.5])
    pre = torch.from_numpy(oracle.moe_fwd(x, W1e, W2e, counts)[0]).to(torch.bfloat16)
    full = oracle.moe_bwd_full(x, W1e, W2e, pre, dy, counts)
    p_f, _, y_f = oracle.moe_fwd(x, W1e, W2e, counts)
    rows = [0, 7, 8, 20]
    p_r, y_r, gp_r, h_r, dx_r = oracle.moe_rows(x, W1e, W2e, pre, dy, counts, rows)
    np.testing.assert_array_equal(p_r, p_f[rows])
    np.testing.assert_array_equal(y_r, y_f[rows])
    np.testing.assert_array_equal(gp_r, full[1][rows])
    np.testing.assert_array_equal(dx_r, full[3][rows])
    cols = [1, 23]
    dW2c, dW1l, dW1g = oracle.moe_cols(x, W2e, pre, dy, counts, 2, cols)
    np.testing.assert_array_equal(dW2c, full[5][2][:, cols].T)
    np.testing.assert_array_equal(dW1l, full[4][2][cols])
    np.testing.assert_array_equal(dW1g, full[4][2][[24 + c for c in cols]])
    assert not oracle.moe_cols(x, W2e, pre, dy, counts, 1, cols)[1].any()


# ----------------------------------------------------------------------------
# FP8 E4M3 codes and the FP8 forward
# ----------------------------------------------------------------------------

def test_e4m3_decode_matches_torch_and_the_format():
    tv = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    ov = np.array([oracle.e4m3_decode(c) for c in range(256)])
    assert np.array_equal(np.isnan(ov), np.isnan(tv))
    fin = ~np.isnan(ov)
    np.testing.assert_array_equal(ov[fin], tv[fin])
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6 and oracle.e4m3_decode(0x38) == 1.0
    assert np.isnan(oracle.e4m3_decode(0x7F)) and np.isnan(oracle.e4m3_decode(0xFF))


def test_e4m3_encode_round_trip_ties_and_saturation():
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if not math.isnan(v):
            assert oracle.e4m3_encode(v) == c, c
    enc = oracle.e4m3_encode
    assert enc(2.0 ** -10) == 0x00             # half the smallest subnormal: tie -> even (0)
    assert enc(3 * 2.0 ** -10) == 0x02         # tie between codes 1 and 2 -> 2
    assert enc(2.0 ** -10 + 2.0 ** -30) == 0x01
    assert enc(1.0625) == 0x38                 # tie between 1 and 1.125 -> 1 (even)
    assert enc(1.1875) == 0x3A                 # tie between 1.125 and 1.25 -> 1.25
    assert enc(449.0) == 0x7E and enc(464.0) == 0x7E and enc(1e9) == 0x7E and enc(-1e9) == 0xFE
    assert enc(float("nan")) == 0x7F


def test_e4m3_encode_matches_torch_in_range():
    g = torch.Generator().manual_seed(9)
    v = torch.randn(3000, generator=g) * torch.exp2(torch.randint(-12, 8, (3000,), generator=g).float())
    v = v.clamp(-440.0, 440.0)
    # every midpoint between neighbouring positive codes, both signs
    vals = torch.arange(0, 0x7E, dtype=torch.uint8).view(torch.float8_e4m3fn).float()
    mids = (vals[:-1] + vals[1:]) / 2
    v = torch.cat([v, mids, -mids])
    want = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(a)) for a in v.double().numpy()])
    np.testing.assert_array_equal(got, want)


def test_fp8_forward_against_the_bf16_oracle_and_fp64_matmul():
    # Power-of-two scales make the dequantised inputs exact, so the FP8 forward's
    # preact must equal the bf16 oracle's preact on the dequantised fp64 inputs; its h
    # before quantisation, rounded to bf16, the bf16 oracle's h; its h8 the nearest
    # E4M3 code of h / s_h (within half a code spacing, or saturated); and its y the
    # fp64 product of the dequantised h8 and W2.
    s = workloads.Shape(33, 48, 40, 24)
    x8, W1_8, W2_8, sc = workloads.make_fp8_block(s, seed=90, s_h=1.0 / 256)   # saturates above 1.75
    p8, hpre, h8, y8 = oracle.fwd_fp8(x8, W1_8, W2_8, **sc)
    deq = lambda t, sv: torch.from_numpy(  # noqa: E731
        np.array([oracle.e4m3_decode(c) for c in t.view(torch.uint8).flatten().tolist()]).reshape(t.shape) * sv)
    x, W1, W2 = deq(x8, sc["s_x"]), deq(W1_8, sc["s_w1"]), deq(W2_8, sc["s_w2"])
    p_ref, h_ref, _ = oracle.fwd(x, W1, W2)
    np.testing.assert_array_equal(p8, p_ref)
    np.testing.assert_array_equal(np.vectorize(oracle.round_bf16)(hpre), h_ref)
    hq = np.vectorize(oracle.e4m3_decode)(h8.astype(np.int64))
    q = hpre / sc["s_h"]
    sat = np.abs(q) >= 448
    assert sat.any() and (~sat).any()
    np.testing.assert_array_equal(hq[sat], np.sign(q[sat]) * 448)
    a = np.abs(q[~sat])
    spacing = np.where(a < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -6))) - 3))
    assert (np.abs(hq[~sat] - q[~sat]) <= spacing / 2).all()
    y_ref = (hq * sc["s_h"]) @ W2.numpy().T
    np.testing.assert_array_equal(y8, y_ref)
    # row subsets agree with the full computation
    r = oracle.fwd_fp8(x8, W1_8, W2_8, rows=[0, 17, 32], **sc)
    np.testing.assert_array_equal(r[2], h8[[0, 17, 32]])
    np.testing.assert_array_equal(r[3], y8[[0, 17, 32]])


def test_identity_down_projection_passes_dy_through():
    # W2 = I (H = Dout): grad_h = dy @ W2 = dy exactly, so the backward's grad_preact is
    # [dy * silu(gate) | dy * left * silu'(gate)] element by element
    s = workloads.Shape(12, 16, 24, 24)
    _, x, W1, _, dy = workloads.make_block(s, seed=79)
    W2 = torch.eye(24).to(torch.bfloat16)
    preact = workloads.make_preact(s, seed=79)
    gh, gp, _, _ = oracle.bwd_rows(W1, W2, preact, dy)
    np.testing.assert_array_equal(gh, dy.double().numpy())
    p = preact.double().numpy()
    left, gate = p[:, :24], p[:, 24:]
    sg = 1.0 / (1.0 + np.exp(-gate))
    want_l = np.vectorize(oracle.round_bf16)(dy.double().numpy() * gate * sg)
    np.testing.assert_allclose(gp[:, :24], want_l, rtol=0, atol=0)
    # dgate with its single bf16 rounding: silu' written in the drop-h report's form
    # sigma + silu * (1 - sigma) (the oracle evaluates sigma * (1 + g * (1 - sigma))),
    # times left and grad_h = dy, rounded once
    silu_p = sg + gate * sg * (1.0 - sg)
    want_g = np.vectorize(oracle.round_bf16)(dy.double().numpy() * left * silu_p)
    np.testing.assert_allclose(gp[:, 24:], want_g, rtol=0, atol=0)
    # the rounding point matters: the unrounded products differ from the stored values
    assert np.any(dy.double().numpy() * left * silu_p != gp[:, 24:])
