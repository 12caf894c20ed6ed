"""Host logic of the lookahead predictor (no GPU): the least-squares map that
carries a layer's input to the next layer's input."""
import torch

from activation_sparse_ffn_layer_gb300.lookahead import fit_map


def test_fit_map_recovers_an_exact_linear_relation():
    g = torch.Generator().manual_seed(5)
    d, n = 16, 400
    M = torch.randn(d, d, generator=g, dtype=torch.float64)
    X0 = torch.randn(d, n, generator=g, dtype=torch.float64)
    X1 = M @ X0
    Mf = fit_map(X0, X1, lam=1e-12)
    assert torch.allclose(Mf, M, rtol=1e-8, atol=1e-8)


def test_fit_map_ridge_shrinks_towards_zero():
    g = torch.Generator().manual_seed(6)
    d, n = 8, 100
    X0 = torch.randn(d, n, generator=g, dtype=torch.float64)
    X1 = 3.0 * X0
    small = fit_map(X0, X1, lam=1e-9)
    big = fit_map(X0, X1, lam=10.0)
    assert torch.allclose(small, 3.0 * torch.eye(d, dtype=torch.float64), atol=1e-6)
    assert big.norm() < 0.5 * small.norm()


def test_fit_map_is_the_normal_equations_solution():
    # the fitted map zeroes the gradient of ||X1 - M X0||^2 + reg ||M||^2
    g = torch.Generator().manual_seed(7)
    d, n, lam = 6, 50, 1e-2
    X0 = torch.randn(d, n, generator=g, dtype=torch.float64)
    X1 = torch.randn(d, n, generator=g, dtype=torch.float64)
    M = fit_map(X0, X1, lam=lam)
    reg = lam * torch.trace(X0 @ X0.T) / d
    grad = (M @ X0 - X1) @ X0.T + reg * M
    assert grad.abs().max() < 1e-9
