"""Pins of the fp64 convolution-derivative oracle against facts outside itself
(no GPU): hand-derived worked examples, finite differences, the adjoint identity
of a linear map, 1x1 convolutions as matrix products, torch's float64
convolution and its gradients, and the gather forms against the scatter forms.

The operation is the 2-D convolution whose input and weight derivatives
"Meganeura: Portable GPU Training and Inference through Vulkan and Metal" lists
among its backward nodes (Section 3.1) and names as the kernels owning its
ResNet-50 training gap (Section 7.3)."""
import json
import os

import numpy as np
import pytest

from oracle import conv as oc

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "conv_tiny.json")


def _rand(rng, *shape):
    return rng.standard_normal(shape)


@pytest.mark.parametrize("case", range(2))
def test_golden_worked_examples(case):
    g = json.load(open(GOLDEN))["cases"][case]
    X = np.array(g["X"], dtype=np.float64)[None, :, :, None]
    Wt = np.array(g["Wt"], dtype=np.float64)[None, :, :, None]
    dY = np.array(g["dY"], dtype=np.float64)[None, :, :, None]
    st, pad = g["stride"], g["pad"]
    R, S = Wt.shape[1:3]
    assert np.array_equal(oc.conv2d_fwd(X, Wt, st, pad)[0, :, :, 0], np.array(g["Y"]))
    assert np.array_equal(oc.conv2d_grad_input(dY, Wt, 3, 3, st, pad)[0, :, :, 0],
                          np.array(g["dX"]))
    assert np.array_equal(oc.conv2d_grad_weight(X, dY, R, S, st, pad)[0, :, :, 0],
                          np.array(g["dW"]))


SHAPES = [
    # N, H, W, C, K, R, S, stride, pad
    (2, 5, 6, 3, 4, 3, 2, 1, 1),
    (1, 7, 5, 2, 3, 3, 3, 2, 1),
    (2, 6, 6, 4, 2, 1, 1, 2, 0),
    (1, 9, 8, 3, 2, 5, 4, 3, 2),
    (3, 4, 4, 2, 5, 4, 4, 1, 0),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_finite_differences(shape):
    """sum(G * Y) is linear in X and in Wt, so its central difference equals the
    gradient up to rounding: dL/dX = grad_input(G, Wt), dL/dWt = grad_weight(X, G)."""
    N, H, W, C, K, R, S, st, pad = shape
    rng = np.random.default_rng(hash(shape) % 2**32)
    X, Wt = _rand(rng, N, H, W, C), _rand(rng, K, R, S, C)
    P, Q = oc.out_size(H, W, R, S, st, pad)
    G = _rand(rng, N, P, Q, K)
    dX = oc.conv2d_grad_input(G, Wt, H, W, st, pad)
    dW = oc.conv2d_grad_weight(X, G, R, S, st, pad)
    loss = lambda X_, W_: float(np.sum(G * oc.conv2d_fwd(X_, W_, st, pad)))
    h = 1e-3
    for _ in range(12):
        i = tuple(rng.integers(0, d) for d in X.shape)
        Xp, Xm = X.copy(), X.copy()
        Xp[i] += h
        Xm[i] -= h
        fd = (loss(Xp, Wt) - loss(Xm, Wt)) / (2 * h)
        assert abs(fd - dX[i]) <= 1e-8 * (1 + abs(dX[i])), (i, fd, dX[i])
        j = tuple(rng.integers(0, d) for d in Wt.shape)
        Wp, Wm = Wt.copy(), Wt.copy()
        Wp[j] += h
        Wm[j] -= h
        fd = (loss(X, Wp) - loss(X, Wm)) / (2 * h)
        assert abs(fd - dW[j]) <= 1e-8 * (1 + abs(dW[j])), (j, fd, dW[j])


@pytest.mark.parametrize("shape", SHAPES)
def test_adjoint_identity(shape):
    """<Y(X, Wt), G> = <X, dX(G, Wt)> = <Wt, dW(X, G)>."""
    N, H, W, C, K, R, S, st, pad = shape
    rng = np.random.default_rng(7 + hash(shape) % 2**31)
    X, Wt = _rand(rng, N, H, W, C), _rand(rng, K, R, S, C)
    P, Q = oc.out_size(H, W, R, S, st, pad)
    G = _rand(rng, N, P, Q, K)
    a = np.sum(oc.conv2d_fwd(X, Wt, st, pad) * G)
    b = np.sum(X * oc.conv2d_grad_input(G, Wt, H, W, st, pad))
    c = np.sum(Wt * oc.conv2d_grad_weight(X, G, R, S, st, pad))
    assert abs(a - b) <= 1e-10 * (1 + abs(a)) and abs(a - c) <= 1e-10 * (1 + abs(a))


def test_one_by_one_is_a_matrix_product():
    """A 1x1 convolution with stride 1 and no padding is Y = X Wt^T over pixels:
    dX = dY Wt and dW = dY^T X (numpy matmul)."""
    rng = np.random.default_rng(11)
    N, H, W, C, K = 2, 3, 5, 6, 4
    X, Wt = _rand(rng, N, H, W, C), _rand(rng, K, 1, 1, C)
    dY = _rand(rng, N, H, W, K)
    Xm, dYm, Wm = X.reshape(-1, C), dY.reshape(-1, K), Wt.reshape(K, C)
    np.testing.assert_allclose(oc.conv2d_fwd(X, Wt, 1, 0).reshape(-1, K), Xm @ Wm.T, rtol=1e-12,
                               atol=1e-12)
    np.testing.assert_allclose(oc.conv2d_grad_input(dY, Wt, H, W, 1, 0).reshape(-1, C), dYm @ Wm,
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oc.conv2d_grad_weight(X, dY, 1, 1, 1, 0).reshape(K, C),
                               dYm.T @ Xm, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("shape", SHAPES)
def test_torch_float64(shape):
    """torch's float64 conv2d (NCHW) and its input/weight gradients."""
    torch = pytest.importorskip("torch")
    N, H, W, C, K, R, S, st, pad = shape
    rng = np.random.default_rng(23 + hash(shape) % 2**31)
    X, Wt = _rand(rng, N, H, W, C), _rand(rng, K, R, S, C)
    P, Q = oc.out_size(H, W, R, S, st, pad)
    dY = _rand(rng, N, P, Q, K)
    tX = torch.from_numpy(X).permute(0, 3, 1, 2)
    tW = torch.from_numpy(Wt).permute(0, 3, 1, 2)
    tG = torch.from_numpy(dY).permute(0, 3, 1, 2)
    Y = torch.nn.functional.conv2d(tX, tW, stride=st, padding=pad).permute(0, 2, 3, 1).numpy()
    np.testing.assert_allclose(oc.conv2d_fwd(X, Wt, st, pad), Y, rtol=1e-12, atol=1e-12)
    gi = torch.nn.grad.conv2d_input(tX.shape, tW, tG, stride=st, padding=pad)
    gw = torch.nn.grad.conv2d_weight(tX, tW.shape, tG, stride=st, padding=pad)
    np.testing.assert_allclose(oc.conv2d_grad_input(dY, Wt, H, W, st, pad),
                               gi.permute(0, 2, 3, 1).numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oc.conv2d_grad_weight(X, dY, R, S, st, pad),
                               gw.permute(0, 2, 3, 1).numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("shape", SHAPES)
def test_gather_forms_match_scatter_forms(shape):
    N, H, W, C, K, R, S, st, pad = shape
    rng = np.random.default_rng(31 + hash(shape) % 2**31)
    X, Wt = _rand(rng, N, H, W, C), _rand(rng, K, R, S, C)
    P, Q = oc.out_size(H, W, R, S, st, pad)
    dY = _rand(rng, N, P, Q, K)
    dX = oc.conv2d_grad_input(dY, Wt, H, W, st, pad)
    dW = oc.conv2d_grad_weight(X, dY, R, S, st, pad)
    pi = np.stack([rng.integers(0, d, 40) for d in dX.shape], axis=1)
    pw = np.stack([rng.integers(0, d, 40) for d in dW.shape], axis=1)
    np.testing.assert_allclose(oc.conv2d_grad_input_at(dY, Wt, H, W, st, pad, pi),
                               dX[tuple(pi.T)], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oc.conv2d_grad_weight_at(X, dY, R, S, st, pad, pw),
                               dW[tuple(pw.T)], rtol=1e-12, atol=1e-12)


def test_rejects_bad_shapes():
    X = np.zeros((1, 2, 2, 1))
    with pytest.raises(RuntimeError):
        oc.conv2d_fwd(X, np.zeros((1, 3, 3, 1)), 1, 0)  # kernel larger than the padded image
    with pytest.raises(ValueError):
        oc.conv2d_grad_input(np.zeros((1, 2, 2, 1)), np.zeros((1, 2, 2, 1)), 2, 2, 1, 0)
    with pytest.raises(RuntimeError):
        oc.conv2d_grad_input_at(np.zeros((1, 1, 1, 1)), np.zeros((1, 2, 2, 1)), 2, 2, 1, 0,
                                [[0, 5, 0, 0]])
