"""Pins of the fp64 oracle against facts fixed by the mathematics, not by the
oracle itself (no GPU needed).

The pages ("Meganeura: Portable GPU Training and Inference through Vulkan and
Metal") print no attention formula and no worked example; what they fix is that
attention is one node with an analytic derivative (Section 3.1), split into a
forward, a dQ and a fused dK+dV kernel (Section 3.3), with an exact CPU
reference as the independent check (Section 5.2). Each test below would fail
for a plausible slip in the oracle: a dropped term, a wrong sign, a transposed
operand, an off-by-one causal mask, a base-2 LSE, a missing scale.
"""
import math

import numpy as np
import pytest

import oracle
from attention_forward_backward_gb300 import synth

RNG = np.random.default_rng(12345)


def rand(*shape, gain=1.0):
    return RNG.standard_normal(shape) * gain


def loss(Q, K, V, dO, causal, scale):
    O, _ = oracle.attn_fwd(Q, K, V, causal, scale)
    return float(np.sum(O * dO))


# ---------------------------------------------------------------- gradients
@pytest.mark.parametrize("L", [1, 3, 5, 8])
@pytest.mark.parametrize("D", [2, 4])
@pytest.mark.parametrize("causal", [True, False])
def test_central_finite_differences(L, D, causal):
    """dQ, dK, dV equal central differences of loss = sum(dO * O)."""
    Q, K, V, dO = (rand(1, 2, L, D) for _ in range(4))
    scale = 0.7
    g = oracle.attn_bwd(Q, K, V, dO, causal, scale)
    h = 1e-6
    for name, X in (("dQ", Q), ("dK", K), ("dV", V)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            orig = X[idx]
            X[idx] = orig + h
            lp = loss(Q, K, V, dO, causal, scale)
            X[idx] = orig - h
            lm = loss(Q, K, V, dO, causal, scale)
            X[idx] = orig
            num[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(num - g[name])) / max(np.max(np.abs(num)), 1e-30)
        # L = 1 has identically zero dQ and dK: compare absolutely there.
        if np.max(np.abs(num)) < 1e-8:
            assert np.max(np.abs(g[name])) < 1e-12, name
        else:
            assert err < 1e-6, (name, err)


def test_backward_forward_agree():
    """The O and LSE the backward recomputes equal the forward's."""
    Q, K, V, dO = (rand(2, 3, 17, 8) for _ in range(4))
    O, LSE = oracle.attn_fwd(Q, K, V, True, 0.3)
    g = oracle.attn_bwd(Q, K, V, dO, True, 0.3)
    np.testing.assert_array_equal(O, g["O"])
    np.testing.assert_array_equal(LSE, g["LSE"])
    np.testing.assert_allclose(g["Dvec"], np.sum(dO * O, axis=-1), rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- softmax
@pytest.mark.parametrize("causal", [True, False])
def test_softmax_rows_sum_to_one(causal):
    """With V = all ones every output element is sum_j P_ij, which must be 1."""
    L, D = 33, 6
    Q, K = rand(2, L, D, gain=3.0), rand(2, L, D, gain=3.0)
    V = np.ones((2, L, D))
    O, LSE = oracle.attn_fwd(Q, K, V, causal, 0.5)
    np.testing.assert_allclose(O, 1.0, rtol=0, atol=1e-12)


def test_lse_is_natural_log_of_scaled_scores():
    """LSE_i = ln sum_j exp(scale q_i.k_j) (natural log, scaled logits).

    Evaluated independently with math.fsum over math.exp of each logit."""
    L, D, scale = 9, 5, 0.37
    Q, K, V = rand(L, D), rand(L, D), rand(L, D)
    _, LSE = oracle.attn_fwd(Q, K, V, True, scale)
    for i in range(L):
        ref = math.log(math.fsum(math.exp(scale * float(np.dot(Q[i], K[j])))
                                 for j in range(i + 1)))
        assert abs(LSE[i] - ref) < 1e-12


# ---------------------------------------------------------------- causal cases
def test_causal_first_row():
    """Row 0 sees only key 0: O[0] = V[0] exactly, LSE[0] = s_00, dQ[0] = 0."""
    L, D, scale = 12, 7, 0.9
    Q, K, V, dO = (rand(L, D) for _ in range(4))
    g = oracle.attn_bwd(Q, K, V, dO, True, scale)
    np.testing.assert_array_equal(g["O"][0], V[0])
    assert abs(g["LSE"][0] - scale * float(np.dot(Q[0], K[0]))) < 1e-13
    np.testing.assert_allclose(g["dQ"][0], 0.0, atol=1e-15)
    # the last key is seen only by the last query
    p_last = math.exp(scale * float(np.dot(Q[-1], K[-1])) - g["LSE"][-1])
    np.testing.assert_allclose(g["dV"][-1], p_last * dO[-1], rtol=1e-12, atol=1e-14)


def test_causal_mask_is_top_left_inclusive():
    """Changing a key after position i must not change output row i."""
    L, D = 10, 4
    Q, K, V = rand(L, D), rand(L, D), rand(L, D)
    O1, L1 = oracle.attn_fwd(Q, K, V, True, 0.5)
    K2, V2 = K.copy(), V.copy()
    K2[6:] += 5.0
    V2[6:] -= 3.0
    O2, L2 = oracle.attn_fwd(Q, K2, V2, True, 0.5)
    np.testing.assert_array_equal(O1[:6], O2[:6])
    np.testing.assert_array_equal(L1[:6], L2[:6])
    assert np.max(np.abs(O1[6:] - O2[6:])) > 1e-3


# ---------------------------------------------------------------- dV, dO = 1
@pytest.mark.parametrize("causal", [True, False])
def test_dv_with_unit_dO_is_column_sums_of_P(causal):
    """dV = P^T dO; with dO = 1 each dV_j is the column sum of P (all d equal)
    and the column sums add up to L (each row of P sums to one)."""
    L, D, scale = 21, 6, 0.4
    Q, K, V = rand(L, D), rand(L, D), rand(L, D)
    dO = np.ones((L, D))
    g = oracle.attn_bwd(Q, K, V, dO, causal, scale)
    col = g["dV"][:, 0]
    np.testing.assert_allclose(g["dV"], np.repeat(col[:, None], D, axis=1), rtol=1e-13)
    assert abs(col.sum() - L) < 1e-11
    # column sums from the oracle's own forward: P_ij = O of a one-hot V
    for j in (0, L // 2, L - 1):
        Vj = np.zeros((L, 1))
        Vj[j] = 1.0
        Pcol, _ = oracle.attn_fwd(Q, K, np.repeat(Vj, D, axis=1), causal, scale)
        assert abs(Pcol[:, 0].sum() - col[j]) < 1e-12


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("causal", [True, False])
def test_sum_of_dK_is_zero(causal):
    """Rows of dS sum to zero (softmax Jacobian), hence sum_j dK_j = 0."""
    Q, K, V, dO = (rand(3, 25, 8) for _ in range(4))
    g = oracle.attn_bwd(Q, K, V, dO, causal, 0.6)
    s = np.sum(g["dK"], axis=-2)
    assert np.max(np.abs(s)) < 1e-12 * max(1.0, np.max(np.abs(g["dK"])))


def test_equal_keys_closed_forms():
    """All keys equal: P is uniform over allowed keys, so O_i is the (prefix)
    mean of V, and dQ = scale * K_0 * sum_j dS_ij = 0."""
    L, D = 15, 5
    Q, V, dO = rand(L, D), rand(L, D), rand(L, D)
    K = np.repeat(rand(1, D), L, axis=0)
    for causal in (True, False):
        g = oracle.attn_bwd(Q, K, V, dO, causal, 0.8)
        if causal:
            mean = np.cumsum(V, axis=0) / np.arange(1, L + 1)[:, None]
        else:
            mean = np.repeat(V.mean(axis=0, keepdims=True), L, axis=0)
        np.testing.assert_allclose(g["O"], mean, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(g["dQ"], 0.0, atol=1e-13)


def test_single_key():
    """L = 1: O = V, dV = dO, dQ = dK = 0, LSE = s_00."""
    Q, K, V, dO = (rand(2, 1, 6) for _ in range(4))
    for causal in (True, False):
        g = oracle.attn_bwd(Q, K, V, dO, causal, 1.3)
        np.testing.assert_array_equal(g["O"], V)
        np.testing.assert_allclose(g["dV"], dO, rtol=1e-15)
        np.testing.assert_array_equal(g["dQ"], 0.0)
        np.testing.assert_array_equal(g["dK"], 0.0)
        np.testing.assert_allclose(g["LSE"][:, 0], 1.3 * np.sum(Q[:, 0] * K[:, 0], axis=-1),
                                   rtol=1e-14)


def test_key_shift_metamorphic():
    """K_j + c for every j leaves P and O unchanged and shifts LSE_i by
    scale * (Q_i . c)."""
    L, D, scale = 19, 6, 0.45
    Q, K, V = rand(L, D), rand(L, D), rand(L, D)
    c = rand(D)
    for causal in (True, False):
        O1, L1 = oracle.attn_fwd(Q, K, V, causal, scale)
        O2, L2 = oracle.attn_fwd(Q, K + c, V, causal, scale)
        np.testing.assert_allclose(O2, O1, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(L2 - L1, scale * Q @ c, rtol=1e-11, atol=1e-12)


def test_two_key_closed_form():
    """Two keys, no mask, D = 1: P_i1 = sigmoid(s_i1 - s_i0), so
    O_i = V_0 + sigmoid(s_i1 - s_i0) (V_1 - V_0); LSE_i = s_i0 + ln(1 + e^(s_i1 - s_i0))."""
    Q = np.array([[0.5], [-1.25]])
    K = np.array([[2.0], [-0.75]])
    V = np.array([[3.0], [-1.0]])
    scale = 0.8
    O, LSE = oracle.attn_fwd(Q, K, V, False, scale)
    for i in range(2):
        s0, s1 = scale * Q[i, 0] * K[0, 0], scale * Q[i, 0] * K[1, 0]
        sig = 1.0 / (1.0 + math.exp(-(s1 - s0)))
        assert abs(O[i, 0] - (V[0, 0] + sig * (V[1, 0] - V[0, 0]))) < 1e-14
        assert abs(LSE[i] - (s0 + math.log1p(math.exp(s1 - s0)))) < 1e-14


def test_rows_variant_matches_full():
    Q, K, V = rand(40, 8), rand(40, 8), rand(40, 8)
    rows = [0, 1, 17, 39]
    O, LSE = oracle.attn_fwd(Q, K, V, True, 0.35)
    Or, Lr = oracle.attn_fwd_rows(Q, K, V, rows, True, 0.35)
    np.testing.assert_array_equal(Or, O[rows])
    np.testing.assert_array_equal(Lr, LSE[rows])


def test_thread_count_does_not_change_results():
    Q, K, V, dO = (rand(2, 2, 31, 8) for _ in range(4))
    a = oracle.attn_bwd(Q, K, V, dO, True, 0.5, nthreads=1)
    b = oracle.attn_bwd(Q, K, V, dO, True, 0.5, nthreads=4)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


def test_large_logits_are_stable():
    """Logit std ~ 40: the max-shifted LSE stays finite, rows still sum to 1."""
    Q, K = rand(64, 16, gain=10.0), rand(64, 16, gain=10.0)
    O, LSE = oracle.attn_fwd(Q, K, np.ones((64, 16)), True, 0.25)
    assert np.all(np.isfinite(LSE))
    np.testing.assert_allclose(O, 1.0, atol=1e-12)


# ---------------------------------------------------------------- library cross-check
@pytest.mark.parametrize("causal", [True, False])
def test_torch_float64_sdpa_autograd(causal):
    """Third implementation: torch CPU float64 SDPA + autograd on tiny shapes."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    B, H, L, D, scale = 2, 3, 11, 5, 0.55
    Q, K, V, dO = (rand(B, H, L, D) for _ in range(4))
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    out = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    out.backward(torch.tensor(dO, dtype=torch.float64))
    g = oracle.attn_bwd(Q, K, V, dO, causal, scale)
    np.testing.assert_allclose(g["O"], out.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dQ"], tq.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(g["dK"], tk.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(g["dV"], tv.grad.numpy(), rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- the input generator
def test_splitmix64_published_vector():
    """First outputs of SplitMix64 seeded with 1234567, as published with the
    reference C implementation of the generator."""
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    assert [int(v) for v in synth.splitmix64(1234567, 0, 5)] == want


def test_normals_are_standard_and_deterministic():
    a = synth.normal_f32(4242, 1 << 18)
    b = synth.normal_f32(4242, 1 << 18, chunk=1000)
    np.testing.assert_array_equal(a, b)
    assert abs(float(a.mean())) < 0.01 and abs(float(a.std()) - 1.0) < 0.01


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.concatenate([synth.normal_f32(5, 4096) * 3,
                        # exact ties: halfway between two bf16 values
                        np.array([1.0 + 2**-8, 1.0 + 3 * 2**-8, -(1.0 + 2**-8)], np.float32)])
    ours = synth.round_to_bf16(x)
    ref = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


# ---------------------------------------------------------------- cross attention and mask alignment
MASKS_EX = ("none", "causal", "causal_bottom_right")


def loss_ex(Q, K, V, dO, mask, scale):
    O, _ = oracle.attn_fwd_ex(Q, K, V, mask, scale)
    return float(np.sum(O * dO))


@pytest.mark.parametrize("Lq,Lk", [(3, 5), (5, 3), (1, 4), (4, 1)])
@pytest.mark.parametrize("mask", MASKS_EX)
def test_cross_attention_finite_differences(Lq, Lk, mask):
    """Lq != Lk: dQ, dK, dV equal central differences of sum(dO * O) for every
    mask alignment, including rows with an empty softmax (their O is constant 0,
    so they contribute nothing)."""
    D, scale, h = 3, 0.6, 1e-6
    Q, dO = rand(1, 2, Lq, D), rand(1, 2, Lq, D)
    K, V = rand(1, 2, Lk, D), rand(1, 2, Lk, D)
    g = oracle.attn_bwd_ex(Q, K, V, dO, mask, scale)
    for name, X in (("dQ", Q), ("dK", K), ("dV", V)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            orig = X[idx]
            X[idx] = orig + h
            lp = loss_ex(Q, K, V, dO, mask, scale)
            X[idx] = orig - h
            lm = loss_ex(Q, K, V, dO, mask, scale)
            X[idx] = orig
            num[idx] = (lp - lm) / (2 * h)
        if np.max(np.abs(num)) < 1e-8:
            assert np.max(np.abs(g[name])) < 1e-12, name
        else:
            err = np.max(np.abs(num - g[name])) / np.max(np.abs(num))
            assert err < 1e-6, (name, err)


def test_mask_alignments_coincide_when_square():
    """With Lq = Lk the top-left and bottom-right causal masks are the same mask,
    and the self-attention entry points agree with the general ones."""
    Q, K, V, dO = (rand(2, 2, 9, 4) for _ in range(4))
    a = oracle.attn_bwd_ex(Q, K, V, dO, "causal", 0.4)
    b = oracle.attn_bwd_ex(Q, K, V, dO, "causal_bottom_right", 0.4)
    c = oracle.attn_bwd(Q, K, V, dO, True, 0.4)
    for k in ("O", "LSE", "dQ", "dK", "dV"):
        np.testing.assert_array_equal(a[k], b[k])
        np.testing.assert_array_equal(a[k], c[k])


def test_single_query_bottom_right_sees_every_key():
    """One query aligned at the bottom right attends to all Lk keys: the same as
    no mask, and (for the top-left alignment) only key 0."""
    Q, dO = rand(1, 1, 1, 6), rand(1, 1, 1, 6)
    K, V = rand(1, 1, 13, 6), rand(1, 1, 13, 6)
    br = oracle.attn_bwd_ex(Q, K, V, dO, "causal_bottom_right", 0.5)
    full = oracle.attn_bwd_ex(Q, K, V, dO, "none", 0.5)
    for k in ("O", "LSE", "dQ", "dK", "dV"):
        np.testing.assert_array_equal(br[k], full[k])
    tl = oracle.attn_bwd_ex(Q, K, V, dO, "causal", 0.5)
    np.testing.assert_allclose(tl["O"][0, 0, 0], V[0, 0, 0], rtol=0, atol=1e-15)
    assert np.all(tl["dK"][0, 0, 1:] == 0) and np.all(tl["dV"][0, 0, 1:] == 0)


def test_empty_rows_contribute_nothing():
    """Bottom-right alignment with Lq > Lk leaves the first Lq - Lk rows without
    keys: O = 0, LSE = -inf, dQ = 0, and dK, dV equal those of the problem
    without those rows (same alignment, Lq' = Lk)."""
    Lq, Lk, D = 11, 4, 5
    Q, dO = rand(1, 2, Lq, D), rand(1, 2, Lq, D)
    K, V = rand(1, 2, Lk, D), rand(1, 2, Lk, D)
    g = oracle.attn_bwd_ex(Q, K, V, dO, "causal_bottom_right", 0.45)
    e = Lq - Lk
    assert np.all(g["O"][:, :, :e] == 0) and np.all(g["dQ"][:, :, :e] == 0)
    assert np.all(np.isneginf(g["LSE"][:, :, :e])) and np.all(np.isfinite(g["LSE"][:, :, e:]))
    r = oracle.attn_bwd_ex(Q[:, :, e:], K, V, dO[:, :, e:], "causal_bottom_right", 0.45)
    for k in ("dK", "dV"):
        np.testing.assert_allclose(g[k], r[k], rtol=1e-13, atol=1e-14)
    for k in ("O", "LSE", "dQ"):
        np.testing.assert_allclose(g[k][:, :, e:], r[k], rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("mask", MASKS_EX)
def test_torch_float64_sdpa_cross_attention(mask):
    """Third implementation for Lq != Lk: torch CPU float64 SDPA with an explicit
    boolean mask of each alignment, + autograd (no empty rows here)."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    B, H, Lq, Lk, D, scale = 2, 2, 7, 10, 4, 0.5
    Q, dO = rand(B, H, Lq, D), rand(B, H, Lq, D)
    K, V = rand(B, H, Lk, D), rand(B, H, Lk, D)
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    allow = {"none": np.ones((Lq, Lk), bool), "causal": j <= i,
             "causal_bottom_right": j <= i + (Lk - Lq)}[mask]
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    out = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.tensor(allow), scale=scale)
    out.backward(torch.tensor(dO, dtype=torch.float64))
    g = oracle.attn_bwd_ex(Q, K, V, dO, mask, scale)
    np.testing.assert_allclose(g["O"], out.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dQ"], tq.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(g["dK"], tk.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(g["dV"], tv.grad.numpy(), rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- key padding
def loss_padded(Q, K, V, dO, kv_len, mask, scale):
    O, _ = oracle.attn_fwd_padded(Q, K, V, kv_len, mask, scale)
    return float(np.sum(O * dO))


@pytest.mark.parametrize("mask", MASKS_EX)
def test_padded_finite_differences(mask):
    """Per-batch key padding: dQ, dK, dV equal central differences of
    sum(dO * O) over every input element, padding rows included (their exact
    gradient is 0: perturbing a padding key changes nothing)."""
    B, H, Lq, Lk, D, scale, h = 3, 1, 4, 5, 2, 0.7, 1e-6
    kv_len = [5, 2, 0]
    Q, dO = rand(B, H, Lq, D), rand(B, H, Lq, D)
    K, V = rand(B, H, Lk, D), rand(B, H, Lk, D)
    g = oracle.attn_bwd_padded(Q, K, V, dO, kv_len, mask, scale)
    for name, X in (("dQ", Q), ("dK", K), ("dV", V)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            orig = X[idx]
            X[idx] = orig + h
            lp = loss_padded(Q, K, V, dO, kv_len, mask, scale)
            X[idx] = orig - h
            lm = loss_padded(Q, K, V, dO, kv_len, mask, scale)
            X[idx] = orig
            num[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(num - g[name])) / max(np.max(np.abs(num)), 1e-300)
        assert err < 1e-6, (name, err)
    for b, n in enumerate(kv_len):
        assert np.all(g["dK"][b, :, n:] == 0) and np.all(g["dV"][b, :, n:] == 0)


@pytest.mark.parametrize("mask", MASKS_EX)
def test_torch_float64_sdpa_padded(mask):
    """Third implementation: torch CPU float64 SDPA with the boolean mask
    (key j < kv_len[b]) AND the alignment of the mask computed from kv_len[b],
    + autograd, on a batch whose every row keeps at least one key."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    B, H, Lq, Lk, D, scale = 3, 2, 5, 9, 4, 0.5
    kv_len = [9, 6, 5]
    Q, dO = rand(B, H, Lq, D), rand(B, H, Lq, D)
    K, V = rand(B, H, Lk, D), rand(B, H, Lk, D)
    allow = np.zeros((B, 1, Lq, Lk), bool)
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    for b, n in enumerate(kv_len):
        a = j < n
        if mask == "causal":
            a = a & (j <= i)
        elif mask == "causal_bottom_right":
            a = a & (j <= i + (n - Lq))
        allow[b, 0] = a
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    out = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.tensor(allow), scale=scale)
    out.backward(torch.tensor(dO, dtype=torch.float64))
    g = oracle.attn_bwd_padded(Q, K, V, dO, kv_len, mask, scale)
    np.testing.assert_allclose(g["O"], out.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dQ"], tq.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(g["dK"], tk.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(g["dV"], tv.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_padded_closed_forms():
    """kv_len = Lk is the unpadded problem; kv_len = 1 leaves one key, so every
    row that sees it has O = V_0, dQ = dK = 0 and dV_0 = the sum of those rows'
    dO; kv_len = 0 leaves none: O = 0, LSE = -inf, every gradient 0; padding
    rows' contents do not matter."""
    B, H, Lq, Lk, D, scale = 3, 2, 6, 7, 3, 0.8
    Q, dO = rand(B, H, Lq, D), rand(B, H, Lq, D)
    K, V = rand(B, H, Lk, D), rand(B, H, Lk, D)
    g = oracle.attn_bwd_padded(Q, K, V, dO, [Lk, 1, 0], "none", scale)
    full = oracle.attn_bwd_ex(Q[:1], K[:1], V[:1], dO[:1], "none", scale)
    for k in ("O", "LSE", "dQ", "dK", "dV"):
        np.testing.assert_array_equal(g[k][:1], full[k])
    np.testing.assert_allclose(g["O"][1], np.broadcast_to(V[1, :, :1], (H, Lq, D)), atol=1e-15)
    assert np.all(g["dQ"][1] == 0) and np.all(g["dK"][1] == 0)
    np.testing.assert_allclose(g["dV"][1, :, 0], dO[1].sum(axis=1), rtol=1e-13, atol=1e-14)
    assert np.all(g["dV"][1, :, 1:] == 0)
    assert np.all(g["O"][2] == 0) and np.all(np.isneginf(g["LSE"][2]))
    for k in ("dQ", "dK", "dV"):
        assert np.all(g[k][2] == 0)
    K2, V2 = K.copy(), V.copy()
    K2[1, :, 1:] = 1e6 * rand(H, Lk - 1, D)
    V2[1, :, 1:] = -1e6
    g2 = oracle.attn_bwd_padded(Q, K2, V2, dO, [Lk, 1, 0], "none", scale)
    for k in ("O", "LSE", "dQ", "dK", "dV"):
        np.testing.assert_array_equal(g2[k][1:], g[k][1:])


def test_padded_bottom_right_uses_own_length():
    """Bottom-right alignment under padding: batch element b aligns its last
    query with its own last real key (offset kv_len[b] - Lq); with Lq > kv_len[b]
    the first Lq - kv_len[b] rows have an empty softmax."""
    B, H, Lq, Lk, D, scale = 2, 1, 5, 8, 4, 0.6
    Q, dO = rand(B, H, Lq, D), rand(B, H, Lq, D)
    K, V = rand(B, H, Lk, D), rand(B, H, Lk, D)
    g = oracle.attn_bwd_padded(Q, K, V, dO, [8, 3], "causal_bottom_right", scale)
    # batch 1: 3 keys, 5 queries: rows 0, 1 see nothing; row 4 sees keys 0..2
    assert np.all(np.isneginf(g["LSE"][1, :, :2])) and np.all(g["O"][1, :, :2] == 0)
    r = oracle.attn_fwd_ex(Q[1, :, 4:], K[1, :, :3], V[1, :, :3], "none", scale)
    np.testing.assert_allclose(g["O"][1, :, 4:], r[0], rtol=1e-14, atol=1e-15)
    # batch 0 (unpadded): the ordinary bottom-right problem
    r0 = oracle.attn_bwd_ex(Q[:1], K[:1], V[:1], dO[:1], "causal_bottom_right", scale)
    np.testing.assert_array_equal(g["dK"][:1], r0["dK"])
