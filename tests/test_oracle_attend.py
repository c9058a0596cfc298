"""Pins for the oracle's masked attention (MInference 1.0 overview, section 1
"Problem Formulation": A(M) = Softmax(Q K^T / sqrt(d) - c (1 - M)) V).

Each test ties the oracle to something other than itself: a library routine
(torch SDPA, torch.softmax of the page's formula with a large finite c), a
closed form, or scalar brute force on a tiny input.
"""
import math

import numpy as np
import pytest
import torch

from oracle import msa_oracle as O

D = 128


def rand_qkv(N, seed, d=D):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((N, d))
    k = rng.standard_normal((N, d))
    v = rng.standard_normal((N, d))
    return q, k, v


def test_dense_causal_matches_torch_sdpa():
    q, k, v = rand_qkv(300, 1)  # ragged against the 64-row block
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, None], torch.from_numpy(k)[None, None],
        torch.from_numpy(v)[None, None], is_causal=True)[0, 0].numpy()
    out = O.dense_causal(q, k, v, O.default_scale(D))
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_page_formula_with_large_c_matches_exclusion():
    """The page writes the mask as a penalty c(1-M); with c = 1e4 the penalised
    entries underflow to exactly 0, which is the oracle's exclusion rule."""
    N = 200
    q, k, v = rand_qkv(N, 2)
    rng = np.random.default_rng(3)
    M = rng.random((N, N)) < 0.3
    M &= np.tril(np.ones((N, N), dtype=bool))
    M[np.arange(N), np.arange(N)] = True  # no empty row
    scale = 1 / math.sqrt(D)
    c = 1e4
    logits = torch.from_numpy(q @ k.T * scale - c * (1.0 - M))
    ref = (torch.softmax(logits, dim=-1) @ torch.from_numpy(v)).numpy()
    out, counts = O.attend_rows(q, k, v, range(N), lambda i: M[i], scale)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    assert (counts == M.sum(1)).all()
    # the index-list form of the same mask gives the same numbers
    out_b, counts_b = O.attend_rows(q, k, v, range(N), lambda i: np.nonzero(M[i])[0], scale)
    np.testing.assert_allclose(out_b, out, rtol=0, atol=1e-14)


def test_identity_values_expose_probabilities_brute_force():
    """N <= d and v_j = e_j make out = P; every entry checked by scalar loops."""
    N = 96
    q, k, _ = rand_qkv(N, 4)
    v = np.eye(N, D)
    scale = 1 / math.sqrt(D)
    rng = np.random.default_rng(5)
    M = rng.random((N, N)) < 0.5
    M[np.arange(N), np.arange(N)] = True
    out, _ = O.attend_rows(q, k, v, range(N), lambda i: M[i], scale)
    for i in range(N):
        J = [j for j in range(i + 1) if M[i, j]]
        zs = {j: sum(q[i, c] * k[j, c] for c in range(D)) * scale for j in J}
        zmax = max(zs.values())
        den = sum(math.exp(z - zmax) for z in zs.values())
        for j in range(N):
            expect = math.exp(zs[j] - zmax) / den if j in zs else 0.0
            assert abs(out[i, j] - expect) < 1e-12
        assert abs(out[i, :N].sum() - 1.0) < 1e-12


def test_constant_values_give_constant_output():
    N = 256
    q, k, _ = rand_qkv(N, 6)
    c = np.random.default_rng(7).standard_normal(D)
    v = np.tile(c, (N, 1))
    out = O.dense_causal(q, k, v, 0.3)
    np.testing.assert_allclose(out, np.tile(c, (N, 1)), rtol=0, atol=1e-12)


def test_zero_keys_average_the_admitted_values():
    """K = 0 makes every admitted logit equal, so out_i is the plain mean of
    v_j over the admitted set: this pins mask membership and the causal cut."""
    N = 320
    q, _, v = rand_qkv(N, 8)
    k = np.zeros((N, D))
    mask = O.block_mask_from_blocks([np.array([0]), np.array([0, 1]), np.array([2]),
                                     np.array([0, 3]), np.array([1, 2, 4])], N)
    out, counts = O.attend_blocks(q, k, v, mask, 0.1)
    for i in [0, 5, 63, 64, 100, 127, 128, 191, 192, 250, 255, 256, 300, 319]:
        m = i // 64
        allow = np.nonzero(mask(m))[0]
        J = allow[allow <= i]
        assert counts[i] == J.size
        np.testing.assert_allclose(out[i], v[J].mean(0), rtol=0, atol=1e-12)


def test_single_key_rows_copy_the_value():
    N = 128
    q, k, v = rand_qkv(N, 9)
    out, counts = O.attend_rows(q, k, v, range(N), lambda i: np.array([i // 2]), 0.2)
    assert (counts == 1).all()
    np.testing.assert_array_equal(out, v[np.arange(N) // 2])


def test_empty_rows_output_zero():
    N = 128
    q, k, v = rand_qkv(N, 10)
    # keys admitted only from 100 on: rows < 100 have none after the causal cut
    mask = lambda m: np.arange(N) >= 100
    out, counts = O.attend_blocks(q, k, v, mask, 0.2)
    assert (counts[:100] == 0).all() and (out[:100] == 0).all()
    assert (counts[100:] == np.arange(1, 29)).all()


def test_attend_rows_and_blocks_agree():
    N = 200
    q, k, v = rand_qkv(N, 11)
    rng = np.random.default_rng(12)
    bm = rng.random((4, N)) < 0.4
    out_b, cnt_b = O.attend_blocks(q, k, v, lambda m: bm[m], 0.09)
    out_r, cnt_r = O.attend_rows(q, k, v, range(N), lambda i: bm[i // 64], 0.09)
    np.testing.assert_allclose(out_b, out_r, rtol=1e-12, atol=1e-13)
    assert (cnt_b == cnt_r).all()


def test_half_ulp_bound_helper():
    """The output bound's half-ulp term: bf16 spacing is 2^(e-7) on [2^e, 2^(e+1))."""
    from tests.parity import half_ulp_bf16
    for x, expect in [(1.0, 2 ** -8), (1.99, 2 ** -8), (2.0, 2 ** -7), (4.14, 2 ** -6),
                      (-4.14, 2 ** -6), (0.3, 2 ** -10)]:
        assert half_ulp_bf16(x) == expect
    # rounding 4.14387 to bf16 (step 1/32 there) lands within half a step
    r = torch.tensor(4.14387, dtype=torch.float64).to(torch.bfloat16).double().item()
    assert abs(r - 4.14387) <= half_ulp_bf16(4.14387)
