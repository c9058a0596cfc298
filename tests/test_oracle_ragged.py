"""Pins for the oracle at sequence lengths that are not a multiple of 64.

Reading (MInference 1.0 overview, section 2.2; the page's block kernels work on
padded blocks): index formats are built over the sequence padded to the next
multiple of 64, the causal cut removes padded keys, padded rows produce no
output; block-sparse pooling averages the real rows of a partial block.
"""
import math

import numpy as np
import pytest
import torch

from oracle import msa_oracle as O

D = 128


def test_padded_last_block_keeps_the_full_block_rule():
    """N = 69: row block 1 has 5 real rows (64..68).  Offset 10 reaches keys
    54..58 from those rows, all in key block 0, but over the padded block
    (rows 64..127) it also crosses key block 1: the tile (1, 1) is active."""
    a = O.vs_active_tiles(np.array([10]), 69)
    assert a[1, 0] and a[1, 1]
    # the same rule as any full block: distances {0, 1}
    assert (a == O.vs_active_tiles(np.array([10]), 128)).all()


@pytest.mark.parametrize("N", [1, 37, 100, 300])
def test_dense_causal_matches_sdpa_at_ragged_length(N):
    rng = np.random.default_rng(N)
    q, k, v = (rng.standard_normal((N, D)) for _ in range(3))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, None], torch.from_numpy(k)[None, None],
        torch.from_numpy(v)[None, None], is_causal=True)[0, 0].numpy()
    np.testing.assert_allclose(O.dense_causal(q, k, v, O.default_scale(D)), ref,
                               rtol=1e-10, atol=1e-12)


def test_pooling_averages_the_real_rows():
    N = 150  # blocks of 64, 64 and 22 rows
    x = np.arange(N, dtype=np.float64)[:, None] * np.ones((1, D))
    pooled = O.mean_pool(x, N)
    np.testing.assert_allclose(pooled[:, 0], [31.5, 95.5, (128 + 149) / 2])


@pytest.mark.parametrize("N", [5, 40, 64, 70])
def test_estimate_short_sequences(N):
    rng = np.random.default_rng(N)
    q, k = rng.standard_normal((N, D)), rng.standard_normal((N, D))
    v, s, A = O.estimate_vs(q, k, 64, O.default_scale(D))
    L = min(64, N)
    assert A.shape == (L, N)
    assert abs(v.sum() - L) < 1e-10 and abs(s.sum() - L) < 1e-10


@pytest.mark.parametrize("N", [70, 199])
def test_mask_nnz_at_ragged_length(N):
    rng = np.random.default_rng(N)
    allow = rng.random(((N + 63) // 64, N)) < 0.5
    mask = lambda m: allow[m]
    ref = sum(int(allow[i // 64, j]) for i in range(N) for j in range(i + 1))
    assert O.mask_nnz(mask, N) == ref


@pytest.mark.parametrize("N", [70, 199])
def test_streaming_and_block_sets_at_ragged_length(N):
    """Closed forms hold at a partial last block: local >= NB gives every
    causal pair; the block-sparse diagonal is always kept."""
    NB = (N + 63) // 64
    sel = [O.streaming_blocks(m, 0, NB) for m in range(NB)]
    assert O.mask_nnz(O.block_mask_from_blocks(sel, N), N) == N * (N + 1) // 2
    rng = np.random.default_rng(N)
    q, k = rng.standard_normal((N, D)), rng.standard_normal((N, D))
    blocks, _ = O.block_sparse_blocks(q, k, 1)
    assert all(list(b) == [m] for m, b in enumerate(blocks))
