"""The seeded input recipes that both the oracle and the kernels consume.

These check the structure each recipe promises (shapes, length rules, NaN
garbage past each length, determinism per seed, the temporal correlation of
the decode series, the M = total / N shape of the serving trace) at reduced
sizes on CPU.  None of the method's arithmetic is involved.
"""

import numpy as np
import pytest
import torch

import workloads


def _valid_prefix_clean(X, ke):
    X = X.numpy()
    ke = ke.numpy()
    for r in range(X.shape[0]):
        L = int(np.clip(ke[r], 0, X.shape[1]))
        assert not np.isnan(X[r, :L]).any()  # indexer and iid prefixes hold no NaN
        if L < X.shape[1]:
            assert np.isnan(X[r, L:]).all()


@pytest.mark.parametrize("name,M,N,K", [("short_iid", 4, 8192, 256),
                                        ("decode_batch", 8, 8192, 512),
                                        ("prefill_causal", 16, 8192, 512),
                                        ("long_decode", 4, 16384, 512)])
def test_recipe_shapes_lengths_and_padding(name, M, N, K):
    X, ke, KK = workloads.generate(name, M=M, N=N, K=K)
    assert X.shape == (M, N) and X.dtype == torch.float32
    assert ke.shape == (M,) and ke.dtype == torch.int32 and KK == K
    k = ke.numpy()
    if name == "short_iid":
        assert (k == N).all()
    elif name == "prefill_causal":
        assert np.array_equal(k, N - M + np.arange(M) + 1)
    elif name == "decode_batch":
        assert (k >= K).all() and (k <= N).all()
    else:  # long_decode: the same fraction of the width as 500000 / 524288
        assert (k >= -(-N * 500000 // 524288)).all() and (k <= N).all()
    _valid_prefix_clean(X, ke)


def test_adversarial_recipe_forced_lengths_and_levels():
    M, N, K = 16, 4096, 64
    X, ke, _ = workloads.generate("adversarial", M=M, N=N, K=K)
    k = ke.numpy()
    assert list(k[:4]) == [1, 7, K - 1, K]  # lengths around K are always present
    assert (k >= 1).all() and (k <= N).all()
    Xn = X.numpy()
    for r in range(M):
        L = int(k[r])
        if L < N:
            assert np.isnan(Xn[r, L:]).all()


def test_recipes_are_deterministic_per_seed():
    a = workloads.generate("decode_batch", M=4, N=4096, K=256)
    b = workloads.generate("decode_batch", M=4, N=4096, K=256)
    c = workloads.generate("decode_batch", M=4, N=4096, K=256, seed=12345)
    assert torch.equal(a[1], b[1]) and np.array_equal(a[0].numpy(), b[0].numpy(), equal_nan=True)
    assert not np.array_equal(a[0].numpy(), c[0].numpy(), equal_nan=True)


def test_decode_series_is_correlated_and_lengths_grow():
    M, N, K, steps = 4, 4096, 128, 3
    Xs, kes = workloads.decode_batch_series(M, N, K, steps, seed=5)
    assert len(Xs) == steps and len(kes) == steps
    for t in range(1, steps):
        assert torch.equal(kes[t], (kes[t - 1] + 1).clamp(max=N))
        L = int(kes[t - 1].min())
        a = Xs[t - 1][:, :L].numpy().ravel()
        b = Xs[t][:, :L].numpy().ravel()
        assert np.corrcoef(a, b)[0, 1] > 0.9  # a small drift per step
    _valid_prefix_clean(Xs[-1], kes[-1])


def test_trace_sequence_shapes():
    widths = (512, 2048, 8192)
    calls = workloads.trace_sequence(1 << 14, 64, 3, widths=widths)
    assert len(calls) == len(widths)
    for (X, ke), N in zip(calls, widths):
        assert X.shape == (max(1, (1 << 14) // N), N)
        k = ke.numpy()
        assert (k >= N // 2).all() and (k <= N).all()
        _valid_prefix_clean(X, ke)
