"""The allocation-free entry point, exact_topk_kv_split_noalloc.

It exists for callers that cannot allocate device memory where they need the
selection: plugins whose host framework owns every device allocation, and
loops that cannot afford cudaMalloc's implicit device synchronization.  Its
counters and workspace come from one static device array inside the library.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process,
where its first call performs the per-device set-up.
"""

import ctypes

import numpy as np
import pytest
import torch

import exact_top_selection_gb300 as etk
import workloads
from gpu_helpers import CANARY, bits, compare_rows

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p


def _noalloc(X, ke, out, nv, K, stream):
    M, N = X.shape
    return etk.library().exact_topk_kv_split_noalloc(
        P(X.data_ptr()), M, N, P(ke.data_ptr()), P(out.data_ptr()),
        None if nv is None else P(nv.data_ptr()), K, P(stream.cuda_stream))


def _existing(X, ke, nv, K):
    """The same selection through exact_topk with caller-owned buffers."""
    M, N = X.shape
    cb, wb = etk.workspace_size(M, N, K)
    counters = torch.zeros(cb, dtype=torch.uint8, device=X.device)
    workspace = torch.empty(max(wb, 16), dtype=torch.uint8, device=X.device)
    out = torch.full((M, K), CANARY, dtype=torch.int32, device=X.device)
    etk.topk(X, ke, out, nv, K, counters, workspace)
    return out


def _same_as_existing(X, ke, K, a, b, M_live):
    """Row by row, the two entry points select the same value multiset (the
    indices may differ only inside a tie at rank K) and the same pad rows."""
    for r in range(M_live):
        L = int(min(max(int(ke[r]), 0), X.shape[1]))
        if L <= K:
            assert np.array_equal(np.sort(a[r]), np.sort(b[r])), r
            continue
        assert np.array_equal(np.sort(bits(X[r][a[r]])), np.sort(bits(X[r][b[r]]))), r


def _case(name, M, N, K, M_live, seed):
    X, ke, K = workloads.generate(name, M=M, N=N, K=K, device="cpu", seed=seed)
    ke = ke.clone()
    if name != "long_decode":
        # ragged rows, including a few with ke <= K (padded with -1) and one
        # empty and one out-of-range length
        ke[1] = K // 3
        ke[2] = 0
        ke[3] = N + 17  # clamped to N: the whole row is valid, so its NaN tail
        X[3] = torch.nan_to_num(X[3], nan=0.25)  # becomes a run of equal scores
    return X, ke, K, M_live


@pytest.mark.parametrize("name,M,N,K,M_live", [
    ("decode_batch", 16, 65536, 2048, 13),
    ("adversarial", 32, 40000, 512, 32),
    ("long_decode", 4, 524288, 2048, 4),
])
def test_noalloc_matches_oracle_and_existing_entry_point_on_two_calls_in_a_row(
        name, M, N, K, M_live):
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    X, ke, K, M_live = _case(name, M, N, K, M_live, seed=20261000 + M)
    Xd, ked = X.to(dev), ke.to(dev)
    nv = torch.tensor([M_live], dtype=torch.int32, device=dev)
    Xn, ken = X.numpy(), ke.numpy()
    ref = _existing(Xd, ked, nv, K).cpu().numpy()
    for call in range(2):  # the second call finds the first call's array contents
        out = torch.full((M, K), CANARY, dtype=torch.int32, device=dev)
        assert _noalloc(Xd, ked, out, nv, K, stream) == 0
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        # bit-exact value multisets against the CPU oracle, the pad rule, and
        # untouched rows at and beyond the live count
        compare_rows(Xn, ken, K, got, M_live=M_live)
        _same_as_existing(Xn, ken, K, got, ref, M_live)


def test_noalloc_rejects_shapes_beyond_its_scratch_and_launches_nothing():
    dev = torch.device("cuda")
    M, N, K = 600, 100000, 64  # needs about M * N * 8 bytes = 480 MB > 64 MiB
    X = torch.zeros(M, N, device=dev)
    ke = torch.full((M,), N, dtype=torch.int32, device=dev)
    out = torch.full((M, K), CANARY, dtype=torch.int32, device=dev)
    rc = _noalloc(X, ke, out, None, K, torch.cuda.current_stream())
    assert rc == -5
    torch.cuda.synchronize()
    assert (out.cpu().numpy() == CANARY).all()


def test_noalloc_rejects_a_misaligned_output_before_enqueuing_anything():
    dev = torch.device("cuda")
    M, N, K = 4, 65536, 256
    X = torch.randn(M, N, device=dev)
    ke = torch.full((M,), N, dtype=torch.int32, device=dev)
    buf = torch.full((M * K + 1,), CANARY, dtype=torch.int32, device=dev)
    lib = etk.library()
    misaligned = P(buf.data_ptr() + 2)
    rc = lib.exact_topk_kv_split_noalloc(P(X.data_ptr()), M, N, P(ke.data_ptr()), misaligned,
                                         None, K, P(torch.cuda.current_stream().cuda_stream))
    assert rc == -6
    torch.cuda.synchronize()
    assert (buf.cpu().numpy() == CANARY).all()
