"""The allocation-free entry point, exact_topk_kv_split_noalloc.

It exists for callers that cannot allocate device memory where they need the
selection (an already-open stream capture, a host framework that owns every
allocation, a loop that cannot afford cudaMalloc's device synchronization):
its counters and workspace come from one static device array inside the
library.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes on its own in a
fresh process, where its first call performs the per-device set-up.
"""

import ctypes

import numpy as np
import pytest
import torch

import exact_top_selection_gb300 as etk
import workloads
from gpu_helpers import CANARY, bits

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p


def _noalloc(X, ke, out, nv, K, stream):
    M, N = X.shape
    return etk.library().exact_topk_kv_split_noalloc(
        P(X.data_ptr()), M, N, P(ke.data_ptr()), P(out.data_ptr()),
        None if nv is None else P(nv.data_ptr()), K, P(stream.cuda_stream))


def _existing(X, ke, nv, K):
    M, N = X.shape
    cb, wb = etk.workspace_size(M, N, K)
    counters = torch.zeros(cb, dtype=torch.uint8, device=X.device)
    workspace = torch.empty(max(wb, 16), dtype=torch.uint8, device=X.device)
    out = torch.full((M, K), CANARY, dtype=torch.int32, device=X.device)
    etk.topk(X, ke, out, nv, K, counters, workspace)
    return out


def _same_value_multisets(X, ke, K, a, b):
    X = X.cpu().numpy()
    ke = ke.cpu().numpy()
    a = a.cpu().numpy()
    b = b.cpu().numpy()
    for r in range(X.shape[0]):
        L = int(min(max(int(ke[r]), 0), X.shape[1]))
        if L <= K:
            assert sorted(a[r][a[r] >= 0].tolist()) == list(range(L))
            assert int((a[r] == -1).sum()) == K - L
            assert np.array_equal(np.sort(a[r]), np.sort(b[r]))
            continue
        assert len(set(a[r].tolist())) == K and (a[r] >= 0).all() and (a[r] < L).all()
        assert np.array_equal(np.sort(bits(X[r][a[r]])), np.sort(bits(X[r][b[r]]))), r


def test_noalloc_matches_existing_entry_point_on_two_calls_in_a_row():
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    cases = [("decode_batch", 16, 65536, 2048), ("long_decode", 4, 524288, 2048)]
    for name, M, N, K in cases:
        X, ke, K = workloads.generate(name, M=M, N=N, K=K, device="cuda")
        nv = torch.tensor([M], dtype=torch.int32, device=dev)
        ref = _existing(X, ke, nv, K)
        out = torch.full((M, K), CANARY, dtype=torch.int32, device=dev)
        assert _noalloc(X, ke, out, nv, K, stream) == 0
        torch.cuda.synchronize()
        _same_value_multisets(X, ke, K, out, ref)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    dev = torch.device("cuda")
    M, N, K = 600, 100000, 64  # needs about M * N * 8 bytes = 480 MB > 64 MiB
    X = torch.zeros(M, N, device=dev)
    ke = torch.full((M,), N, dtype=torch.int32, device=dev)
    out = torch.full((M, K), CANARY, dtype=torch.int32, device=dev)
    rc = _noalloc(X, ke, out, None, K, torch.cuda.current_stream())
    assert rc == -5
    torch.cuda.synchronize()
    assert (out.cpu().numpy() == CANARY).all()
