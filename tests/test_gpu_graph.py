"""CUDA-graph capture and replay (section 2.1 "Deployment requirements": the
operator must be capturable; section 5.5: counters are restored on device so
replays need no host work).  One capture per kernel family, replayed over
different inputs written into the captured buffers and a different live-row
count; every replay is checked against the oracle and must leave the counter
buffer at zero."""

import numpy as np
import pytest
import torch

import exact_top_selection_gb300 as etk
import workloads
from gpu_helpers import CANARY, assert_counters_zero, compare_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("family,N,K", [(etk.FAMILY_PERSISTENT_SAMPLED, 70000, 2048),
                                        (etk.FAMILY_KV_SPLIT, 140000, 2048),
                                        (etk.FAMILY_CLUSTER_SPLIT, 70000, 2048),
                                        (etk.FAMILY_ROW_LOCAL_EXACT, 8192, 256),
                                        (etk.FAMILY_ROW_LOCAL_EXACT, 20000, 512)])
def test_capture_and_replay(family, N, K):
    dev = torch.device("cuda")
    M = 24
    runner = etk.ExactTopK(M, N, K, device=dev, family=family)
    X = torch.empty(M, N, device=dev)
    ke = torch.empty(M, dtype=torch.int32, device=dev)
    nv = torch.tensor([M], dtype=torch.int32, device=dev)
    out = torch.full((M, K), CANARY, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream()
    X.copy_(workloads.iid_rows(M, N, 1, device="cpu"))
    ke.fill_(N)
    with torch.cuda.stream(stream):
        runner(X, ke, num_valid_rows=nv, out=out, stream=stream)   # pre-capture call
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        runner(X, ke, num_valid_rows=nv, out=out, stream=stream)
    rng = np.random.default_rng(5)
    for rep in range(4):
        Xh = workloads.iid_rows(M, N, 100 + rep, device="cpu",
                                dist="int" if rep == 2 else "normal").numpy()
        keh = rng.integers(0, N + 1, M).astype(np.int32)
        m_live = M if rep != 3 else 9
        X.copy_(torch.from_numpy(Xh))
        ke.copy_(torch.from_numpy(keh))
        nv.fill_(m_live)
        out.fill_(CANARY)
        g.replay()
        torch.cuda.synchronize()
        compare_rows(Xh, keh, K, out.cpu().numpy(), M_live=m_live)
        assert_counters_zero(runner.counters.cpu().numpy())


def test_back_to_back_replays_share_counters():
    # Many replays of one graph without any host work in between: the queue
    # and arrival counters must be restored by every launch.
    dev = torch.device("cuda")
    M, N, K = 200, 66000, 2048
    X, ke, K = workloads.generate("prefill_causal", M=M, N=N, K=K, device="cuda")
    runner = etk.ExactTopK(M, N, K, device=dev)
    out = torch.empty(M, K, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        runner(X, ke, out=out, stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(10):
            runner(X, ke, out=out, stream=stream)
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    compare_rows(X.cpu().numpy(), ke.cpu().numpy(), K, out.cpu().numpy())
    assert_counters_zero(runner.counters.cpu().numpy())
