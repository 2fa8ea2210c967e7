"""Full-size parity: the five workloads at their full sizes, in the launch
configuration bench.py times (default plan), every row checked against the
CPU oracle (bit-exact value multisets, eq. 30, pad rule) and every row's route
trace checked against the oracle's written-out method."""

import numpy as np
import pytest
import torch

import exact_top_selection_gb300 as etk
import workloads
from gpu_helpers import (CANARY, assert_counters_zero, compare_rows, compare_trace,
                         oracle_trace_for_plan)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", workloads.ORDER)
def test_full_size_workload(name):
    dev = torch.device("cuda")
    X, ke, K = workloads.generate(name, device="cuda")
    M, N = X.shape
    runner = etk.ExactTopK(M, N, K, device=dev)
    out = torch.full((M, K), CANARY, dtype=torch.int32, device=dev)
    tr = torch.full((M, 8), CANARY, dtype=torch.int32, device=dev)
    nv = torch.tensor([M], dtype=torch.int32, device=dev)
    runner(X, ke, num_valid_rows=nv, out=out)          # as timed: no trace
    out2 = torch.full((M, K), CANARY, dtype=torch.int32, device=dev)
    runner(X, ke, num_valid_rows=nv, out=out2, trace=tr)
    torch.cuda.synchronize()
    Xh, keh = X.cpu().numpy(), ke.cpu().numpy()
    del X
    compare_rows(Xh, keh, K, out.cpu().numpy())
    compare_rows(Xh, keh, K, out2.cpu().numpy())
    assert_counters_zero(runner.counters.cpu().numpy())
    _, tr_ref = oracle_trace_for_plan(Xh, keh, K, runner.plan)
    compare_trace(tr.cpu().numpy(), tr_ref)
