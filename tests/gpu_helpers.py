"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and compare it with the CPU oracle row by row."""

import numpy as np
import torch

import exact_top_selection_gb300 as etk
import oracle

CANARY = -7


def bits(x):
    return np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)


def run_gpu(X, ke, K, num_valid=None, prev=None, row_pitch=None, trace=True, **plan_kw):
    """Runs one call with an explicit plan; returns (out, trace, plan, counters)."""
    dev = torch.device("cuda")
    Xd = X if isinstance(X, torch.Tensor) and X.is_cuda else torch.as_tensor(X).to(dev)
    M = Xd.shape[0]
    ked = torch.as_tensor(ke, dtype=torch.int32).to(dev)
    runner = etk.ExactTopK(M, Xd.shape[1], K, device=dev, row_pitch=row_pitch, **plan_kw)
    out = torch.full((M, K), CANARY, dtype=torch.int32, device=dev)
    tr = torch.full((M, 8), CANARY, dtype=torch.int32, device=dev) if trace else None
    nv = None if num_valid is None else torch.tensor([num_valid], dtype=torch.int32, device=dev)
    pv = None if prev is None else torch.as_tensor(prev, dtype=torch.int32).to(dev).contiguous()
    runner(Xd, ked, num_valid_rows=nv, out=out, prev_topk=pv, trace=tr)
    torch.cuda.synchronize()
    return (out.cpu().numpy(), None if tr is None else tr.cpu().numpy(), runner.plan,
            runner.counters.cpu().numpy())


def assert_counters_zero(counters):
    assert not counters.any(), f"counters not restored: {np.nonzero(counters)[0][:8]}"


def compare_rows(X, ke, K, out, M_live=None, ref=None, check_rows=None):
    """Bit-exact value-multiset parity against the definition oracle, plus the
    exactness criterion, the pad rule and untouched dead rows."""
    X = np.asarray(X)
    M, N = X.shape
    if M_live is None:
        M_live = M
    if ref is None:
        ref = oracle.topk_rows(X, ke, K, M_live=M_live)
    rows = range(M) if check_rows is None else check_rows
    for r in rows:
        if r >= M_live:
            assert (out[r] == CANARY).all(), f"row {r} >= M_live was written"
            continue
        L = int(min(max(int(ke[r]), 0), N))
        o = out[r]
        if L <= K:
            assert sorted(o[o >= 0].tolist()) == list(range(L)), f"row {r}: pad row indices"
            assert int((o == -1).sum()) == K - L, f"row {r}: pad count"
            continue
        assert (o >= 0).all() and (o < L).all(), f"row {r}: index out of [0, L)"
        assert len(np.unique(o)) == K, f"row {r}: duplicate indices"
        got = np.sort(bits(X[r][o]))
        exp = np.sort(bits(X[r][ref[r]]))
        if not np.array_equal(got, exp):
            diff = np.nonzero(got != exp)[0]
            raise AssertionError(f"row {r} (L={L}): value multiset differs at {diff.size} places")


def compare_trace(tr_gpu, tr_ref, rows=None):
    rows = range(tr_gpu.shape[0]) if rows is None else rows
    for r in rows:
        if not np.array_equal(tr_gpu[r], tr_ref[r]):
            raise AssertionError(f"row {r}: trace {tr_gpu[r].tolist()} != oracle {tr_ref[r].tolist()}"
                                 f" (fields {oracle.TRACE_FIELDS})")


def oracle_trace_for_plan(X, ke, K, plan, prev=None, M_live=None):
    sampled = plan.family != etk.FAMILY_ROW_LOCAL_EXACT
    return oracle.method_trace(X, ke, K, plan.stride, plan.dual, rho0=(plan.rho0_num, plan.rho0_den),
                               rho1=(plan.rho1_num, plan.rho1_den), sampled=sampled, guess=prev,
                               M_live=M_live)
