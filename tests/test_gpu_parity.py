"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

The bar: bit-exact multisets of selected FP32 values per row (ties at rank K
may pick different indices), exactness criterion eq. 30 of section 6.1, the
-1 pad rule of section 2.1, untouched rows beyond the live count, counters
restored to zero, and the per-row route trace (Table 2 of section 4.6)
identical to the oracle's written-out method.
"""

import numpy as np
import pytest
import torch

import exact_top_selection_gb300 as etk
import oracle
import workloads
from gpu_helpers import (CANARY, assert_counters_zero, compare_rows, compare_trace,
                         oracle_trace_for_plan, run_gpu)

pytestmark = pytest.mark.gpu

FAMILIES = [etk.FAMILY_PERSISTENT_SAMPLED, etk.FAMILY_KV_SPLIT, etk.FAMILY_ROW_LOCAL_EXACT,
            etk.FAMILY_CLUSTER_SPLIT]
SAMPLED_FAMILIES = [etk.FAMILY_PERSISTENT_SAMPLED, etk.FAMILY_KV_SPLIT, etk.FAMILY_CLUSTER_SPLIT]


def _rows(M, N, seed, dist):
    X = workloads.iid_rows(M, N, seed, dist=dist).numpy()
    return X


def _ke(M, N, K, seed):
    rng = np.random.default_rng(seed)
    ke = rng.integers(0, N + 1, M).astype(np.int32)
    special = [0, 1, K - 1, K, K + 1, N, N + 5, -3]
    for i, v in enumerate(special[:M]):
        ke[i] = v
    return ke


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("N,K", [(1, 1), (7, 4), (64, 1), (4095, 256), (8191, 7), (8192, 256),
                                 (12345, 2048), (40000, 2048)])
def test_small_shapes_every_family(family, N, K):
    M = 24
    X = _rows(M, N, 1000 + N + K, "normal")
    ke = _ke(M, N, K, N * 7 + K)
    out, tr, plan, ctr = run_gpu(X, ke, K, family=family, stride=16 if N < 20000 else 0)
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
    compare_trace(tr, tr_ref)


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("dist", ["int", "uniform"])
def test_tie_heavy_rows(family, dist):
    M, N, K = 20, 30000, 2048
    X = _rows(M, N, 77, dist)
    ke = _ke(M, N, K, 78)
    out, tr, plan, ctr = run_gpu(X, ke, K, family=family)
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
    compare_trace(tr, tr_ref)


@pytest.mark.parametrize("name", workloads.ORDER)
@pytest.mark.parametrize("family", [0] + FAMILIES)
def test_scaled_workloads(name, family):
    # The five workload recipes at sizes the oracle finishes in seconds, still
    # spanning several tiles and a ragged tail.
    w = workloads.WORKLOADS[name]
    M = min(w.M, 48)
    N = min(w.N, 40000 if w.N > 8192 else w.N)
    K = min(w.K, 1024)
    Xt, ket, K = workloads.generate(name, M=M, N=N, K=K, device="cpu")
    X, ke = Xt.numpy(), ket.numpy()
    out, tr, plan, ctr = run_gpu(X, ke, K, family=family)
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
    compare_trace(tr, tr_ref)


@pytest.mark.parametrize("family", SAMPLED_FAMILIES)
@pytest.mark.parametrize("dual", [0, 1])
def test_forced_routes(family, dual):
    # Table 2's routes, forced by planting large values on or off the sampled
    # residue class (the view phase is a pure function of the row, eq. 13).
    K, s, N = 64, 16, 8192
    q0 = -(-3 * K // (2 * s))
    q1 = -(-7 * K // (4 * s))
    rng = np.random.default_rng(8)
    base = rng.standard_normal(N).astype(np.float32)

    def planted(r, off_hi, off_mid):
        row = base.copy()
        a = oracle.view_phase(r, s)
        on = np.arange(a, N, s)
        off = np.array([i for i in range(N) if i % s != a])
        row[on[:q0]] = 100.0
        row[on[q0:q1]] = 90.0
        row[off[:off_hi]] = 100.0
        row[off[off_hi:off_hi + off_mid]] = 90.0
        return row

    X = np.stack([base, planted(1, 30, 50), planted(2, 30, 0), base])
    ke = np.array([N, N, N, 100], np.int32)
    out, tr, plan, ctr = run_gpu(X, ke, K, family=family, stride=s, dual=dual, splits=3)
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
    compare_trace(tr, tr_ref)
    if dual:
        assert tr[:, 0].tolist() == [1, 2, 3, 5]
    else:
        assert tr[:3, 0].tolist() == [1, 4, 4]


@pytest.mark.parametrize("family", SAMPLED_FAMILIES)
@pytest.mark.parametrize("dual", [0, 1])
def test_exact_recovery_after_a_short_phase2(family, dual):
    # Phase 2 falls short of K (the view over-counts the largest scores) while
    # the view shows the next coarse bins filled.  Row 0: those bins complete
    # the Top-K; row 2: they complete it with one key to spare; row 1: they do
    # not, and the whole row's coarse histogram decides.  Values, tau*, |E0|
    # and |Q0| must match the oracle's full-row recovery on every row.
    K, s, N = 64, 16, 8192
    q0 = -(-3 * K // (2 * s))
    q1 = -(-7 * K // (4 * s))
    rng = np.random.default_rng(11)
    base = rng.standard_normal(N).astype(np.float32)

    def planted(r, near_on, near_off):
        row = base.copy()
        a = oracle.view_phase(r, s)
        on = np.arange(a, N, s)
        off = np.array([i for i in range(N) if i % s != a])
        row[on[:q0]] = 100.0
        row[on[q0:q1]] = 90.0
        row[off[:30]] = 100.0
        row[on[q1:q1 + near_on]] = 80.0
        row[off[30:30 + near_off]] = 80.0
        return row

    X = np.stack([planted(0, 8, 60), planted(1, 8, 0), planted(2, 8, 20), base])
    ke = np.full(4, N, np.int32)
    out, tr, plan, ctr = run_gpu(X, ke, K, family=family, stride=s, dual=dual, splits=3)
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
    compare_trace(tr, tr_ref)
    exact = 3 if dual else 4
    assert tr[:, 0].tolist() == [exact, exact, exact, 1]
    # E0: the 100s and the 90s; Q0: the 80s
    assert tr[[0, 2], 6].tolist() == [37, 37]
    assert tr[[0, 2], 7].tolist() == [68, 28]


@pytest.mark.parametrize("family", SAMPLED_FAMILIES)
def test_guess_source(family):
    M, N, K = 12, 20000, 512
    X = _rows(M, N, 5, "normal")
    ke = np.full(M, N, np.int32)
    ke[7] = 300
    ref = oracle.topk_rows(X, ke, K)
    guess = ref.copy()
    rng = np.random.default_rng(3)
    guess[1] = rng.permutation(N)[:K]        # poor but valid
    guess[2, 5] = -1                          # invalid entry -> sampled route
    guess[3] = np.argmax(X[3])                # K copies of one index -> exact recovery
    guess[4, :] = np.arange(K)                # arbitrary valid
    guess[5, 0] = N + 10                      # out of range -> sampled route
    guess[7] = 0                              # pad row ignores the guess
    out, tr, plan, ctr = run_gpu(X, ke, K, prev=guess, family=family)
    compare_rows(X, ke, K, out, ref=ref)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan, prev=guess)
    compare_trace(tr, tr_ref)
    assert tr[0, 0] == 6 and tr[3, 0] == 7


@pytest.mark.parametrize("family", SAMPLED_FAMILIES)
def test_guess_decode_series(family):
    # A decode batch over correlated steps: each step's output is the next
    # step's guess source; every step is exact and routes like the oracle.
    M, N, K, steps = 6, 40000, 512, 4
    Xs, kes = workloads.decode_batch_series(M, N, K, steps, seed=91, device="cpu")
    prev = None
    for t in range(steps):
        X, ke = Xs[t].numpy(), kes[t].numpy()
        out, tr, plan, ctr = run_gpu(X, ke, K, prev=prev, family=family)
        compare_rows(X, ke, K, out)
        assert_counters_zero(ctr)
        _, tr_ref = oracle_trace_for_plan(X, ke, K, plan, prev=prev)
        compare_trace(tr, tr_ref)
        if t:
            # rows long enough now and one step ago take a guess route
            rows = (np.clip(ke, 0, N) > K) & (np.clip(kes[t - 1].numpy(), 0, N) > K)
            assert np.isin(tr[rows, 0], [6, 7]).all(), tr[:, 0]
        prev = out


@pytest.mark.parametrize("family", FAMILIES)
def test_live_rows_and_canary(family):
    M, N, K = 16, 9000, 100
    X = _rows(M, N, 11, "normal")
    ke = np.full(M, N, np.int32)
    for m_live in (0, 1, 9, 16, 40):
        out, tr, plan, ctr = run_gpu(X, ke, K, num_valid=m_live, family=family)
        eff = min(max(m_live, 0), M)
        compare_rows(X, ke, K, out, M_live=eff)
        assert (tr[eff:] == CANARY).all()
        assert_counters_zero(ctr)


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("pitch_extra,offset", [(1, 0), (3, 1), (0, 2)])
def test_unaligned_rows(family, pitch_extra, offset):
    # Rows at a pitch that is not a multiple of 4 floats, and a base pointer
    # that is only 4-byte aligned: scalar head/tail plus 128-bit body.
    M, N, K = 10, 20001, 300
    pitch = N + pitch_extra
    rng = np.random.default_rng(pitch_extra * 10 + offset)
    flat = rng.standard_normal(M * pitch + offset).astype(np.float32)
    dev = torch.device("cuda")
    flat_d = torch.as_tensor(flat).to(dev)
    Xd = flat_d[offset:offset + M * pitch].view(M, pitch)[:, :N]
    X = Xd.cpu().numpy()
    ke = _ke(M, N, K, 5)
    out, tr, plan, ctr = run_gpu(Xd, ke, K, row_pitch=pitch, family=family)
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 64])
def test_kv_split_counts(splits):
    M, N, K = 6, 70000, 2048
    Xt, ket, K = workloads.generate("long_decode", M=M, N=N, K=K)
    X, ke = Xt.numpy(), ket.numpy()
    out, tr, plan, ctr = run_gpu(X, ke, K, family=etk.FAMILY_KV_SPLIT, splits=splits)
    assert plan.splits == splits
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
    compare_trace(tr, tr_ref)


@pytest.mark.parametrize("splits", [5, 6, 8])
def test_cluster_split_counts(splits):
    # Cluster sizes from the fewest segments that hold a row up to the
    # portable limit; short rows leave trailing CTAs with empty segments.
    M, N, K = 10, 70000, 2048
    Xt, ket, K = workloads.generate("decode_batch", M=M, N=N, K=K)
    X, ke = Xt.numpy(), ket.numpy()
    # lengths raised past the generated ones would expose the NaN padding
    X = np.where(np.isnan(X), np.float32(0.0), X)
    ke[:4] = [2049, 3000, 16400, N]
    out, tr, plan, ctr = run_gpu(X, ke, K, family=etk.FAMILY_CLUSTER_SPLIT, splits=splits)
    assert plan.splits == splits
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
    compare_trace(tr, tr_ref)


def test_cluster_split_widest_rows():
    # Eight resident segments of 16384 scores each: the widest row a cluster
    # holds, with ragged lengths down to a single segment.
    M, N, K = 12, 131072, 2048
    Xt, ket, K = workloads.generate("decode_batch", M=M, N=N, K=K)
    X, ke = Xt.numpy(), ket.numpy()
    X = np.where(np.isnan(X), np.float32(0.0), X)
    ke[:6] = [N, N - 1, 16384, 16385, 114689, 40000]
    out, tr, plan, ctr = run_gpu(X, ke, K, family=etk.FAMILY_CLUSTER_SPLIT)
    assert plan.splits == 8
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
    compare_trace(tr, tr_ref)


@pytest.mark.parametrize("family", FAMILIES)
def test_frontier_spill_constant_and_tie_rows(family):
    # Constant rows and huge tie bands push |Q0| to L, beyond on-chip capacity,
    # through the global frontier slices.
    M, N, K = 8, 60000, 2048
    X = np.zeros((M, N), np.float32)
    X[0] = 0.5
    X[1] = np.where(np.arange(N) % 3 == 0, 2.0, 1.0)
    X[2, :] = -np.inf
    X[3] = np.float32(1e-40)
    X[4] = np.where(np.arange(N) % 2 == 0, -0.0, 0.0)
    X[5] = (np.arange(N) % 7).astype(np.float32)
    X[6, :5000] = 3.0
    X[7] = np.random.default_rng(1).integers(0, 2, N).astype(np.float32)
    ke = np.array([N, N, N - 1, 50000, N, 33333, N, 45000], np.int32)
    out, tr, plan, ctr = run_gpu(X, ke, K, family=family)
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
    compare_trace(tr, tr_ref)


def test_worker_count_does_not_change_values():
    M, N, K = 40, 66000, 2048
    Xt, ket, K = workloads.generate("prefill_causal", M=M, N=N, K=K)
    X, ke = Xt.numpy(), ket.numpy()
    ref = oracle.topk_rows(X, ke, K)
    traces = []
    for w in (1, 7, 0):
        out, tr, plan, ctr = run_gpu(X, ke, K, family=etk.FAMILY_PERSISTENT_SAMPLED, workers=w)
        compare_rows(X, ke, K, out, ref=ref)
        assert_counters_zero(ctr)
        traces.append(tr)
    assert all(np.array_equal(traces[0], t) for t in traces[1:])


def test_persistent_long_views_and_mixed_rows():
    # Views longer than the TMA boxes cover (N / s = 3125 lines: the first
    # 1024 entries from the boxes, the rest loaded directly), on few workers so
    # that every CTA takes many rows through both tails (refinement beside the
    # next row's Phase 1, and the whole-CTA tail of pad rows and spilled
    # frontiers), with NaN garbage past ke that the boxes read but must not use.
    M, N, K = 36, 100000, 2048
    rng = np.random.default_rng(2026)
    X = rng.standard_normal((M, N)).astype(np.float32)
    ke = rng.integers(K + 1, N + 1, M).astype(np.int32)
    ke[3], ke[11], ke[20] = 0, K, 5
    X[7] = 1.25                                  # constant: |Q0| = L, spilled
    X[15] = (np.arange(N) % 3).astype(np.float32)  # three-level ties
    ke[7], ke[15], ke[30] = N, N, N
    for r in range(M):
        X[r, ke[r]:] = np.nan
    for workers in (3, 0):
        out, tr, plan, ctr = run_gpu(X, ke, K, family=etk.FAMILY_PERSISTENT_SAMPLED, stride=32,
                                     workers=workers)
        compare_rows(X, ke, K, out)
        assert_counters_zero(ctr)
        _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
        compare_trace(tr, tr_ref)


def test_trace_sequence_default_planner():
    # A serving-style sequence (N growing, M = 2^22 / N, ragged lengths, NaN
    # tails, K = min(2048, N / 4)) through the default planner: the calls land
    # on all four kernel families and every row matches the oracle.
    calls = workloads.trace_sequence(1 << 22, 2048, 314, device="cpu",
                                     widths=(512, 16384, 65536, 262144, 1048576))
    families = set()
    for X, ke in calls:
        K = min(2048, X.shape[1] // 4)
        out, tr, plan, ctr = run_gpu(X.numpy(), ke.numpy(), K)
        families.add(plan.family)
        compare_rows(X.numpy(), ke.numpy(), K, out)
        assert_counters_zero(ctr)
    assert families == {etk.FAMILY_ROW_LOCAL_EXACT, etk.FAMILY_PERSISTENT_SAMPLED,
                        etk.FAMILY_CLUSTER_SPLIT, etk.FAMILY_KV_SPLIT}


def test_default_entry_point_matches_plan_entry_point():
    # exact_topk (default plan, PR-style API) vs the oracle, through the
    # workspace_size / topk pair exactly as the pages' API describes.
    M, N, K = 64, 65536, 2048
    Xt, ket, K = workloads.generate("decode_batch", M=M, N=N, K=K)
    dev = torch.device("cuda")
    Xd, ked = Xt.to(dev), ket.to(dev)
    cb, wb = etk.workspace_size(M, N, K)
    counters = torch.zeros(cb, dtype=torch.uint8, device=dev)
    workspace = torch.empty(wb, dtype=torch.uint8, device=dev)
    out = torch.full((M, K), CANARY, dtype=torch.int32, device=dev)
    nv = torch.tensor([M], dtype=torch.int32, device=dev)
    for _ in range(3):
        etk.topk(Xd, ked, out, nv, K, counters, workspace)
    torch.cuda.synchronize()
    compare_rows(Xt.numpy(), ket.numpy(), K, out.cpu().numpy())
    assert_counters_zero(counters.cpu().numpy())


def test_host_errors_launch_nothing():
    dev = torch.device("cuda")
    M, N, K = 4, 1000, 10
    X = torch.randn(M, N, device=dev)
    ke = torch.full((M,), N, dtype=torch.int32, device=dev)
    out = torch.full((M, K), CANARY, dtype=torch.int32, device=dev)
    cb, wb = etk.workspace_size(M, N, K)
    counters = torch.zeros(cb, dtype=torch.uint8, device=dev)
    ws = torch.empty(max(wb, 16), dtype=torch.uint8, device=dev)
    lib = etk.library()
    import ctypes
    P = ctypes.c_void_p
    stream = P(torch.cuda.current_stream().cuda_stream)
    assert lib.exact_topk(None, M, N, P(ke.data_ptr()), P(out.data_ptr()), None, K,
                          P(counters.data_ptr()), cb, P(ws.data_ptr()), wb, None, stream) == -1
    assert lib.exact_topk(P(X.data_ptr()), M, N, P(ke.data_ptr()), P(out.data_ptr()), None, 0,
                          P(counters.data_ptr()), cb, P(ws.data_ptr()), wb, None, stream) == -3
    assert lib.exact_topk(P(X.data_ptr()), M, N, P(ke.data_ptr()), P(out.data_ptr()), None, K,
                          P(counters.data_ptr()), cb - 16 if cb >= 16 else 0, P(ws.data_ptr()),
                          wb, None, stream) == -4
    assert lib.exact_topk(P(X.data_ptr() + 2), M, N, P(ke.data_ptr()), P(out.data_ptr()), None,
                          K, P(counters.data_ptr()), cb, P(ws.data_ptr()), wb, None,
                          stream) == -6
    torch.cuda.synchronize()
    assert (out.cpu().numpy() == CANARY).all()


@pytest.mark.parametrize("splits", [10, 13, 16])
def test_cluster_split_wide_counts(splits):
    # Clusters above the portable size of 8 CTAs; segments longer than the
    # 16384 scores a CTA holds read the rest from global memory.
    M, N, K = 6, 300000, 2048
    Xt, ket, K = workloads.generate("long_decode", M=M, N=N, K=K)
    X, ke = Xt.numpy(), ket.numpy()
    X = np.where(np.isnan(X), np.float32(0.0), X)
    ke[:4] = [N, 16385, 270001, 2049]
    out, tr, plan, ctr = run_gpu(X, ke, K, family=etk.FAMILY_CLUSTER_SPLIT, splits=splits)
    assert plan.splits == splits
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
    compare_trace(tr, tr_ref)


def test_cluster_split_rows_of_524288():
    # The widest rows a cluster takes (16 CTAs x 32768 scores), with ragged
    # lengths down to one held segment.
    M, N, K = 6, 524288, 2048
    Xt, ket, K = workloads.generate("long_decode", M=M, N=N, K=K, seed=77)
    X, ke = Xt.numpy(), ket.numpy()
    X = np.where(np.isnan(X), np.float32(0.0), X)
    ke[:5] = [N, N - 3, 16 * 16384 + 5, 16384, 300017]
    out, tr, plan, ctr = run_gpu(X, ke, K, family=etk.FAMILY_CLUSTER_SPLIT)
    assert plan.splits == 16
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
    compare_trace(tr, tr_ref)


def test_cluster_split_wide_unaligned_rows():
    # Row starts that are only 4-byte aligned: no bulk copy, scalar loads for
    # the held part and for the part read from global memory.
    M, N, K = 4, 300001, 1024
    pitch = N + 1
    rng = np.random.default_rng(99)
    flat = rng.standard_normal(M * pitch + 1).astype(np.float32)
    dev = torch.device("cuda")
    flat_d = torch.as_tensor(flat).to(dev)
    Xd = flat_d[1:1 + M * pitch].view(M, pitch)[:, :N]
    X = Xd.cpu().numpy()
    ke = np.array([N, 200003, 17, 290000], np.int32)
    out, tr, plan, ctr = run_gpu(Xd, ke, K, row_pitch=pitch, family=etk.FAMILY_CLUSTER_SPLIT)
    assert plan.splits == 16
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
    compare_trace(tr, tr_ref)


def test_cluster_split_wide_tie_and_constant_rows():
    # Frontiers far beyond the merged list on wide rows: the cluster-summed
    # digit rounds and the commit read every segment's global part.
    M, N, K = 6, 400000, 2048
    X = np.zeros((M, N), np.float32)
    X[0] = 0.5
    X[1] = np.where(np.arange(N) % 3 == 0, 2.0, 1.0)
    X[2] = np.random.default_rng(5).integers(0, 4, N).astype(np.float32)
    X[3, :] = -np.inf
    X[4] = np.random.default_rng(6).standard_normal(N).astype(np.float32)
    X[4, 390000:] = 7.0                       # a tie band of 10000 maxima in the last segment
    X[5] = np.where(np.arange(N) % 2 == 0, -0.0, 0.0)
    ke = np.array([N, N, 399999, 333333, N, 250000], np.int32)
    out, tr, plan, ctr = run_gpu(X, ke, K, family=etk.FAMILY_CLUSTER_SPLIT)
    assert plan.splits == 16
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
    compare_trace(tr, tr_ref)


@pytest.mark.parametrize("dual", [0, 1])
def test_cluster_split_wide_forced_routes(dual):
    # Table 2's routes on rows wide enough for 16-CTA clusters, forced by
    # planting values on or off the sampled residue class.
    K, s, N = 64, 16, 400000
    q0 = -(-3 * K // (2 * s))
    q1 = -(-7 * K // (4 * s))
    rng = np.random.default_rng(18)
    base = rng.standard_normal(N).astype(np.float32)

    def planted(r, off_hi, off_mid):
        row = base.copy()
        a = oracle.view_phase(r, s)
        on = np.arange(a, N, s)
        off = np.setdiff1d(np.arange(N), on)[::997]  # spread over every segment
        row[on[:q0]] = 100.0
        row[on[q0:q1]] = 90.0
        row[off[:off_hi]] = 100.0
        row[off[off_hi:off_hi + off_mid]] = 90.0
        return row

    X = np.stack([base, planted(1, 30, 50), planted(2, 30, 0), base])
    ke = np.array([N, N, N, 100], np.int32)
    out, tr, plan, ctr = run_gpu(X, ke, K, family=etk.FAMILY_CLUSTER_SPLIT, stride=s, dual=dual)
    assert plan.splits == 16
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
    compare_trace(tr, tr_ref)
    if dual:
        assert tr[:, 0].tolist() == [1, 2, 3, 5]
    else:
        assert tr[:3, 0].tolist() == [1, 4, 4]


@pytest.mark.parametrize("splits", [1, 4, 7])
def test_stream_floor_reads_exactly_the_valid_prefixes(splits):
    # The streaming-floor kernel (a measurement utility): its per-segment
    # checksums equal XORs over the segments of each row's valid prefix.
    M, N = 5, 70001
    rng = np.random.default_rng(splits)
    X = rng.standard_normal((M, N)).astype(np.float32)
    ke = np.array([N, 0, 1, 33333, N + 9], np.int32)
    dev = torch.device("cuda")
    out = etk.stream_floor(torch.as_tensor(X).to(dev), torch.as_tensor(ke).to(dev), splits)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint32)
    bits = X.view(np.uint32)
    for r in range(M):
        L = int(min(max(int(ke[r]), 0), N))
        seg = ((L + splits - 1) // splits + 7) // 8 * 8
        for q in range(splits):
            lo, hi = min(L, q * seg), min(L, q * seg + seg)
            exp = np.bitwise_xor.reduce(bits[r, lo:hi]) if hi > lo else np.uint32(0)
            assert got[r, q] == exp, (r, q)


@pytest.mark.parametrize("workers", [1, 0])
def test_persistent_rows_deferred_at_their_band(workers):
    # Two-level rows whose view holds just enough ones for tau0 (Phase 2 runs
    # on chip) but not for tau1, whose bin then holds the whole row: such a
    # row leaves its band to the heavy-row epilogue.  Fewer and more ones
    # than K, mixed with ordinary rows.
    M, N, K, s = 12, 100000, 512, 64
    q0 = -(-3 * K // (2 * s))
    rng = np.random.default_rng(515)
    X = rng.standard_normal((M, N)).astype(np.float32)
    ke = np.full(M, N, np.int32)
    for r in range(0, M, 2):
        a = oracle.view_phase(r, s)
        on = np.arange(a, N, s)
        off = np.setdiff1d(np.arange(N), on)
        n = K + (r // 2) % 3 * 4 - 5  # K - 5, K - 1, K + 3
        X[r] = 0.0
        X[r, rng.permutation(on)[:q0]] = 1.0
        X[r, rng.permutation(off)[:n - q0]] = 1.0
    ke[4] = N - 3333
    X[4, ke[4]:] = np.nan
    out, tr, plan, ctr = run_gpu(X, ke, K, family=etk.FAMILY_PERSISTENT_SAMPLED, stride=s,
                                 dual=1, workers=workers)
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
    compare_trace(tr, tr_ref)
    # fewer ones than K: the band, run by the heavy-row epilogue; more: the
    # primary route on chip; row 4 (cut short) is deferred at its Phase 1
    assert tr[0:M:2, 0].tolist() == [2, 2, 1, 2, 2, 1]


@pytest.mark.parametrize("workers", [1, 3, 0])
def test_persistent_heavy_rows_deferred_and_overflowing(workers):
    # Rows whose view predicts a frontier far beyond on-chip capacity
    # (constant, -inf, signed-zero, two-level, subnormal and near-tie rows)
    # are finished after the CTA's other rows, by passes over the row itself;
    # on one worker more than its 63-entry list of such rows exist, and the
    # rest take the frontier route.  Mixed with ordinary, padded and empty
    # rows; lengths up to 100000 straddle the deferral threshold.
    M, N, K = 140, 100000, 512
    rng = np.random.default_rng(4242)
    X = rng.standard_normal((M, N)).astype(np.float32)
    ke = rng.integers(K + 1, N + 1, M).astype(np.int32)
    for r in range(M):
        kind = r % 7
        if kind == 0:
            X[r] = 0.75
        elif kind == 1:
            X[r] = -np.inf
        elif kind == 2:
            X[r] = np.where(rng.integers(0, 2, N) == 1, np.float32(-0.0), np.float32(0.0))
        elif kind == 3:
            X[r] = 0.0
            X[r, rng.permutation(N)[:K + (r % 5) - 2]] = 1.0
        elif kind == 4:  # subnormals of both signs: sign bit over a 23-bit mantissa
            X[r] = (rng.integers(1, 1 << 23, N).astype(np.uint32) |
                    (rng.integers(0, 2, N).astype(np.uint32) << np.uint32(31))).view(np.float32)
        elif kind == 5:  # K - 10 ones over two adjacent values, each far beyond capacity
            X[r] = np.where(rng.integers(0, 2, N) == 1, np.float32(0.5),
                            np.nextafter(np.float32(0.5), np.float32(1.0)))
            X[r, rng.permutation(N)[:K - 10]] = 1.0
    ke[5], ke[11], ke[17] = 0, K, 7
    for r in range(M):
        X[r, ke[r]:] = np.nan
    out, tr, plan, ctr = run_gpu(X, ke, K, family=etk.FAMILY_PERSISTENT_SAMPLED, workers=workers)
    compare_rows(X, ke, K, out)
    assert_counters_zero(ctr)
    _, tr_ref = oracle_trace_for_plan(X, ke, K, plan)
    compare_trace(tr, tr_ref)
