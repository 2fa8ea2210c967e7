"""CPU-only checks of the C ABI library: it loads without a GPU, exports every
entry point include/exact_topk.h declares, and its host logic (planner,
argument validation, error strings) behaves as documented.  No compute call
is made here."""

import ctypes
import os
import re

import pytest

import exact_top_selection_gb300 as etk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GB300 = etk.DeviceInfo(152, 3, 3, 1, 2)


def declared_functions():
    with open(os.path.join(ROOT, "include", "exact_topk.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_]+\**\s+\**(exact_topk\w*)\s*\(", text,
                                 re.M)))


def test_header_declares_the_expected_entry_points():
    assert set(declared_functions()) == set(etk.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(etk.library_path() if os.path.exists(etk.library_path()) else
                      etk.library()._name)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_error_strings():
    assert etk.version() == 10000
    for code in range(0, -9, -1):
        assert etk.error_string(code) and etk.error_string(code) != "unknown exact_topk status"
    assert etk.error_string(-99) == "unknown exact_topk status"


@pytest.mark.parametrize("M,N,K,family,stride,dual", [
    (4, 8192, 256, etk.FAMILY_ROW_LOCAL_EXACT, 64, 0),
    (64, 65536, 2048, etk.FAMILY_CLUSTER_SPLIT, 128, 1),
    (64, 131072, 2048, etk.FAMILY_CLUSTER_SPLIT, 128, 1),
    # a KV-split would give these rows one segment each: persistent instead
    (151, 131072, 2048, etk.FAMILY_PERSISTENT_SAMPLED, 128, 1),
    (128, 131072, 2048, etk.FAMILY_PERSISTENT_SAMPLED, 128, 1),
    (64, 262144, 2048, etk.FAMILY_KV_SPLIT, 128, 1),
    # narrow rows: exact kernel for one wave of rows or rows under 1K columns
    (100, 8192, 256, etk.FAMILY_ROW_LOCAL_EXACT, 64, 0),
    (5000, 512, 64, etk.FAMILY_ROW_LOCAL_EXACT, 64, 0),
    (5000, 2048, 64, etk.FAMILY_PERSISTENT_SAMPLED, 64, 0),
    (4096, 4096, 2048, etk.FAMILY_PERSISTENT_SAMPLED, 64, 0),
    (2048, 8192, 2048, etk.FAMILY_PERSISTENT_SAMPLED, 64, 0),
    (8, 140000, 2048, etk.FAMILY_KV_SPLIT, 128, 1),
    (4096, 131072, 2048, etk.FAMILY_PERSISTENT_SAMPLED, 128, 1),
    (8, 524288, 2048, etk.FAMILY_KV_SPLIT, 128, 1),
    (20, 300000, 2048, etk.FAMILY_KV_SPLIT, 128, 1),
    (256, 131072, 2048, etk.FAMILY_PERSISTENT_SAMPLED, 128, 1),
    (1000, 40000, 2048, etk.FAMILY_PERSISTENT_SAMPLED, 64, 0),
])
def test_planner_families(M, N, K, family, stride, dual):
    p = etk.make_plan(M, N, K, device_info=GB300)
    assert (p.family, p.stride, p.dual) == (family, stride, dual)
    # q = ceil(rho K / s) with rho = 3/2 and rho1 = 7/4 (sections 4.2, 6.4)
    assert p.q0 == -(-3 * K // (2 * stride)) and p.q1 == -(-7 * K // (4 * stride))
    assert p.counter_bytes >= 4 * (4 + M) and p.counter_bytes % 16 == 0
    if family == etk.FAMILY_KV_SPLIT:
        assert p.workers == M * p.splits and 1 <= p.splits <= 64
        assert p.workspace_bytes >= M * N * 8 + M * p.splits * 8
    elif family == etk.FAMILY_CLUSTER_SPLIT:
        # the fewest 16384-score segments that hold a row; no workspace
        assert p.splits == -(-N // 16384) and p.workers == M * p.splits
        assert p.workspace_bytes == 0 and p.cand_capacity == 16384
    elif N > p.cand_capacity:
        assert p.workers == min(M, 152 * (3 if family == 1 else 1))
        assert p.workspace_bytes >= p.workers * N * 8
    elif family == etk.FAMILY_PERSISTENT_SAMPLED:
        # no frontier slices; one 32-byte record per row for deferred rows
        assert p.workspace_bytes == -(-M * 32 // 256) * 256
    else:
        assert p.workspace_bytes == 0


def test_planner_takes_wide_clusters_on_request():
    # clusters of up to 16 CTAs hold 16384 scores each and read up to as many
    # again from global memory: rows up to 16 x 32768 scores
    p = etk.make_plan(8, 524288, 2048, device_info=GB300, family=etk.FAMILY_CLUSTER_SPLIT)
    assert (p.splits, p.workers, p.workspace_bytes) == (16, 128, 0)
    p = etk.make_plan(8, 300000, 2048, device_info=GB300, family=etk.FAMILY_CLUSTER_SPLIT,
                      splits=10)
    assert p.splits == 10
    for bad in (dict(splits=9), dict(splits=17)):
        with pytest.raises(etk.ExactTopKError) as e:
            etk.make_plan(8, 300000, 2048, device_info=GB300, family=etk.FAMILY_CLUSTER_SPLIT,
                          **bad)
        assert e.value.code == -7
    with pytest.raises(etk.ExactTopKError):
        etk.make_plan(8, 524289, 2048, device_info=GB300, family=etk.FAMILY_CLUSTER_SPLIT)


def test_planner_overrides_and_errors():
    p = etk.make_plan(10, 100000, 100, device_info=GB300, family=etk.FAMILY_KV_SPLIT, splits=7,
                      stride=32, dual=0, rho0=(5, 4))
    assert (p.family, p.splits, p.stride, p.dual, p.rho0_num, p.rho0_den) == (2, 7, 32, 0, 5, 4)
    assert p.q0 == -(-5 * 100 // (4 * 32))
    bad = [dict(num_rows=0, max_kv_len=10, top_k=1), dict(num_rows=1, max_kv_len=0, top_k=1),
           dict(num_rows=1, max_kv_len=10, top_k=1, row_pitch=9)]
    for kw in bad:
        with pytest.raises(etk.ExactTopKError) as e:
            etk.make_plan(device_info=GB300, **kw)
        assert e.value.code == -2
    for k in (0, 16385):
        with pytest.raises(etk.ExactTopKError) as e:
            etk.make_plan(4, 100, k, device_info=GB300)
        assert e.value.code == -3
    for kw in (dict(stride=3), dict(stride=8192), dict(family=9), dict(splits=300,
               family=etk.FAMILY_KV_SPLIT), dict(dual=2), dict(family=etk.FAMILY_CLUSTER_SPLIT,
               splits=3), dict(family=etk.FAMILY_CLUSTER_SPLIT, splits=17)):
        with pytest.raises(etk.ExactTopKError) as e:
            etk.make_plan(4, 100000, 16, device_info=GB300, **kw)
        assert e.value.code == -7


def _fake(addr):
    return ctypes.c_void_p(addr)


def test_run_validates_arguments_without_touching_the_gpu():
    # Fake, never-dereferenced addresses: every call below must be rejected on
    # the host before any CUDA call.
    lib = etk.library()
    p = etk.make_plan(64, 65536, 2048, device_info=GB300, family=etk.FAMILY_KV_SPLIT)
    X, ke, out, ctr, ws = (_fake(0x100000 * i) for i in range(1, 6))
    cb, wb = p.counter_bytes, p.workspace_bytes
    run = lambda *a: lib.exact_topk_run(ctypes.byref(p), *a)
    assert run(None, ke, out, None, ctr, cb, ws, wb, None, None, None) == -1
    assert run(X, ke, out, None, None, cb, ws, wb, None, None, None) == -1
    assert run(X, ke, out, None, ctr, cb - 16, ws, wb, None, None, None) == -4
    assert run(X, ke, out, None, ctr, cb, ws, wb - 1, None, None, None) == -5
    assert run(_fake(0x100002), ke, out, None, ctr, cb, ws, wb, None, None, None) == -6
    assert run(X, ke, out, None, _fake(0x100008), cb, ws, wb, None, None, None) == -6
    q = etk.Plan.from_buffer_copy(p)
    q.cand_capacity = 5
    assert lib.exact_topk_run(ctypes.byref(q), X, ke, out, None, ctr, cb, ws, wb, None, None,
                              None) == -7
    q = etk.Plan.from_buffer_copy(p)
    q.workspace_bytes = 1
    assert lib.exact_topk_run(ctypes.byref(q), X, ke, out, None, ctr, cb, ws, wb, None, None,
                              None) == -7
    assert lib.exact_topk(None, 4, 100, ke, out, None, 10, ctr, 64, ws, 0, None, None) == -1
