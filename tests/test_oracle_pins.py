"""Pins the CPU oracle to facts that do not come from the oracle itself.

Citations are to "Sample-Guided Exact Top-K Selection for Long-Context Sparse
Attention": section 2.1 (operator contract), section 4.2 (coarse map, eqs.
11-15), section 4.3 (admitted tail, Lemma 4.1, eqs. 16-21), section 4.4
(radix refinement, eqs. 22-25, Theorem 4.2), section 6.1 (exactness
criterion, eq. 30) and Table 2 (routes).

Independent references used here: brute-force enumeration of K-subsets,
numpy's sort, numpy's IEEE binary16 cast, closed-form rows, hand-computed
fixtures under tests/golden/, and invariants stated on the pages.
"""

import itertools
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32(bits):
    return np.array(bits, dtype=np.uint32).view(np.float32)


def bits(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def numeric_topk_values(row, K):
    """K largest values of a row by numpy's numeric sort (-0 == +0)."""
    return np.sort(row.astype(np.float64))[::-1][:K]


def selected_values(row, idx):
    idx = np.asarray(idx)
    return row[idx[idx >= 0]]


def is_exact(row, L, K, idx):
    """Exactness criterion of eq. (30) plus the sentinel rule of section 2.1."""
    idx = np.asarray(idx)
    if L <= K:
        return sorted(idx[idx >= 0].tolist()) == list(range(L)) and int((idx == -1).sum()) == K - L
    if (idx < 0).any() or (idx >= L).any() or len(set(idx.tolist())) != K:
        return False
    sel = np.zeros(L, dtype=bool)
    sel[idx] = True
    v = row[:L].astype(np.float64)
    return v[sel].min() >= (v[~sel].max() if (~sel).any() else -np.inf)


# ---------------------------------------------------------------- FP16 projection


def test_f16_projection_matches_numpy_random_patterns():
    rng = np.random.default_rng(1)
    u = rng.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    x = x[~np.isnan(x)]
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = oracle.f16_bits_array(x)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(hex(int(bits(x[i]))), hex(int(ref[i])), hex(int(got[i]))) for i in bad[:5]]


def test_f16_projection_matches_numpy_at_rounding_boundaries():
    # Every binary32 exponent crossed with the mantissa patterns that sit on,
    # just below and just above each rounding midpoint of the binary16 grid,
    # for both the normal (13 dropped bits) and subnormal half ranges.
    lows = []
    for drop in range(13, 25):
        half = 1 << (drop - 1)
        for base in (0, 1 << drop, 3 << drop, (1 << 23) - (1 << drop)):
            for d in (-1, 0, 1):
                lows.append((base + half + d) & 0x7FFFFF)
    lows += [0, 1, 0x7FFFFF, 0x400000]
    exps = np.arange(0, 255, dtype=np.uint32)
    man = np.array(sorted(set(lows)), dtype=np.uint32)
    u = (exps[:, None] << 23 | man[None, :]).ravel()
    u = np.concatenate([u, u | 0x80000000])
    x = u.view(np.float32)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = oracle.f16_bits_array(x)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(hex(int(u[i])), hex(int(ref[i])), hex(int(got[i]))) for i in bad[:5]]


# ---------------------------------------------------------------- coarse map (eq. 11)


def _golden_coarse():
    rows = []
    with open(os.path.join(GOLDEN, "coarse_bins.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b, c = line.split()
            rows.append((int(a, 16), int(b, 16), int(c)))
    return rows


@pytest.mark.parametrize("u,h,c", _golden_coarse())
def test_coarse_bin_golden(u, h, c):
    x = f32([u])[0]
    assert oracle.f16_bits(x) == h
    assert oracle.coarse_bin(x) == c


def test_coarse_bins_cover_every_half_in_descending_order():
    # Every non-NaN binary16 value, sorted by numpy in descending numeric
    # order (+0 placed before -0), must receive kappa_down16 = 0x3FF + rank:
    # the 0x3FF smaller keys belong to positive NaN patterns.  Hence bin b
    # holds exactly the 32 consecutive halves of ranks 32b - 0x3FF .. +31.
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = h.view(np.float16)
    keep = ~np.isnan(v)
    h, v = h[keep], v[keep]
    signbit = (h >> 15).astype(np.int64)
    order = np.lexsort((signbit, -v.astype(np.float64)))  # value desc, then +0 before -0
    halves = h[order].view(np.float16).astype(np.float32)
    got = oracle.coarse_bin_array(halves)
    rank = np.arange(halves.size)
    assert np.array_equal(got, (0x3FF + rank) >> 5)


def test_coarse_map_is_monotone_eq12():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(200000).astype(np.float32) * 10.0 ** rng.integers(-40, 39, 200000),
                        f32([0, 0x80000000, 0x7F800000, 0xFF800000, 1, 0x80000001])]).astype(np.float32)
    x = x[np.isfinite(x) | np.isinf(x)]
    c = oracle.coarse_bin_array(x)
    order = np.argsort(-x.astype(np.float64), kind="stable")
    cs = c[order]
    # x_i > x_j  =>  c(x_i) <= c(x_j): along descending values the bins never decrease.
    assert (np.diff(cs) >= 0).all()


# ---------------------------------------------------------------- inclusive cutoff (section 4.3)


@pytest.mark.parametrize("tau", [31, 32, 100, 543, 574, 575, 900, 1023, 1024, 1500, 2015, 2016, 2047])
def test_cutoff_is_largest_key_of_admitted_prefix(tau):
    T = oracle.cutoff_for_bin(tau)
    x_T = f32([_bits_from_desc(T)])[0]
    assert oracle.coarse_bin(x_T) <= tau
    if T < 0xFF800000:
        x_next = f32([_bits_from_desc(T + 1)])[0]
        assert oracle.coarse_bin(x_next) > tau


def _bits_from_desc(k):
    a = (~k) & 0xFFFFFFFF
    return (a & 0x7FFFFFFF) if a & 0x80000000 else (~a) & 0xFFFFFFFF


def test_cutoff_compare_reproduces_coarse_prefix():
    # Comparing desc32 keys with the cutoff admits exactly {c(x) <= tau}
    # (section 5.3: the raw FP32 compare "reproduces the selected coarse
    # prefix, including its boundary value").
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(100000) * 4).astype(np.float32)
    x = np.concatenate([x, np.nextafter(x, np.float32(np.inf)), np.nextafter(x, np.float32(-np.inf))])
    c = oracle.coarse_bin_array(x)
    u = bits(x).astype(np.uint64)
    asc = np.where(u & 0x80000000, (~u) & 0xFFFFFFFF, u | 0x80000000)
    desc = (~asc) & 0xFFFFFFFF
    for tau in (500, 540, 543, 560, 1023, 1024, 1100, 1500):
        T = oracle.cutoff_for_bin(tau)
        assert np.array_equal(desc <= T, c <= tau)


# ---------------------------------------------------------------- definition: Top-K


def test_definition_against_brute_force_subsets():
    rng = np.random.default_rng(4)
    for trial in range(300):
        L = int(rng.integers(0, 10))
        K = int(rng.integers(1, 12))
        row = rng.integers(-2, 3, size=max(L, 1)).astype(np.float32)
        X = np.full((1, max(L, 1) + 2), np.nan, dtype=np.float32)
        X[0, :L] = row[:L]
        out = oracle.topk_rows(X, np.array([L], np.int32), K)[0]
        if L <= K:
            assert sorted(out[out >= 0].tolist()) == list(range(L))
            assert int((out == -1).sum()) == K - L
            continue
        exact_sets = []
        for S in itertools.combinations(range(L), K):
            rest = [j for j in range(L) if j not in S]
            if min(row[list(S)]) >= max(row[rest]):
                exact_sets.append(set(S))
        assert set(out.tolist()) in exact_sets


def test_definition_against_numpy_sort():
    rng = np.random.default_rng(5)
    for trial in range(40):
        N = int(rng.integers(1, 65536))
        K = int(rng.choice([1, 7, 64, 256, 2048]))
        kind = trial % 4
        if kind == 0:
            row = rng.standard_normal(N).astype(np.float32)
        elif kind == 1:
            row = rng.integers(-5, 5, N).astype(np.float32)
        elif kind == 2:
            row = f32(rng.integers(0, 1 << 32, N, dtype=np.uint64).astype(np.uint32))
            row[np.isnan(row)] = 0.0
        else:
            row = (rng.standard_normal(N) * 1e-39).astype(np.float32)  # subnormals
        X = row[None, :]
        out = oracle.topk_rows(X, np.array([N], np.int32), K)[0]
        assert is_exact(row, N, K, out)
        got = np.sort(selected_values(row, out).astype(np.float64))[::-1]
        assert np.array_equal(got, numeric_topk_values(row, min(K, N)))


def test_definition_closed_form_permutation_rows():
    # x_i = f(pi(i)) with f strictly increasing selects {i : pi(i) >= L - K}.
    rng = np.random.default_rng(6)
    for L, K in [(10, 3), (1000, 1), (5000, 2048), (65536, 2048), (3000, 2999)]:
        pi = rng.permutation(L)
        row = (pi.astype(np.float64) * 0.25 - 100.0).astype(np.float32)  # exact in float32
        out = oracle.topk_rows(row[None, :], np.array([L], np.int32), K)[0]
        assert set(out.tolist()) == set(np.nonzero(pi >= L - K)[0].tolist())


def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "special_rows.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, K, ke, row, exp, pad = [p.strip() for p in line.split("|")]
            rows.append((name, int(K), int(ke), [int(t, 16) for t in row.split()],
                         [int(t, 16) for t in exp.split()], int(pad)))
    return rows


@pytest.mark.parametrize("name,K,ke,row,exp,pad", _golden_rows(), ids=[r[0] for r in _golden_rows()])
def test_definition_golden_special_rows(name, K, ke, row, exp, pad):
    X = f32(row)[None, :]
    out = oracle.topk_rows(X, np.array([ke], np.int32), K)[0]
    got = bits(X[0][out[out >= 0]])
    # sort selected bit patterns by value descending, -0 below +0
    key = np.where(got & 0x80000000, (~got) & 0xFFFFFFFF, got | 0x80000000)
    got = got[np.argsort(-key.astype(np.int64), kind="stable")]
    assert got.tolist() == exp
    assert int((out == -1).sum()) == pad


def test_definition_constant_and_two_level_rows():
    L, K = 5000, 2048
    row = np.full(L, 0.5, np.float32)
    out = oracle.topk_rows(row[None, :], np.array([L], np.int32), K)[0]
    assert len(set(out.tolist())) == K and (out >= 0).all() and (out < L).all()
    for ones in (10, 2047, 2048, 2049, 4000):
        row = np.zeros(L, np.float32)
        row[np.random.default_rng(ones).permutation(L)[:ones]] = 1.0
        out = oracle.topk_rows(row[None, :], np.array([L], np.int32), K)[0]
        assert int(row[out].sum()) == min(K, ones)


def test_definition_clamps_lengths_and_leaves_dead_rows():
    X = np.arange(40, dtype=np.float32).reshape(4, 10)
    ke = np.array([-3, 25, 4, 10], np.int32)
    out = oracle.topk_rows(X, ke, 3, M_live=3)
    assert (out[0] == -1).all()
    assert sorted(out[1].tolist()) == [7, 8, 9]
    assert sorted(out[2].tolist()) == [1, 2, 3]
    assert (out[3] == -7).all()  # row >= M_live untouched


# ---------------------------------------------------------------- method oracle


def test_view_phase_is_a_permutation_per_block_of_rows():
    # "Every block of s rows consequently uses each phase once" (section 4.2).
    for s in (16, 64, 128, 256):
        for block in range(3):
            phases = [oracle.view_phase(block * s + t, s) for t in range(s)]
            assert sorted(phases) == list(range(s))


def _method_rows(rng, n_rows, N, kind):
    if kind == "normal":
        X = rng.standard_normal((n_rows, N)).astype(np.float32)
    elif kind == "quantized":
        X = (np.clip(np.round(rng.standard_normal((n_rows, N)) * 32), -128, 127) / 32).astype(np.float32)
    elif kind == "ties":
        X = rng.integers(0, 3, (n_rows, N)).astype(np.float32)
    else:
        X = np.exp(rng.standard_normal((n_rows, N)) * 3).astype(np.float32)
    return X


@pytest.mark.parametrize("kind", ["normal", "quantized", "ties", "lognormal"])
@pytest.mark.parametrize("s,dual,K", [(16, True, 64), (64, False, 256), (128, True, 256), (32, True, 1)])
def test_method_matches_definition(kind, s, dual, K):
    rng = np.random.default_rng(hash((kind, s, K)) & 0xFFFF)
    M, N = 24, 6000
    X = _method_rows(rng, M, N, kind)
    ke = rng.integers(0, N + 1, M).astype(np.int32)
    ke[:3] = [N, K, K + 1]
    ref = oracle.topk_rows(X, ke, K)
    out, tr = oracle.method_trace(X, ke, K, s, dual)
    for r in range(M):
        L = int(ke[r])
        assert is_exact(X[r], L, K, out[r]), (r, tr[r])
        a = np.sort(bits(selected_values(X[r], out[r])))
        b = np.sort(bits(selected_values(X[r], ref[r])))
        assert np.array_equal(a, b)


def test_method_trace_invariants():
    rng = np.random.default_rng(7)
    M, N, K, s = 64, 20000, 256, 64
    X = rng.standard_normal((M, N)).astype(np.float32)
    ke = rng.integers(0, N + 1, M).astype(np.int32)
    out, tr = oracle.method_trace(X, ke, K, s, True)
    q0 = -(-3 * K // (2 * s))
    q1 = -(-7 * K // (4 * s))
    for r in range(M):
        L = int(ke[r])
        route, tau0, tau1, c0, c1, tstar, e0, q0n = tr[r].tolist()
        if L <= K:
            assert route == oracle.ROUTE_PAD
            continue
        c = oracle.coarse_bin_array(X[r, :L])
        a = oracle.view_phase(r, s)
        sample = np.sort(c[a::s])
        if sample.size < q1:
            assert route == oracle.ROUTE_DIRECT_EXACT
        else:
            # tau0 is the q0-th smallest sampled coarse bin (eq. 15).
            assert tau0 == sample[q0 - 1] and tau1 == sample[q1 - 1]
            assert c0 == int((c <= tau0).sum())
            if c0 >= K:
                assert route == oracle.ROUTE_PRIMARY and q0n == c0 and e0 == 0
                # Lemma 4.1: the admitted tail contains a Top-K solution.
                v = X[r, :L].astype(np.float64)
                adm = c <= tau0
                assert v[adm].min() >= (v[~adm].max() if (~adm).any() else -np.inf)
            else:
                assert c1 == int((c <= tau1).sum())
                assert route in (oracle.ROUTE_BAND, oracle.ROUTE_EXACT_AFTER_BAND)
                assert (route == oracle.ROUTE_BAND) == (c1 >= K)
        if route in (oracle.ROUTE_DIRECT_EXACT, oracle.ROUTE_EXACT_AFTER_BAND):
            # eq. 20: tau* = min{b : C(b) >= K}
            assert int((c <= tstar).sum()) >= K and int((c < tstar).sum()) < K
            assert e0 == int((c < tstar).sum()) and q0n == int((c == tstar).sum())


def test_method_forced_routes():
    # Table 2 routes forced by construction.  The view phase a_r is a pure
    # function of r (eq. 13), so large values planted on the sampled residue
    # class make the sample overestimate the tail and the primary underfill.
    K, s, N = 64, 16, 8192
    q0 = -(-3 * K // (2 * s))  # 6
    q1 = -(-7 * K // (4 * s))  # 7
    rng = np.random.default_rng(8)
    base = rng.standard_normal(N).astype(np.float32)

    def planted(r, off_view_hi, off_view_mid):
        row = base.copy()
        a = oracle.view_phase(r, s)
        on = np.arange(a, N, s)
        off = np.array([i for i in range(N) if i % s != a])
        row[on[:q0]] = 100.0
        row[on[q0:q1]] = 90.0
        row[off[:off_view_hi]] = 100.0
        row[off[off_view_hi:off_view_hi + off_view_mid]] = 90.0
        return row

    rows = [base.copy(),                 # r=0: typical row, primary
            planted(1, 30, 50),          # r=1: C(tau0)=36 < K <= C(tau1)=87: band
            planted(2, 30, 0),           # r=2: C(tau1)=37 < K: exact after band
            base.copy()]                 # r=3: |V| < q1: direct exact
    X = np.stack(rows)
    ke = np.array([N, N, N, 100], np.int32)  # r=3: phase 12, 6 sampled values < q1
    out, tr = oracle.method_trace(X, ke, K, s, True)
    assert tr[:, 0].tolist() == [oracle.ROUTE_PRIMARY, oracle.ROUTE_BAND,
                                 oracle.ROUTE_EXACT_AFTER_BAND, oracle.ROUTE_DIRECT_EXACT]
    assert tr[1, 3] == 36 and tr[1, 4] == 87 and tr[2, 4] == 37
    _, tr = oracle.method_trace(X, ke, K, s, False)
    assert tr[1, 0] == oracle.ROUTE_EXACT_NO_BAND and tr[2, 0] == oracle.ROUTE_EXACT_NO_BAND
    ref = oracle.topk_rows(X, ke, K)
    for r in range(4):
        assert is_exact(X[r], int(ke[r]), K, out[r])
        assert np.array_equal(np.sort(bits(X[r][out[r]])), np.sort(bits(X[r][ref[r]])))


def test_method_guess_routes():
    rng = np.random.default_rng(9)
    M, N, K = 6, 4000, 128
    X = rng.standard_normal((M, N)).astype(np.float32)
    ke = np.full(M, N, np.int32)
    ref = oracle.topk_rows(X, ke, K)
    guess = ref.copy()
    guess[1] = rng.permutation(N)[:K]          # a poor guess is still certified (loose)
    guess[2, 5] = -1                            # an invalid entry: falls back to sampling
    guess[3, 7] = guess[3, 8]                   # duplicates can underfill only if C < K
    guess[4] = np.arange(K)                     # arbitrary valid guess
    out, tr = oracle.method_trace(X, ke, K, 16, True, guess=guess)
    assert tr[0, 0] == oracle.ROUTE_GUESS and tr[0, 3] >= K
    assert tr[1, 0] == oracle.ROUTE_GUESS
    assert tr[2, 0] in (oracle.ROUTE_PRIMARY, oracle.ROUTE_BAND, oracle.ROUTE_EXACT_AFTER_BAND)
    for r in range(M):
        assert is_exact(X[r], N, K, out[r])
    # A guess made of K copies of one index can only certify by luck.
    g2 = np.tile(np.argmax(X, axis=1)[:, None], (1, K)).astype(np.int32)
    out, tr = oracle.method_trace(X, ke, K, 16, True, guess=g2)
    assert (tr[:, 0] == oracle.ROUTE_GUESS_EXACT).all()
    for r in range(M):
        assert is_exact(X[r], N, K, out[r])


def test_method_thread_count_does_not_change_results():
    rng = np.random.default_rng(10)
    X = rng.standard_normal((33, 3000)).astype(np.float32)
    ke = rng.integers(0, 3001, 33).astype(np.int32)
    o1, t1 = oracle.method_trace(X, ke, 100, 16, True, nthreads=1)
    o8, t8 = oracle.method_trace(X, ke, 100, 16, True, nthreads=8)
    assert np.array_equal(o1, o8) and np.array_equal(t1, t8)
