"""Seeded synthetic score matrices for exact row-wise Top-K.

This module holds input generators only: none of the selection method's
arithmetic lives here.  Both the CUDA path's tests/bench and the CPU oracle
receive the same materialized matrices from it.

The five named workloads stand in for the indexer-score captures the paper
measures on ("Sample-Guided Exact Top-K Selection for Long-Context Sparse
Attention", section 6.1), which are not available.  Their score model is the
indexer of section 2.1 eq. (1): per row r, 16 heads with query vectors
q_{r,h} ~ N(0, 1)^64 and weights w_{r,h} ~ U(0, 1); one shared key set
k_j ~ N(0, 1)^64 (a single KV cache); score s_{r,j} = sum_h w_{r,h} *
ReLU(q_{r,h} . k_j), computed in FP32 without TF32.

Padded columns (j >= ke[r]) are filled with NaN bit patterns, so a kernel
that reads past the valid prefix produces wrong results instead of passing by
accident.
"""

from __future__ import annotations

import dataclasses
import math

import torch

HEADS = 16
HEAD_DIM = 64


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    kind: str  # "iid", "indexer", "indexer_causal", "adversarial"
    seed: int
    description: str


WORKLOADS = {
    "short_iid": Workload("short_iid", 4, 8192, 256, "iid", 20260001,
                          "M=4 rows, N=8192, ke=8192, K=256; i.i.d. N(0,1) FP32"),
    "decode_batch": Workload("decode_batch", 64, 65536, 2048, "indexer", 20260002,
                             "decode batch M=64, N=65536, ke~U[2048,65536], K=2048; indexer-like"),
    "prefill_causal": Workload("prefill_causal", 4096, 131072, 2048, "indexer_causal", 20260003,
                               "prefill causal M=4096, N=131072, ke[r]=N-M+r+1, K=2048; indexer-like"
                               " + 0.1*sin(j/4096), NaN padding"),
    "long_decode": Workload("long_decode", 8, 524288, 2048, "indexer", 20260004,
                            "long-context decode M=8, N=524288, ke~U[500000,524288], K=2048;"
                            " indexer-like"),
    "adversarial": Workload("adversarial", 256, 131072, 2048, "adversarial", 20260005,
                            "adversarial M=256, N=131072, ke~U[1,131072], K=2048; 256-level"
                            " quantized scores, constant rows, +-0/+-inf/subnormal rows"),
}

ORDER = ["short_iid", "decode_batch", "prefill_causal", "long_decode", "adversarial"]


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randint(g, lo, hi, n, device):
    """Uniform integers in [lo, hi] (inclusive)."""
    return torch.randint(int(lo), int(hi) + 1, (n,), generator=g, device=device, dtype=torch.int64)


def indexer_scores(M, N, g, device, chunk_rows=None):
    """s_{r,j} = sum_h w_{r,h} ReLU(q_{r,h} . k_j), FP32 without TF32."""
    keys = torch.randn(N, HEAD_DIM, generator=g, device=device, dtype=torch.float32)
    q = torch.randn(M, HEADS, HEAD_DIM, generator=g, device=device, dtype=torch.float32)
    w = torch.rand(M, HEADS, generator=g, device=device, dtype=torch.float32)
    out = torch.empty(M, N, device=device, dtype=torch.float32)
    if chunk_rows is None:
        budget = (1 << 29) if device != "cpu" and str(device).startswith("cuda") else (1 << 26)
        chunk_rows = max(1, budget // (HEADS * N * 4))
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        for r0 in range(0, M, chunk_rows):
            r1 = min(M, r0 + chunk_rows)
            s = torch.relu(q[r0:r1].reshape(-1, HEAD_DIM) @ keys.T).reshape(r1 - r0, HEADS, N)
            out[r0:r1] = torch.einsum("rhn,rh->rn", s, w[r0:r1])
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    return out


def nan_garbage(n, g, device):
    """NaN bit patterns: quiet NaN, all-ones, and random payloads of either sign."""
    kind = torch.randint(0, 3, (n,), generator=g, device=device, dtype=torch.int64)
    payload = torch.randint(1, 1 << 22, (n,), generator=g, device=device, dtype=torch.int64)
    sign = torch.randint(0, 2, (n,), generator=g, device=device, dtype=torch.int64) << 31
    rnd = sign | 0x7F800000 | payload
    bits = torch.where(kind == 0, torch.full_like(payload, 0x7FC00000),
                       torch.where(kind == 1, torch.full_like(payload, 0xFFFFFFFF), rnd))
    return _bits_to_f32(bits)


def _bits_to_f32(bits_i64):
    b = bits_i64 & 0xFFFFFFFF
    b = torch.where(b >= (1 << 31), b - (1 << 32), b)
    return b.to(torch.int32).view(torch.float32)


def pad_with_nan(X, ke, g):
    """Overwrites X[r, ke[r]:] with NaN garbage."""
    M, N = X.shape
    cols = torch.arange(N, device=X.device).unsqueeze(0)
    mask = cols >= ke.to(X.device).unsqueeze(1).to(torch.int64)
    n = int(mask.sum().item())
    if n:
        X[mask] = nan_garbage(n, g, X.device)
    return X


def _adversarial(M, N, K, g, device, ke):
    z = torch.randn(M, N, generator=g, device=device, dtype=torch.float32)
    X = torch.clamp(torch.round(z * 32.0), -128.0, 127.0) / 32.0  # 256 levels
    for r in range(M):
        L = int(ke[r])
        if L <= 0:
            continue
        kind = r % 16
        row = X[r, :L]
        if kind == 0:  # constant row
            row.fill_(0.5)
        elif kind == 1:  # a few +inf
            n = min(L, 64)
            pos = torch.randperm(L, generator=g, device=device)[:n]
            row[pos] = math.inf
        elif kind == 2:  # +inf straddling rank K
            n = min(L, K + (r // 16) % 3 - 1)
            pos = torch.randperm(L, generator=g, device=device)[:n]
            row[pos] = math.inf
        elif kind == 3:  # -inf only
            row.fill_(-math.inf)
        elif kind == 4:  # signed zeros only
            sgn = torch.randint(0, 2, (L,), generator=g, device=device, dtype=torch.int64)
            row.copy_(torch.where(sgn == 1, torch.tensor(-0.0, device=device),
                                  torch.tensor(0.0, device=device)))
        elif kind == 5:  # subnormals of both signs and zeros
            mant = torch.randint(0, 1 << 23, (L,), generator=g, device=device, dtype=torch.int64)
            sgn = torch.randint(0, 2, (L,), generator=g, device=device, dtype=torch.int64) << 31
            mant = torch.where(mant % 7 == 0, torch.zeros_like(mant), mant)
            row.copy_(_bits_to_f32(sgn | mant))
        elif kind == 6:  # two levels: about K ones, rest zeros
            n = min(L, K + (r // 16) % 5 - 2)
            row.fill_(0.0)
            pos = torch.randperm(L, generator=g, device=device)[:n]
            row[pos] = 1.0
        elif kind == 7:  # many equal maxima: a tie band far larger than K
            n = min(L, 3 * K)
            pos = torch.randperm(L, generator=g, device=device)[:n]
            row[pos] = 3.96875
    return X


def make_ke(w: Workload, M, N, K, g, device):
    if w.kind == "iid":
        return torch.full((M,), N, dtype=torch.int32, device=device)
    if w.kind == "indexer_causal":
        r = torch.arange(M, device=device, dtype=torch.int64)
        return (N - M + r + 1).clamp(min=0).to(torch.int32)
    if w.name == "long_decode":  # ke in [500000, 524288] at full width, same fraction when scaled
        lo = max(min(K, N), (N * 500000 + 524287) // 524288)
        return _randint(g, lo, N, M, device).to(torch.int32)
    if w.kind == "indexer":
        lo = min(K, N)
        return _randint(g, lo, N, M, device).to(torch.int32)
    # adversarial
    ke = _randint(g, 1, N, M, device)
    forced = [1, 7, K - 1, K]
    for r, v in enumerate(forced[:M]):
        ke[r] = min(v, N)
    return ke.to(torch.int32)


def generate(name_or_workload, M=None, N=None, K=None, device="cpu", seed=None):
    """Materializes (X [M, N] float32, ke [M] int32, K) for a named workload.

    M, N, K default to the workload's full sizes; smaller values give scaled
    versions with the same value model and length recipe."""
    w = WORKLOADS[name_or_workload] if isinstance(name_or_workload, str) else name_or_workload
    M = w.M if M is None else int(M)
    N = w.N if N is None else int(N)
    K = w.K if K is None else int(K)
    seed = w.seed if seed is None else int(seed)
    device = str(device)
    g = _gen(device, seed)
    ke = make_ke(w, M, N, K, g, device)
    if w.kind == "iid":
        X = torch.randn(M, N, generator=g, device=device, dtype=torch.float32)
    elif w.kind in ("indexer", "indexer_causal"):
        X = indexer_scores(M, N, g, device)
        if w.kind == "indexer_causal":
            j = torch.arange(N, device=device, dtype=torch.float32)
            X += 0.1 * torch.sin(j / 4096.0)
    else:
        X = _adversarial(M, N, K, g, device, ke.cpu())
    pad_with_nan(X, ke, g)
    return X, ke, K


def iid_rows(M, N, seed, device="cpu", dist="normal"):
    """Plain i.i.d. rows for tests: 'normal', 'uniform', 'int' (small integers, many ties)."""
    g = _gen(device, seed)
    if dist == "normal":
        return torch.randn(M, N, generator=g, device=device, dtype=torch.float32)
    if dist == "uniform":
        return torch.rand(M, N, generator=g, device=device, dtype=torch.float32)
    if dist == "int":
        return torch.randint(-3, 4, (M, N), generator=g, device=device).to(torch.float32)
    raise ValueError(dist)


def decode_batch_series(M, N, K, steps, seed, device="cpu", drift=0.05):
    """A decode batch followed over `steps` steps: indexer-like scores that drift
    by `drift` * N(0,1) per step, lengths ~ U[K, N - steps] that grow by one
    position per step (one new token), NaN padding beyond each length.

    Returns lists (X_t, ke_t) of device tensors; step t+1 is correlated with
    step t, which is what a previous-step Top-K guess relies on."""
    g = _gen(device, seed)
    X = indexer_scores(M, N, g, device)
    ke0 = _randint(g, min(K, N), max(min(K, N), N - steps), M, device).to(torch.int32)
    Xs, kes = [], []
    for t in range(steps):
        if t:
            X = X + drift * torch.randn(M, N, generator=g, device=device, dtype=torch.float32)
        ke_t = (ke0 + t).clamp(max=N).to(torch.int32)
        Xt = X.clone()
        pad_with_nan(Xt, ke_t, g)
        Xs.append(Xt)
        kes.append(ke_t)
    return Xs, kes


def decode_series(M, N, K, steps, seed, device="cpu", drift=0.05):
    """Temporally correlated decode steps: step t+1 = step t + drift * noise.

    Yields (X_t, ke_t); lengths grow by one position per step, as in decoding."""
    g = _gen(device, seed)
    base = indexer_scores(M, N, g, device)
    lo = max(K + 1, N - steps - 64)
    ke = _randint(g, lo, N - steps, M, device).to(torch.int32)
    X = base.clone()
    for t in range(steps):
        if t:
            X = X + drift * torch.randn(M, N, generator=g, device=device, dtype=torch.float32)
        ke_t = (ke + t).clamp(max=N).to(torch.int32)
        Xt = X.clone()
        pad_with_nan(Xt, ke_t, g)
        yield Xt, ke_t


TRACE_WIDTHS = (4096, 8192, 16384, 32768, 65536, 131072, 262144, 524288)


def trace_sequence(total, K, seed, device="cpu", widths=TRACE_WIDTHS):
    """A serving-style sequence of calls whose row width grows while the row
    count shrinks with it (M = total // N, at least one row), the shape of an
    engine moving from prefill chunks to long decode contexts.  Lengths are
    uniform in [N/2, N] (at least one position), scores indexer-like with NaN
    garbage beyond each length.

    Returns a list of (X, ke) device tensors, one per call."""
    g = _gen(device, seed)
    calls = []
    for N in widths:
        M = max(1, total // N)
        X = indexer_scores(M, N, g, device)
        ke = _randint(g, max(1, N // 2), N, M, device).to(torch.int32)
        pad_with_nan(X, ke, g)
        calls.append((X, ke))
    return calls
