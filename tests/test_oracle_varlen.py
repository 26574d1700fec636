"""Pins of the packed variable-length oracle (``oracle.recurrence_varlen``).

The pages name dynamic sequence packing ("Mamba-2架构深度解析" §5) without
defining it; the reading here is that each packed sequence is its own
recurrence, restarting from its own initial state at its first token.  These
tests pin the oracle to that definition without going through the C oracle:
a pure-Python fp64 loop over the recurrence, written out per token, plus
properties any correct packing has.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _inputs(T, H, P, N, G, nseq, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, P, generator=g, dtype=torch.float64).float()
    dt = (torch.rand(T, H, generator=g, dtype=torch.float64) * 0.2 + 0.01).float()
    A = (-torch.rand(H, generator=g, dtype=torch.float64) * 2 - 0.1).float()
    B = torch.randn(T, G, N, generator=g, dtype=torch.float64).float()
    C = torch.randn(T, G, N, generator=g, dtype=torch.float64).float()
    D = torch.randn(H, generator=g, dtype=torch.float64).float()
    init = torch.randn(nseq, H, P, N, generator=g, dtype=torch.float64).float()
    return x, dt, A, B, C, D, init


def _brute(x, dt, A, B, C, D, init, cu):
    """Per token, per (h, p): s = exp(dt A) s + dt x B; y = C . s + D x; s restarts at each sequence."""
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    y = np.zeros((T, H, P))
    fin = np.zeros((len(cu) - 1, H, P, N))
    for s in range(len(cu) - 1):
        for h in range(H):
            g = h // (H // G)
            for p in range(P):
                st = [float(init[s, h, p, n]) if init is not None else 0.0 for n in range(N)]
                for t in range(cu[s], cu[s + 1]):
                    a = math.exp(float(dt[t, h]) * float(A[h]))
                    for n in range(N):
                        st[n] = a * st[n] + float(dt[t, h]) * float(x[t, h, p]) * float(B[t, g, n])
                    y[t, h, p] = sum(float(C[t, g, n]) * st[n] for n in range(N)) + float(D[h]) * float(x[t, h, p])
                fin[s, h, p] = st
    return y, fin


CU = [0, 5, 5, 6, 14, 14]  # lengths 5, 0, 1, 8, 0


def test_varlen_matches_the_definition_written_out():
    x, dt, A, B, C, D, init = _inputs(14, 4, 3, 5, 2, len(CU) - 1, seed=1)
    y, f = oracle.recurrence_varlen(x, dt, A, B, C, D, init, CU)
    yb, fb = _brute(x, dt, A, B, C, D, init, CU)
    assert np.max(np.abs(y - yb)) <= 1e-12 * max(1.0, np.max(np.abs(yb)))
    assert np.max(np.abs(f - fb)) <= 1e-12 * max(1.0, np.max(np.abs(fb)))
    # empty sequences keep their initial state
    assert np.array_equal(f[1], init[1].double().numpy()) and np.array_equal(f[4], init[4].double().numpy())


def test_a_missing_state_reset_would_be_caught():
    # the same tokens as one sequence (no reset at the boundaries) differ from the packed result
    x, dt, A, B, C, D, init = _inputs(14, 4, 3, 5, 2, len(CU) - 1, seed=1)
    y, _ = oracle.recurrence_varlen(x, dt, A, B, C, D, init, CU)
    y1, _ = _brute(x, dt, A, B, C, D, init[:1], [0, 14])
    assert np.max(np.abs(y[5:] - y1[5:])) > 1e-3


def test_sequences_are_independent_of_their_neighbours():
    x, dt, A, B, C, D, init = _inputs(14, 2, 3, 4, 1, len(CU) - 1, seed=2)
    y, f = oracle.recurrence_varlen(x, dt, A, B, C, D, init, CU)
    # reversing the order of the sequences reverses the blocks of the result
    lens = [b - a for a, b in zip(CU, CU[1:])]
    order = list(range(len(lens)))[::-1]
    idx = torch.cat([torch.arange(CU[s], CU[s + 1]) for s in order]).long()
    cu2 = [0]
    for s in order:
        cu2.append(cu2[-1] + lens[s])
    y2, f2 = oracle.recurrence_varlen(x[idx], dt[idx], A, B[idx], C[idx], D, init[order], cu2)
    assert np.array_equal(y2, y[idx.numpy()])
    assert np.array_equal(f2, f[order])


def test_equal_lengths_match_the_batch_layout():
    b, L, H, P, N, G = 3, 7, 2, 3, 4, 1
    x, dt, A, B, C, D, init = _inputs(b * L, H, P, N, G, b, seed=3)
    y, f = oracle.recurrence_varlen(x, dt, A, B, C, D, init, [0, L, 2 * L, 3 * L])
    yb, fb = oracle.recurrence(x.reshape(b, L, H, P), dt.reshape(b, L, H), A, B.reshape(b, L, G, N),
                               C.reshape(b, L, G, N), D, init)
    assert np.array_equal(y, yb.reshape(b * L, H, P)) and np.array_equal(f, fb)


@pytest.mark.parametrize("cu", [[1, 4], [0, 3, 2], [0, 3, 5]])
def test_bad_offsets_are_rejected(cu):
    x, dt, A, B, C, D, init = _inputs(4, 1, 2, 2, 1, len(cu) - 1, seed=4)
    with pytest.raises(ValueError):
        oracle.recurrence_varlen(x, dt, A, B, C, D, None, cu)
