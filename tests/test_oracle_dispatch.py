"""Pins for the oracle's dispatch (expert-contiguous packing) and combine
(weighted scatter-add), from page "M6.1 - Routed Capacity: MoE Experts,
Routers, and Token Dispatch", sections 0x05A-0x05F."""
import os

import numpy as np
import pytest

from oracle import moe_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _layout_fixture():
    routes, packed, offsets = [], None, None
    for line in open(os.path.join(GOLD, "dispatch_layout.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        if f[0] == "packed":
            packed = [int(r[1:]) for r in f[1:]]
        elif f[0] == "offsets":
            offsets = [int(v) for v in f[1:]]
        else:
            routes.append((int(f[1]), int(f[2]), int(f[3]), float(f[4])))
    T = 1 + max(r[0] for r in routes)
    K = 1 + max(r[1] for r in routes)
    ids = np.zeros((T, K), dtype=np.int32)
    gates = np.zeros((T, K))
    for t, k, e, g in routes:
        ids[t, k] = e
        gates[t, k] = g
    return ids, gates, packed, offsets


def test_dispatch_reproduces_the_pages_layout():
    ids, _, packed, offsets = _layout_fixture()
    meta = O.dispatch(ids, 3)
    assert meta["offsets"].tolist() == offsets
    K = ids.shape[1]
    # route r = t*K + k in token-major order
    got_routes = (meta["route_token"] * K + meta["route_slot"]).tolist()
    assert got_routes == packed
    assert meta["counts"].tolist() == [3, 3, 0]
    # the inverse map sends each (token, slot) to its packed row
    for row, (t, k) in enumerate(zip(meta["route_token"], meta["route_slot"])):
        assert meta["token_slot_row"][t, k] == row


def _trace_fixture():
    H, experts, Y = [], {}, []
    for line in open(os.path.join(GOLD, "combine_trace.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        if f[0] == "H":
            H.append([float(v) for v in f[1:]])
        elif f[0] == "expert":
            experts[int(f[1])] = (float(f[2]), np.array([float(f[3]), float(f[4])]))
        elif f[0] == "Y":
            Y.append([float(v) for v in f[1:]])
    fns = [(lambda a, c: (lambda x: a * x + c))(*experts[e]) for e in range(len(experts))]
    return np.array(H), fns, np.array(Y)


def test_combine_reproduces_the_pages_numeric_trace():
    ids, gates, _, _ = _layout_fixture()
    H, fns, Y = _trace_fixture()
    got = O.moe_apply(H, ids, gates, fns)
    np.testing.assert_allclose(got, Y, rtol=0, atol=1e-12)


def test_planted_combine_mistakes_break_the_trace(monkeypatch):
    """The page's failure lab: an overwrite instead of an add, or the gate of the
    other slot, keeps every shape valid but must miss the printed output."""
    ids, gates, _, _ = _layout_fixture()
    H, fns, Y = _trace_fixture()

    def overwrite_apply(h, ids_, gates_, experts):
        meta = O.dispatch(ids_, len(experts))
        xp = h[meta["route_token"]]
        g = gates_[meta["route_token"], meta["route_slot"]]
        y = np.zeros_like(h, dtype=np.float64)
        off = meta["offsets"]
        for e in range(len(experts)):
            for j in range(off[e], off[e + 1]):
                y[meta["route_token"][j]] = g[j] * experts[e](xp[j])      # planted: = instead of +=
        return y

    assert not np.allclose(overwrite_apply(H, ids, gates, fns), Y)
    swapped = gates[:, ::-1].copy()                                      # planted: other slot's gate
    assert not np.allclose(O.moe_apply(H, ids, swapped, fns), Y)
    dup = ids.copy()
    dup[0, 1] = dup[0, 0]                                                # planted: duplicated route
    assert not np.allclose(O.moe_apply(H, dup, gates, fns), Y)


@pytest.mark.parametrize("T,E,K", [(1, 8, 2), (37, 16, 3), (200, 128, 6), (64, 512, 22), (0, 8, 2)])
def test_dispatch_invariants(T, E, K):
    rng = np.random.default_rng(T * 1000 + E)
    ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]) if T else np.zeros((0, K), np.int32)
    meta = O.dispatch(ids, E)
    off, cnt = meta["offsets"], meta["counts"]
    assert cnt.sum() == T * K and off[E] == T * K and off[0] == 0
    assert np.all(np.diff(off) == cnt)
    # every token appears exactly K times (P^T P = diag(K)), once per slot
    assert np.all(np.bincount(meta["route_token"], minlength=T) == K)
    for e in range(E):
        toks = meta["route_token"][off[e]:off[e + 1]]
        assert np.all(np.diff(toks) > 0)                                # ascending, no repeats
        assert np.all(ids[toks, meta["route_slot"][off[e]:off[e + 1]]] == e)
    assert sorted(meta["token_slot_row"].reshape(-1).tolist()) == list(range(T * K))
