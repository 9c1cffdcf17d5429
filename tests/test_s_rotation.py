"""The forward kernel's S lookahead (head dim 64), restated on the host.

With two query tiles of d = 64, Tensor Memory holds three S buffers, used in
turn in the order the MMA thread issues the S products, and a tile's
S(j + 1) is issued before its P(j) V.  The softmax warps of a tile do not
see that order: they work out which buffer holds their S from the work
items alone.  This file restates the MMA thread's issue order (blocks in
order, tile 0 before tile 1, S_t(j + 1) ahead of P_t(j) V, the next item's
S_t(0) behind this item's last P_t V) and checks, over random item
sequences of both masks:
  - the S products go out in the order of the (item, block, tile) units,
    so the issue count mod 3 is the buffer;
  - the softmax's incremental buffer formula gives the same buffer;
  - an S product never overwrites a buffer whose P V has not been issued
    yet (S(x) comes after P(x - 3) V);
  - a tile's S for block k + 2 is issued only after its P V for block k,
    which is what keeps a barrier kept in two sets from running two phases
    ahead of its waiter, and what lets the softmax write alpha of block
    k + 2 into the array of block k without waiting (that P V waited for
    the correction warps' read of it).
No GPU needed."""
import random

import pytest


def _items(causal, nkv, pairs):
    """n[0], n[1] (key blocks of the two query tiles) of each work item."""
    out = []
    for pair in pairs:
        qt0 = 2 * pair
        if causal:
            out.append((min(qt0 + 1, nkv), min(qt0 + 2, nkv)))
        else:
            out.append((nkv, nkv))
    return out


def _issue_order(items, rng):
    """Events ('S' | 'PV', item, block, tile) in the MMA thread's order.  The
    next item's S_t(0) may go out in tile t's slot of the last block (when
    its K and Q are already there: chosen at random here) or after it."""
    ev = []
    s0_issued = False
    for ii, n in enumerate(items):
        nmax = max(n)
        has_next = ii + 1 < len(items)
        if not s0_issued:
            ev += [("S", ii, 0, 0), ("S", ii, 0, 1)]
        s0_issued = False
        for j in range(nmax):
            ahead = j + 1 == nmax and has_next
            done = [False, False]
            for t in range(2):
                if j + 1 < n[t]:
                    ev.append(("S", ii, j + 1, t))
                if j < n[t]:
                    ev.append(("PV", ii, j, t))
                if ahead and (t == 0 or done[0]) and rng.random() < 0.5:
                    ev.append(("S", ii + 1, 0, t))
                    done[t] = True
            if ahead:
                for t in range(2):
                    if not done[t]:
                        ev.append(("S", ii + 1, 0, t))
                s0_issued = True
    return ev


def _units(items):
    return [(ii, j, t) for ii, n in enumerate(items) for j in range(max(n))
            for t in range(2) if j < n[t]]


def _softmax_buffers(items, t):
    """The softmax of tile t: buffer of each of its blocks, as the kernel
    computes it (seq3 = S products of the earlier items mod 3)."""
    out, seq3 = {}, 0
    for ii, (n0, n1) in enumerate(items):
        sb = (seq3 + t) % 3
        for j in range((n0, n1)[t]):
            out[(ii, j, t)] = sb
            sb = (sb + (2 if t == 0 else (2 if j + 1 < n0 else 1))) % 3
        seq3 = (seq3 + n0 + n1) % 3
    return out


@pytest.mark.parametrize("seed", range(4))
def test_s_rotation_invariants(seed):
    rng = random.Random(seed)
    for _ in range(400):
        causal = rng.random() < 0.5
        nkv = rng.randint(1, 9)
        pairs = [rng.randrange((nkv + 1) // 2) for _ in range(rng.randint(1, 6))]
        items = _items(causal, nkv, pairs)
        ev = _issue_order(items, rng)
        units = _units(items)
        idx = {u: i for i, u in enumerate(units)}
        s_units = [idx[e[1:]] for e in ev if e[0] == "S"]
        assert s_units == list(range(len(units))), "S products out of unit order"
        for t in range(2):
            for u, b in _softmax_buffers(items, t).items():
                assert b == idx[u] % 3, (items, u)
        pos = {(e[0],) + e[1:]: i for i, e in enumerate(ev)}
        for u, x in idx.items():
            if x >= 3:
                assert pos[("PV",) + units[x - 3]] < pos[("S",) + u], (items, u)
        for t in range(2):
            tu = [u for u in units if u[2] == t]
            for k in range(len(tu) - 2):
                assert pos[("PV",) + tu[k]] < pos[("S",) + tu[k + 2]], (items, t, k)


def test_plain_order_breaks_rule():
    """Pin: the same check catches an order that overwrites a P still
    waiting for its P V (S_t(j + 2) issued two blocks ahead)."""
    items = _items(False, 4, [0])
    units = _units(items)
    idx = {u: i for i, u in enumerate(units)}
    ev = [("S", 0, 0, 0), ("S", 0, 0, 1), ("S", 0, 1, 0), ("S", 0, 1, 1), ("S", 0, 2, 0)]
    pv_before = {e[1:] for e in ev if e[0] == "PV"}
    bad = [u for e in ev if e[0] == "S" for u in [e[1:]]
           if idx[u] >= 3 and units[idx[u] - 3] not in pv_before]
    assert bad == [(0, 1, 1), (0, 2, 0)]
