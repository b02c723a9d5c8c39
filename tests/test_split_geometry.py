"""The K-split geometry of the weight-streaming kernels (SplitGeom in
csrc/kernels.h), restated here and checked for the properties the kernels and
the SwiGLU/combine kernels rely on: every k-block of every unit falls to exactly
one CTA, in order; a unit's pieces get slots 0..n_u-1 in K order; n_u never
exceeds the 16 partial-sum slots the workspace holds; and every CTA's share
differs from the mean by less than one k-block.  CPU only."""
import random

import pytest

MAX_SLOTS = 16


def sk_start(c, W, G):
    return c * W // G


def sk_cta_of(x, W, G):
    return -(-((x + 1) * G) // W) - 1


def sk_grid(W, kb, grid):
    m = (kb + MAX_SLOTS - 2) // (MAX_SLOTS - 1)
    return max(1, min(grid, W // m))


def segments(U, kb, grid):
    """(cta, unit, kb0, kb1, slot) as the kernel's walker produces them."""
    W = U * kb
    G = sk_grid(W, kb, grid)
    out = []
    for c in range(G):
        cur, end = sk_start(c, W, G), sk_start(c + 1, W, G)
        while cur < end:
            u, kb0 = divmod(cur, kb)
            kb1 = min(kb, kb0 + (end - cur))
            out.append((c, u, kb0, kb1, c - sk_cta_of(u * kb, W, G)))
            cur += kb1 - kb0
    return out, W, G


CASES = [(224, 64), (64, 224), (896, 64), (256, 224), (1, 4), (2, 4), (3, 224), (7, 6), (112, 64), (32, 224)]


@pytest.mark.parametrize("U,kb", CASES)
def test_every_kblock_once_and_slots_in_k_order(U, kb):
    segs, W, G = segments(U, kb, 148)
    seen = {}
    for c, u, kb0, kb1, slot in segs:
        assert 0 <= kb0 < kb1 <= kb and 0 <= slot < MAX_SLOTS
        for k in range(kb0, kb1):
            assert (u, k) not in seen
            seen[(u, k)] = slot
    assert len(seen) == U * kb
    for u in range(U):
        n_u = sk_cta_of((u + 1) * kb - 1, W, G) - sk_cta_of(u * kb, W, G) + 1
        slots = [seen[(u, k)] for k in range(kb)]
        assert slots == sorted(slots) and set(slots) == set(range(n_u))   # 0..n_u-1, in K order


@pytest.mark.parametrize("U,kb", CASES)
def test_shares_are_balanced(U, kb):
    segs, W, G = segments(U, kb, 148)
    share = {}
    for c, u, kb0, kb1, slot in segs:
        share[c] = share.get(c, 0) + kb1 - kb0
    assert max(share.values()) - min(share.values()) <= 1
    assert G == 148 or W // G >= (kb + MAX_SLOTS - 2) // (MAX_SLOTS - 1)


def test_slot_bound_over_random_geometries():
    rng = random.Random(0)
    for _ in range(2000):
        U, kb, grid = rng.randint(1, 4000), rng.choice([1, 2, 4, 6, 14, 32, 56, 64, 112, 224, 448]), 148
        W = U * kb
        G = sk_grid(W, kb, grid)
        for u in rng.sample(range(U), min(U, 20)):
            n_u = sk_cta_of((u + 1) * kb - 1, W, G) - sk_cta_of(u * kb, W, G) + 1
            assert 1 <= n_u <= MAX_SLOTS
        for x in rng.sample(range(W), min(W, 20)):
            c = sk_cta_of(x, W, G)
            assert sk_start(c, W, G) <= x < sk_start(c + 1, W, G)
