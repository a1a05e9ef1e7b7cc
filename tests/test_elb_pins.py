"""Pins of the ELB oracle: a hand-worked example, invariants and brute force.  CPU only."""
import itertools
import json
import os

import numpy as np

from oracle import elb_oracle as B

HERE = os.path.dirname(os.path.abspath(__file__))


def test_hand_example():
    g = json.load(open(os.path.join(HERE, "golden", "elb_example.json")))
    c = B.accumulate(np.array(g["ids"]), g["E"])
    assert c.tolist() == g["counts"]
    ex, vals = B.top_m(c, g["M"])
    assert ex.tolist() == g["top_experts"] and vals.tolist() == g["top_counts"]


def test_count_invariants():
    rng = np.random.default_rng(3)
    L, S, k, E = 5, 32, 4, 60
    ids = np.stack([np.stack([rng.choice(E, k, replace=False) for _ in range(S)]) for _ in range(L)])
    c = B.accumulate(ids, E)
    assert (c.sum(axis=1) == S * k).all()          # distinct valid ids: k per step
    assert c.max() <= S and c.min() >= 0
    # accumulating in two halves equals accumulating at once
    assert np.array_equal(B.accumulate(ids[:, S // 2:], E, B.accumulate(ids[:, :S // 2], E)), c)


def test_top_m_brute_force():
    rng = np.random.default_rng(4)
    for _ in range(50):
        E = int(rng.integers(1, 8))
        c = rng.integers(0, 3, size=(1, E))
        M = int(rng.integers(1, 10))
        ex, vals = B.top_m(c, M)
        # brute force: the first min(M,E) of all orderings that are sorted by (-count, id)
        best = min(itertools.permutations(range(E)), key=lambda p: [(-c[0, e], e) for e in p])
        assert ex[0].tolist() == list(best[:min(M, E)])
        assert vals[0].tolist() == [int(c[0, e]) for e in best[:min(M, E)]]


def test_planted_mistake_is_caught():
    """Counting duplicates within a step changes the hand example."""
    g = json.load(open(os.path.join(HERE, "golden", "elb_example.json")))
    ids = np.array(g["ids"])
    bad = np.zeros((2, g["E"]), dtype=np.int64)
    for j in range(2):
        for row in ids[j]:
            for e in row:
                if 0 <= e < g["E"]:
                    bad[j, e] += 1
    assert bad.tolist() != g["counts"]
