"""CPU oracle for Specter's expert lookahead buffer (ELB) counting and top-M selection.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference arm may import this module.  The CUDA library never calls it and
shares no code, table or constant with it.

  [Specter]  "Specter: Fast MoE Inference via Quantization-Enabled Multi-Step Speculative
             Offloading" (paper summary page), method step (2): over the draft steps
             i = 1..t, the analyzer keeps per layer j and expert e the count
             ELB(t)_cnt[j, e] = sum_i I[e in ELB_route[i, j]]; step (3): at a chunk boundary
             the planner snapshots the buffer and takes each layer's top-M experts.

Readings of open points:
  * ELB_route[i, j] is the set of expert ids the draft routes to at step i in layer j (the
    k ids of that step's token); an expert counts once per step;
  * ids outside [0, E) are not counted;
  * top-M orders by count, descending; equal counts go to the lower expert id; when fewer than
    M experts exist the list is E long.
Pins: tests/test_elb_pins.py (a hand-worked example, invariants, brute force).
"""
from __future__ import annotations

import numpy as np


def accumulate(ids: np.ndarray, E: int, counts: np.ndarray | None = None) -> np.ndarray:
    """ids (L, S, k) routed ids of S draft steps per layer -> counts (L, E) int64 (added to
    `counts` when given)."""
    ids = np.asarray(ids)
    L, S, _ = ids.shape
    out = np.zeros((L, E), dtype=np.int64) if counts is None else np.array(counts, dtype=np.int64)
    for j in range(L):
        for i in range(S):
            for e in set(int(v) for v in ids[j, i]):
                if 0 <= e < E:
                    out[j, e] += 1
    return out


def top_m(counts: np.ndarray, M: int):
    """counts (L, E) -> (experts (L, min(M, E)), their counts), by descending count, then id."""
    counts = np.asarray(counts)
    L, E = counts.shape
    m = min(M, E)
    experts = np.zeros((L, m), dtype=np.int64)
    vals = np.zeros((L, m), dtype=np.int64)
    for j in range(L):
        order = sorted(range(E), key=lambda e: (-int(counts[j, e]), e))[:m]
        experts[j] = order
        vals[j] = [counts[j, e] for e in order]
    return experts, vals
