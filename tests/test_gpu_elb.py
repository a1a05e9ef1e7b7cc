"""ELB counting and top-M on the GPU against the CPU oracle: bit-exact integers."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import elb_oracle as B

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def M():
    from weight_only_int4_route_gb300 import moe
    moe.lib()
    return moe


def test_hand_example(M):
    g = json.load(open(os.path.join(HERE, "golden", "elb_example.json")))
    ids = torch.tensor(g["ids"], dtype=torch.int32, device=DEV)
    counts = torch.zeros((2, g["E"]), dtype=torch.int32, device=DEV)
    M.elb_accumulate(ids, g["E"], counts)
    assert counts.cpu().tolist() == g["counts"]
    ex, vals = M.elb_topm(counts, g["M"])
    assert ex.cpu().tolist() == g["top_experts"] and vals.cpu().tolist() == g["top_counts"]


@pytest.mark.parametrize("L,S,k,E,M_", [(24, 32, 4, 60, 8), (26, 16, 6, 64, 12), (32, 16, 2, 16, 4),
                                         (3, 700, 8, 256, 300), (1, 1, 1, 1, 1)])
def test_random_routes_match_oracle(M, L, S, k, E, M_):
    rng = np.random.default_rng(L * 1000 + S + E)
    ids = np.stack([np.stack([rng.choice(E, min(k, E), replace=False) for _ in range(S)]) for _ in range(L)])
    if k > 1 and S > 3:
        ids[:, 3, 1] = ids[:, 3, 0]          # a duplicate within a step
        ids[:, 2, 0] = E + 5                 # an id outside [0, E)
    start = rng.integers(0, 5, size=(L, E))
    counts = torch.from_numpy(start.astype(np.int32)).to(DEV)
    M.elb_accumulate(torch.from_numpy(ids.astype(np.int32)).to(DEV), E, counts)
    ref = B.accumulate(ids, E, start)
    assert np.array_equal(counts.cpu().numpy(), ref)
    ex, vals = M.elb_topm(counts, M_)
    rex, rvals = B.top_m(ref, M_)
    assert np.array_equal(ex.cpu().numpy(), rex) and np.array_equal(vals.cpu().numpy(), rvals)
    # the fused launch gives the same counts and selection
    c2 = torch.from_numpy(start.astype(np.int32)).to(DEV)
    ex2 = torch.empty_like(ex)
    v2 = torch.empty_like(vals)
    M.elb_step(torch.from_numpy(ids.astype(np.int32)).to(DEV), E, c2, M_, ex2, v2)
    assert np.array_equal(c2.cpu().numpy(), ref)
    assert np.array_equal(ex2.cpu().numpy(), rex) and np.array_equal(v2.cpu().numpy(), rvals)
