"""BF16 bit-field codec on the GPU against the CPU oracle: bit-exact."""
import numpy as np
import pytest
import torch

from oracle import bitfield_oracle as B

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def M():
    from weight_only_int4_route_gb300 import moe
    moe.lib()
    return moe


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_every_pattern(M):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    exp, sm = M.bf16_split(t)
    e_ref, s_ref = B.split(bits)
    assert np.array_equal(exp.cpu().numpy(), e_ref) and np.array_equal(sm.cpu().numpy(), s_ref)
    back = M.bf16_recombine(exp, sm)
    assert np.array_equal(_bits(back), B.recombine(e_ref, s_ref))


@pytest.mark.parametrize("n", [0, 1, 15, 16, 17, 1000, 4096 + 7, 3_000_001])
def test_random_weights_and_tails(M, n):
    g = torch.Generator().manual_seed(n)
    w = (torch.randn(n, generator=g) * 0.02).to(torch.bfloat16)
    e_ref, s_ref = B.split(_bits(w))
    exp, sm = M.bf16_split(w.to(DEV))
    assert np.array_equal(exp.cpu().numpy(), e_ref) and np.array_equal(sm.cpu().numpy(), s_ref)
    back = M.bf16_recombine(exp, sm)
    assert torch.equal(back.cpu().view(torch.int16), w.view(torch.int16))
