"""The workspace-free INT4 grouped GEMM (moe_grouped_gemm_w4a16_static).

It serves callers that cannot allocate device memory themselves; its split-K scratch is a
fixed array inside the library.  Its results must match moe_grouped_gemm_w4a16 given a
workspace, on two calls in a row (the shared array keeps the previous call's contents), and
a call needing more scratch than the array holds must be refused before any launch.
This file is collected last so that a stop-at-first-failure run has run everything else."""
import ctypes

import pytest
import torch

from _helpers import assert_close_layer, have_gpu
from weight_only_int4_route_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

DEV = "cuda:0"


@pytest.fixture(scope="module")
def M():
    from weight_only_int4_route_gb300 import build, moe
    build.build()
    moe.lib()
    return moe


def _case(cfg, which, counts, seed):
    E = len(counts)
    K, N, act = (cfg.d, cfg.F1, cfg.act) if which == 1 else (cfg.F, cfg.d, "none")
    q = synth.codes(cfg, "q1" if which == 1 else "q2", (E, K, N))
    s = synth.scales(cfg, "s1" if which == 1 else "s2", E, K, N)
    off = torch.zeros(E + 1, dtype=torch.int32)
    off[1:] = torch.cumsum(torch.tensor(counts), 0)
    g = torch.Generator().manual_seed(seed)
    a = torch.randn((sum(counts), K), generator=g).to(cfg.torch_dtype)
    return a, q, s, off, K, N, act


@pytest.mark.parametrize("which", [1, 2])
def test_static_scratch_matches_workspace_entry(M, which):
    cfg = synth.CONFIGS["qwen"]
    counts = [0] * 60
    for e in (3, 17, 41, 59):   # a decode step: 4 routed rows on 4 experts
        counts[e] = 1
    for call in range(2):       # two calls in a row through the shared array
        a, q, s, off, K, N, act = _case(cfg, which, counts, seed=100 * which + call)
        R, E = a.shape[0], len(counts)
        assert M.lib().moe_grouped_gemm_workspace_size(R, E, K, N, 4, M.ACT[act]) > 0, "case must use scratch"
        packed = M.pack_weights(q.to(DEV), s.to(DEV), 4, cfg.group)
        ref = M.grouped_gemm(a.to(DEV), packed, 4, E, K, N, cfg.group, off.to(DEV), act, torch.float32)
        got = M.grouped_gemm_static(a.to(DEV), packed, E, K, N, cfg.group, off.to(DEV), act, torch.float32)
        torch.cuda.synchronize()
        assert M.device_error(DEV) == 0
        assert_close_layer(got.cpu(), ref.cpu().double(), f"static scratch call {call}")


def test_static_scratch_refuses_oversize(M):
    # one expert with 60 rows, a long reduction and a channel count the tensor-memory kernel
    # does not take (not a multiple of 128): the warp-MMA plan splits K and its fp32 partial
    # sums (splits x 60 x 4160) exceed the 2 MiB array
    R, E, K, N = 60, 1, 8192, 4160
    need = M.lib().moe_grouped_gemm_workspace_size(R, E, K, N, 4, 0)
    assert need > (2 << 20)
    nul = ctypes.c_void_p(16)   # never dereferenced: the call is refused on the host
    st = M.lib().moe_grouped_gemm_w4a16_static(nul, 0, nul, E, K, N, 0, nul, R, 0, nul, 0, None)
    assert st == -2 and b"scratch" in M.lib().moe_last_error_string()
