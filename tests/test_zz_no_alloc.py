"""The workspace-free INT4 grouped GEMM (moe_grouped_gemm_w4a16_static).

It serves callers that cannot allocate device memory themselves; its split-K scratch is a
fixed array inside the library.  Both entry points run the same plan and the same kernels
with the same reduction order, so its results must equal moe_grouped_gemm_w4a16's given a
workspace bit for bit, on two calls in a row (the shared array keeps the previous call's
contents), and match the float64 oracle within the layer tolerance.  A call needing more
scratch than the array holds must be refused before any launch.
This file is collected last so that a stop-at-first-failure run has run everything else."""
import ctypes

import pytest
import torch

from _helpers import assert_close_layer, have_gpu
from oracle import moe_oracle as O
from weight_only_int4_route_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

DEV = "cuda:0"
STATIC_BYTES = 2 << 20   # size of the library's built-in scratch array


@pytest.fixture(scope="module")
def M():
    from weight_only_int4_route_gb300 import build, moe
    build.build()
    moe.lib()
    return moe


def _oracle(a, q, s, group, off, act):
    out = []
    for e in range(q.shape[0]):
        lo, hi = int(off[e]), int(off[e + 1])
        w = O.dequant(q[e:e + 1], s[e:e + 1], group)[0]
        out.append(O.activation(a[lo:hi].double() @ w, act))
    return torch.cat(out)


def _case(cfg, K, N, act, counts, seed):
    E = len(counts)
    g = torch.Generator().manual_seed(seed)
    q = torch.randint(-7, 8, (E, K, N), generator=g, dtype=torch.int8)
    G = 1 if cfg.group == 0 else K // cfg.group
    s = ((torch.rand((E, G, N), generator=g) * 0.015 + 0.005) * (256.0 / K) ** 0.5).to(cfg.torch_dtype)
    off = torch.zeros(E + 1, dtype=torch.int32)
    off[1:] = torch.cumsum(torch.tensor(counts), 0)
    a = torch.randn((sum(counts), K), generator=g).to(cfg.torch_dtype)
    return a, q, s, off


# (config, K, N, act, rows per expert, path the plan takes)
CASES = {
    # a decode step on the Qwen-shaped FC1 / FC2: 4 routed rows on 4 experts (decode stream
    # kernel, K split into fp32 partials)
    "decode_fc1": ("qwen", 2048, 2816, "swiglu", {3: 1, 17: 1, 41: 1, 59: 1}, 60, "gemv"),
    "decode_fc2": ("qwen", 1408, 2048, "none", {3: 1, 17: 1, 41: 1, 59: 1}, 60, "gemv"),
    # a few dozen rows per expert on a channel count the tensor-memory kernel does not take: the
    # warp-MMA kernel splits K and its partials go through the array
    "mma_split_k": ("encdec_int4", 2048, 192, "none", {0: 30, 1: 20}, 2, "mma"),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_static_scratch_matches_workspace_entry(M, case):
    name, K, N, act, rows, E, path = CASES[case]
    cfg = synth.CONFIGS[name]
    counts = [rows.get(e, 0) for e in range(E)]
    R = sum(counts)
    assert M.gemm_path(R, E, K, N, 4, cfg.group, act) == path
    need = M.lib().moe_grouped_gemm_workspace_size(R, E, K, N, 4, M.ACT[act])
    assert 0 < need <= STATIC_BYTES, need
    for call in range(2):       # two calls in a row through the shared array
        a, q, s, off = _case(cfg, K, N, act, counts, seed=1000 * len(case) + call)
        packed = M.pack_weights(q.to(DEV), s.to(DEV), 4, cfg.group)
        ref = M.grouped_gemm(a.to(DEV), packed, 4, E, K, N, cfg.group, off.to(DEV), act, torch.float32)
        got = M.grouped_gemm_static(a.to(DEV), packed, E, K, N, cfg.group, off.to(DEV), act, torch.float32)
        torch.cuda.synchronize()
        assert M.device_error(DEV) == 0
        assert torch.equal(got, ref), f"{case}: static scratch call {call} differs from the workspace call"
        assert_close_layer(got.cpu(), _oracle(a, q, s, cfg.group, off, act), f"{case} call {call} vs oracle")


def test_static_scratch_refuses_oversize(M):
    # one expert with 60 rows, a long reduction and a channel count the tensor-memory kernel
    # does not take (not a multiple of 128): the warp-MMA plan splits K and its fp32 partial
    # sums (splits x 60 x 4160) exceed the 2 MiB array
    R, E, K, N = 60, 1, 8192, 4160
    need = M.lib().moe_grouped_gemm_workspace_size(R, E, K, N, 4, 0)
    assert need > STATIC_BYTES
    nul = ctypes.c_void_p(16)   # never dereferenced: the call is refused on the host
    st = M.lib().moe_grouped_gemm_w4a16_static(nul, 0, nul, E, K, N, 0, nul, R, 0, nul, 0, None)
    assert st == -2 and b"scratch" in M.lib().moe_last_error_string()
