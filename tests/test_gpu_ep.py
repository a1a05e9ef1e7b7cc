"""Expert-parallel layer on the GPU kernels, ranks run in one process (the exchanges are list
transpositions; one GPU per call): every rank's output against the oracle layer over all tokens,
and against the single-GPU layer call on the same tokens."""
import dataclasses

import pytest
import torch

from oracle import moe_oracle as O
from weight_only_int4_route_gb300 import synth

from _helpers import assert_close_layer, have_gpu, layer_inputs

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

DEV = "cuda:0"


@pytest.fixture(scope="module")
def M():
    from weight_only_int4_route_gb300 import build, moe
    build.build()
    moe.lib()
    return moe


def _cuts(T, world):
    base, extra = divmod(T, world)
    c = [0]
    for r in range(world):
        c.append(c[-1] + base + (1 if r < extra else 0))
    return c


CASES = [("tiny", 16, 2), ("tiny", 16, 3), ("encdec_int4", 320, 2), ("encdec_int8", 40, 4), ("qwen", 64, 2),
         ("dsv2", 32, 3), ("phi", 32, 2)]


@pytest.mark.parametrize("name,T,world", CASES)
def test_expert_parallel_matches_oracle_and_single_gpu(M, name, T, world):
    from weight_only_int4_route_gb300 import ep
    cfg = synth.CONFIGS[name]
    w, x = layer_inputs(cfg, T)
    ref = O.moe_layer(x, w, cfg)
    xd = x.to(DEV)
    shards = [ep.cuda_shard(cfg, w, r, world, DEV) for r in range(world)]
    c = _cuts(T, world)
    outs = ep.ep_forward_local(shards, [xd[c[r]:c[r + 1]] for r in range(world)], ep.CudaOps())
    torch.cuda.synchronize()
    assert M.device_error() == 0
    got = torch.cat(outs, 0)
    assert got.dtype == cfg.torch_dtype and got.shape == (T, cfg.d)
    assert_close_layer(got, ref["out"], f"{name} T={T} world={world}")
    # the same tokens through the single-GPU layer call
    layer = M.Layer(M.PackedLayer.from_weights(cfg, w, DEV), T)
    single = layer.forward(xd)
    torch.cuda.synchronize()
    d = (got.float() - single.float()).abs().max().item()
    assert d <= 2e-2 * single.float().abs().max().item(), d


def test_expert_parallel_skewed_routing(M):
    """Every token's experts live on rank 0: rank 1 receives nothing and gets all its rows back."""
    from weight_only_int4_route_gb300 import ep
    cfg = synth.CONFIGS["tiny"]
    w, x = layer_inputs(cfg, 16)
    bias = torch.zeros(cfg.E)
    bias[0], bias[1] = 60.0, 50.0
    w = dataclasses.replace(w, bias=bias)
    ref = O.moe_layer(x, w, cfg)
    assert set(ref["ids"].flatten().tolist()) == {0, 1}
    xd = x.to(DEV)
    shards = [ep.cuda_shard(cfg, w, r, 2, DEV) for r in range(2)]
    outs = ep.ep_forward_local(shards, [xd[:7], xd[7:]], ep.CudaOps())
    torch.cuda.synchronize()
    assert M.device_error() == 0
    assert_close_layer(torch.cat(outs, 0), ref["out"], "skewed")


def test_expert_parallel_more_ranks_than_experts(M):
    """E = 8 over 10 ranks: two ranks own no expert and only route and combine."""
    from weight_only_int4_route_gb300 import ep
    cfg = synth.CONFIGS["tiny"]
    w, x = layer_inputs(cfg, 20)
    ref = O.moe_layer(x, w, cfg)
    xd = x.to(DEV)
    world = 10
    shards = [ep.cuda_shard(cfg, w, r, world, DEV) for r in range(world)]
    assert sum(1 for s in shards if s.E_local == 0) == 2
    c = _cuts(20, world)
    outs = ep.ep_forward_local(shards, [xd[c[r]:c[r + 1]] for r in range(world)], ep.CudaOps())
    torch.cuda.synchronize()
    assert_close_layer(torch.cat(outs, 0), ref["out"], "E < world")
