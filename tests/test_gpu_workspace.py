"""One layer workspace, sized by moe_layer_workspace_size for max_T tokens, serves a forward
call of every T <= max_T (the Python Layer relies on it), and each result matches the oracle."""
import pytest
import torch

from _helpers import assert_close_layer, have_gpu, layer_inputs
from oracle import moe_oracle as O
from weight_only_int4_route_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

DEV = "cuda:0"


@pytest.fixture(scope="module")
def M():
    from weight_only_int4_route_gb300 import build, moe
    build.build()
    moe.lib()
    yield moe


@pytest.mark.parametrize("name,max_T", [("phi", 12), ("qwen", 12), ("encdec_int4", 40), ("dsv2", 9)])
def test_every_smaller_batch_fits(M, name, max_T):
    cfg = synth.CONFIGS[name]
    w, x = layer_inputs(cfg, max_T)
    layer = M.Layer(M.PackedLayer.from_weights(cfg, w, DEV), max_T)
    assert layer.ws.numel() == layer.workspace_bytes(max_T)
    xd = x.to(DEV)
    for T in range(1, max_T + 1):
        assert layer.workspace_bytes(T) <= layer.ws.numel(), T
        out = layer.forward(xd[:T].contiguous())   # refused with MOE_ERR_WORKSPACE if it did not fit
        if T in (1, max_T // 2, max_T):
            torch.cuda.synchronize()
            assert M.device_error(DEV) == 0
            ref = O.moe_layer(x[:T], w, cfg)
            assert_close_layer(out.cpu(), ref["out"], f"{name} T={T}")
    torch.cuda.synchronize()
    assert M.device_error(DEV) == 0
