"""The decode step as one kernel launch (moe_set_decode_mode 2; automatic mode picks it for small steps).

The single launch runs router, top-k, sort, FC1 + activation, FC2, the shared expert and the
combine ("Specter" summary page, technical novelty: one launch for all expert sub-computations
of a draft step).  Checked against the float64 oracle (routing bit for bit, output within the
layer tolerance) and against the kernel chain (same routing, outputs within the tolerance; the
two sum in different orders), on every decode-sized configuration and on edge cases; repeated
and back-to-back calls give the same bits; the launch count is one."""
import pytest
import torch

from _helpers import GATE_RTOL, assert_close_layer, have_gpu, layer_inputs
from oracle import moe_oracle as O
from weight_only_int4_route_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

DEV = "cuda:0"


@pytest.fixture(scope="module")
def M():
    from weight_only_int4_route_gb300 import build, moe
    build.build()
    moe.lib()
    prev = moe.set_decode_mode("launch")   # the one-launch kernel for every decode-sized step here
    yield moe
    moe.set_decode_mode(prev)


def _layer(M, cfg, w, T):
    from weight_only_int4_route_gb300.moe import Layer, PackedLayer
    return Layer(PackedLayer.from_weights(cfg, w, DEV), T)


def _check(M, cfg, T, renormalize=False):
    from weight_only_int4_route_gb300.moe import Layer, PackedLayer
    w, x = layer_inputs(cfg, T)
    layer = Layer(PackedLayer.from_weights(cfg, w, DEV), T, renormalize=renormalize)
    assert layer.launch_count(T) == 1
    xd = x.to(DEV)
    out = layer.forward(xd).clone()
    torch.cuda.synchronize()
    assert M.device_error(DEV) == 0
    ref = O.moe_layer(x, w, cfg, renormalize=renormalize)
    rt = layer.routing(T)
    assert torch.equal(rt["ids"].cpu(), ref["ids"])
    assert torch.equal(rt["offsets"].cpu(), ref["offsets"])
    assert torch.equal(rt["perm"].cpu(), ref["perm"])
    assert torch.equal(rt["inv_perm"].cpu(), ref["inv_perm"])
    assert ((rt["gate"].cpu().double() - ref["gate"]).abs() / ref["gate"]).max().item() <= GATE_RTOL
    assert_close_layer(out.cpu(), ref["out"], f"{cfg.name} T={T} one launch")
    # the same call again: the same bits (units are taken dynamically, the arithmetic is fixed)
    again = layer.forward(xd)
    torch.cuda.synchronize()
    assert torch.equal(again, out)
    # the kernel chain on the same inputs: the same routing, outputs within the tolerance
    prev = M.set_decode_mode("chain")
    try:
        chain = layer.forward(xd).clone()
        torch.cuda.synchronize()
    finally:
        M.set_decode_mode(prev)
    assert_close_layer(chain.cpu(), ref["out"], f"{cfg.name} T={T} chain")
    assert M.device_error(DEV) == 0
    return out


@pytest.mark.parametrize("name,T", [("tiny", 16), ("tiny", 1), ("qwen", 1), ("qwen", 8), ("qwen", 32),
                                    ("dsv2", 32), ("phi", 1), ("phi", 16), ("phi", 32)])
def test_decode_layer_matches_oracle(M, name, T):
    _check(M, synth.CONFIGS[name], T)


@pytest.mark.parametrize("case", ["gelu_fp16_int4", "one_expert", "k_equals_E", "renormalize", "odd_T", "max_rows"])
def test_decode_layer_edge_cases(M, case):
    if case == "gelu_fp16_int4":     # encoder-decoder shape, exact-erf GELU, per-channel scales, 16-bit router
        _check(M, synth.custom("encdec_int4", index=21), 24)
    elif case == "one_expert":       # E = 1, k = 1: a dense FFN
        _check(M, synth.custom("tiny", E=1, k=1, index=22), 9)
    elif case == "k_equals_E":       # every expert selected
        _check(M, synth.custom("tiny", E=4, k=4, index=23), 7)
    elif case == "renormalize":
        _check(M, synth.custom("qwen", index=24), 5, renormalize=True)
    elif case == "odd_T":            # rows not filling the n-tiles, shared expert with 3 tokens
        _check(M, synth.custom("qwen", index=25), 3)
    elif case == "max_rows":         # T * k = 256 rows over 64 experts, row chunks of several experts split
        _check(M, synth.custom("dsv2", k=8, index=26), 32)


def test_decode_layer_skewed_routing(M):
    """A large logit bias sends every token to one expert: that expert's rows span several row
    chunks, every other expert but the second choice is empty."""
    cfg = synth.custom("phi", index=27)
    T = 29
    w, x = layer_inputs(cfg, T)
    w.bias = torch.zeros(cfg.E)
    w.bias[3] = 50.0
    layer = _layer(M, cfg, w, T)
    out = layer.forward(x.to(DEV))
    torch.cuda.synchronize()
    ref = O.moe_layer(x, w, cfg)
    assert int(ref["counts"][3]) == T
    assert torch.equal(layer.routing(T)["offsets"].cpu(), ref["offsets"])
    assert_close_layer(out.cpu(), ref["out"], "skewed one launch")
    assert M.device_error(DEV) == 0


def test_decode_layers_back_to_back_share_workspace(M):
    """Several layers with distinct weights run back to back on one workspace with no host
    synchronization (each launch leaves the control words zero for the next), then a smaller T on
    the same workspace: every output equals the oracle's."""
    from weight_only_int4_route_gb300.moe import Layer, PackedLayer
    cfg = synth.CONFIGS["qwen"]
    T = 8
    ws = None
    layers, weights = [], []
    for i in range(3):
        w = synth.layer_weights(cfg, i)
        weights.append(w)
        layer = Layer(PackedLayer.from_weights(cfg, w, DEV), T, workspace=ws)
        ws = layer.ws
        layers.append(layer)
    x = synth.activations(cfg, T)
    for w in weights:
        x = O.gap_filtered(x, w.wr, w.bias, cfg.k, lambda n, a: synth.redraw_rows(cfg, T, n, a))
    xd = x.to(DEV)
    outs = [torch.empty((T, cfg.d), dtype=cfg.torch_dtype, device=DEV) for _ in layers]
    for _ in range(3):
        for layer, o in zip(layers, outs):
            layer.forward(xd, o)
    torch.cuda.synchronize()
    assert M.device_error(DEV) == 0
    for w, o in zip(weights, outs):
        assert_close_layer(o.cpu(), O.moe_layer(x, w, cfg)["out"], "stacked")
    small = layers[0].forward(xd[:2])
    torch.cuda.synchronize()
    assert_close_layer(small.cpu(), O.moe_layer(x[:2], weights[0], cfg)["out"], "T=2 on the T=8 workspace")
