"""The quantized tcgen05 GEMM as CTA pairs (clusters of two CTAs, M = 256) against the same GEMM
on single CTAs (bit for bit), against the oracle, and exact on integer inputs."""
import pytest
import torch

from oracle import moe_oracle as O
from weight_only_int4_route_gb300 import synth

from _helpers import assert_close_layer, have_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

DEV = "cuda:0"


@pytest.fixture(scope="module")
def M():
    from weight_only_int4_route_gb300 import build, moe
    build.build()
    moe.lib()
    yield moe
    moe.set_gemm_pairs(False)   # the default


def _offsets(counts):
    off = torch.zeros(len(counts) + 1, dtype=torch.int32)
    off[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int64), 0).to(torch.int32)
    return off


def _both(M, a, packed, bits, E, K, N, group, off, act, odt):
    M.set_gemm_pairs(False)
    single = M.grouped_gemm(a, packed, bits, E, K, N, group, off, act, odt)
    M.set_gemm_pairs(True)
    pair = M.grouped_gemm(a, packed, bits, E, K, N, group, off, act, odt)
    M.set_gemm_pairs(False)
    torch.cuda.synchronize()
    assert M.device_error(DEV) == 0
    return single, pair


@pytest.mark.parametrize("name,which", [("encdec_int4", 1), ("encdec_int4", 2), ("encdec_int8", 1), ("qwen", 1),
                                        ("qwen", 2), ("phi", 1), ("dsv2", 2)])
@pytest.mark.parametrize("counts", [[120, 117, 0, 131], [1, 17, 40, 0], [160, 161, 320, 9], [700, 0, 0, 33]])
def test_pairs_match_single_and_oracle(M, name, which, counts):
    cfg = synth.CONFIGS[name]
    E = len(counts)
    K, N, act = (cfg.d, cfg.F1, cfg.act) if which == 1 else (cfg.F, cfg.d, "none")
    q = synth.codes(cfg, "q1" if which == 1 else "q2", (E, K, N))
    s = synth.scales(cfg, "s1" if which == 1 else "s2", E, K, N)
    R = sum(counts)
    a = synth.normal(cfg, "x", (R, K), 1.0, cfg.torch_dtype, extra=which + 10 * E)
    off = _offsets(counts)
    packed = M.pack_weights(q.to(DEV), s.to(DEV), cfg.bits, cfg.group)
    if M.gemm_path(R, E, K, N, cfg.bits, cfg.group, act) != "tcgen05":
        pytest.skip("not a tcgen05 shape")
    odt = cfg.torch_dtype if which == 1 else torch.float32
    single, pair = _both(M, a.to(DEV), packed, cfg.bits, E, K, N, cfg.group, off.to(DEV), act, odt)
    assert torch.equal(single, pair), "pairs and single CTAs differ"
    assert_close_layer(pair, _oracle(a, q, s, cfg.group, off, act), f"{name} fc{which}")


def _oracle(a, q, s, group, off, act):
    """Per expert: act(a[rows] . dq(W_e)) in float64."""
    out = []
    for e in range(q.shape[0]):
        lo, hi = int(off[e]), int(off[e + 1])
        w = O.dequant(q[e:e + 1], s[e:e + 1], group)[0]
        out.append(O.activation(a[lo:hi].double() @ w, act))
    return torch.cat(out)


@pytest.mark.parametrize("bits,group,dtype", [(4, 0, torch.float16), (4, 128, torch.bfloat16),
                                              (8, 0, torch.float16), (8, 128, torch.bfloat16)])
@pytest.mark.parametrize("counts,N", [([300, 0, 1250, 3], 256), ([130, 129, 128, 64, 17], 512),
                                      ([33, 0, 47], 256)])
@pytest.mark.parametrize("act", ["none", "relu", "swiglu"])
def test_pairs_exact_integers(M, bits, group, dtype, counts, N, act):
    """Integer activations, power-of-two scales: every sum is exact, so the pairs' result equals
    the oracle bit for bit."""
    gen = torch.Generator().manual_seed(sum(counts) + bits + N)
    E, K = len(counts), 512
    R = sum(counts)
    a = torch.randint(-1, 2, (R, K), generator=gen).to(dtype)
    lo, hi = (-8, 8) if bits == 4 else (-128, 128)
    q = torch.randint(lo, hi, (E, K, N), generator=gen, dtype=torch.int8)
    G = 1 if group == 0 else K // 128
    s = (2.0 ** torch.randint(-7, -4, (E, G, N), generator=gen).double()).to(dtype)
    packed = M.pack_weights(q.to(DEV), s.to(DEV), bits, group)
    off = _offsets(counts)
    assert M.gemm_path(R, E, K, N, bits, group, act) == "tcgen05"
    odt = torch.float32
    single, pair = _both(M, a.to(DEV), packed, bits, E, K, N, group, off.to(DEV), act, odt)
    assert torch.equal(single, pair)
    if act != "swiglu":   # SiLU is not exact; the other activations keep integer sums exact
        assert torch.equal(pair.cpu().double(), _oracle(a, q, s, group, off, act))


def test_pairs_repeat_bit_identical(M):
    cfg = synth.CONFIGS["encdec_int4"]
    counts = [120] * 32
    E, K, N = 32, cfg.d, cfg.F1
    q = synth.codes(cfg, "q1", (E, K, N))
    s = synth.scales(cfg, "s1", E, K, N)
    a = synth.normal(cfg, "x", (sum(counts), K), 1.0, cfg.torch_dtype, extra=99).to(DEV)
    packed = M.pack_weights(q.to(DEV), s.to(DEV), 4, 0)
    off = _offsets(counts).to(DEV)
    M.set_gemm_pairs(True)
    first = M.grouped_gemm(a, packed, 4, E, K, N, 0, off, "gelu", torch.float16)
    for _ in range(200):
        assert torch.equal(M.grouped_gemm(a, packed, 4, E, K, N, 0, off, "gelu", torch.float16), first)
    M.set_gemm_pairs(False)
    assert M.device_error(DEV) == 0


def test_layer_with_pairs_matches_single(M):
    """The whole layer (routing, both GEMMs, combine) gives the same bits with and without pairs."""
    from _helpers import layer_inputs
    for name, T in (("qwen", 512), ("encdec_int4", 1280), ("phi", 256)):
        cfg = synth.CONFIGS[name]
        w, x = layer_inputs(cfg, T)
        layer = M.Layer(M.PackedLayer.from_weights(cfg, w, DEV), T)
        xd = x.to(DEV)
        M.set_gemm_pairs(False)
        single = layer.forward(xd).clone()
        M.set_gemm_pairs(True)
        pair = layer.forward(xd)
        M.set_gemm_pairs(False)
        torch.cuda.synchronize()
        assert M.device_error(DEV) == 0
        assert torch.equal(single, pair), name
