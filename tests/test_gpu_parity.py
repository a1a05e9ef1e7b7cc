"""GPU parity: every C-ABI call against the CPU oracle on the same seeded inputs.

Bit-exact: packed words, dequantized weights, expert ids, offsets, permutations,
gathered rows, and GEMMs whose products and partial sums are exact (integer inputs).
Within tolerance: gates (fp32 vs float64) and layer outputs (rel L2 <= 5e-3,
max-abs <= 2e-2 * max|ref|)."""
import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from weight_only_int4_route_gb300 import synth

from _helpers import GATE_RTOL, assert_close_layer, have_gpu, layer_inputs

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

DEV = "cuda:0"


@pytest.fixture(scope="module")
def M():
    from weight_only_int4_route_gb300 import build, moe
    build.build()
    moe.lib()
    return moe


def _codes(bits, shape, gen):
    lo, hi = (-8, 8) if bits == 4 else (-128, 128)
    return torch.randint(lo, hi, shape, generator=gen, dtype=torch.int8)


def _scales(shape, dtype, gen):
    return (torch.rand(shape, generator=gen) * 0.05 + 0.001).to(dtype)


# ------------------------------------------------------------------ pack / dequant


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("group", [0, 128])
def test_pack_words_match_oracle(M, bits, dtype, group):
    gen = torch.Generator().manual_seed(100 + bits + group)
    E, K, N = 3, 384, 136
    q = _codes(bits, (E, K, N), gen)
    s = _scales((E, 1 if group == 0 else K // 128, N), dtype, gen)
    packed = M.pack_weights(q.to(DEV), s.to(DEV), bits, group).cpu()
    ref_words = O.pack_int4(q.numpy()) if bits == 4 else O.pack_int8(q.numpy())
    nbytes = ref_words.nbytes
    got_words = packed[:nbytes].numpy().view(np.uint32).reshape(ref_words.shape)
    assert np.array_equal(got_words, ref_words)
    off = M.lib().moe_packed_scale_offset(E, K, N, bits)
    assert torch.equal(packed[off:off + s.numel() * 2].view(dtype).view(s.shape), s)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("group", [0, 128])
def test_dequant_bit_exact(M, bits, dtype, group):
    gen = torch.Generator().manual_seed(200 + bits + group)
    E, K, N = 2, 512, 264
    q = _codes(bits, (E, K, N), gen)
    s = _scales((E, 1 if group == 0 else K // 128, N), dtype, gen)
    packed = M.pack_weights(q.to(DEV), s.to(DEV), bits, group)
    for out_dt in (dtype, torch.float32):
        got = M.dequant(packed, E, K, N, bits, group, dtype, out_dt).cpu()
        ref = O.dequant_rounded(q, s, group, out_dt)
        assert torch.equal(got.view(torch.int16 if out_dt != torch.float32 else torch.int32),
                           ref.view(torch.int16 if out_dt != torch.float32 else torch.int32)), out_dt


@pytest.mark.parametrize("name", ["encdec_int8", "encdec_int4", "qwen", "phi"])
def test_dequant_config_shapes(M, name):
    """Algorithm 1 bit-exact on each config's FC1 and FC2 shapes (one expert)."""
    cfg = synth.CONFIGS[name]
    for K, N in ((cfg.d, cfg.F1), (cfg.F, cfg.d)):
        q = synth.codes(cfg, "q1", (1, K, N))
        s = synth.scales(cfg, "s1", 1, K, N)
        packed = M.pack_weights(q.to(DEV), s.to(DEV), cfg.bits, cfg.group)
        got = M.dequant(packed, 1, K, N, cfg.bits, cfg.group, cfg.torch_dtype, cfg.torch_dtype).cpu()
        ref = O.dequant_rounded(q, s, cfg.group, cfg.torch_dtype)
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), (name, K, N)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_i2f_every_code_every_slot(M, dtype):
    """Every INT4 code in every nibble slot and every INT8 code in every byte decodes to itself."""
    for bits, codes in ((4, range(-8, 8)), (8, range(-128, 128))):
        per = 8 if bits == 4 else 4
        vals = torch.tensor(list(codes), dtype=torch.int8)
        K = 128 * ((len(vals) * per + 127) // 128)
        q = torch.zeros((1, K, 8), dtype=torch.int8)
        # run j, element i carries code vals[(j + i) % len]: every code visits every slot
        for j in range(K // per):
            for i in range(per):
                q[0, j * per + i, :] = vals[(j + i) % len(vals)]
        s = torch.ones((1, 1, 8), dtype=dtype)
        packed = M.pack_weights(q.to(DEV), s.to(DEV), bits, 0)
        got = M.dequant(packed, 1, K, 8, bits, 0, dtype, torch.float32).cpu()
        assert torch.equal(got, q.to(torch.float32))


# ------------------------------------------------------------------ router


@pytest.mark.parametrize("name,T", [("tiny", 16), ("encdec_int4", 40), ("encdec_int4", 333), ("qwen", 32),
                                    ("qwen", 4096), ("dsv2", 512), ("phi", 17)])
def test_route_matches_oracle(M, name, T):
    cfg = synth.CONFIGS[name]
    w, x = layer_inputs(cfg, T)
    bias = None if w.bias is None else w.bias.to(DEV)
    ids, gate = M.route_topk(x.to(DEV), w.wr.to(DEV), bias, cfg.k)
    lg, rids, rgate = O.route(x, w.wr, w.bias, cfg.k)
    assert torch.equal(ids.cpu(), rids)
    rel = ((gate.cpu().double() - rgate).abs() / rgate).max().item()
    assert rel <= GATE_RTOL, rel


def test_route_renormalize_and_max_experts(M):
    cfg = synth.custom("qwen", d=256, E=256, k=8, router_dtype="bf16")
    w, x = layer_inputs(cfg, 50)
    ids, gate = M.route_topk(x.to(DEV), w.wr.to(DEV), None, cfg.k, renormalize=True)
    _, rids, rgate = O.route(x, w.wr, None, cfg.k, renormalize=True)
    assert torch.equal(ids.cpu(), rids)
    assert ((gate.cpu().double() - rgate).abs() / rgate).max().item() <= GATE_RTOL


# ------------------------------------------------------------------ permute


@pytest.mark.parametrize("T,k,E,skew", [(16, 2, 8, False), (1, 4, 60, False), (1000, 6, 64, False),
                                        (777, 1, 32, True), (300, 1, 1, False), (70, 8, 256, False)])
def test_permute_bit_exact(M, T, k, E, skew):
    gen = torch.Generator().manual_seed(T * 31 + k)
    if skew:   # most rows on expert 3, several experts empty
        ids = torch.where(torch.rand((T, k), generator=gen) < 0.8, 3,
                          torch.randint(0, E // 2, (T, k), generator=gen)).to(torch.int32)
    else:
        ids = torch.stack([torch.randperm(E, generator=gen)[:k] for _ in range(T)]).to(torch.int32)
    x = torch.randn((T, 264), generator=gen).to(torch.bfloat16)
    offsets, perm, inv, xp = M.permute(ids.to(DEV), x.to(DEV), E)
    _, roff, rperm, rinv = O.sort_by_expert(ids, E)
    assert torch.equal(offsets.cpu(), roff)
    assert torch.equal(perm.cpu(), rperm)
    assert torch.equal(inv.cpu(), rinv)
    assert torch.equal(xp.cpu(), O.permute_rows(x, rperm, k))


def test_unpermute_of_permute_is_identity(M):
    """k = 1, gate 1: combine(permute(x)) returns x bit-exactly."""
    gen = torch.Generator().manual_seed(9)
    T, E = 513, 7
    ids = torch.randint(0, E, (T, 1), generator=gen).to(torch.int32)
    x = torch.randn((T, 128), generator=gen).to(torch.float16)
    _, _, inv, xp = M.permute(ids.to(DEV), x.to(DEV), E)
    out = M.unpermute_combine(xp, inv, torch.ones((T, 1), device=DEV), None, torch.float16)
    assert torch.equal(out.cpu(), x)


@pytest.mark.parametrize("T,k,d", [(37, 3, 96), (5, 40, 260), (300, 1, 1024)])
def test_combine_matches_oracle(M, T, k, d):
    """Weighted un-permute: d not a multiple of the 128-column group, and k above 32."""
    gen = torch.Generator().manual_seed(10 + T + k + d)
    y = torch.randn((T * k, d), generator=gen, dtype=torch.float32)
    inv = torch.randperm(T * k, generator=gen).to(torch.int32)
    gate = torch.rand((T, k), generator=gen)
    sh = torch.randn((T, d), generator=gen).to(torch.bfloat16)
    out = M.unpermute_combine(y.to(DEV), inv.to(DEV), gate.to(DEV), sh.to(DEV), torch.float32).cpu()
    ref = sum(gate[:, j:j + 1].double() * y.double()[inv.view(T, k)[:, j].long()] for j in range(k)) + sh.double()
    assert (out.double() - ref).abs().max().item() <= 1e-5 * ref.abs().max().item()


# ------------------------------------------------------------------ grouped GEMM


def _rows_offsets(counts):
    off = torch.zeros(len(counts) + 1, dtype=torch.int32)
    off[1:] = torch.cumsum(torch.tensor(counts), 0)
    return off


def _oracle_gemm(a, q, s, group, offsets, act):
    out = []
    for e in range(q.shape[0]):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        w = O.dequant(q[e:e + 1], s[e:e + 1], group)[0] if s is not None else q[e].double()
        out.append(O.activation(a[lo:hi].double() @ w, act))
    return torch.cat(out)


@pytest.mark.parametrize("bits,group,dtype", [(4, 0, torch.float16), (4, 128, torch.bfloat16),
                                              (8, 0, torch.float16), (8, 128, torch.bfloat16),
                                              (4, 128, torch.float16), (16, 0, torch.bfloat16)])
@pytest.mark.parametrize("counts,N", [([0, 1, 17, 40], 192), ([300, 0, 1250, 3], 192), ([300, 0, 1250, 3], 256),
                                      ([130, 129, 128, 64, 1], 384)])
@pytest.mark.parametrize("act", ["none", "relu"])
def test_gemm_exact_integers(M, bits, group, dtype, counts, N, act):
    """Integer activations and power-of-two scales: every product and fp32 partial sum
    is exact, so the GPU result equals the oracle bit for bit (both kernels)."""
    gen = torch.Generator().manual_seed(sum(counts) + bits)
    E, K = len(counts), 512
    R = sum(counts)
    a = torch.randint(-1, 2, (R, K), generator=gen).to(dtype)
    if bits == 16:
        q = torch.randint(-8, 9, (E, K, N), generator=gen).to(dtype)
        s = None
        packed = M.pack_weights(q.to(DEV), None, 16, 0)
    else:
        q = _codes(bits, (E, K, N), gen)
        G = 1 if group == 0 else K // 128
        s = (2.0 ** torch.randint(-7, -4, (E, G, N), generator=gen).double()).to(dtype)
        packed = M.pack_weights(q.to(DEV), s.to(DEV), bits, group)
    off = _rows_offsets(counts)
    path = M.gemm_path(R, E, K, N, bits, group, act)
    if N % 128 == 0 and R / max(1, sum(c > 0 for c in counts)) >= 64:
        assert path == "tcgen05"
    got = M.grouped_gemm(a.to(DEV), packed, bits, E, K, N, group, off.to(DEV), act, torch.float32).cpu()
    assert M.device_error(DEV) == 0
    ref = _oracle_gemm(a, q, s, group, off, act)
    assert torch.equal(got.double(), ref), path


def _gemv_counts(case):
    if case == "few_rows":            # one n8 tile per row chunk, two m16 tiles per unit
        return [1, 0, 3, 2, 5, 0, 7, 8], 1024, 256
    if case == "two_tiles":           # two n8 tiles per row chunk
        return [9, 16, 12, 0, 10], 512, 192
    if case == "many_experts":        # expert table past 128 entries, rows only at high ids
        c = [0] * 200
        c[3], c[150], c[199], c[130] = 1, 2, 1, 3
        return c, 256, 64
    if case == "split_k":             # two rows, long K: the plan splits K
        return [2, 1], 4096, 128
    raise ValueError(case)


@pytest.mark.parametrize("bits,group,dtype", [(4, 128, torch.bfloat16), (4, 0, torch.float16),
                                              (8, 128, torch.float16), (8, 0, torch.bfloat16),
                                              (16, 0, torch.bfloat16)])
@pytest.mark.parametrize("case", ["few_rows", "two_tiles", "many_experts", "split_k"])
@pytest.mark.parametrize("act", ["none", "relu"])
def test_decode_gemm_exact_integers(M, bits, group, dtype, case, act):
    """Decode-sized batches (a few rows per expert) on the weight-stream kernel: integer
    activations and power-of-two scales keep every sum exact, so the result is bit-exact."""
    counts, K, N = _gemv_counts(case)
    gen = torch.Generator().manual_seed(len(counts) * 7 + K + N + bits)
    E, R = len(counts), sum(counts)
    a = torch.randint(-1, 2, (R, K), generator=gen).to(dtype)
    if bits == 16:
        q = torch.randint(-8, 9, (E, K, N), generator=gen).to(dtype)
        s = None
        packed = M.pack_weights(q.to(DEV), None, 16, 0)
    else:
        q = _codes(bits, (E, K, N), gen)
        G = 1 if group == 0 else K // 128
        s = (2.0 ** torch.randint(-7, -4, (E, G, N), generator=gen).double()).to(dtype)
        packed = M.pack_weights(q.to(DEV), s.to(DEV), bits, group)
    off = _rows_offsets(counts)
    assert M.gemm_path(R, E, K, N, bits, group, act) == "gemv"
    got = M.grouped_gemm(a.to(DEV), packed, bits, E, K, N, group, off.to(DEV), act, torch.float32).cpu()
    assert M.device_error(DEV) == 0
    assert torch.equal(got.double(), _oracle_gemm(a, q, s, group, off, act))


@pytest.mark.parametrize("name,which", [("tiny", 1), ("tiny", 2), ("encdec_int8", 1), ("encdec_int4", 2),
                                        ("qwen", 1), ("qwen", 2), ("phi", 1)])
@pytest.mark.parametrize("counts", [[3, 0, 1, 2], [12, 9, 0, 16], [40, 7, 0, 129], [300, 150, 0, 77]])
def test_gemm_config_shapes_vs_oracle(M, name, which, counts):
    """FC1 (with its activation) or FC2 on each config's real (K, N), 4 experts."""
    cfg = synth.CONFIGS[name]
    E = len(counts)
    K, N, act = (cfg.d, cfg.F1, cfg.act) if which == 1 else (cfg.F, cfg.d, "none")
    q = synth.codes(cfg, "q1" if which == 1 else "q2", (E, K, N))
    s = synth.scales(cfg, "s1" if which == 1 else "s2", E, K, N)
    R = sum(counts)
    a = synth.normal(cfg, "x", (R, K), 1.0, cfg.torch_dtype, extra=which)
    off = _rows_offsets(counts)
    packed = M.pack_weights(q.to(DEV), s.to(DEV), cfg.bits, cfg.group)
    got = M.grouped_gemm(a.to(DEV), packed, cfg.bits, E, K, N, cfg.group, off.to(DEV), act, cfg.torch_dtype)
    ref = _oracle_gemm(a, q, s, cfg.group, off, act)
    assert M.device_error(DEV) == 0
    assert_close_layer(got, ref, f"{name} fc{which} {M.gemm_path(R, E, K, N, cfg.bits, cfg.group, act)}")


def test_shared_expert_vs_oracle(M):
    cfg = synth.CONFIGS["qwen"]
    w = synth.layer_weights(cfg)
    for T in (1, 8, 17, 32, 63, 100, 700):   # gemv up to 16 rows, tcgen05 from 17
        x = synth.activations(cfg, T)
        gu = M.pack_weights(w.ws_gu.to(DEV)[None], None, 16, 0)
        dn = M.pack_weights(w.ws_d.to(DEV)[None], None, 16, 0)
        got = M.shared_expert(x.to(DEV), gu, dn, cfg.Fs, torch.float32)
        assert_close_layer(got, O.shared_expert(x, w.ws_gu, w.ws_d), f"shared T={T}")


# ------------------------------------------------------------------ whole layer


def _run_layer(M, cfg, w, x, max_T=None):
    from weight_only_int4_route_gb300.moe import Layer, PackedLayer
    layer = Layer(PackedLayer.from_weights(cfg, w, DEV), max_T or max(1, x.shape[0]))
    out = layer.forward(x.to(DEV))
    torch.cuda.synchronize()
    return layer, out


def _check_layer(M, cfg, T, subset=None):
    w, x = layer_inputs(cfg, T)
    layer, out = _run_layer(M, cfg, w, x)
    ref = O.moe_layer(x, w, cfg, token_subset=subset)
    rt = layer.routing(T)
    assert torch.equal(rt["ids"].cpu(), ref["ids"])
    assert torch.equal(rt["offsets"].cpu(), ref["offsets"])
    assert torch.equal(rt["perm"].cpu(), ref["perm"])
    assert torch.equal(rt["inv_perm"].cpu(), ref["inv_perm"])
    assert ((rt["gate"].cpu().double() - ref["gate"]).abs() / ref["gate"]).max().item() <= GATE_RTOL
    assert M.device_error(DEV) == 0
    got = out.cpu() if subset is None else out.cpu()[subset]
    return assert_close_layer(got, ref["out"], f"{cfg.name} T={T}")


@pytest.mark.parametrize("name,T", [("tiny", 16), ("tiny", 1), ("encdec_int8", 40), ("encdec_int4", 40),
                                    ("encdec_int4", 77), ("encdec_int8", 320), ("encdec_int4", 320),
                                    ("encdec_int4", 1280), ("encdec_int8", 640),
                                    ("qwen", 1), ("qwen", 8), ("qwen", 32), ("dsv2", 32), ("phi", 1), ("phi", 16),
                                    ("phi", 32)])
def test_layer_matches_oracle(M, name, T):
    _check_layer(M, synth.CONFIGS[name], T)


@pytest.mark.parametrize("name,T", [("encdec_int4", 3840), ("encdec_int8", 3840), ("encdec_int8", 1280),
                                    ("qwen", 4096), ("dsv2", 512), ("phi", 8192)])
def test_layer_full_size_sampled(M, name, T):
    """Full workload size in the same launch configuration the benchmark times: routing
    compared in full, outputs on 256 seeded token samples (the layer is per-token
    independent, so the oracle computes only those tokens)."""
    subset = torch.randperm(T, generator=torch.Generator().manual_seed(T))[:256].sort().values
    _check_layer(M, synth.CONFIGS[name], T, subset)


def test_layer_edge_cases(M):
    # single expert (E = 1, k = 1): a dense FFN
    _check_layer(M, synth.custom("tiny", E=1, k=1, index=7), 33)
    # every expert selected (k = E)
    _check_layer(M, synth.custom("tiny", E=4, k=4, index=8), 21)
    # skewed routing: a huge logit bias sends every token to one expert, the rest are empty
    cfg = synth.custom("encdec_int4", index=9)
    w, x = layer_inputs(cfg, 150)
    w.bias = torch.zeros(cfg.E)
    w.bias[5] = 100.0
    layer, out = _run_layer(M, cfg, w, x)
    ref = O.moe_layer(x, w, cfg)
    assert int(ref["counts"][5]) == 150
    assert torch.equal(layer.routing(150)["offsets"].cpu(), ref["offsets"])
    assert_close_layer(out.cpu(), ref["out"], "skewed")


def test_layer_zero_tokens(M):
    cfg = synth.CONFIGS["tiny"]
    w, _ = layer_inputs(cfg, 4)
    from weight_only_int4_route_gb300.moe import Layer, PackedLayer
    layer = Layer(PackedLayer.from_weights(cfg, w, DEV), 4)
    x = torch.empty((0, cfg.d), dtype=cfg.torch_dtype, device=DEV)
    out = layer.forward(x)
    assert out.shape == (0, cfg.d)


def test_tcgen05_gemm_repeatable(M):
    """The tensor-memory GEMM run many times on one prefill shape: no bounded wait may expire
    and every result is bit-identical (fixed reduction order, no atomics)."""
    cfg = synth.CONFIGS["encdec_int4"]
    E, K, N, T = cfg.E, cfg.F, cfg.d, 3840
    counts = [T // E] * E
    R = sum(counts)
    assert M.gemm_path(R, E, K, N, cfg.bits, cfg.group, "none") == "tcgen05"
    gen = torch.Generator().manual_seed(77)
    q = _codes(cfg.bits, (E, K, N), gen)
    s = _scales((E, 1, N), cfg.torch_dtype, gen)
    packed = M.pack_weights(q.to(DEV), s.to(DEV), cfg.bits, cfg.group)
    a = torch.randn((R, K), generator=gen).to(cfg.torch_dtype).to(DEV)
    off = _rows_offsets(counts).to(DEV)
    first = M.grouped_gemm(a, packed, cfg.bits, E, K, N, cfg.group, off, "none", torch.float32)
    for _ in range(400):
        again = M.grouped_gemm(a, packed, cfg.bits, E, K, N, cfg.group, off, "none", torch.float32)
        assert torch.equal(again, first)
    assert M.device_error(DEV) == 0


@pytest.mark.parametrize("R,N,path", [(16, 128, "gemv"), (48, 192, "mma"), (1024, 128, "tcgen05")])
def test_gelu_epilogue_accuracy(M, R, N, path):
    """out[r, n] = GELU(x_r) through each GEMM path (one weight of 1, fp32 output): the kernels'
    GELU against the float64 erf form within 1e-6 * max(1, |x|)."""
    E, K = 1, 128
    x = torch.linspace(-9.0, 9.0, R).to(torch.float16)
    a = torch.zeros((R, K), dtype=torch.float16)
    a[:, 0] = x
    q = torch.zeros((E, K, N), dtype=torch.int8)
    q[0, 0, :] = 1
    s = torch.ones((E, 1, N), dtype=torch.float16)
    packed = M.pack_weights(q.to(DEV), s.to(DEV), 4, 0)
    off = torch.tensor([0, R], dtype=torch.int32)
    assert M.gemm_path(R, E, K, N, 4, 0, "gelu") == path
    got = M.grouped_gemm(a.to(DEV), packed, 4, E, K, N, 0, off.to(DEV), "gelu", torch.float32).cpu().double()
    assert M.device_error(DEV) == 0
    ref = O.gelu(x.double())[:, None].expand(R, N)
    err = (got - ref).abs() / x.double().abs().clamp(min=1.0)[:, None]
    assert err.max().item() <= 1e-6, (path, err.max().item())



@pytest.mark.parametrize("name", ["encdec_int4", "encdec_int8"])
def test_fused_top1_combine_is_bit_identical(M, name):
    """Top-1 without a shared expert: FC2's epilogue writes the gated rows to their tokens. The
    layer output equals, bit for bit, the separate calls: route, permute, FC1, FC2 (fp32), combine."""
    cfg = synth.CONFIGS[name]
    T = 1280
    w, x = layer_inputs(cfg, T)
    layer, out = _run_layer(M, cfg, w, x)
    assert layer.launch_count(T) == 6    # router (2), permute (2), FC1, FC2: no combine launch
    packed = PackedLayer_from(cfg, w)
    xd = x.to(DEV)
    ids, gate = M.route_topk(xd, packed.wr, None, cfg.k)
    offs, perm, inv, xp = M.permute(ids, xd, cfg.E)
    h = M.grouped_gemm(xp, packed.w1, cfg.bits, cfg.E, cfg.d, cfg.F1, cfg.group, offs, cfg.act, cfg.torch_dtype)
    y = M.grouped_gemm(h, packed.w2, cfg.bits, cfg.E, cfg.F, cfg.d, cfg.group, offs, "none", torch.float32)
    sep = M.unpermute_combine(y, inv, gate, None, cfg.torch_dtype)
    assert M.device_error(DEV) == 0
    assert torch.equal(out, sep)


def PackedLayer_from(cfg, w):
    from weight_only_int4_route_gb300.moe import PackedLayer
    return PackedLayer.from_weights(cfg, w, DEV)



@pytest.mark.parametrize("name,T", [("qwen", 8), ("phi", 1), ("encdec_int4", 40), ("dsv2", 32), ("qwen", 1)])
def test_layer_graph_matches_forward(M, name, T):
    """The chain captured as one CUDA graph gives the eager forward's output bit for bit, also
    after a new input is written into the graph's input buffer, and each replay matches the
    float64 oracle (routing exactly, output within the layer tolerance)."""
    from weight_only_int4_route_gb300.moe import Layer, LayerGraph, PackedLayer
    cfg = synth.CONFIGS[name]
    w, x = layer_inputs(cfg, T)
    layer = Layer(PackedLayer.from_weights(cfg, w, DEV), T)
    g = LayerGraph(layer, T)
    for rep in range(2):
        xi = x
        if rep == 1:   # a second input, gap-filtered like the first
            xi = O.gap_filtered(synth.normal(cfg, "x", (T, cfg.d), 1.0, cfg.torch_dtype, extra=99), w.wr, w.bias,
                                cfg.k, lambda n, a: synth.redraw_rows(cfg, T + 99, n, a))
        g.x.copy_(xi.to(DEV))
        got = g.launch().clone()
        torch.cuda.synchronize()
        oracle = O.moe_layer(xi, w, cfg)
        rt = layer.routing(T)
        assert torch.equal(rt["ids"].cpu(), oracle["ids"]), rep
        assert torch.equal(rt["perm"].cpu(), oracle["perm"]), rep
        assert_close_layer(got.cpu(), oracle["out"], f"{name} T={T} graph replay {rep}")
        ref = layer.forward(xi.to(DEV))
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
    assert M.device_error(DEV) == 0
    g.close()


def _gap_filtered_all(cfg, x, weights, T):
    """x with every token's top-(k+1) logits at least the test gap apart under each router."""
    for _ in range(16):
        before = x.clone()
        for i, w in enumerate(weights):
            x = O.gap_filtered(x, w.wr, w.bias, cfg.k, lambda n, a, i=i: synth.redraw_rows(cfg, T + 7 * i, n, a))
        if torch.equal(before, x):
            return x
    raise RuntimeError("gap filter over several routers did not settle")


@pytest.mark.slow
def test_phi_stack_matches_oracle(M):
    """The benchmark's step on the Phi-shaped stack: 32 layers with distinct weights, T = 8192,
    one shared workspace, layers run back to back on one stream (each reads the same input and
    writes its own output).  Layers 0 and 31 are drawn on the CPU so the oracle can recompute
    them: routing compared in full, outputs on 256 seeded tokens each."""
    from weight_only_int4_route_gb300.moe import Layer, PackedLayer
    cfg = synth.CONFIGS["phi"]
    T, L = 8192, cfg.layers
    checked = {0: synth.layer_weights(cfg, 0), L - 1: synth.layer_weights(cfg, L - 1)}
    x = _gap_filtered_all(cfg, synth.activations(cfg, T), list(checked.values()), T)
    packed = []
    for i in range(L):
        wi = checked[i] if i in checked else synth.layer_weights(cfg, i, device=DEV)
        packed.append(PackedLayer.from_weights(cfg, wi, DEV))
        del wi
    layers = [Layer(p, T) for p in packed[:1]]
    ws = layers[0].ws
    layers += [Layer(p, T, workspace=ws) for p in packed[1:]]
    xd = x.to(DEV)
    outs = [torch.empty((T, cfg.d), dtype=cfg.torch_dtype, device=DEV) for _ in range(L)]
    for rep in range(2):   # a repeated step must give the same bits
        for li, layer in enumerate(layers):
            layer.forward(xd, outs[li])
        torch.cuda.synchronize()
        if rep == 0:
            first = [outs[i].clone() for i in checked]
    assert M.device_error(DEV) == 0
    assert all(torch.equal(outs[i], f) for i, f in zip(checked, first))
    subset = torch.randperm(T, generator=torch.Generator().manual_seed(31))[:256].sort().values
    for i, w in checked.items():
        ref = O.moe_layer(x, w, cfg, token_subset=subset)
        # the shared workspace holds the routing of the last layer run
        if i == L - 1:
            rt = layers[i].routing(T)
            assert torch.equal(rt["ids"].cpu(), ref["ids"])
            assert torch.equal(rt["offsets"].cpu(), ref["offsets"])
            assert torch.equal(rt["perm"].cpu(), ref["perm"])
        assert_close_layer(outs[i].cpu()[subset], ref["out"], f"phi stack layer {i}")


@pytest.mark.parametrize("name,T", [("qwen", 8), ("dsv2", 300)])
def test_forked_shared_expert_matches_serial(M, name, T):
    """With a shared expert, moe_layer_forward runs it on a second stream beside the routed
    chain and joins before the combine; the profiled forward (stage events) runs the same
    kernels in one stream.  Both give the same output bit for bit, over repeated calls."""
    from weight_only_int4_route_gb300.moe import STAGES, Layer, PackedLayer
    cfg = synth.CONFIGS[name]
    assert cfg.Fs > 0
    w, x = layer_inputs(cfg, T)
    layer = Layer(PackedLayer.from_weights(cfg, w, DEV), T)
    xd = x.to(DEV)
    events = [torch.cuda.Event(enable_timing=True) for _ in STAGES]
    for e in events:   # torch creates the CUDA event on its first record
        e.record()
    prev = M.set_decode_mode("chain")   # the kernel chain, also for a decode-sized T
    try:
        serial = layer.forward_profiled(xd, torch.empty((T, cfg.d), dtype=x.dtype, device=DEV), events).clone()
        for _ in range(3):
            forked = layer.forward(xd)
            torch.cuda.synchronize()
            assert torch.equal(forked, serial)
    finally:
        M.set_decode_mode(prev)
    assert M.device_error(DEV) == 0


def test_gelu_same_bits_on_every_path(M):
    """The tensor-memory GEMM evaluates GELU two at a time with paired fp32 instructions, the
    decode GEMM one at a time; the operations and their order are the same, so the outputs are
    the same bits (one weight of 1: every GEMM result is x itself)."""
    E, K, N = 1, 128, 128

    def run(x):
        R = x.shape[0]
        a = torch.zeros((R, K), dtype=torch.float16)
        a[:, 0] = x
        q = torch.zeros((E, K, N), dtype=torch.int8)
        q[0, 0, :] = 1
        s = torch.ones((E, 1, N), dtype=torch.float16)
        packed = M.pack_weights(q.to(DEV), s.to(DEV), 4, 0)
        off = torch.tensor([0, R], dtype=torch.int32)
        out = M.grouped_gemm(a.to(DEV), packed, 4, E, K, N, 0, off.to(DEV), "gelu", torch.float32).cpu()
        return out, M.gemm_path(R, E, K, N, 4, 0, "gelu")

    x = torch.linspace(-9.0, 9.0, 1024).to(torch.float16)
    tc, p_tc = run(x)
    pick = torch.arange(0, 1024, 64)
    gv, p_gv = run(x[pick])
    assert (p_tc, p_gv) == ("tcgen05", "gemv")
    assert M.device_error(DEV) == 0
    assert torch.equal(tc[pick], gv)


def test_silu_same_bits_on_every_path(M):
    """SwiGLU through the tensor-memory GEMM (SiLU two at a time, paired fp32) and through the
    decode GEMM (one at a time): gate = x, up = 1, so the output is SiLU(x) on both, bit for bit."""
    E, K, N = 1, 128, 256
    F = N // 2

    def run(x):
        R = x.shape[0]
        a = torch.zeros((R, K), dtype=torch.bfloat16)
        a[:, 0] = x
        a[:, 1] = 1.0
        q = torch.zeros((E, K, N), dtype=torch.int8)
        q[0, 0, :F] = 1     # gate channels read x
        q[0, 1, F:] = 1     # up channels read 1
        s = torch.ones((E, K // 128, N), dtype=torch.bfloat16)
        packed = M.pack_weights(q.to(DEV), s.to(DEV), 4, 128)
        off = torch.tensor([0, R], dtype=torch.int32)
        out = M.grouped_gemm(a.to(DEV), packed, 4, E, K, N, 128, off.to(DEV), "swiglu", torch.float32).cpu()
        return out, M.gemm_path(R, E, K, N, 4, 128, "swiglu")

    x = torch.linspace(-12.0, 12.0, 1024).to(torch.bfloat16)
    tc, p_tc = run(x)
    pick = torch.arange(0, 1024, 64)
    gv, p_gv = run(x[pick])
    assert (p_tc, p_gv) == ("tcgen05", "gemv")
    assert M.device_error(DEV) == 0
    assert torch.equal(tc[pick], gv)
    ref = x.double() / (1.0 + torch.exp(-x.double()))
    assert (tc.double() - ref[:, None]).abs().max().item() <= 1e-6 * max(1.0, ref.abs().max().item())


@pytest.mark.parametrize("name,T", [("qwen", 300), ("encdec_int4", 40), ("dsv2", 32)])
def test_back_to_back_layers_keep_stream_order(M, name, T):
    """Layer calls issued back to back on alternating inputs, sharing one workspace and with no
    host synchronization between them (kernels launched with programmatic stream serialization,
    the shared expert forked onto a second stream) give every call the same bits as a call run
    alone: each kernel waits for its predecessor before touching memory."""
    from weight_only_int4_route_gb300.moe import Layer, PackedLayer
    cfg = synth.CONFIGS[name]
    w, x0 = layer_inputs(cfg, T)
    x1 = synth.normal(cfg, "x", (T, cfg.d), 1.0, cfg.torch_dtype, extra=123)
    layer = Layer(PackedLayer.from_weights(cfg, w, DEV), T)
    xs = [x0.to(DEV), x1.to(DEV)]
    ref = []
    for x in xs:
        ref.append(layer.forward(x).clone())
        torch.cuda.synchronize()
    outs = [layer.forward(xs[i % 2]) for i in range(24)]
    torch.cuda.synchronize()
    assert M.device_error(DEV) == 0
    for i, o in enumerate(outs):
        assert torch.equal(o, ref[i % 2]), i
