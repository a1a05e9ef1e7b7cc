"""Pins for the CPU oracle: each check ties an oracle function to something other
than itself (hand-computed values, exhaustive identities, brute force, textbook
routines, closed forms).  A second group plants plausible mistakes in the
oracle and shows that a pin catches each one."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from weight_only_int4_route_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- P1 dequant


def test_alg1_per_channel_hand_tensor():
    g = golden("alg1_dequant.json")["per_channel"]
    q = torch.tensor(g["W"], dtype=torch.int8)
    s = torch.tensor(g["S"], dtype=torch.float16)
    got = O.dequant(q, s, 0)
    assert torch.equal(got, torch.tensor(g["W_dq"], dtype=torch.float64))


def test_alg1_group128_hand_entries():
    g = golden("alg1_dequant.json")["group128"]
    m = torch.arange(g["M"])
    q = ((m % 15) - 7).to(torch.int8)[None, :, None].expand(1, g["M"], g["N"]).contiguous()
    s = torch.tensor(g["S"], dtype=torch.float16)
    got = O.dequant(q, s, 128)
    for ent in g["entries"]:
        assert int(q[0, ent["m"], ent["n"]]) == ent["W"]
        assert float(got[0, ent["m"], ent["n"]]) == ent["W_dq"], ent


def test_dequant_rounded_is_single_rounding():
    """RN(q*s) to fp16/bf16 is the representable value nearest to the exact
    product, computed with Python fractions (no float arithmetic in the check)."""
    from fractions import Fraction
    gen = torch.Generator().manual_seed(5)
    q = torch.randint(-127, 128, (1, 64, 8), dtype=torch.int8, generator=gen)
    for dt in (torch.float16, torch.bfloat16):
        s = (torch.rand((1, 1, 8), generator=gen) * 0.02 + 1e-3).to(dt)
        got = O.dequant_rounded(q, s, 0, dt)
        for m in range(0, 64, 7):
            for n in range(8):
                exact = Fraction(int(q[0, m, n])) * Fraction(float(s[0, 0, n]))
                v = got[0, m, n]
                bits = int(v.view(torch.int16).item())
                for nb_bits in (bits + 1, bits - 1):
                    nb = torch.tensor([nb_bits], dtype=torch.int16).view(dt)[0]
                    if torch.isfinite(nb.float()):
                        assert abs(Fraction(float(v)) - exact) <= abs(Fraction(float(nb)) - exact), (m, n, dt)


# ---------------------------------------------------------------- P2 encoding / I2F


def test_i2f_constants_from_page():
    g = golden("i2f_words.json")
    assert np.array([int(g["fp16_1024_bits"], 16)], np.uint16).view(np.float16)[0] == 1024
    assert np.array([int(g["fp16_1152_bits"], 16)], np.uint16).view(np.float16)[0] == 1152
    assert (np.array([int(g["bf16_128_bits"], 16) << 16], np.uint32).view(np.float32)[0]) == 128


def test_int4_word_example_by_hand():
    g = golden("i2f_words.json")["int4_example"]
    el = np.array(g["elements_e0_to_e7"], dtype=np.int8).reshape(1, 8, 1)
    w = O.pack_int4(el)
    assert w.shape == (1, 1, 1) and int(w[0, 0, 0]) == int(g["word"], 16)
    assert np.array_equal(O.unpack_int4(w, 8), el)
    assert O.i2f_int4_word(int(g["word"], 16), "f16") == [float(v) for v in g["elements_e0_to_e7"]]


def test_int8_word_example_by_hand():
    g = golden("i2f_words.json")["int8_example"]
    el = np.array(g["elements_e0_to_e3"], dtype=np.int8).reshape(1, 4, 1)
    w = O.pack_int8(el)
    assert int(w[0, 0, 0]) == int(g["word"], 16)
    assert O.i2f_int8_word(int(g["word"], 16), "f16") == [float(v) for v in g["elements_e0_to_e3"]]


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_i2f_int4_exhaustive_every_slot(fmt):
    """Every code -8..7 in every element position decodes to itself."""
    for pos in range(8):
        for q in range(-8, 8):
            el = np.zeros((1, 8, 1), dtype=np.int8)
            el[0, pos, 0] = q
            word = int(O.pack_int4(el)[0, 0, 0])
            vals = O.i2f_int4_word(word, fmt)
            want = [0.0] * 8
            want[pos] = float(q)
            assert vals == want, (fmt, pos, q)
            if fmt == "f16":
                assert O.i2f_int4_word_upper(word) == want


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_i2f_int8_exhaustive_every_slot(fmt):
    for pos in range(4):
        for q in range(-128, 128):
            el = np.zeros((1, 4, 1), dtype=np.int8)
            el[0, pos, 0] = q
            word = int(O.pack_int8(el)[0, 0, 0])
            want = [0.0] * 4
            want[pos] = float(q)
            assert O.i2f_int8_word(word, fmt) == want


def test_pack_roundtrip_random():
    gen = np.random.default_rng(3)
    q4 = gen.integers(-8, 8, size=(3, 64, 24)).astype(np.int8)
    assert np.array_equal(O.unpack_int4(O.pack_int4(q4), 64), q4)
    q8 = gen.integers(-128, 128, size=(3, 64, 24)).astype(np.int8)
    assert np.array_equal(O.unpack_int8(O.pack_int8(q8), 64), q8)


def test_pack_int4_layout_positions():
    """Element (e, k, n) lands in word (e, n, k // 8) at nibble slot sigma^-1(k % 8)."""
    el = np.zeros((2, 16, 3), dtype=np.int8) - 8          # u = 0 everywhere
    el[1, 13, 2] = 7                                     # u = 15 at k = 13 -> word 1, element 5 -> slot 6
    w = O.pack_int4(el)
    nz = np.argwhere(w != 0)
    assert nz.tolist() == [[1, 2, 1]]
    assert int(w[1, 2, 1]) == 0xF << (4 * 6)


# ---------------------------------------------------------------- P3 router


def test_topk_brute_force_tiny():
    gen = torch.Generator().manual_seed(11)
    for E, k in [(4, 1), (6, 2), (8, 2), (8, 3), (7, 4)]:
        lg = torch.randn((50, E), generator=gen, dtype=torch.float64)
        ids = O.topk_ids(lg, k)
        for t in range(50):
            assert ids[t].tolist() == O.brute_force_topk(lg[t].tolist(), k)


def test_topk_ties_lower_id_first():
    lg = torch.tensor([[0.5, 1.0, 1.0, 0.2, 1.0]], dtype=torch.float64)
    assert O.topk_ids(lg, 3).tolist() == [[1, 2, 4]]


def test_softmax_closed_form_and_invariants():
    g = golden("closed_forms.json")["softmax2"]
    lg = torch.tensor([[g["a"], g["b"]]], dtype=torch.float64)
    p = O.softmax(lg)
    assert abs(float(p[0, 0]) - g["p_a"]) < 1e-15
    gen = torch.Generator().manual_seed(2)
    lg = torch.randn((20, 9), generator=gen, dtype=torch.float64) * 3
    p = O.softmax(lg)
    assert torch.allclose(p.sum(1), torch.ones(20, dtype=torch.float64), atol=1e-14)
    # ratio invariant p_i / p_j = exp(l_i - l_j)
    assert torch.allclose(p[:, 0] / p[:, 1], torch.exp(lg[:, 0] - lg[:, 1]), rtol=1e-13)


def test_gate_no_renorm_keeps_switch_prob_below_one():
    gen = torch.Generator().manual_seed(4)
    lg = torch.randn((10, 32), generator=gen, dtype=torch.float64)
    ids = O.topk_ids(lg, 1)
    g = O.gate_weights(lg, ids)
    assert bool((g < 1).all()) and bool((g > 0).all())
    g2 = O.gate_weights(lg, O.topk_ids(lg, 3), renormalize=True)
    assert torch.allclose(g2.sum(1), torch.ones(10, dtype=torch.float64))


def test_router_logits_small_by_hand():
    x = torch.tensor([[1.0, -2.0]], dtype=torch.float16)
    wr = torch.tensor([[0.5, 1.0, -1.0], [0.25, 0.0, 2.0]], dtype=torch.float32)
    b = torch.tensor([0.0, -1.0, 10.0])
    assert O.router_logits(x, wr, b).tolist() == [[0.0, 0.0, 5.0]]


# ---------------------------------------------------------------- P4 sort / permute


def test_sort_matches_textbook_stable_sort():
    gen = torch.Generator().manual_seed(7)
    for T, k, E in [(1, 1, 4), (16, 2, 8), (33, 4, 60), (20, 6, 64)]:
        ids = torch.stack([torch.randperm(E, generator=gen)[:k] for _ in range(T)]).to(torch.int32)
        counts, offsets, perm, inv_perm = O.sort_by_expert(ids, E)
        flat = ids.reshape(-1).tolist()
        want = sorted(range(T * k), key=lambda f: flat[f])         # Python's sort is stable
        assert perm.tolist() == want
        assert int(offsets[-1]) == T * k and int(offsets[0]) == 0
        assert counts.tolist() == [flat.count(e) for e in range(E)]
        for p in range(T * k):
            assert int(inv_perm[int(perm[p])]) == p
        for e in range(E):
            seg = perm[offsets[e]:offsets[e + 1]].tolist()
            assert all(flat[f] == e for f in seg) and seg == sorted(seg)


def test_unpermute_of_permute_is_identity_k1():
    gen = torch.Generator().manual_seed(8)
    T, E, d = 37, 5, 6
    x = torch.randn((T, d), generator=gen).to(torch.float16)
    ids = torch.randint(0, E, (T, 1), generator=gen).to(torch.int32)
    _, _, perm, inv_perm = O.sort_by_expert(ids, E)
    xp = O.permute_rows(x, perm, 1)
    assert torch.equal(xp[inv_perm.long()], x)


# ---------------------------------------------------------------- activations


def test_activation_closed_forms():
    g = golden("closed_forms.json")
    for a, v in g["gelu"]:
        assert abs(float(O.gelu(torch.tensor(a, dtype=torch.float64))) - v) < 1e-15
    for a, v in g["silu"]:
        assert abs(float(O.silu(torch.tensor(a, dtype=torch.float64))) - v) < 1e-15
    h = torch.linspace(-6, 6, 101, dtype=torch.float64)
    assert torch.allclose(O.gelu(h) - O.gelu(-h), h, atol=1e-14)       # erf is odd
    assert torch.allclose(O.silu(h) - O.silu(-h), h, atol=1e-14)
    hh = torch.cat([h[:, None], (h + 1)[:, None]], 1)                  # swiglu: gate first, then up
    assert torch.allclose(O.activation(hh, "swiglu")[:, 0], O.silu(h) * (h + 1))


# ---------------------------------------------------------------- P5 layer reductions


def _tiny_weights(cfg, gen, same_experts=False):
    E, d, F, F1 = cfg.E, cfg.d, cfg.F, cfg.F1
    q1 = torch.randint(-7, 8, (E, d, F1), generator=gen, dtype=torch.int8)
    q2 = torch.randint(-7, 8, (E, F, d), generator=gen, dtype=torch.int8)
    G1 = 1 if cfg.group == 0 else d // cfg.group
    G2 = 1 if cfg.group == 0 else F // cfg.group
    s1 = (torch.rand((E, G1, F1), generator=gen) * 0.05 + 0.01).to(cfg.torch_dtype)
    s2 = (torch.rand((E, G2, d), generator=gen) * 0.05 + 0.01).to(cfg.torch_dtype)
    if same_experts:
        q1, q2, s1, s2 = (t[:1].expand_as(t).contiguous() for t in (q1, q2, s1, s2))
    wr = (torch.randn((d, E), generator=gen) / math.sqrt(d)).to(cfg.router_torch_dtype)
    return synth.LayerWeights(wr, None, q1, s1, q2, s2, None, None)


def test_dense_ffn_hand_example():
    g = golden("dense_ffn_2x2.json")
    cfg = synth.custom("tiny", d=2, F=2, E=1, k=1, act="relu")
    w = synth.LayerWeights(torch.zeros((2, 1), dtype=torch.float32), None,
                           torch.tensor([g["W1"]], dtype=torch.int8), torch.tensor([[g["S1"]]], dtype=torch.float16),
                           torch.tensor([g["W2"]], dtype=torch.int8), torch.tensor([[g["S2"]]], dtype=torch.float16),
                           None, None)
    x = torch.tensor([g["x"]], dtype=torch.float16)
    r = O.moe_layer(x, w, cfg)
    assert r["out"][0].tolist() == g["out"]
    assert O.dequant(w.q1, w.s1, 0)[0].tolist() == g["W1_dq"]


def test_single_expert_equals_python_loop_ffn():
    """E = 1, k = 1: the layer is one dense FFN (gate = softmax of one logit = 1),
    checked against a pure-Python triple loop on the codes and scales."""
    gen = torch.Generator().manual_seed(21)
    for act in ("relu", "gelu", "swiglu"):
        cfg = synth.custom("tiny", d=8, F=6, E=1, k=1, act=act)
        w = _tiny_weights(cfg, gen)
        x = torch.randn((3, 8), generator=gen).to(torch.float16)
        got = O.moe_layer(x, w, cfg)["out"]
        for t in range(3):
            xs = [float(v) for v in x[t]]
            h = []
            for n in range(cfg.F1):
                h.append(sum(xs[m] * int(w.q1[0, m, n]) * float(w.s1[0, 0, n]) for m in range(8)))
            if act == "relu":
                a = [max(v, 0.0) for v in h]
            elif act == "gelu":
                a = [0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in h]
            else:
                a = [h[i] / (1 + math.exp(-h[i])) * h[6 + i] for i in range(6)]
            for n in range(8):
                ref = sum(a[m] * int(w.q2[0, m, n]) * float(w.s2[0, 0, n]) for m in range(6))
                assert abs(float(got[t, n]) - ref) <= 1e-12 * max(1.0, abs(ref))


def test_identical_experts_scale_by_gate_sum():
    gen = torch.Generator().manual_seed(22)
    cfg = synth.custom("tiny", d=16, F=8, E=6, k=3, act="gelu")
    w = _tiny_weights(cfg, gen, same_experts=True)
    x = torch.randn((9, 16), generator=gen).to(torch.float16)
    r = O.moe_layer(x, w, cfg)
    one = synth.custom("tiny", d=16, F=8, E=1, k=1, act="gelu")
    w1 = synth.LayerWeights(w.wr[:, :1], None, w.q1[:1], w.s1[:1], w.q2[:1], w.s2[:1], None, None)
    ffn = O.moe_layer(x, w1, one)["out"]
    assert torch.allclose(r["out"], r["gate"].sum(1, keepdim=True) * ffn, rtol=1e-12, atol=1e-14)


def test_grouped_equals_per_token_gemv():
    """[Specter] step 5: regrouping tokens by expert is mathematically equivalent."""
    gen = torch.Generator().manual_seed(23)
    for name, kw in [("tiny", dict(d=32, F=16, E=5, k=2)),
                     ("qwen", dict(d=256, F=128, E=6, k=3, Fs=128)),
                     ("encdec_int8", dict(d=32, F=64, E=4, k=1))]:
        cfg = synth.custom(name, **kw)
        w = _tiny_weights(cfg, gen)
        if cfg.Fs:
            w.ws_gu = (torch.randn((cfg.d, 2 * cfg.Fs), generator=gen) / 16).to(cfg.torch_dtype)
            w.ws_d = (torch.randn((cfg.Fs, cfg.d), generator=gen) / 16).to(cfg.torch_dtype)
        x = torch.randn((11, cfg.d), generator=gen).to(cfg.torch_dtype)
        a = O.moe_layer(x, w, cfg)["out"]
        b = O.moe_layer_per_token(x, w, cfg)
        assert torch.allclose(a, b, rtol=1e-12, atol=1e-12)


def test_token_subset_matches_full():
    gen = torch.Generator().manual_seed(24)
    cfg = synth.custom("tiny", d=32, F=16, E=5, k=2)
    w = _tiny_weights(cfg, gen)
    x = torch.randn((20, 32), generator=gen).to(torch.float16)
    full = O.moe_layer(x, w, cfg)["out"]
    sub = torch.tensor([3, 0, 17, 9])
    part = O.moe_layer(x, w, cfg, token_subset=sub)["out"]
    assert torch.equal(part, full[sub])


def test_gap_filter_removes_near_ties():
    cfg = synth.CONFIGS["tiny"]
    w = synth.layer_weights(cfg)
    x = synth.activations(cfg, 64)
    xf = O.gap_filtered(x, w.wr, w.bias, cfg.k, lambda n, a: synth.redraw_rows(cfg, 64, n, a), gap=0.05)
    assert bool(O.topk_gap_ok(O.router_logits(xf, w.wr, w.bias), cfg.k, 0.05).all())


# ---------------------------------------------------------------- comparison metrics


def test_rel_l2_hand_values():
    """rel_l2(got, ref) = ||got - ref||_2 / ||ref||_2, by hand: got = (3, 4), ref = (0, 2) gives
    ||(3, 2)|| / 2 = sqrt(13) / 2; got = ref gives 0; got = 0 gives 1; got = 2 ref gives 1."""
    g, r = torch.tensor([3.0, 4.0]), torch.tensor([0.0, 2.0])
    assert O.rel_l2(g, r) == pytest.approx(math.sqrt(13.0) / 2.0, rel=1e-15)
    assert O.rel_l2(r, g) == pytest.approx(math.sqrt(13.0) / 5.0, rel=1e-15)   # not symmetric
    x = torch.tensor([[1.5, -2.0], [0.25, 7.0]], dtype=torch.float64)
    assert O.rel_l2(x, x) == 0.0
    assert O.rel_l2(torch.zeros_like(x), x) == pytest.approx(1.0, rel=1e-15)
    assert O.rel_l2(2 * x, x) == pytest.approx(1.0, rel=1e-15)
    # a 2-D input is one vector: the Frobenius norm over every element
    assert O.rel_l2(x + torch.tensor([[3.0, 0.0], [0.0, 4.0]]), x) == pytest.approx(
        5.0 / math.sqrt(1.5 ** 2 + 2.0 ** 2 + 0.25 ** 2 + 7.0 ** 2), rel=1e-15)


def test_max_abs_rel_hand_values():
    """max_abs_rel(got, ref) = max|got - ref| / max|ref|, by hand: got = (3, 4), ref = (0, 2) gives
    max(3, 2) / 2 = 1.5; a sign flip of the largest entry of ref = (1, -8) gives 16 / 8 = 2."""
    g, r = torch.tensor([3.0, 4.0]), torch.tensor([0.0, 2.0])
    assert O.max_abs_rel(g, r) == 1.5
    assert O.max_abs_rel(r, g) == 0.75
    assert O.max_abs_rel(torch.tensor([1.0, 8.0]), torch.tensor([1.0, -8.0])) == 2.0
    assert O.max_abs_rel(r, r) == 0.0


# ---------------------------------------------------------------- planted mistakes


def test_planted_wrong_interleave_is_caught(monkeypatch):
    monkeypatch.setattr(O, "SIGMA", (0, 1, 2, 3, 4, 5, 6, 7))
    with pytest.raises(AssertionError):
        test_int4_word_example_by_hand()


def test_planted_wrong_group_row_is_caught(monkeypatch):
    monkeypatch.setattr(O, "scale_row", lambda m, group: torch.zeros_like(m))
    with pytest.raises(AssertionError):
        test_alg1_group128_hand_entries()


def test_planted_ascending_topk_is_caught(monkeypatch):
    monkeypatch.setattr(O, "topk_ids", lambda lg, k: torch.sort(lg, dim=1, stable=True).indices[:, :k].to(torch.int32))
    with pytest.raises(AssertionError):
        test_topk_brute_force_tiny()


def test_planted_unstable_sort_is_caught(monkeypatch):
    def bad(ids, E):
        c, o, p, ip = orig(ids, E)
        p2 = p.clone()
        for e in range(E):
            p2[o[e]:o[e + 1]] = p[o[e]:o[e + 1]].flip(0)
        return c, o, p2, ip
    orig = O.sort_by_expert
    monkeypatch.setattr(O, "sort_by_expert", bad)
    with pytest.raises(AssertionError):
        test_sort_matches_textbook_stable_sort()


def test_planted_transposed_operand_is_caught(monkeypatch):
    orig = O.expert_ffn
    monkeypatch.setattr(O, "expert_ffn", lambda xe, w1, w2, act: orig(xe, w1, w2.flip(1), act))
    with pytest.raises(AssertionError):
        test_single_expert_equals_python_loop_ffn()


def test_planted_missing_gate_is_caught(monkeypatch):
    monkeypatch.setattr(O, "gate_weights", lambda lg, ids, renormalize=False: torch.ones(ids.shape, dtype=torch.float64))
    with pytest.raises(AssertionError):
        test_gate_no_renorm_keeps_switch_prob_below_one()


def test_planted_metric_denominator_swap_is_caught(monkeypatch):
    """Dividing by the result under test instead of the reference would let a too-large output pass."""
    monkeypatch.setattr(O, "rel_l2", lambda g, r: float(torch.linalg.vector_norm(g.double() - r.double())
                                                       / torch.linalg.vector_norm(g.double())))
    monkeypatch.setattr(O, "max_abs_rel", lambda g, r: float((g.double() - r.double()).abs().max()
                                                            / g.double().abs().max()))
    with pytest.raises(AssertionError):
        test_rel_l2_hand_values()
    with pytest.raises(AssertionError):
        test_max_abs_rel_hand_values()


def test_planted_vacuous_metric_is_caught(monkeypatch):
    """A metric that compares the reference with itself (always 0) fails the hand values."""
    monkeypatch.setattr(O, "rel_l2", lambda g, r: float(torch.linalg.vector_norm(r.double() - r.double())
                                                       / torch.linalg.vector_norm(r.double())))
    monkeypatch.setattr(O, "max_abs_rel", lambda g, r: float((r.double() - r.double()).abs().max()
                                                            / r.double().abs().max()))
    with pytest.raises(AssertionError):
        test_rel_l2_hand_values()
    with pytest.raises(AssertionError):
        test_max_abs_rel_hand_values()
