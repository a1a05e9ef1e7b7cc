"""CPU oracle for the weight-only quantized MoE expert layer.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference arm may import this module.  The CUDA library never
calls it, and it shares no code, table or constant with the CUDA sources.

Everything here is plain PyTorch CPU arithmetic in float64 (numpy for bit
patterns), written as the definitions the pages give, in their order:

  [FT]       "Who Says Elephants Can't Run: Bringing Large Scale MoE Models
             into Cloud Scale Production" (paper review page).
  [Specter]  "Specter: Fast MoE Inference via Quantization-Enabled Multi-Step
             Speculative Offloading" (paper summary page).

Pins (tests/test_oracle_pins.py) tie each function to something other than
itself: hand-computed Algorithm 1 tensors, exhaustive integer-to-float
identities over every code, brute-force top-k, textbook stable sorting,
closed forms of the activations and the E=1 dense-FFN reduction.

Readings of open points:
  * Algorithm 1's W (E, M, N): M is the reduction (input) dim, N the output
    channel; per-channel scales are (E, 1, N).  Group-128 scales are
    (E, K/128, N) and scale rows g(m) = m // 128.  Scales carry the
    activation dtype (fp16 or bf16).
  * Codes are stored offset-binary: u = q + 8 (INT4), u = q + 128 (INT8);
    1152 = 1024 + 128 in [FT] fixes the INT8 bias, INT4 uses 8 by analogy.
  * The INT4 word interleave [e0,e2,e4,e6,e1,e3,e5,e7] is read as: e0..e7
    are 8 consecutive reduction-dim elements of one output channel, and
    nibble slot p (bits 4p..4p+3) of the 32-bit word holds e_{sigma(p)},
    sigma = (0, 2, 4, 6, 1, 3, 5, 7).
  * Router: logits = x . Wr (+ bias) ; top-k by logit, descending, ties to
    the lower expert id ; gate = softmax over all E evaluated at the chosen
    ids, no renormalisation unless asked.
  * Shared expert: ungated (gate 1) SwiGLU FFN in 16-bit weights.
  * GELU is the exact erf form; SiLU(x) = x / (1 + exp(-x)); SwiGLU takes the
    first F FC1 columns as the gate and the next F as the up projection.
"""
from __future__ import annotations

import itertools
from typing import Callable, Optional

import numpy as np
import torch

F64 = torch.float64

# --------------------------------------------------------------------------
# Dequantisation -- [FT] §3 core formulas, expert quantization, Algorithm 1
# --------------------------------------------------------------------------


def scale_row(m: torch.Tensor, group: int) -> torch.Tensor:
    """Row of the scale tensor used by reduction index m: 0 per channel, m // group otherwise."""
    return torch.zeros_like(m) if group == 0 else m // group


def dequant(q: torch.Tensor, s: torch.Tensor, group: int) -> torch.Tensor:
    """W_dq[e, m, n] = IntToFloat(W[e, m, n]) * S[e, g(m), n]  (Algorithm 1, exact in float64)."""
    E, K, N = q.shape
    rows = scale_row(torch.arange(K), group)
    return q.to(F64) * s.to(F64)[:, rows, :]


def dequant_rounded(q: torch.Tensor, s: torch.Tensor, group: int, out_dtype: torch.dtype) -> torch.Tensor:
    """Algorithm 1 rounded once to out_dtype: RN_even(q * s).

    q * s has at most 8 + 11 significant bits, so it is exact in float32 and the
    float64 -> float32 step torch takes before narrowing is exact; the only
    rounding is the final one."""
    return dequant(q, s, group).to(out_dtype)


# --------------------------------------------------------------------------
# Storage encoding -- [FT] §3, optimized I2F, 8-bit and 4-bit dequantization
# --------------------------------------------------------------------------

INT4_BIAS = 8
INT8_BIAS = 128
# nibble slot p of a word holds element SIGMA[p] of the 8-element run
SIGMA = (0, 2, 4, 6, 1, 3, 5, 7)


def slot_of_element(i: int) -> int:
    return SIGMA.index(i)


def pack_int4(q: np.ndarray) -> np.ndarray:
    """(E, K, N) int8 codes in [-8, 7] -> (E, N, K/8) uint32 words, interleaved nibbles."""
    q = np.asarray(q)
    E, K, N = q.shape
    assert K % 8 == 0 and q.min() >= -8 and q.max() <= 7
    u = (q.astype(np.int64) + INT4_BIAS).astype(np.uint64)
    runs = u.transpose(0, 2, 1).reshape(E, N, K // 8, 8)      # runs[e, n, j, i] = u[e, 8j+i, n]
    word = np.zeros((E, N, K // 8), dtype=np.uint64)
    for i in range(8):
        word |= runs[..., i] << np.uint64(4 * slot_of_element(i))
    return word.astype(np.uint32)


def unpack_int4(words: np.ndarray, K: int) -> np.ndarray:
    """Inverse of pack_int4: (E, N, K/8) uint32 -> (E, K, N) int8."""
    w = np.asarray(words).astype(np.uint64)
    E, N, J = w.shape
    assert J * 8 == K
    out = np.zeros((E, N, J, 8), dtype=np.int64)
    for i in range(8):
        out[..., i] = ((w >> np.uint64(4 * slot_of_element(i))) & np.uint64(0xF)).astype(np.int64) - INT4_BIAS
    return out.reshape(E, N, K).transpose(0, 2, 1).astype(np.int8)


def pack_int8(q: np.ndarray) -> np.ndarray:
    """(E, K, N) int8 codes -> (E, N, K/4) uint32 words; byte b holds element 4j+b as q + 128."""
    q = np.asarray(q)
    E, K, N = q.shape
    assert K % 4 == 0
    u = (q.astype(np.int64) + INT8_BIAS).astype(np.uint64)
    runs = u.transpose(0, 2, 1).reshape(E, N, K // 4, 4)
    word = np.zeros((E, N, K // 4), dtype=np.uint64)
    for b in range(4):
        word |= runs[..., b] << np.uint64(8 * b)
    return word.astype(np.uint32)


def unpack_int8(words: np.ndarray, K: int) -> np.ndarray:
    w = np.asarray(words).astype(np.uint64)
    E, N, J = w.shape
    out = np.zeros((E, N, J, 4), dtype=np.int64)
    for b in range(4):
        out[..., b] = ((w >> np.uint64(8 * b)) & np.uint64(0xFF)).astype(np.int64) - INT8_BIAS
    return out.reshape(E, N, K).transpose(0, 2, 1).astype(np.int8)


def _f16(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16)


def _bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (bf16 is the top half of float32)."""
    return (np.asarray(bits, dtype=np.uint32) << np.uint32(16)).view(np.float32)


def i2f_int4_word(word: int, fmt: str = "f16") -> list:
    """Magic-number decode of one INT4 word into its 8 values e0..e7, as on the page.

    Pair p (p = 0..3) sits in nibble slots p and p + 4, i.e. bits 4p and 16 + 4p,
    which hold e_{2p} and e_{2p+1}.  Masking those bits and OR-ing them into the
    mantissa of 1024.0 (fp16, 0x6400) or 128.0 (bf16, 0x4300) gives 1024 + u /
    128 + u exactly; subtracting 1024 + 8 / 128 + 8 leaves u - 8 = q."""
    out = [None] * 8
    for p in range(4):
        lanes = (word >> (4 * p)) & 0x000F000F
        if fmt == "f16":
            h = lanes | 0x64006400
            lo, hi = _f16(np.array([h & 0xFFFF, h >> 16]))
            vals = (lo - np.float16(1024 + INT4_BIAS), hi - np.float16(1024 + INT4_BIAS))
        else:
            h = lanes | 0x43004300
            lo, hi = _bf16(np.array([h & 0xFFFF, h >> 16]))
            vals = (lo - np.float32(128 + INT4_BIAS), hi - np.float32(128 + INT4_BIAS))
        out[2 * p], out[2 * p + 1] = float(vals[0]), float(vals[1])
    return out


def i2f_int4_word_upper(word: int) -> list:
    """fp16 variant that skips one shift: the odd nibble slots stay in place.

    (w & 0x00F000F0) | 0x6400_6400 is 1024 + 16u exactly; times 1/16 minus 72
    gives u - 8 (both steps exact: a power-of-two scale and a small integer)."""
    out = [None] * 8
    for p in range(4):
        if p % 2 == 0:
            lanes = (word >> (4 * p)) & 0x000F000F
            h = lanes | 0x64006400
            v = _f16(np.array([h & 0xFFFF, h >> 16])) - np.float16(1024 + INT4_BIAS)
        else:
            lanes = (word >> (4 * (p - 1))) & 0x00F000F0
            h = lanes | 0x64006400
            v = _f16(np.array([h & 0xFFFF, h >> 16])) * np.float16(1.0 / 16) - np.float16(64 + INT4_BIAS)
        out[2 * p], out[2 * p + 1] = float(v[0]), float(v[1])
    return out


def i2f_int8_word(word: int, fmt: str = "f16") -> list:
    """[FT] 8-bit path: byte u -> fp16 (1024 + u) - 1152 = u - 128.

    bf16 has 7 mantissa bits, so a byte does not fit the mantissa of 128.0; the
    bf16 reading uses the float32 magic 2^23 instead: (2^23 + u) - (2^23 + 128)."""
    out = []
    for b in range(4):
        u = (word >> (8 * b)) & 0xFF
        if fmt == "f16":
            out.append(float(_f16(np.array([0x6400 | u]))[0] - np.float16(1152)))
        else:
            v = np.array([0x4B000000 | u], dtype=np.uint32).view(np.float32)[0]
            out.append(float(v - np.float32(8388608 + 128)))
    return out


# --------------------------------------------------------------------------
# Router -- [Specter] background on MoE (router scores, top-k); [FT] model
# table (top-1 Switch gating); [FT] §3 workflow (gating output tuple)
# --------------------------------------------------------------------------


def router_logits(x: torch.Tensor, wr: torch.Tensor, bias: Optional[torch.Tensor] = None) -> torch.Tensor:
    """logits[t, e] = sum_m x[t, m] * Wr[m, e] (+ b[e]), float64."""
    lg = x.to(F64) @ wr.to(F64)
    if bias is not None:
        lg = lg + bias.to(F64)[None, :]
    return lg


def topk_ids(logits: torch.Tensor, k: int) -> torch.Tensor:
    """The k largest logits per row, descending; equal logits keep the lower expert id first."""
    order = torch.sort(-logits, dim=1, stable=True).indices
    return order[:, :k].to(torch.int32)


def softmax(logits: torch.Tensor) -> torch.Tensor:
    z = logits - logits.max(dim=1, keepdim=True).values
    ez = torch.exp(z)
    return ez / ez.sum(dim=1, keepdim=True)


def gate_weights(logits: torch.Tensor, ids: torch.Tensor, renormalize: bool = False) -> torch.Tensor:
    """expert_scale: softmax over all E experts taken at the chosen ids."""
    g = softmax(logits).gather(1, ids.long())
    if renormalize:
        g = g / g.sum(dim=1, keepdim=True)
    return g


def route(x, wr, bias, k, renormalize=False):
    lg = router_logits(x, wr, bias)
    ids = topk_ids(lg, k)
    return lg, ids, gate_weights(lg, ids, renormalize)


def topk_gap_ok(logits: torch.Tensor, k: int, gap: float = 1e-3) -> torch.Tensor:
    """Rows whose k+1 largest logits are pairwise at least `gap` apart (no near-ties)."""
    m = min(k + 1, logits.shape[1])
    top = torch.sort(logits, dim=1, descending=True).values[:, :m]
    if m < 2:
        return torch.ones(logits.shape[0], dtype=torch.bool)
    return (top[:, :-1] - top[:, 1:]).min(dim=1).values >= gap


def gap_filtered(x: torch.Tensor, wr, bias, k: int, redraw: Callable[[int, int], torch.Tensor],
                 gap: float = 1e-3, max_attempts: int = 64) -> torch.Tensor:
    """Replace token rows whose top-(k+1) logits have a near-tie until none is left.

    redraw(n_rows, attempt) returns n fresh rows (from the seeded generator)."""
    x = x.clone()
    for attempt in range(max_attempts):
        bad = (~topk_gap_ok(router_logits(x, wr, bias), k, gap)).nonzero().flatten()
        if bad.numel() == 0:
            return x
        x[bad] = redraw(bad.numel(), attempt).to(x.dtype)
    raise RuntimeError("logit-gap filter did not converge")


# --------------------------------------------------------------------------
# Token routing by expert -- [FT] §3 workflow (append row index, sort by
# expert_idx, permute the activation matrix); [Specter] step 5 (group tokens
# by expert so the per-token GEMV becomes a per-expert GEMM)
# --------------------------------------------------------------------------


def sort_by_expert(ids: torch.Tensor, E: int):
    """Stable sort of flat indices f = t*k + j by expert id.

    Returns counts (E), offsets (E+1), perm (R): perm[p] = f, inv_perm (R): inv_perm[f] = p."""
    flat = ids.reshape(-1).long()
    counts = torch.stack([(flat == e).sum() for e in range(E)]).to(torch.int32)
    offsets = torch.zeros(E + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(counts, 0)
    perm = torch.cat([(flat == e).nonzero().flatten() for e in range(E)]).to(torch.int32)
    inv_perm = torch.empty_like(perm)
    inv_perm[perm.long()] = torch.arange(perm.numel(), dtype=torch.int32)
    return counts, offsets, perm, inv_perm


def permute_rows(x: torch.Tensor, perm: torch.Tensor, k: int) -> torch.Tensor:
    """Xp[p] = x[perm[p] // k]."""
    return x[(perm.long() // k)]


# --------------------------------------------------------------------------
# Expert FFN and activations
# --------------------------------------------------------------------------


def relu(h):
    return torch.clamp(h, min=0.0)


def gelu(h):
    """Exact GELU: h * Phi(h) = 0.5 h (1 + erf(h / sqrt 2))."""
    return 0.5 * h * (1.0 + torch.erf(h / torch.sqrt(torch.tensor(2.0, dtype=F64))))


def silu(h):
    return h / (1.0 + torch.exp(-h))


def activation(h: torch.Tensor, act: str) -> torch.Tensor:
    if act == "relu":
        return relu(h)
    if act == "gelu":
        return gelu(h)
    if act == "swiglu":
        F = h.shape[-1] // 2
        return silu(h[..., :F]) * h[..., F:]
    if act == "none":
        return h
    raise ValueError(act)


def expert_ffn(xe: torch.Tensor, w1: torch.Tensor, w2: torch.Tensor, act: str) -> torch.Tensor:
    """act(x . W1) . W2 in float64, no intermediate rounding."""
    return activation(xe.to(F64) @ w1, act) @ w2


def shared_expert(x: torch.Tensor, ws_gu: torch.Tensor, ws_d: torch.Tensor) -> torch.Tensor:
    """Unquantized 16-bit SwiGLU shared expert, ungated: (silu(x Wg) * (x Wu)) Wd."""
    return expert_ffn(x, ws_gu.to(F64), ws_d.to(F64), "swiglu")


# --------------------------------------------------------------------------
# Whole layer -- [FT] §3 workflow and Figure 1 (route, sort, grouped GEMM,
# un-permute with expert_scale); [Specter] core method (router and shared
# expert stay in 16-bit, only the expert MLPs are quantized)
# --------------------------------------------------------------------------


def moe_layer(x, w, cfg, token_subset: Optional[torch.Tensor] = None, renormalize: bool = False):
    """Reference MoE layer.

    x: (T, d) 16-bit; w: synth.LayerWeights; cfg: synth.LayerConfig.
    Routing, counts, offsets and permutation are computed for all T tokens.
    If token_subset is given, expert outputs and the combined output are
    computed only for those tokens (the layer is independent per token).
    Returns a dict with logits, ids, gate, counts, offsets, perm, inv_perm
    and out (len(subset) or T, d) float64, unrounded."""
    T, k, E = x.shape[0], cfg.k, cfg.E
    logits, ids, gate = route(x, w.wr, w.bias, k, renormalize)
    counts, offsets, perm, inv_perm = sort_by_expert(ids, E)
    toks = torch.arange(T) if token_subset is None else token_subset.long()
    want = torch.zeros(T, dtype=torch.bool)
    want[toks] = True
    y = torch.zeros(T * k, cfg.d, dtype=F64)                    # Yp, permuted order
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if lo == hi:
            continue                                            # empty expert: weights never touched
        f = perm[lo:hi].long()
        sel = want[f // k]
        if not bool(sel.any()):
            continue
        rows = torch.arange(lo, hi)[sel]
        w1 = dequant(w.q1[e:e + 1], w.s1[e:e + 1], cfg.group)[0]
        w2 = dequant(w.q2[e:e + 1], w.s2[e:e + 1], cfg.group)[0]
        y[rows] = expert_ffn(permute_rows(x, perm[rows], k), w1, w2, cfg.act)
    out = torch.zeros(len(toks), cfg.d, dtype=F64)
    for j in range(k):
        p = inv_perm[toks * k + j].long()
        out += gate[toks, j].unsqueeze(1) * y[p]
    if w.ws_gu is not None:
        out += shared_expert(x[toks], w.ws_gu, w.ws_d)
    return dict(logits=logits, ids=ids, gate=gate, counts=counts, offsets=offsets, perm=perm,
                inv_perm=inv_perm, out=out, y=y, tokens=toks)


def moe_layer_per_token(x, w, cfg, renormalize: bool = False) -> torch.Tensor:
    """Same layer without any reordering: every token runs its k experts one by one
    (the per-token GEMV form that [Specter] step 5 regroups into GEMMs)."""
    T, k = x.shape[0], cfg.k
    _, ids, gate = route(x, w.wr, w.bias, k, renormalize)
    out = torch.zeros(T, cfg.d, dtype=F64)
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            w1 = dequant(w.q1[e:e + 1], w.s1[e:e + 1], cfg.group)[0]
            w2 = dequant(w.q2[e:e + 1], w.s2[e:e + 1], cfg.group)[0]
            out[t] += float(gate[t, j]) * expert_ffn(x[t:t + 1], w1, w2, cfg.act)[0]
    if w.ws_gu is not None:
        out += shared_expert(x, w.ws_gu, w.ws_d)
    return out


# --------------------------------------------------------------------------
# Comparison metrics used by the parity tests
# --------------------------------------------------------------------------


def rel_l2(got: torch.Tensor, ref: torch.Tensor) -> float:
    g, r = got.to(F64), ref.to(F64)
    return float(torch.linalg.vector_norm(g - r) / max(float(torch.linalg.vector_norm(r)), 1e-300))


def max_abs_rel(got: torch.Tensor, ref: torch.Tensor) -> float:
    g, r = got.to(F64), ref.to(F64)
    return float((g - r).abs().max() / max(float(r.abs().max()), 1e-300))


def brute_force_topk(logits_row, k: int):
    """Every k-subset by total logit; ordered by logit desc, ties by lower id (tiny E only)."""
    E = len(logits_row)
    best = max(itertools.combinations(range(E), k), key=lambda c: (sum(logits_row[i] for i in c), [-i for i in c]))
    return sorted(best, key=lambda i: (-logits_row[i], i))
