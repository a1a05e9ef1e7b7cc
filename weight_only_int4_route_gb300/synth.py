"""Seeded synthetic inputs for the quantized MoE expert layer.

This module only draws random numbers with the shapes and value ranges of the
five layer configurations; it holds none of the layer's arithmetic (no
dequantisation, routing, sorting or matrix products).  Both the CUDA path and
the CPU oracle take their inputs from here.

Each tensor has its own torch.Generator, seeded from (config seed, layer,
tensor id, token count), so a tensor never depends on which other tensors were
drawn before it.  Values drawn on the CPU and on a CUDA device differ (torch's
generators differ per device); tests draw on the CPU and copy to the device.

Distributions (readings of the page texts, restated for each config):
  * activations x ~ N(0, 1) in the activation dtype;
  * INT4 codes uniform on [-7, 7], INT8 codes uniform on [-127, 127],
    one signed code per byte, logical shape (E, K, N) with K the reduction
    dimension ("Who Says Elephants Can't Run", Expert quantization,
    Algorithm 1: W of shape (E, M, N), scales (E, 1, N));
  * scales U[0.005, 0.02] * sqrt(256 / K) * (sigma_4 / sigma_code) in the
    activation dtype, shape (E, 1, N) per channel or (E, K/128, N) for
    group 128 (GPTQ group size 128, Specter: background on GPTQ INT4);
  * router weights N(0, std = 1/sqrt(d)) in fp32 (tiny config) or the
    activation dtype; Zipf(s) logit bias b[e] = -s * ln(rank[e]) with a
    seeded permutation of ranks 1..E;
  * shared-expert weights N(0, std = 1/sqrt(K)) in the activation dtype.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}

# Standard deviation of a code drawn uniformly from [-7, 7] and [-127, 127].
SIGMA_CODE = {4: math.sqrt(((2 * 7 + 1) ** 2 - 1) / 12.0), 8: math.sqrt(((2 * 127 + 1) ** 2 - 1) / 12.0)}
QMAX = {4: 7, 8: 127}


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    d: int                 # hidden size (FC1 reduction dim, FC2 output dim)
    F: int                 # expert intermediate size
    E: int                 # routed experts
    k: int                 # experts per token
    act: str               # "relu" | "gelu" | "swiglu"
    bits: int              # 4 | 8
    group: int             # 0 = per output channel, 128 = group of 128 input rows
    dtype: str             # activation / scale / shared-weight dtype: "f16" | "bf16"
    router_dtype: str      # "f32" | "f16" | "bf16"
    Fs: int = 0            # shared-expert intermediate size (0 = none)
    zipf: float = 0.0      # Zipf exponent of the router logit bias (0 = none)
    layers: int = 1        # stacked layers timed back to back
    T: tuple = ()          # token counts of the workload
    index: int = 0         # config index, seeds derive from it

    @property
    def F1(self) -> int:
        """FC1 output width: 2F for SwiGLU (gate columns then up columns), else F."""
        return 2 * self.F if self.act == "swiglu" else self.F

    @property
    def seed(self) -> int:
        return 1234 + self.index

    @property
    def torch_dtype(self) -> torch.dtype:
        return _DT[self.dtype]

    @property
    def router_torch_dtype(self) -> torch.dtype:
        return _DT[self.router_dtype]


CONFIGS = {
    "tiny": LayerConfig("tiny", d=256, F=512, E=8, k=2, act="relu", bits=4, group=0,
                        dtype="f16", router_dtype="f32", T=(16,), index=0),
    "encdec_int8": LayerConfig("encdec_int8", d=1024, F=4096, E=32, k=1, act="gelu", bits=8, group=0,
                               dtype="f16", router_dtype="f16", T=(40, 320, 1280, 3840), index=1),
    "encdec_int4": LayerConfig("encdec_int4", d=1024, F=4096, E=32, k=1, act="gelu", bits=4, group=0,
                               dtype="f16", router_dtype="f16", T=(40, 320, 1280, 3840), index=1),
    "qwen": LayerConfig("qwen", d=2048, F=1408, E=60, k=4, act="swiglu", bits=4, group=128,
                        dtype="bf16", router_dtype="bf16", Fs=4 * 1408, T=(1, 8, 32, 4096), index=2),
    "dsv2": LayerConfig("dsv2", d=2048, F=1408, E=64, k=6, act="swiglu", bits=4, group=128,
                        dtype="bf16", router_dtype="bf16", Fs=2 * 1408, zipf=1.1, T=(32, 512), index=3),
    "phi": LayerConfig("phi", d=4096, F=6400, E=16, k=2, act="swiglu", bits=4, group=128,
                       dtype="bf16", router_dtype="bf16", layers=32, T=(1, 16, 32, 8192), index=4),
}

# tensor ids for generator sub-seeds
_TID = {"x": 1, "wr": 2, "bias": 3, "q1": 4, "s1": 5, "q2": 6, "s2": 7, "wsgu": 8, "wsd": 9, "xfix": 10}


def generator(cfg: LayerConfig, tensor: str, layer: int = 0, extra: int = 0,
              device: str | torch.device = "cpu") -> torch.Generator:
    """Independent generator for one tensor of one layer."""
    seed = (cfg.seed * 1_000_003 + _TID[tensor] * 10_007 + layer * 101 + extra * 7919) % (2 ** 63 - 1)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def codes(cfg: LayerConfig, which: str, shape: Sequence[int], layer: int = 0, device="cpu") -> torch.Tensor:
    """Signed integer codes, one per int8, uniform on [-qmax, qmax]."""
    qmax = QMAX[cfg.bits]
    g = generator(cfg, which, layer, device=device)
    return torch.randint(-qmax, qmax + 1, tuple(shape), dtype=torch.int8, generator=g, device=device)


def scales(cfg: LayerConfig, which: str, E: int, K: int, N: int, layer: int = 0, device="cpu") -> torch.Tensor:
    G = 1 if cfg.group == 0 else K // cfg.group
    amp = math.sqrt(256.0 / K) * (SIGMA_CODE[4] / SIGMA_CODE[cfg.bits])
    g = generator(cfg, which, layer, device=device)
    u = torch.rand((E, G, N), generator=g, device=device, dtype=torch.float32)
    return ((0.005 + 0.015 * u) * amp).to(cfg.torch_dtype)


def normal(cfg: LayerConfig, which: str, shape, std: float, dtype: torch.dtype, layer: int = 0,
           extra: int = 0, device="cpu") -> torch.Tensor:
    g = generator(cfg, which, layer, extra, device=device)
    return (torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32) * std).to(dtype)


@dataclasses.dataclass
class LayerWeights:
    """One layer's inputs in their logical (page) layout."""
    wr: torch.Tensor                 # (d, E) router weights
    bias: Optional[torch.Tensor]     # (E,) fp32 logit bias or None
    q1: torch.Tensor                 # (E, d, F1) int8 codes
    s1: torch.Tensor                 # (E, G1, F1) scales
    q2: torch.Tensor                 # (E, F, d) int8 codes
    s2: torch.Tensor                 # (E, G2, d) scales
    ws_gu: Optional[torch.Tensor]    # (d, 2Fs) shared gate|up weights
    ws_d: Optional[torch.Tensor]     # (Fs, d) shared down weights


def zipf_bias(cfg: LayerConfig, layer: int = 0, device="cpu") -> Optional[torch.Tensor]:
    if cfg.zipf == 0.0:
        return None
    g = generator(cfg, "bias", layer, device="cpu")
    rank = torch.randperm(cfg.E, generator=g).to(torch.float64) + 1.0
    return (-cfg.zipf * torch.log(rank)).to(torch.float32).to(device)


def layer_weights(cfg: LayerConfig, layer: int = 0, device="cpu") -> LayerWeights:
    d, F, F1, E = cfg.d, cfg.F, cfg.F1, cfg.E
    wr = normal(cfg, "wr", (d, E), 1.0 / math.sqrt(d), cfg.router_torch_dtype, layer, device=device)
    q1 = codes(cfg, "q1", (E, d, F1), layer, device)
    s1 = scales(cfg, "s1", E, d, F1, layer, device)
    q2 = codes(cfg, "q2", (E, F, d), layer, device)
    s2 = scales(cfg, "s2", E, F, d, layer, device)
    ws_gu = ws_d = None
    if cfg.Fs:
        ws_gu = normal(cfg, "wsgu", (d, 2 * cfg.Fs), 1.0 / math.sqrt(d), cfg.torch_dtype, layer, device=device)
        ws_d = normal(cfg, "wsd", (cfg.Fs, d), 1.0 / math.sqrt(cfg.Fs), cfg.torch_dtype, layer, device=device)
    return LayerWeights(wr, zipf_bias(cfg, layer, device), q1, s1, q2, s2, ws_gu, ws_d)


def activations(cfg: LayerConfig, T: int, device="cpu") -> torch.Tensor:
    """x (T, d) ~ N(0, 1) in the activation dtype."""
    return normal(cfg, "x", (T, cfg.d), 1.0, cfg.torch_dtype, extra=T, device=device)


def redraw_rows(cfg: LayerConfig, T: int, n_rows: int, attempt: int, device="cpu") -> torch.Tensor:
    """Fresh N(0,1) rows used to replace tokens rejected by a test's logit-gap filter."""
    return normal(cfg, "xfix", (n_rows, cfg.d), 1.0, cfg.torch_dtype, extra=T * 1000 + attempt, device=device)


def custom(name: str, **kw) -> LayerConfig:
    """A config derived from a named one with some fields replaced (test shapes)."""
    return dataclasses.replace(CONFIGS[name], **kw)
