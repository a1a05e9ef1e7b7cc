"""Shared helpers for the parity tests: seeded inputs with the top-k logit-gap filter,
tolerance checks, and GPU availability."""
from __future__ import annotations

import torch

from oracle import moe_oracle as O
from weight_only_int4_route_gb300 import synth

# Layer-output tolerance (relative L2 and max-abs relative to max |ref|).
REL_L2 = 5e-3
MAX_ABS = 2e-2
# Router gate tolerance.  The GPU accumulates the d <= 4096 bf16/fp16 products of a logit in
# fp32 on the tensor cores, then takes an fp32 exp and divide; a gate's relative error is at
# most about twice the absolute logit error.  Measured against the float64 oracle the worst
# gate over 16,384 (Phi-shaped, d = 4096) is 1.6e-5 relative, so 1e-4 keeps a 6x margin.  Expert
# ids stay bit-exact because the inputs keep a 1e-3 gap between the top k+1 logits.
GATE_RTOL = 1e-4
GAP = 1e-3


def have_gpu() -> bool:
    return torch.cuda.is_available()


def layer_inputs(cfg, T, device="cpu", gap=GAP):
    """Weights and gap-filtered activations for one layer (drawn on the CPU)."""
    w = synth.layer_weights(cfg)
    x = synth.activations(cfg, T)
    if T > 0:
        x = O.gap_filtered(x, w.wr, w.bias, cfg.k, lambda n, a: synth.redraw_rows(cfg, T, n, a), gap)
    return w, x


def assert_close_layer(got: torch.Tensor, ref: torch.Tensor, what: str = ""):
    rl2 = O.rel_l2(got.double().cpu(), ref)
    mar = O.max_abs_rel(got.double().cpu(), ref)
    assert rl2 <= REL_L2 and mar <= MAX_ABS, f"{what}: rel_l2={rl2:.3e} max_abs_rel={mar:.3e}"
    return rl2, mar
