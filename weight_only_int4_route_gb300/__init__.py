"""GB300-native weight-only INT4/INT8 MoE expert layer.

The compute path lives in the C-ABI library libmoe.so (hand-written sm_103a
CUDA, see include/moe.h).  `weight_only_int4_route_gb300.moe` is the thin
ctypes binding; `synth` draws the seeded synthetic inputs.  Importing the
package loads nothing; the library is loaded on first use of `moe`.
"""
__all__ = ["synth", "moe"]
