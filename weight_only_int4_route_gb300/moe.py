"""ctypes binding of libmoe (include/moe.h): argument marshalling only.

Every function below checks shapes, allocates outputs with torch on the input's device
and forwards raw device pointers to the C ABI on torch's current CUDA stream.  All
arithmetic happens in libmoe's CUDA kernels; there is no CPU fallback, and importing
this module fails if libmoe.so has not been built.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import re
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")
LIB_CHECKED_PATH = os.path.join(_PKG, "libmoe_checked.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "moe.h")

F16, BF16, F32 = 0, 1, 2
ACT = {"none": 0, "relu": 1, "gelu": 2, "swiglu": 3}
_TORCH2MOE = {torch.float16: F16, torch.bfloat16: BF16, torch.float32: F32}
_MOE2TORCH = {v: k for k, v in _TORCH2MOE.items()}

_c_i64, _c_int, _c_size, _vp = ctypes.c_int64, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str, message: str):
        super().__init__(f"{what} failed with status {status}: {message}")
        self.status = status


class LayerDesc(ctypes.Structure):
    _fields_ = [("d", _c_i64), ("F", _c_i64), ("E", _c_i64), ("k", ctypes.c_int32), ("act", ctypes.c_int32),
                ("bits", ctypes.c_int32), ("group", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("router_dtype", ctypes.c_int32), ("renormalize", ctypes.c_int32), ("Fs", _c_i64)]


class LayerWeightsC(ctypes.Structure):
    _fields_ = [("w_router", _vp), ("router_bias", _vp), ("w1", _vp), ("w2", _vp),
                ("ws_gate_up", _vp), ("ws_down", _vp)]


class LayerRouting(ctypes.Structure):
    _fields_ = [("ids", _vp), ("gate_w", _vp), ("offsets", _vp), ("perm", _vp), ("inv_perm", _vp)]


_SIGS = {
    "moe_last_error_string": (ctypes.c_char_p, []),
    "moe_version": (_c_int, []),
    "moe_device_error": (_c_int, [_vp, ctypes.POINTER(ctypes.c_int32)]),
    "moe_checked_build": (_c_int, []),
    "moe_set_decode_mode": (_c_int, [_c_int]),
    "moe_set_gemm_pairs": (_c_int, [_c_int]),
    "moe_check_status": (_c_int, [_vp, ctypes.POINTER(ctypes.c_int32)]),
    "moe_packed_size": (_c_size, [_c_i64, _c_i64, _c_i64, _c_int, _c_int]),
    "moe_packed_scale_offset": (_c_size, [_c_i64, _c_i64, _c_i64, _c_int]),
    "moe_pack_weights": (_c_int, [_vp, _vp, _c_int, _c_i64, _c_i64, _c_i64, _c_int, _c_int, _vp, _c_size, _vp]),
    "moe_dequant": (_c_int, [_vp, _c_int, _c_i64, _c_i64, _c_i64, _c_int, _c_int, _c_int, _vp, _vp]),
    "moe_route_topk_workspace_size": (_c_size, [_c_i64, _c_i64, _c_i64]),
    "moe_route_topk": (_c_int, [_vp, _c_int, _vp, _c_int, _vp, _c_i64, _c_i64, _c_i64, _c_int, _c_int, _vp, _vp, _vp, _c_size, _vp]),
    "moe_permute_workspace_size": (_c_size, [_c_i64, _c_i64, _c_int]),
    "moe_permute": (_c_int, [_vp, _vp, _c_int, _c_i64, _c_i64, _c_i64, _c_int, _vp, _vp, _vp, _vp, _vp, _c_size, _vp]),
    "moe_gemm_path": (_c_int, [_c_i64, _c_i64, _c_i64, _c_i64, _c_int, _c_int, _c_int]),
    "moe_grouped_gemm_workspace_size": (_c_size, [_c_i64, _c_i64, _c_i64, _c_i64, _c_int, _c_int]),
    "moe_grouped_gemm_w4a16": (_c_int, [_vp, _c_int, _vp, _c_i64, _c_i64, _c_i64, _c_int, _vp, _c_i64, _c_int, _vp, _c_int, _vp, _c_size, _vp]),
    "moe_grouped_gemm_w8a16": (_c_int, [_vp, _c_int, _vp, _c_i64, _c_i64, _c_i64, _c_int, _vp, _c_i64, _c_int, _vp, _c_int, _vp, _c_size, _vp]),
    "moe_grouped_gemm_w4a16_static": (_c_int, [_vp, _c_int, _vp, _c_i64, _c_i64, _c_i64, _c_int, _vp, _c_i64, _c_int, _vp, _c_int, _vp]),
    "moe_grouped_gemm_w16a16": (_c_int, [_vp, _c_int, _vp, _c_i64, _c_i64, _c_i64, _vp, _c_i64, _c_int, _vp, _c_int, _vp, _c_size, _vp]),
    "moe_unpermute_combine": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _c_int, _c_i64, _c_i64, _c_int, _vp, _c_int, _vp]),
    "moe_shared_expert_workspace_size": (_c_size, [_c_i64, _c_i64, _c_i64]),
    "moe_shared_expert": (_c_int, [_vp, _c_int, _vp, _vp, _c_i64, _c_i64, _c_i64, _vp, _c_int, _vp, _c_size, _vp]),
    "moe_layer_workspace_size": (_c_size, [ctypes.POINTER(LayerDesc), _c_i64]),
    "moe_layer_routing_view": (_c_int, [ctypes.POINTER(LayerDesc), _c_i64, _vp, ctypes.POINTER(LayerRouting)]),
    "moe_layer_launch_count": (_c_int, [ctypes.POINTER(LayerDesc), _c_i64]),
    "moe_layer_forward": (_c_int, [ctypes.POINTER(LayerDesc), ctypes.POINTER(LayerWeightsC), _vp, _c_i64, _vp, _vp, _c_size, _vp]),
    "moe_bf16_recombine": (_c_int, [_vp, _vp, _c_i64, _vp, _vp]),
    "moe_bf16_split": (_c_int, [_vp, _c_i64, _vp, _vp, _vp]),
    "moe_elb_accumulate": (_c_int, [_vp, _c_i64, _c_i64, _c_int, _c_i64, _vp, _vp]),
    "moe_elb_topm": (_c_int, [_vp, _c_i64, _c_i64, _c_int, _vp, _vp, _vp]),
    "moe_elb_step": (_c_int, [_vp, _c_i64, _c_i64, _c_int, _c_i64, _vp, _c_int, _vp, _vp, _vp]),
    "moe_layer_graph_create": (_c_int, [ctypes.POINTER(LayerDesc), ctypes.POINTER(LayerWeightsC), _vp, _c_i64, _vp,
                                        _vp, ctypes.c_size_t, _vp, ctypes.POINTER(_vp)]),
    "moe_layer_graph_launch": (_c_int, [_vp, _vp]),
    "moe_layer_graph_destroy": (_c_int, [_vp]),
    "moe_layer_forward_profiled": (_c_int, [ctypes.POINTER(LayerDesc), ctypes.POINTER(LayerWeightsC), _vp, _c_i64, _vp, _vp,
                                            _c_size, _vp, ctypes.POINTER(_vp)]),
}

# stage boundaries recorded by moe_layer_forward_profiled (enum in include/moe.h)
STAGES = ("start", "routed", "permuted", "fc1", "fc2", "shared", "done")

_lib: Optional[ctypes.CDLL] = None
_lib_checked: Optional[ctypes.CDLL] = None


def header_symbols() -> list[str]:
    """Every function declared in include/moe.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def _load(path: str) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(f"{os.path.basename(path)} is not built ({path}); run weight_only_int4_route_gb300/build.py "
                           "or __graft_entry__.build() -- there is no fallback path")
    L = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib() -> ctypes.CDLL:
    """The library (libmoe.so)."""
    global _lib
    if _lib is None:
        _lib = _load(LIB_PATH)
    return _lib


def lib_checked() -> ctypes.CDLL:
    """The bounds-checked build of the same library (libmoe_checked.so), for tests and debugging."""
    global _lib_checked
    if _lib_checked is None:
        _lib_checked = _load(LIB_CHECKED_PATH)
    return _lib_checked


_DECODE_MODES = {"auto": 0, "chain": 1, "launch": 2}


def set_decode_mode(mode: str) -> str:
    """'auto' (the default: one kernel launch for small decode steps, else the chain), 'chain' (the
    kernel chain) or 'launch' (one launch whenever the layer allows it); returns the previous mode."""
    prev = lib().moe_set_decode_mode(_DECODE_MODES[mode])
    if prev < 0:
        _check(prev, "moe_set_decode_mode")
    return {v: k for k, v in _DECODE_MODES.items()}[prev]


def set_gemm_pairs(on: bool) -> bool:
    """CTA pairs (M = 256) for the quantized tcgen05 GEMM on or off (process-wide); returns the
    previous setting."""
    prev = lib().moe_set_gemm_pairs(1 if on else 0)
    if prev < 0:
        _check(prev, "moe_set_gemm_pairs")
    return bool(prev)


def check_status(device="cuda:0", L: Optional[ctypes.CDLL] = None) -> tuple[int, int]:
    """(status, flags) of moe_check_status on the current stream: synchronizes, reads and clears
    the library's device check word (always 0 in the plain build)."""
    v = ctypes.c_int32(0)
    st = (L or lib()).moe_check_status(_stream(torch.device(device)), ctypes.byref(v))
    return int(st), int(v.value)


def _check(st: int, what: str):
    if st != 0:
        raise MoeError(st, what, lib().moe_last_error_string().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dt(t: torch.Tensor) -> int:
    return _TORCH2MOE[t.dtype]


def device_error(device="cuda:0") -> int:
    """Synchronize the current stream and return (and clear) the library's device error code."""
    v = ctypes.c_int32(0)
    _check(lib().moe_device_error(_stream(torch.device(device)), ctypes.byref(v)), "moe_device_error")
    return int(v.value)


# ---------------------------------------------------------------- weights


def packed_size(E, K, N, bits, group) -> int:
    return int(lib().moe_packed_size(E, K, N, bits, group))


def pack_weights(codes: torch.Tensor, scales: Optional[torch.Tensor], bits: int, group: int,
                 w_dtype: Optional[torch.dtype] = None) -> torch.Tensor:
    """codes (E, K, N) int8 (or 16-bit weights for bits 16) -> packed uint8 buffer."""
    E, K, N = codes.shape
    w_dtype = w_dtype or (codes.dtype if bits == 16 else scales.dtype)
    out = torch.empty(packed_size(E, K, N, bits, group), dtype=torch.uint8, device=codes.device)
    _check(lib().moe_pack_weights(_ptr(codes.contiguous()), _ptr(None if scales is None else scales.contiguous()),
                                  _TORCH2MOE[w_dtype], E, K, N, bits, group, _ptr(out), out.numel(),
                                  _stream(codes.device)), "moe_pack_weights")
    return out


def dequant(packed, E, K, N, bits, group, w_dtype: torch.dtype, out_dtype: torch.dtype) -> torch.Tensor:
    out = torch.empty((E, K, N), dtype=out_dtype, device=packed.device)
    _check(lib().moe_dequant(_ptr(packed), _TORCH2MOE[w_dtype], E, K, N, bits, group, _TORCH2MOE[out_dtype],
                             _ptr(out), _stream(packed.device)), "moe_dequant")
    return out


# ---------------------------------------------------------------- routing


def route_topk(x: torch.Tensor, wr: torch.Tensor, bias: Optional[torch.Tensor], k: int, renormalize=False):
    T, d = x.shape
    E = wr.shape[1]
    ids = torch.empty((T, k), dtype=torch.int32, device=x.device)
    gate = torch.empty((T, k), dtype=torch.float32, device=x.device)
    wsb = int(lib().moe_route_topk_workspace_size(T, d, E))
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=x.device)
    _check(lib().moe_route_topk(_ptr(x), _dt(x), _ptr(wr), _dt(wr), _ptr(bias), T, d, E, k, int(renormalize),
                                _ptr(ids), _ptr(gate), _ptr(ws), ws.numel(), _stream(x.device)), "moe_route_topk")
    return ids, gate


def permute(ids: torch.Tensor, x: torch.Tensor, E: int):
    T, k = ids.shape
    d = x.shape[1]
    dev = x.device
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    inv = torch.empty(T * k, dtype=torch.int32, device=dev)
    xp = torch.empty((T * k, d), dtype=x.dtype, device=dev)
    wsb = int(lib().moe_permute_workspace_size(T, E, k))
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    _check(lib().moe_permute(_ptr(ids), _ptr(x), _dt(x), T, d, E, k, _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(xp),
                             _ptr(ws), ws.numel(), _stream(dev)), "moe_permute")
    return offsets, perm, inv, xp


# ---------------------------------------------------------------- GEMM / combine / shared


def grouped_gemm(a: torch.Tensor, packed: torch.Tensor, bits: int, E: int, K: int, N: int, group: int,
                 offsets: Optional[torch.Tensor], act: str, out_dtype: torch.dtype) -> torch.Tensor:
    R = a.shape[0]
    n_out = N // 2 if act == "swiglu" else N
    out = torch.empty((R, n_out), dtype=out_dtype, device=a.device)
    wsb = int(lib().moe_grouped_gemm_workspace_size(R, E, K, N, bits, ACT[act]))
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=a.device)
    args = (_ptr(a), _dt(a), _ptr(packed), E, K, N)
    tail = (_ptr(offsets), R, ACT[act], _ptr(out), _TORCH2MOE[out_dtype], _ptr(ws), ws.numel(), _stream(a.device))
    if bits == 4:
        st = lib().moe_grouped_gemm_w4a16(*args, group, *tail)
    elif bits == 8:
        st = lib().moe_grouped_gemm_w8a16(*args, group, *tail)
    else:
        st = lib().moe_grouped_gemm_w16a16(*args, *tail)
    _check(st, f"moe_grouped_gemm (bits {bits})")
    return out


def grouped_gemm_static(a: torch.Tensor, packed: torch.Tensor, E: int, K: int, N: int, group: int,
                        offsets: torch.Tensor, act: str, out_dtype: torch.dtype) -> torch.Tensor:
    """INT4 grouped GEMM whose scratch lives in the library (no workspace argument)."""
    R = a.shape[0]
    out = torch.empty((R, N // 2 if act == "swiglu" else N), dtype=out_dtype, device=a.device)
    _check(lib().moe_grouped_gemm_w4a16_static(_ptr(a), _dt(a), _ptr(packed), E, K, N, group, _ptr(offsets), R,
                                               ACT[act], _ptr(out), _TORCH2MOE[out_dtype], _stream(a.device)),
           "moe_grouped_gemm_w4a16_static")
    return out


def gemm_path(R, E, K, N, bits, group, act: str) -> str:
    """'tcgen05', 'gemv' or 'mma': the kernel a grouped GEMM of this shape dispatches to."""
    return {0: "mma", 1: "tcgen05", 2: "gemv"}[lib().moe_gemm_path(R, E, K, N, bits, group, ACT[act])]


def unpermute_combine(yp: torch.Tensor, inv_perm: torch.Tensor, gate: torch.Tensor,
                      shared: Optional[torch.Tensor], out_dtype: torch.dtype) -> torch.Tensor:
    T, k = gate.shape
    d = yp.shape[1]
    out = torch.empty((T, d), dtype=out_dtype, device=yp.device)
    _check(lib().moe_unpermute_combine(_ptr(yp), _dt(yp), _ptr(inv_perm), _ptr(gate), _ptr(shared),
                                       F32 if shared is None else _dt(shared), T, d, k, _ptr(out),
                                       _TORCH2MOE[out_dtype], _stream(yp.device)), "moe_unpermute_combine")
    return out


def shared_expert(x: torch.Tensor, wgu_packed: torch.Tensor, wd_packed: torch.Tensor, Fs: int,
                  out_dtype: torch.dtype) -> torch.Tensor:
    T, d = x.shape
    out = torch.empty((T, d), dtype=out_dtype, device=x.device)
    wsb = int(lib().moe_shared_expert_workspace_size(T, d, Fs))
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=x.device)
    _check(lib().moe_shared_expert(_ptr(x), _dt(x), _ptr(wgu_packed), _ptr(wd_packed), T, d, Fs, _ptr(out),
                                   _TORCH2MOE[out_dtype], _ptr(ws), ws.numel(), _stream(x.device)),
           "moe_shared_expert")
    return out


# ---------------------------------------------------------------- whole layer


@dataclasses.dataclass
class PackedLayer:
    """One layer's device-resident weights in libmoe's packed format."""
    cfg: object
    wr: torch.Tensor
    bias: Optional[torch.Tensor]
    w1: torch.Tensor
    w2: torch.Tensor
    ws_gu: Optional[torch.Tensor]
    ws_d: Optional[torch.Tensor]

    @staticmethod
    def from_weights(cfg, w, device) -> "PackedLayer":
        dev = torch.device(device)
        w1 = pack_weights(w.q1.to(dev), w.s1.to(dev), cfg.bits, cfg.group)
        w2 = pack_weights(w.q2.to(dev), w.s2.to(dev), cfg.bits, cfg.group)
        gu = dn = None
        if cfg.Fs:
            gu = pack_weights(w.ws_gu.to(dev)[None], None, 16, 0)
            dn = pack_weights(w.ws_d.to(dev)[None], None, 16, 0)
        bias = None if w.bias is None else w.bias.to(dev)
        return PackedLayer(cfg, w.wr.to(dev).contiguous(), bias, w1, w2, gu, dn)


def layer_desc(cfg, renormalize: bool = False) -> LayerDesc:
    return LayerDesc(cfg.d, cfg.F, cfg.E, cfg.k, ACT[cfg.act], cfg.bits, cfg.group,
                     _TORCH2MOE[cfg.torch_dtype], _TORCH2MOE[cfg.router_torch_dtype], int(renormalize), cfg.Fs)


class Layer:
    """moe_layer_forward with a reusable workspace for token counts up to max_T."""

    def __init__(self, packed: PackedLayer, max_T: int, renormalize: bool = False,
                 workspace: Optional[torch.Tensor] = None):
        self.p = packed
        self.cfg = packed.cfg
        self.desc = layer_desc(self.cfg, renormalize)
        self.max_T = max_T
        self.ws_bytes = int(lib().moe_layer_workspace_size(ctypes.byref(self.desc), max_T))
        if workspace is None:
            workspace = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=packed.w1.device)
        assert workspace.numel() >= self.ws_bytes
        self.ws = workspace
        p = packed
        self.wc = LayerWeightsC(p.wr.data_ptr(), None if p.bias is None else p.bias.data_ptr(), p.w1.data_ptr(),
                                p.w2.data_ptr(), None if p.ws_gu is None else p.ws_gu.data_ptr(),
                                None if p.ws_d is None else p.ws_d.data_ptr())

    def launch_count(self, T: int) -> int:
        return int(lib().moe_layer_launch_count(ctypes.byref(self.desc), T))

    def workspace_bytes(self, T: int) -> int:
        return int(lib().moe_layer_workspace_size(ctypes.byref(self.desc), T))

    def forward(self, x: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
        T = x.shape[0]
        assert T <= self.max_T and x.dtype == self.cfg.torch_dtype and x.is_contiguous()
        if out is None:
            out = torch.empty((T, self.cfg.d), dtype=x.dtype, device=x.device)
        _check(lib().moe_layer_forward(ctypes.byref(self.desc), ctypes.byref(self.wc), _ptr(x), T, _ptr(out),
                                       _ptr(self.ws), self.ws.numel(), _stream(x.device)), "moe_layer_forward")
        return out

    def forward_profiled(self, x: torch.Tensor, out: torch.Tensor, events) -> torch.Tensor:
        """forward() that records the STAGES events (torch.cuda.Event, already created) between stages."""
        T = x.shape[0]
        arr = (_vp * len(STAGES))(*[ctypes.c_void_p(e.cuda_event) for e in events])
        _check(lib().moe_layer_forward_profiled(ctypes.byref(self.desc), ctypes.byref(self.wc), _ptr(x), T, _ptr(out),
                                                _ptr(self.ws), self.ws.numel(), _stream(x.device), arr),
               "moe_layer_forward_profiled")
        return out

    def routing(self, T: int) -> dict:
        """Views of the routing results left in the workspace by the last forward(T tokens)."""
        v = LayerRouting()
        _check(lib().moe_layer_routing_view(ctypes.byref(self.desc), T, _ptr(self.ws), ctypes.byref(v)),
               "moe_layer_routing_view")
        base = self.ws.data_ptr()
        k, E = self.cfg.k, self.cfg.E

        def view(ptr, n, dtype):
            off = ptr - base
            esz = torch.tensor([], dtype=dtype).element_size()
            return self.ws[off:off + n * esz].view(dtype)

        return dict(ids=view(v.ids, T * k, torch.int32).view(T, k), gate=view(v.gate_w, T * k, torch.float32).view(T, k),
                    offsets=view(v.offsets, E + 1, torch.int32), perm=view(v.perm, T * k, torch.int32),
                    inv_perm=view(v.inv_perm, T * k, torch.int32))


class LayerGraph:
    """A Layer's whole chain for a fixed T captured into one CUDA graph (moe_layer_graph_*).

    The graph reads `self.x` and writes `self.out` (device buffers owned here): copy the step's
    input into `x`, call `launch()`, read `out`."""

    def __init__(self, layer: "Layer", T: int):
        assert 0 < T <= layer.max_T
        dev = layer.p.w1.device
        self.layer, self.T = layer, T
        self.x = torch.zeros((T, layer.cfg.d), dtype=layer.cfg.torch_dtype, device=dev)
        self.out = torch.empty((T, layer.cfg.d), dtype=layer.cfg.torch_dtype, device=dev)
        self.handle = _vp()
        side = torch.cuda.Stream(device=dev)            # capture needs a created stream
        side.wait_stream(torch.cuda.current_stream(dev))
        _check(lib().moe_layer_graph_create(ctypes.byref(layer.desc), ctypes.byref(layer.wc), _ptr(self.x), T,
                                            _ptr(self.out), _ptr(layer.ws), layer.ws.numel(),
                                            ctypes.c_void_p(side.cuda_stream), ctypes.byref(self.handle)),
               "moe_layer_graph_create")
        torch.cuda.current_stream(dev).wait_stream(side)

    def launch(self) -> torch.Tensor:
        _check(lib().moe_layer_graph_launch(self.handle, _stream(self.x.device)), "moe_layer_graph_launch")
        return self.out

    def close(self):
        if self.handle:
            lib().moe_layer_graph_destroy(self.handle)
            self.handle = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def bf16_split(t: torch.Tensor):
    """BF16 tensor -> (exponent bytes, sign|mantissa bytes), uint8 of t.numel() each."""
    assert t.dtype == torch.bfloat16 and t.is_contiguous()
    n = t.numel()
    exp = torch.empty(n, dtype=torch.uint8, device=t.device)
    sm = torch.empty(n, dtype=torch.uint8, device=t.device)
    _check(lib().moe_bf16_split(_ptr(t), n, _ptr(exp), _ptr(sm), _stream(t.device)), "moe_bf16_split")
    return exp, sm


def bf16_recombine(exp: torch.Tensor, sm: torch.Tensor) -> torch.Tensor:
    """(exponent bytes, sign|mantissa bytes) -> BF16 tensor of the same length."""
    assert exp.dtype == sm.dtype == torch.uint8 and exp.numel() == sm.numel()
    out = torch.empty(exp.numel(), dtype=torch.bfloat16, device=exp.device)
    _check(lib().moe_bf16_recombine(_ptr(exp), _ptr(sm), exp.numel(), _ptr(out), _stream(exp.device)),
           "moe_bf16_recombine")
    return out


def elb_accumulate(ids: torch.Tensor, E: int, counts: torch.Tensor) -> torch.Tensor:
    """ids (L, S, k) int32 draft-step routes; counts (L, E) int32, updated in place."""
    L, S, k = ids.shape
    assert ids.dtype == counts.dtype == torch.int32 and counts.shape == (L, E)
    _check(lib().moe_elb_accumulate(_ptr(ids), L, S, k, E, _ptr(counts), _stream(ids.device)), "moe_elb_accumulate")
    return counts


def elb_topm(counts: torch.Tensor, M: int):
    """counts (L, E) int32 -> (experts, counts) of each layer's top-M, (L, min(M, E)) int32."""
    L, E = counts.shape
    m = min(M, E)
    ex = torch.empty((L, m), dtype=torch.int32, device=counts.device)
    vals = torch.empty((L, m), dtype=torch.int32, device=counts.device)
    _check(lib().moe_elb_topm(_ptr(counts), L, E, M, _ptr(ex), _ptr(vals), _stream(counts.device)), "moe_elb_topm")
    return ex, vals


def elb_step(ids: torch.Tensor, E: int, counts: torch.Tensor, M: int, experts: torch.Tensor, vals: torch.Tensor):
    """elb_accumulate followed by elb_topm in one launch, into preallocated (L, min(M, E)) outputs."""
    L, S, k = ids.shape
    _check(lib().moe_elb_step(_ptr(ids), L, S, k, E, _ptr(counts), M, _ptr(experts), _ptr(vals), _stream(ids.device)),
           "moe_elb_step")
    return experts, vals
