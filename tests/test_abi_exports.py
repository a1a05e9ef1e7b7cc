"""CPU-only checks of the C ABI: the library loads, exports every symbol the header
declares, and its host-side queries and argument validation answer without a GPU
(no compute call is made here)."""
import ctypes

import pytest

from weight_only_int4_route_gb300 import build as B
from weight_only_int4_route_gb300 import moe as M


@pytest.fixture(scope="module")
def L():
    B.build()
    return M.lib()


def test_every_header_symbol_is_exported(L):
    names = M.header_symbols()
    assert len(names) >= 21
    missing = [n for n in names if not hasattr(L, n)]
    assert missing == []
    assert set(names) == set(M._SIGS), "binding and header disagree"


def test_checked_library_exports_the_same_symbols():
    """The bounds-checked build (MOE_CHECKED=1) is the same ABI: every header symbol, and it
    says that it is the checked build (the plain one says it is not)."""
    B.build(checked=True)
    C = M.lib_checked()
    assert [n for n in M.header_symbols() if not hasattr(C, n)] == []
    assert C.moe_checked_build() == 1
    assert M.lib().moe_checked_build() == 0
    assert C.moe_check_status(None, None) == -1   # host_flags NULL: refused on the host


def test_version_and_error_string(L):
    assert L.moe_version() == 1
    assert isinstance(L.moe_last_error_string(), bytes)


def test_packed_sizes(L):
    # INT4: E*N*K/2 bytes of words, then 256-aligned (E, G, N) 16-bit scales
    assert L.moe_packed_scale_offset(2, 256, 64, 4) == 2 * 64 * 128
    assert L.moe_packed_size(2, 256, 64, 4, 0) == 2 * 64 * 128 + 256
    assert L.moe_packed_size(2, 256, 64, 4, 128) == 2 * 64 * 128 + 512
    assert L.moe_packed_size(3, 256, 64, 8, 0) == 3 * 64 * 256 + 512
    assert L.moe_packed_size(1, 256, 64, 16, 0) == 256 * 64 * 2
    assert L.moe_packed_size(1, 100, 64, 4, 0) == 0          # K % 8 != 0
    assert L.moe_packed_size(1, 256, 60, 4, 0) == 0          # N % 8 != 0
    assert L.moe_packed_size(1, 192, 64, 4, 128) == 0        # K % 128 != 0 with group 128


def test_permute_workspace_size(L):
    assert L.moe_permute_workspace_size(16, 8, 2) == 2 * 256
    assert L.moe_permute_workspace_size(4096, 60, 4) == 2 * ((64 * 60 * 4 + 255) // 256 * 256)


def test_invalid_arguments_are_rejected_on_host(L):
    nul = ctypes.c_void_p(0)
    # bad bits
    assert L.moe_pack_weights(nul, nul, 0, 1, 256, 64, 5, 0, nul, 0, nul) == -1
    assert b"bits" in L.moe_last_error_string()
    # bad dtype
    assert L.moe_route_topk(nul, 7, nul, 0, nul, 4, 256, 8, 2, 0, nul, nul, nul, 0, nul) == -1
    # k > E
    assert L.moe_route_topk(nul, 0, nul, 0, nul, 4, 256, 8, 9, 0, nul, nul, nul, 0, nul) == -1
    # T == 0 is a no-op
    assert L.moe_route_topk(nul, 0, nul, 0, nul, 0, 256, 8, 2, 0, nul, nul, nul, 0, nul) == 0
    # K not a multiple of 128
    assert L.moe_grouped_gemm_w4a16(nul, 0, nul, 2, 200, 64, 0, nul, 4, 0, nul, 0, nul, 0, nul) == -1
    # unsupported N
    assert L.moe_grouped_gemm_w4a16(nul, 0, nul, 2, 256, 40, 0, nul, 4, 0, nul, 0, nul, 0, nul) == -2
    # offsets NULL with E > 1
    assert L.moe_grouped_gemm_w8a16(nul, 0, nul, 2, 256, 64, 0, nul, 4, 0, nul, 0, nul, 0, nul) == -1
    # misaligned pointer
    bad = ctypes.c_void_p(0x1003)
    assert L.moe_unpermute_combine(bad, 2, bad, bad, nul, 2, 4, 64, 1, bad, 0, nul) == -1
    # layer graph: no handle pointer, T == 0, the legacy default stream; NULL destroy is a no-op
    assert L.moe_layer_graph_create(None, None, nul, 4, nul, nul, 0, nul, None) == -1
    h = ctypes.c_void_p()
    assert L.moe_layer_graph_create(None, None, nul, 0, nul, nul, 0, nul, ctypes.byref(h)) == -1 and not h.value
    assert L.moe_layer_graph_create(None, None, nul, 4, nul, nul, 0, nul, ctypes.byref(h)) == -1 and not h.value
    assert L.moe_layer_graph_launch(nul, nul) == -1
    assert L.moe_layer_graph_destroy(nul) == 0
    # bit-field codec: negative n, misaligned planes; n == 0 is a no-op
    assert L.moe_bf16_recombine(nul, nul, -1, nul, nul) == -1
    assert L.moe_bf16_recombine(bad, bad, 64, bad, nul) == -1
    assert L.moe_bf16_split(nul, 0, nul, nul, nul) == 0
    # ELB: E above 256, k out of range; L == 0 is a no-op
    assert L.moe_elb_accumulate(nul, 2, 4, 2, 300, nul, nul) == -1
    assert L.moe_elb_accumulate(nul, 2, 4, 0, 8, nul, nul) == -1
    assert L.moe_elb_topm(nul, 0, 8, 2, nul, nul, nul) == 0


def test_layer_workspace_query(L):
    from weight_only_int4_route_gb300 import synth
    for name, cfg in synth.CONFIGS.items():
        desc = M.layer_desc(cfg)
        n = L.moe_layer_workspace_size(ctypes.byref(desc), max(cfg.T))
        assert n > 0, name
    bad = M.layer_desc(synth.CONFIGS["tiny"])
    bad.k = 99
    assert L.moe_layer_workspace_size(ctypes.byref(bad), 16) == 0


def test_layer_workspace_size_serves_every_smaller_batch(L):
    """moe_layer_workspace_size(desc, T) is the largest requirement over T' <= T (a smaller batch
    can need more: its split-K plans write partial sums in more slices), so it never decreases
    in T and a workspace sized for T serves every call with fewer tokens."""
    from weight_only_int4_route_gb300 import synth
    for name, cfg in synth.CONFIGS.items():
        d = M.layer_desc(cfg)
        sizes = [L.moe_layer_workspace_size(ctypes.byref(d), T) for T in range(1, 257)]
        assert all(s > 0 for s in sizes), name
        assert all(b >= a for a, b in zip(sizes, sizes[1:])), name
        assert L.moe_layer_workspace_size(ctypes.byref(d), 4096) >= sizes[-1], name
        big = [L.moe_layer_workspace_size(ctypes.byref(d), T) for T in (65535, 65536, 65537, 200000)]
        assert all(b >= a for a, b in zip(big, big[1:])), name


@pytest.mark.parametrize("R,E,K,N,bits,group,act,path", [
    (64, 8, 1024, 2048, 4, 0, "none", "gemv"),          # 8 rows per expert
    (128, 8, 1024, 2048, 4, 0, "none", "gemv"),         # 16: the last decode-stream size
    (136, 8, 1024, 2048, 4, 0, "none", "tcgen05"),      # 17: tensor memory from here
    (10, 100, 1024, 2048, 4, 0, "none", "gemv"),        # fewer rows than experts: 1 per active expert
    (136, 8, 1024, 192, 4, 0, "none", "mma"),           # N % 128 != 0: the warp-MMA tile kernel
    (4000, 8, 1000, 2048, 4, 0, "none", "mma"),         # K % 128 != 0
    (136, 8, 1024, 2816, 4, 128, "swiglu", "tcgen05"),  # SWIGLU: (N/2) % 64 == 0 suffices
    (4000, 8, 1024, 2048, 8, 128, "gelu", "tcgen05"),
    (16, 8, 1024, 2048, 16, 0, "none", "gemv"),         # 16-bit weights: the same thresholds
    (17, 1, 2048, 11264, 16, 0, "swiglu", "tcgen05"),
])
def test_gemm_path_follows_the_documented_rule(L, R, E, K, N, bits, group, act, path):
    """moe_gemm_path: a = ceil(R / min(E, R)) rows per active expert; a <= 16 the decode
    weight-stream kernel, a >= 17 the tcgen05 kernel where K % 128 == 0 and N % 128 == 0 (SWIGLU:
    (N/2) % 64 == 0), else the warp-MMA kernel.  Host-side planning only."""
    assert M.gemm_path(R, E, K, N, bits, group, act) == path

