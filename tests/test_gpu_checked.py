"""Out-of-range indices on the GPU, in the plain and in the bounds-checked build.

The inputs are made wrong on the host (expert ids outside [0, E), offsets that decrease,
permutation entries past the end); no kernel is made to fault.  The plain build drops rows
whose expert id is out of range and skips permutation entries outside [0, T*k); the checked
build (libmoe_checked.so, compiled with MOE_CHECKED=1) does the same and also reports each
kind of violation through moe_check_status, and a GEMM with unusable offsets computes
nothing.  Valid rows are unaffected in both."""
import ctypes

import pytest
import torch

from _helpers import have_gpu
from oracle import moe_oracle as O

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a CUDA GPU")]

DEV = "cuda:0"
ERR_DEVICE_CHECK = -5
BIT_ID, BIT_OFFSETS, BIT_PERM = 1, 2, 4


@pytest.fixture(scope="module")
def M():
    from weight_only_int4_route_gb300 import build, moe
    build.build()
    build.build(checked=True)
    moe.lib()
    moe.lib_checked()
    return moe


def _permute(M, L, ids, x, E):
    T, k = ids.shape
    d = x.shape[1]
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=DEV)
    perm = torch.full((T * k,), -7, dtype=torch.int32, device=DEV)
    inv = torch.full((T * k,), -7, dtype=torch.int32, device=DEV)
    xp = torch.zeros((T * k, d), dtype=x.dtype, device=DEV)
    ws = torch.empty(max(int(L.moe_permute_workspace_size(T, E, k)), 16), dtype=torch.uint8, device=DEV)
    st = L.moe_permute(M._ptr(ids), M._ptr(x), M._dt(x), T, d, E, k, M._ptr(offsets), M._ptr(perm), M._ptr(inv),
                       M._ptr(xp), M._ptr(ws), ws.numel(), M._stream(torch.device(DEV)))
    assert st == 0, L.moe_last_error_string()
    return offsets, perm, inv, xp


@pytest.mark.parametrize("T,k,E", [(40, 2, 8), (700, 3, 16)])   # one-CTA and tiled permute paths
@pytest.mark.parametrize("checked", [False, True])
def test_out_of_range_ids_are_dropped(M, T, k, E, checked):
    L = M.lib_checked() if checked else M.lib()
    gen = torch.Generator().manual_seed(T + k)
    ids = torch.randint(0, E, (T, k), generator=gen, dtype=torch.int32)
    bad = torch.rand((T, k), generator=gen) < 0.1
    ids[bad] = torch.where(torch.rand(int(bad.sum()), generator=gen) < 0.5, -3, E + 5).to(torch.int32)
    x = torch.randn((T, 256), generator=gen).to(torch.bfloat16)
    offsets, perm, inv, xp = _permute(M, L, ids.to(DEV), x.to(DEV), E)
    st, flags = M.check_status(DEV, L)
    if checked:
        assert st == ERR_DEVICE_CHECK and flags == BIT_ID
    else:
        assert st == 0 and flags == 0
    # valid rows: the stable sort of the valid ids alone
    flat = ids.flatten()
    valid = (flat >= 0) & (flat < E)
    nvalid = int(valid.sum())
    counts = torch.stack([(flat == e).sum() for e in range(E)]).to(torch.int32)
    roff = torch.zeros(E + 1, dtype=torch.int32)
    roff[1:] = torch.cumsum(counts, 0)
    rperm = torch.cat([(flat == e).nonzero().flatten() for e in range(E)]).to(torch.int32)
    assert torch.equal(offsets.cpu(), roff) and int(roff[E]) == nvalid
    assert torch.equal(perm.cpu()[:nvalid], rperm)
    inv_c = inv.cpu()
    assert bool((inv_c[~valid] == -1).all()), "dropped rows must have inv_perm == -1"
    assert torch.equal(inv_c[rperm.long()], torch.arange(nvalid, dtype=torch.int32))
    assert torch.equal(xp.cpu()[:nvalid], O.permute_rows(x, rperm, k))
    # the combine skips the dropped rows: with gate 1 and y = xp, token t gets the sum of its valid rows
    gate = torch.ones((T, k), device=DEV)
    out = torch.empty((T, 256), dtype=torch.float32, device=DEV)
    st = L.moe_unpermute_combine(M._ptr(xp), M._dt(xp), M._ptr(inv), M._ptr(gate), None, 2, T, 256, k, M._ptr(out),
                                 2, M._stream(torch.device(DEV)))
    assert st == 0
    ref = (x.double()[:, None, :] * valid.view(T, k, 1).double()).sum(1)
    assert torch.allclose(out.cpu().double(), ref, rtol=0, atol=1e-5)
    st, flags = M.check_status(DEV, L)
    assert (st, flags) == ((ERR_DEVICE_CHECK, BIT_PERM) if checked else (0, 0))


@pytest.mark.parametrize("R_rows,path_N", [(8, 256), (200, 256), (60, 192)])   # decode, tcgen05, warp-MMA kernels
def test_checked_gemm_rejects_unusable_offsets(M, R_rows, path_N):
    """Offsets that decrease or run past R: the checked GEMM computes nothing and reports it; the
    same GEMM with valid offsets reports nothing (no false positive)."""
    L = M.lib_checked()
    E, K, N = 4, 256, path_N
    R = 4 * R_rows
    gen = torch.Generator().manual_seed(R + N)
    q = torch.randint(-7, 8, (E, K, N), generator=gen, dtype=torch.int8)
    s = (torch.rand((E, 1, N), generator=gen) * 0.01 + 0.001).to(torch.float16)
    packed = M.pack_weights(q.to(DEV), s.to(DEV), 4, 0)
    a = torch.randn((R, K), generator=gen).to(torch.float16).to(DEV)
    sentinel = 12345.0
    for offs, expect in (([0, R_rows, 2 * R_rows, 3 * R_rows, R], 0),            # valid
                         ([0, 2 * R_rows, R_rows, 3 * R_rows, R], BIT_OFFSETS),   # decreasing
                         ([0, R_rows, 2 * R_rows, 3 * R_rows, R + 9], BIT_OFFSETS)):   # past R
        off = torch.tensor(offs, dtype=torch.int32, device=DEV)
        out = torch.full((R, N), sentinel, dtype=torch.float32, device=DEV)
        wsb = int(L.moe_grouped_gemm_workspace_size(R, E, K, N, 4, 0))
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=DEV)
        st = L.moe_grouped_gemm_w4a16(M._ptr(a), 0, M._ptr(packed), E, K, N, 0, M._ptr(off), R, 0, M._ptr(out), 2,
                                      M._ptr(ws), ws.numel(), M._stream(torch.device(DEV)))
        assert st == 0
        st, flags = M.check_status(DEV, L)
        assert flags == expect, (offs, flags)
        if expect:
            assert st == ERR_DEVICE_CHECK
            # split-K plans still run their reduction over the (never written) partials; every
            # single-pass kernel leaves the output untouched
            if wsb == 0:
                assert bool((out == sentinel).all())
        else:
            assert st == 0 and not bool((out == sentinel).any())
    assert M.device_error(DEV) == 0
