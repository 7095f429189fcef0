"""The allocation-free selection entry point against the regular one.

gdnbeam_select_topw_noalloc serves callers that cannot hand the library a
scratch buffer (a plugin given only its input and output tensors, a process
whose device memory another allocator has reserved); it runs the same
selection on a fixed area inside the library. Two calls in a row, on
different inputs, must give exactly what gdnbeam_select_topw gives with a
caller-provided buffer — the area keeps the previous call's contents, so the
second call checks that nothing leaks from one call into the next.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import linear_attention_beam_gb300 as gb

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _inputs(seed, R, W_t, V, dtype):
    g = torch.Generator(device=DEV).manual_seed(seed)
    td = torch.bfloat16 if dtype == gb.BF16 else torch.float32
    z = (torch.randn(R * W_t, V, generator=g, device=DEV) * 2).to(td)
    z[:, ::7] = z[:, :1]  # ties inside rows
    lse = torch.logsumexp(z.float(), dim=1).contiguous()
    cum = torch.randn(R * W_t, generator=g, device=DEV)
    bias = torch.randn(R * W_t, generator=g, device=DEV)
    return z.contiguous(), lse, cum, bias


def _outputs(R, W_next):
    return (torch.empty(R, W_next, dtype=torch.int32, device=DEV),
            torch.empty(R, W_next, dtype=torch.int32, device=DEV),
            torch.empty(R, W_next, dtype=torch.float32, device=DEV))


@pytest.mark.parametrize("R,W_t,W_next,V,dtype", [(4, 512, 512, 8192, gb.BF16), (3, 37, 64, 513, gb.F32)])
def test_noalloc_selection_matches_the_scratch_version_twice(R, W_t, W_next, V, dtype):
    lib = gb.load()
    assert lib.gdnbeam_select_scratch_bytes(R, W_t, W_next, V) <= lib.gdnbeam_select_noalloc_max_bytes()
    scratch = torch.empty(lib.gdnbeam_select_scratch_bytes(R, W_t, W_next, V), dtype=torch.uint8, device=DEV)
    for call in range(2):
        z, lse, cum, bias = _inputs(100 + call, R, W_t, V, dtype)
        b = bias if call == 1 else None
        ref = _outputs(R, W_next)
        got = _outputs(R, W_next)
        assert lib.gdnbeam_select_topw(R, W_t, W_next, V, dtype, gb.ptr(z), gb.ptr(lse), gb.ptr(cum), gb.ptr(b),
                                       gb.ptr(ref[0]), gb.ptr(ref[1]), gb.ptr(ref[2]), gb.ptr(scratch),
                                       scratch.numel(), None) == 0
        assert lib.gdnbeam_select_topw_noalloc(R, W_t, W_next, V, dtype, gb.ptr(z), gb.ptr(lse), gb.ptr(cum),
                                               gb.ptr(b), gb.ptr(got[0]), gb.ptr(got[1]), gb.ptr(got[2]),
                                               None) == 0
        torch.cuda.synchronize()
        assert lib.gdnbeam_device_status(1) == 0
        for a, c in zip(ref, got):
            np.testing.assert_array_equal(a.cpu().numpy(), c.cpu().numpy())


def test_noalloc_selection_refuses_oversized_calls():
    lib = gb.load()
    R, W_t, W_next, V = 64, 512, 512, 8192  # needs far more than the fixed area
    assert lib.gdnbeam_select_scratch_bytes(R, W_t, W_next, V) > lib.gdnbeam_select_noalloc_max_bytes()
    z = torch.zeros(1, dtype=torch.bfloat16, device=DEV)
    f = torch.zeros(1, device=DEV)
    i = torch.zeros(1, dtype=torch.int32, device=DEV)
    st = lib.gdnbeam_select_topw_noalloc(R, W_t, W_next, V, gb.BF16, gb.ptr(z), gb.ptr(f), None, None,
                                         gb.ptr(i), gb.ptr(i), gb.ptr(f), None)
    assert st == gb.EWORKSPACE


@pytest.mark.parametrize("dtype", [gb.BF16, gb.F32])
def test_noalloc_selection_after_the_exact_fallback(dtype):
    # all-equal logits overflow the on-chip candidate buffer and take the
    # two-stage exact path, which leaves its flags in the shared area; the
    # next call, on ordinary inputs, must not be steered by them
    lib = gb.load()
    R, W_t, W_next, V = 2, 64, 5, 100
    scratch = torch.empty(lib.gdnbeam_select_scratch_bytes(R, W_t, W_next, V), dtype=torch.uint8, device=DEV)
    td = torch.bfloat16 if dtype == gb.BF16 else torch.float32
    ties = (torch.zeros(R * W_t, V, dtype=td, device=DEV), torch.zeros(R * W_t, device=DEV),
            torch.zeros(R * W_t, device=DEV), None)
    for call, (z, lse, cum, b) in enumerate([ties, _inputs(7, R, W_t, V, dtype), ties]):
        ref = _outputs(R, W_next)
        got = _outputs(R, W_next)
        assert lib.gdnbeam_select_topw(R, W_t, W_next, V, dtype, gb.ptr(z), gb.ptr(lse), gb.ptr(cum), gb.ptr(b),
                                       gb.ptr(ref[0]), gb.ptr(ref[1]), gb.ptr(ref[2]), gb.ptr(scratch),
                                       scratch.numel(), None) == 0
        assert lib.gdnbeam_select_topw_noalloc(R, W_t, W_next, V, dtype, gb.ptr(z), gb.ptr(lse), gb.ptr(cum),
                                               gb.ptr(b), gb.ptr(got[0]), gb.ptr(got[1]), gb.ptr(got[2]),
                                               None) == 0
        torch.cuda.synchronize()
        assert lib.gdnbeam_device_status(1) == 0
        for a, c in zip(ref, got):
            np.testing.assert_array_equal(a.cpu().numpy(), c.cpu().numpy())
        if call != 1:  # every candidate ties: the lowest flat indices win
            for r in range(R):
                np.testing.assert_array_equal(got[0][r].cpu().numpy(), [0] * 5)
                np.testing.assert_array_equal(got[1][r].cpu().numpy(), [0, 1, 2, 3, 4])
