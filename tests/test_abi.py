"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, and its host-side logic (configuration checks, memory accounting,
call sequencing, argument checks) behaves as documented. No kernel runs."""
import ctypes as C
import json
import os
import re

import pytest

import linear_attention_beam_gb300 as gb
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdnbeam.h")


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdnbeam_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_function():
    lib = gb.load()
    names = header_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    # and the binding declares a signature for each
    assert set(names) <= set(gb._SIGS)


def test_binding_constants_match_the_header():
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    vals = {k: int(v) for k, v in re.findall(r"\b(GDNBEAM_[A-Z0-9_]+)\s*=\s*(-?\d+)", src)}
    for name in ("OK", "EINVAL", "EUNSUPPORTED", "EWORKSPACE", "ESTATE", "ECUDA", "EDEVICE", "ENOMEM",
                 "F32", "BF16", "DERR_TOKEN", "DERR_PARENT", "DERR_SLOT", "DERR_NONFINITE",
                 "DERR_TIMEOUT", "DERR_SELECT"):
        assert vals["GDNBEAM_" + name] == getattr(gb, name), name


def cfg(wl, **kw):
    d = dict(R=wl.R, layers=wl.layers, H=wl.H, d_k=wl.d_k, d_v=wl.d_v, d_model=wl.d_model, V=wl.V,
             T=wl.T, W_max=wl.W_max, L_max=wl.L, dtype=gb.BF16 if wl.dtype == "bf16" else gb.F32,
             residual=int(wl.residual), H_k=wl.Hk)
    d.update(kw)
    return gb.Config(**d)


def footprint(c):
    f = gb.Footprint()
    st = gb.load().gdnbeam_footprint_of(C.byref(c), C.byref(f))
    return st, f


@pytest.mark.parametrize("wl", list(synth.WORKLOADS.values()), ids=list(synth.WORKLOADS))
def test_every_workload_is_accepted(wl):
    st, f = footprint(cfg(wl))
    assert st == 0 and f.workspace_bytes > 0


def test_record_size_and_capacity_match_the_page():
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "onela_record_sizes.json")))
    # one request, one layer, one head, d = 128, W = 512, T = 2 decode calls (3 selections)
    c = gb.Config(R=1, layers=1, H=1, d_k=128, d_v=128, d_model=128, V=1024, T=3, W_max=512,
                  L_max=16, dtype=gb.BF16, residual=0)
    st, f = footprint(c)
    assert st == 0
    assert f.record_elements == g["gtr_elements"]
    # S_ctx: one fp32 d_v x d_k state for the request and head
    assert f.sctx_bytes == 4 * g["fullstate_elements"]
    W, Tdec = 512, 2
    elems = W * 128 * 128 / (128 * 128 + W * Tdec * f.record_elements)
    assert abs(elems - g["capacity_ratio_W512_T2_approx"]) < 1.0
    # bytes as laid out: bf16 vectors plus an fp32 decay per record; a
    # FullState decoder would hold one bf16 state per beam
    assert f.records_bytes == Tdec * W * (2 * (128 + 128) + 4)
    assert f.fullstate_bytes == W * 2 * g["fullstate_elements"]
    ratio_bytes = f.fullstate_bytes / (f.sctx_bytes + f.records_bytes)
    assert 25 < ratio_bytes < g["capacity_ratio_W512_T2_approx"]


@pytest.mark.parametrize("field,value,status", [
    ("d_k", 96, gb.EUNSUPPORTED), ("d_k", 512, gb.EUNSUPPORTED), ("d_v", 1024, gb.EUNSUPPORTED),
    ("T", 9, gb.EUNSUPPORTED),
    ("V", 20000, gb.EUNSUPPORTED), ("layers", 2, gb.EUNSUPPORTED), ("dtype", 7, gb.EUNSUPPORTED),
    ("R", 0, gb.EINVAL), ("W_max", 0, gb.EINVAL), ("V", 1, gb.EINVAL), ("state_path", 3, gb.EUNSUPPORTED),
    ("state_path", -1, gb.EUNSUPPORTED)])
def test_config_rejections(field, value, status):
    c = cfg(synth.TINY)
    setattr(c, field, value)
    assert footprint(c)[0] == status


def test_wide_heads_are_accepted_on_the_replay_path_only():
    for dk, dv in ((256, 256), (128, 512), (256, 512)):
        assert footprint(cfg(synth.TINY, d_k=dk, d_v=dv, d_model=dv))[0] == 0
        for sp in (1, 2):  # the baselines keep whole states on chip
            assert footprint(cfg(synth.TINY, d_k=dk, d_v=dv, d_model=dv, state_path=sp))[0] == gb.EUNSUPPORTED


def test_state_path_workspaces():
    # FullState keeps two per-beam state buffers; ReplaySSM only a storage copy
    # of S_ctx beside the records; the replay path neither
    wl = synth.BATCHED
    sizes = [footprint(cfg(wl, state_path=sp))[1].workspace_bytes for sp in (0, 1, 2)]
    per_beam_states = wl.R * wl.W_max * wl.layers * wl.H * wl.d_v * wl.d_k * 2
    sctx_copy = wl.R * wl.layers * wl.H * wl.d_v * wl.d_k * 2
    assert sizes[1] - sizes[0] >= 2 * per_beam_states + sctx_copy
    assert sctx_copy <= sizes[2] - sizes[0] < sctx_copy + (1 << 20)


def test_residual_needs_matching_width():
    c = cfg(synth.DEEP, d_model=1000)
    assert footprint(c)[0] == gb.EUNSUPPORTED


FAKE_WS = 1 << 40  # never dereferenced by the host-side checks below


def make_ctx(wl=synth.TINY):
    lib = gb.load()
    c = cfg(wl)
    st, f = footprint(c)
    w = gb.Weights(E=FAKE_WS, W_proj=FAKE_WS, W_o=FAKE_WS)
    h = C.c_void_p()
    assert lib.gdnbeam_create(C.byref(c), C.byref(w), FAKE_WS, f.workspace_bytes, C.byref(h)) == 0
    return lib, h, f


def test_create_checks_workspace():
    lib = gb.load()
    c = cfg(synth.TINY)
    _, f = footprint(c)
    w = gb.Weights(E=FAKE_WS, W_proj=FAKE_WS, W_o=FAKE_WS)
    h = C.c_void_p()
    assert lib.gdnbeam_create(C.byref(c), C.byref(w), FAKE_WS, f.workspace_bytes - 1, C.byref(h)) == gb.EWORKSPACE
    assert not h.value
    assert lib.gdnbeam_create(C.byref(c), C.byref(w), FAKE_WS + 8, f.workspace_bytes, C.byref(h)) == gb.EINVAL
    assert lib.gdnbeam_create(C.byref(c), None, FAKE_WS, f.workspace_bytes, C.byref(h)) == gb.EINVAL


def test_call_sequence_is_enforced_on_the_host():
    lib, h, _ = make_ctx()
    tok = FAKE_WS
    # decode before prefill
    assert lib.gdnbeam_step(h, 0, 8, None, tok, FAKE_WS, FAKE_WS, None, None) == gb.ESTATE
    # out-of-range call index, beam count, missing parents
    assert lib.gdnbeam_step(h, 2, 8, None, tok, FAKE_WS, FAKE_WS, None, None) == gb.EINVAL
    assert lib.gdnbeam_step(h, 0, 9, None, tok, FAKE_WS, FAKE_WS, None, None) == gb.EINVAL
    assert lib.gdnbeam_step(h, 1, 8, None, tok, FAKE_WS, FAKE_WS, None, None) == gb.EINVAL
    assert lib.gdnbeam_prefill_state(h, FAKE_WS, 33, FAKE_WS, FAKE_WS, None) == gb.EINVAL  # L > L_max
    assert lib.gdnbeam_read_sctx(h, FAKE_WS, None) == gb.ESTATE
    assert lib.gdnbeam_get_paths(h, 8, FAKE_WS, FAKE_WS, FAKE_WS, None) == gb.ESTATE
    # selection arguments
    assert lib.gdnbeam_select(h, -1, 2, 8, FAKE_WS, FAKE_WS, None, None, FAKE_WS, FAKE_WS, FAKE_WS, None) == gb.EINVAL
    assert lib.gdnbeam_select(h, 0, 8, 9, FAKE_WS, FAKE_WS, None, None, FAKE_WS, FAKE_WS, FAKE_WS, None) == gb.EINVAL
    assert lib.gdnbeam_select(h, 5, 8, 8, FAKE_WS, FAKE_WS, None, None, FAKE_WS, FAKE_WS, FAKE_WS, None) == gb.EINVAL
    assert lib.gdnbeam_reset(h, None) == 0
    assert "select=" in lib.gdnbeam_variant(h).decode()
    lib.gdnbeam_destroy(h)


def test_select_topw_argument_checks():
    lib = gb.load()
    sb = lib.gdnbeam_select_scratch_bytes(2, 4, 3, 10)
    assert sb >= 2 * 4 * 3 * 8  # at least the per-row precut keys of the exact fallback
    a = FAKE_WS
    assert lib.gdnbeam_select_topw(2, 4, 3, 10, gb.BF16, a, a, None, None, a, a, a, a, sb - 1, None) == gb.EWORKSPACE
    assert lib.gdnbeam_select_topw(2, 1, 11, 10, gb.BF16, a, a, None, None, a, a, a, a, 10 ** 9, None) == gb.EINVAL
    assert lib.gdnbeam_select_topw(2, 4, 3, 10, 5, a, a, None, None, a, a, a, a, sb, None) == gb.EUNSUPPORTED


def test_strerror():
    lib = gb.load()
    assert lib.gdnbeam_strerror(gb.ESTATE).decode() == "call out of sequence"


def test_hot_path_uses_tensor_core_kernels():
    lib, h, _ = make_ctx(synth.BATCHED)
    v = lib.gdnbeam_variant(h).decode()
    assert "proj=tc" in v and "logits=tc" in v, v
    lib.gdnbeam_destroy(h)
    lib, h, _ = make_ctx(synth.TINY)
    assert "proj=simt" in lib.gdnbeam_variant(h).decode()
    lib.gdnbeam_destroy(h)


def test_per_request_reset_and_prefill_argument_checks():
    # three requests: releasing one blocks decoding until it is prefilled
    # again; bad request lists are refused before anything is launched
    wl = synth.TINY.with_(R=3)
    lib, h, _ = make_ctx(wl)
    i32 = lambda *v: (C.c_int32 * len(v))(*v)
    mask = i32(0, 1, 0)
    assert lib.gdnbeam_reset(h, mask) == 0
    assert lib.gdnbeam_step(h, 0, 8, None, FAKE_WS, FAKE_WS, FAKE_WS, None, None) == gb.ESTATE
    assert lib.gdnbeam_read_sctx(h, FAKE_WS, None) == gb.ESTATE
    pr = lambda ids, n, L=8: lib.gdnbeam_prefill_requests(h, ids, n, FAKE_WS, L, FAKE_WS, FAKE_WS, None)
    assert pr(i32(1), 0) == 0                 # nothing to do
    assert pr(i32(3), 1) == gb.EINVAL         # id out of range
    assert pr(i32(-1), 1) == gb.EINVAL
    assert pr(i32(1, 1), 2) == gb.EINVAL      # listed twice
    assert pr(i32(0, 1, 2, 0), 4) == gb.EINVAL  # more ids than requests
    assert pr(i32(1), 1, L=33) == gb.EINVAL   # L > L_max
    assert pr(None, 1) == gb.EINVAL
    assert lib.gdnbeam_prefill_requests(h, i32(1), 1, None, 8, FAKE_WS, FAKE_WS, None) == gb.EINVAL
    assert lib.gdnbeam_reset(None, None) == gb.EINVAL
    lib.gdnbeam_destroy(h)
