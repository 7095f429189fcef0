"""A whole decode step (every decode call, its selection and the final paths)
captured once in a CUDA graph and replayed gives the same bits as the same
calls made one by one: the library's calls on the step path only enqueue
work on the caller's stream, with sizes and pointers fixed at the call."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import synth
from gpu_util import DEV, decoder_for, device_status_clear, to_dev

pytestmark = pytest.mark.gpu

CASES = {
    # tensor-core paths (bf16, heads of 128), bias on the cumulative scores
    "gqa_w128": synth.GQA.with_(R=2, bias_var=4.0),
    # stacked layers with a residual stream
    "deep_small": synth.DEEP.with_(name="deep_small", R=2, W=(64, 128, 128, 128), L=256),
    # CUDA-core paths (fp32)
    "tiny_f32": synth.TINY,
}


@pytest.mark.parametrize("name", list(CASES))
def test_graph_replay_matches_eager_calls(name):
    wl = CASES[name]
    p = synth.make_params(wl)
    dec = decoder_for(wl, p)
    stream = torch.cuda.Stream(DEV)
    prompts = to_dev(synth.make_prompt(wl), torch.int32)
    bias = synth.make_bias(wl)
    biases = [to_dev(np.ascontiguousarray(bias[t, :, :wl.W[t]])) if bias is not None else None
              for t in range(wl.T - 1)]
    T = wl.T
    with torch.cuda.stream(stream):
        dec.prefill(prompts, stream=stream)
        root = dec.select(-1, 1, wl.W[0], dec.root_logits, dec.root_lse, stream=stream)
        outs = [tuple(torch.empty(wl.R, wl.W[s], dtype=d, device=DEV)
                      for d in (torch.int32, torch.int32, torch.float32)) for s in range(T)]
        sid = torch.empty(wl.R, wl.W[T - 1], T, dtype=torch.int32, device=DEV)

    def step(st):
        par, tok, cum = root
        for t in range(T - 1):
            lg, ls = dec.step(t, wl.W[t], par if t else None, tok, stream=st)
            par, tok, cum = dec.select(t, wl.W[t], wl.W[t + 1], lg, ls, cum, biases[t],
                                       out=outs[t + 1], stream=st)
        dec.get_paths(wl.W[T - 1], par, tok, sid=sid, stream=st)

    with torch.cuda.stream(stream):
        step(stream)
    torch.cuda.synchronize()
    assert dec.status(stream) == 0
    eager = [x.clone() for o in outs[1:] for x in o] + [sid.clone()]
    for o in outs[1:]:
        for x in o:
            x.fill_(-7)
    sid.fill_(-7)

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
        step(stream)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert device_status_clear() == 0
    replayed = [x for o in outs[1:] for x in o] + [sid]
    for a, b in zip(eager, replayed):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("name", list(CASES))
def test_serve_graph_matches_decode(name):
    # BeamDecoder.serve captures a whole batch (prompt upload, prefill, root
    # selection, decode calls, selections, paths and scores download) once per
    # shape and replays it: two batches of different prompts, served one
    # after the other, give bit for bit what an ordinary decode of each gives
    wl = CASES[name]
    p = synth.make_params(wl)
    dec = decoder_for(wl, p)
    bias = synth.make_bias(wl)
    bias_dev = to_dev(bias) if bias is not None else None
    rng = np.random.default_rng(5)
    batches = [synth.make_prompt(wl), rng.integers(0, wl.V, size=(wl.R, wl.L)).astype(np.int32)]
    expect = []
    for prompts in batches:
        dec.prefill(to_dev(prompts, torch.int32))
        res = dec.decode(wl.W, bias=bias_dev)
        torch.cuda.synchronize()
        assert dec.status() == 0
        expect.append((res.sid.cpu().clone(), res.cum[-1].cpu().clone()))
    for rep in range(2):  # first use (ordinary run, then capture), then replays
        for prompts, (sid_e, cum_e) in zip(batches, expect):
            sid, cum = dec.serve(torch.as_tensor(prompts), wl.W, bias_dev)
            assert torch.equal(sid, sid_e), (rep, "sid")
            assert torch.equal(cum.view(torch.int32), cum_e.view(torch.int32)), (rep, "cum")
    # the same batches served as ordinary calls
    for prompts, (sid_e, cum_e) in zip(batches, expect):
        sid, cum = dec.serve(torch.as_tensor(prompts), wl.W, bias_dev, graph=False)
        assert torch.equal(sid, sid_e) and torch.equal(cum.view(torch.int32), cum_e.view(torch.int32))
