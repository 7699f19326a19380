"""CUDA-graph capture of the attention calls.

The window + tail call forks the handle's copy stream off the capturing
stream with an event and joins it back through the copy_done / compute_done
events, so the whole call -- host-to-device tile copies, decode launches,
combine -- records into one graph.  Scratch is grown by an eager call first
(growth during capture is refused with SKV_ECAPTURE, also checked here).
Replays must reproduce the eager results bit for bit, also after the inputs
change in place."""
import numpy as np
import pytest

from split_kv_flash_attn_gb300 import workloads as wl
from tests.gpu_util import dev, pinned

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import split_kv_flash_attn_gb300 as m
    return m


def _capture(torch, fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        fn()
    return g


@pytest.mark.parametrize("quant", [False, True])
def test_window_tail_graph_replay(skv, quant):
    import torch
    h = skv.Handle(0)
    if quant:
        w = wl.long_context_decode(n_kv=5000, wc=1000, tile_rows=1024, H=40, Hk=8, D=128)
    else:
        w = wl.tiny_decode()
    q, kw, vw = dev(w.q), dev(w.k), dev(w.v)
    kt, vt = pinned(w.k_tail), pinned(w.v_tail)
    o = torch.empty((w.S, w.nq, w.H, w.D), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.S, w.nq, w.H), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def call():
        skv.attn_window_tail(h, q, kw, vw, kt, vt, Hk=w.Hk, tile_rows=w.tile_rows, k_type=w.k_type,
                             v_type=w.v_type, o=o, lse=lse, stream=s)

    with torch.cuda.stream(s):
        call()                                   # eager: grows the workspace and the ring
    torch.cuda.synchronize()
    o_ref, l_ref = o.clone(), lse.clone()
    g = _capture(torch, call, s)
    o.zero_()
    lse.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    # new inputs in place (query and pinned tail): the replay reads them
    q.copy_(torch.flip(q, dims=[2]))
    kt.copy_(torch.roll(kt, 1, dims=0))
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    o_new, l_new = o.clone(), lse.clone()
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_new) and torch.equal(lse, l_new)
    assert not torch.equal(o_new, o_ref)
    h.close()


def test_decode_and_prefill_graph_replay(skv):
    import torch
    h = skv.Handle(0)
    w = wl.unified_decode(n_cache=8192, S=4, rows_per_seq=1500, H=32, Hk=8, D=128, salt=4)
    q, k, v, rows = dev(w.q), dev(w.k), dev(w.v), dev(w.kv_rows)
    p = wl.prefill_chunk(n_kv=2048, wc=2048, nq=64, H=32, Hk=8, D=128)
    pq, pk, pv, pp = dev(p.q), dev(p.k), dev(p.v), dev(p.q_pos)
    s = torch.cuda.Stream()
    outs = {}

    def call():
        outs["d"] = skv.attn_partial(h, q, k, v, Hk=8, kv_rows=rows, o=outs["d"][0], lse=outs["d"][1], stream=s)
        outs["p"] = skv.attn_partial(h, pq, pk, pv, Hk=8, q_pos=pp, o=outs["p"][0], lse=outs["p"][1], stream=s)

    outs["d"] = (torch.empty((4, 1, 32, 128), device="cuda"), torch.empty((4, 1, 32), device="cuda"))
    outs["p"] = (torch.empty((1, 64, 32, 128), device="cuda"), torch.empty((1, 64, 32), device="cuda"))
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    ref = {k_: (a.clone(), b.clone()) for k_, (a, b) in outs.items()}
    g = _capture(torch, call, s)
    for a, b in outs.values():
        a.zero_()
        b.zero_()
    g.replay()
    torch.cuda.synchronize()
    for k_ in outs:
        assert torch.equal(outs[k_][0], ref[k_][0]) and torch.equal(outs[k_][1], ref[k_][1]), k_
    assert h.status() == 0
    h.close()


def test_growth_during_capture_is_refused(skv):
    import torch
    h = skv.Handle(0)                            # fresh handle: no workspace yet
    w = wl.unified_decode(n_cache=8192, S=4, rows_per_seq=1500, H=32, Hk=8, D=128, salt=5)
    q, k, v, rows = dev(w.q), dev(w.k), dev(w.v), dev(w.kv_rows)
    s = torch.cuda.Stream()
    errors = []

    def call():
        try:
            skv.attn_partial(h, q, k, v, Hk=8, kv_rows=rows, stream=s)
        except skv.SplitKVError as e:
            errors.append(e.status)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
        call()
    assert errors == [5]                         # SKV_ECAPTURE
    h.close()
