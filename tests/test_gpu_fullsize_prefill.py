"""Parity of the tensor-core prefill path at the sizes bench.py times.

* The prefill chunk: 512 causal tokens at positions 65024..65535 x 32 heads
  over 65536 fp16 keys (32768 in device memory + a 32768-row pinned tail in
  8192-row tiles).  All 512 x 32 rows (every KV head, all 128 query tiles)
  against the oracle, and against the split-KV decode kernel (one query token
  per sequence, 512 sequences, the same keys and causal positions).
* The same shape over q8_0-K / q4_0-V rows (32768 rows on the device): every
  token of KV heads 0 and 7 against the oracle.
* Row-list prefill over the unified cache: 8 sequences x 64 tokens, each over
  its own 32768-row list of the 262144-row fp16 cache: every token of KV heads
  0 and 7 against the oracle.
The oracle works one KV head group at a time (the cache cut down to that
head's columns), which keeps each check to seconds of CPU time."""
import numpy as np
import pytest

from split_kv_flash_attn_gb300 import workloads as wl
from tests.gpu_util import check_attention, dev, head_columns, oracle_one_head, pinned, vmax_of

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

HEADS = (0, 7)


@pytest.fixture(scope="module")
def skv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import split_kv_flash_attn_gb300 as m
    return m


@pytest.fixture(scope="module")
def h(skv):
    return skv.Handle(0)


def _check_heads(oracle_mod, w, o, l, heads, k_type, v_type, what, **regions_and_keys):
    G = w.H // w.Hk
    o = o.cpu()
    l = l.cpu()
    sv = wl.segment_bytes(v_type, w.D)
    for kh in heads:
        want_o, want_l = oracle_one_head(oracle_mod, w, kh, k_type=k_type, v_type=v_type, **regions_and_keys)
        vs = [regions_and_keys["v0"]] + ([regions_and_keys["v1"]] if regions_and_keys.get("v1") is not None else [])
        vmax = max(vmax_of(oracle_mod, v_type, head_columns(v, kh, sv), w.D) for v in vs)
        check_attention(o[:, :, kh * G:(kh + 1) * G], l[:, :, kh * G:(kh + 1) * G], want_o, want_l, vmax,
                        f"{what}, KV head {kh}")


def test_prefill_chunk_full_size(skv, h, oracle_mod):
    import torch
    w = wl.prefill_chunk()
    o, l = skv.attn_window_tail(h, dev(w.q), dev(w.k), dev(w.v), pinned(w.k_tail), pinned(w.v_tail), Hk=w.Hk,
                                tile_rows=w.tile_rows, q_pos=dev(w.q_pos))
    torch.cuda.synchronize()
    assert h.status() == 0
    _check_heads(oracle_mod, w, o, l, range(w.Hk), wl.F16, wl.F16, "prefill chunk", k0=w.k, v0=w.v, k1=w.k_tail,
                 v1=w.v_tail, n_keys=w.n_keys, q_pos=w.q_pos)

    # every token through the decode kernel: token t becomes sequence t with
    # one query token at its own causal position, over the same 65536 keys
    K = dev(np.concatenate([w.k, w.k_tail]))
    V = dev(np.concatenate([w.v, w.v_tail]))
    q_tok = dev(w.q.reshape(w.nq, 1, w.H, w.D))
    pos_tok = dev(w.q_pos.reshape(w.nq, 1))
    o_dec, l_dec = skv.attn_partial(h, q_tok, K, V, Hk=w.Hk, q_pos=pos_tok)
    torch.cuda.synchronize()
    vmax = float(np.abs(np.concatenate([w.v, w.v_tail]).view(np.float16)).max())
    check_attention(o.reshape(w.nq, 1, w.H, w.D), l.reshape(w.nq, 1, w.H),
                    o_dec.cpu().numpy().astype(np.float64), l_dec.cpu().numpy().astype(np.float64), vmax,
                    "prefill chunk vs decode kernel, every token and head")
    assert h.status() == 0


def test_prefill_quant_window_full_size(skv, h, oracle_mod):
    import torch
    w = wl.prefill_quant_window()
    o, l = skv.attn_partial(h, dev(w.q), dev(w.k), dev(w.v), Hk=w.Hk, k_type=w.k_type, v_type=w.v_type,
                            q_pos=dev(w.q_pos))
    torch.cuda.synchronize()
    assert h.status() == 0
    _check_heads(oracle_mod, w, o, l, HEADS, w.k_type, w.v_type, "q8_0/q4_0 prefill", k0=w.k, v0=w.v,
                 n_keys=w.n_keys, q_pos=w.q_pos)


def test_prefill_row_lists_full_size(skv, h, oracle_mod):
    import torch
    w = wl.prefill_row_lists()
    o, l = skv.attn_partial(h, dev(w.q), dev(w.k), dev(w.v), Hk=w.Hk, kv_rows=dev(w.kv_rows), q_pos=dev(w.q_pos))
    torch.cuda.synchronize()
    assert h.status() == 0
    _check_heads(oracle_mod, w, o, l, HEADS, wl.F16, wl.F16, "row-list prefill", k0=w.k, v0=w.v, n_keys=w.n_keys,
                 kv_rows=w.kv_rows, q_pos=w.q_pos)
