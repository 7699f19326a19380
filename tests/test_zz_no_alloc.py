"""skv_attn_partial_static: decode attention that allocates nothing.

For callers that cannot call cudaMalloc (an engine serving all device memory
from a pool it reserved up front, a path that cannot take the synchronisation
an allocation may cause, or code without a library handle), the library offers
this one entry point whose scratch is a fixed array in device global memory.

The test calls it through the C ABI:
* twice in a row -- a row-list decode with fp16 rows, then a dense decode with
  q8_0/q4_0 rows, both split across many CTAs so the fixed scratch is used and
  reused -- and compares each result with the fp64 oracle and with
  skv_attn_partial's on the same inputs, within the attention tolerance of the
  other GPU tests;
* on a short range that plans a single split (o/lse written directly, no
  scratch touched), and on many query rows whose planned split partials would
  not fit the array (the call re-plans to fewer splits), both against the
  oracle;
* with more units than the array's stated maximum: SKV_ENOMEM, nothing run.
It is self-contained so it passes alone in a fresh process as well as after
the rest of the suite (this file is collected last)."""
import ctypes

import numpy as np
import pytest

from split_kv_flash_attn_gb300 import workloads as wl
from tests.gpu_util import check_attention, dev, vmax_of

pytestmark = pytest.mark.gpu

SKV_ENOMEM = 4


def _call_static(skv, lib, q, k, v, Hk, k_type, v_type, kv_rows=None, n_keys=None, expect=0):
    import torch
    S, nq, H, D = (int(x) for x in q.shape)
    sh = skv.SkvShape(S, nq, H, Hk, D, 1.0 / np.sqrt(D), k_type, v_type,
                      Hk * skv.segment_bytes(k_type, D), Hk * skv.segment_bytes(v_type, D))
    o = torch.full((S, nq, H, D), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((S, nq, H), float("nan"), dtype=torch.float32, device="cuda")
    if n_keys is None:
        n_keys = int(kv_rows.shape[-1]) if kv_rows is not None else int(k.shape[0])
    rows_ld = int(kv_rows.shape[-1]) if kv_rows is not None else 0
    rc = lib.skv_attn_partial_static(ctypes.byref(sh), q.data_ptr(), k.data_ptr(), v.data_ptr(), None, 0, None, 0,
                                     kv_rows.data_ptr() if kv_rows is not None else None, rows_ld, 0, 0, n_keys,
                                     o.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == expect, f"skv_attn_partial_static returned {rc}, expected {expect}"
    return o, lse


def _oracle_dense(oracle_mod, q, K, V, Hk, k_type, v_type, n_keys=None):
    D = q.shape[-1]
    return oracle_mod.attention(q, D=D, H=q.shape[2], Hk=Hk, scale=1.0 / np.sqrt(D), k_type=k_type, v_type=v_type,
                                k0=K, v0=V, n_rows0=K.shape[0], k_row_bytes0=K.shape[1], v_row_bytes0=V.shape[1],
                                n_keys=K.shape[0] if n_keys is None else n_keys)


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import split_kv_flash_attn_gb300 as skv
    from split_kv_flash_attn_gb300 import _lib
    return skv, _lib.lib()


def test_static_scratch_twice_against_oracle_and_attn_partial(env, oracle_mod):
    import torch
    skv, lib = env
    h = skv.Handle(0)

    # call 1: fp16 unified cache through row lists (with padding)
    w = wl.unified_decode(n_cache=16384, S=8, rows_per_seq=1900, H=32, Hk=8, D=128, salt=9)
    q, k, v, rows = dev(w.q), dev(w.k), dev(w.v), dev(w.kv_rows)
    o1, l1 = _call_static(skv, lib, q, k, v, w.Hk, wl.F16, wl.F16, kv_rows=rows)

    # call 2, right after: dense q8_0 K / q4_0 V rows, a different split plan
    rng = wl.generator(3, salt=21)
    q2 = wl.normal_f16(rng, (1, 1, 40, 128))
    K2 = wl.cache_rows(rng, wl.Q8_0, 6000, 8, 128)
    V2 = wl.cache_rows(rng, wl.Q4_0, 6000, 8, 128)
    q2d, k2d, v2d = dev(q2), dev(K2), dev(V2)
    o2, l2 = _call_static(skv, lib, q2d, k2d, v2d, 8, wl.Q8_0, wl.Q4_0)
    torch.cuda.synchronize()

    want1 = oracle_mod.attention(w.q, D=w.D, H=w.H, Hk=w.Hk, scale=w.scale, k0=w.k, v0=w.v, n_rows0=w.k.shape[0],
                                 k_row_bytes0=w.k.shape[1], v_row_bytes0=w.v.shape[1], n_keys=w.n_keys,
                                 kv_rows=w.kv_rows)
    vmax1 = vmax_of(oracle_mod, wl.F16, w.v, w.D)
    check_attention(o1, l1, *want1, vmax1, "static call 1 vs oracle")
    want2 = _oracle_dense(oracle_mod, q2, K2, V2, 8, wl.Q8_0, wl.Q4_0)
    vmax2 = vmax_of(oracle_mod, wl.Q4_0, V2, 128)
    check_attention(o2, l2, *want2, vmax2, "static call 2 vs oracle")

    # the same inputs through the handle's entry point
    r1o, r1l = skv.attn_partial(h, q, k, v, Hk=w.Hk, kv_rows=rows)
    r2o, r2l = skv.attn_partial(h, q2d, k2d, v2d, Hk=8, k_type=wl.Q8_0, v_type=wl.Q4_0)
    torch.cuda.synchronize()
    check_attention(o1, l1, r1o.cpu().numpy().astype(np.float64), r1l.cpu().numpy().astype(np.float64), vmax1,
                    "static call 1 vs skv_attn_partial")
    check_attention(o2, l2, r2o.cpu().numpy().astype(np.float64), r2l.cpu().numpy().astype(np.float64), vmax2,
                    "static call 2 vs skv_attn_partial")
    h.close()


def test_static_scratch_single_split_and_replanned(env, oracle_mod):
    skv, lib = env
    rng = wl.generator(1, salt=33)
    # one 64-key tile: a single split, written straight to o/lse
    q = wl.normal_f16(rng, (1, 1, 4, 64))
    K = wl.cache_rows(rng, wl.F16, 64, 1, 64)
    V = wl.cache_rows(rng, wl.F16, 64, 1, 64)
    o, l = _call_static(skv, lib, dev(q), dev(K), dev(V), 1, wl.F16, wl.F16)
    check_attention(o, l, *_oracle_dense(oracle_mod, q, K, V, 1, wl.F16, wl.F16), vmax_of(oracle_mod, wl.F16, V, 64),
                    "single split")
    # 64 tokens x 32 heads x 4 sequences = 8192 query rows of 512 B: every
    # split's partials take 4 MiB, so the planned split count is cut to fit
    qm = wl.normal_f16(rng, (4, 64, 32, 128))
    Km = wl.cache_rows(rng, wl.F16, 4096, 8, 128)
    Vm = wl.cache_rows(rng, wl.F16, 4096, 8, 128)
    o, l = _call_static(skv, lib, dev(qm), dev(Km), dev(Vm), 8, wl.F16, wl.F16)
    check_attention(o, l, *_oracle_dense(oracle_mod, qm, Km, Vm, 8, wl.F16, wl.F16),
                    vmax_of(oracle_mod, wl.F16, Vm, 128), "re-planned splits")


def test_static_scratch_rejects_units_beyond_maximum(env):
    import torch
    skv, lib = env
    # 1024 sequences x 8 KV heads x one 8-column group = 8192 units > 4096
    q = torch.zeros((1024, 1, 32, 128), dtype=torch.float16, device="cuda")
    kv = torch.zeros((256, 8 * 128), dtype=torch.float16, device="cuda")
    o, l = _call_static(skv, lib, q, kv, kv, 8, wl.F16, wl.F16, n_keys=256, expect=SKV_ENOMEM)
    torch.cuda.synchronize()
    assert torch.isnan(o).all() and torch.isnan(l).all(), "a rejected call must not write its outputs"
