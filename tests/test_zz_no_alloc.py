"""skv_attn_partial_static: decode attention that allocates nothing.

For callers that cannot call cudaMalloc (an engine serving all device memory
from a pool it reserved up front, a path that cannot take the synchronisation
an allocation may cause, or code without a library handle), the library offers
this one entry point whose scratch is a fixed array in device global memory.

The test calls it through the C ABI twice in a row -- a row-list decode with
fp16 rows, then a dense decode with q8_0/q4_0 rows, both split across many
CTAs so the fixed scratch is used and reused -- and compares each result with
skv_attn_partial's on the same inputs, within the attention tolerance of the
other GPU tests.  It is self-contained so it passes alone in a fresh process
as well as after the rest of the suite (this file is collected last)."""
import ctypes

import numpy as np
import pytest

from split_kv_flash_attn_gb300 import workloads as wl
from tests.gpu_util import check_attention, dev, vmax_of

pytestmark = pytest.mark.gpu


def _call_static(skv, lib, q, k, v, Hk, k_type, v_type, kv_rows=None):
    import torch
    S, nq, H, D = (int(x) for x in q.shape)
    sh = skv.SkvShape(S, nq, H, Hk, D, 1.0 / np.sqrt(D), k_type, v_type,
                      Hk * skv.segment_bytes(k_type, D), Hk * skv.segment_bytes(v_type, D))
    o = torch.full((S, nq, H, D), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((S, nq, H), float("nan"), dtype=torch.float32, device="cuda")
    n_keys = int(kv_rows.shape[-1]) if kv_rows is not None else int(k.shape[0])
    rows_ld = n_keys if kv_rows is not None else 0
    rc = lib.skv_attn_partial_static(ctypes.byref(sh), q.data_ptr(), k.data_ptr(), v.data_ptr(), None, 0, None, 0,
                                     kv_rows.data_ptr() if kv_rows is not None else None, rows_ld, 0, 0, n_keys,
                                     o.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, f"skv_attn_partial_static returned {rc}"
    return o, lse


def test_static_scratch_matches_attn_partial_twice(oracle_mod):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import split_kv_flash_attn_gb300 as skv
    from split_kv_flash_attn_gb300 import _lib
    lib = _lib.lib()
    h = skv.Handle(0)

    # call 1: fp16 unified cache through row lists (with padding)
    w = wl.unified_decode(n_cache=16384, S=8, rows_per_seq=1900, H=32, Hk=8, D=128, salt=9)
    q, k, v, rows = dev(w.q), dev(w.k), dev(w.v), dev(w.kv_rows)
    o1, l1 = _call_static(skv, lib, q, k, v, w.Hk, wl.F16, wl.F16, kv_rows=rows)
    r1o, r1l = skv.attn_partial(h, q, k, v, Hk=w.Hk, kv_rows=rows)
    torch.cuda.synchronize()
    vmax1 = vmax_of(oracle_mod, wl.F16, w.v, w.D)
    check_attention(o1, l1, r1o.cpu().numpy().astype(np.float64), r1l.cpu().numpy().astype(np.float64), vmax1,
                    "static call 1")

    # call 2, right after: dense q8_0 K / q4_0 V rows, a different split plan
    rng = wl.generator(3, salt=21)
    q2 = wl.normal_f16(rng, (1, 1, 40, 128))
    K2 = wl.cache_rows(rng, wl.Q8_0, 6000, 8, 128)
    V2 = wl.cache_rows(rng, wl.Q4_0, 6000, 8, 128)
    q2d, k2d, v2d = dev(q2), dev(K2), dev(V2)
    o2, l2 = _call_static(skv, lib, q2d, k2d, v2d, 8, wl.Q8_0, wl.Q4_0)
    r2o, r2l = skv.attn_partial(h, q2d, k2d, v2d, Hk=8, k_type=wl.Q8_0, v_type=wl.Q4_0)
    torch.cuda.synchronize()
    vmax2 = vmax_of(oracle_mod, wl.Q4_0, V2, 128)
    check_attention(o2, l2, r2o.cpu().numpy().astype(np.float64), r2l.cpu().numpy().astype(np.float64), vmax2,
                    "static call 2")
    h.close()
