"""The failure path of a bounded device-side wait, on the GPU, without a fault.

A self-test kernel waits, with the bounded mbarrier wait of the tensor-core
pipelines, on a barrier that nothing arrives on; the wait gives up after its
budget and sets the handle's status word.  The host reads SKV_ETIMEOUT, the
word is cleared by the read, and the same handle and context keep computing
correct attention afterwards.  Nothing here traps, faults or waits unbounded.
"""
import math

import pytest

from split_kv_flash_attn_gb300 import workloads as wl
from tests.gpu_util import check_attention, dev, vmax_of

pytestmark = pytest.mark.gpu

SKV_EINVAL, SKV_ETIMEOUT = 1, 7


@pytest.fixture(scope="module")
def skv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import split_kv_flash_attn_gb300 as m
    return m


def test_wait_gives_up_and_context_survives(skv, oracle_mod):
    import time
    h = skv.Handle(0)
    assert h.status() == 0
    t0 = time.perf_counter()
    skv.selftest_wait_timeout(h, 5_000_000)           # 5 ms budget
    with pytest.raises(skv.SplitKVError) as e:
        h.status()
    waited = time.perf_counter() - t0
    assert e.value.status == SKV_ETIMEOUT
    assert 0.004 <= waited < 2.0                       # it waited its budget, and no more than a bounded time
    assert h.status() == 0                             # the read cleared the word
    # the context and the handle still compute correct attention
    D, H, Hk, n = 128, 16, 4, 700
    rng = wl.generator(2, salt=4242)
    q = wl.normal_f16(rng, (1, 1, H, D))
    K = wl.cache_rows(rng, wl.F16, n, Hk, D)
    V = wl.cache_rows(rng, wl.F16, n, Hk, D)
    o, lse = skv.attn_partial(h, dev(q), dev(K), dev(V), Hk=Hk)
    want_o, want_l = oracle_mod.attention(q, D=D, H=H, Hk=Hk, scale=1 / math.sqrt(D), k0=K, v0=V, n_rows0=n,
                                          k_row_bytes0=K.shape[1], v_row_bytes0=V.shape[1], n_keys=n)
    check_attention(o, lse, want_o, want_l, vmax_of(oracle_mod, wl.F16, V, D), "after a timeout")
    assert h.status() == 0


def test_budget_out_of_range_rejected(skv):
    h = skv.Handle(0)
    for bad in (0, 999, 2_000_000_000):
        with pytest.raises(skv.SplitKVError) as e:
            skv.selftest_wait_timeout(h, bad)
        assert e.value.status == SKV_EINVAL
    assert h.status() == 0
