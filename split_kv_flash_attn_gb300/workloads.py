"""Seeded synthetic inputs for the five split-KV attention workloads.

This module only draws random numbers and lays them out as bytes.  It holds
none of the attention arithmetic, so both the CUDA path and the CPU oracle can
take their inputs from it without sharing any of the method.

Every workload draws from one NumPy ``PCG64`` generator seeded ``1000 + i``
(i = workload number, 1..5), in a fixed order: Q, then K, then V, then the row
lists or block selections.  fp16 values are drawn as float32 standard normals
and rounded to fp16 (round-to-nearest-even).  Quantised rows are packed in the
ggml block layout: q8_0 = [fp16 scale][32 x int8], q4_0 = [fp16 scale][16 bytes,
value j in the low nibble of byte j and value j+16 in the high nibble].

Cache rows are cell-major: row r holds KV heads 0..Hk-1 one after the other,
each head's D values as one segment.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

F16, Q8_0, Q4_0 = 0, 1, 2
SEED_BASE = 1000


def generator(workload: int, salt: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(SEED_BASE + workload + 7919 * salt))


def segment_bytes(type_: int, D: int) -> int:
    return {F16: 2 * D, Q8_0: 34 * (D // 32), Q4_0: 18 * (D // 32)}[type_]


def normal_f16(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32).astype(np.float16)


def _scales_f16(rng, n_blocks, lo=0.005, hi=0.02):
    return rng.uniform(lo, hi, n_blocks).astype(np.float16)


def q8_0_rows(rng: np.random.Generator, n_rows: int, Hk: int, D: int,
              chunk: int = 1 << 16) -> np.ndarray:
    """[n_rows, Hk*D/32*34] uint8: int8 codes ~U[-127,127], fp16 scale ~U[0.005,0.02]."""
    nb = Hk * (D // 32)
    out = np.empty((n_rows, nb, 34), dtype=np.uint8)
    for r0 in range(0, n_rows, chunk):
        r1 = min(n_rows, r0 + chunk)
        d = _scales_f16(rng, (r1 - r0) * nb).reshape(r1 - r0, nb)
        q = rng.integers(-127, 128, size=(r1 - r0, nb, 32), dtype=np.int8)
        out[r0:r1, :, 0:2] = d.view(np.uint8).reshape(r1 - r0, nb, 2)
        out[r0:r1, :, 2:] = q.view(np.uint8)
    return out.reshape(n_rows, nb * 34)


def q4_0_rows(rng: np.random.Generator, n_rows: int, Hk: int, D: int,
              chunk: int = 1 << 16) -> np.ndarray:
    """[n_rows, Hk*D/32*18] uint8: 4-bit codes u ~U[0,15], fp16 scale ~U[0.005,0.02]."""
    nb = Hk * (D // 32)
    out = np.empty((n_rows, nb, 18), dtype=np.uint8)
    for r0 in range(0, n_rows, chunk):
        r1 = min(n_rows, r0 + chunk)
        d = _scales_f16(rng, (r1 - r0) * nb).reshape(r1 - r0, nb)
        u = rng.integers(0, 16, size=(r1 - r0, nb, 32), dtype=np.uint8)
        out[r0:r1, :, 0:2] = d.view(np.uint8).reshape(r1 - r0, nb, 2)
        out[r0:r1, :, 2:] = u[:, :, :16] | (u[:, :, 16:] << 4)
    return out.reshape(n_rows, nb * 18)


def cache_rows(rng, type_: int, n_rows: int, Hk: int, D: int) -> np.ndarray:
    """Cell-major cache rows as a 2-D uint8 array [n_rows, row_bytes]."""
    if type_ == F16:
        return normal_f16(rng, (n_rows, Hk * D)).view(np.uint8).reshape(n_rows, Hk * D * 2)
    if type_ == Q8_0:
        return q8_0_rows(rng, n_rows, Hk, D)
    if type_ == Q4_0:
        return q4_0_rows(rng, n_rows, Hk, D)
    raise ValueError(type_)


@dataclass
class Workload:
    """A drawn workload.  Arrays are numpy; ``meta`` holds the sizes."""
    name: str
    S: int
    nq: int
    H: int
    Hk: int
    D: int
    k_type: int
    v_type: int
    q: np.ndarray                    # float16 [S, nq, H, D]
    k: np.ndarray                    # uint8 rows (region 0: window or whole cache)
    v: np.ndarray
    k_tail: np.ndarray | None = None  # uint8 rows of the host tail
    v_tail: np.ndarray | None = None
    kv_rows: np.ndarray | None = None  # int32 [S, n_keys] or [S, Hk, n_keys]
    q_pos: np.ndarray | None = None
    n_keys: int = 0
    tile_rows: int = 0
    extra: dict | None = None

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))


def pad_rows(lists: np.ndarray, multiple: int = 256) -> np.ndarray:
    """Append -1 entries so the last axis is a multiple of ``multiple``."""
    n = lists.shape[-1]
    m = -(-n // multiple) * multiple
    if m == n:
        return lists.astype(np.int32)
    pad = np.full(lists.shape[:-1] + (m - n,), -1, dtype=np.int32)
    return np.concatenate([lists.astype(np.int32), pad], axis=-1)


# ---------------------------------------------------------------- workloads

def tiny_decode(seed_workload: int = 1, n_kv: int = 256, wc: int = 128, H: int = 4,
                Hk: int = 1, D: int = 64) -> Workload:
    """Workload 1: one sequence, one token, window wc on device + host tail."""
    rng = generator(seed_workload)
    q = normal_f16(rng, (1, 1, H, D))
    k = cache_rows(rng, F16, n_kv, Hk, D)
    v = cache_rows(rng, F16, n_kv, Hk, D)
    return Workload("tiny_decode", 1, 1, H, Hk, D, F16, F16, q,
                    k[:wc].copy(), v[:wc].copy(), k[wc:].copy(), v[wc:].copy(),
                    n_keys=n_kv, tile_rows=n_kv - wc, extra={"wc": wc, "n_kv": n_kv})


def unified_decode(n_cache: int = 262144, S: int = 8, rows_per_seq: int = 32768,
                   H: int = 32, Hk: int = 8, D: int = 128, pad_to: int = 256,
                   seed_workload: int = 2, salt: int = 0) -> Workload:
    """Workload 2: a shared cell-major cache; each sequence owns ``rows_per_seq``
    distinct random rows (a random permutation of the cache cut into S lists
    when S*rows_per_seq == n_cache), sorted ascending, padded with -1."""
    assert S * rows_per_seq <= n_cache
    rng = generator(seed_workload, salt)
    q = normal_f16(rng, (S, 1, H, D))
    k = cache_rows(rng, F16, n_cache, Hk, D)
    v = cache_rows(rng, F16, n_cache, Hk, D)
    perm = rng.permutation(n_cache)[: S * rows_per_seq].reshape(S, rows_per_seq)
    lists = pad_rows(np.sort(perm, axis=1), pad_to)
    return Workload("unified_decode", S, 1, H, Hk, D, F16, F16, q, k, v,
                    kv_rows=lists, n_keys=lists.shape[1],
                    extra={"n_cache": n_cache, "rows_per_seq": rows_per_seq})


def long_context_decode(n_kv: int = 1048576, wc: int = 131072, tile_rows: int = 32768,
                        H: int = 40, Hk: int = 8, D: int = 128,
                        seed_workload: int = 3) -> Workload:
    """Workload 3: K q8_0, V q4_0; window [0,wc) on device, tail [wc,n_kv) on host."""
    rng = generator(seed_workload)
    q = normal_f16(rng, (1, 1, H, D))
    k = q8_0_rows(rng, n_kv, Hk, D)
    v = q4_0_rows(rng, n_kv, Hk, D)
    return Workload("long_context_decode", 1, 1, H, Hk, D, Q8_0, Q4_0, q,
                    k[:wc], v[:wc], k[wc:], v[wc:], n_keys=n_kv, tile_rows=tile_rows,
                    extra={"wc": wc, "n_kv": n_kv})


def prefill_chunk(n_kv: int = 65536, wc: int = 32768, nq: int = 512, H: int = 32,
                  Hk: int = 8, D: int = 128, tile_rows: int = 8192,
                  seed_workload: int = 4) -> Workload:
    """Workload 4: nq new tokens at positions n_kv-nq .. n_kv-1, causal."""
    rng = generator(seed_workload)
    q = normal_f16(rng, (1, nq, H, D))
    k = cache_rows(rng, F16, n_kv, Hk, D)
    v = cache_rows(rng, F16, n_kv, Hk, D)
    q_pos = (n_kv - nq + np.arange(nq, dtype=np.int32)).reshape(1, nq)
    return Workload("prefill_chunk", 1, nq, H, Hk, D, F16, F16, q,
                    k[:wc], v[:wc], k[wc:], v[wc:], q_pos=q_pos, n_keys=n_kv,
                    tile_rows=tile_rows, extra={"wc": wc, "n_kv": n_kv})


def prefill_quant_window(n: int = 32768, nq: int = 512, H: int = 32, Hk: int = 8, D: int = 128,
                         k_type: int = Q8_0, v_type: int = Q4_0, salt: int = 77) -> Workload:
    """Prefill over quantised rows: nq causal tokens at positions n-nq .. n-1
    over n q8_0-K / q4_0-V rows held on the device (the prefill chunk's shape
    over the long-context workload's row types)."""
    rng = generator(4, salt)
    q = normal_f16(rng, (1, nq, H, D))
    k = cache_rows(rng, k_type, n, Hk, D)
    v = cache_rows(rng, v_type, n, Hk, D)
    q_pos = (n - nq + np.arange(nq, dtype=np.int32)).reshape(1, nq)
    return Workload("prefill_quant_window", 1, nq, H, Hk, D, k_type, v_type, q, k, v, q_pos=q_pos, n_keys=n)


def prefill_row_lists(nq: int = 64, salt: int = 78, **unified) -> Workload:
    """Prefill through row lists: the unified-cache workload's cache and lists
    (``unified_decode(**unified)``), with nq causal tokens per sequence at the
    last nq positions of its list."""
    w = unified_decode(**unified)
    rng = generator(4, salt)
    q = normal_f16(rng, (w.S, nq, w.H, w.D))
    n_list = w.kv_rows.shape[1]
    q_pos = np.tile(np.arange(n_list - nq, n_list, dtype=np.int32), (w.S, 1))
    return Workload("prefill_row_lists", w.S, nq, w.H, w.Hk, w.D, F16, F16, q, w.k, w.v, kv_rows=w.kv_rows,
                    q_pos=q_pos, n_keys=n_list, extra=w.extra)


def block_sparse_decode(n_kv: int = 262144, S: int = 4, H: int = 32, Hk: int = 4,
                        D: int = 128, block_rows: int = 64, n_sel: int = 512,
                        cache_pages: int = 2048, seed_workload: int = 5) -> Workload:
    """Workload 5: paged host cache [block][Hk][block_rows][D] fp16; per (seq,
    KV head) ``n_sel`` distinct blocks drawn uniformly, sorted, expanded to rows."""
    rng = generator(seed_workload)
    n_blocks = n_kv // block_rows
    q = normal_f16(rng, (S, 1, H, D))
    k = normal_f16(rng, (n_blocks, Hk, block_rows, D))
    v = normal_f16(rng, (n_blocks, Hk, block_rows, D))
    sel = np.empty((S, Hk, n_sel), dtype=np.int32)
    for s in range(S):
        for kh in range(Hk):
            sel[s, kh] = np.sort(rng.choice(n_blocks, size=n_sel, replace=False))
    rows = (sel[..., None] * block_rows + np.arange(block_rows, dtype=np.int32)).reshape(S, Hk, -1)
    return Workload("block_sparse_decode", S, 1, H, Hk, D, F16, F16, q,
                    k.view(np.uint8).reshape(-1), v.view(np.uint8).reshape(-1),
                    kv_rows=rows.astype(np.int32), n_keys=rows.shape[-1],
                    extra={"n_kv": n_kv, "block_rows": block_rows, "n_blocks": n_blocks,
                           "sel": sel, "cache_pages": cache_pages})


def redraw_selection(sel: np.ndarray, n_blocks: int, frac: float,
                     rng: np.random.Generator) -> np.ndarray:
    """Replace ``frac`` of each (seq, head) selection with unused blocks (drift step)."""
    out = sel.copy()
    S, Hk, n = sel.shape
    n_new = int(round(frac * n))
    for s in range(S):
        for kh in range(Hk):
            cur = set(out[s, kh].tolist())
            drop = rng.choice(n, size=n_new, replace=False)
            pool = np.setdiff1d(np.arange(n_blocks), np.fromiter(cur, np.int64))
            add = rng.choice(pool, size=n_new, replace=False)
            row = out[s, kh].copy()
            row[drop] = add
            out[s, kh] = np.sort(row)
    return out


def new_kv_values(rng: np.random.Generator, n: int, Hk: int, D: int, outlier_channels: int = 4):
    """fp32 K and V values [n][Hk][D] for appends: standard normals, with a few
    K channels per head scaled up 8x (the outlier channels of key activations)
    and one row in 16 of V scaled by 1e-3 (tiny blocks reach fp16 subnormal
    scales).  Returns (k, v)."""
    k = rng.standard_normal((n, Hk, D), dtype=np.float32)
    v = rng.standard_normal((n, Hk, D), dtype=np.float32)
    for h in range(Hk):
        ch = rng.choice(D, size=min(outlier_channels, D), replace=False)
        k[:, h, ch] *= 8.0
    v[::16] *= 1e-3
    return k, v
