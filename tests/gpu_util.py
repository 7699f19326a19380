"""Helpers shared by the GPU parity tests: device copies and the tolerance
check.  Tolerances: max|dO| <= 2e-3 * max|V| and |dlse| <= 1e-4 absolute;
rows with no visible key must give O = 0 and lse = -inf exactly."""
import numpy as np

TOL_O_REL = 2e-3
TOL_LSE = 1e-4


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def pinned(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def check_attention(o_gpu, lse_gpu, o_ref, lse_ref, vmax, what=""):
    o = o_gpu.detach().cpu().numpy().astype(np.float64).reshape(o_ref.shape)
    lse = lse_gpu.detach().cpu().numpy().astype(np.float64).reshape(lse_ref.shape)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: -inf rows differ"
    assert np.all(o[empty] == 0.0), f"{what}: empty rows must give O = 0"
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    if (~empty).any():
        do = np.abs(o[~empty] - o_ref[~empty]).max()
        dl = np.abs(lse[~empty] - lse_ref[~empty]).max()
        assert do <= TOL_O_REL * vmax, f"{what}: max|dO| = {do:.3e} > {TOL_O_REL} * {vmax:.3f}"
        assert dl <= TOL_LSE, f"{what}: max|dlse| = {dl:.3e}"
        return do / vmax, dl
    return 0.0, 0.0


def vmax_of(oracle_mod, type_, raw_rows, D):
    """max|V| over a cache given as raw rows (decoded by the oracle)."""
    raw = np.ascontiguousarray(raw_rows).reshape(-1).view(np.uint8)
    if type_ == oracle_mod.F16:
        return float(np.abs(raw.view(np.float16).astype(np.float64)).max())
    n_vals = raw.size // (34 if type_ == oracle_mod.Q8_0 else 18) * 32
    return float(np.abs(oracle_mod.dequant(type_, raw, n_vals)).max())


def head_columns(rows, kh, seg):
    """The bytes of KV head kh (segment size seg) of cell-major rows, as rows
    of their own (a one-head cache the oracle can read with Hk = 1)."""
    return np.ascontiguousarray(np.asarray(rows).reshape(rows.shape[0], -1)[:, kh * seg:(kh + 1) * seg])


def oracle_one_head(oracle_mod, w, kh, *, k_type, v_type, k0, v0, k1=None, v1=None, **kw):
    """Oracle rows of the G query heads of KV head kh (all tokens, all
    sequences): the cache regions are cut down to that head's columns."""
    G = w.H // w.Hk
    sk, sv = oracle_mod.segment_bytes(k_type, w.D), oracle_mod.segment_bytes(v_type, w.D)
    qh = np.ascontiguousarray(w.q[:, :, kh * G:(kh + 1) * G])
    regions = dict(k0=head_columns(k0, kh, sk), v0=head_columns(v0, kh, sv), n_rows0=k0.shape[0],
                   k_row_bytes0=sk, v_row_bytes0=sv)
    if k1 is not None:
        regions.update(k1=head_columns(k1, kh, sk), v1=head_columns(v1, kh, sv), n_rows1=k1.shape[0],
                       k_row_bytes1=sk, v_row_bytes1=sv)
    return oracle_mod.attention(qh, D=w.D, H=G, Hk=1, scale=w.scale, k_type=k_type, v_type=v_type, **regions, **kw)
