"""Shared helpers for the GPU parity tests (inputs come from synth, expected
values only from the oracle)."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import context_causal_attention_tcgen05_gb300 as cpa

# Spec tolerances: max |err| of attention outputs (bf16 2e-2, fp32 1e-4), of lse 5e-3.
TOL_OUT = {torch.bfloat16: 2e-2, torch.float32: 1e-4}
TOL_LSE = 5e-3


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not os.path.exists(cpa.library_path()):
        from context_causal_attention_tcgen05_gb300 import build_lib
        build_lib.build()
    cpa.load_library()


def f64(t):
    return t.detach().float().cpu().double().numpy()


def max_err(gpu, ref):
    g = f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    both_inf = np.isneginf(g) & np.isneginf(r)
    with np.errstate(invalid="ignore"):  # -inf - -inf where both are -inf: masked by both_inf
        d = np.abs(np.where(both_inf, 0.0, g - r))
    return float(np.nan_to_num(d, nan=np.inf).max()) if d.size else 0.0


# (test, quantity, max error, bound) of every checked result, printed in the
# terminal summary so the margins to the bounds are visible in a quiet run.
MARGINS = []


def _record(what, err, bound):
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0].split("::")[-1]
    MARGINS.append((test, what, float(err), float(bound)))


def assert_close(gpu_out, gpu_lse, ref_out, ref_lse, dtype, what=""):
    eo = max_err(gpu_out, ref_out)
    el = max_err(gpu_lse, ref_lse)
    _record(f"{what} out", eo, TOL_OUT[dtype])
    _record(f"{what} lse", el, TOL_LSE)
    assert eo <= TOL_OUT[dtype], f"{what}: out max err {eo}"
    assert el <= TOL_LSE, f"{what}: lse max err {el}"
    return eo, el


def check_grad(name, got, ref, tol):
    """Gradient bound (reading R11): max |err| <= tol * max(1, max |ref|)."""
    e = max_err(got, ref)
    bound = tol * max(1.0, float(np.abs(np.asarray(ref, dtype=np.float64)).max()) if np.size(ref) else 1.0)
    _record(name, e, bound)
    assert e <= bound, f"{name}: max err {e} > bound {bound}"
    return e


def oracle_bwd_by_kv_head(q, k, v, do, workers=4, **kw):
    """oracle.attention_bwd applied to each key/value head with its G query heads
    (one call per head on a thread pool) and reassembled.  The definition treats
    heads independently, so this is the same gradient as one call on all heads."""
    import oracle

    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv

    def one(hk):
        hs = slice(hk * G, (hk + 1) * G)
        return oracle.attention_bwd(q[:, hs], k[:, hk:hk + 1], v[:, hk:hk + 1], do[:, hs], **kw)

    with ThreadPoolExecutor(max(1, min(workers, Hkv))) as ex:
        parts = list(ex.map(one, range(Hkv)))
    return tuple(np.concatenate([p[i] for p in parts], axis=1) for i in range(3))


def check_ok():
    st = cpa.cp_check_device_status()
    assert st == 0, f"device status {st}: {cpa.cp_last_error()}"


def sample_rows(S, P, layout, n_random=256, seed=1):
    """Chunk-boundary rows of the layout plus random rows (sorted, unique)."""
    rows = set()
    nchunks = 2 * P if layout in ("zigzag", "dual_chunk_swap") else P
    C = S // nchunks
    for c in range(nchunks):
        for r in (c * C, c * C + 1, c * C + C // 2, (c + 1) * C - 2, (c + 1) * C - 1):
            if 0 <= r < S:
                rows.add(r)
    rng = np.random.default_rng(seed)
    rows.update(rng.integers(0, S, size=n_random).tolist())
    return np.array(sorted(rows), dtype=np.int64)
