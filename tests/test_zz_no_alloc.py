"""The block backward that allocates no device memory (cp_attn_block_bwd_noalloc).

Some callers cannot allocate device memory or pass a workspace: code behind a
plugin or custom-operator interface that hands over only input and output
buffers, runtimes that fix their device memory plan ahead of time.  This entry
point keeps its scratch in an array built into the library.  It is called here
through the C ABI twice in a row, on different inputs, and must agree with
cp_attn_block_bwd_typed (which uses a caller workspace) and with the oracle's
gradient within the backward tolerance; a second call must not see the first
call's leftovers in the shared array.  Sizes beyond the built-in scratch are
refused.  This file is collected last so a stopping run has covered
everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

import context_causal_attention_tcgen05_gb300 as cpa
import oracle
from gpu_common import check_ok, max_err, need_gpu
from synth import cu_seqlens_from_lengths, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _bound(ref, tol):
    return tol * max(1.0, float(np.abs(ref).max()))


@pytest.mark.parametrize("dtype,D,tol", [(torch.bfloat16, 128, 2e-2), (torch.float32, 64, 1e-4),
                                         (torch.bfloat16, 64, 2e-2)],
                         ids=["bf16_d128", "f32_d64", "bf16_d64"])
@pytest.mark.parametrize("docs_window", [False, True], ids=["causal", "docs_window"])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(dtype, D, tol, docs_window):
    S, Hq, Hkv = 384, 8, 2
    # documents cover every position the call sees: keys 0..383, queries 64..447
    cu = cu_seqlens_from_lengths([100, 1, 150, 133, 64]) if docs_window else None
    W = 90 if docs_window else 0
    cu_d = None if cu is None else torch.from_numpy(cu).cuda()
    for seed in (11, 12):  # two calls in a row, different inputs
        qh, kh, vh, doh = make_inputs(S, Hq, Hkv, D, dtype, seed=seed, with_dout=True)
        q, k, v, do = qh.cuda(), kh.cuda(), vh.cuda(), doh.cuda()
        o, l = cpa.cp_attn_block_fwd(q, k, v, True, 64, 0, cu_seqlens=cu_d, window=W)
        want = cpa.cp_attn_block_bwd_typed(q, k, v, o, do, l, True, 64, 0, cu_seqlens=cu_d, window=W)
        got = cpa.cp_attn_block_bwd_noalloc(q, k, v, o, do, l, True, 64, 0, cu_seqlens=cu_d, window=W)
        check_ok()
        ref = oracle.attention_bwd(qh, kh, vh, doh, True, 64, 0, cu_seqlens=cu, window=W)
        for name, g, w, r in zip(("dq", "dk", "dv"), got, want, ref):
            e_ws = max_err(g, w.float().cpu().double().numpy())
            e_or = max_err(g, r)
            print(f"noalloc {name} seed {seed}: vs workspace form {e_ws:.3g}, vs oracle {e_or:.3g} "
                  f"(bound {_bound(r, tol):.3g})")
            assert e_ws <= _bound(r, tol), f"{name} seed {seed}: {e_ws}"
            assert e_or <= _bound(r, tol), f"{name} seed {seed}: {e_or}"


def test_noalloc_output_overlapping_dout_twice():
    # dq written over dout's storage: the tensor-core kernels still read dout, so the
    # call takes its fp32 accumulators from the shared array and casts after them;
    # the second call (other inputs) must not see the first call's accumulators
    S, Hq, Hkv, D = 256, 4, 2, 128
    lib = cpa.load_library()
    for seed in (21, 22):
        qh, kh, vh, doh = make_inputs(S, Hq, Hkv, D, torch.bfloat16, seed=seed, with_dout=True)
        q, k, v = qh.cuda(), kh.cuda(), vh.cuda()
        buf = doh.cuda()  # dout, then dq in the same storage
        o, l = cpa.cp_attn_block_fwd(q, k, v, True)
        dk, dv = torch.empty_like(k), torch.empty_like(v)
        m = cpa._mask(True, 0, 0, 1, 1, None, 0)
        st = lib.cp_attn_block_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                           buf.data_ptr(), l.data_ptr(), S, S, Hq, Hkv, D, cpa.CP_BF16,
                                           ctypes.byref(m), 0.0, buf.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                           torch.cuda.current_stream().cuda_stream)
        assert st == 0, cpa.cp_last_error()
        check_ok()
        ref = oracle.attention_bwd(qh, kh, vh, doh, True)
        for name, g, r in zip(("dq", "dk", "dv"), (buf, dk, dv), ref):
            e = max_err(g, r)
            print(f"noalloc overlapping {name} seed {seed}: {e:.3g} (bound {_bound(r, 2e-2):.3g})")
            assert e <= _bound(r, 2e-2), f"{name} seed {seed}: {e}"


def test_noalloc_refuses_sizes_beyond_its_scratch():
    S, Hq, Hkv, D = 8192, 32, 8, 128  # dQ alone needs 128 MiB of fp32 scratch
    q = torch.empty(S, Hq, D, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(S, Hkv, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(Hq, S, dtype=torch.float32, device="cuda")
    with pytest.raises(cpa.CpAttnError) as ei:
        cpa.cp_attn_block_bwd_noalloc(q, k, k, q, q, lse)
    assert ei.value.status == -5
    assert "built-in scratch" in str(ei.value)
