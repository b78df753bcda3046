"""The allocation-free block backward (cp_attn_block_bwd_noalloc).

Some callers cannot allocate device memory or pass a workspace (plugin and
custom-operator interfaces that hand over only inputs and outputs, runtimes
with a fixed memory plan).  This entry point keeps its scratch in an array
built into the library.  Here it is called through the C ABI twice in a row,
on different inputs, and must agree with cp_attn_block_bwd (which uses a
caller workspace) within the backward tolerance; a second call must not see
the first call's leftovers.  Sizes beyond the built-in scratch are refused.
This file is collected last so a stopping run has covered everything else.
"""
import numpy as np
import pytest
import torch

import context_causal_attention_tcgen05_gb300 as cpa
from gpu_common import check_ok, max_err, need_gpu
from synth import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.mark.parametrize("dtype,D,tol", [(torch.bfloat16, 128, 2e-2), (torch.float32, 64, 1e-4)],
                         ids=["bf16_d128", "f32_d64"])
def test_noalloc_matches_workspace_entry_point_twice(dtype, D, tol):
    S, Hq, Hkv = 384, 8, 2
    for seed in (11, 12):  # two calls in a row, different inputs
        q, k, v, do = (t.cuda() for t in make_inputs(S, Hq, Hkv, D, dtype, seed=seed, with_dout=True))
        o, l = cpa.cp_attn_block_fwd(q, k, v, True, 64, 0)
        want = cpa.cp_attn_block_bwd(q, k, v, o, do, l, True, 64, 0)
        got = cpa.cp_attn_block_bwd_noalloc(q, k, v, o, do, l, True, 64, 0)
        check_ok()
        for name, g, w in zip(("dq", "dk", "dv"), got, want):
            ref = w.float().cpu().double().numpy()
            e = max_err(g, ref)
            assert e <= tol * max(1.0, float(np.abs(ref).max())), f"{name} seed {seed}: {e}"


def test_noalloc_refuses_sizes_beyond_its_scratch():
    S, Hq, Hkv, D = 8192, 32, 8, 128  # dQ alone needs 128 MiB of fp32 scratch
    q = torch.empty(S, Hq, D, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(S, Hkv, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(Hq, S, dtype=torch.float32, device="cuda")
    with pytest.raises(cpa.CpAttnError) as ei:
        cpa.cp_attn_block_bwd_noalloc(q, k, k, q, q, lse)
    assert ei.value.status == -5
    assert "built-in scratch" in str(ei.value)
