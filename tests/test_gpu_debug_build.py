"""The index-checking debug build (-DCP_DEBUG, libcp_attn_debug.so).

Every kernel of that build checks the indices it computes against its
buffers' extents; a failed check records CP_ERR_DEVICE_INDEX and the access is
skipped.  Here the debug build runs every kernel family on small ragged cases
in a child process: results must meet the same bounds against the oracle, and
no check may fire.  (No out-of-range case is run on purpose.)
"""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_build_runs_clean():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from context_causal_attention_tcgen05_gb300 import build_lib

    lib = build_lib.DEBUG_LIB_PATH
    if not os.path.exists(lib):
        build_lib.build(debug=True)
    env = dict(os.environ, CP_ATTN_LIBRARY=lib)
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_child.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    print(r.stdout[-4000:], r.stderr[-2000:])
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "debug build: 0 failures" in r.stdout
