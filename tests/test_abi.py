"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/cp_attn.h declares, and refuses bad arguments with the
documented status before touching the device."""
import ctypes

import pytest

import context_causal_attention_tcgen05_gb300 as cpa


@pytest.fixture(scope="module")
def lib():
    import os
    if not os.path.exists(cpa.library_path()):
        from context_causal_attention_tcgen05_gb300 import build_lib
        build_lib.build()
    return cpa.load_library()


def test_every_header_function_is_exported(lib):
    names = cpa.header_functions()
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert cpa.cp_status_string(0) == "CP_OK"
    assert cpa.cp_status_string(-8) == "CP_ERR_DEVICE_TIMEOUT"
    assert cpa.cp_version().count(".") == 2


P16 = ctypes.c_void_p(1 << 20)  # 16-byte aligned fake device address; never dereferenced


def _fwd(lib, **kw):
    args = dict(q=P16, k=P16, v=P16, Sq=128, Sk=128, Hq=8, Hkv=8, D=128, dtype=1, mask=None,
                scale=0.0, out=P16, lse=P16, stream=None)
    args.update(kw)
    return lib.cp_attn_block_fwd(*args.values())


def test_block_fwd_refusals(lib):
    assert _fwd(lib, dtype=7) == -3                       # CP_ERR_DTYPE
    assert _fwd(lib, D=96) == -3                          # bf16 needs D in {64,128}
    assert _fwd(lib, dtype=0, D=48) == -2                 # fp32 D not supported
    assert _fwd(lib, Hq=6, Hkv=4) == -2                   # Hq % Hkv
    assert _fwd(lib, Sq=-1) == -1
    assert _fwd(lib, q=ctypes.c_void_p(0)) == -1          # NULL q
    assert _fwd(lib, k=ctypes.c_void_p((1 << 20) + 8)) == -4  # misaligned
    assert "aligned" in cpa.cp_last_error()
    m = cpa.cp_mask()
    m.causal, m.q_stride, m.k_stride = 1, 0, 1
    assert _fwd(lib, mask=ctypes.byref(m)) == -1          # stride 0
    m.q_stride, m.window = 1, -4
    assert _fwd(lib, mask=ctypes.byref(m)) == -1          # negative window
    m.causal, m.window = 0, 16
    assert _fwd(lib, mask=ctypes.byref(m)) == -5          # a window needs the causal rule
    assert "causal" in cpa.cp_last_error()
    assert ctypes.sizeof(cpa.cp_mask) == 56               # the window fits the struct's padding
    assert _fwd(lib, Sq=0) == 0                           # empty is a no-op


def _ring(lib, **kw):
    args = dict(q=P16, k=P16, v=P16, S=8192, Hq=32, Hkv=32, D=128, dtype=1, P=8, reorder=1, mode=0,
                cu=None, n_docs=0, out=P16, lse=P16, ws=P16, ws_bytes=1 << 40, stream=None)
    args.update(kw)
    return lib.cp_ring_attention(*args.values())


def test_ring_refusals(lib):
    assert _ring(lib, S=8200) == -2                       # S % 2P
    assert _ring(lib, P=0) == -1
    assert _ring(lib, P=33) == -1
    assert _ring(lib, reorder=9) == -1
    assert _ring(lib, mode=5) == -1
    assert _ring(lib, P=20, S=20 * 64) == -5              # zigzag limited to P <= 16
    # packing only with a load-balanced ring (MaxText packing PR)
    assert _ring(lib, reorder=0, cu=P16, n_docs=3) == -5
    assert "load-balanced" in cpa.cp_last_error()
    assert _ring(lib, ws_bytes=100) == -6                 # workspace too small
    assert _ring(lib, ws=ctypes.c_void_p(0)) == -6


def test_ring_to_seq_refusals(lib):
    # sequence-order output needs runs of consecutive positions: striped (and AUTO with
    # documents, which resolves to striped) is refused before any device work
    f = lib.cp_ring_attention_reordered_to_seq
    args = lambda S=8192, P=8, reorder=1, cu=None, n_docs=0: (
        P16, P16, P16, S, 32, 32, 128, cpa.CP_BF16, P, reorder, cu, n_docs, P16, P16, None)
    assert f(*args(reorder=2)) == -5
    assert "consecutive positions" in cpa.cp_last_error()
    assert f(*args(reorder=3, cu=P16, n_docs=3)) == -5
    assert f(*args(S=8200)) == -2                          # S % 2P
    assert f(*args(P=0)) == -1
    assert f(*args(reorder=9)) == -1


def test_ulysses_refusals(lib):
    f = lib.cp_ulysses_attention
    # q k v S Hq Hkv D dtype P cu n_docs window out lse ws ws_bytes stream
    base = [P16, P16, P16, 32768, 32, 8, 128, 1, 16, None, 0, 0, P16, P16, P16, 1 << 40, None]
    a = list(base)
    a[5] = 6
    st = f(*a)  # Hkv=6, P=16: neither a divisor nor a multiple of the key/value heads
    assert st == -2 and "Hkv" in cpa.cp_last_error()
    a = list(base)
    a[5] = 32
    a[3] = 32769
    assert f(*a) == -2                                    # S % P
    a = list(base)  # Hkv=8 < P=16 is accepted (heads replicated): it reaches the workspace check
    a[15] = 100
    assert f(*a) == -6
    a = list(base)
    a[11] = -1                                            # negative window
    assert f(*a) == -1
    need = ctypes.c_size_t()
    assert lib.cp_workspace_size(2, 32768, 32, 8, 128, 1, 16, 0, ctypes.byref(need)) == 0
    need_plain = ctypes.c_size_t()
    assert lib.cp_workspace_size(2, 32768, 32, 16, 128, 1, 16, 0, ctypes.byref(need_plain)) == 0
    assert need.value == need_plain.value  # 8 heads x 2 copies hold as much as 16 heads


def test_usp_refusals(lib):
    f = lib.cp_usp_attention
    # q k v S Hq Hkv D dtype Pu Pr reorder cu n_docs out lse ws ws_bytes stream
    base = [P16, P16, P16, 8192, 32, 8, 128, 1, 4, 4, 1, None, 0, P16, P16, P16, 1 << 40, None]
    a = list(base)
    a[5] = 6                                              # Hkv % P_ulysses
    assert f(*a) == -2
    a = list(base)
    a[8], a[9] = 8, 16                                    # P_ulysses * P_ring > 64
    assert f(*a) == -1
    a = list(base)
    a[3] = 40                                             # zigzag rule holds, (S / P_ring) % P_ulysses does not
    assert f(*a) == -2
    a = list(base)
    a[16] = 100                                           # workspace too small
    assert f(*a) == -6
    need = ctypes.c_size_t()
    assert lib.cp_workspace_size(6, 8192, 32, 8, 128, 1, 4, 0, ctypes.byref(need)) == 0 and need.value > 0


def test_ulysses_bwd_refusals(lib):
    f = lib.cp_ulysses_attention_bwd
    # q k v out lse dout S Hq Hkv D dtype P cu n_docs window dq dk dv ws ws_bytes stream
    base = [P16, P16, P16, P16, P16, P16, 4096, 32, 8, 128, 1, 16, None, 0, 0, P16, P16, P16, P16, 1 << 40, None]
    a = list(base)
    a[8] = 6
    assert f(*a) == -2 and "Hkv" in cpa.cp_last_error()
    a = list(base)
    a[7] = 24                                             # Hq % P
    assert f(*a) == -2
    a = list(base)
    a[19] = 100                                           # workspace too small
    assert f(*a) == -6
    a = list(base)
    a[4] = None                                           # lse required
    assert f(*a) == -1
    need = ctypes.c_size_t()
    assert lib.cp_workspace_size(5, 4096, 32, 8, 128, 1, 16, 0, ctypes.byref(need)) == 0
    assert need.value > 0


def test_permute_refusals(lib):
    assert lib.cp_ulysses_seq2head(P16, P16, 64, 6, 128, 4, 1, None) == -2   # H % P
    assert lib.cp_zigzag_reorder(P16, P16, 60, 8, 128, 4, 1, None) == -2     # S % 2P
    assert lib.cp_striped_reorder(P16, P16, 64, 1, 4, 4, 1, None) == -4      # 8-byte rows
    assert lib.cp_zigzag_reorder(P16, P16, 64, 8, 128, 4, 1, None) == -1     # x, y overlap
    assert lib.cp_zigzag_reorder(P16, P16, 0, 8, 128, 4, 1, None) == 0       # empty


def test_batched_ring_permute_refusals(lib):
    P32 = ctypes.c_void_p((1 << 20) + (1 << 30))  # a second fake address, far from P16
    qkv = lambda S=64, Hq=8, Hkv=8, D=128, dt=1, P=4, reo=1, dst=P32: lib.cp_ring_reorder_qkv(
        P16, P16, P16, dst, dst, dst, S, Hq, Hkv, D, dt, P, reo, None)
    assert qkv(reo=0) == -1          # contiguous: nothing to reorder
    assert qkv(reo=3) == -1          # AUTO needs documents to resolve
    assert qkv(S=60) == -2           # S % 2P
    assert qkv(S=60, reo=2, dst=P16) == -1  # striped needs only S % P; then the overlap check
    assert qkv(D=4, Hkv=1) == -4     # 8-byte rows of k/v
    assert qkv(dt=7) == -3
    assert qkv(dst=P16) == -1        # source and destination overlap
    assert qkv(S=0) == 0             # empty
    odd = ctypes.c_void_p((1 << 20) + (1 << 30) + 8)  # 8-byte aligned only
    assert qkv(dst=odd) == -4        # 16-byte vectors need 16-byte aligned tensors
    rst = lambda S=64, lse_re=P16, lse=P32, P=4, reo=1: lib.cp_ring_restore(
        P16, lse_re, P32, lse, S, 8, 128, 1, P, reo, None)
    assert rst(lse=None) == -1       # lse_re without lse
    assert rst(reo=0) == -1
    assert rst(S=60) == -2
    assert rst(S=0) == 0
    assert lib.cp_ring_restore(P16, P16, odd, P32, 64, 8, 128, 1, 4, 1, None) == -4  # out misaligned


def test_merge_and_workspace_refusals(lib):
    assert lib.cp_lse_merge(P16, P16, P16, P16, P16, P16, 16, 4, 100, 1, None) == -4
    assert lib.cp_lse_merge(P16, P16, P16, P16, P16, P16, 16, 4, 128, 5, None) == -3
    out = ctypes.c_size_t(0)
    assert lib.cp_workspace_size(9, 8192, 32, 32, 128, 1, 8, 0, ctypes.byref(out)) == -1
    assert lib.cp_workspace_size(0, 8192, 32, 32, 128, 1, 8, 0, ctypes.byref(out)) == 0
    fused = out.value
    assert lib.cp_workspace_size(0, 8192, 32, 32, 128, 1, 8, 1, ctypes.byref(out)) == 0
    assert out.value > fused  # stepwise keeps fp32 partials
    assert lib.cp_debug_bounded_wait(0, None) == -1


def _bwd(lib, **kw):
    args = dict(q=P16, k=P16, v=P16, out=P16, dout=P16, lse=P16, Sq=128, Sk=128, Hq=8, Hkv=8, D=128,
                dtype=1, mask=None, scale=0.0, dq=ctypes.c_void_p(1 << 30), dk=ctypes.c_void_p(1 << 31),
                dv=ctypes.c_void_p(1 << 32), acc=0, ws=ctypes.c_void_p(1 << 33), ws_bytes=1 << 20,
                stream=None)
    args.update(kw)
    return lib.cp_attn_block_bwd(*args.values())


def test_accumulating_block_bwd_refusals(lib):
    # the accumulating form (fp32 gradient buffers + accumulate flag): refused before any launch
    assert _bwd(lib, acc=2) == -1                         # accumulate is 0 or 1
    assert _bwd(lib, dq=P16) == -1                        # dq_acc overlaps q
    assert "overlap" in cpa.cp_last_error()
    assert _bwd(lib, dk=ctypes.c_void_p(1 << 30)) == -1   # dk_acc overlaps dq_acc
    assert _bwd(lib, ws_bytes=100) == -6                  # Delta needs 4*Hq*Sq bytes
    assert _bwd(lib, ws=ctypes.c_void_p(0)) == -6
    assert _bwd(lib, dv=ctypes.c_void_p((1 << 32) + 4)) == -4  # misaligned
    assert _bwd(lib, D=96) == -3
    assert _bwd(lib, Sq=0, Sk=0) == 0                     # empty is a no-op


def test_noalloc_refuses_absurd_sizes_without_a_device(lib):
    # the shared validation runs first: sizes whose scratch arithmetic could wrap are
    # refused by the S*H < 2^31 and int32-position rules, never by a wrapped size
    f = lib.cp_attn_block_bwd_noalloc
    base = [P16, P16, P16, P16, P16, P16, 1 << 40, 128, 8, 8, 128, 1, None, 0.0, P16, P16, P16, None]
    assert f(*base) == -5 and "2^31" in cpa.cp_last_error()
    m = cpa.cp_mask()
    m.causal, m.q_stride, m.k_stride, m.q_offset = 1, 1, 1, -(1 << 63)
    a = list(base)
    a[6], a[12] = 128, ctypes.byref(m)
    assert f(*a) == -5 and "int32" in cpa.cp_last_error()
    m.q_offset, m.q_stride = 0, 1 << 62                   # stride * (Sq - 1) would overflow int64
    assert f(*a) == -5
    a = list(base)
    a[6], a[7] = 8192, 8192                               # valid, but beyond the built-in scratch
    a[8], a[9] = 32, 8
    assert f(*a) == -5 and "built-in scratch" in cpa.cp_last_error()
