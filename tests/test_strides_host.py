"""Host-side checks of the strided entry points (CPU only).

Every call here is rejected by the argument checks, which run before any CUDA
call, so no kernel is ever launched on the fake (aligned, never dereferenced)
addresses used below."""
import ctypes

from io_aware_exact_14_gb300 import fa

BASE = 1 << 32   # fake 16-byte-aligned device addresses; the checks never dereference them


def _st(b, h, n):
    return fa.FaStrides(b, h, n)


def _fwd(q, qs, k, ks, v, vs, o, os_, lse, B=2, H=3, N=300, d=64):
    a = lambda s: ctypes.addressof(s) if s is not None else None
    return fa.load().fa_fwd_strided(q, a(qs), k, a(ks), v, a(vs), o, a(os_), lse, B, H, N, d, 0.125, 0, None)


def test_rejects_bad_strides():
    B, H, N, d = 2, 3, 300, 64
    good = _st(H * N * d, N * d, d)
    far = BASE + (1 << 28)
    for bad in (_st(H * N * d, N * d, d + 4),      # not a multiple of 8 elements (16 bytes)
                _st(H * N * d, N * d, d - 8),      # rows closer than d
                _st(0, N * d, d),                  # zero stride
                _st(-H * N * d, N * d, d)):        # negative stride
        st = _fwd(BASE, bad, BASE + (1 << 24), good, BASE + (2 << 24), good, far, good, far + (1 << 26))
        assert st == fa.FA_ERR_INVALID_ARG


def test_rejects_outputs_sharing_elements():
    B, H, N, d = 2, 3, 300, 64
    bnhd = _st(N * H * d, d, H * d)                # [B, N, H, d] storage seen as [B, H, N, d]
    q, k, v = BASE, BASE + (1 << 24), BASE + (2 << 24)
    lse = BASE + (3 << 24)
    # O written over q itself
    assert _fwd(q, bnhd, k, bnhd, v, bnhd, q, bnhd, lse) == fa.FA_ERR_INVALID_ARG
    # O interleaved with q half a row apart (shares elements)
    assert _fwd(q, bnhd, k, bnhd, v, bnhd, q + d, bnhd, lse) == fa.FA_ERR_INVALID_ARG
    # packed gradients whose slots are closer than d elements overlap
    packed = _st(N * 3 * H * d, d, 3 * H * d)
    g = fa.load().fa_bwd_strided
    a = ctypes.addressof
    dq = BASE + (4 << 24)
    st = g(q, a(bnhd), k, a(bnhd), v, a(bnhd), v + (1 << 22), a(bnhd), lse, v + (2 << 22), a(bnhd),
           dq, a(packed), dq + 2 * (d // 2), a(packed), dq + 2 * H * d * 2, a(packed),
           B, H, N, d, 0.125, 0, BASE + (5 << 24), 1 << 20, None)
    assert st == fa.FA_ERR_INVALID_ARG
