"""The C-ABI library: it builds, loads, exports what include/fa.h declares, and
rejects bad arguments before touching a device (CPU only, no compute calls)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from io_aware_exact_14_gb300 import build, fa
    build.build()
    return fa.load()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_status_string", "fa_debug_status"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    from io_aware_exact_14_gb300 import fa
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in fa.SIGNATURES, f"binding lacks {name}"


FAKE = 0x10000  # never dereferenced: every call below fails validation first
BAD_ALIGN = FAKE + 8


def fwd(lib, q=FAKE, k=FAKE + 0x100000, v=FAKE + 0x200000, o=FAKE + 0x300000, lse=FAKE + 0x400000,
        B=1, H=1, N=128, d=64, scale=0.125, causal=0):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, None)


def test_fwd_argument_checks(lib):
    assert fwd(lib, d=100) == 2           # FA_ERR_UNSUPPORTED: not a multiple of 8
    assert fwd(lib, d=264) == 2           # above 256
    assert fwd(lib, d=260) == 2
    assert fwd(lib, d=4) == 2
    assert fwd(lib, d=0) == 2
    assert fwd(lib, N=0, q=0, k=0, v=0, o=0, lse=0) == 0  # empty problem is a no-op
    assert fwd(lib, q=0) == 1             # FA_ERR_INVALID_ARG: null
    assert fwd(lib, lse=0) == 1
    assert fwd(lib, v=BAD_ALIGN) == 1     # misaligned tensor
    assert fwd(lib, lse=FAKE + 0x400002) == 1
    assert fwd(lib, B=0) == 1
    assert fwd(lib, N=-1) == 1
    assert fwd(lib, scale=0.0) == 1
    assert fwd(lib, scale=float("nan")) == 1
    assert fwd(lib, scale=-0.125) == 1
    assert fwd(lib, o=FAKE) == 1          # output aliases q
    assert fwd(lib, lse=FAKE + 0x300000 + 64) == 1  # lse overlaps o
    assert fwd(lib, B=1 << 16, H=1 << 16) == 2      # beyond the grid limit


def test_bwd_argument_checks(lib):
    p = [FAKE + i * 0x100000 for i in range(12)]
    ws = lib.fa_bwd_workspace_bytes(1, 1, 128, 64)
    assert ws == 512  # 128 fp32 row terms, 256-byte rounded
    assert lib.fa_bwd_workspace_bytes(2, 3, 100, 128) == ((2 * 3 * 100 * 4 + 255) // 256) * 256
    assert lib.fa_bwd_workspace_bytes(1, 1, 0, 64) == 0
    assert lib.fa_bwd_workspace_bytes(1, 1, 128, 100) == 0
    assert lib.fa_bwd_workspace_bytes(1, 1, 128, 96) == 512

    def bwd(**kw):
        a = dict(q=p[0], k=p[1], v=p[2], o=p[3], lse=p[4], do=p[5], dq=p[6], dk=p[7], dv=p[8],
                 B=1, H=1, N=128, d=64, scale=0.125, causal=1, ws=p[9], wsb=ws)
        a.update(kw)
        return lib.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"], a["dv"],
                          a["B"], a["H"], a["N"], a["d"], a["scale"], a["causal"], a["ws"], a["wsb"], None)

    assert bwd(d=84) == 2
    assert bwd(d=264) == 2
    assert lib.fa_bwd_workspace_bytes(1, 1, 128, 256) == 512
    assert lib.fa_bwd_workspace_bytes(1, 1, 128, 264) == 0
    assert bwd(N=0, q=0) == 0
    assert bwd(dq=0) == 1
    assert bwd(do=BAD_ALIGN) == 1
    assert bwd(ws=0) == 4                 # FA_ERR_WORKSPACE
    assert bwd(wsb=ws - 4) == 4
    assert bwd(ws=p[9] + 4) == 4
    assert bwd(dk=p[0]) == 1              # output aliases an input
    assert bwd(dv=p[6]) == 1              # two outputs alias
    assert bwd(ws=p[4]) == 1              # workspace aliases lse
    assert lib.fa_bwd_preprocess(p[3], p[5], 0, 1, 1, 128, 64, None) == 1
    assert lib.fa_bwd_dkdv(p[0], p[1], p[2], p[4], p[5], p[10], p[7], p[0], 1, 1, 128, 64, 0.1, 0, None) == 1
    assert lib.fa_bwd_dq(p[0], p[1], p[2], p[4], p[5], p[10], p[6], 1, 1, 128, 64, 0.0, 0, None) == 1


def test_noalloc_rejects_oversized_problem_without_a_device(lib):
    p = [FAKE + i * 0x100000 for i in range(9)]
    assert lib.fa_bwd_noalloc(*p, 1, 64, 32769, 64, 0.125, 0, None) == 4   # 2^21 + 64 rows
    assert b"exceeds the built-in scratch" in lib.fa_last_error_detail()
    assert lib.fa_bwd_noalloc(*p, 1, 1, 128, 100, 0.125, 0, None) == 2
    assert lib.fa_bwd_noalloc(0, *p[1:], 1, 1, 128, 64, 0.125, 0, None) == 1


def test_status_strings(lib):
    for s in range(6):
        text = lib.fa_status_string(s).decode()
        assert text.startswith("FA_")
    assert lib.fa_status_string(99).decode() == "unknown fa_status"


class _Dropout(ctypes.Structure):
    _fields_ = [("p", ctypes.c_float), ("seed", ctypes.c_ulonglong), ("offset", ctypes.c_uint)]


def test_dropout_argument_checks(lib):
    """A NULL fa_dropout or p outside [0, 1) is rejected before any device access;
    so are the usual pointer and size errors."""
    def fwd_d(drop, **kw):
        a = dict(q=FAKE, k=FAKE + 0x100000, v=FAKE + 0x200000, o=FAKE + 0x300000, lse=FAKE + 0x400000, d=64)
        a.update(kw)
        ptr = ctypes.addressof(drop) if drop is not None else None
        return lib.fa_fwd_dropout(a["q"], a["k"], a["v"], a["o"], a["lse"], 1, 1, 128, a["d"], 0.125, 0, ptr, None)

    assert fwd_d(None) == 1
    for p in (1.0, 1.5, -0.1, float("nan"), float("inf")):
        assert fwd_d(_Dropout(p, 1, 0)) == 1, p
    assert fwd_d(_Dropout(0.1, 1, 0), q=0) == 1
    assert fwd_d(_Dropout(0.1, 1, 0), d=264) == 2   # above the widest head
    assert fwd_d(_Dropout(0.1, 1, 0), d=100) == 2   # not a multiple of 8
    assert fwd_d(_Dropout(0.1, 1, 0), o=FAKE) == 1
    p = [FAKE + i * 0x100000 for i in range(12)]
    ws = lib.fa_bwd_workspace_bytes(1, 1, 128, 64)
    drop = _Dropout(0.2, 5, 0)
    assert lib.fa_bwd_dropout(*p[:9], 1, 1, 128, 64, 0.125, 1, None, p[9], ws, None) == 1
    assert lib.fa_bwd_dropout(*p[:9], 1, 1, 128, 64, 0.125, 1, ctypes.addressof(_Dropout(1.0, 5, 0)), p[9], ws,
                              None) == 1
    assert lib.fa_bwd_dropout(*p[:9], 1, 1, 128, 64, 0.125, 1, ctypes.addressof(drop), 0, ws, None) == 4
    assert lib.fa_bwd_dropout(*p[:6], p[0], *p[7:9], 1, 1, 128, 64, 0.125, 1, ctypes.addressof(drop), p[9], ws,
                              None) == 1


def test_fp8_argument_checks(lib):
    x, out, ds = FAKE, FAKE + 0x100000, FAKE + 0x200000
    assert lib.fa_fp8_quantize(x, out, ds, 1, 1, 128, 40, 0, 0, 0, None) == 2    # d not a multiple of 16
    assert lib.fa_fp8_quantize(x, out, ds, 1, 1, 128, 96, 0, 1, 5, None) == 2    # rotation needs d = 64, 128 or 256
    assert lib.fa_fp8_quantize(x, out, ds, 1, 1, 128, 272, 0, 0, 0, None) == 2   # above the widest head
    assert lib.fa_fp8_quantize(0, out, ds, 1, 1, 128, 64, 0, 0, 0, None) == 1
    assert lib.fa_fp8_quantize(x, x, ds, 1, 1, 128, 64, 0, 0, 0, None) == 1     # out aliases x
    assert lib.fa_fp8_quantize(x, out, ds, 1, 1, 0, 64, 0, 0, 0, None) == 0      # empty
    assert lib.fa_fp8_vt_ld(1) == 16 and lib.fa_fp8_vt_ld(32) == 32 and lib.fa_fp8_vt_ld(33) == 48
    p = [FAKE + i * 0x100000 for i in range(8)]
    assert lib.fa_fwd_fp8(*p, 1, 1, 128, 40, 0.1, 0, None) == 2
    assert lib.fa_fwd_fp8(*p, 1, 1, 128, 272, 0.1, 0, None) == 2
    assert lib.fa_fwd_fp8(*p, 1, 1, 128, 64, 0.0, 0, None) == 1
    assert lib.fa_fwd_fp8(*p[:6], p[0], p[7], 1, 1, 128, 64, 0.1, 0, None) == 1   # o aliases q8
    assert lib.fa_fwd_fp8(0, *p[1:], 1, 1, 128, 64, 0.1, 0, None) == 1


def _prototypes():
    """name -> parameter count of every function prototype in include/fa.h."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER, encoding="utf-8").read(), flags=re.S)
    protos = {}
    for m in re.finditer(r"\b(fa_[a-z_0-9]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        params = m.group(2).strip()
        protos[m.group(1)] = 0 if params in ("", "void") else len(params.split(","))
    return protos


def test_binding_signatures_match_header_prototypes():
    """Every ctypes signature passes exactly as many arguments as the C
    prototype takes (a mismatch would hand the library garbage)."""
    from io_aware_exact_14_gb300 import fa
    protos = _prototypes()
    assert set(protos) == set(declared_functions())
    for name, n in protos.items():
        assert name in fa.SIGNATURES, name
        assert len(fa.SIGNATURES[name][1]) == n, (name, len(fa.SIGNATURES[name][1]), n)


def _splitkv_ws(B, H, Nq, Nk, d, splits):
    n_kt = (Nk + 127) // 128
    w = min(splits, n_kt)
    per = -(-n_kt // w)
    n_used = -(-n_kt // per)
    rows = B * H * Nq * n_used * (4 if Nq <= 32 and d <= 64 else 1)   # four results per chunk there
    kd = 64 if d <= 64 else (128 if d <= 128 else 256)
    r256 = lambda x: (x + 255) // 256 * 256
    return r256(rows * kd * 4) + r256(rows * 4)


def test_splitkv_workspace_sizes(lib):
    """With an explicit chunk count no device is consulted: the size is the
    fp32 partial outputs (padded to the kernel's head width) plus the partial
    LSE of the chunks actually used (four results per chunk for up to 32 query
    rows at d <= 64), each rounded to 256 bytes."""
    for args in [(1, 1, 1, 1000, 128, 3), (2, 3, 5, 4097, 64, 7), (1, 2, 16, 129, 96, 4), (1, 2, 33, 900, 64, 2),
                 (1, 1, 1, 128, 40, 8), (2, 1, 33, 70000, 128, 300), (1, 4, 1, 9000, 256, 6),
                 (2, 2, 130, 300, 200, 2)]:
        assert lib.fa_fwd_splitkv_workspace_bytes(*args) == _splitkv_ws(*args), args
    assert lib.fa_fwd_splitkv_workspace_bytes(1, 1, 1, 0, 128, 4) == 0     # no keys
    assert lib.fa_fwd_splitkv_workspace_bytes(1, 1, 0, 100, 128, 4) == 0   # no queries
    assert lib.fa_fwd_splitkv_workspace_bytes(1, 1, 1, 100, 100, 4) == 0   # d not a multiple of 8
    assert lib.fa_fwd_splitkv_workspace_bytes(1, 1, 1, 100, 264, 4) == 0   # above the widest head


def test_fp8_splitkv_workspace_sizes_and_argument_checks(lib):
    """The e4m3 split path's partial rows are 128 floats wide for d <= 128 and
    256 beyond (four results per chunk for up to 32 query rows at d <= 128);
    its sizes follow the FP8 rule (d a multiple of 16 up to 256); argument
    errors come back before any device access."""
    for B, H, Nq, Nk, d, s in [(1, 1, 1, 1000, 128, 3), (2, 3, 5, 4097, 64, 7), (1, 2, 16, 129, 96, 4),
                               (1, 2, 1, 3000, 256, 5), (2, 1, 40, 900, 192, 2)]:
        n_kt = (Nk + 127) // 128
        per = -(-n_kt // min(s, n_kt))
        rows = B * H * Nq * -(-n_kt // per) * (4 if Nq <= 32 and d <= 128 else 1)
        width = 128 if d <= 128 else 256
        r256 = lambda x: (x + 255) // 256 * 256
        assert lib.fa_fwd_fp8_splitkv_workspace_bytes(B, H, Nq, Nk, d, s) == r256(rows * width * 4) + r256(rows * 4)
    assert lib.fa_fwd_fp8_splitkv_workspace_bytes(1, 1, 1, 100, 40, 4) == 0    # d not a multiple of 16
    assert lib.fa_fwd_fp8_splitkv_workspace_bytes(1, 1, 1, 100, 272, 4) == 0   # above the widest head
    assert lib.fa_fwd_fp8_splitkv_workspace_bytes(1, 1, 1, 0, 128, 4) == 0
    p = [FAKE + i * 0x100000 for i in range(9)]
    call = lambda *a: lib.fa_fwd_fp8_splitkv(*a)
    assert call(*p[:8], 1, 1, 1, 1000, 40, 0.1, 0, 2, p[8], 1 << 20, None) == 2     # d not a multiple of 16
    assert call(0, *p[1:8], 1, 1, 1, 1000, 64, 0.1, 0, 2, p[8], 1 << 20, None) == 1  # NULL q8
    assert call(*p[:6], p[0], p[7], 1, 1, 1, 1000, 64, 0.1, 1, 2, p[8], 1 << 20, None) == 1   # o aliases q8
    assert call(*p[:8], 1, 1, 1, 1000, 64, 0.1, 1, 2, p[8], 16, None) == 4          # workspace too small
    assert call(*p[:8], 1, 1, 0, 1000, 64, 0.1, 0, 2, None, 0, None) == 0            # Nq == 0: no-op
