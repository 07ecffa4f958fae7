"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments with the documented status codes
before touching the GPU (every call below fails validation, so none launches)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nea_attn.h")


@pytest.fixture(scope="module")
def nea():
    from causal_gqa_flashattention_gb300 import build, nea as binding
    build.build()
    binding.lib()
    return binding


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nea_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("nea_attn_fwd", "nea_attn_bwd", "nea_attn_bwd_workspace_bytes",
              "nea_attn_check_status", "nea_status_string", "nea_version",
              "nea_rope_table", "nea_rope_qk", "nea_attn_bwd_rope", "nea_attn_bwd_ex",
              "nea_attn_decode",
              "nea_attn_decode_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(nea):
    L = nea.lib()
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings(nea):
    for code in (0, -1, -2, -3, -4, -5):
        assert nea.status_string(code) not in ("", "unknown status")
    assert nea.status_string(7) == "unknown status"
    assert nea.lib().nea_version() >= 100


GOOD = dict(B=2, H=12, Hkv=4, N=1024, d=64, scale=0.125, causal=1, dtype=0)
P = 1 << 20  # a 16-byte aligned fake address: validation fails before any use


def fwd(nea, ptrs=None, **kw):
    a = dict(GOOD, **kw)
    ptrs = ptrs or [P] * 5
    return nea.lib().nea_attn_fwd(*[ctypes.c_void_p(p) for p in ptrs], a["B"], a["H"], a["Hkv"],
                                  a["N"], a["d"], a["scale"], a["causal"], a["dtype"], None)


def bwd(nea, ptrs=None, ws=P, ws_bytes=1 << 40, **kw):
    a = dict(GOOD, **kw)
    ptrs = ptrs or [P] * 9
    return nea.lib().nea_attn_bwd(*[ctypes.c_void_p(p) for p in ptrs], ctypes.c_void_p(ws),
                                  ws_bytes, a["B"], a["H"], a["Hkv"], a["N"], a["d"], a["scale"],
                                  a["causal"], a["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(H=12, Hkv=5), -1), (dict(B=0), -1), (dict(N=0), -1), (dict(d=0), -1),
    (dict(causal=2), -1), (dict(dtype=3), -1), (dict(scale=0.0), -1),
    (dict(scale=float("nan")), -1), (dict(scale=float("inf")), -1), (dict(scale=-1.0), -1),
    (dict(d=96), -2), (dict(d=32), -2), (dict(B=1 << 14, H=1 << 10, Hkv=1 << 10, N=1 << 24), -2),
    (dict(dtype=1, d=128), -2),
])
def test_invalid_and_unsupported_arguments(nea, kw, code):
    assert fwd(nea, **kw) == code
    assert bwd(nea, **kw) == code


@pytest.mark.parametrize("which", range(5))
def test_null_and_misaligned_pointers_fwd(nea, which):
    ptrs = [P] * 5
    ptrs[which] = 0
    assert fwd(nea, ptrs) == -1
    ptrs[which] = P + 8
    assert fwd(nea, ptrs) == -1


@pytest.mark.parametrize("which", range(9))
def test_null_and_misaligned_pointers_bwd(nea, which):
    ptrs = [P] * 9
    ptrs[which] = 0
    assert bwd(nea, ptrs) == -1
    ptrs[which] = P + 4
    assert bwd(nea, ptrs) == -1


def test_workspace_checks(nea):
    need = nea.bwd_workspace_bytes(2, 12, 4, 1024, 64, 0)
    rows = 2 * 12 * 1024
    assert need >= rows * 4 * 2 + rows * 64 * 4
    assert bwd(nea, ws=0) == -5
    assert bwd(nea, ws=P + 16) == -5          # not 256-byte aligned
    assert bwd(nea, ws_bytes=need - 1) == -5
    # fp32: D, L2 and the transposed Q, dO, K
    need32 = nea.bwd_workspace_bytes(2, 12, 4, 1024, 64, 1)
    assert need32 >= rows * 4 * 2 + 2 * rows * 64 * 4 + 2 * 4 * 1024 * 64 * 4
    assert nea.bwd_workspace_bytes(2, 12, 4, 1024, 128, 1) == 0   # fp32 supports d = 64 only
    assert nea.bwd_workspace_bytes(2, 12, 5, 1024, 64, 0) == 0
    # ragged N: per-row terms padded to whole 128-row tiles, dQ accumulator not
    need_r = nea.bwd_workspace_bytes(2, 12, 4, 1000, 64, 0)
    assert need_r >= 2 * (2 * 12 * 1024 * 4) + 2 * 12 * 1000 * 64 * 4
    assert need_r <= need


def test_rope_argument_checks(nea):
    """Host-side validation of the RoPE calls: rejected before any launch."""
    L = nea.lib()
    vp = ctypes.c_void_p
    assert L.nea_rope_table(vp(0), 128, 64, 10000.0, None) == -1          # null
    assert L.nea_rope_table(vp(P + 4), 128, 64, 10000.0, None) == -1      # misaligned
    assert L.nea_rope_table(vp(P), 128, 63, 10000.0, None) == -1          # odd d
    assert L.nea_rope_table(vp(P), 0, 64, 10000.0, None) == -1            # N < 1
    assert L.nea_rope_table(vp(P), 128, 64, 0.0, None) == -1              # base <= 0
    assert L.nea_rope_table(vp(P), 128, 64, float("nan"), None) == -1
    a = GOOD
    args = lambda ptrs, **kw: [vp(x) for x in ptrs] + [dict(a, **kw)[n] for n in
                                                      ("B", "H", "Hkv", "N", "d", "dtype")] + [None]
    assert L.nea_rope_qk(*args([P, P, P, P, 0])) == -1                     # null table
    assert L.nea_rope_qk(*args([P, P, P + 8, P, P])) == -1                 # misaligned Qr
    assert L.nea_rope_qk(*args([P] * 5, H=12, Hkv=5)) == -1                # bad group
    assert L.nea_rope_qk(*args([P] * 5, d=96)) == -2                       # unsupported d
    bw = [vp(P)] * 6 + [vp(0)] + [vp(P)] * 4
    assert L.nea_attn_bwd_rope(*bw, 1 << 40, 2, 12, 4, 1024, 64, 0.125, 1, 0, None) == -1


def test_decode_argument_checks(nea):
    L = nea.lib()
    vp = ctypes.c_void_p

    def dec(ptrs=None, ws=P, wsb=1 << 40, B=2, H=12, Hkv=4, nq=1, Lmax=1024, d=64, scale=0.125,
            dtype=0):
        ptrs = ptrs or [P] * 6
        return L.nea_attn_decode(*[vp(x) for x in ptrs], vp(ws), wsb, B, H, Hkv, nq, Lmax, d,
                                 scale, dtype, None)
    assert dec(ptrs=[P, P, P, 0, P, P]) == -1            # null lens
    assert dec(ptrs=[P, P, P, P + 2, P, P]) == -1        # misaligned lens
    assert dec(ptrs=[P + 8, P, P, P, P, P]) == -1        # misaligned Q
    assert dec(H=12, Hkv=5) == -1
    assert dec(nq=0) == -1
    assert dec(nq=8, Lmax=4) == -1                        # cache shorter than the new tokens
    assert dec(scale=0.0) == -1
    assert dec(d=96) == -2
    assert dec(nq=11) == -2                               # 3 * 11 query rows > 32
    assert dec(ws=0) == -5
    assert dec(wsb=16) == -5
    need = nea.decode_workspace_bytes(2, 12, 4, 1, 1024, 64)
    assert need >= 2 * 12 * 8 * 64 * 4 + 2 * 12 * 8 * 8
    assert nea.decode_workspace_bytes(2, 12, 4, 11, 1024, 64) == 0


def test_bwd_ex_argument_checks(nea):
    L = nea.lib()
    vp = ctypes.c_void_p
    ptrs = [vp(P)] * 6

    def ex(flags, cs=P, ws=P):
        return L.nea_attn_bwd_ex(*ptrs, vp(cs), flags, vp(P), vp(P), vp(P), vp(ws), 1 << 40,
                                 2, 12, 4, 1024, 64, 0.125, 1, 0, None)
    assert ex(2) == -1               # unknown flag bit
    assert ex(-1) == -1
    assert ex(1, cs=P + 4) == -1     # misaligned RoPE table
    assert ex(1, ws=0) == -5         # no workspace
    assert L.nea_attn_bwd_ex(*ptrs, vp(0), 1, vp(P), vp(P), vp(P), vp(P), 1 << 40, 2, 12, 5,
                             1024, 64, 0.125, 1, 0, None) == -1   # bad group
