"""C-ABI checks that need no GPU: the library loads, exports every function
include/gqa_attn.h declares, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa_attn.h")


@pytest.fixture(scope="module")
def lib():
    from causal_gqa_attention_fwd_gb300 import build
    build.build()
    import causal_gqa_attention_fwd_gb300 as g
    return g.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"GQA_ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for n in ("attn_fwd", "attn_bwd", "attn_varlen_fwd", "attn_varlen_bwd", "attn_bwd_workspace_size",
              "attn_varlen_bwd_workspace_size", "attn_status_string", "attn_get_device_status"):
        assert n in names


def test_exports_every_declared_symbol(lib):
    import causal_gqa_attention_fwd_gb300 as g
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
        assert n in g._binding.SIGNATURES, f"{n} has no binding"


def test_library_does_not_need_libcuda_at_load():
    import subprocess
    from causal_gqa_attention_fwd_gb300 import LIB_PATH
    out = subprocess.run(["ldd", LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out


NULL = None
A = 256   # a 16-byte-aligned fake device address: never dereferenced, rejected earlier or not launched


def fwd(lib, *, ptrs=(A, A, A, A, A), B=1, Hq=4, Hkv=2, T=16, D=64, causal=1, scale=0.125):
    return lib.attn_fwd(*ptrs, B, Hq, Hkv, T, D, causal, scale, None)


def test_fwd_validation(lib):
    assert fwd(lib, Hq=3, Hkv=2) == 2                    # Hq % Hkv
    assert fwd(lib, Hq=0) == 2
    assert fwd(lib, B=-1) == 2
    assert fwd(lib, D=96) == 3
    assert fwd(lib, D=256) == 3
    assert fwd(lib, ptrs=(NULL, A, A, A, A)) == 1
    assert fwd(lib, ptrs=(A, A, A, A, NULL)) == 1
    assert fwd(lib, ptrs=(A + 8, A, A, A, A)) == 4     # misaligned
    assert fwd(lib, ptrs=(A, A, A, A, A + 4)) == 4
    assert fwd(lib, ptrs=(NULL,) * 5, T=0) == 0          # empty: no-op
    assert fwd(lib, ptrs=(NULL,) * 5, B=0) == 0
    assert fwd(lib, scale=float("nan")) == 2


def vfwd(lib, *, ptrs=(A, A, A, A, A, A), n=2, total=10, maxlen=6, Hq=4, Hkv=2, D=128):
    return lib.attn_varlen_fwd(*ptrs, n, total, maxlen, Hq, Hkv, D, 1, 0.1, None)


def test_varlen_fwd_validation(lib):
    assert vfwd(lib, maxlen=11) == 2                     # longer than the batch
    assert vfwd(lib, n=-1) == 2
    assert vfwd(lib, ptrs=(A, A, A, A, A, NULL)) == 1    # cu_seqlens
    assert vfwd(lib, D=32) == 3
    assert vfwd(lib, ptrs=(NULL,) * 6, n=0, total=0, maxlen=0) == 0


def bwd(lib, *, ptrs=(A,) * 10, ws_bytes=1 << 40, B=1, Hq=4, Hkv=2, T=16, D=64):
    return lib.attn_bwd(*ptrs, ws_bytes, B, Hq, Hkv, T, D, 1, 0.125, None)


def test_bwd_validation(lib):
    assert bwd(lib, Hq=5) == 2
    assert bwd(lib, D=80) == 3
    p = list((A,) * 10)
    p[5] = NULL                                            # dout
    assert bwd(lib, ptrs=tuple(p)) == 1
    p = list((A,) * 10)
    p[8] = A + 2                                           # dv misaligned
    assert bwd(lib, ptrs=tuple(p)) == 4
    p = list((A,) * 10)
    p[9] = NULL                                            # workspace
    assert bwd(lib, ptrs=tuple(p)) == 6
    assert bwd(lib, ws_bytes=16) == 6                      # too small
    p = list((A,) * 10)
    p[9] = A + 16                                          # workspace not 256-aligned
    assert bwd(lib, ptrs=tuple(p)) == 6
    assert bwd(lib, ptrs=(NULL,) * 10, T=0) == 0


def test_noalloc_validation(lib):
    # returns before any CUDA call: shape, scratch limit, NULL pointers
    args = (A,) * 9
    assert lib.attn_bwd_noalloc(*args, 1, 3, 2, 16, 64, 1, 0.1, None) == 2
    assert lib.attn_bwd_noalloc(*args, 2, 1024, 8, 2048, 64, 1, 0.1, None) == 10
    assert lib.attn_bwd_noalloc(*((NULL,) * 9), 1, 4, 2, 0, 64, 1, 0.1, None) == 0
    assert lib.attn_bwd_noalloc(*((NULL,) * 9), 1, 4, 2, 16, 64, 1, 0.1, None) == 1
    assert lib.attn_bwd_noalloc_scratch_bytes() == 16 << 20


def test_workspace_sizes(lib):
    # Delta + LSE*log2e: 256-aligned f32 rows each; rows = B*Hq*roundup(T,128);
    # then 256 bytes for the dQ kernel's tile counter
    rows = 2 * 32 * 4096
    assert lib.attn_bwd_workspace_size(2, 32, 8, 4096, 128) == 2 * rows * 4 + 256
    rows = 1 * 4 * 256
    assert lib.attn_bwd_workspace_size(1, 4, 2, 129, 64) == 2 * rows * 4 + 256
    assert lib.attn_bwd_workspace_size(1, 3, 2, 16, 64) == 0
    pad = -(-(17000 + 132 * 16 + 256) // 128) * 128        # packed rows per head
    assert lib.attn_varlen_bwd_workspace_size(16, 17000, 16, 8, 128) == 2 * (-(-16 * pad * 4 // 256) * 256) + 256
    assert lib.attn_varlen_bwd_workspace_size(16, 17000, 16, 8, 64) == 2 * (-(-16 * pad * 4 // 256) * 256) + 256
    assert lib.attn_varlen_bwd_workspace_size(2, 10, 4, 2, 96) == 0
    # rotary backward: the two rotated f16 copies (256-aligned) before attn_bwd's workspace
    qk = -(-(2 * 32 * 4096 * 128 * 2) // 256) * 256 + 2 * 8 * 4096 * 128 * 2
    assert lib.attn_bwd_rope_workspace_size(2, 32, 8, 4096, 128) == (-(-qk // 256) * 256 +
                                                                     lib.attn_bwd_workspace_size(2, 32, 8, 4096, 128))


def test_inject_timeout_validation(lib):
    # test-only failure injection: kernel 0 (none) .. 3, limit 1..5000 ms; arming is host state only
    assert lib.attn_test_inject_timeout(4, 50) == 2
    assert lib.attn_test_inject_timeout(-1, 50) == 2
    assert lib.attn_test_inject_timeout(1, 0) == 2
    assert lib.attn_test_inject_timeout(1, 6000) == 2
    assert lib.attn_test_inject_timeout(2, 50) == 0
    assert lib.attn_test_inject_timeout(0, 1) == 0            # disarm


def test_debug_build_exports_the_same_symbols(lib):
    from causal_gqa_attention_fwd_gb300 import build
    dbg = ctypes.CDLL(build.build(debug=True))
    for n in declared_functions():
        assert hasattr(dbg, n), f"{n} not exported by the debug build"
    dbg.attn_is_debug_build.restype = ctypes.c_int
    assert dbg.attn_is_debug_build() == 1
    assert lib.attn_is_debug_build() == 0


def test_status_strings(lib):
    import causal_gqa_attention_fwd_gb300 as g
    for code in range(14):
        s = g.status_string(code)
        assert s and s != "unknown status"
    assert g.status_string(99) == "unknown status"


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from causal_gqa_attention_fwd_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        _binding.lib()


def dec(lib, *, ptrs=(A,) * 7, ws_bytes=1 << 40, B=1, Hq=4, Hkv=2, Tq=1, S=4096, D=64, scale=0.125, rope=(None, 0)):
    return lib.attn_decode_fwd(*ptrs, ws_bytes, B, Hq, Hkv, Tq, S, D, scale, *rope, None)


def test_decode_validation(lib):
    assert dec(lib, Tq=5, S=4) == 2                        # more new queries than the cache holds
    assert dec(lib, Hq=6, Hkv=4) == 2
    assert dec(lib, D=96) == 3
    assert dec(lib, B=-1) == 2
    assert dec(lib, scale=float("inf")) == 2
    p = list((A,) * 7)
    p[3] = NULL                                            # cache_lens
    assert dec(lib, ptrs=tuple(p)) == 1
    p = list((A,) * 7)
    p[1] = A + 8                                           # k_cache misaligned
    assert dec(lib, ptrs=tuple(p)) == 4
    p = list((A,) * 7)
    p[3] = A + 2                                           # cache_lens not 4-byte aligned
    assert dec(lib, ptrs=tuple(p)) == 4
    p = list((A,) * 7)
    p[6] = NULL                                            # workspace needed (split key range)
    assert dec(lib, ptrs=tuple(p)) == 6
    assert dec(lib, ws_bytes=64) == 6
    assert dec(lib, ptrs=(NULL,) * 7, B=0) == 0
    assert dec(lib, ptrs=(NULL,) * 7, Tq=0) == 0
    assert dec(lib, rope=(A + 4, 4096)) == 4                 # rotary table not 16-byte aligned
    assert dec(lib, rope=(A, 4095)) == 2                     # table shorter than the cache capacity


def ws_decode(units, slots, rows_ws, D):
    """partial O (f32, 256-byte aligned) + (max, sum) pairs per (unit, slot, row); none when
    a unit cannot be cut (one slot)"""
    if slots <= 1:
        return 0
    rows = units * slots * rows_ws
    return (rows * D * 4 + 255) // 256 * 256 + rows * 8


def test_decode_workspace_size(lib):
    # units = B * Hkv * ceil(G*Tq / 16); slots per unit = min(ceil(S / 128), 160); rows = min(G*Tq, 16)
    assert lib.attn_decode_workspace_size(1, 4, 2, 1, 4096, 64) == ws_decode(2, 32, 2, 64)
    assert lib.attn_decode_workspace_size(4, 8, 2, 1, 128, 128) == 0                            # one chunk
    assert lib.attn_decode_workspace_size(4, 8, 2, 1, 256, 128) == ws_decode(8, 2, 4, 128)
    assert lib.attn_decode_workspace_size(8, 32, 8, 1, 32768, 128) == ws_decode(64, 160, 4, 128)
    assert lib.attn_decode_workspace_size(2, 16, 2, 4, 640, 128) == ws_decode(8, 5, 16, 128)   # R = 32
    assert lib.attn_decode_workspace_size(8, 12, 2, 1, 2048, 128) == ws_decode(16, 16, 6, 128)
    assert lib.attn_decode_workspace_size(1, 1, 1, 1, 1 << 20, 64) == ws_decode(1, 160, 1, 64)
    assert lib.attn_decode_workspace_size(1, 4, 2, 1, 4096, 80) == 0                            # invalid D


def paged(lib, *, ptrs=(A,) * 8, ws_bytes=1 << 40, B=1, Hq=4, Hkv=2, Tq=1, psz=64, num_pages=8, max_pages=8, D=64,
          rope=(None, 0)):
    return lib.attn_decode_paged_fwd(*ptrs, ws_bytes, B, Hq, Hkv, Tq, psz, num_pages, max_pages, D, 0.125, *rope, None)


def test_decode_paged_validation(lib):
    assert paged(lib, psz=48) == 2                          # page size: 16, 32, 64 or a multiple of 128
    assert paged(lib, psz=8) == 2
    assert paged(lib, psz=0) == 2                           # no capacity
    assert paged(lib, num_pages=0) == 2
    assert paged(lib, Tq=3, psz=16, max_pages=0) == 2
    assert paged(lib, D=80) == 3
    p = list((A,) * 8)
    p[3] = NULL                                             # block_table
    assert paged(lib, ptrs=tuple(p)) == 1
    p = list((A,) * 8)
    p[3] = A + 2                                            # block_table not 4-byte aligned
    assert paged(lib, ptrs=tuple(p)) == 4
    p = list((A,) * 8)
    p[1] = A + 8                                            # k_pages misaligned
    assert paged(lib, ptrs=tuple(p)) == 4
    p = list((A,) * 8)
    p[7] = NULL                                             # workspace (8 pages of 64 = 4 chunks: units can be cut)
    assert paged(lib, ptrs=tuple(p)) == 6
    assert paged(lib, ptrs=(NULL,) * 8, B=0) == 0
    assert paged(lib, rope=(A, 511)) == 2                     # capacity 8 pages x 64


def test_decode_fp8_validation(lib):
    f = lambda **kw: lib.attn_decode_fp8_fwd(A, A, A, kw.get("ks", 0.01), 0.01, A, A, A, A, 1 << 40, 1, 4, 2, 1,
                                             4096, kw.get("D", 64), 0.125, None, 0, None)
    assert f(D=96) == 3
    assert f(ks=float("nan")) == 2
    g = lambda **kw: lib.attn_decode_paged_fp8_fwd(A, A, A, 0.01, 0.01, A, A, A, A, A, 1 << 40, 1, 4, 2, 1,
                                                   kw.get("psz", 64), 8, 8, 64, 0.125, None, 0, None)
    assert g(psz=40) == 2


def test_fwd_rope_validation(lib):
    """Rotary forward: the table and the workspace are checked before any
    launch (and before the architecture check)."""
    def f(ptrs=(A, A, A, A, A), ws=A, ws_bytes=1 << 40, tab=A, npos=4096, T=1000, D=128, Hq=4, Hkv=2):
        return lib.attn_fwd_rope(*ptrs, ws, ws_bytes, 2, Hq, Hkv, T, D, 1, 0.1, tab, npos, None)
    assert f(D=96) == 3
    assert f(Hq=3) == 2
    assert f(tab=NULL) == 1
    assert f(tab=A + 4) == 4
    assert f(npos=999) == 2                              # table shorter than T
    assert f(ws=NULL) == 6
    assert f(ws_bytes=lib.attn_fwd_rope_workspace_size(2, 4, 2, 1000, 128) - 1) == 6
    assert f(ws=A + 16) == 4                             # workspace needs 256-byte alignment
    assert f(ptrs=(NULL,) * 5, T=0, tab=NULL, ws=NULL) == 0    # empty: no-op


def test_fwd_rope_workspace_size(lib):
    # rotated f16 q (256-byte aligned section) then rotated f16 k
    assert lib.attn_fwd_rope_workspace_size(2, 4, 2, 1000, 128) == 2 * 4 * 1000 * 128 * 2 + 2 * 2 * 1000 * 128 * 2
    assert lib.attn_fwd_rope_workspace_size(1, 1, 1, 3, 64) == 512 + 3 * 64 * 2
    assert lib.attn_fwd_rope_workspace_size(1, 4, 2, 100, 96) == 0


def test_varlen_fwd_rope_validation(lib):
    def f(ptrs=(A,) * 6, n=2, total=10, maxlen=6, tab=A, npos=6, ws=A, ws_bytes=1 << 40, D=128):
        return lib.attn_varlen_fwd_rope(*ptrs, n, total, maxlen, 4, 2, D, 1, 0.1, tab, npos, ws, ws_bytes, None)
    assert f(D=96) == 3
    assert f(tab=NULL) == 1
    assert f(npos=5) == 2                                # table shorter than max_seqlen
    assert f(maxlen=11) == 2                             # max_seqlen > total
    assert f(ws=NULL) == 6
    assert f(ws=A + 32) == 4
    assert f(ptrs=(NULL,) * 6, n=0, tab=NULL, ws=NULL) == 0
    assert lib.attn_varlen_fwd_rope_workspace_size(10, 4, 2, 128) == 10 * 4 * 128 * 2 + 10 * 2 * 128 * 2


def test_python_binding_exposes_every_workspace_size():
    """Each *_workspace_size entry point of the header has a same-named
    Python function in the package, returning what the C call returns."""
    import causal_gqa_attention_fwd_gb300 as g
    lib = g.lib()
    cases = {
        "attn_fwd_rope_workspace_size": (2, 4, 2, 1000, 128),
        "attn_varlen_fwd_rope_workspace_size": (1000, 4, 2, 128),
        "attn_bwd_workspace_size": (2, 4, 2, 1000, 128),
        "attn_bwd_rope_workspace_size": (2, 4, 2, 1000, 128),
        "attn_varlen_bwd_workspace_size": (3, 1000, 4, 2, 128),
        "attn_varlen_bwd_rope_workspace_size": (3, 1000, 4, 2, 128),
        "attn_decode_workspace_size": (2, 8, 2, 1, 4096, 128),
    }
    for name, args in cases.items():
        assert getattr(g, name)(*args) == int(getattr(lib, name)(*args)) > 0, name
