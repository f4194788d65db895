"""CPU-only checks of the C-ABI library: it builds, loads, exports every
symbol that include/pkv.h declares, and rejects bad arguments on the host
(before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_attention_11_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                            src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_three_operations():
    names = declared_functions()
    for n in ("paged_kv_append", "paged_attn_decode", "paged_attn_varlen",
              "paged_attn_decode_workspace_size", "pkv_status_string", "pkv_last_cuda_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"libpkv.so does not export {n}"


def test_status_strings(lib):
    lib.pkv_status_string.restype = ctypes.c_char_p
    assert lib.pkv_status_string(0) == b"PKV_OK"
    assert lib.pkv_status_string(1) == b"PKV_ERR_INVALID"
    assert lib.pkv_status_string(2) == b"PKV_ERR_UNSUPPORTED"
    assert lib.pkv_status_string(3) == b"PKV_ERR_CUDA"


def _bind(lib):
    import paged_kv_attention_11_gb300._binding as b
    for name, args in b._SIGS.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = b._RES.get(name, ctypes.c_int)
    return lib


def test_host_validation_rejects_before_cuda(lib):
    L = _bind(lib)
    P = 0x1000  # fake, never dereferenced: validation fails first
    # append: negative token count, zero heads
    assert L.paged_kv_append(P, P, P, P, P, -1, 8, 128, 16, 64, None, None) == 1
    assert L.paged_kv_append(P, P, P, P, P, 4, 0, 128, 16, 64, None, None) == 1
    # append: head_dim not a multiple of 8 -> unsupported
    assert L.paged_kv_append(P, P, P, P, P, 4, 8, 100, 16, 64, None, None) == 2
    # append of zero rows is a no-op
    assert L.paged_kv_append(None, None, None, None, None, 0, 8, 128, 16, 64, None, None) == 0
    # decode: H_q not a multiple of H_kv
    assert L.paged_attn_decode(P, P, P, P, P, 4, P, 2, 6, 4, 128, 16, 64, 64, 0.1, 0, P,
                               1 << 20, None, None) == 1
    # decode: head_dim 96 / page size 8 / group of 16 unsupported
    assert L.paged_attn_decode(P, P, P, P, P, 4, P, 2, 8, 2, 96, 16, 64, 64, 0.1, 0, P,
                               1 << 20, None, None) == 2
    assert L.paged_attn_decode(P, P, P, P, P, 4, P, 2, 8, 2, 128, 8, 64, 64, 0.1, 0, P,
                               1 << 20, None, None) == 2
    assert L.paged_attn_decode(P, P, P, P, P, 4, P, 2, 32, 2, 128, 16, 64, 64, 0.1, 0, P,
                               1 << 20, None, None) == 2
    # decode: NaN scale, missing pointers
    assert L.paged_attn_decode(P, P, P, P, P, 4, P, 2, 8, 2, 128, 16, 64, 64, float("nan"), 0,
                               P, 1 << 20, None, None) == 1
    assert L.paged_attn_decode(None, P, P, P, P, 4, P, 2, 8, 2, 128, 16, 64, 64, 0.1, 0, P,
                               1 << 20, None, None) == 1
    # decode: misaligned q
    assert L.paged_attn_decode(P, P + 2, P, P, P, 4, P, 2, 8, 2, 128, 16, 64, 64, 0.1, 0, P,
                               1 << 20, None, None) == 1
    # varlen: window without causal, causal not 0/1
    assert L.paged_attn_varlen(P, P, P, P, P, P, P, 4, 2, 64, 64, 100, 8, 2, 128, 16, 64,
                               0.1, 0, 16, None, None) == 1
    assert L.paged_attn_varlen(P, P, P, P, P, P, P, 4, 2, 64, 64, 100, 8, 2, 128, 16, 64,
                               0.1, 2, 0, None, None) == 1
    # varlen: group that does not divide 128
    assert L.paged_attn_varlen(P, P, P, P, P, P, P, 4, 2, 64, 64, 100, 6, 2, 128, 16, 64,
                               0.1, 1, 0, None, None) == 2
    # zero-size batches are no-ops
    assert L.paged_attn_decode(None, None, None, None, None, 4, None, 0, 8, 2, 128, 16, 64, 0,
                               0.1, 0, None, 0, None, None) == 0


def test_rope_entry_points_validate_on_host(lib):
    L = _bind(lib)
    P = 0x1000  # fake, never dereferenced: validation fails first
    nan = float("nan")

    def app(q=P, T=4, H_q=8, H_kv=2, D=128, max_pos=64, eps=1e-6, cs=P, slots=P):
        return L.paged_kv_append_rope(q, P, P, P, P, slots, P, cs, max_pos, None, None, eps, T,
                                      H_q, H_kv, D, 16, 64, None, None)
    assert app(T=-1) == 1
    assert app(max_pos=0) == 1
    assert app(eps=nan) == 1 and app(eps=-1.0) == 1
    assert app(H_q=0) == 1                 # q given without heads
    assert app(H_kv=0) == 1
    assert app(D=96) == 2                  # head_dim outside {64, 128, 256}
    assert app(cs=P + 4) == 1              # misaligned table
    assert app(slots=None) == 1            # missing slot mapping
    assert app(T=1 << 28) == 2             # more vectors than one launch indexes
    assert app(T=0, q=None, cs=None, slots=None) == 0   # no tokens: no-op
    # the table: odd head_dim, non-positive / NaN / infinite theta, misaligned
    assert L.pkv_rope_table(P, 16, 127, 1e6, None) == 1
    assert L.pkv_rope_table(P, 16, 128, 0.0, None) == 1
    assert L.pkv_rope_table(P, 16, 128, nan, None) == 1
    assert L.pkv_rope_table(P, 16, 128, float("inf"), None) == 1
    assert L.pkv_rope_table(P + 8, 16, 128, 1e6, None) == 1
    assert L.pkv_rope_table(None, 0, 128, 1e6, None) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import paged_kv_attention_11_gb300._binding as b
    monkeypatch.setattr(b, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(b, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        b.lib()


def test_product_package_does_not_import_oracle():
    pkg = os.path.join(ROOT, "paged_kv_attention_11_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.replace("oracles", ""), f


def _declared_signatures():
    """name -> list of parameter C types, from include/pkv.h."""
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    sigs = {}
    for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(([^)]*)\)\s*;",
                         src, flags=re.M):
        params = [p.strip() for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        sigs[m.group(1)] = params
    return sigs


def _ctype_of(param: str):
    if "*" in param:
        return ctypes.c_void_p
    base = param.rsplit(" ", 1)[0].replace("const ", "").strip()
    return {"int32_t": ctypes.c_int32, "int64_t": ctypes.c_int64, "float": ctypes.c_float,
            "double": ctypes.c_double, "size_t": ctypes.c_size_t}[base]


def test_binding_signatures_match_the_header():
    # every ctypes prototype in the binding has the header's arity and types
    import paged_kv_attention_11_gb300._binding as b
    sigs = _declared_signatures()
    assert set(b._SIGS) == set(sigs), set(b._SIGS) ^ set(sigs)
    for name, args in b._SIGS.items():
        want = [_ctype_of(p) for p in sigs[name]]
        assert args == want, (name, args, want)


def test_shared_prefix_decode_validates_on_host(lib):
    L = _bind(lib)
    P = 0x1000  # fake, never dereferenced: validation fails first

    def call(gs=4, pl=P, H_q=32, H_kv=8, D=128, ws=P, B=8):
        return L.paged_attn_decode_shared_prefix(P, P, P, P, P, 4, P, B, gs, pl, H_q, H_kv, D,
                                                 16, 64, 64, 0.1, ws, 1 << 24, None, None)
    assert call(gs=0) == 1                 # empty groups
    assert call(pl=None) == 1              # missing prefix lengths
    assert call(ws=P + 64) == 1            # workspace not 256-byte aligned
    assert call(H_q=30) == 1               # H_q not a multiple of H_kv
    assert call(gs=8) == 2                 # 8 members x 4 heads: 32 rows > 16 at head_dim 128
    assert call(D=512, H_q=8, H_kv=8, gs=1) == 2   # head_dim 512 has no prefix pass
    assert call(B=0, gs=4) == 0            # empty batch: no-op
    # head_dim 1024 is no shape of either call
    assert L.paged_attn_varlen(P, P, P, P, P, P, P, 4, 2, 64, 64, 100, 8, 2, 1024, 16, 64,
                               0.1, 1, 0, None, None) == 2
    assert L.paged_attn_decode(P, P, P, P, P, 4, P, 2, 8, 2, 1024, 16, 64, 64, 0.1, 0, P,
                               1 << 20, None, None) == 2


def test_decode_append_validates_on_host(lib):
    L = _bind(lib)
    P = 0x1000  # fake, never dereferenced: validation fails first

    def call(kn=P, vn=P, H_q=32, D=128, ws=P, B=8, scale=0.1):
        return L.paged_attn_decode_append(P, P, kn, vn, P, P, P, 4, P, B, H_q, 8, D, 16, 64, 64,
                                          scale, 0, ws, 1 << 24, None, None)
    assert call(kn=None) == 1              # missing new K rows
    assert call(vn=P + 8) == 1             # misaligned new V rows
    assert call(ws=P + 64) == 1            # workspace not 256-byte aligned
    assert call(H_q=30) == 1               # H_q not a multiple of H_kv
    assert call(scale=float("nan")) == 1
    assert call(D=96) == 2                 # head_dim outside the decode shapes
    assert call(B=0, kn=None, vn=None) == 0  # empty batch: no-op


def test_mixed_append_validates_on_host(lib):
    L = _bind(lib)
    P = 0x1000  # fake, never dereferenced: validation fails first

    def call(kn=P, vn=P, sm=P, T=16, ws=P, D=128, H_q=32, B=8):
        return L.paged_attn_mixed_append(
            P, P, P, 4, P, B, 64, P, P, P, P, P, 4, 2, 64, 128, 100,
            kn, vn, sm, T, P, P, H_q, 8, D, 16, 64, 0.1, 0, 0, ws, 1 << 24, None, None)
    assert call(kn=None) == 1              # missing new K rows
    assert call(vn=P + 8) == 1             # misaligned new V rows
    assert call(sm=None) == 1              # missing slot mapping
    assert call(T=-1) == 1                 # negative token count
    assert call(ws=None) == 1              # appending needs the workspace (grid barrier)
    assert call(ws=P + 64) == 1            # workspace not 256-byte aligned
    assert call(H_q=30) == 1               # H_q not a multiple of H_kv
    assert call(D=64) == 2                 # head_dim other than 128


def test_copy_validates_on_host(lib):
    # sizes, alignment and overlap are checked before any CUDA call
    L = _bind(lib)
    a, b = 1 << 20, 1 << 21
    assert L.pkv_copy(b, a, 8, None) == 1          # not a multiple of 16
    assert L.pkv_copy(b + 8, a, 16, None) == 1     # misaligned destination
    assert L.pkv_copy(b, a + 4, 16, None) == 1     # misaligned source
    assert L.pkv_copy(a + 16, a, 64, None) == 1    # overlapping ranges
    assert L.pkv_copy(None, a, 16, None) == 1
    assert L.pkv_copy(b, a, 0, None) == 0          # nothing to copy
