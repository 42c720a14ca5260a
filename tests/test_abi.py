"""The C-ABI library loads and exports what include/relattn.h declares.

Runs without a GPU: only host-side entry points are called (no kernel).
"""

import ctypes
import os
import re
import subprocess

import pytest

from paged_relative_bias_gb300 import build as B
from paged_relative_bias_gb300 import relattn as R

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "relattn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(relattn_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return R.lib()


def test_header_lists_the_entry_points():
    names = declared_functions()
    assert "relattn_decode" in names and "relattn_prefill" in names
    assert set(names) == set(R.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.lib_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (relattn_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_no_torch_types_in_the_abi():
    text = open(HEADER).read()
    for bad in ("torch", "at::", "Tensor", "c10"):
        assert bad not in text


def test_status_strings_and_version(lib):
    assert R.status_string(0) == "ok"
    assert "invalid" in R.status_string(1)
    assert "unsupported" in R.status_string(2)
    assert "workspace" in R.status_string(3)
    assert "CUDA" in R.status_string(4)
    assert lib.relattn_abi_version() == 100


def test_invalid_arguments_rejected_on_host(lib):
    """Null or inconsistent arguments fail before any CUDA work."""
    dims = R.Dims(1, 4, 2, 0, 0, 0)
    good = R.KVCacheDesc(16, 16, 2, 128, 1, 128, 128)
    rc = lib.relattn_decode(None, None, ctypes.byref(good), None, None, 0, 64,
                            ctypes.byref(dims), None, None, 0, None)
    assert rc == R.ERR_INVALID_ARG
    bad_bs = R.KVCacheDesc(16, 16, 2, 64, 1, 128, 128)
    rc = lib.relattn_decode(16, 16, ctypes.byref(bad_bs), 16, 16, 0, 64,
                            ctypes.byref(dims), 16, 16, 1 << 20, None)
    assert rc == R.ERR_UNSUPPORTED
    bad_dv = R.KVCacheDesc(16, 16, 2, 128, 1, 128, 96)
    rc = lib.relattn_decode(16, 16, ctypes.byref(bad_dv), 16, 16, 0, 64,
                            ctypes.byref(dims), 16, 16, 1 << 20, None)
    assert rc == R.ERR_UNSUPPORTED
    misaligned = R.KVCacheDesc(17, 16, 2, 128, 1, 128, 128)
    rc = lib.relattn_decode(16, 16, ctypes.byref(misaligned), 16, 16, 0, 64,
                            ctypes.byref(dims), 16, 16, 1 << 20, None)
    assert rc == R.ERR_INVALID_ARG
    gqa = R.Dims(1, 5, 2, 0, 0, 0)  # 5 query heads over 2 KV heads
    two = R.KVCacheDesc(16, 16, 2, 128, 2, 128, 128)
    rc = lib.relattn_decode(16, 16, ctypes.byref(two), 16, 16, 0, 64,
                            ctypes.byref(gqa), 16, 16, 1 << 20, None)
    assert rc == R.ERR_INVALID_ARG
    wide = R.Dims(1, 34, 2, 0, 0, 0)  # 17 query heads per KV head
    rc = lib.relattn_decode(16, 16, ctypes.byref(two), 16, 16, 0, 64,
                            ctypes.byref(wide), 16, 16, 1 << 20, None)
    assert rc == R.ERR_UNSUPPORTED
    rc = lib.relattn_prefill(None, None, None, None, None, ctypes.byref(good), None, None,
                             0, 64, ctypes.byref(dims), None, None, 0, None)
    assert rc == R.ERR_INVALID_ARG


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(R, "_LIB", None)
    monkeypatch.setattr(R, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        R.lib()


def test_bound_decode_marshals_like_the_wrapper(monkeypatch):
    """bind_decode checks its inputs once and then makes the same C call,
    with the same arguments, as relattn_decode (a fake library records them)."""
    import torch
    calls = []

    class Fake:
        def __getattr__(self, name):
            def f(*args):
                calls.append((name, args[:-1]))
                return 0
            f.__name__ = name
            return f

    monkeypatch.setattr(R, "_LIB", Fake())
    monkeypatch.setattr(R, "lib", lambda: R._LIB)
    monkeypatch.setattr(R, "_stream", lambda dev: 0)
    B, Hq, Hkv = 2, 8, 2
    q = torch.zeros((B, Hq, 128), dtype=torch.bfloat16)
    rel = torch.zeros((B, Hq, 64), dtype=torch.float32)
    kc = torch.zeros((4, 128, Hkv, 128), dtype=torch.bfloat16)
    vc = torch.zeros((4, 128, Hkv, 128), dtype=torch.bfloat16)
    bt = torch.zeros((B, 2), dtype=torch.int32)
    sl = torch.ones((B,), dtype=torch.int32)
    out = torch.empty((B, Hq, 128), dtype=torch.bfloat16)
    ws = torch.empty(4096, dtype=torch.uint8)
    R.relattn_decode(q, rel, kc, vc, bt, sl, 0, 64, out=out, workspace=ws)
    run = R.bind_decode(q, rel, kc, vc, bt, sl, 0, 64, out, ws)
    assert len(calls) == 1  # binding makes no call
    run()
    run()
    assert [c[0] for c in calls] == ["relattn_decode"] * 3

    def plain(args):  # pointers and ints; structures by their fields
        return [tuple(getattr(a._obj, f[0]) for f in a._obj._fields_) if hasattr(a, "_obj")
                else a for a in args]

    assert plain(calls[1][1]) == plain(calls[0][1]) == plain(calls[2][1])
    with pytest.raises(ValueError):
        R.bind_decode(q, rel[:, :, :32], kc, vc, bt, sl, 0, 64, out, ws)


def test_ctypes_structures_match_the_header():
    """The binding's ctypes mirrors of the header's structures have the same
    fields, in the same order, with the same C types."""
    text = open(os.path.join(ROOT, "include", "relattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    ctype = {"int32_t": ctypes.c_int32, "float": ctypes.c_float}
    mirrors = {"relattn_kv_cache": R.KVCacheDesc, "relattn_dims": R.Dims,
               "relattn_options": R.Options}
    for name, cls in mirrors.items():
        body = re.search(r"typedef struct %s \{(.*?)\} %s;" % (name, name), text, re.S).group(1)
        fields = []
        for decl in filter(None, (d.strip() for d in body.split(";"))):
            m = re.match(r"(?:const\s+)?(\w+)\s*(\*?)\s*(\w+)$", " ".join(decl.split()))
            assert m, decl
            base, star, field = m.groups()
            fields.append((field, ctypes.c_void_p if star else ctype[base]))
        assert [(f, t) for f, t in cls._fields_] == fields, name


def test_options_and_cache_write_rejected_on_host(lib):
    """relattn_options and relattn_cache_write arguments that are not offered
    fail before any CUDA work (no GPU is needed to see the codes)."""
    dims = R.Dims(1, 4, 2, 16, 16, 0)
    cache = R.KVCacheDesc(16, 16, 2, 128, 1, 128, 128)
    e4m3_64 = R.KVCacheDesc(16, 16, 2, 128, 1, 128, 64)

    def opts(rel=R.DTYPE_F32, out=R.DTYPE_BF16, sink=None, kv=R.DTYPE_BF16, ks=1.0, vs=1.0,
             ls=None):
        return R.Options(rel, out, sink, None, kv, ks, vs, ls)

    def decode_ex(o):
        return lib.relattn_decode_ex(16, 16, ctypes.byref(o), ctypes.byref(cache), 16, 16, 1, 0,
                                     64, ctypes.byref(dims), 16, 16, 1 << 20, None)

    assert decode_ex(opts(rel=7)) == R.ERR_INVALID_ARG            # unknown rel type
    assert decode_ex(opts(out=R.DTYPE_E4M3)) == R.ERR_INVALID_ARG  # e4m3 is no output type
    assert decode_ex(opts(sink=18)) == R.ERR_INVALID_ARG           # sink not 4-byte aligned
    assert decode_ex(opts(ls=18)) == R.ERR_INVALID_ARG             # factors not aligned
    assert decode_ex(opts(kv=R.DTYPE_E4M3, ks=0.0)) == R.ERR_INVALID_ARG  # scale must be > 0
    assert decode_ex(opts(kv=5)) == R.ERR_INVALID_ARG

    def write(k=16, v=16, o=None, c=cache, d=dims, ws=16, ws_bytes=256):
        return lib.relattn_cache_write(k, v, None if o is None else ctypes.byref(o), 16,
                                       ctypes.byref(c), 16, 16, ctypes.byref(d), ws, ws_bytes,
                                       None)

    assert write(k=None) == R.ERR_INVALID_ARG
    assert write(k=24) == R.ERR_INVALID_ARG                      # k not 16-byte aligned
    assert write(ws_bytes=128) == R.ERR_WORKSPACE                # below the status word
    assert write(o=opts(rel=9)) == R.ERR_INVALID_ARG
    assert write(o=opts(kv=R.DTYPE_E4M3, ks=0.5, vs=0.5), c=e4m3_64) == R.ERR_UNSUPPORTED
    assert write(d=R.Dims(70000, 4, 2, 16, 16, 0)) == R.ERR_UNSUPPORTED  # > 65535 sequences
    assert write(d=R.Dims(0, 4, 2, 0, 0, 0)) == R.OK             # nothing to write: no launch
