"""Python binding of the relattn C ABI (``include/relattn.h``).

Argument marshalling only: every step of the attention runs in the CUDA
library ``lib/librelattn.so``.  Tensors are torch device tensors; their data
pointers and the current CUDA stream are handed to the C entry points.  There
is no fallback: if the library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_int32, c_size_t, c_uint32, c_void_p

import torch

from . import build as _build

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_WORKSPACE = 3
ERR_CUDA = 4

DEV_BAD_BLOCK_ID = 0x1
DEV_BAD_LENGTH = 0x2
DEV_WAIT_TIMEOUT = 0x4
DEV_Q_RANGE = 0x8

EXPORTS = (
    "relattn_workspace_size",
    "relattn_workspace_init",
    "relattn_decode",
    "relattn_prefill",
    "relattn_read_status",
    "relattn_status_string",
    "relattn_debug_walk_decode",
    "relattn_debug_walk_prefill",
    "relattn_abi_version",
    "relattn_decode_noalloc",
    "relattn_decode_multi",
    "relattn_decode_ex",
    "relattn_prefill_ex",
    "relattn_cache_write",
    "relattn_debug_wait_timeout",
    "relattn_debug_decode_give_up",
    "relattn_debug_walk_decode_ex",
    "relattn_debug_walk_prefill_ex",
    "relattn_decode_noalloc_status",
)

DTYPE_F32 = 0
DTYPE_BF16 = 1
DTYPE_E4M3 = 2
_CACHE_DTYPES = (torch.bfloat16, torch.float8_e4m3fn)
_DTYPE_CODE = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16}


class KVCacheDesc(ctypes.Structure):
    _fields_ = [("k", c_void_p), ("v", c_void_p), ("num_blocks", c_int32),
                ("block_size", c_int32), ("num_kv_heads", c_int32),
                ("d_qk", c_int32), ("d_v", c_int32)]


class Dims(ctypes.Structure):
    _fields_ = [("batch", c_int32), ("num_q_heads", c_int32),
                ("max_blocks_per_seq", c_int32), ("num_tokens", c_int32),
                ("max_q_len", c_int32), ("num_ctas", c_int32)]


class Options(ctypes.Structure):
    _fields_ = [("rel", c_int32), ("out", c_int32), ("sink", c_void_p), ("gate", c_void_p),
                ("kv", c_int32), ("k_scale", c_float), ("v_scale", c_float),
                ("logit_scale", c_void_p)]


class RelattnError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} (code {code})")
        self.code = code


_LIB = None


def library_path() -> str:
    return _build.lib_path()


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"relattn CUDA library not found at {path}; build it with "
            "`python -m paged_relative_bias_gb300.build` (there is no CPU fallback)")
    L = ctypes.CDLL(path)
    P, S = POINTER(KVCacheDesc), POINTER(Dims)
    L.relattn_workspace_size.argtypes = [S, P]
    L.relattn_workspace_size.restype = c_size_t
    L.relattn_workspace_init.argtypes = [c_void_p, c_size_t, c_void_p]
    L.relattn_workspace_init.restype = c_int
    L.relattn_decode.argtypes = [c_void_p, c_void_p, P, c_void_p, c_void_p, c_int32,
                                 c_int32, S, c_void_p, c_void_p, c_size_t, c_void_p]
    L.relattn_decode.restype = c_int
    L.relattn_prefill.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, P,
                                  c_void_p, c_void_p, c_int32, c_int32, S, c_void_p,
                                  c_void_p, c_size_t, c_void_p]
    L.relattn_prefill.restype = c_int
    L.relattn_read_status.argtypes = [c_void_p, POINTER(c_uint32), c_void_p]
    L.relattn_read_status.restype = c_int
    L.relattn_status_string.argtypes = [c_int]
    L.relattn_status_string.restype = c_char_p
    L.relattn_debug_walk_decode.argtypes = [c_void_p, c_void_p, c_int32, P, S, c_void_p,
                                            c_int32, c_void_p, c_void_p, c_size_t, c_void_p]
    L.relattn_debug_walk_decode.restype = c_int
    L.relattn_debug_walk_prefill.argtypes = [c_void_p, c_void_p, c_void_p, c_int32, P, S,
                                             c_void_p, c_int32, c_void_p, c_void_p,
                                             c_size_t, c_void_p]
    L.relattn_debug_walk_prefill.restype = c_int
    L.relattn_debug_walk_prefill_ex.argtypes = [c_void_p, c_void_p, c_void_p, c_int32,
                                                POINTER(Options), P, S, c_void_p, c_int32,
                                                c_void_p, c_void_p, c_size_t, c_void_p]
    L.relattn_debug_walk_prefill_ex.restype = c_int
    L.relattn_decode_noalloc_status.argtypes = [c_void_p, c_void_p]
    L.relattn_decode_noalloc_status.restype = c_int
    L.relattn_decode_noalloc.argtypes = [c_void_p, c_void_p, P, c_void_p, c_void_p, c_int32,
                                         c_int32, S, c_void_p, c_void_p]
    L.relattn_decode_noalloc.restype = c_int
    L.relattn_decode_multi.argtypes = [c_void_p, c_void_p, P, c_void_p, c_void_p, c_int32,
                                       c_int32, c_int32, S, c_void_p, c_void_p, c_size_t,
                                       c_void_p]
    L.relattn_decode_multi.restype = c_int
    L.relattn_decode_ex.argtypes = [c_void_p, c_void_p, POINTER(Options), P, c_void_p,
                                    c_void_p, c_int32, c_int32, c_int32, S, c_void_p, c_void_p,
                                    c_size_t, c_void_p]
    L.relattn_decode_ex.restype = c_int
    L.relattn_prefill_ex.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, POINTER(Options),
                                     c_void_p, P, c_void_p, c_void_p, c_int32, c_int32, S,
                                     c_void_p, c_void_p, c_size_t, c_void_p]
    L.relattn_prefill_ex.restype = c_int
    L.relattn_cache_write.argtypes = [c_void_p, c_void_p, POINTER(Options), c_void_p, P,
                                      c_void_p, c_void_p, S, c_void_p, c_size_t, c_void_p]
    L.relattn_cache_write.restype = c_int
    L.relattn_debug_wait_timeout.argtypes = [c_void_p, c_size_t, c_void_p]
    L.relattn_debug_wait_timeout.restype = c_int
    L.relattn_debug_decode_give_up.argtypes = [c_void_p, c_void_p, P, c_void_p, c_void_p,
                                               c_int32, c_int32, S, c_void_p, c_void_p,
                                               c_size_t, c_int32, c_void_p]
    L.relattn_debug_decode_give_up.restype = c_int
    L.relattn_debug_walk_decode_ex.argtypes = [c_void_p, c_void_p, c_int32, c_int32,
                                               POINTER(Options), P, S, c_void_p, c_int32,
                                               c_void_p, c_void_p, c_size_t, c_void_p]
    L.relattn_debug_walk_decode_ex.restype = c_int
    L.relattn_abi_version.argtypes = []
    L.relattn_abi_version.restype = c_int
    _LIB = L
    return L


def status_string(code: int) -> str:
    return lib().relattn_status_string(code).decode()


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise RelattnError(rc, what)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _need(t: torch.Tensor, name: str, dtype, dims: int, device) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dimensions, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def cache_desc(k_cache: torch.Tensor, v_cache: torch.Tensor) -> KVCacheDesc:
    """bf16 caches are [NB, 128, Hkv, d]; e4m3 caches are head-major,
    [NB, Hkv, 128, d]."""
    if k_cache.dtype == torch.float8_e4m3fn:
        return KVCacheDesc(k_cache.data_ptr(), v_cache.data_ptr(), k_cache.shape[0],
                           k_cache.shape[2], k_cache.shape[1], k_cache.shape[3],
                           v_cache.shape[3])
    return KVCacheDesc(k_cache.data_ptr(), v_cache.data_ptr(), k_cache.shape[0],
                       k_cache.shape[1], k_cache.shape[2], k_cache.shape[3],
                       v_cache.shape[3])


def workspace_size(dims: Dims, cache: KVCacheDesc) -> int:
    n = lib().relattn_workspace_size(ctypes.byref(dims), ctypes.byref(cache))
    if n == 0:
        raise RelattnError(ERR_INVALID_ARG, "relattn_workspace_size")
    return int(n)


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-filled workspace buffer (allocated by torch, initialised by the library)."""
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    _check(lib().relattn_workspace_init(ws.data_ptr(), nbytes, _stream(ws.device)),
           "relattn_workspace_init")
    return ws


def read_status(workspace: torch.Tensor) -> int:
    st = c_uint32(0)
    _check(lib().relattn_read_status(workspace.data_ptr(), ctypes.byref(st),
                                     _stream(workspace.device)), "relattn_read_status")
    return int(st.value)


def clear_status(workspace: torch.Tensor) -> None:
    _check(lib().relattn_workspace_init(workspace.data_ptr(), workspace.numel(),
                                        _stream(workspace.device)), "relattn_workspace_init")


def decode_dims(q, block_table, num_ctas=0) -> Dims:
    return Dims(q.shape[0], q.shape[1], block_table.shape[1], 0, 0, num_ctas)


def _options(rel, out_dtype, sink=None, gate=None, rows_shape=None, device=None,
             k_cache=None, k_scale=None, v_scale=None, logit_scale=None) -> Options:
    """The *_ex options; sink / gate are float32 [rows..., Hq] tensors or None,
    logit_scale a float32 [rows...] tensor or None; an e4m3 cache
    (float8_e4m3fn tensors) needs its two scales."""
    if rel.dtype not in _DTYPE_CODE:
        raise TypeError(f"rel must be float32 or bfloat16, got {rel.dtype}")
    if out_dtype not in _DTYPE_CODE:
        raise TypeError(f"out must be bfloat16 or float32, got {out_dtype}")
    for name, t in (("sink", sink), ("gate", gate)):
        if t is not None:
            _need(t, name, torch.float32, len(rows_shape), device)
            if tuple(t.shape) != tuple(rows_shape):
                raise ValueError(f"{name} must be {list(rows_shape)}, got {tuple(t.shape)}")
    if logit_scale is not None:
        _need(logit_scale, "logit_scale", torch.float32, len(rows_shape) - 1, device)
        if tuple(logit_scale.shape) != tuple(rows_shape[:-1]):
            raise ValueError(f"logit_scale must be {list(rows_shape[:-1])}, "
                             f"got {tuple(logit_scale.shape)}")
    kv, ks, vs = DTYPE_BF16, 1.0, 1.0
    if k_cache is not None and k_cache.dtype == torch.float8_e4m3fn:
        if k_scale is None or v_scale is None:
            raise ValueError("an e4m3 cache needs k_scale and v_scale")
        kv, ks, vs = DTYPE_E4M3, float(k_scale), float(v_scale)
    return Options(_DTYPE_CODE[rel.dtype], _DTYPE_CODE[out_dtype], _ptr(sink), _ptr(gate), kv,
                   ks, vs, _ptr(logit_scale))


def _need_cache(k_cache, v_cache, device) -> None:
    if k_cache.dtype not in _CACHE_DTYPES or v_cache.dtype != k_cache.dtype:
        raise TypeError("k_cache / v_cache must both be bfloat16 or both float8_e4m3fn")
    _need(k_cache, "k_cache", k_cache.dtype, 4, device)
    _need(v_cache, "v_cache", v_cache.dtype, 4, device)


def _plain(rel, out_dtype, sink, gate, k_cache=None, logit_scale=None) -> bool:
    return (rel.dtype == torch.float32 and out_dtype == torch.bfloat16 and sink is None
            and gate is None and logit_scale is None
            and (k_cache is None or k_cache.dtype == torch.bfloat16))


def relattn_decode(q, rel, k_cache, v_cache, block_table, seq_lens, window: int,
                   rel_extent: int, out=None, workspace=None, num_ctas: int = 0,
                   out_dtype=torch.bfloat16, sink=None, gate=None, k_scale=None,
                   v_scale=None, logit_scale=None):
    """Paged relative-bias decode; see ``relattn_decode`` in include/relattn.h.

    rel may be float32 or bfloat16 and out bfloat16 or float32 (``out``'s own
    dtype when it is given); sink / gate are optional float32 [B, Hq] logits
    (the gated output with a sink); float8_e4m3fn caches take k_scale and
    v_scale; logit_scale is an optional float32 [B] of log-position factors.
    Anything but fp32 rel, bf16 out, a bf16 cache and none of the optional
    inputs goes through ``relattn_decode_ex``.
    """
    if not _plain(rel, out.dtype if out is not None else out_dtype, sink, gate, k_cache,
                  logit_scale):
        if q.dim() != 3 or rel.dim() != 3:
            raise ValueError("q must be [B, Hq, d_qk] and rel [B, Hq, rel_extent]")
        o = relattn_decode_multi(q[:, None], rel[:, None], k_cache, v_cache, block_table,
                                 seq_lens, window, rel_extent,
                                 out=None if out is None else out[:, None],
                                 workspace=workspace, num_ctas=num_ctas, out_dtype=out_dtype,
                                 sink=None if sink is None else sink[:, None],
                                 gate=None if gate is None else gate[:, None],
                                 k_scale=k_scale, v_scale=v_scale,
                                 logit_scale=None if logit_scale is None
                                 else logit_scale[:, None])
        return o[:, 0]
    fn, args, out = _decode_call(q, rel, k_cache, v_cache, block_table, seq_lens, window,
                                 rel_extent, out, workspace, num_ctas)
    _check(fn(*args, _stream(q.device)), fn.__name__)
    return out


def _decode_call(q, rel, k_cache, v_cache, block_table, seq_lens, window, rel_extent, out,
                 workspace, num_ctas):
    """(C function, its arguments but the stream, out) of a plain decode."""
    dev = q.device
    B, Hq, dqk = q.shape
    _need(q, "q", torch.bfloat16, 3, dev)
    _need(rel, "rel", torch.float32, 3, dev)
    _need(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _need(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _need(block_table, "block_table", torch.int32, 2, dev)
    _need(seq_lens, "seq_lens", torch.int32, 1, dev)
    if tuple(rel.shape) != (B, Hq, rel_extent):
        raise ValueError("rel must be [B, Hq, rel_extent]")
    if seq_lens.shape[0] != B or block_table.shape[0] != B:
        raise ValueError("seq_lens / block_table batch mismatch")
    cache = cache_desc(k_cache, v_cache)
    dims = decode_dims(q, block_table, num_ctas)
    if out is None:
        out = torch.empty((B, Hq, v_cache.shape[3]), dtype=torch.bfloat16, device=dev)
    else:
        _need(out, "out", torch.bfloat16, 3, dev)
    if workspace is None:
        workspace = new_workspace(workspace_size(dims, cache), dev)
    return lib().relattn_decode, (
        q.data_ptr(), rel.data_ptr(), ctypes.byref(cache), block_table.data_ptr(),
        seq_lens.data_ptr(), int(window), int(rel_extent), ctypes.byref(dims),
        out.data_ptr(), workspace.data_ptr(), workspace.numel()), out


def relattn_decode_noalloc(q, rel, k_cache, v_cache, block_table, seq_lens, window: int,
                           rel_extent: int, out, num_ctas: int = 0):
    """Decode whose split state lives in the library's own device array.

    For callers that cannot allocate device memory: nothing is allocated here
    either, so ``out`` must be given.  Calls share that array; order them on
    one stream.
    """
    dev = q.device
    B, Hq, _ = q.shape
    _need(q, "q", torch.bfloat16, 3, dev)
    _need(rel, "rel", torch.float32, 3, dev)
    _need(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _need(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _need(block_table, "block_table", torch.int32, 2, dev)
    _need(seq_lens, "seq_lens", torch.int32, 1, dev)
    _need(out, "out", torch.bfloat16, 3, dev)
    cache = cache_desc(k_cache, v_cache)
    dims = decode_dims(q, block_table, num_ctas)
    _check(lib().relattn_decode_noalloc(
        q.data_ptr(), rel.data_ptr(), ctypes.byref(cache), block_table.data_ptr(),
        seq_lens.data_ptr(), int(window), int(rel_extent), ctypes.byref(dims),
        out.data_ptr(), _stream(dev)), "relattn_decode_noalloc")
    return out


def noalloc_status(device=None) -> int:
    """Status bits of the last relattn_decode_noalloc call on the device
    (synchronises the current stream)."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    st = (ctypes.c_uint32 * 1)()
    with torch.cuda.device(dev):
        _check(lib().relattn_decode_noalloc_status(ctypes.addressof(st), _stream(dev)),
               "relattn_decode_noalloc_status")
    return int(st[0])


def relattn_decode_multi(q, rel, k_cache, v_cache, block_table, seq_lens, window: int,
                         rel_extent: int, out=None, workspace=None, num_ctas: int = 0,
                         out_dtype=torch.bfloat16, sink=None, gate=None, k_scale=None,
                         v_scale=None, logit_scale=None):
    """Decode of k query tokens per sequence (speculative verification).

    q is [B, k, Hq, d_qk], rel [B, k, Hq, rel_extent], out [B, k, Hq, d_v];
    token i of sequence b sits at position seq_lens[b] - k + i.  rel may be
    float32 or bfloat16, out bfloat16 or float32, sink / gate optional
    float32 [B, k, Hq] logits and logit_scale an optional float32 [B, k]
    (``relattn_decode_ex``).
    """
    fn, args, out = _decode_multi_call(q, rel, k_cache, v_cache, block_table, seq_lens, window,
                                       rel_extent, out, workspace, num_ctas, out_dtype, sink,
                                       gate, k_scale, v_scale, logit_scale)
    _check(fn(*args, _stream(q.device)), fn.__name__)
    return out


def _decode_multi_call(q, rel, k_cache, v_cache, block_table, seq_lens, window, rel_extent,
                       out, workspace, num_ctas, out_dtype, sink, gate, k_scale, v_scale,
                       logit_scale):
    """(C function, its arguments but the stream, out) of a multi-token or
    typed decode."""
    dev = q.device
    _need(q, "q", torch.bfloat16, 4, dev)
    B, kq, Hq, _ = q.shape
    out_dtype = out.dtype if out is not None else out_dtype
    io = _options(rel, out_dtype, sink, gate, (B, kq, Hq), dev, k_cache, k_scale, v_scale,
                  logit_scale)
    _need(rel, "rel", rel.dtype, 4, dev)
    _need_cache(k_cache, v_cache, dev)
    _need(block_table, "block_table", torch.int32, 2, dev)
    _need(seq_lens, "seq_lens", torch.int32, 1, dev)
    if tuple(rel.shape) != (B, kq, Hq, rel_extent):
        raise ValueError("rel must be [B, k, Hq, rel_extent]")
    if seq_lens.shape[0] != B or block_table.shape[0] != B:
        raise ValueError("seq_lens / block_table batch mismatch")
    cache = cache_desc(k_cache, v_cache)
    dims = Dims(B, Hq, block_table.shape[1], 0, 0, num_ctas)
    if out is None:
        out = torch.empty((B, kq, Hq, v_cache.shape[3]), dtype=out_dtype, device=dev)
    else:
        _need(out, "out", out_dtype, 4, dev)
    if workspace is None:
        workspace = new_workspace(workspace_size(dims, cache), dev)
    if _plain(rel, out_dtype, sink, gate, k_cache, logit_scale):
        return lib().relattn_decode_multi, (
            q.data_ptr(), rel.data_ptr(), ctypes.byref(cache), block_table.data_ptr(),
            seq_lens.data_ptr(), int(kq), int(window), int(rel_extent), ctypes.byref(dims),
            out.data_ptr(), workspace.data_ptr(), workspace.numel()), out
    return lib().relattn_decode_ex, (
        q.data_ptr(), rel.data_ptr(), ctypes.byref(io), ctypes.byref(cache),
        block_table.data_ptr(), seq_lens.data_ptr(), int(kq), int(window),
        int(rel_extent), ctypes.byref(dims), out.data_ptr(), workspace.data_ptr(),
        workspace.numel()), out


def bind_decode(q, rel, k_cache, v_cache, block_table, seq_lens, window: int,
                rel_extent: int, out, workspace, num_ctas: int = 0, sink=None, gate=None,
                k_scale=None, v_scale=None, logit_scale=None):
    """Check and marshal one decode call for buffers that stay in place (a
    serving loop that refills q, rel, seq_lens and block_table between
    steps); returns run(), which enqueues that same C-ABI call on the
    device's current stream and raises on a non-zero return code.  q is
    [B, Hq, d_qk] (``relattn_decode``) or [B, k, Hq, d_qk]
    (``relattn_decode_multi``); every tensor must outlive run.
    """
    if q.dim() == 3 and _plain(rel, out.dtype, sink, gate, k_cache, logit_scale):
        fn, args, out = _decode_call(q, rel, k_cache, v_cache, block_table, seq_lens, window,
                                     rel_extent, out, workspace, num_ctas)
    else:
        if q.dim() == 3:
            q, rel, out = q[:, None], rel[:, None], out[:, None]
            sink = None if sink is None else sink[:, None]
            gate = None if gate is None else gate[:, None]
            logit_scale = None if logit_scale is None else logit_scale[:, None]
        fn, args, out = _decode_multi_call(q, rel, k_cache, v_cache, block_table, seq_lens,
                                           window, rel_extent, out, workspace, num_ctas,
                                           out.dtype, sink, gate, k_scale, v_scale,
                                           logit_scale)
    dev = q.device
    keep = (q, rel, k_cache, v_cache, block_table, seq_lens, out, workspace, sink, gate,
            logit_scale)

    def run():
        _check(fn(*args, _stream(dev)), fn.__name__)
        return keep

    return run


def prefill_dims(q, block_table, ctx_lens, max_q_len: int, num_ctas=0) -> Dims:
    return Dims(ctx_lens.shape[0], q.shape[1], block_table.shape[1], q.shape[0],
                int(max_q_len), num_ctas)


def relattn_cache_write(k, v, cu_seqlens, k_cache, v_cache, block_table, ctx_lens,
                        max_q_len: int, k_scale=None, v_scale=None, workspace=None):
    """Write new tokens' keys and values into the paged cache without
    attending (see ``relattn_cache_write`` in include/relattn.h): copied into a
    bf16 cache, or quantised into a head-major float8_e4m3fn cache with its
    k_scale / v_scale.  k is [T, Hkv, d_qk], v [T, Hkv, d_v], both bf16."""
    dev = k.device
    _need(k, "k", torch.bfloat16, 3, dev)
    _need(v, "v", torch.bfloat16, 3, dev)
    _need_cache(k_cache, v_cache, dev)
    _need(block_table, "block_table", torch.int32, 2, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1, dev)
    _need(ctx_lens, "ctx_lens", torch.int32, 1, dev)
    T, B = k.shape[0], ctx_lens.shape[0]
    if v.shape[0] != T:
        raise ValueError("k / v must have one row per new token")
    if cu_seqlens.shape[0] != B + 1 or block_table.shape[0] != B:
        raise ValueError("cu_seqlens / block_table batch mismatch")
    io = _options(torch.empty(0, dtype=torch.float32), torch.bfloat16, k_cache=k_cache,
                  k_scale=k_scale, v_scale=v_scale)
    cache = cache_desc(k_cache, v_cache)
    dims = Dims(B, k.shape[1], block_table.shape[1], T, int(max_q_len), 0)
    if workspace is None:
        workspace = new_workspace(256, dev)
    _check(lib().relattn_cache_write(
        k.data_ptr(), v.data_ptr(), ctypes.byref(io), cu_seqlens.data_ptr(), ctypes.byref(cache),
        block_table.data_ptr(), ctx_lens.data_ptr(), ctypes.byref(dims), workspace.data_ptr(),
        workspace.numel(), _stream(dev)), "relattn_cache_write")
    return workspace


def relattn_prefill(q, k, v, rel, cu_seqlens, k_cache, v_cache, block_table, ctx_lens,
                    window: int, rel_extent: int, max_q_len: int, out=None,
                    workspace=None, out_dtype=torch.bfloat16, sink=None, gate=None,
                    logit_scale=None, k_scale=None, v_scale=None, num_ctas: int = 0):
    """Chunked prefill with a cached prefix; writes k, v into the cache.

    rel may be float32 or bfloat16, out bfloat16 or float32 (``out``'s own
    dtype when it is given), sink / gate optional float32 [T, Hq] logits,
    logit_scale an optional float32 [T] of log-position factors; a
    float8_e4m3fn cache (head-major) takes its k_scale and v_scale.  Anything
    but fp32 rel, bf16 out, a bf16 cache and none of the optional inputs goes
    through ``relattn_prefill_ex``.
    """
    dev = q.device
    T, Hq, dqk = q.shape
    out_dtype = out.dtype if out is not None else out_dtype
    io = _options(rel, out_dtype, sink, gate, (T, Hq), dev, k_cache, k_scale, v_scale,
                  logit_scale)
    _need(q, "q", torch.bfloat16, 3, dev)
    _need(k, "k", torch.bfloat16, 3, dev)
    _need(v, "v", torch.bfloat16, 3, dev)
    _need(rel, "rel", rel.dtype, 3, dev)
    _need_cache(k_cache, v_cache, dev)
    _need(block_table, "block_table", torch.int32, 2, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1, dev)
    _need(ctx_lens, "ctx_lens", torch.int32, 1, dev)
    if tuple(rel.shape) != (T, Hq, rel_extent):
        raise ValueError("rel must be [T, Hq, rel_extent]")
    if k.shape[0] != T or v.shape[0] != T:
        raise ValueError("k / v must have one row per new token")
    B = ctx_lens.shape[0]
    if cu_seqlens.shape[0] != B + 1 or block_table.shape[0] != B:
        raise ValueError("cu_seqlens / block_table batch mismatch")
    cache = cache_desc(k_cache, v_cache)
    dims = prefill_dims(q, block_table, ctx_lens, max_q_len, num_ctas)
    if out is None:
        out = torch.empty((T, Hq, v_cache.shape[3]), dtype=out_dtype, device=dev)
    else:
        _need(out, "out", out_dtype, 3, dev)
    if workspace is None:
        workspace = new_workspace(workspace_size(dims, cache), dev)
    if _plain(rel, out_dtype, sink, gate, k_cache, logit_scale):
        _check(lib().relattn_prefill(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), rel.data_ptr(), cu_seqlens.data_ptr(),
            ctypes.byref(cache), block_table.data_ptr(), ctx_lens.data_ptr(), int(window),
            int(rel_extent), ctypes.byref(dims), out.data_ptr(), workspace.data_ptr(),
            workspace.numel(), _stream(dev)), "relattn_prefill")
    else:
        _check(lib().relattn_prefill_ex(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), rel.data_ptr(), ctypes.byref(io),
            cu_seqlens.data_ptr(), ctypes.byref(cache), block_table.data_ptr(),
            ctx_lens.data_ptr(), int(window), int(rel_extent), ctypes.byref(dims),
            out.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream(dev)),
            "relattn_prefill_ex")
    return out


def debug_walk_decode(block_table, seq_lens, window: int, k_cache, v_cache, num_q_heads: int,
                      num_ctas: int = 0, max_records: int = 1 << 20):
    """Replay of the decode kernel's block walk: int32 [n, 6] records."""
    dev = block_table.device
    cache = cache_desc(k_cache, v_cache)
    dims = Dims(block_table.shape[0], num_q_heads, block_table.shape[1], 0, 0, num_ctas)
    ws = new_workspace(workspace_size(dims, cache), dev)
    rec = torch.zeros((max_records, 6), dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(lib().relattn_debug_walk_decode(
        block_table.data_ptr(), seq_lens.data_ptr(), int(window), ctypes.byref(cache),
        ctypes.byref(dims), rec.data_ptr(), max_records, cnt.data_ptr(), ws.data_ptr(),
        ws.numel(), _stream(dev)), "relattn_debug_walk_decode")
    n = int(cnt.item())
    if n > max_records:
        raise RuntimeError("walk produced more records than the buffer holds")
    return rec[:n].cpu(), read_status(ws)


def debug_walk_decode_ex(block_table, seq_lens, num_query_tokens: int, window: int, k_cache,
                         v_cache, num_q_heads: int, num_ctas: int = 0,
                         max_records: int = 1 << 20):
    """Replay of the decode kernel's walk for k query tokens per sequence over
    the cache's type: int32 [n, 8] records (cta, sequence, first token of the
    chunk, KV head, key tile, physical block, first key brought, keys)."""
    dev = block_table.device
    cache = cache_desc(k_cache, v_cache)
    dims = Dims(block_table.shape[0], num_q_heads, block_table.shape[1], 0, 0, num_ctas)
    ws = new_workspace(workspace_size(dims, cache), dev)
    opts = Options(DTYPE_F32, DTYPE_BF16, None, None,
                   DTYPE_E4M3 if k_cache.dtype == torch.float8_e4m3fn else DTYPE_BF16,
                   1.0, 1.0, None)
    rec = torch.zeros((max_records, 8), dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(lib().relattn_debug_walk_decode_ex(
        block_table.data_ptr(), seq_lens.data_ptr(), int(num_query_tokens), int(window),
        ctypes.byref(opts), ctypes.byref(cache), ctypes.byref(dims), rec.data_ptr(),
        max_records, cnt.data_ptr(), ws.data_ptr(), ws.numel(), _stream(dev)),
        "relattn_debug_walk_decode_ex")
    n = int(cnt.item())
    if n > max_records:
        raise RuntimeError("walk produced more records than the buffer holds")
    return rec[:n].cpu(), read_status(ws)


def debug_walk_prefill(cu_seqlens, ctx_lens, block_table, window: int, k_cache, v_cache,
                       num_q_heads: int, max_q_len: int, max_records: int = 1 << 20,
                       rel_dtype=None):
    """Replay of the prefill kernel's block walk: int32 [n, 6] records.

    rel_dtype None: the two-heads kernel (relattn_debug_walk_prefill); else
    the kernel relattn_prefill runs for a rel of that dtype
    (relattn_debug_walk_prefill_ex)."""
    dev = block_table.device
    cache = cache_desc(k_cache, v_cache)
    num_tokens = int(cu_seqlens[-1].item())  # test hook: a host read is fine here
    dims = Dims(ctx_lens.shape[0], num_q_heads, block_table.shape[1], num_tokens,
                int(max_q_len), 0)
    ws = new_workspace(workspace_size(dims, cache), dev)
    rec = torch.zeros((max_records, 6), dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    if rel_dtype is None:
        _check(lib().relattn_debug_walk_prefill(
            cu_seqlens.data_ptr(), ctx_lens.data_ptr(), block_table.data_ptr(), int(window),
            ctypes.byref(cache), ctypes.byref(dims), rec.data_ptr(), max_records,
            cnt.data_ptr(), ws.data_ptr(), ws.numel(), _stream(dev)),
            "relattn_debug_walk_prefill")
    else:
        opts = Options(_DTYPE_CODE[rel_dtype], DTYPE_BF16, None, None, DTYPE_BF16, 1.0, 1.0, None)
        _check(lib().relattn_debug_walk_prefill_ex(
            cu_seqlens.data_ptr(), ctx_lens.data_ptr(), block_table.data_ptr(), int(window),
            ctypes.byref(opts), ctypes.byref(cache), ctypes.byref(dims), rec.data_ptr(),
            max_records, cnt.data_ptr(), ws.data_ptr(), ws.numel(), _stream(dev)),
            "relattn_debug_walk_prefill_ex")
    n = int(cnt.item())
    if n > max_records:
        raise RuntimeError("walk produced more records than the buffer holds")
    return rec[:n].cpu(), read_status(ws)
