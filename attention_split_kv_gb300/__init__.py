"""Python binding of libattn (C ABI in include/attn.h).

Argument marshalling only: every step of the attention path runs in the CUDA
kernels of ``libattn.so``.  There is no fallback: importing works without the
library (so sizes can be planned on a machine without a GPU), but every call
that needs it raises ``AttnLibraryMissing`` if ``libattn.so`` was not built.

Functions keep the C names; pointer arguments accept torch tensors (their
``data_ptr()``), plain integers (device addresses) or None (NULL).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = [
    "ATTN_OK", "ATTN_EINVAL", "ATTN_EUNSUPPORTED", "ATTN_ECUDA", "ATTN_EBOUNDS", "ATTN_ETIMEOUT",
    "ATTN_KV_F16", "ATTN_KV_INT8", "ATTN_F16", "ATTN_F32", "AttnError", "AttnLibraryMissing",
    "lib_path", "load", "build", "exported_symbols",
    "attn_version", "attn_last_error", "attn_decode_workspace_size", "attn_decode",
    "attn_decode_ring", "attn_decode_ex", "attn_decode_tiered", "attn_decode_tiered_workspace_size",
    "attn_decode_noalloc", "attn_prefill", "attn_prefill_paged", "attn_decode_validate", "attn_device_status",
    "attn_testing_set_waits", "decode", "decode_tiered", "prefill", "prefill_paged",
]

ATTN_OK, ATTN_EINVAL, ATTN_EUNSUPPORTED, ATTN_ECUDA, ATTN_EBOUNDS, ATTN_ETIMEOUT = range(6)
ATTN_KV_F16, ATTN_KV_INT8 = 0, 1
ATTN_F16, ATTN_F32 = 0, 1
_STATUS = {0: "ATTN_OK", 1: "ATTN_EINVAL", 2: "ATTN_EUNSUPPORTED", 3: "ATTN_ECUDA", 4: "ATTN_EBOUNDS",
           5: "ATTN_ETIMEOUT"}

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libattn.so")
_lib = None

# every entry point include/attn.h declares
exported_symbols = ("attn_version", "attn_last_error", "attn_decode_workspace_size", "attn_decode",
                    "attn_decode_ring", "attn_decode_ex", "attn_decode_tiered", "attn_decode_tiered_workspace_size",
                    "attn_decode_noalloc", "attn_prefill", "attn_prefill_paged", "attn_decode_validate",
                    "attn_device_status", "attn_testing_set_waits")


class AttnLibraryMissing(RuntimeError):
    pass


class AttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (_STATUS.get(status, str(status)), message))
        self.status = status


def lib_path() -> str:
    return _LIB_PATH


def build(force: bool = False, verbose: bool = False) -> str:
    from . import _build
    return _build.build(force=force, verbose=verbose)


def load():
    """Load libattn.so (raises AttnLibraryMissing if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise AttnLibraryMissing("libattn.so is not built (run attention_split_kv_gb300.build())")
    lib = ctypes.CDLL(_LIB_PATH)
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.attn_version.restype = ctypes.c_char_p
    lib.attn_last_error.restype = ctypes.c_char_p
    lib.attn_decode_workspace_size.argtypes = [I, I, I, I, I, I]
    lib.attn_decode_workspace_size.restype = SZ
    lib.attn_decode.argtypes = [P, P, P, P, P, I, I, I, I, P, P, I, I, I, I, I, I, F, F, I, P, P, P, SZ, P]
    lib.attn_decode.restype = I
    lib.attn_decode_ring.argtypes = [P, P, P, P, I, P, P, I, I, I, I, I, I, F, F, I, P, P, P, SZ, P]
    lib.attn_decode_ring.restype = I
    lib.attn_decode_tiered_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.attn_decode_tiered_workspace_size.restype = SZ
    lib.attn_decode_tiered.argtypes = [P, I, P, P, P, P, I, P, P, I, I, I, I, P, P, P, P, I, I, I, I, I, I, F, F,
                                       I, P, I, P, P, SZ, P]
    lib.attn_decode_ex.argtypes = [P, I, P, P, P, P, I, I, I, I, I, P, P, I, I, I, I, I, I, F, F, I, P, I, P, P, SZ,
                                   P]
    lib.attn_decode_ex.restype = I
    lib.attn_decode_tiered.restype = I
    lib.attn_decode_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, P, P, I, I, I, I, I, I, F, F, I, P, P, P]
    lib.attn_decode_noalloc.restype = I
    lib.attn_prefill.argtypes = [P, P, P, I, I, I, I, I, I, F, F, P, P, P]
    lib.attn_prefill.restype = I
    lib.attn_prefill_paged.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, F, F, P, P, P]
    lib.attn_prefill_paged.restype = I
    lib.attn_decode_validate.argtypes = [P, P, I, I, I, I, I, ctypes.POINTER(ctypes.c_int), P]
    lib.attn_decode_validate.restype = I
    lib.attn_device_status.argtypes = [P]
    lib.attn_device_status.restype = I
    lib.attn_testing_set_waits.argtypes = [ctypes.c_ulonglong, I]
    lib.attn_testing_set_waits.restype = I
    _lib = lib
    return lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int):
    if status != ATTN_OK:
        raise AttnError(status, load().attn_last_error().decode())


def attn_version() -> str:
    return load().attn_version().decode()


def attn_last_error() -> str:
    return load().attn_last_error().decode()


def attn_decode_workspace_size(batch, n_heads, n_kv_heads, head_dim, max_kv, split_keys=0) -> int:
    return int(load().attn_decode_workspace_size(batch, n_heads, n_kv_heads, head_dim, max_kv, split_keys))


def attn_decode(q, k_cache, v_cache, kv_len, page_table, page_size, max_pages_per_seq, n_pages, max_kv,
                k_scales, v_scales, kv_dtype, batch, n_heads, n_kv_heads, head_dim, window, softcap, scale,
                split_keys, out, lse_out, workspace, workspace_bytes, stream=None) -> None:
    _check(load().attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), _ptr(page_table),
                              int(page_size), int(max_pages_per_seq), int(n_pages), int(max_kv),
                              _ptr(k_scales), _ptr(v_scales), int(kv_dtype), int(batch), int(n_heads),
                              int(n_kv_heads), int(head_dim), int(window), float(softcap), float(scale),
                              int(split_keys), _ptr(out), _ptr(lse_out), _ptr(workspace),
                              int(workspace_bytes), _stream(stream)))


def attn_decode_ring(q, k_ring, v_ring, seq_len, ring_size, k_scales, v_scales, kv_dtype, batch, n_heads,
                     n_kv_heads, head_dim, window, softcap, scale, split_keys, out, lse_out, workspace,
                     workspace_bytes, stream=None) -> None:
    _check(load().attn_decode_ring(_ptr(q), _ptr(k_ring), _ptr(v_ring), _ptr(seq_len), int(ring_size),
                                   _ptr(k_scales), _ptr(v_scales), int(kv_dtype), int(batch), int(n_heads),
                                   int(n_kv_heads), int(head_dim), int(window), float(softcap), float(scale),
                                   int(split_keys), _ptr(out), _ptr(lse_out), _ptr(workspace),
                                   int(workspace_bytes), _stream(stream)))


def attn_decode_tiered_workspace_size(batch, n_heads, n_kv_heads, head_dim, cold_max_kv, hot_ring,
                                      split_keys=0) -> int:
    return int(load().attn_decode_tiered_workspace_size(batch, n_heads, n_kv_heads, head_dim, cold_max_kv,
                                                        hot_ring, split_keys))


def attn_decode_ex(q, q_dtype, k_cache, v_cache, kv_len, page_table, page_size, max_pages_per_seq, n_pages, max_kv,
                   ring_size, k_scales, v_scales, kv_dtype, batch, n_heads, n_kv_heads, head_dim, window, softcap,
                   scale, split_keys, out, out_dtype, lse_out, workspace, workspace_bytes, stream=None) -> None:
    _check(load().attn_decode_ex(_ptr(q), int(q_dtype), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), _ptr(page_table),
                                 int(page_size), int(max_pages_per_seq), int(n_pages), int(max_kv), int(ring_size),
                                 _ptr(k_scales), _ptr(v_scales), int(kv_dtype), int(batch), int(n_heads),
                                 int(n_kv_heads), int(head_dim), int(window), float(softcap), float(scale),
                                 int(split_keys), _ptr(out), int(out_dtype), _ptr(lse_out), _ptr(workspace),
                                 int(workspace_bytes), _stream(stream)))


def _dtype_of(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return ATTN_F32
    if t.dtype == torch.float16:
        return ATTN_F16
    raise AttnError(ATTN_EINVAL, "q and out must be float16 or float32, not %s" % t.dtype)


def attn_decode_tiered(q, q_dtype, cold_k, cold_v, cold_k_scales, cold_v_scales, cold_dtype, cold_len,
                       cold_page_table, cold_page_size, cold_max_pages_per_seq, cold_n_pages, cold_max_kv, hot_k,
                       hot_v, hot_len, hot_start, hot_ring, batch, n_heads, n_kv_heads, head_dim, window, softcap,
                       scale, split_keys, out, out_dtype, lse_out, workspace, workspace_bytes, stream=None) -> None:
    _check(load().attn_decode_tiered(_ptr(q), int(q_dtype), _ptr(cold_k), _ptr(cold_v), _ptr(cold_k_scales),
                                     _ptr(cold_v_scales),
                                     int(cold_dtype), _ptr(cold_len), _ptr(cold_page_table), int(cold_page_size),
                                     int(cold_max_pages_per_seq), int(cold_n_pages), int(cold_max_kv), _ptr(hot_k),
                                     _ptr(hot_v), _ptr(hot_len), _ptr(hot_start), int(hot_ring), int(batch),
                                     int(n_heads), int(n_kv_heads), int(head_dim), int(window), float(softcap),
                                     float(scale), int(split_keys), _ptr(out), int(out_dtype), _ptr(lse_out),
                                     _ptr(workspace), int(workspace_bytes), _stream(stream)))


def decode_tiered(case, out=None, lse_out=None, workspace=None, split_keys: int = 0, stream=None, out_f32=False):
    """attn_decode_tiered on a TieredCase-like object (tensors already on the GPU);
    q f16 or f32 as the case holds it, out f16 (or f32 with ``out_f32``)."""
    import torch
    dev = case.q.device
    B, Hq, Hkv, D = case.batch, case.n_heads, case.n_kv_heads, case.head_dim
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32 if out_f32 else torch.float16, device=dev)
    ws_bytes = attn_decode_tiered_workspace_size(B, Hq, Hkv, D, case.cap, case.hot_ring, split_keys)
    if ws_bytes == 0:
        raise AttnError(ATTN_EINVAL, "invalid sizes for the tiered decode workspace")
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    attn_decode_tiered(case.q, _dtype_of(case.q), case.k, case.v, case.k_scales, case.v_scales,
                       ATTN_KV_INT8 if case.int8 else ATTN_KV_F16, case.kv_len, case.page_table, case.page_size,
                       case.max_pages, case.n_pages, case.cap, case.hot_k, case.hot_v, case.hot_len,
                       case.hot_start, case.hot_ring, B, Hq, Hkv, D, case.window, case.softcap, case.scale,
                       split_keys, out, _dtype_of(out), lse_out, workspace, workspace.numel(), stream)
    return out


def attn_decode_noalloc(q, k_cache, v_cache, kv_len, page_table, page_size, max_pages_per_seq, n_pages,
                        max_kv, k_scales, v_scales, kv_dtype, batch, n_heads, n_kv_heads, head_dim, window,
                        softcap, scale, split_keys, out, lse_out, stream=None) -> None:
    """attn_decode without a caller workspace: the library's fixed 16 MiB
    device scratch array is used instead (for callers that cannot allocate)."""
    _check(load().attn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), _ptr(page_table),
                                      int(page_size), int(max_pages_per_seq), int(n_pages), int(max_kv),
                                      _ptr(k_scales), _ptr(v_scales), int(kv_dtype), int(batch), int(n_heads),
                                      int(n_kv_heads), int(head_dim), int(window), float(softcap), float(scale),
                                      int(split_keys), _ptr(out), _ptr(lse_out), _stream(stream)))


def attn_prefill(q, k, v, seq_len, n_heads, n_kv_heads, head_dim, causal, window, softcap, scale,
                 out, lse_out=None, stream=None) -> None:
    _check(load().attn_prefill(_ptr(q), _ptr(k), _ptr(v), int(seq_len), int(n_heads), int(n_kv_heads),
                               int(head_dim), int(bool(causal)), int(window), float(softcap), float(scale),
                               _ptr(out), _ptr(lse_out), _stream(stream)))


def attn_decode_validate(kv_len, page_table, batch, page_size, max_pages_per_seq, n_pages, max_kv,
                         stream=None):
    """Returns (status, first bad sequence or -1); never raises on EBOUNDS/EINVAL."""
    bad = ctypes.c_int(-1)
    st = load().attn_decode_validate(_ptr(kv_len), _ptr(page_table), int(batch), int(page_size),
                                     int(max_pages_per_seq), int(n_pages), int(max_kv), ctypes.byref(bad),
                                     _stream(stream))
    if st == ATTN_ECUDA:
        _check(st)
    return st, bad.value


def attn_device_status(stream=None) -> int:
    return int(load().attn_device_status(_stream(stream)))


# ---------------------------------------------------------------- conveniences
def attn_testing_set_waits(wait_limit_ns: int, stall_first_tile: int) -> int:
    """Testing hook: pipeline-wait time limit (0 = the default) and the first-tile stall."""
    return load().attn_testing_set_waits(int(wait_limit_ns), int(stall_first_tile))


def decode(case, out=None, lse_out=None, workspace=None, split_keys: int = 0, max_kv: Optional[int] = None,
           stream=None, out_f32=False):
    """attn_decode on a DecodeCase-like object (tensors already on the GPU);
    attn_decode_ring when the case holds a ring cache (``case.ring > 0``).

    Allocates ``out`` (and the workspace) with torch when not given.
    """
    import torch
    dev = case.q.device
    B, Hq, Hkv, D = case.batch, case.n_heads, case.n_kv_heads, case.head_dim
    ring = int(getattr(case, "ring", 0) or 0)
    if max_kv is None:
        max_kv = ring if ring else case.cap
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32 if out_f32 else torch.float16, device=dev)
    ws_bytes = attn_decode_workspace_size(B, Hq, Hkv, D, max_kv, split_keys)
    if ws_bytes == 0:
        raise AttnError(ATTN_EINVAL, "invalid sizes for the decode workspace")
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    qt, ot = _dtype_of(case.q), _dtype_of(out)
    if qt != ATTN_F16 or ot != ATTN_F16:
        attn_decode_ex(case.q, qt, case.k, case.v, case.kv_len, case.page_table, case.page_size, case.max_pages,
                       case.n_pages, max_kv, ring, case.k_scales, case.v_scales,
                       ATTN_KV_INT8 if case.int8 else ATTN_KV_F16, B, Hq, Hkv, D, case.window, case.softcap,
                       case.scale, split_keys, out, ot, lse_out, workspace, workspace.numel(), stream)
        return out
    if ring:
        attn_decode_ring(case.q, case.k, case.v, case.kv_len, ring, case.k_scales, case.v_scales,
                         ATTN_KV_INT8 if case.int8 else ATTN_KV_F16, B, Hq, Hkv, D, case.window, case.softcap,
                         case.scale, split_keys, out, lse_out, workspace, workspace.numel(), stream)
        return out
    attn_decode(case.q, case.k, case.v, case.kv_len, case.page_table, case.page_size, case.max_pages,
                case.n_pages, max_kv, case.k_scales, case.v_scales,
                ATTN_KV_INT8 if case.int8 else ATTN_KV_F16, B, Hq, Hkv, D, case.window, case.softcap,
                case.scale, split_keys, out, lse_out, workspace, workspace.numel(), stream)
    return out


def prefill(case, out=None, lse_out=None, stream=None):
    """attn_prefill on a PrefillCase-like object (tensors already on the GPU)."""
    import torch
    if out is None:
        out = torch.empty_like(case.q)
    attn_prefill(case.q, case.k, case.v, case.seq_len, case.n_heads, case.n_kv_heads, case.head_dim,
                 case.causal, case.window, case.softcap, case.scale, out, lse_out, stream)
    return out


def attn_prefill_paged(q, k_cache, v_cache, q_start, kv_len, page_table, page_size, max_pages, n_pages, batch,
                       total_q, max_q, n_heads, n_kv_heads, head_dim, window, softcap, scale, out, lse_out,
                       stream=None) -> None:
    _check(load().attn_prefill_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(q_start), _ptr(kv_len),
                                     _ptr(page_table), int(page_size), int(max_pages), int(n_pages), int(batch),
                                     int(total_q), int(max_q), int(n_heads), int(n_kv_heads), int(head_dim),
                                     int(window), float(softcap), float(scale), _ptr(out), _ptr(lse_out),
                                     _stream(stream)))


def prefill_paged(case, out=None, lse_out=None, stream=None):
    """attn_prefill_paged on a ChunkCase-like object (tensors already on the GPU)."""
    import torch
    if out is None:
        out = torch.empty_like(case.q)
    attn_prefill_paged(case.q, case.k, case.v, case.q_start, case.kv_len, case.page_table, case.page_size,
                       case.max_pages, int(case.k.shape[0]), case.batch, case.total_q, case.max_q, case.n_heads,
                       case.n_kv_heads, case.head_dim, case.window, case.softcap, case.scale, out, lse_out, stream)
    return out
