"""Single-token decode attention over a KV cache on GB300 (sm_103a).

Thin ctypes binding over ``libkvdecode.so`` (C ABI declared in
``include/kvdecode.h``). Every step of the path runs in the library's CUDA
kernels; this module only checks tensor metadata and marshals pointers and
sizes. PyTorch supplies device memory and streams. There is no CPU fallback:
if the library is missing or stale, loading fails with an error.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import numpy as np

from . import roofline  # noqa: F401  (host-side byte model)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvdecode.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE_TOO_SMALL, ERR_CUDA = range(5)
OUT_BF16, OUT_F32 = 0, 1
STATUS_SEQ_LEN_CLAMPED = 0x1
STATUS_POS_OUT_OF_RANGE = 0x2
STATUS_UMAX_FALLBACK = 0x10

# Every symbol include/kvdecode.h declares.
EXPORTED = (
    "kvd_decode_plan", "kvd_kv_append", "kvd_decode_attention", "kvd_split_kv_chunk",
    "kvd_split_kv_merge", "kvd_schedule_describe", "kvd_kernel_info", "kvd_status_string",
    "kvd_version", "kvd_decode_attention_static", "kvd_decode_step", "kvd_kv_append_paged",
    "kvd_decode_attention_paged", "kvd_decode_step_paged", "kvd_kv_quantize_q8", "kvd_kv_append_q8",
    "kvd_decode_attention_q8", "kvd_decode_step_q8", "kvd_decode_plan_multi", "kvd_kv_append_multi",
    "kvd_decode_attention_multi", "kvd_decode_step_multi", "kvd_decode_ex", "kvd_kv_append_q8_paged",
    "kvd_decode_attention_umax", "kvd_decode_step_umax", "kvd_step_staging_bytes", "kvd_decode_step_host",
    "kvd_kv_quantize_fp8", "kvd_kv_append_fp8", "kvd_kv_append_fp8_paged", "kvd_merge_attention",
    "kvd_probe_read",
)
STATIC_WORKSPACE_BYTES = 16 << 20  # KVD_STATIC_WORKSPACE_BYTES

_lock = threading.Lock()
_lib = None


class KvdError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def load(path: str = LIB_PATH):
    """Load libkvdecode.so. Raises if it has not been built (no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m kv_cache_decode_gb300._build` "
                "(or __graft_entry__.build()); there is no CPU fallback")
        from . import _build
        if path == LIB_PATH and not _build.up_to_date():
            raise RuntimeError(f"{path} is older than its sources: rebuild it")
        _lib = _declare(ctypes.CDLL(path))
        return _lib


class _CCache(ctypes.Structure):
    """struct kvd_cache of kvdecode.h."""
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("k_scales", ctypes.c_void_p),
                ("v_scales", ctypes.c_void_p), ("block_table", ctypes.c_void_p), ("s_max", ctypes.c_int),
                ("max_blocks", ctypes.c_int), ("page_size", ctypes.c_int), ("num_pages", ctypes.c_int),
                ("fp8", ctypes.c_int)]


def _declare(lib):
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    PI, PSZ = ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_size_t)
    lib.kvd_decode_plan.argtypes = [I, I, I, I, I, I, I, I, PI, PSZ]
    lib.kvd_kv_append.argtypes = [P, P, P, P, P, I, I, I, I, P, P]
    dec = [P, P, P, P, I, I, I, I, I, I, F, I, P, SZ, P, I, P, P, P]
    for name in ("kvd_decode_attention", "kvd_split_kv_chunk", "kvd_split_kv_merge"):
        getattr(lib, name).argtypes = dec
    lib.kvd_decode_attention_static.argtypes = [P, P, P, P, I, I, I, I, I, I, F, I, P, I, P, P, P]
    lib.kvd_decode_attention_static.restype = I
    # append arguments (k_cache, v_cache, k_new, v_new, pos), then q, seq_lens and the rest
    lib.kvd_decode_step.argtypes = [P, P, P, P, P, P, P] + dec[4:]
    lib.kvd_decode_step.restype = I
    # paged: the cache becomes (pool, block_table) and s_max becomes (max_blocks, page_size, num_pages)
    lib.kvd_kv_append_paged.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P]
    lib.kvd_kv_append_paged.restype = I
    dec_paged = [P, P, P, P, P, I, I, I, I] + dec[6:]
    lib.kvd_decode_attention_paged.argtypes = dec_paged
    lib.kvd_decode_attention_paged.restype = I
    lib.kvd_decode_step_paged.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I] + dec[6:]
    lib.kvd_decode_step_paged.restype = I
    # int8: codes in place of the cache, plus the two scale arrays
    lib.kvd_kv_quantize_q8.argtypes = [P, P, P, P, I, I, I, I, I, P]
    lib.kvd_kv_quantize_q8.restype = I
    lib.kvd_kv_append_q8.argtypes = [P, P, P, P, P, P, P, I, I, I, I, P, P]
    lib.kvd_kv_append_q8.restype = I
    lib.kvd_kv_append_q8_paged.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, P, P]
    lib.kvd_kv_quantize_fp8.argtypes = lib.kvd_kv_quantize_q8.argtypes
    lib.kvd_kv_quantize_fp8.restype = I
    lib.kvd_kv_append_fp8.argtypes = lib.kvd_kv_append_q8.argtypes
    lib.kvd_kv_append_fp8.restype = I
    lib.kvd_kv_append_fp8_paged.argtypes = lib.kvd_kv_append_q8_paged.argtypes
    lib.kvd_kv_append_fp8_paged.restype = I
    lib.kvd_kv_append_q8_paged.restype = I
    # unified maximum: decode_attention / decode_step with phi after scale
    lib.kvd_decode_attention_umax.argtypes = dec[:11] + [F] + dec[11:]
    lib.kvd_decode_attention_umax.restype = I
    lib.kvd_decode_step_umax.argtypes = [P, P, P, P, P, P, P] + dec[4:11] + [F] + dec[11:]
    lib.kvd_decode_step_umax.restype = I
    lib.kvd_merge_attention.argtypes = [P, P, I, ctypes.c_longlong, I, I, P, I, P, P]
    lib.kvd_merge_attention.restype = I
    lib.kvd_probe_read.argtypes = [P, SZ, I, P, P, P]
    lib.kvd_probe_read.restype = I
    lib.kvd_step_staging_bytes.argtypes = [I, I, I, I, I]
    lib.kvd_step_staging_bytes.restype = SZ
    lib.kvd_decode_step_host.argtypes = [P, P, P, P, P, P, P, P, SZ, I, I, I, I, I, I, I, F, I, P, SZ, P, P, I, P,
                                         P, P]
    lib.kvd_decode_step_host.restype = I
    lib.kvd_decode_attention_q8.argtypes = [P, P, P, P, P] + dec[3:]
    lib.kvd_decode_attention_q8.restype = I
    lib.kvd_decode_step_q8.argtypes = [P, P, P, P, P, P, P, P, P] + dec[4:]
    lib.kvd_decode_step_q8.restype = I
    # multi-token: n_tokens after batch
    lib.kvd_decode_plan_multi.argtypes = [I, I, I, I, I, I, I, I, I, PI, PSZ]
    lib.kvd_decode_plan_multi.restype = I
    lib.kvd_kv_append_multi.argtypes = [P, P, P, P, P, I, I, I, I, I, P, P]
    lib.kvd_kv_append_multi.restype = I
    lib.kvd_decode_attention_multi.argtypes = dec[:5] + [I] + dec[5:]
    lib.kvd_decode_attention_multi.restype = I
    lib.kvd_decode_step_multi.argtypes = [P, P, P, P, P, P, P, I, I] + dec[5:]
    lib.kvd_decode_step_multi.restype = I
    lib.kvd_decode_ex.argtypes = [ctypes.POINTER(_CCache), P, P, I, I, I, I, I, I, F, I, P, SZ, P, I, P, P, P, P,
                                  P, P]
    lib.kvd_decode_ex.restype = I
    lib.kvd_schedule_describe.argtypes = [P, I, I, I, I, I, I, I, I, P, I, PI, PI]
    lib.kvd_kernel_info.argtypes = [I, I, I, I, PI, PI, PI, PI, PI, PI]
    lib.kvd_status_string.argtypes = [I]
    lib.kvd_status_string.restype = ctypes.c_char_p
    lib.kvd_version.argtypes = []
    lib.kvd_version.restype = ctypes.c_char_p
    for name in EXPORTED[:7]:
        getattr(lib, name).restype = I
    return lib


def status_string(status: int) -> str:
    try:
        return load().kvd_status_string(int(status)).decode()
    except Exception:  # pragma: no cover - library missing
        return "status"


def version() -> str:
    return load().kvd_version().decode()


def _out_code(out_dtype) -> int:
    if out_dtype in (OUT_BF16, "bf16", "bfloat16"):
        return OUT_BF16
    if out_dtype in (OUT_F32, "f32", "float32", "fp32"):
        return OUT_F32
    import torch
    if out_dtype is torch.bfloat16:
        return OUT_BF16
    if out_dtype is torch.float32:
        return OUT_F32
    raise ValueError(f"unknown out_dtype {out_dtype!r}")


def _check(rc: int, what: str):
    if rc != OK:
        raise KvdError(rc, what)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    h = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return h or None


# ---------------------------------------------------------------------------
# Host-only queries
# ---------------------------------------------------------------------------

def decode_plan(batch: int, n_heads_q: int, n_heads_kv: int, head_dim: int, max_seq_len: int,
                num_sms: int = 0, n_split: int = 0, out_dtype="bf16") -> Tuple[int, int]:
    """(n_split, workspace_bytes) for a decode_attention call of this shape."""
    lib = load()
    n = ctypes.c_int(0)
    ws = ctypes.c_size_t(0)
    _check(lib.kvd_decode_plan(batch, n_heads_q, n_heads_kv, head_dim, max_seq_len, num_sms,
                               n_split, _out_code(out_dtype), ctypes.byref(n), ctypes.byref(ws)),
           "kvd_decode_plan")
    return n.value, ws.value


def kernel_info(n_heads_q: int, n_heads_kv: int, head_dim: int, out_dtype="bf16") -> dict:
    lib = load()
    th, sm, tt, cps, su, sc = (ctypes.c_int(0) for _ in range(6))
    _check(lib.kvd_kernel_info(n_heads_q, n_heads_kv, head_dim, _out_code(out_dtype),
                               ctypes.byref(th), ctypes.byref(sm), ctypes.byref(tt),
                               ctypes.byref(cps), ctypes.byref(su), ctypes.byref(sc)),
           "kvd_kernel_info")
    return {"threads": th.value, "smem_bytes": sm.value, "tile_tokens": tt.value,
            "ctas_per_sm": cps.value, "seg_unit": su.value, "seg_cost": sc.value}


def schedule_describe(seq_lens, s_max: int, max_seq_len: int, n_heads_q: int, n_heads_kv: int,
                      head_dim: int, n_split: int, out_dtype="bf16"):
    """Host replica of the device schedule: (rows [n, 8] int32, n_split_eff).

    Row = (cta, b, h, tok_lo, tok_hi, kind, slot, c_last); kind 0 final,
    1 partial by owner, 2 partial by another CTA, 3 empty pair.
    """
    lib = load()
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    n_rows = ctypes.c_int(0)
    eff = ctypes.c_int(0)
    args = [lens.ctypes.data_as(ctypes.c_void_p), int(lens.size), s_max, max_seq_len, n_heads_q,
            n_heads_kv, head_dim, n_split, _out_code(out_dtype)]
    _check(lib.kvd_schedule_describe(*args, None, 0, ctypes.byref(n_rows), ctypes.byref(eff)),
           "kvd_schedule_describe")
    rows = np.zeros((max(n_rows.value, 1), 8), dtype=np.int32)
    _check(lib.kvd_schedule_describe(*args, rows.ctypes.data_as(ctypes.c_void_p), n_rows.value,
                                     ctypes.byref(n_rows), ctypes.byref(eff)),
           "kvd_schedule_describe")
    return rows[:n_rows.value], eff.value


# ---------------------------------------------------------------------------
# GPU entry points (torch CUDA tensors in, results written in place)
# ---------------------------------------------------------------------------

def _require(t, name, dtype=None, ndim=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def kv_append(k_cache, v_cache, k_new, v_new, pos, status=None, stream=None):
    """k_cache[b, pos[b], h, :] = k_new[b, h, :] (and V), on the GPU."""
    import torch
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _require(t, n, torch.bfloat16, 4)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _require(t, n, torch.bfloat16, 3)
    _require(pos, "pos", torch.int32, 1)
    B, S, Hkv, D = k_cache.shape
    if v_cache.shape != k_cache.shape or k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D) \
            or pos.shape != (B,):
        raise ValueError("kv_append: inconsistent shapes")
    _check(load().kvd_kv_append(k_cache.data_ptr(), v_cache.data_ptr(), k_new.data_ptr(),
                                v_new.data_ptr(), pos.data_ptr(), B, S, Hkv, D, _ptr(status),
                                _stream_handle(stream)), "kvd_kv_append")


def _decode_args(q, k_cache, v_cache, seq_lens, max_seq_len, scale, n_split, workspace, out,
                 lse, status, stream):
    import torch
    _require(q, "q", torch.bfloat16, 3)
    _require(k_cache, "k_cache", torch.bfloat16, 4)
    _require(v_cache, "v_cache", torch.bfloat16, 4)
    _require(seq_lens, "seq_lens", torch.int32, 1)
    _require(out, "out", None, 3)
    B, Hq, D = q.shape
    _, S, Hkv, Dk = k_cache.shape
    if k_cache.shape[0] != B or Dk != D or v_cache.shape != k_cache.shape or \
            seq_lens.shape != (B,) or out.shape != (B, Hq, D):
        raise ValueError("decode_attention: inconsistent shapes")
    if out.dtype == torch.bfloat16:
        code = OUT_BF16
    elif out.dtype == torch.float32:
        code = OUT_F32
    else:
        raise TypeError("out must be bfloat16 or float32")
    if lse is not None:
        _require(lse, "lse", torch.float32, 2)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(),
                                                           workspace.numel() * workspace.element_size())
    return [q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), seq_lens.data_ptr(), B, S,
            int(max_seq_len), Hq, Hkv, D, float(scale), int(n_split), ws_ptr, ws_bytes,
            out.data_ptr(), code, _ptr(lse), _ptr(status), _stream_handle(stream)]


def alloc_workspace(q, k_cache, max_seq_len: int, n_split: int = 0, out_dtype="bf16"):
    """A device workspace big enough for decode_attention with these arguments."""
    import torch
    B, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    with torch.cuda.device(q.device):
        _, nbytes = decode_plan(B, Hq, Hkv, D, max_seq_len, 0, n_split, out_dtype)
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)


def decode_attention(q, k_cache, v_cache, seq_lens, max_seq_len: int, scale: float, out,
                     workspace=None, n_split: int = 0, lse=None, status=None, stream=None):
    """out[b, h] = softmax(scale * q[b, h] . K[b, :L_b, h // G]) V[b, :L_b, h // G]."""
    args = _decode_args(q, k_cache, v_cache, seq_lens, max_seq_len, scale, n_split, workspace,
                        out, lse, status, stream)
    _check(load().kvd_decode_attention(*args), "kvd_decode_attention")


def decode_attention_static(q, k_cache, v_cache, seq_lens, max_seq_len: int, scale: float, out,
                            n_split: int = 0, lse=None, status=None, stream=None):
    """decode_attention using the library's own static scratch array (no workspace
    argument, nothing allocated). Calls that overlap on the GPU share that array."""
    a = _decode_args(q, k_cache, v_cache, seq_lens, max_seq_len, scale, n_split, None, out, lse,
                     status, stream)
    args = a[:12] + a[14:]  # drop workspace pointer and size
    _check(load().kvd_decode_attention_static(*args), "kvd_decode_attention_static")


def _paged_args(k_pages, v_pages, block_table, B, what):
    import torch
    _require(k_pages, "k_pages", torch.bfloat16, 4)
    _require(v_pages, "v_pages", torch.bfloat16, 4)
    _require(block_table, "block_table", torch.int32, 2)
    num_pages, page, Hkv, D = k_pages.shape
    if v_pages.shape != k_pages.shape or block_table.shape[0] != B:
        raise ValueError(f"{what}: inconsistent shapes")
    return block_table.shape[1], page, num_pages, Hkv, D


def kv_append_paged(k_pages, v_pages, k_new, v_new, block_table, pos, status=None, stream=None):
    """Paged kv_append: the new rows go to row pos[b] % page of page
    block_table[b, pos[b] // page] of the pools [num_pages, page, Hkv, D]."""
    import torch
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _require(t, n, torch.bfloat16, 3)
    _require(pos, "pos", torch.int32, 1)
    B = k_new.shape[0]
    max_blocks, page, num_pages, Hkv, D = _paged_args(k_pages, v_pages, block_table, B, "kv_append_paged")
    if k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D) or pos.shape != (B,):
        raise ValueError("kv_append_paged: inconsistent shapes")
    _check(load().kvd_kv_append_paged(k_pages.data_ptr(), v_pages.data_ptr(), k_new.data_ptr(),
                                      v_new.data_ptr(), block_table.data_ptr(), pos.data_ptr(), B,
                                      max_blocks, page, num_pages, Hkv, D, _ptr(status),
                                      _stream_handle(stream)), "kvd_kv_append_paged")


def _decode_paged_args(q, k_pages, v_pages, block_table, seq_lens, max_seq_len, scale, n_split,
                       workspace, out, lse, status, stream):
    B = q.shape[0]
    max_blocks, page, num_pages, _, _ = _paged_args(k_pages, v_pages, block_table, B, "decode_attention_paged")
    import torch
    _require(q, "q", torch.bfloat16, 3)
    _require(seq_lens, "seq_lens", torch.int32, 1)
    _require(out, "out", None, 3)
    _, Hq, D = q.shape
    Hkv = k_pages.shape[2]
    if k_pages.shape[3] != D or seq_lens.shape != (B,) or out.shape != (B, Hq, D):
        raise ValueError("decode_attention_paged: inconsistent shapes")
    if out.dtype == torch.bfloat16:
        code = OUT_BF16
    elif out.dtype == torch.float32:
        code = OUT_F32
    else:
        raise TypeError("out must be bfloat16 or float32")
    if lse is not None:
        _require(lse, "lse", torch.float32, 2)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(),
                                                           workspace.numel() * workspace.element_size())
    head = [B, max_blocks, page, num_pages]
    tail = [int(max_seq_len), Hq, Hkv, D, float(scale), int(n_split), ws_ptr, ws_bytes, out.data_ptr(),
            code, _ptr(lse), _ptr(status), _stream_handle(stream)]
    return head, tail


def decode_attention_paged(q, k_pages, v_pages, block_table, seq_lens, max_seq_len: int, scale: float,
                           out, workspace=None, n_split: int = 0, lse=None, status=None, stream=None):
    """decode_attention over a paged cache: pools [num_pages, page, Hkv, D] and
    block_table [B, max_blocks] (token t of sequence b is row t % page of page
    block_table[b, t // page]). Workspace as for decode_attention."""
    head, tail = _decode_paged_args(q, k_pages, v_pages, block_table, seq_lens, max_seq_len, scale,
                                    n_split, workspace, out, lse, status, stream)
    _check(load().kvd_decode_attention_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                                             block_table.data_ptr(), seq_lens.data_ptr(), *head, *tail),
           "kvd_decode_attention_paged")


def decode_step_paged(q, k_pages, v_pages, k_new, v_new, pos, block_table, seq_lens, max_seq_len: int,
                      scale: float, out, workspace=None, n_split: int = 0, lse=None, status=None,
                      stream=None):
    """kv_append_paged then decode_attention_paged as one call (kvd_decode_step_paged)."""
    import torch
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _require(t, n, torch.bfloat16, 3)
    _require(pos, "pos", torch.int32, 1)
    B = q.shape[0]
    Hkv, D = k_pages.shape[2], k_pages.shape[3]
    if k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D) or pos.shape != (B,):
        raise ValueError("decode_step_paged: inconsistent shapes")
    head, tail = _decode_paged_args(q, k_pages, v_pages, block_table, seq_lens, max_seq_len, scale,
                                    n_split, workspace, out, lse, status, stream)
    _check(load().kvd_decode_step_paged(k_pages.data_ptr(), v_pages.data_ptr(), k_new.data_ptr(),
                                        v_new.data_ptr(), pos.data_ptr(), q.data_ptr(),
                                        block_table.data_ptr(), seq_lens.data_ptr(), *head, *tail),
           "kvd_decode_step_paged")


def _code_dtypes(fmt):
    """Tensor dtypes an 8-bit cache's codes may have: int8, or for fp8 E4M3
    bytes (uint8) or torch's float8_e4m3fn (the same bits)."""
    import torch
    if fmt == "int8":
        return (torch.int8,)
    if fmt == "fp8":
        return (torch.uint8, torch.float8_e4m3fn)
    raise ValueError(f"unknown 8-bit cache format {fmt!r}")


def _is_fp8(codes) -> bool:
    import torch
    return codes.dtype in (torch.uint8, torch.float8_e4m3fn)


def _q8_args(k_codes, v_codes, k_scales, v_scales, fmt="int8"):
    import torch
    _require(k_codes, "k_codes", _code_dtypes(fmt), 4)
    _require(v_codes, "v_codes", _code_dtypes(fmt), 4)
    _require(k_scales, "k_scales", torch.float32, 3)
    _require(v_scales, "v_scales", torch.float32, 3)
    if v_codes.shape != k_codes.shape or k_scales.shape != k_codes.shape[:3] or v_scales.shape != k_scales.shape:
        raise ValueError(f"{fmt} cache: codes [B, S_max, Hkv, D] and scales [B, S_max, Hkv] disagree")


def _quantize8(cache, codes, scales, seq_lens, max_seq_len, stream, fmt):
    import torch
    _require(cache, "cache", torch.bfloat16, 4)
    _require(codes, "codes", _code_dtypes(fmt), 4)
    _require(scales, "scales", torch.float32, 3)
    _require(seq_lens, "seq_lens", torch.int32, 1)
    B, S, Hkv, D = cache.shape
    if codes.shape != cache.shape or scales.shape != (B, S, Hkv) or seq_lens.shape != (B,):
        raise ValueError(f"kv_quantize_{fmt}: inconsistent shapes")
    name = "kvd_kv_quantize_q8" if fmt == "int8" else "kvd_kv_quantize_fp8"
    _check(getattr(load(), name)(cache.data_ptr(), codes.data_ptr(), scales.data_ptr(), seq_lens.data_ptr(), B, S,
                                 int(max_seq_len), Hkv, D, _stream_handle(stream)), name)


def kv_quantize_q8(cache, codes, scales, seq_lens, max_seq_len: int, stream=None):
    """int8 codes/scales of rows t < seq_lens[b] of a bf16 cache [B, S_max, Hkv, D]."""
    _quantize8(cache, codes, scales, seq_lens, max_seq_len, stream, "int8")


def kv_quantize_fp8(cache, codes, scales, seq_lens, max_seq_len: int, stream=None):
    """fp8 E4M3 codes (uint8 or float8_e4m3fn) and scales of rows t < seq_lens[b]
    of a bf16 cache [B, S_max, Hkv, D] (kvd_kv_quantize_fp8)."""
    _quantize8(cache, codes, scales, seq_lens, max_seq_len, stream, "fp8")


def _append8(k_codes, v_codes, k_scales, v_scales, k_new, v_new, pos, status, stream, fmt):
    import torch
    _q8_args(k_codes, v_codes, k_scales, v_scales, fmt)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _require(t, n, torch.bfloat16, 3)
    _require(pos, "pos", torch.int32, 1)
    B, S, Hkv, D = k_codes.shape
    if k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D) or pos.shape != (B,):
        raise ValueError(f"kv_append_{fmt}: inconsistent shapes")
    name = "kvd_kv_append_q8" if fmt == "int8" else "kvd_kv_append_fp8"
    _check(getattr(load(), name)(k_codes.data_ptr(), v_codes.data_ptr(), k_scales.data_ptr(), v_scales.data_ptr(),
                                 k_new.data_ptr(), v_new.data_ptr(), pos.data_ptr(), B, S, Hkv, D, _ptr(status),
                                 _stream_handle(stream)), name)


def kv_append_q8(k_codes, v_codes, k_scales, v_scales, k_new, v_new, pos, status=None, stream=None):
    """The new bf16 rows quantized and written at pos[b] of the int8 cache."""
    _append8(k_codes, v_codes, k_scales, v_scales, k_new, v_new, pos, status, stream, "int8")


def kv_append_fp8(k_codes, v_codes, k_scales, v_scales, k_new, v_new, pos, status=None, stream=None):
    """The new bf16 rows quantized to fp8 E4M3 and written at pos[b] (kvd_kv_append_fp8)."""
    _append8(k_codes, v_codes, k_scales, v_scales, k_new, v_new, pos, status, stream, "fp8")


def _append8_paged(k_code_pages, v_code_pages, k_scale_pages, v_scale_pages, k_new, v_new, block_table, pos,
                   status, stream, fmt):
    import torch
    _q8_args(k_code_pages, v_code_pages, k_scale_pages, v_scale_pages, fmt)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _require(t, n, torch.bfloat16, 3)
    _require(pos, "pos", torch.int32, 1)
    _require(block_table, "block_table", torch.int32, 2)
    num_pages, page, Hkv, D = k_code_pages.shape
    B = k_new.shape[0]
    if (k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D) or pos.shape != (B,)
            or block_table.shape[0] != B):
        raise ValueError(f"kv_append_{fmt}_paged: inconsistent shapes")
    name = "kvd_kv_append_q8_paged" if fmt == "int8" else "kvd_kv_append_fp8_paged"
    _check(getattr(load(), name)(k_code_pages.data_ptr(), v_code_pages.data_ptr(), k_scale_pages.data_ptr(),
                                 v_scale_pages.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), block_table.data_ptr(),
                                 pos.data_ptr(), B, block_table.shape[1], page, num_pages, Hkv, D, _ptr(status),
                                 _stream_handle(stream)), name)


def kv_append_q8_paged(k_code_pages, v_code_pages, k_scale_pages, v_scale_pages, k_new, v_new, block_table, pos,
                       status=None, stream=None):
    """The new bf16 rows quantized and written, as kv_append_paged places them,
    into int8 page pools: codes [num_pages, page, Hkv, D], scales
    [num_pages, page, Hkv]."""
    _append8_paged(k_code_pages, v_code_pages, k_scale_pages, v_scale_pages, k_new, v_new, block_table, pos,
                   status, stream, "int8")


def kv_append_fp8_paged(k_code_pages, v_code_pages, k_scale_pages, v_scale_pages, k_new, v_new, block_table, pos,
                        status=None, stream=None):
    """kv_append_q8_paged for fp8 E4M3 page pools (kvd_kv_append_fp8_paged)."""
    _append8_paged(k_code_pages, v_code_pages, k_scale_pages, v_scale_pages, k_new, v_new, block_table, pos,
                   status, stream, "fp8")


def _decode_q8_args(q, k_codes, v_codes, k_scales, v_scales, seq_lens, max_seq_len, scale, n_split, workspace,
                    out, lse, status, stream):
    """(seq_lens pointer, batch, s_max, ...) as for kvd_decode_attention, after the int8 cache."""
    import torch
    _q8_args(k_codes, v_codes, k_scales, v_scales)
    _require(q, "q", torch.bfloat16, 3)
    _require(seq_lens, "seq_lens", torch.int32, 1)
    _require(out, "out", None, 3)
    B, Hq, D = q.shape
    _, S, Hkv, Dk = k_codes.shape
    if k_codes.shape[0] != B or Dk != D or seq_lens.shape != (B,) or out.shape != (B, Hq, D):
        raise ValueError("decode_attention_q8: inconsistent shapes")
    if out.dtype == torch.bfloat16:
        code = OUT_BF16
    elif out.dtype == torch.float32:
        code = OUT_F32
    else:
        raise TypeError("out must be bfloat16 or float32")
    if lse is not None:
        _require(lse, "lse", torch.float32, 2)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(),
                                                           workspace.numel() * workspace.element_size())
    return [seq_lens.data_ptr(), B, S, int(max_seq_len), Hq, Hkv, D, float(scale), int(n_split), ws_ptr, ws_bytes,
            out.data_ptr(), code, _ptr(lse), _ptr(status), _stream_handle(stream)]


def decode_attention_q8(q, k_codes, v_codes, k_scales, v_scales, seq_lens, max_seq_len: int, scale: float, out,
                        workspace=None, n_split: int = 0, lse=None, status=None, stream=None):
    """decode_attention over an int8 cache (codes [B, S_max, Hkv, D] int8, scales
    [B, S_max, Hkv] float32; a row reads back as scale * code). Any group."""
    tail = _decode_q8_args(q, k_codes, v_codes, k_scales, v_scales, seq_lens, max_seq_len, scale, n_split,
                           workspace, out, lse, status, stream)
    _check(load().kvd_decode_attention_q8(q.data_ptr(), k_codes.data_ptr(), v_codes.data_ptr(),
                                          k_scales.data_ptr(), v_scales.data_ptr(), *tail),
           "kvd_decode_attention_q8")


def decode_step_q8(q, k_codes, v_codes, k_scales, v_scales, k_new, v_new, pos, seq_lens, max_seq_len: int,
                   scale: float, out, workspace=None, n_split: int = 0, lse=None, status=None, stream=None):
    """kv_append_q8 then decode_attention_q8 as one call (kvd_decode_step_q8)."""
    import torch
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _require(t, n, torch.bfloat16, 3)
    _require(pos, "pos", torch.int32, 1)
    B, S, Hkv, D = k_codes.shape
    if k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D) or pos.shape != (B,):
        raise ValueError("decode_step_q8: inconsistent shapes")
    tail = _decode_q8_args(q, k_codes, v_codes, k_scales, v_scales, seq_lens, max_seq_len, scale, n_split,
                           workspace, out, lse, status, stream)
    _check(load().kvd_decode_step_q8(k_codes.data_ptr(), v_codes.data_ptr(), k_scales.data_ptr(),
                                     v_scales.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), pos.data_ptr(),
                                     q.data_ptr(), *tail), "kvd_decode_step_q8")


def decode_plan_multi(batch: int, n_tokens: int, n_heads_q: int, n_heads_kv: int, head_dim: int,
                      max_seq_len: int, num_sms: int = 0, n_split: int = 0, out_dtype="bf16") -> Tuple[int, int]:
    """(n_split, workspace_bytes) for a multi-token call of this shape."""
    lib = load()
    n = ctypes.c_int(0)
    ws = ctypes.c_size_t(0)
    _check(lib.kvd_decode_plan_multi(batch, n_tokens, n_heads_q, n_heads_kv, head_dim, max_seq_len, num_sms,
                                     n_split, _out_code(out_dtype), ctypes.byref(n), ctypes.byref(ws)),
           "kvd_decode_plan_multi")
    return n.value, ws.value


def kv_append_multi(k_cache, v_cache, k_new, v_new, pos, status=None, stream=None):
    """The T new rows of each sequence (k_new [B, T, Hkv, D]) at pos[b] + i."""
    import torch
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _require(t, n, torch.bfloat16, 4)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _require(t, n, torch.bfloat16, 4)
    _require(pos, "pos", torch.int32, 1)
    B, S, Hkv, D = k_cache.shape
    T = k_new.shape[1]
    if v_cache.shape != k_cache.shape or k_new.shape != (B, T, Hkv, D) or v_new.shape != k_new.shape \
            or pos.shape != (B,):
        raise ValueError("kv_append_multi: inconsistent shapes")
    _check(load().kvd_kv_append_multi(k_cache.data_ptr(), v_cache.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                      pos.data_ptr(), B, T, S, Hkv, D, _ptr(status), _stream_handle(stream)),
           "kvd_kv_append_multi")


def _decode_multi_args(q, k_cache, v_cache, seq_lens, max_seq_len, scale, n_split, workspace, out, lse, status,
                       stream):
    import torch
    _require(q, "q", torch.bfloat16, 4)
    _require(out, "out", None, 4)
    B, T, Hq, D = q.shape
    if out.shape != q.shape:
        raise ValueError("decode_attention_multi: out must be [B, T, Hq, D]")
    if lse is not None:
        _require(lse, "lse", torch.float32, 3)
        if lse.shape != (B, T, Hq):
            raise ValueError("decode_attention_multi: lse must be [B, T, Hq]")
    # the single-token checks on [B, T*Hq, D] views (rows of one sequence are contiguous)
    a = _decode_args(q.view(B, T * Hq, D), k_cache, v_cache, seq_lens, max_seq_len, scale, n_split, workspace,
                     out.view(B, T * Hq, D), None if lse is None else lse.view(B, T * Hq), status, stream)
    a[7] = Hq  # n_heads_q proper
    return a[:5] + [T] + a[5:]


def decode_attention_multi(q, k_cache, v_cache, seq_lens, max_seq_len: int, scale: float, out, workspace=None,
                           n_split: int = 0, lse=None, status=None, stream=None):
    """T query tokens per sequence (q, out [B, T, Hq, D]); token i attends to the
    first seq_lens[b] - T + 1 + i cached tokens. T from 1 to 64."""
    args = _decode_multi_args(q, k_cache, v_cache, seq_lens, max_seq_len, scale, n_split, workspace, out, lse,
                              status, stream)
    _check(load().kvd_decode_attention_multi(*args), "kvd_decode_attention_multi")


def decode_step_multi(q, k_cache, v_cache, k_new, v_new, pos, seq_lens, max_seq_len: int, scale: float, out,
                      workspace=None, n_split: int = 0, lse=None, status=None, stream=None):
    """kv_append_multi then decode_attention_multi as one call (kvd_decode_step_multi)."""
    import torch
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _require(t, n, torch.bfloat16, 4)
    _require(pos, "pos", torch.int32, 1)
    a = _decode_multi_args(q, k_cache, v_cache, seq_lens, max_seq_len, scale, n_split, workspace, out, lse,
                           status, stream)
    B, T, Hq, D = q.shape
    if k_new.shape != (B, T, k_cache.shape[2], D) or v_new.shape != k_new.shape or pos.shape != (B,):
        raise ValueError("decode_step_multi: inconsistent shapes")
    # (k_cache, v_cache, k_new, v_new, pos, q, seq_lens, batch, T, ...)
    args = [a[1], a[2], k_new.data_ptr(), v_new.data_ptr(), pos.data_ptr(), a[0], a[3], a[4], a[5]] + a[6:]
    _check(load().kvd_decode_step_multi(*args), "kvd_decode_step_multi")


def decode_ex(q, k, v, seq_lens, max_seq_len: int, scale: float, out, *, k_scales=None, v_scales=None,
              block_table=None, k_new=None, v_new=None, pos=None, workspace=None, n_split: int = 0, lse=None,
              status=None, stream=None):
    """Any supported combination in one call (kvd_decode_ex): q [B, Hq, D] or
    [B, T, Hq, D]; k, v a contiguous cache [B, S_max, Hkv, D] (bf16, or 8-bit
    codes with k_scales/v_scales [B, S_max, Hkv]: int8 codes, or fp8 E4M3 codes
    as uint8 or float8_e4m3fn) or, with block_table [B, max_blocks], page pools
    [num_pages, page, Hkv, D] (bf16, or 8-bit codes with scale pools
    [num_pages, page, Hkv]); k_new, v_new ([B, Hkv, D] or [B, T, Hkv, D]) and pos
    to append first. Workspace: decode_plan_multi."""
    import torch
    T = q.shape[1] if q.dim() == 4 else 1
    B, Hq, D = q.shape[0], q.shape[-2], q.shape[-1]
    Hkv = k.shape[2]
    c = _CCache()
    c.k, c.v = k.data_ptr(), v.data_ptr()
    c.k_scales, c.v_scales = _ptr(k_scales), _ptr(v_scales)
    c.fp8 = 1 if (k_scales is not None and _is_fp8(k)) else 0
    if block_table is not None:
        _require(block_table, "block_table", torch.int32, 2)
        c.block_table, c.max_blocks, c.page_size, c.num_pages = (block_table.data_ptr(), block_table.shape[1],
                                                                   k.shape[1], k.shape[0])
    else:
        c.s_max = k.shape[1]
    if out.shape != q.shape or k.shape[3] != D or v.shape != k.shape:
        raise ValueError("decode_ex: inconsistent shapes")
    code = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32 if out.dtype == torch.float32 else None
    if code is None:
        raise TypeError("out must be bfloat16 or float32")
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(),
                                                           workspace.numel() * workspace.element_size())
    _check(load().kvd_decode_ex(ctypes.byref(c), q.data_ptr(), seq_lens.data_ptr(), B, T, int(max_seq_len), Hq,
                                Hkv, D, float(scale), int(n_split), ws_ptr, ws_bytes, out.data_ptr(), code,
                                _ptr(lse), _ptr(k_new), _ptr(v_new), _ptr(pos), _ptr(status),
                                _stream_handle(stream)), "kvd_decode_ex")


def decode_step(q, k_cache, v_cache, k_new, v_new, pos, seq_lens, max_seq_len: int, scale: float,
                out, workspace=None, n_split: int = 0, lse=None, status=None, stream=None):
    """kv_append(k_cache, v_cache, k_new, v_new, pos) then decode_attention(...), as one
    call whose attention launch starts while the append runs (kvd_decode_step)."""
    import torch
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _require(t, n, torch.bfloat16, 3)
    _require(pos, "pos", torch.int32, 1)
    B, S, Hkv, D = k_cache.shape
    if k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D) or pos.shape != (B,):
        raise ValueError("decode_step: inconsistent shapes")
    a = _decode_args(q, k_cache, v_cache, seq_lens, max_seq_len, scale, n_split, workspace, out,
                     lse, status, stream)
    args = [a[1], a[2], k_new.data_ptr(), v_new.data_ptr(), pos.data_ptr(), a[0], a[3]] + a[4:]
    _check(load().kvd_decode_step(*args), "kvd_decode_step")


def decode_attention_umax(q, k_cache, v_cache, seq_lens, max_seq_len: int, scale: float, phi: float, out,
                          workspace=None, n_split: int = 0, lse=None, status=None, stream=None):
    """decode_attention with the unified-maximum softmax: every split's partial
    softmax is taken against phi (logit units) while a row's scores allow,
    so the merge is a plain sum (kvd_decode_attention_umax)."""
    a = _decode_args(q, k_cache, v_cache, seq_lens, max_seq_len, scale, n_split, workspace, out, lse, status,
                     stream)
    _check(load().kvd_decode_attention_umax(*(a[:11] + [float(phi)] + a[11:])), "kvd_decode_attention_umax")


def decode_step_umax(q, k_cache, v_cache, k_new, v_new, pos, seq_lens, max_seq_len: int, scale: float, phi: float,
                     out, workspace=None, n_split: int = 0, lse=None, status=None, stream=None):
    """decode_step with the unified-maximum softmax (kvd_decode_step_umax)."""
    import torch
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _require(t, n, torch.bfloat16, 3)
    _require(pos, "pos", torch.int32, 1)
    B, S, Hkv, D = k_cache.shape
    if k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D) or pos.shape != (B,):
        raise ValueError("decode_step_umax: inconsistent shapes")
    a = _decode_args(q, k_cache, v_cache, seq_lens, max_seq_len, scale, n_split, workspace, out, lse, status,
                     stream)
    args = [a[1], a[2], k_new.data_ptr(), v_new.data_ptr(), pos.data_ptr(), a[0], a[3]] + a[4:11] + [float(phi)] + a[11:]
    _check(load().kvd_decode_step_umax(*args), "kvd_decode_step_umax")


def merge_attention(outs, lses, out, lse=None, stream=None):
    """Results over disjoint token shards combined by their normalisers
    (kvd_merge_attention): outs [n, ..., D] bf16 or fp32 and lses [n, ...] fp32
    as the attention calls return out and lse; out [..., D] bf16 or fp32."""
    import torch
    _require(outs, "outs", (torch.bfloat16, torch.float32))
    _require(lses, "lses", torch.float32)
    _require(out, "out", (torch.bfloat16, torch.float32))
    n, D = outs.shape[0], outs.shape[-1]
    if lses.shape != outs.shape[:-1] or out.shape != outs.shape[1:]:
        raise ValueError("merge_attention: outs [n, ..., D], lses [n, ...] and out [..., D] disagree")
    if lse is not None:
        _require(lse, "lse", torch.float32)
        if lse.shape != lses.shape[1:]:
            raise ValueError("merge_attention: lse must be shaped like lses[0]")
    rows = out.numel() // D
    code = lambda t: OUT_BF16 if t.dtype == torch.bfloat16 else OUT_F32
    _check(load().kvd_merge_attention(outs.data_ptr(), lses.data_ptr(), n, rows, D, code(outs), out.data_ptr(),
                                      code(out), _ptr(lse), _stream_handle(stream)), "kvd_merge_attention")


def probe_read(src, nbytes: int = 0, ctas: int = 0, sink=None, status=None, stream=None):
    """One read-only streaming pass over a device tensor's bytes (kvd_probe_read):
    a measurement aid giving the read ceiling of a kernel that reads those
    bytes once. nbytes = 0 reads the whole tensor."""
    n = nbytes or src.numel() * src.element_size()
    _check(load().kvd_probe_read(src.data_ptr(), n, ctas, _ptr(sink), _ptr(status), _stream_handle(stream)),
           "kvd_probe_read")


def step_staging_bytes(batch: int, n_tokens: int, n_heads_q: int, n_heads_kv: int, head_dim: int) -> int:
    """Device staging bytes decode_step_host needs (kvd_step_staging_bytes)."""
    return int(load().kvd_step_staging_bytes(batch, n_tokens, n_heads_q, n_heads_kv, head_dim))


class HostStep:
    """A step from host inputs to a host result (kvd_decode_step_host) with its
    buffers bound once: the CPU tensors q_host [B, Hq, D] or [B, T, Hq, D]
    (bf16), k_new_host, v_new_host ([B, Hkv, D] or [B, T, Hkv, D]), pos_host,
    seq_lens_host (int32 [B]), the device cache, the device buffer `staging`
    (step_staging_bytes), `out` and its CPU copy out_host. Each call copies the
    host inputs' current contents in, runs the step and copies `out` back, on
    `stream` (pin the host tensors for asynchronous copies); nothing is
    synchronised. With out=None the kernels write the result straight into the
    pinned out_host. Arguments are checked here and by the library on every call."""

    def __init__(self, q_host, k_new_host, v_new_host, pos_host, seq_lens_host, k_cache, v_cache, staging,
                 max_seq_len: int, scale: float, out, out_host, workspace=None, n_split: int = 0, lse=None,
                 status=None, stream=None):
        import torch
        for t, n in ((q_host, "q_host"), (k_new_host, "k_new_host"), (v_new_host, "v_new_host")):
            if t.dtype != torch.bfloat16 or t.device.type != "cpu" or not t.is_contiguous():
                raise TypeError(f"{n} must be a contiguous bfloat16 CPU tensor")
        for t, n in ((pos_host, "pos_host"), (seq_lens_host, "seq_lens_host")):
            if t.dtype != torch.int32 or t.device.type != "cpu" or not t.is_contiguous():
                raise TypeError(f"{n} must be a contiguous int32 CPU tensor")
        # out None: the kernels write the result straight into out_host (pinned)
        if out is None and not out_host.is_pinned():
            raise ValueError("out=None needs a pinned out_host")
        like = out if out is not None else out_host
        if out_host.device.type != "cpu" or out_host.dtype != like.dtype or out_host.shape != like.shape:
            raise TypeError("out_host must be a CPU tensor like out")
        _require(k_cache, "k_cache", torch.bfloat16, 4)
        _require(v_cache, "v_cache", torch.bfloat16, 4)
        T = q_host.shape[1] if q_host.dim() == 4 else 1
        B, Hq, D = q_host.shape[0], q_host.shape[-2], q_host.shape[-1]
        S, Hkv = k_cache.shape[1], k_cache.shape[2]
        code = OUT_BF16 if like.dtype == torch.bfloat16 else OUT_F32 if like.dtype == torch.float32 else None
        if code is None or like.shape != q_host.shape:
            raise TypeError("out must be bfloat16 or float32, shaped like q")
        ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(),
                                                               workspace.numel() * workspace.element_size())
        self._keep = (q_host, k_new_host, v_new_host, pos_host, seq_lens_host, k_cache, v_cache, staging, out,
                      out_host, workspace, lse, status)
        self._fn = load().kvd_decode_step_host
        self._args = (k_cache.data_ptr(), v_cache.data_ptr(), q_host.data_ptr(), k_new_host.data_ptr(),
                      v_new_host.data_ptr(), pos_host.data_ptr(), seq_lens_host.data_ptr(), staging.data_ptr(),
                      staging.numel() * staging.element_size(), B, T, S, int(max_seq_len), Hq, Hkv, D,
                      float(scale), int(n_split), ws_ptr, ws_bytes, None if out is None else out.data_ptr(),
                      out_host.data_ptr(), code,
                      _ptr(lse), _ptr(status), _stream_handle(stream))

    def __call__(self):
        _check(self._fn(*self._args), "kvd_decode_step_host")


def alloc_host_packet(batch: int, n_tokens: int, n_heads_q: int, n_heads_kv: int, head_dim: int):
    """One pinned host buffer laid out like decode_step_host's staging buffer,
    and its views (q, k_new, v_new, pos, seq_lens; shapes as decode_step_host
    takes them). A HostStep over these views copies its inputs in one copy."""
    import torch
    B, T = batch, n_tokens
    al = lambda n: -(-n // 256) * 256
    nq, nk, ni = B * T * n_heads_q * head_dim * 2, B * T * n_heads_kv * head_dim * 2, B * 4
    packet = torch.empty(step_staging_bytes(B, T, n_heads_q, n_heads_kv, head_dim), dtype=torch.uint8).pin_memory()
    offs = [0, al(nq), al(nq) + al(nk), al(nq) + 2 * al(nk), al(nq) + 2 * al(nk) + al(ni)]
    qs = (B, n_heads_q, head_dim) if T == 1 else (B, T, n_heads_q, head_dim)
    ks = (B, n_heads_kv, head_dim) if T == 1 else (B, T, n_heads_kv, head_dim)
    q = packet[offs[0]:offs[0] + nq].view(torch.bfloat16).view(qs)
    kn = packet[offs[1]:offs[1] + nk].view(torch.bfloat16).view(ks)
    vn = packet[offs[2]:offs[2] + nk].view(torch.bfloat16).view(ks)
    pos = packet[offs[3]:offs[3] + ni].view(torch.int32)
    lens = packet[offs[4]:offs[4] + ni].view(torch.int32)
    return packet, q, kn, vn, pos, lens


def decode_step_host(q_host, k_new_host, v_new_host, pos_host, seq_lens_host, k_cache, v_cache, staging,
                     max_seq_len: int, scale: float, out, out_host, workspace=None, n_split: int = 0, lse=None,
                     status=None, stream=None):
    """One HostStep call: copy the host inputs in, run the step, copy out back."""
    HostStep(q_host, k_new_host, v_new_host, pos_host, seq_lens_host, k_cache, v_cache, staging, max_seq_len,
             scale, out, out_host, workspace, n_split, lse, status, stream)()


def split_kv_chunk(q, k_cache, v_cache, seq_lens, max_seq_len: int, scale: float, out,
                   workspace=None, n_split: int = 0, lse=None, status=None, stream=None):
    """First launch of decode_attention only (the split-KV chunk kernel)."""
    args = _decode_args(q, k_cache, v_cache, seq_lens, max_seq_len, scale, n_split, workspace,
                        out, lse, status, stream)
    _check(load().kvd_split_kv_chunk(*args), "kvd_split_kv_chunk")


def split_kv_merge(q, k_cache, v_cache, seq_lens, max_seq_len: int, scale: float, out,
                   workspace=None, n_split: int = 0, lse=None, status=None, stream=None):
    """Second launch of decode_attention only (the log-sum-exp merge kernel)."""
    args = _decode_args(q, k_cache, v_cache, seq_lens, max_seq_len, scale, n_split, workspace,
                        out, lse, status, stream)
    _check(load().kvd_split_kv_merge(*args), "kvd_split_kv_merge")
