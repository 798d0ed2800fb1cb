"""Python binding of the GB300 grouped-query decode-attention library.

Argument marshalling only: tensors are passed to the C ABI in
``include/gqa_decode.h`` as raw device pointers with the current CUDA stream;
every step of the computation runs in the library's CUDA kernels. PyTorch
provides device memory and streams. There is no fallback: if the compiled
library is missing, loading raises.

Entry points (same names as the C ABI, without the ``gqa_`` prefix where it
would repeat the module name):

* ``kv_append``            -- write the new token(s) of every sequence into the paged cache
* ``gqa_decode``           -- grouped-query decode attention over the paged cache
                              (one or T causal new tokens per sequence, optional
                              sliding window)
* ``kv_append_varlen``     -- the same for a different number of new tokens per sequence
* ``gqa_prefill``          -- causal attention of prompts (any length) over the paged cache
* ``decode_workspace_size``-- workspace bytes ``gqa_decode`` needs
* ``kv_pool_elements``     -- elements a pool of ``num_blocks`` blocks holds (K and V)
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import threading
from typing import Optional

import torch

from . import build as _build

BLOCK_SIZE = 16
DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2, torch.int8: 3,
              torch.float8_e4m3fn: 4}

GQA_DEVERR_BLOCK_INDEX = 1
GQA_DEVERR_CONTEXT_LEN = 2
GQA_DEVERR_POSITION = 4
GQA_DEVERR_TIMEOUT = 8

KERNEL_AUTO, KERNEL_MMA, KERNEL_FMA = 0, 1, 2
GQA_DTYPE_I4 = 5
GQA_DTYPE_I4_KC = 6


class GqaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class KVCacheDesc(ctypes.Structure):
    """Mirror of gqa_kv_cache_t."""
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int64), ("num_kv_heads", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("stride_block", ctypes.c_int64),
                ("stride_head", ctypes.c_int64), ("stride_token", ctypes.c_int64),
                ("k_residual", ctypes.c_void_p), ("residual_rows", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class DecodeOpts(ctypes.Structure):
    """Mirror of gqa_decode_opts_t."""
    _fields_ = [("tokens_per_seq", ctypes.c_int32), ("sliding_window", ctypes.c_int32),
                ("kernel", ctypes.c_int32), ("max_warps", ctypes.c_int32),
                ("min_blocks_per_warp", ctypes.c_int32), ("row_layout", ctypes.c_int32),
                ("event_main_begin", ctypes.c_void_p), ("event_main_end", ctypes.c_void_p)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load the compiled library (build it first with ``build.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library not built: {path} is missing "
                                   "(run gqa_decode_attention_kv_gb300.build.build())")
            lib = ctypes.CDLL(path)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            lib.gqa_status_string.argtypes = [ctypes.c_int]
            lib.gqa_status_string.restype = ctypes.c_char_p
            lib.gqa_version.argtypes = []
            lib.gqa_version.restype = ctypes.c_int
            lib.gqa_kv_pool_elements.argtypes = [i64, i32, i32]
            lib.gqa_kv_pool_elements.restype = i64
            lib.gqa_kv_append.argtypes = [ctypes.POINTER(KVCacheDesc), vp, vp, i32, vp, i32, vp,
                                          i32, i32, vp, vp]
            lib.gqa_kv_append.restype = ctypes.c_int
            lib.gqa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
            lib.gqa_decode_workspace_size.restype = ctypes.c_size_t
            lib.gqa_decode.argtypes = [ctypes.POINTER(KVCacheDesc), vp, i32, i32, vp, i32, vp, i32,
                                       ctypes.c_float, vp, i32, vp, ctypes.c_size_t,
                                       ctypes.POINTER(DecodeOpts), vp, vp]
            lib.gqa_decode.restype = ctypes.c_int
            lib.gqa_decode_noalloc.argtypes = [ctypes.POINTER(KVCacheDesc), vp, i32, i32, vp, i32,
                                               vp, i32, ctypes.c_float, vp, i32,
                                               ctypes.POINTER(DecodeOpts), vp, vp]
            lib.gqa_decode_noalloc.restype = ctypes.c_int
            lib.gqa_kv_append_varlen.argtypes = [ctypes.POINTER(KVCacheDesc), vp, vp, i32, vp, i32, vp,
                                                 i32, vp, i32, vp, vp]
            lib.gqa_kv_append_varlen.restype = ctypes.c_int
            lib.gqa_prefill.argtypes = [ctypes.POINTER(KVCacheDesc), vp, i32, i32, vp, i32, vp, i32, vp,
                                        i32, ctypes.c_float, i32, vp, i32, i32, vp, vp]
            lib.gqa_prefill.restype = ctypes.c_int
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().gqa_status_string(int(status)).decode()


def version() -> int:
    return int(load().gqa_version())


def kv_pool_elements(num_blocks: int, num_kv_heads: int, head_dim: int) -> int:
    return int(load().gqa_kv_pool_elements(num_blocks, num_kv_heads, head_dim))


@dataclasses.dataclass
class PagedKVCache:
    """Device tensors of one paged KV cache plus their element strides.

    Default layout is the pool ``[num_blocks, K, 16, d]``; any layout whose
    element of (block p, kv-head g, slot s, dim i) is at
    ``p*stride_block + g*stride_head + s*stride_token + i`` works."""
    k: torch.Tensor
    v: torch.Tensor
    num_blocks: int
    num_kv_heads: int
    head_dim: int
    stride_block: int
    stride_head: int
    stride_token: int
    k_scale: Optional[torch.Tensor] = None
    v_scale: Optional[torch.Tensor] = None
    dtype_code: Optional[int] = None   # set for storage the tensor dtype does not name (int4)
    k_residual: Optional[torch.Tensor] = None   # KIVI-style cache: fp32 [rows, K, 16, d]

    @staticmethod
    def allocate(num_blocks: int, num_kv_heads: int, head_dim: int, dtype,
                 device="cuda", residual_rows: int = 0) -> "PagedKVCache":
        """dtype: a torch dtype; "int4" for two 4-bit codes per byte (uint8
        storage [num_blocks, K, 16, d/2]; strides still count 4-bit elements);
        "int4kc" for the same codes with K scaled per (block, kv-head, channel)
        (k_scale [num_blocks, K, d]) and a zeroed fp32 residual of
        ``residual_rows`` sequences."""
        int4 = dtype in ("int4", "int4kc")
        kc = dtype == "int4kc"
        shape = (num_blocks, num_kv_heads, BLOCK_SIZE, head_dim // 2 if int4 else head_dim)
        k = torch.empty(shape, dtype=torch.uint8 if int4 else dtype, device=device)
        v = torch.empty_like(k)
        ks = vs = res = None
        if int4 or dtype in (torch.int8, torch.float8_e4m3fn):
            vs = torch.empty((num_blocks, num_kv_heads, BLOCK_SIZE), dtype=torch.float16, device=device)
            ks = torch.empty((num_blocks, num_kv_heads, head_dim), dtype=torch.float16,
                             device=device) if kc else torch.empty_like(vs)
        if kc:
            res = torch.zeros((residual_rows, num_kv_heads, BLOCK_SIZE, head_dim), dtype=torch.float32,
                              device=device)
        code = GQA_DTYPE_I4_KC if kc else GQA_DTYPE_I4 if int4 else None
        return PagedKVCache(k, v, num_blocks, num_kv_heads, head_dim,
                            num_kv_heads * BLOCK_SIZE * head_dim, BLOCK_SIZE * head_dim, head_dim,
                            ks, vs, code, res)

    @property
    def dtype(self) -> torch.dtype:
        return self.k.dtype

    def desc(self) -> KVCacheDesc:
        return KVCacheDesc(
            self.k.data_ptr(), self.v.data_ptr(),
            self.k_scale.data_ptr() if self.k_scale is not None else None,
            self.v_scale.data_ptr() if self.v_scale is not None else None,
            self.num_blocks, self.num_kv_heads, BLOCK_SIZE, self.head_dim,
            self.dtype_code if self.dtype_code is not None else DTYPE_CODE[self.k.dtype],
            self.stride_block, self.stride_head, self.stride_token,
            self.k_residual.data_ptr() if self.k_residual is not None else None,
            int(self.k_residual.shape[0]) if self.k_residual is not None else 0, 0)


def _stream_ptr(stream) -> Optional[int]:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dev(t: Optional[torch.Tensor], name: str, index: bool = False, optional: bool = False):
    """Device pointer of a tensor the library reads or writes as a packed array.

    The C ABI sees a bare pointer, so what it cannot check is checked here:
    the tensor must be contiguous, an index array must be int32, and the memory
    must be on a CUDA device."""
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (the library reads it as a packed array)")
    if index and t.dtype != torch.int32:
        raise ValueError(f"{name} must be int32, not {t.dtype}")
    if not index and t.dtype not in DTYPE_CODE and t.dtype != torch.uint8:
        raise ValueError(f"{name} has unsupported dtype {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t.data_ptr()


def _on_cache_device(cache: "PagedKVCache", **tensors):
    """Every array must sit on the cache's device, and that device must be the
    current one: the library launches on the current device and reads the
    pointers it is given there."""
    dev = cache.k.device
    cur = torch.cuda.current_device() if torch.cuda.is_available() else None
    if dev.type == "cuda" and cur is not None and dev.index != cur:
        raise ValueError(f"the cache is on {dev} but the current device is cuda:{cur}")
    for name, t in tensors.items():
        if t is not None and t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the cache on {dev}")


def _check_table_and_lens(block_tables: torch.Tensor, lens: torch.Tensor, batch: int, lens_name: str,
                          lens_min: int):
    if block_tables.dim() != 2 or block_tables.shape[0] < batch:
        raise ValueError(f"block_tables must be [>= {batch}, max_blocks], not {tuple(block_tables.shape)}")
    if lens.dim() != 1 or lens.numel() < lens_min:
        raise ValueError(f"{lens_name} must be 1-D with >= {lens_min} entries, not {tuple(lens.shape)}")


def _check_query(cache: "PagedKVCache", q: torch.Tensor, dims: tuple):
    if q.dim() not in dims:
        raise ValueError(f"q must have {' or '.join(str(x) for x in dims)} dims, not {q.dim()}")
    H, d = int(q.shape[-2]), int(q.shape[-1])
    if d != cache.head_dim:
        raise ValueError(f"q's head_dim {d} differs from the cache's {cache.head_dim}")
    if H % cache.num_kv_heads:
        raise ValueError(f"{H} query heads are not a multiple of {cache.num_kv_heads} kv-heads")


def _check_out(q: torch.Tensor, out: Optional[torch.Tensor]):
    if out is not None and tuple(out.shape) != tuple(q.shape):
        raise ValueError(f"out must have q's shape {tuple(q.shape)}, not {tuple(out.shape)}")


def _check_new_rows(cache: "PagedKVCache", k_new: torch.Tensor, v_new: torch.Tensor, dims: tuple):
    if k_new.dim() not in dims or tuple(v_new.shape) != tuple(k_new.shape):
        raise ValueError(f"k_new and v_new must share one shape with {dims} dims, "
                         f"not {tuple(k_new.shape)} and {tuple(v_new.shape)}")
    if tuple(k_new.shape[-2:]) != (cache.num_kv_heads, cache.head_dim):
        raise ValueError(f"new rows end in {tuple(k_new.shape[-2:])}, the cache's heads and "
                         f"head_dim are {(cache.num_kv_heads, cache.head_dim)}")


def _check(status: int, where: str):
    if status != 0:
        raise GqaError(status, where)


def kv_append(cache: PagedKVCache, k_new: torch.Tensor, v_new: torch.Tensor,
              block_tables: torch.Tensor, positions: torch.Tensor,
              err: Optional[torch.Tensor] = None, stream=None) -> None:
    """Write k_new/v_new [B, K, d] (one token) or [B, T, K, d] (T tokens) at
    positions positions[b] .. positions[b]+T-1 of each sequence's paged cache."""
    T = 1 if k_new.dim() == 3 else int(k_new.shape[1])
    args = (_dev(k_new, "k_new"), _dev(v_new, "v_new"), _dev(block_tables, "block_tables", True),
            _dev(positions, "positions", True), _dev(err, "err", True, True))
    _check_new_rows(cache, k_new, v_new, (3, 4))
    B = int(positions.shape[0]) if positions.dim() == 1 else -1
    if B < 0 or int(k_new.shape[0]) != B:
        raise ValueError(f"positions must be [B] with B = k_new.shape[0] = {int(k_new.shape[0])}")
    _check_table_and_lens(block_tables, positions, B, "positions", B)
    _on_cache_device(cache, k_new=k_new, v_new=v_new, block_tables=block_tables,
                     positions=positions, err=err)
    desc = cache.desc()
    st = load().gqa_kv_append(ctypes.byref(desc), args[0], args[1], DTYPE_CODE[k_new.dtype], args[2],
                              int(block_tables.shape[1]), args[3], int(positions.shape[0]),
                              T, args[4], _stream_ptr(stream))
    _check(st, "gqa_kv_append")


def decode_workspace_size(batch: int, num_heads: int, num_kv_heads: int, head_dim: int,
                          device: int = -1, tokens_per_seq: int = 1) -> int:
    return int(load().gqa_decode_workspace_size(batch, num_heads, num_kv_heads, head_dim,
                                                tokens_per_seq, device))


_ws_cache: dict = {}


def workspace_for(batch: int, num_heads: int, num_kv_heads: int, head_dim: int,
                  device: torch.device, tokens_per_seq: int = 1, stream=None) -> torch.Tensor:
    """A cached, zero-initialised device workspace large enough for this shape,
    one per (device, stream): calls on one stream run in order, so they may
    share it; calls on different streams get different workspaces. The buffer
    is allocated on that stream, so a larger one replacing it is ordered after
    the calls already queued there."""
    dev = torch.device(device)
    idx = dev.index if dev.index is not None else torch.cuda.current_device()
    need = decode_workspace_size(batch, num_heads, num_kv_heads, head_dim, idx, tokens_per_seq)
    if need == 0:
        raise ValueError("no workspace size for this shape")
    s = stream if stream is not None else torch.cuda.current_stream(torch.device("cuda", idx))
    key = (idx, s.cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < need:
        # zero-filled once: the library keeps its run-time work counter at zero between calls
        with torch.cuda.stream(s):
            buf = torch.zeros(need, dtype=torch.uint8, device=dev)
        _ws_cache[key] = buf
    return buf


def gqa_decode(cache: PagedKVCache, q: torch.Tensor, block_tables: torch.Tensor,
               context_lens: torch.Tensor, scale: float, out: Optional[torch.Tensor] = None,
               out_dtype: torch.dtype = torch.float32, workspace: Optional[torch.Tensor] = None,
               kernel: int = KERNEL_AUTO, max_warps: int = 0, min_blocks_per_warp: int = 0,
               events: Optional[tuple] = None, err: Optional[torch.Tensor] = None,
               stream=None, window: int = 0, row_layout: int = 0) -> torch.Tensor:
    """out[b,h] = softmax(scale * q[b,h] . K_g^T) V_g over context_lens[b] cached tokens.

    q is [B, H, d] (one new token per sequence) or [B, T, H, d] (T new tokens,
    causal among themselves); ``window`` > 0 keeps each query's last ``window``
    positions. ``out`` has q's shape."""
    T = 1 if q.dim() == 3 else int(q.shape[1])
    B, H, d = q.shape[0], q.shape[-2], q.shape[-1]
    qp, tp, lp = _dev(q, "q"), _dev(block_tables, "block_tables", True), _dev(context_lens, "context_lens", True)
    ep = _dev(err, "err", True, True)
    _check_query(cache, q, (3, 4))
    _check_table_and_lens(block_tables, context_lens, B, "context_lens", B)
    _check_out(q, out)
    _on_cache_device(cache, q=q, block_tables=block_tables, context_lens=context_lens, out=out,
                     workspace=workspace, err=err)
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    if workspace is None:
        workspace = workspace_for(B, H, cache.num_kv_heads, d, q.device, T, stream)
    op, wp = _dev(out, "out"), _dev(workspace, "workspace")
    opts = DecodeOpts(T, window, kernel, max_warps, min_blocks_per_warp, row_layout, None, None)
    if events is not None:
        opts.event_main_begin = events[0].cuda_event
        opts.event_main_end = events[1].cuda_event
    desc = cache.desc()
    st = load().gqa_decode(ctypes.byref(desc), qp, DTYPE_CODE[q.dtype], H, tp,
                           int(block_tables.shape[1]), lp, B, float(scale),
                           op, DTYPE_CODE[out.dtype], wp, workspace.numel() * workspace.element_size(),
                           ctypes.byref(opts), ep, _stream_ptr(stream))
    _check(st, "gqa_decode")
    return out


def gqa_decode_noalloc(cache: PagedKVCache, q: torch.Tensor, block_tables: torch.Tensor,
                       context_lens: torch.Tensor, scale: float, out: Optional[torch.Tensor] = None,
                       out_dtype: torch.dtype = torch.float32, kernel: int = KERNEL_AUTO,
                       err: Optional[torch.Tensor] = None, stream=None,
                       window: int = 0) -> torch.Tensor:
    """gqa_decode with the library's built-in scratch instead of a workspace.

    For callers that may not allocate device memory; the output tensor is still
    the caller's (pass ``out`` to avoid even that allocation here). Calls that
    overlap on the GPU share one scratch array and race."""
    T = 1 if q.dim() == 3 else int(q.shape[1])
    B, H, d = q.shape[0], q.shape[-2], q.shape[-1]
    qp, tp, lp = _dev(q, "q"), _dev(block_tables, "block_tables", True), _dev(context_lens, "context_lens", True)
    ep = _dev(err, "err", True, True)
    _check_query(cache, q, (3, 4))
    _check_table_and_lens(block_tables, context_lens, B, "context_lens", B)
    _check_out(q, out)
    _on_cache_device(cache, q=q, block_tables=block_tables, context_lens=context_lens, out=out, err=err)
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    op = _dev(out, "out")
    opts = DecodeOpts(T, window, kernel, 0, 0, 0, None, None)
    desc = cache.desc()
    st = load().gqa_decode_noalloc(ctypes.byref(desc), qp, DTYPE_CODE[q.dtype], H,
                                   tp, int(block_tables.shape[1]),
                                   lp, B, float(scale), op,
                                   DTYPE_CODE[out.dtype], ctypes.byref(opts), ep,
                                   _stream_ptr(stream))
    _check(st, "gqa_decode_noalloc")
    return out


def kv_append_varlen(cache: PagedKVCache, k_new: torch.Tensor, v_new: torch.Tensor,
                     token_start: torch.Tensor, max_new_tokens: int, block_tables: torch.Tensor,
                     positions: torch.Tensor, err: Optional[torch.Tensor] = None, stream=None) -> None:
    """Write rows token_start[b] .. token_start[b+1]-1 of k_new/v_new [total, K, d] at
    positions positions[b], positions[b]+1, ... of sequence b."""
    args = (_dev(k_new, "k_new"), _dev(v_new, "v_new"), _dev(token_start, "token_start", True),
            _dev(block_tables, "block_tables", True), _dev(positions, "positions", True),
            _dev(err, "err", True, True))
    _check_new_rows(cache, k_new, v_new, (3,))
    B = int(positions.shape[0]) if positions.dim() == 1 else -1
    if B < 0:
        raise ValueError("positions must be 1-D")
    _check_table_and_lens(block_tables, positions, B, "positions", B)
    if token_start.dim() != 1 or token_start.numel() < B + 1:
        raise ValueError(f"token_start must be 1-D with >= {B + 1} entries")
    _on_cache_device(cache, k_new=k_new, v_new=v_new, token_start=token_start,
                     block_tables=block_tables, positions=positions, err=err)
    desc = cache.desc()
    st = load().gqa_kv_append_varlen(ctypes.byref(desc), args[0], args[1],
                                     DTYPE_CODE[k_new.dtype], args[2], int(max_new_tokens),
                                     args[3], int(block_tables.shape[1]), args[4],
                                     int(positions.shape[0]), args[5], _stream_ptr(stream))
    _check(st, "gqa_kv_append_varlen")


def gqa_prefill(cache: PagedKVCache, q: torch.Tensor, q_start: torch.Tensor, max_new_tokens: int,
                block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                out: Optional[torch.Tensor] = None, out_dtype: torch.dtype = torch.float32,
                window: int = 0, err: Optional[torch.Tensor] = None, stream=None,
                kernel: int = 0) -> torch.Tensor:
    """Causal attention of each sequence's new tokens (rows q_start[b] .. of q
    [total, H, d]) over its paged cache, new tokens included. kernel: 0 auto,
    1 tcgen05 one-tile (32-token chunks), 2 warp-level mma.sync, 3 tcgen05
    two-tile (64-token chunks, head_dim 128), 4 tcgen05 one-tile with 64-token
    chunks and two CTAs per SM (head_dim 128)."""
    args = (_dev(q, "q"), _dev(q_start, "q_start", True), _dev(block_tables, "block_tables", True),
            _dev(context_lens, "context_lens", True), _dev(err, "err", True, True))
    _check_query(cache, q, (3,))
    B = int(context_lens.shape[0]) if context_lens.dim() == 1 else -1
    if B < 0:
        raise ValueError("context_lens must be 1-D")
    _check_table_and_lens(block_tables, context_lens, B, "context_lens", B)
    if q_start.dim() != 1 or q_start.numel() < B + 1:
        raise ValueError(f"q_start must be 1-D with >= {B + 1} entries")
    _check_out(q, out)
    _on_cache_device(cache, q=q, q_start=q_start, block_tables=block_tables,
                     context_lens=context_lens, out=out, err=err)
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    op = _dev(out, "out")
    desc = cache.desc()
    st = load().gqa_prefill(ctypes.byref(desc), args[0], DTYPE_CODE[q.dtype], int(q.shape[1]),
                            args[1], int(max_new_tokens), args[2],
                            int(block_tables.shape[1]), args[3], B, float(scale), int(window),
                            op, DTYPE_CODE[out.dtype], int(kernel), args[4], _stream_ptr(stream))
    _check(st, "gqa_prefill")
    return out


def cache_from_case(case) -> PagedKVCache:
    """Wrap the device tensors of a generated decode case (gqa_inputs.DecodeCase)."""
    return PagedKVCache(case.k_cache, case.v_cache, case.num_blocks, case.num_kv_heads,
                        case.head_dim, case.stride_block, case.stride_head, case.stride_token,
                        case.k_scale, case.v_scale,
                        {"i4": GQA_DTYPE_I4, "i4kc": GQA_DTYPE_I4_KC}.get(case.cache_dtype),
                        getattr(case, "k_residual", None))
