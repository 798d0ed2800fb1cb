"""CPU oracle for one GQA decode step over a KV cache (fp64, plain and slow).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it. The CUDA library never imports, links or
calls anything here, and nothing here imports the CUDA library.

Functions and the passages they follow:

* ``decode``             -- GQA attention, "分组查询注意力 (GQA)", 技术原理 steps 2-4
                            and its attention equation (C, fp64, ``gqa_oracle.c``).
* ``gather_dense``       -- the block-table lookup of "LLM 推理性能优化实战" section 8.2:
                            token t of a sequence lives in physical block
                            ``table[t // 16]``, slot ``t % 16`` (block_size 16, the
                            KV-cache essay's "block_size=16" paragraph).
* ``append``             -- the paged write of one new token per sequence: slot
                            ``pos % 16`` of block ``table[pos // 16]``.
* ``quantize_int8`` / ``dequantize_int8`` -- symmetric per-(token, kv-head) int8,
                            "LLM 推理性能优化实战" sections 15.1, 15.2 and 15.5
                            (rounding rule in ``gqa_oracle.c``).
* ``quantize_fp8`` / ``dequantize_fp8`` -- FP8 E4M3 KV codes with per-(token,
                            kv-head) fp16 scales (section 15.5's FP8 option).
* ``quantize_int4_channels`` / ``gather_channel_scales`` / ``append_int4_channels``
                         -- the KIVI-style K cache of section 15.5 (K per channel, V per
                            token, INT4): one scale per (block, kv-head, channel).
* ``quantised_sequence`` -- what a code cache holds for one sequence's K or V rows
                            written from position 0 (the rules above, row by row or,
                            for the KIVI-style K, block by block per channel).
* ``kv_cache_elements``  -- the KV-size closed form 2 * layers * K * d * S * B,
                            "分组查询注意力 (GQA)" 关键参数 item 2 and
                            "LLM 推理性能优化实战" section 6.1.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lib = None
_lock = threading.Lock()

BLOCK_SIZE = 16


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain C99, no fast-math, no contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-O2", "-fno-fast-math",
           "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            i32 = ctypes.c_int32
            lib.oracle_gqa_decode.argtypes = [dp, dp, dp, ip, i32, i32, i32, i32, i32, i32, i32,
                                              ctypes.c_double, dp, i32]
            lib.oracle_gqa_decode.restype = ctypes.c_int
            lib.oracle_quantize_int8.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_int64,
                                                 ctypes.c_int32, ctypes.POINTER(ctypes.c_int8),
                                                 ctypes.POINTER(ctypes.c_uint16)]
            lib.oracle_quantize_int8.restype = None
            lib.oracle_f32_to_f16_bits.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_f16_bits.restype = ctypes.c_uint16
            lib.oracle_f16_bits_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_bits_to_f32.restype = ctypes.c_float
            lib.oracle_quantize_int4.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_int64,
                                                 ctypes.c_int32, ctypes.POINTER(ctypes.c_int8),
                                                 ctypes.POINTER(ctypes.c_uint16)]
            lib.oracle_quantize_int4.restype = None
            lib.oracle_quantize_int4_channels.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_int32,
                                                          ctypes.c_int32, ctypes.POINTER(ctypes.c_int8),
                                                          ctypes.POINTER(ctypes.c_uint16)]
            lib.oracle_quantize_int4_channels.restype = None
            lib.oracle_quantize_fp8.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_int64,
                                                ctypes.c_int32, ctypes.POINTER(ctypes.c_uint8),
                                                ctypes.POINTER(ctypes.c_uint16)]
            lib.oracle_quantize_fp8.restype = None
            lib.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_e4m3.restype = ctypes.c_uint8
            lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_f64.restype = ctypes.c_double
            lib.oracle_num_cpus.argtypes = []
            lib.oracle_num_cpus.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_cpus() -> int:
    return int(_load().oracle_num_cpus())


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def decode(q, k, v, lens, scale: float, nthreads: int = 0, window: int = 0) -> np.ndarray:
    """Attention of each sequence's new token(s) over its cache, from the definition.

    q: [B, H, d] (one new token per sequence) or [B, T, H, d] (T new tokens);
    k, v: dense [B, S_max, K, d]; lens: [B], counting the new tokens. Query i of
    sequence b sits at position lens[b] - T + i and attends positions up to its
    own (causal among the new tokens), the last ``window`` of them when window > 0.
    Head h reads KV head h // (H/K). Inputs are converted to fp64 exactly
    (bf16/fp16/fp32 values are all representable). Returns fp64 shaped like q.
    """
    q = np.ascontiguousarray(np.asarray(q, dtype=np.float64))
    k = np.ascontiguousarray(np.asarray(k, dtype=np.float64))
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
    lens = np.ascontiguousarray(np.asarray(lens, dtype=np.int32))
    single = q.ndim == 3
    q4 = q[:, None] if single else q
    B, T, H, d = q4.shape
    q4 = np.ascontiguousarray(q4)
    if k.ndim != 4 or k.shape[0] != B or k.shape[3] != d or v.shape != k.shape:
        raise ValueError("k/v must be [B, S_max, K, d] matching q")
    S_max, K = k.shape[1], k.shape[2]
    out = np.empty((B, T, H, d), dtype=np.float64)
    rc = _load().oracle_gqa_decode(_ptr(q4, ctypes.c_double), _ptr(k, ctypes.c_double),
                                   _ptr(v, ctypes.c_double), _ptr(lens, ctypes.c_int32),
                                   B, T, H, K, d, S_max, int(window), float(scale),
                                   _ptr(out, ctypes.c_double), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_gqa_decode failed with {rc}")
    return out[:, 0] if single else out


def gather_dense(pool, block_table, lens, stride_block: int, stride_head: int,
                 stride_token: int, num_kv_heads: int, head_dim: int,
                 batch_index=None) -> np.ndarray:
    """Dense [B, S_max, K, d] view of sequences held in a paged pool.

    ``pool`` is the flat element array of the cache; token t of sequence b, head g,
    element i sits at ``table[b, t // 16] * stride_block + g * stride_head +
    (t % 16) * stride_token + i``. Returns the pool's dtype (no arithmetic)."""
    flat = np.asarray(pool).reshape(-1)
    table = np.asarray(block_table)
    lens = np.asarray(lens).reshape(-1)
    rows = range(len(lens)) if batch_index is None else batch_index
    rows = list(rows)
    S_max = int(max([int(lens[b]) for b in rows] + [0]))
    K, d = num_kv_heads, head_dim
    out = np.zeros((len(rows), S_max, K, d), dtype=flat.dtype)
    i = np.arange(d)
    for n, b in enumerate(rows):
        L = int(lens[b])
        if L == 0:
            continue
        t = np.arange(L)
        phys = table[b, t // BLOCK_SIZE].astype(np.int64)
        base = (phys * stride_block + (t % BLOCK_SIZE) * stride_token)        # [L]
        idx = base[:, None, None] + (np.arange(K) * stride_head)[None, :, None] + i[None, None, :]
        out[n, :L] = flat[idx]
    return out


def gather_scales(scale_pool, block_table, lens, num_kv_heads: int, batch_index=None):
    """Dense [B, S_max, K] view of per-(token, kv-head) scales held as [NB, K, 16]."""
    sp = np.asarray(scale_pool)
    table = np.asarray(block_table)
    lens = np.asarray(lens).reshape(-1)
    rows = list(range(len(lens)) if batch_index is None else batch_index)
    S_max = int(max([int(lens[b]) for b in rows] + [0]))
    out = np.zeros((len(rows), S_max, num_kv_heads), dtype=sp.dtype)
    for n, b in enumerate(rows):
        L = int(lens[b])
        t = np.arange(L)
        phys = table[b, t // BLOCK_SIZE].astype(np.int64)
        out[n, :L] = sp[phys, :, t % BLOCK_SIZE]
    return out


def append(pool, new, block_table, positions, stride_block: int, stride_head: int,
           stride_token: int):
    """Write new[b, g, :] into slot positions[b] % 16 of block table[b, positions[b] // 16].

    ``pool``: flat element array (modified in place, any dtype); ``new``: [B, K, d]
    of the pool's dtype. Returns the pool."""
    flat = np.asarray(pool).reshape(-1)
    new = np.asarray(new)
    B, K, d = new.shape
    for b in range(B):
        pos = int(positions[b])
        phys = int(block_table[b, pos // BLOCK_SIZE])
        for g in range(K):
            off = phys * stride_block + g * stride_head + (pos % BLOCK_SIZE) * stride_token
            flat[off:off + d] = new[b, g]
    return pool


def append_scales(scale_pool, new_scales, block_table, positions):
    """Scale counterpart of ``append`` for a [NB, K, 16] scale array."""
    sp = np.asarray(scale_pool)
    for b in range(new_scales.shape[0]):
        pos = int(positions[b])
        phys = int(block_table[b, pos // BLOCK_SIZE])
        sp[phys, :, pos % BLOCK_SIZE] = new_scales[b]
    return scale_pool


def quantize_int8(x) -> tuple[np.ndarray, np.ndarray]:
    """Rows of x (last axis = d, converted to fp32) -> (int8 codes, fp16 scale bits as uint16)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    d = x.shape[-1]
    rows = x.size // d if d else 0
    codes = np.empty(x.shape, dtype=np.int8)
    scales = np.empty(x.shape[:-1], dtype=np.uint16)
    _load().oracle_quantize_int8(_ptr(x, ctypes.c_float), rows, d,
                                 _ptr(codes, ctypes.c_int8), _ptr(scales, ctypes.c_uint16))
    return codes, scales


def quantize_int4(x) -> tuple[np.ndarray, np.ndarray]:
    """Rows of x -> (codes in [-7, 7] as int8, one per element; fp16 scale bits as uint16)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    d = x.shape[-1]
    rows = x.size // d if d else 0
    codes = np.empty(x.shape, dtype=np.int8)
    scales = np.empty(x.shape[:-1], dtype=np.uint16)
    _load().oracle_quantize_int4(_ptr(x, ctypes.c_float), rows, d,
                                 _ptr(codes, ctypes.c_int8), _ptr(scales, ctypes.c_uint16))
    return codes, scales


def quantize_int4_channels(x) -> tuple[np.ndarray, np.ndarray]:
    """One block's K values [n, d] (n <= 16 present tokens) -> (codes [n, d] in
    [-7, 7] as int8, [d] fp16 scale bits as uint16): one scale per channel over
    the block's tokens (the KIVI-style K of section 15.5; rule in gqa_oracle.c)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    n, d = x.shape
    codes = np.zeros((n, d), dtype=np.int8)
    scales = np.zeros(d, dtype=np.uint16)
    if n:
        _load().oracle_quantize_int4_channels(_ptr(x, ctypes.c_float), n, d,
                                              _ptr(codes, ctypes.c_int8), _ptr(scales, ctypes.c_uint16))
    return codes, scales


def gather_channel_scales(scale_pool, block_table, lens, batch_index=None):
    """Dense [B, S_max, K, d] view of per-(block, kv-head, channel) scales held as
    [NB, K, d]: every token of a block carries its block's channel scales."""
    sp = np.asarray(scale_pool)
    table = np.asarray(block_table)
    lens = np.asarray(lens).reshape(-1)
    rows = list(range(len(lens)) if batch_index is None else batch_index)
    S_max = int(max([int(lens[b]) for b in rows] + [0]))
    out = np.zeros((len(rows), S_max) + sp.shape[1:], dtype=sp.dtype)
    for n, b in enumerate(rows):
        L = int(lens[b])
        t = np.arange(L)
        out[n, :L] = sp[table[b, t // BLOCK_SIZE].astype(np.int64)]
    return out


def append_int4_channels(pool_bytes, scale_pool, residual, k_rows, block_table, positions,
                         counts, stride_block: int, stride_head: int, stride_token: int):
    """The KIVI-style K append: sequence b adds counts[b] tokens (rows of
    k_rows[b], each [K, d] fp32) at positions[b] ..; every block they touch is
    re-quantised per channel over all the tokens it then holds, the older ones
    taken from residual[b] (fp32 [K, 16, d], the unquantised K of the block
    that was filling), and the rows of a block left unfinished are kept in
    residual[b]. pool_bytes: flat uint8 K pool (strides in 4-bit elements);
    scale_pool: [NB, K, d] uint16 fp16 bits. All modified in place."""
    flat = np.asarray(pool_bytes).reshape(-1)
    sp = np.asarray(scale_pool)
    res = np.asarray(residual)
    for b in range(len(counts)):
        n, p0 = int(counts[b]), int(positions[b])
        if n == 0:
            continue
        rows = np.asarray(k_rows[b], dtype=np.float32)
        K = rows.shape[1]
        for jb in range(p0 // BLOCK_SIZE, (p0 + n - 1) // BLOCK_SIZE + 1):
            first = jb * BLOCK_SIZE
            tend = min(BLOCK_SIZE, p0 + n - first)
            phys = int(block_table[b, jb])
            for g in range(K):
                x = np.stack([res[b, g, t] if first + t < p0 else rows[first + t - p0, g]
                              for t in range(tend)])
                codes, sbits = quantize_int4_channels(x)
                packed = pack_int4(codes)
                for t in range(tend):
                    off = (phys * stride_block + g * stride_head + t * stride_token) // 2
                    flat[off:off + packed.shape[1]] = packed[t]
                sp[phys, g] = sbits
                if tend < BLOCK_SIZE:
                    res[b, g, :tend] = x
    return pool_bytes


def pack_int4(codes) -> np.ndarray:
    """[..., d] codes in [-8, 7] -> [..., d/2] bytes: element 2j in the low nibble,
    2j+1 in the high nibble, each as a two's-complement nibble."""
    c = np.asarray(codes).astype(np.int16)
    lo = c[..., 0::2] & 0xF
    hi = c[..., 1::2] & 0xF
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_int4(packed) -> np.ndarray:
    """Inverse of pack_int4: [..., d/2] bytes -> [..., d] int8 codes."""
    b = np.asarray(packed, dtype=np.uint8).astype(np.int16)
    nib = np.stack([b & 0xF, b >> 4], axis=-1).reshape(*b.shape[:-1], 2 * b.shape[-1])
    return np.where(nib >= 8, nib - 16, nib).astype(np.int8)


def quantize_fp8(x) -> tuple[np.ndarray, np.ndarray]:
    """Rows of x -> (e4m3 codes as uint8, fp16 scale bits as uint16)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    d = x.shape[-1]
    rows = x.size // d if d else 0
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty(x.shape[:-1], dtype=np.uint16)
    _load().oracle_quantize_fp8(_ptr(x, ctypes.c_float), rows, d,
                                _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint16))
    return codes, scales


def e4m3_to_f64(codes) -> np.ndarray:
    """Exact values of e4m3 codes (uint8) as fp64 (NaN for the NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([_load().oracle_e4m3_to_f64(i) for i in range(256)], dtype=np.float64)
    return table[c]


def f32_to_e4m3(x) -> np.ndarray:
    """Nearest-even e4m3 codes of fp32 values, saturated to +-448."""
    a = np.asarray(x, dtype=np.float32)
    lib = _load()
    return np.asarray([lib.oracle_f32_to_e4m3(float(v)) for v in a.reshape(-1)],
                      dtype=np.uint8).reshape(a.shape)


def dequantize_fp8(codes, scale_values) -> np.ndarray:
    """e4m3(code) * scale in fp64 (exact)."""
    return e4m3_to_f64(codes) * np.asarray(scale_values, dtype=np.float64)[..., None]


def f16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of fp16 bit patterns (uint16) as fp64."""
    b = np.asarray(bits, dtype=np.uint16)
    lib = _load()
    flat = [lib.oracle_f16_bits_to_f32(int(v)) for v in b.reshape(-1)]
    return np.asarray(flat, dtype=np.float64).reshape(b.shape)


def f32_to_f16_bits(x) -> np.ndarray:
    """Round fp32 values to fp16 (nearest-even); returns the bit patterns."""
    a = np.asarray(x, dtype=np.float32)
    lib = _load()
    flat = [lib.oracle_f32_to_f16_bits(float(v)) for v in a.reshape(-1)]
    return np.asarray(flat, dtype=np.uint16).reshape(a.shape)


def dequantize_int4(packed, scale_values) -> np.ndarray:
    """Packed int4 rows [..., d/2] -> code * scale in fp64 (exact)."""
    return dequantize_int8(unpack_int4(packed), scale_values)


def dequantize_int8(codes, scale_values) -> np.ndarray:
    """codes[..., i] * scale[...] in fp64 (exact: both factors are short)."""
    c = np.asarray(codes, dtype=np.float64)
    s = np.asarray(scale_values, dtype=np.float64)
    return c * s[..., None]


def f16_bits_value(bits) -> np.ndarray:
    """fp16 bit patterns as fp64 values (numpy's binary16 decode; exact)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def quantised_sequence(rows, cache_dtype: str, per_channel: bool = False):
    """Codes, scales and exact values a code cache holds for the rows [L, K, d]
    of one sequence written at positions 0 .. L-1.

    cache_dtype "i8" / "fp8" / "i4": one fp16 scale per (token, kv-head), the
    rules of ``quantize_int8`` / ``quantize_fp8`` / ``quantize_int4``.
    ``per_channel`` (the K of the KIVI-style cache, "i4kc"): each 16-token
    block of each kv-head is quantised per channel over the tokens it holds
    (``quantize_int4_channels``); the last block may be partial.
    Returns (values fp64 [L, K, d], codes [L, K, d] (int8, or uint8 e4m3
    codes), scale bits uint16 ([L, K], or [ceil(L/16), K, d] per channel))."""
    x = np.ascontiguousarray(np.asarray(rows, dtype=np.float32))
    L, K, d = x.shape
    if per_channel:
        nblk = -(-L // BLOCK_SIZE)
        codes = np.zeros((L, K, d), dtype=np.int8)
        sbits = np.zeros((nblk, K, d), dtype=np.uint16)
        for jb in range(nblk):
            t0, t1 = jb * BLOCK_SIZE, min(L, (jb + 1) * BLOCK_SIZE)
            for g in range(K):
                c, s = quantize_int4_channels(x[t0:t1, g])
                codes[t0:t1, g] = c
                sbits[jb, g] = s
        per_tok = np.repeat(f16_bits_value(sbits), BLOCK_SIZE, axis=0)[:L]      # [L, K, d]
        return codes.astype(np.float64) * per_tok, codes, sbits
    if cache_dtype == "i8":
        codes, sbits = quantize_int8(x)
        return dequantize_int8(codes, f16_bits_value(sbits)), codes, sbits
    if cache_dtype == "fp8":
        codes, sbits = quantize_fp8(x)
        return dequantize_fp8(codes, f16_bits_value(sbits)), codes, sbits
    if cache_dtype in ("i4", "i4kc"):
        codes, sbits = quantize_int4(x)
        return dequantize_int8(codes, f16_bits_value(sbits)), codes, sbits
    raise ValueError(f"not a code cache: {cache_dtype!r}")


def kv_cache_elements(layers: int, kv_heads: int, head_dim: int, seq_len: int,
                      batch: int) -> int:
    """Elements of K and V cached for ``batch`` sequences of ``seq_len`` tokens:
    2 * layers * kv_heads * head_dim * seq_len * batch."""
    return 2 * layers * kv_heads * head_dim * seq_len * batch


def blocks_for_tokens(n_tokens: int) -> int:
    """Physical 16-token blocks a sequence of n_tokens occupies (last one may be partial)."""
    return -(-int(n_tokens) // BLOCK_SIZE)
