"""Test helpers: run the CPU oracle on a generated decode case and compare.

The oracle sees exactly the values the GPU reads: the pool is copied to the
host as fp32 (exact for bf16/f16/fp32) or int8 codes with fp16 scales, and the
oracle gathers the dense sequences through the block table itself."""
from __future__ import annotations

import numpy as np
import torch

TOL = 2e-3   # max-abs error bound for fp32 output (bf16/f16 inputs, fp32 accumulation)


def _host(t: torch.Tensor) -> np.ndarray:
    t = t.detach()
    if t.dtype in (torch.int8, torch.uint8):
        return t.cpu().numpy()
    if t.dtype == torch.float8_e4m3fn:
        return t.cpu().view(torch.uint8).numpy()       # raw codes; the oracle decodes them
    return t.float().cpu().numpy()


def oracle_for_case(case, rows=None, nthreads: int = 0, host_pools=None, window: int = 0) -> np.ndarray:
    """fp64 oracle output [len(rows), (T,) H, d] for the sequences in ``rows``."""
    import oracle
    lens = case.context_lens.cpu().numpy()
    table = case.block_table.cpu().numpy()
    rows = list(range(case.batch)) if rows is None else list(rows)
    kp, vp = host_pools if host_pools is not None else (_host(case.k_cache), _host(case.v_cache))
    K, d = case.num_kv_heads, case.head_dim
    if case.cache_dtype in ("i4", "i4kc"):
        # bytes: element strides halve, a row is d/2 bytes
        kb = oracle.gather_dense(kp, table, lens, case.stride_block // 2, case.stride_head // 2,
                                 case.stride_token // 2, K, d // 2, rows)
        vb = oracle.gather_dense(vp, table, lens, case.stride_block // 2, case.stride_head // 2,
                                 case.stride_token // 2, K, d // 2, rows)
        vs = oracle.gather_scales(case.v_scale.float().cpu().numpy(), table, lens, K, rows)
        if case.cache_dtype == "i4kc":     # K: code * its block's channel scale
            kcs = oracle.gather_channel_scales(case.k_scale.float().cpu().numpy().astype(np.float64),
                                               table, lens, rows)
            kd = oracle.unpack_int4(kb).astype(np.float64) * kcs
        else:
            ks = oracle.gather_scales(case.k_scale.float().cpu().numpy(), table, lens, K, rows)
            kd = oracle.dequantize_int4(kb, ks)
        q = case.q.detach().float().cpu().numpy().astype(np.float64)[rows]
        return oracle.decode(q, kd, oracle.dequantize_int4(vb, vs),
                             lens[rows], case.scale, nthreads, window=window)
    kd = oracle.gather_dense(kp, table, lens, case.stride_block, case.stride_head,
                             case.stride_token, K, d, rows).astype(np.float64)
    vd = oracle.gather_dense(vp, table, lens, case.stride_block, case.stride_head,
                             case.stride_token, K, d, rows).astype(np.float64)
    if case.cache_dtype in ("i8", "fp8"):
        ks = oracle.gather_scales(case.k_scale.float().cpu().numpy(), table, lens, K, rows)
        vs = oracle.gather_scales(case.v_scale.float().cpu().numpy(), table, lens, K, rows)
        if case.cache_dtype == "i8":
            kd = oracle.dequantize_int8(kd, ks)
            vd = oracle.dequantize_int8(vd, vs)
        else:
            kd = oracle.dequantize_fp8(oracle.gather_dense(kp, table, lens, case.stride_block,
                                       case.stride_head, case.stride_token, K, d, rows), ks)
            vd = oracle.dequantize_fp8(oracle.gather_dense(vp, table, lens, case.stride_block,
                                       case.stride_head, case.stride_token, K, d, rows), vs)
    q = case.q.detach().float().cpu().numpy().astype(np.float64)[rows]
    return oracle.decode(q, kd, vd, lens[rows], case.scale, nthreads, window=window)


def source_rows(case, b):
    """Host copies of sequence b's unquantised K and V rows ([L, K, d] fp32) of a
    case drawn with source="normal"."""
    st = case.src_start.cpu()
    lo, hi = int(st[b]), int(st[b + 1])
    return case.k_src[lo:hi].cpu().numpy(), case.v_src[lo:hi].cpu().numpy()


def fill_from_source(gq, case):
    """Quantise a source="normal" case's rows into its device cache with the
    library's varlen append (every sequence written from position 0)."""
    lens = case.context_lens
    zeros = torch.zeros_like(lens)
    gq.kv_append_varlen(gq.cache_from_case(case), case.k_src, case.v_src, case.src_start,
                        int(lens.max().item()) if lens.numel() else 0, case.block_table, zeros)


def oracle_for_source_case(case, rows, nthreads: int = 0, window: int = 0) -> np.ndarray:
    """fp64 oracle output for the sequences in ``rows`` of a case whose cache is
    filled from unquantised rows: the oracle quantises those rows itself
    (oracle.quantised_sequence) and never reads the device cache."""
    import oracle
    lens = case.context_lens.cpu().numpy()
    rows = list(rows)
    S = max([int(lens[b]) for b in rows] + [0])
    K, d = case.num_kv_heads, case.head_dim
    kd = np.zeros((len(rows), S, K, d))
    vd = np.zeros((len(rows), S, K, d))
    for n, b in enumerate(rows):
        ks, vs = source_rows(case, b)
        L = ks.shape[0]
        kd[n, :L] = oracle.quantised_sequence(ks, case.cache_dtype, case.cache_dtype == "i4kc")[0]
        vd[n, :L] = oracle.quantised_sequence(vs, case.cache_dtype)[0]
    q = case.q.detach().float().cpu().numpy().astype(np.float64)[rows]
    return oracle.decode(q, kd, vd, lens[rows], case.scale, nthreads, window=window)


def cache_codes_of(case, b, which: str):
    """Codes ([L, K, d]) and scale bits the device cache holds for sequence b:
    per token [L, K], or for the KIVI-style K per block [nblk, K, d]."""
    import oracle
    lens = case.context_lens.cpu().numpy()
    L = int(lens[b])
    nblk = -(-L // 16)
    ids = case.block_table[b, :nblk].long()
    pool = (case.k_cache if which == "k" else case.v_cache).index_select(0, ids)
    sc = (case.k_scale if which == "k" else case.v_scale).index_select(0, ids)
    pool = pool.view(torch.uint8) if pool.dtype == torch.float8_e4m3fn else pool
    pool = pool.cpu().numpy()                           # [nblk, K, 16, row]
    sbits = sc.cpu().view(torch.int16).numpy().view(np.uint16)
    codes = pool.transpose(0, 2, 1, 3).reshape(nblk * 16, pool.shape[1], pool.shape[3])[:L]
    if case.cache_dtype in ("i4", "i4kc"):
        codes = oracle.unpack_int4(codes)
    if which == "k" and case.cache_dtype == "i4kc":
        return codes, sbits                             # [nblk, K, d]
    return codes, sbits.transpose(0, 2, 1).reshape(nblk * 16, -1)[:L]


def max_abs_err(gpu_out: torch.Tensor, ref: np.ndarray, rows=None) -> float:
    got = gpu_out.detach().float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[list(rows)]
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), "non-finite output"
    return float(np.abs(got - ref).max()) if got.size else 0.0
