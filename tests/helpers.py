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


def max_abs_err(gpu_out: torch.Tensor, ref: np.ndarray, rows=None) -> float:
    got = gpu_out.detach().float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[list(rows)]
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), "non-finite output"
    return float(np.abs(got - ref).max()) if got.size else 0.0
