"""GQA decode on the GPU against the fp64 CPU oracle, through the C ABI.

Bar: max-abs error <= 2e-3 on fp32 output (bf16/f16/int8 inputs, fp32
accumulation; the oracle reads the same rounded or dequantised values).
Paging is exact: a shuffled block table gives the same bytes as the identity
table when the split layout is the same."""
import math

import numpy as np
import pytest
import torch

import gqa_inputs as gi
from helpers import (TOL, cache_codes_of, fill_from_source, max_abs_err, oracle_for_case,
                     oracle_for_source_case, source_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    from gqa_decode_attention_kv_gb300 import build
    build.build()
    import gqa_decode_attention_kv_gb300 as m
    return m


def _run(gq, case, **kw):
    out = gq.gqa_decode(gq.cache_from_case(case), case.q, case.block_table, case.context_lens,
                        case.scale, **kw)
    torch.cuda.synchronize()
    return out


KERNELS = [1, 2]      # tensor-core, CUDA-core


# --------------------------------------------------------------------------- small, full compare


def test_tiny_fp32_contiguous_workload(gq):
    case = gi.case_for(gi.WORKLOADS["tiny_f32_contiguous"], seed=0, device="cuda")
    out = _run(gq, case)
    assert max_abs_err(out, oracle_for_case(case)) <= TOL


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype,d,H,K", [
    ("bf16", 128, 32, 8), ("bf16", 128, 64, 8), ("bf16", 64, 16, 4), ("f16", 128, 32, 8),
    ("bf16", 128, 8, 8), ("bf16", 128, 16, 8), ("f16", 64, 8, 1),
])
def test_ragged_multi_tile(gq, kernel, dtype, d, H, K):
    _ragged(gq, kernel, dtype, d, H, K)


@pytest.mark.parametrize("dtype,d,H,K,kernel", [
    ("bf16", 128, 64, 4, 1), ("bf16", 128, 48, 4, 1), ("bf16", 128, 64, 2, 1),
    ("bf16", 128, 64, 1, 1), ("f16", 64, 32, 1, 1), ("f32", 64, 64, 1, 2), ("f32", 128, 16, 1, 2),
])
@pytest.mark.parametrize("layout", [1, 2])
def test_groups_larger_than_one_warp(gq, dtype, d, H, K, kernel, layout):
    """G = 16, 12, 32, 64: every 8 heads stream the tiles on their own (layout 1),
    or the CTA's warps split the heads and share one ring (layout 2)."""
    _ragged(gq, kernel, dtype, d, H, K, row_layout=layout)


def _ragged(gq, kernel, dtype, d, H, K, **kw):
    lens = [1, 15, 16, 17, 33, 200, 511, 0, 1000]
    case = gi.make_case(len(lens), H, K, d, lens, dtype, seed=21, device="cuda")
    ref = oracle_for_case(case)
    for mw in (0, 1, 5, 37):          # 0 = fill the GPU; 1 = one warp does everything
        out = _run(gq, case, kernel=kernel, max_warps=mw, min_blocks_per_warp=1, **kw)
        err = max_abs_err(out, ref)
        assert err <= TOL, (mw, err)


@pytest.mark.parametrize("layout", [0, 1, 2])
def test_int8_wide_group(gq, layout):
    lens = [1, 16, 17, 300, 2047, 0, 64]
    case = gi.make_case(len(lens), 64, 2, 128, lens, "i8", q_dtype="bf16", seed=35, device="cuda")
    ref = oracle_for_case(case)
    for mw in (0, 3):
        out = _run(gq, case, max_warps=mw, min_blocks_per_warp=1, row_layout=layout)
        assert max_abs_err(out, ref) <= TOL


@pytest.mark.parametrize("dtype", ["i8", "fp8", "bf16"])
def test_head_dim_64_groups_above_8_on_the_cuda_core_kernel(gq, dtype):
    """G = 16 with head_dim 64: the CUDA-core kernel serves it as 8-row unit streams."""
    lens = [1, 17, 300, 0, 64]
    case = gi.make_case(len(lens), 32, 2, 64, lens, dtype, seed=36, device="cuda")
    ref = oracle_for_case(case)
    for mw in (0, 3):
        out = _run(gq, case, kernel=2, max_warps=mw, min_blocks_per_warp=1)
        assert max_abs_err(out, ref) <= TOL


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("d", [128, 64])
def test_int8_cache(gq, kernel, d):
    if kernel == 1 and d == 64:
        pytest.skip("the tensor-core int8 kernel covers head_dim 128")
    lens = [1, 16, 17, 300, 2047, 0, 64]
    case = gi.make_case(len(lens), 64, 8, d, lens, "i8", q_dtype="bf16", seed=22, device="cuda")
    ref = oracle_for_case(case)
    for mw in (0, 3):
        out = _run(gq, case, kernel=kernel, max_warps=mw, min_blocks_per_warp=1)
        assert max_abs_err(out, ref) <= TOL


@pytest.mark.parametrize("kernel,d", [(1, 128), (2, 128), (2, 64)])
def test_fp8_cache(gq, kernel, d):
    lens = [1, 16, 17, 300, 2047, 0, 64]
    case = gi.make_case(len(lens), 64, 8, d, lens, "fp8", q_dtype="bf16", seed=36, device="cuda")
    ref = oracle_for_case(case)
    for mw in (0, 3):
        out = _run(gq, case, kernel=kernel, max_warps=mw, min_blocks_per_warp=1)
        assert max_abs_err(out, ref) <= TOL


def test_fp8_wide_group_f16_query(gq):
    lens = [33, 700, 5]
    case = gi.make_case(3, 64, 4, 128, lens, "fp8", q_dtype="f16", seed=37, device="cuda")
    assert max_abs_err(_run(gq, case), oracle_for_case(case)) <= TOL


@pytest.mark.parametrize("kernel,d", [(1, 128), (2, 128), (2, 64)])
def test_int4_cache(gq, kernel, d):
    lens = [1, 16, 17, 300, 2047, 0, 64]
    case = gi.make_case(len(lens), 64, 8, d, lens, "i4", q_dtype="bf16", seed=38, device="cuda")
    ref = oracle_for_case(case)
    for mw in (0, 3):
        out = _run(gq, case, kernel=kernel, max_warps=mw, min_blocks_per_warp=1)
        assert max_abs_err(out, ref) <= TOL


@pytest.mark.parametrize("layout", [0, 1, 2])
def test_int4_wide_group_f16_query(gq, layout):
    lens = [33, 700, 5, 0]
    case = gi.make_case(4, 64, 4, 128, lens, "i4", q_dtype="f16", seed=39, device="cuda")
    assert max_abs_err(_run(gq, case, row_layout=layout), oracle_for_case(case)) <= TOL


# bound per cache: the f16 low part of p s_v resolves 2^-24 absolute, which the
# small FP8 scales (~0.008) turn into ~1e-4 of output; int8 and INT4 scales leave
# the fp32 accumulation (~1e-5) as the floor
_SAME_ROW_BOUND = {"i8": 1e-4, "i4": 1e-4, "i4kc": 1e-4, "fp8": TOL / 4}


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["i8", "fp8", "i4", "i4kc"])
def test_one_value_row_everywhere_comes_back_exactly(gq, dtype, kernel):
    """Every cached token holds the same V codes and scale: whatever the scores,
    the output is that row. The tensor-core kernel feeds the weights p s_v to
    P.V as an f16 high plus low part, so what remains is the low part's
    resolution and the fp32 accumulation; the high part alone would miss by
    about 2^-12 |v| (5e-4 to 8e-4 at these values)."""
    lens = [2, 3, 9, 17, 300]
    case = gi.make_case(len(lens), 32, 8, 128, lens, dtype, q_dtype="bf16", seed=41, device="cuda")
    case.q = (case.q.float() * 3).to(torch.bfloat16)          # a few tokens carry the weight
    blk = int(case.block_table[0, 0])
    case.v_cache.copy_(case.v_cache[blk, 0, 0].expand_as(case.v_cache))
    case.v_scale.fill_(float(case.v_scale[blk, 0, 0]))
    ref = oracle_for_case(case)
    for mw in (0, 3):
        out = _run(gq, case, kernel=kernel, max_warps=mw, min_blocks_per_warp=1)
        assert max_abs_err(out, ref) <= _SAME_ROW_BOUND[dtype]


def test_int8_cache_with_f16_query(gq):
    lens = [40, 333]
    case = gi.make_case(2, 32, 8, 128, lens, "i8", q_dtype="f16", seed=23, device="cuda")
    assert max_abs_err(_run(gq, case), oracle_for_case(case)) <= TOL


def test_shuffled_table_matches_identity_table_bit_for_bit(gq):
    lens = [100, 257, 31]
    a = gi.make_case(3, 32, 8, 128, lens, "bf16", seed=24, device="cuda", shuffle=False)
    b = gi.make_case(3, 32, 8, 128, lens, "bf16", seed=24, device="cuda", shuffle=True)
    # same logical contents: move b's identity-layout data into its shuffled blocks
    ta, tb = a.block_table.long(), b.block_table.long()
    for t_src, t_dst in ((a.k_cache, b.k_cache), (a.v_cache, b.v_cache)):
        for s in range(3):
            nb = -(-lens[s] // 16)
            t_dst[tb[s, :nb]] = t_src[ta[s, :nb]]
    b.q = a.q
    oa = _run(gq, a, max_warps=9)
    ob = _run(gq, b, max_warps=9)
    assert torch.equal(oa.view(torch.int32), ob.view(torch.int32))


def test_split_count_does_not_change_the_answer(gq):
    case = gi.make_case(2, 32, 8, 128, [4096, 1500], "bf16", seed=25, device="cuda")
    ref = oracle_for_case(case)
    outs = [_run(gq, case, max_warps=mw, min_blocks_per_warp=1) for mw in (1, 2, 16, 100, 0)]
    for o in outs:
        assert max_abs_err(o, ref) <= TOL
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 1e-4


@pytest.mark.parametrize("lens,K,window,queries,max_warps,d", [
    ([20000], 1, 0, 1, 0, 128),              # one pair, hundreds of pieces: 32 warps per row
    ([20000], 1, 0, 1, 30, 128),             # about 45 pieces per row: 8 warps per row
    ([20000] + [1] * 63, 8, 0, 1, 0, 128),   # few pieces expected, one long row: chunks of 32
    ([20000], 1, 5000, 1, 0, 128),           # a window over the long row
    ([3000, 40], 1, 64, 4, 0, 128),          # causal new tokens under a window
    ([20000], 1, 0, 1, 0, 64),               # head_dim 64: half the lanes hold dims
    ([20000] + [1] * 63, 8, 0, 1, 0, 64),
])
def test_combine_forms_match_the_oracle(gq, lens, K, window, queries, max_warps, d):
    """Rows merged by one warp (pieces in chunks of 32), by 8 warps or by 32 warps
    sharing a CTA, each against the oracle element by element."""
    case = gi.make_case(len(lens), 8, K, d, lens, "bf16", seed=33, device="cuda", queries=queries)
    ref = oracle_for_case(case, window=window)
    out = _run(gq, case, window=window, max_warps=max_warps, min_blocks_per_warp=1)
    assert max_abs_err(out, ref) <= TOL


def test_one_token_context_returns_v(gq):
    case = gi.make_case(4, 32, 8, 128, [1, 1, 1, 1], "bf16", seed=26, device="cuda")
    out = _run(gq, case)
    table = case.block_table.long()
    v0 = case.v_cache[table[:, 0], :, 0, :].float()                 # [B, K, d]
    expect = v0.repeat_interleave(4, dim=1)                          # head h reads group h // 4
    assert torch.equal(out, expect)


def test_zero_query_averages_values(gq):
    case = gi.make_case(3, 16, 4, 128, [7, 130, 64], "bf16", seed=27, device="cuda", q_zero=True)
    ref = oracle_for_case(case)
    assert max_abs_err(_run(gq, case), ref) <= TOL


def test_empty_contexts_give_zero_rows(gq):
    case = gi.make_case(3, 16, 4, 128, [0, 50, 0], "bf16", seed=28, device="cuda")
    out = _run(gq, case)
    assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[2]) == 0
    assert max_abs_err(out, oracle_for_case(case)) <= TOL


def test_all_contexts_empty(gq):
    case = gi.make_case(2, 8, 2, 64, [0, 0], "f32", seed=29, device="cuda")
    out = _run(gq, case, out=torch.full((2, 8, 64), 7.0, device="cuda"))
    assert torch.count_nonzero(out) == 0


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_half_precision_output(gq, out_dtype):
    case = gi.make_case(3, 32, 8, 128, [1, 90, 700], "bf16", seed=30, device="cuda")
    ref = oracle_for_case(case)
    out = _run(gq, case, out_dtype=out_dtype)
    got = out.float().cpu().numpy()
    # bound: 2e-3 plus half a unit in the last place of the stored value
    ulp_bits = 8 if out_dtype == torch.bfloat16 else 11
    half_ulp = np.abs(ref) * 2.0 ** -ulp_bits
    assert np.all(np.abs(got - ref) <= TOL + half_ulp)


def test_large_scores_are_stable(gq):
    case = gi.make_case(2, 32, 8, 128, [300, 5000], "bf16", seed=31, device="cuda")
    case.q = (case.q.float() * 30).to(torch.bfloat16)       # scores of order +-300
    ref = oracle_for_case(case)
    assert max_abs_err(_run(gq, case), ref) <= TOL


def test_device_errors_are_flagged_not_trapped(gq):
    case = gi.make_case(3, 32, 8, 128, [40, 40, 40], "bf16", seed=32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    table = case.block_table.clone()
    table[1, 1] = -5
    lens = case.context_lens.clone()
    lens[2] = 10_000
    out = gq.gqa_decode(gq.cache_from_case(case), case.q, table, lens, case.scale, err=err)
    torch.cuda.synchronize()
    flags = int(err.item())
    assert flags & gq.GQA_DEVERR_BLOCK_INDEX and flags & gq.GQA_DEVERR_CONTEXT_LEN
    assert not flags & gq.GQA_DEVERR_TIMEOUT
    ref = oracle_for_case(case, rows=[0])
    assert max_abs_err(out, ref, rows=[0]) <= TOL           # healthy sequence still right


def test_append_then_decode_steps(gq, oracle_mod):
    """Several decode steps: append each new token, advance, decode. The oracle
    replays the appends into its own host copy of the pool."""
    lens0 = [14, 30, 1]
    steps = 5
    case = gi.make_case(3, 32, 8, 128, lens0, "bf16", seed=33, device="cuda", extra_tokens=steps)
    cache = gq.cache_from_case(case)
    host_k = case.k_cache.float().cpu().numpy().copy()
    host_v = case.v_cache.float().cpu().numpy().copy()
    table = case.block_table.cpu().numpy()
    lens = case.context_lens.clone()
    gen = torch.Generator(device="cuda").manual_seed(5)
    for step in range(steps):
        kn = torch.randn(case.k_new.shape, generator=gen, device="cuda").to(torch.bfloat16)
        vn = torch.randn(case.k_new.shape, generator=gen, device="cuda").to(torch.bfloat16)
        gq.kv_append(cache, kn, vn, case.block_table, lens)
        pos = [n + step for n in lens0]
        oracle_mod.append(host_k, kn.float().cpu().numpy(), table, pos, case.stride_block,
                          case.stride_head, case.stride_token)
        oracle_mod.append(host_v, vn.float().cpu().numpy(), table, pos, case.stride_block,
                          case.stride_head, case.stride_token)
        lens += 1
        case.context_lens = lens
        out = _run(gq, case)
        ref = oracle_for_case(case, host_pools=(host_k, host_v))
        assert max_abs_err(out, ref) <= TOL, step


def test_int8_append_then_decode(gq, oracle_mod):
    """Quantise on append (GPU) and compare the decode with the oracle, which
    quantises the same new rows with its own rule."""
    lens0 = [20, 47]
    case = gi.make_case(2, 64, 8, 128, lens0, "i8", q_dtype="bf16", seed=34, device="cuda",
                        extra_tokens=1, new_dtype="bf16")
    cache = gq.cache_from_case(case)
    kpool = case.k_cache.cpu().numpy().copy()
    vpool = case.v_cache.cpu().numpy().copy()
    ksc = case.k_scale.cpu().view(torch.int16).numpy().view(np.uint16).copy()
    vsc = case.v_scale.cpu().view(torch.int16).numpy().view(np.uint16).copy()
    gq.kv_append(cache, case.k_new, case.v_new, case.block_table, case.context_lens)
    table = case.block_table.cpu().numpy()
    for new, pool, sc in ((case.k_new, kpool, ksc), (case.v_new, vpool, vsc)):
        codes, sbits = oracle_mod.quantize_int8(new.float().cpu().numpy())
        oracle_mod.append(pool.reshape(-1), codes, table, lens0, case.stride_block,
                          case.stride_head, case.stride_token)
        oracle_mod.append_scales(sc, sbits, table, lens0)
    case.context_lens = case.context_lens + 1
    out = _run(gq, case)
    # oracle on its own quantised pool
    case_o = gi.DecodeCase(**{**case.__dict__})
    case_o.k_cache = torch.from_numpy(kpool)
    case_o.v_cache = torch.from_numpy(vpool)
    case_o.k_scale = torch.from_numpy(ksc.view(np.float16))
    case_o.v_scale = torch.from_numpy(vsc.view(np.float16))
    assert max_abs_err(out, oracle_for_case(case_o)) <= TOL


# --------------------------------------------------------------------------- full-size workloads


def _sampled(gq, wl, rows, seed=0, **kw):
    """Decode a full-size workload with the default launch, then check the
    sampled sequences (every head) against the oracle. Code caches drawn as
    N(0, 1) rows are quantised into the cache by the library's append; the
    oracle quantises the sampled rows itself, and the cache must hold exactly
    its codes and scales for them."""
    case = gi.case_for(wl, seed=seed, device="cuda")
    if case.k_src is not None:
        fill_from_source(gq, case)
        torch.cuda.synchronize()
        _codes_match_the_oracle(case, rows)
        out = _run(gq, case, window=wl.window, **kw)
        ref = oracle_for_source_case(case, rows, window=wl.window)
        return max_abs_err(out, ref, rows=rows)
    out = _run(gq, case, window=wl.window, **kw)
    ref = oracle_for_case(case, rows=rows, host_pools=_host_pools(case), window=wl.window)
    return max_abs_err(out, ref, rows=rows)


def _codes_match_the_oracle(case, rows):
    import oracle
    for b in rows:
        for which, src in zip("kv", source_rows(case, b)):
            kc = which == "k" and case.cache_dtype == "i4kc"
            _, codes, sbits = oracle.quantised_sequence(src, case.cache_dtype, kc)
            got_codes, got_bits = cache_codes_of(case, b, which)
            if case.cache_dtype == "fp8":
                got_codes = got_codes.view(np.uint8)
            assert np.array_equal(got_codes, codes), (b, which)
            assert np.array_equal(got_bits, sbits), (b, which)


def _host_pools(case):
    def host(t):
        if t.dtype in (torch.int8, torch.uint8):
            return t.cpu().numpy()
        if t.dtype == torch.float8_e4m3fn:
            return t.cpu().view(torch.uint8).numpy()
        return t.float().cpu().numpy()
    return host(case.k_cache), host(case.v_cache)


@pytest.mark.parametrize("name,rows", [
    ("llama3_8b_bf16_b64_s4096", [0, 17, 63]),
    ("llama70b_bf16_b32_ragged", [0, 5, 31]),
    ("long_ctx_bf16_b1_s131072", [0]),
    ("int8kv_b128_ragged", [0, 64, 127]),
    ("fp8kv_b128_ragged", [0, 77, 127]),
    ("int4kv_b128_ragged", [0, 100, 127]),
    ("int4kc_b128_ragged", [0, 50, 127]),
    ("spec_verify_bf16_b64_s4096_t4", [0, 40, 63]),
    ("mistral7b_swa_bf16_b64_s16384_w4096", [0, 63]),
])
def test_full_size_workloads_sampled(gq, name, rows):
    assert _sampled(gq, gi.WORKLOADS[name], rows) <= TOL


def test_full_size_long_context_b4_sampled(gq):
    assert _sampled(gq, gi.WORKLOADS["long_ctx_bf16_b4_s131072"], [3]) <= TOL


@pytest.mark.parametrize("kv_heads", [64, 32, 16, 8, 1])
def test_kv_head_sweep_sampled(gq, kv_heads):
    """H=64 with K from MHA (G=1) to MQA (G=64) on the 70B-shaped ragged lengths
    (first 6 sequences, so the MHA point stays a few GB)."""
    import dataclasses
    wl = dataclasses.replace(gi.kv_sweep_workload(kv_heads), batch=6)
    assert _sampled(gq, wl, [1, 5]) <= TOL


def test_step_replays_from_a_cuda_graph(gq):
    """append + decode captured in a CUDA graph (the kernels keep their
    programmatic-launch edges) replays to the eager result bit for bit."""
    lens = [100, 4000, 17, 1]
    case = gi.make_case(len(lens), 32, 8, 128, lens, "bf16", seed=41, device="cuda", extra_tokens=1)
    cache = gq.cache_from_case(case)
    pos = case.context_lens.clone()
    after = case.context_lens + 1
    out = torch.empty(case.q.shape, dtype=torch.float32, device="cuda")
    ws = gq.workspace_for(len(lens), 32, 8, 128, torch.device("cuda"), 1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step():
        gq.kv_append(cache, case.k_new, case.v_new, case.block_table, pos, err=err)
        gq.gqa_decode(cache, case.q, case.block_table, after, case.scale, out=out, workspace=ws, err=err)

    step()
    torch.cuda.synchronize()
    eager = out.clone()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            for _ in range(3):
                step()
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out, eager)


def test_alternating_caches_keep_their_own_tensor_maps(gq):
    """The library remembers encoded tensor maps by the cache's address, shape and
    strides. Decoding two caches of the same shape in turn, and a third cache
    with more blocks, must each give exactly what a first call on it gives."""
    lens = [300, 17, 1000]
    cases = [gi.make_case(len(lens), 32, 8, 128, lens, "bf16", seed=60 + i, device="cuda") for i in range(2)]
    cases.append(gi.make_case(len(lens), 32, 8, 128, lens, "bf16", seed=62, device="cuda", spare_blocks=40))
    first = [_run(gq, case).clone() for case in cases]
    for _ in range(2):
        for case, ref in zip(cases, first):
            assert torch.equal(_run(gq, case), ref)
    for case, ref in zip(cases, first):
        assert max_abs_err(ref, oracle_for_case(case)) <= TOL
