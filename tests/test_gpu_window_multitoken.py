"""Sliding-window and multi-token decode on the GPU against the fp64 oracle,
through the C ABI.

Sliding window ("LLM 推理性能优化实战", section 6.4.1): each query attends
only the last W positions up to its own. Several new tokens per sequence
(speculative verification, section 14.2; chunked prefill next to decode,
section 11.7): the T queries sit at positions L-T .. L-1 and are causal among
themselves. Bar: max-abs 2e-3 on fp32 output, as for the plain decode."""
import numpy as np
import pytest
import torch

import gqa_inputs as gi
from helpers import TOL, max_abs_err, oracle_for_case

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


LENS = [1, 5, 15, 16, 17, 31, 33, 100, 300, 0, 1000]


# --------------------------------------------------------------------------- sliding window


@pytest.mark.parametrize("window", [1, 5, 16, 17, 100, 4096])
@pytest.mark.parametrize("dtype,kernel", [("bf16", 1), ("bf16", 2), ("f16", 1), ("f32", 2),
                                          ("i8", 1), ("fp8", 1), ("i4", 1), ("i4", 2)])
def test_sliding_window(gq, dtype, kernel, window):
    case = gi.make_case(len(LENS), 32, 8, 128, LENS, dtype, seed=61, device="cuda")
    ref = oracle_for_case(case, window=window)
    for mw in (0, 3):
        out = _run(gq, case, kernel=kernel, window=window, max_warps=mw, min_blocks_per_warp=1)
        assert max_abs_err(out, ref) <= TOL, (mw,)


def test_window_never_reads_blocks_before_it(gq):
    """Table entries wholly before the window may hold anything: poison them with
    out-of-range indices; the answer must not change and no error is flagged."""
    W = 40
    case = gi.make_case(len(LENS), 16, 4, 128, LENS, "bf16", seed=62, device="cuda")
    ref = _run(gq, case, window=W)
    table = case.block_table.clone()
    for b, L in enumerate(LENS):
        first = max(0, L - W) // 16
        table[b, :first] = case.num_blocks + 1000
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gq.gqa_decode(gq.cache_from_case(case), case.q, table, case.context_lens, case.scale,
                        window=W, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out, ref)


def test_window_covering_the_context_equals_full_attention(gq):
    case = gi.make_case(len(LENS), 32, 8, 128, LENS, "bf16", seed=63, device="cuda")
    full = _run(gq, case)
    assert torch.equal(_run(gq, case, window=max(LENS)), full)


def test_window_of_one_returns_the_newest_value(gq):
    lens = [1, 7, 16, 33]
    case = gi.make_case(len(lens), 8, 2, 128, lens, "bf16", seed=64, device="cuda")
    out = _run(gq, case, window=1)
    ref = oracle_for_case(case, window=1)
    assert np.array_equal(out.cpu().numpy().astype(np.float64), ref)     # p = 1: o = v exactly


def test_window_wide_group(gq):
    case = gi.make_case(len(LENS), 64, 2, 128, LENS, "bf16", seed=65, device="cuda")
    ref = oracle_for_case(case, window=50)
    assert max_abs_err(_run(gq, case, window=50), ref) <= TOL


# --------------------------------------------------------------------------- several new tokens


@pytest.mark.parametrize("T", [2, 4, 8])
@pytest.mark.parametrize("dtype,kernel", [("bf16", 1), ("f16", 1), ("bf16", 2), ("f32", 2),
                                          ("i8", 1), ("fp8", 1), ("i4", 1)])
def test_multi_token_causal(gq, dtype, kernel, T):
    lens = [1, 2, T, T + 1, 16, 17, 64, 300, 0, 1000]
    if kernel == 2 and dtype != "f32" and 4 * T > 8:
        pytest.skip("CUDA-core kernel serves more than 8 rows per kv-head only for fp32 caches")
    case = gi.make_case(len(lens), 32, 8, 128, lens, dtype, seed=66, device="cuda", queries=T)
    ref = oracle_for_case(case)
    for mw in (0, 5):
        out = _run(gq, case, kernel=kernel, max_warps=mw, min_blocks_per_warp=1)
        assert out.shape == case.q.shape
        assert max_abs_err(out, ref) <= TOL, (mw,)


@pytest.mark.parametrize("T,window", [(4, 7), (8, 3), (2, 100), (8, 16)])
def test_multi_token_with_window(gq, T, window):
    lens = [1, 3, 9, 16, 40, 257, 0]
    case = gi.make_case(len(lens), 16, 4, 128, lens, "bf16", seed=67, device="cuda", queries=T)
    ref = oracle_for_case(case, window=window)
    assert max_abs_err(_run(gq, case, window=window), ref) <= TOL


@pytest.mark.parametrize("layout", [0, 1, 2])
@pytest.mark.parametrize("H,K,T,dtype", [(64, 8, 8, "bf16"), (32, 4, 8, "i8"), (8, 8, 4, "f16"),
                                         (16, 1, 4, "bf16"), (24, 8, 4, "fp8")])
def test_multi_token_rows_span_several_warps(gq, H, K, T, dtype, layout):
    """G*T query rows per kv-head up to 64, as 8-row unit streams (layout 1) or
    with the warps of one CTA sharing the tiles (layout 2)."""
    lens = [3, 16, 100, 513]
    case = gi.make_case(len(lens), H, K, 128, lens, dtype, seed=68, device="cuda", queries=T)
    ref = oracle_for_case(case)
    for mw in (0, 7):
        out = _run(gq, case, row_layout=layout, max_warps=mw, min_blocks_per_warp=1)
        assert max_abs_err(out, ref) <= TOL, (mw,)


def test_last_new_token_equals_a_single_token_decode(gq):
    """Query T-1 sees the whole context: the same answer as a one-token decode."""
    T, lens = 4, [20, 77, 300]
    case = gi.make_case(len(lens), 32, 8, 128, lens, "bf16", seed=69, device="cuda", queries=T)
    multi = _run(gq, case)
    one = gq.gqa_decode(gq.cache_from_case(case), case.q[:, T - 1].contiguous(), case.block_table,
                        case.context_lens, case.scale)
    torch.cuda.synchronize()
    assert (multi[:, T - 1] - one).abs().max().item() <= 2e-5


def test_multi_token_append_then_decode(gq, oracle_mod):
    """Append T tokens per sequence (bit-exact against the host scatter), then
    decode them against the oracle."""
    T = 4
    lens = [0, 5, 13, 16, 60]
    case = gi.make_case(len(lens), 16, 4, 128, lens, "bf16", seed=70, device="cuda",
                        extra_tokens=T, queries=T)
    cache = gq.cache_from_case(case)
    before = case.k_cache.detach().cpu().view(torch.int16).numpy().reshape(-1).copy()
    gq.kv_append(cache, case.k_new, case.v_new, case.block_table, case.context_lens.clone())
    torch.cuda.synchronize()
    table = case.block_table.cpu().numpy()
    kn = case.k_new.detach().cpu().view(torch.int16).numpy()
    for i in range(T):
        oracle_mod.append(before, kn[:, i], table, [L + i for L in lens], case.stride_block,
                          case.stride_head, case.stride_token)
    got = case.k_cache.detach().cpu().view(torch.int16).numpy().reshape(-1)
    assert np.array_equal(got, before)
    case.context_lens += T
    ref = oracle_for_case(case)
    assert max_abs_err(_run(gq, case), ref) <= TOL


@pytest.mark.parametrize("cache", ["i8", "fp8", "i4"])
def test_multi_token_append_quantises_bit_exactly(gq, oracle_mod, cache):
    T = 3
    lens = [2, 15, 31]
    case = gi.make_case(len(lens), 16, 4, 128, lens, cache, q_dtype="bf16", seed=71, device="cuda",
                        extra_tokens=T, queries=T, new_dtype="f32")
    hk = case.k_cache.detach().cpu().view(torch.uint8).numpy().reshape(-1).copy()
    hks = case.k_scale.detach().cpu().view(torch.int16).numpy().view(np.uint16).copy()
    gq.kv_append(gq.cache_from_case(case), case.k_new, case.v_new, case.block_table,
                 case.context_lens.clone())
    torch.cuda.synchronize()
    quantize = {"i8": oracle_mod.quantize_int8, "fp8": oracle_mod.quantize_fp8,
                "i4": oracle_mod.quantize_int4}[cache]
    div = 2 if cache == "i4" else 1                  # 4-bit pools are written as bytes
    table = case.block_table.cpu().numpy()
    for i in range(T):
        codes, sbits = quantize(case.k_new[:, i].float().cpu().numpy())
        rows = oracle_mod.pack_int4(codes) if cache == "i4" else codes.view(np.uint8)
        pos = [L + i for L in lens]
        oracle_mod.append(hk, rows, table, pos, case.stride_block // div,
                          case.stride_head // div, case.stride_token // div)
        oracle_mod.append_scales(hks, sbits, table, pos)
    assert np.array_equal(case.k_cache.detach().cpu().view(torch.uint8).numpy().reshape(-1), hk)
    assert np.array_equal(case.k_scale.detach().cpu().view(torch.int16).numpy().view(np.uint16), hks)


def test_multi_token_without_workspace(gq):
    T, lens = 4, [9, 100, 1]
    case = gi.make_case(len(lens), 32, 8, 128, lens, "bf16", seed=72, device="cuda", queries=T)
    out = gq.gqa_decode_noalloc(gq.cache_from_case(case), case.q, case.block_table,
                                case.context_lens, case.scale, window=20)
    torch.cuda.synchronize()
    assert max_abs_err(out, oracle_for_case(case, window=20)) <= TOL
