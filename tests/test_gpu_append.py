"""Paged KV append on the GPU, bit-exact against the oracle's host scatter (and,
for int8 and FP8 caches, against the oracle's quantiser). Calls go through the C ABI."""
import numpy as np
import pytest
import torch

import gqa_inputs as gi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    from gqa_decode_attention_kv_gb300 import build
    build.build()
    import gqa_decode_attention_kv_gb300 as m
    return m


def _raw(t):
    """Bytes of a tensor as a flat uint8 numpy array (no value conversion)."""
    return t.detach().contiguous().cpu().view(torch.uint8).numpy().reshape(-1)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 128), ("f32", 64), ("bf16", 64)])
def test_append_float_cache_is_bit_exact(gq, oracle_mod, dtype, d):
    lens = [0, 5, 15, 16, 17, 31, 32, 33, 100]
    case = gi.make_case(len(lens), 8, 4, d, lens, dtype, seed=11, device="cuda", extra_tokens=1)
    cache = gq.cache_from_case(case)
    ref_k = case.k_cache.detach().cpu().clone()
    ref_v = case.v_cache.detach().cpu().clone()
    pos = case.context_lens.clone()
    gq.kv_append(cache, case.k_new, case.v_new, case.block_table, pos)
    torch.cuda.synchronize()
    table = case.block_table.cpu().numpy()
    # oracle scatter on raw 16/32-bit words: no value conversion anywhere
    word = {2: np.uint16, 4: np.uint32}[case.k_cache.element_size()]
    hk = _raw(ref_k).view(word).copy()
    hv = _raw(ref_v).view(word).copy()
    oracle_mod.append(hk, _raw(case.k_new).view(word).reshape(case.k_new.shape), table, lens,
                      case.stride_block, case.stride_head, case.stride_token)
    oracle_mod.append(hv, _raw(case.v_new).view(word).reshape(case.v_new.shape), table, lens,
                      case.stride_block, case.stride_head, case.stride_token)
    got_k = _raw(case.k_cache).view(word)
    got_v = _raw(case.v_cache).view(word)
    # NaN payloads compare as bits, so untouched poisoned slots must match too
    assert np.array_equal(got_k, hk)
    assert np.array_equal(got_v, hv)


@pytest.mark.parametrize("cache", ["i8", "fp8", "i4"])
@pytest.mark.parametrize("in_dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("d", [128, 64])
def test_append_coded_cache_quantises_bit_exactly(gq, oracle_mod, cache, in_dtype, d):
    lens = [3, 16, 40, 1, 0, 255]
    case = gi.make_case(len(lens), 16, 8, d, lens, cache, q_dtype="bf16", seed=12, device="cuda",
                        extra_tokens=1, new_dtype=in_dtype)
    # a few awkward rows: all zeros, a tiny-magnitude row, a large one
    kn = case.k_new.clone()
    kn[0, 0].zero_()
    kn[1, 1] *= 1e-6
    kn[2, 2] *= 300.0
    case.k_new = kn
    before = [_raw(t).copy() for t in (case.k_cache, case.v_cache, case.k_scale, case.v_scale)]
    gq.kv_append(gq.cache_from_case(case), case.k_new, case.v_new, case.block_table,
                 case.context_lens.clone())
    torch.cuda.synchronize()
    table = case.block_table.cpu().numpy()
    quantize = {"i8": oracle_mod.quantize_int8, "fp8": oracle_mod.quantize_fp8,
                "i4": oracle_mod.quantize_int4}[cache]
    hk = before[0].view(np.uint8).copy()
    hv = before[1].view(np.uint8).copy()
    hks = before[2].view(np.uint16).reshape(case.k_scale.shape).copy()
    hvs = before[3].view(np.uint16).reshape(case.v_scale.shape).copy()
    # a 4-bit pool is written as bytes: packed rows, element strides halved
    div = 2 if cache == "i4" else 1
    for new, pool, sc in ((case.k_new, hk, hks), (case.v_new, hv, hvs)):
        codes, sbits = quantize(new.float().cpu().numpy())
        rows = oracle_mod.pack_int4(codes) if cache == "i4" else codes.view(np.uint8)
        oracle_mod.append(pool, rows, table, lens, case.stride_block // div,
                          case.stride_head // div, case.stride_token // div)
        oracle_mod.append_scales(sc, sbits, table, lens)
    assert np.array_equal(_raw(case.k_cache), hk)
    assert np.array_equal(_raw(case.v_cache), hv)
    assert np.array_equal(_raw(case.k_scale).view(np.uint16).reshape(hks.shape), hks)
    assert np.array_equal(_raw(case.v_scale).view(np.uint16).reshape(hvs.shape), hvs)


def test_append_contiguous_layout(gq, oracle_mod):
    """The un-paged [B, S_pad, K, d] layout with an identity table."""
    case = gi.make_case(2, 8, 2, 64, [37, 99], "f32", seed=13, device="cuda", contiguous=True,
                        extra_tokens=1)
    ref = case.k_cache.detach().cpu().numpy().copy()
    gq.kv_append(gq.cache_from_case(case), case.k_new, case.v_new, case.block_table,
                 case.context_lens.clone())
    torch.cuda.synchronize()
    for b, L in enumerate([37, 99]):
        ref[b, L] = case.k_new[b].cpu().numpy()
    got = case.k_cache.cpu().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.nan_to_num(got), np.nan_to_num(ref))


def test_append_flags_bad_positions_and_tables(gq):
    case = gi.make_case(3, 8, 2, 128, [5, 5, 5], "bf16", seed=14, device="cuda", extra_tokens=1)
    before = case.k_cache.detach().clone()
    table = case.block_table.clone()
    table[1, 0] = case.num_blocks + 7            # out-of-range physical block
    pos = torch.tensor([5, 5, 10_000], dtype=torch.int32, device="cuda")  # seq 2 past the table
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gq.kv_append(gq.cache_from_case(case), case.k_new, case.v_new, table, pos, err=err)
    torch.cuda.synchronize()
    flags = int(err.item())
    assert flags & gq.GQA_DEVERR_BLOCK_INDEX and flags & gq.GQA_DEVERR_POSITION
    # sequence 0 was written; nothing else changed
    changed = (case.k_cache.view(torch.int16) != before.view(torch.int16)).reshape(case.num_blocks, -1).any(1)
    assert changed.sum().item() == 1 and changed[int(table[0, 0])]
