"""The KIVI-style 4-bit cache on the GPU against the oracle, through the C ABI.

"LLM 推理性能优化实战" section 15.5 names KIVI: K quantised to INT4 per channel,
V per token. Here a channel's group is the tokens of one 16-token block of one
kv-head: K carries one fp16 scale per (block, kv-head, channel), V one per
(token, kv-head). The append re-quantises every block its tokens reach from
the unquantised K (old slots from the fp32 residual row of the sequence) and
must match the oracle's per-channel append bit for bit, residual included;
the decode must match the fp64 oracle on the dequantised cache within 2e-3."""
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


def _bits(t):
    return t.detach().contiguous().cpu().view(torch.uint8).numpy().copy()


def _host_state(case):
    return (_bits(case.k_cache), _bits(case.v_cache), _bits(case.k_scale).view(np.uint16).reshape(case.k_scale.shape),
            _bits(case.v_scale).view(np.uint16).reshape(case.v_scale.shape),
            case.k_residual.detach().cpu().numpy().copy())


def _oracle_append(oracle_mod, case, state, k_rows, v_rows, positions, counts):
    """Oracle model of one append: K per channel by blocks, V per token."""
    hk, hv, hks, hvs, res = state
    table = case.block_table.cpu().numpy()
    sb, sh, st = case.stride_block, case.stride_head, case.stride_token
    oracle_mod.append_int4_channels(hk, hks, res, k_rows, table, positions, counts, sb, sh, st)
    for b, n in enumerate(counts):
        for i in range(int(n)):
            codes, sbits = oracle_mod.quantize_int4(v_rows[b][i])
            pos = [int(positions[b]) + i]
            oracle_mod.append(hv, oracle_mod.pack_int4(codes)[None], table[b:b + 1], pos,
                              sb // 2, sh // 2, st // 2)
            oracle_mod.append_scales(hvs, sbits[None], table[b:b + 1], pos)


def _assert_state(case, state):
    hk, hv, hks, hvs, res = state
    assert np.array_equal(_bits(case.k_cache), hk)
    assert np.array_equal(_bits(case.v_cache), hv)
    assert np.array_equal(_bits(case.k_scale).view(np.uint16).reshape(hks.shape), hks)
    assert np.array_equal(_bits(case.v_scale).view(np.uint16).reshape(hvs.shape), hvs)
    assert np.array_equal(case.k_residual.cpu().numpy().view(np.uint32), res.view(np.uint32))


@pytest.mark.parametrize("T", [1, 3, 17])
@pytest.mark.parametrize("in_dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("d", [128, 64])
def test_append_requantises_blocks_bit_exactly(gq, oracle_mod, T, in_dtype, d):
    """T new tokens per sequence from lengths that start a block, sit inside
    one, end one, or cross one (T = 17 spans two boundaries)."""
    lens = [0, 1, 15, 16, 31, 40, 200]
    case = gi.make_case(len(lens), 16, 4, d, lens, "i4kc", q_dtype="bf16", seed=90 + T, device="cuda",
                        extra_tokens=T, queries=T, new_dtype=in_dtype)
    # awkward rows: a zero token, a tiny one, a large one, one outlier channel
    kn = case.k_new.clone()
    k4 = kn.view(len(lens), T, 4, d)
    k4[0, 0].zero_()
    k4[1, 0, 1] *= 1e-6
    k4[2, 0, 2] *= 300.0
    k4[3, :, :, 5] *= 40.0
    case.k_new = kn
    state = _host_state(case)
    gq.kv_append(gq.cache_from_case(case), case.k_new, case.v_new, case.block_table, case.context_lens.clone())
    torch.cuda.synchronize()
    k_rows = [case.k_new[b].float().cpu().numpy().reshape(T, 4, d) for b in range(len(lens))]
    v_rows = [case.v_new[b].float().cpu().numpy().reshape(T, 4, d) for b in range(len(lens))]
    _oracle_append(oracle_mod, case, state, k_rows, v_rows, lens, [T] * len(lens))
    _assert_state(case, state)


def test_token_by_token_appends_then_decode(gq, oracle_mod):
    """40 single-token steps from empty sequences: after every step the pool
    equals the oracle's, and the decode of the grown cache matches the oracle."""
    B, H, K, d = 3, 32, 8, 128
    case = gi.make_case(B, H, K, d, [0, 0, 0], "i4kc", seed=95, device="cuda", extra_tokens=40)
    case.k_residual.zero_()
    cache = gq.cache_from_case(case)
    state = _host_state(case)
    g = torch.Generator(device="cuda").manual_seed(96)
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    for step in range(40):
        kn = torch.randn((B, K, d), generator=g, device="cuda").to(torch.bfloat16)
        vn = torch.randn((B, K, d), generator=g, device="cuda").to(torch.bfloat16)
        gq.kv_append(cache, kn, vn, case.block_table, lens)
        _oracle_append(oracle_mod, case, state, [kn[b].float().cpu().numpy()[None] for b in range(B)],
                       [vn[b].float().cpu().numpy()[None] for b in range(B)], [step] * B, [1] * B)
        lens += 1
        if step in (0, 14, 15, 16, 39):
            torch.cuda.synchronize()
            _assert_state(case, state)
            case.context_lens = lens.clone()
            out = gq.gqa_decode(cache, case.q, case.block_table, case.context_lens, case.scale)
            assert max_abs_err(out, oracle_for_case(case)) <= TOL, step


def test_varlen_append_of_prompts(gq, oracle_mod):
    """Prompts of mixed lengths (0, short, several blocks) after mixed prefixes."""
    news = [0, 5, 16, 33, 100]
    prior = [7, 0, 9, 16, 21]
    K, d = 4, 128
    case = gi.make_case(len(news), 16, K, d, prior, "i4kc", seed=97, device="cuda", extra_tokens=max(news))
    g = torch.Generator(device="cuda").manual_seed(98)
    total = sum(news)
    kn = torch.randn((total, K, d), generator=g, device="cuda")
    vn = torch.randn((total, K, d), generator=g, device="cuda")
    starts = torch.tensor(np.concatenate([[0], np.cumsum(news)]), dtype=torch.int32, device="cuda")
    state = _host_state(case)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gq.kv_append_varlen(gq.cache_from_case(case), kn, vn, starts, max(news), case.block_table,
                        case.context_lens.clone(), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    s = starts.cpu().numpy()
    k_rows = [kn[s[b]:s[b + 1]].cpu().numpy() for b in range(len(news))]
    v_rows = [vn[s[b]:s[b + 1]].cpu().numpy() for b in range(len(news))]
    _oracle_append(oracle_mod, case, state, k_rows, v_rows, prior, news)
    _assert_state(case, state)
    case.context_lens += torch.tensor(news, dtype=torch.int32, device="cuda")
    out = gq.gqa_decode(gq.cache_from_case(case), case.q, case.block_table, case.context_lens, case.scale)
    assert max_abs_err(out, oracle_for_case(case)) <= TOL


LENS = [1, 5, 15, 16, 17, 31, 33, 100, 300, 0, 1000, 2047]


@pytest.mark.parametrize("kernel,d", [(1, 128), (2, 128), (2, 64), (0, 64)])
@pytest.mark.parametrize("H,K", [(32, 8), (64, 8), (8, 8), (64, 4)])
def test_decode_matches_oracle(gq, kernel, d, H, K):
    case = gi.make_case(len(LENS), H, K, d, LENS, "i4kc", seed=99, device="cuda")
    ref = oracle_for_case(case)
    for mw in (0, 5):
        out = gq.gqa_decode(gq.cache_from_case(case), case.q, case.block_table, case.context_lens,
                            case.scale, kernel=kernel, max_warps=mw, min_blocks_per_warp=1)
        torch.cuda.synchronize()
        assert max_abs_err(out, ref) <= TOL, (mw,)


@pytest.mark.parametrize("layout", [0, 1, 2])
def test_decode_wide_groups_and_f16_queries(gq, layout):
    case = gi.make_case(4, 64, 2, 128, [33, 700, 5, 0], "i4kc", q_dtype="f16", seed=100, device="cuda")
    out = gq.gqa_decode(gq.cache_from_case(case), case.q, case.block_table, case.context_lens, case.scale,
                        row_layout=layout)
    torch.cuda.synchronize()
    assert max_abs_err(out, oracle_for_case(case)) <= TOL


@pytest.mark.parametrize("T,window,kernel", [(1, 37, 1), (4, 0, 1), (4, 100, 1), (8, 16, 1), (1, 20, 2),
                                             (2, 0, 2)])
def test_decode_with_window_and_several_queries(gq, T, window, kernel):
    lens = [1, 3, 9, 16, 40, 257, 0, 1000]
    case = gi.make_case(len(lens), 16, 4, 128, lens, "i4kc", seed=101, device="cuda", queries=T)
    out = gq.gqa_decode(gq.cache_from_case(case), case.q, case.block_table, case.context_lens, case.scale,
                        window=window, kernel=kernel)
    torch.cuda.synchronize()
    assert max_abs_err(out, oracle_for_case(case, window=window)) <= TOL


def test_large_channel_scales_and_tiny_ones(gq):
    """Channel scales spread over many binades: the f16 product q*s the
    tensor-core path forms stays within the bound."""
    lens = [64, 500]
    case = gi.make_case(2, 32, 8, 128, lens, "i4kc", seed=102, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(103)
    spread = 2.0 ** torch.randint(-12, 4, case.k_scale.shape, generator=g, device="cuda")
    case.k_scale = (case.k_scale.float() * spread).to(torch.float16)
    out = gq.gqa_decode(gq.cache_from_case(case), case.q, case.block_table, case.context_lens, case.scale)
    torch.cuda.synchronize()
    assert max_abs_err(out, oracle_for_case(case)) <= TOL
