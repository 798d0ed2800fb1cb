"""Pins for the CPU oracle: each check ties it to something other than itself --
figures the pages print, closed forms, library routines (torch SDPA, numpy's
fp16 rounding) and invariants that a dropped term, a wrong sign, index or
transposed operand would break. CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import gqa_inputs as gi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa_reference(q, k, v, lens, scale):
    """Library reference: torch SDPA in fp64 on CPU, K/V repeat-interleaved to H heads."""
    B, H, d = q.shape
    K = k.shape[2]
    G = H // K
    out = np.zeros((B, H, d))
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        qb = torch.from_numpy(q[b]).reshape(1, H, 1, d)
        kb = torch.from_numpy(k[b, :L]).permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
        vb = torch.from_numpy(v[b, :L]).permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
        o = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, scale=scale)
        out[b] = o.reshape(H, d).numpy()
    return out


# --------------------------------------------------------------------------- decode


@pytest.mark.parametrize("B,H,K,d,lens", [
    (2, 8, 2, 64, [37, 100]),          # the tiny contiguous workload's shape
    (3, 8, 8, 16, [1, 5, 33]),         # G = 1: plain multi-head attention
    (2, 8, 1, 32, [17, 9]),            # K = 1: multi-query attention
    (1, 12, 3, 128, [70]),
])
def test_decode_matches_torch_sdpa_with_repeat_interleave(oracle_mod, B, H, K, d, lens):
    q = _rand((B, H, d), 1)
    k = _rand((B, max(lens), K, d), 2)
    v = _rand((B, max(lens), K, d), 3)
    scale = 1.0 / math.sqrt(d)
    got = oracle_mod.decode(q, k, v, lens, scale)
    ref = _sdpa_reference(q, k, v, lens, scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_decode_matches_sdpa_native_gqa(oracle_mod):
    """torch's own grouped-query mode (enable_gqa) fixes the head-to-group map."""
    B, H, K, d, S = 2, 8, 2, 32, 11
    q, k, v = _rand((B, H, d), 4), _rand((B, S, K, d), 5), _rand((B, S, K, d), 6)
    got = oracle_mod.decode(q, k, v, [S, S], 0.3)
    qt = torch.from_numpy(q).unsqueeze(2)
    kt = torch.from_numpy(k).permute(0, 2, 1, 3)
    vt = torch.from_numpy(v).permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=0.3, enable_gqa=True)
    np.testing.assert_allclose(got, ref.squeeze(2).numpy(), rtol=0, atol=1e-12)


def test_group_mapping_is_contiguous_not_modulo(oracle_mod):
    """Head h must read KV head h // G. Give each KV head a constant V value equal to
    its index: the output of head h is then exactly h // G."""
    B, H, K, d, S = 1, 8, 2, 4, 6
    q = _rand((B, H, d), 7)
    k = _rand((B, S, K, d), 8)
    v = np.zeros((B, S, K, d))
    for g in range(K):
        v[:, :, g, :] = g
    out = oracle_mod.decode(q, k, v, [S], 0.5)
    for h in range(H):
        assert np.all(out[0, h] == h // (H // K))


def test_one_token_context_returns_v_exactly(oracle_mod):
    q, k, v = _rand((2, 4, 8), 9), _rand((2, 3, 2, 8), 10), _rand((2, 3, 2, 8), 11)
    out = oracle_mod.decode(q, k, v, [1, 1], 0.7)
    for b in range(2):
        for h in range(4):
            assert np.array_equal(out[b, h], v[b, 0, h // 2])


def test_zero_query_gives_mean_of_values(oracle_mod):
    q = np.zeros((1, 4, 16))
    k, v = _rand((1, 40, 2, 16), 12), _rand((1, 40, 2, 16), 13)
    out = oracle_mod.decode(q, k, v, [29], 1.0)
    for h in range(4):
        np.testing.assert_allclose(out[0, h], v[0, :29, h // 2].mean(axis=0), rtol=0, atol=1e-14)


def test_two_token_closed_form_fixes_sign_and_scale(oracle_mod):
    """d=1, k_1=1, k_2=0: s_1 = scale*a, s_2 = 0, so o = (v1 e^{s1} + v2) / (e^{s1} + 1)."""
    a, scale = 3.0, 0.25
    q = np.array([[[a]]])
    k = np.array([[[[1.0]], [[0.0]]]])
    v = np.array([[[[2.0]], [[-5.0]]]])
    out = oracle_mod.decode(q, k, v, [2], scale)
    s1 = scale * a
    expect = (2.0 * math.exp(s1) - 5.0) / (math.exp(s1) + 1.0)
    assert out[0, 0, 0] == pytest.approx(expect, abs=1e-15)


def test_large_scores_do_not_overflow_and_pick_dominant_key(oracle_mod):
    d = 8
    k = np.zeros((1, 5, 1, d))
    k[0, :, 0, 0] = [1.0, 2.0, 3.0, 50.0, 4.0]
    v = _rand((1, 5, 1, d), 14)
    q = np.zeros((1, 1, d))
    q[0, 0, 0] = 100.0                      # scores up to 5000: exp would overflow unshifted
    out = oracle_mod.decode(q, k, v, [5], 1.0)
    np.testing.assert_array_equal(out[0, 0], v[0, 3, 0])


def test_permuting_tokens_leaves_output_unchanged(oracle_mod):
    q, k, v = _rand((1, 4, 16), 15), _rand((1, 23, 2, 16), 16), _rand((1, 23, 2, 16), 17)
    perm = np.random.default_rng(18).permutation(23)
    a = oracle_mod.decode(q, k, v, [23], 0.25)
    b = oracle_mod.decode(q, k[:, perm], v[:, perm], [23], 0.25)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


def test_tokens_past_length_are_ignored(oracle_mod):
    q, k, v = _rand((2, 4, 8), 19), _rand((2, 30, 2, 8), 20), _rand((2, 30, 2, 8), 21)
    a = oracle_mod.decode(q, k, v, [12, 30], 0.5)
    k2, v2 = k.copy(), v.copy()
    k2[0, 12:] = np.nan
    v2[0, 12:] = np.nan
    b = oracle_mod.decode(q, k2, v2, [12, 30], 0.5)
    np.testing.assert_array_equal(a, b)


def test_empty_context_gives_zero(oracle_mod):
    q, k, v = _rand((2, 2, 8), 22), _rand((2, 4, 1, 8), 23), _rand((2, 4, 1, 8), 24)
    out = oracle_mod.decode(q, k, v, [0, 4], 0.5)
    assert np.all(out[0] == 0.0) and np.all(np.isfinite(out[1]))


def _sdpa_masked(q4, k, v, lens, scale, window):
    """Library reference for T queries per sequence: torch SDPA (fp64, CPU) with an
    explicit boolean mask; query i of sequence b is at position lens[b] - T + i."""
    B, T, H, d = q4.shape
    G = H // k.shape[2]
    out = np.zeros(q4.shape)
    for b in range(B):
        L = int(lens[b])
        pos = L - T + np.arange(T)
        t = np.arange(L)
        allow = t[None, :] <= pos[:, None]
        if window:
            allow &= t[None, :] > pos[:, None] - window
        rows = allow.any(1)
        if not rows.any():
            continue
        qb = torch.from_numpy(q4[b][rows]).permute(1, 0, 2).unsqueeze(0)           # [1, H, T', d]
        kb = torch.from_numpy(k[b, :L]).permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
        vb = torch.from_numpy(v[b, :L]).permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
        o = torch.nn.functional.scaled_dot_product_attention(
            qb, kb, vb, attn_mask=torch.from_numpy(allow[rows]), scale=scale)
        out[b][rows] = o[0].permute(1, 0, 2).numpy()
    return out


@pytest.mark.parametrize("window,lens", [
    (1, [1, 7, 40]), (5, [3, 5, 6, 100]), (16, [16, 17, 33]), (37, [36, 37, 38, 200]),
])
def test_sliding_window_matches_sdpa_with_band_mask(oracle_mod, window, lens):
    B, H, K, d = len(lens), 8, 2, 32
    q = _rand((B, H, d), 41)
    k = _rand((B, max(lens), K, d), 42)
    v = _rand((B, max(lens), K, d), 43)
    got = oracle_mod.decode(q, k, v, lens, 0.2, window=window)
    ref = _sdpa_masked(q[:, None], k, v, lens, 0.2, window)[:, 0]
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    # same as full attention over the last `window` tokens, cut out by hand
    for b, L in enumerate(lens):
        lo = max(0, L - window)
        cut = oracle_mod.decode(q[b:b + 1], k[b:b + 1, lo:L], v[b:b + 1, lo:L], [L - lo], 0.2)
        np.testing.assert_allclose(got[b:b + 1], cut, rtol=0, atol=1e-12)


def test_window_of_one_returns_the_newest_value_exactly(oracle_mod):
    lens = [1, 9, 30]
    k = _rand((3, 30, 2, 16), 44)
    v = _rand((3, 30, 2, 16), 45)
    got = oracle_mod.decode(_rand((3, 4, 16), 46), k, v, lens, 1.0, window=1)
    for b, L in enumerate(lens):
        assert np.array_equal(got[b], np.repeat(v[b, L - 1], 2, axis=0))


def test_window_covering_the_context_is_full_attention(oracle_mod):
    lens = [5, 64]
    q, k, v = _rand((2, 4, 16), 47), _rand((2, 64, 2, 16), 48), _rand((2, 64, 2, 16), 49)
    full = oracle_mod.decode(q, k, v, lens, 0.3)
    assert np.array_equal(oracle_mod.decode(q, k, v, lens, 0.3, window=64), full)
    assert np.array_equal(oracle_mod.decode(q, k, v, lens, 0.3, window=1000), full)


@pytest.mark.parametrize("T,window", [(2, 0), (4, 0), (8, 0), (3, 5), (8, 4)])
def test_multi_token_matches_sdpa_with_causal_mask(oracle_mod, T, window):
    lens = [T, T + 1, 17, 50]
    B, H, K, d = len(lens), 8, 2, 32
    q = _rand((B, T, H, d), 50)
    k = _rand((B, max(lens), K, d), 51)
    v = _rand((B, max(lens), K, d), 52)
    got = oracle_mod.decode(q, k, v, lens, 0.25, window=window)
    ref = _sdpa_masked(q, k, v, lens, 0.25, window)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_each_new_token_sees_exactly_its_prefix(oracle_mod):
    """Query i of T equals a one-token decode over the prefix ending at its position."""
    T, lens = 4, [6, 21]
    q = _rand((2, T, 8, 16), 53)
    k, v = _rand((2, 21, 4, 16), 54), _rand((2, 21, 4, 16), 55)
    got = oracle_mod.decode(q, k, v, lens, 0.5)
    for b, L in enumerate(lens):
        for i in range(T):
            one = oracle_mod.decode(q[b:b + 1, i], k[b:b + 1], v[b:b + 1], [L - T + i + 1], 0.5)
            np.testing.assert_array_equal(got[b:b + 1, i], one)
    # causality: changing the last new token's K/V leaves the earlier queries alone
    k2, v2 = k.copy(), v.copy()
    k2[0, lens[0] - 1] += 3.0
    v2[0, lens[0] - 1] -= 2.0
    got2 = oracle_mod.decode(q, k2, v2, lens, 0.5)
    assert np.array_equal(got2[0, :T - 1], got[0, :T - 1])
    assert not np.array_equal(got2[0, T - 1], got[0, T - 1])


def test_queries_before_the_sequence_start_give_zero(oracle_mod):
    """lens < T: the queries at negative positions attend nothing."""
    T = 4
    q = _rand((1, T, 4, 8), 56)
    k, v = _rand((1, 2, 2, 8), 57), _rand((1, 2, 2, 8), 58)
    got = oracle_mod.decode(q, k, v, [2], 1.0)
    assert np.array_equal(got[0, :2], np.zeros((2, 4, 8)))
    assert np.array_equal(got[0, 2], np.repeat(v[0, 0], 2, axis=0))   # one token: o = v


def test_thread_count_does_not_change_result(oracle_mod):
    q, k, v = _rand((3, 8, 32), 25), _rand((3, 50, 2, 32), 26), _rand((3, 50, 2, 32), 27)
    a = oracle_mod.decode(q, k, v, [50, 7, 31], 0.2, nthreads=1)
    b = oracle_mod.decode(q, k, v, [50, 7, 31], 0.2, nthreads=5)
    np.testing.assert_array_equal(a, b)


# --------------------------------------------------------------------------- paging


def test_gather_with_identity_table_is_a_reshape(oracle_mod):
    B, S_pad, K, d = 2, 48, 2, 8
    dense = _rand((B, S_pad, K, d), 28)
    table = np.arange(B * 3).reshape(B, 3)
    got = oracle_mod.gather_dense(dense, table, [40, 48], 16 * K * d, d, K * d, K, d)
    np.testing.assert_array_equal(got[0, :40], dense[0, :40])
    np.testing.assert_array_equal(got[1], dense[1])


def test_append_then_gather_round_trips_through_a_shuffled_pool(oracle_mod):
    """Scatter a sequence token by token into a pool with a shuffled table, then
    gather it back: the block/slot arithmetic must invert exactly."""
    B, K, d, S = 3, 2, 8, 37
    nb_per = -(-S // 16)
    NB = B * nb_per + 2
    rng = np.random.default_rng(29)
    perm = rng.permutation(NB)
    table = perm[:B * nb_per].reshape(B, nb_per)
    pool = np.full((NB, K, 16, d), np.nan)
    seq = _rand((B, S, K, d), 30)
    for t in range(S):
        oracle_mod.append(pool, seq[:, t], table, [t] * B, K * 16 * d, 16 * d, d)
    got = oracle_mod.gather_dense(pool, table, [S] * B, K * 16 * d, 16 * d, d, K, d)
    np.testing.assert_array_equal(got, seq)
    # exactly the slots written are non-NaN: B * S tokens * K heads * d elements
    assert np.count_nonzero(~np.isnan(pool)) == B * S * K * d


def _labelled_scale_pool(nb, K):
    """[nb, K, 16] pool whose entry (block p, kv-head g, slot s) holds 1000*p + 100*g + s,
    so every gathered value names the slot it came from."""
    return np.array([[[1000 * p + 100 * g + s for s in range(16)] for g in range(K)]
                     for p in range(nb)], dtype=np.int64)


def test_scale_gather_reads_the_slots_the_table_names(oracle_mod):
    """Per-(token, kv-head) scales gathered through a shuffled table, checked
    against expected values written out by hand: sequence 0 holds 18 tokens in
    blocks 2 then 0, sequence 1 holds 3 tokens in block 3."""
    pool = _labelled_scale_pool(4, 2)
    table = np.array([[2, 0], [3, -1]], dtype=np.int32)
    got = oracle_mod.gather_scales(pool, table, [18, 3], 2)
    assert got.shape == (2, 18, 2)
    seq0_head0 = list(range(2000, 2016)) + [0, 1]
    seq0_head1 = list(range(2100, 2116)) + [100, 101]
    seq1_head0 = [3000, 3001, 3002] + [0] * 15          # past the length: left at zero
    seq1_head1 = [3100, 3101, 3102] + [0] * 15
    np.testing.assert_array_equal(got[0, :, 0], seq0_head0)
    np.testing.assert_array_equal(got[0, :, 1], seq0_head1)
    np.testing.assert_array_equal(got[1, :, 0], seq1_head0)
    np.testing.assert_array_equal(got[1, :, 1], seq1_head1)
    # a subset of rows, in the order asked for
    sub = oracle_mod.gather_scales(pool, table, [18, 3], 2, batch_index=[1])
    assert sub.shape == (1, 3, 2)
    np.testing.assert_array_equal(sub[0], [[3000, 3100], [3001, 3101], [3002, 3102]])


def test_scale_append_writes_only_the_named_slot(oracle_mod):
    """Appending at positions 17 and 2 writes block table[0][1] = 0, slot 1 and
    block table[1][0] = 3, slot 2, for both kv-heads, and nothing else."""
    pool = _labelled_scale_pool(4, 2)
    before = pool.copy()
    table = np.array([[2, 0], [3, -1]], dtype=np.int32)
    new = np.array([[-7, -8], [-9, -10]], dtype=np.int64)         # [B, K]
    oracle_mod.append_scales(pool, new, table, [17, 2])
    expect = before.copy()
    expect[0, 0, 1], expect[0, 1, 1] = -7, -8
    expect[3, 0, 2], expect[3, 1, 2] = -9, -10
    np.testing.assert_array_equal(pool, expect)
    # and the gather sees the new values at those positions
    got = oracle_mod.gather_scales(pool, table, [18, 3], 2)
    np.testing.assert_array_equal(got[0, 17], [-7, -8])
    np.testing.assert_array_equal(got[1, 2], [-9, -10])


def test_block_padding_example_from_the_pages(oracle_mod):
    with open(os.path.join(GOLDEN, "block_padding.json")) as f:
        gold = json.load(f)
    for case in gold["cases"]:
        nb = oracle_mod.blocks_for_tokens(case["tokens"])
        assert nb == case["blocks"]
        assert nb * gold["block_size"] == case["slots"]
        assert nb * gold["block_size"] - case["tokens"] == case["wasted"]
        assert case["wasted"] <= gold["block_size"] - 1


# --------------------------------------------------------------------------- KV size


def test_kv_size_closed_form_reproduces_printed_figures(oracle_mod):
    with open(os.path.join(GOLDEN, "kv_size_figures.json")) as f:
        gold = json.load(f)
    for key, g in gold.items():
        if key.startswith("_"):
            continue
        n = oracle_mod.kv_cache_elements(g["layers"], g["kv_heads"], g["head_dim"],
                                         g["seq_len"], g["batch"])
        n_bytes = n * g.get("bytes_per_element", 1)
        unit = {"1e9 elements": 1e9, "1e9 bytes": 1e9, "MiB": 2 ** 20}[g["unit"]]
        scaled = n_bytes / unit
        trunc = math.floor(scaled * 10 ** g["decimals"]) / 10 ** g["decimals"]
        assert trunc == pytest.approx(g["printed"]), key
    mha = oracle_mod.kv_cache_elements(80, 64, 128, 2048, 1)
    gqa = oracle_mod.kv_cache_elements(80, 8, 128, 2048, 1)
    assert (mha, gqa) == (2_684_354_560, 335_544_320)
    assert mha == 8 * gqa                                  # KV bytes scale as 1/G


# --------------------------------------------------------------------------- fp16 / int8


def test_fp16_rounding_matches_numpy_everywhere(oracle_mod):
    rng = np.random.default_rng(31)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 4000),
        np.array([0.0, -0.0, 65504.0, 65519.996, 65520.0, 1e6, -1e6, 2 ** -24, 2 ** -25,
                  3 * 2 ** -26, 2 ** -14, 2 ** -14 - 2 ** -25, 6.1e-5, 1.0 + 2 ** -11,
                  1.0 + 3 * 2 ** -11, 1.0 + 2 ** -11 + 2 ** -20, np.inf, -np.inf], dtype=np.float32),
    ])
    got = oracle_mod.f32_to_f16_bits(vals)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, ref)
    back = oracle_mod.f16_bits_to_f64(ref)
    np.testing.assert_array_equal(back, ref.view(np.float16).astype(np.float64))


def test_int8_rounding_worked_example():
    """amax = 127 gives scale exactly 1.0, so codes are rint(x) with ties to even."""
    import oracle
    x = np.array([[127.0, -63.5, 0.5, 1.5, 2.5, -2.5, 126.4, 0.0]], dtype=np.float32)
    codes, scale = oracle.quantize_int8(x)
    assert scale[0] == np.float16(1.0).view(np.uint16)
    assert codes[0].tolist() == [127, -64, 0, 2, 2, -2, 126, 0]


def test_int8_quantisation_invariants(oracle_mod):
    rng = np.random.default_rng(32)
    x = rng.standard_normal((500, 128)).astype(np.float32) * np.float32(10.0) ** rng.integers(-3, 4, (500, 1))
    codes, sbits = oracle_mod.quantize_int8(x)
    s = oracle_mod.f16_bits_to_f64(sbits)
    # the row maximum lands on +-127 (scale is amax/127 within fp16 rounding)
    assert np.all(np.abs(codes.astype(np.int32)).max(axis=1) == 127)
    assert codes.min() >= -127
    # reconstruction error of each element is at most half a step
    err = np.abs(x.astype(np.float64) - codes * s[:, None])
    assert np.all(err <= s[:, None] / 2 * (1 + 1e-6))
    # symmetric: negating the input negates the codes and keeps the scale
    c2, s2 = oracle_mod.quantize_int8(-x)
    np.testing.assert_array_equal(c2, -codes)
    np.testing.assert_array_equal(s2, sbits)
    # a power-of-two rescale moves only the scale, while the scale stays a normal
    # fp16 number (below 2**-14 fp16 has a fixed absolute step, so rounding differs)
    c3, s3 = oracle_mod.quantize_int8(x * np.float32(4.0))
    normal = s >= 2.0 ** -14
    assert normal.sum() > 300
    np.testing.assert_array_equal(c3[normal], codes[normal])
    np.testing.assert_array_equal(oracle_mod.f16_bits_to_f64(s3)[normal], 4 * s[normal])
    # an all-zero row quantises to scale 0 and codes 0
    cz, sz = oracle_mod.quantize_int8(np.zeros((1, 64), dtype=np.float32))
    assert sz[0] == 0 and not cz.any()


def test_int4_rounding_worked_example(oracle_mod):
    """amax = 7 gives scale exactly 1.0, so codes are rint(x) with ties to even."""
    x = np.array([[7.0, -6.5, 0.5, 1.5, 2.5, -2.5, 3.5, 0.0]], dtype=np.float32)
    codes, scale = oracle_mod.quantize_int4(x)
    assert scale[0] == np.float16(1.0).view(np.uint16)
    assert codes[0].tolist() == [7, -6, 0, 2, 2, -2, 4, 0]


def test_int4_quantisation_invariants(oracle_mod):
    rng = np.random.default_rng(33)
    x = rng.standard_normal((500, 128)).astype(np.float32) * np.float32(10.0) ** rng.integers(-3, 4, (500, 1))
    codes, sbits = oracle_mod.quantize_int4(x)
    s = oracle_mod.f16_bits_to_f64(sbits)
    assert np.all(np.abs(codes.astype(np.int32)).max(axis=1) == 7)
    assert codes.min() >= -7 and codes.max() <= 7
    err = np.abs(x.astype(np.float64) - codes * s[:, None])
    assert np.all(err <= s[:, None] / 2 * (1 + 1e-6))
    c2, s2 = oracle_mod.quantize_int4(-x)
    np.testing.assert_array_equal(c2, -codes)
    np.testing.assert_array_equal(s2, sbits)
    cz, sz = oracle_mod.quantize_int4(np.zeros((1, 64), dtype=np.float32))
    assert sz[0] == 0 and not cz.any()
    # the int4 step is 127/7 times the int8 one (before fp16 rounding of each)
    _, s8 = oracle_mod.quantize_int8(x)
    ratio = s / oracle_mod.f16_bits_to_f64(s8)
    normal = oracle_mod.f16_bits_to_f64(s8) >= 2.0 ** -14
    np.testing.assert_allclose(ratio[normal], 127 / 7, rtol=2 ** -10)


def test_int4_packing_bytes(oracle_mod):
    """Element 2j in the low nibble, two's complement: -7 -> 0x9, -1 -> 0xF, -4 -> 0xC."""
    codes = np.array([[-7, 7, 0, -1, 3, -4]], dtype=np.int8)
    packed = oracle_mod.pack_int4(codes)
    assert packed[0].tolist() == [0x79, 0xF0, 0xC3]
    every = np.array([[a, b] for a in range(-8, 8) for b in range(-8, 8)], dtype=np.int8).reshape(1, -1)
    np.testing.assert_array_equal(oracle_mod.unpack_int4(oracle_mod.pack_int4(every)), every)
    assert sorted(set(oracle_mod.pack_int4(every)[0].tolist())) == list(range(256))


def test_int4_dequantised_attention_matches_sdpa(oracle_mod):
    rng = np.random.default_rng(34)
    kv = rng.standard_normal((1, 20, 2, 64)).astype(np.float32)
    codes, sbits = oracle_mod.quantize_int4(kv)
    deq = oracle_mod.dequantize_int4(oracle_mod.pack_int4(codes), oracle_mod.f16_bits_to_f64(sbits))
    assert deq.shape == kv.shape
    np.testing.assert_array_equal(deq, codes * oracle_mod.f16_bits_to_f64(sbits)[..., None])
    q = rng.standard_normal((1, 8, 64))
    got = oracle_mod.decode(q, deq, deq, [20], 0.125)
    ref = _sdpa_reference(q, deq, deq, [20], 0.125)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_dequantised_attention_equals_attention_on_dequantised_values(oracle_mod):
    """The int8 path is the float path fed q*s: the dequantised cache is exact in fp64."""
    rng = np.random.default_rng(33)
    x = rng.standard_normal((1, 20, 2, 64)).astype(np.float32)
    codes, sb = oracle_mod.quantize_int8(x)
    kv = oracle_mod.dequantize_int8(codes, oracle_mod.f16_bits_to_f64(sb))
    q = _rand((1, 4, 64), 34)
    got = oracle_mod.decode(q, kv, kv, [20], 0.125)
    ref = _sdpa_reference(q, kv, kv, [20], 0.125)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    assert np.abs(kv - x).max() <= oracle_mod.f16_bits_to_f64(sb).max() / 2 * (1 + 1e-6)


# --------------------------------------------------------------------------- KIVI-style K (per channel)


def test_int4_channel_rounding_worked_example(oracle_mod):
    """Worked by hand: channel 0 = (0.7, -1.4, 0.35) has amax 1.4, scale
    fp16(0.2) = 0.199951171875 (0x3266), and 0.7/s = 3.5009 -> 4, -1.4/s =
    -7.0017 -> -7, 0.35/s = 1.7504 -> 2. Channel 1 = (1, 0.5, -0.25): scale
    fp16(1/7) = 0.142822265625 (0x3092), codes 7, 4 (3.5009), -2 (-1.7504).
    Channel 2 = (3.5, -7, 0): amax 7 gives scale 1, codes rint with ties to even."""
    x = np.array([[0.7, 1.0, 3.5], [-1.4, 0.5, -7.0], [0.35, -0.25, 0.0]], dtype=np.float32)
    codes, sbits = oracle_mod.quantize_int4_channels(x)
    assert sbits.tolist() == [0x3266, 0x3092, 0x3C00]
    assert codes.tolist() == [[4, 7, 4], [-7, 4, -7], [2, -2, 0]]


def test_int4_channel_scales_follow_channels_not_tokens(oracle_mod):
    """Channel i scaled by 2^i: the scales double channel by channel and the
    codes of every channel are the same column (a token-wise grouping would
    give each token one scale instead)."""
    rng = np.random.default_rng(35)
    base = rng.uniform(0.5, 2.0, (16, 1)).astype(np.float32)
    x = base * (np.float32(2.0) ** np.arange(8, dtype=np.float32))[None, :]
    codes, sbits = oracle_mod.quantize_int4_channels(x)
    s = oracle_mod.f16_bits_to_f64(sbits)
    np.testing.assert_array_equal(s[1:] / s[:-1], np.full(7, 2.0))
    for i in range(1, 8):
        np.testing.assert_array_equal(codes[:, i], codes[:, 0])


def test_int4_channel_quantisation_invariants(oracle_mod):
    rng = np.random.default_rng(36)
    for n in (1, 2, 7, 16):
        x = rng.standard_normal((n, 128)).astype(np.float32) * np.float32(10.0) ** rng.integers(-3, 4, (1, 128))
        codes, sbits = oracle_mod.quantize_int4_channels(x)
        s = oracle_mod.f16_bits_to_f64(sbits)
        # each channel's largest magnitude lands on +-7; codes stay in [-7, 7]
        assert np.all(np.abs(codes.astype(np.int32)).max(axis=0) == 7)
        assert codes.min() >= -7 and codes.max() <= 7
        # reconstruction error is at most half a step of the element's channel
        err = np.abs(x.astype(np.float64) - codes * s[None, :])
        assert np.all(err <= s[None, :] / 2 * (1 + 1e-6))
        # changing one channel changes no other channel's codes or scale
        y = x.copy()
        y[:, 5] *= np.float32(-3.0)
        c2, s2 = oracle_mod.quantize_int4_channels(y)
        keep = np.arange(128) != 5
        np.testing.assert_array_equal(c2[:, keep], codes[:, keep])
        np.testing.assert_array_equal(s2[keep], sbits[keep])
        # the per-channel codes of x are the per-token codes of x transposed
        ct, st = oracle_mod.quantize_int4(x.T)
        np.testing.assert_array_equal(ct.T, codes)
        np.testing.assert_array_equal(st, sbits)
    cz, sz = oracle_mod.quantize_int4_channels(np.zeros((3, 64), dtype=np.float32))
    assert not sz.any() and not cz.any()


def test_channel_scale_gather_and_append_on_a_tiny_pool(oracle_mod):
    """Token by token through a shuffled pool: after each append the block a
    token landed in holds the per-channel codes of everything in it so far
    (re-quantised from the unquantised values), finished blocks keep theirs,
    and the gathered scales follow the block table."""
    rng = np.random.default_rng(37)
    K, d, NB = 2, 8, 6
    table = np.array([[4, 1, 3]], dtype=np.int32)
    sb_, sh_, st_ = K * 16 * d, 16 * d, d
    pool = np.zeros(NB * sb_ // 2, dtype=np.uint8)
    scales = np.zeros((NB, K, d), dtype=np.uint16)
    resid = np.zeros((1, K, 16, d), dtype=np.float32)
    xs = rng.standard_normal((40, K, d)).astype(np.float32)
    for pos in range(40):
        oracle_mod.append_int4_channels(pool, scales, resid, [xs[pos:pos + 1]], table, [pos], [1],
                                        sb_, sh_, st_)
        jb, L = pos // 16, pos + 1
        for g in range(K):
            blk = xs[16 * jb:L, g]
            codes, sbits = oracle_mod.quantize_int4_channels(blk)
            ph = table[0, jb]
            np.testing.assert_array_equal(scales[ph, g], sbits)
            got = pool[(ph * sb_ + g * sh_) // 2:(ph * sb_ + g * sh_) // 2 + len(blk) * d // 2]
            np.testing.assert_array_equal(oracle_mod.unpack_int4(got.reshape(len(blk), d // 2)), codes)
    # all 40 appended one at a time == the same 40 appended in one call
    pool2 = np.zeros_like(pool)
    scales2 = np.zeros_like(scales)
    resid2 = np.zeros_like(resid)
    oracle_mod.append_int4_channels(pool2, scales2, resid2, [xs], table, [0], [40], sb_, sh_, st_)
    np.testing.assert_array_equal(pool2, pool)
    np.testing.assert_array_equal(scales2, scales)
    np.testing.assert_array_equal(resid2[0, :, :8], resid[0, :, :8])
    dense = oracle_mod.gather_channel_scales(scales, table, [40])
    assert dense.shape == (1, 40, K, d)
    for t in (0, 15, 16, 39):
        np.testing.assert_array_equal(dense[0, t], scales[table[0, t // 16]])


# --------------------------------------------------------------------------- generator


def test_generator_poisons_only_unowned_slots(oracle_mod):
    case = gi.make_case(3, 4, 2, 16, [5, 16, 33], "f32", seed=3)
    pool = case.k_cache.numpy()
    dense = oracle_mod.gather_dense(pool, case.block_table.numpy(), case.context_lens.numpy(),
                                    case.stride_block, case.stride_head, case.stride_token, 2, 16)
    for b, L in enumerate([5, 16, 33]):
        assert np.isfinite(dense[b, :L]).all()
    owned = 5 + 16 + 33
    assert np.count_nonzero(~np.isnan(pool)) == owned * 2 * 16


@pytest.mark.parametrize("dtype,code_lo,code_hi,s_lo,s_hi", [
    ("i8", -127, 127, 0.015, 0.035), ("fp8", -448.0, 448.0, 0.006, 0.010),
    ("i4", -7, 7, 0.35, 0.50), ("i4kc", -7, 7, 0.35, 0.50),
])
def test_generator_recipe(oracle_mod, dtype, code_lo, code_hi, s_lo, s_hi):
    """The seeded inputs are what the input recipe states: a shuffled table that
    hands every physical block to one sequence, codes and scales in the stated
    ranges, NaN scales on the slots no sequence holds, and the same case for
    the same seed."""
    lens = [5, 16, 33, 0]
    case = gi.make_case(4, 8, 2, 128, lens, dtype, seed=7)
    table = case.block_table.numpy()
    owned = table[table >= 0]
    assert sorted(owned.tolist()) == list(range(case.num_blocks))    # each block exactly once
    assert not np.array_equal(owned, np.sort(owned))                  # and shuffled
    if dtype in ("i4", "i4kc"):
        codes = oracle_mod.unpack_int4(case.v_cache.numpy())
    elif dtype == "fp8":
        codes = oracle_mod.e4m3_to_f64(case.v_cache.view(torch.uint8).numpy())
    else:
        codes = case.v_cache.numpy()
    assert codes.min() >= code_lo and codes.max() <= code_hi
    vs = case.v_scale.float().numpy()
    held = oracle_mod.gather_scales(vs, table, np.array(lens), 2)
    for b, L in enumerate(lens):
        assert np.isfinite(held[b, :L]).all()
        assert ((held[b, :L] >= s_lo - 1e-3) & (held[b, :L] <= s_hi + 1e-3)).all()
    assert np.isnan(vs).sum() == (case.num_blocks * 16 - sum(lens)) * 2     # the rest are poisoned
    again = gi.make_case(4, 8, 2, 128, lens, dtype, seed=7)
    for x, y in ((case.q, again.q), (case.k_cache, again.k_cache), (case.v_scale, again.v_scale)):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))


@pytest.mark.parametrize("dtype", ["i8", "fp8", "i4", "i4kc"])
def test_generator_normal_source_recipe(dtype):
    """source="normal": unquantised K/V rows N(0, 1) in fp32, one per cached
    token, packed by sequence; the cache itself is left for the consumer to
    fill (codes zero, every scale NaN), and the same seed gives the same rows."""
    lens = [5, 16, 33, 0, 300]
    case = gi.make_case(5, 8, 2, 128, lens, dtype, seed=9, source="normal")
    assert case.k_src.shape == (sum(lens), 2, 128) and case.k_src.dtype == torch.float32
    assert case.v_src.shape == case.k_src.shape
    assert case.src_start.tolist() == [0, 5, 21, 54, 54, 354]
    for src in (case.k_src, case.v_src):
        assert abs(float(src.mean())) < 0.02 and abs(float(src.std()) - 1.0) < 0.02
    assert not torch.equal(case.k_src, case.v_src)
    assert not case.k_cache.view(torch.uint8).any() and not case.v_cache.view(torch.uint8).any()
    assert torch.isnan(case.k_scale).all() and torch.isnan(case.v_scale).all()
    again = gi.make_case(5, 8, 2, 128, lens, dtype, seed=9, source="normal")
    assert torch.equal(case.k_src, again.k_src) and torch.equal(case.v_src, again.v_src)
    wl = gi.WORKLOADS["int8kv_b128_ragged"]
    assert wl.source == "normal" and wl.cache_dtype == "i8"


def test_quantised_sequence_per_token_rules(oracle_mod):
    """Rows of one sequence quantise independently by the per-token rules: each
    row's largest magnitude lands on the top code (+-127, +-448, +-7) and every
    value is within half a step of its input."""
    rng = np.random.default_rng(51)
    x = rng.standard_normal((21, 3, 64)).astype(np.float32)
    for dtype, top in (("i8", 127), ("fp8", 448), ("i4", 7)):
        vals, codes, sbits = oracle_mod.quantised_sequence(x, dtype)
        assert vals.shape == x.shape and sbits.shape == (21, 3)
        s = oracle_mod.f16_bits_value(sbits)
        assert np.all(s > 0)
        arg = np.abs(x).argmax(axis=-1)
        top_vals = np.take_along_axis(vals, arg[..., None], -1)[..., 0]
        np.testing.assert_allclose(np.abs(top_vals), top * s, rtol=0, atol=0)
        if dtype == "fp8":
            # e4m3 spacing near |x|/s is at most 2^-3 of it: relative error <= 1/16
            assert np.all(np.abs(vals - x) <= np.abs(x) / 16 + s[..., None] * 2.0 ** -9)
        else:
            assert np.all(np.abs(vals - x) <= s[..., None] / 2 * (1 + 1e-3))


def test_quantised_sequence_per_channel_matches_token_by_token_appends(oracle_mod):
    """The KIVI-style K written from position 0 in one go equals 37 single-token
    appends through a shuffled pool (the last block left partial): same codes,
    same per-(block, channel) scales."""
    rng = np.random.default_rng(52)
    K, d, L = 2, 8, 37
    x = rng.standard_normal((L, K, d)).astype(np.float32)
    _, codes, sbits = oracle_mod.quantised_sequence(x, "i4kc", per_channel=True)
    assert codes.shape == (L, K, d) and sbits.shape == (3, K, d)
    table = np.array([[5, 0, 2]], dtype=np.int32)
    sb_, sh_, st_ = K * 16 * d, 16 * d, d
    pool = np.zeros(6 * sb_ // 2, dtype=np.uint8)
    scales = np.zeros((6, K, d), dtype=np.uint16)
    resid = np.zeros((1, K, 16, d), dtype=np.float32)
    for pos in range(L):
        oracle_mod.append_int4_channels(pool, scales, resid, [x[pos:pos + 1]], table, [pos], [1],
                                        sb_, sh_, st_)
    dense = oracle_mod.gather_dense(pool, table, [L], sb_ // 2, sh_ // 2, st_ // 2, K, d // 2)[0]
    np.testing.assert_array_equal(oracle_mod.unpack_int4(dense), codes)
    np.testing.assert_array_equal(scales[table[0]], sbits)


# --------------------------------------------------------------------------- fp8 (e4m3)


def test_e4m3_decoding_matches_torch_for_every_code(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle_mod.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref)) and np.isnan(mine).sum() == 2
    np.testing.assert_array_equal(mine[~np.isnan(mine)], ref[~np.isnan(ref)])
    assert oracle_mod.e4m3_to_f64(np.uint8(0x7E)) == 448.0          # largest finite value
    assert oracle_mod.e4m3_to_f64(np.uint8(0x01)) == 2.0 ** -9       # smallest subnormal


def test_e4m3_rounding_matches_torch_in_range(oracle_mod):
    rng = np.random.default_rng(41)
    x = np.concatenate([
        (rng.standard_normal(20000) * 10.0 ** rng.integers(-4, 3, 20000)).astype(np.float32),
        # exact midpoints between neighbouring codes: ties must go to the even code
        np.array([(oracle_mod.e4m3_to_f64(np.uint8(c)) + oracle_mod.e4m3_to_f64(np.uint8(c + 1))) / 2
                  for c in range(0, 0x7E)], dtype=np.float32),
    ]).clip(-460.0, 460.0)
    mine = oracle_mod.f32_to_e4m3(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(mine, ref)
    # beyond the range the reading saturates to +-448
    assert oracle_mod.f32_to_e4m3(np.float32(1e6)) == 0x7E
    assert oracle_mod.f32_to_e4m3(np.float32(-1e6)) == 0xFE


def test_fp8_quantisation_invariants(oracle_mod):
    rng = np.random.default_rng(42)
    x = rng.standard_normal((300, 128)).astype(np.float32) * np.float32(10.0) ** rng.integers(-2, 3, (300, 1))
    codes, sbits = oracle_mod.quantize_fp8(x)
    s = oracle_mod.f16_bits_to_f64(sbits)
    vals = oracle_mod.e4m3_to_f64(codes)
    # each row's largest magnitude lands on +-448 (scale is amax/448 to fp16 precision)
    assert np.all(np.abs(vals).max(axis=1) == 448.0)
    # relative error of each element within half an e4m3 step (2^-4) above the subnormals
    recon = vals * s[:, None]
    big = np.abs(x) >= 2.0 ** -6 * s[:, None]
    assert np.all(np.abs(recon - x)[big] <= np.abs(x)[big] * 2.0 ** -4 * 1.0001)
    c2, s2 = oracle_mod.quantize_fp8(-x)
    np.testing.assert_array_equal(c2 ^ 0x80, codes)                 # sign bit only
    np.testing.assert_array_equal(s2, sbits)
    cz, sz = oracle_mod.quantize_fp8(np.zeros((1, 64), dtype=np.float32))
    assert sz[0] == 0 and not cz.any()
