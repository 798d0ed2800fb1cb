"""Paged prefill on the GPU against the fp64 oracle, through the C ABI.

Prefill ("LLM 推理性能优化实战" sections 9.2-9.4) is the multi-token decode
definition with T = the prompt length: the n_b new tokens of sequence b sit at
positions L_b - n_b .. L_b - 1 and attend causally to the cache (optionally the
last W positions). The oracle runs that definition per sequence. Bar: max-abs
2e-3 on fp32 output; the varlen append is bit-exact against the host scatter."""
import numpy as np
import pytest
import torch

import gqa_inputs as gi
from helpers import TOL, max_abs_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    from gqa_decode_attention_kv_gb300 import build
    build.build()
    import gqa_decode_attention_kv_gb300 as m
    return m


def _case(lens, news, H, K, d, dtype, seed):
    """A paged cache holding lens[b] tokens per sequence (the last news[b] of
    them the prompt's) and the prompts' queries, packed [total, H, d]."""
    case = gi.make_case(len(lens), H, K, d, lens, dtype, seed=seed, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(seed + 1000)
    total = int(sum(news))
    q = torch.randn((total, H, d), generator=g, device="cuda").to(gi.DTYPES[dtype])
    q_start = torch.tensor(np.concatenate([[0], np.cumsum(news)]), dtype=torch.int32, device="cuda")
    return case, q, q_start


def _reference(oracle_mod, case, q, news, window=0):
    """fp64 oracle rows [total, H, d]: sequence by sequence, T = news[b]."""
    kp = case.k_cache.detach().float().cpu().numpy()
    vp = case.v_cache.detach().float().cpu().numpy()
    table = case.block_table.cpu().numpy()
    lens = case.context_lens.cpu().numpy()
    qh = q.detach().float().cpu().numpy().astype(np.float64)
    out, row = [], 0
    for b, n in enumerate(news):
        kd = oracle_mod.gather_dense(kp, table, lens, case.stride_block, case.stride_head,
                                     case.stride_token, case.num_kv_heads, case.head_dim, [b])
        vd = oracle_mod.gather_dense(vp, table, lens, case.stride_block, case.stride_head,
                                     case.stride_token, case.num_kv_heads, case.head_dim, [b])
        if n:
            o = oracle_mod.decode(qh[row:row + n][None], kd, vd, [lens[b]], case.scale, window=window)
            out.append(o[0])
        row += n
    return np.concatenate(out) if out else np.zeros((0,) + q.shape[1:])


def _run(gq, case, q, q_start, news, **kw):
    out = gq.gqa_prefill(gq.cache_from_case(case), q, q_start, max(news), case.block_table,
                         case.context_lens, case.scale, **kw)
    torch.cuda.synchronize()
    return out


KERNELS = [3, 4, 1, 2]   # tcgen05 two-tile and its one-tile-per-CTA twin (head_dim 128; 64 takes the
                         # 32-token form), tcgen05 32-token one-tile, mma.sync


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("H,K,d", [(32, 8, 128), (8, 8, 128), (64, 4, 128), (16, 4, 64), (8, 1, 64)])
def test_prefill_mixed_prompts(gq, oracle_mod, dtype, H, K, d, kernel):
    news = [1, 5, 16, 17, 64, 100, 33]
    prior = [0, 7, 40, 0, 500, 3, 16]
    lens = [n + p for n, p in zip(news, prior)]
    case, q, q_start = _case(lens, news, H, K, d, dtype, seed=81)
    ref = _reference(oracle_mod, case, q, news)
    assert max_abs_err(_run(gq, case, q, q_start, news, kernel=kernel), ref) <= TOL


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("window", [1, 16, 37, 200])
def test_prefill_sliding_window(gq, oracle_mod, window, kernel):
    news = [3, 64, 129, 300]
    prior = [10, 0, 77, 256]
    lens = [n + p for n, p in zip(news, prior)]
    case, q, q_start = _case(lens, news, 32, 8, 128, "bf16", seed=82)
    ref = _reference(oracle_mod, case, q, news, window=window)
    assert max_abs_err(_run(gq, case, q, q_start, news, window=window, kernel=kernel), ref) <= TOL


@pytest.mark.parametrize("kernel", KERNELS)
def test_prefill_long_prompt_and_empty_sequences(gq, oracle_mod, kernel):
    news = [0, 1000, 0, 513]
    lens = [5, 1000, 0, 1030]
    case, q, q_start = _case(lens, news, 32, 8, 128, "bf16", seed=83)
    ref = _reference(oracle_mod, case, q, news)
    assert max_abs_err(_run(gq, case, q, q_start, news, kernel=kernel), ref) <= TOL


@pytest.mark.parametrize("kernel", [3, 4])
@pytest.mark.parametrize("H,K", [(48, 8), (96, 2), (64, 1), (128, 1)])
def test_prefill_group_sizes(gq, oracle_mod, H, K, kernel):
    """G = 6 and 48 (a warp's 32 rows are not whole tokens: the 64-token forms
    store them row by row) and G = 64 and 128 (each warp's rows are 32 heads
    of one token: stored as one box per 16 columns), ragged prompts."""
    news = [1, 40, 130, 7]
    prior = [0, 9, 33, 100]
    lens = [n + p for n, p in zip(news, prior)]
    case, q, q_start = _case(lens, news, H, K, 128, "bf16", seed=95)
    ref = _reference(oracle_mod, case, q, news)
    assert max_abs_err(_run(gq, case, q, q_start, news, kernel=kernel), ref) <= TOL


@pytest.mark.parametrize("kernel", [3, 4])
def test_prefill_many_items_per_persistent_cta(gq, oracle_mod, kernel):
    """40 ragged prompts (0..300 new tokens over 0..70 cached ones). The
    64-token forms' persistent CTAs (one or two per SM) deal out 1600 or 3200
    (query tile, kv-head, sequence) items, so every CTA walks several of them,
    skips those past a short prompt's end, and carries its barrier phases and
    stage ring from one item to the next."""
    rng = np.random.default_rng(91)
    news = rng.integers(0, 301, size=40).tolist()
    news[5], news[17] = 0, 300
    prior = rng.integers(0, 71, size=40).tolist()
    lens = [n + p for n, p in zip(news, prior)]
    case, q, q_start = _case(lens, news, 32, 8, 128, "bf16", seed=93)
    ref = _reference(oracle_mod, case, q, news)
    assert max_abs_err(_run(gq, case, q, q_start, news, kernel=kernel), ref) <= TOL


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("sign", [-1.0, 0.0])
def test_prefill_negative_and_zero_scale(gq, oracle_mod, kernel, sign):
    """A negative scale flips which key dominates (the wide kernel takes the
    raw minimum then); a zero scale weights every attended position alike."""
    news = [70, 200, 1]
    lens = [90, 200, 40]
    case, q, q_start = _case(lens, news, 32, 8, 128, "bf16", seed=95)
    case.scale = sign * case.scale
    ref = _reference(oracle_mod, case, q, news)
    assert max_abs_err(_run(gq, case, q, q_start, news, kernel=kernel), ref) <= TOL


def test_prefill_kernels_agree_on_large_scores(gq, oracle_mod):
    """Scores spread over hundreds of log2 units: the lazy rescale of the tensor-
    memory accumulator has to fire; both kernels match the oracle."""
    news = [130, 257]
    lens = [130, 300]
    case, q, q_start = _case(lens, news, 16, 4, 128, "bf16", seed=89)
    q = (q.float() * 40.0).to(torch.bfloat16)
    ref = _reference(oracle_mod, case, q, news)
    for kernel in KERNELS:
        assert max_abs_err(_run(gq, case, q, q_start, news, kernel=kernel), ref) <= TOL, kernel


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_prefill_half_outputs(gq, oracle_mod, out_dtype):
    news = [20, 70]
    lens = [25, 90]
    case, q, q_start = _case(lens, news, 32, 8, 128, "bf16", seed=84)
    ref = _reference(oracle_mod, case, q, news)
    out = _run(gq, case, q, q_start, news, out_dtype=out_dtype)
    got = out.float().cpu().numpy().astype(np.float64)
    ulp = np.abs(ref) * (2.0 ** -8 if out_dtype == torch.bfloat16 else 2.0 ** -11)
    assert np.all(np.abs(got - ref) <= TOL + ulp)


def test_prefill_last_token_equals_decode(gq, oracle_mod):
    """The last prompt token attends the whole cache: a one-token decode of it."""
    news = [50, 200]
    lens = [60, 200]
    case, q, q_start = _case(lens, news, 32, 8, 128, "bf16", seed=85)
    out = _run(gq, case, q, q_start, news)
    last = torch.stack([q[int(q_start[b + 1]) - 1] for b in range(2)])
    one = gq.gqa_decode(gq.cache_from_case(case), last, case.block_table, case.context_lens, case.scale)
    torch.cuda.synchronize()
    got = torch.stack([out[int(q_start[b + 1]) - 1] for b in range(2)])
    assert (got - one).abs().max().item() <= 2e-5


def test_varlen_append_then_prefill(gq, oracle_mod):
    """Write each prompt's K/V with the varlen append (bit-exact), then prefill."""
    news = [7, 40, 0, 33]
    prior = [0, 20, 9, 100]
    lens = list(prior)
    case = gi.make_case(len(lens), 16, 4, 128, lens, "bf16", seed=86, device="cuda",
                        extra_tokens=max(news))
    g = torch.Generator(device="cuda").manual_seed(87)
    total = sum(news)
    kn = torch.randn((total, 4, 128), generator=g, device="cuda").to(torch.bfloat16)
    vn = torch.randn((total, 4, 128), generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn((total, 16, 128), generator=g, device="cuda").to(torch.bfloat16)
    starts = torch.tensor(np.concatenate([[0], np.cumsum(news)]), dtype=torch.int32, device="cuda")
    before_k = case.k_cache.detach().cpu().view(torch.int16).numpy().reshape(-1).copy()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache = gq.cache_from_case(case)
    gq.kv_append_varlen(cache, kn, vn, starts, max(news), case.block_table, case.context_lens.clone(),
                        err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    table = case.block_table.cpu().numpy()
    kh = kn.cpu().view(torch.int16).numpy()
    row = 0
    for b, n in enumerate(news):
        for i in range(n):
            oracle_mod.append(before_k, kh[row + i][None], table[b:b + 1], [prior[b] + i],
                              case.stride_block, case.stride_head, case.stride_token)
        row += n
    assert np.array_equal(case.k_cache.detach().cpu().view(torch.int16).numpy().reshape(-1), before_k)
    case.context_lens += torch.tensor(news, dtype=torch.int32, device="cuda")
    ref = _reference(oracle_mod, case, q, news)
    out = gq.gqa_prefill(cache, q, starts, max(news), case.block_table, case.context_lens, case.scale,
                         err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert max_abs_err(out, ref) <= TOL


def test_prefill_flags_bad_lengths(gq):
    news = [10, 10]
    lens = [20, 20]
    case, q, q_start = _case(lens, news, 8, 2, 128, "bf16", seed=88)
    bad = case.context_lens.clone()
    bad[1] = 5                                   # fewer cached tokens than new ones
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gq.gqa_prefill(gq.cache_from_case(case), q, q_start, 10, case.block_table, bad, case.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & gq.GQA_DEVERR_CONTEXT_LEN


def test_full_size_prefill_workload_sampled(gq, oracle_mod):
    """The bench's prefill workload in its launch configuration; the last 24
    prompt tokens of two sequences against the oracle."""
    wl = gi.WORKLOADS["llama3_8b_prefill_bf16_b8_p2048"]
    case = gi.case_for(wl, seed=0, device="cuda")
    B, T, H, d = wl.batch, wl.queries, wl.num_heads, wl.head_dim
    q = case.q.reshape(B * T, H, d)
    starts = torch.arange(0, B * T + 1, T, dtype=torch.int32, device="cuda")
    out = gq.gqa_prefill(gq.cache_from_case(case), q, starts, T, case.block_table, case.context_lens,
                         case.scale)
    torch.cuda.synchronize()
    kp = case.k_cache.float().cpu().numpy()
    vp = case.v_cache.float().cpu().numpy()
    table = case.block_table.cpu().numpy()
    lens = case.context_lens.cpu().numpy()
    for b in (0, B - 1):
        kd = oracle_mod.gather_dense(kp, table, lens, case.stride_block, case.stride_head,
                                     case.stride_token, wl.num_kv_heads, d, [b])
        vd = oracle_mod.gather_dense(vp, table, lens, case.stride_block, case.stride_head,
                                     case.stride_token, wl.num_kv_heads, d, [b])
        qb = q[b * T:(b + 1) * T].float().cpu().numpy().astype(np.float64)
        # the last 24 queries: T' = 24 new tokens at the end of the same context
        ref = oracle_mod.decode(qb[T - 24:][None], kd, vd, [lens[b]], case.scale)[0]
        got = out[b * T + T - 24:(b + 1) * T].float().cpu().numpy().astype(np.float64)
        assert np.abs(got - ref).max() <= TOL


@pytest.mark.parametrize("kernel", KERNELS)
def test_prefill_on_the_unpaged_layout(gq, oracle_mod, kernel):
    """The contiguous [B, S_pad, K, d] buffer with an identity table: token,
    head and block strides differ from the pool's, and the page copies follow."""
    news = [40, 7, 100]
    prior = [60, 0, 13]
    lens = [n + p for n, p in zip(news, prior)]
    case = gi.make_case(len(lens), 32, 8, 128, lens, "bf16", seed=90, device="cuda", contiguous=True)
    g = torch.Generator(device="cuda").manual_seed(91)
    q = torch.randn((sum(news), 32, 128), generator=g, device="cuda").to(torch.bfloat16)
    q_start = torch.tensor(np.concatenate([[0], np.cumsum(news)]), dtype=torch.int32, device="cuda")
    ref = _reference(oracle_mod, case, q, news)
    assert max_abs_err(_run(gq, case, q, q_start, news, kernel=kernel), ref) <= TOL
