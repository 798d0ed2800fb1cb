"""Host arithmetic of the benchmark: the bytes and flops that roofline.achieved
divides by, checked against hand counts, and the gate that keeps an ncu traffic
figure to the kernel source it was taken on."""
import dataclasses

import bench
import gqa_inputs as gi


def _one_head(name, **kw):
    return dataclasses.replace(gi.WORKLOADS[name], num_heads=1, num_kv_heads=1, **kw)


def test_default_decode_bytes_hand_count():
    wl = gi.WORKLOADS["llama3_8b_bf16_b64_s4096"]
    B, S, H, K, d = 64, 4096, 32, 8, 128
    kv = B * S * 2 * K * d * 2            # K and V rows, bf16, every cached token once
    q = B * H * d * 2                     # bf16 queries in
    o = B * H * d * 4                     # fp32 output out
    meta = B * (S // 16) * 4 + B * 4      # one table entry per block, one length per sequence
    got = bench.algorithmic_bytes(wl, [S] * B)
    assert got["kv"] == kv
    assert got["blocks"] == B * S // 16
    assert got["decode"] == kv + q + o + meta == 1075380480


def test_window_counts_only_the_band():
    # L = 100, W = 37: positions 63..99, in blocks 3..6
    wl = _one_head("mistral7b_swa_bf16_b64_s16384_w4096", window=37)
    got = bench.algorithmic_bytes(wl, [100])
    assert got["tokens"] == 37
    assert got["blocks"] == 4
    assert got["kv"] == 37 * 2 * 128 * 2


def test_code_cache_scale_bytes():
    # int8: codes of K and V plus one fp16 scale each per token
    i8 = _one_head("int8kv_b128_ragged")
    assert bench.algorithmic_bytes(i8, [40])["kv"] == 40 * (2 * 128 + 2 * 2)
    # KIVI-style INT4: half-byte codes, a V scale per token, d K scales per block
    kc = _one_head("int4kc_b128_ragged")
    assert bench.algorithmic_bytes(kc, [40])["kv"] == 40 * (128 + 2) + 3 * 128 * 2


def test_prefill_flops_closed_forms():
    wl = gi.WORKLOADS["llama3_8b_prefill_bf16_b8_p2048"]
    T, H, d = 2048, 32, 128
    # fresh prompts: row i attends i + 1 positions, 4 d flops per head and position
    assert bench.prefill_flops(wl, [T] * 8) == 4 * d * H * 8 * T * (T + 1) // 2 == 275012124672
    # a 30-token window over a fresh 100-token prompt: rows 0..29 attend i + 1, the rest 30
    w = dataclasses.replace(wl, queries=100, window=30)
    assert bench.prefill_flops(w, [100]) == 4 * d * H * (30 * 31 // 2 + 70 * 30)
    # 100 new tokens after 50 cached ones: row i attends 51 + i
    w2 = dataclasses.replace(wl, queries=100)
    assert bench.prefill_flops(w2, [150]) == 4 * d * H * sum(51 + i for i in range(100))


def test_traffic_is_read_only_for_the_source_it_was_taken_on(tmp_path):
    src = bench.kernel_source_hash()
    f = tmp_path / "traffic.txt"
    f.write_text(
        "# comment: ignored\n"
        f"workload: w\nkernel_variant: auto\nsource_hash: {src}\ntraffic_bytes_per_launch: 123\n\n"
        "workload: w2\nkernel_variant: auto\nsource_hash: 0000000000000000\n"
        "traffic_bytes_per_launch: 456\n")
    assert bench.read_traffic("w", "auto", str(f)) == 123.0
    assert bench.read_traffic("w2", "auto", str(f)) is None     # taken on other sources
    assert bench.read_traffic("w", "1", str(f)) is None         # another kernel variant
    assert bench.read_traffic("other", "auto", str(f)) is None
    assert bench.read_traffic("w", "auto", str(tmp_path / "missing.txt")) is None
    # the prefill kernel's figure is keyed to its own sources
    assert bench.read_traffic("w", "auto", str(f), bench.PREFILL_SOURCES) is None


def test_oracle_inputs_follow_the_cache_layout(oracle_mod):
    """The CPU baseline gathers its sequences from the cache block by block: on
    the un-paged [B, S_pad, K, d] buffer and on a paged pool alike it must hand
    the oracle the same inputs the parity tests build (so the same output)."""
    import numpy as np
    from helpers import oracle_for_case
    wl = gi.WORKLOADS["tiny_f32_contiguous"]
    case = gi.case_for(wl, seed=0, device="cpu", extra_tokens=0)
    q, kd, vd, sl = bench._oracle_inputs(wl, case, [0, 1])
    np.testing.assert_array_equal(oracle_mod.decode(q, kd, vd, sl, case.scale), oracle_for_case(case))
    paged = dataclasses.replace(wl, cache_dtype="bf16", q_dtype="bf16", contiguous=False, batch=3)
    case = gi.make_case(3, 8, 2, 64, [20, 33, 5], "bf16", seed=3)
    q, kd, vd, sl = bench._oracle_inputs(paged, case, [0, 2])
    np.testing.assert_array_equal(oracle_mod.decode(q, kd, vd, sl, case.scale),
                                  oracle_for_case(case, rows=[0, 2]))
