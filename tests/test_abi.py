"""The C-ABI library builds, loads and exports every function include/gqa_decode.h
declares; host-side logic and argument checks answer without a GPU (every case
here fails validation before any CUDA call, or needs none)."""
import ctypes
import os
import re

import pytest

import gqa_decode_attention_kv_gb300 as gq
from gqa_decode_attention_kv_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa_decode.h")

OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gq.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert "gqa_decode" in names and "gqa_kv_append" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in the header but not exported"


def test_library_exports_nothing_else():
    out = os.popen(f"nm -D --defined-only {gbuild.LIB_PATH}").read()
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert exported == set(declared_functions())


def test_status_strings_and_version(lib):
    assert gq.status_string(0) == "ok"
    assert "unsupported" in gq.status_string(2)
    assert gq.status_string(999) == "unknown status"
    assert gq.version() >= 100


def test_pool_elements_match_the_kv_size_closed_form(lib, oracle_mod):
    # Llama-2-70B: 80 layers x 2048 tokens = 128 blocks per layer at batch 1
    blocks = 80 * oracle_mod.blocks_for_tokens(2048)
    mha = gq.kv_pool_elements(blocks, 64, 128)
    gqa = gq.kv_pool_elements(blocks, 8, 128)
    assert mha == oracle_mod.kv_cache_elements(80, 64, 128, 2048, 1) == 2_684_354_560
    assert gqa == oracle_mod.kv_cache_elements(80, 8, 128, 2048, 1) == 335_544_320
    assert gq.kv_pool_elements(-1, 8, 128) == -1


def _desc(**kw):
    base = dict(k=0x10000, v=0x20000, k_scale=None, v_scale=None, num_blocks=64, num_kv_heads=8,
                block_size=16, head_dim=128, dtype=2, stride_block=8 * 16 * 128,
                stride_head=16 * 128, stride_token=128)
    base.update(kw)
    return gq.KVCacheDesc(**base)


def _decode(lib, desc, q=0x30000, q_dtype=2, H=32, table=0x40000, maxb=8, lens=0x50000, B=4,
            scale=0.1, out=0x60000, out_dtype=0, ws=0x70000, ws_bytes=1 << 20, T=0, window=0,
            layout=0):
    opts = gq.DecodeOpts(T, window, 0, 0, 0, layout, None, None)
    return lib.gqa_decode(ctypes.byref(desc), q, q_dtype, H, table, maxb, lens, B, scale, out,
                          out_dtype, ws, ws_bytes, ctypes.byref(opts), None, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(k=None), INVALID),
    (dict(block_size=32), UNSUPPORTED),
    (dict(head_dim=96), UNSUPPORTED),
    (dict(dtype=7), INVALID),
    (dict(k=0x10008), INVALID),                      # not 16-byte aligned
    (dict(stride_token=100), INVALID),               # shorter than a row
    (dict(stride_head=16 * 128 + 4), INVALID),       # 8 bytes: not a multiple of 16 bytes
    (dict(dtype=3), INVALID),                        # int8 cache without scales
    (dict(num_blocks=0), INVALID),
])
def test_cache_description_checks(lib, kw, expect):
    assert _decode(lib, _desc(**kw)) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(H=30), INVALID),                           # H not a multiple of K
    (dict(H=8 * 128), UNSUPPORTED),                  # G = 128 > 64
    (dict(B=9000), UNSUPPORTED),
    (dict(q=0x30004), INVALID),
    (dict(ws=0x70010), INVALID),                     # workspace not 256-byte aligned
    (dict(q_dtype=1), UNSUPPORTED),                  # fp16 q against a bf16 cache
    (dict(out_dtype=3), UNSUPPORTED),
    (dict(scale=float("nan")), INVALID),
    (dict(out=None), INVALID),
    (dict(B=0), OK),                                 # empty batch: nothing to launch
    (dict(T=-1), INVALID),
    (dict(window=-5), INVALID),
    (dict(T=17), UNSUPPORTED),                       # G*T = 4*17 = 68 query rows > 64
    (dict(T=16, B=0), OK),                           # 64 rows: allowed
    (dict(window=7, B=0), OK),
    (dict(layout=3), INVALID),
])
def test_decode_argument_checks(lib, kw, expect):
    assert _decode(lib, _desc(), **kw) == expect


def test_append_argument_checks(lib):
    d = _desc()
    f = lib.gqa_kv_append
    assert f(ctypes.byref(d), 0x1000, 0x2000, 2, 0x3000, 8, 0x4000, 0, 1, None, None) == OK
    assert f(ctypes.byref(d), 0x1004, 0x2000, 2, 0x3000, 8, 0x4000, 4, 1, None, None) == INVALID
    assert f(ctypes.byref(d), 0x1000, 0x2000, 0, 0x3000, 8, 0x4000, 4, 1, None, None) == UNSUPPORTED
    assert f(ctypes.byref(d), None, 0x2000, 2, 0x3000, 8, 0x4000, 4, 1, None, None) == INVALID
    assert f(ctypes.byref(d), 0x1000, 0x2000, 2, 0x3000, 8, 0x4000, 4, -1, None, None) == INVALID
    i8 = _desc(dtype=3, k_scale=0x80000, v_scale=0x90000)
    assert f(ctypes.byref(i8), 0x1000, 0x2000, 3, 0x3000, 8, 0x4000, 4, 1, None, None) == UNSUPPORTED


def test_kivi_cache_appends_need_the_residual(lib):
    """GQA_DTYPE_I4_KC: appends read and write k_residual (one row per batch
    row); a missing, misaligned or too short residual is refused before any
    launch, by both append entry points."""
    base = dict(dtype=6, k_scale=0x80000, v_scale=0x90000)
    f, fv = lib.gqa_kv_append, lib.gqa_kv_append_varlen
    for kw in (dict(), dict(k_residual=0xA0008, residual_rows=4), dict(k_residual=0xA0000, residual_rows=3)):
        d = _desc(**base, **kw)
        assert f(ctypes.byref(d), 0x1000, 0x2000, 2, 0x3000, 8, 0x4000, 4, 1, None, None) == INVALID
        assert fv(ctypes.byref(d), 0x1000, 0x2000, 2, 0x5000, 3, 0x3000, 8, 0x4000, 4, None, None) == INVALID
    # an empty batch needs no residual
    d = _desc(**base)
    assert f(ctypes.byref(d), 0x1000, 0x2000, 2, 0x3000, 8, 0x4000, 0, 1, None, None) == OK


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(gq, "_lib", None)
    monkeypatch.setattr(gbuild, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        gq.load()


def test_binding_rejects_arrays_the_library_cannot_read():
    """The C ABI sees bare pointers; the binding refuses what they cannot
    describe: strided views, index arrays that are not int32, host memory."""
    import torch
    with pytest.raises(ValueError, match="contiguous"):
        gq._dev(torch.zeros(4, 6).t(), "q")
    with pytest.raises(ValueError, match="int32"):
        gq._dev(torch.zeros(4, dtype=torch.int64), "context_lens", index=True)
    with pytest.raises(ValueError, match="dtype"):
        gq._dev(torch.zeros(4, dtype=torch.float64), "q")
    with pytest.raises(ValueError, match="CUDA"):
        gq._dev(torch.zeros(4, dtype=torch.int32), "context_lens", index=True)
    with pytest.raises(ValueError, match="required"):
        gq._dev(None, "q")
    assert gq._dev(None, "err", index=True, optional=True) is None
    # the public calls check before they touch the cache or the library
    q = torch.zeros(3, 8, 64, dtype=torch.bfloat16)
    lens = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        gq.gqa_prefill(None, q, lens, 3, lens.reshape(1, 1), lens, 0.125)
    with pytest.raises(ValueError, match="contiguous"):
        gq.gqa_decode(None, q.transpose(0, 1), lens.reshape(1, 1), lens, 0.125)
    with pytest.raises(ValueError, match="contiguous"):
        gq.kv_append(None, q.transpose(0, 1), q, lens.reshape(1, 1), lens)


def _cpu_cache(K=2, d=64, nb=4):
    import torch
    k = torch.zeros(nb, K, 16, d, dtype=torch.bfloat16)
    return gq.PagedKVCache(k, k.clone(), nb, K, d, K * 16 * d, 16 * d, d)


def test_binding_rejects_a_query_the_cache_cannot_serve():
    """The library takes head_dim from the cache and the batch from q, so a q
    of another head_dim, or a head count that is not a multiple of the
    kv-heads, would be read out of bounds: refused before any call."""
    import torch
    cache = _cpu_cache()
    gq._check_query(cache, torch.zeros(3, 8, 64), (3, 4))           # fits
    with pytest.raises(ValueError, match="head_dim"):
        gq._check_query(cache, torch.zeros(3, 8, 128), (3, 4))
    with pytest.raises(ValueError, match="multiple"):
        gq._check_query(cache, torch.zeros(3, 7, 64), (3, 4))
    with pytest.raises(ValueError, match="dims"):
        gq._check_query(cache, torch.zeros(3, 2, 8, 64), (3,))


def test_binding_rejects_short_tables_and_lengths():
    import torch
    lens = torch.zeros(4, dtype=torch.int32)
    gq._check_table_and_lens(torch.zeros(4, 9, dtype=torch.int32), lens, 4, "context_lens", 4)
    with pytest.raises(ValueError, match="block_tables"):
        gq._check_table_and_lens(torch.zeros(3, 9, dtype=torch.int32), lens, 4, "context_lens", 4)
    with pytest.raises(ValueError, match="block_tables"):
        gq._check_table_and_lens(torch.zeros(36, dtype=torch.int32), lens, 4, "context_lens", 4)
    with pytest.raises(ValueError, match="context_lens"):
        gq._check_table_and_lens(torch.zeros(4, 9, dtype=torch.int32), lens[:3], 4, "context_lens", 4)
    with pytest.raises(ValueError, match="q_start|positions"):
        gq._check_table_and_lens(torch.zeros(4, 9, dtype=torch.int32), lens, 4, "positions", 5)


def test_binding_rejects_an_output_of_another_shape():
    import torch
    q = torch.zeros(3, 8, 64)
    gq._check_out(q, None)
    gq._check_out(q, torch.zeros(3, 8, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="out"):
        gq._check_out(q, torch.zeros(3, 8, 32))


def test_binding_rejects_new_rows_of_another_shape():
    import torch
    cache = _cpu_cache()
    x = torch.zeros(5, 2, 64)
    gq._check_new_rows(cache, x, x.clone(), (3, 4))
    with pytest.raises(ValueError, match="share one shape"):
        gq._check_new_rows(cache, x, torch.zeros(5, 2, 32), (3, 4))
    with pytest.raises(ValueError, match="heads and head_dim"):
        gq._check_new_rows(cache, torch.zeros(5, 4, 64), torch.zeros(5, 4, 64), (3, 4))
    with pytest.raises(ValueError, match="dims"):
        gq._check_new_rows(cache, torch.zeros(5, 1, 2, 64), torch.zeros(5, 1, 2, 64), (3,))


def test_binding_rejects_arrays_on_another_device():
    """Every array must sit where the cache is (meta tensors stand in for a
    second device here)."""
    import torch
    cache = _cpu_cache()
    gq._on_cache_device(cache, q=torch.zeros(2), err=None)
    with pytest.raises(ValueError, match="q is on meta"):
        gq._on_cache_device(cache, q=torch.zeros(2, device="meta"))
