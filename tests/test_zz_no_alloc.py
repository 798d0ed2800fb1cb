"""gqa_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (it keeps its split-KV scratch in a fixed array inside the
library). Checked through the C ABI against gqa_decode on the same inputs, on
two calls in a row, since every call reuses the same scratch array: both
entry points run the same kernels on the same partition, so the outputs must
agree bit for bit. Collected
last on purpose: it must pass alone in a fresh process and after the rest."""
import ctypes

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


def _noalloc_raw(gq, case, out):
    """Call the C entry point directly with ctypes (no Python-side allocation)."""
    lib = gq.load()
    desc = gq.cache_from_case(case).desc()
    B, H, _ = case.q.shape
    return lib.gqa_decode_noalloc(ctypes.byref(desc), case.q.data_ptr(), gq.DTYPE_CODE[case.q.dtype],
                                  H, case.block_table.data_ptr(), int(case.block_table.shape[1]),
                                  case.context_lens.data_ptr(), B, float(case.scale), out.data_ptr(),
                                  gq.DTYPE_CODE[out.dtype], None, None,
                                  torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("cache_dtype", ["bf16", "i8"])
def test_noalloc_matches_workspace_decode_on_two_calls(gq, cache_dtype):
    lens = [4096, 17, 1, 2500, 0, 900, 3333, 64]
    case = gi.make_case(len(lens), 64, 8, 128, lens, cache_dtype, q_dtype="bf16", seed=41,
                        device="cuda")
    ref = gq.gqa_decode(gq.cache_from_case(case), case.q, case.block_table, case.context_lens,
                        case.scale)
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _noalloc_raw(gq, case, out) == 0
        torch.cuda.synchronize()
        # same kernels, same partition, same split slots: the same bits
        assert torch.equal(out, ref)


def test_noalloc_rejects_shapes_beyond_its_scratch(gq):
    # 8191 sequences x 8 kv-heads x 8 heads of partials do not fit in the built-in array
    B = 8191
    lens = [16] * B
    case = gi.make_case(B, 64, 8, 128, lens, "bf16", seed=42, device="cuda", poison=False)
    out = torch.empty((B, 64, 128), device="cuda")
    assert _noalloc_raw(gq, case, out) == 3          # GQA_ERR_WORKSPACE
