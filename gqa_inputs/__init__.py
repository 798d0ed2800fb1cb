"""Seeded synthetic inputs for one GQA decode step over a paged KV cache.

This module only draws random numbers and lays them out in memory. It holds no
attention, softmax, quantisation or paging arithmetic of the method: both the
CUDA path (through the C-ABI) and the CPU oracle consume what it produces, and
neither of them is imported here.

Layouts produced (element strides, innermost last):

* paged pool ``[num_blocks, K, 16, d]`` (one 16-token tile per (block, kv-head),
  the head-before-sequence order of the cache tensor on "LLM 推理性能优化实战",
  section 5.2) with a per-sequence block table ``[B, max_blocks]`` int32 that
  maps logical block ``j`` to a physical block (section 8.2 of the same page);
  physical blocks are a seeded permutation, so neighbouring logical blocks are
  scattered through the pool;
* contiguous cache ``[B, S_pad, K, d]`` (the ``[batch, seq, num_kv_heads,
  head_dim]`` index of section 7 of that page), described to the library as a
  pool whose block stride is ``16*K*d`` with an identity block table.

Slots that no sequence owns (the tail of a sequence's last block and blocks no
table references) are filled with NaN (float caches) or with NaN scales (int8
caches), so that any read past ``context_lens`` poisons the output.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

BLOCK_SIZE = 16

# dtype names shared with the C-ABI enum (gqa_dtype_t in include/gqa_decode.h)
DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "i8": torch.int8,
          "fp8": torch.float8_e4m3fn, "i4": torch.uint8, "i4kc": torch.uint8}   # i4*: two codes per byte
DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2, "i8": 3, "fp8": 4, "i4": 5, "i4kc": 6}
# code caches with fp16 scales: per (token, kv-head); for the K of "i4kc"
# (KIVI-style) per (block, kv-head, channel)
CODED = ("i8", "fp8", "i4", "i4kc")
PACKED4 = ("i4", "i4kc")     # two 4-bit codes per byte

@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode-step workload: shapes, length recipe and storage types."""
    name: str
    batch: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    cache_dtype: str            # "f32" | "f16" | "bf16" | "i8" | "fp8" | "i4" | "i4kc"
    q_dtype: str                # "f32" | "f16" | "bf16"
    lens: str                   # "fixed:<a,b,...>" | "const:<S>" | "uniform:<lo>:<hi>"
    contiguous: bool = False    # un-paged [B, S_pad, K, d] buffer + identity table
    queries: int = 1            # new tokens per sequence (causal among themselves)
    window: int = 0             # sliding window in tokens; 0 = full attention
    kind: str = "decode"        # "decode" (gqa_decode) or "prefill" (gqa_prefill: queries = prompt)
    # code caches: "codes" = codes and scales drawn directly (ranges in make_case);
    # "normal" = K/V rows drawn N(0, 1) in fp32 and left for the consumer to
    # quantise into the cache (make_case's ``source``)
    source: str = "codes"

    @property
    def group_size(self) -> int:
        return self.num_heads // self.num_kv_heads


# The decode-step workloads. Names say what they are; sizes are the ones the
# tests and the benchmark use.
WORKLOADS = {
    "tiny_f32_contiguous": Workload("tiny_f32_contiguous", 2, 8, 2, 64, "f32", "f32",
                                    "fixed:37,100", contiguous=True),
    "llama3_8b_bf16_b64_s4096": Workload("llama3_8b_bf16_b64_s4096", 64, 32, 8, 128,
                                         "bf16", "bf16", "const:4096"),
    "llama70b_bf16_b32_ragged": Workload("llama70b_bf16_b32_ragged", 32, 64, 8, 128,
                                         "bf16", "bf16", "uniform:128:32768"),
    "long_ctx_bf16_b1_s131072": Workload("long_ctx_bf16_b1_s131072", 1, 32, 8, 128,
                                         "bf16", "bf16", "const:131072"),
    "long_ctx_bf16_b4_s131072": Workload("long_ctx_bf16_b4_s131072", 4, 32, 8, 128,
                                         "bf16", "bf16", "const:131072"),
    # K/V drawn N(0, 1), then quantised per (token, kv-head) into the cache
    "int8kv_b128_ragged": Workload("int8kv_b128_ragged", 128, 64, 8, 128, "i8", "bf16",
                                   "uniform:2048:8192", source="normal"),
    "fp8kv_b128_ragged": Workload("fp8kv_b128_ragged", 128, 64, 8, 128, "fp8", "bf16",
                                  "uniform:2048:8192", source="normal"),
    "int4kv_b128_ragged": Workload("int4kv_b128_ragged", 128, 64, 8, 128, "i4", "bf16",
                                   "uniform:2048:8192", source="normal"),
    # KIVI-style 4-bit cache (K per channel, V per token), same shape
    "int4kc_b128_ragged": Workload("int4kc_b128_ragged", 128, 64, 8, 128, "i4kc", "bf16",
                                   "uniform:2048:8192", source="normal"),
    # four new tokens per sequence (speculative verification of three drafts),
    # Llama-3-8B shape; the lengths include the new tokens
    "spec_verify_bf16_b64_s4096_t4": Workload("spec_verify_bf16_b64_s4096_t4", 64, 32, 8, 128,
                                              "bf16", "bf16", "const:4096", queries=4),
    # prefill of 8 fresh 2048-token prompts, Llama-3-8B attention shape
    "llama3_8b_prefill_bf16_b8_p2048": Workload("llama3_8b_prefill_bf16_b8_p2048", 8, 32, 8, 128,
                                                "bf16", "bf16", "const:2048", queries=2048,
                                                kind="prefill"),
    # sliding window of 4096 tokens over 16K-token contexts, Mistral-7B shape
    "mistral7b_swa_bf16_b64_s16384_w4096": Workload("mistral7b_swa_bf16_b64_s16384_w4096", 64, 32, 8,
                                                    128, "bf16", "bf16", "const:16384", window=4096),
}


def kv_sweep_workload(num_kv_heads: int) -> Workload:
    """The 70B-shaped ragged workload at H=64 with a different KV-head count
    (64 = MHA, 1 = MQA); used to show KV bytes scaling as 1/G."""
    base = WORKLOADS["llama70b_bf16_b32_ragged"]
    return dataclasses.replace(base, name=f"llama70b_bf16_b32_ragged_k{num_kv_heads}",
                               num_kv_heads=num_kv_heads)


def draw_lens(spec: str, batch: int, seed: int) -> torch.Tensor:
    """Context lengths (tokens already in the cache, including the new one)."""
    kind, _, rest = spec.partition(":")
    if kind == "fixed":
        vals = [int(x) for x in rest.split(",")]
        if len(vals) != batch:
            raise ValueError("fixed length list does not match the batch")
        return torch.tensor(vals, dtype=torch.int32)
    if kind == "const":
        return torch.full((batch,), int(rest), dtype=torch.int32)
    if kind == "uniform":
        lo, hi = (int(x) for x in rest.split(":"))
        g = torch.Generator().manual_seed(seed * 7919 + 17)
        return torch.randint(lo, hi + 1, (batch,), generator=g, dtype=torch.int32)
    raise ValueError(f"unknown length recipe {spec!r}")


@dataclasses.dataclass
class DecodeCase:
    """Everything one decode step reads, plus the new token for an append."""
    batch: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    cache_dtype: str
    q_dtype: str
    scale: float
    q: torch.Tensor                 # [B, H, d] q_dtype ([B, T, H, d] for T > 1 queries)
    k_cache: torch.Tensor           # pool or contiguous buffer, cache dtype
    v_cache: torch.Tensor
    k_scale: Optional[torch.Tensor]  # [num_blocks, K, 16] fp16 (code caches; [num_blocks, K, d] for i4kc)
    v_scale: Optional[torch.Tensor]
    num_blocks: int
    stride_block: int               # element strides of the cache description
    stride_head: int
    stride_token: int
    block_table: torch.Tensor       # [B, max_blocks] int32
    context_lens: torch.Tensor      # [B] int32, tokens valid for the decode
    k_new: torch.Tensor             # [B, K, d] new token(s) (input dtype of append; [B, T, K, d])
    v_new: torch.Tensor
    queries: int = 1                # T new tokens per sequence
    k_residual: Optional[torch.Tensor] = None   # i4kc: fp32 [B, K, 16, d], unquantised K of the open block
    # source="normal" code caches: the unquantised rows the cache is to hold,
    # fp32 [sum(lens), K, d], rows src_start[b] .. src_start[b+1]-1 being
    # positions 0 .. lens[b]-1 of sequence b (codes and scales still empty)
    k_src: Optional[torch.Tensor] = None
    v_src: Optional[torch.Tensor] = None
    src_start: Optional[torch.Tensor] = None    # [B+1] int32

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])


def _randn(shape, gen, device, dtype):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


def make_case(batch: int, num_heads: int, num_kv_heads: int, head_dim: int,
              lens: Sequence[int] | torch.Tensor, cache_dtype: str = "bf16",
              q_dtype: Optional[str] = None, seed: int = 0, device: str = "cpu",
              contiguous: bool = False, shuffle: bool = True, spare_blocks: int = 0,
              extra_tokens: int = 0, max_blocks: Optional[int] = None, poison: bool = True,
              new_dtype: Optional[str] = None, q_zero: bool = False, queries: int = 1,
              source: str = "codes") -> DecodeCase:
    """Draw one seeded decode case.

    ``lens`` are the lengths the decode attends to. Sequence ``b`` owns
    ``ceil((lens[b] + extra_tokens) / 16)`` physical blocks, so ``extra_tokens=1``
    leaves room to append a token at position ``lens[b]``. ``queries`` = T > 1
    draws T query tokens and T new K/V tokens per sequence ([B, T, ...] shapes).
    Values: Q, K, V ~ N(0, 1) rounded to their storage dtype; int8 caches hold
    uniform codes in [-127, 127] with fp16 scales in [0.015, 0.035] (the scale a
    row of 128 N(0,1) draws gets from its max magnitude); FP8 caches hold e4m3
    codes of N(0, 128^2) draws clipped to +-448 with fp16 scales in
    [0.006, 0.010]; int4 caches hold uniform codes in [-7, 7], two per byte
    (the row's last dim is d/2), with fp16 scales in [0.35, 0.50] (amax/7 of
    128 N(0,1) draws); "i4kc" caches hold the same codes with K scales per
    (block, kv-head, channel) and V scales per (token, kv-head), both in
    [0.35, 0.50], and an fp32 residual [B, K, 16, d] of N(0,1) draws standing
    for the unquantised K of each sequence's open block (drawn independently
    of that block's codes: decode reads only codes and scales, an append
    re-quantises the block from the residual).

    ``source="normal"`` (code caches only) draws instead the unquantised K/V
    rows of every cached token, N(0, 1) in fp32, packed ``[sum(lens), K, d]``
    in ``k_src``/``v_src`` with row offsets ``src_start``: the codes are left
    zero and every scale NaN until the consumer quantises the rows into the
    cache (the CUDA path through its append, the oracle with its own rule);
    a slot the quantisation does not reach keeps its NaN scale."""
    if q_dtype is None:
        q_dtype = "bf16" if cache_dtype in CODED else cache_dtype
    if new_dtype is None:
        new_dtype = q_dtype if cache_dtype in CODED else cache_dtype
    lens_t = torch.as_tensor(lens, dtype=torch.int32).reshape(-1).cpu()
    if lens_t.numel() != batch:
        raise ValueError("lens must have one entry per sequence")
    K, d, bs = num_kv_heads, head_dim, BLOCK_SIZE
    own = [-(-(int(lens_t[b]) + extra_tokens) // bs) for b in range(batch)]
    if max_blocks is None:
        max_blocks = max([1] + own)
    if max(own, default=0) > max_blocks:
        raise ValueError("max_blocks is smaller than a sequence's block count")
    if source not in ("codes", "normal"):
        raise ValueError(f"unknown source {source!r}")
    normal = source == "normal" and cache_dtype in CODED
    gen_cpu = torch.Generator().manual_seed(seed)
    dev = torch.device(device)
    gen_dev = gen_cpu if dev.type == "cpu" else torch.Generator(device=dev).manual_seed(seed)

    if contiguous:
        s_pad = max_blocks * bs
        num_blocks = batch * max_blocks
        table = torch.arange(num_blocks, dtype=torch.int32).reshape(batch, max_blocks)
        shape = (batch, s_pad, K, d)
        sb, sh, st = bs * K * d, d, K * d
    else:
        total = sum(own) + spare_blocks
        num_blocks = max(total, 1)
        perm = (torch.randperm(num_blocks, generator=gen_cpu, dtype=torch.int64) if shuffle
                else torch.arange(num_blocks, dtype=torch.int64)).to(torch.int32)
        table = torch.full((batch, max_blocks), -1, dtype=torch.int32)
        off = 0
        for b in range(batch):
            table[b, :own[b]] = perm[off:off + own[b]]
            off += own[b]
        shape = (num_blocks, K, bs, d)
        sb, sh, st = K * bs * d, bs * d, d

    if normal:
        es_shape = shape[:-1] + (d // 2,) if cache_dtype in PACKED4 else shape
        kc = torch.zeros(es_shape, dtype=DTYPES[cache_dtype], device=dev)
        vc = torch.zeros_like(kc)
        sshape = (num_blocks, K, bs)
        kshape = (num_blocks, K, d) if cache_dtype == "i4kc" else sshape
        ks = torch.full(kshape, float("nan"), dtype=torch.float16, device=dev)
        vs = torch.full(sshape, float("nan"), dtype=torch.float16, device=dev)
    elif cache_dtype == "i8":
        kc = torch.randint(-127, 128, shape, generator=gen_dev, device=dev, dtype=torch.int8)
        vc = torch.randint(-127, 128, shape, generator=gen_dev, device=dev, dtype=torch.int8)
        sshape = (num_blocks, K, bs)
        ks = (torch.rand(sshape, generator=gen_dev, device=dev) * 0.02 + 0.015).to(torch.float16)
        vs = (torch.rand(sshape, generator=gen_dev, device=dev) * 0.02 + 0.015).to(torch.float16)
    elif cache_dtype in PACKED4:
        pshape = shape[:-1] + (d // 2,)
        def packed():
            lo = torch.randint(-7, 8, pshape, generator=gen_dev, device=dev, dtype=torch.int32)
            hi = torch.randint(-7, 8, pshape, generator=gen_dev, device=dev, dtype=torch.int32)
            return ((lo & 0xF) | ((hi & 0xF) << 4)).to(torch.uint8)
        kc, vc = packed(), packed()
        sshape = (num_blocks, K, bs)
        kshape = (num_blocks, K, d) if cache_dtype == "i4kc" else sshape
        ks = (torch.rand(kshape, generator=gen_dev, device=dev) * 0.15 + 0.35).to(torch.float16)
        vs = (torch.rand(sshape, generator=gen_dev, device=dev) * 0.15 + 0.35).to(torch.float16)
    elif cache_dtype == "fp8":
        def codes():
            x = torch.randn(shape, generator=gen_dev, device=dev) * 128.0
            return x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
        kc, vc = codes(), codes()
        sshape = (num_blocks, K, bs)
        ks = (torch.rand(sshape, generator=gen_dev, device=dev) * 0.004 + 0.006).to(torch.float16)
        vs = (torch.rand(sshape, generator=gen_dev, device=dev) * 0.004 + 0.006).to(torch.float16)
    else:
        dt = DTYPES[cache_dtype]
        kc = _randn(shape, gen_dev, dev, dt)
        vc = _randn(shape, gen_dev, dev, dt)
        ks = vs = None

    if poison and not normal:
        _poison_unowned(kc, vc, ks, vs, table, lens_t, contiguous, cache_dtype)
    k_src = v_src = src_start = None
    if normal:
        total = int(lens_t.sum())
        k_src = _randn((total, K, d), gen_dev, dev, torch.float32)
        v_src = _randn((total, K, d), gen_dev, dev, torch.float32)
        src_start = torch.zeros(batch + 1, dtype=torch.int32)
        src_start[1:] = torch.cumsum(lens_t, 0)
        src_start = src_start.to(dev)

    tq = (queries,) if queries > 1 else ()
    q = _randn((batch, *tq, num_heads, d), gen_dev, dev, DTYPES[q_dtype])
    if q_zero:
        q.zero_()
    k_new = _randn((batch, *tq, K, d), gen_dev, dev, DTYPES[new_dtype])
    v_new = _randn((batch, *tq, K, d), gen_dev, dev, DTYPES[new_dtype])
    res = None
    if cache_dtype == "i4kc":
        res = (torch.zeros((batch, K, bs, d), dtype=torch.float32, device=dev) if normal
               else _randn((batch, K, bs, d), gen_dev, dev, torch.float32))
    return DecodeCase(batch, num_heads, K, d, cache_dtype, q_dtype, 1.0 / math.sqrt(d),
                      q, kc, vc, ks, vs, num_blocks, sb, sh, st, table.to(dev),
                      lens_t.to(dev), k_new, v_new, queries, res, k_src, v_src, src_start)


def _poison_unowned(kc, vc, ks, vs, table, lens, contiguous, cache_dtype):
    """NaN-fill every (block, slot) no sequence holds a valid token in."""
    bs = BLOCK_SIZE
    nb = table.shape[0] * table.shape[1] if contiguous else kc.shape[0]
    fill = torch.zeros(nb, dtype=torch.int64)       # valid slots per physical block
    for b in range(table.shape[0]):
        n = int(lens[b])
        full, rem = divmod(n, bs)
        ids = table[b, :full].to(torch.int64)
        fill[ids] = bs
        if rem:
            fill[int(table[b, full])] = rem
    slot = torch.arange(bs).unsqueeze(0)
    bad = (slot >= fill.unsqueeze(1)).to(kc.device)          # [nb, 16]
    if contiguous:
        B, s_pad = kc.shape[0], kc.shape[1]
        bad_tok = bad.reshape(B, s_pad)                       # blocks are consecutive per row
        mask = bad_tok[:, :, None, None].expand_as(kc)
    else:
        mask = bad[:, None, :, None].expand_as(kc)
    if cache_dtype in CODED:
        smask = bad[:, None, :].expand_as(vs)
        vs.masked_fill_(smask, float("nan"))
        if cache_dtype == "i4kc":      # channel scales: of blocks holding no valid token
            ks.masked_fill_(bad.all(dim=1)[:, None, None].to(ks.device).expand_as(ks), float("nan"))
        else:
            ks.masked_fill_(smask, float("nan"))
    else:
        kc.masked_fill_(mask, float("nan"))
        vc.masked_fill_(mask, float("nan"))


def case_for(workload: Workload, seed: int = 0, device: str = "cpu", **kw) -> DecodeCase:
    lens = draw_lens(workload.lens, workload.batch, seed)
    return make_case(workload.batch, workload.num_heads, workload.num_kv_heads,
                     workload.head_dim, lens, workload.cache_dtype, workload.q_dtype,
                     seed=seed, device=device, contiguous=workload.contiguous,
                     queries=workload.queries, **{"source": workload.source, **kw})
