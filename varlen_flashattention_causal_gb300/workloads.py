"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds input generation only -- lengths, block tables, slot
mappings and N(0, 1) tensors -- and none of the attention arithmetic.  Both
the CUDA path and the CPU oracle consume what it produces.

Every workload is drawn from ``torch.Generator`` seeded with
``SEED0 + index`` where index is the workload's position in the list below.
Shapes follow the workloads the source pages discuss (packed prefill of a
6-token and a 4-token request, Llama-3-8B-like GQA decode, long-context
decode, chunked prefill over a cached prefix, cascade decode over a shared
system prompt, an fp8 KV mixed batch):

0 tiny      B=4 lens {6,4,17,33}, Hq 8 / Hkv 2, D 64, bs 16, 16-block pool,
            then one decode step per request
1 decode    B=64, 1 query token, Hq 32 / Hkv 8, D 128, ctx ~ U[512, 4096],
            bs 16, 40960-block pool
2 longctx   B=4, ctx {32k, 64k, 96k, 128k} (k = 1024), Hq 64 / Hkv 8, D 128,
            bs in {16, 64, 256}, pool = 1.25 x the blocks used
3 chunked   B=16, new ~ U[1024, 8192] on cached ctx ~ U[0, 4096], Hq 32 /
            Hkv 8, D 128, bs 64
  cascade   64 requests share a 4096-token prefix (same block ids in every
            row), private suffix ~ U[256, 1024] incl. the current token,
            q_len 1, bs 64
4 fp8mixed  128 decode requests ctx log-uniform [128, 16384] + 4 prefill
            chunks of 2048 (no cached context), e4m3 cache with per-tensor
            scales amax/448, bs 32

Block tables are consecutive slices of one random permutation of the pool;
entries a request does not own are -1.  Slot mappings follow the serving
engine's placement rule: position p of request r goes to slot
block_table[r][p // bs] * bs + p % bs.
"""
from dataclasses import dataclass, field
import math
from typing import List, Optional

import torch

SEED0 = 20261202


def generator(index: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(SEED0 + index)
    return g


def randn(shape, g, device="cpu", dtype=torch.bfloat16):
    """N(0, 1) drawn in fp32 and rounded to ``dtype``."""
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


@dataclass
class Batch:
    """One attention call's worth of synthetic input (CPU or device tensors)."""
    name: str
    Hq: int
    Hkv: int
    D: int
    bs: int
    num_blocks: int
    q_lens: List[int]
    kv_lens: List[int]
    causal: bool = True
    # device-independent tensors
    cu_seqlens_q: Optional[torch.Tensor] = None   # int32 [B+1]
    seqused_k: Optional[torch.Tensor] = None      # int32 [B]
    block_table: Optional[torch.Tensor] = None    # int32 [B, max_blocks]
    q: Optional[torch.Tensor] = None              # [T, Hq, D]
    # K/V of every cached token (context + new), token-major, and where the
    # KV write puts each one
    k_tok: Optional[torch.Tensor] = None          # [Tkv, Hkv, D]
    v_tok: Optional[torch.Tensor] = None
    slot_mapping: Optional[torch.Tensor] = None   # int64 [Tkv]
    kv_dtype: str = "bf16"                        # "bf16" | "fp16" | "fp8"
    k_scale: float = 1.0
    v_scale: float = 1.0
    extra: dict = field(default_factory=dict)

    @property
    def B(self):
        return len(self.q_lens)

    @property
    def T(self):
        return sum(self.q_lens)

    @property
    def softmax_scale(self):
        return 1.0 / math.sqrt(self.D)

    @property
    def max_seqlen_q(self):
        return max(self.q_lens) if self.q_lens else 0

    @property
    def max_seqlen_k(self):
        return max(self.kv_lens) if self.kv_lens else 0


def block_tables(kv_lens, bs, pool_blocks, g, shared_prefix_blocks=0):
    """Consecutive slices of randperm(pool_blocks); -1 where unused.

    With shared_prefix_blocks = n, the first n entries of every row are the
    same n block ids (a common prefix stored once)."""
    perm = torch.randperm(pool_blocks, generator=g)
    need = [(L + bs - 1) // bs for L in kv_lens]
    width = max(need) if need else 1
    bt = torch.full((len(kv_lens), max(width, 1)), -1, dtype=torch.int32)
    pos = 0
    if shared_prefix_blocks:
        shared = perm[:shared_prefix_blocks].to(torch.int32)
        pos = shared_prefix_blocks
    for r, n in enumerate(need):
        if shared_prefix_blocks:
            own = n - shared_prefix_blocks
            bt[r, :shared_prefix_blocks] = shared
            bt[r, shared_prefix_blocks:n] = perm[pos:pos + own].to(torch.int32)
            pos += own
        else:
            bt[r, :n] = perm[pos:pos + n].to(torch.int32)
            pos += n
    assert pos <= pool_blocks, "pool too small"
    return bt


def slots(block_table, r, positions, bs):
    """Engine-side slot placement for positions of request r (int64)."""
    p = torch.as_tensor(positions, dtype=torch.int64)
    return block_table[r].to(torch.int64)[p // bs] * bs + p % bs


def _finish(b: Batch, g, device, cached_positions, gen_kv=True):
    """Fill cu_seqlens, seqused_k, q and the token-major K/V + slots."""
    B = b.B
    b.cu_seqlens_q = torch.zeros(B + 1, dtype=torch.int32)
    b.cu_seqlens_q[1:] = torch.cumsum(torch.tensor(b.q_lens, dtype=torch.int64), 0).to(torch.int32)
    b.seqused_k = torch.tensor(b.kv_lens, dtype=torch.int32)
    b.q = randn((b.T, b.Hq, b.D), g, device)
    if gen_kv:
        sl = [slots(b.block_table, r, pos, b.bs) for r, pos in enumerate(cached_positions)]
        b.slot_mapping = torch.cat(sl) if sl else torch.zeros(0, dtype=torch.int64)
        n = b.slot_mapping.numel()
        b.k_tok = randn((n, b.Hkv, b.D), g, device)
        b.v_tok = randn((n, b.Hkv, b.D), g, device)
        if b.kv_dtype == "fp8":
            # per-tensor scales: the largest magnitude maps to e4m3's 448
            b.k_scale = float(b.k_tok.float().abs().max()) / 448.0
            b.v_scale = float(b.v_tok.float().abs().max()) / 448.0
    return b


def tiny(device="cpu"):
    """Workload 0: returns (prefill batch, decode batch) sharing one pool.

    The prefill writes each prompt's K/V, then attends causally; the decode
    step appends one token per request at position len and attends over
    len + 1 keys."""
    g = generator(0)
    lens = [6, 4, 17, 33]
    Hq, Hkv, D, bs, nb = 8, 2, 64, 16, 16
    bt = block_tables([L + 1 for L in lens], bs, nb, g)
    pre = Batch("tiny-prefill", Hq, Hkv, D, bs, nb, list(lens), list(lens), block_table=bt)
    _finish(pre, g, device, [range(L) for L in lens])
    dec = Batch("tiny-decode", Hq, Hkv, D, bs, nb, [1] * 4, [L + 1 for L in lens], block_table=bt)
    _finish(dec, g, device, [[L] for L in lens])
    return pre, dec


def decode_llama8b(device="cpu", B=64, lo=512, hi=4096, pool=40960, gen_kv=True):
    """Workload 1: Llama-3-8B-shaped paged decode (query = last position)."""
    g = generator(1)
    ctx = torch.randint(lo, hi + 1, (B,), generator=g).tolist()
    Hq, Hkv, D, bs = 32, 8, 128, 16
    bt = block_tables(ctx, bs, pool, g)
    b = Batch("decode-llama8b", Hq, Hkv, D, bs, pool, [1] * B, ctx, block_table=bt)
    return _finish(b, g, device, [range(L) for L in ctx], gen_kv=gen_kv)


LONGCTX = [32 * 1024, 64 * 1024, 96 * 1024, 128 * 1024]


def decode_longctx(bs=16, device="cpu", ctx=None, gen_kv=True):
    """Workload 2: long-context split-KV decode at block size bs."""
    g = generator(2)
    ctx = list(LONGCTX if ctx is None else ctx)
    Hq, Hkv, D = 64, 8, 128
    used = sum((L + bs - 1) // bs for L in ctx)
    pool = (used * 5 + 3) // 4
    bt = block_tables(ctx, bs, pool, g)
    b = Batch("decode-longctx-bs%d" % bs, Hq, Hkv, D, bs, pool, [1] * len(ctx), ctx, block_table=bt)
    return _finish(b, g, device, [range(L) for L in ctx], gen_kv=gen_kv)


def chunked_prefill(device="cpu", B=16, gen_kv=True, new_range=(1024, 8192), ctx_range=(0, 4096)):
    """Workload 3a: chunked causal prefill over a cached prefix (bs 64)."""
    g = generator(3)
    new = torch.randint(new_range[0], new_range[1] + 1, (B,), generator=g).tolist()
    ctx = torch.randint(ctx_range[0], ctx_range[1] + 1, (B,), generator=g).tolist()
    Hq, Hkv, D, bs = 32, 8, 128, 64
    kv = [c + n for c, n in zip(ctx, new)]
    used = sum((L + bs - 1) // bs for L in kv)
    pool = (used * 5 + 3) // 4
    bt = block_tables(kv, bs, pool, g)
    b = Batch("chunked-prefill", Hq, Hkv, D, bs, pool, new, kv, block_table=bt)
    b.extra["ctx"] = ctx
    return _finish(b, g, device, [range(L) for L in kv], gen_kv=gen_kv)


def cascade_decode(device="cpu", B=64, prefix=4096, lo=256, hi=1024):
    """Workload 3b: decode where every request shares a prefix of `prefix`
    tokens stored once; suffix lengths include the current token."""
    g = generator(3 + 100)
    suf = torch.randint(lo, hi + 1, (B,), generator=g).tolist()
    Hq, Hkv, D, bs = 32, 8, 128, 64
    assert prefix % bs == 0
    kv = [prefix + s for s in suf]
    npre = prefix // bs
    used = npre + sum((L + bs - 1) // bs - npre for L in kv)
    pool = (used * 5 + 3) // 4
    bt = block_tables(kv, bs, pool, g, shared_prefix_blocks=npre)
    b = Batch("cascade-decode", Hq, Hkv, D, bs, pool, [1] * B, kv, block_table=bt)
    b.extra["prefix"] = prefix
    b.extra["suffix"] = suf
    # prefix tokens are written once (through row 0), suffix tokens per row
    positions = [range(L) if r == 0 else range(prefix, L) for r, L in enumerate(kv)]
    return _finish(b, g, device, positions)


def fp8_mixed(device="cpu", n_dec=128, n_pre=4, pre_len=2048, lo=128, hi=16384, gen_kv=True):
    """Workload 4: fp8 e4m3 KV cache, decode requests + prefill chunks in
    one batch (decodes first)."""
    g = generator(4)
    u = torch.rand((n_dec,), generator=g, dtype=torch.float64)
    ctx = torch.round(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))).to(torch.int64).tolist()
    Hq, Hkv, D, bs = 32, 8, 128, 32
    q_lens = [1] * n_dec + [pre_len] * n_pre
    kv = ctx + [pre_len] * n_pre
    used = sum((L + bs - 1) // bs for L in kv)
    pool = (used * 5 + 3) // 4
    bt = block_tables(kv, bs, pool, g)
    b = Batch("fp8-mixed", Hq, Hkv, D, bs, pool, q_lens, kv, block_table=bt, kv_dtype="fp8")
    return _finish(b, g, device, [range(L) for L in kv], gen_kv=gen_kv)


def swa_decode(device="cpu", B=64, lo=4096, hi=32768, window=4096, gen_kv=True):
    """Sliding-window decode with attention sinks: each query sees its last
    `window` keys (window_left = window - 1); Hq 32 / Hkv 8, D 128, bs 16,
    contexts U[lo, hi]; one N(0, 1) sink logit per query head."""
    g = generator(5)
    ctx = torch.randint(lo, hi + 1, (B,), generator=g).tolist()
    Hq, Hkv, D, bs = 32, 8, 128, 16
    used = sum((L + bs - 1) // bs for L in ctx)
    pool = (used * 5 + 3) // 4
    bt = block_tables(ctx, bs, pool, g)
    b = Batch("swa-decode", Hq, Hkv, D, bs, pool, [1] * B, ctx, block_table=bt)
    b.extra["window"] = (window - 1, -1)
    b.extra["sinks"] = torch.randn((Hq,), generator=g, dtype=torch.float32)
    return _finish(b, g, device, [range(L) for L in ctx], gen_kv=gen_kv)


def verify_decode(device="cpu", B=64, q_lo=2, q_hi=8, lo=512, hi=8192, gen_kv=True):
    """Multi-token verification (speculative decoding): q_len U[q_lo, q_hi]
    new tokens per request at the end of a paged context U[lo, hi] (the
    new tokens' keys included), Hq 32 / Hkv 8, D 128, bs 16, causal."""
    g = generator(6)
    ql = torch.randint(q_lo, q_hi + 1, (B,), generator=g).tolist()
    ctx = torch.randint(lo, hi + 1, (B,), generator=g).tolist()
    kv = [c + q for c, q in zip(ctx, ql)]
    Hq, Hkv, D, bs = 32, 8, 128, 16
    used = sum((L + bs - 1) // bs for L in kv)
    pool = (used * 5 + 3) // 4
    bt = block_tables(kv, bs, pool, g)
    b = Batch("verify-decode", Hq, Hkv, D, bs, pool, ql, kv, block_table=bt)
    return _finish(b, g, device, [range(L) for L in kv], gen_kv=gen_kv)


def make_batch(q_lens, kv_lens, Hq, Hkv, D, bs, seed, pool=None, causal=True,
               kv_dtype="bf16", device="cpu", name="custom", q_dtype=torch.bfloat16):
    """A seeded batch of any shape (tests).  All kv_lens tokens of every
    request are cached (written through the slot mapping); the queries are
    the last q_len positions of each request."""
    g = torch.Generator()
    g.manual_seed(SEED0 + 1000 + seed)
    need = sum((L + bs - 1) // bs for L in kv_lens)
    pool = pool if pool is not None else max(1, need + (need + 3) // 4)
    bt = block_tables(list(kv_lens), bs, pool, g)
    b = Batch(name, Hq, Hkv, D, bs, pool, list(q_lens), list(kv_lens), causal=causal,
              block_table=bt, kv_dtype=kv_dtype)
    _finish(b, g, device, [range(L) for L in kv_lens])
    if q_dtype != torch.bfloat16:
        b.q = b.q.to(q_dtype)
        b.k_tok = b.k_tok.to(q_dtype)
        b.v_tok = b.v_tok.to(q_dtype)
    return b
