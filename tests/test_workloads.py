"""The synthetic workloads have the shapes and structure of the configurations
they stand in for (head counts, head size, block size, pool, length ranges,
shared prefix, fp8 cache), their block tables are valid page maps, and they
are reproducible from their seeds.  No GPU."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from varlen_flashattention_causal_gb300 import workloads as W  # noqa: E402


def _pages(b):
    """Physical block ids each request's keys use, in order."""
    bt = b.block_table
    return [bt[r, :(L + b.bs - 1) // b.bs].tolist() for r, L in enumerate(b.kv_lens)]


def _check_page_map(b, shared_prefix_blocks=0):
    pages = _pages(b)
    seen = {}
    for r, ids in enumerate(pages):
        assert all(0 <= i < b.num_blocks for i in ids)
        for i in ids[shared_prefix_blocks:]:
            assert i not in seen, "block %d of request %d already used by request %d" % (i, r, seen[i])
            seen[i] = r
    if shared_prefix_blocks:
        first = pages[0][:shared_prefix_blocks]
        assert all(ids[:shared_prefix_blocks] == first for ids in pages)
        assert not set(first) & set(seen)
    assert int(b.cu_seqlens_q[-1]) == b.T
    assert b.cu_seqlens_q.tolist() == [sum(b.q_lens[:r]) for r in range(b.B + 1)]
    assert b.seqused_k.tolist() == b.kv_lens
    assert all(k >= q for q, k in zip(b.q_lens, b.kv_lens))


def test_tiny_prefill_then_one_decode_step():
    pre, dec = W.tiny()
    assert pre.q_lens == pre.kv_lens == [6, 4, 17, 33]
    assert (pre.Hq, pre.Hkv, pre.D, pre.bs, pre.num_blocks) == (8, 2, 64, 16, 16)
    assert dec.q_lens == [1, 1, 1, 1] and dec.kv_lens == [7, 5, 18, 34]
    _check_page_map(pre)
    _check_page_map(dec)
    # the decode step's block table continues each prompt's block list
    assert torch.equal(pre.block_table, dec.block_table)
    # its single new token per request goes to slot (position len)
    for r, L in enumerate(pre.kv_lens):
        blk = int(dec.block_table[r, L // dec.bs])
        assert int(dec.slot_mapping[r]) == blk * dec.bs + L % dec.bs


def test_llama8b_decode_shape():
    b = W.decode_llama8b(gen_kv=False)
    assert (b.B, b.Hq, b.Hkv, b.D, b.bs, b.num_blocks) == (64, 32, 8, 128, 16, 40960)
    assert b.q_lens == [1] * 64
    assert all(512 <= L <= 4096 for L in b.kv_lens)
    assert len(set(b.kv_lens)) > 32                     # spread over the range, not constant
    _check_page_map(b)


@pytest.mark.parametrize("bs", [16, 64, 256])
def test_long_context_shape(bs):
    b = W.decode_longctx(bs=bs, gen_kv=False)
    assert (b.B, b.Hq, b.Hkv, b.D, b.bs) == (4, 64, 8, 128, bs)
    assert b.kv_lens == [32 * 1024, 64 * 1024, 96 * 1024, 128 * 1024]
    assert b.num_blocks >= sum(-(-L // bs) for L in b.kv_lens)
    _check_page_map(b)


def test_chunked_prefill_shape():
    b = W.chunked_prefill(gen_kv=False)
    assert (b.B, b.Hq, b.Hkv, b.D, b.bs) == (16, 32, 8, 128, 64)
    ctx = b.extra["ctx"]
    assert all(1024 <= q <= 8192 for q in b.q_lens)
    assert all(0 <= c <= 4096 for c in ctx)
    assert b.kv_lens == [c + q for c, q in zip(ctx, b.q_lens)]
    _check_page_map(b)


def test_cascade_shares_the_prefix_blocks():
    b = W.cascade_decode()
    P = b.extra["prefix"]
    assert (b.B, P, b.bs) == (64, 4096, 64)
    assert b.q_lens == [1] * 64
    suffix = b.extra["suffix"]
    assert all(256 <= s <= 1024 for s in suffix)
    assert b.kv_lens == [P + s for s in suffix]
    _check_page_map(b, shared_prefix_blocks=P // b.bs)


def test_fp8_mixed_batch_shape():
    b = W.fp8_mixed(gen_kv=False)
    assert (b.Hq, b.Hkv, b.D, b.bs, b.kv_dtype) == (32, 8, 128, 32, "fp8")
    assert b.q_lens == [1] * 128 + [2048] * 4
    dec = b.kv_lens[:128]
    assert all(128 <= L <= 16384 for L in dec)
    assert b.kv_lens[128:] == [2048] * 4
    # log-uniform: about as many contexts below the geometric mean as above
    gm = (128 * 16384) ** 0.5
    below = sum(L < gm for L in dec)
    assert 40 <= below <= 88
    _check_page_map(b)


def test_workloads_are_reproducible():
    a, b = W.decode_llama8b(gen_kv=False), W.decode_llama8b(gen_kv=False)
    assert a.kv_lens == b.kv_lens and torch.equal(a.block_table, b.block_table) and torch.equal(a.q, b.q)
    c, d = W.chunked_prefill(gen_kv=False), W.chunked_prefill(gen_kv=False)
    assert c.q_lens == d.q_lens and torch.equal(c.block_table, d.block_table)
