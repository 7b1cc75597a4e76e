"""Pins for the fp64 CPU oracle: checks against what the pages and the
mathematics fix, never against the oracle itself.

Each test names the passage it follows ("vLLM 中 Attention Kernel 如何并行处理
多个请求" is abbreviated "multi-request page"; "FlashAttention deep dive" is
the vLLM backend page).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from varlen_flashattention_causal_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def cache_of(b, dtype=torch.bfloat16):
    """Build CPU caches for batch b with the oracle's own KV write."""
    if b.kv_dtype == "fp8":
        dtype = torch.float8_e4m3fn
    kc = torch.zeros((b.num_blocks, b.bs, b.Hkv, b.D), dtype=dtype)
    vc = torch.zeros_like(kc)
    oracle.kv_write(b.k_tok, b.v_tok, kc, vc, b.slot_mapping, b.k_scale, b.v_scale)
    return kc, vc


def run(b, kc=None, vc=None, **kw):
    if kc is None:
        kc, vc = cache_of(b)
    return oracle.attention(b.q, kc, vc, b.cu_seqlens_q, b.seqused_k, b.block_table,
                            b.softmax_scale, causal=b.causal, k_scale=b.k_scale,
                            v_scale=b.v_scale, **kw)


def key_rows(b, r):
    """Token-major K/V rows of request r (the order they were written)."""
    start = sum(b.kv_lens[:r])
    n = b.kv_lens[r]
    return b.k_tok[start:start + n], b.v_tok[start:start + n]


def read_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# --------------------------------------------------------------- worked examples

def test_packed_6_4_mask_is_the_pages_matrix():
    """multi-request page, sec. 1: the block-diagonal lower-triangular mask."""
    rows = read_golden("packed_6_4_mask.txt")
    want = np.array([[int(x) for x in r[1:]] for r in rows], dtype=bool)
    q = np.zeros((10, 1, 4))
    k = np.zeros((10, 1, 4))
    _, _, mask = oracle.dense_masked_attention(q, k, k, [0, 6, 10], [0, 6, 10], 1.0)
    assert (mask == want).all()


def test_packed_6_4_oracle_equals_brute_force_and_isolation():
    """multi-request page, sec. 1 and 5: packing A (6) and B (4) together
    gives the same result as running each alone; changing B's inputs leaves
    A's outputs bit-identical and vice versa."""
    b = W.make_batch([6, 4], [6, 4], Hq=4, Hkv=2, D=16, bs=16, seed=1)
    out, lse = run(b)
    ref, ref_lse, _ = oracle.dense_masked_attention(
        b.q.double(), b.k_tok.double(), b.v_tok.double(), [0, 6, 10], [0, 6, 10], b.softmax_scale)
    np.testing.assert_allclose(out.numpy(), ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.numpy(), ref_lse, rtol=0, atol=1e-12)

    # perturb request B only (its queries and its cached K/V)
    b2 = W.make_batch([6, 4], [6, 4], Hq=4, Hkv=2, D=16, bs=16, seed=1)
    b2.q[6:] = W.randn((4, 4, 16), torch.Generator().manual_seed(7))
    b2.k_tok[6:] = -b2.k_tok[6:]
    b2.v_tok[6:] = 3 * b2.v_tok[6:]
    out2, lse2 = run(b2)
    assert torch.equal(out2[:6], out[:6]) and torch.equal(lse2[:6], lse[:6])
    assert not torch.equal(out2[6:], out[6:])
    # and the other way round
    b3 = W.make_batch([6, 4], [6, 4], Hq=4, Hkv=2, D=16, bs=16, seed=1)
    b3.k_tok[:6] = 2 * b3.k_tok[:6]
    out3, lse3 = run(b3)
    assert torch.equal(out3[6:], out[6:]) and torch.equal(lse3[6:], lse[6:])

    # each request alone
    for r, (lo, hi) in enumerate([(0, 6), (6, 10)]):
        single = W.make_batch([hi - lo], [hi - lo], Hq=4, Hkv=2, D=16, bs=16, seed=1)
        single.q = b.q[lo:hi].clone()
        single.k_tok, single.v_tok = key_rows(b, r)
        o1, l1 = run(single)
        assert torch.equal(o1, out[lo:hi]) and torch.equal(l1, lse[lo:hi])


def test_multi_token_verify_equals_six_decodes():
    """multi-request page, sec. 10: 6 new positions over 20,000 cached
    tokens.  Each query row equals an independent decode at its position,
    and sees exactly the number of keys the page's picture gives."""
    g = read_golden("verify_6_over_20000.txt")
    ctx, q_len = int(g[0][1]), int(g[1][1])
    nvis = {int(a): int(c) for a, c in g[2:]}
    b = W.make_batch([q_len], [ctx + q_len], Hq=2, Hkv=1, D=16, bs=64, seed=2)
    kc, vc = cache_of(b)
    out, lse = run(b, kc, vc)
    for i in range(q_len):
        dec = W.make_batch([1], [nvis[i]], Hq=2, Hkv=1, D=16, bs=64, seed=2)
        dec.q = b.q[i:i + 1].clone()
        dec.block_table = b.block_table
        dec.num_blocks = b.num_blocks
        o, l = run(dec, kc, vc)
        np.testing.assert_allclose(o.numpy(), out[i:i + 1].numpy(), rtol=0, atol=1e-13)
        np.testing.assert_allclose(l.numpy(), lse[i:i + 1].numpy(), rtol=0, atol=1e-12)
    # the visible-count column: with q = 0 every visible key scores 0, so
    # lse = ln(number of visible keys)
    b.q.zero_()
    _, lse0 = run(b, kc, vc)
    for i in range(q_len):
        assert abs(float(lse0[i, 0]) - math.log(nvis[i])) < 1e-12


def test_decode_rows_see_every_key():
    """multi-request page, sec. 9: decode requests with contexts of 20,000 and
    35,000 tokens have attention rows of 20,001 and 35,001 keys, all visible.
    With q = 0 every score ties, so lse = ln(row length) and out is the mean
    of all V rows; and the causal result equals the non-causal one exactly."""
    g = read_golden("decode_20000_35000.txt")
    ctx = [int(r[1]) for r in g]
    row = [int(r[2]) for r in g]
    assert row == [c + 1 for c in ctx]
    b = W.make_batch([1, 1], row, Hq=2, Hkv=1, D=16, bs=64, seed=40)
    kc, vc = cache_of(b)
    out, lse = run(b, kc, vc)
    b_nc = W.make_batch([1, 1], row, Hq=2, Hkv=1, D=16, bs=64, seed=40, causal=False)
    out_nc, lse_nc = run(b_nc, kc, vc)
    assert torch.equal(out, out_nc) and torch.equal(lse, lse_nc)
    b.q.zero_()
    out0, lse0 = run(b, kc, vc)
    for r, n in enumerate(row):
        _, v = key_rows(b, r)
        assert v.shape[0] == n
        for h in range(2):
            assert abs(float(lse0[r, h]) - math.log(n)) < 1e-12
            np.testing.assert_allclose(out0[r, h].numpy(), v[:, 0].double().mean(0).numpy(), rtol=0, atol=1e-14)


def test_split_into_the_pages_segments():
    """multi-request page, sec. 12: a 12,288-key decode row cut into the
    page's three 4096-key segments.  Each segment's local max m_s, exponent
    sum l_s and weighted output O_s are computed by brute force from the key
    rows, then reduced by the page's formulas m = max m_s,
    l = sum e^{m_s - m} l_s, O = sum e^{m_s - m} O_s / l.  That equals the
    oracle's unsplit result, and so does the oracle's pairwise log-sum-exp
    merge of its own per-segment results."""
    segs = [(int(a), int(c)) for _, a, c in read_golden("split_segments_4096.txt")]
    n = segs[-1][1] + 1
    b = W.make_batch([1], [n], Hq=2, Hkv=1, D=16, bs=64, seed=41)
    kc, vc = cache_of(b)
    full, full_lse = run(b, kc, vc)
    k, v = key_rows(b, 0)
    for h in range(2):
        q = b.q[0, h].double().numpy()
        parts = []
        for lo, hi in segs:
            s = b.softmax_scale * (k[lo:hi + 1, 0].double().numpy() @ q)
            m_s = s.max()
            e = np.exp(s - m_s)
            parts.append((m_s, e.sum(), e @ v[lo:hi + 1, 0].double().numpy()))
        m = max(p[0] for p in parts)
        l = sum(math.exp(m_s - m) * l_s for m_s, l_s, _ in parts)
        o = sum(math.exp(m_s - m) * o_s for m_s, _, o_s in parts) / l
        np.testing.assert_allclose(o, full[0, h].numpy(), rtol=0, atol=1e-13)
        assert abs(m + math.log(l) - float(full_lse[0, h])) < 1e-11
    # the oracle's own segments (keys lo..hi through the block table), merged
    state = None
    for lo, hi in segs:
        bt = b.block_table[:, lo // b.bs:].contiguous()
        o_s, l_s = oracle.attention(b.q, kc, vc, b.cu_seqlens_q, torch.tensor([hi - lo + 1], dtype=torch.int32),
                                    bt, b.softmax_scale, causal=False)
        o_s, l_s = o_s.view(-1, 16), l_s.view(-1)
        state = (o_s, l_s) if state is None else oracle.merge_states(state[0], state[1], o_s, l_s)
    np.testing.assert_allclose(state[0].numpy(), full.view(-1, 16).numpy(), rtol=0, atol=1e-13)
    np.testing.assert_allclose(state[1].numpy(), full_lse.view(-1).numpy(), rtol=0, atol=1e-11)


def test_paged_lookup_example():
    """multi-request page, sec. 11: position 1024 -> physical block 37 for
    request A and 912 for request B; the KV write puts the token there and
    the attention read finds it there."""
    g = read_golden("paged_lookup.txt")
    pos, blkA, blkB = int(g[0][1]), int(g[1][1]), int(g[2][1])
    bs, Hkv, D = 16, 1, 16
    nb = 1024
    logical = pos // bs
    bt = torch.full((2, logical + 1), -1, dtype=torch.int32)
    rng = torch.Generator().manual_seed(3)
    others = [x for x in torch.randperm(nb, generator=rng).tolist() if x not in (blkA, blkB)]
    bt[0, :logical] = torch.tensor(others[:logical], dtype=torch.int32)
    bt[1, :logical] = torch.tensor(others[logical:2 * logical], dtype=torch.int32)
    bt[0, logical], bt[1, logical] = blkA, blkB
    slot = torch.tensor([blkA * bs + pos % bs, blkB * bs + pos % bs], dtype=torch.int64)
    k = W.randn((2, Hkv, D), rng)
    v = W.randn((2, Hkv, D), rng)
    kc = torch.zeros((nb, bs, Hkv, D), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    oracle.kv_write(k, v, kc, vc, slot)
    assert torch.equal(kc[blkA, pos % bs], k[0]) and torch.equal(kc[blkB, pos % bs], k[1])
    assert torch.equal(vc[blkA, pos % bs], v[0]) and torch.equal(vc[blkB, pos % bs], v[1])
    assert int(torch.count_nonzero(kc.float())) == int(torch.count_nonzero(k.float()))
    # read back through the block table: with q = 0 all pos + 1 visible keys
    # score equally and every other cached row is zero
    q = torch.zeros((2, 1, D), dtype=torch.bfloat16)
    cu = torch.tensor([0, 1, 2], dtype=torch.int32)
    su = torch.tensor([pos + 1, pos + 1], dtype=torch.int32)
    out, _ = oracle.attention(q, kc, vc, cu, su, bt, 1.0, causal=True)
    np.testing.assert_allclose(out[:, 0].numpy(), (v[:, 0].double() / (pos + 1)).numpy(),
                               rtol=0, atol=1e-15)


# -------------------------------------------------------------- closed forms

def test_single_key_returns_v0_exactly():
    """Row 0 of a causal request with no cached context sees only key 0:
    out = V_0 exactly and lse = scale * q . K_0."""
    b = W.make_batch([5, 3], [5, 3], Hq=4, Hkv=2, D=32, bs=16, seed=4)
    out, lse = run(b)
    for r, t in enumerate([0, 5]):
        k, v = key_rows(b, r)
        for h in range(4):
            g = h // 2
            assert torch.equal(out[t, h], v[0, g].double())
            s = b.softmax_scale * float((b.q[t, h].double() * k[0, g].double()).sum())
            assert abs(float(lse[t, h]) - s) < 1e-12


def test_two_keys_closed_form():
    """Two visible keys: out = sigmoid(s0 - s1) V_0 + sigmoid(s1 - s0) V_1."""
    b = W.make_batch([2], [2], Hq=1, Hkv=1, D=8, bs=16, seed=5)
    out, lse = run(b)
    k, v = key_rows(b, 0)
    qd, kd, vd = b.q[1, 0].double(), k[:, 0].double(), v[:, 0].double()
    s0 = b.softmax_scale * float(qd @ kd[0])
    s1 = b.softmax_scale * float(qd @ kd[1])
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    want = w0 * vd[0] + (1.0 - w0) * vd[1]
    np.testing.assert_allclose(out[1, 0].numpy(), want.numpy(), rtol=0, atol=1e-14)
    assert abs(float(lse[1, 0]) - (s0 + math.log1p(math.exp(s1 - s0)))) < 1e-13


@pytest.mark.parametrize("ctx", [0, 13])
def test_equal_scores_give_mean_of_visible_values(ctx):
    """q = 0 makes every visible score 0: out = mean of the visible V rows
    and lse = ln(#visible).  With cached context ctx, query i sees ctx+i+1
    keys (bottom-right alignment, multi-request page sec. 10).  Both the
    paged oracle and the dense formulation."""
    q_len = 7
    b = W.make_batch([q_len], [ctx + q_len], Hq=2, Hkv=2, D=16, bs=16, seed=6)
    b.q.zero_()
    out, lse = run(b)
    dense, dense_lse, _ = _dense(b)
    _, v = key_rows(b, 0)
    for i in range(q_len):
        n = ctx + i + 1
        for h in range(2):
            want = v[:n, h].double().mean(0).numpy()
            np.testing.assert_allclose(out[i, h].numpy(), want, rtol=0, atol=1e-14)
            np.testing.assert_allclose(dense[i, h], want, rtol=0, atol=1e-14)
            assert abs(float(lse[i, h]) - math.log(n)) < 1e-13
            assert abs(float(dense_lse[i, h]) - math.log(n)) < 1e-13


def test_gqa_head_mapping():
    """Query head h reads KV head h // (Hq / Hkv).  Each KV head holds a
    different constant value row, so with q = 0 the output of head h is
    exactly that constant, in the paged oracle and in the dense formulation."""
    Hq, Hkv = 8, 2
    b = W.make_batch([3], [3], Hq=Hq, Hkv=Hkv, D=16, bs=16, seed=7)
    b.q.zero_()
    for g in range(Hkv):
        b.v_tok[:, g, :] = float(g + 1)
    out, _ = run(b)
    dense, _, _ = _dense(b)
    for h in range(Hq):
        want = torch.full((3, 16), float(h // (Hq // Hkv) + 1), dtype=torch.float64)
        assert torch.equal(out[:, h], want)
        assert torch.equal(torch.from_numpy(dense[:, h]), want)


def test_non_causal_sees_every_key():
    """causal=False (the cascade prefix stage): every query sees all keys."""
    b = W.make_batch([4], [9], Hq=2, Hkv=1, D=16, bs=16, seed=8, causal=False)
    b.q.zero_()
    out, lse = run(b)
    _, v = key_rows(b, 0)
    for i in range(4):
        np.testing.assert_allclose(out[i, 0].numpy(), v[:, 0].double().mean(0).numpy(), atol=1e-14)
        assert abs(float(lse[i, 0]) - math.log(9)) < 1e-13


def test_empty_kv_gives_zero_and_minus_inf():
    """No visible key: out 0, lse -inf (reading adopted for kv_len = 0)."""
    b = W.make_batch([1, 1], [0, 4], Hq=2, Hkv=1, D=16, bs=16, seed=9)
    out, lse = run(b)
    assert torch.equal(out[0], torch.zeros((2, 16), dtype=torch.float64))
    assert lse[0].tolist() == [-math.inf, -math.inf]
    assert torch.isfinite(lse[1]).all()


# ------------------------------------------------------------ brute force

@pytest.mark.parametrize("seed,causal,dtype", [(10, True, torch.bfloat16), (11, True, torch.bfloat16),
                                               (12, False, torch.bfloat16), (13, True, torch.float16)])
def test_oracle_equals_dense_brute_force(seed, causal, dtype):
    """Random varlen batch with cached context and GQA: the per-row paged
    oracle equals the dense whole-matrix formulation, for bf16 and fp16
    storage (the dense side widens with torch's own conversion)."""
    rng = np.random.default_rng(seed)
    B = 4
    q_lens = rng.integers(1, 9, B).tolist()
    ctx = rng.integers(0, 20, B).tolist()
    kv = [c + q for c, q in zip(ctx, q_lens)]
    b = W.make_batch(q_lens, kv, Hq=6, Hkv=2, D=32, bs=16, seed=seed, causal=causal, q_dtype=dtype)
    kc, vc = cache_of(b, dtype)
    out, lse = run(b, kc, vc)
    # the cached rows of request r are its kv_len tokens in position order
    cuk = [0] + np.cumsum(kv).tolist()
    ref, ref_lse, _ = oracle.dense_masked_attention(
        b.q.double(), b.k_tok.double(), b.v_tok.double(),
        b.cu_seqlens_q.tolist(), cuk, b.softmax_scale, causal=causal)
    np.testing.assert_allclose(out.numpy(), ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.numpy(), ref_lse, rtol=0, atol=1e-12)


def test_online_softmax_recurrence_matches():
    """multi-request page, sec. 7: the online recurrence over K/V tiles
    (m_new = max(m, rowmax S), alpha = e^(m - m_new), l = alpha l + sum p,
    O = alpha O + p V, out = O / l) equals the oracle's two-pass softmax for
    any tiling."""
    b = W.make_batch([5], [40], Hq=1, Hkv=1, D=16, bs=16, seed=13)
    out, lse = run(b)
    k, v = key_rows(b, 0)
    kd, vd = k[:, 0].double().numpy(), v[:, 0].double().numpy()
    for tile in (1, 3, 16, 40):
        for i in range(5):
            qi = b.q[i, 0].double().numpy()
            n = 35 + i + 1
            m, l, o = -np.inf, 0.0, np.zeros(16)
            for j0 in range(0, n, tile):
                s = b.softmax_scale * (kd[j0:min(n, j0 + tile)] @ qi)
                m_new = max(m, s.max())
                alpha = math.exp(m - m_new) if m > -np.inf else 0.0
                p = np.exp(s - m_new)
                l = alpha * l + p.sum()
                o = alpha * o + p @ vd[j0:min(n, j0 + tile)]
                m = m_new
            np.testing.assert_allclose(o / l, out[i, 0].numpy(), rtol=0, atol=1e-13)
            assert abs(m + math.log(l) - float(lse[i, 0])) < 1e-12


# ------------------------------------------------------------- invariances

def test_paged_equals_contiguous_and_any_block_size():
    """vAttention notes (virtually contiguous KV) and multi-request page
    sec. 11: the block-table walk is pure addressing, so a randomly permuted
    paged layout at any block size gives bit-identical fp64 results to a
    contiguous layout (one block per request)."""
    q_lens, kv = [3, 1, 6], [50, 17, 70]
    ref = W.make_batch(q_lens, kv, Hq=4, Hkv=2, D=16, bs=16, seed=14)
    out_ref, lse_ref = run(ref)
    for bs in (32, 64, 256, 80):
        b = W.make_batch(q_lens, kv, Hq=4, Hkv=2, D=16, bs=bs, seed=14)
        b.q, b.k_tok, b.v_tok = ref.q, ref.k_tok, ref.v_tok
        o, l = run(b)
        assert torch.equal(o, out_ref) and torch.equal(l, lse_ref)
    # contiguous: request r is physical block r, block size >= every kv_len
    bsz = 80
    c = W.make_batch(q_lens, kv, Hq=4, Hkv=2, D=16, bs=bsz, seed=14)
    c.q, c.k_tok, c.v_tok = ref.q, ref.k_tok, ref.v_tok
    c.num_blocks = 3
    c.block_table = torch.arange(3, dtype=torch.int32).view(3, 1)
    c.slot_mapping = torch.cat([torch.arange(L) + r * bsz for r, L in enumerate(kv)]).to(torch.int64)
    o, l = run(c)
    assert torch.equal(o, out_ref) and torch.equal(l, lse_ref)


def _decode_split(b, kc, vc, split_blocks):
    """Attention of the decode query over keys [0, a) and [a, kv) separately,
    using a column-offset view of the block table for the second part
    (the cascade suffix trick, FlashAttention deep dive, cascade stage 2)."""
    a = split_blocks * b.bs
    lo = oracle.attention(b.q, kc, vc, b.cu_seqlens_q, torch.tensor([a], dtype=torch.int32),
                          b.block_table, b.softmax_scale, causal=False)
    hi_bt = b.block_table[:, split_blocks:].contiguous()
    hi = oracle.attention(b.q, kc, vc, b.cu_seqlens_q, b.seqused_k - a, hi_bt,
                          b.softmax_scale, causal=False)
    return lo, hi


def test_split_kv_merge_equals_unsplit():
    """multi-request page sec. 12 and the merge formula of the vLLM backend
    page: splitting the keys into segments and merging by log-sum-exp gives
    the unsplit result."""
    b = W.make_batch([1], [300], Hq=4, Hkv=2, D=32, bs=16, seed=15)
    kc, vc = cache_of(b)
    full, full_lse = run(b, kc, vc)
    for split_blocks in (1, 7, 18):
        (o1, l1), (o2, l2) = _decode_split(b, kc, vc, split_blocks)
        o, l = oracle.merge_states(o1.view(-1, 32), l1.view(-1), o2.view(-1, 32), l2.view(-1))
        np.testing.assert_allclose(o.numpy(), full.view(-1, 32).numpy(), rtol=0, atol=1e-13)
        np.testing.assert_allclose(l.numpy(), full_lse.view(-1).numpy(), rtol=0, atol=1e-12)
    # three segments, merged pairwise in either order
    a, c = 5 * 16, 12 * 16
    segs = []
    for lo_b, hi_tok in ((0, a), (5, c - a), (12, 300 - c)):
        bt = b.block_table[:, lo_b:].contiguous()
        segs.append(oracle.attention(b.q, kc, vc, b.cu_seqlens_q,
                                     torch.tensor([hi_tok], dtype=torch.int32), bt,
                                     b.softmax_scale, causal=False))
    (o1, l1), (o2, l2), (o3, l3) = [(o.view(-1, 32), l.view(-1)) for o, l in segs]
    o12, l12 = oracle.merge_states(o1, l1, o2, l2)
    oa, la = oracle.merge_states(o12, l12, o3, l3)
    o23, l23 = oracle.merge_states(o2, l2, o3, l3)
    ob, lb = oracle.merge_states(o1, l1, o23, l23)
    for o, l in ((oa, la), (ob, lb)):
        np.testing.assert_allclose(o.numpy(), full.view(-1, 32).numpy(), rtol=0, atol=1e-13)
        np.testing.assert_allclose(l.numpy(), full_lse.view(-1).numpy(), rtol=0, atol=1e-12)


def test_cascade_prefix_suffix_merge_equals_full():
    """vLLM backend page, cascade attention: stage 1 (all queries vs the
    shared prefix, non-causal, block_table[:1]), stage 2 (each request's
    suffix, causal, block_table[:, num_common_kv_blocks:]), stage 3 (merge)
    equals attention over prefix + suffix."""
    b = W.cascade_decode(B=6, prefix=128, lo=20, hi=70)
    b.bs = 64
    kc, vc = cache_of(b)
    full, full_lse = run(b, kc, vc)
    T, Hq, D = b.q.shape
    pre = oracle.attention(b.q, kc, vc, torch.tensor([0, T], dtype=torch.int32),
                           torch.tensor([128], dtype=torch.int32), b.block_table[:1],
                           b.softmax_scale, causal=False)
    nblk = 128 // b.bs
    suf = oracle.attention(b.q, kc, vc, b.cu_seqlens_q, b.seqused_k - 128,
                           b.block_table[:, nblk:].contiguous(), b.softmax_scale, causal=True)
    o, l = oracle.merge_states(pre[0].view(-1, D), pre[1].view(-1), suf[0].view(-1, D), suf[1].view(-1))
    np.testing.assert_allclose(o.numpy(), full.view(-1, D).numpy(), rtol=0, atol=1e-13)
    np.testing.assert_allclose(l.numpy(), full_lse.view(-1).numpy(), rtol=0, atol=1e-12)


def test_decode_equals_last_prefill_row():
    """multi-request page sec. 9: the decode query is the last row of the
    causal matrix, whose mask is all ones."""
    b = W.make_batch([9], [9], Hq=4, Hkv=1, D=16, bs=16, seed=16)
    kc, vc = cache_of(b)
    out, lse = run(b, kc, vc)
    d = W.make_batch([1], [9], Hq=4, Hkv=1, D=16, bs=16, seed=16)
    d.q = b.q[8:9].clone()
    d.block_table, d.num_blocks = b.block_table, b.num_blocks
    o, l = run(d, kc, vc)
    assert torch.equal(o[0], out[8]) and torch.equal(l[0], lse[8])


def test_row_subset_matches_full():
    b = W.make_batch([4, 6], [10, 6], Hq=2, Hkv=1, D=16, bs=16, seed=17)
    out, lse = run(b)
    rows = [9, 0, 4]
    o, l = run(b, rows=rows)
    assert torch.equal(o, out[rows]) and torch.equal(l, lse[rows])


# ------------------------------------------------------------------- merge

def test_merge_special_cases():
    rng = np.random.default_rng(18)
    o1, o2 = rng.normal(size=(3, 8)), rng.normal(size=(3, 8))
    l1 = np.array([-np.inf, 0.5, -np.inf])
    l2 = np.array([1.25, -np.inf, -np.inf])
    o, l = oracle.merge_states(torch.tensor(o1), torch.tensor(l1), torch.tensor(o2), torch.tensor(l2))
    assert np.array_equal(o[0].numpy(), o2[0]) and l[0] == 1.25
    assert np.array_equal(o[1].numpy(), o1[1]) and l[1] == 0.5
    assert np.array_equal(o[2].numpy(), np.zeros(8)) and l[2] == -np.inf
    # equal lse: plain average, lse + ln 2
    le = np.array([0.3, 0.3, 0.3])
    o, l = oracle.merge_states(torch.tensor(o1), torch.tensor(le), torch.tensor(o2), torch.tensor(le))
    np.testing.assert_allclose(o.numpy(), 0.5 * (o1 + o2), rtol=0, atol=1e-15)
    np.testing.assert_allclose(l.numpy(), 0.3 + math.log(2.0), rtol=0, atol=1e-15)
    # large lse values do not overflow
    lb = np.array([900.0, 1000.0, -1000.0])
    o, l = oracle.merge_states(torch.tensor(o1), torch.tensor(lb), torch.tensor(o2), torch.tensor(lb - 1.0))
    w = 1.0 / (1.0 + math.exp(-1.0))
    np.testing.assert_allclose(o.numpy(), w * o1 + (1 - w) * o2, rtol=0, atol=1e-12)


# -------------------------------------------------------------------- fp8

def _e4m3_brute(x: float) -> int:
    """Nearest e4m3 code by exhaustive search over the finite positive codes,
    ties to the even code (= even mantissa, codes are monotone in value),
    |x| >= 448 saturating."""
    a = abs(x)
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0
    vals = [(c, _e4m3_value_by_definition(c)) for c in range(0x7F)]
    if a >= 448.0:
        return sign | 0x7E
    best = min(vals, key=lambda cv: (abs(a - cv[1]), cv[0] & 1))
    return sign | best[0]


def _e4m3_value_by_definition(c):
    e, m = (c >> 3) & 15, c & 7
    v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
    return -v if c & 0x80 else v


def test_e4m3_decode_known_values():
    """FlashAttention deep dive, FP8 support: float8_e4m3fn (bias 7, no inf)."""
    assert oracle.e4m3_to_double(0x7E) == 448.0
    assert oracle.e4m3_to_double(0xFE) == -448.0
    assert oracle.e4m3_to_double(0x38) == 1.0
    assert oracle.e4m3_to_double(0x08) == 2.0 ** -6
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9
    assert oracle.e4m3_to_double(0x00) == 0.0
    assert math.isnan(oracle.e4m3_to_double(0x7F))
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert oracle.e4m3_to_double(c) == _e4m3_value_by_definition(c)
    # torch's independent table
    codes = torch.tensor([c for c in range(256) if c & 0x7F != 0x7F], dtype=torch.uint8)
    tv = codes.view(torch.float8_e4m3fn).double()
    assert [oracle.e4m3_to_double(int(c)) for c in codes] == tv.tolist()


def _fp16_value_by_definition(c):
    """IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits."""
    e, m = (c >> 10) & 31, c & 1023
    v = m * 2.0 ** -24 if e == 0 else (1 + m / 1024.0) * 2.0 ** (e - 15)
    return -v if c & 0x8000 else v


def test_fp16_storage_decodes_by_definition():
    """fp16 queries and caches ("FlashAttention deep dive", flash_attn_varlen_func:
    fp16 or bf16 inputs) are widened exactly.  A request with one visible key
    returns V_0 exactly, so a value row holding every finite binary16 code
    comes back as the codes' values; and with K_0 = 1 and scale 1 a query
    holding one code c has lse = value(c) exactly."""
    codes = np.array([c for c in range(1 << 16) if (c >> 10) & 31 != 31], dtype=np.uint16)
    want = [_fp16_value_by_definition(int(c)) for c in codes]
    assert want[:2] == [0.0, 2.0 ** -24] and 65504.0 in want and -1.0 in want
    as_fp16 = torch.from_numpy(codes.view(np.float16).copy())
    assert as_fp16.double().tolist() == want                  # torch's own widening agrees
    n = len(codes)
    one = torch.tensor([0], dtype=torch.int32)
    # values: one request, one key, D = every code
    q = torch.zeros((1, 1, n), dtype=torch.float16)
    kc = torch.zeros((1, 1, 1, n), dtype=torch.float16)
    vc = as_fp16.view(1, 1, 1, n)
    out, lse = oracle.attention(q, kc, vc, torch.tensor([0, 1]), torch.tensor([1]), one.view(1, 1), 1.0)
    assert out[0, 0].tolist() == want and float(lse[0, 0]) == 0.0
    # queries: n one-token requests on the same cached key K_0 = 1.0
    q = as_fp16.view(n, 1, 1)
    kc = torch.ones((1, 1, 1, 1), dtype=torch.float16)
    vc = torch.zeros_like(kc)
    cu = torch.arange(n + 1, dtype=torch.int32)
    out, lse = oracle.attention(q, kc, vc, cu, torch.ones(n, dtype=torch.int32),
                                torch.zeros((n, 1), dtype=torch.int32), 1.0)
    assert lse[:, 0].tolist() == want


def test_e4m3_encode_matches_brute_force_and_torch():
    rng = np.random.default_rng(19)
    xs = list(rng.normal(scale=50.0, size=600)) + list(rng.normal(scale=0.01, size=300))
    # exact midpoints between neighbouring codes (ties) and the subnormal range
    for c in range(0x7D):
        lo, hi = _e4m3_value_by_definition(c), _e4m3_value_by_definition(c + 1)
        xs += [0.5 * (lo + hi), -0.5 * (lo + hi), lo, hi * 0.999]
    xs += [0.0, -0.0, 447.9, 448.0, 449.0, 463.9, 464.0, 1e6, -1e6, 2.0 ** -10, 2.0 ** -11]
    xs = [float(np.float32(x)) for x in xs]
    for x in xs:
        assert oracle.e4m3_from_float(x) == _e4m3_brute(x), x
    inrange = torch.tensor([x for x in xs if abs(x) <= 448.0], dtype=torch.float32)
    want = inrange.to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    got = [oracle.e4m3_from_float(float(x)) for x in inrange]
    assert got == want


def test_fp8_kv_write_quantizes_x_over_scale():
    """FlashAttention deep dive, KV cache update: reshape_and_cache_flash
    with k_scale / v_scale.  Reading adopted: store e4m3(x / scale) with the
    division in fp32.  Keys use k_scale and values v_scale (the batch's two
    per-tensor scales differ)."""
    b = W.make_batch([2], [20], Hq=2, Hkv=2, D=16, bs=16, seed=20, kv_dtype="fp8")
    assert b.k_scale != b.v_scale
    kc, vc = cache_of(b)
    kb, vb = kc.view(torch.uint8), vc.view(torch.uint8)
    for t in range(20):
        slot = int(b.slot_mapping[t])
        for h in range(2):
            for d in range(16):
                x = np.float32(b.k_tok[t, h, d].float().item()) / np.float32(b.k_scale)
                assert int(kb[slot // 16, slot % 16, h, d]) == _e4m3_brute(float(x))
                y = np.float32(b.v_tok[t, h, d].float().item()) / np.float32(b.v_scale)
                assert int(vb[slot // 16, slot % 16, h, d]) == _e4m3_brute(float(y))
    # dequantised attention with an fp8 cache is the bf16 formula applied to
    # the widened values times the scale
    out, _ = run(b, kc, vc)
    deq_k = kc.double() * b.k_scale
    deq_v = vc.double() * b.v_scale
    q, s = b.q.double(), b.softmax_scale
    bt = b.block_table[0]
    rows_k = torch.stack([deq_k[bt[j // 16], j % 16] for j in range(20)])
    rows_v = torch.stack([deq_v[bt[j // 16], j % 16] for j in range(20)])
    for i in range(2):
        for h in range(2):
            n = 18 + i + 1
            sc = s * (rows_k[:n, h] @ q[i, h])
            p = torch.softmax(sc, 0)
            np.testing.assert_allclose(out[i, h].numpy(), (p @ rows_v[:n, h]).numpy(), atol=1e-12)


def test_kv_write_skips_negative_slots_and_rejects_out_of_range():
    k = W.randn((3, 1, 16), torch.Generator().manual_seed(21))
    kc = torch.zeros((2, 16, 1, 16), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    oracle.kv_write(k, k, kc, vc, torch.tensor([5, -1, 17]))
    assert torch.equal(kc[0, 5, 0], k[0, 0]) and torch.equal(kc[1, 1, 0], k[2, 0])
    assert int(torch.count_nonzero(kc.float())) == 32
    with pytest.raises(ValueError):
        oracle.kv_write(k, k, kc, vc, torch.tensor([0, 1, 32]))


# ------------------------------------------ variants: window, soft cap, sinks
# "FlashAttention deep dive", flash_attn_varlen_func arguments window_size,
# softcap and s_aux, and its table of supported variants (sliding window,
# soft cap, attention sinks); readings in oracle/attn_oracle.c.

def _dense(b, **kw):
    cuk = [0] + np.cumsum(b.kv_lens).tolist()
    return oracle.dense_masked_attention(b.q.double(), b.k_tok.double(), b.v_tok.double(),
                                         b.cu_seqlens_q.tolist(), cuk, b.softmax_scale,
                                         causal=b.causal, **kw)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("window,softcap,with_sinks", [
    ((3, -1), 0.0, False), ((0, -1), 0.0, False), ((5, 2), 0.0, False), ((-1, 1), 0.0, False),
    ((-1, -1), 2.5, False), ((-1, -1), 0.0, True), ((4, 0), 1.5, True), ((2, 3), 0.7, True)])
def test_variants_equal_dense_brute_force(causal, window, softcap, with_sinks):
    """The paged per-row oracle with a window, a soft cap and sinks equals
    the dense whole-matrix formulation (mask matrix, np.tanh on the score
    matrix, the sink as an extra score column with a zero value row)."""
    rng = np.random.default_rng(30 + int(causal))
    q_lens = [5, 1, 9, 3]
    kv = [12, 7, 9, 20]
    b = W.make_batch(q_lens, kv, Hq=6, Hkv=2, D=32, bs=16, seed=31, causal=causal)
    sinks = rng.normal(0.0, 1.5, 6) if with_sinks else None
    out, lse = run(b, window=window, softcap=softcap, sinks=sinks)
    ref, ref_lse, _ = _dense(b, window=window, softcap=softcap, sinks=sinks)
    np.testing.assert_allclose(out.numpy(), ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.numpy(), ref_lse, rtol=0, atol=1e-12)


def test_window_zero_left_returns_the_diagonal_value():
    """Causal with a window of no keys to the left: query i sees only its
    own position ctx + i, so out = V_{ctx+i} exactly and lse = its score."""
    b = W.make_batch([4, 2], [10, 2], Hq=2, Hkv=1, D=16, bs=16, seed=32)
    out, lse = run(b, window=(0, -1))
    t = 0
    for r, (ql, kl) in enumerate(zip(b.q_lens, b.kv_lens)):
        k, v = key_rows(b, r)
        for i in range(ql):
            j = kl - ql + i
            for h in range(2):
                assert torch.equal(out[t, h], v[j, 0].double())
                s = b.softmax_scale * float((b.q[t, h].double() * k[j, 0].double()).sum())
                assert abs(float(lse[t, h]) - s) < 1e-12
            t += 1


@pytest.mark.parametrize("window", [(0, 0), (2, 1), (-1, 3), (4, -1), (1, 40)])
def test_window_without_causal_bounds_both_sides(window):
    """Non-causal with a window (left, right): the query at absolute position
    p = ctx + i sees keys max(0, p - left) .. min(kv_len - 1, p + right).
    With q = 0 the scores tie: out = mean of those V rows, lse = ln(count);
    window (0, 0) returns V_p exactly.  Paged oracle and dense formulation."""
    left, right = window
    b = W.make_batch([5, 3], [12, 3], Hq=2, Hkv=1, D=16, bs=16, seed=35, causal=False)
    b.q.zero_()
    out, lse = run(b, window=window)
    dense, dense_lse, _ = _dense(b, window=window)
    t = 0
    for r, (ql, kl) in enumerate(zip(b.q_lens, b.kv_lens)):
        _, v = key_rows(b, r)
        for i in range(ql):
            p = kl - ql + i
            lo = 0 if left < 0 else max(0, p - left)
            hi = kl - 1 if right < 0 else min(kl - 1, p + right)
            want = v[lo:hi + 1, 0].double().mean(0)
            for h in range(2):
                if window == (0, 0):
                    assert torch.equal(out[t, h], v[p, 0].double())
                np.testing.assert_allclose(out[t, h].numpy(), want.numpy(), rtol=0, atol=1e-14)
                np.testing.assert_allclose(dense[t, h], want.numpy(), rtol=0, atol=1e-14)
                assert abs(float(lse[t, h]) - math.log(hi - lo + 1)) < 1e-13
                assert abs(float(dense_lse[t, h]) - math.log(hi - lo + 1)) < 1e-13
            t += 1


def test_wide_window_and_minus_inf_sink_change_nothing():
    """A window wider than every request, and sinks of -inf, select the
    same keys and weights as plain attention: results are identical."""
    b = W.make_batch([6, 1, 3], [9, 30, 3], Hq=4, Hkv=2, D=16, bs=16, seed=33)
    kc, vc = cache_of(b)
    out0, lse0 = run(b, kc, vc)
    out1, lse1 = run(b, kc, vc, window=(64, 64))
    out2, lse2 = run(b, kc, vc, sinks=[-math.inf] * 4)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
    assert torch.equal(out0, out2) and torch.equal(lse0, lse2)


def test_huge_softcap_is_no_cap():
    """c * tanh(s / c) -> s as c grows (the error is about s^3 / (3 c^2))."""
    b = W.make_batch([5], [11], Hq=2, Hkv=1, D=32, bs=16, seed=34)
    out0, lse0 = run(b)
    out1, lse1 = run(b, softcap=1e6)
    assert float((out0 - out1).abs().max()) < 1e-9
    assert float((lse0 - lse1).abs().max()) < 1e-9


@pytest.mark.parametrize("cap", [0.5, 3.0, 30.0])
def test_softcap_of_a_single_key_is_the_capped_logit(cap):
    """FlashAttention deep dive, argument table (softcap), as read: the cap
    maps the scaled logit s = scale * q . K to c * tanh(s / c).  Row 0 of a
    request without context sees only key 0, so its lse is exactly that
    capped logit and its output is V_0."""
    b = W.make_batch([3], [3], Hq=2, Hkv=1, D=32, bs=16, seed=42)
    b.q = (b.q.float() * 4).to(torch.bfloat16)          # raw logits of a few units
    out, lse = run(b, softcap=cap)
    k, v = key_rows(b, 0)
    for h in range(2):
        s = b.softmax_scale * float((b.q[0, h].double() * k[0, 0].double()).sum())
        assert abs(float(lse[0, h]) - cap * math.tanh(s / cap)) < 1e-12
        assert torch.equal(out[0, h], v[0, 0].double())


def test_softcap_bounds_every_logit():
    """With cap c every logit lies in (-c, c), so lse <= c + log(#keys)
    however large the raw scores are."""
    b = W.make_batch([3], [40], Hq=2, Hkv=1, D=32, bs=16, seed=35)
    b.q = (b.q.float() * 50).to(torch.bfloat16)       # raw scores in the hundreds
    out, lse = run(b, softcap=2.0)
    for i in range(3):
        nk = 40 - 3 + i + 1
        assert float(lse[i].max()) <= 2.0 + math.log(nk) + 1e-12


def test_sink_is_a_merge_with_an_empty_value_state():
    """A sink z joins the normalisation with value 0: the result equals the
    log-sum-exp merge ("FlashAttention deep dive", 合并算法) of the plain
    state with the state (out 0, lse z)."""
    b = W.make_batch([4, 2], [13, 2], Hq=4, Hkv=2, D=16, bs=16, seed=36)
    kc, vc = cache_of(b)
    z = [0.5, -2.0, 3.0, 1.0]
    out, lse = run(b, kc, vc, sinks=z)
    po, pl = run(b, kc, vc)
    T = b.q.shape[0]
    zl = torch.tensor(z, dtype=torch.float64).repeat(T)
    mo, ml = oracle.merge_states(po.reshape(-1, 16), pl.reshape(-1), torch.zeros(T * 4, 16,
                                 dtype=torch.float64), zl)
    assert float((out.reshape(-1, 16) - mo).abs().max()) < 1e-12
    assert float((lse.reshape(-1) - ml).abs().max()) < 1e-12


def test_sink_without_keys_gives_zero_and_the_sink():
    """No visible key but a sink: out = 0 and lse = z."""
    b = W.make_batch([2, 1], [2, 0], Hq=2, Hkv=1, D=16, bs=16, seed=37, causal=False)
    out, lse = run(b, sinks=[0.25, -1.0])
    assert torch.equal(out[2], torch.zeros(2, 16, dtype=torch.float64))
    assert lse[2].tolist() == [0.25, -1.0]


# ------------------------------------------------ fp8 queries with q_scale
# "FlashAttention deep dive", FA3 FP8 support (q_descale beside the k/v
# descales); "Making FlashAttention-4 faster for inference", PR 2109 (FP8
# inputs).  Value of an e4m3 query element = code * q_scale.

def test_fp8_query_with_scale_equals_its_bf16_value():
    """Scaling e4m3 codes by a power of two is exact in bf16 (4 significant
    bits into 8), so attention with (e4m3 q, q_scale = 2^-3) equals attention
    with the bf16 tensor holding code * 2^-3, bit for bit."""
    b = W.make_batch([5, 1, 9], [12, 30, 9], Hq=4, Hkv=2, D=32, bs=16, seed=38)
    kc, vc = cache_of(b)
    q8 = (b.q.float() * 8.0).to(torch.float8_e4m3fn)
    qv = (q8.float() * 0.125).to(torch.bfloat16)
    assert torch.equal(qv.float(), q8.float() * 0.125)
    out8, lse8 = oracle.attention(q8, kc, vc, b.cu_seqlens_q, b.seqused_k, b.block_table, b.softmax_scale,
                                  q_scale=0.125)
    b.q = qv
    outb, lseb = run(b, kc, vc)
    assert torch.equal(out8, outb) and torch.equal(lse8, lseb)


def test_fp8_query_scale_is_a_logit_scale():
    """q_scale multiplies every logit like softmax_scale does: (q_scale s,
    softmax_scale t) and (1, s * t) agree to rounding."""
    b = W.make_batch([4, 2], [20, 7], Hq=2, Hkv=1, D=16, bs=16, seed=39)
    kc, vc = cache_of(b)
    q8 = b.q.to(torch.float8_e4m3fn)
    o1, l1 = oracle.attention(q8, kc, vc, b.cu_seqlens_q, b.seqused_k, b.block_table, 0.25, q_scale=0.7)
    o2, l2 = oracle.attention(q8, kc, vc, b.cu_seqlens_q, b.seqused_k, b.block_table, 0.25 * 0.7)
    assert float((o1 - o2).abs().max()) < 1e-12 and float((l1 - l2).abs().max()) < 1e-12
