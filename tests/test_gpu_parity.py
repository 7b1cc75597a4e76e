"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs.

Tolerances: max-abs 1e-2 on out and lse for bf16/fp16 inputs (fp32
accumulation, N(0, 1) data); 4e-2 for the e4m3 KV path, where the oracle is
fed the same dequantised e4m3 values.  The bound is on the arithmetic: each
output element may in addition carry the rounding of the exact result to
the output type (half an ulp: 2^-9 of the magnitude for bf16), since a bf16
output above 2.56 cannot always lie within 1e-2 of the exact value.  KV
writes (slot_mapping scatter, e4m3 quantisation) must be bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import varlen_flashattention_causal_gb300 as va
from varlen_flashattention_causal_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = 1e-2
TOL_FP8 = 4e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from varlen_flashattention_causal_gb300 import build
    build.build()
    va.attn_device_error_flag(reset=True)
    yield
    torch.cuda.synchronize()


def cache_dtype(b):
    return torch.float8_e4m3fn if b.kv_dtype == "fp8" else b.k_tok.dtype


# Dirty memory.  A serving engine reuses cache pages and scratch across
# requests, so unwritten cache rows, workspace bytes and the memory around
# an output hold whatever was there before ("vLLM 中 Attention Kernel 如何
# 并行处理多个请求", sec. 11: pages are handed from request to request).
# The tests therefore fill caches, workspaces and output surroundings with
# quiet-NaN bit patterns: a kernel that reads an unwritten cache row into a
# result (even as 0 * NaN), reads workspace it did not write, or writes
# outside its output shows up as a NaN or as a changed guard.
NAN_BITS = {torch.bfloat16: (torch.int16, 0x7FC0), torch.float16: (torch.int16, 0x7E00),
            torch.float8_e4m3fn: (torch.uint8, 0x7F), torch.float32: (torch.int32, 0x7FC00000)}
GUARD = 3          # NaN rows before and after every output and lse buffer
PAD = 8            # NaN columns after each token row of a strided output


def nan_filled(shape, dtype, device="cuda"):
    it, bits = NAN_BITS[dtype]
    return torch.full(shape, bits, dtype=it, device=device).view(dtype)


def is_nan_pattern(t):
    it, bits = NAN_BITS[t.dtype]
    return bool((t.contiguous().view(it) == bits).all())


def same_bytes(a, b):
    return torch.equal(a.detach().cpu().contiguous().view(torch.uint8), b.detach().cpu().contiguous().view(torch.uint8))


def gpu_cache(b):
    kc = nan_filled((b.num_blocks, b.bs, b.Hkv, b.D), cache_dtype(b))
    vc = nan_filled((b.num_blocks, b.bs, b.Hkv, b.D), cache_dtype(b))
    va.kv_cache_write(b.k_tok.cuda(), b.v_tok.cuda(), kc, vc, b.slot_mapping.cuda(), b.k_scale, b.v_scale)
    return kc, vc


def cpu_cache(b):
    kc = nan_filled((b.num_blocks, b.bs, b.Hkv, b.D), cache_dtype(b), "cpu")
    vc = nan_filled((b.num_blocks, b.bs, b.Hkv, b.D), cache_dtype(b), "cpu")
    oracle.kv_write(b.k_tok, b.v_tok, kc, vc, b.slot_mapping, b.k_scale, b.v_scale)
    return kc, vc


class Guarded:
    """out [T, Hq, D] and lse [T, Hq] views into NaN-filled buffers with
    GUARD rows on each side (and, unless `contiguous`, PAD columns after each
    token row, so out has a token stride above Hq * D), plus a NaN-filled
    workspace of `ws_bytes` followed by guard bytes.  verify() checks that
    nothing outside out, lse and the workspace was written."""

    def __init__(self, T, Hq, D, dtype, ws_bytes=0, contiguous=False):
        pad = 0 if contiguous else PAD
        self.T, self.row = T, Hq * D
        self.o_full = nan_filled((T + 2 * GUARD, Hq * D + pad), dtype)
        self.out = self.o_full[GUARD:GUARD + T, :Hq * D].view(T, Hq, D)
        self.l_full = nan_filled((T + 2 * GUARD, Hq), torch.float32)
        self.lse = self.l_full[GUARD:GUARD + T]
        self.ws_full = torch.full((ws_bytes + 4096,), 0xFF, dtype=torch.uint8, device="cuda")
        self.ws = self.ws_full[:ws_bytes] if ws_bytes else None

    def verify(self):
        torch.cuda.synchronize()
        T = self.T
        assert is_nan_pattern(self.o_full[:GUARD]) and is_nan_pattern(self.o_full[GUARD + T:]), "write above/below out"
        if self.o_full.shape[1] > self.row:
            assert is_nan_pattern(self.o_full[:, self.row:]), "write into the padding of a token row"
        assert is_nan_pattern(self.l_full[:GUARD]) and is_nan_pattern(self.l_full[GUARD + T:]), "write around lse"
        assert bool((self.ws_full[self.ws_full.numel() - 4096:] == 0xFF).all()), "write past the workspace"


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def ws_bytes_for(T, Hq, D, B, max_q, max_k, Hkv, num_splits, q_dtype=None, kv_dtype=None):
    ns = num_splits if num_splits > 0 else va.attn_num_splits(B, max_q, max_k, Hq, Hkv, _sms(), D, q_dtype,
                                                              kv_dtype)
    return va.attn_workspace_size(T, Hq, D, ns)


def gpu_attn(b, kc, vc, num_splits=0, causal=None, q=None, block_table=None, seqused_k=None,
             cu=None, max_q=None, max_k=None, q_descale=1.0, **ext):
    """attn_varlen_prefill(_ext) on dirty memory: out and lse inside NaN guards
    (out with a padded token stride), a NaN-filled workspace; checks the
    guards after the call."""
    q = (b.q if q is None else q).cuda()
    T, Hq, D = q.shape
    odt = torch.bfloat16 if q.dtype == torch.float8_e4m3fn else q.dtype
    bt = (b.block_table if block_table is None else block_table).cuda()
    su = (b.seqused_k if seqused_k is None else seqused_k).cuda()
    cu = (b.cu_seqlens_q if cu is None else cu).cuda()
    mq = b.max_seqlen_q if max_q is None else max_q
    mk = b.max_seqlen_k if max_k is None else max_k
    g = Guarded(T, Hq, D, odt, ws_bytes_for(T, Hq, D, su.numel(), mq, mk, b.Hkv, num_splits, va._dt(q),
                                            va._dt(kc)))
    va.attn_varlen_prefill(q, kc, vc, g.out, cu, su, bt, mq, mk, b.softmax_scale,
                           causal=b.causal if causal is None else causal, lse_out=g.lse,
                           q_descale=q_descale,
                           k_descale=b.k_scale if b.kv_dtype == "fp8" else 1.0,
                           v_descale=b.v_scale if b.kv_dtype == "fp8" else 1.0,
                           num_splits=num_splits, workspace=g.ws, **ext)
    g.verify()
    return g.out, g.lse


def gpu_decode(b, kc, vc, num_splits=0, q=None):
    """attn_paged_decode on dirty memory (contiguous out inside NaN guard
    rows, NaN-filled workspace); checks the guards after the call."""
    q = (b.q if q is None else q).cuda()
    B, Hq, D = q.shape
    g = Guarded(B, Hq, D, q.dtype, ws_bytes_for(B, Hq, D, B, 1, b.max_seqlen_k, b.Hkv, num_splits, va._dt(q),
                                                va._dt(kc)),
                contiguous=True)
    va.attn_paged_decode(q, kc, vc, g.out, b.seqused_k.cuda(), b.block_table.cuda(), b.max_seqlen_k,
                         b.softmax_scale, lse_out=g.lse, num_splits=num_splits, workspace=g.ws,
                         k_descale=b.k_scale if b.kv_dtype == "fp8" else 1.0,
                         v_descale=b.v_scale if b.kv_dtype == "fp8" else 1.0)
    g.verify()
    return g.out, g.lse


def ref_attn(b, kc, vc, rows=None, causal=None):
    return oracle.attention(b.q, kc, vc, b.cu_seqlens_q, b.seqused_k, b.block_table, b.softmax_scale,
                            causal=b.causal if causal is None else causal,
                            k_scale=b.k_scale if b.kv_dtype == "fp8" else 1.0,
                            v_scale=b.v_scale if b.kv_dtype == "fp8" else 1.0, rows=rows)


def max_err(gpu, ref):
    g = gpu.detach().double().cpu()
    r = ref.double()
    both_inf = torch.isinf(g) & torch.isinf(r) & (torch.sign(g) == torch.sign(r))
    d = (g - r).abs()
    d[both_inf] = 0.0
    return float(d.max()) if d.numel() else 0.0


def half_ulp(ref, dtype):
    """Half a unit in the last place of `dtype` at the magnitude of each
    reference value: the error of rounding the exact result to the output
    type, which no kernel can avoid (bf16 keeps 8 significant bits, so an
    output of 4.05 cannot be closer than 0.0128 to the exact 4.0497)."""
    mant = {torch.bfloat16: 8, torch.float16: 11}.get(dtype)
    if mant is None:
        return torch.zeros_like(ref)
    e = torch.floor(torch.log2(ref.abs().clamp_min(1e-30)))
    return torch.pow(2.0, e - mant)


def check(out, lse, ref_out, ref_lse, tol, rows=None):
    """max-abs error within `tol` (the arithmetic's bound), plus the output
    type's own rounding of the reference (half an ulp, per element)."""
    if rows is not None:
        out, lse = out[rows], lse[rows]
    g = out.detach().double().cpu()
    r = ref_out.double()
    excess = (g - r).abs() - half_ulp(r, out.dtype)
    eo, el = float(excess.max()) if excess.numel() else 0.0, max_err(lse, ref_lse)
    assert eo <= tol and el <= tol, "max-abs error beyond output rounding: out %.3g lse %.3g (tol %.3g)" % (
        eo, el, tol)
    assert torch.isfinite(out.float()).all()
    return eo, el


def assert_no_device_error():
    assert va.attn_device_error_flag(reset=True) == 0


# ------------------------------------------------------------------ KV write

@pytest.mark.parametrize("kv_dtype,src", [("bf16", torch.bfloat16), ("fp16", torch.float16), ("fp8", torch.bfloat16)])
def test_kv_write_bit_exact(kv_dtype, src):
    b = W.make_batch([3, 1, 9], [70, 33, 200], Hq=8, Hkv=4, D=128, bs=32, seed=1, kv_dtype=kv_dtype, q_dtype=src)
    # padding tokens (slot -1) must be skipped
    b.slot_mapping = b.slot_mapping.clone()
    b.slot_mapping[::17] = -1
    g = gpu_cache(b)
    c = cpu_cache(b)
    assert torch.equal(g[0].view(torch.uint8).cpu(), c[0].view(torch.uint8))
    assert torch.equal(g[1].view(torch.uint8).cpu(), c[1].view(torch.uint8))
    assert_no_device_error()


def test_kv_write_strided_source_and_bad_slot():
    b = W.make_batch([2], [40], Hq=4, Hkv=2, D=64, bs=16, seed=2)
    # key/value as views into a wider per-token buffer (token stride > Hkv*D)
    wide = torch.zeros((40, 3, 2, 64), dtype=torch.bfloat16)
    wide[:, 0], wide[:, 2] = b.k_tok, b.v_tok
    wide = wide.cuda()
    kc = torch.zeros((b.num_blocks, 16, 2, 64), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    slots = b.slot_mapping.clone()
    slots[5] = b.num_blocks * 16 + 3          # outside the cache: must not be written
    va.kv_cache_write(wide[:, 0], wide[:, 2], kc, vc, slots.cuda())
    assert va.attn_device_error_flag(reset=True) & va.ERR_SLOT
    c = cpu_cache(b)
    ok = torch.ones(40, dtype=torch.bool)
    ok[5] = False
    good = b.slot_mapping[ok]
    kc_flat, ck_flat = kc.view(-1, 2, 64).cpu(), c[0].view(-1, 2, 64)
    assert torch.equal(kc_flat[good], ck_flat[good])
    s5 = int(b.slot_mapping[5])
    assert int(torch.count_nonzero(kc_flat[s5].float())) == 0


# --------------------------------------------------------------- workload 0

def test_tiny_packed_prefill_then_decode():
    pre, dec = W.tiny()
    kc, vc = gpu_cache(pre)
    ck, cv = cpu_cache(pre)
    out, lse = gpu_attn(pre, kc, vc)
    ro, rl = ref_attn(pre, ck, cv)
    check(out, lse, ro, rl, TOL)
    # one decode step: write each request's new token, attend over len + 1
    va.kv_cache_write(dec.k_tok.cuda(), dec.v_tok.cuda(), kc, vc, dec.slot_mapping.cuda())
    oracle.kv_write(dec.k_tok, dec.v_tok, ck, cv, dec.slot_mapping)
    assert same_bytes(kc, ck) and same_bytes(vc, cv)
    ro, rl = ref_attn(dec, ck, cv)
    out, lse = gpu_attn(dec, kc, vc)
    check(out, lse, ro, rl, TOL)
    o2, l2 = gpu_decode(dec, kc, vc)
    check(o2, l2, ro, rl, TOL)
    assert_no_device_error()


# --------------------------------------------------------- randomised cases

CASES = [
    # q_lens, kv_lens, Hq, Hkv, D, bs, causal
    ([6, 4], [6, 4], 4, 4, 64, 16, True),                       # the pages' 6 + 4 example, MHA
    ([1, 1, 1, 1, 1], [1, 17, 64, 65, 300], 8, 2, 128, 16, True),  # decode incl. kv_len 1
    ([5, 1, 70, 3], [5, 90, 200, 3], 8, 2, 64, 48, True),        # chunked prefill, odd block size
    ([16, 2, 33], [100, 2, 33], 16, 2, 128, 64, True),           # G = 8
    ([129, 64, 1], [129, 500, 257], 4, 1, 128, 256, True),       # several row blocks, ragged tails
    ([7, 9], [20, 9], 6, 3, 64, 32, False),                      # non-causal (cascade prefix stage)
    ([2, 3], [2, 3], 1, 1, 128, 16, True),                       # one head
    # rows-heavy requests (q_len * G > 64) run on the tcgen05 kernel
    ([300, 70], [300, 500], 8, 2, 128, 16, True),                # 16-row pages, 4 per K/V tile
    ([200], [100], 4, 1, 128, 64, True),                         # more queries than keys
    ([90, 150], [90, 150], 2, 2, 128, 32, False),                # G = 1, non-causal
    ([128, 129, 3], [1000, 129, 40], 16, 1, 128, 48, True),      # G = 16, block size 48
    ([70, 1], [0, 33], 8, 2, 128, 16, True),                     # kv_len 0 with many rows
    ([520], [777], 8, 2, 128, 256, True),                        # pages larger than a tile
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("num_splits", [1, 2, 7, 0])
def test_random_batches_against_oracle(case, num_splits):
    q_lens, kv_lens, Hq, Hkv, D, bs, causal = CASES[case]
    b = W.make_batch(q_lens, kv_lens, Hq, Hkv, D, bs, seed=100 + case, causal=causal)
    kc, vc = gpu_cache(b)
    ro, rl = ref_attn(b, *cpu_cache(b))
    out, lse = gpu_attn(b, kc, vc, num_splits=num_splits)
    check(out, lse, ro, rl, TOL)
    assert_no_device_error()


def test_fp16_path():
    b = W.make_batch([5, 1, 40], [50, 70, 40], 8, 2, 128, 32, seed=7, q_dtype=torch.float16)
    kc, vc = gpu_cache(b)
    ro, rl = ref_attn(b, *cpu_cache(b))
    for ns in (1, 3):
        out, lse = gpu_attn(b, kc, vc, num_splits=ns)
        assert out.dtype == torch.float16
        check(out, lse, ro, rl, TOL)


def test_fp16_single_token_calls():
    """A call in which every request has one query token (fp16): the 16-row
    CTAs run the two-stage configuration."""
    b = W.make_batch([1, 1, 1, 1], [300, 1, 77, 1000], 8, 2, 128, 16, seed=9, q_dtype=torch.float16)
    kc, vc = gpu_cache(b)
    ro, rl = ref_attn(b, *cpu_cache(b))
    for ns in (1, 4, 0):
        out, lse = gpu_attn(b, kc, vc, num_splits=ns)
        assert out.dtype == torch.float16
        check(out, lse, ro, rl, TOL)
    assert_no_device_error()


@pytest.mark.parametrize("D", [64, 128])
def test_fp8_kv_small(D):
    b = W.make_batch([1, 1, 12, 3], [200, 33, 64, 3], 8, 2, D, 32, seed=8, kv_dtype="fp8")
    kc, vc = gpu_cache(b)
    ck, cv = cpu_cache(b)
    assert torch.equal(kc.view(torch.uint8).cpu(), ck.view(torch.uint8))
    ro, rl = ref_attn(b, ck, cv)
    for ns in (1, 4):
        out, lse = gpu_attn(b, kc, vc, num_splits=ns)
        check(out, lse, ro, rl, TOL_FP8)


def test_fp8_kv_verify_rows():
    """e4m3 cache under verify-sized requests only (at most 8 query tokens,
    so at most 32 packed rows in the call): the 16-row CTAs and the 32-row
    CTAs whose key-slice pairs fetch and widen only their own rows, with bf16
    and with e4m3 queries."""
    b = W.make_batch([1, 5, 8, 3, 7, 1], [300, 64, 500, 40, 129, 2], 32, 8, 128, 16, seed=18, kv_dtype="fp8")
    kc, vc = gpu_cache(b)
    ck, cv = cpu_cache(b)
    ro, rl = ref_attn(b, ck, cv)
    for ns in (1, 0):
        out, lse = gpu_attn(b, kc, vc, num_splits=ns)
        check(out, lse, ro, rl, TOL_FP8)
    qs = float(b.q.float().abs().max()) / 448.0
    q8 = (b.q.float() / qs).to(torch.float8_e4m3fn)
    out, lse = _q8_call(b, q8, qs, kc, vc)
    ro8, rl8 = oracle.attention(q8, ck, cv, b.cu_seqlens_q, b.seqused_k, b.block_table, b.softmax_scale,
                                k_scale=b.k_scale, v_scale=b.v_scale, q_scale=qs)
    check(out, lse, ro8, rl8, TOL_FP8)
    assert_no_device_error()


@pytest.mark.parametrize("G,q_lens", [(1, [1, 8, 5, 9, 2]), (2, [1, 4, 3, 5, 1]), (4, [1, 2, 2, 3, 1]),
                                       (8, [1, 1, 2, 1, 1])])
@pytest.mark.parametrize("q_kind", ["bf16", "fp16", "e4m3"])
def test_fp8_rows_up_to_eight(G, q_lens, q_kind):
    """e4m3 cache, head size 128, requests of up to 8 packed rows (the
    transposed decode kernel: S^T = K Q^T, O^T = V^T P^T, 8-row CTAs) beside
    requests of 9 to 36 rows (the 16- and 64-row kernels), for G = 1, 2, 4, 8:
    the causal diagonal inside a tile (q_len > 1), kv_len below one tile,
    ragged tails, split and unsplit, against the oracle."""
    Hkv = 4
    kv_lens = [700, 64, 33, 1000, 9]
    qdt = torch.float16 if q_kind == "fp16" else torch.bfloat16
    b = W.make_batch(q_lens, kv_lens, G * Hkv, Hkv, 128, 16, seed=70 + G, kv_dtype="fp8", q_dtype=qdt)
    kc, vc = gpu_cache(b)
    ck, cv = cpu_cache(b)
    q, qs = b.q, 1.0
    if q_kind == "e4m3":
        qs = float(b.q.float().abs().max()) / 448.0
        q = (b.q.float() / qs).to(torch.float8_e4m3fn)
    ro, rl = oracle.attention(q, ck, cv, b.cu_seqlens_q, b.seqused_k, b.block_table, b.softmax_scale,
                              k_scale=b.k_scale, v_scale=b.v_scale, q_scale=qs)
    for ns in (1, 0, 5):
        out, lse = gpu_attn(b, kc, vc, num_splits=ns, q=q, q_descale=qs)
        check(out, lse, ro, rl, TOL_FP8)
    assert_no_device_error()


def test_fp8_paged_decode_entry_point():
    """attn_paged_decode (one token per request, no cu_seqlens) on an e4m3
    cache with bf16 queries, G = 4, split and unsplit, against the oracle."""
    b = W.make_batch([1] * 6, [1, 63, 64, 65, 777, 2048], 32, 8, 128, 16, seed=77, kv_dtype="fp8")
    kc, vc = gpu_cache(b)
    ro, rl = ref_attn(b, *cpu_cache(b))
    for ns in (1, 0, 4):
        out, lse = gpu_decode(b, kc, vc, num_splits=ns)
        check(out, lse, ro, rl, TOL_FP8)
    assert_no_device_error()


# ------------------------------------------------------------- edge cases

def test_empty_and_degenerate_requests():
    # request 1 has kv_len 0, request 2 has no query tokens, request 3 has
    # more queries than keys (negative context: its first rows see nothing)
    q_lens, kv_lens = [3, 1, 0, 5, 2], [10, 0, 7, 3, 2]
    b = W.make_batch(q_lens, kv_lens, 4, 2, 64, 16, seed=9)
    kc, vc = gpu_cache(b)
    ro, rl = ref_attn(b, *cpu_cache(b))
    for ns in (1, 3):
        out, lse = gpu_attn(b, kc, vc, num_splits=ns)
        check(out, lse, ro, rl, TOL)
        assert torch.equal(out[3].float().cpu(), torch.zeros(4, 64))
        assert torch.isinf(lse[3]).all() and (lse[3] < 0).all()
        assert torch.isinf(lse[4:6]).all()          # queries 0, 1 of request 3 see nothing
    assert_no_device_error()


def test_paged_layout_invariance_is_bitwise():
    """Same K/V in two different random block permutations (same block
    size and launch plan) gives bit-identical results."""
    b1 = W.make_batch([1, 4, 9], [300, 77, 160], 8, 2, 128, 16, seed=10)
    b2 = W.make_batch([1, 4, 9], [300, 77, 160], 8, 2, 128, 16, seed=11)
    b2.q, b2.k_tok, b2.v_tok = b1.q, b1.k_tok, b1.v_tok
    assert not torch.equal(b1.block_table, b2.block_table)
    o1, l1 = gpu_attn(b1, *gpu_cache(b1), num_splits=3)
    o2, l2 = gpu_attn(b2, *gpu_cache(b2), num_splits=3)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # a different block size changes only the rounding, within tolerance
    b3 = W.make_batch([1, 4, 9], [300, 77, 160], 8, 2, 128, 256, seed=12)
    b3.q, b3.k_tok, b3.v_tok = b1.q, b1.k_tok, b1.v_tok
    o3, l3 = gpu_attn(b3, *gpu_cache(b3), num_splits=3)
    assert max_err(o3, o1.double().cpu()) <= TOL and max_err(l3, l1.double().cpu()) <= TOL


def test_decode_equals_last_row_of_prefill():
    b = W.make_batch([64], [64], 8, 2, 128, 16, seed=12)
    kc, vc = gpu_cache(b)
    out, lse = gpu_attn(b, kc, vc, num_splits=1)
    d_out, d_lse = gpu_decode(b, kc, vc, num_splits=1, q=b.q[63:64])
    assert max_err(d_out[0], out[63].double().cpu()) <= 4e-3
    assert max_err(d_lse[0], lse[63].double().cpu()) <= 1e-4


def test_out_of_range_block_id_reads_zeros_and_is_flagged():
    """A block id outside [0, num_blocks) is never dereferenced: its rows
    read as zero K and V, and the device error word records it."""
    b = W.make_batch([1, 1], [64, 64], 4, 1, 64, 16, seed=13)
    kc, vc = gpu_cache(b)
    bad = b.block_table.clone()
    bad[1, 2] = b.num_blocks + 5         # keys 32..47 of request 1 point outside the pool
    out, lse = gpu_attn(b, kc, vc, block_table=bad, num_splits=1)
    assert va.attn_device_error_flag(reset=True) & va.ERR_BLOCK_ID
    assert torch.isfinite(out.float()).all()
    ck, cv = cpu_cache(b)
    ro, rl = ref_attn(b, ck, cv)
    check(out[:1], lse[:1], ro[:1], rl[:1], TOL)          # request 0 untouched
    # request 1 equals the oracle on a cache whose block 2 of that row is zero
    blk = int(b.block_table[1, 2])
    ck[blk] = 0
    cv[blk] = 0
    ro, rl = ref_attn(b, ck, cv)
    check(out[1:], lse[1:], ro[1:], rl[1:], TOL)


def test_out_of_range_block_id_fp8_decode_rows():
    """The same contract on the e4m3 decode path (rows <= 8, head size 128):
    the bad block's 16 slots read as zero K and V, the error word records it,
    the other requests are untouched."""
    b = W.make_batch([1, 1, 2], [100, 64, 90], 16, 4, 128, 16, seed=14, kv_dtype="fp8")
    kc, vc = gpu_cache(b)
    bad = b.block_table.clone()
    bad[1, 1] = b.num_blocks + 7         # keys 16..31 of request 1
    out, lse = gpu_attn(b, kc, vc, block_table=bad, num_splits=1)
    assert va.attn_device_error_flag(reset=True) & va.ERR_BLOCK_ID
    assert torch.isfinite(out.float()).all()
    ck, cv = cpu_cache(b)
    ro, rl = ref_attn(b, ck, cv)
    keep = torch.tensor([True, False, True, True])    # tokens of requests 0 and 2
    check(out[keep], lse[keep], ro[keep], rl[keep], TOL_FP8)
    blk = int(b.block_table[1, 1])
    ck[blk] = 0
    cv[blk] = 0
    ro, rl = ref_attn(b, ck, cv)
    check(out[1:2], lse[1:2], ro[1:2], rl[1:2], TOL_FP8)


def test_debug_validation_refuses_bad_tables_and_launches_nothing(monkeypatch):
    """With ATTN_DEBUG_VALIDATE=1 the entry points copy their integer tables
    to the host and refuse a call that breaks the contract (ATTN_ERR_TABLE)
    before anything is launched: out, lse, the workspace and the cache keep
    their bytes and the device error word stays clear.  A valid call runs
    and gives the same bytes as without the check, and a call captured into
    a CUDA graph is not checked (no host synchronisation under capture)."""
    b = W.make_batch([5, 1, 140], [64, 300, 140], 8, 2, 128, 16, seed=21)
    kc, vc = gpu_cache(b)
    ref_out, ref_lse = gpu_attn(b, kc, vc, num_splits=1)
    va.attn_device_error_flag(reset=True)
    monkeypatch.setenv("ATTN_DEBUG_VALIDATE", "1")
    out, lse = gpu_attn(b, kc, vc, num_splits=1)
    assert same_bytes(out, ref_out) and same_bytes(lse, ref_lse)

    bt, su, cu = b.block_table.clone(), b.seqused_k.clone(), b.cu_seqlens_q.clone()
    bt[1, 3] = b.num_blocks                      # a block id the request reads, outside the pool
    su_short = su.clone()
    su_short[2] = 139                            # 140 new tokens, 139 cached keys
    cu_bad = cu.clone()
    cu_bad[0] = 1                                # cu_seqlens_q must start at 0
    T, Hq, D = b.q.shape
    cases = [dict(bt=bt), dict(mk=b.max_seqlen_k - 1), dict(mq=b.max_seqlen_q - 1), dict(su=su_short),
             dict(cu=cu_bad)]
    for c in cases:
        g = Guarded(T, Hq, D, b.q.dtype, va.attn_workspace_size(T, Hq, D, 1))
        with pytest.raises(va.AttnError) as e:
            va.attn_varlen_prefill(b.q.cuda(), kc, vc, g.out, c.get("cu", cu).cuda(), c.get("su", su).cuda(),
                                   c.get("bt", b.block_table).cuda(), c.get("mq", b.max_seqlen_q),
                                   c.get("mk", b.max_seqlen_k), b.softmax_scale, lse_out=g.lse,
                                   num_splits=1, workspace=g.ws)
        assert e.value.status == va.ATTN_ERR_TABLE, c.keys()
        g.verify()
        assert is_nan_pattern(g.out) and is_nan_pattern(g.lse)
        assert bool((g.ws_full == 0xFF).all())
    # decode with the bad block id
    qd = b.q[:3].contiguous().cuda()
    od = nan_filled((3, Hq, D), b.q.dtype)
    with pytest.raises(va.AttnError) as e:
        va.attn_paged_decode(qd, kc, vc, od, su.cuda(), bt.cuda(), b.max_seqlen_k, b.softmax_scale, num_splits=1)
    assert e.value.status == va.ATTN_ERR_TABLE and is_nan_pattern(od)
    # KV write with a slot past the cache
    k0, v0 = kc.clone(), vc.clone()
    slots = b.slot_mapping.clone()
    slots[7] = b.num_blocks * b.bs
    with pytest.raises(va.AttnError) as e:
        va.kv_cache_write(b.k_tok.cuda(), b.v_tok.cuda(), kc, vc, slots.cuda())
    assert e.value.status == va.ATTN_ERR_TABLE
    assert same_bytes(kc, k0) and same_bytes(vc, v0)
    torch.cuda.synchronize()
    assert va.attn_device_error_flag(reset=True) == 0

    # under capture: not checked, and the replay gives the same bytes
    g = Guarded(T, Hq, D, b.q.dtype, va.attn_workspace_size(T, Hq, D, 1))
    args = (b.q.cuda(), kc, vc, g.out, cu.cuda(), su.cuda(), b.block_table.cuda(), b.max_seqlen_q,
            b.max_seqlen_k, b.softmax_scale)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            va.attn_varlen_prefill(*args, lse_out=g.lse, num_splits=1, workspace=g.ws)
    graph.replay()
    g.verify()
    assert same_bytes(g.out, ref_out) and same_bytes(g.lse, ref_lse)


# ------------------------------------------------------------------- merge

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_merge_states_against_oracle(dtype):
    g = torch.Generator().manual_seed(14)
    T, Hq, D = 37, 8, 128
    o1 = torch.randn((T, Hq, D), generator=g).to(dtype)
    o2 = torch.randn((T, Hq, D), generator=g).to(dtype)
    l1 = torch.randn((T, Hq), generator=g) * 5
    l2 = torch.randn((T, Hq), generator=g) * 5
    l1[0, :3] = -math.inf
    l2[0, 1:5] = -math.inf
    g = Guarded(T, Hq, D, dtype, contiguous=True)
    out, lo = g.out, g.lse
    va.attn_merge_states(out, lo, o1.cuda(), l1.cuda(), o2.cuda(), l2.cuda())
    g.verify()
    ro, rl = oracle.merge_states(o1.view(-1, D), l1.view(-1), o2.view(-1, D), l2.view(-1))
    tol = 1e-2 if dtype != torch.float32 else 1e-5
    assert max_err(out.view(-1, D), ro) <= tol
    assert max_err(lo.view(-1), rl) <= 1e-5
    # in place: out aliases o1
    a = o1.cuda()
    va.attn_merge_states(a, None, a, l1.cuda(), o2.cuda(), l2.cuda())
    assert torch.equal(a, out)


# ------------------------------------------------------ full-size workloads

def _rows_sample(b, n, seed):
    """Seeded sample of packed rows: every request's first and last query
    plus uniformly drawn rows."""
    cu = b.cu_seqlens_q.tolist()
    rows = set()
    for r in range(b.B):
        if cu[r + 1] > cu[r]:
            rows.update([cu[r], cu[r + 1] - 1])
    g = torch.Generator().manual_seed(seed)
    rows.update(torch.randint(0, b.T, (n,), generator=g).tolist())
    return sorted(rows)


def test_workload1_llama8b_decode_full():
    b = W.decode_llama8b()
    kc, vc = gpu_cache(b)
    ck, cv = cpu_cache(b)
    assert same_bytes(kc, ck) and same_bytes(vc, cv)
    ro, rl = ref_attn(b, ck, cv)
    out, lse = gpu_decode(b, kc, vc)
    check(out, lse, ro, rl, TOL)
    assert_no_device_error()


@pytest.fixture(scope="module")
def longctx_ref():
    b = W.decode_longctx(bs=16)
    ck, cv = cpu_cache(b)
    ro, rl = ref_attn(b, ck, cv)
    return b, ro, rl


@pytest.mark.parametrize("bs", [16, 64, 256])
def test_workload2_longctx_decode_full(longctx_ref, bs):
    # the oracle is layout-invariant (pinned), so the bs = 16 reference
    # serves every block size
    b16, ro, rl = longctx_ref
    b = W.decode_longctx(bs=bs, gen_kv=False)
    b.q = b16.q
    positions = [range(L) for L in b.kv_lens]
    b.slot_mapping = torch.cat([W.slots(b.block_table, r, p, bs) for r, p in enumerate(positions)])
    b.k_tok, b.v_tok = b16.k_tok, b16.v_tok
    kc, vc = gpu_cache(b)
    out, lse = gpu_decode(b, kc, vc)
    check(out, lse, ro, rl, TOL)
    assert_no_device_error()


def segment_keys(max_k, n, tile=64):
    """Keys per split-KV segment for n segments of a call whose longest
    request has max_k keys: the keys cut evenly, rounded up to whole 64-key
    tiles (the library's host planning rule for an explicit num_splits)."""
    per = -(-max_k // n)
    return -(-per // tile) * tile


def boundary_rows(b, n_segments=1, per_request=256, seed=3, tile_rows=128):
    """Token rows of a prefill batch where a tiled kernel is most likely to
    go wrong, plus a seeded random sample.  For every request:
      - both sides of every 128-packed-row Q-tile boundary (packed rows
        128k - 1 and 128k, i.e. tokens (128k - 1) // G and 128k // G); every
        second one is also a 256-row work-item boundary;
      - with n_segments > 1: the tokens whose causal limit ctx + i is the
        last key of a segment, the first key of the next one, and the first
        key of the segment's last 64-key tile;
      - its first and last token, and per_request seeded random tokens.
    Returns sorted packed token indices."""
    G = b.Hq // b.Hkv
    cu = b.cu_seqlens_q.tolist()
    g = torch.Generator().manual_seed(W.SEED0 + 900 + seed)
    chunk = segment_keys(b.max_seqlen_k, n_segments) if n_segments > 1 else None
    rows = set()
    for r in range(b.B):
        q0, ql, kv = cu[r], cu[r + 1] - cu[r], b.kv_lens[r]
        if ql <= 0:
            continue
        ctx = kv - ql
        local = {0, ql - 1}
        for pr in range(tile_rows, ql * G, tile_rows):
            local.update([(pr - 1) // G, pr // G])
        if chunk:
            for end in range(chunk, kv + chunk, chunk):
                local.update([end - 1 - ctx, end - ctx, end - 64 - ctx])
        local.update(torch.randint(0, ql, (per_request,), generator=g).tolist())
        rows.update(q0 + i for i in local if 0 <= i < ql)
    return sorted(rows)


@pytest.fixture(scope="module")
def chunked_ref():
    """The chunked prefill batch and the oracle on the union of the boundary
    rows of every split setting tested below (computed once: about 7,800
    token rows x 32 heads over up to 12k keys, fp64)."""
    b = W.chunked_prefill()
    rows = sorted(set(boundary_rows(b, 1)) | set(boundary_rows(b, 3)))
    ro, rl = ref_attn(b, *cpu_cache(b), rows=rows)
    return b, rows, ro, rl


@pytest.mark.parametrize("num_splits", [1, 3, 0])
def test_workload3_chunked_prefill_full_sampled(chunked_ref, num_splits):
    """The chunked prefill workload at full size (16 requests, 1k-8k new
    tokens on 0-4k cached), compared with the oracle on every Q-tile and
    work-item boundary row, the rows at split-segment edges and 256 seeded
    rows per request (all heads, out and lse); caches, workspace and the
    memory around out are dirty (NaN patterns)."""
    b, rows, ro, rl = chunked_ref
    kc, vc = gpu_cache(b)
    out, lse = gpu_attn(b, kc, vc, num_splits=num_splits)
    mine = boundary_rows(b, n_segments=num_splits)
    at = {r: i for i, r in enumerate(rows)}
    idx = torch.tensor([at[r] for r in mine])
    check(out, lse, ro[idx], rl[idx], TOL, rows=mine)
    assert_no_device_error()


def test_workload3_cascade_decode_full():
    b = W.cascade_decode()
    kc, vc = gpu_cache(b)
    ck, cv = cpu_cache(b)
    ro, rl = ref_attn(b, ck, cv)            # plain attention over prefix + suffix
    P = b.extra["prefix"]
    nblk = P // b.bs
    T, Hq, D = b.q.shape
    q = b.q.cuda()
    # stage 1: every query against the shared prefix, non-causal, first row of the block table
    pre_o = torch.empty_like(q)
    pre_l = torch.empty((T, Hq), dtype=torch.float32, device="cuda")
    va.attn_varlen_prefill(q, kc, vc, pre_o, torch.tensor([0, T], dtype=torch.int32, device="cuda"),
                           torch.tensor([P], dtype=torch.int32, device="cuda"), b.block_table[:1].cuda(),
                           T, P, b.softmax_scale, causal=False, lse_out=pre_l)
    # stage 2: each request's own suffix, causal, column-offset block table view
    suf_o = torch.empty_like(q)
    suf_l = torch.empty((T, Hq), dtype=torch.float32, device="cuda")
    bt = b.block_table.cuda()
    va.attn_varlen_prefill(q, kc, vc, suf_o, b.cu_seqlens_q.cuda(), (b.seqused_k - P).cuda(), bt[:, nblk:],
                           1, b.max_seqlen_k - P, b.softmax_scale, causal=True, lse_out=suf_l)
    out = torch.empty_like(q)
    lse = torch.empty((T, Hq), dtype=torch.float32, device="cuda")
    va.attn_merge_states(out, lse, pre_o, pre_l, suf_o, suf_l)
    check(out, lse, ro, rl, TOL)
    assert_no_device_error()

    # the same step captured in a CUDA graph with the prefix call on a second
    # stream (joined before the merge), as the benchmark times it: with the
    # automatic split counts the same kernels compute the same items, so the
    # result is bit-identical; with 4 prefix and 2 suffix segments (the
    # benchmark's pair) it matches the oracle
    pre_o2, suf_o2, out2 = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    pre_l2, suf_l2, lse2 = (torch.empty((T, Hq), dtype=torch.float32, device="cuda") for _ in range(3))
    cu0 = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    su0 = torch.tensor([P], dtype=torch.int32, device="cuda")
    cu, su = b.cu_seqlens_q.cuda(), (b.seqused_k - P).cuda()
    side = torch.cuda.Stream()
    for ns_pre, ns_suf in ((0, 0), (4, 2)):
        def step():
            cur = torch.cuda.current_stream()
            side.wait_stream(cur)
            with torch.cuda.stream(side):
                va.attn_varlen_prefill(q, kc, vc, pre_o2, cu0, su0, bt[:1], T, P, b.softmax_scale, causal=False,
                                       lse_out=pre_l2, num_splits=ns_pre)
            va.attn_varlen_prefill(q, kc, vc, suf_o2, cu, su, bt[:, nblk:], 1, b.max_seqlen_k - P,
                                   b.softmax_scale, causal=True, lse_out=suf_l2, num_splits=ns_suf)
            cur.wait_stream(side)
            va.attn_merge_states(out2, lse2, pre_o2, pre_l2, suf_o2, suf_l2)

        warm = torch.cuda.Stream()
        warm.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(warm):
            step()
        torch.cuda.current_stream().wait_stream(warm)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            out2.zero_()
            g.replay()
            torch.cuda.synchronize()
            if ns_pre == 0:
                assert torch.equal(out2, out) and torch.equal(lse2, lse)
            else:
                check(out2, lse2, ro, rl, TOL)
        assert_no_device_error()


def test_cascade_entry_point_against_oracle():
    """attn_cascade: the shared prefix and every request's suffix in one
    call, their segments merged by one combine ("FlashAttention deep
    dive", Cascade Attention), against plain attention over prefix + suffix:
    the library's split counts and explicit ones, with and without a second
    stream for the prefix half, and as a CUDA graph replayed three times
    (bit-identical to the eager call with the same counts)."""
    b = W.cascade_decode()
    kc, vc = gpu_cache(b)
    ck, cv = cpu_cache(b)
    ro, rl = ref_attn(b, ck, cv)
    P = b.extra["prefix"]
    nblk = P // b.bs
    T, Hq, D = b.q.shape
    q, bt = b.q.cuda(), b.block_table.cuda()
    cu0 = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    pk = torch.tensor([P], dtype=torch.int32, device="cuda")
    cu, su = b.cu_seqlens_q.cuda(), (b.seqused_k - P).cuda()
    auto = va.attn_cascade_splits(b.B, T, 1, P, b.max_seqlen_k - P, Hq, b.Hkv, D)
    aux = torch.cuda.Stream()

    def call(g, nsp, nss, use_aux):
        va.attn_cascade(q, kc, vc, g.out, cu0, pk, bt[0], P, cu, su, bt[:, nblk:], 1, b.max_seqlen_k - P,
                        b.softmax_scale, lse_out=g.lse, prefix_splits=nsp, suffix_splits=nss, workspace=g.ws,
                        aux_stream=aux if use_aux else None)

    ref_auto = None
    for nsp, nss, use_aux in ((0, 0, True), (0, 0, False), (1, 1, True), (4, 2, True), (8, 8, False)):
        tot = (nsp or auto[0]) + (nss or auto[1])
        g = Guarded(T, Hq, D, b.q.dtype, va.attn_workspace_size(T, Hq, D, tot))
        call(g, nsp, nss, use_aux)
        g.verify()
        check(g.out, g.lse, ro, rl, TOL)
        if nsp == 0 and use_aux:
            ref_auto = (g.out.clone(), g.lse.clone())
        elif nsp == 0:
            assert torch.equal(g.out, ref_auto[0]) and torch.equal(g.lse, ref_auto[1])
    assert_no_device_error()

    g = Guarded(T, Hq, D, b.q.dtype, va.attn_workspace_size(T, Hq, D, auto[0] + auto[1]))
    warm = torch.cuda.Stream()
    warm.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(warm):
        call(g, 0, 0, True)
    torch.cuda.current_stream().wait_stream(warm)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(g, 0, 0, True)
    for _ in range(3):
        g.out.fill_(0)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(g.out, ref_auto[0]) and torch.equal(g.lse, ref_auto[1])
    g.verify()
    assert_no_device_error()


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_cascade_entry_point_other_shapes(kv_dtype):
    """attn_cascade beyond decode: suffixes of several query tokens (one
    request above 64 packed rows, so the suffix half also runs a tensor-core
    class beside the prefix half's), on a bf16 or e4m3 cache, and an empty
    prefix (prefix_len 0: the prefix half contributes no key)."""
    bs = 32
    P = 4 * bs
    q_lens = [1, 3, 40, 7]
    suf = [50, 3, 300, 20]
    kv = [P + s for s in suf]
    g = W.generator(171)
    npre = P // bs
    used = npre + sum((L + bs - 1) // bs - npre for L in kv)
    bt = W.block_tables(kv, bs, used + 8, g, shared_prefix_blocks=npre)
    b = W.Batch("cascade-shapes", 32, 8, 128, bs, used + 8, q_lens, kv, block_table=bt, kv_dtype=kv_dtype)
    # the shared prefix's keys are written once (row 0), each suffix's per row
    b = W._finish(b, g, "cpu", [range(L) if r == 0 else range(P, L) for r, L in enumerate(kv)])
    kc, vc = gpu_cache(b)
    ck, cv = cpu_cache(b)
    ro, rl = ref_attn(b, ck, cv)
    tol = TOL_FP8 if kv_dtype == "fp8" else TOL
    T, Hq, D = b.q.shape
    q, btd = b.q.cuda(), b.block_table.cuda()
    cu = b.cu_seqlens_q.cuda()
    kd = b.k_scale if kv_dtype == "fp8" else 1.0
    vd = b.v_scale if kv_dtype == "fp8" else 1.0
    for pl in (P, 0):
        nb = pl // bs
        cu0 = torch.tensor([0, T], dtype=torch.int32, device="cuda")
        pk = torch.tensor([pl], dtype=torch.int32, device="cuda")
        su = (b.seqused_k - pl).cuda()
        for nsp, nss in ((0, 0), (2, 3)):
            auto = va.attn_cascade_splits(b.B, T, max(q_lens), pl, max(kv) - pl, Hq, b.Hkv, D,
                                          q_dtype=va.ATTN_BF16, kv_dtype=va.ATTN_FP8_E4M3 if kv_dtype == "fp8" else va.ATTN_BF16)
            tot = (nsp or auto[0]) + (nss or auto[1])
            g = Guarded(T, Hq, D, b.q.dtype, va.attn_workspace_size(T, Hq, D, tot))
            va.attn_cascade(q, kc, vc, g.out, cu0, pk, btd[0], pl, cu, su, btd[:, nb:], max(q_lens), max(kv) - pl,
                            b.softmax_scale, lse_out=g.lse, k_descale=kd, v_descale=vd, prefix_splits=nsp,
                            suffix_splits=nss, workspace=g.ws, aux_stream=torch.cuda.Stream())
            g.verify()
            check(g.out, g.lse, ro, rl, tol)
    assert_no_device_error()


def test_workload4_fp8_mixed_full_sampled():
    b = W.fp8_mixed()
    kc, vc = gpu_cache(b)
    ck, cv = cpu_cache(b)
    assert torch.equal(kc.view(torch.uint8).cpu(), ck.view(torch.uint8))
    assert torch.equal(vc.view(torch.uint8).cpu(), cv.view(torch.uint8))
    out, lse = gpu_attn(b, kc, vc)
    # every decode row; the chunks' Q-tile and item boundary rows plus 32
    # seeded rows each
    rows = boundary_rows(b, per_request=32, seed=4)
    ro, rl = ref_attn(b, ck, cv, rows=rows)
    check(out, lse, ro, rl, TOL_FP8, rows=rows)
    assert_no_device_error()


def test_short_segments_repeated_are_stable():
    """Many tensor-core CTAs with only two K/V tiles each (64 queries x 4
    heads against 4096 keys, 32 segments), called repeatedly: every call
    must match the oracle -- a pipeline that reads O before its last P V
    lands would fail intermittently here."""
    b = W.make_batch([64], [4096], 32, 8, 128, 64, seed=15, causal=False)
    kc, vc = gpu_cache(b)
    ro, rl = ref_attn(b, *cpu_cache(b))
    for it in range(12):
        out, lse = gpu_attn(b, kc, vc, num_splits=(32, 0, 16)[it % 3])
        check(out, lse, ro, rl, TOL)
    assert_no_device_error()


@pytest.mark.parametrize("q_dtype,bs", [(torch.bfloat16, 32), (torch.float16, 16), (torch.bfloat16, 48),
                                        (torch.bfloat16, 256)])
def test_fp8_kv_rows_heavy(q_dtype, bs):
    """e4m3 caches under rows-heavy requests (the tensor-core path widens
    the staged e4m3 tiles to fp16): prefill, chunked prefill with context,
    a ragged tail, next to decode rows in the same batch."""
    b = W.make_batch([300, 70, 1, 129], [300, 500, 1000, 200], 8, 2, 128, bs, seed=16, kv_dtype="fp8",
                     q_dtype=q_dtype)
    kc, vc = gpu_cache(b)
    ck, cv = cpu_cache(b)
    assert torch.equal(kc.view(torch.uint8).cpu(), ck.view(torch.uint8))
    ro, rl = ref_attn(b, ck, cv)
    for ns in (1, 3, 0):
        out, lse = gpu_attn(b, kc, vc, num_splits=ns)
        assert out.dtype == q_dtype
        check(out, lse, ro, rl, TOL_FP8)
    assert_no_device_error()


def test_cuda_graph_capture_and_replay():
    """A whole step -- the KV write of the batch's tokens, then one mixed
    call (decode rows, a chunk with context, a prefill; split-KV and its
    combine) -- captured once in a CUDA graph and replayed.  Capture fails
    if the path synchronises the host or allocates; every replay reuses the
    tensor-core kernel's ticket counter, which must have rewound itself."""
    b = W.make_batch([300, 1, 1, 40, 1], [700, 900, 64, 40, 2000], 32, 8, 128, 16, seed=17)
    kc, vc = gpu_cache(b)
    ro, rl = ref_attn(b, *cpu_cache(b))
    dev = torch.device("cuda")
    q = b.q.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    cu, su, bt = b.cu_seqlens_q.to(dev), b.seqused_k.to(dev), b.block_table.to(dev)
    kt, vt, sl = b.k_tok.to(dev), b.v_tok.to(dev), b.slot_mapping.to(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ns = va.attn_num_splits(b.B, b.max_seqlen_q, b.max_seqlen_k, b.Hq, b.Hkv, sms)
    ws = torch.empty(max(1, va.attn_workspace_size(b.T, b.Hq, b.D, max(ns, 2))), dtype=torch.uint8, device=dev)

    def step():
        va.kv_cache_write(kt, vt, kc, vc, sl)
        va.attn_varlen_prefill(q, kc, vc, out, cu, su, bt, b.max_seqlen_q, b.max_seqlen_k, b.softmax_scale,
                               causal=True, lse_out=lse, num_splits=0, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(4):
        out.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        check(out, lse, ro, rl, TOL)
    assert_no_device_error()


def test_tensor_core_repeated_calls_on_one_workspace():
    """Many consecutive calls on one workspace: each call zeroes the
    tensor-core kernel's work counter in the workspace before its launch,
    so no call inherits a counter from the one before and every output is
    bitwise the first (which matches the oracle)."""
    b = W.make_batch([130, 200, 1], [400, 260, 300], 8, 2, 128, 16, seed=18)
    kc, vc = gpu_cache(b)
    ro, rl = ref_attn(b, *cpu_cache(b))
    dev = torch.device("cuda")
    q, cu, su, bt = b.q.to(dev), b.cu_seqlens_q.to(dev), b.seqused_k.to(dev), b.block_table.to(dev)
    ws = torch.full((va.attn_workspace_size(b.T, b.Hq, b.D, 2),), 0xFF, dtype=torch.uint8, device=dev)
    first = {}
    for it in range(140):
        ns = 1 + it % 2
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
        va.attn_varlen_prefill(q, kc, vc, out, cu, su, bt, b.max_seqlen_q, b.max_seqlen_k, b.softmax_scale,
                               lse_out=lse, num_splits=ns, workspace=ws)
        if ns not in first:
            check(out, lse, ro, rl, TOL)
            first[ns] = (out, lse)
        else:
            o0, l0 = first[ns]
            assert torch.equal(out, o0) and torch.equal(lse, l0), "call %d differs" % it
    assert_no_device_error()


def test_graph_replays_beside_eager_calls_on_another_stream():
    """A captured mixed-batch step replayed on one stream while eager
    tensor-core calls run on another, interleaved without synchronisation.
    Each call has its own workspace, and the tensor-core kernel's work
    counter lives there, so the two never share a counter: both outputs
    match the oracle after 4 replays beside 4 x 20 eager calls."""
    dev = torch.device("cuda")
    a = W.make_batch([300, 1, 1, 40, 1, 129], [700, 900, 64, 40, 2000, 129], 32, 8, 128, 16, seed=19)
    e = W.make_batch([200, 90, 1, 333], [260, 400, 77, 333], 16, 4, 128, 32, seed=20)
    kca, vca = gpu_cache(a)
    kce, vce = gpu_cache(e)
    roa, rla = ref_attn(a, *cpu_cache(a))
    roe, rle = ref_attn(e, *cpu_cache(e))
    sms = _sms()

    def bufs(b):
        q = b.q.to(dev)
        ns = va.attn_num_splits(b.B, b.max_seqlen_q, b.max_seqlen_k, b.Hq, b.Hkv, sms)
        ws = torch.full((va.attn_workspace_size(b.T, b.Hq, b.D, max(ns, 2)),), 0xFF, dtype=torch.uint8,
                        device=dev)
        return (q, torch.empty_like(q), torch.empty(q.shape[:2], dtype=torch.float32, device=dev),
                b.cu_seqlens_q.to(dev), b.seqused_k.to(dev), b.block_table.to(dev), ws)

    qa, oa, la, cua, sua, bta, wsa = bufs(a)
    qe, oe, le, cue, sue, bte, wse = bufs(e)

    def step_a():
        va.attn_varlen_prefill(qa, kca, vca, oa, cua, sua, bta, a.max_seqlen_q, a.max_seqlen_k, a.softmax_scale,
                               lse_out=la, num_splits=0, workspace=wsa)

    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s1):
        step_a()
    torch.cuda.current_stream().wait_stream(s1)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step_a()
    torch.cuda.synchronize()
    s2.wait_stream(torch.cuda.current_stream())
    for _ in range(4):
        with torch.cuda.stream(s1):
            g.replay()
        with torch.cuda.stream(s2):
            for _ in range(20):
                va.attn_varlen_prefill(qe, kce, vce, oe, cue, sue, bte, e.max_seqlen_q, e.max_seqlen_k,
                                       e.softmax_scale, lse_out=le, num_splits=0, workspace=wse)
    torch.cuda.synchronize()
    check(oa, la, roa, rla, TOL)
    check(oe, le, roe, rle, TOL)
    assert_no_device_error()


# ------------------------------------------ variants: window, soft cap, sinks

VARIANT_CASES = [
    dict(window=(48, -1)),
    dict(window=(0, -1)),
    dict(window=(100, 7), causal=False),
    dict(window=(-1, 5), causal=False),
    dict(softcap=3.0),
    dict(sinks=True),
    dict(window=(33, -1), softcap=2.0, sinks=True),
]


@pytest.mark.parametrize("num_splits", [1, 3, 0])
@pytest.mark.parametrize("case", range(len(VARIANT_CASES)))
def test_variants_against_oracle(case, num_splits):
    """Sliding window, soft cap and sinks ("FlashAttention deep dive",
    window_size / softcap / s_aux) on a batch that mixes decode rows,
    short and long prefill rows (both kernels), with and without split-KV."""
    kw = dict(VARIANT_CASES[case])
    causal = kw.pop("causal", True)
    b = W.make_batch([1, 7, 300, 1, 129, 20], [500, 7, 600, 2000, 129, 333], 32, 8, 128, 16, seed=40 + case,
                     causal=causal)
    kc, vc = gpu_cache(b)
    sinks = None
    if kw.pop("sinks", False):
        g = torch.Generator().manual_seed(W.SEED0 + 700 + case)
        sinks = (torch.randn(32, generator=g) * 2.0).float()
    window = kw.get("window", (-1, -1))
    softcap = kw.get("softcap", 0.0)
    out, lse = gpu_attn(b, kc, vc, num_splits=num_splits, causal=causal, window=window, softcap=softcap,
                        sinks=None if sinks is None else sinks.cuda())
    ro, rl = oracle.attention(b.q, *cpu_cache(b), b.cu_seqlens_q, b.seqused_k, b.block_table, b.softmax_scale,
                              causal=causal, window=window, softcap=softcap,
                              sinks=None if sinks is None else sinks.double())
    check(out, lse, ro, rl, TOL)
    assert_no_device_error()


@pytest.mark.parametrize("D,kv_dtype", [(64, "bf16"), (128, "fp8")])
def test_variants_other_paths(D, kv_dtype):
    """The same variants on head size 64 (rows-heavy requests on the
    mma.sync kernel) and on an e4m3 cache (both kernels widen e4m3)."""
    b = W.make_batch([1, 40, 200, 1], [900, 60, 250, 3000], 16, 4, D, 32, seed=48, kv_dtype=kv_dtype)
    kc, vc = gpu_cache(b)
    ck, cv = cpu_cache(b)
    g = torch.Generator().manual_seed(W.SEED0 + 750)
    sinks = (torch.randn(16, generator=g) * 2.0).float()
    fp8 = kv_dtype == "fp8"
    for window, softcap, use_sinks in [((64, -1), 0.0, False), ((-1, -1), 4.0, True), ((17, -1), 1.5, True)]:
        for ns in (1, 0):
            out, lse = gpu_attn(b, kc, vc, num_splits=ns, window=window, softcap=softcap,
                                sinks=sinks.cuda() if use_sinks else None)
            ro, rl = oracle.attention(b.q, ck, cv, b.cu_seqlens_q, b.seqused_k, b.block_table, b.softmax_scale,
                                      k_scale=b.k_scale if fp8 else 1.0, v_scale=b.v_scale if fp8 else 1.0,
                                      window=window, softcap=softcap,
                                      sinks=sinks.double() if use_sinks else None)
            check(out, lse, ro, rl, TOL_FP8 if fp8 else TOL)
    assert_no_device_error()


def test_workload_swa_decode_with_sinks():
    """Sliding-window decode with sinks (the swa bench workload, smaller):
    window of 1000 keys over contexts of 2k-8k, split-KV over the window."""
    b = W.swa_decode(B=8, lo=2048, hi=8192, window=1000)
    kc, vc = gpu_cache(b)
    win, sinks = b.extra["window"], b.extra["sinks"]
    for ns in (0, 1):
        out, lse = gpu_attn(b, kc, vc, num_splits=ns, window=win, sinks=sinks.cuda())
        ro, rl = oracle.attention(b.q, *cpu_cache(b), b.cu_seqlens_q, b.seqused_k, b.block_table, b.softmax_scale,
                                  window=win, sinks=sinks.double())
        check(out, lse, ro, rl, TOL)
    assert_no_device_error()


@pytest.mark.parametrize("num_splits", [0, 1])
def test_workload_verify_full(num_splits):
    """Multi-token verification at the benchmarked shape (64 requests, 2-8
    query tokens each over paged contexts of 0.5k-8k keys), every row:
    requests of up to 16 packed rows run on 16-row CTAs, longer ones on
    32-row CTAs, all in one call, with the automatic split counts and
    without splitting."""
    b = W.verify_decode()
    kc, vc = gpu_cache(b)
    out, lse = gpu_attn(b, kc, vc, num_splits=num_splits)
    ro, rl = ref_attn(b, *cpu_cache(b))
    check(out, lse, ro, rl, TOL)
    assert_no_device_error()


# ------------------------------------------------ e4m3 queries (q_descale)

@pytest.mark.parametrize("bs,num_splits", [(16, 0), (32, 1), (16, 3)])
def test_fp8_query_against_oracle(bs, num_splits):
    """e4m3 queries with q_descale over an e4m3 cache ("FlashAttention deep
    dive", FA3 FP8: q/k/v descales): decode, verify and prefill rows in one
    call, Q K^T on e4m3 operands, bf16 output; the oracle gets the same
    e4m3 codes and scales."""
    b = W.make_batch([1, 7, 300, 1, 129, 20, 3], [500, 7, 600, 2000, 129, 333, 40], 32, 8, 128, bs, seed=60,
                     kv_dtype="fp8")
    kc, vc = gpu_cache(b)
    ck, cv = cpu_cache(b)
    qs = float(b.q.float().abs().max()) / 448.0
    q8 = (b.q.float() / qs).to(torch.float8_e4m3fn)
    out, lse = gpu_attn(b, kc, vc, num_splits=num_splits, q=q8, q_descale=qs)
    ro, rl = oracle.attention(q8, ck, cv, b.cu_seqlens_q, b.seqused_k, b.block_table, b.softmax_scale,
                              k_scale=b.k_scale, v_scale=b.v_scale, q_scale=qs)
    check(out, lse, ro, rl, TOL_FP8)
    assert_no_device_error()


def _q8_call(b, q8, qs, kc, vc, num_splits=0):
    return gpu_attn(b, kc, vc, num_splits=num_splits, q=q8, q_descale=qs)


@pytest.mark.parametrize("bs", [64, 256])
def test_fp8_query_tensor_core_page_sizes(bs):
    """e4m3 queries on requests above 64 packed rows (the tensor-core
    kernel: S = Q K^T as kind::f8f6f4 MMAs, K read from its 128-byte-
    swizzled staging slot, page loads of gcd(bs, 64) rows), ragged lengths,
    against the oracle with the same e4m3 codes and scales."""
    b = W.make_batch([130, 17, 300, 64], [130, 400, 1000, 700], 32, 8, 128, bs, seed=62, kv_dtype="fp8")
    kc, vc = gpu_cache(b)
    ck, cv = cpu_cache(b)
    qs = float(b.q.float().abs().max()) / 448.0
    q8 = (b.q.float() / qs).to(torch.float8_e4m3fn)
    for ns in (1, 0):
        out, lse = _q8_call(b, q8, qs, kc, vc, ns)
        ro, rl = oracle.attention(q8, ck, cv, b.cu_seqlens_q, b.seqused_k, b.block_table, b.softmax_scale,
                                  k_scale=b.k_scale, v_scale=b.v_scale, q_scale=qs)
        check(out, lse, ro, rl, TOL_FP8)
    assert_no_device_error()


def test_fp8_query_mixed_workload_sampled():
    """The fp8 mixed batch (128 decode rows + four 2048-token prefill chunks,
    e4m3 cache, bs 32) with e4m3 queries: every decode row and sampled
    prefill rows against the oracle."""
    b = W.fp8_mixed()
    kc, vc = gpu_cache(b)
    ck, cv = cpu_cache(b)
    qs = float(b.q.float().abs().max()) / 448.0
    q8 = (b.q.float() / qs).to(torch.float8_e4m3fn)
    out, lse = _q8_call(b, q8, qs, kc, vc)
    rows = boundary_rows(b, per_request=32, seed=5)
    ro, rl = oracle.attention(q8, ck, cv, b.cu_seqlens_q, b.seqused_k, b.block_table, b.softmax_scale,
                              k_scale=b.k_scale, v_scale=b.v_scale, q_scale=qs, rows=rows)
    check(out, lse, ro, rl, TOL_FP8, rows=rows)
    assert_no_device_error()


def test_fp8_query_with_variants():
    """e4m3 queries with a sliding window, a soft cap and sinks."""
    b = W.make_batch([1, 12, 90, 1], [800, 60, 200, 1500], 32, 8, 128, 16, seed=61, kv_dtype="fp8")
    kc, vc = gpu_cache(b)
    ck, cv = cpu_cache(b)
    qs = float(b.q.float().abs().max()) / 448.0
    q8 = (b.q.float() / qs).to(torch.float8_e4m3fn)
    g = torch.Generator().manual_seed(W.SEED0 + 760)
    sinks = (torch.randn(32, generator=g) * 2.0).float()
    for ns in (1, 0):
        out, lse = gpu_attn(b, kc, vc, num_splits=ns, q=q8, q_descale=qs, window=(100, -1), softcap=5.0,
                            sinks=sinks.cuda())
        ro, rl = oracle.attention(q8, ck, cv, b.cu_seqlens_q, b.seqused_k, b.block_table, b.softmax_scale,
                                  k_scale=b.k_scale, v_scale=b.v_scale, q_scale=qs, window=(100, -1),
                                  softcap=5.0, sinks=sinks.double())
        check(out, lse, ro, rl, TOL_FP8)
    assert_no_device_error()
