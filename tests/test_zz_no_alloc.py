"""attn_paged_decode_noalloc: decode for callers that cannot allocate.

Some callers of this library may not allocate device memory at all -- a
plugin living inside a framework that owns every device allocation, or a
serving loop that cannot afford the device synchronisation cudaMalloc and
cudaFree may cause.  For them attn_paged_decode_noalloc keeps its split-KV
scratch in a fixed array inside libattn.so instead of a caller workspace.

This file checks, through the C ABI, that two calls in a row give the same
result as the regular attn_paged_decode (within the parity tolerance, and
bitwise at the same explicit split count), that the leftover contents of the
shared array from the first call do not leak into the second, that a batch
whose automatic split count would overflow the array runs with fewer
segments and still matches, and that an explicit split count too large for
the array is refused.
It is named to run after every other test file, and needs nothing from them.
"""
import pytest
import torch

import varlen_flashattention_causal_gb300 as va
from varlen_flashattention_causal_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _cache(b):
    kc = torch.zeros((b.num_blocks, b.bs, b.Hkv, b.D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    va.kv_cache_write(b.k_tok.cuda(), b.v_tok.cuda(), kc, vc, b.slot_mapping.cuda())
    return kc, vc


def _decode(fn, b, kc, vc, **kw):
    q = b.q.cuda()
    out = torch.empty_like(q)
    lse = torch.empty((b.B, b.Hq), dtype=torch.float32, device="cuda")
    fn(q, kc, vc, out, b.seqused_k.cuda(), b.block_table.cuda(), b.max_seqlen_k, b.softmax_scale,
       lse_out=lse, **kw)
    return out, lse


def _maxerr(a, b):
    return float((a.double() - b.double()).abs().max())


def test_noalloc_decode_matches_regular_entry_point_twice():
    from varlen_flashattention_causal_gb300 import build
    build.build()
    # first call: the Llama-3-8B-shaped decode batch; second call: a
    # different batch (longer contexts, fewer requests) on the same array
    first = W.decode_llama8b()
    second = W.make_batch([1] * 6, [9000, 17, 4096, 1, 20000, 333], 32, 8, 128, 16, seed=77)
    for b in (first, second):
        kc, vc = _cache(b)
        ref_o, ref_l = _decode(va.attn_paged_decode, b, kc, vc)
        got_o, got_l = _decode(va.attn_paged_decode_noalloc, b, kc, vc)
        torch.cuda.synchronize()
        assert _maxerr(got_o, ref_o) <= TOL
        assert _maxerr(got_l, ref_l) <= TOL
        assert torch.isfinite(got_o.float()).all() and torch.isfinite(got_l).all()
        # with the same explicit split count both run the very same kernels
        # on the same partial layout, so the results are bitwise equal
        o1, l1 = _decode(va.attn_paged_decode, b, kc, vc, num_splits=4)
        o2, l2 = _decode(va.attn_paged_decode_noalloc, b, kc, vc, num_splits=4)
        assert torch.equal(o2, o1) and torch.equal(l2, l1)
        del kc, vc
    assert va.attn_device_error_flag(reset=True) == 0


def test_noalloc_caps_the_automatic_split_count_to_its_array():
    """64 requests, the longest of 16k keys: the automatic choice for this
    batch is 8 segments, whose partials (about 8.1 MiB) do not fit in the
    8 MiB array, so the entry point runs fewer segments.  Its result must
    still match the regular entry point given a workspace for all 8 (within
    the parity tolerance: different segment boundaries round differently)."""
    from varlen_flashattention_causal_gb300 import build
    build.build()
    b = W.make_batch([1] * 64, [16384, 12000, 5000, 1] + [300] * 60, 32, 8, 128, 16, seed=79)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ns = va.attn_num_splits(b.B, 1, b.max_seqlen_k, b.Hq, b.Hkv, sms)
    assert va.attn_workspace_size(b.B, b.Hq, b.D, ns) > va.NOALLOC_SCRATCH_BYTES
    kc, vc = _cache(b)
    ref_o, ref_l = _decode(va.attn_paged_decode, b, kc, vc, num_splits=ns)
    got_o, got_l = _decode(va.attn_paged_decode_noalloc, b, kc, vc)
    torch.cuda.synchronize()
    assert _maxerr(got_o, ref_o) <= TOL and _maxerr(got_l, ref_l) <= TOL
    assert torch.isfinite(got_o.float()).all() and torch.isfinite(got_l).all()
    assert va.attn_device_error_flag(reset=True) == 0


def test_noalloc_refuses_splits_beyond_its_array():
    from varlen_flashattention_causal_gb300 import build
    build.build()
    b = W.make_batch([1] * 64, [1024] * 64, 32, 8, 128, 16, seed=78)
    kc, vc = _cache(b)
    # 64 tokens x 32 heads x 256 segments of fp32 partials is far above 8 MiB
    assert va.attn_workspace_size(b.B, b.Hq, b.D, 256) > va.NOALLOC_SCRATCH_BYTES
    with pytest.raises(va.AttnError) as e:
        _decode(va.attn_paged_decode_noalloc, b, kc, vc, num_splits=256)
    assert e.value.status == 7          # ATTN_ERR_WORKSPACE
