"""Failure detection on the GPU without a fault: a bounded wait on a flag
that nothing sets gives up after its limit, reports ERR_TIMEOUT through the
device error word, and leaves the context usable for the next call."""
import os
import sys
import time

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import varlen_flashattention_causal_gb300 as va  # noqa: E402
from varlen_flashattention_causal_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_the_context_survives():
    from varlen_flashattention_causal_gb300 import build
    build.build()
    torch.cuda.synchronize()
    va.attn_device_error_flag(reset=True)
    t0 = time.perf_counter()
    va.attn_selftest_wait_timeout()
    flag = va.attn_device_error_flag(reset=True)        # synchronises the device
    waited = time.perf_counter() - t0
    assert flag == va.ERR_TIMEOUT
    assert 1.5 < waited < 60.0
    assert va.attn_device_error_flag() == 0

    # the next call runs normally and matches the oracle
    b = W.make_batch([1] * 4, [40, 130, 7, 300], 8, 2, 128, 16, seed=90)
    kc = torch.zeros((b.num_blocks, b.bs, b.Hkv, b.D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    va.kv_cache_write(b.k_tok.cuda(), b.v_tok.cuda(), kc, vc, b.slot_mapping.cuda())
    q = b.q.cuda()
    out = torch.empty_like(q)
    lse = torch.empty((b.T, b.Hq), dtype=torch.float32, device="cuda")
    va.attn_paged_decode(q, kc, vc, out, b.seqused_k.cuda(), b.block_table.cuda(), max(b.kv_lens),
                         b.softmax_scale, lse_out=lse)
    ref, ref_lse = oracle.attention(b.q, kc, vc, b.cu_seqlens_q, b.seqused_k, b.block_table, b.softmax_scale)
    assert float((out.double().cpu() - ref).abs().max()) < 1e-2
    assert float((lse.double().cpu() - ref_lse).abs().max()) < 1e-2
    assert va.attn_device_error_flag() == 0
