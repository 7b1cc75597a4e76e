"""fp64 CPU oracle for varlen / paged causal attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (``varlen_flashattention_causal_gb300``) never does, and the two
share no code: this side is a plain restatement of what the source pages
define, in fp64.

Two independent formulations live here:

* ``attention`` / ``merge_states`` / ``kv_write`` -- ctypes wrappers over
  ``attn_oracle.c`` (per query row: walk the block table, two-pass softmax).
* ``dense_masked_attention`` -- numpy brute force that materialises the whole
  packed score matrix with the block-diagonal, lower-triangular mask drawn in
  "vLLM 中 Attention Kernel 如何并行处理多个请求", sec. 1 (S = [[S_A, -inf],
  [-inf, S_B]]), for tiny cases only.  It never looks at a block table.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, the pages' worked examples, brute force, invariants).
"""
import ctypes
import os

import numpy as np
import torch

from .build import build_oracle

BF16, FP16, E4M3, FP32 = 0, 1, 2, 3

_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_oracle())
        c = ctypes
        lib.oracle_attention.restype = c.c_int
        lib.oracle_attention.argtypes = [
            c.c_void_p, c.c_int, c.c_int64,
            c.c_void_p, c.c_void_p, c.c_int, c.c_double, c.c_double,
            c.c_void_p, c.c_void_p, c.c_void_p, c.c_int64,
            c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int,
            c.c_double, c.c_int, c.c_void_p, c.c_int64,
            c.c_void_p, c.c_void_p, c.c_int]
        lib.oracle_attention_ext.restype = c.c_int
        lib.oracle_attention_ext.argtypes = [
            c.c_void_p, c.c_int, c.c_int64,
            c.c_void_p, c.c_void_p, c.c_int, c.c_double, c.c_double,
            c.c_void_p, c.c_void_p, c.c_void_p, c.c_int64,
            c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int,
            c.c_double, c.c_int, c.c_int64, c.c_int64, c.c_double, c.c_void_p, c.c_double,
            c.c_void_p, c.c_int64, c.c_void_p, c.c_void_p, c.c_int]
        lib.oracle_merge_states.restype = None
        lib.oracle_merge_states.argtypes = [
            c.c_int64, c.c_int, c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p,
            c.c_void_p, c.c_void_p]
        lib.oracle_kv_write.restype = c.c_int
        lib.oracle_kv_write.argtypes = [
            c.c_void_p, c.c_void_p, c.c_int, c.c_int64, c.c_void_p, c.c_void_p,
            c.c_int, c.c_void_p, c.c_int64, c.c_int, c.c_int, c.c_int, c.c_int,
            c.c_float, c.c_float]
        lib.oracle_e4m3_from_float.restype = c.c_uint8
        lib.oracle_e4m3_from_float.argtypes = [c.c_float]
        lib.oracle_e4m3_to_double.restype = c.c_double
        lib.oracle_e4m3_to_double.argtypes = [c.c_uint8]
        _lib = lib
    return _lib


def _code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float16:
        return FP16
    if t.dtype in (torch.float8_e4m3fn, torch.uint8):
        return E4M3
    if t.dtype == torch.float32:
        return FP32
    raise TypeError("oracle: unsupported storage dtype %s" % t.dtype)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _host(t, dtype=None):
    t = t.detach().to("cpu")
    if dtype is not None:
        t = t.to(dtype)
    return t.contiguous()


def attention(q, k_cache, v_cache, cu_seqlens_q, seqused_k, block_table,
              softmax_scale, causal=True, k_scale=1.0, v_scale=1.0,
              rows=None, nthreads=0, window=(-1, -1), softcap=0.0, sinks=None, q_scale=1.0):
    """fp64 attention over a paged cache.

    q: [T, Hq, D] (bf16/fp16); k_cache, v_cache: [num_blocks, bs, Hkv, D]
    (bf16/fp16/e4m3); cu_seqlens_q: [B+1]; seqused_k: [B]; block_table:
    [B, max_blocks] (int32).  rows: optional packed token indices to
    evaluate.  window = (left, right) keys around the query's absolute
    position (-1 unlimited), softcap (0 = none), sinks [Hq] (one logit per
    query head, or None): the variants of "FlashAttention deep dive",
    flash_attn_varlen_func (window_size, softcap, s_aux) as read in
    attn_oracle.c.  q may be e4m3 with q_scale (its value is code *
    q_scale).  Returns (out [n, Hq, D] float64, lse [n, Hq] float64).
    """
    lib = _load()
    q = _host(q)
    k_cache, v_cache = _host(k_cache), _host(v_cache)
    cu = _host(cu_seqlens_q, torch.int32)
    su = _host(seqused_k, torch.int32)
    bt = _host(block_table, torch.int32)
    T, Hq, D = q.shape
    nb, bs, Hkv, Dk = k_cache.shape
    assert Dk == D and v_cache.shape == k_cache.shape and bt.dim() == 2
    B = su.numel()
    rws = None if rows is None else _host(torch.as_tensor(rows), torch.int64)
    n = T if rws is None else rws.numel()
    out = torch.empty((n, Hq, D), dtype=torch.float64)
    lse = torch.empty((n, Hq), dtype=torch.float64)
    plain = tuple(window) == (-1, -1) and not softcap and sinks is None and q_scale == 1.0
    if plain:
        st = lib.oracle_attention(
            q.data_ptr(), _code(q), Hq * D,
            k_cache.data_ptr(), v_cache.data_ptr(), _code(k_cache),
            float(k_scale), float(v_scale),
            cu.data_ptr(), su.data_ptr(), bt.data_ptr(), bt.shape[1],
            B, Hq, Hkv, D, bs, nb, float(softmax_scale), int(bool(causal)),
            _ptr(rws), n, out.data_ptr(), lse.data_ptr(), int(nthreads))
    else:
        sk = None if sinks is None else _host(torch.as_tensor(sinks), torch.float64)
        assert sk is None or sk.numel() == Hq
        st = lib.oracle_attention_ext(
            q.data_ptr(), _code(q), Hq * D,
            k_cache.data_ptr(), v_cache.data_ptr(), _code(k_cache),
            float(k_scale), float(v_scale),
            cu.data_ptr(), su.data_ptr(), bt.data_ptr(), bt.shape[1],
            B, Hq, Hkv, D, bs, nb, float(softmax_scale), int(bool(causal)),
            int(window[0]), int(window[1]), float(softcap), _ptr(sk), float(q_scale),
            _ptr(rws), n, out.data_ptr(), lse.data_ptr(), int(nthreads))
    if st != 0:
        raise ValueError("oracle_attention failed with status %d" % st)
    return out, lse


def merge_states(o1, lse1, o2, lse2):
    """fp64 log-sum-exp merge of two attention states ([n, D] / [n] shaped)."""
    lib = _load()
    o1 = _host(o1, torch.float64)
    o2 = _host(o2, torch.float64)
    l1 = _host(lse1, torch.float64)
    l2 = _host(lse2, torch.float64)
    D = o1.shape[-1]
    n = l1.numel()
    assert o1.numel() == n * D and o2.numel() == n * D and l2.numel() == n
    out = torch.empty(o1.shape, dtype=torch.float64)
    lse = torch.empty(l1.shape, dtype=torch.float64)
    lib.oracle_merge_states(n, D, o1.data_ptr(), l1.data_ptr(), o2.data_ptr(),
                            l2.data_ptr(), out.data_ptr(), lse.data_ptr())
    return out, lse


def kv_write(key, value, k_cache, v_cache, slot_mapping, k_scale=1.0, v_scale=1.0):
    """Scatter key/value [T, Hkv, D] into CPU caches [nb, bs, Hkv, D] in place."""
    lib = _load()
    key, value = _host(key), _host(value)
    sm = _host(slot_mapping, torch.int64)
    assert k_cache.device.type == "cpu" and k_cache.is_contiguous()
    assert v_cache.device.type == "cpu" and v_cache.is_contiguous()
    T, Hkv, D = key.shape
    nb, bs, Hc, Dc = k_cache.shape
    assert Hc == Hkv and Dc == D
    st = lib.oracle_kv_write(
        key.data_ptr(), value.data_ptr(), _code(key), Hkv * D,
        k_cache.data_ptr(), v_cache.data_ptr(), _code(k_cache), sm.data_ptr(),
        T, Hkv, D, bs, nb, float(k_scale), float(v_scale))
    if st != 0:
        raise ValueError("oracle_kv_write failed with status %d" % st)


def e4m3_from_float(x: float) -> int:
    """e4m3 code of an fp32 value (nearest, ties to even, saturating)."""
    return int(_load().oracle_e4m3_from_float(float(x)))


def e4m3_to_double(code: int) -> float:
    return float(_load().oracle_e4m3_to_double(int(code)))


def dense_masked_attention(q, k, v, cu_seqlens_q, cu_seqlens_k, softmax_scale,
                           causal=True, window=(-1, -1), softcap=0.0, sinks=None):
    """Brute force over the whole packed problem (tiny cases only).

    q: [T, Hq, D]; k, v: [Tk, Hkv, D] hold every request's keys back to back
    (request r owns key rows [cu_seqlens_k[r], cu_seqlens_k[r+1])), no
    paging.  One T x Tk score matrix per head is built, entries between
    different requests are set to -inf, and, when causal, so are keys after
    the query's absolute position ctx + i (ctx = kv_len - q_len); a window
    (left, right) masks keys outside [pos - left, pos + right].  softcap
    maps the scaled scores through c * tanh(s / c).  sinks append one extra
    score column per head (the sink logit) whose value row is zero.  Then a
    dense row softmax and P @ V.  Returns float64 numpy (out, lse, mask).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    cq = [int(x) for x in cu_seqlens_q]
    ck = [int(x) for x in cu_seqlens_k]
    T, Hq, D = q.shape
    Tk, Hkv, _ = k.shape
    G = Hq // Hkv
    req_q = np.zeros(T, dtype=np.int64)
    loc_q = np.zeros(T, dtype=np.int64)
    ctx_q = np.zeros(T, dtype=np.int64)
    for r in range(len(cq) - 1):
        req_q[cq[r]:cq[r + 1]] = r
        loc_q[cq[r]:cq[r + 1]] = np.arange(cq[r + 1] - cq[r])
        ctx_q[cq[r]:cq[r + 1]] = (ck[r + 1] - ck[r]) - (cq[r + 1] - cq[r])
    req_k = np.zeros(Tk, dtype=np.int64)
    loc_k = np.zeros(Tk, dtype=np.int64)
    for r in range(len(ck) - 1):
        req_k[ck[r]:ck[r + 1]] = r
        loc_k[ck[r]:ck[r + 1]] = np.arange(ck[r + 1] - ck[r])
    mask = req_q[:, None] == req_k[None, :]
    pos = (ctx_q + loc_q)[:, None]
    if causal:
        mask &= loc_k[None, :] <= pos
    if window[0] >= 0:
        mask &= loc_k[None, :] >= pos - window[0]
    if window[1] >= 0:
        mask &= loc_k[None, :] <= pos + window[1]
    out = np.zeros((T, Hq, D))
    lse = np.full((T, Hq), -np.inf)
    for h in range(Hq):
        g = h // G
        s = softmax_scale * (q[:, h, :] @ k[:, g, :].T)
        if softcap:
            s = softcap * np.tanh(s / softcap)
        s = np.where(mask, s, -np.inf)
        vg = v[:, g, :]
        if sinks is not None:
            s = np.concatenate([s, np.full((T, 1), float(sinks[h]))], axis=1)
            vg = np.concatenate([vg, np.zeros((1, D))], axis=0)
        m = s.max(axis=1, keepdims=True)
        live = np.isfinite(m[:, 0])
        m = np.where(np.isfinite(m), m, 0.0)
        e = np.exp(s - m)
        l = e.sum(axis=1)
        p = e / np.where(l > 0, l, 1.0)[:, None]
        out[:, h, :] = p @ vg
        lse[:, h] = np.where(live, m[:, 0] + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return out, lse, mask
