"""Varlen causal FlashAttention over a paged KV cache on GB300 (sm_103a).

Thin ctypes binding over ``libattn.so``: each function has the name of the
C entry point it wraps (declared in ``include/attn.h``) and only marshals
arguments -- every step of the computation runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors; the call is enqueued on the
current torch stream unless ``stream`` is given.  There is no CPU fallback:
if the library is missing or the device is not sm_103, calls raise.

Build the library with ``varlen_flashattention_causal_gb300.build.build()``
(``__graft_entry__.build()`` does it too).
"""
import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "AttnError", "attn_varlen_prefill", "attn_varlen_prefill_ext", "attn_paged_decode",
    "attn_paged_decode_noalloc", "attn_merge_states", "kv_cache_write", "attn_workspace_size",
    "attn_num_splits", "attn_num_splits_typed", "attn_tile_kind", "attn_status_string", "attn_device_error_flag",
    "attn_selftest_wait_timeout", "attn_validate_tables", "attn_validate_slots", "attn_cascade",
    "attn_cascade_splits",
    "attn_debug_validate_enabled", "library_path",
]

ATTN_BF16, ATTN_FP16, ATTN_FP8_E4M3, ATTN_FP32 = 0, 1, 2, 3
ERR_BLOCK_ID, ERR_SLOT, ERR_TIMEOUT = 1, 2, 4
ATTN_ERR_TABLE = 10

_lib = None


class AttnError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (fn, attn_status_string(status), status))


def library_path():
    return _build.LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise RuntimeError("libattn.so is not built (run varlen_flashattention_causal_gb300.build.build())")
    lib = ctypes.CDLL(_build.LIB)
    c = ctypes
    vp, i64, i32, f32, sz = c.c_void_p, c.c_int64, c.c_int, c.c_float, c.c_size_t
    lib.attn_varlen_prefill.restype = i32
    lib.attn_varlen_prefill.argtypes = [
        vp, i64, vp, vp, vp, i64, vp, vp, vp, vp, i64,
        i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32,
        f32, i32, f32, f32, i32, vp, sz, vp]
    lib.attn_varlen_prefill_ext.restype = i32
    lib.attn_varlen_prefill_ext.argtypes = [
        vp, i64, vp, vp, vp, i64, vp, vp, vp, vp, i64,
        i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32,
        f32, i32, f32, f32, f32, i32, i32, f32, vp, i32, vp, sz, vp]
    lib.attn_paged_decode.restype = i32
    lib.attn_paged_decode.argtypes = [
        vp, vp, vp, vp, vp, vp, vp, i64,
        i32, i32, i32, i32, i32, i32, i32, i32, i32,
        f32, f32, f32, i32, vp, sz, vp]
    lib.attn_paged_decode_noalloc.restype = i32
    lib.attn_paged_decode_noalloc.argtypes = [
        vp, vp, vp, vp, vp, vp, vp, i64,
        i32, i32, i32, i32, i32, i32, i32, i32, i32,
        f32, f32, f32, i32, vp]
    lib.attn_merge_states.restype = i32
    lib.attn_merge_states.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]
    lib.kv_cache_write.restype = i32
    lib.kv_cache_write.argtypes = [vp, i64, vp, i64, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, f32, vp]
    lib.attn_workspace_size.restype = sz
    lib.attn_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.attn_num_splits.restype = i32
    lib.attn_num_splits.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.attn_num_splits_typed.restype = i32
    lib.attn_num_splits_typed.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32]
    lib.attn_tile_kind.restype = i32
    lib.attn_tile_kind.argtypes = [i32, i32, i32, i32, i32]
    lib.attn_status_string.restype = c.c_char_p
    lib.attn_status_string.argtypes = [i32]
    lib.attn_device_error_flag.restype = i32
    lib.attn_device_error_flag.argtypes = [i32]
    lib.attn_selftest_wait_timeout.restype = i32
    lib.attn_selftest_wait_timeout.argtypes = [vp]
    lib.attn_cascade.restype = i32
    lib.attn_cascade.argtypes = [
        vp, i64, vp, vp, vp, i64, vp, vp, vp, vp, i32, vp, vp, vp, i64,
        i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32,
        f32, f32, f32, i32, i32, vp, sz, vp, vp]
    lib.attn_cascade_splits.restype = i32
    lib.attn_cascade_splits.argtypes = [i32] * 11 + [c.POINTER(i32), c.POINTER(i32)]
    lib.attn_validate_tables.restype = i32
    lib.attn_validate_tables.argtypes = [vp, vp, vp, i64, i32, i32, i32, i32, i32, i32, i32]
    lib.attn_validate_slots.restype = i32
    lib.attn_validate_slots.argtypes = [vp, i32, i32, i32]
    lib.attn_debug_validate_enabled.restype = i32
    lib.attn_debug_validate_enabled.argtypes = []
    _lib = lib
    return lib


def _dt(t):
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float16:
        return ATTN_FP16
    if t.dtype in (torch.float8_e4m3fn, torch.uint8):
        return ATTN_FP8_E4M3
    if t.dtype == torch.float32:
        return ATTN_FP32
    raise TypeError("unsupported dtype %s" % t.dtype)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn, st):
    if st != 0:
        raise AttnError(fn, st)


def _i32(t, name):
    if t.dtype != torch.int32 or not t.is_contiguous():
        raise TypeError("%s must be a contiguous int32 tensor" % name)
    return t


def _workspace(T, Hq, D, ns, device, workspace):
    if workspace is not None:
        return workspace, workspace.numel() * workspace.element_size()
    # at least the tensor-core kernel's work counter, then the split partials
    n = attn_workspace_size(T, Hq, D, ns)
    return torch.empty(n, dtype=torch.uint8, device=device), n


def _sms(device):
    return torch.cuda.get_device_properties(device).multi_processor_count


def attn_varlen_prefill(q, k_cache, v_cache, out, cu_seqlens_q, seqused_k, block_table,
                        max_seqlen_q, max_seqlen_k, softmax_scale, causal=True, lse_out=None,
                        k_descale=1.0, v_descale=1.0, num_splits=0, workspace=None, stream=None,
                        window=(-1, -1), softcap=0.0, sinks=None, q_descale=1.0):
    """flash_attn_varlen_func over a paged cache (see include/attn.h).

    q, out: [T, Hq, D] (token stride may exceed Hq * D); k_cache, v_cache:
    [num_blocks, block_size, Hkv, D]; cu_seqlens_q [B+1], seqused_k [B],
    block_table [B, >=max_blocks] int32 (row stride taken from the tensor);
    lse_out: optional [T, Hq] fp32.  num_splits 0 = automatic; the
    workspace is allocated here when not given.  Variants
    (attn_varlen_prefill_ext): window = (left, right) keys around each
    query's position (-1 unlimited), softcap (0 = off), sinks: optional
    [Hq] fp32 CUDA tensor of per-head sink logits.  q may be
    float8_e4m3fn (with an e4m3 cache, head size 128) scaled by q_descale;
    out is then bf16.
    """
    lib = _load()
    T, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    B = seqused_k.numel()
    _i32(cu_seqlens_q, "cu_seqlens_q")
    _i32(seqused_k, "seqused_k")
    if block_table.dtype != torch.int32 or block_table.stride(-1) != 1:
        raise TypeError("block_table must be int32 with unit column stride")
    # the workspace is sized for the largest split count the library may
    # choose; with num_splits = 0 it picks a count per request class itself
    ns = num_splits if num_splits > 0 else attn_num_splits(B, max_seqlen_q, max_seqlen_k, Hq, Hkv,
                                                           _sms(q.device), D, _dt(q), _dt(k_cache))
    ws, ws_bytes = _workspace(T, Hq, D, ns, q.device, workspace)
    if sinks is not None and (sinks.dtype != torch.float32 or sinks.numel() != Hq or not sinks.is_contiguous()
                              or not sinks.is_cuda):
        raise TypeError("sinks must be a contiguous CUDA float32 tensor of Hq elements")
    st = lib.attn_varlen_prefill_ext(
        _p(q), q.stride(0), _p(k_cache), _p(v_cache), _p(out), out.stride(0), _p(lse_out),
        _p(cu_seqlens_q), _p(seqused_k), _p(block_table), block_table.stride(0),
        B, T, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, D, bs, nb,
        _dt(q), _dt(k_cache), float(softmax_scale), int(bool(causal)), float(q_descale),
        float(k_descale), float(v_descale), int(window[0]), int(window[1]), float(softcap), _p(sinks),
        int(num_splits), _p(ws), ws_bytes, _stream(stream))
    _check("attn_varlen_prefill", st)
    return out


# The C ABI has a separate entry point for the variants and e4m3 queries;
# attn_varlen_prefill above already calls it and takes its arguments
# (window, softcap, sinks, q_descale), so the Python name is the same call.
attn_varlen_prefill_ext = attn_varlen_prefill


def attn_paged_decode(q, k_cache, v_cache, out, seq_lens, block_table, max_seq_len,
                      softmax_scale, lse_out=None, k_descale=1.0, v_descale=1.0,
                      num_splits=0, workspace=None, stream=None):
    """One query token per request: q, out [B, Hq, D] contiguous."""
    lib = _load()
    B, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    _i32(seq_lens, "seq_lens")
    if block_table.dtype != torch.int32 or block_table.stride(-1) != 1:
        raise TypeError("block_table must be int32 with unit column stride")
    ns = num_splits if num_splits > 0 else attn_num_splits(B, 1, max_seq_len, Hq, Hkv, _sms(q.device), D,
                                                           _dt(q), _dt(k_cache))
    ws, ws_bytes = _workspace(B, Hq, D, ns, q.device, workspace)
    st = lib.attn_paged_decode(
        _p(q), _p(k_cache), _p(v_cache), _p(out), _p(lse_out), _p(seq_lens), _p(block_table),
        block_table.stride(0), B, int(max_seq_len), Hq, Hkv, D, bs, nb, _dt(q), _dt(k_cache),
        float(softmax_scale), float(k_descale), float(v_descale), int(num_splits), _p(ws), ws_bytes,
        _stream(stream))
    _check("attn_paged_decode", st)
    return out


def attn_cascade_splits(B, total_q, max_seqlen_q, prefix_len, max_suffix_len, Hq, Hkv, D, q_dtype=ATTN_BF16,
                        kv_dtype=ATTN_BF16, num_sms=None):
    """(prefix_splits, suffix_splits) attn_cascade chooses by itself."""
    if num_sms is None:
        num_sms = _sms(torch.device("cuda", torch.cuda.current_device()))
    a, b = ctypes.c_int(0), ctypes.c_int(0)
    st = _load().attn_cascade_splits(int(B), int(total_q), int(max_seqlen_q), int(prefix_len), int(max_suffix_len),
                                     int(Hq), int(Hkv), int(D), int(q_dtype), int(kv_dtype), int(num_sms),
                                     ctypes.byref(a), ctypes.byref(b))
    if st != 0:
        raise ValueError("attn_cascade_splits: invalid sizes")
    return a.value, b.value


def attn_cascade(q, k_cache, v_cache, out, cu_prefix_query_lens, prefix_kv_lens, prefix_block_table, prefix_len,
                 cu_seqlens_q, suffix_kv_lens, suffix_block_table, max_seqlen_q, max_suffix_len, softmax_scale,
                 lse_out=None, k_descale=1.0, v_descale=1.0, prefix_splits=0, suffix_splits=0, workspace=None,
                 stream=None, aux_stream=None):
    """Cascade attention in one call (see include/attn.h): prefix shared by
    every request (cu_prefix_query_lens = [0, T], prefix_kv_lens =
    [prefix_len], one row of block ids) plus each request's causal suffix,
    merged in one combine.  aux_stream: optional second stream for the
    prefix half.  The workspace is allocated here when not given."""
    lib = _load()
    T, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    B = suffix_kv_lens.numel()
    for t, n in ((cu_prefix_query_lens, "cu_prefix_query_lens"), (prefix_kv_lens, "prefix_kv_lens"),
                 (prefix_block_table, "prefix_block_table"), (cu_seqlens_q, "cu_seqlens_q"),
                 (suffix_kv_lens, "suffix_kv_lens")):
        _i32(t, n)
    if suffix_block_table.dtype != torch.int32 or suffix_block_table.stride(-1) != 1:
        raise TypeError("suffix_block_table must be int32 with unit column stride")
    if prefix_splits > 0 and suffix_splits > 0:
        ns = prefix_splits + suffix_splits
    else:
        a, b = attn_cascade_splits(B, T, max_seqlen_q, prefix_len, max_suffix_len, Hq, Hkv, D, _dt(q),
                                   _dt(k_cache), _sms(q.device))
        ns = (prefix_splits or a) + (suffix_splits or b)
    ws, ws_bytes = _workspace(T, Hq, D, ns, q.device, workspace)
    aux = None if aux_stream is None else _stream(aux_stream)
    st = lib.attn_cascade(
        _p(q), q.stride(0), _p(k_cache), _p(v_cache), _p(out), out.stride(0), _p(lse_out),
        _p(cu_prefix_query_lens), _p(prefix_kv_lens), _p(prefix_block_table), int(prefix_len),
        _p(cu_seqlens_q), _p(suffix_kv_lens), _p(suffix_block_table), suffix_block_table.stride(0),
        B, T, int(max_seqlen_q), int(max_suffix_len), Hq, Hkv, D, bs, nb, _dt(q), _dt(k_cache),
        float(softmax_scale), float(k_descale), float(v_descale), int(prefix_splits), int(suffix_splits),
        _p(ws), ws_bytes, _stream(stream), aux)
    _check("attn_cascade", st)
    return out


def attn_merge_states(out, lse_out, o1, lse1, o2, lse2, stream=None):
    """merge_attn_states: o* [T, Hq, D] (bf16/fp16/fp32), lse* [T, Hq] fp32."""
    lib = _load()
    T, Hq, D = o1.shape
    st = lib.attn_merge_states(_p(out), _p(lse_out), _p(o1), _p(lse1), _p(o2), _p(lse2),
                               T, Hq, D, _dt(o1), _stream(stream))
    _check("attn_merge_states", st)
    return out


def kv_cache_write(key, value, k_cache, v_cache, slot_mapping, k_scale=1.0, v_scale=1.0, stream=None):
    """reshape_and_cache_flash: key/value [T, Hkv, D] -> caches via slot_mapping (int64)."""
    lib = _load()
    T, Hkv, D = key.shape
    nb, bs, _, _ = k_cache.shape
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_contiguous():
        raise TypeError("slot_mapping must be a contiguous int64 tensor")
    st = lib.kv_cache_write(_p(key), key.stride(0), _p(value), value.stride(0), _p(k_cache), _p(v_cache),
                            _p(slot_mapping), T, Hkv, D, bs, nb, _dt(key), _dt(k_cache),
                            float(k_scale), float(v_scale), _stream(stream))
    _check("kv_cache_write", st)


def attn_workspace_size(total_q, Hq, D, num_splits):
    return int(_load().attn_workspace_size(int(total_q), int(Hq), int(D), int(num_splits)))


def attn_num_splits(B, max_seqlen_q, max_seqlen_k, Hq, Hkv, num_sms, D=None, q_dtype=None, kv_dtype=None):
    """The automatic split count; with D / q_dtype / kv_dtype (ATTN_* codes)
    given, attn_num_splits_typed for them (defaults 128, bf16, bf16)."""
    if D is None and q_dtype is None and kv_dtype is None:
        return int(_load().attn_num_splits(int(B), int(max_seqlen_q), int(max_seqlen_k), int(Hq), int(Hkv),
                                           int(num_sms)))
    return int(_load().attn_num_splits_typed(int(B), int(max_seqlen_q), int(max_seqlen_k), int(Hq), int(Hkv),
                                             128 if D is None else int(D),
                                             ATTN_BF16 if q_dtype is None else int(q_dtype),
                                             ATTN_BF16 if kv_dtype is None else int(kv_dtype), int(num_sms)))


def attn_num_splits_typed(B, max_seqlen_q, max_seqlen_k, Hq, Hkv, D, q_dtype, kv_dtype, num_sms):
    return attn_num_splits(B, max_seqlen_q, max_seqlen_k, Hq, Hkv, num_sms, D, q_dtype, kv_dtype)


def attn_tile_kind(q_lo, q_hi, k_lo, k_hi, ctx):
    return int(_load().attn_tile_kind(q_lo, q_hi, k_lo, k_hi, ctx))


def attn_status_string(status):
    return _load().attn_status_string(int(status)).decode()


def attn_device_error_flag(reset=False):
    v = int(_load().attn_device_error_flag(int(bool(reset))))
    if v < 0:
        raise RuntimeError("attn_device_error_flag: CUDA call failed")
    return v


def attn_selftest_wait_timeout(stream=None):
    """Launch the bounded-wait self-test: a wait on a phase nothing completes
    gives up after its limit (2 s) and raises ERR_TIMEOUT in the device error
    word (read it with attn_device_error_flag)."""
    _check("attn_selftest_wait_timeout", _load().attn_selftest_wait_timeout(_stream(stream)))


def _host_i32(t, name):
    t = torch.as_tensor(t)
    if t.device.type != "cpu" or t.dtype != torch.int32:
        raise TypeError("%s must be an int32 CPU tensor" % name)
    return t


def attn_validate_tables(cu_seqlens_q, seqused_k, block_table, max_seqlen_q, max_seqlen_k, block_size,
                         num_blocks, causal=True, total_q=None):
    """Check host copies of a call's integer tables (the ATTN_DEBUG_VALIDATE
    checks); returns the attn_status code (0 = ok, ATTN_ERR_TABLE = 10).
    cu_seqlens_q may be None (decode: one query row per request)."""
    su = _host_i32(seqused_k, "seqused_k").contiguous()
    bt = _host_i32(block_table, "block_table")
    if bt.dim() != 2 or bt.stride(1) != 1:
        raise TypeError("block_table must be 2-D with unit column stride")
    B = su.numel()
    cu = None if cu_seqlens_q is None else _host_i32(cu_seqlens_q, "cu_seqlens_q").contiguous()
    if total_q is None:
        total_q = B if cu is None else int(cu[-1])
    return int(_load().attn_validate_tables(_p(cu), _p(su), _p(bt), bt.stride(0), B, int(total_q),
                                            int(max_seqlen_q), int(max_seqlen_k), int(block_size),
                                            int(num_blocks), int(bool(causal))))


def attn_validate_slots(slot_mapping, block_size, num_blocks):
    """Check a host slot_mapping (int64); returns the attn_status code."""
    sm = torch.as_tensor(slot_mapping)
    if sm.device.type != "cpu" or sm.dtype != torch.int64:
        raise TypeError("slot_mapping must be an int64 CPU tensor")
    sm = sm.contiguous()
    return int(_load().attn_validate_slots(_p(sm), sm.numel(), int(block_size), int(num_blocks)))


def attn_debug_validate_enabled():
    return bool(_load().attn_debug_validate_enabled())


NOALLOC_SCRATCH_BYTES = 8 << 20   # ATTN_NOALLOC_SCRATCH_BYTES in include/attn.h


def attn_paged_decode_noalloc(q, k_cache, v_cache, out, seq_lens, block_table, max_seq_len,
                              softmax_scale, lse_out=None, k_descale=1.0, v_descale=1.0,
                              num_splits=0, stream=None):
    """attn_paged_decode for callers that cannot allocate device memory.

    Some callers may not allocate: a plugin inside a framework that owns all
    device memory, or a serving loop that cannot afford the device
    synchronisation cudaMalloc/cudaFree may cause.  This wrapper allocates
    nothing (no workspace tensor either): the split-KV scratch is a fixed
    8 MiB array inside libattn.so.  Calls on one device share that array,
    so calls that overlap on the GPU race; serialise them.  An explicit
    num_splits too large for the array raises AttnError (ATTN_ERR_WORKSPACE).
    """
    lib = _load()
    B, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    _i32(seq_lens, "seq_lens")
    if block_table.dtype != torch.int32 or block_table.stride(-1) != 1:
        raise TypeError("block_table must be int32 with unit column stride")
    st = lib.attn_paged_decode_noalloc(_p(q), _p(k_cache), _p(v_cache), _p(out), _p(lse_out), _p(seq_lens), _p(block_table),
            block_table.stride(0), B, int(max_seq_len), Hq, Hkv, D, bs, nb, _dt(q), _dt(k_cache),
            float(softmax_scale), float(k_descale), float(v_descale), int(num_splits), _stream(stream))
    _check("attn_paged_decode_noalloc", st)
    return out
