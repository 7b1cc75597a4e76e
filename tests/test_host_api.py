"""Host-side checks of libattn.so that need no GPU: the library builds and
loads, exports every entry point include/attn.h declares, rejects bad
arguments with the documented status before launching anything, and its
host mirrors of the planning rules follow the pages' examples."""
import ctypes
import os
import re

import pytest
import torch

import varlen_flashattention_causal_gb300 as va
from varlen_flashattention_causal_gb300 import build as vb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

OK, ERR_NULL, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_BS, ERR_HD, ERR_WS, ERR_CUDA, ERR_DEV = range(10)
BF16, FP16, E4M3, FP32 = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    vb.build()
    return va._load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_ ]*?\*?\s*\b([a-z_][a-z0-9_]*)\s*\(",
                                 src, flags=re.M)))


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"attn_varlen_prefill", "attn_paged_decode", "attn_merge_states", "kv_cache_write",
            "attn_workspace_size", "attn_status_string"} <= set(names)
    raw = ctypes.CDLL(vb.LIB)
    for n in names:
        assert hasattr(raw, n), n


def test_status_strings(lib):
    for s in range(11):
        assert va.attn_status_string(s) != "unknown status"
    assert va.attn_status_string(ERR_HD).startswith("head size")


# A 16-byte-aligned placeholder address.  Every call below that gets it stops
# before any launch on any machine: at a host validation error, at an empty
# batch (B = 0 or T = 0 returns ATTN_OK before the device is looked up), or
# at the workspace check, which also precedes every launch.
FAKE = ctypes.c_void_p(4096)

try:
    import torch
    _HAVE_GPU = torch.cuda.is_available()
except Exception:  # pragma: no cover
    _HAVE_GPU = False


def prefill(lib, **kw):
    a = dict(q=FAKE, qs=8 * 128, k=FAKE, v=FAKE, out=FAKE, os=8 * 128, lse=None, cu=FAKE, su=FAKE,
             bt=FAKE, bts=4, B=2, T=10, mq=6, mk=6, Hq=8, Hkv=2, D=128, bs=16, nb=4, qd=BF16,
             kd=BF16, scale=0.125, causal=1, kds=1.0, vds=1.0, ns=1, ws=None, wsb=0)
    a.update(kw)
    return lib.attn_varlen_prefill(a["q"], a["qs"], a["k"], a["v"], a["out"], a["os"], a["lse"], a["cu"],
                                   a["su"], a["bt"], a["bts"], a["B"], a["T"], a["mq"], a["mk"], a["Hq"],
                                   a["Hkv"], a["D"], a["bs"], a["nb"], a["qd"], a["kd"], a["scale"],
                                   a["causal"], a["kds"], a["vds"], a["ns"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), ERR_NULL),
    (dict(k=None), ERR_NULL),
    (dict(bt=None), ERR_NULL),
    (dict(cu=None), ERR_NULL),
    (dict(D=96), ERR_HD),
    (dict(D=256), ERR_HD),
    (dict(bs=24), ERR_BS),
    (dict(bs=0), ERR_BS),
    (dict(Hq=6, Hkv=4), ERR_SHAPE),
    (dict(qs=8 * 128 - 8), ERR_SHAPE),
    (dict(B=-1), ERR_SHAPE),
    (dict(B=65536), ERR_SHAPE),
    (dict(Hq=65536 * 2, Hkv=2, qs=65536 * 2 * 128, os=65536 * 2 * 128), ERR_SHAPE),
    (dict(qd=E4M3, kd=BF16), ERR_DTYPE),
    (dict(qd=E4M3, kd=E4M3, D=64, qs=8 * 64, os=8 * 64), ERR_DTYPE),
    (dict(qd=E4M3, kd=E4M3, qs=8 * 128 + 8), ERR_ALIGN),
    (dict(qd=BF16, kd=FP16), ERR_DTYPE),
    (dict(qd=FP32, kd=FP32), ERR_DTYPE),
    (dict(q=ctypes.c_void_p(4104)), ERR_ALIGN),
    (dict(qs=8 * 128 + 4), ERR_ALIGN),
    (dict(ns=4, ws=None, wsb=0), None),     # no device here: reaches CUDA or fails on workspace
    # a request may have more than 64 packed rows (17 tokens x 4 heads): the
    # tensor-core kernel's work counter needs the first 256 workspace bytes,
    # checked before the device is looked up
    (dict(mq=17), ERR_WS),
    (dict(mq=17, ws=FAKE, wsb=255), ERR_WS),
    (dict(mq=17, ws=ctypes.c_void_p(4100), wsb=256), ERR_ALIGN),
    (dict(mq=17, ws=FAKE, wsb=256), "device"),
    # head size 64 never runs the tensor-core kernel: no workspace needed
    (dict(mq=17, D=64, qs=8 * 64, os=8 * 64), "device"),
])
def test_prefill_validation(lib, kw, status):
    if status == "device" and _HAVE_GPU:
        # these pass every host check and would launch on the placeholder
        # pointers: they are meaningful (and safe) only without a device
        pytest.skip("would launch kernels on placeholder pointers")
    st = prefill(lib, **kw)
    if status is None:
        assert st in (ERR_WS, ERR_CUDA, ERR_DEV)
    elif status == "device":
        # host checks passed; the call stopped at the device lookup
        assert st in (ERR_CUDA, ERR_DEV)
    else:
        assert st == status


def test_empty_batch_is_a_no_op(lib):
    assert prefill(lib, B=0, T=0) == OK


def test_decode_validation(lib):
    st = lib.attn_paged_decode(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 4, 2, 100, 8, 2, 80, 16, 4,
                               BF16, BF16, 0.1, 1.0, 1.0, 0, None, 0, None)
    assert st == ERR_HD
    st = lib.attn_paged_decode(FAKE, FAKE, None, FAKE, None, FAKE, FAKE, 4, 2, 100, 8, 2, 64, 16, 4,
                               BF16, BF16, 0.1, 1.0, 1.0, 0, None, 0, None)
    assert st == ERR_NULL


def test_kv_write_validation(lib):
    # key, ks, value, vs, k_cache, v_cache, slots, T, Hkv, D, bs, nb, src, kv, k_scale, v_scale, stream
    args = [FAKE, 256, FAKE, 256, FAKE, FAKE, FAKE, 3, 2, 128, 16, 4, BF16, BF16, 1.0, 1.0, None]

    def call(**edit):
        a = list(args)
        for i, v in edit.items():
            a[int(i[1:])] = v
        return lib.kv_cache_write(*a)

    assert call(a10=33) == ERR_BS
    assert call(a9=100) == ERR_HD
    assert call(a13=FP16) == ERR_DTYPE
    assert call(a12=E4M3, a13=E4M3) == ERR_DTYPE
    assert call(a13=E4M3, a14=0.0) == ERR_SHAPE
    assert call(a6=None) == ERR_NULL
    assert call(a1=100) == ERR_SHAPE
    assert call(a1=264, a4=ctypes.c_void_p(4100)) == ERR_ALIGN
    assert call(a7=0) == OK


def test_merge_validation(lib):
    assert lib.attn_merge_states(FAKE, None, FAKE, FAKE, FAKE, FAKE, 4, 8, 128, E4M3, None) == ERR_DTYPE
    assert lib.attn_merge_states(FAKE, None, None, FAKE, FAKE, FAKE, 4, 8, 128, BF16, None) == ERR_NULL
    assert lib.attn_merge_states(FAKE, None, FAKE, FAKE, FAKE, FAKE, 4, 8, 72, BF16, None) == ERR_HD
    assert lib.attn_merge_states(FAKE, None, FAKE, FAKE, FAKE, FAKE, 0, 8, 128, BF16, None) == OK


def test_tile_kind_follows_the_pages_walkthrough(lib):
    """"vLLM 中 Attention Kernel 如何并行处理多个请求", sec. 3-4: BLOCK_M =
    BLOCK_N = 4 over request A (6 tokens): (q0-3, k0-3) diagonal, (q0-3,
    k4-5) skipped, (q4-5, k0-3) full, (q4-5, k4-5) diagonal."""
    kinds = {"skip": 0, "full": 1, "diagonal": 2}
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "tile_walk_4x4.txt"))
            if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 4
    for q_lo, q_hi, k_lo, k_hi, kind in rows:
        assert va.attn_tile_kind(int(q_lo), int(q_hi), int(k_lo), int(k_hi), 0) == kinds[kind]


def test_tile_kind_with_context_and_brute_force(lib):
    # with cached context the diagonal moves right by ctx (sec. 10); check
    # every small tile against the element mask by enumeration
    for ctx in (0, 3, 20):
        for q_lo in range(0, 8, 2):
            for q_hi in range(q_lo + 1, 10, 3):
                for k_lo in range(0, 30, 5):
                    for k_hi in range(k_lo + 1, 32, 7):
                        vis = [[k <= ctx + i for k in range(k_lo, k_hi)] for i in range(q_lo, q_hi)]
                        flat = [v for row in vis for v in row]
                        want = 1 if all(flat) else (0 if not any(flat) else 2)
                        assert va.attn_tile_kind(q_lo, q_hi, k_lo, k_hi, ctx) == want


def test_workspace_and_split_rules(lib):
    # 256 bytes for the tensor-core kernel's work counter, then the partials
    assert va.attn_workspace_size(64, 32, 128, 1) == 256
    assert va.attn_workspace_size(0, 32, 128, 5) == 256
    n = va.attn_workspace_size(64, 32, 128, 5)
    assert n >= 256 + 64 * 32 * 5 * (128 + 1) * 4 and n % 256 == 0
    # decode with few (request, KV head) pairs and long contexts splits;
    # big prefill batches do not
    assert va.attn_num_splits(4, 1, 131072, 64, 8, 152) > 8
    assert va.attn_num_splits(1024, 1, 512, 32, 8, 152) == 1   # enough CTAs, short keys
    assert va.attn_num_splits(1, 1, 100, 32, 8, 152) == 1     # too short to split
    # one long request among many short ones is still cut into segments
    assert va.attn_num_splits(1024, 1, 16384, 32, 8, 152) >= 8
    # the decode benchmark shape (64 requests up to 4060 keys, 8 KV heads):
    # 4 segments, the flat optimum of a 1-16 sweep on this chip
    assert va.attn_num_splits(64, 1, 4060, 32, 8, 152) == 4
    for B, L in ((64, 4096), (4, 32768), (128, 16384), (1, 2048)):
        s = va.attn_num_splits(B, 1, L, 32, 8, 152)
        assert 1 <= s <= 256 and (L // 64) >= s or s == 1
    # the typed form: bf16 at head size 128 is attn_num_splits itself; an
    # e4m3 cache runs decode rows on the transposed kernel, whose target is
    # eight CTAs an SM (5 segments on the decode benchmark shape)
    E4M3 = va.ATTN_FP8_E4M3
    assert va.attn_num_splits_typed(64, 1, 4060, 32, 8, 128, va.ATTN_BF16, va.ATTN_BF16, 152) == 4
    assert va.attn_num_splits_typed(64, 1, 4060, 32, 8, 128, va.ATTN_BF16, E4M3, 152) == 5
    assert va.attn_num_splits_typed(64, 1, 4060, 32, 8, 128, E4M3, E4M3, 152) == 5
    assert va.attn_num_splits_typed(64, 1, 4060, 32, 8, 64, va.ATTN_BF16, E4M3, 152) == 4   # 16-row kernel
    assert va.attn_num_splits_typed(64, 1, 4060, 30, 8, 128, va.ATTN_BF16, E4M3, 152) == 1  # Hq % Hkv


def prefill_ext(lib, wl=-1, wr=-1, cap=0.0, sinks=None, **kw):
    a = dict(q=FAKE, qs=8 * 128, k=FAKE, v=FAKE, out=FAKE, os=8 * 128, lse=None, cu=FAKE, su=FAKE,
             bt=FAKE, bts=4, B=2, T=10, mq=6, mk=6, Hq=8, Hkv=2, D=128, bs=16, nb=4, qd=BF16,
             kd=BF16, scale=0.125, causal=1, kds=1.0, vds=1.0, ns=1, ws=None, wsb=0)
    a.update(kw)
    return lib.attn_varlen_prefill_ext(a["q"], a["qs"], a["k"], a["v"], a["out"], a["os"], a["lse"], a["cu"],
                                       a["su"], a["bt"], a["bts"], a["B"], a["T"], a["mq"], a["mk"], a["Hq"],
                                       a["Hkv"], a["D"], a["bs"], a["nb"], a["qd"], a["kd"], a["scale"],
                                       a["causal"], a.get("qds", 1.0), a["kds"], a["vds"], wl, wr, cap, sinks,
                                       a["ns"], a["ws"],
                                       a["wsb"], None)


@pytest.mark.parametrize("wl,wr,cap,status", [
    (-2, -1, 0.0, ERR_SHAPE), (-1, -3, 0.0, ERR_SHAPE), (-1, -1, -1.0, ERR_SHAPE),
    (-1, -1, float("nan"), ERR_SHAPE), (-1, -1, float("inf"), ERR_SHAPE),
    (0, 0, 0.0, OK), (16, -1, 30.0, OK)])
def test_variant_validation(lib, wl, wr, cap, status):
    """attn_varlen_prefill_ext: window bounds below -1 and negative, NaN or
    infinite soft caps are refused before any launch.  Valid ones pass
    validation: with an empty batch the call then returns ATTN_OK at once,
    before it looks for a device, so no placeholder pointer can reach a
    launch on any machine."""
    kw = {} if status != OK else dict(B=0, T=0)
    assert prefill_ext(lib, wl=wl, wr=wr, cap=cap, **kw) == status


# ------------------------------------------------ the Python binding's marshalling

def test_binding_has_the_c_names():
    """Every function include/attn.h declares has a Python function of the
    same name in the binding, and every name the binding exports exists."""
    for n in declared_functions():
        assert callable(getattr(va, n, None)), n
    for n in va.__all__:
        assert hasattr(va, n), n


def _cpu(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def _status_of(call):
    with pytest.raises(va.AttnError) as e:
        call()
    return e.value.status


def test_bindings_pass_arguments_in_the_declared_order(lib):
    """Each Python wrapper hands its C entry point the declared number, types
    and order of arguments.  Each call below uses small CPU tensors with one
    argument chosen to fail one host check (head size, block size, dtype,
    window, soft cap, scale), and must raise AttnError with exactly that
    status.  Host validation precedes every device access, so these
    pointers are never dereferenced and nothing is launched on any machine."""
    cu = torch.tensor([0, 3], dtype=torch.int32)
    su = torch.tensor([3], dtype=torch.int32)
    bt = torch.zeros((1, 4), dtype=torch.int32)

    def prefill(fn=va.attn_varlen_prefill, D=128, bs=16, qdt=torch.bfloat16, kdt=torch.bfloat16, **kw):
        q, kc, out = _cpu(3, 8, D, dtype=qdt), _cpu(4, bs, 2, D, dtype=kdt), _cpu(3, 8, D)
        return lambda: fn(q, kc, kc, out, cu, su, bt, 3, 3, 0.1, num_splits=1, stream=0, **kw)

    assert _status_of(prefill(D=96)) == ERR_HD
    assert _status_of(prefill(bs=24)) == ERR_BS
    assert _status_of(prefill(kdt=torch.float16)) == ERR_DTYPE
    assert _status_of(prefill(qdt=torch.float8_e4m3fn)) == ERR_DTYPE
    assert _status_of(prefill(window=(-2, -1))) == ERR_SHAPE
    assert _status_of(prefill(window=(-1, -5))) == ERR_SHAPE
    assert _status_of(prefill(softcap=-1.0)) == ERR_SHAPE
    assert _status_of(prefill(fn=va.attn_varlen_prefill_ext, D=64, bs=8)) == ERR_BS

    sl = torch.tensor([5, 7], dtype=torch.int32)
    bt2 = torch.zeros((2, 4), dtype=torch.int32)
    for fn, extra in ((va.attn_paged_decode, {}), (va.attn_paged_decode_noalloc, {})):
        def decode(D=128, bs=16, kdt=torch.bfloat16):
            q, kc, out = _cpu(2, 8, D), _cpu(4, bs, 2, D, dtype=kdt), _cpu(2, 8, D)
            return lambda: fn(q, kc, kc, out, sl, bt2, 7, 0.1, num_splits=1, stream=0, **extra)
        assert _status_of(decode(D=96)) == ERR_HD
        assert _status_of(decode(bs=48 + 8)) == ERR_BS
        assert _status_of(decode(kdt=torch.float16)) == ERR_DTYPE

    def merge(D=128, dt=torch.bfloat16):
        o, l = _cpu(4, 8, D, dtype=dt), _cpu(4, 8, dtype=torch.float32)
        return lambda: va.attn_merge_states(o, None, o, l, o, l, stream=0)
    assert _status_of(merge(D=72)) == ERR_HD
    assert _status_of(merge(dt=torch.float8_e4m3fn)) == ERR_DTYPE

    slots = torch.zeros(3, dtype=torch.int64)

    def write(D=128, bs=16, src=torch.bfloat16, kdt=torch.bfloat16, **kw):
        k, kc = _cpu(3, 2, D, dtype=src), _cpu(4, bs, 2, D, dtype=kdt)
        return lambda: va.kv_cache_write(k, k, kc, kc, slots, stream=0, **kw)
    assert _status_of(write(D=96)) == ERR_HD
    assert _status_of(write(bs=40)) == ERR_BS
    assert _status_of(write(src=torch.float16)) == ERR_DTYPE
    assert _status_of(write(kdt=torch.float8_e4m3fn, k_scale=0.0)) == ERR_SHAPE
    assert _status_of(write(kdt=torch.float8_e4m3fn, v_scale=-1.0)) == ERR_SHAPE


# ------------------------------------------------ debug validation of the integer tables

def _tables():
    """Two requests ("vLLM 中 Attention Kernel 如何并行处理多个请求" sec. 5: packed
    rows; sec. 11: block table): q_len 3 and 5, kv_len 20 and 5 at block size
    16, a 4-column table whose unused columns hold garbage."""
    cu = torch.tensor([0, 3, 8], dtype=torch.int32)
    su = torch.tensor([20, 5], dtype=torch.int32)
    bt = torch.tensor([[7, 2, -99, 12345], [4, 99999, -1, 0]], dtype=torch.int32)
    return cu, su, bt


def _v(cu, su, bt, mq=5, mk=20, bs=16, nb=8, causal=True, total_q=None):
    return va.attn_validate_tables(cu, su, bt, mq, mk, bs, nb, causal, total_q)


def test_validate_tables_accepts_a_valid_batch(lib):
    cu, su, bt = _tables()
    assert _v(cu, su, bt) == 0
    # only the first ceil(kv_len / block_size) entries of a row are read
    assert _v(cu, su, bt[:, :2].contiguous()) == 0
    # bounds above the truth are fine; decode form (one row per request)
    assert _v(cu, su, bt, mq=100, mk=1000) == 0
    assert _v(None, su, bt, mq=1) == 0
    assert _v(cu, su.new_zeros(2), bt, causal=False) == 0


@pytest.mark.parametrize("edit", [
    "cu0", "cu_end", "cu_back", "mq_small", "mk_small", "kv_neg", "causal_short", "block_neg",
    "block_big", "stride_short", "decode_total"])
def test_validate_tables_rejects_each_broken_rule(lib, edit):
    cu, su, bt = _tables()
    kw = {}
    if edit == "cu0":
        cu[0] = 1
    elif edit == "cu_end":
        kw["total_q"] = 9                       # q holds 9 rows, cu_seqlens_q ends at 8
    elif edit == "cu_back":
        cu[1] = 9                                # request 1 gets q_len -1
        kw["mq"] = 100
    elif edit == "mq_small":
        kw["mq"] = 4                             # q_len 5 > max_seqlen_q
    elif edit == "mk_small":
        kw["mk"] = 19                            # kv_len 20 > max_seqlen_k
    elif edit == "kv_neg":
        su[1] = -1
    elif edit == "causal_short":
        su[1] = 4                                # 5 new tokens but 4 cached keys
    elif edit == "block_neg":
        bt[0, 1] = -1
    elif edit == "block_big":
        bt[1, 0] = 8                             # num_blocks = 8
    elif edit == "stride_short":
        bt = bt[:, :1]                           # request 0 needs two columns
        bt = torch.as_strided(bt.contiguous().view(-1), (2, 1), (1, 1))
    elif edit == "decode_total":
        assert _v(None, su, bt, mq=1, total_q=3) == va.ATTN_ERR_TABLE
        return
    assert _v(cu, su, bt, **kw) == va.ATTN_ERR_TABLE
    # the same batch without the mask accepts short caches
    if edit == "causal_short":
        assert _v(cu, su, bt, causal=False, **kw) == 0


def test_validate_tables_on_a_generated_batch(lib):
    from varlen_flashattention_causal_gb300 import workloads as W
    b = W.make_batch([37, 1, 64, 0], [300, 129, 64, 17], Hq=8, Hkv=2, D=64, bs=16, seed=3)
    nb = 1 + max(int(b.block_table[r, :(L + 15) // 16].max()) for r, L in enumerate(b.kv_lens))
    st = va.attn_validate_tables(b.cu_seqlens_q, b.seqused_k, b.block_table, b.max_seqlen_q,
                                 b.max_seqlen_k, 16, nb)
    assert st == 0
    assert va.attn_validate_tables(b.cu_seqlens_q, b.seqused_k, b.block_table, b.max_seqlen_q,
                                   b.max_seqlen_k, 16, nb - 1) == va.ATTN_ERR_TABLE


def test_validate_slots(lib):
    ok = torch.tensor([0, -1, 127, 64], dtype=torch.int64)
    assert va.attn_validate_slots(ok, 16, 8) == 0
    for bad in (-2, 128, 1 << 40):
        t = ok.clone()
        t[2] = bad
        assert va.attn_validate_slots(t, 16, 8) == va.ATTN_ERR_TABLE


def test_debug_switch_reads_the_environment(lib, monkeypatch):
    monkeypatch.delenv("ATTN_DEBUG_VALIDATE", raising=False)
    assert not va.attn_debug_validate_enabled()
    monkeypatch.setenv("ATTN_DEBUG_VALIDATE", "0")
    assert not va.attn_debug_validate_enabled()
    monkeypatch.setenv("ATTN_DEBUG_VALIDATE", "1")
    assert va.attn_debug_validate_enabled()


# ------------------------------------------------ cascade entry point (host side)

def _casc(D=128, bs=16, qdt=torch.bfloat16, kdt=torch.bfloat16, P=32):
    q, kc, out = _cpu(3, 8, D, dtype=qdt), _cpu(8, bs, 2, D, dtype=kdt), _cpu(3, 8, D)
    cu0 = torch.tensor([0, 3], dtype=torch.int32)
    pk = torch.tensor([P], dtype=torch.int32)
    pbt = torch.zeros(4, dtype=torch.int32)
    cu = torch.tensor([0, 1, 2, 3], dtype=torch.int32)
    su = torch.tensor([5, 5, 5], dtype=torch.int32)
    bt = torch.zeros((3, 4), dtype=torch.int32)
    return lambda: va.attn_cascade(q, kc, kc, out, cu0, pk, pbt, P, cu, su, bt, 1, 5, 0.1, prefix_splits=1,
                                   suffix_splits=1, stream=0)


def test_cascade_host_checks(lib):
    """attn_cascade checks both halves on the host before anything runs:
    head size, block size, dtypes, and a prefix that does not end on a block
    boundary ("FlashAttention deep dive", Cascade Attention: the common
    prefix is a whole number of blocks)."""
    assert _status_of(_casc(D=96)) == ERR_HD
    assert _status_of(_casc(bs=24)) == ERR_BS
    assert _status_of(_casc(P=40)) == ERR_SHAPE
    assert _status_of(_casc(kdt=torch.float16)) == ERR_DTYPE
    assert _status_of(_casc(qdt=torch.float8_e4m3fn, kdt=torch.float8_e4m3fn)) == ERR_DTYPE


def test_cascade_split_rule(lib):
    """The library's split counts for the two halves of a cascade call: each
    at least one, more prefix segments for a longer prefix, more suffix
    segments for longer suffixes, and none above the 256 clamp."""
    a, b = va.attn_cascade_splits(64, 64, 1, 4096, 1024, 32, 8, 128, num_sms=152)
    assert 1 <= a <= 256 and 1 <= b <= 256
    a2, _ = va.attn_cascade_splits(64, 64, 1, 65536, 1024, 32, 8, 128, num_sms=152)
    _, b2 = va.attn_cascade_splits(64, 64, 1, 4096, 16384, 32, 8, 128, num_sms=152)
    assert a2 >= a and b2 >= b
    for args in ((0, 64, 1, 4096, 1024, 32, 8, 128), (64, 64, 1, 4096, 1024, 32, 7, 128)):
        with pytest.raises(ValueError):
            va.attn_cascade_splits(*args, num_sms=152)
