// attn_api.cu -- the C ABI of libattn (declared in include/attn.h): host-side
// argument validation, split planning and kernel launches.  No entry point
// allocates device memory or synchronises the host.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/attn.h"
#include "internal.h"
#include "sm100.cuh"

using namespace attn;

// device error word (bit flags from internal.h); kernels get its address
__device__ unsigned g_attn_error_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 256;
constexpr int kTileN = 64;          // keys per K/V tile of the mma kernel

// Filled on a device's first call.  Calls may come from several host
// threads: the fields are written once, under g_dev_fill, before `ready` is
// published with release order; readers that see `ready` (acquire) see them.
struct DevInfo {
    std::atomic<int> ready{0};
    int sms = 0;
    int major = 0, minor = 0;
    unsigned *err = nullptr;
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_fill;

attn_status device_info(DevInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    DevInfo &d = g_dev[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_dev_fill);
        if (!d.ready.load(std::memory_order_relaxed)) {
            int sms = 0, major = 0, minor = 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return ATTN_ERR_CUDA;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
                return ATTN_ERR_CUDA;
            if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
                return ATTN_ERR_CUDA;
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_attn_error_word) != cudaSuccess || !p) return ATTN_ERR_CUDA;
            d.sms = sms;
            d.major = major;
            d.minor = minor;
            d.err = static_cast<unsigned *>(p);
            d.ready.store(1, std::memory_order_release);
        }
    }
    if (d.major != 10 || d.minor != 3) return ATTN_ERR_DEVICE;
    *out = &d;
    return ATTN_OK;
}

// Failure-detection self-test: one thread waits, through the bounded wait
// of the tensor-core kernel's pipeline, on phase 0 of an mbarrier that
// expects one arrival and never gets it.  After the wait limit it gives up
// and raises the timeout bit of the error word.
__global__ void wait_timeout_selftest_kernel(unsigned *err) {
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
    sm100::mbar_init(b, 1);
    sm100::fence_mbar_init();
    abort_flag = 0;
    if (!sm100::mbar_wait(b, 0, &abort_flag)) atomicOr(err, ERR_TIMEOUT);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool is16(attn_dtype t) { return t == ATTN_BF16 || t == ATTN_FP16; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t part_o_bytes(int T, int Hq, int D, int ns) { return align256((size_t)T * Hq * ns * D * sizeof(float)); }

// Workspace layout: the tensor-core kernel's work counters in the first
// kSchedBytes (zeroed by the call that uses them), then the split-KV
// partials (O_s, then LSE_s) when a call splits.
constexpr size_t kSchedBytes = 256;

// Request classes by packed row count (q_len * G):
//   0  rows <= 16: decode and short verify rows, mma.sync kernel with 16-row
//      CTAs (one token x up to 16 heads of a group).  On an e4m3 cache with
//      head size 128 this class ends at 8 rows and runs the transposed
//      decode kernel (8-row CTAs); class 1 then starts at 9 rows;
//   1  17 .. 64 rows: longer verify rows and short chunks, mma.sync kernel
//      with 32- or 64-row CTAs (memory-bound work, where a 128-row
//      tensor-core tile would mostly be padding);
//   2  more than 64 rows: prefill and chunks, tcgen05 kernel.  When the
//      tcgen05 kernel does not take the shape (head size 64, G not dividing
//      128) class 1 extends to every request above 16 rows instead.
constexpr int kLightRows = 16;
constexpr int kMidRows = 64;

// Split rule.  `base` CTAs run without splitting; `target` is the CTA count
// that fills every SM twice.  Too few CTAs: cut each request's keys into
// more segments, each at least `min_tiles` K/V tiles.  With `len_tiles` > 0
// segments are also capped at that many tiles, so one long request in a
// batch of short ones does not become the critical path.
int split_rule(long long base, int max_seqlen_k, long long target, int min_tiles, int len_tiles) {
    if (base <= 0 || max_seqlen_k <= 0) return 1;
    const int tiles = (max_seqlen_k + kTileN - 1) / kTileN;
    long long s = 1;
    if (base < target) s = (2 * target + base - 1) / base;
    if (len_tiles > 0) s = std::max<long long>(s, (tiles + len_tiles - 1) / len_tiles);
    s = std::min<long long>(s, std::max(1, tiles / min_tiles));
    s = std::min<long long>(s, kMaxSplits);
    return (int)std::max<long long>(s, 1);
}

struct ClassPlan {
    bool on;       // launched
    int lo, hi;    // packed-row range of the class
    bool tc;       // tcgen05 kernel (else mma.sync with rpc rows per CTA)
    bool dec;      // transposed decode kernel (class 0 on e4m3 caches)
    int rpc;       // rows per CTA
    int ns;        // segments (automatic choice)
};
struct Plan {
    ClassPlan c[3];
};

// uniform: every request has exactly max_q query tokens (so all requests
// fall in one class); only host scalars are used, nothing is read back
Plan make_plan(int B, int max_q, int max_k, bool uniform, int Hq, int Hkv, int D, int q_dtype, int kv_dtype,
               int sms) {
    Plan pl{};
    const int G = Hq / Hkv;
    const int max_rows = std::max(1, max_q) * G;
    const bool heavy_tc = tc_supported(D, q_dtype, kv_dtype, G);
    const bool dec = dec_supported(D, q_dtype, kv_dtype);
    const int light = dec ? dec_rows_per_cta() : kLightRows;
    const int hi[3] = {light, heavy_tc ? kMidRows : INT32_MAX, INT32_MAX};
    for (int k = 0; k < 3; ++k) {
        ClassPlan &c = pl.c[k];
        c.lo = k == 0 ? 0 : hi[k - 1] + 1;
        c.hi = hi[k];
        if (k == 2 && !heavy_tc) continue;                 // folded into class 1
        // uniform lengths: only max_rows's class; otherwise every class from
        // the smallest request (one token: G rows) to the largest
        c.on = uniform ? (max_rows >= c.lo && max_rows <= c.hi) : (max_rows >= c.lo && G <= c.hi);
        if (!c.on) continue;
        c.tc = (k == 2);
        c.dec = (k == 0 && dec);
        const int rows_cap = std::min(max_rows, c.hi);
        // (class 1 on 16-row CTAs, each row block re-reading K/V from L2,
        // measured slower than one CTA for all of a request's rows)
        c.rpc = c.tc ? tc_rows_per_cta() : (k == 0 ? light : mma_rows_per_cta(rows_cap));
        const long long rb = (rows_cap + c.rpc - 1) / c.rpc;
        if (k == 0)        // decode-like rows: also bound the keys per segment (32 tiles)
            // (the transposed decode kernel fits five CTAs an SM and measured
            // best with more, shorter segments: 0.64 / 0.68 of the copy peak
            // against 0.62 / 0.64 at the 16-row kernel's target on the fp8
            // decode batch)
            c.ns = split_rule((long long)B * Hkv * rb, max_k, (c.dec ? 8LL : 6LL) * sms, 2, 32);
        else if (!c.tc)
            c.ns = split_rule((long long)B * Hkv * rb, max_k, 4LL * sms, 2, rb == 1 ? 32 : 0);
        else
            c.ns = split_rule((long long)B * Hkv * rb, max_k, 2LL * sms, 4, 0);
    }
    return pl;
}

attn_status check_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

struct FwdArgs {
    const void *q;
    int64_t q_stride;
    const void *k_cache, *v_cache;
    void *out;
    int64_t out_stride;
    float *lse;
    const int32_t *cu_seqlens_q, *seqused_k, *block_table;
    int64_t bt_stride;
    int B, T, max_q, max_k, Hq, Hkv, D, bs, num_blocks;
    attn_dtype q_dtype, kv_dtype;
    float scale;
    int causal;
    float q_descale = 1.f, k_descale, v_descale;
    int num_splits;
    void *ws;
    size_t ws_bytes;
    cudaStream_t stream;
    int window_left = -1, window_right = -1;
    float softcap = 0.f;
    const float *sinks = nullptr;
};

attn_status validate_fwd(const FwdArgs &a) {
    if (!a.q || !a.k_cache || !a.v_cache || !a.out || !a.seqused_k || !a.block_table) return ATTN_ERR_NULL;
    if (a.B > 0 && a.cu_seqlens_q == nullptr && a.max_q != 1) return ATTN_ERR_NULL;
    if (a.D != 64 && a.D != 128) return ATTN_ERR_HEAD_SIZE;
    if (a.bs <= 0 || a.bs % 16 != 0) return ATTN_ERR_BLOCK_SIZE;
    // 16-bit q with a cache of the same type or e4m3; e4m3 q with an e4m3
    // cache and head size 128 (out is then bf16)
    const bool q8 = a.q_dtype == ATTN_FP8_E4M3;
    if (!is16(a.q_dtype) && !q8) return ATTN_ERR_DTYPE;
    if (!(a.kv_dtype == a.q_dtype || a.kv_dtype == ATTN_FP8_E4M3)) return ATTN_ERR_DTYPE;
    if (q8 && a.D != 128) return ATTN_ERR_DTYPE;
    if (a.B < 0 || a.B > 65535 || a.T < 0 || a.Hq <= 0 || a.Hq > 65535 || a.Hkv <= 0 || a.Hq % a.Hkv != 0 ||
        a.num_blocks < 0 || a.max_q < 0 || a.max_k < 0 || a.bt_stride < 0 || a.num_splits < 0)
        return ATTN_ERR_SHAPE;
    if (a.q_stride < (int64_t)a.Hq * a.D || a.out_stride < (int64_t)a.Hq * a.D) return ATTN_ERR_SHAPE;
    if ((long long)a.max_q * (a.Hq / a.Hkv) > (1LL << 30)) return ATTN_ERR_SHAPE;
    if (!aligned16(a.q) || !aligned16(a.k_cache) || !aligned16(a.v_cache) || !aligned16(a.out) ||
        (a.q_stride % (q8 ? 16 : 8)) != 0 || (a.out_stride % 8) != 0)
        return ATTN_ERR_ALIGN;
    if (!(a.scale == a.scale) || !(a.k_descale == a.k_descale) || !(a.v_descale == a.v_descale) ||
        !(a.q_descale == a.q_descale))
        return ATTN_ERR_SHAPE;
    if (a.window_left < -1 || a.window_right < -1 || !(a.softcap >= 0.f) || isinf(a.softcap)) return ATTN_ERR_SHAPE;
    return ATTN_OK;
}

// ATTN_DEBUG_VALIDATE=1: copy the integer tables of the call to the host,
// after the work already queued on the stream (which may be writing them),
// and check them with attn_validate_tables.  The block table is copied row
// by row, ceil(kv_len / block_size) entries a row: exactly the entries the
// kernels would read, and only once every kv_len is known to be within
// max_seqlen_k.  A stream that is being captured cannot be synchronised,
// so calls captured into a graph are not checked.
attn_status debug_check_fwd(const FwdArgs &a) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(a.stream, &cs) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) return ATTN_OK;
    std::vector<int32_t> cu(a.cu_seqlens_q ? a.B + 1 : 0), used(a.B);
    if (a.cu_seqlens_q && cudaMemcpyAsync(cu.data(), a.cu_seqlens_q, cu.size() * sizeof(int32_t),
                                          cudaMemcpyDefault, a.stream) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (cudaMemcpyAsync(used.data(), a.seqused_k, used.size() * sizeof(int32_t), cudaMemcpyDefault, a.stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(a.stream) != cudaSuccess)
        return ATTN_ERR_CUDA;
    for (int r = 0; r < a.B; ++r) {
        if (used[r] < 0 || used[r] > a.max_k) return ATTN_ERR_TABLE;
        // rows of a [B, W] table: a row never reaches into the next one
        if (a.B > 1 && (used[r] + a.bs - 1) / a.bs > a.bt_stride) return ATTN_ERR_TABLE;
    }
    const int w = (a.max_k + a.bs - 1) / a.bs;
    std::vector<int32_t> bt((size_t)a.B * std::max(w, 1), 0);
    for (int r = 0; r < a.B; ++r) {
        const int n = (used[r] + a.bs - 1) / a.bs;
        if (n > 0 && cudaMemcpyAsync(bt.data() + (size_t)r * w, a.block_table + (int64_t)r * a.bt_stride,
                                     n * sizeof(int32_t), cudaMemcpyDefault, a.stream) != cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    if (cudaStreamSynchronize(a.stream) != cudaSuccess) return ATTN_ERR_CUDA;
    return attn_validate_tables(a.cu_seqlens_q ? cu.data() : nullptr, used.data(), bt.data(), std::max(w, 1), a.B,
                                a.T, a.max_q, a.max_k, a.bs, a.num_blocks, a.causal);
}

// window bounds that exclude nothing become -1; the keys one CTA can see
// (with a left window bound, at most the window plus the CTA's query span and
// the right bound, from a tile-aligned start) size the split segments
struct Span {
    int wl, wr, max_k_eff;
};
Span key_span(const FwdArgs &a) {
    Span sp;
    sp.wl = (a.window_left >= a.max_k) ? -1 : a.window_left;
    sp.wr = (a.window_right >= a.max_k) ? -1 : a.window_right;
    long long span_k = a.max_k;
    if (sp.wl >= 0 && (a.causal || sp.wr >= 0))
        span_k = std::min<long long>(span_k, (long long)sp.wl + a.max_q + std::max(sp.wr, 0) + kTileN);
    sp.max_k_eff = (int)span_k;
    return sp;
}

Plan plan_for(const FwdArgs &a, const Span &sp, int sms) {
    const bool uniform = (long long)a.T == (long long)a.B * a.max_q;
    return make_plan(a.B, a.max_q, sp.max_k_eff, uniform, a.Hq, a.Hkv, a.D, a.q_dtype, a.kv_dtype, sms);
}

// the kernel parameters every class of a call shares
FwdParams base_params(const FwdArgs &a, const Span &sp, const DevInfo *dev) {
    FwdParams p{};
    p.q = a.q;
    p.q_stride = a.q_stride;
    p.k_cache = a.k_cache;
    p.v_cache = a.v_cache;
    p.out = a.out;
    p.out_stride = a.out_stride;
    p.lse = a.lse;
    p.cu_seqlens_q = a.cu_seqlens_q;
    p.seqused_k = a.seqused_k;
    p.block_table = a.block_table;
    p.bt_stride = a.bt_stride;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.bs = a.bs;
    p.num_blocks = a.num_blocks;
    p.causal = a.causal ? 1 : 0;
    p.scale_log2 = a.scale * a.q_descale * a.k_descale * 1.4426950408889634f;
    p.v_descale = a.v_descale;
    p.err = dev->err;
    p.window_left = sp.wl;
    p.window_right = sp.wr;
    if (a.softcap > 0.f) {
        p.cap_in = a.scale * a.q_descale * a.k_descale / a.softcap;
        p.cap_out = a.softcap * 1.4426950408889634f;
    }
    p.sinks = a.sinks;
    return p;
}

// Launch every class of the plan on `stream`, class k with ns[k] segments.
// A class writes partial states when it is split or when `partials` is set;
// p.sched must already point at a zeroed work counter if a tensor-core class
// is on.
attn_status launch_classes(const FwdArgs &a, const FwdParams &p, const Plan &pl, const int ns[3], int max_k_eff,
                           bool partials, const DevInfo *dev, cudaStream_t stream) {
    const int G = a.Hq / a.Hkv;
    // every segment spans a whole number of K/V tiles
    auto chunk_for = [&](int n) {
        if (n <= 1) return 1 << 30;
        const int per = (max_k_eff + n - 1) / n;
        return ((per + kTileN - 1) / kTileN) * kTileN;
    };
    const int max_rows = std::max(1, a.max_q) * G;
    for (int k = 0; k < 3; ++k) {
        const ClassPlan &c = pl.c[k];
        if (!c.on) continue;
        FwdParams t = p;
        t.nsplit = ns[k];
        t.partials = (partials || ns[k] > 1) ? 1 : 0;
        t.split_chunk = chunk_for(ns[k]);
        t.rows_lo = c.lo;
        t.rows_hi = c.hi;
        t.n_row_blocks = (std::min(max_rows, c.hi) + c.rpc - 1) / c.rpc;
        if ((long long)t.n_row_blocks * ns[k] > 0x7fffffffLL) return ATTN_ERR_SHAPE;
        attn_status st;
        if (c.tc && tc2_supported(a.D, a.q_dtype, a.kv_dtype, G))
            st = check_cuda(launch_fwd_tc2(t, a.q_dtype, a.T, dev->sms, stream));
        else if (c.tc)
            st = check_cuda(launch_fwd_tc(t, a.q_dtype, a.kv_dtype, a.T, dev->sms, stream));
        else if (c.dec && dec_pool_fits(a.num_blocks, a.bs))
            st = check_cuda(launch_fwd_dec(t, a.q_dtype, stream));
        else if (c.dec)   // the 16-row kernel takes any rows <= 8 too
            st = check_cuda(launch_fwd_mma(t, a.D, a.q_dtype, a.kv_dtype, mma_rows_per_cta(c.hi), a.max_q <= 1, stream));
        else
            st = check_cuda(launch_fwd_mma(t, a.D, a.q_dtype, a.kv_dtype, c.rpc, a.max_q <= 1, stream));
        if (st != ATTN_OK) return st;
    }
    return ATTN_OK;
}

// merge the partial states in (part_o, part_lse), part_stride slots per
// (token, head): a token's count by its class (ns), or every token `all`
// slots when all > 0
attn_status launch_combine_for(const FwdArgs &a, const Plan &pl, const int ns[3], int part_stride, float *part_o,
                               float *part_lse, int all, cudaStream_t stream) {
    CombineParams c{};
    c.part_o = part_o;
    c.part_lse = part_lse;
    c.out = a.out;
    c.out_stride = a.out_stride;
    c.lse = a.lse;
    c.cu_seqlens_q = a.cu_seqlens_q;
    c.B = a.B;
    c.T = a.T;
    c.Hq = a.Hq;
    c.D = a.D;
    c.G = a.Hq / a.Hkv;
    c.max_q = a.max_q;
    if (all > 0) {
        c.rows_hi0 = c.rows_hi1 = INT32_MAX;
        c.ns0 = c.ns1 = c.ns2 = all;
    } else {
        c.rows_hi0 = pl.c[0].hi;
        c.rows_hi1 = pl.c[1].hi;
        c.ns0 = ns[0];
        c.ns1 = ns[1];
        c.ns2 = ns[2];
    }
    c.part_stride = part_stride;
    return check_cuda(launch_combine(c, a.q_dtype == ATTN_FP8_E4M3 ? ATTN_BF16 : a.q_dtype, stream));
}

attn_status run_fwd(const FwdArgs &a) {
    attn_status st = validate_fwd(a);
    if (st != ATTN_OK) return st;
    if (a.B == 0 || a.T == 0) return ATTN_OK;
    if (attn_debug_validate_enabled()) {
        st = debug_check_fwd(a);
        if (st != ATTN_OK) return st;
    }
    const int G = a.Hq / a.Hkv;
    // A request of more than kMidRows packed rows may run on the tensor-core
    // kernel, whose work counters live at the start of the workspace: such a
    // call needs one even without split-KV (checked from host scalars alone,
    // before the device is looked up).
    const bool tc_on = tc_supported(a.D, a.q_dtype, a.kv_dtype, G) && (long long)std::max(1, a.max_q) * G > kMidRows;
    if (tc_on) {
        if (!a.ws || a.ws_bytes < kSchedBytes) return ATTN_ERR_WORKSPACE;
        if (!aligned16(a.ws)) return ATTN_ERR_ALIGN;
    }
    DevInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != ATTN_OK) return st;

    const Span sp = key_span(a);
    const Plan pl = plan_for(a, sp, dev->sms);
    int ns[3];
    for (int k = 0; k < 3; ++k)
        ns[k] = !pl.c[k].on ? 1 : (a.num_splits > 0 ? std::min(a.num_splits, kMaxSplits) : pl.c[k].ns);
    auto ns_max = [&]() { return std::max(ns[0], std::max(ns[1], ns[2])); };
    if (a.num_splits <= 0) {
        // automatic: cap to what the workspace holds (its layout is sized by
        // the largest count)
        auto fits = [&](int n) { return n <= 1 || (a.ws && a.ws_bytes >= attn_workspace_size(a.T, a.Hq, a.D, n)); };
        while (!fits(ns_max())) {
            int k = 0;
            for (int j = 1; j < 3; ++j)
                if (ns[j] > ns[k]) k = j;
            --ns[k];
        }
    }
    const int stride = ns_max();
    if (stride > 1) {
        if (!a.ws) return ATTN_ERR_WORKSPACE;
        if (a.ws_bytes < attn_workspace_size(a.T, a.Hq, a.D, stride)) return ATTN_ERR_WORKSPACE;
        if (!aligned16(a.ws)) return ATTN_ERR_ALIGN;
    }

    FwdParams p = base_params(a, sp, dev);
    p.part_stride = stride;
    if (stride > 1) {
        char *base = static_cast<char *>(a.ws) + kSchedBytes;
        p.part_o = reinterpret_cast<float *>(base);
        p.part_lse = reinterpret_cast<float *>(base + part_o_bytes(a.T, a.Hq, a.D, stride));
    }
    if (pl.c[2].on) {
        // the work counters start at zero in every call (a stream-ordered
        // memset: capturable, and no counter state carries over between
        // calls, captured graphs or streams)
        p.sched = static_cast<unsigned long long *>(a.ws);
        st = check_cuda(cudaMemsetAsync(a.ws, 0, 2 * sizeof(unsigned long long), a.stream));
        if (st != ATTN_OK) return st;
    }
    st = launch_classes(a, p, pl, ns, sp.max_k_eff, false, dev, a.stream);
    if (st != ATTN_OK) return st;
    if (stride > 1) st = launch_combine_for(a, pl, ns, stride, p.part_o, p.part_lse, 0, a.stream);
    return st;
}

// ---------------------------------------------------------------- cascade
//
// "FlashAttention deep dive", Cascade Attention: every query attends to a
// prefix shared by all requests (one non-causal call over all query tokens)
// and to its own request's suffix (a causal call), and the two states are
// merged by log-sum-exp.  Here both halves write their segments' partial
// states into one array -- the prefix's ns_p segments in slots [0, ns_p) of
// every (token, head), the suffix's ns_s in [ns_p, ns_p + ns_s) -- and one
// combine merges them all: three launches where the pages' form takes five
// (two split calls with their combines, then the merge).  The prefix half
// runs on a second stream when the caller gives one, so the prefix's
// tensor-core work and the suffix's cache reads overlap.

// Split counts for the two halves sharing the GPU.  The prefix is
// compute-heavy (every query x every prefix key), the suffix reads its
// caches once: each gets a share of the SMs in proportion to its estimated
// time alone (tensor-core work at 0.6 PFLOP/s -- a prefix spread over few
// items runs well below the kernel's full-GPU rate -- and cache bytes at
// 5.5 TB/s), and its segment count fills its share, rounded up for the
// prefix.  On 64 requests over a 4096-key prefix with suffixes of 256-1024
// keys this picks (2, 4): 61.7 us against 60.4 us for the best pair
// measured, (2, 2), and 78 us for the worst, (8, 8).
constexpr double kCascadeFlops = 0.6e15;
constexpr double kCascadeBytes = 5.5e12;
void cascade_splits(const FwdArgs &pre, const FwdArgs &suf, const Plan &pp, const Plan &ps, int sms, int *ns_p,
                    int *ns_s) {
    const int G = pre.Hq / pre.Hkv;
    const double kv_elem = pre.kv_dtype == ATTN_FP8_E4M3 ? 1.0 : 2.0;
    const double t_p = 4.0 * pre.T * pre.Hq * (double)pre.max_k * pre.D / kCascadeFlops;
    const double t_s = (double)suf.B * suf.max_k * suf.Hkv * suf.D * 2.0 * kv_elem / kCascadeBytes +
                       4.0 * suf.T * suf.Hq * (double)suf.max_k * suf.D / kCascadeFlops;
    const double share = (t_p + t_s) > 0.0 ? t_p / (t_p + t_s) : 0.5;
    const int sms_p = std::max(2, std::min(sms - 2, (int)(share * sms + 0.5)));
    const int sms_s = std::max(2, sms - sms_p);
    // prefix: work units per segment (a pair of SMs per item on the tensor
    // cores, else about three CTAs an SM)
    const int rows = std::max(1, pre.T) * G;
    int units = 0;
    double per_unit = 1.0;
    for (int k = 0; k < 3; ++k)
        if (pp.c[k].on && rows >= pp.c[k].lo && rows <= pp.c[k].hi) {
            units = ((rows + pp.c[k].rpc - 1) / pp.c[k].rpc) * pre.Hkv;
            per_unit = pp.c[k].tc ? 2.0 : 1.0 / 3.0;
        }
    const int tiles_p = (pre.max_k + kTileN - 1) / kTileN;
    int np = units > 0 ? (int)std::ceil(sms_p / (per_unit * units)) : 1;
    np = std::max(1, std::min(np, std::max(1, tiles_p / 4)));
    *ns_p = std::min(np, kMaxSplits);
    // suffix: the class-0 rule on its share of the SMs
    int nsx = 1;
    for (int k = 0; k < 3; ++k)
        if (ps.c[k].on) {
            const int rows_cap = std::min(std::max(1, suf.max_q) * G, ps.c[k].hi);
            const long long rb = (rows_cap + ps.c[k].rpc - 1) / ps.c[k].rpc;
            nsx = std::max(nsx, split_rule((long long)suf.B * suf.Hkv * rb, suf.max_k, 6LL * sms_s, 2, 32));
        }
    *ns_s = nsx;
}

struct CascadeArgs {
    FwdArgs pre, suf;             // the two halves (ws, stream, num_splits unused)
    int prefix_splits, suffix_splits;
    void *ws;
    size_t ws_bytes;
    cudaStream_t stream, aux;
};

// host checks of a cascade call; fills the split counts
attn_status check_cascade(CascadeArgs &c, DevInfo **dev_out) {
    attn_status st = validate_fwd(c.pre);
    if (st != ATTN_OK) return st;
    st = validate_fwd(c.suf);
    if (st != ATTN_OK) return st;
    if (c.pre.max_k % c.pre.bs != 0) return ATTN_ERR_SHAPE;   // the suffix starts at a block boundary
    if (c.prefix_splits < 0 || c.suffix_splits < 0) return ATTN_ERR_SHAPE;
    return device_info(dev_out);
}

attn_status run_cascade(CascadeArgs &c) {
    if (c.suf.B == 0 || c.suf.T == 0) return ATTN_OK;
    if (!c.ws || !aligned16(c.ws)) return !c.ws ? ATTN_ERR_WORKSPACE : ATTN_ERR_ALIGN;
    DevInfo *dev = nullptr;
    attn_status st = check_cascade(c, &dev);
    if (st != ATTN_OK) return st;
    if (attn_debug_validate_enabled()) {
        c.pre.stream = c.suf.stream = c.stream;
        st = debug_check_fwd(c.pre);
        if (st == ATTN_OK) st = debug_check_fwd(c.suf);
        if (st != ATTN_OK) return st;
    }
    const Span spp = key_span(c.pre), sps = key_span(c.suf);
    const Plan pp = plan_for(c.pre, spp, dev->sms), ps = plan_for(c.suf, sps, dev->sms);
    int ns_p = 1, ns_s = 1;
    cascade_splits(c.pre, c.suf, pp, ps, dev->sms, &ns_p, &ns_s);
    if (c.prefix_splits > 0) ns_p = std::min(c.prefix_splits, kMaxSplits);
    if (c.suffix_splits > 0) ns_s = std::min(c.suffix_splits, kMaxSplits);
    const int stride = ns_p + ns_s;
    if (c.ws_bytes < attn_workspace_size(c.suf.T, c.suf.Hq, c.suf.D, stride)) return ATTN_ERR_WORKSPACE;

    char *base = static_cast<char *>(c.ws) + kSchedBytes;
    float *part_o = reinterpret_cast<float *>(base);
    float *part_lse = reinterpret_cast<float *>(base + part_o_bytes(c.suf.T, c.suf.Hq, c.suf.D, stride));
    const int D = c.suf.D;
    FwdParams fp = base_params(c.pre, spp, dev), fs = base_params(c.suf, sps, dev);
    fp.part_stride = fs.part_stride = stride;
    fp.part_o = part_o;                       // prefix segments: slots [0, ns_p)
    fp.part_lse = part_lse;
    fs.part_o = part_o + (size_t)ns_p * D;    // suffix segments: slots [ns_p, ns_p + ns_s)
    fs.part_lse = part_lse + ns_p;
    // separate work counters (the halves may run at the same time)
    fp.sched = static_cast<unsigned long long *>(c.ws);
    fs.sched = static_cast<unsigned long long *>(c.ws) + 2;
    int nsp[3] = {ns_p, ns_p, ns_p}, nss[3] = {ns_s, ns_s, ns_s};

    // fork: the prefix half on the aux stream after the work already queued
    // on the main stream; join before the combine.  The two events are this
    // host thread's own (created on its first cascade call on the device),
    // recorded and waited on at once, so calls never share an event.
    const bool fork = c.aux != nullptr && c.aux != c.stream;
    cudaStream_t sp_stream = fork ? c.aux : c.stream;
    static thread_local cudaEvent_t tl_ev[kMaxDevices][2];
    int devno = 0;
    if (cudaGetDevice(&devno) != cudaSuccess || devno < 0 || devno >= kMaxDevices) return ATTN_ERR_CUDA;
    cudaEvent_t *ev = tl_ev[devno];
    if (fork) {
        for (int i = 0; i < 2; ++i)
            if (!ev[i] && cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) return ATTN_ERR_CUDA;
        if (cudaEventRecord(ev[0], c.stream) != cudaSuccess || cudaStreamWaitEvent(c.aux, ev[0], 0) != cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    if (pp.c[2].on) {
        st = check_cuda(cudaMemsetAsync(fp.sched, 0, 2 * sizeof(unsigned long long), sp_stream));
        if (st != ATTN_OK) return st;
    }
    st = launch_classes(c.pre, fp, pp, nsp, spp.max_k_eff, true, dev, sp_stream);
    if (st != ATTN_OK) return st;
    if (ps.c[2].on) {
        st = check_cuda(cudaMemsetAsync(fs.sched, 0, 2 * sizeof(unsigned long long), c.stream));
        if (st != ATTN_OK) return st;
    }
    st = launch_classes(c.suf, fs, ps, nss, sps.max_k_eff, true, dev, c.stream);
    if (st != ATTN_OK) return st;
    if (fork) {
        if (cudaEventRecord(ev[1], c.aux) != cudaSuccess || cudaStreamWaitEvent(c.stream, ev[1], 0) != cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    return launch_combine_for(c.suf, ps, nss, stride, part_o, part_lse, stride, c.stream);
}

}  // namespace

extern "C" {

size_t attn_workspace_size(int total_q, int Hq, int D, int num_splits) {
    if (num_splits <= 1 || total_q <= 0 || Hq <= 0 || D <= 0) return kSchedBytes;
    return kSchedBytes + part_o_bytes(total_q, Hq, D, num_splits) +
           align256((size_t)total_q * Hq * num_splits * sizeof(float));
}

int attn_num_splits_typed(int B, int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D, attn_dtype q_dtype,
                          attn_dtype kv_dtype, int num_sms) {
    if (Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0 || B <= 0) return 1;
    // every request class may be present: the largest count sizes the workspace
    const Plan pl = make_plan(B, max_seqlen_q, max_seqlen_k, false, Hq, Hkv, D, q_dtype, kv_dtype, num_sms);
    int n = 1;
    for (int k = 0; k < 3; ++k)
        if (pl.c[k].on) n = std::max(n, pl.c[k].ns);
    return n;
}

int attn_num_splits(int B, int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int num_sms) {
    return attn_num_splits_typed(B, max_seqlen_q, max_seqlen_k, Hq, Hkv, 128, ATTN_BF16, ATTN_BF16, num_sms);
}

int attn_tile_kind(int q_lo, int q_hi, int k_lo, int k_hi, int ctx) { return tile_kind(q_lo, q_hi, k_lo, k_hi, ctx); }

const char *attn_status_string(attn_status s) {
    switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULL: return "required pointer is NULL";
    case ATTN_ERR_SHAPE: return "inconsistent sizes or strides";
    case ATTN_ERR_DTYPE: return "unsupported dtype combination";
    case ATTN_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case ATTN_ERR_BLOCK_SIZE: return "block_size must be a positive multiple of 16";
    case ATTN_ERR_HEAD_SIZE: return "head size must be 64 or 128";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_CUDA: return "CUDA runtime error";
    case ATTN_ERR_DEVICE: return "current device is not sm_103";
    case ATTN_ERR_TABLE: return "cu_seqlens_q, seqused_k, block_table or slot_mapping breaks the contract";
    }
    return "unknown status";
}

attn_status attn_selftest_wait_timeout(attn_stream_t stream) {
    DevInfo *dev = nullptr;
    const attn_status st = device_info(&dev);
    if (st != ATTN_OK) return st;
    wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(dev->err);
    return check_cuda(cudaGetLastError());
}

int attn_device_error_flag(int reset) {
    unsigned v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbol(&v, g_attn_error_word, sizeof v) != cudaSuccess) return -1;
    if (reset) {
        const unsigned z = 0;
        if (cudaMemcpyToSymbol(g_attn_error_word, &z, sizeof z) != cudaSuccess) return -1;
    }
    return (int)v;
}

attn_status attn_varlen_prefill(const void *q, int64_t q_stride_tok, const void *k_cache, const void *v_cache,
                                void *out, int64_t out_stride_tok, float *lse_out, const int32_t *cu_seqlens_q,
                                const int32_t *seqused_k, const int32_t *block_table, int64_t bt_row_stride, int B,
                                int total_q, int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D,
                                int block_size, int num_blocks, attn_dtype q_dtype, attn_dtype kv_dtype,
                                float softmax_scale, int causal, float k_descale, float v_descale, int num_splits,
                                void *workspace, size_t ws_bytes, attn_stream_t stream) {
    return attn_varlen_prefill_ext(q, q_stride_tok, k_cache, v_cache, out, out_stride_tok, lse_out, cu_seqlens_q,
                                   seqused_k, block_table, bt_row_stride, B, total_q, max_seqlen_q, max_seqlen_k, Hq,
                                   Hkv, D, block_size, num_blocks, q_dtype, kv_dtype, softmax_scale, causal, 1.f,
                                   k_descale, v_descale, -1, -1, 0.f, nullptr, num_splits, workspace, ws_bytes,
                                   stream);
}

attn_status attn_varlen_prefill_ext(const void *q, int64_t q_stride_tok, const void *k_cache, const void *v_cache,
                                    void *out, int64_t out_stride_tok, float *lse_out, const int32_t *cu_seqlens_q,
                                    const int32_t *seqused_k, const int32_t *block_table, int64_t bt_row_stride,
                                    int B, int total_q, int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D,
                                    int block_size, int num_blocks, attn_dtype q_dtype, attn_dtype kv_dtype,
                                    float softmax_scale, int causal, float q_descale, float k_descale,
                                    float v_descale, int window_left, int window_right, float softcap,
                                    const float *sinks,
                                    int num_splits, void *workspace, size_t ws_bytes, attn_stream_t stream) {
    FwdArgs a{};
    a.q = q;
    a.q_stride = q_stride_tok;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.out = out;
    a.out_stride = out_stride_tok;
    a.lse = lse_out;
    a.cu_seqlens_q = cu_seqlens_q;
    a.seqused_k = seqused_k;
    a.block_table = block_table;
    a.bt_stride = bt_row_stride;
    a.B = B;
    a.T = total_q;
    a.max_q = max_seqlen_q;
    a.max_k = max_seqlen_k;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.bs = block_size;
    a.num_blocks = num_blocks;
    a.q_dtype = q_dtype;
    a.kv_dtype = kv_dtype;
    a.scale = softmax_scale;
    a.causal = causal;
    a.k_descale = k_descale;
    a.v_descale = v_descale;
    a.num_splits = num_splits;
    a.ws = workspace;
    a.ws_bytes = ws_bytes;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    a.q_descale = q_descale;
    a.window_left = window_left;
    a.window_right = window_right;
    a.softcap = softcap;
    a.sinks = sinks;
    if (B > 0 && !cu_seqlens_q) return ATTN_ERR_NULL;
    return run_fwd(a);
}

attn_status attn_paged_decode(const void *q, const void *k_cache, const void *v_cache, void *out, float *lse_out,
                              const int32_t *seq_lens, const int32_t *block_table, int64_t bt_row_stride, int B,
                              int max_seq_len, int Hq, int Hkv, int D, int block_size, int num_blocks,
                              attn_dtype q_dtype, attn_dtype kv_dtype, float softmax_scale, float k_descale,
                              float v_descale, int num_splits, void *workspace, size_t ws_bytes,
                              attn_stream_t stream) {
    FwdArgs a{};
    a.q = q;
    a.q_stride = (int64_t)Hq * D;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.out = out;
    a.out_stride = (int64_t)Hq * D;
    a.lse = lse_out;
    a.cu_seqlens_q = nullptr;   // request r owns query row r
    a.seqused_k = seq_lens;
    a.block_table = block_table;
    a.bt_stride = bt_row_stride;
    a.B = B;
    a.T = B;
    a.max_q = 1;
    a.max_k = max_seq_len;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.bs = block_size;
    a.num_blocks = num_blocks;
    a.q_dtype = q_dtype;
    a.kv_dtype = kv_dtype;
    a.scale = softmax_scale;
    a.causal = 1;
    a.k_descale = k_descale;
    a.v_descale = v_descale;
    a.num_splits = num_splits;
    a.ws = workspace;
    a.ws_bytes = ws_bytes;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    return run_fwd(a);
}

static void fill_cascade(CascadeArgs &c, const void *q, int64_t q_stride_tok, const void *k_cache,
                         const void *v_cache, void *out, int64_t out_stride_tok, float *lse_out,
                         const int32_t *cu_prefix_query_lens, const int32_t *prefix_kv_lens,
                         const int32_t *prefix_block_table, int prefix_len, const int32_t *cu_seqlens_q,
                         const int32_t *suffix_kv_lens, const int32_t *suffix_block_table, int64_t bt_row_stride,
                         int B, int total_q, int max_seqlen_q, int max_suffix_len, int Hq, int Hkv, int D,
                         int block_size, int num_blocks, attn_dtype q_dtype, attn_dtype kv_dtype, float softmax_scale,
                         float k_descale, float v_descale) {
    for (int h = 0; h < 2; ++h) {
        FwdArgs &a = h ? c.suf : c.pre;
        a.q = q;
        a.q_stride = q_stride_tok;
        a.k_cache = k_cache;
        a.v_cache = v_cache;
        a.out = out;
        a.out_stride = out_stride_tok;
        a.lse = lse_out;
        a.T = total_q;
        a.Hq = Hq;
        a.Hkv = Hkv;
        a.D = D;
        a.bs = block_size;
        a.num_blocks = num_blocks;
        a.q_dtype = q_dtype;
        a.kv_dtype = kv_dtype;
        a.scale = softmax_scale;
        a.k_descale = k_descale;
        a.v_descale = v_descale;
    }
    // prefix: one "request" holding every query token, non-causal (all prefix
    // keys precede every query), over the shared block row
    c.pre.cu_seqlens_q = cu_prefix_query_lens;
    c.pre.seqused_k = prefix_kv_lens;
    c.pre.block_table = prefix_block_table;
    c.pre.bt_stride = 0;
    c.pre.B = 1;
    c.pre.max_q = total_q;
    c.pre.max_k = prefix_len;
    c.pre.causal = 0;
    // suffix: each request over its own blocks, causal with bottom-right alignment
    c.suf.cu_seqlens_q = cu_seqlens_q;
    c.suf.seqused_k = suffix_kv_lens;
    c.suf.block_table = suffix_block_table;
    c.suf.bt_stride = bt_row_stride;
    c.suf.B = B;
    c.suf.max_q = max_seqlen_q;
    c.suf.max_k = max_suffix_len;
    c.suf.causal = 1;
}

attn_status attn_cascade(const void *q, int64_t q_stride_tok, const void *k_cache, const void *v_cache, void *out,
                         int64_t out_stride_tok, float *lse_out, const int32_t *cu_prefix_query_lens,
                         const int32_t *prefix_kv_lens, const int32_t *prefix_block_table, int prefix_len,
                         const int32_t *cu_seqlens_q, const int32_t *suffix_kv_lens,
                         const int32_t *suffix_block_table, int64_t bt_row_stride, int B, int total_q,
                         int max_seqlen_q, int max_suffix_len, int Hq, int Hkv, int D, int block_size,
                         int num_blocks, attn_dtype q_dtype, attn_dtype kv_dtype, float softmax_scale,
                         float k_descale, float v_descale, int prefix_splits, int suffix_splits, void *workspace,
                         size_t ws_bytes, attn_stream_t stream, attn_stream_t aux_stream) {
    if (B > 0 && (!cu_seqlens_q || !cu_prefix_query_lens || !prefix_kv_lens)) return ATTN_ERR_NULL;
    if (q_dtype == ATTN_FP8_E4M3) return ATTN_ERR_DTYPE;   // no q_descale in this entry point
    CascadeArgs c{};
    fill_cascade(c, q, q_stride_tok, k_cache, v_cache, out, out_stride_tok, lse_out, cu_prefix_query_lens,
                 prefix_kv_lens, prefix_block_table, prefix_len, cu_seqlens_q, suffix_kv_lens, suffix_block_table,
                 bt_row_stride, B, total_q, max_seqlen_q, max_suffix_len, Hq, Hkv, D, block_size, num_blocks,
                 q_dtype, kv_dtype, softmax_scale, k_descale, v_descale);
    c.prefix_splits = prefix_splits;
    c.suffix_splits = suffix_splits;
    c.ws = workspace;
    c.ws_bytes = ws_bytes;
    c.stream = reinterpret_cast<cudaStream_t>(stream);
    c.aux = reinterpret_cast<cudaStream_t>(aux_stream);
    return run_cascade(c);
}

int attn_cascade_splits(int B, int total_q, int max_seqlen_q, int prefix_len, int max_suffix_len, int Hq, int Hkv,
                        int D, int q_dtype, int kv_dtype, int num_sms, int *prefix_splits, int *suffix_splits) {
    if (B <= 0 || total_q <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || num_sms <= 0 || !prefix_splits ||
        !suffix_splits)
        return -1;
    CascadeArgs c{};
    fill_cascade(c, nullptr, 0, nullptr, nullptr, nullptr, 0, nullptr, nullptr, nullptr, nullptr, prefix_len, nullptr,
                 nullptr, nullptr, 0, B, total_q, max_seqlen_q, max_suffix_len, Hq, Hkv, D, 16, 1,
                 (attn_dtype)q_dtype, (attn_dtype)kv_dtype, 1.f, 1.f, 1.f);
    const Span spp = key_span(c.pre), sps = key_span(c.suf);
    const Plan pp = plan_for(c.pre, spp, num_sms), ps = plan_for(c.suf, sps, num_sms);
    cascade_splits(c.pre, c.suf, pp, ps, num_sms, prefix_splits, suffix_splits);
    return 0;
}

attn_status attn_merge_states(void *out, float *lse_out, const void *o1, const float *lse1, const void *o2,
                              const float *lse2, int T, int Hq, int D, attn_dtype dtype, attn_stream_t stream) {
    if (!out || !o1 || !lse1 || !o2 || !lse2) return ATTN_ERR_NULL;
    if (T < 0 || Hq <= 0) return ATTN_ERR_SHAPE;
    if (D != 64 && D != 128) return ATTN_ERR_HEAD_SIZE;
    if (!(dtype == ATTN_BF16 || dtype == ATTN_FP16 || dtype == ATTN_FP32)) return ATTN_ERR_DTYPE;
    if (!aligned16(out) || !aligned16(o1) || !aligned16(o2)) return ATTN_ERR_ALIGN;
    if (T == 0) return ATTN_OK;
    DevInfo *dev = nullptr;
    attn_status st = device_info(&dev);
    if (st != ATTN_OK) return st;
    return check_cuda(launch_merge(out, lse_out, o1, lse1, o2, lse2, T, Hq, D, dtype,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

attn_status kv_cache_write(const void *key, int64_t key_stride_tok, const void *value, int64_t value_stride_tok,
                           void *k_cache, void *v_cache, const int64_t *slot_mapping, int T, int Hkv, int D,
                           int block_size, int num_blocks, attn_dtype src_dtype, attn_dtype kv_dtype, float k_scale,
                           float v_scale, attn_stream_t stream) {
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return ATTN_ERR_NULL;
    if (D != 64 && D != 128) return ATTN_ERR_HEAD_SIZE;
    if (block_size <= 0 || block_size % 16 != 0) return ATTN_ERR_BLOCK_SIZE;
    if (!is16(src_dtype)) return ATTN_ERR_DTYPE;
    if (!(kv_dtype == src_dtype || kv_dtype == ATTN_FP8_E4M3)) return ATTN_ERR_DTYPE;
    if (T < 0 || Hkv <= 0 || num_blocks < 0 || key_stride_tok < (int64_t)Hkv * D ||
        value_stride_tok < (int64_t)Hkv * D)
        return ATTN_ERR_SHAPE;
    if (kv_dtype == ATTN_FP8_E4M3 && !(k_scale > 0.f && v_scale > 0.f)) return ATTN_ERR_SHAPE;
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache) ||
        key_stride_tok % 8 != 0 || value_stride_tok % 8 != 0)
        return ATTN_ERR_ALIGN;
    if (T == 0) return ATTN_OK;
    if (attn_debug_validate_enabled()) {
        // see debug_check_fwd: host copy of the slots, skipped under capture
        const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return ATTN_ERR_CUDA;
        if (cs == cudaStreamCaptureStatusNone) {
            std::vector<int64_t> slots(T);
            if (cudaMemcpyAsync(slots.data(), slot_mapping, slots.size() * sizeof(int64_t), cudaMemcpyDefault, s) !=
                    cudaSuccess ||
                cudaStreamSynchronize(s) != cudaSuccess)
                return ATTN_ERR_CUDA;
            const attn_status vs = attn_validate_slots(slots.data(), T, block_size, num_blocks);
            if (vs != ATTN_OK) return vs;
        }
    }
    DevInfo *dev = nullptr;
    attn_status st = device_info(&dev);
    if (st != ATTN_OK) return st;
    return check_cuda(launch_kv_write(key, key_stride_tok, value, value_stride_tok, k_cache, v_cache, slot_mapping, T,
                                      Hkv, D, block_size, num_blocks, src_dtype, kv_dtype, k_scale, v_scale, dev->err,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
