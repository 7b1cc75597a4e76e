// internal.h -- parameter blocks and launcher declarations shared by the
// translation units of libattn (not part of the public C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

// storage type codes (same numbering as attn_dtype in include/attn.h)
enum : int { DT_BF16 = 0, DT_FP16 = 1, DT_E4M3 = 2, DT_FP32 = 3 };

// error bits of the device error word
enum : unsigned { ERR_BLOCK_ID = 1u, ERR_SLOT = 2u, ERR_TIMEOUT = 4u };

// One attention launch over the requests whose packed row count
// rows = q_len * G lies in [rows_lo, rows_hi].  Packed row p of a request
// is query token p / G, query head kvh * G + p % G (all heads of one KV
// group side by side, so each K/V tile serves G heads).
struct FwdParams {
    const void *q;
    int64_t q_stride;            // elements between consecutive tokens
    const void *k_cache;
    const void *v_cache;
    void *out;
    int64_t out_stride;
    float *lse;                  // [T, Hq] or nullptr
    const int32_t *cu_seqlens_q; // nullptr: request r owns token r (decode)
    const int32_t *seqused_k;
    const int32_t *block_table;
    int64_t bt_stride;
    int B, Hq, Hkv, G, bs, num_blocks;
    int causal;
    float scale_log2;            // softmax_scale * k_descale * log2(e)
    float v_descale;
    int nsplit;                  // KV segments per (request, KV head, row block)
    int split_chunk;             // keys per segment (multiple of the KV tile)
    int part_stride;             // segment slots per (token, head) in the workspace
    float *part_o;               // [T, Hq, part_stride, D] fp32, segment s at slot s
    float *part_lse;             // [T, Hq, part_stride]
    int partials;                // 1: write normalised partial states there instead of
                                 // out / lse (split-KV, and both halves of a cascade call)
    int rows_lo, rows_hi;
    int n_row_blocks;            // row blocks of the largest request of the class
    unsigned *err;
    // variants: keys p - window_left .. p + window_right around the query's
    // absolute position p (-1 = unlimited side); soft cap (cap_in =
    // scale * k_descale / softcap applied to the raw dot product, cap_out =
    // softcap * log2(e); cap_in = 0: off); per-query-head sink logits
    // (natural log; nullptr: none), taken into the state of segment 0
    int window_left, window_right;
    float cap_in, cap_out;
    const float *sinks;
    // tensor-core kernel only: {next ticket, unused} of this call's work
    // counter, in the caller's workspace, zeroed before the launch
    unsigned long long *sched;
};

// Split-KV reduction over the partial states of every token whose request
// ran with more than one segment.  A token's request is found from
// cu_seqlens_q (nullptr: token t is request t); its class -- packed rows
// q_len * G up to rows_hi0, up to rows_hi1, or above -- gives its segment
// count ns0, ns1 or ns2.
struct CombineParams {
    const float *part_o;
    const float *part_lse;
    void *out;
    int64_t out_stride;
    float *lse;
    const int32_t *cu_seqlens_q;
    int B, T, Hq, D, G, max_q;
    int rows_hi0, rows_hi1;
    int ns0, ns1, ns2, part_stride;
};

// Launch with programmatic stream serialisation (the kernel calls
// pdl_wait() before touching global memory); stream-ordered like <<< >>>
// and capturable in a CUDA graph.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// launchers (return the launch error)
// single_token: every request of the call has one query token (max_q 1)
cudaError_t launch_fwd_mma(const FwdParams &p, int D, int q_dtype, int kv_dtype, int rows_per_cta, bool single_token,
                           cudaStream_t stream);
cudaError_t launch_combine(const CombineParams &p, int out_dtype, cudaStream_t stream);
cudaError_t launch_merge(void *out, float *lse_out, const void *o1, const float *lse1, const void *o2,
                         const float *lse2, int T, int Hq, int D, int dtype, cudaStream_t stream);
cudaError_t launch_kv_write(const void *key, int64_t ks, const void *value, int64_t vs, void *k_cache,
                            void *v_cache, const int64_t *slot, int T, int Hkv, int D, int bs, int num_blocks,
                            int src_dtype, int kv_dtype, float k_scale, float v_scale, unsigned *err,
                            cudaStream_t stream);

// Tile classification ("vLLM 中 Attention Kernel 如何并行处理多个请求", sec. 4)
// for query positions [q_lo, q_hi) of a request with cached context ctx
// (query i sees keys j <= ctx + i) against keys [k_lo, k_hi):
// 0 = skip (all in the future), 1 = full (no mask), 2 = diagonal (mask).
__host__ __device__ inline int tile_kind(int q_lo, int q_hi, int k_lo, int k_hi, int ctx) {
    if (q_hi <= q_lo || k_hi <= k_lo) return 0;
    if ((long long)k_lo > (long long)ctx + q_hi - 1) return 0;
    if ((long long)k_hi - 1 <= (long long)ctx + q_lo) return 1;
    return 2;
}

// rows per CTA of the mma kernel for a given largest packed row count
int mma_rows_per_cta(int max_rows);

// decode-shape kernel on transposed tiles (e4m3 cache, head size 128): whether
// it takes the shape, its rows per CTA (requests of up to that many packed
// rows), and its launcher
bool dec_supported(int D, int q_dtype, int kv_dtype);
// its TMA maps address cache slots with 32-bit coordinates: the pool's
// num_blocks * bs slots must stay below 2^31 (else the 16-row kernel runs)
bool dec_pool_fits(int num_blocks, int bs);
int dec_rows_per_cta();
cudaError_t launch_fwd_dec(const FwdParams &p, int q_dtype, cudaStream_t stream);

// tcgen05 kernel: whether it handles this shape, rows per CTA, launcher
bool tc_supported(int D, int q_dtype, int kv_dtype, int G);
int tc_rows_per_cta();
// (persistent: at most num_sms CTAs)
cudaError_t launch_fwd_tc(const FwdParams &p, int q_dtype, int kv_dtype, int64_t T, int num_sms,
                          cudaStream_t stream);
// the same work on pairs of SMs (16-bit q and cache, head size 128): whether
// it takes the shape, and its launcher (persistent clusters of two CTAs)
bool tc2_supported(int D, int q_dtype, int kv_dtype, int G);
cudaError_t launch_fwd_tc2(const FwdParams &p, int q_dtype, int64_t T, int num_sms, cudaStream_t stream);

}  // namespace attn
