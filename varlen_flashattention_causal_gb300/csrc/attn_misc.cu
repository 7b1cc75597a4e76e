// attn_misc.cu -- the memory-bound side kernels of the attention path:
//   * kv_write_kernel   reshape_and_cache_flash ("FlashAttention deep dive",
//                       KV cache update): scatter new K/V rows to their slots,
//                       optionally quantising to e4m3
//   * combine_kernel    split-KV reduction ("vLLM 中 Attention Kernel 如何并行
//                       处理多个请求", sec. 12): merge the per-segment states
//   * merge_kernel      merge_attn_states (cascade attention, stage 3)
#include <algorithm>
#include <climits>

#include "common.cuh"

namespace attn {

// ----------------------------------------------------------------- KV write

// One thread moves 8 consecutive elements (16 source bytes) of one
// (token, KV head) row.  slot < 0 skips the token; a slot past the cache is
// never written and raises ERR_SLOT.
template <int ST, int CT>
__global__ void __launch_bounds__(256) kv_write_kernel(const uint8_t *__restrict__ key, int64_t ks,
                                                        const uint8_t *__restrict__ value, int64_t vs,
                                                        uint8_t *__restrict__ k_cache, uint8_t *__restrict__ v_cache,
                                                        const int64_t *__restrict__ slot_mapping, int T, int Hkv,
                                                        int D, int bs, int num_blocks, float k_scale, float v_scale,
                                                        unsigned *err) {
    pdl_wait();
    pdl_trigger();
    const int chunks = D / 8;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = (int64_t)T * Hkv * chunks;
    if (idx >= total) return;
    const int c = (int)(idx % chunks);
    const int h = (int)((idx / chunks) % Hkv);
    const int64_t t = idx / ((int64_t)chunks * Hkv);
    const int64_t slot = slot_mapping[t];
    if (slot < 0) return;
    if (slot >= (int64_t)num_blocks * bs) {
        raise_error(err, ERR_SLOT);
        return;
    }
    const int64_t src_k = (t * ks + (int64_t)h * D + c * 8) * 2;
    const int64_t src_v = (t * vs + (int64_t)h * D + c * 8) * 2;
    const int64_t dst = (slot * Hkv + h) * D + c * 8;   // elements; slot = block * bs + row
    const int4 kx = ldg_nc16(key + src_k);
    const int4 vx = ldg_nc16(value + src_v);
    if constexpr (CT == ST) {
        *reinterpret_cast<int4 *>(k_cache + dst * 2) = kx;
        *reinterpret_cast<int4 *>(v_cache + dst * 2) = vx;
    } else {
        // e4m3(x / scale): fp32 division (IEEE, round to nearest), then one
        // rounding to e4m3, nearest-even, saturating to +-448
        using T = typename Elem<ST>::T;
        const T *ke = reinterpret_cast<const T *>(&kx);
        const T *ve = reinterpret_cast<const T *>(&vx);
        uint32_t kq[2], vq[2];
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            uint32_t kw = 0, vw = 0;
#pragma unroll
            for (int j = 0; j < 4; j += 2) {
                const float2 kf = make_float2(__fdiv_rn(to_float(ke[w * 4 + j]), k_scale),
                                              __fdiv_rn(to_float(ke[w * 4 + j + 1]), k_scale));
                const float2 vf = make_float2(__fdiv_rn(to_float(ve[w * 4 + j]), v_scale),
                                              __fdiv_rn(to_float(ve[w * 4 + j + 1]), v_scale));
                const uint32_t k2 = __nv_cvt_float2_to_fp8x2(kf, __NV_SATFINITE, __NV_E4M3);
                const uint32_t v2 = __nv_cvt_float2_to_fp8x2(vf, __NV_SATFINITE, __NV_E4M3);
                kw |= (k2 & 0xffffu) << (j * 8);
                vw |= (v2 & 0xffffu) << (j * 8);
            }
            kq[w] = kw;
            vq[w] = vw;
        }
        *reinterpret_cast<uint2 *>(k_cache + dst) = make_uint2(kq[0], kq[1]);
        *reinterpret_cast<uint2 *>(v_cache + dst) = make_uint2(vq[0], vq[1]);
    }
}

cudaError_t launch_kv_write(const void *key, int64_t ks, const void *value, int64_t vs, void *k_cache,
                            void *v_cache, const int64_t *slot, int T, int Hkv, int D, int bs, int num_blocks,
                            int src_dtype, int kv_dtype, float k_scale, float v_scale, unsigned *err,
                            cudaStream_t stream) {
    const int64_t total = (int64_t)T * Hkv * (D / 8);
    if (total == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((total + 255) / 256);
    auto *k = reinterpret_cast<const uint8_t *>(key);
    auto *v = reinterpret_cast<const uint8_t *>(value);
    auto *kc = reinterpret_cast<uint8_t *>(k_cache);
    auto *vc = reinterpret_cast<uint8_t *>(v_cache);
#define KVW(ST, CT)                                                                                          \
    launch_pdl(kv_write_kernel<ST, CT>, dim3(blocks), dim3(256), 0, stream, k, ks, v, vs, kc, vc, slot, T, Hkv, D, \
               bs, num_blocks, k_scale, v_scale, err)
    if (src_dtype == DT_BF16 && kv_dtype == DT_BF16) return KVW(DT_BF16, DT_BF16);
    if (src_dtype == DT_FP16 && kv_dtype == DT_FP16) return KVW(DT_FP16, DT_FP16);
    if (src_dtype == DT_BF16 && kv_dtype == DT_E4M3) return KVW(DT_BF16, DT_E4M3);
    if (src_dtype == DT_FP16 && kv_dtype == DT_E4M3) return KVW(DT_FP16, DT_E4M3);
#undef KVW
    return cudaErrorInvalidValue;
}

// ------------------------------------------------------------ state merges

template <class T>
__device__ __forceinline__ float4 load4(const T *p);
template <>
__device__ __forceinline__ float4 load4<float>(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
template <>
__device__ __forceinline__ float4 load4<__half>(const __half *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

template <class T>
__device__ __forceinline__ void store4(T *p, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float *p, float4 v) {
    *reinterpret_cast<float4 *>(p) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *p, float4 v) {
    *reinterpret_cast<uint2 *>(p) = make_uint2(pack2<true>(v.x, v.y), pack2<true>(v.z, v.w));
}
template <>
__device__ __forceinline__ void store4<__half>(__half *p, float4 v) {
    *reinterpret_cast<uint2 *>(p) = make_uint2(pack2<false>(v.x, v.y), pack2<false>(v.z, v.w));
}

constexpr int kCombineBatch = 8;   // segments whose partial rows a lane loads at once

// Merge of one (token t, query head h) by one warp.  Segment s contributes
// with weight exp(lse_s - lse), lse = log sum_s exp(lse_s); segments with
// lse_s = -inf (no visible key) contribute nothing.
template <class OT>
__device__ __forceinline__ void combine_row(const CombineParams &p, int t, int h, int ns, int lane) {
    const int64_t base = ((int64_t)t * p.Hq + h) * (int64_t)p.part_stride;
    const float *ls = p.part_lse + base;
    const int D = p.D;
    if (ns <= kCombineBatch) {
        // one round trip: every lane loads all ns lse values (one address
        // per segment, broadcast across the warp) with its own O columns,
        // and takes the maximum itself
        const int d = lane * 4;
        const float *po = p.part_o + base * D + d;
        float l[kCombineBatch];
        float4 v[kCombineBatch];
#pragma unroll
        for (int k = 0; k < kCombineBatch; ++k) {
            const bool in = k < ns;
            l[k] = in ? ls[k] : -INFINITY;
            v[k] = (in && d < D) ? *reinterpret_cast<const float4 *>(po + (int64_t)k * D)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < kCombineBatch; ++k) mx = fmaxf(mx, l[k]);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float wsum = 0.f;
        if (mx != -INFINITY) {
#pragma unroll
            for (int k = 0; k < kCombineBatch; ++k) {
                // an empty segment wrote only its lse: its O slot is not used
                const float w = l[k] == -INFINITY ? 0.f : expf(l[k] - mx);
                if (w == 0.f) v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                wsum += w;
                acc.x += w * v[k].x;
                acc.y += w * v[k].y;
                acc.z += w * v[k].z;
                acc.w += w * v[k].w;
            }
        }
        const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
        if (d < D) {
            OT *out = reinterpret_cast<OT *>(p.out) + (int64_t)t * p.out_stride + (int64_t)h * D;
            store4<OT>(out + d, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
        }
        if (lane == 0 && p.lse) p.lse[(int64_t)t * p.Hq + h] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
        return;
    }
    float mx = -INFINITY;
    for (int s = lane; s < ns; s += 32) mx = fmaxf(mx, ls[s]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const int d = lane * 4;                       // this lane's four columns
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (mx != -INFINITY && d < D) {
        const float *po = p.part_o + base * D + d;
        for (int s0 = 0; s0 < ns; s0 += kCombineBatch) {
            // a batch of segments in flight: all loads first, then the sums
            float l[kCombineBatch];
            float4 v[kCombineBatch];
#pragma unroll
            for (int k = 0; k < kCombineBatch; ++k) {
                const bool in = s0 + k < ns;
                l[k] = in ? ls[s0 + k] : -INFINITY;
                v[k] = in ? *reinterpret_cast<const float4 *>(po + (int64_t)(s0 + k) * D)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < kCombineBatch; ++k) {
                // an empty segment wrote only its lse: its O slot is never read
                const float w = l[k] == -INFINITY ? 0.f : expf(l[k] - mx);
                if (w == 0.f) v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                wsum += w;
                acc.x += w * v[k].x;
                acc.y += w * v[k].y;
                acc.z += w * v[k].z;
                acc.w += w * v[k].w;
            }
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    if (d < D) {
        OT *out = reinterpret_cast<OT *>(p.out) + (int64_t)t * p.out_stride + (int64_t)h * D;
        store4<OT>(out + d, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
    }
    if (lane == 0 && p.lse) p.lse[(int64_t)t * p.Hq + h] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

// General form: one warp per (token, query head); the token's request is
// found by binary search in cu_seqlens_q, its class gives the segment
// count, and tokens of requests that ran with one segment are skipped.
template <class OT>
__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
    pdl_wait();
    pdl_trigger();
    const int warp_global = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp_global >= p.T * p.Hq) return;
    const int t = warp_global / p.Hq;
    const int h = warp_global % p.Hq;
    int q_len = 1;
    if (p.cu_seqlens_q) {
        int lo = 0, hi = p.B - 1;                 // last r with cu[r] <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.cu_seqlens_q[mid] <= t) lo = mid;
            else hi = mid - 1;
        }
        q_len = p.cu_seqlens_q[lo + 1] - p.cu_seqlens_q[lo];
    }
    const int rows = q_len * p.G;
    const int ns = rows <= p.rows_hi0 ? p.ns0 : (rows <= p.rows_hi1 ? p.ns1 : p.ns2);
    if (ns <= 1) return;
    combine_row<OT>(p, t, h, ns, lane);
}

// Per-request form, for calls in which no request above 64 packed rows was
// split (the usual case: decode and verify rows next to unsplit prefill
// chunks).  One CTA per (request, 8 query heads, query token): two loads
// give the request's class, so the CTAs of unsplit requests exit at once
// instead of one warp per token and head searching for its request.
constexpr int kCombineHeads = 8;
template <class OT>
__global__ void __launch_bounds__(32 * kCombineHeads) combine_light_kernel(const CombineParams p) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x;
    int t0 = r, q_len = 1;
    if (p.cu_seqlens_q) {
        t0 = p.cu_seqlens_q[r];
        q_len = p.cu_seqlens_q[r + 1] - t0;
    }
    const int rows = q_len * p.G;
    const int ns = rows <= p.rows_hi0 ? p.ns0 : (rows <= p.rows_hi1 ? p.ns1 : p.ns2);
    if (q_len <= 0 || ns <= 1) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y * kCombineHeads + warp;
    if (h >= p.Hq) return;
    for (int i = blockIdx.z; i < q_len; i += gridDim.z) combine_row<OT>(p, t0 + i, h, ns, lane);
}

cudaError_t launch_combine(const CombineParams &p, int out_dtype, cudaStream_t stream) {
    const int64_t threads = (int64_t)p.T * p.Hq * 32;
    if (threads == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((threads + 127) / 128);
    // per-request form when every split request has at most 64 packed rows
    // (so at most 64 tokens for a CTA to walk)
    const bool light = (p.ns2 <= 1) && (p.ns1 <= 1 || p.rows_hi1 <= 64);
    if (light) {
        // tokens of a split request: at most 64 packed rows, so at most 64 / G
        const int zt = std::max(1, std::min(p.max_q, std::max(1, std::max(p.rows_hi0, std::min(p.rows_hi1, 64)) / p.G)));
        // (at most 4 CTAs along the tokens, each walking every 4th token:
        // most requests of a mixed batch have one token, and the extra CTAs
        // of the others would only exit)
        const dim3 g((unsigned)p.B, (unsigned)((p.Hq + kCombineHeads - 1) / kCombineHeads), (unsigned)std::min(zt, 4));
        const dim3 blk(32 * kCombineHeads);
        if (out_dtype == DT_BF16) return launch_pdl(combine_light_kernel<__nv_bfloat16>, g, blk, 0, stream, p);
        if (out_dtype == DT_FP16) return launch_pdl(combine_light_kernel<__half>, g, blk, 0, stream, p);
        return cudaErrorInvalidValue;
    }
    if (out_dtype == DT_BF16) return launch_pdl(combine_kernel<__nv_bfloat16>, dim3(blocks), dim3(128), 0, stream, p);
    if (out_dtype == DT_FP16) return launch_pdl(combine_kernel<__half>, dim3(blocks), dim3(128), 0, stream, p);
    return cudaErrorInvalidValue;
}

// merge_attn_states: two states per (token, head), one warp each
template <class T>
__global__ void __launch_bounds__(128) merge_kernel(T *out, float *lse_out, const T *o1, const float *lse1,
                                                    const T *o2, const float *lse2, int T_, int Hq, int D) {
    pdl_wait();
    pdl_trigger();
    const int warp_global = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp_global >= T_ * Hq) return;
    const int64_t row = warp_global;
    const float a = lse1[row], b = lse2[row];
    const float mx = fmaxf(a, b);
    float w1 = 0.f, w2 = 0.f, l = -INFINITY;
    if (mx != -INFINITY) {
        const float e1 = expf(a - mx), e2 = expf(b - mx);
        const float s = e1 + e2;
        w1 = e1 / s;
        w2 = e2 / s;
        l = mx + logf(s);
    }
    for (int d = lane * 4; d < D; d += 128) {
        const float4 x = load4<T>(o1 + row * D + d);
        const float4 y = load4<T>(o2 + row * D + d);
        float4 z;
        z.x = w1 * x.x + w2 * y.x;
        z.y = w1 * x.y + w2 * y.y;
        z.z = w1 * x.z + w2 * y.z;
        z.w = w1 * x.w + w2 * y.w;
        store4<T>(out + row * D + d, z);   // same lane read these elements: out may alias o1/o2
    }
    if (lane == 0 && lse_out) lse_out[row] = l;
}

cudaError_t launch_merge(void *out, float *lse_out, const void *o1, const float *lse1, const void *o2,
                         const float *lse2, int T, int Hq, int D, int dtype, cudaStream_t stream) {
    const int64_t threads = (int64_t)T * Hq * 32;
    if (threads == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((threads + 127) / 128);
#define MRG(TYPE)                                                                                              \
    launch_pdl(merge_kernel<TYPE>, dim3(blocks), dim3(128), 0, stream, reinterpret_cast<TYPE *>(out), lse_out,  \
               reinterpret_cast<const TYPE *>(o1), lse1, reinterpret_cast<const TYPE *>(o2), lse2, T, Hq, D)
    if (dtype == DT_BF16) return MRG(__nv_bfloat16);
    if (dtype == DT_FP16) return MRG(__half);
    if (dtype == DT_FP32) return MRG(float);
#undef MRG
    return cudaErrorInvalidValue;
}

}  // namespace attn
