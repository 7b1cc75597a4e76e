// attn_noalloc.cu -- attn_paged_decode_noalloc: paged decode whose split-KV
// scratch lives in a fixed device array inside this library, for callers
// that must not allocate device memory themselves.
//
// Some callers cannot hand the library a workspace: plugin code running
// inside a host framework that owns every device allocation and forbids
// raw cudaMalloc, or latency-critical serving loops where cudaMalloc and
// cudaFree may synchronise the device and stall unrelated work.  This entry
// point needs nothing from them beyond the inputs and outputs: the
// per-segment partial results of split-KV go to g_noalloc_scratch below.
//
// The array is a file-scope __device__ variable, so every GPU that loads
// the library holds ATTN_NOALLOC_SCRATCH_BYTES of it until the process
// exits.  Host code must never pass g_noalloc_scratch itself to a kernel:
// on the host that name is a stand-in symbol, not a device address.  The
// device address is obtained once per device with cudaGetSymbolAddress
// (on the first call made while that device is current) and cached.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/attn.h"

static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

// device address of the array, per device; host threads racing on a
// device's first call store the same value, through an atomic
std::atomic<void *> g_scratch_addr[kMaxDevices];

attn_status scratch_for_current_device(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return ATTN_ERR_CUDA;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *addr = p;
    return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_paged_decode_noalloc(
    const void *q, const void *k_cache, const void *v_cache, void *out, float *lse_out,
    const int32_t *seq_lens, const int32_t *block_table, int64_t bt_row_stride,
    int B, int max_seq_len, int Hq, int Hkv, int D, int block_size, int num_blocks,
    attn_dtype q_dtype, attn_dtype kv_dtype, float softmax_scale, float k_descale, float v_descale,
    int num_splits, attn_stream_t stream) {
    // host validation comes first, as in every entry point: with an empty
    // batch the regular entry point runs the same argument checks and
    // returns before it looks up the device
    const attn_status valid =
        attn_paged_decode(q, k_cache, v_cache, out, lse_out, seq_lens, block_table, bt_row_stride, 0, max_seq_len,
                          Hq, Hkv, D, block_size, num_blocks, q_dtype, kv_dtype, softmax_scale, k_descale,
                          v_descale, num_splits, nullptr, 0, stream);
    if (valid != ATTN_OK) return valid;
    if (B <= 0) {
        // nothing to compute (a negative B is refused there)
        return attn_paged_decode(q, k_cache, v_cache, out, lse_out, seq_lens, block_table, bt_row_stride, B,
                                 max_seq_len, Hq, Hkv, D, block_size, num_blocks, q_dtype, kv_dtype,
                                 softmax_scale, k_descale, v_descale, num_splits, nullptr, 0, stream);
    }
    // the regular entry point refuses an explicit split count whose partial
    // results do not fit in ws_bytes (ATTN_ERR_WORKSPACE, before any launch)
    // and caps the automatic choice (num_splits = 0) to what fits
    void *scratch = nullptr;
    const attn_status st = scratch_for_current_device(&scratch);
    if (st != ATTN_OK) return st;
    // every partial slot the kernels read is written earlier in the same
    // call (empty segments write -inf), and a work counter, when used, is
    // zeroed by the call itself, so nothing needs clearing first
    return attn_paged_decode(q, k_cache, v_cache, out, lse_out, seq_lens, block_table, bt_row_stride, B,
                             max_seq_len, Hq, Hkv, D, block_size, num_blocks, q_dtype, kv_dtype, softmax_scale,
                             k_descale, v_descale, num_splits, scratch, (size_t)ATTN_NOALLOC_SCRATCH_BYTES,
                             stream);
}
