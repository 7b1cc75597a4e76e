// attn_validate.cu -- host-side checks of the integer tables of a call
// (cu_seqlens_q, seqused_k, block_table, slot_mapping) against the contract
// of include/attn.h.  The entry points run them on host copies of the
// tables when the environment sets ATTN_DEBUG_VALIDATE=1; they are exported
// on their own so that a caller (or a test without a GPU) can check tables
// it already holds on the host.
//
// The checks cover what the kernels cannot see: a max_seqlen_q or
// max_seqlen_k below the truth (the launch is sized from them and split
// segments would stop short of kv_len), cu_seqlens_q that is not a prefix
// sum ending at total_q ("FlashAttention deep dive", flash_attn_varlen_func
// argument table), a request with fewer cached keys than new queries under
// the causal mask (its new tokens' keys are part of kv_len, "vLLM 中
// Attention Kernel 如何并行处理多个请求" sec. 10), and block ids or slots
// outside the cache (sec. 11), which the kernels also catch but only as a
// device error word after the fact.
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "../../include/attn.h"

extern "C" {

int attn_debug_validate_enabled(void) {
    const char *v = getenv("ATTN_DEBUG_VALIDATE");
    return v && v[0] && strcmp(v, "0") != 0;
}

attn_status attn_validate_tables(const int32_t *cu_seqlens_q, const int32_t *seqused_k, const int32_t *block_table,
                                 int64_t bt_row_stride, int B, int total_q, int max_seqlen_q, int max_seqlen_k,
                                 int block_size, int num_blocks, int causal) {
    if (B < 0 || total_q < 0 || block_size <= 0 || num_blocks < 0 || bt_row_stride < 0) return ATTN_ERR_SHAPE;
    if (B == 0) return ATTN_OK;
    if (!seqused_k || !block_table) return ATTN_ERR_NULL;
    // without cu_seqlens_q every request owns one query row (decode)
    if (cu_seqlens_q) {
        if (cu_seqlens_q[0] != 0 || cu_seqlens_q[B] != total_q) return ATTN_ERR_TABLE;
    } else if (total_q != B) {
        return ATTN_ERR_TABLE;
    }
    for (int r = 0; r < B; ++r) {
        const long long q_len = cu_seqlens_q ? (long long)cu_seqlens_q[r + 1] - cu_seqlens_q[r] : 1;
        const long long kv_len = seqused_k[r];
        if (q_len < 0 || q_len > max_seqlen_q) return ATTN_ERR_TABLE;
        if (kv_len < 0 || kv_len > max_seqlen_k) return ATTN_ERR_TABLE;
        if (causal && kv_len < q_len) return ATTN_ERR_TABLE;
        const long long nblk = (kv_len + block_size - 1) / block_size;
        // rows of a [B, W] table: a row never reaches into the next one
        if (B > 1 && nblk > bt_row_stride) return ATTN_ERR_TABLE;
        const int32_t *row = block_table + (int64_t)r * bt_row_stride;
        for (long long j = 0; j < nblk; ++j)
            if (row[j] < 0 || row[j] >= num_blocks) return ATTN_ERR_TABLE;
    }
    return ATTN_OK;
}

attn_status attn_validate_slots(const int64_t *slot_mapping, int T, int block_size, int num_blocks) {
    if (T < 0 || block_size <= 0 || num_blocks < 0) return ATTN_ERR_SHAPE;
    if (T == 0) return ATTN_OK;
    if (!slot_mapping) return ATTN_ERR_NULL;
    const long long n_slots = (long long)num_blocks * block_size;
    for (int t = 0; t < T; ++t)
        if (slot_mapping[t] < -1 || slot_mapping[t] >= n_slots) return ATTN_ERR_TABLE;   // -1: padding token
    return ATTN_OK;
}

}  // extern "C"
