// attn_dec.cu -- decode-shape attention over an e4m3 paged KV cache on
// transposed mma.sync tiles: S^T = K Q^T and O^T = V^T P^T.
//
// A decode CTA's rows are (query token, head-in-group) pairs, G of them per
// token (four for Llama-3-8B's 32 query / 8 KV heads).  The smallest
// mma.sync tile is 16 wide on its row side (M) and 8 on its column side
// (N).  With the query rows on N and the keys (then the head dims) on M, a
// tile at G = 4 is half padding instead of three quarters.  Against the
// 16-row kernel that halves the tensor work per key and halves the
// accumulators: O^T is 8 rows x 128 dims, 32 fp32 values a lane.  The
// freed registers let five CTAs share an SM.  The loop is bound by
// instruction issue and latency, not by HBM (with every read an L2 hit it
// runs only a few percent faster), so more warps per scheduler and fewer
// instructions per key are what move it.
//
// Work split, gather and masking follow the 16-row kernel.
//  * One CTA is one request x one KV head x one block of 8 packed rows x one
//    KV segment ("vLLM 中 Attention Kernel 如何并行处理多个请求", sec. 3 and 12).
//  * K/V tiles of 64 keys are gathered through the block table (sec. 11)
//    into a two-stage ring.  Each of the 4 warps fetches and consumes only
//    its own 16 keys of every tile, so the main loop has no CTA-wide
//    barrier.  A warp's 16 keys are 16 consecutive slots of one cache block,
//    so one TMA box per tile brings them (for K and one for V), issued by
//    one lane from one block-table entry: the address work of a tile is done
//    once, not per row ("Making FlashAttention-4 faster for inference",
//    transposed address generation, taken to its end).
//  * Causal alignment is bottom-right (sec. 10); only tiles that need a
//    mask get one (sec. 4); the softmax is the online recurrence of sec. 7;
//    partial states are merged by log-sum-exp (sec. 12).
//
// Fragments (lane = 4g + t):
//  * Q K^T runs on e4m3 operands (m16n8k32) with K as stored, never
//    widened.  e4m3 queries enter as they are; 16-bit queries are split
//    once, in the prologue, into e4m3 terms whose sum is the query exactly
//    (hi + lo for bf16, hi + mid + lo for fp16, under a power-of-two row
//    scale), one MMA per term.  The head dimension is read in a permuted
//    order, the same for K and Q (the dot product does not depend on it):
//    k32-step kk of lane quad t takes bytes 32t + 8kk + 0..3 and
//    32t + 8kk + 4..7, so a lane's K fragments of every k-step are 32
//    contiguous bytes of key rows g and g + 8, and its Q^T fragments the
//    same bytes of query row g.
//  * The S^T accumulator holds keys g and g + 8 x rows 2t and 2t + 1.  A
//    row's softmax reduces over the eight lanes of one t.  P^T's B fragment
//    wants the rows on g and the keys on t: one movmatrix.trans per 8 x 8
//    block turns one into the other.
//  * P V: m-tile i of O^T holds dims 16g + 2i (its row g) and 16g + 2i + 1
//    (its row g + 8).  A lane's V^T fragments of all eight m-tiles are then
//    bytes 16g .. 16g + 15 of key rows 2t, 2t + 1, 2t + 8 and 2t + 9,
//    paired by key with prmt and widened in registers.  A lane ends with
//    dims 16g .. 16g + 15 of rows 2t and 2t + 1.
#include <type_traits>

#include "common.cuh"
#include "sm100.cuh"
#include "tma_host.h"

namespace attn {

namespace {

template <int QT_, int MINB_, int STAGES_>
struct DecCfg {
    static constexpr int QT = QT_;
    // CTAs per SM the registers are capped for (fp16 queries hold three
    // e4m3 terms of Q: one CTA fewer, no spills)
    static constexpr int MINB = (QT == DT_FP16) ? MINB_ - 1 : MINB_;
    static constexpr int STAGES = STAGES_;          // K/V tiles in each warp's TMA ring
    static constexpr int D = 128;                   // head size
    static constexpr int ROWS = 8;                  // packed rows per CTA (the N side)
    static constexpr int BN = 64;                   // keys per K/V tile
    static constexpr int NWARP = 4;
    static constexpr int NW = BN / NWARP;           // keys per warp and tile (the M side of S^T)
    static constexpr int KV_ROW = D;                // bytes of one cached e4m3 row (one KV head)
    static constexpr int CH = KV_ROW / 16;          // 16-byte chunks per row
    static constexpr int TILE_RAW = BN * KV_ROW;    // one K (or V) tile as stored
    static constexpr int STAGE_BYTES = 2 * TILE_RAW;
    static constexpr bool Q8 = (QT == DT_E4M3);
    // e4m3 terms Q is split into for Q K^T on e4m3 operands: bf16 (8
    // significant bits) is exact in hi + lo, fp16 (11) in hi + mid + lo
    static constexpr int NQ = (QT == DT_BF16) ? 2 : (QT == DT_FP16) ? 3 : 1;
    using OutT = std::conditional_t<QT == DT_FP16, __half, __nv_bfloat16>;   // e4m3 q: bf16 out
    static constexpr int OSTRIDE = D + 4;           // fp32 epilogue row stride (bank spread)
    static constexpr int EPI_BYTES = NWARP * ROWS * OSTRIDE * 4 + 2 * NWARP * ROWS * 4;
    static constexpr int MAIN_BYTES = STAGES * STAGE_BYTES;
    static constexpr int BARS_OFF = MAIN_BYTES > EPI_BYTES ? MAIN_BYTES : EPI_BYTES;   // mbarriers after the ring
    static constexpr int NBARS = STAGES * NWARP;    // one per (stage, warp)
    // + 1 KB: the ring is aligned up to 1024 bytes (the 128-byte swizzle's period)
    static constexpr int SMEM = 1024 + BARS_OFF + NBARS * 8 + 16;
    static_assert(NW == 16 && CH == 8, "one 16-slot TMA box of 128-byte rows per warp and tile");
};

// transpose of an 8 x 8 matrix of 16-bit values held one row pair per lane
// (lane 4g + t: row g, columns 2t and 2t + 1)
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// byte offset of 16-byte chunk ch of row `row` in a staged tile, chunks
// XOR-swizzled by row & 7: the eight rows (or chunks) that eight lanes of
// one load phase read fall in eight different bank groups
__device__ __forceinline__ uint32_t stage_off(int row, int ch) {
    return (uint32_t)(row * 128 + ((ch ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint4 lds16(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

constexpr float kRescaleLog2Dec = 8.0f;   // reference-maximum threshold (log2 units)

}  // namespace

template <class C>
__global__ void __launch_bounds__(128, C::MINB)
    fwd_dec_kernel(const FwdParams p, const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
    constexpr int D = C::D, ROWS = C::ROWS, BN = C::BN, NW = C::NW, STAGES = C::STAGES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);

    pdl_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t4 = lane & 3;
    const int r = blockIdx.z, kvh = blockIdx.y;
    const int s_idx = blockIdx.x % p.nsplit;
    const int rb = p.n_row_blocks - 1 - (int)(blockIdx.x / p.nsplit);

    int q_start, q_len;
    if (p.cu_seqlens_q) {
        q_start = p.cu_seqlens_q[r];
        q_len = p.cu_seqlens_q[r + 1] - q_start;
    } else {
        q_start = r;
        q_len = 1;
    }
    const int kv_len = p.seqused_k[r];
    const int G = p.G;
    const int rows = q_len * G;
    if (rows < p.rows_lo || rows > p.rows_hi) return;
    const int row0 = rb * ROWS;
    if (row0 >= rows) return;
    const int row_end = min(row0 + ROWS, rows);
    const int ctx = kv_len - q_len;                  // cached context before the queries
    const int i_min = row0 / G, i_max = (row_end - 1) / G;
    // keys any row of the block may see, cut into whole-tile segments
    int kv_end = kv_len;
    if (p.causal) kv_end = min(kv_len, ctx + i_max + 1);
    if (p.window_right >= 0) kv_end = (int)min((long long)kv_end, (long long)ctx + i_max + p.window_right + 1);
    const int kv_beg = (p.window_left >= 0) ? (max(0, ctx + i_min - p.window_left) & ~(BN - 1)) : 0;
    const long long kv_lo_ll = (long long)kv_beg + (long long)s_idx * p.split_chunk;
    const int kv_lo = (int)min(kv_lo_ll, (long long)INT_MAX);
    const int kv_hi = (int)min((long long)kv_end, kv_lo_ll + p.split_chunk);

    if (kv_lo >= kv_hi) {
        // no key in this segment for any row of the block: empty state (a
        // sink alone, in segment 0)
        for (int pr = row0 + tid; pr < row_end; pr += blockDim.x) {
            const int64_t tok = q_start + pr / G;
            const int h = kvh * G + pr % G;
            const float zl = (p.sinks && s_idx == 0) ? p.sinks[h] : -INFINITY;
            if (p.partials) {
                const int64_t slot = (tok * p.Hq + h) * p.part_stride + s_idx;
                p.part_lse[slot] = zl;
                if (zl != -INFINITY)
                    for (int d = 0; d < D; ++d) p.part_o[slot * D + d] = 0.f;
            } else {
                if (p.lse) p.lse[tok * p.Hq + h] = zl;
                using OT = typename C::OutT;
                OT *o = reinterpret_cast<OT *>(p.out) + tok * p.out_stride + (int64_t)h * D;
                for (int d = 0; d < D; ++d) o[d] = OT(0.f);
            }
        }
        return;
    }

    // ---- Q^T fragments of query row g of the block, straight from global
    // memory (rows past the block's end are zero).  Word j of term k holds
    // e4m3 bytes of dims 32t + 4j .. 32t + 4j + 3.  16-bit queries are
    // split into NQ e4m3 terms under a power-of-two row scale 2^e (the row's
    // largest magnitude lands in [128, 256)): hi = e4m3(q 2^e), the next
    // term e4m3 of what is left, and so on -- each term carries 4
    // significant bits, so the sum is q 2^e exactly down to e4m3's
    // subnormal step (2^-9 in the scaled units, 2^-16 of the row maximum).
    uint32_t qf[C::NQ][8];
    float row_scale = 1.f;   // 2^-e of query row g (1 for e4m3 queries)
    {
        const int pr = row0 + g;
        const bool ok = pr < row_end;
        const int64_t tok = q_start + (ok ? pr / G : 0);
        const int h = kvh * G + (ok ? pr % G : 0);
        const int4 z = make_int4(0, 0, 0, 0);
        if constexpr (C::Q8) {
            const uint8_t *src = reinterpret_cast<const uint8_t *>(p.q) + tok * p.q_stride + (int64_t)h * D + 32 * t4;
            const int4 a = ok ? ldg_nc16(src) : z, b = ok ? ldg_nc16(src + 16) : z;
            qf[0][0] = a.x; qf[0][1] = a.y; qf[0][2] = a.z; qf[0][3] = a.w;
            qf[0][4] = b.x; qf[0][5] = b.y; qf[0][6] = b.z; qf[0][7] = b.w;
        } else {
            const uint8_t *src =
                reinterpret_cast<const uint8_t *>(p.q) + (tok * p.q_stride + (int64_t)h * D + 32 * t4) * 2;
            float qv[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int4 v = ok ? ldg_nc16(src + 16 * c) : z;
                const uint32_t w[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float2 f;
                    if constexpr (C::QT == DT_BF16) f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[k]));
                    else f = __half22float2(*reinterpret_cast<const __half2 *>(&w[k]));
                    qv[8 * c + 2 * k] = f.x;
                    qv[8 * c + 2 * k + 1] = f.y;
                }
            }
            float mx = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(qv[i]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const int E = (int)((__float_as_uint(mx) >> 23) & 0xff) - 127;
            const int e = min(max(7 - E, -126), 126);
            const float sc = __uint_as_float((uint32_t)(e + 127) << 23);
            row_scale = __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
            for (int i = 0; i < 32; ++i) qv[i] *= sc;
#pragma unroll
            for (int k = 0; k < C::NQ; ++k) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint32_t word = 0;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        float2 x = make_float2(qv[4 * j + 2 * hh], qv[4 * j + 2 * hh + 1]);
                        const __nv_fp8x2_storage_t b8 = __nv_cvt_float2_to_fp8x2(x, __NV_SATFINITE, __NV_E4M3);
                        word |= (uint32_t)b8 << (16 * hh);
                        if (k + 1 < C::NQ) {
                            // what this term leaves for the next (exact in fp32)
                            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(b8, __NV_E4M3);
                            const float2 back = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
                            qv[4 * j + 2 * hh] = x.x - back.x;
                            qv[4 * j + 2 * hh + 1] = x.y - back.y;
                        }
                    }
                    qf[k][j] = word;
                }
            }
        }
    }
    // the row scales of this lane's accumulator rows 2t and 2t + 1
    const float rs0 = __shfl_sync(0xffffffffu, row_scale, 8 * t4);
    const float rs1 = __shfl_sync(0xffffffffu, row_scale, 8 * t4 + 4);
    const float sl2_0 = p.scale_log2 * rs0, sl2_1 = p.scale_log2 * rs1;
    const float vds = p.v_descale * kE4m3Lo8Scale;   // V widened to fp16 holds value * 2^-8
    const bool capped = p.cap_in > 0.f;
    const float cap_in0 = p.cap_in * rs0, cap_in1 = p.cap_in * rs1;

    // query token (local index) of the two rows this lane owns (2t, 2t + 1)
    // and their visible keys [lo, lim]
    const int ir0 = (row0 + 2 * t4) / G, ir1 = (row0 + 2 * t4 + 1) / G;
    auto last_key = [&](int ir) -> int {
        long long l = p.causal ? (long long)ctx + ir : (long long)INT_MAX;
        if (p.window_right >= 0) l = min(l, (long long)ctx + ir + p.window_right);
        return (int)l;
    };
    const int lim0 = last_key(ir0), lim1 = last_key(ir1);
    const int lo0 = (p.window_left >= 0) ? ctx + ir0 - p.window_left : INT_MIN;
    const int lo1 = (p.window_left >= 0) ? ctx + ir1 - p.window_left : INT_MIN;

    // ---- K/V tile gather through the block table: warp w fetches key rows
    // [16w, 16w + 16) of every tile, the rows it alone reads.  Those 16
    // tokens start at a multiple of 16 and a cache block holds a multiple of
    // 16 tokens, so they are 16 consecutive slots of one block: one TMA box
    // (16 slots x one KV head x 128 bytes) for K and one for V, issued by
    // lane 0 on the warp's own mbarrier of that stage.  The 128-byte
    // swizzle writes chunk c of row r at slot c ^ (r & 7) (the layout the
    // fragment loads expect).  A block id outside the pool is flagged and
    // replaced by a slot past the end of the map, which TMA fills with
    // zeros.  Tiles are fetched in order; the block position of the warp's
    // next tile is carried from call to call (one tile is BN tokens: BN / bs
    // blocks and BN % bs slots on).
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BARS_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + C::NBARS);
    const uint32_t bar_w = smem_u32(bars) + warp * 8;   // stage s: bar_w + 8 NWARP s
    const uint32_t ring = smem_u32(smem) + warp * NW * C::KV_ROW;
    if (tid == 0) *abort_flag = 0;
    if (lane == 0) {
#pragma unroll
        for (int s2 = 0; s2 < STAGES; ++s2) sm100::mbar_init(bar_w + 8 * C::NWARP * s2, 1);
        sm100::fence_mbar_init();
    }
    __syncthreads();   // barriers and the abort flag initialised
    const int64_t bt_base = (int64_t)r * p.bt_stride;
    const int n_slots = p.num_blocks * p.bs;            // the maps' slot extent (checked on the host)
    int ld_t0 = kv_lo + warp * NW;                      // the warp's first token of the next tile
    int ld_bi = ld_t0 / p.bs;                           // its block-table index
    int ld_bw = ld_t0 - ld_bi * p.bs;                   // and slot within that block
    const int adv_q = BN / p.bs, adv_r = BN - adv_q * p.bs;
    auto load_next = [&](int stage) {
        if (lane == 0) {
            const uint32_t bar = bar_w + 8 * C::NWARP * stage;
            if (ld_t0 < kv_hi) {
                const int blk = p.block_table[bt_base + ld_bi];
                int slot = n_slots;
                if ((unsigned)blk < (unsigned)p.num_blocks) slot = blk * p.bs + ld_bw;
                else raise_error(p.err, ERR_BLOCK_ID);
                const uint32_t dst = ring + stage * C::STAGE_BYTES;
                sm100::mbar_expect_tx(bar, 2 * NW * C::KV_ROW);
                sm100::tma_load_3d(dst, &kmap, 0, kvh, slot, bar);
                sm100::tma_load_3d(dst + C::TILE_RAW, &vmap, 0, kvh, slot, bar);
            } else {
                sm100::mbar_arrive(bar);   // nothing of this warp's rows left: complete the phase
            }
        }
        ld_t0 += BN;
        ld_bi += adv_q;
        ld_bw += adv_r;
        if (ld_bw >= p.bs) {
            ld_bw -= p.bs;
            ++ld_bi;
        }
    };

    // tiles that need a mask: those past the segment end, the causal
    // diagonal or the right window edge (n0 > right_lim), and those before
    // the left window edge (n0 < left_lim)
    long long right_lim = (long long)kv_hi - BN;
    if (p.causal) right_lim = min(right_lim, (long long)ctx + i_min - BN + 1);
    if (p.window_right >= 0) right_lim = min(right_lim, (long long)ctx + i_min + p.window_right - BN + 1);
    const long long left_lim = (p.window_left >= 0) ? (long long)ctx + i_max - p.window_left : LLONG_MIN;

    const int n_tiles = (kv_hi - kv_lo + BN - 1) / BN;
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s)
        if (s < n_tiles) load_next(s);

    float o[D / 16][4];   // O^T m-tile i: dims 16g + 2i (0, 1) and 16g + 2i + 1 (2, 3) x rows 2t, 2t + 1
#pragma unroll
    for (int i = 0; i < D / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.f, 0.f};   // this lane's share of the row sums (keys g, g + 8)
    const int kr = warp * NW;  // the warp's first key row in a tile

    int waited = 0;   // tiles whose loads this warp has seen land
    for (int t = 0; t < n_tiles; ++t) {
        if (!sm100::mbar_wait(bar_w + 8 * C::NWARP * (t % STAGES), (t / STAGES) & 1, abort_flag)) break;
        waited = t + 1;
        __syncwarp();          // every lane has read tile t - 1: its stage may be refilled
        {
            const int tn = t + STAGES - 1;
            if (tn < n_tiles) load_next(tn % STAGES);
        }
        const uint8_t *sK = smem + (t % STAGES) * C::STAGE_BYTES;
        const uint8_t *sV = sK + C::TILE_RAW;
        const int n0 = kv_lo + t * BN;

        // S^T = K Q^T for the warp's 16 keys: s[0], s[1] key g, rows 2t,
        // 2t + 1; s[2], s[3] key g + 8
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const uint4 x0 = lds16(sK + stage_off(kr + g, 2 * t4)), x1 = lds16(sK + stage_off(kr + g, 2 * t4 + 1));
            const uint4 y0 = lds16(sK + stage_off(kr + g + 8, 2 * t4));
            const uint4 y1 = lds16(sK + stage_off(kr + g + 8, 2 * t4 + 1));
            const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            const uint32_t yw[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t a[4] = {xw[2 * kk], yw[2 * kk], xw[2 * kk + 1], yw[2 * kk + 1]};
#pragma unroll
                for (int k = 0; k < C::NQ; ++k) mma16832_e4m3(s, a, qf[k][2 * kk], qf[k][2 * kk + 1]);
            }
        }

        // scale to log2 units; mask only tiles crossing the segment end, the
        // causal diagonal or a window edge
        const bool need_mask = (n0 > right_lim) || (n0 < left_lim);
        if (capped) {
#pragma unroll
            for (int e = 0; e < 4; ++e) s[e] = p.cap_out * tanh_ex2(s[e] * ((e & 1) ? cap_in1 : cap_in0));
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) s[e] *= (e & 1) ? sl2_1 : sl2_0;
        }
        if (need_mask) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = n0 + kr + g + 8 * (e >> 1);
                const int lim = (e & 1) ? lim1 : lim0;
                const int lo = (e & 1) ? lo1 : lo0;
                if (key >= kv_hi || key > lim || key < lo) s[e] = -INFINITY;
            }
        }

        // online softmax: a row's 16 keys sit on the eight lanes of one t.
        // m is a reference maximum that moves only when a row's maximum
        // grows by more than 2^8 (log2 units); P is formed against it and O
        // is rescaled only on the rare tiles that move it
        float mx[2] = {fmaxf(s[0], s[2]), fmaxf(s[1], s[3])};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 4));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 8));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 16));
        }
        float base[2], alpha[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const bool bump = mx[h] > m[h] + kRescaleLog2Dec;
            alpha[h] = (bump && m[h] != -INFINITY) ? ex2(m[h] - mx[h]) : 1.f;
            if (bump) m[h] = mx[h];
            base[h] = (m[h] == -INFINITY) ? 0.f : m[h];   // fully masked row so far
        }
        s[0] = ex2(s[0] - base[0]);
        s[1] = ex2(s[1] - base[1]);
        s[2] = ex2(s[2] - base[0]);
        s[3] = ex2(s[3] - base[1]);
        l[0] = l[0] * alpha[0] + (s[0] + s[2]);
        l[1] = l[1] * alpha[1] + (s[1] + s[3]);
        if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
                o[i][0] *= alpha[0];
                o[i][1] *= alpha[1];
                o[i][2] *= alpha[0];
                o[i][3] *= alpha[1];
            }
        }

        // P^T as the B operand: keys 2t, 2t + 1 (b0) and 2t + 8, 2t + 9 (b1)
        // of row g
        const uint32_t b0 = movmatrix_trans(pack2<false>(s[0], s[1]));
        const uint32_t b1 = movmatrix_trans(pack2<false>(s[2], s[3]));

        // O^T += V^T P^T: V^T fragments of key rows 2t, 2t + 1, 2t + 8,
        // 2t + 9, dims 16g .. 16g + 15 (byte d of a chunk is dim 16g + d)
        {
            const uint4 v0 = lds16(sV + stage_off(kr + 2 * t4, g)), v1 = lds16(sV + stage_off(kr + 2 * t4 + 1, g));
            const uint4 v2 = lds16(sV + stage_off(kr + 2 * t4 + 8, g));
            const uint4 v3 = lds16(sV + stage_off(kr + 2 * t4 + 9, g));
            const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
            const uint32_t w2[4] = {v2.x, v2.y, v2.z, v2.w}, w3[4] = {v3.x, v3.y, v3.z, v3.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                // m-tiles 2w and 2w + 1: dims 16g + 4w + {0, 1} and + {2, 3}
                const uint32_t a0[4] = {e4m3_pair_to_h2_lo8<0>(w0[w], w1[w]), e4m3_pair_to_h2_lo8<1>(w0[w], w1[w]),
                                        e4m3_pair_to_h2_lo8<0>(w2[w], w3[w]), e4m3_pair_to_h2_lo8<1>(w2[w], w3[w])};
                mma16816<false>(o[2 * w], a0, b0, b1);
                const uint32_t a1[4] = {e4m3_pair_to_h2_lo8<2>(w0[w], w1[w]), e4m3_pair_to_h2_lo8<3>(w0[w], w1[w]),
                                        e4m3_pair_to_h2_lo8<2>(w2[w], w3[w]), e4m3_pair_to_h2_lo8<3>(w2[w], w3[w])};
                mma16816<false>(o[2 * w + 1], a1, b0, b1);
            }
        }
    }
    pdl_trigger();     // the next kernel may be scheduled; it waits for this grid's completion
    if (waited < n_tiles) {
        // a wait gave up (a stalled copy, which would be a bug): flag it, give
        // the loads still in flight a bounded chance to land, and skip the output
        if (lane == 0) raise_error(p.err, ERR_TIMEOUT);
        const int issued = min(n_tiles, waited + STAGES - 1);
        int own = 0;   // (a local flag: these waits must not end on the shared one)
        for (int t = waited; t < issued; ++t)
            sm100::mbar_wait(bar_w + 8 * C::NWARP * (t % STAGES), (t / STAGES) & 1, &own);
    }
    __syncthreads();   // every staged tile consumed; the ring becomes the epilogue's buffer
    if (*abort_flag) return;

    // ---- epilogue: merge the four warp states of each row, normalise, store
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 4);
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 8);
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 16);
    }
    float *sO = reinterpret_cast<float *>(smem);
    float *sM = sO + C::NWARP * ROWS * C::OSTRIDE;
    float *sL = sM + C::NWARP * ROWS;
    {
        float *r0 = sO + (warp * ROWS + 2 * t4) * C::OSTRIDE + 16 * g;
        float *r1 = r0 + C::OSTRIDE;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            *reinterpret_cast<float4 *>(r0 + 4 * j) = make_float4(o[2 * j][0], o[2 * j][2], o[2 * j + 1][0], o[2 * j + 1][2]);
            *reinterpret_cast<float4 *>(r1 + 4 * j) = make_float4(o[2 * j][1], o[2 * j][3], o[2 * j + 1][1], o[2 * j + 1][3]);
        }
        if (g == 0) {
            sM[warp * ROWS + 2 * t4] = m[0];
            sM[warp * ROWS + 2 * t4 + 1] = m[1];
            sL[warp * ROWS + 2 * t4] = l[0];
            sL[warp * ROWS + 2 * t4 + 1] = l[1];
        }
    }
    __syncthreads();

    constexpr int DV = D / 4;
    for (int idx = tid; idx < ROWS * DV; idx += blockDim.x) {
        const int lr = idx / DV, c4 = idx % DV;
        const int pr = row0 + lr;
        if (pr >= row_end) continue;
        float mf = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::NWARP; ++w) mf = fmaxf(mf, sM[w * ROWS + lr]);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float lf = 0.f;
        if (mf != -INFINITY) {
#pragma unroll
            for (int w = 0; w < C::NWARP; ++w) {
                const float sc = ex2(sM[w * ROWS + lr] - mf);
                lf += sL[w * ROWS + lr] * sc;
                const float4 v = *reinterpret_cast<const float4 *>(&sO[(w * ROWS + lr) * C::OSTRIDE + c4 * 4]);
                acc.x += sc * v.x;
                acc.y += sc * v.y;
                acc.z += sc * v.z;
                acc.w += sc * v.w;
            }
        }
        const int64_t tok = q_start + pr / G;
        const int h = kvh * G + pr % G;
        float sink_scale = 1.f;
        if (p.sinks && s_idx == 0 && p.sinks[h] > -INFINITY) {
            // the sink joins segment 0's state: a virtual key with logit z, value 0
            const float z2 = p.sinks[h] * 1.4426950408889634f;
            const float mn = fmaxf(mf, z2);
            sink_scale = (mf == -INFINITY) ? 0.f : ex2(mf - mn);
            lf = lf * sink_scale + ex2(z2 - mn);
            mf = mn;
        }
        const float inv = lf > 0.f ? vds * sink_scale / lf : 0.f;
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
        const float lse_v = lf > 0.f ? (mf + __log2f(lf)) * 0.6931471805599453f : -INFINITY;
        if (!p.partials) {
            using OT = typename C::OutT;
            OT *dst = reinterpret_cast<OT *>(p.out) + tok * p.out_stride + (int64_t)h * D + c4 * 4;
            uint2 pk;
            pk.x = pack2<C::QT != DT_FP16>(acc.x, acc.y);
            pk.y = pack2<C::QT != DT_FP16>(acc.z, acc.w);
            *reinterpret_cast<uint2 *>(dst) = pk;
            if (c4 == 0 && p.lse) p.lse[tok * p.Hq + h] = lse_v;
        } else {
            const int64_t slot = (tok * p.Hq + h) * p.part_stride + s_idx;
            *reinterpret_cast<float4 *>(p.part_o + slot * D + c4 * 4) = acc;
            if (c4 == 0) p.part_lse[slot] = lse_v;
        }
    }
}

template <class C>
static cudaError_t launch_dec_cfg(const FwdParams &p, cudaStream_t stream) {
    // the caches viewed as [num_blocks * bs slots][Hkv][128 bytes]: a box is
    // 16 slots of one KV head, 128-byte swizzle
    const uint64_t n_slots = (uint64_t)p.num_blocks * p.bs;
    if (n_slots == 0 || n_slots > (uint64_t)INT32_MAX - 1) return cudaErrorInvalidValue;
    CUtensorMap kmap, vmap;
    const uint64_t row = (uint64_t)p.Hkv * C::KV_ROW;
    if (!encode_3d_u8(&kmap, p.k_cache, C::KV_ROW, (uint64_t)p.Hkv, n_slots, C::KV_ROW, row, C::KV_ROW, 1, C::NW, true) ||
        !encode_3d_u8(&vmap, p.v_cache, C::KV_ROW, (uint64_t)p.Hkv, n_slots, C::KV_ROW, row, C::KV_ROW, 1, C::NW, true))
        return cudaErrorInvalidValue;
    auto kern = fwd_dec_kernel<C>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.n_row_blocks * p.nsplit), (unsigned)p.Hkv, (unsigned)p.B);
    return launch_pdl(kern, grid, dim3(128), C::SMEM, stream, p, kmap, vmap);
}

// five CTAs an SM (96 registers a thread, 34 KB of shared memory each) and
// a two-tile ring per warp measured fastest on the fp8 decode and mixed
// batches (four CTAs with three tiles, six with two: slower or equal)
constexpr int kDecMinBlocks = 5;
constexpr int kDecStages = 2;

bool dec_supported(int D, int q_dtype, int kv_dtype) {
    return D == 128 && kv_dtype == DT_E4M3 && (q_dtype == DT_BF16 || q_dtype == DT_FP16 || q_dtype == DT_E4M3);
}

bool dec_pool_fits(int num_blocks, int bs) {
    const long long n = (long long)num_blocks * bs;
    return n > 0 && n < (long long)INT32_MAX;
}

int dec_rows_per_cta() { return 8; }

cudaError_t launch_fwd_dec(const FwdParams &p, int q_dtype, cudaStream_t stream) {
    switch (q_dtype) {
    case DT_BF16: return launch_dec_cfg<DecCfg<DT_BF16, kDecMinBlocks, kDecStages>>(p, stream);
    case DT_FP16: return launch_dec_cfg<DecCfg<DT_FP16, kDecMinBlocks, kDecStages>>(p, stream);
    case DT_E4M3: return launch_dec_cfg<DecCfg<DT_E4M3, kDecMinBlocks, kDecStages>>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
