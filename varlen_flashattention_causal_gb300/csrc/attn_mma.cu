// attn_mma.cu -- FlashAttention-style forward over a paged KV cache with
// warp-level mma.sync (m16n8k16) tensor-core tiles.
//
// This kernel serves the rows-light side of the hot path: decode (one query
// token per request), multi-token verification and short queries.  Its
// tiles are 16 query rows per warp, the smallest tensor-core tile, so the
// G query heads that share a KV head (GQA) are packed into the rows and
// every K/V tile fetched from HBM serves all of them.  The kernel is
// HBM-bound: one K/V row per (token, KV head) is read exactly once.
//
// Work of one CTA ("vLLM 中 Attention Kernel 如何并行处理多个请求", sec. 3 and 12):
// one request x one KV head x one block of packed query rows x one KV
// segment.  Rows are (query token, head-in-group) pairs.  The K/V tiles of
// BN keys are gathered through the block table (sec. 11) with 16-byte
// cp.async copies into a multi-stage shared-memory ring: each warp computes
// the addresses of its rows once (one lane per row) and shares them by
// shuffle, instead of every thread re-deriving 64-bit row pointers
// ("Making FlashAttention-4 faster for inference", transposed address
// generation).  Scores are masked in registers from local positions with
// the bottom-right alignment of sec. 10 (q_abs = ctx + i), only on tiles
// that need it (sec. 4), and the softmax is the online recurrence of sec. 7.
// With WN > 1 the warps split each K/V tile's keys (flash-decoding inside
// the CTA) and merge their states through shared memory at the end; with
// WN = 4 (decode shapes) each warp also fetches exactly its own keys, so the
// warps stream their slices independently, synchronising only at the start
// (Q) and at the end (the merge); with
// partials (nsplit > 1) each CTA writes a normalised partial state that the combine
// kernel merges by log-sum-exp (sec. 12).
#include <type_traits>

#include "common.cuh"

namespace attn {

template <int D_, int WM_, int WN_, int BN_, int STAGES_, int QT_, int KVT_>
struct MmaCfg {
    static constexpr int D = D_, WM = WM_, WN = WN_, BN = BN_, STAGES = STAGES_, QT = QT_, KVT = KVT_;
    static constexpr int ROWS = 16 * WM;
    static constexpr bool MMA_BF16 = (KVT == DT_BF16);   // fp16 and e4m3 caches run f16 MMAs (P V)
    using OutT = std::conditional_t<QT == DT_FP16, __half, __nv_bfloat16>;   // e4m3 q: bf16 out
    static constexpr int KV_BYTES = Elem<KVT>::bytes;
    static constexpr int KV_ROW = D * KV_BYTES;          // bytes of one cached row (one KV head)
    static constexpr int TILE_RAW = BN * KV_ROW;         // one K (or V) tile as stored
    static constexpr int ROW16 = D * 2;                  // one row in 16-bit MMA form
    static constexpr int TILE16 = BN * ROW16;
    static constexpr int Q_BYTES = ROWS * ROW16;
    static constexpr int STAGE_BYTES = 2 * TILE_RAW;
    static constexpr int NW = BN / WN;                   // keys per warp per tile
    static constexpr int NT = NW / 8;                    // n8 tiles of S per warp
    static constexpr int KT = D / 16;                    // k16 steps of Q K^T
    static constexpr int RPW = BN / 4;                   // K/V rows each warp fetches
    static constexpr int CH = KV_ROW / 16;               // 16-byte chunks per cached row
    // One row block of 16 rows: warp w fetches K/V rows [16w, 16w + 16) of
    // every tile and is also the only warp that reads them (its key slice),
    // so the main loop needs no CTA-wide barrier.
    static constexpr bool WARP_LOCAL = (WM == 1 && RPW == NW);
    // Two row blocks of 16 rows (2 x 2 warps): warp w = wm + 2 wn fetches
    // rows [16w, 16w + 16), so the two warps of key slice wn fetch exactly
    // the 32 rows that only they read, and a barrier of that pair (64
    // threads) stands in for the CTA-wide one.
    static constexpr bool PAIR_LOCAL = (WM == 2 && WN == 2 && NW == 2 * RPW);
    // e4m3 K fragments straight from the staged tile (decode shape, D 128):
    // the head dimension is read in a permuted order -- k-step kk of lane
    // quad t covers dims 32t + 4kk .. 32t + 4kk + 3, the same order for the
    // Q fragments, so Q K^T is unchanged -- which makes a lane's B
    // fragments of all eight k-steps 32 contiguous bytes of its key row,
    // widened in registers.  V takes the same route under VDIRECT below.
    static constexpr bool KDIRECT = (KVT == DT_E4M3) && WARP_LOCAL && D == 128 && QT != DT_E4M3;
    // e4m3 queries: Q K^T on e4m3 operands (m16n8k32), the K fragments
    // read straight from the staged bytes with no widening, in the same
    // permuted head order (k-step kk of lane quad t covers dims
    // 32t + 8kk .. 32t + 8kk + 7); output in bf16
    static constexpr bool Q8 = (QT == DT_E4M3);
    static constexpr bool STAGE_SWZ = KDIRECT || Q8;   // staged e4m3 rows chunk-swizzled
    // e4m3 V fragments straight from the staged bytes too (decode shape, D
    // 128, the warp's own 16 keys): the head dimension of P V's output is
    // read in a permuted order -- n8 tile j of lane (g, t) covers dims 16n + j
    // (n = g for V, n = 2t, 2t + 1 for O) -- so a lane's B fragments of all
    // sixteen n8 tiles are bytes 16g .. 16g + 15 of its four key rows (one
    // 16-byte load each), paired by key and widened in registers; the
    // epilogue writes O back in the natural order.  No fp16 V tile, no
    // ldmatrix, and no CTA-wide widening pass.
    static constexpr bool VDIRECT = (KVT == DT_E4M3) && WARP_LOCAL && D == 128 && (KDIRECT || Q8);
    static_assert(!Q8 || (KVT == DT_E4M3 && D == 128), "e4m3 queries need an e4m3 cache and head size 128");
    // e4m3: widened fp16 tiles after the staging ring (K and V; V only with
    // KDIRECT or Q8; none with VDIRECT)
    static constexpr int CONV_BYTES = (KVT == DT_E4M3) ? (VDIRECT ? 0 : (KDIRECT || Q8) ? TILE16 : 2 * TILE16) : 0;
    static constexpr int OSTRIDE = D + 4;                // fp32 epilogue row stride (bank spread)
    static constexpr int EPI_BYTES = WN * ROWS * OSTRIDE * 4 + 2 * WN * ROWS * 4;
    static constexpr int MAIN_BYTES = STAGES * STAGE_BYTES + CONV_BYTES;
    static constexpr int SMEM = Q_BYTES + (MAIN_BYTES > EPI_BYTES ? MAIN_BYTES : EPI_BYTES);
    // decode shape with two stages: more CTAs per SM instead of a deeper
    // ring -- e4m3 cache: 38 KB (52 KB with a widened V tile) and at most
    // 128 registers a thread, four CTAs; 16-bit cache: 68 KB and at most 168
    // registers, three CTAs (two with three stages, at 100 KB)
    static constexpr int MIN_BLOCKS = (WARP_LOCAL && STAGES == 2) ? (KVT == DT_E4M3 ? 4 : 3) : 1;
    static_assert(WM * WN == 4, "4 warps");
    static_assert(NT % 2 == 0, "n-tile pairs");
    static_assert((RPW * CH) % 32 == 0, "whole warp copy rounds");
};

constexpr float kRescaleLog2 = 8.0f;   // reference-maximum threshold (log2 units)

template <class C>
__global__ void __launch_bounds__(128, C::MIN_BLOCKS) fwd_mma_kernel(const FwdParams p) {
    constexpr int D = C::D, ROWS = C::ROWS, BN = C::BN, STAGES = C::STAGES;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *sQ = smem;
    uint8_t *sMain = smem + C::Q_BYTES;

    pdl_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm = warp % C::WM, wn = warp / C::WM;
    const int r = blockIdx.z, kvh = blockIdx.y;
    const int s_idx = blockIdx.x % p.nsplit;
    const int rb = p.n_row_blocks - 1 - (int)(blockIdx.x / p.nsplit);   // longest rows first

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
    // keys any row of the block may see: up to the last row's causal /
    // right-window bound, from the first row's left-window bound (rounded
    // down to a tile); segments cut that range into whole tiles
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

    // ---- Q rows of this block -> shared memory: e4m3 rows of D bytes with
    // 16-byte chunks swizzled by row & 7 (e4m3 queries), else the 16-bit MMA
    // form, swizzled
    if constexpr (C::Q8) {
        for (int c = tid; c < ROWS * (D / 16); c += blockDim.x) {
            const int lr = c / (D / 16), ch = c % (D / 16);
            const int pr = row0 + lr;
            int4 v = make_int4(0, 0, 0, 0);
            if (pr < row_end)
                v = ldg_nc16(reinterpret_cast<const uint8_t *>(p.q) +
                             (int64_t)(q_start + pr / G) * p.q_stride + (int64_t)(kvh * G + pr % G) * D + ch * 16);
            *reinterpret_cast<int4 *>(sQ + lr * D + ((ch ^ (lr & 7)) << 4)) = v;
        }
    }
    for (int c = tid; c < (C::Q8 ? 0 : ROWS * (D / 8)); c += blockDim.x) {
        const int lr = c / (D / 8), ch = c % (D / 8);
        const int pr = row0 + lr;
        int4 v = make_int4(0, 0, 0, 0);
        if (pr < row_end) {
            const uint8_t *src = reinterpret_cast<const uint8_t *>(p.q) +
                                 ((int64_t)(q_start + pr / G) * p.q_stride + (int64_t)(kvh * G + pr % G) * D) * 2 +
                                 ch * 16;
            v = ldg_nc16(src);
            if constexpr (C::QT == DT_BF16 && !C::MMA_BF16) {
                const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&v);
                int4 w;
                uint32_t *wu = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 f = __bfloat1622float2(b[k]);
                    wu[k] = pack2<false>(f.x, f.y);
                }
                v = w;
            }
        }
        *reinterpret_cast<int4 *>(sQ + swz(lr, ch, C::ROW16)) = v;
    }

    // e4m3 tiles hold value * 2^-8 (see e4m3x4_to_h2x2_lo8): scale S and O back
    const float sl2 = (C::KVT == DT_E4M3 && !C::Q8) ? p.scale_log2 * kE4m3Lo8Scale : p.scale_log2;
    const float vds = (C::KVT == DT_E4M3) ? p.v_descale * kE4m3Lo8Scale : p.v_descale;

    // ---- K/V tile gather through the block table
    const int64_t bt_base = (int64_t)r * p.bt_stride;
    const uint8_t *kbase = reinterpret_cast<const uint8_t *>(p.k_cache);
    const uint8_t *vbase = reinterpret_cast<const uint8_t *>(p.v_cache);
    // byte offset of 16-byte chunk ch of row `row` in a staged e4m3 tile:
    // chunks XOR-swizzled by row & 7 with STAGE_SWZ (the direct K fragment
    // loads of eight rows then hit eight different bank groups), plain otherwise
    auto stage8 = [](int row, int ch) -> uint32_t {
        return (uint32_t)(row * C::KV_ROW + ((C::STAGE_SWZ ? (ch ^ (row & 7)) : ch) << 4));
    };
    auto load_tile = [&](int t, int stage) {
        const int n0 = kv_lo + t * BN;
        int64_t off = 0;
        int ok = 0;
        if (lane < C::RPW) {
            const int tok = n0 + warp * C::RPW + lane;
            if (tok < kv_hi) {
                const int blk = p.block_table[bt_base + tok / p.bs];
                if ((unsigned)blk < (unsigned)p.num_blocks) {
                    ok = 1;
                    off = (((int64_t)blk * p.bs + tok % p.bs) * p.Hkv + kvh) * (int64_t)C::KV_ROW;
                } else {
                    raise_error(p.err, ERR_BLOCK_ID);
                }
            }
        }
        uint8_t *sK = sMain + stage * C::STAGE_BYTES;
        uint8_t *sV = sK + C::TILE_RAW;
#pragma unroll
        for (int it = 0; it < C::RPW * C::CH / 32; ++it) {
            const int idx = it * 32 + lane;
            const int lr = idx / C::CH, ch = idx % C::CH;
            const int64_t o = __shfl_sync(0xffffffffu, off, lr);
            const int v = __shfl_sync(0xffffffffu, ok, lr);
            const int row = warp * C::RPW + lr;
            const uint32_t dst = (C::KVT == DT_E4M3) ? stage8(row, ch) : swz(row, ch, C::KV_ROW);
            const int64_t so = v ? o + ch * 16 : 0;
            cp_async16(smem_u32(sK + dst), kbase + so, v ? 16 : 0);
            cp_async16(smem_u32(sV + dst), vbase + so, v ? 16 : 0);
        }
    };

    // e4m3 tiles are widened to fp16 (exact) into a swizzled tile for
    // ldmatrix.  Warp-local mode: each warp widens only its own rows.
    uint8_t *cK = sMain + STAGES * C::STAGE_BYTES;
    uint8_t *cV = (C::KDIRECT || C::Q8) ? cK : cK + C::TILE16;
    auto convert_tile = [&](int stage) {
        const uint8_t *sK = sMain + stage * C::STAGE_BYTES;
        const uint8_t *sV = sK + C::TILE_RAW;
        constexpr bool own_rows = C::WARP_LOCAL || C::PAIR_LOCAL;   // each warp widens the rows it fetched
        constexpr int kChunks = (own_rows ? C::RPW : BN) * (D / 16);
        const int c0 = own_rows ? lane : tid;
        const int cstep = own_rows ? 32 : (int)blockDim.x;
        const int rbase = own_rows ? warp * C::RPW : 0;
        for (int c = c0; c < kChunks; c += cstep) {
            const int row = rbase + c / (D / 16), ch = c % (D / 16);
            // fp16 patterns of value * 2^-8 (the 2^8 is in the scales)
            if constexpr (!C::KDIRECT && !C::Q8) {
                const int4 rk = *reinterpret_cast<const int4 *>(sK + stage8(row, ch));
                int4 k0, k1;
                e4m3x4_to_h2x2_lo8((uint32_t)rk.x, reinterpret_cast<uint32_t &>(k0.x), reinterpret_cast<uint32_t &>(k0.y));
                e4m3x4_to_h2x2_lo8((uint32_t)rk.y, reinterpret_cast<uint32_t &>(k0.z), reinterpret_cast<uint32_t &>(k0.w));
                e4m3x4_to_h2x2_lo8((uint32_t)rk.z, reinterpret_cast<uint32_t &>(k1.x), reinterpret_cast<uint32_t &>(k1.y));
                e4m3x4_to_h2x2_lo8((uint32_t)rk.w, reinterpret_cast<uint32_t &>(k1.z), reinterpret_cast<uint32_t &>(k1.w));
                *reinterpret_cast<int4 *>(cK + swz(row, 2 * ch, C::ROW16)) = k0;
                *reinterpret_cast<int4 *>(cK + swz(row, 2 * ch + 1, C::ROW16)) = k1;
            }
            const int4 rv = *reinterpret_cast<const int4 *>(sV + stage8(row, ch));
            int4 v0, v1;
            e4m3x4_to_h2x2_lo8((uint32_t)rv.x, reinterpret_cast<uint32_t &>(v0.x), reinterpret_cast<uint32_t &>(v0.y));
            e4m3x4_to_h2x2_lo8((uint32_t)rv.y, reinterpret_cast<uint32_t &>(v0.z), reinterpret_cast<uint32_t &>(v0.w));
            e4m3x4_to_h2x2_lo8((uint32_t)rv.z, reinterpret_cast<uint32_t &>(v1.x), reinterpret_cast<uint32_t &>(v1.y));
            e4m3x4_to_h2x2_lo8((uint32_t)rv.w, reinterpret_cast<uint32_t &>(v1.z), reinterpret_cast<uint32_t &>(v1.w));
            *reinterpret_cast<int4 *>(cV + swz(row, 2 * ch, C::ROW16)) = v0;
            *reinterpret_cast<int4 *>(cV + swz(row, 2 * ch + 1, C::ROW16)) = v1;
        }
    };

    const int n_tiles = (kv_hi - kv_lo + BN - 1) / BN;
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < n_tiles) load_tile(s, s);
        cp_async_commit();
    }
    __syncthreads();   // Q visible to every warp

    uint32_t qf[C::KT][4];
    if constexpr (C::Q8) {
        // e4m3 A fragments, permuted head order (see Q8): k-step kk (32
        // dims) of lane (g, t) holds bytes 32t + 8kk .. + 3 (a0, a1) and
        // 32t + 8kk + 4 .. + 7 (a2, a3) of rows g and g + 8
        const int g = lane >> 2, t4 = lane & 3;
        const int r0 = wm * 16 + g, r1 = r0 + 8;
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk) {
            const int ch = 2 * t4 + (kk >> 1), off = (kk & 1) * 8;
            const uint2 x0 = *reinterpret_cast<const uint2 *>(sQ + r0 * D + ((ch ^ (r0 & 7)) << 4) + off);
            const uint2 x1 = *reinterpret_cast<const uint2 *>(sQ + r1 * D + ((ch ^ (r1 & 7)) << 4) + off);
            qf[kk][0] = x0.x;
            qf[kk][1] = x1.x;
            qf[kk][2] = x0.y;
            qf[kk][3] = x1.y;
        }
    } else if constexpr (C::KDIRECT) {
        // permuted head dimension (see KDIRECT): lane (g, t) takes, for
        // k-step kk, dims 32t + 4kk .. 32t + 4kk + 3 of rows g and g + 8
        const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 r0 = *reinterpret_cast<const uint4 *>(sQ + swz(wm * 16 + g, 4 * t4 + c, C::ROW16));
            const uint4 r1 = *reinterpret_cast<const uint4 *>(sQ + swz(wm * 16 + g + 8, 4 * t4 + c, C::ROW16));
            qf[2 * c][0] = r0.x;       // row g, dims 32t + 8c + 0, 1
            qf[2 * c][2] = r0.y;       // row g, dims 32t + 8c + 2, 3
            qf[2 * c][1] = r1.x;       // row g + 8
            qf[2 * c][3] = r1.y;
            qf[2 * c + 1][0] = r0.z;   // k-step 2c + 1: dims 32t + 8c + 4 .. 7
            qf[2 * c + 1][2] = r0.w;
            qf[2 * c + 1][1] = r1.z;
            qf[2 * c + 1][3] = r1.w;
        }
    } else {
#pragma unroll
        for (int kk = 0; kk < C::KT; ++kk) {
            const int row = wm * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int ch = kk * 2 + (lane >> 4);
            ldmatrix_x4(qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], smem_u32(sQ + swz(row, ch, C::ROW16)));
        }
    }

    // query token (local index) of the two rows this thread owns in C frags
    const int ir0 = (row0 + wm * 16 + (lane >> 2)) / G;
    const int ir1 = (row0 + wm * 16 + (lane >> 2) + 8) / G;
    // visible keys of the two rows: [lo, lim]
    auto last_key = [&](int ir) -> int {
        long long l = p.causal ? (long long)ctx + ir : (long long)INT_MAX;
        if (p.window_right >= 0) l = min(l, (long long)ctx + ir + p.window_right);
        return (int)l;
    };
    const int lim0 = last_key(ir0), lim1 = last_key(ir1);
    const int lo0 = (p.window_left >= 0) ? ctx + ir0 - p.window_left : INT_MIN;
    const int lo1 = (p.window_left >= 0) ? ctx + ir1 - p.window_left : INT_MIN;
    // soft cap: raw score -> cap * log2(e) * tanh(score * scale * k_descale / cap)
    const bool capped = p.cap_in > 0.f;
    const float cap_in = (C::KVT == DT_E4M3 && !C::Q8) ? p.cap_in * kE4m3Lo8Scale : p.cap_in;

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.f, 0.f};

    // the threads that wrote what a warp reads next (and will overwrite what
    // it has read): the warp, its key-slice pair, or the CTA
    auto tile_sync = [&]() {
        if constexpr (C::WARP_LOCAL) __syncwarp();
        else if constexpr (C::PAIR_LOCAL) {
            if (wn == 0) named_bar_sync<1, 64>();
            else named_bar_sync<2, 64>();
        }
        else __syncthreads();
    };
    for (int t = 0; t < n_tiles; ++t) {
        cp_async_wait<STAGES - 2>();
        tile_sync();
        {
            const int tn = t + STAGES - 1;
            if (tn < n_tiles) load_tile(tn, tn % STAGES);
            cp_async_commit();
        }
        const uint8_t *tK, *tV;
        if constexpr (C::VDIRECT) {
            // nothing to widen into shared memory: K and V fragments come
            // straight from the staged bytes
            tK = nullptr;
            tV = sMain + (t % STAGES) * C::STAGE_BYTES + C::TILE_RAW;
        } else if constexpr (C::KVT == DT_E4M3) {
            convert_tile(t % STAGES);
            tile_sync();
            tK = cK;
            tV = cV;
        } else {
            tK = sMain + (t % STAGES) * C::STAGE_BYTES;
            tV = tK + C::TILE_RAW;
        }
        const int n0 = kv_lo + t * BN;

        // S = Q K^T for this warp's NW keys
        float s[C::NT][4];
#pragma unroll
        for (int i = 0; i < C::NT; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
        if constexpr (C::Q8) {
            // n-tile j: lane (g, t) holds key row wn * NW + 8j + g, bytes
            // [32t, 32t + 32): its B fragments of all four k32 steps, as stored
            const uint8_t *raw = sMain + (t % STAGES) * C::STAGE_BYTES;
#pragma unroll
            for (int j = 0; j < C::NT; ++j) {
                const int key = wn * C::NW + 8 * j + (lane >> 2);
                const int c0 = 2 * (lane & 3);
                const uint4 w0 = *reinterpret_cast<const uint4 *>(raw + stage8(key, c0));
                const uint4 w1 = *reinterpret_cast<const uint4 *>(raw + stage8(key, c0 + 1));
                mma16832_e4m3(s[j], qf[0], w0.x, w0.y);
                mma16832_e4m3(s[j], qf[1], w0.z, w0.w);
                mma16832_e4m3(s[j], qf[2], w1.x, w1.y);
                mma16832_e4m3(s[j], qf[3], w1.z, w1.w);
            }
        } else if constexpr (C::KDIRECT) {
            // n-tile j: lane (g, t) holds key row wn * NW + 8j + g, bytes
            // [32t, 32t + 32) = its B fragments of all eight k-steps
            const uint8_t *raw = sMain + (t % STAGES) * C::STAGE_BYTES;
#pragma unroll
            for (int j = 0; j < C::NT; ++j) {
                const int key = wn * C::NW + 8 * j + (lane >> 2);
                const int c0 = 2 * (lane & 3);
                const uint4 w0 = *reinterpret_cast<const uint4 *>(raw + stage8(key, c0));
                const uint4 w1 = *reinterpret_cast<const uint4 *>(raw + stage8(key, c0 + 1));
                const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int kk = 0; kk < C::KT; ++kk) {
                    uint32_t b0, b1;
                    e4m3x4_to_h2x2_lo8(w[kk], b0, b1);
                    mma16816<false>(s[j], qf[kk], b0, b1);
                }
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < C::KT; ++kk) {
#pragma unroll
                for (int j = 0; j < C::NT / 2; ++j) {
                    const int key = wn * C::NW + j * 16 + (lane & 7) + (lane >> 4) * 8;
                    const int ch = kk * 2 + ((lane >> 3) & 1);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(b0, b1, b2, b3, smem_u32(tK + swz(key, ch, C::ROW16)));
                    mma16816<C::MMA_BF16>(s[2 * j], qf[kk], b0, b1);
                    mma16816<C::MMA_BF16>(s[2 * j + 1], qf[kk], b2, b3);
                }
            }
        }

        // scale to log2 units; mask only tiles crossing the sequence end or
        // the causal diagonal ("full" tiles skip this, sec. 4)
        const bool need_mask =
            (n0 + BN > kv_hi) || (p.causal && tile_kind(i_min, i_max + 1, n0, n0 + BN, ctx) != 1) ||
            (p.window_left >= 0 && n0 < ctx + i_max - p.window_left) ||
            (p.window_right >= 0 && (long long)n0 + BN - 1 > (long long)ctx + i_min + p.window_right);
        if (capped) {
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[nt][e] = p.cap_out * tanh_ex2(s[nt][e] * cap_in);
        } else {
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[nt][e] *= sl2;
        }
        if (need_mask) {
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = n0 + wn * C::NW + nt * 8 + 2 * (lane & 3) + (e & 1);
                    const int lim = (e >> 1) ? lim1 : lim0;
                    const int lo = (e >> 1) ? lo1 : lo0;
                    if (key >= kv_hi || key > lim || key < lo) s[nt][e] = -INFINITY;
                }
            }
        }

        // online softmax (two rows per thread, four lanes per row).  m is a
        // reference maximum that moves only when a row's maximum grows by
        // more than 2^8 (log2 units): P is formed against it (every value
        // <= 256, exact since l and O share the reference), and O is
        // rescaled only on the rare tiles that move it
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt) {
            mx[0] = fmaxf(mx[0], fmaxf(s[nt][0], s[nt][1]));
            mx[1] = fmaxf(mx[1], fmaxf(s[nt][2], s[nt][3]));
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        }
        float base[2], alpha[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const bool bump = mx[h] > m[h] + kRescaleLog2;
            alpha[h] = (bump && m[h] != -INFINITY) ? ex2(m[h] - mx[h]) : 1.f;
            if (bump) m[h] = mx[h];
            base[h] = (m[h] == -INFINITY) ? 0.f : m[h];      // fully masked row so far
        }
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt) {
            s[nt][0] = ex2(s[nt][0] - base[0]);
            s[nt][1] = ex2(s[nt][1] - base[0]);
            s[nt][2] = ex2(s[nt][2] - base[1]);
            s[nt][3] = ex2(s[nt][3] - base[1]);
            rs[0] += s[nt][0] + s[nt][1];
            rs[1] += s[nt][2] + s[nt][3];
        }
        l[0] = l[0] * alpha[0] + rs[0];
        l[1] = l[1] * alpha[1] + rs[1];
        if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                o[i][0] *= alpha[0];
                o[i][1] *= alpha[0];
                o[i][2] *= alpha[1];
                o[i][3] *= alpha[1];
            }
        }

        // O += P V (P re-used from the S accumulators as A fragments)
#pragma unroll
        for (int kk = 0; kk < C::NW / 16; ++kk) {
            uint32_t a[4];
            a[0] = pack2<C::MMA_BF16>(s[2 * kk][0], s[2 * kk][1]);
            a[1] = pack2<C::MMA_BF16>(s[2 * kk][2], s[2 * kk][3]);
            a[2] = pack2<C::MMA_BF16>(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            a[3] = pack2<C::MMA_BF16>(s[2 * kk + 1][2], s[2 * kk + 1][3]);
            if constexpr (C::VDIRECT) {
                // keys 2t, 2t + 1, 2t + 8, 2t + 9 of the warp's 16, dims 16g .. 16g + 15
                const int g = lane >> 2, t4 = lane & 3;
                const int kb = wn * C::NW + kk * 16 + 2 * t4;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // one half of the 16 bytes at a time (register pressure)
                    const uint2 r0 = *reinterpret_cast<const uint2 *>(tV + stage8(kb, g) + 8 * h);
                    const uint2 r1 = *reinterpret_cast<const uint2 *>(tV + stage8(kb + 1, g) + 8 * h);
                    const uint2 r2 = *reinterpret_cast<const uint2 *>(tV + stage8(kb + 8, g) + 8 * h);
                    const uint2 r3 = *reinterpret_cast<const uint2 *>(tV + stage8(kb + 9, g) + 8 * h);
                    const uint32_t w0[2] = {r0.x, r0.y}, w1[2] = {r1.x, r1.y};
                    const uint32_t w2[2] = {r2.x, r2.y}, w3[2] = {r3.x, r3.y};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        // n8 tile 4w + i (w = 2h + e): dims 16n + 4w + i
                        const int w = 2 * h + e;
                        mma16816<false>(o[4 * w + 0], a, e4m3_pair_to_h2_lo8<0>(w0[e], w1[e]),
                                        e4m3_pair_to_h2_lo8<0>(w2[e], w3[e]));
                        mma16816<false>(o[4 * w + 1], a, e4m3_pair_to_h2_lo8<1>(w0[e], w1[e]),
                                        e4m3_pair_to_h2_lo8<1>(w2[e], w3[e]));
                        mma16816<false>(o[4 * w + 2], a, e4m3_pair_to_h2_lo8<2>(w0[e], w1[e]),
                                        e4m3_pair_to_h2_lo8<2>(w2[e], w3[e]));
                        mma16816<false>(o[4 * w + 3], a, e4m3_pair_to_h2_lo8<3>(w0[e], w1[e]),
                                        e4m3_pair_to_h2_lo8<3>(w2[e], w3[e]));
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {
                    const int key = wn * C::NW + kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int ch = 2 * j + (lane >> 4);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4_trans(b0, b1, b2, b3, smem_u32(tV + swz(key, ch, C::ROW16)));
                    mma16816<C::MMA_BF16>(o[2 * j], a, b0, b1);
                    mma16816<C::MMA_BF16>(o[2 * j + 1], a, b2, b3);
                }
            }
        }
    }
    pdl_trigger();     // the next kernel may be scheduled; it waits for this grid's completion
    cp_async_wait<0>();
    __syncthreads();   // all shared-memory tiles consumed; reuse for the epilogue

    // ---- epilogue: merge the WN warp states of each row, normalise, store
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
    }
    float *sO = reinterpret_cast<float *>(sMain);
    float *sM = sO + C::WN * ROWS * C::OSTRIDE;
    float *sL = sM + C::WN * ROWS;
    {
        const int lr = wm * 16 + (lane >> 2);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            if constexpr (C::VDIRECT) {
                // permuted order: n8 tile i, columns 2t and 2t + 1 are dims
                // 32t + i and 32t + 16 + i
                const int c0 = 32 * (lane & 3) + i;
                sO[(wn * ROWS + lr) * C::OSTRIDE + c0] = o[i][0];
                sO[(wn * ROWS + lr) * C::OSTRIDE + c0 + 16] = o[i][1];
                sO[(wn * ROWS + lr + 8) * C::OSTRIDE + c0] = o[i][2];
                sO[(wn * ROWS + lr + 8) * C::OSTRIDE + c0 + 16] = o[i][3];
            } else {
                const int col = i * 8 + 2 * (lane & 3);
                *reinterpret_cast<float2 *>(&sO[(wn * ROWS + lr) * C::OSTRIDE + col]) = make_float2(o[i][0], o[i][1]);
                *reinterpret_cast<float2 *>(&sO[(wn * ROWS + lr + 8) * C::OSTRIDE + col]) =
                    make_float2(o[i][2], o[i][3]);
            }
        }
        if ((lane & 3) == 0) {
            sM[wn * ROWS + lr] = m[0];
            sM[wn * ROWS + lr + 8] = m[1];
            sL[wn * ROWS + lr] = l[0];
            sL[wn * ROWS + lr + 8] = l[1];
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
        for (int w = 0; w < C::WN; ++w) mf = fmaxf(mf, sM[w * ROWS + lr]);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float lf = 0.f;
        if (mf != -INFINITY) {
#pragma unroll
            for (int w = 0; w < C::WN; ++w) {
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
            if constexpr (C::QT != DT_FP16) {
                pk.x = pack2<true>(acc.x, acc.y);
                pk.y = pack2<true>(acc.z, acc.w);
            } else {
                pk.x = pack2<false>(acc.x, acc.y);
                pk.y = pack2<false>(acc.z, acc.w);
            }
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
static cudaError_t launch_cfg(const FwdParams &p, cudaStream_t stream) {
    auto kern = fwd_mma_kernel<C>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.n_row_blocks * p.nsplit), (unsigned)p.Hkv, (unsigned)p.B);
    return launch_pdl(kern, grid, dim3(128), C::SMEM, stream, p);
}

template <int D, int QT, int KVT>
static cudaError_t launch_rows(const FwdParams &p, int rows_per_cta, bool single_token, cudaStream_t stream) {
    // D 128: three stages (e4m3: plus one widened tile, 68 KB).  16-row CTAs
    // run two, for more CTAs per SM (see MmaCfg::MIN_BLOCKS), on e4m3 caches
    // (faster on the fp8 decode and mixed batches) and on 16-bit caches when
    // every request of the call has one query token (16-bit verify rows of
    // several tokens measured faster with the deeper ring)
    constexpr int STAGES = (D == 128) ? 3 : 4;
    switch (rows_per_cta) {
    case 16:
        if (D == 128 && (KVT == DT_E4M3 || single_token)) return launch_cfg<MmaCfg<D, 1, 4, 64, 2, QT, KVT>>(p, stream);
        return launch_cfg<MmaCfg<D, 1, 4, 64, STAGES, QT, KVT>>(p, stream);
    case 32: return launch_cfg<MmaCfg<D, 2, 2, 64, STAGES, QT, KVT>>(p, stream);
    default: return launch_cfg<MmaCfg<D, 4, 1, 64, STAGES, QT, KVT>>(p, stream);
    }
}

template <int D>
static cudaError_t launch_d(const FwdParams &p, int q_dtype, int kv_dtype, int rows_per_cta, bool single_token,
                            cudaStream_t s) {
    if (q_dtype == DT_E4M3 && kv_dtype == DT_E4M3) {
        if constexpr (D == 128) return launch_rows<D, DT_E4M3, DT_E4M3>(p, rows_per_cta, single_token, s);
        return cudaErrorInvalidValue;
    }
    if (q_dtype == DT_BF16 && kv_dtype == DT_BF16) return launch_rows<D, DT_BF16, DT_BF16>(p, rows_per_cta, single_token, s);
    if (q_dtype == DT_FP16 && kv_dtype == DT_FP16) return launch_rows<D, DT_FP16, DT_FP16>(p, rows_per_cta, single_token, s);
    if (q_dtype == DT_BF16 && kv_dtype == DT_E4M3) return launch_rows<D, DT_BF16, DT_E4M3>(p, rows_per_cta, single_token, s);
    if (q_dtype == DT_FP16 && kv_dtype == DT_E4M3) return launch_rows<D, DT_FP16, DT_E4M3>(p, rows_per_cta, single_token, s);
    return cudaErrorInvalidValue;
}

int mma_rows_per_cta(int max_rows) { return max_rows <= 16 ? 16 : (max_rows <= 32 ? 32 : 64); }

cudaError_t launch_fwd_mma(const FwdParams &p, int D, int q_dtype, int kv_dtype, int rows_per_cta, bool single_token,
                           cudaStream_t stream) {
    if (D == 64) return launch_d<64>(p, q_dtype, kv_dtype, rows_per_cta, single_token, stream);
    if (D == 128) return launch_d<128>(p, q_dtype, kv_dtype, rows_per_cta, single_token, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
