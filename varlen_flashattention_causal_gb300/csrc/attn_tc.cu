// attn_tc.cu -- varlen causal attention over a paged KV cache on the
// Blackwell tensor cores (tcgen05 MMAs, accumulators in TMEM, TMA loads).
//
// This kernel takes the rows-heavy side of the hot path: prefill and
// chunked prefill, where S = Q K^T and O = P V are genuine dense
// contractions.  One CTA owns one request x one KV head x 256 packed query
// rows (two 128-row Q tiles; a row is a (query token, head-in-group) pair,
// so each K/V tile serves all G query heads of its group) x one KV segment.
//
// Roles (10 warps):
//   warp 0      TMA producer: Q once, then K_j and V_j tiles of 64 keys,
//               each gathered page by page through the block table ("vLLM 中
//               Attention Kernel 如何并行处理多个请求", sec. 11) into a ring of
//               ten 16 KB shared-memory slots (five tiles of look-ahead)
//   warp 1      MMA issuer of Q tile A (one thread) and TMEM owner
//   warp 10     MMA issuer of Q tile B (one thread)
//               Per K/V tile j each issuer X runs S_X(j) = Q_X K_j^T, then
//               O_X += P_X(j-1) V_(j-1).  Two issuers keep the tensor pipe fed:
//               a single thread spends tens of cycles per MMA, commit and
//               barrier wait, and with one issuer those stalls show up as
//               idle tensor cycles.  The two chains touch disjoint TMEM
//               columns; a K/V slot is released when both have consumed it.
//   warps 2-5   softmax warpgroup of Q tile A, one thread per row
//   warps 6-9   softmax warpgroup of Q tile B
// TMEM columns: S_A double buffer [0,64) [64,128), S_B [128,192) [192,256),
// O_A [256,384), O_B [384,512).  P_X(j) (bf16/fp16, two per column) is
// written over the first 32 columns of the S buffer it was computed from and
// is the TMEM "A" operand of O_X += P_X V; only K, V (and Q) are read from
// shared memory by the tensor core, which keeps shared-memory bandwidth
// below the MMA rate.  S_X(j+2) reuses the buffer of P_X(j) only after
// O_X += P_X(j) V has been issued, and tcgen05 MMAs of one thread run in
// order.
//
// Softmax (sec. 7): each thread reads its row of S from TMEM, masks it in
// registers from local positions with the bottom-right alignment of
// sec. 10 (only on tiles that are not full, sec. 4), and keeps a running
// maximum m and sum l.  O lives in TMEM and is rescaled only when a row's
// maximum grows by more than 2^8 (in exp2 units); otherwise P is formed
// against the stale maximum, which keeps every exponential <= 256 and is
// exact because l and O share the same reference.
#include "common.cuh"
#include "sm100.cuh"
#include "tma_host.h"

namespace attn {

using namespace sm100;

namespace {

constexpr int kBM = 128;                               // rows per Q tile
constexpr int kBN = 64;                                // keys per K/V tile
constexpr int kD = 128;                                // head size handled here
constexpr uint32_t kQBytes = kBM * kD * 2;             // one Q tile, 32 KB
constexpr uint32_t kQHalf = kBM * 128;                 // 64 columns of a Q tile
constexpr uint32_t kTileBytes = kBN * kD * 2;          // one 16-bit K or V tile, 16 KB
constexpr uint32_t kKVHalf = kBN * 128;                // 64 columns of a K/V tile
constexpr uint32_t kStageBytes = kBN * kD;             // one e4m3 K or V tile, 8 KB
constexpr float kRescaleThreshold = 8.0f;              // log2 units

// Shared memory map (offsets from a 1024-aligned base).  16-bit caches:
// Q_A, Q_B, then a ring of ten 16 KB K/V slots the TMA fills directly.
// e4m3 caches: Q_A, Q_B, a ring of eight 16 KB fp16 slots, and a ring of
// four 8 KB staging slots the TMA fills with e4m3 pages; two converter
// warps widen each staged tile into the fp16 ring (exact: every e4m3
// value is an fp16 value).
template <bool FP8>
struct TcLayout {
    static constexpr int kSlots = FP8 ? 8 : 10;
    static constexpr int kStages = FP8 ? 4 : 0;
    static constexpr int kThreads = FP8 ? 416 : 352;
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffKV = kOffQ + 2 * kQBytes;
    static constexpr uint32_t kOffStage = kOffKV + kSlots * kTileBytes;
    static constexpr uint32_t kOffBar = kOffStage + kStages * kStageBytes;
    static constexpr int kNumBars = 16 + 2 * kSlots + 2 * kStages;
    static constexpr uint32_t kOffMisc = kOffBar + 8 * 48;
    static constexpr uint32_t kSmemBytes = kOffMisc + 64 + 1024;   // + alignment slack
    static_assert(kNumBars <= 48, "barrier area");
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

// TMEM column offsets of S_x buffer b and O_x
__device__ __forceinline__ uint32_t col_s(int x, int b) { return (uint32_t)x * 128u + (uint32_t)b * 64u; }
__device__ __forceinline__ uint32_t col_o(int x) { return 256u + (uint32_t)x * 128u; }

}  // namespace

struct TcParams {
    FwdParams f;
    int kv_rows;        // rows per TMA page load: gcd(block_size, 64)
};

// whole-warp wait: lane 0 polls, the result is broadcast, so every lane
// takes the same path into the warp-collective tcgen05 instructions after it
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// MMA_BF16: tensor-core operand type (bf16, else fp16); OUT_BF16: output
// type (that of q); FP8: e4m3 caches, widened to fp16 in shared memory.
template <bool MMA_BF16, bool OUT_BF16, bool FP8>
__global__ void __launch_bounds__(TcLayout<FP8>::kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ TcParams tp, const __grid_constant__ CUtensorMap qmap,
                  const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
    using Lay = TcLayout<FP8>;
    constexpr int kSlots = Lay::kSlots, kStages = Lay::kStages;
    constexpr uint32_t kOffQ = Lay::kOffQ, kOffKV = Lay::kOffKV, kOffStage = Lay::kOffStage;
    constexpr uint32_t kOffBar = Lay::kOffBar, kOffMisc = Lay::kOffMisc;
    const FwdParams &p = tp.f;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *sm = smem_raw + (sbase - raw);
    auto bar = [&](int i) { return sbase + kOffBar + 8u * (uint32_t)i; };
    constexpr int B_Q = 0;
    auto B_FULL = [](int s) { return 1 + s; };
    auto B_EMPTY = [](int s) { return 1 + kSlots + s; };
    // S_X, P_X and "O_X += P_X V done" barriers exist per TMEM buffer
    // b = j & 1.  A parity wait is only sound if the barrier is neither two
    // phases ahead of nor two phases behind the phase waited for; per buffer,
    // the next phase always needs work the waiter has not released yet, and
    // the previous one is implied by S_X(j) having landed (one issuer's MMAs
    // complete in order).
    auto B_SFULL = [](int x, int b) { return 1 + 2 * kSlots + 2 * x + b; };
    auto B_PFULL = [](int x, int b) { return 5 + 2 * kSlots + 2 * x + b; };
    auto B_ODONE = [](int x, int b) { return 9 + 2 * kSlots + 2 * x + b; };
    auto B_DRAIN = [](int x) { return 13 + 2 * kSlots + x; };
    // e4m3 mode: staging ring (TMA -> converters) and "Q is fp16" barriers
    auto B_STFULL = [](int t) { return 15 + 2 * kSlots + t; };
    auto B_STEMPTY = [](int t) { return 15 + 2 * kSlots + kStages + t; };
    constexpr int B_QREADY = 15 + 2 * kSlots + 2 * kStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + kOffMisc);
    uint32_t *taddr_slot = reinterpret_cast<uint32_t *>(sm + kOffMisc + 8);
    volatile int *never = reinterpret_cast<volatile int *>(sm + kOffMisc + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = blockIdx.z, kvh = blockIdx.y;
    const int s_idx = blockIdx.x % p.nsplit;
    const int rb = p.n_row_blocks - 1 - (int)(blockIdx.x / p.nsplit);

    // ---- per-CTA work (uniform over the CTA)
    const int q_start = p.cu_seqlens_q[r];
    const int q_len = p.cu_seqlens_q[r + 1] - q_start;
    const int kv_len = p.seqused_k[r];
    const int G = p.G;
    const int rows = q_len * G;
    if (rows < p.rows_lo || rows > p.rows_hi) return;
    const int row0 = rb * 2 * kBM;
    if (row0 >= rows) return;
    const int row_end = min(row0 + 2 * kBM, rows);
    const int ntiles_q = (row_end - row0 + kBM - 1) / kBM;   // 1 or 2 active Q tiles
    const int ctx = kv_len - q_len;
    const int i_max = (row_end - 1) / G;
    int kv_end = kv_len;
    if (p.causal) kv_end = min(kv_len, ctx + i_max + 1);
    const int kv_lo = s_idx * p.split_chunk;
    const int kv_hi = min(kv_end, kv_lo + p.split_chunk);
    const int n_kv = kv_hi > kv_lo ? (kv_hi - kv_lo + kBN - 1) / kBN : 0;

    if (n_kv == 0) {
        // no key for any row in this segment: empty state, no TMEM taken
        for (int pr = row0 + tid; pr < row_end; pr += blockDim.x) {
            const int64_t tok = q_start + pr / G;
            const int h = kvh * G + pr % G;
            if (p.nsplit > 1) {
                p.part_lse[(tok * p.Hq + h) * p.part_stride + s_idx] = -INFINITY;
            } else {
                if (p.lse) p.lse[tok * p.Hq + h] = -INFINITY;
                uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(p.out) +
                                                     (tok * p.out_stride + (int64_t)h * kD) * 2);
                for (int c = 0; c < kD / 8; ++c) o[c] = make_uint4(0, 0, 0, 0);
            }
        }
        return;
    }

    if (tid == 0) {
        *abort_flag = 0;
        *never = 0;
        mbar_init(bar(B_Q), 1);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(bar(B_FULL(s)), FP8 ? 2u : 1u);          // TMA bytes, or the two converter warps
            mbar_init(bar(B_EMPTY(s)), (uint32_t)ntiles_q);   // one release per active Q tile
        }
        for (int t = 0; t < kStages; ++t) {
            mbar_init(bar(B_STFULL(t)), 1);
            mbar_init(bar(B_STEMPTY(t)), 2);
        }
        if (FP8) mbar_init(bar(B_QREADY), 2);
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(B_SFULL(x, 0)), 1);
            mbar_init(bar(B_SFULL(x, 1)), 1);
            mbar_init(bar(B_PFULL(x, 0)), 4);
            mbar_init(bar(B_PFULL(x, 1)), 4);
            mbar_init(bar(B_ODONE(x, 0)), 1);
            mbar_init(bar(B_ODONE(x, 1)), 1);
        }
        mbar_init(bar(B_DRAIN(0)), 1);
        mbar_init(bar(B_DRAIN(1)), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(sbase + kOffMisc + 8, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *taddr_slot;

    if (warp == 0) {
        // =================================================== TMA producer
        const int R = tp.kv_rows;
        const int pages = kBN / R;               // page loads per tile (1..4)
        const int64_t bt_base = (int64_t)r * p.bt_stride;
        int issued = -1;                         // last K/V load index issued
        if (lane == 0) {
            tma_prefetch(&qmap);
            tma_prefetch(&kmap);
            tma_prefetch(&vmap);
            mbar_expect_tx(bar(B_Q), (uint32_t)ntiles_q * kQBytes);
            const int tok0 = q_start + row0 / G;
            const int toks_per_tile = kBM / G;
            for (int x = 0; x < ntiles_q; ++x)
                for (int h = 0; h < 2; ++h)
                    tma_load_3d(sbase + kOffQ + x * kQBytes + h * kQHalf, &qmap, h * 64, kvh * G,
                                tok0 + x * toks_per_tile, bar(B_Q));
        }
        // Page coordinates are read from the block table 32 pages at a time
        // (one per lane) and the next batch is requested a whole batch ahead,
        // so the table's load latency never sits between two tiles.
        const int total_pages = n_kv * pages;
        auto page_coord = [&](int g) -> int {       // row of page g in the cache, -1 if absent
            if (g >= total_pages) return -1;
            const int tok = kv_lo + g * R;
            if (tok >= kv_hi) return -1;
            int blk = p.block_table[bt_base + tok / p.bs];
            if ((unsigned)blk >= (unsigned)p.num_blocks) {
                raise_error(p.err, ERR_BLOCK_ID);
                blk = 0;                             // never dereference an id outside the pool
            }
            return blk * p.bs + tok % p.bs;
        };
        int batch = 0;                               // pages [batch, batch + 32) are in cur
        int cur = page_coord(lane);
        int nxt = page_coord(32 + lane);
        for (int j = 0; j < n_kv; ++j) {
            const int g0 = j * pages;
            if (g0 >= batch + 32) {
                batch += 32;
                cur = nxt;
                nxt = page_coord(batch + 32 + lane);
            }
            // lane pp < pages takes page g0 + pp of this tile (a tile never straddles a batch: 32 % pages == 0)
            const int coord = __shfl_sync(0xffffffffu, cur, (g0 - batch + (lane < pages ? lane : 0)) & 31);
            const int mine = lane < pages ? coord : -1;
            const int nvalid = __popc(__ballot_sync(0xffffffffu, mine >= 0));
            bool ok = true;
            for (int kv = 0; kv < 2 && ok; ++kv) {
                const int L = 2 * j + kv;        // load index
                const CUtensorMap *m = kv ? &vmap : &kmap;
                if constexpr (FP8) {
                    // e4m3 pages -> staging slot (one 128-byte row per key, no swizzle)
                    const int st = L % kStages;
                    if (L >= kStages) ok = warp_wait(bar(B_STEMPTY(st)), ((L / kStages) - 1) & 1, abort_flag);
                    if (!ok) break;
                    if (lane == 0) mbar_expect_tx(bar(B_STFULL(st)), (uint32_t)nvalid * R * kD);
                    __syncwarp();
                    if (mine >= 0)
                        tma_load_3d(sbase + kOffStage + st * kStageBytes + lane * R * 128, m, 0, kvh, mine,
                                    bar(B_STFULL(st)));
                } else {
                    const int slot = L % kSlots;
                    if (L >= kSlots) ok = warp_wait(bar(B_EMPTY(slot)), ((L / kSlots) - 1) & 1, abort_flag);
                    if (!ok) break;
                    if (lane == 0) mbar_expect_tx(bar(B_FULL(slot)), (uint32_t)nvalid * R * kD * 2);
                    __syncwarp();
                    if (mine >= 0) {
                        const uint32_t dst = sbase + kOffKV + slot * kTileBytes + lane * R * 128;
                        tma_load_3d(dst, m, 0, kvh, mine, bar(B_FULL(slot)));
                        tma_load_3d(dst + kKVHalf, m, 64, kvh, mine, bar(B_FULL(slot)));
                    }
                }
                issued = L;
            }
            if (!ok) break;
        }
        // drain: every load issued has landed before the CTA exits
        if (lane == 0) {
            if constexpr (FP8) {
                for (int L = max(0, issued - kStages + 1); L <= issued; ++L)
                    mbar_wait(bar(B_STFULL(L % kStages)), (L / kStages) & 1, never);
            } else {
                for (int L = max(0, issued - kSlots + 1); L <= issued; ++L)
                    mbar_wait(bar(B_FULL(L % kSlots)), (L / kSlots) & 1, never);
            }
            mbar_wait(bar(B_Q), 0, never);
        }
    } else if (warp == 1 || warp == 10) {
        // ================================================ MMA issuers (tile x)
        const int x = warp == 1 ? 0 : 1;
        if (lane == 0 && x < ntiles_q) {
            const uint32_t idS = idesc_f16(MMA_BF16, kBM, kBN, false, false);
            const uint32_t idO = idesc_f16(MMA_BF16, kBM, kD, false, true);
            // descriptors of every operand base, built once; a K slice or a
            // ring slot only adds a small offset to the start-address field
            // (addresses stay below 2^18, so the 14-bit field never carries)
            const uint64_t dQ = sdesc_sw128(sbase + kOffQ + x * kQBytes, 16, 1024);
            const uint64_t dK = sdesc_sw128(sbase + kOffKV, 16, 1024);
            const uint64_t dV = sdesc_sw128(sbase + kOffKV, kKVHalf, 1024);
            const uint32_t tOx = tmem + col_o(x);
            bool ok = mbar_wait(bar(FP8 ? B_QREADY : B_Q), 0, abort_flag);
            for (int j = 0; j <= n_kv && ok; ++j) {
                const int sk = (2 * j) % kSlots;                  // K_j
                const int sv = (2 * j + kSlots - 1) % kSlots;     // V_(j-1)
                if (j < n_kv) {
                    ok = mbar_wait(bar(B_FULL(sk)), ((2 * j) / kSlots) & 1, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t b0 = dK + ((sk * kTileBytes) >> 4);
                    const uint32_t d = tmem + col_s(x, j & 1);
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk)
                        umma_ss(d, dQ + (((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4),
                                b0 + (((kk >> 2) * kKVHalf + (kk & 3) * 32) >> 4), idS, kk > 0 ? 1u : 0u);
                    umma_commit(bar(B_SFULL(x, j & 1)));
                    umma_commit(bar(B_EMPTY(sk)));
                }
                if (j > 0) {
                    ok = mbar_wait(bar(B_FULL(sv)), ((2 * j - 1) / kSlots) & 1, abort_flag);
                    if (ok) ok = mbar_wait(bar(B_PFULL(x, (j - 1) & 1)), ((j - 1) >> 1) & 1, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    // A = P_X from TMEM (8 columns per 16 keys), B = V from shared memory
                    const uint64_t b0 = dV + ((sv * kTileBytes) >> 4);
                    const uint32_t a = tmem + col_s(x, (j - 1) & 1);
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        umma_ts(tOx, a + kk * 8, b0 + ((kk * 2048) >> 4), idO, (j == 1 && kk == 0) ? 0u : 1u);
                    umma_commit(bar(B_ODONE(x, (j - 1) & 1)));
                    umma_commit(bar(B_EMPTY(sv)));
                }
            }
            if (*abort_flag) {
                // a stalled pipeline: wait (bounded) for the MMAs this thread issued
                umma_commit(bar(B_DRAIN(x)));
                mbar_wait(bar(B_DRAIN(x)), 0, never);
            }
        }
    } else if (warp >= 2 && warp <= 9) {
        // ================================================ softmax warpgroups
        const int x = (warp - 2) >> 2;              // Q tile 0 (A) or 1 (B)
        const int quarter = warp & 3;               // TMEM lane quarter this warp may access
        const int trow = quarter * 32 + lane;       // row within the Q tile
        const int prow = row0 + x * kBM + trow;     // packed row within the request
        const bool row_ok = prow < row_end;
        const int qi = prow / G;                    // local query index
        const int lim = p.causal ? ctx + qi : INT_MAX;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_base + col_o(x);
        const float sl2 = p.scale_log2;
        float m_ref = -INFINITY;                    // reference maximum (log2 units)
        float l = 0.f;
        bool ok = x < ntiles_q;
        // query range of this Q tile, for the tile classification
        const int tq_lo = (row0 + x * kBM) / G;
        const int tq_hi = (min(row0 + (x + 1) * kBM, row_end) - 1) / G + 1;
        const int nlim = min(kv_hi - 1, lim);       // last visible key of this row in the segment
        for (int j = 0; j < n_kv && ok; ++j) {
            const int n0 = kv_lo + j * kBN;
            const int b = j & 1;
            const uint32_t tS = tmem + lane_base + col_s(x, b);
            const bool need_mask =
                (n0 + kBN > kv_hi) || (p.causal && tile_kind(tq_lo, tq_hi, n0, n0 + kBN, ctx) != 1);
            ok = warp_wait(bar(B_SFULL(x, b)), (j >> 1) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            uint32_t v[kBN];
            {
                uint32_t (&v0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
                uint32_t (&v1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
                tmem_ld32(tS, v0);
                tmem_ld32(tS + 32, v1);
                tmem_wait_ld();
            }
            // masked keys: this row sees keys n0 .. n0 + nv - 1 of the tile
            const int nv = need_mask ? max(0, min(kBN, nlim - n0 + 1)) : kBN;
            float mx8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mx8[k] = -INFINITY;
            if (nv == kBN) {
#pragma unroll
                for (int e = 0; e < kBN; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], __uint_as_float(v[e]));
            } else {
#pragma unroll
                for (int e = 0; e < kBN; ++e) {
                    const float s = e < nv ? __uint_as_float(v[e]) : -INFINITY;
                    v[e] = __float_as_uint(s);
                    mx8[e & 7] = fmaxf(mx8[e & 7], s);
                }
            }
            float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            mx *= sl2;
            // rescale only when the maximum grows past the threshold
            const bool bump = mx > m_ref + kRescaleThreshold;
            const bool corr = bump && m_ref != -INFINITY;
            const float m_new = bump ? mx : m_ref;
            const float alpha = corr ? ex2(m_ref - m_new) : 1.f;
            const float base = (m_new == -INFINITY) ? 0.f : m_new;
            m_ref = m_new;
            uint32_t pk[32];
            float rs8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) rs8[k] = 0.f;
#pragma unroll
            for (int e = 0; e < kBN; e += 2) {
                const float p0 = ex2(fmaf(__uint_as_float(v[e]), sl2, -base));
                const float p1 = ex2(fmaf(__uint_as_float(v[e + 1]), sl2, -base));
                rs8[(e >> 1) & 7] += p0 + p1;
                pk[e / 2] = pack2<MMA_BF16>(p0, p1);
            }
            const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
            l = l * alpha + rs;
            if (__any_sync(0xffffffffu, corr)) {
                // O_X must hold P_X(j-1) V before it is rescaled
                ok = warp_wait(bar(B_ODONE(x, (j - 1) & 1)), ((j - 1) >> 1) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < kD / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + c * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(tO + c * 32, o);
                }
            }
            if (n0 + kBN > kv_hi) {
                // keys past the segment end: their P is exactly 0, but the V
                // rows there may hold anything (unwritten cache rows, pages
                // not loaded) -- zero them so 0 * V cannot produce NaN.  Both
                // warpgroups write the same zeros, each before publishing its
                // own P, because either issuer may read the tile first.
                const int Lv = 2 * j + 1, sv = Lv % kSlots;
                ok = warp_wait(bar(B_FULL(sv)), (Lv / kSlots) & 1, abort_flag);
                if (!ok) break;
                if (trow < kBN && trow >= kv_hi - n0) {
                    uint4 *v0 = reinterpret_cast<uint4 *>(sm + kOffKV + sv * kTileBytes + trow * 128);
                    uint4 *v1 = reinterpret_cast<uint4 *>(sm + kOffKV + sv * kTileBytes + kKVHalf + trow * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c) v0[c] = v1[c] = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            // P -> TMEM over the S buffer it came from (columns 0..31)
            tmem_st32(tS, pk);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PFULL(x, b)));
        }
        // ---- epilogue: O / l -> out (or the split partials)
        if (ok && x < ntiles_q) {
            // O_X += P_X(n-1) V done implies every earlier P V of this tile is done
            ok = warp_wait(bar(B_ODONE(x, (n_kv - 1) & 1)), ((n_kv - 1) >> 1) & 1, abort_flag);
            if (ok) {
                tc_fence_after();
                const float inv = l > 0.f ? p.v_descale / l : 0.f;
                const float lse_v = l > 0.f ? (m_ref + __log2f(l)) * 0.6931471805599453f : -INFINITY;
                const int64_t tok = q_start + qi;
                const int h = kvh * G + prow % G;
#pragma unroll
                for (int c = 0; c < kD / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + c * 32, o);
                    tmem_wait_ld();
                    if (!row_ok) continue;
                    if (p.nsplit == 1) {
                        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(p.out) +
                                                               (tok * p.out_stride + (int64_t)h * kD + c * 32) * 2);
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint4 w;
                            w.x = pack2<OUT_BF16>(__uint_as_float(o[q4 * 8 + 0]) * inv, __uint_as_float(o[q4 * 8 + 1]) * inv);
                            w.y = pack2<OUT_BF16>(__uint_as_float(o[q4 * 8 + 2]) * inv, __uint_as_float(o[q4 * 8 + 3]) * inv);
                            w.z = pack2<OUT_BF16>(__uint_as_float(o[q4 * 8 + 4]) * inv, __uint_as_float(o[q4 * 8 + 5]) * inv);
                            w.w = pack2<OUT_BF16>(__uint_as_float(o[q4 * 8 + 6]) * inv, __uint_as_float(o[q4 * 8 + 7]) * inv);
                            dst[q4] = w;
                        }
                    } else {
                        float4 *dst = reinterpret_cast<float4 *>(
                            p.part_o + ((tok * p.Hq + h) * p.part_stride + s_idx) * kD + c * 32);
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            dst[q4] = make_float4(__uint_as_float(o[q4 * 4]) * inv, __uint_as_float(o[q4 * 4 + 1]) * inv,
                                                  __uint_as_float(o[q4 * 4 + 2]) * inv,
                                                  __uint_as_float(o[q4 * 4 + 3]) * inv);
                    }
                }
                if (row_ok) {
                    if (p.nsplit == 1) {
                        if (p.lse) p.lse[tok * p.Hq + h] = lse_v;
                    } else {
                        p.part_lse[(tok * p.Hq + h) * p.part_stride + s_idx] = lse_v;
                    }
                }
            }
        }
    } else if (FP8) {
        // ============================== e4m3 -> fp16 converters (warps 11, 12)
        const int cid = tid - 352;                 // 0 .. 63
        bool ok = warp_wait(bar(B_Q), 0, abort_flag);
        if (ok) {
            if constexpr (OUT_BF16) {
                // q arrived as bf16; the MMAs run on fp16 operands: convert in place
                uint4 *qv = reinterpret_cast<uint4 *>(sm + kOffQ);
                for (int c = cid; c < ntiles_q * (int)(kQBytes / 16); c += 64) {
                    const uint4 raw = qv[c];
                    const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
                    uint4 w;
                    uint32_t *wu = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 f = __bfloat1622float2(b2[k]);
                        wu[k] = pack2<false>(f.x, f.y);
                    }
                    qv[c] = w;
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_QREADY));
        }
        for (int L = 0; L < 2 * n_kv && ok; ++L) {
            const int st = L % kStages, sl = L % kSlots;
            ok = warp_wait(bar(B_STFULL(st)), (L / kStages) & 1, abort_flag);
            if (ok && L >= kSlots) ok = warp_wait(bar(B_EMPTY(sl)), ((L / kSlots) - 1) & 1, abort_flag);
            if (!ok) break;
            const uint8_t *src = sm + kOffStage + st * kStageBytes;
            uint8_t *dst = sm + kOffKV + sl * kTileBytes;
            for (int i = cid; i < kBN * 8; i += 64) {
                const int row = i >> 3, c = i & 7;          // e4m3 columns 16c .. 16c + 15 of one key
                const uint4 raw = *reinterpret_cast<const uint4 *>(src + row * 128 + c * 16);
                const uint16_t *b = reinterpret_cast<const uint16_t *>(&raw);
                const uint4 lo = make_uint4(e4m3x2_to_h2(b[0]), e4m3x2_to_h2(b[1]), e4m3x2_to_h2(b[2]),
                                            e4m3x2_to_h2(b[3]));
                const uint4 hi = make_uint4(e4m3x2_to_h2(b[4]), e4m3x2_to_h2(b[5]), e4m3x2_to_h2(b[6]),
                                            e4m3x2_to_h2(b[7]));
                // fp16 columns 16c .. 16c + 15: 64-column half c / 4, 16-byte
                // chunks 2 (c % 4) and 2 (c % 4) + 1 of that half, 128-byte swizzle
                const int q = 2 * (c & 3);
                uint8_t *rowp = dst + (c >> 2) * kKVHalf + row * 128;
                *reinterpret_cast<uint4 *>(rowp + ((q ^ (row & 7)) << 4)) = lo;
                *reinterpret_cast<uint4 *>(rowp + (((q + 1) ^ (row & 7)) << 4)) = hi;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(B_STEMPTY(st)));
                mbar_arrive(bar(B_FULL(sl)));
            }
        }
    }

    // ---- teardown: every MMA has completed before TMEM is released
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (tid == 0 && *abort_flag) raise_error(p.err, ERR_TIMEOUT);
}

static int gcd_int(int a, int b) {
    while (b) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return a;
}

bool tc_supported(int D, int q_dtype, int kv_dtype, int G) {
    if (D != kD) return false;
    const bool ok_types = (q_dtype == DT_BF16 && kv_dtype == DT_BF16) || (q_dtype == DT_FP16 && kv_dtype == DT_FP16) ||
                          ((q_dtype == DT_BF16 || q_dtype == DT_FP16) && kv_dtype == DT_E4M3);
    if (!ok_types) return false;
    if (G <= 0 || G > 128 || (128 % G) != 0) return false;
    return true;
}

int tc_rows_per_cta() { return 2 * kBM; }

template <bool MMA_BF16, bool OUT_BF16, bool FP8>
static cudaError_t launch_tc(const TcParams &tp, const CUtensorMap &qmap, const CUtensorMap &kmap,
                             const CUtensorMap &vmap, dim3 grid, cudaStream_t stream) {
    using Lay = TcLayout<FP8>;
    auto kern = fwd_tc_kernel<MMA_BF16, OUT_BF16, FP8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, Lay::kThreads, Lay::kSmemBytes, stream>>>(tp, qmap, kmap, vmap);
    return cudaGetLastError();
}

cudaError_t launch_fwd_tc(const FwdParams &f, int q_dtype, int kv_dtype, int64_t T, cudaStream_t stream) {
    TcParams tp{};
    tp.f = f;
    tp.kv_rows = gcd_int(f.bs, kBN);
    const bool q16 = q_dtype == DT_FP16;
    const bool fp8 = kv_dtype == DT_E4M3;
    CUtensorMap qmap, kmap, vmap;
    // Q viewed as [T][Hq][D]: box = 64 columns x G heads x (128 / G) tokens
    if (!encode_3d_bf16(&qmap, f.q, q16, kD, (uint64_t)f.Hq, (uint64_t)T, (uint64_t)kD * 2,
                        (uint64_t)f.q_stride * 2, 64, (uint32_t)f.G, (uint32_t)(kBM / f.G)))
        return cudaErrorInvalidValue;
    // caches viewed as [num_blocks * bs][Hkv][D]: box = 1 head x R rows and
    // 64 columns (16-bit, swizzled) or all 128 bytes of a row (e4m3)
    const uint64_t nslots = (uint64_t)f.num_blocks * f.bs;
    const uint32_t R = (uint32_t)tp.kv_rows;
    if (fp8) {
        if (!encode_3d_u8(&kmap, f.k_cache, kD, (uint64_t)f.Hkv, nslots, (uint64_t)kD, (uint64_t)f.Hkv * kD, kD, 1, R) ||
            !encode_3d_u8(&vmap, f.v_cache, kD, (uint64_t)f.Hkv, nslots, (uint64_t)kD, (uint64_t)f.Hkv * kD, kD, 1, R))
            return cudaErrorInvalidValue;
    } else {
        if (!encode_3d_bf16(&kmap, f.k_cache, q16, kD, (uint64_t)f.Hkv, nslots, (uint64_t)kD * 2,
                            (uint64_t)f.Hkv * kD * 2, 64, 1, R) ||
            !encode_3d_bf16(&vmap, f.v_cache, q16, kD, (uint64_t)f.Hkv, nslots, (uint64_t)kD * 2,
                            (uint64_t)f.Hkv * kD * 2, 64, 1, R))
            return cudaErrorInvalidValue;
    }
    dim3 grid((unsigned)(f.n_row_blocks * f.nsplit), (unsigned)f.Hkv, (unsigned)f.B);
    if (fp8) {
        // e4m3 caches: fp16 MMAs (the widening is exact); output in q's type
        return q16 ? launch_tc<false, false, true>(tp, qmap, kmap, vmap, grid, stream)
                   : launch_tc<false, true, true>(tp, qmap, kmap, vmap, grid, stream);
    }
    return q16 ? launch_tc<false, false, false>(tp, qmap, kmap, vmap, grid, stream)
               : launch_tc<true, true, false>(tp, qmap, kmap, vmap, grid, stream);
}

}  // namespace attn
