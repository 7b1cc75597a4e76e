// attn_tc.cu -- varlen causal attention over a paged KV cache on the
// Blackwell tensor cores (tcgen05 MMAs, accumulators in TMEM, TMA loads).
//
// This kernel takes the rows-heavy side of the hot path over e4m3 caches:
// prefill and chunked prefill, where S = Q K^T and O = P V are genuine dense
// contractions.  (16-bit caches run on pairs of SMs, attn_tc2.cu; the
// template's 16-bit form is not instantiated.)  A work item is one request x one KV head x 256 packed
// query rows (two 128-row Q tiles; a row is a (query token, head-in-group)
// pair, so each K/V tile serves all G query heads of its group) x one KV
// segment.
//
// The kernel is persistent: one CTA per SM draws work items of its class
// from a ticket counter until none is left.  Items are numbered request by
// request (within a request: KV head, then row block from the last -- the
// most keys under the causal mask -- to the first, then segment).  Requests
// outside the class cost one step of a scan, not CTA launches, which
// matters in batches that mix a few long prefill chunks with many decode
// rows.  TMEM, the barriers and the pipeline state persist across items, so
// the next item's Q and K/V loads overlap the current item's last tiles
// and epilogue.
//
// Roles (11 warps; 15 with e4m3 caches, 12 with e4m3 queries):
//   warp 0      scheduler and TMA producer: finds the CTA's next item,
//               publishes it in a two-entry ring in shared memory, then
//               loads Q once per item and the K_j and V_j tiles of 64 keys,
//               each gathered page by page through the block table ("vLLM
//               中 Attention Kernel 如何并行处理多个请求", sec. 11) into a
//               ring of ten 16 KB shared-memory slots
//   warp 1      MMA issuer of Q tile A (one thread) and TMEM owner
//   warp 10     MMA issuer of Q tile B (one thread)
//               Per K/V tile j each issuer X runs S_X(j) = Q_X K_j^T, then
//               O_X += P_X(j-1) V_(j-1).  Two issuers keep the tensor pipe fed:
//               a single thread spends tens of cycles per MMA, commit and
//               barrier wait, and with one issuer those stalls show up as
//               idle tensor cycles.  The two chains touch disjoint TMEM
//               columns; a K/V slot is released when both have passed it.
//               An issuer whose Q tile is empty in an item (fewer than 129
//               rows) still waits for every slot of the item and releases it.
//   warps 2-5   softmax warpgroup of Q tile A, one thread per row
//   warps 6-9   softmax warpgroup of Q tile B
//   warps 11-14 (e4m3 caches only) converters: Q to fp16 in place, then
//               every staged e4m3 tile to fp16 in a ring slot
//   e4m3 queries (with an e4m3 cache): Q stays e4m3 and S = Q K^T runs as
//               kind::f8f6f4 MMAs (K = 32 a step) with K read straight from
//               its 128-byte-swizzled staging slot (released by the issuers'
//               commits); warp 11 alone widens only the V tiles, into a ring
//               indexed by V tile; P V stays on fp16
//               ("FlashAttention deep dive", FA3 FP8 path)
// TMEM columns: S_A double buffer [0,64) [64,128), S_B [128,192) [192,256),
// O_A [256,384), O_B [384,512).  P_X(j) (bf16/fp16, two per column) is
// written over the first 32 columns of the S buffer it was computed from and
// is the TMEM "A" operand of O_X += P_X V; only K, V (and Q) are read from
// shared memory by the tensor core, which keeps shared-memory bandwidth
// below the MMA rate.  S_X(j+2) reuses the buffer of P_X(j) only after
// O_X += P_X(j) V has been issued, and tcgen05 MMAs of one thread run in
// order.  The first O_X += P V of an item overwrites O_X only after the
// softmax warpgroup has read out the previous item's O_X.
//
// Every barrier phase is counted across items (load index L over all K/V
// loads of the CTA, tile index per chain, item index), so a parity wait
// never runs two phases behind or ahead: each waiter passes every phase of
// its barriers in order, and the phase after next needs the waiter's own
// release.
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

#include <algorithm>

namespace attn {

using namespace sm100;

namespace {

constexpr int kBM = 128;                               // rows per Q tile
constexpr int kBN = 64;                                // keys per K/V tile
constexpr int kD = 128;                                // head size handled here
constexpr uint32_t kQBytes = kBM * kD * 2;             // one Q tile, 32 KB
constexpr uint32_t kQHalf = kBM * 128;                 // 64 columns of a Q tile
constexpr uint32_t kQBytes8 = kBM * kD;                // one e4m3 Q tile, 16 KB (128-byte rows)
constexpr uint32_t kTileBytes = kBN * kD * 2;          // one 16-bit K or V tile, 16 KB
constexpr uint32_t kKVHalf = kBN * 128;                // 64 columns of a K/V tile
constexpr uint32_t kStageBytes = kBN * kD;             // one e4m3 K or V tile, 8 KB
constexpr float kRescaleThreshold = 8.0f;              // log2 units

// Shared memory map (offsets from a 1024-aligned base).  16-bit caches:
// Q_A, Q_B, then a ring of ten 16 KB K/V slots the TMA fills directly.
// e4m3 caches: Q_A, Q_B, a ring of seven 16 KB fp16 slots, and a ring of
// six 8 KB staging slots the TMA fills with e4m3 pages; the converter
// warps widen each staged tile into the fp16 ring (exact: every e4m3
// value is an fp16 value).  The misc area holds the abort flag, the TMEM
// address and the two-entry work-item ring.
// e4m3 queries (Q8, with an e4m3 cache): Q_A, Q_B as e4m3 (16 KB each), a
// ring of eight 16 KB fp16 slots that holds only V (K is read by the tensor
// core straight from its staging slot), and the staging ring.
template <bool FP8, bool Q8 = false>
struct TcLayout {
    static_assert(!Q8 || FP8, "e4m3 queries need an e4m3 cache");
    static constexpr uint32_t kQTile = Q8 ? kQBytes8 : kQBytes;
    static constexpr int kSlots = FP8 ? (Q8 ? 8 : 7) : 10;
    static constexpr int kStages = FP8 ? 6 : 0;
    // converter warps: four for e4m3 caches with 16-bit q (K, V and Q to
    // widen; 13 to 15 warps all leave 128 registers a thread), one with
    // e4m3 q (V only), which keeps the CTA at 12 warps and 168 registers
    static constexpr int kConvWarps = FP8 ? (Q8 ? 1 : 4) : 0;
    static constexpr int kThreads = 352 + 32 * kConvWarps;
    static constexpr int kConsumerWarps = kThreads / 32 - 1;   // every warp but the producer
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffKV = kOffQ + 2 * kQTile;
    static constexpr uint32_t kOffStage = kOffKV + kSlots * kTileBytes;
    static constexpr uint32_t kOffBar = kOffStage + kStages * kStageBytes;
    static constexpr int kNumBars = 23 + 2 * kSlots + 2 * kStages;
    static constexpr uint32_t kOffMisc = kOffBar + 8 * 64;
    static constexpr uint32_t kSmemBytes = kOffMisc + 128 + 1024;   // + alignment slack
    static_assert(kNumBars <= 64, "barrier area");
    // e4m3 q: K loads (even load index) must always land in even stages, whose
    // release count (the two issuers) differs from the V stages' (converters)
    static_assert(!Q8 || kStages % 2 == 0, "K and V keep their stage parity");
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

// TMEM column offsets of S_x buffer b and O_x
__device__ __forceinline__ uint32_t col_s(int x, int b) { return (uint32_t)x * 128u + (uint32_t)b * 64u; }
__device__ __forceinline__ uint32_t col_o(int x) { return 256u + (uint32_t)x * 128u; }

// One work item and the quantities every role derives from it.
struct Item {
    int r, kvh, rb, s;              // request, KV head, row block (256 packed rows), KV segment
    int q_start, q_len, kv_len;
    int row0, row_end, ntiles_q;    // packed rows [row0, row_end), 1 or 2 active Q tiles
    int ctx, kv_lo, kv_hi, n_kv;    // keys [kv_lo, kv_hi) in n_kv tiles
};

__device__ __forceinline__ void derive(const FwdParams &p, Item &it) {
    const int rows = it.q_len * p.G;
    it.row0 = it.rb * 2 * kBM;
    it.row_end = min(it.row0 + 2 * kBM, rows);
    it.ntiles_q = (it.row_end - it.row0 + kBM - 1) / kBM;
    it.ctx = it.kv_len - it.q_len;
    const int i_min = it.row0 / p.G, i_max = (it.row_end - 1) / p.G;
    // keys any row of the item may see: up to the last row's causal /
    // right-window bound, from the first row's left-window bound rounded
    // down to a tile (a multiple of every page-load height)
    int kv_end = it.kv_len;
    if (p.causal) kv_end = min(it.kv_len, it.ctx + i_max + 1);
    if (p.window_right >= 0) kv_end = (int)min((long long)kv_end, (long long)it.ctx + i_max + p.window_right + 1);
    const int kv_beg = (p.window_left >= 0) ? (max(0, it.ctx + i_min - p.window_left) & ~(kBN - 1)) : 0;
    const long long lo = (long long)kv_beg + (long long)it.s * p.split_chunk;
    it.kv_lo = (int)min(lo, (long long)INT_MAX);
    it.kv_hi = (int)min((long long)kv_end, lo + p.split_chunk);
    it.n_kv = it.kv_hi > it.kv_lo ? (it.kv_hi - it.kv_lo + kBN - 1) / kBN : 0;
}

}  // namespace

struct TcParams {
    FwdParams f;
    int kv_rows;                  // rows per TMA page load: gcd(block_size, 64)
};

// max of three (one instruction on this architecture)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// whole-warp wait: lane 0 polls, the result is broadcast, so every lane
// takes the same path into the warp-collective tcgen05 instructions after it
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// MMA_BF16: tensor-core operand type (bf16, else fp16); OUT_BF16: output
// type (that of q); FP8: e4m3 caches, widened to fp16 in shared memory.
template <bool MMA_BF16, bool OUT_BF16, bool FP8, bool Q8 = false>
__global__ void __launch_bounds__(TcLayout<FP8, Q8>::kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ TcParams tp, const __grid_constant__ CUtensorMap qmap,
                  const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
    using Lay = TcLayout<FP8, Q8>;
    constexpr uint32_t kQTile = Lay::kQTile;
    constexpr int kSlots = Lay::kSlots, kStages = Lay::kStages;
    constexpr uint32_t kOffQ = Lay::kOffQ, kOffKV = Lay::kOffKV, kOffStage = Lay::kOffStage;
    constexpr uint32_t kOffBar = Lay::kOffBar, kOffMisc = Lay::kOffMisc;
    const FwdParams &p = tp.f;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *sm = smem_raw + (sbase - raw);
    auto bar = [&](int i) { return sbase + kOffBar + 8u * (uint32_t)i; };
    constexpr int B_Q = 0;                                   // Q tiles landed, one phase per item with keys
    auto B_FULL = [](int s) { return 1 + s; };
    auto B_EMPTY = [](int s) { return 1 + kSlots + s; };
    constexpr int kB = 1 + 2 * kSlots;
    // S_X, P_X and "O_X += P_X V done" barriers exist per TMEM buffer
    // b = (chain tile index) & 1.  Per buffer, the next phase always needs
    // work the waiter has not released yet, and the previous one is implied
    // by S_X(j) having landed (one issuer's MMAs complete in order).
    auto B_SFULL = [](int x, int b) { return kB + 2 * x + b; };
    auto B_PFULL = [](int x, int b) { return kB + 4 + 2 * x + b; };
    auto B_ODONE = [](int x, int b) { return kB + 8 + 2 * x + b; };
    auto B_DRAIN = [](int x) { return kB + 12 + x; };
    auto B_OFREE = [](int x) { return kB + 14 + x; };        // softmax X has read O_X out
    constexpr int B_QFREE = kB + 16;                         // both chains are done with the Q tiles
    auto B_ITEMF = [](int i) { return kB + 17 + i; };        // ring entry i written
    auto B_ITEME = [](int i) { return kB + 19 + i; };        // ring entry i read by every consumer warp
    constexpr int B_QREADY = kB + 21;                        // e4m3 mode: Q converted to fp16
    auto B_STFULL = [](int t) { return kB + 22 + t; };       // e4m3 staging ring
    auto B_STEMPTY = [](int t) { return kB + 22 + kStages + t; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + kOffMisc);
    uint32_t *taddr_slot = reinterpret_cast<uint32_t *>(sm + kOffMisc + 8);
    volatile int *never = reinterpret_cast<volatile int *>(sm + kOffMisc + 16);
    volatile int *ring = reinterpret_cast<volatile int *>(sm + kOffMisc + 32);   // 2 entries x 8 ints

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.G;

    if (tid == 0) {
        *abort_flag = 0;
        *never = 0;
        mbar_init(bar(B_Q), 1);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(bar(B_FULL(s)), FP8 ? (uint32_t)Lay::kConvWarps : 1u);   // TMA bytes, or the converter warps
            mbar_init(bar(B_EMPTY(s)), 2u);                    // one release per chain
        }
        for (int t = 0; t < kStages; ++t) {
            mbar_init(bar(B_STFULL(t)), 1);
            // released by the converter warps, or (e4m3 q, K stages: even t)
            // by the two MMA issuers
            mbar_init(bar(B_STEMPTY(t)), (Q8 && (t & 1) == 0) ? 2u : (uint32_t)Lay::kConvWarps);
        }
        if (FP8) mbar_init(bar(B_QREADY), (uint32_t)Lay::kConvWarps);
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(B_SFULL(x, 0)), 1);
            mbar_init(bar(B_SFULL(x, 1)), 1);
            mbar_init(bar(B_PFULL(x, 0)), 4);
            mbar_init(bar(B_PFULL(x, 1)), 4);
            mbar_init(bar(B_ODONE(x, 0)), 1);
            mbar_init(bar(B_ODONE(x, 1)), 1);
            mbar_init(bar(B_DRAIN(x)), 1);
            mbar_init(bar(B_OFREE(x)), 4);
        }
        mbar_init(bar(B_QFREE), 2);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_ITEMF(i)), 1);
            mbar_init(bar(B_ITEME(i)), (uint32_t)Lay::kConsumerWarps);
        }
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
    // set-up above touched no global memory; the inputs (and the ticket
    // counter) are used only once the previous kernel has completed
    pdl_wait();

    // consumer warps: take item k from the ring; false on abort, it.r < 0
    // ends the walk
    auto read_item = [&](int k, Item &it) -> bool {
        if (!warp_wait(bar(B_ITEMF(k & 1)), (k >> 1) & 1, abort_flag)) return false;
        __syncwarp();
        const volatile int *e = ring + (k & 1) * 8;
        it.r = e[0];
        it.kvh = e[1];
        it.rb = e[2];
        it.s = e[3];
        it.q_start = e[4];
        it.q_len = e[5];
        it.kv_len = e[6];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_ITEME(k & 1)));
        if (it.r >= 0) derive(p, it);
        return true;
    };

    if (warp == 0) {
        // ======================================= scheduler and TMA producer
        const int R = tp.kv_rows;
        const int pages = kBN / R;               // page loads per tile (1..4)
        // Dynamic schedule: the first item of CTA c is item c, every later
        // one a ticket P + n drawn from the launch's counter, so a CTA that
        // drew long items takes fewer.  Tickets of one CTA only grow, which
        // lets the request scan below move forward only: requests are
        // scanned 32 at a time (one per lane), sc_incl being the inclusive
        // prefix of the item counts in the chunk.
        const long long P = gridDim.x;
        int sc_chunk = -32;
        long long sc_base = 0, sc_total = 0, sc_incl = 0, sc_cnt = 0;
        int sc_q0 = 0, sc_ql = 0, sc_kv = 0, sc_nrb = 0;
        int npipe = 0;                           // items with keys published so far
        int Lbase = 0;                           // K/V loads of earlier items
        int issued = -1;                         // last load index issued
        bool ok = true;
        if (lane == 0) {
            tma_prefetch(&qmap);
            tma_prefetch(&kmap);
            tma_prefetch(&vmap);
        }
        for (int k = 0; ok; ++k) {
            // ---- item k of this CTA
            long long v = blockIdx.x;
            if (k > 0) {
                unsigned long long t = 0;
                if (lane == 0) t = atomicAdd(p.sched, 1ull);
                v = P + (long long)__shfl_sync(0xffffffffu, t, 0);
            }
            while (sc_chunk < p.B && v >= sc_base + sc_total) {
                sc_base += sc_total;
                sc_chunk += 32;
                const int r = sc_chunk + lane;
                sc_cnt = 0;
                sc_nrb = 0;
                if (r < p.B) {
                    sc_q0 = p.cu_seqlens_q ? p.cu_seqlens_q[r] : r;
                    sc_ql = (p.cu_seqlens_q ? p.cu_seqlens_q[r + 1] : r + 1) - sc_q0;
                    sc_kv = p.seqused_k[r];
                    const int rows = sc_ql * G;
                    if (rows > 0 && rows >= p.rows_lo && rows <= p.rows_hi) {
                        sc_nrb = (rows + 2 * kBM - 1) / (2 * kBM);
                        sc_cnt = (long long)sc_nrb * p.Hkv * p.nsplit;
                    }
                }
                sc_incl = sc_cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const long long t = __shfl_up_sync(0xffffffffu, sc_incl, o);
                    if (lane >= o) sc_incl += t;
                }
                sc_total = __shfl_sync(0xffffffffu, sc_incl, 31);
            }
            Item it{};
            it.r = -1;
            if (v < sc_base + sc_total) {
                const long long rel = v - sc_base;
                const int src = __ffs(__ballot_sync(0xffffffffu, sc_incl > rel)) - 1;
                const long long u =
                    rel - (__shfl_sync(0xffffffffu, sc_incl, src) - __shfl_sync(0xffffffffu, sc_cnt, src));
                const int nrb = __shfl_sync(0xffffffffu, sc_nrb, src);
                it.r = sc_chunk + src;
                it.q_start = __shfl_sync(0xffffffffu, sc_q0, src);
                it.q_len = __shfl_sync(0xffffffffu, sc_ql, src);
                it.kv_len = __shfl_sync(0xffffffffu, sc_kv, src);
                it.s = (int)(u % p.nsplit);
                const long long t = u / p.nsplit;
                it.rb = nrb - 1 - (int)(t % nrb);
                it.kvh = (int)(t / nrb);
            }
            // ---- publish it: entry k & 1 is free once every consumer warp has read item k - 2
            if (k >= 2) ok = warp_wait(bar(B_ITEME(k & 1)), ((k >> 1) - 1) & 1, abort_flag);
            if (!ok) break;
            if (lane == 0) {
                volatile int *e = ring + (k & 1) * 8;
                e[0] = it.r;
                e[1] = it.kvh;
                e[2] = it.rb;
                e[3] = it.s;
                e[4] = it.q_start;
                e[5] = it.q_len;
                e[6] = it.kv_len;
                mbar_arrive(bar(B_ITEMF(k & 1)));
            }
            __syncwarp();
            if (it.r < 0) break;
            derive(p, it);
            if (it.n_kv == 0) continue;

            // ---- Q tiles, once both chains are done with the previous item's
            if (npipe > 0) ok = warp_wait(bar(B_QFREE), (npipe - 1) & 1, abort_flag);
            if (!ok) break;
            if (lane == 0) {
                mbar_expect_tx(bar(B_Q), (uint32_t)it.ntiles_q * kQTile);
                const int tok0 = it.q_start + it.row0 / G;
                const int toks_per_tile = kBM / G;
                // 16-bit q: two boxes of 64 columns; e4m3 q: one box of 128 bytes
                for (int x = 0; x < it.ntiles_q; ++x)
                    for (int h = 0; h < (Q8 ? 1 : 2); ++h)
                        tma_load_3d(sbase + kOffQ + x * kQTile + h * kQHalf, &qmap, h * 64, it.kvh * G,
                                    tok0 + x * toks_per_tile, bar(B_Q));
            }
            __syncwarp();
            ++npipe;

            // ---- K/V tiles.  Page coordinates are read from the block table
            // 32 pages at a time (one per lane) and the next batch is
            // requested a whole batch ahead, so the table's load latency
            // never sits between two tiles.
            const int64_t bt_base = (int64_t)it.r * p.bt_stride;
            const int total_pages = it.n_kv * pages;
            const int kv_lo = it.kv_lo, kv_hi = it.kv_hi;
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
            for (int j = 0; j < it.n_kv && ok; ++j) {
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
                for (int kv = 0; kv < 2 && ok; ++kv) {
                    const int L = Lbase + 2 * j + kv;    // load index
                    const CUtensorMap *m = kv ? &vmap : &kmap;
                    if constexpr (FP8) {
                        // e4m3 pages -> staging slot (one 128-byte row per key, no swizzle)
                        const int st = L % kStages;
                        if (L >= kStages) ok = warp_wait(bar(B_STEMPTY(st)), ((L / kStages) - 1) & 1, abort_flag);
                        if (!ok) break;
                        if (lane == 0) mbar_expect_tx(bar(B_STFULL(st)), (uint32_t)nvalid * R * kD);
                        __syncwarp();
                        if (mine >= 0)
                            tma_load_3d(sbase + kOffStage + st * kStageBytes + lane * R * 128, m, 0, it.kvh, mine,
                                        bar(B_STFULL(st)));
                    } else {
                        const int slot = L % kSlots;
                        if (L >= kSlots) ok = warp_wait(bar(B_EMPTY(slot)), ((L / kSlots) - 1) & 1, abort_flag);
                        if (!ok) break;
                        if (lane == 0) mbar_expect_tx(bar(B_FULL(slot)), (uint32_t)nvalid * R * kD * 2);
                        __syncwarp();
                        if (mine >= 0) {
                            const uint32_t dst = sbase + kOffKV + slot * kTileBytes + lane * R * 128;
                            tma_load_3d(dst, m, 0, it.kvh, mine, bar(B_FULL(slot)));
                            tma_load_3d(dst + kKVHalf, m, 64, it.kvh, mine, bar(B_FULL(slot)));
                        }
                    }
                    issued = L;
                }
            }
            Lbase += 2 * it.n_kv;
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
            if (npipe > 0) mbar_wait(bar(B_Q), (npipe - 1) & 1, never);
        }
    } else if (warp == 1 || warp == 10) {
        // ================================================ MMA issuers (tile x)
        const int x = warp == 1 ? 0 : 1;
        const uint32_t idS = idesc_f16(MMA_BF16, kBM, kBN, false, false);
        const uint32_t idO = idesc_f16(MMA_BF16, kBM, kD, false, true);
        // descriptors of every operand base, built once; a K slice or a
        // ring slot only adds a small offset to the start-address field
        // (addresses stay below 2^18, so the 14-bit field never carries)
        const uint64_t dQ = sdesc_sw128(sbase + kOffQ + x * kQTile, 16, 1024);
        const uint64_t dK = sdesc_sw128(sbase + kOffKV, 16, 1024);
        const uint64_t dK8 = sdesc_sw128(sbase + kOffStage, 16, 1024);   // e4m3 q: K in its staging slot
        const uint64_t dV = sdesc_sw128(sbase + kOffKV, kKVHalf, 1024);
        const uint32_t tOx = tmem + col_o(x);
        int npipe = 0, Lbase = 0;
        int jx = 0;                              // tiles of this chain in earlier items
        int ax = 0;                              // earlier items in which this chain had rows
        bool ok = true;
        for (int k = 0; ok; ++k) {
            Item it;
            ok = read_item(k, it);
            if (!ok || it.r < 0) break;
            if (it.n_kv == 0) continue;
            const int n_kv = it.n_kv;
            const bool active = x < it.ntiles_q;
            if (lane == 0) {
                ok = mbar_wait(bar(FP8 ? B_QREADY : B_Q), npipe & 1, abort_flag);
                if (ok && !active) {
                    // no rows of this chain in the item: release Q and pass
                    // every slot in order (the other chain's MMAs gate the reuse)
                    mbar_arrive(bar(B_QFREE));
                    for (int L = Lbase; L < Lbase + 2 * n_kv && ok; ++L) {
                        if constexpr (Q8) {
                            if ((L & 1) == 0) {
                                // K_j is read from its staging slot
                                const int st = L % kStages;
                                ok = mbar_wait(bar(B_STFULL(st)), (L / kStages) & 1, abort_flag);
                                if (ok) mbar_arrive(bar(B_STEMPTY(st)));
                            } else {
                                const int v = L >> 1;           // fp16 ring position (V only)
                                ok = mbar_wait(bar(B_FULL(v % kSlots)), (v / kSlots) & 1, abort_flag);
                                if (ok) mbar_arrive(bar(B_EMPTY(v % kSlots)));
                            }
                        } else {
                            ok = mbar_wait(bar(B_FULL(L % kSlots)), (L / kSlots) & 1, abort_flag);
                            if (ok) mbar_arrive(bar(B_EMPTY(L % kSlots)));
                        }
                    }
                }
                for (int j = 0; active && j <= n_kv && ok; ++j) {
                    const int LK = Lbase + 2 * j;          // load index of K_j
                    const int LV = LK - 1;                 // load index of V_(j-1)
                    const int jg = jx + j;                 // chain tile index of K_j
                    if (j < n_kv) {
                        const uint32_t d = tmem + col_s(x, jg & 1);
                        if constexpr (Q8) {
                            // S = Q K^T on e4m3 operands (K = 32 a step), K read
                            // straight from its 128-byte-swizzled staging slot
                            const int st = LK % kStages;
                            ok = mbar_wait(bar(B_STFULL(st)), (LK / kStages) & 1, abort_flag);
                            if (!ok) break;
                            tc_fence_after();
                            const uint64_t b0 = dK8 + ((st * kStageBytes) >> 4);
#pragma unroll
                            for (int kk = 0; kk < kD / 32; ++kk)
                                umma_ss_f8(d, dQ + ((kk * 32) >> 4), b0 + ((kk * 32) >> 4), idS, kk > 0 ? 1u : 0u);
                            umma_commit(bar(B_SFULL(x, jg & 1)));
                            umma_commit(bar(B_STEMPTY(st)));
                        } else {
                            const int sk = LK % kSlots;
                            ok = mbar_wait(bar(B_FULL(sk)), (LK / kSlots) & 1, abort_flag);
                            if (!ok) break;
                            tc_fence_after();
                            const uint64_t b0 = dK + ((sk * kTileBytes) >> 4);
#pragma unroll
                            for (int kk = 0; kk < kD / 16; ++kk)
                                umma_ss(d, dQ + (((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4),
                                        b0 + (((kk >> 2) * kKVHalf + (kk & 3) * 32) >> 4), idS, kk > 0 ? 1u : 0u);
                            umma_commit(bar(B_SFULL(x, jg & 1)));
                            umma_commit(bar(B_EMPTY(sk)));
                        }
                        if (j == n_kv - 1) umma_commit(bar(B_QFREE));
                    }
                    if (j > 0) {
                        const int vpos = Q8 ? (LV >> 1) : LV;    // fp16 ring position of V_(j-1)
                        const int sv = vpos % kSlots;
                        ok = mbar_wait(bar(B_FULL(sv)), (vpos / kSlots) & 1, abort_flag);
                        if (ok) ok = mbar_wait(bar(B_PFULL(x, (jg - 1) & 1)), ((jg - 1) >> 1) & 1, abort_flag);
                        // the item's first P V overwrites O_X: the previous
                        // item's epilogue must have read it out
                        if (ok && j == 1 && ax > 0) ok = mbar_wait(bar(B_OFREE(x)), (ax - 1) & 1, abort_flag);
                        if (!ok) break;
                        tc_fence_after();
                        // A = P_X from TMEM (8 columns per 16 keys), B = V from shared memory
                        const uint64_t b0 = dV + ((sv * kTileBytes) >> 4);
                        const uint32_t a = tmem + col_s(x, (jg - 1) & 1);
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk)
                            umma_ts(tOx, a + kk * 8, b0 + ((kk * 2048) >> 4), idO, (j == 1 && kk == 0) ? 0u : 1u);
                        umma_commit(bar(B_ODONE(x, (jg - 1) & 1)));
                        umma_commit(bar(B_EMPTY(sv)));
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            Lbase += 2 * n_kv;
            ++npipe;
            if (active) {
                jx += n_kv;
                ++ax;
            }
        }
        if (lane == 0 && *abort_flag) {
            // a stalled pipeline: wait (bounded) for the MMAs this thread issued
            umma_commit(bar(B_DRAIN(x)));
            mbar_wait(bar(B_DRAIN(x)), 0, never);
        }
    } else if (warp >= 2 && warp <= 9) {
        // ================================================ softmax warpgroups
        const int x = (warp - 2) >> 2;              // Q tile 0 (A) or 1 (B)
        const int quarter = warp & 3;               // TMEM lane quarter this warp may access
        const int trow = quarter * 32 + lane;       // row within the Q tile
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_base + col_o(x);
        // e4m3 tiles hold value * 2^-8 (see e4m3x4_to_h2x2_lo8): scale S and O back
        const float vds = FP8 ? p.v_descale * kE4m3Lo8Scale : p.v_descale;
        // soft cap: S -> cap * log2(e) * tanh(S * scale * k_descale / cap),
        // already in log2 units; else S * scale * k_descale * log2(e)
        const bool capped = p.cap_in > 0.f;
        // (with e4m3 q, K is not widened: S carries no 2^-8)
        constexpr bool kWideK = FP8 && !Q8;
        const float cap_in = kWideK ? p.cap_in * kE4m3Lo8Scale : p.cap_in;
        const float sl2 = capped ? 1.f : (kWideK ? p.scale_log2 * kE4m3Lo8Scale : p.scale_log2);
        int Lbase = 0, jx = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            Item it;
            ok = read_item(k, it);
            if (!ok || it.r < 0) break;
            if (it.n_kv == 0) {
                // no key for any row in this segment: empty state (a sink
                // alone, in segment 0), no pipeline work
                for (int pr = it.row0 + (tid - 64); pr < it.row_end; pr += 256) {
                    const int64_t tok = it.q_start + pr / G;
                    const int h = it.kvh * G + pr % G;
                    const float zl = (p.sinks && it.s == 0) ? p.sinks[h] : -INFINITY;
                    if (p.partials) {
                        const int64_t slot = (tok * p.Hq + h) * p.part_stride + it.s;
                        p.part_lse[slot] = zl;
                        if (zl != -INFINITY)
                            for (int d = 0; d < kD; ++d) p.part_o[slot * kD + d] = 0.f;
                    } else {
                        if (p.lse) p.lse[tok * p.Hq + h] = zl;
                        uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(p.out) +
                                                             (tok * p.out_stride + (int64_t)h * kD) * 2);
                        for (int c = 0; c < kD / 8; ++c) o[c] = make_uint4(0, 0, 0, 0);
                    }
                }
                continue;
            }
            const int n_kv = it.n_kv, kv_lo = it.kv_lo, kv_hi = it.kv_hi;
            if (x < it.ntiles_q) {
                const int prow = it.row0 + x * kBM + trow;  // packed row within the request
                const bool row_ok = prow < it.row_end;
                const int qi = prow / G;                    // local query index
                long long lim_ll = p.causal ? (long long)it.ctx + qi : (long long)INT_MAX;
                if (p.window_right >= 0) lim_ll = min(lim_ll, (long long)it.ctx + qi + p.window_right);
                const int lim = (int)lim_ll;                // last visible key of this row
                const int lo_key = (p.window_left >= 0) ? it.ctx + qi - p.window_left : INT_MIN;
                float m_ref = -INFINITY;                    // reference maximum (log2 units)
                float l = 0.f;
                // query range of this Q tile, for the tile classification
                const int tq_lo = (it.row0 + x * kBM) / G;
                const int tq_hi = (min(it.row0 + (x + 1) * kBM, it.row_end) - 1) / G + 1;
                const int nlim = min(kv_hi - 1, lim);       // last visible key of this row in the segment
                for (int j = 0; j < n_kv && ok; ++j) {
                    const int n0 = kv_lo + j * kBN;
                    const int jg = jx + j;
                    const int b = jg & 1;
                    const uint32_t tS = tmem + lane_base + col_s(x, b);
                    const bool need_mask =
                        (n0 + kBN > kv_hi) || (p.causal && tile_kind(tq_lo, tq_hi, n0, n0 + kBN, it.ctx) != 1) ||
                        (p.window_left >= 0 && n0 < it.ctx + tq_hi - 1 - p.window_left) ||
                        (p.window_right >= 0 && (long long)n0 + kBN - 1 > (long long)it.ctx + tq_lo + p.window_right);
                    ok = warp_wait(bar(B_SFULL(x, b)), (jg >> 1) & 1, abort_flag);
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
                    if (capped) {
#pragma unroll
                        for (int e = 0; e < kBN; ++e)
                            v[e] = __float_as_uint(p.cap_out * tanh_ex2(__uint_as_float(v[e]) * cap_in));
                    }
                    // masked keys: this row sees keys n0 + e_lo .. n0 + nv - 1 of the tile
                    int nv = kBN, e_lo = 0;
                    if (need_mask) {
                        nv = max(0, min(kBN, nlim - n0 + 1));
                        if (p.window_left >= 0) e_lo = min(kBN, max(0, lo_key - n0));
                    }
                    if (nv < kBN || e_lo > 0) {
#pragma unroll
                        for (int e = 0; e < kBN; ++e)
                            if (e >= nv || e < e_lo) v[e] = __float_as_uint(-INFINITY);
                    }
                    // row maximum: three-input max in four independent chains
                    // (the softmax is issue bound: fewer instructions per element
                    // is what speeds it up)
                    float mx4[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) mx4[c] = fmaxf(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]));
#pragma unroll
                    for (int b8 = 8; b8 < kBN; b8 += 8) {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            mx4[c] = fmax3(mx4[c], __uint_as_float(v[b8 + 2 * c]), __uint_as_float(v[b8 + 2 * c + 1]));
                    }
                    float mx = fmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
                    mx *= sl2;
                    // rescale only when the maximum grows past the threshold
                    const bool bump = mx > m_ref + kRescaleThreshold;
                    const bool corr = bump && m_ref != -INFINITY;
                    const float m_new = bump ? mx : m_ref;
                    const float alpha = corr ? ex2(m_ref - m_new) : 1.f;
                    const float base = (m_new == -INFINITY) ? 0.f : m_new;
                    m_ref = m_new;
                    // P = 2^(s * scale - m): scale-and-shift and the row sum on
                    // packed fp32 pairs (one instruction per two elements)
                    uint32_t pk[32];
                    float2 rs2[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) rs2[c] = make_float2(0.f, 0.f);
                    const float2 sc2 = make_float2(sl2, sl2), nb2 = make_float2(-base, -base);
#pragma unroll
                    for (int e = 0; e < kBN; e += 2) {
                        const float2 x2 =
                            __ffma2_rn(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sc2, nb2);
                        const float p0 = ex2(x2.x);
                        const float p1 = ex2(x2.y);
                        rs2[(e >> 1) & 3] = __fadd2_rn(rs2[(e >> 1) & 3], make_float2(p0, p1));
                        pk[e / 2] = pack2<MMA_BF16>(p0, p1);
                    }
                    const float2 r01 = __fadd2_rn(rs2[0], rs2[1]), r23 = __fadd2_rn(rs2[2], rs2[3]);
                    const float2 r03 = __fadd2_rn(r01, r23);
                    const float rs = r03.x + r03.y;
                    l = l * alpha + rs;
                    if (__any_sync(0xffffffffu, corr)) {
                        // O_X must hold P_X(j-1) V before it is rescaled (corr implies j > 0)
                        ok = warp_wait(bar(B_ODONE(x, (jg - 1) & 1)), ((jg - 1) >> 1) & 1, abort_flag);
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
                        const int Lv = Lbase + 2 * j + 1;
                        const int vpos = Q8 ? (Lv >> 1) : Lv;   // fp16 ring position of V_j
                        const int sv = vpos % kSlots;
                        ok = warp_wait(bar(B_FULL(sv)), (vpos / kSlots) & 1, abort_flag);
                        if (!ok) break;
                        __syncwarp();
                        if (trow < kBN && trow >= kv_hi - n0) {
                            uint4 *v0 = reinterpret_cast<uint4 *>(sm + kOffKV + sv * kTileBytes + trow * 128);
                            uint4 *v1 =
                                reinterpret_cast<uint4 *>(sm + kOffKV + sv * kTileBytes + kKVHalf + trow * 128);
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
                if (ok) {
                    // O_X += P_X(last) V done implies every earlier P V of this item is done
                    const int jl = jx + n_kv - 1;
                    ok = warp_wait(bar(B_ODONE(x, jl & 1)), (jl >> 1) & 1, abort_flag);
                }
                if (ok) {
                    tc_fence_after();
                    const int64_t tok = it.q_start + qi;
                    const int h = it.kvh * G + prow % G;
                    float sink_scale = 1.f;
                    if (row_ok && p.sinks && it.s == 0 && p.sinks[h] > -INFINITY) {
                        // the sink joins segment 0's state: a virtual key with logit z, value 0
                        const float z2 = p.sinks[h] * 1.4426950408889634f;
                        const float mn = fmaxf(m_ref, z2);
                        sink_scale = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - mn);
                        l = l * sink_scale + ex2(z2 - mn);
                        m_ref = mn;
                    }
                    const float inv = l > 0.f ? vds * sink_scale / l : 0.f;
                    const float lse_v = l > 0.f ? (m_ref + __log2f(l)) * 0.6931471805599453f : -INFINITY;
#pragma unroll
                    for (int c = 0; c < kD / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + c * 32, o);
                        tmem_wait_ld();
                        if (!row_ok) continue;
                        if (!p.partials) {
                            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(p.out) +
                                                                   (tok * p.out_stride + (int64_t)h * kD + c * 32) * 2);
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                uint4 w;
                                w.x = pack2<OUT_BF16>(__uint_as_float(o[q4 * 8 + 0]) * inv,
                                                      __uint_as_float(o[q4 * 8 + 1]) * inv);
                                w.y = pack2<OUT_BF16>(__uint_as_float(o[q4 * 8 + 2]) * inv,
                                                      __uint_as_float(o[q4 * 8 + 3]) * inv);
                                w.z = pack2<OUT_BF16>(__uint_as_float(o[q4 * 8 + 4]) * inv,
                                                      __uint_as_float(o[q4 * 8 + 5]) * inv);
                                w.w = pack2<OUT_BF16>(__uint_as_float(o[q4 * 8 + 6]) * inv,
                                                      __uint_as_float(o[q4 * 8 + 7]) * inv);
                                dst[q4] = w;
                            }
                        } else {
                            float4 *dst = reinterpret_cast<float4 *>(
                                p.part_o + ((tok * p.Hq + h) * p.part_stride + it.s) * kD + c * 32);
#pragma unroll
                            for (int q4 = 0; q4 < 8; ++q4)
                                dst[q4] = make_float4(__uint_as_float(o[q4 * 4]) * inv,
                                                      __uint_as_float(o[q4 * 4 + 1]) * inv,
                                                      __uint_as_float(o[q4 * 4 + 2]) * inv,
                                                      __uint_as_float(o[q4 * 4 + 3]) * inv);
                        }
                    }
                    if (row_ok) {
                        if (!p.partials) {
                            if (p.lse) p.lse[tok * p.Hq + h] = lse_v;
                        } else {
                            p.part_lse[(tok * p.Hq + h) * p.part_stride + it.s] = lse_v;
                        }
                    }
                    // O_X has been read out: the chain may start the next item's P V
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_OFREE(x)));
                }
                jx += n_kv;
            }
            Lbase += 2 * n_kv;
        }
    } else if constexpr (FP8) {
        // =========== e4m3 -> fp16 converters (warps 11-14; 11 alone with e4m3 q)
        constexpr int kConvThreads = 32 * Lay::kConvWarps;
        constexpr int kConvChunks = kBN * kD / 16 / kConvThreads;   // 16-byte chunks of a staged tile a thread
        const int cid = tid - 352;                 // 0 .. kConvThreads - 1
        int npipe = 0, Lbase = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            Item it;
            ok = read_item(k, it);
            if (!ok || it.r < 0) break;
            if (it.n_kv == 0) continue;
            ok = warp_wait(bar(B_Q), npipe & 1, abort_flag);
            if (!ok) break;
            __syncwarp();
            if constexpr (OUT_BF16 && !Q8) {
                // q arrived as bf16; the MMAs run on fp16 operands: convert in place
                uint4 *qv = reinterpret_cast<uint4 *>(sm + kOffQ);
                for (int c = cid; c < it.ntiles_q * (int)(kQBytes / 16); c += kConvThreads) {
                    const uint4 raw4 = qv[c];
                    const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&raw4);
                    uint4 w;
                    uint32_t *wu = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(b2[e]);
                        wu[e] = pack2<false>(f.x, f.y);
                    }
                    qv[c] = w;
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_QREADY));
            // every staged tile, or with e4m3 q only the V tiles (odd L; the
            // tensor core reads K in its staging slot), at ring position v
            for (int L = Lbase + (Q8 ? 1 : 0); L < Lbase + 2 * it.n_kv && ok; L += (Q8 ? 2 : 1)) {
                const int v = Q8 ? (L >> 1) : L;
                const int st = L % kStages, sl = v % kSlots;
                ok = warp_wait(bar(B_STFULL(st)), (L / kStages) & 1, abort_flag);
                if (!ok) break;
                __syncwarp();
                // the staged tile goes to registers (8 x 16 bytes a thread) and
                // the stage back to the producer at once, so the TMA loads in
                // flight never wait on the fp16 ring
                const uint8_t *src = sm + kOffStage + st * kStageBytes;
                uint4 raw8[kConvChunks];
#pragma unroll
                for (int u = 0; u < kConvChunks; ++u) {
                    const int i = cid + kConvThreads * u;
                    raw8[u] = *reinterpret_cast<const uint4 *>(src + (i >> 3) * 128 + (i & 7) * 16);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_STEMPTY(st)));
                if (v >= kSlots) ok = warp_wait(bar(B_EMPTY(sl)), ((v / kSlots) - 1) & 1, abort_flag);
                if (!ok) break;
                uint8_t *dst = sm + kOffKV + sl * kTileBytes;
#pragma unroll
                for (int u = 0; u < kConvChunks; ++u) {
                    const int i = cid + kConvThreads * u;
                    const int row = i >> 3, c = i & 7;          // e4m3 columns 16c .. 16c + 15 of one key
                    const uint4 raw4 = raw8[u];
                    uint4 lo, hi;                                // fp16 patterns of value * 2^-8
                    e4m3x4_to_h2x2_lo8(raw4.x, lo.x, lo.y);
                    e4m3x4_to_h2x2_lo8(raw4.y, lo.z, lo.w);
                    e4m3x4_to_h2x2_lo8(raw4.z, hi.x, hi.y);
                    e4m3x4_to_h2x2_lo8(raw4.w, hi.z, hi.w);
                    // fp16 columns 16c .. 16c + 15: 64-column half c / 4, 16-byte
                    // chunks 2 (c % 4) and 2 (c % 4) + 1 of that half, 128-byte swizzle
                    const int q = 2 * (c & 3);
                    uint8_t *rowp = dst + (c >> 2) * kKVHalf + row * 128;
                    *reinterpret_cast<uint4 *>(rowp + ((q ^ (row & 7)) << 4)) = lo;
                    *reinterpret_cast<uint4 *>(rowp + (((q + 1) ^ (row & 7)) << 4)) = hi;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_FULL(sl)));
            }
            Lbase += 2 * it.n_kv;
            ++npipe;
        }
    }

    // ---- teardown: every MMA has completed before TMEM is released
    pdl_trigger();
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
                          ((q_dtype == DT_BF16 || q_dtype == DT_FP16 || q_dtype == DT_E4M3) && kv_dtype == DT_E4M3);
    if (!ok_types) return false;
    if (G <= 0 || G > 128 || (128 % G) != 0) return false;
    return true;
}

int tc_rows_per_cta() { return 2 * kBM; }

template <bool MMA_BF16, bool OUT_BF16, bool FP8, bool Q8 = false>
static cudaError_t launch_tc(const TcParams &tp, const CUtensorMap &qmap, const CUtensorMap &kmap,
                             const CUtensorMap &vmap, dim3 grid, cudaStream_t stream) {
    using Lay = TcLayout<FP8, Q8>;
    auto kern = fwd_tc_kernel<MMA_BF16, OUT_BF16, FP8, Q8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, grid, dim3(Lay::kThreads), Lay::kSmemBytes, stream, tp, qmap, kmap, vmap);
}

cudaError_t launch_fwd_tc(const FwdParams &f, int q_dtype, int kv_dtype, int64_t T, int num_sms,
                          cudaStream_t stream) {
    if (!f.sched) return cudaErrorInvalidValue;
    TcParams tp{};
    tp.f = f;
    tp.kv_rows = gcd_int(f.bs, kBN);
    const bool q16 = q_dtype == DT_FP16;
    const bool q8 = q_dtype == DT_E4M3;
    const bool fp8 = kv_dtype == DT_E4M3;
    CUtensorMap qmap, kmap, vmap;
    // Q viewed as [T][Hq][D]: box = 64 columns (16-bit) or all 128 bytes
    // (e4m3) x G heads x (128 / G) tokens, 128-byte swizzle
    if (q8 ? !encode_3d_u8(&qmap, f.q, kD, (uint64_t)f.Hq, (uint64_t)T, (uint64_t)kD, (uint64_t)f.q_stride, kD,
                           (uint32_t)f.G, (uint32_t)(kBM / f.G), true)
           : !encode_3d_bf16(&qmap, f.q, q16, kD, (uint64_t)f.Hq, (uint64_t)T, (uint64_t)kD * 2,
                             (uint64_t)f.q_stride * 2, 64, (uint32_t)f.G, (uint32_t)(kBM / f.G)))
        return cudaErrorInvalidValue;
    // caches viewed as [num_blocks * bs][Hkv][D]: box = 1 head x R rows and
    // 64 columns (16-bit, swizzled) or all 128 bytes of a row (e4m3)
    const uint64_t nslots = (uint64_t)f.num_blocks * f.bs;
    const uint32_t R = (uint32_t)tp.kv_rows;
    if (fp8) {
        // (e4m3 q: K swizzled for the tensor core, which reads it staged)
        if (!encode_3d_u8(&kmap, f.k_cache, kD, (uint64_t)f.Hkv, nslots, (uint64_t)kD, (uint64_t)f.Hkv * kD, kD, 1, R,
                          q8) ||
            !encode_3d_u8(&vmap, f.v_cache, kD, (uint64_t)f.Hkv, nslots, (uint64_t)kD, (uint64_t)f.Hkv * kD, kD, 1, R))
            return cudaErrorInvalidValue;
    } else {
        if (!encode_3d_bf16(&kmap, f.k_cache, q16, kD, (uint64_t)f.Hkv, nslots, (uint64_t)kD * 2,
                            (uint64_t)f.Hkv * kD * 2, 64, 1, R) ||
            !encode_3d_bf16(&vmap, f.v_cache, q16, kD, (uint64_t)f.Hkv, nslots, (uint64_t)kD * 2,
                            (uint64_t)f.Hkv * kD * 2, 64, 1, R))
            return cudaErrorInvalidValue;
    }
    // persistent: one CTA per SM, never more CTAs than the class can have items
    const long long max_items = (long long)f.n_row_blocks * f.nsplit * f.Hkv * f.B;
    dim3 grid((unsigned)std::max(1LL, std::min<long long>(num_sms, max_items)));
    if (q8)   // e4m3 q and cache: S on e4m3 MMAs, P V on fp16 (V widened); bf16 output
        return launch_tc<false, true, true, true>(tp, qmap, kmap, vmap, grid, stream);
    if (fp8) {
        // e4m3 caches: fp16 MMAs (the widening is exact); output in q's type
        return q16 ? launch_tc<false, false, true>(tp, qmap, kmap, vmap, grid, stream)
                   : launch_tc<false, true, true>(tp, qmap, kmap, vmap, grid, stream);
    }
    // 16-bit caches run on fwd_tc2_kernel (tc2_supported covers every shape
    // this kernel would take)
    return cudaErrorInvalidValue;
}

}  // namespace attn
