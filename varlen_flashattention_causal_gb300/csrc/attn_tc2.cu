// attn_tc2.cu -- the rows-heavy side of the hot path (prefill and chunks
// above 64 packed rows, 16-bit q and cache, head size 128) on pairs of SMs.
//
// Two CTAs of a cluster run every tensor-core MMA together (tcgen05
// .cta_group::2, M = 256): each CTA holds its own 128-row Q tile and half of
// every K and V tile, and one thread of the even CTA issues the MMAs for
// both.  Per 128-key tile:
//   S = Q K^T    A = Q (each CTA its 128 rows, shared memory), B = K split
//                along the keys: each CTA loads 64 keys x 128 dims
//   O += P V     A = P (each CTA its 128 rows, bf16/fp16 in TMEM over its S),
//                B = V split along the head dimension: each CTA loads 128
//                keys x 64 dims
// so each SM reads half of every K/V tile from HBM and feeds the tensor core
// 96 bytes of shared memory per clock at the full MMA rate (a single SM with
// two Q tiles and 64-key tiles needs more than its 128 B/clk for the S MMA).
// TMEM per CTA: three S buffers (3 x 128 columns) and O (128 columns).  The
// issuer runs S two tiles ahead of P V -- S(j), then O += P(j-2) V -- so the
// softmax of a tile has two S MMAs' time to publish P before the tensor
// core needs it.
//
// Work item, schedule, masking and the online softmax are those of the
// single-SM kernel (attn_tc.cu): an item is one request x one KV head x 256
// packed rows (the pair's two Q tiles) x one KV segment; pairs are persistent
// and draw items from the call's ticket counter; keys are masked from local
// positions with the bottom-right alignment of "vLLM 中 Attention Kernel 如何
// 并行处理多个请求" sec. 10, only on tiles that are not full (sec. 4); O is
// rescaled only when a row's maximum grows by more than 2^8.
//
// Roles (12 warps in each CTA of the pair):
//   warp 0      even CTA: scheduler (publishes every item to both CTAs'
//               two-entry rings) and TMA producer of its halves; odd CTA:
//               reads the items and loads its halves
//   warp 1      both: TMEM allocation for the pair; even CTA: issues S = Q K^T
//               (one thread); odd CTA: forwards the completion of its Q and K
//               loads to barriers of the even CTA, so the S issuer knows both
//               halves have landed
//   warp 10     even CTA: issues O += P V (one thread).  Two issuing warps:
//               a warp issuing tcgen05 MMAs is held about 100 cycles per MMA,
//               more than an M = 256 MMA takes, so one issuer would starve
//               the tensor core; S(j) may run ahead of O += P(j-1) V, and
//               the S buffer of tile j is reused once O += P(j-3) V is done
//   warp 11     both: V gate -- waits for each of the CTA's V halves, zeroes
//               its rows past the segment end on a segment's last tile, and
//               reports the half ready to the even CTA's P V issuer
//   warps 2-9   softmax and epilogue of the CTA's own 128 rows in two
//               groups: warps 2-5 take keys 0-63 of every tile and head dims
//               0-63 of O, warps 6-9 keys 64-127 and dims 64-127, one thread
//               per row in each; the groups trade their row maxima every tile
//               and their row sums every item through shared memory, and
//               report each P (and each read-out of O) to barriers of the
//               even CTA
// Every wait is bounded (2 s, then ERR_TIMEOUT and an orderly teardown); the
// CTAs of a pair leave together through a cluster barrier, after the even CTA
// has drained its MMAs, so no MMA or remote arrive touches a CTA that left.
#include "common.cuh"
#include "sm100.cuh"
#include "tma_host.h"

#include <algorithm>
#include <atomic>

namespace attn {

using namespace sm100;

namespace {

constexpr int kPM = 128;                                // rows per CTA (the pair: 256)
constexpr int kPN = 128;                                // keys per K/V tile
constexpr int kPD = 128;                                // head size
constexpr uint32_t kPQBytes = kPM * kPD * 2;            // one Q tile, 32 KB
constexpr uint32_t kPQHalf = kPM * 128;                 // 64 columns of a Q tile, 16 KB
constexpr uint32_t kPSlot = 16384;                      // a K half (64 keys) or a V half (64 dims)
constexpr uint32_t kPKHalf = 64 * 128;                  // 64 columns of a K half, 8 KB
constexpr int kPSlots = 8;                              // ring of K/V halves (four tiles)
constexpr uint32_t kPOffQ = 0;                          // two Q buffers (by item parity)
constexpr uint32_t kPOffKV = kPOffQ + 2 * kPQBytes;
constexpr uint32_t kPOffBar = kPOffKV + kPSlots * kPSlot;
constexpr uint32_t kPOffMisc = kPOffBar + 8 * 64;
constexpr uint32_t kPOffX = kPOffMisc + 128;           // softmax exchange: row maxima, row sums
constexpr uint32_t kPSmem = kPOffX + 3 * 1024 + 1024;    // + alignment slack
constexpr int kPThreads = 384;
constexpr int kPConsumersEven = 11;                     // warps 1-11 read the item ring
constexpr int kPConsumersOdd = 11;                      // warps 0-9 and 11
constexpr float kPRescale = 8.0f;                       // log2 units
constexpr uint16_t kPairMask = 3;
static_assert(kPSmem <= 232448, "shared memory per CTA");

// TMEM columns: S buffer b (three, by tile index mod 3), then O
constexpr int kPSBufs = 3;
__device__ __forceinline__ uint32_t pcol_s(int b) { return (uint32_t)b * 128u; }
constexpr uint32_t kPColO = 384;

struct PItem {
    int r, kvh, rb, s;              // request, KV head, row block (256 packed rows), KV segment
    int q_start, q_len, kv_len;
    int row0, row_end;              // packed rows [row0, row_end) of the pair
    int ctx, kv_lo, kv_hi, n_kv;    // keys [kv_lo, kv_hi) in n_kv tiles of 128
};

__device__ __forceinline__ void pderive(const FwdParams &p, PItem &it) {
    const int rows = it.q_len * p.G;
    it.row0 = it.rb * 2 * kPM;
    it.row_end = min(it.row0 + 2 * kPM, rows);
    it.ctx = it.kv_len - it.q_len;
    const int i_min = it.row0 / p.G, i_max = (it.row_end - 1) / p.G;
    int kv_end = it.kv_len;
    if (p.causal) kv_end = min(it.kv_len, it.ctx + i_max + 1);
    if (p.window_right >= 0) kv_end = (int)min((long long)kv_end, (long long)it.ctx + i_max + p.window_right + 1);
    // (rounded down to 64 keys: a multiple of every page-load height)
    const int kv_beg = (p.window_left >= 0) ? (max(0, it.ctx + i_min - p.window_left) & ~63) : 0;
    const long long lo = (long long)kv_beg + (long long)it.s * p.split_chunk;
    it.kv_lo = (int)min(lo, (long long)INT_MAX);
    it.kv_hi = (int)min((long long)kv_end, lo + p.split_chunk);
    it.n_kv = it.kv_hi > it.kv_lo ? (it.kv_hi - it.kv_lo + kPN - 1) / kPN : 0;
}

__device__ __forceinline__ float pfmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// whole-warp bounded wait: every lane polls (no divergent branch around the
// wait), and the warp agrees on the outcome, so every lane takes the same
// path into the warp-collective tcgen05 instructions after it.  `cluster`:
// with cluster-scope acquire, for the item ring whose entries the even CTA
// writes into the odd CTA's shared memory
__device__ __forceinline__ bool pwarp_wait(uint32_t bar, uint32_t parity, volatile int *abort, bool cluster = false) {
    const bool ok = cluster ? mbar_wait_cl(bar, parity, abort) : mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, ok) != 0;
}

}  // namespace

struct Tc2Params {
    FwdParams f;
    int kv_rows;                  // rows per TMA page load: gcd(block_size, 64)
};

// BF16: operand and output type bf16 (else fp16)
template <bool BF16>
__global__ void __launch_bounds__(kPThreads, 1)
    fwd_tc2_kernel(const __grid_constant__ Tc2Params tp, const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
    const FwdParams &p = tp.f;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *sm = smem_raw + (sbase - raw);
    auto bar = [&](int i) { return sbase + kPOffBar + 8u * (uint32_t)i; };
    // barriers (each CTA has all of them at the same offsets; the comments
    // say which CTA uses them and who arrives)
    constexpr int B_Q = 0;                                    // own Q landed (TMA)
    auto B_FULL = [](int s) { return 1 + s; };                // own K/V half in slot s landed (TMA)
    auto B_EMPTY = [](int s) { return 1 + kPSlots + s; };     // slot s read by the pair's MMAs (commit)
    constexpr int kB = 1 + 2 * kPSlots;
    constexpr int B_PQ = kB;                                  // even: the odd CTA's Q landed (forwarded)
    auto B_PFULLS = [](int s) { return kB + 1 + s; };         // even: the odd CTA's slot s landed
    constexpr int kB2 = kB + 1 + kPSlots;
    // per S buffer b (tile index mod 3; phase = tile index / 3)
    auto B_SFULL = [](int b) { return kB2 + b; };             // S buffer b written (commit, both CTAs)
    auto B_PFULL = [](int b) { return kB2 + 3 + b; };         // even: P over buffer b written (8 warps)
    auto B_ODONE = [](int b) { return kB2 + 6 + b; };         // O += P(buffer b) V done (commit, both)
    constexpr int kB3 = kB2 + 3 * kPSBufs;
    constexpr int B_OFREE = kB3;                              // even: both CTAs read O out (8 warps)
    constexpr int B_QFREE = kB3 + 1;                          // the item's S MMAs done with Q (commit, both)
    auto B_ITEMF = [](int i) { return kB3 + 2 + i; };         // ring entry i written (both)
    auto B_ITEME = [](int i) { return kB3 + 4 + i; };         // even: entry i read by every consumer warp
    constexpr int B_DRAIN = kB3 + 6;                          // both issuers' MMAs are done (commits, both)
    // the two softmax warps of TMEM lane quarter q (one per group, the same
    // rows) posted their tile maxima, by tile parity i
    auto B_XMAX = [](int i, int q) { return kB3 + 13 + kPSlots + 4 * i + q; };
    constexpr int B_XSUM = kB3 + 9;                           // both groups posted row sums (8 warps)
    // Q is double-buffered (buffer = parity of the item's index among items
    // with keys): the next item's Q loads while the current item's S MMAs run
    auto BQ = [](int q) { return q ? kB3 + 10 : B_Q; };       // own Q buffer q landed (TMA)
    auto BPQ = [](int q) { return q ? kB3 + 11 : B_PQ; };     // even: the odd CTA's Q buffer q landed
    auto BQFREE = [](int q) { return q ? kB3 + 12 : B_QFREE; };   // S MMAs done with Q buffer q (commit, both)
    // per K/V slot s holding a V half: both CTAs' halves landed (and, on a
    // segment's last tile, zeroed past its end) -- one arrival from each
    // CTA's V gate warp on the even CTA's copy
    auto B_VREADY = [](int s) { return kB3 + 13 + s; };
    constexpr int kNumBars = kB3 + 13 + kPSlots + 8;
    static_assert(kNumBars <= 64, "barrier area");
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + kPOffMisc);
    uint32_t *taddr_slot = reinterpret_cast<uint32_t *>(sm + kPOffMisc + 8);
    volatile int *never = reinterpret_cast<volatile int *>(sm + kPOffMisc + 16);
    volatile int *ring = reinterpret_cast<volatile int *>(sm + kPOffMisc + 32);   // 2 entries x 8 ints

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.G;
    const uint32_t rank = cluster_ctarank();
    const bool even = rank == 0;
    const uint32_t peer = rank ^ 1u;
    // the even CTA's copy of a barrier (for arrivals from either CTA)
    auto even_bar = [&](int i) { return mapa_shared(bar(i), 0); };

    if (tid == 0) {
        *abort_flag = 0;
        *never = 0;
        mbar_init(bar(B_Q), 1);
        for (int s = 0; s < kPSlots; ++s) {
            mbar_init(bar(B_FULL(s)), 1);
            mbar_init(bar(B_EMPTY(s)), 1);
            mbar_init(bar(B_PFULLS(s)), 1);
        }
        mbar_init(bar(B_PQ), 1);
        for (int b = 0; b < kPSBufs; ++b) {
            mbar_init(bar(B_SFULL(b)), 1);
            mbar_init(bar(B_PFULL(b)), 16);
            mbar_init(bar(B_ODONE(b)), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_ITEMF(i)), 1);
            mbar_init(bar(B_ITEME(i)), (uint32_t)(kPConsumersEven + kPConsumersOdd));
        }
        mbar_init(bar(B_OFREE), 16);
        for (int i = 0; i < 8; ++i) mbar_init(bar(B_XMAX(i >> 2, i & 3)), 2);
        mbar_init(bar(B_XSUM), 8);
        mbar_init(bar(BQ(1)), 1);
        mbar_init(bar(BPQ(1)), 1);
        mbar_init(bar(BQFREE(1)), 1);
        mbar_init(bar(B_QFREE), 1);
        mbar_init(bar(B_DRAIN), 2);
        for (int s = 0; s < kPSlots; ++s) mbar_init(bar(B_VREADY(s)), 2);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc2(sbase + kPOffMisc + 8, 512);
        tmem_relinquish2();
    }
    tc_fence_before();
    // both CTAs' barriers are initialised (and TMEM allocated) before either
    // arrives on the other's barriers
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *taddr_slot;
    pdl_wait();

    // consumer warps: take item k from the local ring; false on abort
    auto read_item = [&](int k, PItem &it) -> bool {
        if (!pwarp_wait(bar(B_ITEMF(k & 1)), (k >> 1) & 1, abort_flag, true)) return false;
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
        if (lane == 0) mbar_arrive_cluster(even_bar(B_ITEME(k & 1)));
        if (it.r >= 0) pderive(p, it);
        return true;
    };

    if (warp == 0) {
        // =================================== scheduler (even) and TMA producer
        const int R = tp.kv_rows;
        const int PT = kPN / R;                  // page loads per 128-key tile (2, 4 or 8)
        const long long P = gridDim.x / 2;      // pairs
        const long long pair = blockIdx.x / 2;
        int sc_chunk = -32;
        long long sc_base = 0, sc_total = 0, sc_incl = 0, sc_cnt = 0;
        int sc_q0 = 0, sc_ql = 0, sc_kv = 0, sc_nrb = 0;
        int npipe = 0, Lbase = 0, issued = -1;
        bool ok = true;
        if (lane == 0) {
            tma_prefetch(&qmap);
            tma_prefetch(&kmap);
            tma_prefetch(&vmap);
        }
        for (int k = 0; ok; ++k) {
            PItem it{};
            it.r = -1;
            if (even) {
                // item k of this pair: the pair index, then tickets
                long long v = pair;
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
                            sc_nrb = (rows + 2 * kPM - 1) / (2 * kPM);
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
                // publish to both rings: entry k & 1 is free once every consumer
                // warp of both CTAs has read item k - 2
                if (k >= 2) ok = pwarp_wait(bar(B_ITEME(k & 1)), ((k >> 1) - 1) & 1, abort_flag);
                if (!ok) break;
                if (lane == 0) {
                    const int vals[7] = {it.r, it.kvh, it.rb, it.s, it.q_start, it.q_len, it.kv_len};
                    const uint32_t e_local = smem_u32(const_cast<int *>(ring + (k & 1) * 8));
                    const uint32_t e_peer = mapa_shared(e_local, peer);
                    volatile int *e = ring + (k & 1) * 8;
#pragma unroll
                    for (int i = 0; i < 7; ++i) {
                        e[i] = vals[i];
                        st_shared_cluster_u32(e_peer + 4u * i, (uint32_t)vals[i]);
                    }
                    // the entry's remote stores are visible before the odd CTA's
                    // consumers see the barrier phase
                    fence_acq_rel_cluster();
                    mbar_arrive(bar(B_ITEMF(k & 1)));
                    mbar_arrive_cluster(mapa_shared(bar(B_ITEMF(k & 1)), peer));
                }
                __syncwarp();
                if (it.r < 0) break;
                pderive(p, it);
            } else {
                ok = read_item(k, it);
                if (!ok || it.r < 0) break;
            }
            if (it.n_kv == 0) continue;

            // ---- own Q tile (rows row0 + 128 rank ..) into buffer npipe & 1,
            // once the pair's S MMAs are done with the item two back
            const int qb = npipe & 1;
            if (npipe >= 2) ok = pwarp_wait(bar(BQFREE(qb)), ((npipe >> 1) - 1) & 1, abort_flag);
            if (!ok) break;
            if (lane == 0) {
                mbar_expect_tx(bar(BQ(qb)), kPQBytes);
                const int tok = it.q_start + (it.row0 + (int)rank * kPM) / G;
                for (int h = 0; h < 2; ++h)
                    tma_load_3d(sbase + kPOffQ + qb * kPQBytes + h * kPQHalf, &qmap, h * 64, it.kvh * G, tok,
                                bar(BQ(qb)));
            }
            __syncwarp();
            ++npipe;

            // ---- K/V halves, page by page through the block table (32 page
            // coordinates per lane batch, the next batch requested ahead)
            const int64_t bt_base = (int64_t)it.r * p.bt_stride;
            const int total_pages = it.n_kv * PT;
            const int kv_lo = it.kv_lo, kv_hi = it.kv_hi;
            auto page_coord = [&](int g) -> int {
                if (g >= total_pages) return -1;
                const int tok = kv_lo + g * R;
                if (tok >= kv_hi) return -1;
                int blk = p.block_table[bt_base + tok / p.bs];
                if ((unsigned)blk >= (unsigned)p.num_blocks) {
                    raise_error(p.err, ERR_BLOCK_ID);
                    blk = 0;
                }
                return blk * p.bs + tok % p.bs;
            };
            int batch = 0;
            int cur = page_coord(lane);
            int nxt = page_coord(32 + lane);
            for (int j = 0; j < it.n_kv && ok; ++j) {
                const int g0 = j * PT;
                if (g0 >= batch + 32) {
                    batch += 32;
                    cur = nxt;
                    nxt = page_coord(batch + 32 + lane);
                }
                for (int kv = 0; kv < 2 && ok; ++kv) {
                    const int L = Lbase + 2 * j + kv;
                    const int slot = L % kPSlots;
                    // K: this CTA's 64 keys of the tile (pages PT/2 * rank ..);
                    // V: all 128 keys of the tile, this CTA's 64 head dims
                    const int npg = kv ? PT : PT / 2;
                    const int pg0 = kv ? 0 : (int)rank * (PT / 2);
                    const int coord = __shfl_sync(0xffffffffu, cur, (g0 - batch + pg0 + (lane < npg ? lane : 0)) & 31);
                    const int mine = lane < npg ? coord : -1;
                    const int nvalid = __popc(__ballot_sync(0xffffffffu, mine >= 0));
                    if (L >= kPSlots) ok = pwarp_wait(bar(B_EMPTY(slot)), ((L / kPSlots) - 1) & 1, abort_flag);
                    if (!ok) break;
                    const uint32_t dst = sbase + kPOffKV + slot * kPSlot + lane * R * 128;
                    if (lane == 0) mbar_expect_tx(bar(B_FULL(slot)), (uint32_t)nvalid * R * 128 * (kv ? 1 : 2));
                    __syncwarp();
                    if (mine >= 0) {
                        if (kv) {
                            tma_load_3d(dst, &vmap, 64 * (int)rank, it.kvh, mine, bar(B_FULL(slot)));
                        } else {
                            tma_load_3d(dst, &kmap, 0, it.kvh, mine, bar(B_FULL(slot)));
                            tma_load_3d(dst + kPKHalf, &kmap, 64, it.kvh, mine, bar(B_FULL(slot)));
                        }
                    }
                    issued = L;
                }
            }
            Lbase += 2 * it.n_kv;
        }
        // drain: every load issued has landed before the CTA leaves
        if (lane == 0) {
            for (int L = max(0, issued - kPSlots + 1); L <= issued; ++L)
                mbar_wait(bar(B_FULL(L % kPSlots)), (L / kPSlots) & 1, never);
            for (int n = max(0, npipe - 2); n < npipe; ++n) mbar_wait(bar(BQ(n & 1)), (n >> 1) & 1, never);
        }
    } else if (warp == 1 && even) {
        // ================================== S = Q K^T issuer of the pair (one thread)
        const uint32_t idS = idesc_f16(BF16, 2 * kPM, kPN, false, false);
        const uint64_t dQb[2] = {sdesc_sw128(sbase + kPOffQ, 16, 1024),
                                 sdesc_sw128(sbase + kPOffQ + kPQBytes, 16, 1024)};
        const uint64_t dKV = sdesc_sw128(sbase + kPOffKV, 16, 1024);
        int npipe = 0, Lbase = 0, jx = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            PItem it;
            ok = read_item(k, it);
            if (!ok || it.r < 0) break;
            if (it.n_kv == 0) continue;
            const int n_kv = it.n_kv;
            const int qb = npipe & 1;
            const uint64_t dQ = dQb[qb];
            if (lane == 0) {
                ok = mbar_wait(bar(BQ(qb)), (npipe >> 1) & 1, abort_flag);
                if (ok) ok = mbar_wait(bar(BPQ(qb)), (npipe >> 1) & 1, abort_flag);
                for (int j = 0; j < n_kv && ok; ++j) {
                    const int LK = Lbase + 2 * j;        // load index of K_j
                    const int jg = jx + j;
                    const int sk = LK % kPSlots;
                    ok = mbar_wait(bar(B_FULL(sk)), (LK / kPSlots) & 1, abort_flag);
                    if (ok) ok = mbar_wait(bar(B_PFULLS(sk)), (LK / kPSlots) & 1, abort_flag);
                    // buffer jg mod 3 holds P(jg - 3) until its P V is done
                    if (ok && jg >= kPSBufs)
                        ok = mbar_wait(bar(B_ODONE((jg - kPSBufs) % kPSBufs)), ((jg - kPSBufs) / kPSBufs) & 1,
                                       abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t d = tmem + pcol_s(jg % kPSBufs);
#pragma unroll
                    for (int kk = 0; kk < kPD / 16; ++kk)
                        umma_ss2(d, dQ + (((kk >> 2) * kPQHalf + (kk & 3) * 32) >> 4),
                                 dKV + ((sk * kPSlot + (kk >> 2) * kPKHalf + (kk & 3) * 32) >> 4), idS,
                                 kk > 0 ? 1u : 0u);
                    umma_commit2(bar(B_SFULL(jg % kPSBufs)), kPairMask);
                    umma_commit2(bar(B_EMPTY(sk)), kPairMask);
                    if (j == n_kv - 1) umma_commit2(bar(BQFREE(qb)), kPairMask);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            Lbase += 2 * n_kv;
            ++npipe;
            jx += n_kv;
        }
        // the pair's MMAs are all done (also on the odd CTA's barrier) before
        // either CTA leaves or frees TMEM
        if (lane == 0) {
            umma_commit2(bar(B_DRAIN), kPairMask);
            mbar_wait(bar(B_DRAIN), 0, never);
        }
    } else if (warp == 10) {
        // ============================ O += P V issuer of the pair (even CTA, one thread)
        const uint32_t idO = idesc_f16(BF16, 2 * kPM, kPD, false, true);
        const uint64_t dV = sdesc_sw128(sbase + kPOffKV, kPSlot, 1024);
        const uint32_t tO = tmem + kPColO;
        int Lbase = 0, jx = 0, ax = 0;
        bool ok = true;
        for (int k = 0; ok && even; ++k) {
            PItem it;
            ok = read_item(k, it);
            if (!ok || it.r < 0) break;
            if (it.n_kv == 0) continue;
            const int n_kv = it.n_kv;
            if (lane == 0) {
                for (int j = 0; j < n_kv && ok; ++j) {
                    const int LV = Lbase + 2 * j + 1;    // load index of V_j
                    const int jg = jx + j;
                    const int sv = LV % kPSlots;
                    // V_j: both CTAs' halves landed and tail-zeroed (V gate warps)
                    ok = mbar_wait_cl(bar(B_VREADY(sv)), (LV / kPSlots) & 1, abort_flag);
                    if (ok) ok = mbar_wait(bar(B_PFULL(jg % kPSBufs)), (jg / kPSBufs) & 1, abort_flag);
                    // the item's first P V overwrites O: both CTAs must have read
                    // the previous item's O out
                    if (ok && j == 0 && ax > 0) ok = mbar_wait(bar(B_OFREE), (ax - 1) & 1, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t a = tmem + pcol_s(jg % kPSBufs);
#pragma unroll
                    for (int kk = 0; kk < kPN / 16; ++kk)
                        umma_ts2(tO, a + kk * 8, dV + ((sv * kPSlot + kk * 2048) >> 4), idO,
                                 (j == 0 && kk == 0) ? 0u : 1u);
                    umma_commit2(bar(B_ODONE(jg % kPSBufs)), kPairMask);
                    umma_commit2(bar(B_EMPTY(sv)), kPairMask);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            Lbase += 2 * n_kv;
            jx += n_kv;
            ++ax;
        }
        if (even && lane == 0) {
            umma_commit2(bar(B_DRAIN), kPairMask);
            mbar_wait(bar(B_DRAIN), 0, never);
        }
    } else if (warp == 1) {
        // ======================= odd CTA: forward own load completions to the even CTA
        int npipe = 0, Lbase = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            PItem it;
            ok = read_item(k, it);
            if (!ok || it.r < 0) break;
            if (it.n_kv == 0) continue;
            if (lane == 0) {
                ok = mbar_wait(bar(BQ(npipe & 1)), (npipe >> 1) & 1, abort_flag);
                if (ok) mbar_arrive_cluster(even_bar(BPQ(npipe & 1)));
                // (K loads only: the V gate warps report the V halves)
                for (int L = Lbase; L < Lbase + 2 * it.n_kv && ok; L += 2) {
                    ok = mbar_wait(bar(B_FULL(L % kPSlots)), (L / kPSlots) & 1, abort_flag);
                    if (ok) mbar_arrive_cluster(even_bar(B_PFULLS(L % kPSlots)));
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            Lbase += 2 * it.n_kv;
            ++npipe;
        }
        if (lane == 0) mbar_wait(bar(B_DRAIN), 0, never);
    } else if (warp == 11) {
        // ============ V gate (both CTAs): each V half of the CTA, once it has
        // landed; on a segment's last tile its rows past the segment end are
        // zeroed first (P is exactly 0 there, but the rows may hold anything --
        // unwritten cache rows, pages not loaded -- and 0 * NaN is NaN).  Both
        // SMs' tensor cores read the half, the peer's through the cluster, so
        // zeroed rows are published with a proxy fence over all state spaces and
        // cluster-scope ordering (a CTA-scope proxy fence measurably left the
        // peer reading stale rows now and then).  The gate then arrives on the
        // even CTA's B_VREADY, which the P V issuer waits for in place of the
        // load completions.  Off the softmax's path, the fences cost little.
        int Lbase = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            PItem it;
            ok = read_item(k, it);
            if (!ok || it.r < 0) break;
            if (it.n_kv == 0) continue;
            for (int j = 0; j < it.n_kv && ok; ++j) {
                const int L = Lbase + 2 * j + 1;          // load index of V_j
                const int sv = L % kPSlots;
                ok = pwarp_wait(bar(B_FULL(sv)), (L / kPSlots) & 1, abort_flag);
                if (!ok) break;
                const int nvalid = it.kv_hi - (it.kv_lo + j * kPN);   // keys of the tile in the segment
                if (nvalid < kPN) {
                    uint4 *half = reinterpret_cast<uint4 *>(sm + kPOffKV + sv * kPSlot);
                    for (int i = nvalid * 8 + lane; i < kPN * 8; i += 32) half[i] = make_uint4(0, 0, 0, 0);
                    fence_proxy_async_all();
                    fence_acq_rel_cluster();
                    __syncwarp();
                    if (lane == 0) {
                        fence_acq_rel_cluster();
                        mbar_arrive_cluster_release(even_bar(B_VREADY(sv)));
                    }
                } else {
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster_release(even_bar(B_VREADY(sv)));
                }
            }
            Lbase += 2 * it.n_kv;
        }
    } else if (warp >= 2 && warp <= 9) {
        // ============ softmax and epilogue (own rows), in two groups of columns
        const int sg = (warp - 2) >> 2;             // 0: keys / dims 0-63, 1: 64-127
        const int quarter = warp & 3;               // TMEM lane quarter this warp may access
        const int trow = quarter * 32 + lane;       // row within the CTA's Q tile
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_base + kPColO + 64u * sg;   // this group's 64 columns of O
        float *xmax = reinterpret_cast<float *>(sm + kPOffX);         // [tile parity][group][row]
        float *xsum = xmax + 4 * kPM;                                  // [group][row]
        const float vds = p.v_descale;
        const bool capped = p.cap_in > 0.f;
        const float sl2 = capped ? 1.f : p.scale_log2;
        const uint32_t pfull_even[kPSBufs] = {even_bar(B_PFULL(0)), even_bar(B_PFULL(1)), even_bar(B_PFULL(2))};
        const uint32_t ofree_even = even_bar(B_OFREE);
        int Lbase = 0, jx = 0, ni = 0;              // ni: items with keys so far
        bool ok = true;
        for (int k = 0; ok; ++k) {
            PItem it;
            ok = read_item(k, it);
            if (!ok || it.r < 0) break;
            const int prow = it.row0 + (int)rank * kPM + trow;   // packed row within the request
            const bool row_ok = prow < it.row_end;
            if (it.n_kv == 0) {
                // no key for any row of the item in this segment: empty state (a
                // sink alone, in segment 0), written by group 0
                if (row_ok && sg == 0) {
                    const int64_t tok = it.q_start + prow / G;
                    const int h = it.kvh * G + prow % G;
                    const float zl = (p.sinks && it.s == 0) ? p.sinks[h] : -INFINITY;
                    if (p.partials) {
                        const int64_t slot = (tok * p.Hq + h) * p.part_stride + it.s;
                        p.part_lse[slot] = zl;
                        if (zl != -INFINITY)
                            for (int d = 0; d < kPD; ++d) p.part_o[slot * kPD + d] = 0.f;
                    } else {
                        if (p.lse) p.lse[tok * p.Hq + h] = zl;
                        uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(p.out) +
                                                             (tok * p.out_stride + (int64_t)h * kPD) * 2);
                        for (int c = 0; c < kPD / 8; ++c) o[c] = make_uint4(0, 0, 0, 0);
                    }
                }
                continue;
            }
            const int n_kv = it.n_kv, kv_lo = it.kv_lo, kv_hi = it.kv_hi;
            const int qi = prow / G;                    // local query index
            long long lim_ll = p.causal ? (long long)it.ctx + qi : (long long)INT_MAX;
            if (p.window_right >= 0) lim_ll = min(lim_ll, (long long)it.ctx + qi + p.window_right);
            const int lim = (int)lim_ll;                // last visible key of this row
            const int lo_key = (p.window_left >= 0) ? it.ctx + qi - p.window_left : INT_MIN;
            float m_ref = -INFINITY;                    // reference maximum (log2 units), same in both groups
            float l = 0.f;                              // this group's part of the row sum
            // query range of this CTA's Q tile, for the tile classification
            const int trow0 = it.row0 + (int)rank * kPM;
            const int tq_lo = trow0 / G;
            const int tq_hi = trow0 < it.row_end ? (min(trow0 + kPM, it.row_end) - 1) / G + 1 : tq_lo;
            const int nlim = min(kv_hi - 1, lim);
            for (int j = 0; j < n_kv && ok; ++j) {
                const int n0 = kv_lo + j * kPN;
                const int g0 = n0 + 64 * sg;            // first key of this group's columns
                const int jg = jx + j;
                const int b = jg % kPSBufs;
                const uint32_t tS = tmem + lane_base + pcol_s(b);
                const bool need_mask =
                    (n0 + kPN > kv_hi) || (p.causal && tile_kind(tq_lo, tq_hi, n0, n0 + kPN, it.ctx) != 1) ||
                    (p.window_left >= 0 && n0 < it.ctx + tq_hi - 1 - p.window_left) ||
                    (p.window_right >= 0 && (long long)n0 + kPN - 1 > (long long)it.ctx + tq_lo + p.window_right);
                ok = pwarp_wait(bar(B_SFULL(b)), (jg / kPSBufs) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                uint32_t v[64];
                {
                    uint32_t (&v0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
                    uint32_t (&v1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
                    tmem_ld32(tS + 64 * sg, v0);
                    tmem_ld32(tS + 64 * sg + 32, v1);
                    tmem_wait_ld();
                }
                if (capped) {
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        v[e] = __float_as_uint(p.cap_out * tanh_ex2(__uint_as_float(v[e]) * p.cap_in));
                }
                // this row sees keys g0 + e_lo .. g0 + nv - 1 of the group's
                // columns (selects, no per-row branch: need_mask is the same for
                // the whole warp)
                if (need_mask) {
                    const int nv = max(0, min(64, nlim - g0 + 1));
                    const int e_lo = (p.window_left >= 0) ? min(64, max(0, lo_key - g0)) : 0;
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        v[e] = (e >= nv || e < e_lo) ? __float_as_uint(-INFINITY) : v[e];
                }
                // this group's row maximum (three-input max, four chains), then
                // the other group's through shared memory
                float mx4[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) mx4[c] = fmaxf(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]));
#pragma unroll
                for (int b8 = 8; b8 < 64; b8 += 8) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        mx4[c] = pfmax3(mx4[c], __uint_as_float(v[b8 + 2 * c]), __uint_as_float(v[b8 + 2 * c + 1]));
                }
                const float mxl = pfmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
                xmax[((jg & 1) * 2 + sg) * kPM + trow] = mxl;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_XMAX(jg & 1, quarter)));
                ok = pwarp_wait(bar(B_XMAX(jg & 1, quarter)), (jg >> 1) & 1, abort_flag);
                if (!ok) break;
                const float mx = fmaxf(mxl, xmax[((jg & 1) * 2 + (sg ^ 1)) * kPM + trow]) * sl2;
                const bool bump = mx > m_ref + kPRescale;
                const bool corr = bump && m_ref != -INFINITY;
                const float m_new = bump ? mx : m_ref;
                const float alpha = corr ? ex2(m_ref - m_new) : 1.f;
                const float base = (m_new == -INFINITY) ? 0.f : m_new;
                m_ref = m_new;
                // P = 2^(s * scale - m) on packed fp32 pairs, row sum alongside
                uint32_t pk[32];
                float2 rs2[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) rs2[c] = make_float2(0.f, 0.f);
                const float2 sc2 = make_float2(sl2, sl2), nb2 = make_float2(-base, -base);
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const float2 x2 =
                        __ffma2_rn(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sc2, nb2);
                    const float p0 = ex2(x2.x);
                    const float p1 = ex2(x2.y);
                    rs2[(e >> 1) & 3] = __fadd2_rn(rs2[(e >> 1) & 3], make_float2(p0, p1));
                    pk[e / 2] = pack2<BF16>(p0, p1);
                }
                const float2 r01 = __fadd2_rn(rs2[0], rs2[1]), r23 = __fadd2_rn(rs2[2], rs2[3]);
                const float2 r03 = __fadd2_rn(r01, r23);
                l = l * alpha + (r03.x + r03.y);
                if (__any_sync(0xffffffffu, corr)) {
                    // O must hold P(j-1) V before it is rescaled (corr implies j > 0);
                    // each group rescales its own 64 columns
                    ok = pwarp_wait(bar(B_ODONE((jg - 1) % kPSBufs)), ((jg - 1) / kPSBufs) & 1, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tO + c * 32, o);
                    }
                }
                // P -> TMEM over the S buffer it came from (packed columns
                // 32 sg .. 32 sg + 31: this group's 64 keys)
                {
                    uint32_t (&p0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&pk[0]);
                    tmem_st32(tS + 32 * sg, p0);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(pfull_even[b]);
            }
            // ---- epilogue: O / l -> out (or the split partials), each group its 64 dims
            if (ok) {
                const int jl = jx + n_kv - 1;
                ok = pwarp_wait(bar(B_ODONE(jl % kPSBufs)), (jl / kPSBufs) & 1, abort_flag);
            }
            if (ok) {
                // the row sum is the two groups' parts
                xsum[sg * kPM + trow] = l;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_XSUM));
                ok = pwarp_wait(bar(B_XSUM), ni & 1, abort_flag);
            }
            if (ok) {
                tc_fence_after();
                l += xsum[(sg ^ 1) * kPM + trow];
                const int64_t tok = it.q_start + qi;
                const int h = it.kvh * G + prow % G;
                float sink_scale = 1.f;
                if (row_ok && p.sinks && it.s == 0 && p.sinks[h] > -INFINITY) {
                    const float z2 = p.sinks[h] * 1.4426950408889634f;
                    const float mn = fmaxf(m_ref, z2);
                    sink_scale = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - mn);
                    l = l * sink_scale + ex2(z2 - mn);
                    m_ref = mn;
                }
                const float inv = l > 0.f ? vds * sink_scale / l : 0.f;
                const float lse_v = l > 0.f ? (m_ref + __log2f(l)) * 0.6931471805599453f : -INFINITY;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + c * 32, o);
                    tmem_wait_ld();
                    if (!row_ok) continue;
                    const int d0 = 64 * sg + c * 32;
                    if (!p.partials) {
                        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(p.out) +
                                                               (tok * p.out_stride + (int64_t)h * kPD + d0) * 2);
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint4 w;
                            w.x = pack2<BF16>(__uint_as_float(o[q4 * 8 + 0]) * inv, __uint_as_float(o[q4 * 8 + 1]) * inv);
                            w.y = pack2<BF16>(__uint_as_float(o[q4 * 8 + 2]) * inv, __uint_as_float(o[q4 * 8 + 3]) * inv);
                            w.z = pack2<BF16>(__uint_as_float(o[q4 * 8 + 4]) * inv, __uint_as_float(o[q4 * 8 + 5]) * inv);
                            w.w = pack2<BF16>(__uint_as_float(o[q4 * 8 + 6]) * inv, __uint_as_float(o[q4 * 8 + 7]) * inv);
                            dst[q4] = w;
                        }
                    } else {
                        float4 *dst = reinterpret_cast<float4 *>(
                            p.part_o + ((tok * p.Hq + h) * p.part_stride + it.s) * kPD + d0);
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            dst[q4] = make_float4(__uint_as_float(o[q4 * 4]) * inv, __uint_as_float(o[q4 * 4 + 1]) * inv,
                                                  __uint_as_float(o[q4 * 4 + 2]) * inv,
                                                  __uint_as_float(o[q4 * 4 + 3]) * inv);
                    }
                }
                if (row_ok && sg == 0) {
                    if (!p.partials) {
                        if (p.lse) p.lse[tok * p.Hq + h] = lse_v;
                    } else {
                        p.part_lse[(tok * p.Hq + h) * p.part_stride + it.s] = lse_v;
                    }
                }
                // O has been read out: the pair may start the next item's P V
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(ofree_even);
            }
            jx += n_kv;
            Lbase += 2 * n_kv;
            ++ni;
        }
    }

    // ---- teardown: the pair's MMAs are done (warp 1 waited for DRAIN in both
    // CTAs) and no thread touches the other CTA after the cluster barrier
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc2(tmem, 512);
    }
    if (tid == 0 && *abort_flag) raise_error(p.err, ERR_TIMEOUT);
}

static int gcd2(int a, int b) {
    while (b) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return a;
}

bool tc2_supported(int D, int q_dtype, int kv_dtype, int G) {
    if (D != kPD) return false;
    if (!((q_dtype == DT_BF16 && kv_dtype == DT_BF16) || (q_dtype == DT_FP16 && kv_dtype == DT_FP16))) return false;
    return G > 0 && G <= 128 && (128 % G) == 0;
}

template <bool BF16>
static cudaError_t launch_tc2_t(const Tc2Params &tp, const CUtensorMap &qmap, const CUtensorMap &kmap,
                                const CUtensorMap &vmap, long long max_items, int num_sms, cudaStream_t stream) {
    auto kern = fwd_tc2_kernel<BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = kPSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    // persistent: as many pairs as can be resident at once (looked up once
    // per device), never more than the class has items
    static std::atomic<int> resident[64];
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int pairs = resident[dev].load(std::memory_order_relaxed);
    if (pairs <= 0) {
        cfg.gridDim = dim3((unsigned)std::max(2, num_sms & ~1));
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
        if (e != cudaSuccess) return e;
        pairs = std::max(1, clusters);
        resident[dev].store(pairs, std::memory_order_relaxed);
    }
    const long long n = std::max(1LL, std::min<long long>(pairs, max_items));
    cfg.gridDim = dim3((unsigned)(2 * n));
    return cudaLaunchKernelEx(&cfg, kern, tp, qmap, kmap, vmap);
}

cudaError_t launch_fwd_tc2(const FwdParams &f, int q_dtype, int64_t T, int num_sms, cudaStream_t stream) {
    if (!f.sched) return cudaErrorInvalidValue;
    Tc2Params tp{};
    tp.f = f;
    tp.kv_rows = gcd2(f.bs, 64);
    const bool q16 = q_dtype == DT_FP16;
    CUtensorMap qmap, kmap, vmap;
    // Q viewed as [T][Hq][D]: box = 64 columns x G heads x (128 / G) tokens
    if (!encode_3d_bf16(&qmap, f.q, q16, kPD, (uint64_t)f.Hq, (uint64_t)T, (uint64_t)kPD * 2, (uint64_t)f.q_stride * 2,
                        64, (uint32_t)f.G, (uint32_t)(kPM / f.G)))
        return cudaErrorInvalidValue;
    // caches viewed as [num_blocks * bs][Hkv][D]: box = R rows x 1 head x 64 columns
    const uint64_t nslots = (uint64_t)f.num_blocks * f.bs;
    const uint32_t R = (uint32_t)tp.kv_rows;
    if (!encode_3d_bf16(&kmap, f.k_cache, q16, kPD, (uint64_t)f.Hkv, nslots, (uint64_t)kPD * 2,
                        (uint64_t)f.Hkv * kPD * 2, 64, 1, R) ||
        !encode_3d_bf16(&vmap, f.v_cache, q16, kPD, (uint64_t)f.Hkv, nslots, (uint64_t)kPD * 2,
                        (uint64_t)f.Hkv * kPD * 2, 64, 1, R))
        return cudaErrorInvalidValue;
    const long long max_items = (long long)f.n_row_blocks * f.nsplit * f.Hkv * f.B;
    return q16 ? launch_tc2_t<false>(tp, qmap, kmap, vmap, max_items, num_sms, stream)
               : launch_tc2_t<true>(tp, qmap, kmap, vmap, max_items, num_sms, stream);
}

}  // namespace attn
