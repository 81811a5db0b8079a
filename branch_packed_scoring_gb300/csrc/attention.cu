// Tree-masked GQA attention over one packed pass (sm_103a, tcgen05 + TMA).
//
// The method ("spinf-serve 0.1.1", PyPI page, "What it does" and "Speed and
// scale"): every question is a branch of the same pass; a branch token attends
// to its own content and causally to its own branch, never to a sibling or to
// another packed input.  The planner encodes that as: key k is visible to the
// rows [k, end[k]), and each scheduled KV tile holds only its own input's keys.
//
// Persistent kernel: one CTA per SM walks a static list of work items, an item
// being one 128-row Q tile of one query head.  Q tiles are taken longest schedule
// first, in rounds over the CTAs with every other round reversed, so the CTAs
// finish together.  Consecutive items are the query heads of one Q tile, so the CTAs
// of a round that share a kv head read its K and V tiles at about the same time (the
// second read comes from L2).  At d_head 256 with two query heads per kv head, an
// item is instead one kv head and a 64-row Q tile, both query heads' 64 rows stacked
// in the MMA's 128 rows: each K/V tile serves both heads, and a 64-row tile meets
// fewer masked keys.  At d_head 128, when a kv group has an even number of query
// heads, CTAs run as cta_group::2 MMA pairs on two heads of one group: the leader
// issues M = 256 products over both CTAs' rows, and each CTA holds half of every K
// tile (64 keys) and V tile (64 columns).  Every CTA loads its own tiles from this
// GPU's memory (no multicast copies).  Warp roles:
//   warp 0      one TMA producer thread for Q (once per item), K and V tiles: it
//               polls the buffers' barriers and issues whichever copy is free first
//               (each tile one 4-D copy of all its 64-column chunks; two K and two V
//               buffers; at d_head 256 outside a cta_group::2 pair the KV tiles are
//               the 64-key halves of the planner's tiles, so that two of each fit)
//   warp 1      TMEM owner and S issuer: S = Q K^T into one of three 128-column
//               (d_head <= 128) or four 64-column (d_head 256) TMEM buffers (SS, fp32)
//   warp 2      PV issuer: O += P V (P read from TMEM, V MN-major from shared
//               memory); two issuing threads, so the tensor core has the other
//               stream's MMAs to run while one thread commits or waits
//   warps 3-10  softmax, two warps per TMEM lane quarter: each thread owns half
//               of one Q row (half of the tile's key columns, D/2 of the O columns):
//               mask, online softmax with the row maximum exchanged between the
//               two halves, P (bf16) into TMEM over its S, rescale O when the
//               reference maximum moves, final O / l staged per warp in shared
//               memory (32 rows x 32 columns at a time) and written by TMA stores
//   warp 11     mask metadata: end[] / pos[] of each KV tile's keys and their
//               minima, loaded from global memory into a 4-slot ring ahead of
//               the softmax
// The tensor core computes S(j+1) and PV(j-1) while the softmax works on tile j;
// the next item's Q load and first S overlap the previous item's epilogue.
//
// Batch invariance ("What it does": an input's scores are bit-identical alone
// or packed with thousands of others): KV tiles start at the first row of the
// input that owns them, so a key always lands in the same MMA column whatever
// precedes its input in the pass; tiles are visited in a fixed order; a tile
// with no visible key for a row is an exact no-op for that row (its maximum
// stays, P is exactly 0 and O is multiplied by exactly 1).  An item's first PV
// product overwrites O and the rest accumulate; a leading tile with no visible key
// leaves exact zeros, to which adding the first visible tile's product gives the
// same bits as writing it.  No result depends on which CTA runs an item.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "runtime.h"

namespace spinf {
namespace {

using namespace dev;

constexpr int kAttnThreads = 384;      // TMA producer, S MMA, PV MMA, 8 softmax warps, mask metadata
constexpr int kSoftmaxThreads = 256;
constexpr int kFirstSoftmaxWarp = 3;
constexpr int kMetaWarp = 11;
constexpr int kPvWarp = 2;
constexpr int kMetaSlots = 4;          // mask-metadata ring: tiles the metadata warp may run ahead
constexpr int kBoxBytes = 128 * 128;   // one TMA box: 128 rows x 64 bf16 (128-byte swizzled rows)
constexpr int kOstageBytes = 32 * 64;  // O staging of one softmax warp: 32 rows x 32 bf16

// Barrier protocol.  A parity wait for the phase of tile G on a ring of n barriers is only
// correct when the barrier's previous phase (tile G - n) is known to have completed and
// its next one (tile G + n) cannot have: with the previous phase still open the wait
// passes at once, with the next one done it blocks.  Every ring below is sized so that
// each wait meets that condition:
//   S_FULL[G % kSBufs]  S(G) is in TMEM: the softmax may read it; the K buffer it read is free
//   P_FULL[G % kSBufs]  every softmax thread has written P(G).  Warps of different lane
//                       quarters are not in lockstep: one may be at most kSBufs - 1 tiles
//                       ahead of another (S(G) needs P(G - kSBufs) consumed), so P_FULL
//                       has kSBufs barriers
//   P_USED[G % kSBufs]  PV(G) has read P(G), so S(G + kSBufs) may overwrite that TMEM
//                       buffer.  MMAs into different accumulators are not ordered by the
//                       tensor core.
//   V_DONE[G % 4]       PV(G) and every earlier PV have finished: O may be read or
//                       rescaled, V buffer G % 2 is free.  While the softmax works on tile
//                       G, S(G) has only proven PV(G - kSBufs) done, so up to kSBufs PVs
//                       (four at d_head 256) may be in flight: with four barriers the
//                       previous phase of PV(G - 1)'s barrier, PV(G - 5), is always done.
//                       (A two-barrier ring by tile parity let a wait for PV(G - 1) pass
//                       while PV(G - 3) was still open at d_head 256: O was then read or
//                       rescaled under in-flight PV products.)
//   MMA_DONE(_PV)       all MMAs of one issuer thread have completed (before TMEM is freed)
enum {
    Q_FULL = 0, Q_EMPTY, S_FULL0, S_FULL1, S_FULL2, S_FULL3, P_FULL0, P_FULL1, P_FULL2, P_FULL3, P_USED0, P_USED1,
    P_USED2, P_USED3, V_DONE0, V_DONE1, V_DONE2, V_DONE3, MMA_DONE, MMA_DONE_PV, N_FIXED_BARS
};
constexpr int kVDone = 4;   // V_DONE ring

// Keys per KV tile: 64 at d_head 256 outside a cta_group::2 pair (Q, two K and two V buffers
// then fit the shared memory: 64 + 4 x 32 KB), else 128.  A 64-key tile is one half of the
// planner's input-anchored 128-key tile, so a key keeps its column whatever is packed.
template <int D, int MODE>
constexpr int kTK = (D == 256 && MODE != 2) ? 64 : 128;

template <int D, int MODE>
struct AttnSmem {
    static constexpr int kChunks = D / 64;
    static constexpr int kTileBytes = kChunks * kBoxBytes;                  // a 128-row Q tile
    static constexpr int kKVTile = kChunks * kTK<D, MODE> * 128;           // a K or V tile
    // a cta_group::2 pair keeps half of every K tile (64 keys) and of every V tile (D/2 columns) per CTA
    static constexpr int kKBytes = MODE == 2 ? kTileBytes / 2 : kKVTile;
    static constexpr int kVBytes = MODE == 2 ? kTileBytes / 2 : kKVTile;
    static constexpr int kStages = 2;   // K and V buffers each
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kTileBytes;                // K stage s at kK + s * kKBytes
    static constexpr int kV = kK + kStages * kKBytes;
    static constexpr int kMeta = kV + kStages * kVBytes;    // int32 [kMetaSlots][2][kTK]: end[], pos[] of a tile's keys
    static constexpr int kMetaHead = kMeta + kMetaSlots * 2 * kTK<D, MODE> * 4;   // int32 [kMetaSlots][4]: min end, min pos, kv0, len
    static constexpr int kXmax = kMetaHead + kMetaSlots * 4 * 4;   // float [2][2][128]: row maxima of the two halves
    static constexpr int kLx = kXmax + 2 * 2 * 128 * 4;     // float [2][128]: the halves' row sums, per item
    static constexpr int kOstage = (kLx + 2 * 128 * 4 + 1023) / 1024 * 1024;  // per softmax warp: 32 x 32 O bf16
    // fixed barriers, then K_FULL, V_FULL [kStages], META_FULL, META_EMPTY [kMetaSlots]
    static constexpr int kBars = kOstage + 8 * kOstageBytes;
    static constexpr int kNumBars = N_FIXED_BARS + 2 * kStages + 2 * kMetaSlots;
    static constexpr int kHolder = kBars + kNumBars * 8;
    static constexpr int kBytes = kHolder + 16;
    static constexpr int kAlloc = kBytes + 1024;            // room to align the base to 1024
    static_assert(kAlloc <= 227 * 1024, "shared memory of one CTA");
};

// TMEM columns: S buffers of one column per key of a KV tile -- tile G uses buffer
// G % kSBufs, and its P (bf16 pairs, half as many columns) overwrites the start of that
// buffer once the softmax has read S -- then O (D columns).  d_head 256: four 64-column
// buffers, O at 256; d_head <= 128: three 128-column buffers, O at 384, so S of tile G
// waits for the PV of tile G - kSBufs (usually long done).  512 columns are allocated, so one CTA per SM (the
// shared-memory request enforces it and no allocation ever waits).
template <int D>
constexpr int kSBufs = D <= 128 ? 3 : 4;
template <int D>
constexpr uint32_t kColO = D <= 128 ? 384 : 256;
constexpr uint32_t kTmemCols = 512;
constexpr int kMinSmem = 116 * 1024;
// Log2 headroom of the lazy softmax reference maximum: P values stay <= 2^8.
constexpr float kRescaleLog2 = 8.f;

struct Item {
    int qt, h, s0, n;
};

// MODE 0: one CTA per item (one query head).  MODE 2: cta_group::2 pairs -- the leader
// issues M = 256 MMAs over both CTAs' rows, each CTA holding half of every K and V tile.
// MODE 3: one CTA per item of two query heads that share a kv head, 64 token rows of each
// stacked in the MMA's 128 rows (Q tiles of 64 rows: fewer masked pairs per executed tile,
// and each K/V tile serves both heads).
template <int D, int MODE>
__global__ void __launch_bounds__(kAttnThreads, 1)
    branch_attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_kh,
                            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                            __nv_bfloat16* __restrict__ o,
                            const int32_t* __restrict__ end, const int32_t* __restrict__ pos,
                            const int32_t* __restrict__ qt_work, const int32_t* __restrict__ tile_kv,
                            const int32_t* __restrict__ tile_len, const int32_t* __restrict__ row_runs, int T,
                            int Hq, int Hkv, int n_items,
                            float scale_log2, int window, int* __restrict__ err) {
    static_assert(MODE == 0 || MODE == 2 || MODE == 3, "one CTA per item, a cta_group::2 pair, or two stacked heads");
    static_assert(MODE != 2 || D >= 128, "a cta_group::2 pair splits V into 64-column boxes");
    using L = AttnSmem<D, MODE>;
    constexpr bool PAIR = MODE == 2;
    constexpr bool CG2 = PAIR;
    constexpr bool QG = MODE == 3;   // MMA row r: token row qt * 64 + (r & 63) of query head 2 * g + (r >> 6)
    constexpr int TK = kTK<D, MODE>;           // keys per KV tile
    constexpr int KH = TK / 2;                 // keys per softmax thread (half of a tile's row)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + L::kQ;
    uint8_t* sK = smem + L::kK;
    uint8_t* sV = smem + L::kV;
    int32_t* meta = reinterpret_cast<int32_t*>(smem + L::kMeta);
    int32_t* meta_head = reinterpret_cast<int32_t*>(smem + L::kMetaHead);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
    uint32_t* holder = reinterpret_cast<uint32_t*>(smem + L::kHolder);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = Hq / Hkv;
    // PAIR: item = (Q tile, pair of heads 2p, 2p+1 of one kv group); this CTA takes head 2p + rank
    const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
    const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int n_units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    const int heads_per_item = PAIR ? 2 : 1;
    const int head_groups = QG ? Hkv : Hq / heads_per_item;   // QG: an item is a kv head g
    // item it = (position it / head_groups in the work order, head group it % head_groups);
    // one 16-byte record {qt, first schedule entry, entry count, 0} per Q tile
    auto item = [&](int it) {
        const int4 w = __ldg(reinterpret_cast<const int4*>(qt_work) + it / head_groups);
        Item I;
        I.qt = w.x;
        I.s0 = w.y;
        I.n = w.z;
        I.h = QG ? it % head_groups : (it % head_groups) * heads_per_item + rank;
        return I;
    };
    // the k-th item of this CTA (pair): rounds of n_units items, every other round
    // reversed, so that long and short items spread evenly over the CTAs
    auto item_index = [&](int k) { return k * n_units + ((k & 1) ? n_units - 1 - unit : unit); };

    uint64_t* k_full = bars + N_FIXED_BARS;
    uint64_t* v_full = k_full + L::kStages;
    static_assert(kSBufs<D> <= kVDone, "the V_DONE ring covers every PV that may be in flight");
    // PV(G) done: barrier V_DONE[G % 4], phase G / 4
    auto v_done = [&](uint32_t G) { return &bars[V_DONE0 + G % kVDone]; };
    auto v_phase = [](uint32_t G) { return (G / kVDone) & 1u; };
    // barrier that says P(G) has been read, and its phase index is G / kSBufs
    auto p_used = [&](uint32_t G) { return &bars[P_USED0 + G % kSBufs<D>]; };
    uint64_t* meta_full = v_full + L::kStages;
    uint64_t* meta_empty = meta_full + kMetaSlots;
    if (threadIdx.x == 0) {
        // P_FULL: every softmax thread, or (CG2) one arrival from each CTA of the pair
        for (int b = 0; b < N_FIXED_BARS; ++b) {
            int count = 1;
            if (b >= P_FULL0 && b <= P_FULL3) count = CG2 ? 2 : kSoftmaxThreads;
            mbar_init(&bars[b], count);
        }
        for (int st = 0; st < L::kStages; ++st) {
            mbar_init(&k_full[st], 1);
            mbar_init(&v_full[st], 1);
        }
        for (int sl = 0; sl < kMetaSlots; ++sl) {
            mbar_init(&meta_full[sl], 32);                       // every lane of the metadata warp
            mbar_init(&meta_empty[sl], kSoftmaxThreads / 32);    // one arrival per softmax warp
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        if constexpr (CG2) {
            tmem_alloc_pair(holder, kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(holder, kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();   // the peer's barriers exist before the pair's copies and commits signal them
    tc_fence_after();
    const uint32_t tmem = *holder;

    if (warp == 0) {
        // ---------------------------------------------------------- Q, K and V producer
        // One thread walks the tile sequence with two cursors, K (with the Q of each item)
        // and V, and issues whichever copy's buffer is free first: a K copy never waits
        // behind a V buffer or the other way round.  Each cursor tests its barrier phases
        // in order, so a barrier is never two phases ahead of the phase tested.
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(CG2 ? &tm_kh : &tm_k);
            tma_prefetch_desc(&tm_v);
            struct Cursor {
                int k;        // item ordinal
                Item I;
                int j;        // tile within the item
                uint32_t G;   // tile of the CTA's sequence
                int kv0;      // first key of tile G
                bool done;
            };
            auto seek = [&](Cursor& c) {   // from item ordinal c.k onwards, the first item with tiles
                for (;; ++c.k) {
                    const int it = item_index(c.k);
                    if (it >= n_items) {
                        c.done = true;
                        return;
                    }
                    c.I = item(it);
                    if (c.I.n > 0) break;
                }
                c.j = 0;
                c.kv0 = __ldg(tile_kv + c.I.s0);
            };
            auto advance = [&](Cursor& c) {
                ++c.G;
                if (++c.j < c.I.n) {
                    c.kv0 = __ldg(tile_kv + c.I.s0 + c.j);
                } else {
                    ++c.k;
                    seek(c);
                }
            };
            Cursor kc{0, Item{0, 0, 0, 0}, 0, 0, 0, false}, vc = kc;
            seek(kc);
            seek(vc);
            uint32_t ic = 0;          // Q copies issued
            bool q_pending = true;    // the K cursor's item still needs its Q
            unsigned long long t_idle = 0;
            while (!kc.done || !vc.done) {
                bool progress = false;
                if (!kc.done) {
                    if (q_pending) {
                        if (ic == 0 || mbar_test(&bars[Q_EMPTY], (ic - 1) & 1)) {   // the previous item's last S is done
                            // one copy per tile: every 64-column chunk at once (4-D view, chunk-major in smem)
                            if constexpr (CG2) {   // both CTAs' Q tiles are counted on the leader's barrier
                                if (rank == 0) mbar_arrive_expect_tx(&bars[Q_FULL], 2 * L::kTileBytes);
                                tma_load_4d_pair(sQ, &tm_q, mapa_shared(smem_u32(&bars[Q_FULL]), 0), 0, kc.I.qt * 128,
                                                 0, kc.I.h);
                            } else {
                                mbar_arrive_expect_tx(&bars[Q_FULL], L::kTileBytes);
                                if constexpr (QG)   // (64 columns, rows, head, chunk) view: both heads' 64 rows
                                    tma_load_4d(sQ, &tm_q, &bars[Q_FULL], 0, kc.I.qt * 64, 2 * kc.I.h, 0);
                                else
                                    tma_load_4d(sQ, &tm_q, &bars[Q_FULL], 0, kc.I.qt * 128, 0, kc.I.h);
                            }
                            ++ic;
                            q_pending = false;
                            progress = true;
                        }
                    } else {
                        const uint32_t G = kc.G, Gp = G - L::kStages;   // S(Gp) was the last reader of the buffer
                        if (G < (uint32_t)L::kStages ||
                            mbar_test(&bars[S_FULL0 + Gp % kSBufs<D>], (Gp / kSBufs<D>) & 1)) {
                            const uint32_t st = G % L::kStages;
                            uint8_t* dst = sK + st * L::kKBytes;
                            if constexpr (CG2) {   // keys [64 rank, 64 rank + 64) of the tile, counted on the leader
                                if (rank == 0) mbar_arrive_expect_tx(&k_full[st], 2 * L::kKBytes);
                                tma_load_4d_pair(dst, &tm_kh, mapa_shared(smem_u32(&k_full[st]), 0), 0,
                                                 kc.kv0 + 64 * rank, 0, kc.I.h / group);
                            } else {
                                mbar_arrive_expect_tx(&k_full[st], L::kKBytes);
                                tma_load_4d(dst, &tm_k, &k_full[st], 0, kc.kv0, 0, QG ? kc.I.h : kc.I.h / group);
                            }
                            const int k_before = kc.k;
                            advance(kc);
                            if (kc.k != k_before) q_pending = true;
                            progress = true;
                        }
                    }
                }
                if (!vc.done) {
                    const uint32_t G = vc.G, Gp = G - L::kStages;   // PV(Gp) was the last reader of the buffer
                    if (G < (uint32_t)L::kStages || mbar_test(v_done(Gp), v_phase(Gp))) {
                        const uint32_t st = G % L::kStages;
                        uint8_t* dst = sV + st * L::kVBytes;
                        if constexpr (CG2) {   // chunks [D/128 rank, D/128 rank + D/128), counted on the leader
                            if (rank == 0) mbar_arrive_expect_tx(&v_full[st], 2 * L::kVBytes);
                            tma_load_4d_pair(dst, &tm_v, mapa_shared(smem_u32(&v_full[st]), 0), 0, vc.kv0,
                                             rank * (L::kChunks / 2), vc.I.h / group);
                        } else {
                            mbar_arrive_expect_tx(&v_full[st], L::kVBytes);
                            tma_load_4d(dst, &tm_v, &v_full[st], 0, vc.kv0, 0, QG ? vc.I.h : vc.I.h / group);
                        }
                        advance(vc);
                        progress = true;
                    }
                }
                if (progress) {
                    t_idle = 0;
                } else {   // bounded like every other wait; back off so the softmax warps sharing
                           // this scheduler keep its issue slots
                    __nanosleep(64);
                    if (*reinterpret_cast<volatile int*>(err) != 0) break;
                    const unsigned long long now = globaltimer();
                    if (t_idle == 0) t_idle = now;
                    else if (now - t_idle > kWaitLimitNs) {
                        atomicCAS(err, 0, kErrTimeout);
                        break;
                    }
                }
            }
            // our last copies have landed before the CTA may retire, and every commit that
            // another thread or CTA makes to our barriers has arrived
            // (CG2: a peer's copies are counted on the leader, whose release implies they landed)
            const uint32_t GK = kc.G, GV = vc.G;
            for (uint32_t b = GK > (uint32_t)L::kStages ? GK - L::kStages : 0; b < GK; ++b)
                if (!CG2 || rank == 0) mbar_drain(&k_full[b % L::kStages], (b / L::kStages) & 1, err);
            for (uint32_t b = GK > (uint32_t)kSBufs<D> ? GK - kSBufs<D> : 0; b < GK; ++b)
                mbar_drain(&bars[S_FULL0 + b % kSBufs<D>], (b / kSBufs<D>) & 1, err);
            for (uint32_t b = GV > (uint32_t)L::kStages ? GV - L::kStages : 0; b < GV; ++b)
                if (!CG2 || rank == 0) mbar_drain(&v_full[b % L::kStages], (b / L::kStages) & 1, err);
            for (uint32_t b = GV > 2u ? GV - 2 : 0; b < GV; ++b) mbar_drain(v_done(b), v_phase(b), err);
            if (ic > 0) {
                if (!CG2 || rank == 0) mbar_drain(&bars[Q_FULL], (ic - 1) & 1, err);
                if (CG2) mbar_drain(&bars[Q_EMPTY], (ic - 1) & 1, err);
            }
        }
    } else if (warp == 1 || warp == kPvWarp) {
        // ---------------------------------------------------------- MMA issuers
        // S = Q K^T from warp 1, O += P V from warp 2: two instruction streams, so the tensor
        // core has the other stream's MMAs to run while one thread commits or waits
        if (lane == 0 && (!CG2 || rank == 0)) {   // a pair's MMAs are all issued by its leader
            constexpr uint32_t idesc_qk = idesc_bf16(CG2 ? 256 : 128, TK, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16(CG2 ? 256 : 128, D, false, true);
            auto commit = [&](uint64_t* bar) {
                if constexpr (CG2) mma_commit_pair(bar); else mma_commit(bar);
            };
            const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
            const bool s_issuer = warp == 1;
            uint32_t G = 0, ic = 0;
            for (int k = 0;; ++k) {
                const int it = item_index(k);
                if (it >= n_items) break;
                const Item I = item(it);
                if (I.n <= 0) continue;
                if (s_issuer) {
                    mbar_wait(&bars[Q_FULL], ic & 1, err);
                    for (int j = 0; j < I.n; ++j) {
                        const uint32_t Gs = G + j;
                        // buffer Gs % kSBufs held P(Gs - kSBufs): that PV has read it
                        if (Gs >= (uint32_t)kSBufs<D>) {
                            const uint32_t Gp = Gs - kSBufs<D>;
                            mbar_wait(p_used(Gp), (Gp / kSBufs<D>) & 1, err);
                        }
                        // an item's first S waits for the previous item's last PV, so that PV runs first
                        // and the softmax warps start their epilogue sooner; this S is not needed before
                        // that epilogue ends
                        if (j == 0 && Gs > 0) mbar_wait(v_done(Gs - 1), v_phase(Gs - 1), err);
                        const uint32_t st = Gs % L::kStages;
                        mbar_wait(&k_full[st], (Gs / L::kStages) & 1, err);
                        tc_fence_after();
                        const uint32_t dS = tmem + (Gs % kSBufs<D>) * TK;
                        const uint32_t aKs = aK + st * L::kKBytes;
                        constexpr int kKBox = CG2 ? kBoxBytes / 2 : TK * 128;   // K boxes hold 64 or 128 keys
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                            const uint32_t koff = (kk >> 2) * kKBox + (kk & 3) * 32;
                            const uint64_t da = sdesc_sw128(aQ + off, 16, 1024), db = sdesc_sw128(aKs + koff, 16, 1024);
                            if constexpr (CG2) mma_f16_ss_pair(dS, da, db, idesc_qk, kk > 0);
                            else mma_f16_ss(dS, da, db, idesc_qk, kk > 0);
                        }
                        commit(&bars[S_FULL0 + Gs % kSBufs<D>]);
                        if (j + 1 == I.n) commit(&bars[Q_EMPTY]);   // Q is free once the item's last S is done
                    }
                } else {
                    for (int j = 0; j < I.n; ++j) {
                        const uint32_t Gj = G + j;
                        uint64_t* pf = &bars[P_FULL0 + Gj % kSBufs<D>];
                        if constexpr (CG2) mbar_wait_cluster(pf, (Gj / kSBufs<D>) & 1, err);   // the peer arrives remotely
                        else mbar_wait(pf, (Gj / kSBufs<D>) & 1, err);
                        const uint32_t st = Gj % L::kStages;
                        mbar_wait(&v_full[st], (Gj / L::kStages) & 1, err);
                        tc_fence_after();
                        const uint32_t aP = tmem + (Gj % kSBufs<D>) * TK;
                        const uint32_t aVs = aV + st * L::kVBytes;
#pragma unroll
                        for (int kk = 0; kk < TK / 16; ++kk) {   // 16 keys: 8 TMEM columns of bf16 pairs of P
                            // V as [chunk][TK keys] boxes: 16 keys of every chunk at kk * 2048
                            const uint64_t db = sdesc_sw128(aVs + kk * 2048, TK * 128, 1024);
                            // an item's first product overwrites O (adding it to zero would give the same bits)
                            const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
                            if constexpr (CG2) mma_f16_ts_pair(tmem + kColO<D>, aP + kk * 8, db, idesc_pv, acc);
                            else mma_f16_ts(tmem + kColO<D>, aP + kk * 8, db, idesc_pv, acc);
                        }
                        commit(v_done(Gj));
                        if constexpr (kSBufs<D> >= 3) commit(&bars[P_USED0 + Gj % kSBufs<D>]);
                    }
                }
                G += I.n;
                ++ic;
            }
            // every MMA of this thread has completed before TMEM is freed
            uint64_t* done = &bars[s_issuer ? MMA_DONE : MMA_DONE_PV];
            commit(done);
            mbar_drain(done, 0, err);
        }
    } else if (warp == kMetaWarp) {
        // ---------------------------------------------------------- mask metadata of each KV tile
        // end[] and pos[] of the tile's keys (keys past the tile's own input: end -1,
        // pos 0), their minima, kv0 and the length, into a ring read by the softmax warps;
        // this warp's global loads run up to kMetaSlots tiles ahead of the softmax
        uint32_t G = 0;
        for (int k = 0;; ++k) {
            const int it = item_index(k);
            if (it >= n_items) break;
            const Item I = item(it);
            if (I.n <= 0) continue;
            for (int j = 0; j < I.n; ++j, ++G) {
                const int slot = G % kMetaSlots;
                const int kv0 = __ldg(tile_kv + I.s0 + j), len = __ldg(tile_len + I.s0 + j);
                constexpr int kPer = TK / 32;   // keys per lane
                int ev[kPer], pv[kPer];
                int emin = INT_MAX, pmin = INT_MAX;
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int key = lane + 32 * i;
                    ev[i] = key < len ? __ldg(end + kv0 + key) : -1;
                    pv[i] = key < len ? __ldg(pos + kv0 + key) : 0;
                    emin = min(emin, ev[i]);
                    pmin = min(pmin, pv[i]);
                }
                emin = __reduce_min_sync(0xffffffffu, emin);
                pmin = __reduce_min_sync(0xffffffffu, pmin);
                if (G >= (uint32_t)kMetaSlots) mbar_wait(&meta_empty[slot], (G / kMetaSlots - 1) & 1, err);
                int32_t* me = meta + slot * 2 * TK;
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    me[lane + 32 * i] = ev[i];
                    me[TK + lane + 32 * i] = pv[i];
                }
                if (lane == 0)
                    *reinterpret_cast<int4*>(meta_head + 4 * slot) = make_int4(emin, pmin, kv0, len);
                mbar_arrive(&meta_full[slot]);
            }
        }
    } else {
        // ---------------------------------------------------------- softmax and epilogue
        const int sw = warp - kFirstSoftmaxWarp;      // 0..7
        const int quarter = warp & 3;                 // TMEM lanes this warp may touch
        const int half = sw >> 2;                     // which half of the row's columns
        const int r = quarter * 32 + lane;            // Q-tile row of this thread
        const int t = sw * 32 + lane;                 // 0..255
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_off + kColO<D> + half * (D / 2);
        const uint32_t pair_bar = 2 + quarter;        // the two warps that share these TMEM lanes
        float* xmax = reinterpret_cast<float*>(smem + L::kXmax);
        float* lx = reinterpret_cast<float*>(smem + L::kLx);

        uint32_t G = 0;
        int k = 0;
        int it = item_index(0);
        Item I = it < n_items ? item(it) : Item{0, 0, 0, 0};
        while (it < n_items) {
            // the next item's record is loaded while this one runs
            const int it_next = item_index(k + 1);
            const Item I_next = it_next < n_items ? item(it_next) : Item{0, 0, 0, 0};
            if (I.n > 0) {
            const int q_row = QG ? I.qt * 64 + (r & 63) : I.qt * 128 + r;
            const bool real = q_row < T;
            const int pos_q = __ldg(pos + q_row);
            // the row's root path as up to four runs of rows [lo, hi) (x < 0: more runs)
            const int4 run01 = __ldg(reinterpret_cast<const int4*>(row_runs) + 2 * q_row);
            const int4 run23 = __ldg(reinterpret_cast<const int4*>(row_runs) + 2 * q_row + 1);
            float m = -INFINITY, l = 0.f;   // l: this half's share of the row sum
            for (int j = 0; j < I.n; ++j, ++G) {
                const int b = G & 1;                  // xmax buffer
                const int sb = G % kSBufs<D>;         // TMEM S buffer
                const int slot = G % kMetaSlots;
                mbar_wait(&meta_full[slot], (G / kMetaSlots) & 1, err);
                const int4 head = *reinterpret_cast<const int4*>(meta_head + 4 * slot);   // min end, min pos, kv0, len
                mbar_wait(&bars[S_FULL0 + sb], (G / kSBufs<D>) & 1, err);
                tc_fence_after();
                const uint32_t tS = tmem + lane_off + sb * TK;
                float s[KH];
                {
                    uint32_t rr[KH];
                    if constexpr (KH == 64) tmem_ld64(tS + half * KH, rr);
                    else tmem_ld32(tS + half * KH, rr);
#pragma unroll
                    for (int i = 0; i < KH; ++i) s[i] = __uint_as_float(rr[i]);
                }
                // visible: kv0 + c <= q_row (causal), q_row < end[key], window on depth.
                // A tile whose every key is visible to this row skips the per-key test.
                const int cmax = real ? q_row - head.z : -1;
                const bool all_visible =
                    cmax >= TK - 1 && head.x > q_row && (window <= 0 || pos_q - head.y < window);
                float mx = -INFINITY;
                // maximum of the KH values, two independent chains of three-input maxima
                auto max64 = [&]() {
                    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
                    for (int i = 0; i < KH; i += 4) {
                        m0 = fmax3(m0, s[i], s[i + 1]);
                        m1 = fmax3(m1, s[i + 2], s[i + 3]);
                    }
                    return fmaxf(m0, m1);
                };
                if (all_visible) {
                    mx = max64();
                } else if ((window <= 0 || pos_q - head.y < window) && run01.x >= 0) {
                    // visible keys of this half from the row's runs: no per-key loads (with a window,
                    // when every key of the tile is within it: no key is shallower than head.y)
                    const int kb = head.z + KH * half;
                    auto bits = [&](int lo, int hi) -> uint64_t {
                        const int a = max(lo - kb, 0), b = min(hi - kb, KH);
                        if (a >= b) return 0ull;
                        const uint64_t upto = b == 64 ? ~0ull : ((1ull << b) - 1ull);
                        return upto & ~((1ull << a) - 1ull);
                    };
                    uint64_t vm = bits(run01.x, run01.y) | bits(run01.z, run01.w) | bits(run23.x, run23.y) |
                                  bits(run23.z, run23.w);
                    // only the tile's own keys: the rest belong to the next input, whose own
                    // anchored tiles cover them
                    const int lim = min(max(head.w - KH * half, 0), KH);
                    if (lim < 64) vm &= (1ull << lim) - 1ull;
                    if (!real) vm = 0ull;
#pragma unroll
                    for (int i = 0; i < KH; ++i) s[i] = ((vm >> i) & 1ull) ? s[i] : -INFINITY;
                    mx = max64();
                } else {
                    const int4* e4 = reinterpret_cast<const int4*>(meta + slot * 2 * TK + half * KH);
                    const int4* p4 = reinterpret_cast<const int4*>(meta + slot * 2 * TK + TK + half * KH);
                    const int cm = cmax - half * KH;
#pragma unroll
                    for (int c4 = 0; c4 < KH / 4; ++c4) {
                        const int4 e = e4[c4];
                        bool v0 = 4 * c4 + 0 <= cm && q_row < e.x;
                        bool v1 = 4 * c4 + 1 <= cm && q_row < e.y;
                        bool v2 = 4 * c4 + 2 <= cm && q_row < e.z;
                        bool v3 = 4 * c4 + 3 <= cm && q_row < e.w;
                        if (window > 0) {
                            const int4 pp = p4[c4];
                            v0 = v0 && pos_q - pp.x < window;
                            v1 = v1 && pos_q - pp.y < window;
                            v2 = v2 && pos_q - pp.z < window;
                            v3 = v3 && pos_q - pp.w < window;
                        }
                        s[4 * c4 + 0] = v0 ? s[4 * c4 + 0] : -INFINITY;
                        s[4 * c4 + 1] = v1 ? s[4 * c4 + 1] : -INFINITY;
                        s[4 * c4 + 2] = v2 ? s[4 * c4 + 2] : -INFINITY;
                        s[4 * c4 + 3] = v3 ? s[4 * c4 + 3] : -INFINITY;
                        mx = fmaxf(mx, fmaxf(fmaxf(s[4 * c4], s[4 * c4 + 1]), fmaxf(s[4 * c4 + 2], s[4 * c4 + 3])));
                    }
                }
                // this warp is done with the metadata slot
                __syncwarp();
                if (lane == 0) mbar_arrive(&meta_empty[slot]);
                // the row maximum of the tile, from both halves
                xmax[(b * 2 + half) * 128 + r] = mx;
                named_bar_sync(pair_bar, 64);
                const float mx_row = fmaxf(xmax[(b * 2) * 128 + r], xmax[(b * 2 + 1) * 128 + r]);
                // Lazy rescaling: P and l are taken relative to a reference maximum m that
                // only moves when the row maximum exceeds it by more than 2^8 (so P <= 256);
                // the final O / l is the same softmax whichever reference was used.
                const float m_hi = fmaxf(m, mx_row);
                const bool grow = m != -INFINITY && (m_hi - m) * scale_log2 > kRescaleLog2;
                const float m_new = (m == -INFINITY || grow) ? m_hi : m;
                uint32_t pk[KH / 2];
                float alpha = 1.f;
                float rowsum = 0.f;
                if (m_new == -INFINITY) {
#pragma unroll
                    for (int i = 0; i < KH / 2; ++i) pk[i] = 0u;
                } else {
                    const float mb = m_new * scale_log2;
                    const float2 sc2 = make_float2(scale_log2, scale_log2), nb2 = make_float2(-mb, -mb);
                    float2 acc = make_float2(0.f, 0.f);   // even and odd columns, added at the end
#pragma unroll
                    for (int c = 0; c < KH / 2; ++c) {
                        const float2 x = ffma2(make_float2(s[2 * c], s[2 * c + 1]), sc2, nb2);
                        const float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                        acc = fadd2(acc, p);
                        pk[c] = pack_bf16x2(p.x, p.y);
                    }
                    rowsum = acc.x + acc.y;
                    if (grow) alpha = fast_exp2(fmaf(m, scale_log2, -mb));
                }
                if (m_new != -INFINITY) {
                    l = l * alpha + rowsum;
                    m = m_new;
                }
                // TMEM traffic is warp-collective: lanes whose maximum did not move multiply by exactly 1.
                // Only a rescale waits for the previous tile's PV (grow is false on an item's first
                // tile); P(j) itself goes to a buffer whose last reader, PV(j-2), finished before S(j).
                if (__any_sync(0xffffffffu, grow)) {
                    mbar_wait(v_done(G - 1), v_phase(G - 1), err);   // G >= 1: grow is false on tile 0
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < D / 64; ++c) {
                        uint32_t rr[32];
                        tmem_ld32(tO + c * 32, rr);
                        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 y = fmul2(make_float2(__uint_as_float(rr[i]), __uint_as_float(rr[i + 1])), a2);
                            rr[i] = __float_as_uint(y.x);
                            rr[i + 1] = __float_as_uint(y.y);
                        }
                        tmem_st32(tO + c * 32, rr);
                    }
                }
                // P of keys [KH half, KH half + KH) -> bf16 pairs in columns [KH/2 half, KH/2 half + KH/2)
                // of this tile's S buffer (both halves have read their S columns before the pair barrier)
                if constexpr (KH == 64) tmem_st32(tS + half * 32, pk);
                else tmem_st16(tS + half * 16, pk);
                tmem_st_wait();
                tc_fence_before();
                if constexpr (CG2) {   // one arrival per CTA on the leader's barrier
                    named_bar_sync(1, kSoftmaxThreads);
                    if (t == 0) {
                        if (rank == 0) mbar_arrive(&bars[P_FULL0 + sb]);
                        else mbar_arrive_cluster(mapa_shared(smem_u32(&bars[P_FULL0 + sb]), 0));
                    }
                } else {
                    mbar_arrive(&bars[P_FULL0 + sb]);
                }
            }
            // epilogue of the item: O / l to global memory, then O back to zero for the next item
            mbar_wait(v_done(G - 1), v_phase(G - 1), err);   // the item's last PV, and so every PV
            tc_fence_after();
            lx[half * 128 + r] = l;
            named_bar_sync(pair_bar, 64);
            const float lrow = lx[r] + lx[128 + r];      // halves added in a fixed order
            const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
            // this warp's 32 rows x D/2 columns, 32 columns at a time: each lane writes its row
            // into a 2 KB staging box, then one TMA store writes the 32 x 32 box to o.  Row x's
            // 16-byte pieces sit at slots piece ^ ((x >> 1) & 3): the 64-byte swizzle of the
            // store's tensor map, and free of bank conflicts for the row writes.  The store has
            // read the box before the next chunk overwrites it; the stores complete before the
            // CTA exits.  (A TMA store measured 1-2.5 % faster than 16-byte stores by the lanes.)
            uint8_t* stage = smem + L::kOstage + sw * kOstageBytes;
            auto store_chunk = [&](const uint32_t* rr, int col) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float2 y = fmul2(make_float2(__uint_as_float(rr[2 * i]), __uint_as_float(rr[2 * i + 1])),
                                           make_float2(inv, inv));
                    w[i] = real ? pack_bf16x2(y.x, y.y) : 0u;
                }
                uint4* srow = reinterpret_cast<uint4*>(stage + lane * 64);
                const int sx = (lane >> 1) & 3;
#pragma unroll
                for (int i = 0; i < 4; ++i) srow[i ^ sx] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {   // one 32-row x 32-column box (64-byte swizzle = the staging layout)
                    if constexpr (QG)
                        tma_store_3d(&tm_o, stage, col, 2 * I.h + (quarter >> 1), I.qt * 64 + (quarter & 1) * 32);
                    else
                        tma_store_3d(&tm_o, stage, col, I.h, I.qt * 128 + quarter * 32);
                    tma_store_commit_and_wait_read();
                }
                __syncwarp();
            };
            if constexpr (D >= 128) {
#pragma unroll 1
                for (int c = 0; c < D / 128; ++c) {   // 64 columns per TMEM load
                    uint32_t rr[64];
                    tmem_ld64(tO + c * 64, rr);
                    store_chunk(rr, half * (D / 2) + c * 64);
                    store_chunk(rr + 32, half * (D / 2) + c * 64 + 32);
                }
            } else {
                uint32_t rr[32];
                tmem_ld32(tO, rr);
                store_chunk(rr, half * (D / 2));
            }
            // lx is read by the partner before either writes it again (next item's epilogue)
            named_bar_sync(pair_bar, 64);
            }
            I = I_next;
            it = it_next;
            ++k;
        }
    }

    if (warp >= kFirstSoftmaxWarp && warp < kMetaWarp && lane == 0) tma_store_wait_all();   // o is written
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();   // nothing of the peer still lands in this CTA
    if (warp == 1) {
        tc_fence_after();
        if constexpr (CG2) tmem_dealloc_pair(tmem, kTmemCols);
        else tmem_dealloc(tmem, kTmemCols);
    }
}

// The schedule a launch walks: the pass's own, or its windowed subset.
struct Sched {
    const int32_t* qt_work;
    const int32_t* tile_kv;
    const int32_t* tile_len;
};

template <int D, int MODE>
spinf_status launch_mode(const Pass& P, const Sched& sc, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tkh,
                         const CUtensorMap& tv, const CUtensorMap& to, __nv_bfloat16* o, int Hq, int Hkv, float scale_log2, int window,
                         int* err, cudaStream_t stream) {
    auto kernel = branch_attention_kernel<D, MODE>;
    const int smem = AttnSmem<D, MODE>::kAlloc > kMinSmem ? AttnSmem<D, MODE>::kAlloc : kMinSmem;
    spinf_status st = set_smem_limit(reinterpret_cast<const void*>(kernel), smem, "cudaFuncSetAttribute(attention)");
    if (st) return st;
    cudaError_t e;
    const int n_items = MODE == 3 ? (P.T_pad / 64) * Hkv : (P.T_pad / 128) * (Hq / (MODE == 0 ? 1 : 2));
    if (MODE != 2) {
        const int grid = std::min(n_items, sm_count());
        kernel<<<grid, kAttnThreads, smem, stream>>>(tq, tk, tkh, tv, to, o, P.dev.end, P.dev.pos, sc.qt_work,
                                                     sc.tile_kv, sc.tile_len, P.dev.row_runs, P.T, Hq, Hkv,
                                                     n_items,
                                                     scale_log2, window, err);
    } else {   // cta_group::2 pairs: clusters of two CTAs, two heads of a kv group per item
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(kAttnThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(2 * std::max(1, sm_count() / 2));
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess || clusters <= 0) {
            cudaGetLastError();
            clusters = std::max(1, sm_count() / 2);
        }
        cfg.gridDim = dim3(2 * std::min(n_items, clusters));
        e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tkh, tv, to, o, (const int32_t*)P.dev.end,
                               (const int32_t*)P.dev.pos, sc.qt_work, sc.tile_kv, sc.tile_len,
                               (const int32_t*)P.dev.row_runs, P.T, Hq, Hkv, n_items, scale_log2, window, err);
        if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    return SPINF_OK;
}

template <int D>
spinf_status launch_attention(const Pass& P, const Sched& sc, const void* q, const void* k, const void* v, void* o, int Hq,
                              int Hkv, float scale, int window, int* err, cudaStream_t stream) {
    CUtensorMap tq, tk, tkh, tv, tvh, tvk;
    // 4-D views (64 columns, rows, 64-column chunks, head): one box holds every chunk of a
    // tile, laid out chunk after chunk (128-byte swizzled rows), as the MMA descriptors expect
    constexpr uint32_t kCh = D / 64;
    const uint64_t dq[4] = {64, (uint64_t)P.T_pad, kCh, (uint64_t)Hq};
    const uint64_t sq[3] = {(uint64_t)Hq * D * 2, 128, (uint64_t)D * 2};
    const uint64_t dk[4] = {64, (uint64_t)P.T_pad, kCh, (uint64_t)Hkv};
    const uint64_t sk[3] = {(uint64_t)Hkv * D * 2, 128, (uint64_t)D * 2};
    const uint32_t box[4] = {64, 128, kCh, 1};
    const uint32_t kbox_half[4] = {64, 64, kCh, 1};                        // keys of one CTA of a pair
    const uint32_t vbox_half[4] = {64, 128, kCh > 1 ? kCh / 2 : 1, 1};     // chunks of one CTA of a pair
    spinf_status st;
    if ((st = make_tmap(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, q, dq, sq, box, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    if ((st = make_tmap(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, k, dk, sk, box, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    if ((st = make_tmap(&tkh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, k, dk, sk, kbox_half, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    if ((st = make_tmap(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v, dk, sk, box, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    if ((st = make_tmap(&tvh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v, dk, sk, vbox_half, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    if ((st = make_tmap(&tvk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v, dk, sk, kbox_half, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(o);
    CUtensorMap to;
    {   // O as (d columns, heads, rows); a store box is 32 columns x 1 head x 32 rows
        const uint64_t dO[3] = {(uint64_t)D, (uint64_t)Hq, (uint64_t)P.T_pad};
        const uint64_t sO[2] = {(uint64_t)D * 2, (uint64_t)Hq * D * 2};
        const uint32_t bO[3] = {32, 1, 32};
        if ((st = make_tmap(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, o, dO, sO, bO, CU_TENSOR_MAP_SWIZZLE_64B)))
            return st;
    }
    const float scale_log2 = scale * 1.4426950408889634f;
    // d_head 128 with an even number of query heads per kv head: a cta_group::2 pair of two
    // heads (the kernel's third map is a K tile's key half).  d_head 256 with two query heads
    // per kv head: both heads' 64-row Q tiles stacked in one CTA's MMA rows.  Otherwise one CTA
    // per head.  d_head 256 copies 64-key K and V tiles (boxes of 64 rows) on the 64-key schedule
    const CUtensorMap& kmap = D == 256 ? tkh : tk;
    const CUtensorMap& vmap = D == 256 ? tvk : tv;
    if constexpr (D == 128)
        if ((Hq / Hkv) % 2 == 0) return launch_mode<D, 2>(P, sc, tq, tk, tkh, tvh, to, ob, Hq, Hkv, scale_log2, window, err, stream);
    if constexpr (D == 256)
        if (Hq / Hkv == 2) {
            // Q as (64 columns, rows, head, 64-column chunk): a box of 64 rows of two adjacent heads
            // lands chunk by chunk as 128 rows (head 2g, then 2g + 1), the MMA's A layout
            CUtensorMap tq2;
            const uint64_t dq2[4] = {64, (uint64_t)P.T_pad, (uint64_t)Hq, kCh};
            const uint64_t sq2[3] = {(uint64_t)Hq * D * 2, (uint64_t)D * 2, 128};
            const uint32_t box2[4] = {64, 64, 2, kCh};
            if ((st = make_tmap(&tq2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, q, dq2, sq2, box2, CU_TENSOR_MAP_SWIZZLE_128B)))
                return st;
            return launch_mode<D, 3>(P, sc, tq2, kmap, tkh, vmap, to, ob, Hq, Hkv, scale_log2, window, err, stream);
        }
    return launch_mode<D, 0>(P, sc, tq, kmap, tkh, vmap, to, ob, Hq, Hkv, scale_log2, window, err, stream);
}

}  // namespace
}  // namespace spinf

using namespace spinf;

extern "C" spinf_status spinf_branch_attention(const spinf_plan* plan, int32_t pass, const void* q, const void* k,
                                               const void* v, void* o, int32_t n_q_heads, int32_t n_kv_heads,
                                               int32_t d_head, float scale, int32_t window, spinf_stream stream) {
    spinf_status st = ensure_device_ready(plan, pass);
    if (st) return st;
    if (!q || !k || !v || !o) return fail(SPINF_E_INVALID, "NULL tensor");
    for (const void* p : {q, k, v, (const void*)o})
        if (reinterpret_cast<uintptr_t>(p) & 15) return fail(SPINF_E_INVALID, "tensor not 16-byte aligned");
    if (n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads || n_q_heads > 65535)
        return fail(SPINF_E_INVALID, "bad head counts");
    if (window < 0) return fail(SPINF_E_INVALID, "negative window");
    const Pass& P = plan->passes[pass];
    if (d_head != 64 && d_head != 128 && d_head != 256) return fail(SPINF_E_UNSUPPORTED, "d_head must be 64, 128 or 256");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // with a window, the schedule without the tiles no row of a Q tile sees within it;
    // d_head 256 walks the 64-key halves of the schedule's tiles (those some row sees), on
    // 64-row Q tiles when a kv head serves two query heads
    Sched sc{P.dev.qt_work, P.dev.tile_kv, P.dev.tile_len};
    if ((window > 0 || d_head == 256) && P.T > 0) {
        std::lock_guard<std::mutex> lock(const_cast<spinf_plan*>(plan)->cache_mu);
        const int q_rows = d_head == 256 && n_q_heads == 2 * n_kv_heads ? 64 : kTile;
        WindowSchedule& w = tile_schedule(const_cast<Pass&>(P), window, d_head == 256 ? 64 : kTile, q_rows);
        if ((st = upload_window(w, s))) return st;
        sc = Sched{w.d_qt_work, w.d_tile_kv, w.d_tile_len};
    }
    if (P.T == 0) return SPINF_OK;
    if (!(scale > 0.f)) scale = 1.0f / std::sqrt(static_cast<float>(d_head));
    switch (d_head) {
        case 64: return launch_attention<64>(P, sc, q, k, v, o, n_q_heads, n_kv_heads, scale, window, plan->d_err, s);
        case 128: return launch_attention<128>(P, sc, q, k, v, o, n_q_heads, n_kv_heads, scale, window, plan->d_err, s);
        case 256: return launch_attention<256>(P, sc, q, k, v, o, n_q_heads, n_kv_heads, scale, window, plan->d_err, s);
        default: return fail(SPINF_E_UNSUPPORTED, "d_head must be 64, 128 or 256");
    }
}
