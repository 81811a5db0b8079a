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
// finish together.  When a kv group has an even number of query heads, CTAs run as
// clusters of two that take two heads of one group on the same Q tile: at d_head
// 64 and 256 each CTA loads half of every K and V tile and multicasts it to both
// (a buffer is refilled once both CTAs' MMAs have released it); at d_head 128 the
// pair is a cta_group::2 MMA pair: the leader issues M = 256 products over both
// CTAs' rows, and each CTA holds half of every K tile (64 keys) and V tile (64
// columns).  Warp roles:
//   warp 0      TMA producer of Q (once per item) and K tiles (two buffers, or one
//               at d_head 256 outside a cta_group::2 pair)
//   warp 1      TMEM owner and MMA issuer: S = Q K^T into one of two TMEM
//               buffers (SS form, fp32), O += P V (P read from TMEM, V MN-major
//               from shared memory)
//   warp 2      TMA producer of V tiles (buffered like K)
//   warps 3-10  softmax, two warps per TMEM lane quarter: each thread owns half
//               of one Q row (64 of the 128 key columns, D/2 of the O columns):
//               mask, online softmax with the row maximum exchanged between the
//               two halves, P (bf16) into TMEM over its S, rescale O when the
//               reference maximum moves, final O / l staged per warp in shared
//               memory and written with coalesced 16-byte stores
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
// stays, P is exactly 0 and O is multiplied by exactly 1).  O starts at zero and
// is always accumulated, so the first visible tile takes the same path alone or
// packed.  No result depends on which CTA runs an item.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"
#include "runtime.h"

namespace spinf {
namespace {

using namespace dev;

constexpr int kAttnThreads = 384;      // Q/K producer, MMA, V producer, 8 softmax warps, mask metadata
constexpr int kSoftmaxThreads = 256;
constexpr int kFirstSoftmaxWarp = 3;
constexpr int kMetaWarp = 11;
constexpr int kMetaSlots = 4;          // mask-metadata ring: tiles the metadata warp may run ahead
constexpr int kBoxBytes = 128 * 128;   // one TMA box: 128 rows x 64 bf16 (128-byte swizzled rows)
constexpr int kOstageBytes = 32 * 64;  // O staging of one softmax warp: 32 rows x 32 bf16

enum { Q_FULL = 0, Q_EMPTY, S_FULL0, S_FULL1, P_FULL, O_DONE, PV_DONE0, PV_DONE1, N_FIXED_BARS };

template <int D, int MODE>
struct AttnSmem {
    static constexpr int kChunks = D / 64;
    static constexpr int kTileBytes = kChunks * kBoxBytes;
    // a cta_group::2 pair keeps half of every K tile (64 keys) and of every V tile (D/2 columns) per CTA
    static constexpr int kKBytes = MODE == 2 ? kTileBytes / 2 : kTileBytes;
    static constexpr int kVBytes = MODE == 2 ? kTileBytes / 2 : kTileBytes;
    static constexpr int kStages = (MODE == 2 || D <= 128) ? 2 : 1;   // K and V buffers each (d 256 alone: one)
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kTileBytes;                // K stage s at kK + s * kKBytes
    static constexpr int kV = kK + kStages * kKBytes;
    static constexpr int kMeta = kV + kStages * kVBytes;    // int32 [kMetaSlots][2][128]: end[], pos[] of a tile's keys
    static constexpr int kMetaHead = kMeta + kMetaSlots * 2 * 128 * 4;   // int32 [kMetaSlots][4]: min end, min pos, kv0, len
    static constexpr int kXmax = kMetaHead + kMetaSlots * 4 * 4;   // float [2][2][128]: row maxima of the two halves
    static constexpr int kLx = kXmax + 2 * 2 * 128 * 4;     // float [2][128]: the halves' row sums, per item
    static constexpr int kOstage = (kLx + 2 * 128 * 4 + 1023) / 1024 * 1024;  // per softmax warp: 32 x 32 O bf16
    // fixed barriers, then K_FULL, K_EMPTY, V_FULL, V_EMPTY [kStages], META_FULL, META_EMPTY [kMetaSlots]
    static constexpr int kBars = kOstage + 8 * kOstageBytes;
    static constexpr int kNumBars = N_FIXED_BARS + 4 * kStages + 2 * kMetaSlots;
    static constexpr int kHolder = kBars + kNumBars * 8;
    static constexpr int kBytes = kHolder + 16;
    static constexpr int kAlloc = kBytes + 1024;            // room to align the base to 1024
    static_assert(kAlloc <= 227 * 1024, "shared memory of one CTA");
};

// TMEM columns: two S buffers [0,128) and [128,256) -- tile G uses buffer G&1,
// and its P (bf16 pairs, 64 columns) overwrites the start of that buffer once
// the softmax has read S -- then O [256, 256 + D).  512 columns, so one CTA per
// SM (the shared-memory request enforces it and no allocation ever waits).
constexpr uint32_t kColO = 256;
constexpr uint32_t kTmemCols = 512;
constexpr int kMinSmem = 116 * 1024;
// Log2 headroom of the lazy softmax reference maximum: P values stay <= 2^8.
constexpr float kRescaleLog2 = 8.f;

struct Item {
    int qt, h, s0, n;
};

// MODE 0: one CTA per item (one query head).  MODE 1: clusters of two CTAs, two heads of a
// kv group, K/V tiles multicast to both.  MODE 2: cta_group::2 pairs -- the leader issues
// M = 256 MMAs over both CTAs' rows, each CTA holding half of every K and V tile.
template <int D, int MODE>
__global__ void __launch_bounds__(kAttnThreads, 1)
    branch_attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_kh,
                            const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ o,
                            const int32_t* __restrict__ end, const int32_t* __restrict__ pos,
                            const int32_t* __restrict__ qt_work, const int32_t* __restrict__ tile_kv,
                            const int32_t* __restrict__ tile_len, int T, int Hq, int Hkv, int n_items,
                            float scale_log2, int window, int* __restrict__ err) {
    static_assert(MODE != 2 || D >= 128, "a cta_group::2 pair splits V into 64-column boxes");
    using L = AttnSmem<D, MODE>;
    constexpr bool PAIR = MODE != 0;
    constexpr bool CG2 = MODE == 2;
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
    const int head_groups = Hq / heads_per_item;
    // item it = (position it / head_groups in the work order, head group it % head_groups);
    // one 16-byte record {qt, first schedule entry, entry count, 0} per Q tile
    auto item = [&](int it) {
        const int4 w = __ldg(reinterpret_cast<const int4*>(qt_work) + it / head_groups);
        Item I;
        I.qt = w.x;
        I.s0 = w.y;
        I.n = w.z;
        I.h = (it % head_groups) * heads_per_item + rank;
        return I;
    };
    // the k-th item of this CTA (pair): rounds of n_units items, every other round
    // reversed, so that long and short items spread evenly over the CTAs
    auto item_index = [&](int k) { return k * n_units + ((k & 1) ? n_units - 1 - unit : unit); };

    uint64_t* k_full = bars + N_FIXED_BARS;
    uint64_t* k_empty = k_full + L::kStages;
    uint64_t* v_full = k_empty + L::kStages;
    uint64_t* v_empty = v_full + L::kStages;
    uint64_t* meta_full = v_empty + L::kStages;
    uint64_t* meta_empty = meta_full + kMetaSlots;
    if (threadIdx.x == 0) {
        // P_FULL: every softmax thread, or (CG2) one arrival from each CTA of the pair
        for (int b = 0; b < N_FIXED_BARS; ++b) mbar_init(&bars[b], b == P_FULL ? (CG2 ? 2 : kSoftmaxThreads) : 1);
        for (int st = 0; st < L::kStages; ++st) {
            mbar_init(&k_full[st], 1);
            mbar_init(&v_full[st], 1);
            mbar_init(&k_empty[st], MODE == 1 ? 2 : 1);   // MODE 1: released by the MMAs of both CTAs
            mbar_init(&v_empty[st], MODE == 1 ? 2 : 1);
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
    if (PAIR) cluster_sync();   // the peer's barriers exist before anything is multicast to them
    tc_fence_after();
    const uint32_t tmem = *holder;
    constexpr uint16_t kBoth = 0x3;

    if (warp == 0) {
        // ---------------------------------------------------------- Q and K producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(CG2 ? &tm_kh : &tm_k);
            uint32_t G = 0, ic = 0;
            for (int k = 0;; ++k) {
                const int it = item_index(k);
                if (it >= n_items) break;
                const Item I = item(it);
                if (I.n <= 0) continue;
                if (ic > 0) mbar_wait(&bars[Q_EMPTY], (ic - 1) & 1, err);   // the last S of the previous item is done
                if constexpr (CG2) {   // both CTAs' Q tiles are counted on the leader's barrier
                    if (rank == 0) mbar_arrive_expect_tx(&bars[Q_FULL], 2 * L::kTileBytes);
                    const uint32_t qf = mapa_shared(smem_u32(&bars[Q_FULL]), 0);
                    for (int c = 0; c < L::kChunks; ++c)
                        tma_load_3d_pair(sQ + c * kBoxBytes, &tm_q, qf, c * 64, I.h, I.qt * 128);
                } else {
                    mbar_arrive_expect_tx(&bars[Q_FULL], L::kTileBytes);
                    for (int c = 0; c < L::kChunks; ++c)
                        tma_load_3d(sQ + c * kBoxBytes, &tm_q, &bars[Q_FULL], c * 64, I.h, I.qt * 128);
                }
                int kv_next = __ldg(tile_kv + I.s0);
                for (int j = 0; j < I.n; ++j, ++G) {
                    const int kv0 = kv_next;
                    if (j + 1 < I.n) kv_next = __ldg(tile_kv + I.s0 + j + 1);
                    const uint32_t st = G % L::kStages;
                    if (G >= (uint32_t)L::kStages) mbar_wait(&k_empty[st], (G / L::kStages - 1) & 1, err);
                    if constexpr (CG2) {   // keys [64 rank, 64 rank + 64) of the tile, counted on the leader
                        if (rank == 0) mbar_arrive_expect_tx(&k_full[st], 2 * L::kKBytes);
                        const uint32_t kf = mapa_shared(smem_u32(&k_full[st]), 0);
                        for (int c = 0; c < L::kChunks; ++c)
                            tma_load_3d_pair(sK + st * L::kKBytes + c * (kBoxBytes / 2), &tm_kh, kf, c * 64,
                                             I.h / group, kv0 + 64 * rank);
                    } else {
                        mbar_arrive_expect_tx(&k_full[st], L::kTileBytes);
                        for (int c = 0; c < L::kChunks; ++c) {
                            uint8_t* dst = sK + st * L::kKBytes + c * kBoxBytes;
                            if (!PAIR) tma_load_3d(dst, &tm_k, &k_full[st], c * 64, I.h / group, kv0);
                            else if ((c & 1) == rank) tma_load_3d_mc(dst, &tm_k, &k_full[st], c * 64, I.h / group, kv0, kBoth);
                        }
                    }
                }
                ++ic;
            }
            // our last copies have landed before the CTA may retire
            // (CG2: a peer's copies are counted on the leader, whose release implies they landed)
            for (uint32_t b = G > (uint32_t)L::kStages ? G - L::kStages : 0; b < G; ++b) {
                if (!CG2 || rank == 0) mbar_wait(&k_full[b % L::kStages], (b / L::kStages) & 1, err);
                mbar_wait(&k_empty[b % L::kStages], (b / L::kStages) & 1, err);   // every release has arrived
            }
            if (ic > 0) {
                if (!CG2 || rank == 0) mbar_wait(&bars[Q_FULL], (ic - 1) & 1, err);
                if (CG2) mbar_wait(&bars[Q_EMPTY], (ic - 1) & 1, err);
            }
        }
    } else if (warp == 2) {
        // ---------------------------------------------------------- V producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_v);
            uint32_t G = 0;
            for (int k = 0;; ++k) {
                const int it = item_index(k);
                if (it >= n_items) break;
                const Item I = item(it);
                if (I.n <= 0) continue;
                int kv_next = __ldg(tile_kv + I.s0);
                for (int j = 0; j < I.n; ++j, ++G) {
                    const int kv0 = kv_next;
                    if (j + 1 < I.n) kv_next = __ldg(tile_kv + I.s0 + j + 1);
                    const uint32_t st = G % L::kStages;
                    if (G >= (uint32_t)L::kStages) mbar_wait(&v_empty[st], (G / L::kStages - 1) & 1, err);
                    if constexpr (CG2) {   // columns [D/2 rank, D/2 rank + D/2) of the tile, counted on the leader
                        if (rank == 0) mbar_arrive_expect_tx(&v_full[st], 2 * L::kVBytes);
                        const uint32_t vf = mapa_shared(smem_u32(&v_full[st]), 0);
                        for (int cc = 0; cc < L::kChunks / 2; ++cc)
                            tma_load_3d_pair(sV + st * L::kVBytes + cc * kBoxBytes, &tm_v, vf,
                                             (rank * (L::kChunks / 2) + cc) * 64, I.h / group, kv0);
                    } else {
                        mbar_arrive_expect_tx(&v_full[st], L::kTileBytes);
                        for (int c = 0; c < L::kChunks; ++c) {
                            uint8_t* dst = sV + st * L::kVBytes + c * kBoxBytes;
                            if (!PAIR) tma_load_3d(dst, &tm_v, &v_full[st], c * 64, I.h / group, kv0);
                            else if ((c & 1) == rank) tma_load_3d_mc(dst, &tm_v, &v_full[st], c * 64, I.h / group, kv0, kBoth);
                        }
                    }
                }
            }
            for (uint32_t b = G > (uint32_t)L::kStages ? G - L::kStages : 0; b < G; ++b) {
                if (!CG2 || rank == 0) mbar_wait(&v_full[b % L::kStages], (b / L::kStages) & 1, err);
                mbar_wait(&v_empty[b % L::kStages], (b / L::kStages) & 1, err);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0 && (!CG2 || rank == 0)) {   // a pair's MMAs are all issued by its leader
            constexpr uint32_t idesc_qk = idesc_bf16(CG2 ? 256 : 128, 128, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16(CG2 ? 256 : 128, D, false, true);
            auto commit = [&](uint64_t* bar) {
                if constexpr (CG2) mma_commit_pair(bar); else mma_commit(bar);
            };
            const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
            // S(Gs) goes to buffer Gs&1, which held P(Gs-2): PV(Gs-2) must be done.  PV_DONE[b]
            // completes once per PV that read buffer b, so its phases cannot be overtaken here.
            auto issue_s = [&](uint32_t Gs) {
                if (Gs >= 2) mbar_wait(&bars[PV_DONE0 + (Gs & 1)], ((Gs - 2) >> 1) & 1, err);
                const uint32_t st = Gs % L::kStages;
                mbar_wait(&k_full[st], (Gs / L::kStages) & 1, err);
                tc_fence_after();
                const uint32_t dS = tmem + (Gs & 1) * 128;
                const uint32_t aKs = aK + st * L::kKBytes;
                constexpr int kKBox = CG2 ? kBoxBytes / 2 : kBoxBytes;   // K boxes hold 64 or 128 keys
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                    const uint32_t koff = (kk >> 2) * kKBox + (kk & 3) * 32;
                    if constexpr (CG2)
                        mma_f16_ss_pair(dS, sdesc_sw128(aQ + off, 16, 1024), sdesc_sw128(aKs + koff, 16, 1024),
                                        idesc_qk, kk > 0);
                    else
                        mma_f16_ss(dS, sdesc_sw128(aQ + off, 16, 1024), sdesc_sw128(aKs + koff, 16, 1024), idesc_qk,
                                   kk > 0);
                }
                if constexpr (MODE == 1) mma_commit_mc(&k_empty[st], kBoth); else commit(&k_empty[st]);
                commit(&bars[S_FULL0 + (Gs & 1)]);
            };
            uint32_t G = 0, ic = 0;
            for (int k = 0;; ++k) {
                const int it = item_index(k);
                if (it >= n_items) break;
                const Item I = item(it);
                if (I.n <= 0) continue;
                const uint32_t G0 = G;
                mbar_wait(&bars[Q_FULL], ic & 1, err);
                issue_s(G0);
                if (I.n == 1) commit(&bars[Q_EMPTY]);
                for (int j = 0; j < I.n; ++j) {
                    const uint32_t Gj = G0 + j;
                    if (j + 1 < I.n) {
                        issue_s(Gj + 1);
                        if (j + 2 == I.n) commit(&bars[Q_EMPTY]);   // Q is free once this S is done
                    }
                    if constexpr (CG2) mbar_wait_cluster(&bars[P_FULL], Gj & 1, err);   // the peer arrives remotely
                    else mbar_wait(&bars[P_FULL], Gj & 1, err);
                    const uint32_t st = Gj % L::kStages;
                    mbar_wait(&v_full[st], (Gj / L::kStages) & 1, err);
                    tc_fence_after();
                    const uint32_t aP = tmem + (Gj & 1) * 128;
                    const uint32_t aVs = aV + st * L::kVBytes;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {   // 16 keys: 8 TMEM columns of bf16 pairs of P
                        const uint64_t db = sdesc_sw128(aVs + kk * 2048, kBoxBytes, 1024);
                        if constexpr (CG2) mma_f16_ts_pair(tmem + kColO, aP + kk * 8, db, idesc_pv, 1);
                        else mma_f16_ts(tmem + kColO, aP + kk * 8, db, idesc_pv, 1);
                    }
                    if constexpr (MODE == 1) mma_commit_mc(&v_empty[st], kBoth); else commit(&v_empty[st]);
                    commit(&bars[O_DONE]);
                    commit(&bars[PV_DONE0 + (Gj & 1)]);
                }
                G += I.n;
                ++ic;
            }
        }
    } else if (warp == kMetaWarp) {
        // ---------------------------------------------------------- mask metadata of each KV tile
        // end[] and pos[] of the tile's 128 keys (keys past the tile's own input: end -1,
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
                int ev[4], pv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int key = lane + 32 * i;
                    ev[i] = key < len ? __ldg(end + kv0 + key) : -1;
                    pv[i] = key < len ? __ldg(pos + kv0 + key) : 0;
                }
                const int emin = __reduce_min_sync(0xffffffffu, min(min(ev[0], ev[1]), min(ev[2], ev[3])));
                const int pmin = __reduce_min_sync(0xffffffffu, min(min(pv[0], pv[1]), min(pv[2], pv[3])));
                if (G >= (uint32_t)kMetaSlots) mbar_wait(&meta_empty[slot], (G / kMetaSlots - 1) & 1, err);
                int32_t* me = meta + slot * 256;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    me[lane + 32 * i] = ev[i];
                    me[128 + lane + 32 * i] = pv[i];
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
        const uint32_t tO = tmem + lane_off + kColO + half * (D / 2);
        const uint32_t pair_bar = 2 + quarter;        // the two warps that share these TMEM lanes
        float* xmax = reinterpret_cast<float*>(smem + L::kXmax);
        float* lx = reinterpret_cast<float*>(smem + L::kLx);

        auto zero_o = [&]() {
            uint32_t z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) tmem_st32(tO + c * 32, z);
            tmem_st_wait();
        };

        zero_o();
        uint32_t G = 0;
        int k = 0;
        int it = item_index(0);
        Item I = it < n_items ? item(it) : Item{0, 0, 0, 0};
        while (it < n_items) {
            // the next item's record is loaded while this one runs
            const int it_next = item_index(k + 1);
            const Item I_next = it_next < n_items ? item(it_next) : Item{0, 0, 0, 0};
            if (I.n > 0) {
            const int q_row = I.qt * 128 + r;
            const bool real = q_row < T;
            const int pos_q = __ldg(pos + q_row);
            float m = -INFINITY, l = 0.f;   // l: this half's share of the row sum
            for (int j = 0; j < I.n; ++j, ++G) {
                const int b = G & 1;
                const int slot = G % kMetaSlots;
                mbar_wait(&meta_full[slot], (G / kMetaSlots) & 1, err);
                const int4 head = *reinterpret_cast<const int4*>(meta_head + 4 * slot);   // min end, min pos, kv0, len
                mbar_wait(&bars[S_FULL0 + b], (G >> 1) & 1, err);
                tc_fence_after();
                const uint32_t tS = tmem + lane_off + b * 128;
                float s[64];
                {
                    uint32_t rr[64];
                    tmem_ld64(tS + half * 64, rr);
#pragma unroll
                    for (int i = 0; i < 64; ++i) s[i] = __uint_as_float(rr[i]);
                }
                // visible: kv0 + c <= q_row (causal), q_row < end[key], window on depth.
                // A tile whose every key is visible to this row skips the per-key test.
                const int cmax = real ? q_row - head.z : -1;
                const bool all_visible =
                    cmax >= 127 && head.x > q_row && (window <= 0 || pos_q - head.y < window);
                float mx = -INFINITY;
                if (all_visible) {
#pragma unroll
                    for (int i = 0; i < 64; ++i) mx = fmaxf(mx, s[i]);
                } else {
                    const int4* e4 = reinterpret_cast<const int4*>(meta + slot * 256 + half * 64);
                    const int4* p4 = reinterpret_cast<const int4*>(meta + slot * 256 + 128 + half * 64);
                    const int cm = cmax - half * 64;
#pragma unroll
                    for (int c4 = 0; c4 < 16; ++c4) {
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
                uint32_t pk[32];
                float alpha = 1.f;
                float rowsum = 0.f;
                if (m_new == -INFINITY) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) pk[i] = 0u;
                } else {
                    const float mb = m_new * scale_log2;
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float p0 = fast_exp2(fmaf(s[2 * c], scale_log2, -mb));
                        const float p1 = fast_exp2(fmaf(s[2 * c + 1], scale_log2, -mb));
                        rowsum += p0;
                        rowsum += p1;
                        pk[c] = pack_bf16x2(p0, p1);
                    }
                    if (grow) alpha = fast_exp2(fmaf(m, scale_log2, -mb));
                }
                if (j > 0) {   // PV of the previous tile has written O and read its P
                    mbar_wait(&bars[O_DONE], (G - 1) & 1, err);
                    tc_fence_after();
                }
                if (m_new != -INFINITY) {
                    l = l * alpha + rowsum;
                    m = m_new;
                }
                // TMEM traffic is warp-collective: lanes whose maximum did not move multiply by exactly 1
                if (__any_sync(0xffffffffu, grow)) {
#pragma unroll 1
                    for (int c = 0; c < D / 64; ++c) {
                        uint32_t rr[32];
                        tmem_ld32(tO + c * 32, rr);
#pragma unroll
                        for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
                        tmem_st32(tO + c * 32, rr);
                    }
                }
                // P of keys [64 half, 64 half + 64) -> bf16 pairs in columns [32 half, 32 half + 32)
                // of this tile's S buffer (both halves have read their S columns before the pair barrier)
                tmem_st32(tS + half * 32, pk);
                tmem_st_wait();
                tc_fence_before();
                if constexpr (CG2) {   // one arrival per CTA on the leader's barrier
                    named_bar_sync(1, kSoftmaxThreads);
                    if (t == 0) {
                        if (rank == 0) mbar_arrive(&bars[P_FULL]);
                        else mbar_arrive_cluster(mapa_shared(smem_u32(&bars[P_FULL]), 0));
                    }
                } else {
                    mbar_arrive(&bars[P_FULL]);
                }
            }
            // epilogue of the item: O / l to global memory, then O back to zero for the next item
            mbar_wait(&bars[O_DONE], (G - 1) & 1, err);
            tc_fence_after();
            lx[half * 128 + r] = l;
            named_bar_sync(pair_bar, 64);
            const float lrow = lx[r] + lx[128 + r];      // halves added in a fixed order
            const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
            // this warp's 32 rows x D/2 columns, 32 columns at a time: each lane writes its row
            // into a 2 KB staging box, then the warp stores 8 rows (4 lanes x 16 bytes each) per
            // instruction.  Row x's 16-byte pieces sit at slots piece ^ ((x >> 1) & 3), so both
            // the row writes and the 8-row reads are free of bank conflicts.
            uint8_t* stage = smem + L::kOstage + sw * kOstageBytes;
            __nv_bfloat16* orow = o + (static_cast<size_t>(I.qt * 128 + quarter * 32) * Hq + I.h) * D;
            const size_t ostride = static_cast<size_t>(Hq) * D;
            auto store_chunk = [&](const uint32_t* rr, int col) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[i] = real ? pack_bf16x2(__uint_as_float(rr[2 * i]) * inv, __uint_as_float(rr[2 * i + 1]) * inv)
                                : 0u;
                uint4* srow = reinterpret_cast<uint4*>(stage + lane * 64);
                const int sx = (lane >> 1) & 3;
#pragma unroll
                for (int i = 0; i < 4; ++i) srow[i ^ sx] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                __syncwarp();
                const int piece = lane & 3;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int x = i * 8 + (lane >> 2);
                    const uint4 val = reinterpret_cast<const uint4*>(stage + x * 64)[piece ^ ((x >> 1) & 3)];
                    *reinterpret_cast<uint4*>(orow + x * ostride + col + piece * 8) = val;
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
            zero_o();
            // lx is read by the partner before either writes it again (next item's epilogue)
            named_bar_sync(pair_bar, 64);
            }
            I = I_next;
            it = it_next;
            ++k;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();   // nothing of the peer still lands in this CTA
    if (warp == 1) {
        tc_fence_after();
        if constexpr (CG2) tmem_dealloc_pair(tmem, kTmemCols);
        else tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, int MODE>
spinf_status launch_mode(const Pass& P, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tkh,
                         const CUtensorMap& tv, __nv_bfloat16* o, int Hq, int Hkv, float scale_log2, int window,
                         int* err, cudaStream_t stream) {
    auto kernel = branch_attention_kernel<D, MODE>;
    const int smem = AttnSmem<D, MODE>::kAlloc > kMinSmem ? AttnSmem<D, MODE>::kAlloc : kMinSmem;
    static bool configured = false;
    cudaError_t e;
    if (!configured) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attention)");
        configured = true;
    }
    const int heads_per_item = MODE == 0 ? 1 : 2;
    const int n_items = (P.T_pad / 128) * (Hq / heads_per_item);
    if (MODE == 0) {
        const int grid = std::min(n_items, sm_count());
        kernel<<<grid, kAttnThreads, smem, stream>>>(tq, tk, tkh, tv, o, P.dev.end, P.dev.pos, P.dev.qt_work,
                                                     P.dev.tile_kv, P.dev.tile_len, P.T, Hq, Hkv, n_items,
                                                     scale_log2, window, err);
    } else {   // clusters of two CTAs, two heads of a kv group per item
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
        e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tkh, tv, o, (const int32_t*)P.dev.end,
                               (const int32_t*)P.dev.pos, (const int32_t*)P.dev.qt_work,
                               (const int32_t*)P.dev.tile_kv, (const int32_t*)P.dev.tile_len, P.T, Hq, Hkv, n_items,
                               scale_log2, window, err);
        if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    return SPINF_OK;
}

template <int D>
spinf_status launch_attention(const Pass& P, const void* q, const void* k, const void* v, void* o, int Hq,
                              int Hkv, float scale, int window, int* err, cudaStream_t stream) {
    CUtensorMap tq, tk, tkh, tv;
    const uint64_t dq[3] = {(uint64_t)D, (uint64_t)Hq, (uint64_t)P.T_pad};
    const uint64_t sq[2] = {(uint64_t)D * 2, (uint64_t)Hq * D * 2};
    const uint64_t dk[3] = {(uint64_t)D, (uint64_t)Hkv, (uint64_t)P.T_pad};
    const uint64_t sk[2] = {(uint64_t)D * 2, (uint64_t)Hkv * D * 2};
    const uint32_t box[3] = {64, 1, 128};
    const uint32_t hbox[3] = {64, 1, 64};   // half a K tile: the keys one CTA of a pair holds
    spinf_status st;
    if ((st = make_tmap(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dq, sq, box, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    if ((st = make_tmap(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k, dk, sk, box, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    if ((st = make_tmap(&tkh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k, dk, sk, hbox, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    if ((st = make_tmap(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, v, dk, sk, box, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(o);
    const float scale_log2 = scale * 1.4426950408889634f;
    // an even number of query heads per kv head pairs two heads per item: d_head 128 as a
    // cta_group::2 pair (half tiles), d_head 64 and 256 as a multicast pair (at 256 the
    // multicast pair measured faster: its softmax warps are not coupled across the two SMs)
    if ((Hq / Hkv) % 2 != 0) return launch_mode<D, 0>(P, tq, tk, tkh, tv, ob, Hq, Hkv, scale_log2, window, err, stream);
    if constexpr (D == 128)
        return launch_mode<D, 2>(P, tq, tk, tkh, tv, ob, Hq, Hkv, scale_log2, window, err, stream);
    else
        return launch_mode<D, 1>(P, tq, tk, tkh, tv, ob, Hq, Hkv, scale_log2, window, err, stream);
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
    if (P.T == 0) return SPINF_OK;
    if (!(scale > 0.f)) scale = 1.0f / std::sqrt(static_cast<float>(d_head));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (d_head) {
        case 64: return launch_attention<64>(P, q, k, v, o, n_q_heads, n_kv_heads, scale, window, plan->d_err, s);
        case 128: return launch_attention<128>(P, q, k, v, o, n_q_heads, n_kv_heads, scale, window, plan->d_err, s);
        case 256: return launch_attention<256>(P, q, k, v, o, n_q_heads, n_kv_heads, scale, window, plan->d_err, s);
        default: return fail(SPINF_E_UNSUPPORTED, "d_head must be 64, 128 or 256");
    }
}
