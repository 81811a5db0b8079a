// Tree-masked GQA attention over one packed pass (sm_103a, tcgen05 + TMA).
//
// The method ("spinf-serve 0.1.1", PyPI page, "What it does" and "Speed and
// scale"): every question is a branch of the same pass; a branch token attends
// to its own content and causally to its own branch, never to a sibling or to
// another packed input.  The planner encodes that as: key k is visible to the
// rows [k, end[k]), and each scheduled KV tile holds only its own input's keys.
//
// Persistent kernel: one CTA per SM walks a static list of work items, an item
// being one 128-row Q tile of one query head (items of the same Q tile and
// neighbouring heads run side by side on neighbouring SMs, so a kv head's tiles
// are read from L2 by its query heads at about the same time).  When a kv group
// has an even number of query heads, CTAs run as clusters of two that take two
// heads of one group on the same Q tile: each CTA loads half of every K and V
// tile and multicasts it to both, so each tile leaves L2 once per pair, and a
// buffer is refilled only when both CTAs' MMAs have released it.  Warp roles:
//   warp 0      TMA producer of Q (once per item) and K tiles (two buffers for
//               d_head <= 128; one for 256, where Q, K and V fill shared memory)
//   warp 1      TMEM owner and MMA issuer: S = Q K^T into one of two TMEM
//               buffers (SS form, fp32), O += P V (P read from TMEM, V MN-major
//               from shared memory)
//   warp 2      TMA producer of V tiles (buffered like K)
//   warps 3-10  softmax, two warps per TMEM lane quarter: each thread owns half
//               of one Q row (64 of the 128 key columns, D/2 of the O columns):
//               mask, online softmax with the row maximum exchanged between the
//               two halves, P (bf16) into TMEM over its S, rescale O when the
//               reference maximum moves, final O / l written by TMA stores of 32 x 32
//               boxes staged per warp
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

constexpr int kAttnThreads = 352;      // Q/K producer, MMA, V producer, 8 softmax warps
constexpr int kSoftmaxThreads = 256;
constexpr int kFirstSoftmaxWarp = 3;
constexpr int kBoxBytes = 128 * 128;   // one TMA box: 128 rows x 64 bf16 (128-byte swizzled rows)
constexpr int kOstageBytes = 32 * 64;  // O store box of one softmax warp: 32 rows x 32 bf16, row-major

enum { Q_FULL = 0, Q_EMPTY, S_FULL0, S_FULL1, P_FULL, O_DONE, PV_DONE0, PV_DONE1, N_FIXED_BARS };

template <int D>
struct AttnSmem {
    static constexpr int kChunks = D / 64;
    static constexpr int kTileBytes = kChunks * kBoxBytes;
    static constexpr int kStages = D <= 128 ? 2 : 1;          // K and V tile buffers each (d 256: no room for two)
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kTileBytes;                // K stage s at kK + s * kTileBytes
    static constexpr int kV = kK + kStages * kTileBytes;
    static constexpr int kKvEnd = kV + kStages * kTileBytes;  // int32 [2][128]
    static constexpr int kKvPos = kKvEnd + 2 * 128 * 4;     // int32 [2][128]
    static constexpr int kXmax = kKvPos + 2 * 128 * 4;      // float [2][2][128]: row maxima of the two halves
    static constexpr int kLx = kXmax + 2 * 2 * 128 * 4;     // float [2][128]: the halves' row sums, per item
    static constexpr int kTmin = kLx + 2 * 128 * 4;         // int [2][8]: per-warp minima of end / pos
    static constexpr int kOstage = (kTmin + 2 * 8 * 4 + 1023) / 1024 * 1024;  // per softmax warp: 32 x 32 O bf16
    static constexpr int kBars = kOstage + 8 * kOstageBytes;   // fixed barriers, then K_FULL, K_EMPTY, V_FULL, V_EMPTY [kStages]
    static constexpr int kNumBars = N_FIXED_BARS + 4 * kStages;
    static constexpr int kHolder = kBars + kNumBars * 8;
    static constexpr int kBytes = kHolder + 16;
    static constexpr int kAlloc = kBytes + 1024;            // room to align the base to 1024
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

__device__ __forceinline__ Item item_at(int it, int Hq, const int32_t* __restrict__ tile_ptr) {
    Item I;
    I.qt = it / Hq;
    I.h = it - I.qt * Hq;
    I.s0 = __ldg(tile_ptr + I.qt);
    I.n = __ldg(tile_ptr + I.qt + 1) - I.s0;
    return I;
}

template <int D, bool PAIR>
__global__ void __launch_bounds__(kAttnThreads, 1)
    branch_attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                            const int32_t* __restrict__ end, const int32_t* __restrict__ pos,
                            const int32_t* __restrict__ tile_ptr, const int32_t* __restrict__ tile_kv,
                            const int32_t* __restrict__ tile_len, int T, int Hq, int Hkv, int n_items,
                            float scale_log2, int window, int* __restrict__ err) {
    using L = AttnSmem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + L::kQ;
    uint8_t* sK = smem + L::kK;
    uint8_t* sV = smem + L::kV;
    int32_t* kv_end = reinterpret_cast<int32_t*>(smem + L::kKvEnd);
    int32_t* kv_pos = reinterpret_cast<int32_t*>(smem + L::kKvPos);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
    uint32_t* holder = reinterpret_cast<uint32_t*>(smem + L::kHolder);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = Hq / Hkv;
    // PAIR: item = (Q tile, pair of heads 2p, 2p+1 of one kv group); this CTA takes head 2p + rank
    const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
    const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int n_units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    const int heads_per_item = PAIR ? 2 : 1;
    auto item = [&](int it) {
        Item I = item_at(it, Hq / heads_per_item, tile_ptr);
        I.h = I.h * heads_per_item + rank;
        return I;
    };

    uint64_t* k_full = bars + N_FIXED_BARS;
    uint64_t* k_empty = k_full + L::kStages;
    uint64_t* v_full = k_empty + L::kStages;
    uint64_t* v_empty = v_full + L::kStages;
    if (threadIdx.x == 0) {
        for (int b = 0; b < N_FIXED_BARS; ++b) mbar_init(&bars[b], b == P_FULL ? kSoftmaxThreads : 1);
        for (int st = 0; st < L::kStages; ++st) {
            mbar_init(&k_full[st], 1);
            mbar_init(&v_full[st], 1);
            mbar_init(&k_empty[st], PAIR ? 2 : 1);   // released by the MMAs of both CTAs of a pair
            mbar_init(&v_empty[st], PAIR ? 2 : 1);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(holder, kTmemCols);
        tmem_relinquish();
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
            tma_prefetch_desc(&tm_k);
            uint32_t G = 0, ic = 0;
            for (int it = unit; it < n_items; it += n_units) {
                const Item I = item(it);
                if (I.n <= 0) continue;
                if (ic > 0) mbar_wait(&bars[Q_EMPTY], (ic - 1) & 1, err);   // the last S of the previous item is done
                mbar_arrive_expect_tx(&bars[Q_FULL], L::kTileBytes);
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_3d(sQ + c * kBoxBytes, &tm_q, &bars[Q_FULL], c * 64, I.h, I.qt * 128);
                int kv_next = __ldg(tile_kv + I.s0);
                for (int j = 0; j < I.n; ++j, ++G) {
                    const int kv0 = kv_next;
                    if (j + 1 < I.n) kv_next = __ldg(tile_kv + I.s0 + j + 1);
                    const uint32_t st = G % L::kStages;
                    if (G >= (uint32_t)L::kStages) mbar_wait(&k_empty[st], (G / L::kStages - 1) & 1, err);
                    mbar_arrive_expect_tx(&k_full[st], L::kTileBytes);
                    for (int c = 0; c < L::kChunks; ++c) {
                        uint8_t* dst = sK + st * L::kTileBytes + c * kBoxBytes;
                        if (!PAIR) tma_load_3d(dst, &tm_k, &k_full[st], c * 64, I.h / group, kv0);
                        else if ((c & 1) == rank) tma_load_3d_mc(dst, &tm_k, &k_full[st], c * 64, I.h / group, kv0, kBoth);
                    }
                }
                ++ic;
            }
            // our last copies have landed before the CTA may retire
            for (uint32_t b = G > (uint32_t)L::kStages ? G - L::kStages : 0; b < G; ++b) {
                mbar_wait(&k_full[b % L::kStages], (b / L::kStages) & 1, err);
                mbar_wait(&k_empty[b % L::kStages], (b / L::kStages) & 1, err);   // every release has arrived
            }
            if (ic > 0) mbar_wait(&bars[Q_FULL], (ic - 1) & 1, err);
        }
    } else if (warp == 2) {
        // ---------------------------------------------------------- V producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_v);
            uint32_t G = 0;
            for (int it = unit; it < n_items; it += n_units) {
                const Item I = item(it);
                if (I.n <= 0) continue;
                int kv_next = __ldg(tile_kv + I.s0);
                for (int j = 0; j < I.n; ++j, ++G) {
                    const int kv0 = kv_next;
                    if (j + 1 < I.n) kv_next = __ldg(tile_kv + I.s0 + j + 1);
                    const uint32_t st = G % L::kStages;
                    if (G >= (uint32_t)L::kStages) mbar_wait(&v_empty[st], (G / L::kStages - 1) & 1, err);
                    mbar_arrive_expect_tx(&v_full[st], L::kTileBytes);
                    for (int c = 0; c < L::kChunks; ++c) {
                        uint8_t* dst = sV + st * L::kTileBytes + c * kBoxBytes;
                        if (!PAIR) tma_load_3d(dst, &tm_v, &v_full[st], c * 64, I.h / group, kv0);
                        else if ((c & 1) == rank) tma_load_3d_mc(dst, &tm_v, &v_full[st], c * 64, I.h / group, kv0, kBoth);
                    }
                }
            }
            for (uint32_t b = G > (uint32_t)L::kStages ? G - L::kStages : 0; b < G; ++b) {
                mbar_wait(&v_full[b % L::kStages], (b / L::kStages) & 1, err);
                mbar_wait(&v_empty[b % L::kStages], (b / L::kStages) & 1, err);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16(128, 128, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16(128, D, false, true);
            const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
            // S(Gs) goes to buffer Gs&1, which held P(Gs-2): PV(Gs-2) must be done.  PV_DONE[b]
            // completes once per PV that read buffer b, so its phases cannot be overtaken here.
            auto issue_s = [&](uint32_t Gs) {
                if (Gs >= 2) mbar_wait(&bars[PV_DONE0 + (Gs & 1)], ((Gs - 2) >> 1) & 1, err);
                const uint32_t st = Gs % L::kStages;
                mbar_wait(&k_full[st], (Gs / L::kStages) & 1, err);
                tc_fence_after();
                const uint32_t dS = tmem + (Gs & 1) * 128;
                const uint32_t aKs = aK + st * L::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                    mma_f16_ss(dS, sdesc_sw128(aQ + off, 16, 1024), sdesc_sw128(aKs + off, 16, 1024), idesc_qk,
                               kk > 0);
                }
                if (PAIR) mma_commit_mc(&k_empty[st], kBoth); else mma_commit(&k_empty[st]);
                mma_commit(&bars[S_FULL0 + (Gs & 1)]);
            };
            uint32_t G = 0, ic = 0;
            for (int it = unit; it < n_items; it += n_units) {
                const Item I = item(it);
                if (I.n <= 0) continue;
                const uint32_t G0 = G;
                mbar_wait(&bars[Q_FULL], ic & 1, err);
                issue_s(G0);
                if (I.n == 1) mma_commit(&bars[Q_EMPTY]);
                for (int j = 0; j < I.n; ++j) {
                    const uint32_t Gj = G0 + j;
                    if (j + 1 < I.n) {
                        issue_s(Gj + 1);
                        if (j + 2 == I.n) mma_commit(&bars[Q_EMPTY]);   // Q is free once this S is done
                    }
                    const uint32_t st = Gj % L::kStages;
                    mbar_wait(&bars[P_FULL], Gj & 1, err);
                    mbar_wait(&v_full[st], (Gj / L::kStages) & 1, err);
                    tc_fence_after();
                    const uint32_t aP = tmem + (Gj & 1) * 128;
                    const uint32_t aVs = aV + st * L::kTileBytes;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_f16_ts(tmem + kColO, aP + kk * 8, sdesc_sw128(aVs + kk * 2048, kBoxBytes, 1024), idesc_pv,
                                   1);
                    if (PAIR) mma_commit_mc(&v_empty[st], kBoth); else mma_commit(&v_empty[st]);
                    mma_commit(&bars[O_DONE]);
                    mma_commit(&bars[PV_DONE0 + (Gj & 1)]);
                }
                G += I.n;
                ++ic;
            }
        }
    } else {
        // ---------------------------------------------------------- softmax and epilogue
        const int sw = warp - kFirstSoftmaxWarp;      // 0..7
        const int quarter = warp & 3;                 // TMEM lanes this warp may touch
        const int half = sw >> 2;                     // which half of the row's columns
        const int r = quarter * 32 + lane;            // Q-tile row of this thread
        const int t = sw * 32 + lane;                 // 0..255 for cooperative loads
        const int key = t & 127;                      // staging: half 0 loads end[], half 1 pos[]
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_off + kColO + half * (D / 2);
        const uint32_t pair_bar = 2 + quarter;        // the two warps that share these TMEM lanes
        float* xmax = reinterpret_cast<float*>(smem + L::kXmax);
        float* lx = reinterpret_cast<float*>(smem + L::kLx);
        int* tmin = reinterpret_cast<int*>(smem + L::kTmin);

        auto zero_o = [&]() {
            uint32_t z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) tmem_st32(tO + c * 32, z);
            tmem_st_wait();
        };
        // end[] (half 0) or pos[] (half 1) of one key of a schedule entry; keys past the
        // tile's own input are read through that input's tiles: never here
        auto stage_value = [&](int e) {
            if (e < 0) return half == 0 ? -1 : 0;
            const int kv0 = __ldg(tile_kv + e), len = __ldg(tile_len + e);
            if (key >= len) return half == 0 ? -1 : 0;
            return half == 0 ? __ldg(end + kv0 + key) : __ldg(pos + kv0 + key);
        };
        // schedule entry of the first tile of the next item with tiles, or -1
        auto first_entry_after = [&](int it) {
            for (it += n_units; it < n_items; it += n_units) {
                const Item I = item(it);
                if (I.n > 0) return I.s0;
            }
            return -1;
        };

        zero_o();
        uint32_t G = 0;
        int next = stage_value(first_entry_after(unit - n_units));
        for (int it = unit; it < n_items; it += n_units) {
            const Item I = item(it);
            if (I.n <= 0) continue;
            const int q_row = I.qt * 128 + r;
            const bool real = q_row < T;
            const int pos_q = __ldg(pos + q_row);
            float m = -INFINITY, l = 0.f;   // l: this half's share of the row sum
            for (int j = 0; j < I.n; ++j, ++G) {
                const int kv0 = __ldg(tile_kv + I.s0 + j);
                const int b = G & 1;
                int32_t* e_buf = kv_end + b * 128;
                int32_t* p_buf = kv_pos + b * 128;
                (half == 0 ? e_buf : p_buf)[key] = next;
                {   // per-warp minimum of end[] (half 0) or pos[] (half 1) over this tile's keys
                    const int wmin = __reduce_min_sync(0xffffffffu, next);
                    if (lane == 0) tmin[b * 8 + sw] = wmin;
                }
                named_bar_sync(1, kSoftmaxThreads);
                next = stage_value(j + 1 < I.n ? I.s0 + j + 1 : first_entry_after(it));
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
                const int cmax = real ? q_row - kv0 : -1;
                const int* tm = tmin + b * 8;
                const int emin = min(min(tm[0], tm[1]), min(tm[2], tm[3]));
                const int pmin = min(min(tm[4], tm[5]), min(tm[6], tm[7]));
                const bool all_visible = cmax >= 127 && emin > q_row && (window <= 0 || pos_q - pmin < window);
                float mx = -INFINITY;
                if (all_visible) {
#pragma unroll
                    for (int i = 0; i < 64; ++i) mx = fmaxf(mx, s[i]);
                } else {
                    const int4* e4 = reinterpret_cast<const int4*>(e_buf + half * 64);
                    const int4* p4 = reinterpret_cast<const int4*>(p_buf + half * 64);
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
                mbar_arrive(&bars[P_FULL]);
            }
            // epilogue of the item: O / l to global memory, then O back to zero for the next item
            mbar_wait(&bars[O_DONE], (G - 1) & 1, err);
            tc_fence_after();
            lx[half * 128 + r] = l;
            named_bar_sync(pair_bar, 64);
            const float lrow = lx[r] + lx[128 + r];      // halves added in a fixed order
            const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
            // this warp's 32 rows x D/2 columns, 32 columns at a time, through a 2 KB staging
            // box and a TMA store (the box's rows are the TMEM lanes of the warp)
            uint8_t* stage = smem + L::kOstage + sw * kOstageBytes;
            const int row0 = I.qt * 128 + quarter * 32;
            auto store_chunk = [&](const uint32_t* rr, int col) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[i] = real ? pack_bf16x2(__uint_as_float(rr[2 * i]) * inv, __uint_as_float(rr[2 * i + 1]) * inv)
                                : 0u;
                uint4* row = reinterpret_cast<uint4*>(stage + lane * 64);
#pragma unroll
                for (int i = 0; i < 4; ++i) row[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(&tm_o, stage, col, I.h, row0);
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
            zero_o();
            // lx is read by the partner before either writes it again (next item's epilogue)
            named_bar_sync(pair_bar, 64);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();   // nothing of the peer still lands in this CTA
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D>
spinf_status launch_attention(const Pass& P, const void* q, const void* k, const void* v, void* o, int Hq,
                              int Hkv, float scale, int window, int* err, cudaStream_t stream) {
    CUtensorMap tq, tk, tv, to;
    const uint64_t dq[3] = {(uint64_t)D, (uint64_t)Hq, (uint64_t)P.T_pad};
    const uint64_t sq[2] = {(uint64_t)D * 2, (uint64_t)Hq * D * 2};
    const uint64_t dk[3] = {(uint64_t)D, (uint64_t)Hkv, (uint64_t)P.T_pad};
    const uint64_t sk[2] = {(uint64_t)D * 2, (uint64_t)Hkv * D * 2};
    const uint32_t box[3] = {64, 1, 128};
    spinf_status st;
    if ((st = make_tmap(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dq, sq, box, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    if ((st = make_tmap(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k, dk, sk, box, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    if ((st = make_tmap(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, v, dk, sk, box, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    const uint32_t obox[3] = {32, 1, 32};   // one softmax warp's rows, 32 columns
    if ((st = make_tmap(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, o, dq, sq, obox, CU_TENSOR_MAP_SWIZZLE_NONE)))
        return st;
    const int smem = AttnSmem<D>::kAlloc > kMinSmem ? AttnSmem<D>::kAlloc : kMinSmem;
    const float scale_log2 = scale * 1.4426950408889634f;
    cudaError_t e;
    if ((Hq / Hkv) % 2 == 0) {   // clusters of two CTAs, two heads of a kv group per item
        auto kernel = branch_attention_kernel<D, true>;
        static bool configured = false;
        if (!configured) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attention)");
            configured = true;
        }
        const int n_items = (P.T_pad / 128) * (Hq / 2);
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
        e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, to, (const int32_t*)P.dev.end, (const int32_t*)P.dev.pos,
                               (const int32_t*)P.dev.tile_ptr, (const int32_t*)P.dev.tile_kv,
                               (const int32_t*)P.dev.tile_len, P.T, Hq, Hkv, n_items, scale_log2, window, err);
        if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    } else {
        auto kernel = branch_attention_kernel<D, false>;
        static bool configured = false;
        if (!configured) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attention)");
            configured = true;
        }
        const int n_items = (P.T_pad / 128) * Hq;
        const int grid = std::min(n_items, sm_count());
        kernel<<<grid, kAttnThreads, smem, stream>>>(tq, tk, tv, to, P.dev.end, P.dev.pos, P.dev.tile_ptr,
                                                     P.dev.tile_kv, P.dev.tile_len, P.T, Hq, Hkv, n_items, scale_log2,
                                                     window, err);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    return SPINF_OK;
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
