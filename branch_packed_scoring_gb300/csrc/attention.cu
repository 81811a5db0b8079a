// Tree-masked GQA attention over one packed pass (sm_103a, tcgen05 + TMA).
//
// The method ("spinf-serve 0.1.1", PyPI page, "What it does" and "Speed and
// scale"): every question is a branch of the same pass; a branch token attends
// to its own content and causally to its own branch, never to a sibling or to
// another packed input.  The planner encodes that as: key k is visible to the
// rows [k, end[k]), and each scheduled KV tile holds only its own input's keys.
//
// One CTA computes one 128-row Q tile of one query head:
//   warp 0      TMA producer: Q once, then K and V tiles (128 keys x d) in the
//               order of the tile's schedule
//   warp 1      TMEM owner and MMA issuer: S = Q K^T into one of two TMEM
//               buffers (SS form, fp32), O += P V (P read from TMEM, V MN-major
//               from shared memory)
//   warps 2-9   softmax, two warps per TMEM lane quarter: each thread owns half
//               of one Q row (64 of the 128 key columns, D/2 of the O columns):
//               mask, online softmax with the row maximum exchanged between the
//               two halves, P (bf16) into TMEM over its S, rescale O when the
//               reference maximum moves, final O / l staged in shared memory
//               and written by a TMA store
// With two S buffers the tensor core computes S(j+1) and PV(j-1) while the
// softmax warps work on tile j.
//
// Batch invariance ("What it does": an input's scores are bit-identical alone
// or packed with thousands of others): KV tiles start at the first row of the
// input that owns them, so a key always lands in the same MMA column whatever
// precedes its input in the pass; tiles are visited in a fixed order; a tile
// with no visible key for a row is an exact no-op for that row (its maximum
// stays, P is exactly 0 and O is multiplied by exactly 1).  O starts at zero and
// is always accumulated, so the first visible tile takes the same path alone or
// packed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"
#include "runtime.h"

namespace spinf {
namespace {

using namespace dev;

constexpr int kAttnThreads = 320;   // producer, MMA, 8 softmax warps
constexpr int kSoftmaxThreads = 256;
constexpr int kBoxBytes = 128 * 128;   // one TMA box: 128 rows x 64 bf16 (128-byte swizzled rows)
constexpr int kSchedSmem = 256;        // schedule entries staged in shared memory (later ones read from global)

enum { Q_FULL = 0, K_FULL, K_EMPTY, V_FULL, V_EMPTY, S_FULL0, S_FULL1, P_FULL, O_DONE, N_BARS };

template <int D>
struct AttnSmem {
    static constexpr int kChunks = D / 64;
    static constexpr int kTileBytes = kChunks * kBoxBytes;
    static constexpr int kQ = 0;                            // Q tile; stages O for the TMA store at the end
    static constexpr int kK = kQ + kTileBytes;
    static constexpr int kV = kK + kTileBytes;
    static constexpr int kKvEnd = kV + kTileBytes;          // int32 [2][128]
    static constexpr int kKvPos = kKvEnd + 2 * 128 * 4;     // int32 [2][128]
    static constexpr int kSched = kKvPos + 2 * 128 * 4;     // int2 [kSchedSmem]: (first row, own keys)
    static constexpr int kXmax = kSched + kSchedSmem * 8;   // float [2][2][128]: row maxima of the two halves
    static constexpr int kLx = kXmax + 2 * 2 * 128 * 4;     // float [2][128]: the halves' row sums, at the end
    static constexpr int kTmin = kLx + 2 * 128 * 4;         // int [2][8]: per-warp minima of end / pos
    static constexpr int kBars = kTmin + 2 * 8 * 4;
    static constexpr int kHolder = kBars + N_BARS * 8;
    static constexpr int kBytes = kHolder + 16;
    static constexpr int kAlloc = kBytes + 1024;            // room to align the base to 1024
};

// TMEM columns: two S buffers [0,128) and [128,256) -- tile j uses buffer j&1,
// and its P (bf16 pairs, 64 columns) overwrites the start of that buffer once
// the softmax has read S -- then O [256, 256 + D).  512 columns, so one CTA per
// SM (the shared-memory request enforces it and no allocation ever waits).
constexpr uint32_t kColO = 256;
constexpr uint32_t kTmemCols = 512;
constexpr int kMinSmem = 116 * 1024;
// Log2 headroom of the lazy softmax reference maximum: P values stay <= 2^8.
constexpr float kRescaleLog2 = 8.f;

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    branch_attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                            const int32_t* __restrict__ end, const int32_t* __restrict__ pos,
                            const int32_t* __restrict__ tile_ptr, const int32_t* __restrict__ tile_kv,
                            const int32_t* __restrict__ tile_len, int T, int Hkv, float scale_log2, int window,
                            int* __restrict__ err) {
    using L = AttnSmem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + L::kQ;
    uint8_t* sK = smem + L::kK;
    uint8_t* sV = smem + L::kV;
    int32_t* kv_end = reinterpret_cast<int32_t*>(smem + L::kKvEnd);
    int32_t* kv_pos = reinterpret_cast<int32_t*>(smem + L::kKvPos);
    int2* sched = reinterpret_cast<int2*>(smem + L::kSched);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
    uint32_t* holder = reinterpret_cast<uint32_t*>(smem + L::kHolder);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = blockIdx.x, h = blockIdx.y;
    const int Hq = gridDim.y;
    const int g = h / (Hq / Hkv);
    const int s0 = tile_ptr[qt];
    const int n = tile_ptr[qt + 1] - s0;

    for (int i = threadIdx.x; i < n && i < kSchedSmem; i += blockDim.x)
        sched[i] = make_int2(tile_kv[s0 + i], tile_len[s0 + i]);
    if (threadIdx.x == 0) {
        for (int b = 0; b < N_BARS; ++b) mbar_init(&bars[b], b == P_FULL ? kSoftmaxThreads : 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;
    auto entry = [&](int j) {
        return j < kSchedSmem ? sched[j] : make_int2(tile_kv[s0 + j], tile_len[s0 + j]);
    };

    if (warp == 0) {
        if (lane == 0 && n > 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            mbar_arrive_expect_tx(&bars[Q_FULL], L::kTileBytes);
            for (int c = 0; c < L::kChunks; ++c) tma_load_3d(sQ + c * kBoxBytes, &tm_q, &bars[Q_FULL], c * 64, h, qt * 128);
            for (int j = 0; j < n; ++j) {
                const int kv0 = entry(j).x;
                if (j > 0) mbar_wait(&bars[K_EMPTY], (j - 1) & 1, err);
                mbar_arrive_expect_tx(&bars[K_FULL], L::kTileBytes);
                for (int c = 0; c < L::kChunks; ++c) tma_load_3d(sK + c * kBoxBytes, &tm_k, &bars[K_FULL], c * 64, g, kv0);
                if (j > 0) mbar_wait(&bars[V_EMPTY], (j - 1) & 1, err);
                mbar_arrive_expect_tx(&bars[V_FULL], L::kTileBytes);
                for (int c = 0; c < L::kChunks; ++c) tma_load_3d(sV + c * kBoxBytes, &tm_v, &bars[V_FULL], c * 64, g, kv0);
            }
            // our last copies have landed before the CTA may retire
            mbar_wait(&bars[K_FULL], (n - 1) & 1, err);
            mbar_wait(&bars[V_FULL], (n - 1) & 1, err);
        }
    } else if (warp == 1) {
        if (lane == 0 && n > 0) {
            constexpr uint32_t idesc_qk = idesc_bf16(128, 128, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16(128, D, false, true);
            const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
            mbar_wait(&bars[Q_FULL], 0, err);
            auto issue_s = [&](int j) {
                mbar_wait(&bars[K_FULL], j & 1, err);
                tc_fence_after();
                const uint32_t dS = tmem + (j & 1) * 128;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                    mma_f16_ss(dS, sdesc_sw128(aQ + off, 16, 1024), sdesc_sw128(aK + off, 16, 1024), idesc_qk,
                               kk > 0);
                }
                mma_commit(&bars[K_EMPTY]);
                mma_commit(&bars[S_FULL0 + (j & 1)]);
            };
            issue_s(0);
            for (int j = 0; j < n; ++j) {
                if (j + 1 < n) {
                    // buffer (j+1)&1 still holds P(j-1) until PV(j-1) has completed
                    if (j >= 1) mbar_wait(&bars[O_DONE], (j - 1) & 1, err);
                    issue_s(j + 1);
                }
                mbar_wait(&bars[P_FULL], j & 1, err);
                mbar_wait(&bars[V_FULL], j & 1, err);
                tc_fence_after();
                const uint32_t aP = tmem + (j & 1) * 128;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_f16_ts(tmem + kColO, aP + kk * 8, sdesc_sw128(aV + kk * 2048, kBoxBytes, 1024), idesc_pv, 1);
                mma_commit(&bars[V_EMPTY]);
                mma_commit(&bars[O_DONE]);
            }
        }
    } else {
        const int quarter = warp & 3;                 // TMEM lanes this warp may touch
        const int half = (warp - 2) >> 2;             // which half of the row's columns
        const int r = quarter * 32 + lane;            // Q-tile row of this thread
        const int t = (warp - 2) * 32 + lane;         // 0..255 for cooperative loads
        const int key = t & 127;                      // staging: half 0 loads end[], half 1 pos[]
        const int q_row = qt * 128 + r;
        const bool real = q_row < T;
        const int pos_q = pos[q_row];
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_off + kColO + half * (D / 2);
        const uint32_t pair_bar = 2 + quarter;        // the two warps that share these TMEM lanes
        float* xmax = reinterpret_cast<float*>(smem + L::kXmax);
        float* lx = reinterpret_cast<float*>(smem + L::kLx);
        int* tmin = reinterpret_cast<int*>(smem + L::kTmin);

        {
            uint32_t z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) tmem_st32(tO + c * 32, z);
            tmem_st_wait();
        }
        // end/pos of the next tile's keys are loaded one tile ahead (keys past the
        // tile's own input are read through that input's tiles: never here)
        auto stage_value = [&](int2 en) {
            if (key >= en.y) return half == 0 ? -1 : 0;
            return half == 0 ? end[en.x + key] : pos[en.x + key];
        };
        int next = n > 0 ? stage_value(entry(0)) : 0;
        float m = -INFINITY, l = 0.f;   // l: this half's share of the row sum
        for (int j = 0; j < n; ++j) {
            const int kv0 = entry(j).x;
            const int b = j & 1;
            int32_t* e_buf = kv_end + b * 128;
            int32_t* p_buf = kv_pos + b * 128;
            (half == 0 ? e_buf : p_buf)[key] = next;
            {   // per-warp minimum of end[] (half 0) or pos[] (half 1) over this tile's keys
                const int wmin = __reduce_min_sync(0xffffffffu, next);
                if (lane == 0) tmin[b * 8 + (warp - 2)] = wmin;
            }
            named_bar_sync(1, kSoftmaxThreads);
            if (j + 1 < n) next = stage_value(entry(j + 1));
            mbar_wait(&bars[S_FULL0 + b], (j >> 1) & 1, err);
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
                mbar_wait(&bars[O_DONE], (j - 1) & 1, err);
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
            // P of keys [64 half, 64 half + 64) -> bf16 pairs in columns [32 half, 32 half + 32) of
            // this tile's S buffer (both halves have read their S columns before the pair barrier)
            tmem_st32(tS + half * 32, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars[P_FULL]);
        }
        if (n > 0) {
            mbar_wait(&bars[O_DONE], (n - 1) & 1, err);
            tc_fence_after();
        }
        // the row sum, halves added in a fixed order
        lx[half * 128 + r] = l;
        named_bar_sync(pair_bar, 64);
        const float lrow = lx[r] + lx[128 + r];
        // O / l in bf16 into the (now free) Q tile, in the TMA box layout: 128-byte rows,
        // 16-byte chunks swizzled by the row's low three bits
        const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
            const int col = half * (D / 2) + c * 32;      // first O column of these 32
            uint32_t rr[32];
            tmem_ld32(tO + c * 32, rr);
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                w[i] = real ? pack_bf16x2(__uint_as_float(rr[2 * i]) * inv, __uint_as_float(rr[2 * i + 1]) * inv) : 0u;
            uint8_t* row = sQ + (col >> 6) * kBoxBytes + r * 128;
            const int chunk0 = (col & 63) >> 3;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int chunk = (chunk0 + i) ^ (r & 7);
                *reinterpret_cast<uint4*>(row + chunk * 16) = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
            }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, kSoftmaxThreads);
        if (t == 0) {
            for (int c = 0; c < L::kChunks; ++c) tma_store_3d(&tm_o, sQ + c * kBoxBytes, c * 64, h, qt * 128);
            tma_store_commit_and_wait_read();
        }
    }

    tc_fence_before();
    __syncthreads();
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
    if ((st = make_tmap(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, o, dq, sq, box, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    const int smem = AttnSmem<D>::kAlloc > kMinSmem ? AttnSmem<D>::kAlloc : kMinSmem;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(branch_attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attention)");
        configured = true;
    }
    const float scale_log2 = scale * 1.4426950408889634f;
    dim3 grid(P.T_pad / 128, Hq);
    branch_attention_kernel<D><<<grid, kAttnThreads, smem, stream>>>(
        tq, tk, tv, to, P.dev.end, P.dev.pos, P.dev.tile_ptr, P.dev.tile_kv, P.dev.tile_len, P.T, Hkv, scale_log2,
        window, err);
    cudaError_t e = cudaGetLastError();
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
