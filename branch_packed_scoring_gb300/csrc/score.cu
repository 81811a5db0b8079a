// Slot scoring: the lm head at the slot rows of a pass, a full-vocabulary
// log-sum-exp, and the log-probabilities of the option tokens.
//
// The method ("spinf-serve 0.1.1", PyPI page, "What it does"): the engine
// returns each option's log-probability at the place where the template ends;
// the man page (PARAMETERS, --lm-head) makes fp32 output of the lm head the
// default.  Logits are never written out: each CTA of the main kernel reduces
// its 128 x 256 logit tile to a (max, sum of exp) pair per row and picks out the
// option-token logits that fall in the tile.
//
//   K4 gather_rows   hidden[slot_row[m]] -> Hs[m]   (e4m3: per-row absmax/448
//                    scale, fp32 division, round-to-nearest-even, saturating)
//   K2 score_main    persistent; z = Hs W^T on tcgen05 (128 slot rows x 256 vocab
//                    rows per tile, fp32 in TMEM, double-buffered), then per row
//                    an online (max, sum exp) over the tile in column order
//   K3 combine       per row, merge the vocabulary chunks in ascending order ->
//                    lse; token_lp = z_gathered - lse
//   K5 extract       searched slots ({*} {n} {$}; PyPI page, "What it does":
//                    the most likely answers with their probabilities): K2
//                    keeps, per searched row and 256-token tile, the best k
//                    allowed tokens; K5 merges the tiles' lists into the row's
//                    top k (z descending, lower id first on ties), lp = z - lse
//   rows outside a plan  spinf_score_rows: the same kernels on caller-given rows
//                    (the decode rows of searched slots), every row searched
//   several passes   spinf_score_passes: the scoring rows of up to 32 passes of
//                    one plan as one list of rows, so that one sweep over the lm
//                    head serves them all and only the last 128-row tile is padded
//
// Every reduction runs in a fixed order that depends only on the row's own
// values and the vocabulary size, so a row's results do not depend on M or on
// which other rows share its tile.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "runtime.h"

namespace spinf {
namespace {

using namespace dev;

constexpr int kBM = 128;   // slot rows per tile (MMA M, TMEM lanes)
constexpr int kBN = 256;   // vocabulary rows per tile (MMA N, TMEM columns)
constexpr int kStages = 4;
constexpr int kABytes = kBM * 128;
constexpr int kBBytes = kBN * 128;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kScoreThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;

enum { FULL0 = 0, EMPTY0 = kStages, ACC_FULL0 = 2 * kStages, ACC_EMPTY0 = 2 * kStages + 2, N_SBARS = 2 * kStages + 4 };

constexpr int kSmemBars = kStages * kStageBytes;
constexpr int kSmemHolder = kSmemBars + N_SBARS * 8;
constexpr int kScoreSmem = kSmemHolder + 16 + 1024;
// searched rows: each epilogue thread stages a 32-logit chunk of its row here (33 floats apart)
constexpr int kSmemXStage = kSmemHolder + 16;
constexpr int kScoreSmemX = kSmemXStage + 128 * 33 * 4 + 1024;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// The scoring rows of one call as one list: rows [m0[b], m0[b + 1]) are the scoring rows
// of the call's b-th pass (its local rows 0, 1, ...), their gathers [g0[b], g0[b + 1]) of
// the call's gathered logits.  A single-pass call has nb = 1.
constexpr int kMaxScorePasses = SPINF_SCORE_MAX_PASSES;
struct RowMap {
    int nb;
    int m0[kMaxScorePasses + 1];
    int g0[kMaxScorePasses + 1];
    const __nv_bfloat16* hidden[kMaxScorePasses];   // [T_pad, D] of each pass, or its slot rows [M_b, D]
    const int32_t* slot_row[kMaxScorePasses];       // [M_b]; nullptr: hidden holds the slot rows in order
    const int32_t* row_gptr[kMaxScorePasses];       // [M_b + 1]
    const int32_t* row_glist[kMaxScorePasses];      // [G_b]
    const int32_t* gather_tok[kMaxScorePasses];     // [G_b]
    float* row_lse[kMaxScorePasses];                // [M_b]
    float* token_lp[kMaxScorePasses];               // [G_b]
};

// Tile order of the main kernel: blocks of up to `rpb` 128-row tiles; within a block, vocabulary
// tile by vocabulary tile, the block's row tiles next to each other.  A block's gathered rows
// stay in L2 while the lm head streams past once per block (one block when all rows fit).
__device__ __forceinline__ void unit_tile(int u, int n_st, int n_vt, int rpb, int& vt, int& st) {
    const int per_block = n_vt * rpb;
    const int rb = u / per_block;
    const int rem = u - rb * per_block;
    const int rows = min(rpb, n_st - rb * rpb);
    vt = rem / rows;
    st = rb * rpb + rem % rows;
}

// Row tiles per block: the gathered rows of a block take at most ~32 MB of the L2.
int rows_per_block(int n_st, int d_model, int elt) {
    const long long tile = (long long)kBM * d_model * elt;
    const long long r = (32ll << 20) / (tile > 0 ? tile : 1);
    return (int)std::max(1ll, std::min<long long>(r, n_st));
}

// The pass b of list row m (m < m0[nb]).
__device__ __forceinline__ int row_pass(const RowMap& rm, int m) {
    int b = 0;
    while (b + 1 < rm.nb && m >= rm.m0[b + 1]) ++b;
    return b;
}

// A one-pass map over the pass's own device descriptors.
RowMap one_pass_map(const Pass& P, const void* hidden, float* row_lse, float* token_lp) {
    RowMap rm{};
    rm.nb = 1;
    rm.m0[1] = (int)P.slot_row.size();
    rm.g0[1] = (int)P.gather_tok.size();
    rm.hidden[0] = static_cast<const __nv_bfloat16*>(hidden);
    rm.slot_row[0] = P.dev.slot_row;
    rm.row_gptr[0] = P.dev.row_gptr;
    rm.row_glist[0] = P.dev.row_glist;
    rm.gather_tok[0] = P.dev.gather_tok;
    rm.row_lse[0] = row_lse;
    rm.token_lp[0] = token_lp;
    return rm;
}

struct ScoreLayout {
    int M, M_pad, G, n_vt, n_st, X, k;
    size_t hs, sa, part, zg, xpart, total;
};

// Workspace layout for M scoring rows, G gathers and X searched slots.
ScoreLayout score_layout_counts(int M, int G, int X, int vocab, int d_model, int w_dtype, int extract_k) {
    ScoreLayout s;
    s.X = X;
    s.k = extract_k;
    s.M = M;
    s.G = G;
    s.M_pad = std::max(1, (s.M + kBM - 1) / kBM) * kBM;
    s.n_st = s.M_pad / kBM;
    s.n_vt = (vocab + kBN - 1) / kBN;
    const size_t elt = w_dtype == SPINF_DTYPE_E4M3 ? 1 : 2;
    s.hs = 0;
    s.sa = s.hs + align256((size_t)s.M_pad * d_model * elt);
    s.part = s.sa + align256((size_t)s.M_pad * 4);
    s.zg = s.part + align256((size_t)s.M_pad * s.n_vt * 8);
    s.xpart = s.zg + align256((size_t)std::max(s.G, 1) * 4);
    s.total = s.xpart + align256((size_t)s.X * s.n_vt * s.k * 8);   // (z, token) per candidate
    return s;
}

ScoreLayout score_layout(const Pass& P, int vocab, int d_model, int w_dtype, int extract_k) {
    return score_layout_counts((int)P.slot_row.size(), (int)P.gather_tok.size(), (int)P.x_m.size(), vocab, d_model,
                               w_dtype, extract_k);
}

// ---------------------------------------------------------------- K4
template <bool FP8>
__global__ void __launch_bounds__(256) gather_rows_kernel(const __grid_constant__ RowMap rm, int M, int D,
                                                          void* __restrict__ out, float* __restrict__ s_act) {
    const int m = blockIdx.x;
    const int nv = D / 8;   // 8 elements per vector
    const uint4* src = nullptr;
    if (m < M) {
        const int b = row_pass(rm, m);
        const int ml = m - rm.m0[b];
        src = reinterpret_cast<const uint4*>(rm.hidden[b] + (size_t)(rm.slot_row[b] ? rm.slot_row[b][ml] : ml) * D);
    }
    if (!FP8) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + (size_t)m * D);
        for (int i = threadIdx.x; i < nv; i += blockDim.x) dst[i] = src ? src[i] : make_uint4(0, 0, 0, 0);
        return;
    }
    __shared__ float red[8];
    float amax = 0.f;
    if (src)
        for (int i = threadIdx.x; i < nv; i += blockDim.x) {
            uint4 u = src[i];
            const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float2 f = __bfloat1622float2(b[j]);
                amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = 0.f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) a = fmaxf(a, red[w]);
        red[0] = a > 0.f ? __fdiv_rn(a, 448.f) : 1.f;
        s_act[m] = red[0];
    }
    __syncthreads();
    const float sc = red[0];
    uint2* dst = reinterpret_cast<uint2*>(static_cast<uint8_t*>(out) + (size_t)m * D);
    for (int i = threadIdx.x; i < nv; i += blockDim.x) {
        uint32_t w[2] = {0u, 0u};
        if (src) {
            uint4 u = src[i];
            const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float2 f = __bfloat1622float2(b[j]);
                float2 q = make_float2(__fdiv_rn(f.x, sc), __fdiv_rn(f.y, sc));
                __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, __NV_E4M3);
                w[j >> 1] |= static_cast<uint32_t>(c) << ((j & 1) * 16);
            }
        }
        dst[i] = make_uint2(w[0], w[1]);
    }
}

// ---------------------------------------------------------------- K2
// Searched rows: a row's best KX candidates of one tile, best first (z descending,
// lower token first on ties; the tile is scanned in ascending token order, so a
// new token goes after an equal one already held).
template <int KX>
struct TopList {
    float z[KX];
    int t[KX];
};

template <int KX>
__device__ __forceinline__ void top_insert(TopList<KX>& L, float v, int tok) {
    bool moved = false;
#pragma unroll
    for (int j = 0; j < KX; ++j) {
        const bool sw = moved || v > L.z[j];
        const float z0 = L.z[j];
        const int t0 = L.t[j];
        if (sw) {
            L.z[j] = v;
            L.t[j] = tok;
            v = z0;
            tok = t0;
        }
        moved = sw;
    }
}

struct ExtractArgs {
    const int32_t* row_x;        // [M] searched slot of each scoring row, or -1
    const int32_t* x_set;        // [X]
    const uint32_t* token_sets;  // [n_sets][words]
    int n_sets;
    int words;                   // ceil(V / 32)
    int k;                       // candidates kept per tile (extract_k)
    uint2* xpart;                // [X][n_vt][k] (z bits, token)
};

// KX: 0 (no searched rows), or the list length (8 or 16) kept per searched row and tile
template <bool FP8, int KX>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_main_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
                      const float* __restrict__ s_act, const float* __restrict__ s_w, float2* __restrict__ part,
                      float* __restrict__ zg, const __grid_constant__ RowMap rm, int M, int V,
                      int n_kb, int n_st, int n_vt, int rpb, const ExtractArgs xa, int* __restrict__ err) {
    constexpr int kPerMma = FP8 ? 32 : 16;           // K elements of one MMA instruction
    constexpr int kMmaPerStage = (FP8 ? 128 : 64) / kPerMma;
    constexpr int kBK = FP8 ? 128 : 64;              // K elements per 128-byte row
    constexpr uint32_t idesc = FP8 ? idesc_e4m3(kBM, kBN) : idesc_bf16(kBM, kBN, false, false);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSmemBars);
    uint32_t* holder = reinterpret_cast<uint32_t*>(smem + kSmemHolder);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = n_vt * n_st;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars[FULL0 + s], 1);
            mbar_init(&bars[EMPTY0 + s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&bars[ACC_FULL0 + a], 1);
            mbar_init(&bars[ACC_EMPTY0 + a], 128);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tm_h);
            tma_prefetch_desc(&tm_w);
            uint32_t it = 0;
            for (int u = blockIdx.x; u < total; u += gridDim.x) {
                int vt, st;
                unit_tile(u, n_st, n_vt, rpb, vt, st);
                for (int kb = 0; kb < n_kb; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    mbar_wait(&bars[EMPTY0 + s], ph ^ 1, err);
                    uint8_t* sa = smem + s * kStageBytes;
                    mbar_arrive_expect_tx(&bars[FULL0 + s], kStageBytes);
                    tma_load_2d(sa, &tm_h, &bars[FULL0 + s], kb * kBK, st * kBM);
                    tma_load_2d(sa + kABytes, &tm_w, &bars[FULL0 + s], kb * kBK, vt * kBN);
                }
            }
            // our last copies have landed before the CTA may retire
            for (uint32_t i = it > (uint32_t)kStages ? it - kStages : 0; i < it; ++i)
                mbar_wait(&bars[FULL0 + i % kStages], (i / kStages) & 1, err);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t it = 0, tcount = 0;
            for (int u = blockIdx.x; u < total; u += gridDim.x, ++tcount) {
                const int acc = tcount & 1;
                const uint32_t aph = (tcount >> 1) & 1;
                mbar_wait(&bars[ACC_EMPTY0 + acc], aph ^ 1, err);
                tc_fence_after();
                const uint32_t d_tmem = tmem + acc * kBN;
                for (int kb = 0; kb < n_kb; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    mbar_wait(&bars[FULL0 + s], ph, err);
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(smem + s * kStageBytes);
                    const uint32_t b_base = a_base + kABytes;
#pragma unroll
                    for (int kk = 0; kk < kMmaPerStage; ++kk) {
                        const uint64_t da = sdesc_sw128(a_base + kk * 32, 16, 1024);
                        const uint64_t db = sdesc_sw128(b_base + kk * 32, 16, 1024);
                        if (FP8) mma_f8_ss(d_tmem, da, db, idesc, (kb | kk) != 0);
                        else mma_f16_ss(d_tmem, da, db, idesc, (kb | kk) != 0);
                    }
                    mma_commit(&bars[EMPTY0 + s]);
                }
                mma_commit(&bars[ACC_FULL0 + acc]);
            }
        }
    } else {
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        uint32_t tcount = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x, ++tcount) {
            int vt, st;
            unit_tile(u, n_st, n_vt, rpb, vt, st);
            const int acc = tcount & 1;
            const uint32_t aph = (tcount >> 1) & 1;
            const int m = st * kBM + r;
            const bool valid = m < M;
            const int v0 = vt * kBN;
            int gc = 0, ge = 0;
            // this row's pass: its gather list (local gather indices) and its logits' base in zg
            const int32_t* row_glist = nullptr;
            const int32_t* gather_tok = nullptr;
            float* zgb = zg;
            if (valid) {   // first gather of this row whose token is >= v0 (tokens sorted per row)
                const int b = row_pass(rm, m), ml = m - rm.m0[b];
                row_glist = rm.row_glist[b];
                gather_tok = rm.gather_tok[b];
                zgb = zg + rm.g0[b];
                int lo = rm.row_gptr[b][ml], hi = rm.row_gptr[b][ml + 1];
                ge = hi;
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (gather_tok[row_glist[mid]] < v0) lo = mid + 1; else hi = mid;
                }
                gc = lo;
            }
            const float sa = (FP8 && valid) ? s_act[m] : 1.f;
            int xr = -1;
            const uint32_t* allow = nullptr;
            TopList<KX ? KX : 1> top;
            float* stage = reinterpret_cast<float*>(smem + kSmemXStage) + (threadIdx.x - 64) * 33;
            uint32_t mw[kBN / 32];   // the tile's allowed-token words, fetched before the accumulator wait
            if constexpr (KX > 0) {
                xr = valid ? xa.row_x[m] : -1;
                if (xr >= 0) {
                    int set = xa.x_set[xr];
                    if (set >= xa.n_sets) {   // a set the call does not hold: every token, and an error
                        atomicExch(err, kErrCheck);
                        set = -1;
                    }
                    if (set >= 0) allow = xa.token_sets + (size_t)set * xa.words;
#pragma unroll
                    for (int c = 0; c < kBN / 32; ++c)
                        mw[c] = !allow ? 0xffffffffu : (v0 + 32 * c < V ? __ldg(allow + ((v0 >> 5) + c)) : 0u);
#pragma unroll
                    for (int j = 0; j < KX; ++j) {
                        top.z[j] = -INFINITY;
                        top.t[j] = -1;
                    }
                }
            }
            mbar_wait(&bars[ACC_FULL0 + acc], aph, err);
            tc_fence_after();
            float mx = -INFINITY, sum = 0.f;
#pragma unroll 1
            for (int c = 0; c < kBN / 32; ++c) {
                uint32_t rr[32];
                tmem_ld32(tmem + lane_off + acc * kBN + c * 32, rr);
                const int vc = v0 + c * 32;
                float z[32];
                float cmax = -INFINITY;
                if (FP8 && vc + 32 <= V) {   // a whole chunk inside the vocabulary: 8 vector scale loads
                    const float4* sw4 = reinterpret_cast<const float4*>(s_w + vc);
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        const float4 sc = __ldg(sw4 + q4);
                        z[4 * q4 + 0] = (__uint_as_float(rr[4 * q4 + 0]) * sc.x) * sa;
                        z[4 * q4 + 1] = (__uint_as_float(rr[4 * q4 + 1]) * sc.y) * sa;
                        z[4 * q4 + 2] = (__uint_as_float(rr[4 * q4 + 2]) * sc.z) * sa;
                        z[4 * q4 + 3] = (__uint_as_float(rr[4 * q4 + 3]) * sc.w) * sa;
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) cmax = fmaxf(cmax, z[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        float x = __uint_as_float(rr[i]);
                        if (FP8) x = (x * (vc + i < V ? s_w[vc + i] : 0.f)) * sa;
                        z[i] = vc + i < V ? x : -INFINITY;
                        cmax = fmaxf(cmax, z[i]);
                    }
                }
                const float nm = fmaxf(mx, cmax);
                float add = 0.f;
#pragma unroll
                for (int i = 0; i < 32; ++i) add += fast_exp2((z[i] - nm) * kLog2e);
                sum = (mx == -INFINITY ? 0.f : sum * fast_exp2((mx - nm) * kLog2e)) + add;
                mx = nm;
                if constexpr (KX > 0) {
                    if (xr >= 0 && vc < V) {
                        // candidates: allowed and above the list's last entry (z = -inf past the
                        // vocabulary never is); they go through one copy of the insertion code,
                        // reading their logits back from this thread's staging row
                        const float thr = top.z[KX - 1];
                        uint32_t cand = 0;
#pragma unroll
                        for (int i = 0; i < 32; ++i) cand |= (z[i] > thr ? 1u : 0u) << i;
                        cand &= mw[0];
                        if (cand) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) stage[i] = z[i];
                            while (cand) {
                                const int i = __ffs(cand) - 1;
                                cand &= cand - 1;
                                const float v = stage[i];
                                if (v > top.z[KX - 1]) top_insert<KX>(top, v, vc + i);
                            }
                        }
                    }
#pragma unroll
                    for (int c = 0; c + 1 < kBN / 32; ++c) mw[c] = mw[c + 1];   // next chunk's word first
                }
                while (gc < ge) {
                    const int g = row_glist[gc];
                    const int tk = gather_tok[g];
                    if (tk >= vc + 32) break;
                    const int idx = tk - vc;
                    float val = z[0];
#pragma unroll
                    for (int i = 1; i < 32; ++i) val = (i == idx) ? z[i] : val;
                    zgb[g] = val;
                    ++gc;
                }
            }
            tc_fence_before();
            mbar_arrive(&bars[ACC_EMPTY0 + acc]);
            if (valid) part[(size_t)m * n_vt + vt] = make_float2(mx, sum);
            if constexpr (KX > 0) {
                if (xr >= 0) {
                    uint2* dst = xa.xpart + ((size_t)xr * n_vt + vt) * xa.k;
#pragma unroll
                    for (int j = 0; j < KX; ++j)
                        if (j < xa.k) dst[j] = make_uint2(__float_as_uint(top.z[j]), (uint32_t)top.t[j]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- K3
__device__ __forceinline__ float2 lse_merge(float2 a, float2 b) {
    if (a.x == -INFINITY) return b;
    if (b.x == -INFINITY) return a;
    const float m = fmaxf(a.x, b.x);
    return make_float2(m, a.y * expf(a.x - m) + b.y * expf(b.x - m));
}

__global__ void __launch_bounds__(128) score_combine_kernel(const float2* __restrict__ part,
                                                            const float* __restrict__ zg,
                                                            const __grid_constant__ RowMap rm, int M, int n_vt) {
    const int m = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (m >= M) return;
    const int b = row_pass(rm, m), ml = m - rm.m0[b];
    const int32_t* row_glist = rm.row_glist[b];
    const float* zgb = zg + rm.g0[b];
    float* token_lp = rm.token_lp[b];
    float2 acc = make_float2(-INFINITY, 0.f);
    for (int vt = lane; vt < n_vt; vt += 32) acc = lse_merge(acc, part[(size_t)m * n_vt + vt]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float2 other;
        other.x = __shfl_xor_sync(0xffffffffu, acc.x, o);
        other.y = __shfl_xor_sync(0xffffffffu, acc.y, o);
        acc = (lane & o) ? lse_merge(other, acc) : lse_merge(acc, other);
    }
    const float lse = acc.x + logf(acc.y);
    if (lane == 0) rm.row_lse[b][ml] = lse;
    for (int i = rm.row_gptr[b][ml] + lane; i < rm.row_gptr[b][ml + 1]; i += 32) {
        const int g = row_glist[i];
        token_lp[g] = zgb[g] - lse;
    }
}

// ---------------------------------------------------------------- K5
// One CTA of 256 threads per searched slot.  Thread t merges the lists of tiles t,
// t + 256, ... (ascending, so an equal z from a later tile -- a higher token -- goes
// after), then the 256 lists are merged pairwise in shared memory, comparing z and, on
// ties, the token id.  Tokens are unique across tiles, so the result is the unique top
// k of the row under that order, whatever the merge tree.
__device__ __forceinline__ bool top_before(float za, int ta, float zb, int tb) {
    return za > zb || (za == zb && ta >= 0 && (tb < 0 || ta < tb));
}

constexpr int kMergeThreads = 256;

template <int KX>
__global__ void __launch_bounds__(kMergeThreads) extract_combine_kernel(const uint2* __restrict__ xpart,
                                                                         const int32_t* __restrict__ x_m, int n_vt,
                                                                         int k, const float* __restrict__ row_lse,
                                                                         int32_t* __restrict__ top_tok,
                                                                         float* __restrict__ top_lp) {
    __shared__ float sz[kMergeThreads][KX];
    __shared__ int st[kMergeThreads][KX];
    const int x = blockIdx.x, t = threadIdx.x;
    TopList<KX> L;
#pragma unroll
    for (int j = 0; j < KX; ++j) {
        L.z[j] = -INFINITY;
        L.t[j] = -1;
    }
    for (int vt = t; vt < n_vt; vt += kMergeThreads) {
        const uint2* src = xpart + ((size_t)x * n_vt + vt) * k;
        uint2 c[KX];
#pragma unroll
        for (int j = 0; j < KX; ++j) c[j] = j < k ? src[j] : make_uint2(__float_as_uint(-INFINITY), ~0u);
#pragma unroll
        for (int j = 0; j < KX; ++j) {   // the tile's list is sorted: stop at the first that does not enter
            const float z = __uint_as_float(c[j].x);
            if (!(z > L.z[KX - 1])) break;
            top_insert<KX>(L, z, (int)c[j].y);
        }
    }
#pragma unroll
    for (int j = 0; j < KX; ++j) {
        sz[t][j] = L.z[j];
        st[t][j] = L.t[j];
    }
    __syncthreads();
    for (int n = kMergeThreads / 2; n >= 1; n >>= 1) {
        if (t < n) {   // merge lists 2t and 2t + 1 into L
            int a = 0, b = 0;
#pragma unroll
            for (int j = 0; j < KX; ++j) {
                const float za = a < KX ? sz[2 * t][a] : -INFINITY, zb = b < KX ? sz[2 * t + 1][b] : -INFINITY;
                const int ta = a < KX ? st[2 * t][a] : -1, tb = b < KX ? st[2 * t + 1][b] : -1;
                const bool take_a = !top_before(zb, tb, za, ta);   // an exhausted list reads (-inf, -1)
                L.z[j] = take_a ? za : zb;
                L.t[j] = take_a ? ta : tb;
                a += take_a ? 1 : 0;
                b += take_a ? 0 : 1;
            }
        }
        __syncthreads();
        if (t < n) {
#pragma unroll
            for (int j = 0; j < KX; ++j) {
                sz[t][j] = L.z[j];
                st[t][j] = L.t[j];
            }
        }
        __syncthreads();
    }
    if (t < k) {
        const float z = sz[0][t];
        const int tok = st[0][t];
        top_tok[(size_t)x * k + t] = tok;
        top_lp[(size_t)x * k + t] = tok >= 0 ? z - row_lse[x_m[x]] : -INFINITY;
    }
}

// The scoring kernels on the rows of `rm` (KX > 0: one pass, `P`'s searched slots).
template <bool FP8, int KX>
spinf_status launch_score_rows(const Pass* P, const RowMap& rm, const ScoreLayout& L, const void* w,
                               const float* w_scale, int D, int V, const spinf_extract_out* ex, uint8_t* ws, int* err,
                               cudaStream_t stream) {
    static_assert(sizeof(RowMap) <= 2200, "the row map travels in the kernels' parameters");
    void* hs = ws + L.hs;
    float* sa = reinterpret_cast<float*>(ws + L.sa);
    float2* part = reinterpret_cast<float2*>(ws + L.part);
    float* zg = reinterpret_cast<float*>(ws + L.zg);
    gather_rows_kernel<FP8><<<L.M_pad, 256, 0, stream>>>(rm, L.M, D, hs, sa);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "gather launch");

    CUtensorMap th, tw;
    const uint64_t elt = FP8 ? 1 : 2;
    const uint64_t dh[2] = {(uint64_t)D, (uint64_t)L.M_pad};
    const uint64_t dw[2] = {(uint64_t)D, (uint64_t)V};
    const uint64_t st[1] = {(uint64_t)D * elt};
    const uint32_t bh[2] = {FP8 ? 128u : 64u, (uint32_t)kBM};
    const uint32_t bw[2] = {FP8 ? 128u : 64u, (uint32_t)kBN};
    const CUtensorMapDataType dt = FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    spinf_status s;
    if ((s = make_tmap(&th, dt, 2, hs, dh, st, bh, CU_TENSOR_MAP_SWIZZLE_128B))) return s;
    if ((s = make_tmap(&tw, dt, 2, w, dw, st, bw, CU_TENSOR_MAP_SWIZZLE_128B))) return s;
    if ((s = set_smem_limit(reinterpret_cast<const void*>(score_main_kernel<FP8, KX>), KX ? kScoreSmemX : kScoreSmem,
                            "cudaFuncSetAttribute(score)")))
        return s;
    const int kbk = FP8 ? 128 : 64;
    const int n_kb = (D + kbk - 1) / kbk;
    const int total = L.n_vt * L.n_st;
    const int grid = std::min(total, sm_count());
    ExtractArgs xa{KX ? P->dev.row_x : nullptr, KX ? P->dev.x_set : nullptr, KX ? ex->token_sets : nullptr,
                   KX ? ex->n_sets : 0, (V + 31) / 32, L.k, reinterpret_cast<uint2*>(ws + L.xpart)};
    score_main_kernel<FP8, KX><<<grid, kScoreThreads, KX ? kScoreSmemX : kScoreSmem, stream>>>(
        th, tw, sa, w_scale, part, zg, rm, L.M, V, n_kb, L.n_st, L.n_vt, rows_per_block(L.n_st, D, FP8 ? 1 : 2), xa,
        err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "score launch");
    score_combine_kernel<<<(L.M + 3) / 4, 128, 0, stream>>>(part, zg, rm, L.M, L.n_vt);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    if constexpr (KX > 0) {
        extract_combine_kernel<KX><<<L.X, kMergeThreads, 0, stream>>>(xa.xpart, P->dev.x_m, L.n_vt, L.k, rm.row_lse[0],
                                                                      ex->top_tok, ex->top_lp);
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "extract launch");
    }
    return SPINF_OK;
}

// The scoring kernels on one pass's rows.
template <bool FP8, int KX>
spinf_status launch_score(const Pass& P, const ScoreLayout& L, const void* hidden, const void* w, const float* w_scale,
                          int D, int V, float* row_lse, float* token_lp, const spinf_extract_out* ex, uint8_t* ws,
                          int* err, cudaStream_t stream) {
    return launch_score_rows<FP8, KX>(&P, one_pass_map(P, hidden, row_lse, token_lp), L, w, w_scale, D, V, ex, ws, err,
                                      stream);
}

}  // namespace
}  // namespace spinf

using namespace spinf;

extern "C" size_t spinf_score_workspace_bytes(const spinf_plan* plan, int32_t pass, int32_t vocab, int32_t d_model,
                                              int32_t w_dtype) {
    if (!plan || pass < 0 || pass >= (int32_t)plan->passes.size() || vocab <= 0 || d_model <= 0) return 0;
    return score_layout(plan->passes[pass], vocab, d_model, w_dtype, plan->extract_k).total;
}

extern "C" spinf_status spinf_score_extract(const spinf_plan* plan, int32_t pass, const void* hidden, const void* w,
                                            const float* w_scale, int32_t w_dtype, int32_t d_model, int32_t vocab,
                                            float* row_lse, float* token_lp, const spinf_extract_out* ex,
                                            void* workspace, size_t workspace_bytes, spinf_stream stream) {
    spinf_status st = ensure_device_ready(plan, pass);
    if (st) return st;
    if (w_dtype != SPINF_DTYPE_BF16 && w_dtype != SPINF_DTYPE_E4M3) return fail(SPINF_E_UNSUPPORTED, "w_dtype");
    if (d_model <= 0 || d_model % 16) return fail(SPINF_E_UNSUPPORTED, "d_model must be a positive multiple of 16");
    if (vocab <= 0) return fail(SPINF_E_INVALID, "vocab must be positive");
    const Pass& P = plan->passes[pass];
    if (P.slot_row.empty()) return SPINF_OK;
    if (!hidden || !w || !row_lse || !token_lp || !workspace) return fail(SPINF_E_INVALID, "NULL buffer");
    if (w_dtype == SPINF_DTYPE_E4M3 && !w_scale) return fail(SPINF_E_INVALID, "e4m3 weights need w_scale");
    if (w_dtype == SPINF_DTYPE_E4M3 && (reinterpret_cast<uintptr_t>(w_scale) & 15))
        return fail(SPINF_E_INVALID, "w_scale must be 16-byte aligned");
    for (const void* p : {hidden, w, (const void*)workspace})
        if (reinterpret_cast<uintptr_t>(p) & 15) return fail(SPINF_E_INVALID, "buffer not 16-byte aligned");
    for (int32_t t : P.gather_tok)
        if (t < 0 || t >= vocab) return fail(SPINF_E_INVALID, "option token outside the vocabulary");
    const ScoreLayout L = score_layout(P, vocab, d_model, w_dtype, plan->extract_k);
    if (workspace_bytes < L.total) return fail(SPINF_E_NOMEM, "workspace too small");
    const bool xt = ex && L.X > 0;
    if (xt) {
        if (!ex->top_tok || !ex->top_lp) return fail(SPINF_E_INVALID, "NULL searched-slot outputs");
        for (int32_t set : P.x_set)
            if (set >= ex->n_sets) return fail(SPINF_E_INVALID, "a searched slot names an unknown token set");
        for (int32_t set : P.x_set)
            if (set >= 0 && !ex->token_sets) return fail(SPINF_E_INVALID, "token_sets is NULL");
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const float* wsc = w_dtype == SPINF_DTYPE_E4M3 ? w_scale : nullptr;
    // list length per searched row and tile: 8 for extract_k <= 8, else 16
    const int kx = !xt ? 0 : L.k <= 8 ? 8 : 16;
    auto go = [&](auto fp8, auto kx_c) {
        return launch_score<decltype(fp8)::value, decltype(kx_c)::value>(P, L, hidden, w, wsc, d_model, vocab, row_lse,
                                                                         token_lp, ex, ws, plan->d_err, s);
    };
    using F = std::false_type;
    using T = std::true_type;
    using K0 = std::integral_constant<int, 0>;
    using K8 = std::integral_constant<int, 8>;
    using K16 = std::integral_constant<int, 16>;
    if (w_dtype == SPINF_DTYPE_E4M3)
        return kx == 0 ? go(T{}, K0{}) : kx == 8 ? go(T{}, K8{}) : go(T{}, K16{});
    return kx == 0 ? go(F{}, K0{}) : kx == 8 ? go(F{}, K8{}) : go(F{}, K16{});
}

extern "C" spinf_status spinf_score(const spinf_plan* plan, int32_t pass, const void* hidden, const void* w,
                                    const float* w_scale, int32_t w_dtype, int32_t d_model, int32_t vocab,
                                    float* row_lse, float* token_lp, void* workspace, size_t workspace_bytes,
                                    spinf_stream stream) {
    return spinf_score_extract(plan, pass, hidden, w, w_scale, w_dtype, d_model, vocab, row_lse, token_lp, nullptr,
                               workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- several passes in one sweep
namespace spinf {
namespace {

// Checks the pass list and counts its rows: M, G in total, and the row map without pointers.
spinf_status passes_map(const spinf_plan* plan, int32_t n, const int32_t* passes, RowMap& rm, int& M, int& G) {
    if (!plan || !passes || n <= 0) return fail(SPINF_E_INVALID, "NULL plan or pass list, or no pass");
    if (n > kMaxScorePasses) return fail(SPINF_E_LIMIT, "more than SPINF_SCORE_MAX_PASSES passes in one call");
    rm = RowMap{};
    rm.nb = n;
    M = G = 0;
    for (int32_t b = 0; b < n; ++b) {
        if (passes[b] < 0 || passes[b] >= (int32_t)plan->passes.size()) return fail(SPINF_E_INVALID, "bad pass index");
        for (int32_t c = 0; c < b; ++c)
            if (passes[c] == passes[b]) return fail(SPINF_E_INVALID, "a pass listed twice");
        const Pass& P = plan->passes[passes[b]];
        rm.m0[b] = M;
        rm.g0[b] = G;
        M += (int)P.slot_row.size();
        G += (int)P.gather_tok.size();
    }
    rm.m0[n] = M;
    rm.g0[n] = G;
    return SPINF_OK;
}

}  // namespace
}  // namespace spinf

extern "C" size_t spinf_score_passes_workspace_bytes(const spinf_plan* plan, int32_t n_passes, const int32_t* passes,
                                                     int32_t vocab, int32_t d_model, int32_t w_dtype) {
    RowMap rm;
    int M = 0, G = 0;
    if (vocab <= 0 || d_model <= 0 || passes_map(plan, n_passes, passes, rm, M, G) != SPINF_OK) return 0;
    return score_layout_counts(M, G, 0, vocab, d_model, w_dtype, plan->extract_k).total;
}

extern "C" spinf_status spinf_score_passes(const spinf_plan* plan, int32_t n_passes, const int32_t* passes,
                                           const void* const* hidden, int32_t hidden_rows, const void* w,
                                           const float* w_scale,
                                           int32_t w_dtype, int32_t d_model, int32_t vocab, float* const* row_lse,
                                           float* const* token_lp, void* workspace, size_t workspace_bytes,
                                           spinf_stream stream) {
    RowMap rm;
    int M = 0, G = 0;
    spinf_status st = passes_map(plan, n_passes, passes, rm, M, G);
    if (st) return st;
    if (!hidden || !row_lse || !token_lp) return fail(SPINF_E_INVALID, "NULL pointer array");
    if (hidden_rows != SPINF_HIDDEN_PASS_ROWS && hidden_rows != SPINF_HIDDEN_SLOT_ROWS)
        return fail(SPINF_E_INVALID, "hidden_rows must be SPINF_HIDDEN_PASS_ROWS or SPINF_HIDDEN_SLOT_ROWS");
    for (int32_t b = 0; b < n_passes; ++b)
        if ((st = ensure_device_ready(plan, passes[b]))) return st;
    if (w_dtype != SPINF_DTYPE_BF16 && w_dtype != SPINF_DTYPE_E4M3) return fail(SPINF_E_UNSUPPORTED, "w_dtype");
    if (d_model <= 0 || d_model % 16) return fail(SPINF_E_UNSUPPORTED, "d_model must be a positive multiple of 16");
    if (vocab <= 0) return fail(SPINF_E_INVALID, "vocab must be positive");
    if (M == 0) return SPINF_OK;
    if (!w || !workspace) return fail(SPINF_E_INVALID, "NULL buffer");
    if (w_dtype == SPINF_DTYPE_E4M3 && !w_scale) return fail(SPINF_E_INVALID, "e4m3 weights need w_scale");
    if (w_dtype == SPINF_DTYPE_E4M3 && (reinterpret_cast<uintptr_t>(w_scale) & 15))
        return fail(SPINF_E_INVALID, "w_scale must be 16-byte aligned");
    for (const void* p : {w, (const void*)workspace})
        if (reinterpret_cast<uintptr_t>(p) & 15) return fail(SPINF_E_INVALID, "buffer not 16-byte aligned");
    for (int32_t b = 0; b < n_passes; ++b) {
        const Pass& P = plan->passes[passes[b]];
        if (P.slot_row.empty()) continue;
        if (!hidden[b] || !row_lse[b] || (!P.gather_tok.empty() && !token_lp[b]))
            return fail(SPINF_E_INVALID, "NULL buffer of pass " + std::to_string(passes[b]));
        if (reinterpret_cast<uintptr_t>(hidden[b]) & 15) return fail(SPINF_E_INVALID, "hidden not 16-byte aligned");
        for (int32_t t : P.gather_tok)
            if (t < 0 || t >= vocab) return fail(SPINF_E_INVALID, "option token outside the vocabulary");
        rm.hidden[b] = static_cast<const __nv_bfloat16*>(hidden[b]);
        rm.slot_row[b] = hidden_rows == SPINF_HIDDEN_SLOT_ROWS ? nullptr : P.dev.slot_row;
        rm.row_gptr[b] = P.dev.row_gptr;
        rm.row_glist[b] = P.dev.row_glist;
        rm.gather_tok[b] = P.dev.gather_tok;
        rm.row_lse[b] = row_lse[b];
        rm.token_lp[b] = token_lp[b];
    }
    const ScoreLayout L = score_layout_counts(M, G, 0, vocab, d_model, w_dtype, plan->extract_k);
    if (workspace_bytes < L.total) return fail(SPINF_E_NOMEM, "workspace too small");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (w_dtype == SPINF_DTYPE_E4M3)
        return launch_score_rows<true, 0>(nullptr, rm, L, w, w_scale, d_model, vocab, nullptr, ws, plan->d_err, s);
    return launch_score_rows<false, 0>(nullptr, rm, L, w, nullptr, d_model, vocab, nullptr, ws, plan->d_err, s);
}

// ---------------------------------------------------------------- rows outside a plan
// Scoring of caller-given hidden rows (the decode rows of searched slots): the rows are
// the scoring rows, every row is searched.  The row tables a pass would hold (identity
// row maps, empty gather lists, the rows' token sets) are written by a small kernel at the
// front of the workspace; the scoring kernels then run as for a pass.
namespace spinf {
namespace {

__global__ void rows_tables_kernel(int n, const int32_t* __restrict__ token_set, int32_t* __restrict__ slot_row,
                                   int32_t* __restrict__ row_x, int32_t* __restrict__ x_m,
                                   int32_t* __restrict__ x_set, int32_t* __restrict__ row_gptr) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= n; i += gridDim.x * blockDim.x) {
        row_gptr[i] = 0;
        if (i < n) {
            slot_row[i] = row_x[i] = x_m[i] = i;
            x_set[i] = token_set ? token_set[i] : -1;
        }
    }
}

struct RowsView {
    Pass P;
    size_t index_bytes = 0;
};

void rows_view(RowsView& rv, int32_t n) {
    Pass& P = rv.P;   // host sizes only: the layout of the scoring workspace
    P.slot_row.resize(n);
    P.x_m.resize(n);
    rv.index_bytes = align256((size_t)n * 4) * 4 + align256((size_t)(n + 1) * 4);
}

}  // namespace
}  // namespace spinf

extern "C" size_t spinf_score_rows_workspace_bytes(int32_t n_rows, int32_t vocab, int32_t d_model, int32_t w_dtype,
                                                   int32_t k) {
    if (n_rows <= 0 || vocab <= 0 || d_model <= 0 || k < 1 || k > 16) return 0;
    RowsView rv;
    rows_view(rv, n_rows);
    return rv.index_bytes + score_layout(rv.P, vocab, d_model, w_dtype, k).total;
}

extern "C" spinf_status spinf_score_rows(const spinf_plan* plan, const void* hidden, int32_t n_rows, const void* w,
                                         const float* w_scale, int32_t w_dtype, int32_t d_model, int32_t vocab,
                                         const int32_t* token_set, const uint32_t* token_sets, int32_t n_sets,
                                         int32_t k, float* row_lse, int32_t* top_tok, float* top_lp, void* workspace,
                                         size_t workspace_bytes, spinf_stream stream) {
    if (!plan || !plan->d_err) return fail(SPINF_E_INVALID, "an uploaded plan is needed (its device error word)");
    if (w_dtype != SPINF_DTYPE_BF16 && w_dtype != SPINF_DTYPE_E4M3) return fail(SPINF_E_UNSUPPORTED, "w_dtype");
    if (d_model <= 0 || d_model % 16) return fail(SPINF_E_UNSUPPORTED, "d_model must be a positive multiple of 16");
    if (vocab <= 0) return fail(SPINF_E_INVALID, "vocab must be positive");
    if (k < 1 || k > 16) return fail(SPINF_E_INVALID, "k must be in 1..16");
    if (n_rows < 0 || n_sets < 0) return fail(SPINF_E_INVALID, "negative count");
    if (n_rows == 0) return SPINF_OK;
    if (!hidden || !w || !row_lse || !top_tok || !top_lp || !workspace) return fail(SPINF_E_INVALID, "NULL buffer");
    if (n_sets > 0 && !token_sets) return fail(SPINF_E_INVALID, "token_sets is NULL");
    if (w_dtype == SPINF_DTYPE_E4M3 && (!w_scale || (reinterpret_cast<uintptr_t>(w_scale) & 15)))
        return fail(SPINF_E_INVALID, "e4m3 weights need a 16-byte aligned w_scale");
    for (const void* p : {hidden, w, (const void*)workspace})
        if (reinterpret_cast<uintptr_t>(p) & 15) return fail(SPINF_E_INVALID, "buffer not 16-byte aligned");
    RowsView rv;
    rows_view(rv, n_rows);
    Pass& P = rv.P;
    const ScoreLayout L = score_layout(P, vocab, d_model, w_dtype, k);
    if (workspace_bytes < rv.index_bytes + L.total) return fail(SPINF_E_NOMEM, "workspace too small");
    uint8_t* base = static_cast<uint8_t*>(workspace);
    const size_t a = align256((size_t)n_rows * 4);
    P.dev.slot_row = reinterpret_cast<int32_t*>(base);
    P.dev.row_x = reinterpret_cast<int32_t*>(base + a);
    P.dev.x_m = reinterpret_cast<int32_t*>(base + 2 * a);
    P.dev.x_set = reinterpret_cast<int32_t*>(base + 3 * a);
    P.dev.row_gptr = reinterpret_cast<int32_t*>(base + 4 * a);
    P.dev.row_glist = P.dev.row_gptr;   // no gathers: never read
    P.dev.gather_tok = P.dev.row_gptr;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    rows_tables_kernel<<<(n_rows + 256) / 256, 256, 0, s>>>(n_rows, token_set, P.dev.slot_row, P.dev.row_x, P.dev.x_m,
                                                           P.dev.x_set, P.dev.row_gptr);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "row tables launch");
    spinf_extract_out ex{token_sets, n_sets, top_tok, top_lp};
    uint8_t* ws = base + rv.index_bytes;
    const float* wsc = w_dtype == SPINF_DTYPE_E4M3 ? w_scale : nullptr;
    using F = std::false_type;
    using T = std::true_type;
    auto go = [&](auto fp8, auto kx_c) {
        return launch_score<decltype(fp8)::value, decltype(kx_c)::value>(P, L, hidden, w, wsc, d_model, vocab, row_lse,
                                                                         nullptr, &ex, ws, plan->d_err, s);
    };
    using K8 = std::integral_constant<int, 8>;
    using K16 = std::integral_constant<int, 16>;
    if (w_dtype == SPINF_DTYPE_E4M3) return k <= 8 ? go(T{}, K8{}) : go(T{}, K16{});
    return k <= 8 ? go(F{}, K8{}) : go(F{}, K16{});
}

// ---------------------------------------------------------------- allocation-free variant
// For callers that may not allocate device memory: the scratch of the scoring
// kernels lives in one file-scope device array per GPU.  Host code must not use
// the array's name as a device address (on the host it only names the symbol);
// its device address is looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_score_scratch[SPINF_SCORE_STATIC_SCRATCH_BYTES];

namespace spinf {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
// per device: the context the address was looked up in, and the address
CUcontext g_scratch_ctx[kMaxDevices] = {};
void* g_scratch_addr[kMaxDevices] = {};

// The calling thread's current driver context (nullptr if the entry point is missing).
CUcontext current_context() {
    using CtxGetCurrent = CUresult (*)(CUcontext*);
    static CtxGetCurrent fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<CtxGetCurrent>(p);
        return static_cast<CtxGetCurrent>(nullptr);
    }();
    CUcontext c = nullptr;
    if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
    return c;
}

// Device address of this GPU's scratch array.  The first call per device looks it up,
// and so does the first call after the device's context changed (a cudaDeviceReset
// makes a new primary context, in which the array has a new address).
spinf_status static_scratch(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(SPINF_E_UNSUPPORTED, "device index beyond the static scratch table");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    // the runtime makes the device's primary context current before the symbol lookup
    void* p = nullptr;
    if (!g_scratch_addr[dev] || g_scratch_ctx[dev] != current_context()) {
        e = cudaGetSymbolAddress(&p, g_score_scratch);
        if (e != cudaSuccess || !p) return cuda_fail(e, "cudaGetSymbolAddress(scoring scratch)");
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = current_context();
    }
    *out = g_scratch_addr[dev];
    return SPINF_OK;
}

}  // namespace
}  // namespace spinf

extern "C" spinf_status spinf_score_static(const spinf_plan* plan, int32_t pass, const void* hidden, const void* w,
                                           const float* w_scale, int32_t w_dtype, int32_t d_model, int32_t vocab,
                                           float* row_lse, float* token_lp, spinf_stream stream) {
    spinf_status st = ensure_device_ready(plan, pass);
    if (st) return st;
    if (w_dtype != SPINF_DTYPE_BF16 && w_dtype != SPINF_DTYPE_E4M3) return fail(SPINF_E_UNSUPPORTED, "w_dtype");
    if (d_model <= 0 || d_model % 16) return fail(SPINF_E_UNSUPPORTED, "d_model must be a positive multiple of 16");
    if (vocab <= 0) return fail(SPINF_E_INVALID, "vocab must be positive");
    const Pass& P = plan->passes[pass];
    if (P.slot_row.empty()) return SPINF_OK;
    const ScoreLayout L = score_layout(P, vocab, d_model, w_dtype, plan->extract_k);
    if (L.total > (size_t)SPINF_SCORE_STATIC_SCRATCH_BYTES)
        return fail(SPINF_E_LIMIT, "this pass needs " + std::to_string(L.total) +
                                       " bytes of scoring scratch; the static area holds " +
                                       std::to_string((size_t)SPINF_SCORE_STATIC_SCRATCH_BYTES) +
                                       " (use spinf_score with a caller workspace)");
    if (!hidden || !w || !row_lse || !token_lp) return fail(SPINF_E_INVALID, "NULL buffer");
    if (w_dtype == SPINF_DTYPE_E4M3 && !w_scale) return fail(SPINF_E_INVALID, "e4m3 weights need w_scale");
    if (w_dtype == SPINF_DTYPE_E4M3 && (reinterpret_cast<uintptr_t>(w_scale) & 15))
        return fail(SPINF_E_INVALID, "w_scale must be 16-byte aligned");
    for (const void* p : {hidden, w})
        if (reinterpret_cast<uintptr_t>(p) & 15) return fail(SPINF_E_INVALID, "buffer not 16-byte aligned");
    for (int32_t t : P.gather_tok)
        if (t < 0 || t >= vocab) return fail(SPINF_E_INVALID, "option token outside the vocabulary");
    void* scratch = nullptr;
    if ((st = static_scratch(&scratch))) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(scratch);
    if (w_dtype == SPINF_DTYPE_E4M3)
        return launch_score<true, 0>(P, L, hidden, w, w_scale, d_model, vocab, row_lse, token_lp, nullptr, ws,
                                         plan->d_err, s);
    return launch_score<false, 0>(P, L, hidden, w, nullptr, d_model, vocab, row_lse, token_lp, nullptr, ws,
                                      plan->d_err, s);
}
