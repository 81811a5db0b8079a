// The steps around the attention call that complete a packed layer: the QKV
// projection with rotary position embedding at tree positions, the output
// projection, and the fp8 form of both with static scales.
//
// The method ("spinf-serve 0.1.1", PyPI page, "What it does"): every question is
// a branch of the packed pass, and an input's scores are the same alone or
// packed.  A token's position is therefore its depth on its own root path (the
// plan's pos[]), never its row in the pass: a branch token gets the positions its
// unpacked sequence (content, question, option prefix) would give it.  The fp8
// scheme that keeps scores bit-identical alone or packed ("spinf-serve" man page,
// DESCRIPTION, --quant fp8s) has static scales: one per activation tensor, one
// per weight output channel, fixed before the request.
//
//   linear_kernel<FP8, MODE>   persistent tcgen05 GEMM y = x w^T: 128 rows x 256
//                              output features per tile, fp32 in TMEM (two
//                              accumulators), a 4-stage TMA ring, the output
//                              staged per warp and written by TMA stores.  MODE 0
//                              writes y; MODE 1 (QKV) turns the q and k columns by
//                              the row's tree position in the epilogue and writes
//                              q, k, v in the attention kernel's layouts.
//   quantize_static_kernel     bf16 -> e4m3 codes with a static scale
//   rope_tree_kernel           the rotary embedding alone, in place on q and k
//
// Each output element is one fixed-order reduction over the input features, by
// the same tile code wherever its row sits, so a row's output does not depend on
// the other rows of the call (no split of the reduction, no algorithm choice by
// size).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "runtime.h"

namespace spinf {
namespace {

using namespace dev;

// ---------------------------------------------------------------- rotary table
// cos and sin of pos * theta^(-2i/d) for every pos of the pass (0..max pos), i < d/2,
// formed in fp64 on the host and rounded to fp32: the fused projection and the
// stand-alone rotation read the same values.  Frequency-major ([i][pos], `stride` =
// max pos + 1): the rows of a tile mostly hold consecutive positions (a content, a
// template), so one warp load of a frequency touches one or two lines.
spinf_status rope_table(Pass& P, int32_t d, float theta, cudaStream_t stream, const float2** out, int* stride) {
    for (auto& t : P.ropes)
        if (t->d == d && t->theta == theta && t->dev) {
            *out = t->dev;
            *stride = t->stride;
            return SPINF_OK;
        }
    auto t = std::make_unique<RopeTable>();
    t->d = d;
    t->theta = theta;
    int32_t max_pos = 0;
    for (int32_t r = 0; r < P.T_pad; ++r) max_pos = std::max(max_pos, P.pos[r]);
    const int32_t half = d / 2;
    t->stride = max_pos + 1;
    t->host.resize((size_t)t->stride * half);
    const double lt = std::log2(static_cast<double>(theta));
    for (int32_t i = 0; i < half; ++i) {
        const double inv_freq = std::exp2(-lt * (2.0 * i) / d);
        for (int32_t p = 0; p <= max_pos; ++p) {
            const double a = p * inv_freq;
            t->host[(size_t)i * t->stride + p] =
                make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
        }
    }
    void* mem = nullptr;
    cudaError_t e = cudaMalloc(&mem, t->host.size() * sizeof(float2));
    if (e != cudaSuccess) return fail(SPINF_E_NOMEM, "device allocation of a rotary table failed");
    e = cudaMemcpyAsync(mem, t->host.data(), t->host.size() * sizeof(float2), cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) {
        cudaFree(mem);
        return cuda_fail(e, "rotary table upload");
    }
    t->dev = static_cast<float2*>(mem);
    *out = t->dev;
    *stride = t->stride;
    P.ropes.push_back(std::move(t));
    return SPINF_OK;
}

// One CTA per packed row; the row's table entries are shared by its heads.
__global__ void rope_tree_kernel(__nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ k,
                                 const int32_t* __restrict__ pos, const float2* __restrict__ table, int stride,
                                 int Hq, int Hkv, int d) {
    const int row = blockIdx.x, half = d / 2;
    const float2* cs = table + __ldg(pos + row);   // entry i at cs[i * stride]
    const int pairs_q = Hq * half, pairs = (Hq + Hkv) * half;
    for (int j = threadIdx.x; j < pairs; j += blockDim.x) {
        const bool is_q = j < pairs_q;
        const int jj = is_q ? j : j - pairs_q;
        const int h = jj / half, i = jj - h * half;
        __nv_bfloat16* base = is_q ? q + (static_cast<size_t>(row) * Hq + h) * d
                                   : k + (static_cast<size_t>(row) * Hkv + h) * d;
        const float x0 = __bfloat162float(base[i]), x1 = __bfloat162float(base[i + half]);
        const float2 r = __ldg(cs + (size_t)i * stride);
        base[i] = __float2bfloat16_rn(x0 * r.x - x1 * r.y);
        base[i + half] = __float2bfloat16_rn(x1 * r.x + x0 * r.y);
    }
}

// ---------------------------------------------------------------- static e4m3 codes
__global__ void quantize_static_kernel(const __nv_bfloat16* __restrict__ x, float scale, uint8_t* __restrict__ out,
                                       int64_t n8) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 u = reinterpret_cast<const uint4*>(x)[i];
        const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(b[j]);
            const float2 qv = make_float2(__fdiv_rn(f.x, scale), __fdiv_rn(f.y, scale));
            const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(qv, __NV_SATFINITE, __NV_E4M3);
            w[j >> 1] |= static_cast<uint32_t>(c) << ((j & 1) * 16);
        }
        reinterpret_cast<uint2*>(out)[i] = make_uint2(w[0], w[1]);
    }
}

// ---------------------------------------------------------------- projection GEMM
constexpr int kLM = 128;   // rows per tile (MMA M, TMEM lanes)
constexpr int kLN = 256;   // output features per tile (MMA N)
constexpr int kLStages = 4;
constexpr int kLA = kLM * 128;
constexpr int kLB = kLN * 128;
constexpr int kLStage = kLA + kLB;
constexpr int kLThreads = 192;
enum { LFULL0 = 0, LEMPTY0 = kLStages, LACC_FULL0 = 2 * kLStages, LACC_EMPTY0 = 2 * kLStages + 2,
       LN_BARS = 2 * kLStages + 4 };
constexpr int kLSmemBars = kLStages * kLStage;
constexpr int kLSmemHolder = kLSmemBars + (LN_BARS + 1) * 8;
// output staging: per epilogue warp two 32-row x 32-column bf16 boxes, written by TMA stores
constexpr int kLStageBytes = 32 * 32 * 2;
constexpr int kLStageOff = (kLSmemHolder + 16 + 1023) / 1024 * 1024;
constexpr int kLSmem = kLStageOff + 4 * 2 * kLStageBytes + 1024;
static_assert(kLSmem <= 227 * 1024, "shared memory of one CTA");

// Where the product's columns go.  MODE 0: all to y[0] (row stride ld[0]).  MODE 1:
// product column n belongs to output o = 0 (q), 1 (k) or 2 (v) by base[]; columns
// below n_rot (q and k) are turned by the row's position, pairs (i, i + d/2) of
// each d-column head.
struct LinearOut {
    __nv_bfloat16* y[3];
    int ld[3];
    int base[3];
    int n_rot;
    int d;
    const float2* cs;      // [d / 2][stride] (cos, sin), frequency-major
    int stride;            // max pos + 1
    const int32_t* pos;    // [rows]
};

// Tile order.  rpb == 0: row tile by row tile, every feature tile of a row tile next to each other,
// so each row tile is read from HBM once and the weights stay in L2 (when they fit beside the
// output stream).  rpb > 0: blocks of up to rpb row tiles; within a block, feature tile by
// feature tile, the block's row tiles next to each other: a block's rows (at most ~32 MB) stay in
// L2 while weights too large to stay there stream past once per block.
__device__ __forceinline__ void linear_tile(int u, int n_mt, int n_nt, int rpb, int& mt, int& nt) {
    if (rpb == 0) {
        mt = u / n_nt;
        nt = u % n_nt;
        return;
    }
    const int per_block = n_nt * rpb;
    const int rb = u / per_block;
    const int rem = u - rb * per_block;
    const int rows = min(rpb, n_mt - rb * rpb);
    nt = rem / rows;
    mt = rb * rpb + rem % rows;
}

template <bool FP8, int MODE>
__global__ void __launch_bounds__(kLThreads, 1)
    linear_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                  const __grid_constant__ CUtensorMap tm_y0, const __grid_constant__ CUtensorMap tm_y1,
                  const __grid_constant__ CUtensorMap tm_y2,
                  const float* __restrict__ w_scale, float x_scale, const LinearOut out, int rows, int N, int n_kb,
                  int n_mt, int n_nt, int rpb, int* __restrict__ err) {
    constexpr int kPerMma = FP8 ? 32 : 16;
    constexpr int kMmaPerStage = (FP8 ? 128 : 64) / kPerMma;
    constexpr int kBK = FP8 ? 128 : 64;
    constexpr uint32_t idesc = FP8 ? idesc_e4m3(kLM, kLN) : idesc_bf16(kLM, kLN, false, false);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kLSmemBars);
    uint32_t* holder = reinterpret_cast<uint32_t*>(smem + kLSmemHolder);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = n_mt * n_nt;
    const int first = (int)blockIdx.x;
    const int stride = (int)gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kLStages; ++s) {
            mbar_init(&bars[LFULL0 + s], 1);
            mbar_init(&bars[LEMPTY0 + s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&bars[LACC_FULL0 + a], 1);
            mbar_init(&bars[LACC_EMPTY0 + a], 128);
        }
        mbar_init(&bars[LN_BARS], 1);
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
            tma_prefetch_desc(&tm_x);
            tma_prefetch_desc(&tm_w);
            uint32_t it = 0;
            for (int u = first; u < total; u += stride) {
                int mt, nt;
                linear_tile(u, n_mt, n_nt, rpb, mt, nt);
                for (int kb = 0; kb < n_kb; ++kb, ++it) {
                    const int s = it % kLStages;
                    mbar_wait(&bars[LEMPTY0 + s], ((it / kLStages) & 1) ^ 1, err);
                    uint8_t* sa = smem + s * kLStage;
                    // the stage receives the whole tile: the row block and the weight tile
                    mbar_arrive_expect_tx(&bars[LFULL0 + s], kLStage);
                    tma_load_2d(sa, &tm_x, &bars[LFULL0 + s], kb * kBK, mt * kLM);
                    tma_load_2d(sa + kLA, &tm_w, &bars[LFULL0 + s], kb * kBK, nt * kLN);
                }
            }
            for (uint32_t i = it > (uint32_t)kLStages ? it - kLStages : 0; i < it; ++i)
                mbar_drain(&bars[LFULL0 + i % kLStages], (i / kLStages) & 1, err);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t it = 0, tcount = 0;
            for (int u = first; u < total; u += stride, ++tcount) {
                const int acc = tcount & 1;
                mbar_wait(&bars[LACC_EMPTY0 + acc], ((tcount >> 1) & 1) ^ 1, err);
                tc_fence_after();
                const uint32_t d_tmem = tmem + acc * kLN;
                for (int kb = 0; kb < n_kb; ++kb, ++it) {
                    const int s = it % kLStages;
                    mbar_wait(&bars[LFULL0 + s], (it / kLStages) & 1, err);
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(smem + s * kLStage);
                    const uint32_t b_base = a_base + kLA;
#pragma unroll
                    for (int kk = 0; kk < kMmaPerStage; ++kk) {
                        const uint64_t da = sdesc_sw128(a_base + kk * 32, 16, 1024);
                        const uint64_t db = sdesc_sw128(b_base + kk * 32, 16, 1024);
                        if (FP8) mma_f8_ss(d_tmem, da, db, idesc, (kb | kk) != 0);
                        else mma_f16_ss(d_tmem, da, db, idesc, (kb | kk) != 0);
                    }
                    mma_commit(&bars[LEMPTY0 + s]);
                }
                mma_commit(&bars[LACC_FULL0 + acc]);
            }
            // every MMA (and so every commit to this CTA's barriers) has completed before exit
            mma_commit(&bars[LN_BARS]);
            mbar_drain(&bars[LN_BARS], 0, err);
        }
    } else {
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        uint8_t* stage_base = smem + kLStageOff + (warp - 2) * 2 * kLStageBytes;
        int sb = 0;   // the staging box the next chunk goes to
        uint32_t tcount = 0;
        for (int u = first; u < total; u += stride, ++tcount) {
            int mt, nt;
            linear_tile(u, n_mt, n_nt, rpb, mt, nt);
            const int acc = tcount & 1;
            const int row = mt * kLM + r;
            const int n0 = nt * kLN;
            const bool valid = row < rows;
            const float2* cs = nullptr;
            if (MODE == 1 && valid) cs = out.cs + __ldg(out.pos + row);   // entry i at cs[i * stride]
            mbar_wait(&bars[LACC_FULL0 + acc], (tcount >> 1) & 1, err);
            tc_fence_after();
            const uint32_t t0 = tmem + lane_off + acc * kLN;
            // product columns n0 + 32c .. + 31 (< N) of the raw accumulator, scaled for e4m3
            auto scale = [&](int c, const uint32_t (&rr)[32], float (&v)[32]) {
                if constexpr (FP8) {
                    // the chunk's 32 channel scales as 8 vector loads (N is a multiple of 32)
                    const float4* ws4 = reinterpret_cast<const float4*>(w_scale + n0 + c * 32);
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        const float4 sc = __ldg(ws4 + q4);
                        v[4 * q4 + 0] = (__uint_as_float(rr[4 * q4 + 0]) * sc.x) * x_scale;
                        v[4 * q4 + 1] = (__uint_as_float(rr[4 * q4 + 1]) * sc.y) * x_scale;
                        v[4 * q4 + 2] = (__uint_as_float(rr[4 * q4 + 2]) * sc.z) * x_scale;
                        v[4 * q4 + 3] = (__uint_as_float(rr[4 * q4 + 3]) * sc.w) * x_scale;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(rr[i]);
                }
            };
            const int half = MODE == 1 ? out.d / 2 : 0;
            // the 32 columns from product column n of this warp's 32 rows: each lane writes its row
            // into a staging box (16-byte pieces at slots piece ^ ((row >> 1) & 3), the 64-byte
            // swizzle of the output maps), then one TMA store writes the box; rows past the end are
            // clipped by the map.  A box is rewritten only after its previous store has read it.
            auto put = [&](int n, const float (&v)[32]) {
                const int o = MODE == 0 ? 0 : n < out.base[1] ? 0 : n < out.base[2] ? 1 : 2;
                const int col = n - (o == 0 ? out.base[0] : o == 1 ? out.base[1] : out.base[2]);
                uint8_t* st = stage_base + sb * kLStageBytes;
                if (lane == 0) tma_store_wait_read1();
                __syncwarp();
                uint4* srow = reinterpret_cast<uint4*>(st + lane * 64);
                const int sx = (lane >> 1) & 3;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    srow[i ^ sx] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                              pack_bf16x2(v[8 * i + 4], v[8 * i + 5]),
                                              pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && mt * kLM + quarter * 32 < rows) {   // a box wholly past the last row is not stored
                    tma_store_2d(o == 0 ? &tm_y0 : o == 1 ? &tm_y1 : &tm_y2, st, col, mt * kLM + quarter * 32);
                    tma_store_commit();
                }
                sb ^= 1;
            };
#pragma unroll 1
            for (int c = 0; c < kLN / 32; ++c) {
                const int n = n0 + c * 32;
                if (n >= N) break;
                if (MODE == 1 && n < out.n_rot) {   // q or k: chunk c and its partner half a head later
                    const int j = (n - (n < out.base[1] ? out.base[0] : out.base[1])) % out.d;
                    if (j >= half) continue;   // written with its first half
                    float2 tab[32];            // (cos, sin), fetched before the TMEM wait
                    if (valid) {
                        const float2* c0 = cs + (size_t)j * out.stride;
#pragma unroll
                        for (int i = 0; i < 32; ++i) tab[i] = __ldg(c0 + (size_t)i * out.stride);
                    }
                    uint32_t ra[32], rb[32];
                    tmem_ld32x2(t0 + c * 32, t0 + (c + half / 32) * 32, ra, rb);
                    float x0[32], x1[32];
                    scale(c, ra, x0);
                    scale(c + half / 32, rb, x1);
                    if (valid) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float a = x0[i], b = x1[i];
                            x0[i] = a * tab[i].x - b * tab[i].y;
                            x1[i] = b * tab[i].x + a * tab[i].y;
                        }
                    }
                    put(n, x0);
                    put(n + half, x1);
                    continue;
                }
                // no turn: this chunk and (when it is not a turned one) the next, one TMEM wait
                const bool two = c + 1 < kLN / 32 && n + 32 < N && !(MODE == 1 && n + 32 < out.n_rot);
                uint32_t ra[32], rb[32];
                if (two) tmem_ld32x2(t0 + c * 32, t0 + (c + 1) * 32, ra, rb);
                else tmem_ld32(t0 + c * 32, ra);
                float v[32];
                scale(c, ra, v);
                put(n, v);
                if (two) {
                    scale(c + 1, rb, v);
                    put(n + 32, v);
                    ++c;
                }
            }
            tc_fence_before();
            mbar_arrive(&bars[LACC_EMPTY0 + acc]);
        }
        if (lane == 0) tma_store_wait_all();   // this warp's stores have completed before the CTA retires
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <bool FP8, int MODE>
spinf_status launch_linear(const void* x, const void* w, const float* w_scale, float x_scale, const LinearOut& out,
                           int64_t rows, int64_t K, int64_t N, int* err, cudaStream_t stream) {
    CUtensorMap tx, tw;
    const uint64_t elt = FP8 ? 1 : 2;
    const uint64_t dx[2] = {(uint64_t)K, (uint64_t)rows};
    const uint64_t dw[2] = {(uint64_t)K, (uint64_t)N};
    const uint64_t st[1] = {(uint64_t)K * elt};
    const uint32_t bx[2] = {FP8 ? 128u : 64u, (uint32_t)kLM};
    const uint32_t bw[2] = {FP8 ? 128u : 64u, (uint32_t)kLN};
    const CUtensorMapDataType dt = FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    spinf_status s;
    if ((s = make_tmap(&tx, dt, 2, x, dx, st, bx, CU_TENSOR_MAP_SWIZZLE_128B))) return s;
    if ((s = make_tmap(&tw, dt, 2, w, dw, st, bw, CU_TENSOR_MAP_SWIZZLE_128B))) return s;
    if ((s = set_smem_limit(reinterpret_cast<const void*>(linear_kernel<FP8, MODE>), kLSmem,
                            "cudaFuncSetAttribute(linear)")))
        return s;
    cudaError_t e;
    const int kbk = FP8 ? 128 : 64;
    const int n_kb = (int)((K + kbk - 1) / kbk);
    const int n_mt = (int)((rows + kLM - 1) / kLM), n_nt = (int)((N + kLN - 1) / kLN);
    const int grid = std::min(n_mt * n_nt, sm_count());
    // weights of more than 48 MB do not stay in L2 beside the output stream (measured: the bf16
    // QKV weights, 63 MB, were read ~14 times from HBM in row-tile order); smaller ones do
    const long long row_tile = (long long)kLM * K * (long long)elt;
    const bool big_w = (long long)N * K * (long long)elt > (48ll << 20);
    const int rpb = big_w ? (int)std::max(1ll, std::min<long long>((32ll << 20) / std::max(1ll, row_tile), n_mt)) : 0;
    // outputs as 2-D (columns, rows) maps, 32 x 32 boxes with the 64-byte swizzle of the staging
    CUtensorMap ty[3];
    const int n_out = MODE == 0 ? 1 : 3;
    for (int o = 0; o < 3; ++o) {
        if (o >= n_out) {
            ty[o] = ty[0];
            continue;
        }
        const int64_t width = MODE == 0 ? N : (o == 0 ? out.base[1] : o == 1 ? out.base[2] - out.base[1] : N - out.base[2]);
        const uint64_t dy[2] = {(uint64_t)width, (uint64_t)rows};
        const uint64_t sy[1] = {(uint64_t)out.ld[o] * 2};
        const uint32_t by[2] = {32u, 32u};
        if ((s = make_tmap(&ty[o], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, out.y[o], dy, sy, by, CU_TENSOR_MAP_SWIZZLE_64B)))
            return s;
    }
    linear_kernel<FP8, MODE><<<grid, kLThreads, kLSmem, stream>>>(tx, tw, ty[0], ty[1], ty[2], w_scale, x_scale, out,
                                                                 (int)rows, (int)N, n_kb, n_mt, n_nt, rpb, err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "linear launch");
    return SPINF_OK;
}

spinf_status check_dtype_args(int32_t w_dtype, const float* w_scale, float x_scale) {
    if (w_dtype != SPINF_DTYPE_BF16 && w_dtype != SPINF_DTYPE_E4M3) return fail(SPINF_E_UNSUPPORTED, "w_dtype");
    if (w_dtype == SPINF_DTYPE_E4M3 && (!w_scale || !(x_scale > 0.f) || !std::isfinite(x_scale)))
        return fail(SPINF_E_INVALID, "e4m3 needs w_scale and a positive finite x_scale");
    if (w_dtype == SPINF_DTYPE_E4M3 && (reinterpret_cast<uintptr_t>(w_scale) & 15))
        return fail(SPINF_E_INVALID, "w_scale must be 16-byte aligned");
    return SPINF_OK;
}

}  // namespace
}  // namespace spinf

using namespace spinf;

extern "C" spinf_status spinf_rope_tree(const spinf_plan* plan, int32_t pass, void* q, void* k, int32_t n_q_heads,
                                        int32_t n_kv_heads, int32_t d_head, float theta, spinf_stream stream) {
    spinf_status st = ensure_device_ready(plan, pass);
    if (st) return st;
    if (!q || !k) return fail(SPINF_E_INVALID, "NULL tensor");
    if (n_q_heads <= 0 || n_kv_heads <= 0 || d_head <= 0 || d_head % 2 || d_head > 1024)
        return fail(SPINF_E_INVALID, "bad head counts or d_head");
    if (!(theta > 1.f) || !std::isfinite(theta)) return fail(SPINF_E_INVALID, "theta must be > 1");
    Pass& P = const_cast<Pass&>(plan->passes[pass]);
    if (P.T_pad == 0) return SPINF_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float2* table = nullptr;
    int stride = 0;
    {
        std::lock_guard<std::mutex> lock(const_cast<spinf_plan*>(plan)->cache_mu);
        if ((st = rope_table(P, d_head, theta, s, &table, &stride))) return st;
    }
    rope_tree_kernel<<<P.T_pad, 256, 0, s>>>(static_cast<__nv_bfloat16*>(q), static_cast<__nv_bfloat16*>(k),
                                             P.dev.pos, table, stride, n_q_heads, n_kv_heads, d_head);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "rope launch");
    return SPINF_OK;
}

extern "C" spinf_status spinf_quantize_static(const void* x, float x_scale, void* codes, int64_t n,
                                              spinf_stream stream) {
    if (!x || !codes) return fail(SPINF_E_INVALID, "NULL tensor");
    if (n < 0 || n % 8) return fail(SPINF_E_INVALID, "n must be a non-negative multiple of 8");
    if (!(x_scale > 0.f) || !std::isfinite(x_scale)) return fail(SPINF_E_INVALID, "x_scale must be positive");
    if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(codes) & 7))
        return fail(SPINF_E_INVALID, "x must be 16-byte and codes 8-byte aligned");
    if (n == 0) return SPINF_OK;
    const int64_t n8 = n / 8;
    const int grid = (int)std::min<int64_t>((n8 + 255) / 256, (int64_t)sm_count() * 8);
    quantize_static_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16*>(x), x_scale, static_cast<uint8_t*>(codes), n8);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    return SPINF_OK;
}

extern "C" spinf_status spinf_linear(const spinf_plan* plan, const void* x, const void* w, const float* w_scale,
                                     float x_scale, int32_t w_dtype, void* y, int64_t rows, int64_t in_features,
                                     int64_t out_features, spinf_stream stream) {
    if (!plan || !plan->d_err) return fail(SPINF_E_INVALID, "an uploaded plan is needed (its device error word)");
    spinf_status st = check_dtype_args(w_dtype, w_scale, x_scale);
    if (st) return st;
    if (!x || !w || !y) return fail(SPINF_E_INVALID, "NULL tensor");
    const bool fp8 = w_dtype == SPINF_DTYPE_E4M3;
    if (rows < 0 || rows > INT32_MAX || in_features <= 0 || in_features % (fp8 ? 16 : 8) || out_features <= 0 ||
        out_features % 32 || out_features > INT32_MAX)
        return fail(SPINF_E_INVALID, "bad sizes (in_features a multiple of 8, 16 for e4m3; out_features of 32)");
    for (const void* p : {x, w, (const void*)y})
        if (reinterpret_cast<uintptr_t>(p) & 15) return fail(SPINF_E_INVALID, "tensor not 16-byte aligned");
    if (rows == 0) return SPINF_OK;
    LinearOut out{};
    out.y[0] = static_cast<__nv_bfloat16*>(y);
    out.ld[0] = (int)out_features;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (fp8) return launch_linear<true, 0>(x, w, w_scale, x_scale, out, rows, in_features, out_features, plan->d_err, s);
    return launch_linear<false, 0>(x, w, nullptr, 1.f, out, rows, in_features, out_features, plan->d_err, s);
}

extern "C" spinf_status spinf_qkv_rope(const spinf_plan* plan, int32_t pass, const void* x, const void* w,
                                       const float* w_scale, float x_scale, int32_t w_dtype, int32_t d_model,
                                       int32_t n_q_heads, int32_t n_kv_heads, int32_t d_head, float theta, void* q,
                                       void* k, void* v, spinf_stream stream) {
    spinf_status st = ensure_device_ready(plan, pass);
    if (st) return st;
    if ((st = check_dtype_args(w_dtype, w_scale, x_scale))) return st;
    if (!x || !w || !q || !k || !v) return fail(SPINF_E_INVALID, "NULL tensor");
    const bool fp8 = w_dtype == SPINF_DTYPE_E4M3;
    if (d_head != 64 && d_head != 128 && d_head != 256) return fail(SPINF_E_UNSUPPORTED, "d_head must be 64, 128 or 256");
    if (n_q_heads <= 0 || n_kv_heads <= 0) return fail(SPINF_E_INVALID, "bad head counts");
    if (d_model <= 0 || d_model % (fp8 ? 16 : 8)) return fail(SPINF_E_INVALID, "bad d_model");
    if (!(theta > 1.f) || !std::isfinite(theta)) return fail(SPINF_E_INVALID, "theta must be > 1");
    for (const void* p : {x, w, (const void*)q, (const void*)k, (const void*)v})
        if (reinterpret_cast<uintptr_t>(p) & 15) return fail(SPINF_E_INVALID, "tensor not 16-byte aligned");
    Pass& P = const_cast<Pass&>(plan->passes[pass]);
    if (P.T_pad == 0) return SPINF_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float2* table = nullptr;
    int stride = 0;
    {
        std::lock_guard<std::mutex> lock(const_cast<spinf_plan*>(plan)->cache_mu);
        if ((st = rope_table(P, d_head, theta, s, &table, &stride))) return st;
    }
    LinearOut out{};
    out.y[0] = static_cast<__nv_bfloat16*>(q);
    out.y[1] = static_cast<__nv_bfloat16*>(k);
    out.y[2] = static_cast<__nv_bfloat16*>(v);
    out.ld[0] = n_q_heads * d_head;
    out.ld[1] = out.ld[2] = n_kv_heads * d_head;
    out.base[0] = 0;
    out.base[1] = n_q_heads * d_head;
    out.base[2] = (n_q_heads + n_kv_heads) * d_head;
    out.n_rot = out.base[2];
    out.d = d_head;
    out.cs = table;
    out.stride = stride;
    out.pos = P.dev.pos;
    const int64_t N = (int64_t)(n_q_heads + 2 * n_kv_heads) * d_head;
    if (fp8) return launch_linear<true, 1>(x, w, w_scale, x_scale, out, P.T_pad, d_model, N, plan->d_err, s);
    return launch_linear<false, 1>(x, w, nullptr, 1.f, out, P.T_pad, d_model, N, plan->d_err, s);
}
