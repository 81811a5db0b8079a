// Decoding steps of searched slots on the cached keys and values of a packed pass.
//
// The method ("spinf-serve 0.1.1", PyPI page, "What it does" and "Speed and
// scale"): extraction slots ({*} text, {n} numbers, {$} amounts) are decoded on
// the same read of the content -- the content and the questions are not read
// again, and the slots of many inputs are decoded together.  A decode row extends
// the root path of a searched slot's row (its anchor) by the tokens chosen at
// earlier steps; it attends to the keys the anchor sees in the pass (read from the
// pass's K and V, not recomputed), then to the decode rows of its own chain, down
// to itself.  So its output is that of the same tokens written into the template
// and laid out in a pass.
//
//   decode_attention_kernel<D>  one CTA per (decode row, kv head), one warp per
//                               query head of the group.  Keys are visited in a
//                               fixed order (the anchor's path in ascending rows,
//                               then the chain from its first token): a row's output
//                               does not depend on the other rows of the step.
//                               Memory-bound: each key row is read once per group.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <type_traits>
#include <utility>
#include <vector>

#include "internal.h"
#include "ptx.cuh"
#include "runtime.h"

namespace spinf {
namespace {

constexpr int kMaxChain = 64;   // decoded tokens per chain (a searched answer is short)

// D / 32 consecutive elements of a bf16 row as fp32 (one 4-, 8- or 16-byte load per lane).
template <int D>
__device__ __forceinline__ void load_row(const __nv_bfloat16* __restrict__ p, float (&x)[D / 32]) {
    constexpr int E = D / 32;
    if constexpr (E == 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(b[j]);
            x[2 * j] = f.x;
            x[2 * j + 1] = f.y;
        }
    } else if constexpr (E == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float2 f = __bfloat1622float2(b[j]);
            x[2 * j] = f.x;
            x[2 * j + 1] = f.y;
        }
    } else {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
        x[0] = f.x;
        x[1] = f.y;
    }
}

// Thread 0 walks the row's chain and fetches its anchor's runs into shared memory,
// checking every index against its array; a row that fails a check is written as
// zeros and raises the plan's error word (SPINF_E_DEVICE_CHECK).  The row's keys (the
// anchor's path, then the chain) are split into kSlices contiguous slices, one warp per
// slice; a warp serves all G query heads of the kv head, so each key and value row is
// loaded once.  The slices' (max, sum, accumulator) are merged in slice order, so the
// result depends on the row's keys and the head grouping only.
// 8 slices, or 4 when 8 slices' partial accumulators would not fit 40 KB of shared memory
template <int D, int G>
constexpr int slices() { return G * D * 4 * 8 <= 40960 ? 8 : 4; }

template <int D, int G>
__global__ void __launch_bounds__(32 * slices<D, G>()) decode_attention_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_pass,
    const __nv_bfloat16* __restrict__ v_pass, const __nv_bfloat16* __restrict__ k_dec,
    const __nv_bfloat16* __restrict__ v_dec, const int32_t* __restrict__ anchor, const int32_t* __restrict__ parent,
    const int32_t* __restrict__ q_row, int n_dec, const int32_t* __restrict__ row_runs, int T,
    __nv_bfloat16* __restrict__ o, int Hkv, float scale_log2, int* __restrict__ err) {
    constexpr int E = D / 32;
    constexpr int kSlices = slices<D, G>();
    const int i = blockIdx.x, g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hq = Hkv * G;
    __shared__ int32_t dsc[8 + 1 + kMaxChain];   // the anchor's 4 runs, chain length, chain rows
    __shared__ int ok;
    __shared__ float part_m[kSlices][G], part_l[kSlices][G];
    __shared__ float part_acc[kSlices][G][D];
    if (threadIdx.x == 0) {
        int good = 1, n = 0;
        int32_t walk[kMaxChain];
        const int r = q_row[i];
        if (r < 0 || r >= n_dec) good = 0;
        for (int c = r; good && c >= 0;) {
            if (n == kMaxChain) { good = 0; break; }
            walk[n++] = c;
            const int p = parent[c];
            if (p >= c) good = 0;
            c = p;
        }
        int a = good ? anchor[walk[n - 1]] : -1;
        for (int j = 0; good && j < n; ++j)
            if (anchor[walk[j]] != a) good = 0;
        if (good && (a < 0 || a >= T)) good = 0;
        if (good) {
            for (int j = 0; j < 8; ++j) dsc[j] = row_runs[8 * (size_t)a + j];
            if (dsc[0] < 0) good = 0;
        }
        dsc[8] = good ? n : 0;
        for (int j = 0; good && j < n; ++j) dsc[9 + j] = walk[n - 1 - j];   // first decoded token first
        if (!good) {
            for (int j = 0; j < 8; ++j) dsc[j] = 0;
            atomicExch(err, dev::kErrCheck);
        }
        ok = good;
    }
    __syncthreads();
    // the group's queries in shared memory (fp32), read back as 16-byte pieces by the score lanes
    __shared__ __align__(16) float qs[G][D];
    for (int x = threadIdx.x; x < G * D; x += blockDim.x)
        qs[x / D][x % D] = __bfloat162float(q[((size_t)i * Hq + g * G) * D + x]);
    __syncthreads();
    float acc[G][E], m[G], l[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        m[hh] = -INFINITY;
        l[hh] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[hh][e] = 0.f;
    }
    // keys four at a time.  Scores: lane group lg = lane / 8 takes key lg, each lane 8 of every
    // 64 columns (one 128-byte line per group and load), summed over the group's 8 lanes; then
    // per head one max and one rescale for the four (scores in log2 units).  Values: lanes over
    // the head dimension, every key's row loaded before the scores are used.
    constexpr int kB = 4;
    const int lg = lane >> 3, ls = lane & 7;
    auto batch = [&](auto rows, int nb) {
        float vx[kB][E];
#pragma unroll
        for (int b = 0; b < kB; ++b)
            if (b < nb) load_row<D>(rows(b).second + lane * E, vx[b]);
        float pd[G];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) pd[hh] = 0.f;
        if (lg < nb) {
            const __nv_bfloat16* kr = rows(lg).first;
            uint4 kp[D / 64];
#pragma unroll
            for (int c = 0; c < D / 64; ++c) kp[c] = *reinterpret_cast<const uint4*>(kr + 64 * c + 8 * ls);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&kp[c]);
                float kx[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 f = __bfloat1622float2(b2[j]);
                    kx[2 * j] = f.x;
                    kx[2 * j + 1] = f.y;
                }
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const float4 q0 = *reinterpret_cast<const float4*>(&qs[hh][64 * c + 8 * ls]);
                    const float4 q1 = *reinterpret_cast<const float4*>(&qs[hh][64 * c + 8 * ls + 4]);
                    float t = pd[hh];
                    t = fmaf(q0.x, kx[0], t);
                    t = fmaf(q0.y, kx[1], t);
                    t = fmaf(q0.z, kx[2], t);
                    t = fmaf(q0.w, kx[3], t);
                    t = fmaf(q1.x, kx[4], t);
                    t = fmaf(q1.y, kx[5], t);
                    t = fmaf(q1.z, kx[6], t);
                    t = fmaf(q1.w, kx[7], t);
                    pd[hh] = t;
                }
            }
        }
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
#pragma unroll
            for (int off = 4; off > 0; off >>= 1) pd[hh] += __shfl_xor_sync(0xffffffffu, pd[hh], off);
            float s[kB];
            float mb = m[hh];
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                const float t = __shfl_sync(0xffffffffu, pd[hh], 8 * b);
                s[b] = b < nb ? t * scale_log2 : -INFINITY;
                mb = fmaxf(mb, s[b]);
            }
            const float corr = dev::fast_exp2(m[hh] - mb);
            l[hh] *= corr;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[hh][e] *= corr;
#pragma unroll
            for (int b = 0; b < kB; ++b)
                if (b < nb) {   // keys in order within the four
                    const float p = dev::fast_exp2(s[b] - mb);
                    l[hh] += p;
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[hh][e] = fmaf(p, vx[b][e], acc[hh][e]);
                }
            m[hh] = mb;
        }
    };
    using Rows = std::pair<const __nv_bfloat16*, const __nv_bfloat16*>;
    // this warp's slice [k0, k1) of the row's keys: the anchor's runs farthest first, then the chain
    int total = dsc[8];
    for (int run = 0; run < 4; ++run) total += dsc[2 * run + 1] - dsc[2 * run];
    const int per = (total + kSlices - 1) / kSlices;
    const int k0 = min(total, warp * per), k1 = min(total, k0 + per);
    int off = 0;
    for (int run = 3; run >= 0; --run) {
        const int lo = dsc[2 * run], len = dsc[2 * run + 1] - lo;
        const int a = max(k0, off), b = min(k1, off + len);
        for (int x = a; x < b; x += kB)
            batch([&](int j) {
                const size_t ro = ((size_t)(lo + x - off + j) * Hkv + g) * D;
                return Rows(k_pass + ro, v_pass + ro);
            }, min(kB, b - x));
        off += len;
    }
    {
        const int a = max(k0, off), b = min(k1, off + dsc[8]);
        for (int x = a; x < b; x += kB)
            batch([&](int j) {
                const size_t ro = ((size_t)dsc[9 + x - off + j] * Hkv + g) * D;
                return Rows(k_dec + ro, v_dec + ro);
            }, min(kB, b - x));
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        if (lane == 0) {
            part_m[warp][hh] = m[hh];
            part_l[warp][hh] = l[hh];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) part_acc[warp][hh][lane * E + e] = acc[hh][e];
    }
    __syncthreads();
    // warp hh < G merges head hh's slices in slice order
    if (warp >= G) return;
    const int hh = warp;
    float M = -INFINITY;
    for (int t = 0; t < kSlices; ++t) M = fmaxf(M, part_m[t][hh]);
    float L = 0.f, out[E];
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = 0.f;
    for (int t = 0; t < kSlices; ++t) {
        const float c = part_m[t][hh] == -INFINITY ? 0.f : dev::fast_exp2(part_m[t][hh] - M);
        L += part_l[t][hh] * c;
#pragma unroll
        for (int e = 0; e < E; ++e) out[e] = fmaf(part_acc[t][hh][lane * E + e], c, out[e]);
    }
    const float inv = ok && L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat16* dst = o + ((size_t)i * Hq + g * G + hh) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2)
        *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(out[e] * inv, out[e + 1] * inv);
}

}  // namespace
}  // namespace spinf

using namespace spinf;

extern "C" spinf_status spinf_decode_attention(const spinf_plan* plan, int32_t pass, const void* q, const void* k_pass,
                                               const void* v_pass, const void* k_dec, const void* v_dec,
                                               int32_t n_dec, const int32_t* anchor, const int32_t* parent,
                                               const int32_t* q_row, int32_t n_q, void* o, int32_t n_q_heads,
                                               int32_t n_kv_heads, int32_t d_head, float scale, spinf_stream stream) {
    spinf_status st = ensure_device_ready(plan, pass);
    if (st) return st;
    if (n_q < 0 || n_dec < 0) return fail(SPINF_E_INVALID, "negative row counts");
    if (n_q == 0) return SPINF_OK;
    if (!q || !k_pass || !v_pass || !k_dec || !v_dec || !o || !anchor || !parent || !q_row)
        return fail(SPINF_E_INVALID, "NULL argument");
    if (d_head != 64 && d_head != 128 && d_head != 256) return fail(SPINF_E_UNSUPPORTED, "d_head must be 64, 128 or 256");
    if (n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads)
        return fail(SPINF_E_UNSUPPORTED, "query heads must be a multiple of kv heads");
    if (n_kv_heads > 65535) return fail(SPINF_E_UNSUPPORTED, "too many kv heads");
    for (const void* p : {q, k_pass, v_pass, k_dec, v_dec, (const void*)o})
        if (reinterpret_cast<uintptr_t>(p) & 15) return fail(SPINF_E_INVALID, "tensor not 16-byte aligned");
    const Pass& P = plan->passes[pass];
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float sc = scale > 0.f ? scale : 1.f / std::sqrt(static_cast<float>(d_head));
    const int G = n_q_heads / n_kv_heads;
    const dim3 grid(n_q, n_kv_heads);
    const float sl2 = sc * 1.4426950408889634f;
    auto go = [&](auto kernel, int slices_) {
        kernel<<<grid, dim3(32 * slices_), 0, s>>>(static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k_pass),
                                      static_cast<const __nv_bfloat16*>(v_pass), static_cast<const __nv_bfloat16*>(k_dec),
                                      static_cast<const __nv_bfloat16*>(v_dec), anchor, parent, q_row, n_dec,
                                      P.dev.row_runs, P.T, static_cast<__nv_bfloat16*>(o), n_kv_heads, sl2, plan->d_err);
    };
    auto by_d = [&](auto g_c) {
        constexpr int GG = decltype(g_c)::value;
        if (d_head == 64) go(decode_attention_kernel<64, GG>, slices<64, GG>());
        else if (d_head == 128) go(decode_attention_kernel<128, GG>, slices<128, GG>());
        else go(decode_attention_kernel<256, GG>, slices<256, GG>());
    };
    switch (G) {
        case 1: by_d(std::integral_constant<int, 1>{}); break;
        case 2: by_d(std::integral_constant<int, 2>{}); break;
        case 4: by_d(std::integral_constant<int, 4>{}); break;
        case 5: by_d(std::integral_constant<int, 5>{}); break;
        case 8: by_d(std::integral_constant<int, 8>{}); break;
        default: return fail(SPINF_E_UNSUPPORTED, "query heads per kv head must be 1, 2, 4, 5 or 8");
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return SPINF_OK;
}
