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
#include <vector>

#include "internal.h"
#include "runtime.h"

namespace spinf {
namespace {

constexpr int kMaxChain = 64;                 // decoded tokens per chain (a searched answer is short)
constexpr int kDescInts = 8 + 1 + kMaxChain;  // per query: 4 pass runs, chain length, chain rows

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

template <int D>
__global__ void __launch_bounds__(256) decode_attention_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_pass,
    const __nv_bfloat16* __restrict__ v_pass, const __nv_bfloat16* __restrict__ k_dec,
    const __nv_bfloat16* __restrict__ v_dec, const int32_t* __restrict__ desc, __nv_bfloat16* __restrict__ o, int Hq,
    int Hkv, float scale) {
    constexpr int E = D / 32;
    const int i = blockIdx.x, g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = g * (Hq / Hkv) + warp;
    const int32_t* dsc = desc + (size_t)i * kDescInts;
    float qv[E], acc[E];
    load_row<D>(q + ((size_t)i * Hq + h) * D + lane * E, qv);
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float m = -INFINITY, l = 0.f;
    auto visit = [&](const __nv_bfloat16* kr, const __nv_bfloat16* vr) {
        float kx[E], vx[E];
        load_row<D>(kr + lane * E, kx);
        load_row<D>(vr + lane * E, vx);
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) s = fmaf(qv[e], kx[e], s);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        s *= scale;
        const float mn = fmaxf(m, s);
        const float corr = expf(m - mn), p = expf(s - mn);
        l = l * corr + p;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = acc[e] * corr + p * vx[e];
        m = mn;
    };
    // the anchor's path in the pass: runs stored nearest first, visited farthest first
    for (int run = 3; run >= 0; --run)
        for (int kk = dsc[2 * run]; kk < dsc[2 * run + 1]; ++kk)
            visit(k_pass + ((size_t)kk * Hkv + g) * D, v_pass + ((size_t)kk * Hkv + g) * D);
    const int n_chain = dsc[8];
    for (int c = 0; c < n_chain; ++c) {
        const int r = dsc[9 + c];
        visit(k_dec + ((size_t)r * Hkv + g) * D, v_dec + ((size_t)r * Hkv + g) * D);
    }
    const float inv = 1.f / l;
    __nv_bfloat16* dst = o + ((size_t)i * Hq + h) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2)
        *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
}

}  // namespace
}  // namespace spinf

using namespace spinf;

extern "C" size_t spinf_decode_workspace_bytes(int32_t n_q) {
    return n_q > 0 ? ((size_t)n_q * kDescInts * sizeof(int32_t) + 255) / 256 * 256 : 0;
}

extern "C" spinf_status spinf_decode_attention(const spinf_plan* plan, int32_t pass, const void* q, const void* k_pass,
                                               const void* v_pass, const void* k_dec, const void* v_dec,
                                               int32_t n_dec, const int32_t* anchor, const int32_t* parent,
                                               const int32_t* q_row, int32_t n_q, void* o, int32_t n_q_heads,
                                               int32_t n_kv_heads, int32_t d_head, float scale, void* workspace,
                                               size_t workspace_bytes, spinf_stream stream) {
    spinf_status st = ensure_device_ready(plan, pass);
    if (st) return st;
    if (n_q < 0 || n_dec < 0) return fail(SPINF_E_INVALID, "negative row counts");
    if (n_q == 0) return SPINF_OK;
    if (!q || !k_pass || !v_pass || !k_dec || !v_dec || !o || !anchor || !parent || !q_row || !workspace)
        return fail(SPINF_E_INVALID, "NULL argument");
    if (d_head != 64 && d_head != 128 && d_head != 256) return fail(SPINF_E_UNSUPPORTED, "d_head must be 64, 128 or 256");
    if (n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads || n_q_heads / n_kv_heads > 8)
        return fail(SPINF_E_UNSUPPORTED, "query heads must be 1..8 per kv head");
    for (const void* p : {q, k_pass, v_pass, k_dec, v_dec, (const void*)o})
        if (reinterpret_cast<uintptr_t>(p) & 15) return fail(SPINF_E_INVALID, "tensor not 16-byte aligned");
    if (workspace_bytes < spinf_decode_workspace_bytes(n_q)) return fail(SPINF_E_NOMEM, "workspace too small");
    const Pass& P = plan->passes[pass];
    // per query: the anchor's pass runs and its decode chain, checked here on the host
    std::vector<int32_t> desc((size_t)n_q * kDescInts, 0);
    for (int32_t i = 0; i < n_q; ++i) {
        const int32_t r = q_row[i];
        if (r < 0 || r >= n_dec) return fail(SPINF_E_INVALID, "q_row outside the decode rows");
        int32_t* d = &desc[(size_t)i * kDescInts];
        std::vector<int32_t> ch;
        for (int32_t c = r; c >= 0; c = parent[c]) {
            if (parent[c] >= c) return fail(SPINF_E_INVALID, "a decode row's parent must be an earlier row");
            if ((int)ch.size() == kMaxChain) return fail(SPINF_E_LIMIT, "decode chain longer than 64 tokens");
            ch.push_back(c);
        }
        const int32_t a = anchor[ch.back()];
        for (int32_t c : ch)
            if (anchor[c] != a) return fail(SPINF_E_INVALID, "a decode chain must keep one anchor");
        if (a < 0 || a >= P.T) return fail(SPINF_E_INVALID, "anchor outside the pass");
        const int32_t* runs = &P.row_runs[8 * (size_t)a];
        if (runs[0] < 0) return fail(SPINF_E_UNSUPPORTED, "anchor's root path has more than four runs");
        for (int j = 0; j < 8; ++j) d[j] = runs[j];
        d[8] = (int32_t)ch.size();
        for (size_t c = 0; c < ch.size(); ++c) d[9 + c] = ch[ch.size() - 1 - c];   // first decoded token first
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // pageable source: the call returns once the bytes are staged, so `desc` may go
    cudaError_t e = cudaMemcpyAsync(workspace, desc.data(), desc.size() * sizeof(int32_t), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode descriptor upload");
    const float sc = scale > 0.f ? scale : 1.f / std::sqrt(static_cast<float>(d_head));
    const dim3 grid(n_q, n_kv_heads), block(32 * (n_q_heads / n_kv_heads));
    auto go = [&](auto kernel) {
        kernel<<<grid, block, 0, s>>>(static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k_pass),
                                      static_cast<const __nv_bfloat16*>(v_pass), static_cast<const __nv_bfloat16*>(k_dec),
                                      static_cast<const __nv_bfloat16*>(v_dec), static_cast<const int32_t*>(workspace),
                                      static_cast<__nv_bfloat16*>(o), n_q_heads, n_kv_heads, sc);
    };
    if (d_head == 64) go(decode_attention_kernel<64>);
    else if (d_head == 128) go(decode_attention_kernel<128>);
    else go(decode_attention_kernel<256>);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return SPINF_OK;
}
