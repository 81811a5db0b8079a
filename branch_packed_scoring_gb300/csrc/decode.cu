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
//   decode_attention_kernel<D, G>  one CTA per (block of consecutive decode rows,
//                               kv head); the rows that share an anchor (a beam's
//                               rows, laid out next to each other) read each key
//                               row of their anchor's path once, by bulk copies
//                               into per-warp double buffers.  Keys are visited in
//                               a fixed order (the anchor's path in ascending rows,
//                               then the chain from its first token) and merged
//                               in a fixed order: a row's output does not depend
//                               on the other rows of the step.
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

// One CTA per (block of consecutive decode rows, kv head).  The block's rows and the G query
// heads of the kv head fill up to kNS query-vector slots (n = row * G + head).  Lane r of warp 0
// walks row r's chain and checks every index against its array; a row that fails is written as
// zeros and raises the plan's error word (SPINF_E_DEVICE_CHECK).  Consecutive good rows with one
// anchor form a sub-group: they share their anchor's path, and each key row of it is read once for
// all their slots.
//
// Keys travel in tiles of kKT rows.  Warp w takes the path tiles w, w + kWarps, ... of every
// sub-group, then the chain tiles of rows w, w + kWarps, ...; each warp copies its own tiles (K
// rows, then V rows) with untiled bulk copies into a double buffer, one tile ahead of the one it
// computes.  Scores: lanes over the head dimension, four keys x kNS slots of partial dot products
// reduced across the warp by halving exchanges, so that lane l ends with the score of key l / 8
// and slot l % 8.  Softmax state (running max and sum) is kept per slot, the accumulator with
// lanes over the head dimension.  A slot whose row is not in the tile's sub-group (or chain) is
// masked: its state does not move.  Each warp keeps its path partial and its rows' chain
// partials; they are merged per slot in a fixed order (path slices by warp, then the chain).
// So a row's output depends on its anchor's path, its chain and the head grouping only, never on
// the other rows of the call or where it sits among them.
constexpr int kWarps = 4;    // warps per CTA
constexpr int kKT = 8;       // keys per tile
constexpr int kNS = 8;       // query-vector slots per CTA

// decode rows per CTA: as many whole head groups as fit the slots
template <int G>
__host__ __device__ constexpr int rows_per_cta() { return G >= kNS ? 1 : kNS / G; }

template <int D>
struct DecodeSmem {
    static constexpr int kRowB = D * 2;                              // one key or value row (bf16)
    static constexpr int kTile = 2 * kKT * kRowB;                    // a tile: K rows, then V rows
    static constexpr int kSlots = kWarps + 1;                        // a path partial per warp, then chains
    static constexpr int kPartAcc = kWarps * 2 * kTile;              // float [kSlots][kNS][D]
    static constexpr int kPartM = kPartAcc + kSlots * kNS * D * 4;   // float [kSlots][kNS]
    static constexpr int kPartL = kPartM + kSlots * kNS * 4;         // float [kSlots][kNS]
    static constexpr int kPw = kKT * kNS + kNS;                      // per warp: p [kKT][kNS], corr [kNS]
    static constexpr int kP = kPartL + kSlots * kNS * 4;
    static constexpr int kBars = (kP + kWarps * kPw * 4 + 7) / 8 * 8;   // uint64 [kWarps][2]
    static constexpr int kBytes = kBars + kWarps * 2 * 8;
};

struct DecodeRow {
    int ok, anchor, nc, plen;     // checks passed, anchor row, chain length, root-path length
    int runs[8];                  // the anchor's root path: four runs [lo, hi), farthest first
    int chain[kMaxChain];         // decode rows of the chain, first token first
};

// A tile of one warp: kind 0 = path tile t of sub-group a, 1 = chain tile t of row a, 2 = none.
struct Tile {
    int kind, a, t;
};

template <int D, int G>
__global__ void __launch_bounds__(32 * kWarps, 2) decode_attention_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_pass,
    const __nv_bfloat16* __restrict__ v_pass, const __nv_bfloat16* __restrict__ k_dec,
    const __nv_bfloat16* __restrict__ v_dec, const int32_t* __restrict__ anchor, const int32_t* __restrict__ parent,
    const int32_t* __restrict__ q_row, int n_dec, int n_q, const int32_t* __restrict__ row_runs, int T,
    __nv_bfloat16* __restrict__ o, int Hkv, float scale_log2, int* __restrict__ err) {
    using L = DecodeSmem<D>;
    constexpr int E = D / 32;
    constexpr int R = rows_per_cta<G>();
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ DecodeRow rows[R];
    __shared__ int sg_lo[R], sg_hi[R], sg_plen[R], n_sg;
    float* part_acc = reinterpret_cast<float*>(dsm + L::kPartAcc);
    float* part_m = reinterpret_cast<float*>(dsm + L::kPartM);
    float* part_l = reinterpret_cast<float*>(dsm + L::kPartL);
    uint64_t* bars = reinterpret_cast<uint64_t*>(dsm + L::kBars);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.y, i0 = blockIdx.x * R, Hq = Hkv * G;
    float* pw = reinterpret_cast<float*>(dsm + L::kP) + warp * L::kPw;

    if (warp == 0 && lane < R) {
        DecodeRow& rw = rows[lane];
        const int i = i0 + lane;
        int good = i < n_q, n = 0, a = -1;
        if (good) {
            int c = q_row[i];
            if (c < 0 || c >= n_dec) good = 0;
            while (good && c >= 0) {
                if (n == kMaxChain) {
                    good = 0;
                    break;
                }
                rw.chain[n++] = c;
                const int p = parent[c];
                if (p >= c) good = 0;
                c = p;
            }
        }
        if (good) {
            a = anchor[rw.chain[n - 1]];
            for (int j = 0; good && j < n; ++j)
                if (anchor[rw.chain[j]] != a) good = 0;
            if (a < 0 || a >= T) good = 0;
        }
        int plen = 0;
        if (good) {
            for (int j = 0; j < 8; ++j) rw.runs[j] = row_runs[8 * (size_t)a + j];
            if (rw.runs[0] < 0) good = 0;
            for (int run = 0; run < 4; ++run) plen += rw.runs[2 * run + 1] - rw.runs[2 * run];
        }
        if (good)
            for (int j = 0; j < n / 2; ++j) {
                const int t = rw.chain[j];
                rw.chain[j] = rw.chain[n - 1 - j];
                rw.chain[n - 1 - j] = t;
            }
        if (!good && i < n_q) atomicExch(err, dev::kErrCheck);
        rw.ok = good;
        rw.anchor = a;
        rw.nc = good ? n : 0;
        rw.plen = good ? plen : 0;
    }
    if (lane == 0) {
        dev::mbar_init(&bars[2 * warp], 1);
        dev::mbar_init(&bars[2 * warp + 1], 1);
        dev::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int ns = 0;
        for (int r = 0; r < R;) {
            if (!rows[r].ok) {
                ++r;
                continue;
            }
            int b = r + 1;
            while (b < R && rows[b].ok && rows[b].anchor == rows[r].anchor) ++b;
            sg_lo[ns] = r;
            sg_hi[ns] = b;
            sg_plen[ns] = rows[r].plen;
            ++ns;
            r = b;
        }
        n_sg = ns;
    }
    // the slots' queries, lanes over the head dimension (zero for slots without a good row)
    float qr[kNS][E];
#pragma unroll
    for (int n = 0; n < kNS; ++n) {
        const int r = n / G, i = i0 + r;
        if (r < R && i < n_q && rows[r].ok) {
            load_row<D>(q + ((size_t)i * Hq + g * G + n % G) * D + lane * E, qr[n]);
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) qr[n][e] = 0.f;
        }
    }
    __syncthreads();

    auto settle = [&](Tile& it) {   // move on to the first tile that exists at or after `it`
        for (;;) {
            if (it.kind == 0) {
                if (it.a >= n_sg) {
                    it = Tile{1, warp, 0};
                    continue;
                }
                if (it.t * kKT < sg_plen[it.a]) return;
                it = Tile{0, it.a + 1, warp};
                continue;
            }
            if (it.kind == 1) {
                if (it.a >= R) {
                    it.kind = 2;
                    return;
                }
                if (rows[it.a].ok && it.t * kKT < rows[it.a].nc) return;
                it = Tile{1, it.a + kWarps, 0};
                continue;
            }
            return;
        }
    };
    auto advance = [&](Tile& it) {
        it.t += it.kind == 0 ? kWarps : 1;
        settle(it);
    };
    auto n_valid = [&](const Tile& it) {
        const int total = it.kind == 0 ? sg_plen[it.a] : rows[it.a].nc;
        return min(kKT, total - it.t * kKT);
    };
    // source rows of key j of a tile
    auto key_rows = [&](const Tile& it, int j, const __nv_bfloat16*& kr, const __nv_bfloat16*& vr) {
        const int x = it.t * kKT + j;
        if (it.kind == 0) {
            const int* runs = rows[sg_lo[it.a]].runs;
            int off = 0, row = 0;
            for (int run = 3; run >= 0; --run) {
                const int lo = runs[2 * run], len = runs[2 * run + 1] - lo;
                if (x < off + len) {
                    row = lo + x - off;
                    break;
                }
                off += len;
            }
            const size_t ro = ((size_t)row * Hkv + g) * D;
            kr = k_pass + ro;
            vr = v_pass + ro;
        } else {
            const size_t ro = ((size_t)rows[it.a].chain[x] * Hkv + g) * D;
            kr = k_dec + ro;
            vr = v_dec + ro;
        }
    };
    auto buffer = [&](int b) { return dsm + (warp * 2 + b) * L::kTile; };
    auto issue = [&](const Tile& it, int b) {   // lanes 0-7 copy K rows, 8-15 V rows
        const int nv = n_valid(it);
        __syncwarp();
        dev::fence_proxy_async_smem();   // this warp's reads of the buffer come before the copies' writes
        if (lane == 0) dev::mbar_arrive_expect_tx(&bars[2 * warp + b], nv * 2 * L::kRowB);
        __syncwarp();
        if (lane < 2 * kKT && (lane & (kKT - 1)) < nv) {
            const int j = lane & (kKT - 1);
            const __nv_bfloat16 *kr, *vr;
            key_rows(it, j, kr, vr);
            dev::bulk_g2s(buffer(b) + (lane >= kKT ? kKT * L::kRowB : 0) + j * L::kRowB, lane >= kKT ? vr : kr,
                     L::kRowB, &bars[2 * warp + b]);
        }
    };

    // softmax state: m, l of slot lane % 8 (the same in the four lanes of a slot), acc per slot
    float m = -INFINITY, l = 0.f, acc[kNS][E];
#pragma unroll
    for (int n = 0; n < kNS; ++n)
#pragma unroll
        for (int e = 0; e < E; ++e) acc[n][e] = 0.f;
    auto reset = [&]() {
        m = -INFINITY;
        l = 0.f;
#pragma unroll
        for (int n = 0; n < kNS; ++n)
#pragma unroll
            for (int e = 0; e < E; ++e) acc[n][e] = 0.f;
    };
    auto store = [&](int slot, int r0, int r1) {   // the partial of the slots of rows [r0, r1)
#pragma unroll
        for (int n = 0; n < kNS; ++n)
            if (n / G >= r0 && n / G < r1)
#pragma unroll
                for (int e = 0; e < E; ++e) part_acc[(slot * kNS + n) * D + lane * E + e] = acc[n][e];
        const int n = lane & (kNS - 1);
        if (lane < kNS && n / G >= r0 && n / G < r1) {
            part_m[slot * kNS + n] = m;
            part_l[slot * kNS + n] = l;
        }
    };

    Tile cur{0, 0, warp};
    settle(cur);
    Tile pre = cur;
    int issued = 0;
    for (int b = 0; b < 2 && pre.kind < 2; ++b, ++issued) {
        issue(pre, b);
        advance(pre);
    }
    bool path_stored = false;
    for (int lt = 0; cur.kind < 2; ++lt) {
        if (cur.kind == 1 && !path_stored) {
            store(warp, 0, R);
            reset();
            path_stored = true;
        }
        const int b = lt & 1, nv = n_valid(cur);
        const int r0 = cur.kind == 0 ? sg_lo[cur.a] : cur.a, r1 = cur.kind == 0 ? sg_hi[cur.a] : cur.a + 1;
        dev::mbar_drain(&bars[2 * warp + b], (lt >> 1) & 1, err);
        const __nv_bfloat16* kt = reinterpret_cast<const __nv_bfloat16*>(buffer(b));
        const __nv_bfloat16* vt = kt + kKT * D;
        // scores of keys kk and kk + 4 for slot lane % 8 (stale rows past nv give masked scores)
        float sc[2] = {0.f, 0.f};
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            if (hb == 1 && nv <= 4) break;
            float v[4 * kNS];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                float kx[E];
                load_row<D>(kt + (hb * 4 + kk) * D + lane * E, kx);
#pragma unroll
                for (int n = 0; n < kNS; ++n) {
                    float2 t = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < E; e += 2)
                        t = dev::ffma2(make_float2(qr[n][e], qr[n][e + 1]), make_float2(kx[e], kx[e + 1]), t);
                    v[kk * kNS + n] = t.x + t.y;
                }
            }
            // halving exchanges: after the step with offset o a lane keeps the half of its values
            // whose index bit o matches its lane bit o, added to the partner's copy of that half
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const bool up = lane & o;
#pragma unroll
                for (int x = 0; x < o; ++x) {
                    const float send = up ? v[x] : v[x + o];
                    const float keep = up ? v[x + o] : v[x];
                    v[x] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            sc[hb] = v[0];
        }
        const int kk = lane >> 3, n = lane & (kNS - 1);
        const bool act = n / G >= r0 && n / G < r1;
        const bool va = act && kk < nv, vb = act && kk + 4 < nv;
        const float sa = va ? sc[0] * scale_log2 : -INFINITY;
        const float sb = vb ? sc[1] * scale_log2 : -INFINITY;
        float tm = fmaxf(sa, sb);
        tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
        tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
        const float mn = fmaxf(m, tm);
        const float corr = mn == -INFINITY ? 1.f : dev::fast_exp2(m - mn);
        const float pa = va ? dev::fast_exp2(sa - mn) : 0.f;
        const float pb = vb ? dev::fast_exp2(sb - mn) : 0.f;
        float ps = pa + pb;
        ps += __shfl_xor_sync(0xffffffffu, ps, 8);
        ps += __shfl_xor_sync(0xffffffffu, ps, 16);
        l = l * corr + ps;
        m = mn;
        pw[lane] = pa;              // p of key kk, slot n
        pw[32 + lane] = pb;         // p of key kk + 4, slot n
        if (lane < kNS) pw[kKT * kNS + lane] = corr;
        __syncwarp();
        {
            float cr[kNS];
            *reinterpret_cast<float4*>(cr) = *reinterpret_cast<const float4*>(pw + kKT * kNS);
            *reinterpret_cast<float4*>(cr + 4) = *reinterpret_cast<const float4*>(pw + kKT * kNS + 4);
#pragma unroll
            for (int s = 0; s < kNS; ++s)
#pragma unroll
                for (int e = 0; e < E; e += 2) {
                    const float2 r = dev::fmul2(make_float2(acc[s][e], acc[s][e + 1]), make_float2(cr[s], cr[s]));
                    acc[s][e] = r.x;
                    acc[s][e + 1] = r.y;
                }
        }
        for (int j = 0; j < nv; ++j) {   // keys in order
            float vx[E], pj[kNS];
            load_row<D>(vt + j * D + lane * E, vx);
            *reinterpret_cast<float4*>(pj) = *reinterpret_cast<const float4*>(pw + j * kNS);
            *reinterpret_cast<float4*>(pj + 4) = *reinterpret_cast<const float4*>(pw + j * kNS + 4);
#pragma unroll
            for (int s = 0; s < kNS; ++s)
#pragma unroll
                for (int e = 0; e < E; e += 2) {
                    const float2 r = dev::ffma2(make_float2(pj[s], pj[s]), make_float2(vx[e], vx[e + 1]),
                                                make_float2(acc[s][e], acc[s][e + 1]));
                    acc[s][e] = r.x;
                    acc[s][e + 1] = r.y;
                }
        }
        // the buffer is free again: bring the tile after the next one into it
        if (pre.kind < 2) {
            issue(pre, b);
            advance(pre);
            ++issued;
        }
        advance(cur);
    }
    if (!path_stored) store(warp, 0, R);
    else
        for (int r = warp; r < R; r += kWarps)
            if (rows[r].ok) store(kWarps, r, r + 1);
    // every copy this warp issued has landed (waits that ran out above leave none in flight)
    for (int b = 0; b < 2; ++b) {
        const int last = issued - 1 - ((issued - 1 - b) & 1);   // the last tile issued into buffer b
        if (last >= 0) dev::mbar_drain(&bars[2 * warp + b], (last >> 1) & 1, err);
    }
    __syncthreads();
    // merge per slot in slot order: path slices by warp, then the chain
    for (int n = warp; n < kNS; n += kWarps) {
        const int r = n / G, i = i0 + r;
        if (r >= R || i >= n_q) continue;
        __nv_bfloat16* dst = o + ((size_t)i * Hq + g * G + n % G) * D + lane * E;
        float out[E];
#pragma unroll
        for (int e = 0; e < E; ++e) out[e] = 0.f;
        if (rows[r].ok) {
            float M = -INFINITY;
            for (int s = 0; s < L::kSlots; ++s) M = fmaxf(M, part_m[s * kNS + n]);
            float Ls = 0.f;
            for (int s = 0; s < L::kSlots; ++s) {
                const float pm = part_m[s * kNS + n];
                const float c = pm == -INFINITY ? 0.f : dev::fast_exp2(pm - M);
                Ls += part_l[s * kNS + n] * c;
#pragma unroll
                for (int e = 0; e < E; ++e) out[e] = fmaf(part_acc[(s * kNS + n) * D + lane * E + e], c, out[e]);
            }
            const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) out[e] *= inv;
        }
#pragma unroll
        for (int e = 0; e < E; e += 2)
            *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(out[e], out[e + 1]);
    }
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
    const float sl2 = sc * 1.4426950408889634f;
    auto go = [&](auto d_c, auto g_c) -> spinf_status {
        constexpr int DD = decltype(d_c)::value, GG = decltype(g_c)::value;
        constexpr int R = rows_per_cta<GG>();
        auto kernel = decode_attention_kernel<DD, GG>;
        const int smem = DecodeSmem<DD>::kBytes;
        spinf_status st2 = set_smem_limit(reinterpret_cast<const void*>(kernel), smem, "cudaFuncSetAttribute(decode)");
        if (st2) return st2;
        const dim3 grid((n_q + R - 1) / R, n_kv_heads);
        kernel<<<grid, dim3(32 * kWarps), smem, s>>>(
            static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k_pass),
            static_cast<const __nv_bfloat16*>(v_pass), static_cast<const __nv_bfloat16*>(k_dec),
            static_cast<const __nv_bfloat16*>(v_dec), anchor, parent, q_row, n_dec, n_q, P.dev.row_runs, P.T,
            static_cast<__nv_bfloat16*>(o), n_kv_heads, sl2, plan->d_err);
        return SPINF_OK;
    };
    auto by_d = [&](auto g_c) -> spinf_status {
        if (d_head == 64) return go(std::integral_constant<int, 64>{}, g_c);
        if (d_head == 128) return go(std::integral_constant<int, 128>{}, g_c);
        return go(std::integral_constant<int, 256>{}, g_c);
    };
    switch (G) {
        case 1: st = by_d(std::integral_constant<int, 1>{}); break;
        case 2: st = by_d(std::integral_constant<int, 2>{}); break;
        case 4: st = by_d(std::integral_constant<int, 4>{}); break;
        case 5: st = by_d(std::integral_constant<int, 5>{}); break;
        case 8: st = by_d(std::integral_constant<int, 8>{}); break;
        default: return fail(SPINF_E_UNSUPPORTED, "query heads per kv head must be 1, 2, 4, 5 or 8");
    }
    if (st) return st;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return SPINF_OK;
}
