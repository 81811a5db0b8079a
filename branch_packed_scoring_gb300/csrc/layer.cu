// The steps around the attention call that complete a packed layer: rotary
// position embedding at tree positions, and the bf16 linear maps of the QKV and
// output projections.
//
// The method ("spinf-serve 0.1.1", PyPI page, "What it does"): every question is
// a branch of the packed pass, and an input's scores are the same alone or
// packed.  A token's position is therefore its depth on its own root path (the
// plan's pos[]), never its row in the pass: a branch token gets the positions its
// unpacked sequence (content, question, option prefix) would give it.
#include <cublasLt.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "internal.h"
#include "runtime.h"

namespace spinf {
namespace {

// One CTA per packed row.  Rotate-half convention: the pairs (x[i], x[i + d/2]),
// i < d/2, turn by pos * theta^(-2i/d).  The angles are formed and reduced in fp64
// (pos reaches the tens of thousands), then the rotation runs in fp32 per head.
__global__ void rope_tree_kernel(__nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ k,
                                 const int32_t* __restrict__ pos, int Hq, int Hkv, int d, double log2_theta) {
    extern __shared__ float cs[];   // [d/2] cos, then [d/2] sin
    const int row = blockIdx.x, half = d / 2;
    const double p = static_cast<double>(__ldg(pos + row));
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        const double inv_freq = exp2(-log2_theta * (2.0 * i) / d);
        double s, c;
        sincos(p * inv_freq, &s, &c);
        cs[i] = static_cast<float>(c);
        cs[half + i] = static_cast<float>(s);
    }
    __syncthreads();
    const int pairs_q = Hq * half, pairs = (Hq + Hkv) * half;
    for (int j = threadIdx.x; j < pairs; j += blockDim.x) {
        const bool is_q = j < pairs_q;
        const int jj = is_q ? j : j - pairs_q;
        const int h = jj / half, i = jj - h * half;
        __nv_bfloat16* base = is_q ? q + (static_cast<size_t>(row) * Hq + h) * d
                                   : k + (static_cast<size_t>(row) * Hkv + h) * d;
        const float x0 = __bfloat162float(base[i]), x1 = __bfloat162float(base[i + half]);
        const float c = cs[i], s = cs[half + i];
        base[i] = __float2bfloat16_rn(x0 * c - x1 * s);
        base[i + half] = __float2bfloat16_rn(x1 * c + x0 * s);
    }
}

struct LtHandle {
    cublasLtHandle_t h = nullptr;
    int device = -1;
};

cublasLtHandle_t lt_handle(int device) {
    static std::mutex mu;
    static LtHandle handles[64];
    std::lock_guard<std::mutex> lock(mu);
    if (device < 0 || device >= 64) return nullptr;
    if (!handles[device].h) {
        if (cublasLtCreate(&handles[device].h) != CUBLAS_STATUS_SUCCESS) handles[device].h = nullptr;
        handles[device].device = device;
    }
    return handles[device].h;
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
    if (!(theta > 1.f)) return fail(SPINF_E_INVALID, "theta must be > 1");
    const Pass& P = plan->passes[pass];
    if (P.T_pad == 0) return SPINF_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    rope_tree_kernel<<<P.T_pad, 256, d_head * sizeof(float), s>>>(static_cast<__nv_bfloat16*>(q),
                                                                  static_cast<__nv_bfloat16*>(k), P.dev.pos,
                                                                  n_q_heads, n_kv_heads, d_head,
                                                                  std::log2(static_cast<double>(theta)));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "rope launch");
    return SPINF_OK;
}

extern "C" spinf_status spinf_linear(const void* x, const void* w, void* y, int64_t rows, int64_t in_features,
                                     int64_t out_features, spinf_stream stream) {
    if (!x || !w || !y) return fail(SPINF_E_INVALID, "NULL tensor");
    if (rows < 0 || in_features <= 0 || out_features <= 0 || in_features % 8 || out_features % 8)
        return fail(SPINF_E_INVALID, "bad sizes (features must be positive multiples of 8)");
    for (const void* p : {x, w, (const void*)y})
        if (reinterpret_cast<uintptr_t>(p) & 15) return fail(SPINF_E_INVALID, "tensor not 16-byte aligned");
    if (rows == 0) return SPINF_OK;
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaGetDevice");
    cublasLtHandle_t h = lt_handle(dev);
    if (!h) return fail(SPINF_E_CUDA, "cublasLtCreate failed");
    // column-major view: Y^T[out, rows] = W[out, in] (row-major, i.e. W^T col-major, transposed) x X^T[in, rows]
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
    spinf_status st = SPINF_OK;
    auto ok = [&](cublasStatus_t r, const char* what) {
        if (r != CUBLAS_STATUS_SUCCESS && st == SPINF_OK) st = fail(SPINF_E_CUDA, std::string("cublasLt: ") + what);
        return r == CUBLAS_STATUS_SUCCESS;
    };
    const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
    if (ok(cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F), "desc") &&
        ok(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof ta), "transa") &&
        ok(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof tb), "transb") &&
        ok(cublasLtMatrixLayoutCreate(&la, CUDA_R_16BF, in_features, out_features, in_features), "layout a") &&
        ok(cublasLtMatrixLayoutCreate(&lb, CUDA_R_16BF, in_features, rows, in_features), "layout b") &&
        ok(cublasLtMatrixLayoutCreate(&lc, CUDA_R_16BF, out_features, rows, out_features), "layout c")) {
        const float alpha = 1.f, beta = 0.f;
        ok(cublasLtMatmul(h, op, &alpha, w, la, x, lb, &beta, y, lc, y, lc, nullptr, nullptr, 0,
                          reinterpret_cast<cudaStream_t>(stream)),
           "matmul");
    }
    if (lc) cublasLtMatrixLayoutDestroy(lc);
    if (lb) cublasLtMatrixLayoutDestroy(lb);
    if (la) cublasLtMatrixLayoutDestroy(la);
    if (op) cublasLtMatmulDescDestroy(op);
    return st;
}
