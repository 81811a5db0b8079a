// Runtime glue of the C ABI: descriptor upload, the device error word, TMA
// tensor-map encoding, plan teardown and the result fingerprint.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "internal.h"
#include "ptx.cuh"
#include "runtime.h"

namespace spinf {

spinf_status cuda_fail(cudaError_t e, const char* what) {
    return fail(SPINF_E_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

spinf_status make_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swizzle) {
    auto fn = encode_fn();
    if (!fn) return fail(SPINF_E_CUDA, "cuTensorMapEncodeTiled is not available");
    cuuint64_t d[5], s[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) s[i] = strides_bytes[i];
    }
    CUresult r = fn(map, dtype, rank, const_cast<void*>(base), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(SPINF_E_INVALID, "tensor map encoding failed (alignment or sizes)");
    return SPINF_OK;
}

spinf_status ensure_device_ready(const spinf_plan* plan, int32_t pass) {
    if (!plan) return fail(SPINF_E_INVALID, "plan is NULL");
    if (pass < 0 || pass >= (int32_t)plan->passes.size()) return fail(SPINF_E_INVALID, "bad pass index");
    if (!plan->passes[pass].dev.block || !plan->d_err) return fail(SPINF_E_INVALID, "pass not uploaded");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != plan->device) return fail(SPINF_E_INVALID, "pass uploaded to another device");
    return SPINF_OK;
}

spinf_status upload_window(WindowSchedule& w, cudaStream_t stream) {
    if (w.block || w.in_pass_block) return SPINF_OK;
    const std::vector<int32_t>* arrays[3] = {&w.qt_work, &w.tile_kv, &w.tile_len};
    int32_t** dst[3] = {&w.d_qt_work, &w.d_tile_kv, &w.d_tile_len};
    size_t off[3], total = 0;
    for (int i = 0; i < 3; ++i) {
        off[i] = total;
        total += (arrays[i]->size() * sizeof(int32_t) + 255) / 256 * 256;
    }
    void* block = nullptr;
    cudaError_t e = cudaMalloc(&block, total > 0 ? total : 256);
    if (e != cudaSuccess) return fail(SPINF_E_NOMEM, "device allocation of a window schedule failed");
    w.staging.assign(total, 0);
    for (int i = 0; i < 3; ++i) {
        if (!arrays[i]->empty()) std::memcpy(w.staging.data() + off[i], arrays[i]->data(), arrays[i]->size() * 4);
        *dst[i] = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(block) + off[i]);
    }
    if (total && (e = cudaMemcpyAsync(block, w.staging.data(), total, cudaMemcpyHostToDevice, stream)) != cudaSuccess) {
        cudaFree(block);
        return cuda_fail(e, "window schedule upload");
    }
    w.block = block;
    return SPINF_OK;
}

spinf_status set_smem_limit(const void* kernel, int bytes, const char* what) {
    static std::mutex mu;
    static std::vector<std::pair<int, const void*>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(mu);
    for (const auto& d : done)
        if (d.first == dev && d.second == kernel) return SPINF_OK;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return cuda_fail(e, what);
    done.emplace_back(dev, kernel);
    return SPINF_OK;
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

}  // namespace spinf

using namespace spinf;

namespace {

// The descriptor arrays of one pass, in upload order, with their device pointers.  The
// pass's 64-key schedule (what d_head 256 attention walks without a window) travels in the
// same block, so that an attention call allocates and uploads nothing.
struct DescriptorSet {
    const std::vector<int32_t>* arrays[21];
    int32_t** dst[21];
    int n = 21;
    size_t off[21];
    size_t total = 0;
    WindowSchedule* w64[2] = {nullptr, nullptr};
};

DescriptorSet descriptor_set(const spinf_plan* plan, Pass& P) {
    std::lock_guard<std::mutex> lock(const_cast<spinf_plan*>(plan)->cache_mu);   // the plan's schedule cache
    WindowSchedule& w = tile_schedule(P, 0, 64);          // 128-row Q tiles (one query head per CTA)
    WindowSchedule& w2 = tile_schedule(P, 0, 64, 64);     // 64-row Q tiles (two stacked query heads)
    DescriptorSet d{{&P.end, &P.pos, &P.tile_ptr, &P.tile_kv, &P.tile_len, &P.slot_row, &P.gather_m, &P.gather_tok,
                     &P.row_gptr, &P.row_glist, &P.qt_work, &P.row_runs, &P.row_x, &P.x_m, &P.x_set, &w.qt_work,
                     &w.tile_kv, &w.tile_len, &w2.qt_work, &w2.tile_kv, &w2.tile_len},
                    {&P.dev.end, &P.dev.pos, &P.dev.tile_ptr, &P.dev.tile_kv, &P.dev.tile_len, &P.dev.slot_row,
                     &P.dev.gather_m, &P.dev.gather_tok, &P.dev.row_gptr, &P.dev.row_glist, &P.dev.qt_work,
                     &P.dev.row_runs, &P.dev.row_x, &P.dev.x_m, &P.dev.x_set, &w.d_qt_work, &w.d_tile_kv,
                     &w.d_tile_len, &w2.d_qt_work, &w2.d_tile_kv, &w2.d_tile_len}};
    // a schedule already uploaded on its own keeps its own copy
    d.w64[0] = w.block ? nullptr : &w;
    d.w64[1] = w2.block ? nullptr : &w2;
    for (int i = 0; i < d.n; ++i) {
        d.off[i] = d.total;
        d.total += (d.arrays[i]->size() * sizeof(int32_t) + 255) / 256 * 256;
    }
    return d;
}

// Points the pass's device views into `block` and enqueues the one copy, from a
// staging buffer the plan keeps (so the copy may still be in flight on return), or from
// the caller's page-locked `stage` when one is given.
spinf_status copy_descriptors(Pass& P, const DescriptorSet& d, void* block, cudaStream_t s,
                              unsigned char* stage = nullptr) {
    unsigned char* host = stage;
    if (!host) {
        P.staging.assign(d.total, 0);
        host = P.staging.data();
    } else {
        std::memset(host, 0, d.total);
    }
    for (int i = 0; i < d.n; ++i) {
        if (!d.arrays[i]->empty()) std::memcpy(host + d.off[i], d.arrays[i]->data(), d.arrays[i]->size() * 4);
        *d.dst[i] = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(block) + d.off[i]);
    }
    if (d.total) {
        cudaError_t e = cudaMemcpyAsync(block, host, d.total, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "descriptor upload");
    }
    for (WindowSchedule* w : d.w64)
        if (w) w->in_pass_block = true;
    return SPINF_OK;
}

spinf_status check_device(spinf_plan* plan, int32_t pass, int* dev) {
    if (!plan) return fail(SPINF_E_INVALID, "plan is NULL");
    if (pass < 0 || pass >= (int32_t)plan->passes.size()) return fail(SPINF_E_INVALID, "bad pass index");
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (plan->device >= 0 && plan->device != *dev) return fail(SPINF_E_INVALID, "plan belongs to another device");
    return SPINF_OK;
}

}  // namespace

extern "C" spinf_status spinf_plan_upload(spinf_plan* plan, int32_t pass, spinf_stream stream) {
    int dev = -1;
    spinf_status st = check_device(plan, pass, &dev);
    if (st) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (!plan->d_err) {
        e = cudaMalloc(&plan->d_err, sizeof(int32_t));
        if (e != cudaSuccess) return fail(SPINF_E_NOMEM, "device allocation of the error word failed");
        plan->err_owned = true;
        e = cudaMemsetAsync(plan->d_err, 0, sizeof(int32_t), s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
        plan->device = dev;
    }
    Pass& P = plan->passes[pass];
    if (P.dev.block) return SPINF_OK;
    const DescriptorSet d = descriptor_set(plan, P);
    void* block = nullptr;
    e = cudaMalloc(&block, d.total > 0 ? d.total : 256);
    if (e != cudaSuccess) return fail(SPINF_E_NOMEM, "device allocation of pass descriptors failed");
    if ((st = copy_descriptors(P, d, block, s))) {
        cudaFree(block);
        return st;
    }
    P.dev.block = block;
    P.dev.owned = true;
    return SPINF_OK;
}

extern "C" size_t spinf_plan_descriptor_bytes(const spinf_plan* plan, int32_t pass) {
    if (!plan || pass < 0 || pass >= (int32_t)plan->passes.size()) return 0;
    return descriptor_set(plan, const_cast<Pass&>(plan->passes[pass])).total + 256;   // + the error word
}

namespace {

spinf_status upload_into(spinf_plan* plan, int32_t pass, void* buffer, size_t bytes, unsigned char* stage,
                         size_t stage_bytes, spinf_stream stream) {
    if (!plan) return fail(SPINF_E_INVALID, "plan is NULL");
    if (pass < 0 || pass >= (int32_t)plan->passes.size()) return fail(SPINF_E_INVALID, "bad pass index");
    if (!buffer || (reinterpret_cast<uintptr_t>(buffer) & 255))
        return fail(SPINF_E_INVALID, "descriptor buffer is NULL or not 256-byte aligned");
    Pass& P = plan->passes[pass];
    if (P.dev.block) return fail(SPINF_E_INVALID, "pass already uploaded");
    const DescriptorSet d = descriptor_set(plan, P);
    if (bytes < d.total + 256) return fail(SPINF_E_INVALID, "descriptor buffer too small");
    if (stage && stage_bytes < d.total) return fail(SPINF_E_INVALID, "staging buffer too small");
    int dev = -1;
    spinf_status st = check_device(plan, pass, &dev);
    if (st) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!plan->d_err) {   // the error word sits after this pass's descriptors
        plan->d_err = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(buffer) + d.total);
        plan->err_owned = false;
        cudaError_t e = cudaMemsetAsync(plan->d_err, 0, sizeof(int32_t), s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
        plan->device = dev;
    }
    if ((st = copy_descriptors(P, d, buffer, s, stage))) return st;
    P.dev.block = buffer;
    P.dev.owned = false;
    return SPINF_OK;
}

}  // namespace

extern "C" spinf_status spinf_plan_upload_to(spinf_plan* plan, int32_t pass, void* buffer, size_t bytes,
                                             spinf_stream stream) {
    return upload_into(plan, pass, buffer, bytes, nullptr, 0, stream);
}

// A copy from pageable memory returns to the host only once the driver has staged it, and
// the staging waits behind the transfers already queued on the copy engine: a caller that
// overlaps the next request's activation copies with this one's kernels would stall there.
// From page-locked memory the copy is enqueued and the call returns at once.
extern "C" spinf_status spinf_plan_upload_pinned(spinf_plan* plan, int32_t pass, void* buffer, size_t bytes,
                                                 void* staging, size_t staging_bytes, spinf_stream stream) {
    if (!staging) return fail(SPINF_E_INVALID, "staging buffer is NULL");
    cudaPointerAttributes a{};
    cudaError_t e = cudaPointerGetAttributes(&a, staging);
    if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes(staging)");
    if (a.type != cudaMemoryTypeHost) return fail(SPINF_E_INVALID, "staging buffer is not page-locked host memory");
    return upload_into(plan, pass, buffer, bytes, static_cast<unsigned char*>(staging), staging_bytes, stream);
}

extern "C" spinf_status spinf_device_status(const spinf_plan* plan, spinf_stream stream) {
    if (!plan) return fail(SPINF_E_INVALID, "plan is NULL");
    if (!plan->d_err) return SPINF_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, plan->d_err, sizeof word, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "device status");
    if (word == 0) return SPINF_OK;
    e = cudaMemsetAsync(plan->d_err, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "device status reset");
    if (word == SPINF_E_DEVICE_TIMEOUT) return fail(SPINF_E_DEVICE_TIMEOUT, "a device wait timed out");
    return fail(SPINF_E_DEVICE_CHECK, "a device-side check failed");
}

namespace spinf {

// One thread waits, with the kernels' bounded wait, on a barrier nothing arrives on.
__global__ void selftest_wait_kernel(int* err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    dev::mbar_init(&bar, 1);
    dev::fence_mbar_init();
    dev::mbar_wait_for(&bar, 0, err, limit_ns);
}

}  // namespace spinf

extern "C" spinf_status spinf_device_selftest(const spinf_plan* plan, int32_t wait_ms, spinf_stream stream) {
    if (!plan || !plan->d_err) return fail(SPINF_E_INVALID, "plan has no device error word (upload a pass first)");
    if (wait_ms < 1 || wait_ms > 10000) return fail(SPINF_E_INVALID, "wait_ms must be in [1, 10000]");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    selftest_wait_kernel<<<1, 32, 0, s>>>(plan->d_err, static_cast<unsigned long long>(wait_ms) * 1000000ull);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
    return SPINF_OK;
}

extern "C" void spinf_plan_free(spinf_plan* plan) {
    if (!plan) return;
    for (Pass& P : plan->passes) {
        if (P.dev.block && P.dev.owned) cudaFree(P.dev.block);
        for (auto& w : P.windows)
            if (w->block) cudaFree(w->block);
        for (auto& r : P.ropes)
            if (r->dev) cudaFree(r->dev);
    }
    if (plan->d_err && plan->err_owned) cudaFree(plan->d_err);
    delete plan;
}

extern "C" const char* spinf_fingerprint(void) {
    return "spinf-gb300 k1=branch_attention/tcgen05 q128xkv128 (kv64 at d256; 2 heads x q64 when Hq=2Hkv) "
           "input-anchored fp32-acc bf16-p tma-store;"
           " k2=score/tcgen05 m128xv256xk64 fp32-acc lse-chunk256 fixed-order, multi-pass sweep in row blocks;"
           " fp8=e4m3 row-absmax/448 rne-sat;"
           " lin=tcgen05 m128xn256 fixed-order, rope fp64-table fp32-rotate, fp8 static scales; sm_103a";
}
