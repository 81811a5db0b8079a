// Host helpers shared by the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace spinf {

spinf_status cuda_fail(cudaError_t e, const char* what);

// Encode a tiled TMA tensor map.  dims/box are innermost first; strides_bytes
// has rank-1 entries (the stride of dimensions 1..rank-1).
spinf_status make_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swizzle);

// The pass exists, was uploaded, and belongs to the current device.
spinf_status ensure_device_ready(const spinf_plan* plan, int32_t pass);

int sm_count();

// Raise `kernel`'s dynamic shared-memory limit to `bytes` on the current device, once per
// (device, kernel): the attribute belongs to a device context, so a process that drives
// several GPUs sets it on each.  Thread-safe.
spinf_status set_smem_limit(const void* kernel, int bytes, const char* what);

// Device copies of a windowed schedule (allocated and copied on `stream` on first use).
spinf_status upload_window(WindowSchedule& w, cudaStream_t stream);

}  // namespace spinf
