// pkv_host.cuh -- host-side helpers shared by the libpkv entry points:
// per-device properties, TMA tensor-map encoding and status mapping.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

struct DeviceInfo {
    int device = -1;
    int num_sms = 0;
    size_t max_smem_optin = 0;
};

// Properties of the current device (cached per device).  Returns false if
// the CUDA runtime cannot answer.
bool current_device_info(DeviceInfo *out);

// Encode a 2-D tiled tensor map over `rows` rows of `row_bytes` bytes
// starting at `base`, with a box of box_inner elements x box_rows rows.
// elem_bytes is 1 (uint8) or 2 (fp16).  swizzle_bytes is 64 or 128.
// Returns false if the driver rejects the description.  The last 16 maps
// encoded are kept and handed out again for the same description.
bool encode_tmap_2d(CUtensorMap *map, const void *base, int elem_bytes, uint64_t inner_elems,
                    uint64_t rows, uint32_t box_inner, uint32_t box_rows, int swizzle_bytes);

inline bool aligned(const void *p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

}  // namespace pkv
