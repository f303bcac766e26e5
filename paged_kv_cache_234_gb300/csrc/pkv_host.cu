// pkv_host.cu -- host-side helpers: device properties, TMA tensor maps,
// status strings.
#include <mutex>

#include "pkv_host.cuh"

namespace pkv {

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_info[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Recently encoded tensor maps.  A map depends only on the description it
// was encoded from (base address, geometry, box, swizzle), so a call over
// the same pools reuses it instead of encoding it again on the host.
struct TmapEntry {
    bool valid = false;
    const void *base = nullptr;
    int elem_bytes = 0, swizzle = 0;
    uint64_t inner = 0, rows = 0;
    uint32_t box_inner = 0, box_rows = 0;
    CUtensorMap map;
};
constexpr int kTmapEntries = 16;
TmapEntry g_tmaps[kTmapEntries];
int g_tmap_next = 0;
std::mutex g_tmap_mu;
}  // namespace

bool current_device_info(DeviceInfo *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &d = g_info[dev];
    if (d.device != dev) {
        int sms = 0, optin = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return false;
        if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
            return false;
        d.num_sms = sms;
        d.max_smem_optin = static_cast<size_t>(optin);
        d.device = dev;
    }
    *out = d;
    return true;
}

bool encode_tmap_2d(CUtensorMap *map, const void *base, int elem_bytes, uint64_t inner_elems,
                    uint64_t rows, uint32_t box_inner, uint32_t box_rows, int swizzle_bytes)
{
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return false;
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
    }
    {
        std::lock_guard<std::mutex> lock(g_tmap_mu);
        for (const TmapEntry &e : g_tmaps) {
            if (e.valid && e.base == base && e.elem_bytes == elem_bytes &&
                e.swizzle == swizzle_bytes && e.inner == inner_elems && e.rows == rows &&
                e.box_inner == box_inner && e.box_rows == box_rows) {
                *map = e.map;
                return true;
            }
        }
    }
    const cuuint64_t dims[2] = {inner_elems, rows};
    const cuuint64_t strides[1] = {inner_elems * static_cast<uint64_t>(elem_bytes)};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt =
        elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const CUtensorMapSwizzle sw =
        swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const CUresult r = g_encode(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    std::lock_guard<std::mutex> lock(g_tmap_mu);
    TmapEntry &e = g_tmaps[g_tmap_next];
    g_tmap_next = (g_tmap_next + 1) % kTmapEntries;
    e.base = base;
    e.elem_bytes = elem_bytes;
    e.swizzle = swizzle_bytes;
    e.inner = inner_elems;
    e.rows = rows;
    e.box_inner = box_inner;
    e.box_rows = box_rows;
    e.map = *map;
    e.valid = true;
    return true;
}

}  // namespace pkv

extern "C" const char *pkv_status_string(pkv_status status)
{
    switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported size or configuration";
    case PKV_ERR_MISALIGNED: return "misaligned pointer";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_CUDA: return "CUDA runtime or launch failure";
    case PKV_ERR_EXHAUSTED: return "no free block (or host memory) for the request";
    }
    return "unknown status";
}
