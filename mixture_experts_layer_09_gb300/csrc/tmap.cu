// tmap.cu -- host-side creation of TMA tensor maps (cuTensorMapEncodeTiled through the runtime's
// driver entry point, so the library needs no link against libcuda), with a small cache keyed by
// every encoding parameter so that repeated calls on the same tensors do not re-encode.
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(ptr);
    }();
    return fn;
}

struct Key {
    const void* base;
    int dtype;
    uint64_t inner, rows, row_bytes;
    uint32_t box_inner, box_rows;
    int swizzle;
    int device;
    bool operator==(const Key& o) const {
        return base == o.base && dtype == o.dtype && inner == o.inner && rows == o.rows && row_bytes == o.row_bytes &&
               box_inner == o.box_inner && box_rows == o.box_rows && swizzle == o.swizzle && device == o.device;
    }
};
struct Entry {
    Key key;
    CUtensorMap map;
};
std::mutex g_mu;
std::vector<Entry> g_cache;  // small, most recent last
constexpr size_t kCacheMax = 256;
}  // namespace

bool tmap_2d(CUtensorMap* out, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t rows,
             uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
    int dev = 0;
    cudaGetDevice(&dev);
    const Key key{base, static_cast<int>(dtype), inner, rows, row_bytes, box_inner, box_rows, static_cast<int>(swizzle),
                  dev};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (size_t i = g_cache.size(); i-- > 0;)
            if (g_cache[i].key == key) {
                *out = g_cache[i].map;
                return true;
            }
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows < 1 ? 1 : rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t es[2] = {1, 1};
    CUtensorMap m;
    if (fn(&m, dtype, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_cache.size() >= kCacheMax) g_cache.erase(g_cache.begin());
    g_cache.push_back(Entry{key, m});
    *out = m;
    return true;
}

}  // namespace moe
