// Host helpers shared by the kernel launchers: TMA tensor-map encoding (through the driver
// entry point fetched by the runtime, so the library links no libcuda) and the SM count.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <map>
#include <mutex>
#include <set>
#include <utility>

#include "kvc_internal.h"

namespace kvc {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

bool make_map_3d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t d0, uint64_t d1,
                 uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1,
                 uint32_t b2, CUtensorMapSwizzle sw) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    static std::mutex mu;
    static std::map<int, int> count;   // per device
    std::lock_guard<std::mutex> lock(mu);
    auto it = count.find(dev);
    if (it != count.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    count[dev] = n;
    return n;
}

int allow_dynamic_smem(const void *kernel, int bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVC_ECUDA;
    static std::mutex mu;
    static std::set<std::pair<const void *, int>> done;   // (kernel, device) pairs already raised
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({kernel, dev})) return KVC_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return KVC_ECUDA;
    done.insert({kernel, dev});
    return KVC_OK;
}

}  // namespace kvc
