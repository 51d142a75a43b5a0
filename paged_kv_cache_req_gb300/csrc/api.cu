// Status plumbing and device queries shared by the libpkv entry points.
#include <cstdarg>
#include <cstdio>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "pkv_internal.cuh"

namespace pkv {

static thread_local char g_last_error[512] = "";

pkv_status fail(pkv_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

pkv_status ok() {
    g_last_error[0] = '\0';
    return PKV_OK;
}

pkv_status check_launch(const char *what) {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return ok();
}

pkv_status launch_status(cudaError_t e, const char *what) {
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    }
    return check_launch(what);
}

bool encode_tmap_bf16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims, const uint64_t *strides,
                      const uint32_t *box, int swizzle_bytes) {
    using encode_fn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static encode_fn fn = nullptr;
    static std::mutex mu;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!fn) {
            void *ptr = nullptr;
            cudaDriverEntryPointQueryResult q{};
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !ptr)
                return false;
            fn = reinterpret_cast<encode_fn>(ptr);
        }
    }
    cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void *>(base),
                          reinterpret_cast<const cuuint64_t *>(dims), reinterpret_cast<const cuuint64_t *>(strides),
                          reinterpret_cast<const cuuint32_t *>(box), elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

std::atomic<int64_t> *device_memo(const void *key, int tag) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void *, int>, std::atomic<int64_t>> memo;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    return &memo[std::make_tuple(dev, key, tag)];   // map nodes never move
}

namespace {
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitNs};
}  // namespace

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

int sm_count() {
    static std::mutex mu;
    static std::vector<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= static_cast<int>(cache.size())) cache.resize(dev + 1, 0);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace pkv

extern "C" const char *pkv_status_string(pkv_status status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported shape";
        case PKV_ERR_CAPACITY: return "buffer too small";
        case PKV_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

extern "C" const char *pkv_last_error(void) { return pkv::g_last_error; }

extern "C" int32_t pkv_abi_version(void) { return PKV_ABI_VERSION; }

extern "C" pkv_status pkv_set_wait_limit(uint64_t nanoseconds) {
    pkv::g_wait_limit_ns.store(nanoseconds ? nanoseconds : pkv::kDefaultWaitNs, std::memory_order_relaxed);
    return pkv::ok();
}

extern "C" uint64_t pkv_wait_limit(void) { return pkv::wait_limit_ns(); }
