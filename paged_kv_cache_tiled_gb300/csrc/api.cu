// libfattn host runtime: status strings, the per-device error word, device
// checks, tensor-map encoding and the debug wait bound.
#include <mutex>
#include <utility>
#include <vector>

#include "host_common.cuh"

namespace fa {

__device__ unsigned g_error_word;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
int g_arch_ok[kMaxDevices] = {};  // 0 unknown, 1 ok, 2 unsupported
// kernels whose dynamic shared-memory limit has been raised, per device:
// (kernel, bytes) pairs (the attribute is a per-device setting)
std::vector<std::pair<const void*, int>> g_smem_attr[kMaxDevices];
unsigned long long g_wait_ns = 4000000000ull;
int g_force_timeout = 0;
thread_local int t_launches = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}
}  // namespace

unsigned* error_word_ptr(fa_status* st) {
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) {
        *st = FA_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess || !p) {
            *st = FA_ERR_CUDA;
            return nullptr;
        }
        g_err_ptr[dev] = static_cast<unsigned*>(p);
    }
    *st = FA_OK;
    return g_err_ptr[dev];
}

fa_status make_ctx(DevCtx* ctx) {
    fa_status st;
    ctx->err = error_word_ptr(&st);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        ctx->wait_ns = g_wait_ns;
        ctx->force_timeout = g_force_timeout;
    }
    return st;
}

int sm_count() {
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sms[dev] = n > 0 ? n : 1;
    }
    return g_sms[dev];
}

fa_status check_device() {
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_arch_ok[dev]) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return FA_ERR_CUDA;
        g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    return g_arch_ok[dev] == 1 ? FA_OK : FA_ERR_UNSUPPORTED;
}

fa_status raise_dynamic_smem(const void* kernel, int bytes) {
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    for (const auto& e : g_smem_attr[dev])
        if (e.first == kernel && e.second >= bytes) return FA_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return FA_ERR_CUDA;
    g_smem_attr[dev].emplace_back(kernel, bytes);
    return FA_OK;
}

void set_launch_count(int n) { t_launches = n; }

fa_status encode_tmap_bf16_4d(CUtensorMap* map, const void* base, const uint64_t dims[4],
                              const uint64_t strides_bytes[3], const uint32_t box[4]) {
    return encode_tmap_4d(map, base, dims, strides_bytes, box, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          CU_TENSOR_MAP_SWIZZLE_128B);
}

// The driver's tensor-map encoder, looked up once (null if unavailable).
static EncodeTiledFn encoder() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess && fn)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return g_encode;
}

fa_status encode_tmap_4d(CUtensorMap* map, const void* base, const uint64_t dims[4], const uint64_t strides_bytes[3],
                         const uint32_t box[4], CUtensorMapDataType dtype, CUtensorMapSwizzle swizzle) {
    if (!encoder()) return FA_ERR_CUDA;
    cuuint64_t gdim[4] = {dims[0], dims[1], dims[2], dims[3]};
    cuuint64_t gstr[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
    cuuint32_t bdim[4] = {box[0], box[1], box[2], box[3]};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(map, dtype, 4, const_cast<void*>(base), gdim, gstr, bdim, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_INVALID_ARG;
}

fa_status encode_tmap_bf16_5d(CUtensorMap* map, const void* base, const uint64_t dims[5], const uint64_t strides_bytes[4],
                              const uint32_t box[5]) {
    if (!encoder()) return FA_ERR_CUDA;
    cuuint64_t gdim[5] = {dims[0], dims[1], dims[2], dims[3], dims[4]};
    cuuint64_t gstr[4] = {strides_bytes[0], strides_bytes[1], strides_bytes[2], strides_bytes[3]};
    cuuint32_t bdim[5] = {box[0], box[1], box[2], box[3], box[4]};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), gdim, gstr, bdim, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_INVALID_ARG;
}

}  // namespace fa

extern "C" {

const char* fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
        case FA_ERR_BOUNDS: return "FA_ERR_BOUNDS";
        case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
        case FA_ERR_NO_BLOCKS: return "FA_ERR_NO_BLOCKS";
    }
    return "FA_ERR_UNKNOWN";
}

fa_status fa_get_error(fa_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
    fa_status st;
    unsigned* p = fa::error_word_ptr(&st);
    if (st != FA_OK) return st;
    unsigned word = 0;
    if (cudaMemcpy(&word, p, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
    unsigned zero = 0;
    if (cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
    if (word & fa::ERR_BOUNDS_BIT) return FA_ERR_BOUNDS;
    if (word & fa::ERR_TIMEOUT_BIT) return FA_ERR_TIMEOUT;
    return FA_OK;
}

void fa_debug_set_wait_limit(unsigned long long ns) {
    std::lock_guard<std::mutex> lk(fa::g_mu);
    fa::g_wait_ns = ns;
}

void fa_debug_force_timeout(int enable) {
    std::lock_guard<std::mutex> lk(fa::g_mu);
    fa::g_force_timeout = enable ? 1 : 0;
}

int fa_last_launch_count(void) { return fa::t_launches; }

}  // extern "C"
