// pa_abi.cu -- status strings, error plumbing, device queries, tensor maps.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "pa_internal.cuh"

namespace pa {

namespace {
thread_local char g_msg[512] = "";
std::atomic<int> g_checked{0};
std::mutex g_mu;
constexpr int kMaxDevices = 64;
DevError *g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
}  // namespace

// One error record per device; zero-initialised when the module loads.
__device__ DevError g_dev_error;

pa_status fail(pa_status status, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return status;
}

pa_status cuda_fail(cudaError_t err, const char *what) {
    return fail(PA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(err), cudaGetErrorName(err));
}

pa_status check_launch(const char *kernel) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, kernel);
    return PA_OK;
}

static int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

DevError *device_error_ptr() {
    int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_err_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dev_error) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<DevError *>(p);
    }
    return g_err_ptr[dev];
}

int sm_count() {
    int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

bool checked_mode() { return g_checked.load(std::memory_order_relaxed) != 0; }

static pa_status get_encoder() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return PA_OK;
}

pa_status encode_tensor_map_3d(CUtensorMap *map, const void *base, int64_t dim0, int64_t dim1, int64_t dim2,
                               int64_t stride1_bytes, int64_t stride2_bytes, int32_t box0, int32_t box2,
                               bool swizzle128) {
    pa_status st = get_encoder();
    if (st != PA_OK) return st;
    const cuuint64_t dims[3] = {(cuuint64_t)dim0, (cuuint64_t)dim1, (cuuint64_t)dim2};
    const cuuint64_t strides[2] = {(cuuint64_t)stride1_bytes, (cuuint64_t)stride2_bytes};
    const cuuint32_t box[3] = {(cuuint32_t)box0, 1u, (cuuint32_t)box2};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for dims %lld x %lld x %lld", (int)r,
                    (long long)dim0, (long long)dim1, (long long)dim2);
    return PA_OK;
}

pa_status encode_halves_map(CUtensorMap *map, const void *base, int64_t num_rows, int64_t row_stride_bytes,
                            int32_t num_heads, int32_t box_rows, int32_t box_halves) {
    pa_status st = get_encoder();
    if (st != PA_OK) return st;
    // Dims innermost first: 64 elements of a row half, row, half, head.
    const cuuint64_t dims[4] = {64u, (cuuint64_t)num_rows, 2u, (cuuint64_t)num_heads};
    const cuuint64_t strides[3] = {(cuuint64_t)row_stride_bytes, 128u, 256u};
    const cuuint32_t box[4] = {64u, (cuuint32_t)box_rows, (cuuint32_t)box_halves, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for %lld rows x %d heads", (int)r,
                    (long long)num_rows, num_heads);
    return PA_OK;
}

pa_status encode_kv_tensor_map_halves(CUtensorMap *map, const void *base, int64_t num_slots,
                                      int32_t num_kv_heads, int32_t box_rows) {
    return encode_halves_map(map, base, num_slots, (int64_t)num_kv_heads * 256, num_kv_heads, box_rows, 2);
}

}  // namespace pa

extern "C" {

int pa_version(void) { return 10000; }

const char *pa_status_str(pa_status s) {
    switch (s) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_DEVICE_CHECK: return "PA_ERR_DEVICE_CHECK";
    }
    return "PA_ERR_UNKNOWN";
}

const char *pa_last_error_message(void) { return pa::g_msg; }

pa_status pa_set_checked(int32_t enabled) {
    pa::g_checked.store(enabled ? 1 : 0);
    return PA_OK;
}

pa_status pa_get_device_error(pa_stream_t stream, int32_t *code, int64_t *where) {
    if (code) *code = 0;
    if (where) *where = 0;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return pa::cuda_fail(e, "cudaStreamSynchronize");
    pa::DevError rec;
    e = cudaMemcpyFromSymbol(&rec, pa::g_dev_error, sizeof rec);
    if (e != cudaSuccess) return pa::cuda_fail(e, "reading the device error record");
    if (rec.code == 0) return PA_OK;
    pa::DevError zero = {0, 0, 0};
    e = cudaMemcpyToSymbol(pa::g_dev_error, &zero, sizeof zero);
    if (e != cudaSuccess) return pa::cuda_fail(e, "clearing the device error record");
    if (code) *code = rec.code;
    if (where) *where = rec.where;
    return pa::fail(PA_ERR_DEVICE_CHECK, "device error %d at %lld", rec.code, (long long)rec.where);
}

}  // extern "C"
