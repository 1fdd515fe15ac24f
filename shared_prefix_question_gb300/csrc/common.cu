// common.cu -- status strings, the device error word, tensor-map encoding.
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace blink {

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}
}  // namespace

bool encode_tmap_3d_bf16(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2)
{
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace blink

extern "C" const char *blink_status_string(blink_status s)
{
    switch (s) {
    case BLINK_OK: return "ok";
    case BLINK_INVALID_ARG: return "invalid argument";
    case BLINK_OUT_OF_RANGE: return "argument outside the supported limits";
    case BLINK_WORKSPACE_TOO_SMALL: return "workspace too small";
    case BLINK_CUDA_ERROR: return "CUDA runtime error";
    case BLINK_DEVICE_FLAG: return "device-side check failed (length, label id or offsets)";
    case BLINK_DEVICE_TIMEOUT: return "bounded wait inside a kernel ran out";
    default: return "unknown status";
    }
}

extern "C" blink_status blink_read_device_status(void *d_ws, int32_t clear, cudaStream_t stream)
{
    if (!d_ws) return BLINK_INVALID_ARG;
    int32_t word = 0;
    if (cudaMemcpyAsync(&word, d_ws, sizeof word, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return BLINK_CUDA_ERROR;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return BLINK_CUDA_ERROR;
    if (clear && word != 0) {
        if (cudaMemsetAsync(d_ws, 0, sizeof word, stream) != cudaSuccess) return BLINK_CUDA_ERROR;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return BLINK_CUDA_ERROR;
    }
    if (word == 0) return BLINK_OK;
    if (word == BLINK_DEVICE_TIMEOUT) return BLINK_DEVICE_TIMEOUT;
    return BLINK_DEVICE_FLAG;
}

namespace blink {
namespace {

// One thread waits, with the same bounded wait every kernel uses, on a barrier that nothing
// arrives at; the wait gives up after limit_ns and latches BLINK_DEVICE_TIMEOUT.
__global__ void selftest_wait_kernel(int *err, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
    ptx::mbar_wait(&bar, 0, &abort_flag, err, BLINK_DEVICE_TIMEOUT, limit_ns);
}

}  // namespace
}  // namespace blink

extern "C" blink_status blink_selftest_wait_timeout(uint32_t limit_us, void *d_ws, size_t ws_bytes, cudaStream_t stream)
{
    using namespace blink;
    if (!d_ws) return BLINK_INVALID_ARG;
    if (ws_bytes < kHeaderBytes) return BLINK_WORKSPACE_TOO_SMALL;
    if (limit_us < 1 || limit_us > 1000000) return BLINK_OUT_OF_RANGE;
    auto *hdr = static_cast<WorkspaceHeader *>(d_ws);
    if (cudaMemsetAsync(&hdr->error, 0, sizeof(int32_t), stream) != cudaSuccess) return BLINK_CUDA_ERROR;
    selftest_wait_kernel<<<1, 32, 0, stream>>>(&hdr->error, static_cast<uint64_t>(limit_us) * 1000u);
    if (cudaGetLastError() != cudaSuccess) return BLINK_CUDA_ERROR;
    return blink_read_device_status(d_ws, 1, stream);
}
