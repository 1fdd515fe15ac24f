// common.cu -- status strings, the device error word, tensor-map encoding.
#include <mutex>

#include "common.cuh"

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
