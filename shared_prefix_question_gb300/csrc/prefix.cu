// prefix.cu -- the prefix side of the path: the shared-prefix length (blink.py `_shared_prefix_len`)
// and writing token rows of K/V into a region of the KV arena (simit engine.py `KVArena` copies).
#include <climits>
#include <cstdint>

#include "common.cuh"

namespace blink {
namespace {

constexpr int kLcpThreads = 256;
constexpr int kLcpChunk = 1024;     // positions compared by one block per step (4 per thread)
constexpr int kLcpBlocksPerSeq = 8;  // blocks sharing one sequence's chunks

// Block (x, i): sequence i against sequence 0, over chunks x, x + 8, ... of 1024 positions; the
// first differing position (or the shorter length) is folded into the global minimum.  Each
// sequence's block 0 also folds len - 1, so every sequence keeps at least one token.  The common
// prefix of all sequences is the minimum over i of the common prefix of sequences 0 and i.
__global__ void __launch_bounds__(kLcpThreads)
    lcp_kernel(const int32_t *__restrict__ tokens, int64_t n_tokens, const int32_t *__restrict__ cu, int n,
               int *__restrict__ out, int *__restrict__ err)
{
    __shared__ int s_first;
    const int i = blockIdx.y;
    const int base0 = __ldg(cu);  // token offsets are relative to cu[0]
    const int len0 = __ldg(cu + 1) - base0;
    const int bi = __ldg(cu + i) - base0;
    const int len = __ldg(cu + i + 1) - __ldg(cu + i);
    if (len0 < 1 || static_cast<int64_t>(len0) > n_tokens || len < 1 || bi < 0 ||
        static_cast<int64_t>(bi) + len > n_tokens) {
        if (threadIdx.x == 0) atomicCAS(err, 0, BLINK_DEVICE_FLAG);
        return;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicMin(out, len - 1);
    if (i == 0) return;
    const int lim = min(len0, len);
    for (int c0 = blockIdx.x * kLcpChunk; c0 < lim; c0 += gridDim.x * kLcpChunk) {
        if (threadIdx.x == 0) s_first = *reinterpret_cast<volatile int *>(out);
        __syncthreads();
        const int known = s_first;  // a mismatch at or past the current minimum changes nothing
        __syncthreads();
        if (c0 >= known) break;
        int first = INT_MAX;
#pragma unroll
        for (int u = 0; u < kLcpChunk / kLcpThreads; ++u) {
            const int j = c0 + u * kLcpThreads + threadIdx.x;
            if (j < lim && first == INT_MAX && __ldg(tokens + j) != __ldg(tokens + bi + j)) first = j;
        }
        if (first != INT_MAX) atomicMin(out, first);
        if (__syncthreads_or(first != INT_MAX)) break;  // later chunks of this block cannot be smaller
    }
    // No difference before lim: the common prefix of the pair is lim, which the len - 1 folds
    // already undercut, so nothing more to fold.
}

// Copies n rows of `row_elems` bf16 values (16-byte chunks) from src (row stride src_stride) to
// dst (row stride dst_stride), for K and V.
__global__ void arena_copy_kernel(const uint16_t *__restrict__ k_src, const uint16_t *__restrict__ v_src,
                                  int64_t src_stride, uint16_t *__restrict__ k_dst, uint16_t *__restrict__ v_dst,
                                  int64_t dst_stride, int64_t n, int row_chunks)
{
    const int64_t total = n * row_chunks;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = e / row_chunks;
        const int c = static_cast<int>(e - r * row_chunks);
        const uint4 *ks = reinterpret_cast<const uint4 *>(k_src + r * src_stride) + c;
        const uint4 *vs = reinterpret_cast<const uint4 *>(v_src + r * src_stride) + c;
        uint4 *kd = reinterpret_cast<uint4 *>(k_dst + r * dst_stride) + c;
        uint4 *vd = reinterpret_cast<uint4 *>(v_dst + r * dst_stride) + c;
        const uint4 a = __ldcs(ks), b = __ldcs(vs);
        __stcs(kd, a);
        __stcs(vd, b);
    }
}

int sm_count_prefix()
{
    int dev = 0, c = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return c;
}

}  // namespace
}  // namespace blink

extern "C" size_t blink_shared_prefix_len_workspace(void) { return blink::kHeaderBytes; }

extern "C" blink_status blink_shared_prefix_len(const int32_t *d_tokens, int64_t n_tokens, const int32_t *d_cu,
                                                int32_t n, int32_t *d_len, int32_t *h_len, void *d_ws, size_t ws_bytes,
                                                cudaStream_t stream)
{
    using namespace blink;
    if (!d_tokens || !d_cu || !d_len || !d_ws) return BLINK_INVALID_ARG;
    if (n < 1 || n > BLINK_MAX_PLAN_SEQUENCES) return BLINK_OUT_OF_RANGE;
    if (n_tokens < 1) return BLINK_INVALID_ARG;
    if (ws_bytes < kHeaderBytes) return BLINK_WORKSPACE_TOO_SMALL;
    auto *hdr = static_cast<WorkspaceHeader *>(d_ws);
    if (n < 2) {  // fewer than two sequences share nothing
        if (cudaMemsetAsync(d_len, 0, sizeof(int32_t), stream) != cudaSuccess) return BLINK_CUDA_ERROR;
    } else {
        // 0x7F7F7F7F: larger than any length, the start of the minimum
        if (cudaMemsetAsync(d_len, 0x7F, sizeof(int32_t), stream) != cudaSuccess) return BLINK_CUDA_ERROR;
        dim3 grid(kLcpBlocksPerSeq, static_cast<unsigned>(n));
        lcp_kernel<<<grid, kLcpThreads, 0, stream>>>(d_tokens, n_tokens, d_cu, n, d_len, &hdr->error);
        if (cudaGetLastError() != cudaSuccess) return BLINK_CUDA_ERROR;
    }
    if (h_len) {
        int32_t word = 0;
        if (cudaMemcpyAsync(h_len, d_len, sizeof(int32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
            return BLINK_CUDA_ERROR;
        if (cudaMemcpyAsync(&word, &hdr->error, sizeof word, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
            return BLINK_CUDA_ERROR;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return BLINK_CUDA_ERROR;
        if (word != 0) return BLINK_DEVICE_FLAG;
    }
    return BLINK_OK;
}

extern "C" blink_status blink_kv_to_arena(const blink_bf16 *k_src, const blink_bf16 *v_src, int64_t src_row_stride,
                                          int64_t n_rows, int32_t row_elems, blink_bf16 *k_arena, blink_bf16 *v_arena,
                                          int64_t arena_row_stride, int64_t arena_slots, int64_t dst_slot,
                                          cudaStream_t stream)
{
    using namespace blink;
    if (!k_src || !v_src || !k_arena || !v_arena) return BLINK_INVALID_ARG;
    if (n_rows < 0 || row_elems < 8 || row_elems % 8 != 0) return BLINK_INVALID_ARG;
    if (src_row_stride < row_elems || arena_row_stride < row_elems || src_row_stride % 8 != 0 ||
        arena_row_stride % 8 != 0)
        return BLINK_INVALID_ARG;
    if (!aligned16(k_src) || !aligned16(v_src) || !aligned16(k_arena) || !aligned16(v_arena)) return BLINK_INVALID_ARG;
    if (dst_slot < 0 || dst_slot + n_rows > arena_slots) return BLINK_OUT_OF_RANGE;
    if (n_rows == 0) return BLINK_OK;
    const int row_chunks = row_elems / 8;
    const int sms = sm_count_prefix();
    const int64_t total = n_rows * row_chunks;
    int64_t grid = (total + 255) / 256;
    if (sms > 0 && grid > 8LL * sms) grid = 8LL * sms;
    arena_copy_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(
        k_src, v_src, src_row_stride, k_arena + dst_slot * arena_row_stride, v_arena + dst_slot * arena_row_stride,
        arena_row_stride, n_rows, row_chunks);
    if (cudaGetLastError() != cudaSuccess) return BLINK_CUDA_ERROR;
    return BLINK_OK;
}
