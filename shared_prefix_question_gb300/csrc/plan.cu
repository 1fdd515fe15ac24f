// plan.cu -- token-budget pack plan on the device (blink.py `_batches`, `_padded`).
//
// One thread block does the whole plan in shared memory:
//   1. keys (len - 1) << 15 | index are unique, so an ascending sort of the keys is exactly the
//      stable length order the pages' `sorted` gives (ties keep request order).  Bitonic sort.
//   2. varlen offsets: a block-wide exclusive scan of the sorted lengths.
//   3. close(s) = the slot where a forward opened at slot s must close.  Because the sorted
//      lengths ascend, "len_e * (e - s + 1) > budget" is monotone in e, so close(s) is a binary
//      search (capped at s + max_rows and n).
//   4. the forwards are the chain 0, close(0), close(close(0)), ...; it is built by pointer
//      doubling: with J = close^(2^j) known, chain[2^j + k] = J[chain[k]] and J <- J o J.
//   5. per-slot forward ids (binary search in the chain), widths, last-token indices.
// The result is bit-identical to the sequential greedy rule.
#include <cstdint>

#include "common.cuh"

namespace blink {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kMaxLen = BLINK_MAX_INPUT_TOKENS;

__device__ __forceinline__ int key_len(uint32_t key) { return static_cast<int>(key >> 15) + 1; }
__device__ __forceinline__ int key_idx(uint32_t key) { return static_cast<int>(key & 0x7FFFu); }

__global__ void __launch_bounds__(kPlanThreads, 1)
    plan_kernel(const int32_t *__restrict__ lengths, int n, int npow2, int budget, int max_rows,
                int32_t *__restrict__ order, int32_t *__restrict__ slot_of, int32_t *__restrict__ fwd_of_slot, int32_t *__restrict__ fwd_slot_start,
                int32_t *__restrict__ fwd_width, int32_t *__restrict__ cu_seqlens, int32_t *__restrict__ last_varlen,
                int32_t *__restrict__ last_padded, int32_t *__restrict__ n_forwards)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    // Region A: keys[npow2] (u32), later reused as J1[n+1] (u16) and chain[n+1] (u16).
    // Region B: J0[n+1] (u16).
    const size_t chain_off = static_cast<size_t>(n + 1 + 7) / 8 * 8;  // in u16 elements
    const size_t region_a = max(static_cast<size_t>(npow2) * 4, chain_off * 4);
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem_raw);
    uint16_t *jb = reinterpret_cast<uint16_t *>(smem_raw + region_a);
    uint16_t *ja = reinterpret_cast<uint16_t *>(smem_raw);
    uint16_t *chain = reinterpret_cast<uint16_t *>(smem_raw) + chain_off;
    __shared__ int s_bad;
    __shared__ int s_scan[kPlanThreads];
    __shared__ int s_nf;

    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    if (tid == 0) s_bad = 0;
    __syncthreads();

    // 1. keys
    for (int i = tid; i < npow2; i += nt) {
        uint32_t k = 0xFFFFFFFFu;
        if (i < n) {
            int L = lengths[i];
            if (L < 1 || L > kMaxLen) {
                s_bad = 1;
                L = 1;
            }
            k = (static_cast<uint32_t>(L - 1) << 15) | static_cast<uint32_t>(i);
        }
        keys[i] = k;
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) n_forwards[0] = -1;
        return;
    }
    for (int k = 2; k <= npow2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < npow2; i += nt) {
                int ixj = i ^ j;
                if (ixj > i) {
                    uint32_t a = keys[i], b = keys[ixj];
                    bool up = (i & k) == 0;
                    if ((a > b) == up) {
                        keys[i] = b;
                        keys[ixj] = a;
                    }
                }
            }
            __syncthreads();
        }
    }

    // 2. order and varlen offsets (each thread scans a contiguous run of slots)
    const int per = (n + nt - 1) / nt;
    const int s0 = tid * per;
    const int s1 = min(n, s0 + per);
    int run = 0;
    for (int s = s0; s < s1; ++s) {
        order[s] = key_idx(keys[s]);
        slot_of[key_idx(keys[s])] = s;
        run += key_len(keys[s]);
    }
    s_scan[tid] = run;
    __syncthreads();
    for (int off = 1; off < nt; off <<= 1) {  // Hillis-Steele inclusive scan of the run sums
        int v = tid >= off ? s_scan[tid - off] : 0;
        __syncthreads();
        s_scan[tid] += v;
        __syncthreads();
    }
    int base = s_scan[tid] - run;
    for (int s = s0; s < s1; ++s) {
        cu_seqlens[s] = base;
        base += key_len(keys[s]);
        last_varlen[s] = base - 1;
    }
    if (tid == nt - 1) cu_seqlens[n] = s_scan[nt - 1];

    // 3. close(s) into J0
    for (int s = tid; s < n; s += nt) {
        int hi = n;
        if (max_rows > 0 && s + max_rows < hi) hi = s + max_rows;
        // first e in (s, hi) with len_e * (e - s + 1) > budget, else hi
        int lo = s + 1, h = hi;
        while (lo < h) {
            int mid = (lo + h) >> 1;
            long long need = static_cast<long long>(key_len(keys[mid])) * static_cast<long long>(mid - s + 1);
            if (need > budget)
                h = mid;
            else
                lo = mid + 1;
        }
        jb[s] = static_cast<uint16_t>(lo);
    }
    if (tid == 0) jb[n] = static_cast<uint16_t>(n);
    __syncthreads();  // keys are dead from here; region A becomes J1 + chain

    // 4. the chain from slot 0, by pointer doubling
    if (tid == 0) chain[0] = 0;
    __syncthreads();
    uint16_t *jsrc = jb, *jdst = ja;
    int known = 1;
    while (true) {
        if (chain[known - 1] == n) break;  // every computed entry already reaches the end
        // extend: chain[known + k] = J(chain[k]), J = close^known
        for (int k = tid; k < known; k += nt) {
            int dst = known + k;
            if (dst <= n) chain[dst] = jsrc[chain[k]];
        }
        // J <- J o J
        for (int s = tid; s <= n; s += nt) jdst[s] = jsrc[jsrc[s]];
        __syncthreads();
        uint16_t *t = jsrc;
        jsrc = jdst;
        jdst = t;
        known = min(2 * known, n + 1);
    }
    // number of forwards = first k with chain[k] == n
    if (tid == 0) {
        int lo = 0, hi = known - 1;
        while (lo < hi) {
            int mid = (lo + hi) >> 1;
            if (chain[mid] == n)
                hi = mid;
            else
                lo = mid + 1;
        }
        s_nf = lo;
        n_forwards[0] = lo;
    }
    __syncthreads();
    const int nf = s_nf;

    // 5. forward tables and per-slot indices
    for (int f = tid; f <= n; f += nt) fwd_slot_start[f] = f <= nf ? chain[f] : n;
    for (int f = tid; f < n; f += nt) {
        int w = 0;
        if (f < nf) w = lengths[order[chain[f + 1] - 1]];
        fwd_width[f] = w;
    }
    for (int s = tid; s < n; s += nt) {
        int lo = 0, hi = nf - 1;  // last f with chain[f] <= s
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (chain[mid] <= s)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int f = lo;
        fwd_of_slot[s] = f;
        const int row = s - chain[f];
        const int width = lengths[order[chain[f + 1] - 1]];
        last_padded[s] = row * width + lengths[order[s]] - 1;
    }
}

}  // namespace
}  // namespace blink

extern "C" blink_status blink_pack_plan(const int32_t *d_lengths, int32_t n, int32_t budget, int32_t max_rows,
                                        int32_t *d_order, int32_t *d_slot_of, int32_t *d_fwd_of_slot,
                                        int32_t *d_fwd_slot_start,
                                        int32_t *d_fwd_width, int32_t *d_cu_seqlens, int32_t *d_last_varlen,
                                        int32_t *d_last_padded, int32_t *d_n_forwards, int32_t *h_n_forwards,
                                        cudaStream_t stream)
{
    using namespace blink;
    if (!d_lengths || !d_order || !d_slot_of || !d_fwd_of_slot || !d_fwd_slot_start || !d_fwd_width || !d_cu_seqlens ||
        !d_last_varlen || !d_last_padded || !d_n_forwards)
        return BLINK_INVALID_ARG;
    if (budget < 1 || max_rows < 0) return BLINK_INVALID_ARG;
    if (n < 1 || n > BLINK_MAX_PLAN_SEQUENCES) return BLINK_OUT_OF_RANGE;

    int npow2 = 1;
    while (npow2 < n) npow2 <<= 1;
    // must match the kernel's carve-up: region A (keys, later J1 + chain), then J0
    const size_t chain_off = static_cast<size_t>(n + 1 + 7) / 8 * 8;
    const size_t keys_bytes = static_cast<size_t>(npow2) * 4;
    const size_t region_a = keys_bytes > chain_off * 4 ? keys_bytes : chain_off * 4;
    const size_t smem = region_a + static_cast<size_t>(n + 1) * 2 + 16;
    if (cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) != cudaSuccess)
        return BLINK_CUDA_ERROR;
    int threads = npow2 / 2;
    if (threads < 64) threads = 64;
    if (threads > kPlanThreads) threads = kPlanThreads;
    plan_kernel<<<1, threads, smem, stream>>>(d_lengths, n, npow2, budget, max_rows, d_order, d_slot_of, d_fwd_of_slot,
                                              d_fwd_slot_start, d_fwd_width, d_cu_seqlens, d_last_varlen,
                                              d_last_padded, d_n_forwards);
    if (cudaGetLastError() != cudaSuccess) return BLINK_CUDA_ERROR;
    if (h_n_forwards) {
        if (cudaMemcpyAsync(h_n_forwards, d_n_forwards, sizeof(int32_t), cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess)
            return BLINK_CUDA_ERROR;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return BLINK_CUDA_ERROR;
        if (*h_n_forwards < 0) return BLINK_DEVICE_FLAG;
    }
    return BLINK_OK;
}
