// plan.cu -- token-budget pack plan on the device (blink.py `_batches`, `_padded`).
//
// One thread block does the plan in shared memory:
//   1. keys (len - 1) << 15 | index are unique, so an ascending sort of the keys is exactly the
//      stable length order the pages' `sorted` gives (ties keep request order).  Up to
//      kSmemSortMax keys the block sorts them itself (bitonic); above that the whole GPU sorts
//      first: blocks sort runs of kRun keys, then log2(n / kRun) merge rounds place every key at
//      its index in its run plus its rank in the partner run (keys are unique: no ties).
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
constexpr int kSmemSortMax = 2048;  // above this many lengths the sort runs over the whole GPU
constexpr int kRun = 1024;          // keys per block-sorted run

__device__ __forceinline__ int warp_inclusive_sum(int v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

__device__ __forceinline__ uint32_t make_key(int L, int i)
{
    if (L < 1 || L > kMaxLen) L = 1;  // flagged by the plan kernel, which re-reads the lengths
    return (static_cast<uint32_t>(L - 1) << 15) | static_cast<uint32_t>(i);
}

// Block b sorts keys of lengths [b kRun, (b + 1) kRun) ascending (bitonic, in shared memory) and
// writes its run to out.  The padding keys (all ones) sort last and are not written; with
// n < 32768 every real key is below them.
__global__ void __launch_bounds__(kRun / 2)
    plan_run_sort_kernel(const int32_t *__restrict__ lengths, int n, uint32_t *__restrict__ out)
{
    __shared__ uint32_t k[kRun];
    const int base = blockIdx.x * kRun;
    for (int i = threadIdx.x; i < kRun; i += blockDim.x)
        k[i] = base + i < n ? make_key(__ldg(lengths + base + i), base + i) : 0xFFFFFFFFu;
    __syncthreads();
    for (int size = 2; size <= kRun; size <<= 1) {
        for (int j = size >> 1; j > 0; j >>= 1) {
            const int p = threadIdx.x;  // one compare-exchange pair per thread
            const int i = (p / j) * 2 * j + (p % j);
            const uint32_t a = k[i], b = k[i + j];
            if ((a > b) == ((i & size) == 0)) {
                k[i] = b;
                k[i + j] = a;
            }
            __syncthreads();
        }
    }
    for (int i = threadIdx.x; i < kRun; i += blockDim.x)
        if (base + i < n) out[base + i] = k[i];
}

// One merge round: sorted runs of R keys (the last one may be short) pair up into runs of 2R.
// A key at position p of run r goes to (r & ~1) R + p + (number of keys below it in run r ^ 1).
// Block b handles kRun consecutive keys of one run (R >= kRun) and stages the partner run (up to
// R keys) in shared memory.
__global__ void __launch_bounds__(kRun)
    plan_merge_kernel(const uint32_t *__restrict__ src, uint32_t *__restrict__ dst, int n, int R)
{
    extern __shared__ uint32_t partner[];
    const int i0 = blockIdx.x * kRun;
    const int run = i0 / R;
    const int p_lo = (run ^ 1) * R;
    const int p_n = max(0, min(R, n - p_lo));
    for (int e = threadIdx.x; e < p_n; e += blockDim.x) partner[e] = src[p_lo + e];
    __syncthreads();
    const int i = i0 + threadIdx.x;
    if (i >= n) return;
    const uint32_t key = src[i];
    int lo = 0, hi = p_n;  // first partner key above key
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (partner[mid] < key)
            lo = mid + 1;
        else
            hi = mid;
    }
    dst[(run & ~1) * R + (i - run * R) + lo] = key;
}

__device__ __forceinline__ int key_len(uint32_t key) { return static_cast<int>(key >> 15) + 1; }
__device__ __forceinline__ int key_idx(uint32_t key) { return static_cast<int>(key & 0x7FFFu); }

__global__ void __launch_bounds__(kPlanThreads, 1)
    plan_kernel(const int32_t *__restrict__ lengths, const uint32_t *__restrict__ sorted, int n, int npow2,
                int budget, int max_rows,
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

    // 1. keys: sorted here, or already sorted over the whole GPU (`sorted`); the lengths are
    // checked here in both cases
    for (int i = tid; i < npow2; i += nt) {
        uint32_t k = 0xFFFFFFFFu;
        if (i < n) {
            const int L = lengths[i];
            if (L < 1 || L > kMaxLen) s_bad = 1;
            k = sorted ? sorted[i] : make_key(L, i);
        }
        keys[i] = k;
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) n_forwards[0] = -1;
        return;
    }
    if (!sorted) {
        for (int k = 2; k <= npow2; k <<= 1) {
            for (int j = k >> 1; j > 0; j >>= 1) {
                for (int p = tid; p < npow2 / 2; p += nt) {  // one compare-exchange pair per step
                    const int i = (p / j) * 2 * j + (p % j);
                    const uint32_t a = keys[i], b = keys[i + j];
                    if ((a > b) == ((i & k) == 0)) {
                        keys[i] = b;
                        keys[i + j] = a;
                    }
                }
                __syncthreads();
            }
        }
    }

    // 2. order and varlen offsets.  Warp w owns slots [w C, (w + 1) C); its lanes take 32
    // consecutive slots at a time (coalesced stores), prefix-summed with shuffles.
    const int lane = tid & 31, wid = tid >> 5, nw = nt >> 5;
    const int chunk = ((n + nw - 1) / nw + 31) / 32 * 32;
    const int c0 = min(n, wid * chunk), c1 = min(n, c0 + chunk);
    {
        int tot = 0;
        for (int s = c0 + lane; s < c1; s += 32) tot += key_len(keys[s]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xFFFFFFFFu, tot, o);
        if (lane == 0) s_scan[wid] = tot;
        __syncthreads();
        if (wid == 0) {  // exclusive scan of the warp totals
            const int v = lane < nw ? s_scan[lane] : 0;
            const int incl = warp_inclusive_sum(v, lane);
            if (lane < nw) s_scan[lane] = incl - v;
            if (lane == 31) s_scan[32] = incl;
        }
        __syncthreads();
        int base = s_scan[wid];
        for (int g0 = c0; g0 < c1; g0 += 32) {
            const int s = g0 + lane;
            const bool in = s < c1;
            const uint32_t key = in ? keys[s] : 0u;
            const int len = in ? key_len(key) : 0;
            const int incl = warp_inclusive_sum(len, lane);
            if (in) {
                const int idx = key_idx(key);
                order[s] = idx;
                slot_of[idx] = s;
                cu_seqlens[s] = base + incl - len;
                last_varlen[s] = base + incl - 1;
            }
            base += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (tid == 0) cu_seqlens[n] = s_scan[32];
    }

    // 3. close(s) into J0.  close is non-decreasing in s (a later start needs no fewer slots to
    // pass the budget, and its row cap ends later), so each thread takes a run of consecutive
    // slots and gallops forward from the previous answer.
    {
        const int per = (n + nt - 1) / nt;
        const int s0 = tid * per, s1 = min(n, s0 + per);
        int prev = 0;
        for (int s = s0; s < s1; ++s) {
            int hi = n;
            if (max_rows > 0 && s + max_rows < hi) hi = s + max_rows;
            // first e in (s, hi) with len_e * (e - s + 1) > budget, else hi
            auto over = [&](int e) {
                return static_cast<long long>(key_len(keys[e])) * static_cast<long long>(e - s + 1) > budget;
            };
            int lo = max(prev, s + 1);
            if (lo > hi) lo = hi;
            int b = lo, step = 1;
            while (b < hi && !over(b)) {  // after this: over() is false below lo, and b == hi or over(b)
                lo = b + 1;
                b += step;
                step <<= 1;
                if (b > hi) b = hi;
            }
            int h = b;
            while (lo < h) {
                const int mid = (lo + h) >> 1;
                if (over(mid))
                    h = mid;
                else
                    lo = mid + 1;
            }
            jb[s] = static_cast<uint16_t>(lo);
            prev = lo;
        }
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

    // 5. forward tables and per-slot indices.  The sorted length of slot s is
    // cu_seqlens[s + 1] - cu_seqlens[s] (written by this block above: visible after the barrier).
    for (int f = tid; f <= n; f += nt) fwd_slot_start[f] = f <= nf ? chain[f] : n;
    for (int f = tid; f < n; f += nt) {
        int w = 0;
        if (f < nf) {
            const int e = chain[f + 1];  // a forward's width is the length of its last slot
            w = cu_seqlens[e] - cu_seqlens[e - 1];
        }
        fwd_width[f] = w;
    }
    // Forward of each slot: mark every forward's first slot (J0's space is free now) and
    // prefix-count the marks over the same warp chunks as step 2.
    uint16_t *mark = jb;
    for (int s2 = tid; s2 < n; s2 += nt) mark[s2] = 0;
    __syncthreads();
    for (int f = tid; f < nf; f += nt) mark[chain[f]] = 1;
    __syncthreads();
    {
        int tot = 0;
        for (int s2 = c0 + lane; s2 < c1; s2 += 32) tot += mark[s2];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xFFFFFFFFu, tot, o);
        if (lane == 0) s_scan[wid] = tot;
        __syncthreads();
        if (wid == 0) {
            const int v = lane < nw ? s_scan[lane] : 0;
            const int incl = warp_inclusive_sum(v, lane);
            if (lane < nw) s_scan[lane] = incl - v;
        }
        __syncthreads();
        int base = s_scan[wid];
        for (int g0 = c0; g0 < c1; g0 += 32) {
            const int s2 = g0 + lane;
            const bool in = s2 < c1;
            const int mk = in ? mark[s2] : 0;
            const int incl = warp_inclusive_sum(mk, lane);
            if (in) {
                const int f = base + incl - 1;  // slot 0 always starts forward 0
                fwd_of_slot[s2] = f;
                const int row = s2 - chain[f];
                const int e = chain[f + 1];
                const int width = cu_seqlens[e] - cu_seqlens[e - 1];
                last_padded[s2] = row * width + (cu_seqlens[s2 + 1] - cu_seqlens[s2]) - 1;
            }
            base += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
    }
}

}  // namespace
}  // namespace blink

// The plan's scratch is its own output arrays (the whole-GPU sort ping-pongs between
// d_fwd_of_slot and d_last_padded before the plan kernel writes them), so no workspace.
extern "C" size_t blink_pack_plan_workspace(int32_t n)
{
    (void)n;
    return 0;
}

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
    // Above kSmemSortMax lengths the keys are sorted over the whole GPU first.  d_fwd_of_slot and
    // d_last_padded are the two sort buffers: the plan kernel loads the sorted keys into shared
    // memory before it writes either of them.
    const uint32_t *sorted = nullptr;
    if (n > kSmemSortMax) {
        auto *buf0 = reinterpret_cast<uint32_t *>(d_fwd_of_slot);
        auto *buf1 = reinterpret_cast<uint32_t *>(d_last_padded);
        const int runs = (n + kRun - 1) / kRun;
        plan_run_sort_kernel<<<runs, kRun / 2, 0, stream>>>(d_lengths, n, buf0);
        uint32_t *src = buf0, *dst = buf1;
        for (int R = kRun; R < n; R <<= 1) {
            const size_t psmem = static_cast<size_t>(R) * sizeof(uint32_t);
            if (psmem > 48 * 1024 &&
                cudaFuncSetAttribute(plan_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(psmem)) != cudaSuccess)
                return BLINK_CUDA_ERROR;
            plan_merge_kernel<<<runs, kRun, psmem, stream>>>(src, dst, n, R);
            uint32_t *t = src;
            src = dst;
            dst = t;
        }
        sorted = src;
    }
    int threads = npow2 / 2;
    if (threads < 64) threads = 64;
    if (threads > kPlanThreads) threads = kPlanThreads;
    plan_kernel<<<1, threads, smem, stream>>>(d_lengths, sorted, n, npow2, budget, max_rows, d_order, d_slot_of,
                                              d_fwd_of_slot,
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
