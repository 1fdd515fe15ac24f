// readout.cu -- fused label readout (blink.py `_read` / `_read_batched` and `softmax`).
//
// Work unit: one (question, offered label) pair, i.e. one row of the CSR label list.  A warp
// takes a row, streams that label's unembedding row with 16-byte loads (the HBM-bound part),
// dots it with the question's last hidden state in FP32 and stages the logit in the output.
// The warp that completes a question's last row (an atomic ticket per question, no spinning)
// then applies the temperature softmax over that question's logits in place.  Consecutive rows
// of a block belong to the same question, so the hidden state is reused from L1.
//
// For large label counts (HBM-bound) the warps only write their logits and a second,
// one-warp-per-question launch runs the softmaxes: waiting on the ticket's result lengthened
// every warp more than the second launch costs.
#include <cstdint>
#include <mutex>

#include "answer.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace blink {
namespace {

constexpr int kReadoutWarps = 8;
// From this many labels on, the softmaxes run in a second launch instead of behind a ticket.
constexpr int kSplitFinishLabels = 8192;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// 16 bytes of a label row, read once per use (no L1 allocation); no access when pred is false
// (the result is then zero).
__device__ __forceinline__ uint4 ld_row_if(const void *p, bool pred)
{
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %5, 0;\n\t"
        "@q ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];\n\t}"
        : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
        : "l"(p), "r"(static_cast<uint32_t>(pred)));
    return v;
}

// 16 bytes of a hidden row (shared by the labels of one question, so it may stay in L1); no
// access when pred is false.  Written like the row load so both issue in program order.
__device__ __forceinline__ uint4 ld_hidden_if(const void *p, bool pred)
{
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %5, 0;\n\t"
        "@q ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];\n\t}"
        : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
        : "l"(p), "r"(static_cast<uint32_t>(pred)));
    return v;
}

__device__ __forceinline__ float dot8(uint4 a, uint4 b, float acc)
{
    acc = fmaf(bf16_lo(a.x), bf16_lo(b.x), acc);
    acc = fmaf(bf16_hi(a.x), bf16_hi(b.x), acc);
    acc = fmaf(bf16_lo(a.y), bf16_lo(b.y), acc);
    acc = fmaf(bf16_hi(a.y), bf16_hi(b.y), acc);
    acc = fmaf(bf16_lo(a.z), bf16_lo(b.z), acc);
    acc = fmaf(bf16_hi(a.z), bf16_hi(b.z), acc);
    acc = fmaf(bf16_lo(a.w), bf16_lo(b.w), acc);
    acc = fmaf(bf16_hi(a.w), bf16_hi(b.w), acc);
    return acc;
}

// Largest b in [0, B) with off[b] <= r (off ascending); clamps to a valid index on bad input.
__device__ __forceinline__ int question_of(const int32_t *__restrict__ off, int B, int r)
{
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(off + mid) <= r)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Six resident blocks per SM (at most 40 registers a thread): measured fastest on the HBM-bound
// readout-stress input (65k random 10 KB rows) among 3 to 8 blocks.
// Temperature softmax of question b's logits probs[lo, hi) in place, then the typed answer if
// asked for (one warp).
__device__ __forceinline__ void finish_question(int b, int lo, int hi, int lane, float log2e_over_t,
                                                float *__restrict__ probs, const int32_t *__restrict__ qtype,
                                                float *__restrict__ answers, int *__restrict__ err)
{
    float v[8];
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int k = lo + lane + 32 * j;
        v[j] = k < hi ? __ldcg(probs + k) * log2e_over_t : -INFINITY;
        m = fmaxf(m, v[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int k = lo + lane + 32 * j;
        v[j] = k < hi ? exp2f(v[j] - m) : 0.f;
        s += v[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    const float inv = 1.0f / s;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int k = lo + lane + 32 * j;
        if (k < hi) probs[k] = v[j] * inv;
    }
    if (qtype && answers) write_answer(v, inv, hi - lo, lane, __ldg(qtype + b), answers + 3 * b, err);
}

// kFused: the warp that completes a question (atomic ticket) runs its softmax; otherwise every
// warp only writes its logit and readout_finish_kernel runs the softmaxes afterwards (for large
// label counts, where the ticket's wait on every warp costs more than a second launch).
template <bool kFused>
__global__ void __launch_bounds__(kReadoutWarps * 32, 6)
    readout_kernel(const uint16_t *__restrict__ hidden, int64_t hstride, int hidden_rows,
                   const int32_t *__restrict__ last_idx, const int32_t *__restrict__ slot_of,
                   const uint16_t *__restrict__ unembed, int V, int H,
                   const int32_t *__restrict__ label_off, const int32_t *__restrict__ label_ids, int B, int sum_k,
                   float log2e_over_t, float *__restrict__ probs, float *__restrict__ logits,
                   const int32_t *__restrict__ qtype, float *__restrict__ answers,
                   uint32_t *__restrict__ counters, int *__restrict__ err)
{
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // readout_finish_kernel is launched as this kernel's programmatic dependent: it may be
    // scheduled once every block has started, and waits for this grid's end before it reads.
    if constexpr (!kFused) ptx::grid_launch_dependents();

    // Distributed check of the CSR offsets: block c checks questions c, c + grid, ...
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b <= B; b += gridDim.x * blockDim.x) {
        bool ok = true;
        if (b == 0) ok = __ldg(label_off) == 0;
        if (b == B) ok = ok && __ldg(label_off + B) == sum_k;
        if (b < B) {
            int k = __ldg(label_off + b + 1) - __ldg(label_off + b);
            ok = ok && k >= 1 && k <= BLINK_MAX_OPTIONS;
        }
        if (!ok) atomicCAS(err, 0, BLINK_DEVICE_FLAG);
    }

    const int r = blockIdx.x * kReadoutWarps + warp;
    if (r >= sum_k) return;
    const int b = question_of(label_off, B, r);
    const int lo = max(0, min(sum_k, __ldg(label_off + b)));
    const int hi = max(lo, min(sum_k, __ldg(label_off + b + 1)));
    const int K = hi - lo;
    if (r < lo || r >= hi) {  // malformed offsets: the row is not inside its question
        if (lane == 0) atomicCAS(err, 0, BLINK_DEVICE_FLAG);
        return;
    }
    const int id = __ldg(label_ids + r);
    int li = b;
    if (slot_of) {
        li = __ldg(slot_of + b);
        if (li < 0 || li >= B) li = -1;
    }
    const int hrow = li < 0 ? -1 : __ldg(last_idx + li);
    const bool bad = id < 0 || id >= V || hrow < 0 || hrow >= hidden_rows;

    float acc = 0.f;
    if (!bad) {
        const uint4 *w = reinterpret_cast<const uint4 *>(unembed + static_cast<int64_t>(id) * H);
        const uint4 *h = reinterpret_cast<const uint4 *>(hidden + static_cast<int64_t>(hrow) * hstride);
        const int nchunk = H >> 3;  // 8 bf16 per 16-byte chunk
        // eight 16-byte chunks of the label row and of the hidden row per lane and batch, the
        // last batch predicated: a 10 KB row costs three round trips to memory
        for (int c = lane; c < nchunk; c += 256) {
            uint4 wv[8], hv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) wv[u] = ld_row_if(w + c + 32 * u, c + 32 * u < nchunk);
#pragma unroll
            for (int u = 0; u < 8; ++u) hv[u] = ld_hidden_if(h + c + 32 * u, c + 32 * u < nchunk);
#pragma unroll
            for (int u = 0; u < 8; ++u) acc = dot8(wv[u], hv[u], acc);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);

    if (!kFused) {  // the logit is final here; readout_finish_kernel runs the softmax
        if (lane == 0) {
            const float z = bad ? __int_as_float(0x7FC00000) : acc;
            probs[r] = z;
            if (logits) logits[r] = z;
            if (bad) atomicCAS(err, 0, BLINK_DEVICE_FLAG);
        }
        return;
    }
    uint32_t ticket = 0;
    if (lane == 0) {
        const float z = bad ? __int_as_float(0x7FC00000) : acc;
        probs[r] = z;  // staged here until the question's softmax
        if (logits) logits[r] = z;
        if (bad) atomicCAS(err, 0, BLINK_DEVICE_FLAG);
        asm volatile("atom.release.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(ticket) : "l"(counters + b), "r"(static_cast<uint32_t>(K - 1)) : "memory");
    }
    ticket = __shfl_sync(0xFFFFFFFFu, ticket, 0);
    if (ticket != static_cast<uint32_t>(K - 1)) return;

    // This warp completed question b: acquire every other row's staged logit, then finish.
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    finish_question(b, lo, hi, lane, log2e_over_t, probs, qtype, answers, err);
}

// One warp per question: the softmax (and answer) over the logits readout_kernel<false> wrote.
__global__ void __launch_bounds__(kReadoutWarps * 32)
    readout_finish_kernel(const int32_t *__restrict__ label_off, int B, int sum_k, float log2e_over_t,
                          float *__restrict__ probs, const int32_t *__restrict__ qtype, float *__restrict__ answers,
                          int *__restrict__ err)
{
    ptx::grid_dep_wait();  // the logits of readout_kernel<false>, launched just before
    const int b = blockIdx.x * kReadoutWarps + (threadIdx.x >> 5);
    if (b >= B) return;
    const int lo = max(0, min(sum_k, __ldg(label_off + b)));
    const int hi = max(lo, min(sum_k, __ldg(label_off + b + 1)));
    if (hi - lo < 1 || hi - lo > BLINK_MAX_OPTIONS) return;  // flagged by the offsets check
    finish_question(b, lo, hi, threadIdx.x & 31, log2e_over_t, probs, qtype, answers, err);
}

// readout_finish_kernel as the programmatic dependent of the readout_kernel<false> launch just
// before it on `stream`: its blocks are scheduled while the logit launch drains.
cudaError_t launch_finish(const int32_t *label_off, int B, int sum_k, float log2e_over_t, float *probs,
                          const int32_t *qtype, float *answers, int *err, cudaStream_t stream)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((B + kReadoutWarps - 1) / kReadoutWarps));
    cfg.blockDim = dim3(kReadoutWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, readout_finish_kernel, label_off, B, sum_k, log2e_over_t, probs, qtype, answers,
                              err);
}

}  // namespace
}  // namespace blink

extern "C" size_t blink_label_readout_workspace(int32_t B)
{
    if (B < 1) return 0;
    return blink::kHeaderBytes + blink::align_up(static_cast<size_t>(B) * sizeof(uint32_t), 256);
}

extern "C" blink_status blink_label_readout(const blink_bf16 *hidden, int64_t hidden_row_stride, int32_t hidden_rows,
                                            const int32_t *d_last_idx, const int32_t *d_slot_of,
                                            const blink_bf16 *unembed, int32_t V, int32_t H,
                                            const int32_t *d_label_off, const int32_t *d_label_ids, int32_t B,
                                            int32_t sum_k, float temperature, float *d_probs, float *h_probs,
                                            float *d_logits, const int32_t *d_qtype, float *d_answers,
                                            float *h_answers, void *d_ws, size_t ws_bytes, cudaStream_t stream)
{
    using namespace blink;
    if (!hidden || !d_last_idx || !unembed || !d_label_off || !d_label_ids || !d_probs || !d_ws)
        return BLINK_INVALID_ARG;
    if ((d_qtype == nullptr) != (d_answers == nullptr) || (h_answers && !d_answers)) return BLINK_INVALID_ARG;
    if (!(temperature > 0.f) || !(temperature < INFINITY)) return BLINK_INVALID_ARG;  // blink.py `decide`
    if (V < 1 || H < 8 || H % 8 != 0 || hidden_rows < 1 || hidden_row_stride < H || hidden_row_stride % 8 != 0)
        return BLINK_INVALID_ARG;
    if (!aligned16(hidden) || !aligned16(unembed)) return BLINK_INVALID_ARG;
    if (B < 1 || B > BLINK_MAX_PLAN_SEQUENCES) return BLINK_OUT_OF_RANGE;
    if (sum_k < B || static_cast<int64_t>(sum_k) > static_cast<int64_t>(B) * BLINK_MAX_OPTIONS)
        return BLINK_OUT_OF_RANGE;
    if (ws_bytes < blink_label_readout_workspace(B)) return BLINK_WORKSPACE_TOO_SMALL;

    auto *hdr = static_cast<WorkspaceHeader *>(d_ws);
    auto *counters = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(d_ws) + kHeaderBytes);
    const int grid = (sum_k + kReadoutWarps - 1) / kReadoutWarps;
    const float log2e_over_t = kLog2e / temperature;
    if (sum_k >= kSplitFinishLabels) {  // no tickets: no counters to clear
        readout_kernel<false><<<grid, kReadoutWarps * 32, 0, stream>>>(
            hidden, hidden_row_stride, hidden_rows, d_last_idx, d_slot_of, unembed, V, H, d_label_off, d_label_ids, B,
            sum_k, log2e_over_t, d_probs, d_logits, d_qtype, d_answers, counters, &hdr->error);
        if (cudaGetLastError() != cudaSuccess) return BLINK_CUDA_ERROR;
        if (launch_finish(d_label_off, B, sum_k, log2e_over_t, d_probs, d_qtype, d_answers, &hdr->error, stream) !=
            cudaSuccess)
            return BLINK_CUDA_ERROR;
    } else {
        if (cudaMemsetAsync(counters, 0, static_cast<size_t>(B) * sizeof(uint32_t), stream) != cudaSuccess)
            return BLINK_CUDA_ERROR;
        readout_kernel<true><<<grid, kReadoutWarps * 32, 0, stream>>>(
            hidden, hidden_row_stride, hidden_rows, d_last_idx, d_slot_of, unembed, V, H, d_label_off, d_label_ids, B,
            sum_k, log2e_over_t, d_probs, d_logits, d_qtype, d_answers, counters, &hdr->error);
    }
    if (cudaGetLastError() != cudaSuccess) return BLINK_CUDA_ERROR;
    if (h_probs || h_answers) {
        int32_t word = 0;
        if (h_probs && cudaMemcpyAsync(h_probs, d_probs, static_cast<size_t>(sum_k) * sizeof(float),
                                       cudaMemcpyDeviceToHost, stream) != cudaSuccess)
            return BLINK_CUDA_ERROR;
        if (h_answers && cudaMemcpyAsync(h_answers, d_answers, static_cast<size_t>(B) * 3 * sizeof(float),
                                         cudaMemcpyDeviceToHost, stream) != cudaSuccess)
            return BLINK_CUDA_ERROR;
        if (cudaMemcpyAsync(&word, &hdr->error, sizeof word, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
            return BLINK_CUDA_ERROR;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return BLINK_CUDA_ERROR;
        if (word != 0) return word == BLINK_DEVICE_TIMEOUT ? BLINK_DEVICE_TIMEOUT : BLINK_DEVICE_FLAG;
    }
    return BLINK_OK;
}

// ---------------------------------------------------------------------------------------------
// The same readout for callers that cannot allocate device memory: the scratch (error word and
// one ticket per question) lives in a static device array owned by this file.
// ---------------------------------------------------------------------------------------------
namespace blink {
namespace {

constexpr int kStaticMaxDevices = 64;
constexpr int kStaticHeaderWords = 64;  // 256 bytes: the error word, then reserved
// Held by every GPU that loads the library, until the process exits.
static __device__ __align__(256) uint32_t g_readout_scratch[kStaticHeaderWords + BLINK_STATIC_SCRATCH_QUESTIONS];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Identifier of the current context (0 if the driver cannot say).  A device reset or a new
// context on the same ordinal loads the module again, at a new address, under a new identifier.
unsigned long long current_context_id()
{
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

std::mutex g_scratch_mutex;
void *g_scratch_addr[kStaticMaxDevices] = {};
unsigned long long g_scratch_ctx[kStaticMaxDevices] = {};

// Device address of g_readout_scratch in the current device's context (the array's name is
// only a host-side stand-in in host code).  Looked up once per device and context: the first
// call on a device, and the first after a device reset, look it up again.
void *scratch_address()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kStaticMaxDevices) return nullptr;
    // 0 before the runtime has made the device's context current (the lookup below does that)
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev] || ctx == 0 || g_scratch_ctx[dev] != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_readout_scratch) != cudaSuccess) return nullptr;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = current_context_id();
    }
    return g_scratch_addr[dev];
}

}  // namespace
}  // namespace blink

extern "C" blink_status blink_label_readout_noalloc(const blink_bf16 *hidden, int64_t hidden_row_stride,
                                                    int32_t hidden_rows, const int32_t *d_last_idx,
                                                    const int32_t *d_slot_of, const blink_bf16 *unembed, int32_t V,
                                                    int32_t H, const int32_t *d_label_off, const int32_t *d_label_ids,
                                                    int32_t B, int32_t sum_k, float temperature, float *d_probs,
                                                    float *h_probs, float *d_logits, cudaStream_t stream)
{
    using namespace blink;
    if (!hidden || !d_last_idx || !unembed || !d_label_off || !d_label_ids || !d_probs) return BLINK_INVALID_ARG;
    if (!(temperature > 0.f) || !(temperature < INFINITY)) return BLINK_INVALID_ARG;
    if (V < 1 || H < 8 || H % 8 != 0 || hidden_rows < 1 || hidden_row_stride < H || hidden_row_stride % 8 != 0)
        return BLINK_INVALID_ARG;
    if (!aligned16(hidden) || !aligned16(unembed)) return BLINK_INVALID_ARG;
    if (B < 1 || B > BLINK_STATIC_SCRATCH_QUESTIONS) return BLINK_OUT_OF_RANGE;
    if (sum_k < B || static_cast<int64_t>(sum_k) > static_cast<int64_t>(B) * BLINK_MAX_OPTIONS)
        return BLINK_OUT_OF_RANGE;

    void *scratch = scratch_address();
    if (!scratch) return BLINK_CUDA_ERROR;
    auto *err = static_cast<int *>(scratch);
    auto *counters = static_cast<uint32_t *>(scratch) + kStaticHeaderWords;
    const int grid = (sum_k + kReadoutWarps - 1) / kReadoutWarps;
    const float log2e_over_t = kLog2e / temperature;
    // Calls share the array: clear this call's error word (and its tickets) first.  Large label
    // counts take the same two-launch form as blink_label_readout, which uses no tickets.
    const bool split = sum_k >= kSplitFinishLabels;
    const size_t clear_words = kStaticHeaderWords + (split ? 0 : static_cast<size_t>(B));
    if (cudaMemsetAsync(scratch, 0, clear_words * sizeof(uint32_t), stream) != cudaSuccess) return BLINK_CUDA_ERROR;
    if (split) {
        readout_kernel<false><<<grid, kReadoutWarps * 32, 0, stream>>>(
            hidden, hidden_row_stride, hidden_rows, d_last_idx, d_slot_of, unembed, V, H, d_label_off, d_label_ids, B,
            sum_k, log2e_over_t, d_probs, d_logits, nullptr, nullptr, counters, err);
        if (cudaGetLastError() != cudaSuccess) return BLINK_CUDA_ERROR;
        if (launch_finish(d_label_off, B, sum_k, log2e_over_t, d_probs, nullptr, nullptr, err, stream) != cudaSuccess)
            return BLINK_CUDA_ERROR;
    } else {
        readout_kernel<true><<<grid, kReadoutWarps * 32, 0, stream>>>(
            hidden, hidden_row_stride, hidden_rows, d_last_idx, d_slot_of, unembed, V, H, d_label_off, d_label_ids, B,
            sum_k, log2e_over_t, d_probs, d_logits, nullptr, nullptr, counters, err);
    }
    if (cudaGetLastError() != cudaSuccess) return BLINK_CUDA_ERROR;
    if (h_probs) {
        int32_t word = 0;
        if (cudaMemcpyAsync(h_probs, d_probs, static_cast<size_t>(sum_k) * sizeof(float), cudaMemcpyDeviceToHost,
                            stream) != cudaSuccess)
            return BLINK_CUDA_ERROR;
        if (cudaMemcpyAsync(&word, err, sizeof word, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
            return BLINK_CUDA_ERROR;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return BLINK_CUDA_ERROR;
        if (word != 0) return word == BLINK_DEVICE_TIMEOUT ? BLINK_DEVICE_TIMEOUT : BLINK_DEVICE_FLAG;
    }
    return BLINK_OK;
}
