// debias.cu -- the log-space readout of the ruling engine (engine.py `_score_plain` and `answer`):
// every question is scored in several passes, one per order of its options; per pass the answer
// codes' logits go through a log-softmax, the content-free prior of that answer count is
// subtracted position by position, and each option's values are averaged over the passes
// before the temperature softmax (and, optionally, blink.py's typed answer).
//
// One warp per question; the per-option sums live in shared memory (one 256-entry row per warp),
// so the position -> option map of a pass can be any permutation.
#include <cstdint>

#include "answer.cuh"
#include "common.cuh"

namespace blink {
namespace {

constexpr int kDebiasWarps = 8;
constexpr int kMaxK = BLINK_MAX_OPTIONS;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__global__ void __launch_bounds__(kDebiasWarps * 32)
    debias_kernel(const float *__restrict__ logits, const int32_t *__restrict__ pass_off,
                  const int32_t *__restrict__ key_of_pos, int n_pass, const int32_t *__restrict__ question_pass,
                  const int32_t *__restrict__ raw_off, int B, int sum_k, const float *__restrict__ prior,
                  float log2e_over_t, float *__restrict__ raw, float *__restrict__ probs,
                  const int32_t *__restrict__ qtype, float *__restrict__ answers, int *__restrict__ err)
{
    __shared__ float acc_all[kDebiasWarps][256];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    float *acc = acc_all[warp];
    for (int q = blockIdx.x * kDebiasWarps + warp; q < B; q += gridDim.x * kDebiasWarps) {
        const int lo = __ldg(raw_off + q), hi = __ldg(raw_off + q + 1);
        const int K = hi - lo;
        const int p0 = __ldg(question_pass + q), p1 = __ldg(question_pass + q + 1);
        if (K < 1 || K > kMaxK || lo < 0 || hi > sum_k || p0 < 0 || p1 <= p0 || p1 > n_pass) {
            if (lane == 0) atomicCAS(err, 0, BLINK_DEVICE_FLAG);
            continue;
        }
        for (int i = lane; i < K; i += 32) acc[i] = 0.f;
        __syncwarp();
        bool bad = false;
        for (int p = p0; p < p1; ++p) {
            const int base = __ldg(pass_off + p);
            if (__ldg(pass_off + p + 1) - base != K) {
                bad = true;
                continue;
            }
            float z[8];
            float m = -INFINITY;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int pos = lane + 32 * j;
                z[j] = pos < K ? __ldg(logits + base + pos) : -INFINITY;
                m = fmaxf(m, z[j]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) s += lane + 32 * j < K ? exp2f((z[j] - m) * kLog2e) : 0.f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
            const float lse = m + log2f(s) * kLn2;  // natural-log log-sum-exp of the pass
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int pos = lane + 32 * j;
                if (pos < K) {
                    const int key = __ldg(key_of_pos + base + pos);
                    float lp = z[j] - lse;
                    if (prior) lp -= __ldg(prior + (K - 1) * kMaxK + pos);
                    if (key >= 0 && key < K)
                        acc[key] += lp;  // a permutation: no two lanes share a key
                    else
                        bad = true;
                }
            }
            __syncwarp();
        }
        if (__any_sync(0xFFFFFFFFu, bad)) {
            if (lane == 0) atomicCAS(err, 0, BLINK_DEVICE_FLAG);
            for (int i = lane; i < K; i += 32) probs[lo + i] = __int_as_float(0x7FC00000);
            continue;
        }
        // mean over the passes, then the temperature softmax
        const float inv_r = 1.0f / static_cast<float>(p1 - p0);
        float v[8];
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int i = lane + 32 * j;
            if (i < K) {
                const float r = acc[i] * inv_r;
                if (raw) raw[lo + i] = r;
                v[j] = r * log2e_over_t;
            } else {
                v[j] = -INFINITY;
            }
            mx = fmaxf(mx, v[j]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            v[j] = lane + 32 * j < K ? exp2f(v[j] - mx) : 0.f;
            s += v[j];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
        const float inv = 1.0f / s;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int i = lane + 32 * j;
            if (i < K) probs[lo + i] = v[j] * inv;
        }
        if (qtype && answers) write_answer(v, inv, K, lane, __ldg(qtype + q), answers + 3 * q, err);
        __syncwarp();
    }
}

}  // namespace
}  // namespace blink

extern "C" size_t blink_rotation_debias_workspace(void) { return blink::kHeaderBytes; }

extern "C" blink_status blink_rotation_debias(const float *d_logits, const int32_t *d_pass_off,
                                              const int32_t *d_key_of_pos, int32_t n_pass,
                                              const int32_t *d_question_pass, const int32_t *d_raw_off, int32_t B,
                                              int32_t sum_k, const float *d_prior, float temperature, float *d_raw,
                                              float *d_probs, float *h_probs, const int32_t *d_qtype,
                                              float *d_answers, float *h_answers, void *d_ws, size_t ws_bytes,
                                              cudaStream_t stream)
{
    using namespace blink;
    if (!d_logits || !d_pass_off || !d_key_of_pos || !d_question_pass || !d_raw_off || !d_probs || !d_ws)
        return BLINK_INVALID_ARG;
    if (!(temperature > 0.f) || !(temperature < INFINITY)) return BLINK_INVALID_ARG;
    if ((d_qtype == nullptr) != (d_answers == nullptr) || (h_answers && !d_answers)) return BLINK_INVALID_ARG;
    if (B < 1 || B > BLINK_MAX_PLAN_SEQUENCES || n_pass < B) return BLINK_OUT_OF_RANGE;
    if (sum_k < B || static_cast<int64_t>(sum_k) > static_cast<int64_t>(B) * BLINK_MAX_OPTIONS)
        return BLINK_OUT_OF_RANGE;
    if (ws_bytes < kHeaderBytes) return BLINK_WORKSPACE_TOO_SMALL;
    auto *hdr = static_cast<WorkspaceHeader *>(d_ws);
    const int grid = (B + kDebiasWarps - 1) / kDebiasWarps;
    debias_kernel<<<grid, kDebiasWarps * 32, 0, stream>>>(d_logits, d_pass_off, d_key_of_pos, n_pass, d_question_pass,
                                                         d_raw_off, B, sum_k, d_prior, kLog2e / temperature, d_raw,
                                                         d_probs, d_qtype, d_answers, &hdr->error);
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
        if (word != 0) return BLINK_DEVICE_FLAG;
    }
    return BLINK_OK;
}
