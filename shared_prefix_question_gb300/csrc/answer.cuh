// answer.cuh -- blink.py `answer_for` for one question, computed by the warp that holds the
// question's probabilities (lane l holds labels l, l + 32, ..., up to 8 per lane).
#pragma once
#include <cstdint>

#include "../../include/blink.h"

namespace blink {

// v[j] * inv is the probability of label lane + 32 j (0 past the question's K labels).
// Writes out[0..2] = {index, confidence, value} (lane 0):
//   choice (qt 0): the first label with the largest probability, (p_best - 1/K) / (1 - 1/K)
//                  (1 when K = 1), p_best;
//   noul   (qt 1): same index, NaN, p of the first label ("yes");
//   score  (qt 2): same index (ties to the lowest level), the confidence clamped to [0, 1], the
//                  expected level sum_i i p_i.
// Probabilities are renormalised by their sum first.  An unknown type latches *err.
__device__ __forceinline__ void write_answer(const float (&v)[8], float inv, int K, int lane, int qt, float *out,
                                             int *err)
{
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) z += v[j] * inv;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
    const float rz = z > 0.f ? 1.0f / z : 1.0f;
    float best = -1.f, ev = 0.f;
    int best_k = 0x7FFFFFFF;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int kl = lane + 32 * j;  // label index inside the question
        if (kl < K) {
            const float pk = v[j] * inv * rz;
            if (pk > best) {  // increasing kl: the first of equal values stays
                best = pk;
                best_k = kl;
            }
            ev = fmaf(static_cast<float>(kl), pk, ev);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ob = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        const int ok = __shfl_xor_sync(0xFFFFFFFFu, best_k, o);
        if (ob > best || (ob == best && ok < best_k)) {
            best = ob;
            best_k = ok;
        }
        ev += __shfl_xor_sync(0xFFFFFFFFu, ev, o);
    }
    const float p_first = __shfl_sync(0xFFFFFFFFu, v[0] * inv * rz, 0);
    if (lane == 0) {
        const float inv_k = 1.0f / static_cast<float>(K);
        const float conf = K > 1 ? (best - inv_k) / (1.0f - inv_k) : 1.0f;
        float c = conf, val = best;
        if (qt == 1) {
            c = __int_as_float(0x7FC00000);
            val = p_first;
        } else if (qt == 2) {
            c = fminf(1.0f, fmaxf(0.0f, conf));
            val = ev;
        } else if (qt != 0) {
            atomicCAS(err, 0, BLINK_DEVICE_FLAG);
            c = val = __int_as_float(0x7FC00000);
        }
        out[0] = static_cast<float>(best_k);
        out[1] = c;
        out[2] = val;
    }
}

}  // namespace blink
