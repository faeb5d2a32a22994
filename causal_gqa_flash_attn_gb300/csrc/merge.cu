// merge.cu -- merge of two attention states by their log-sum-exps
// ("vt/ops.h" (vllm-cpp-sys), MergeAttnStates, after section 2.2 of the paper
// it cites): two softmax attention results over disjoint key sets, each with
// the log-sum-exp of its scores, become the result over the union.
//
// Per token t and head h (outputs [T][H][D] fp32, lses [H][T] fp32):
//   - tokens t >= with_context (when with_context >= 0) take the suffix output
//     and its lse unchanged;
//   - an lse of +inf counts as -inf;
//   - both -inf (neither side has a key): the prefix output and lse -inf;
//   - otherwise m = max(lp, ls), wp = exp(lp - m), ws = exp(ls - m),
//     out = prefix * wp / (wp + ws) + suffix * ws / (wp + ws),
//     lse = log(wp + ws) + m.
// Arithmetic is fp32. The work is a stream over 3 D floats per (t, h): one
// thread per 4 consecutive floats of a row, 128-bit loads and stores, a grid of
// a few blocks per SM striding over the rows.
#include "fa_device.cuh"
#include "fa_internal.h"

#include <cmath>

namespace fa {
namespace {

constexpr int kMergeThreads = 256;

__global__ void __launch_bounds__(kMergeThreads)
    merge_attn_states_kernel(float *__restrict__ out, float *__restrict__ out_lse,
                             const float4 *__restrict__ prefix, const float *__restrict__ prefix_lse,
                             const float4 *__restrict__ suffix, const float *__restrict__ suffix_lse,
                             int T, int H, int D4, int with_context) {
    const long long total = static_cast<long long>(T) * H * D4;
    for (long long i = blockIdx.x * static_cast<long long>(kMergeThreads) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * kMergeThreads) {
        const long long row = i / D4;  // t * H + h
        const int d4 = static_cast<int>(i - row * D4);
        const int t = static_cast<int>(row / H), h = static_cast<int>(row - static_cast<long long>(t) * H);
        const long long li = static_cast<long long>(h) * T + t;
        float4 r;
        float lse;
        if (with_context >= 0 && t >= with_context) {
            r = __ldg(suffix + i);
            lse = __ldg(suffix_lse + li);
        } else {
            float lp = __ldg(prefix_lse + li), ls = __ldg(suffix_lse + li);
            if (lp == INFINITY) lp = -INFINITY;
            if (ls == INFINITY) ls = -INFINITY;
            const float m = fmaxf(lp, ls);
            if (m == -INFINITY) {
                r = __ldg(prefix + i);
                lse = -INFINITY;
            } else {
                const float wp = expf(lp - m), ws = expf(ls - m), tot = wp + ws;
                const float a = wp / tot, b = ws / tot;
                const float4 x = __ldg(prefix + i), y = __ldg(suffix + i);
                r = make_float4(x.x * a + y.x * b, x.y * a + y.y * b, x.z * a + y.z * b,
                                x.w * a + y.w * b);
                lse = logf(tot) + m;
            }
        }
        reinterpret_cast<float4 *>(out)[i] = r;
        if (out_lse && d4 == 0) out_lse[li] = lse;
    }
}

}  // namespace

cudaError_t launch_merge_attn_states(float *out, float *out_lse, const float *prefix,
                                     const float *prefix_lse, const float *suffix,
                                     const float *suffix_lse, int T, int H, int D,
                                     int with_context, cudaStream_t stream) {
    const long long items = static_cast<long long>(T) * H * (D / 4);
    long long blocks = (items + kMergeThreads - 1) / kMergeThreads;
    const long long cap = static_cast<long long>(device_sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    merge_attn_states_kernel<<<static_cast<int>(blocks), kMergeThreads, 0, stream>>>(
        out, out_lse, reinterpret_cast<const float4 *>(prefix), prefix_lse,
        reinterpret_cast<const float4 *>(suffix), suffix_lse, T, H, D / 4, with_context);
    return cudaGetLastError();
}

}  // namespace fa
