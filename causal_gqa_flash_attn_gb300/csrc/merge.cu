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
// warp per (t, h) row (its index arithmetic and weights once), each lane
// 128-bit loads of up to four float4s of the row issued together, a grid of a
// few blocks per SM striding over the rows.
#include "fa_device.cuh"
#include "fa_internal.h"

#include <cmath>

namespace fa {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;

// D4C: float4s per row when fixed at compile time (head_dim 64, 128, 256),
// else 0 and the row is walked in pieces of 32 float4s (d4 of them in all).
template <int D4C>
__global__ void __launch_bounds__(kMergeThreads)
    merge_attn_states_kernel(float *__restrict__ out, float *__restrict__ out_lse,
                             const float4 *__restrict__ prefix,
                             const float *__restrict__ prefix_lse,
                             const float4 *__restrict__ suffix,
                             const float *__restrict__ suffix_lse, int T, int H, int d4,
                             int with_context) {
    constexpr int PER = D4C > 0 ? (D4C + 31) / 32 : 1;  // float4s of a row per lane and piece
    const int D4 = D4C > 0 ? D4C : d4;
    const int lane = threadIdx.x & 31;
    const long long rows = static_cast<long long>(T) * H;
    const long long step = static_cast<long long>(gridDim.x) * kMergeWarps;
    for (long long row = blockIdx.x * static_cast<long long>(kMergeWarps) + (threadIdx.x >> 5);
         row < rows; row += step) {
        const int t = static_cast<int>(row / H);
        const int h = static_cast<int>(row - static_cast<long long>(t) * H);
        const long long li = static_cast<long long>(h) * T + t;
        // the row's case (warp-uniform): 0 the suffix as it is, 1 the prefix as it
        // is (neither side has a key), 2 the weighted sum
        int mode = 0;
        float a = 0.0f, b = 0.0f, lse;
        if (with_context >= 0 && t >= with_context) {
            lse = __ldg(suffix_lse + li);
        } else {
            float lp = __ldg(prefix_lse + li), ls = __ldg(suffix_lse + li);
            if (lp == INFINITY) lp = -INFINITY;
            if (ls == INFINITY) ls = -INFINITY;
            const float m = fmaxf(lp, ls);
            if (m == -INFINITY) {
                mode = 1;
                lse = -INFINITY;
            } else {
                mode = 2;
                const float wp = expf(lp - m), ws = expf(ls - m), tot = wp + ws;
                a = wp / tot;
                b = ws / tot;
                lse = logf(tot) + m;
            }
        }
        for (int c0 = 0; c0 < D4; c0 += 32 * PER) {  // a single piece when D4C > 0
            const float4 *px = prefix + row * D4 + c0, *sx = suffix + row * D4 + c0;
            float4 *ox = reinterpret_cast<float4 *>(out) + row * D4 + c0;
            const int rem = D4 - c0;  // this piece's float4s are those below rem
            float4 x[PER], y[PER];
#pragma unroll
            for (int k = 0; k < PER; ++k)
                if (lane + 32 * k < rem) {
                    if (mode != 0) x[k] = __ldg(px + lane + 32 * k);
                    if (mode != 1) y[k] = __ldg(sx + lane + 32 * k);
                }
#pragma unroll
            for (int k = 0; k < PER; ++k)
                if (lane + 32 * k < rem)
                    ox[lane + 32 * k] =
                        mode == 0 ? y[k]
                        : mode == 1
                            ? x[k]
                            : make_float4(x[k].x * a + y[k].x * b, x[k].y * a + y[k].y * b,
                                          x[k].z * a + y[k].z * b, x[k].w * a + y[k].w * b);
        }
        if (out_lse && lane == 0) out_lse[li] = lse;
    }
}

}  // namespace

cudaError_t launch_merge_attn_states(float *out, float *out_lse, const float *prefix,
                                     const float *prefix_lse, const float *suffix,
                                     const float *suffix_lse, int T, int H, int D,
                                     int with_context, cudaStream_t stream) {
    const long long rows = static_cast<long long>(T) * H;
    long long blocks = (rows + kMergeWarps - 1) / kMergeWarps;
    const long long cap = static_cast<long long>(device_sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    auto kernel = D == 64    ? merge_attn_states_kernel<16>
                  : D == 128 ? merge_attn_states_kernel<32>
                  : D == 256 ? merge_attn_states_kernel<64>
                             : merge_attn_states_kernel<0>;
    kernel<<<static_cast<int>(blocks), kMergeThreads, 0, stream>>>(
        out, out_lse, reinterpret_cast<const float4 *>(prefix), prefix_lse,
        reinterpret_cast<const float4 *>(suffix), suffix_lse, T, H, D / 4, with_context);
    return cudaGetLastError();
}

}  // namespace fa
