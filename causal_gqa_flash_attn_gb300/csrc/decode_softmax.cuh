// decode_softmax.cuh -- the online-softmax step shared by the decode kernels
// ("attention.cu", "Decode-mode flash attention": running max, rescale of the
// accumulators when the max grows, and the exp of each score against it).
#pragma once

#include "fa_device.cuh"

namespace fa {

// Online-softmax fold of one group of scores of two heads (exp2 domain).
// sv: this thread's scores (-inf when masked), n of them per head.
template <int MT, int NT, int N>
__device__ __forceinline__ void fold_scores(float (&sv)[2][N], float sl2, float thr,
                                            float &mu0, float &mu1, float &mt0, float &mt1,
                                            float &ls0, float &ls1, float (&o)[MT][NT][4],
                                            int nt, float (&pv)[2][N]) {
    float *mu[2] = {&mu0, &mu1};
    float *mtr[2] = {&mt0, &mt1};
    float *ls[2] = {&ls0, &ls1};
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        float mx = sv[hh][0];
#pragma unroll
        for (int k = 1; k < N; ++k) mx = fmaxf(mx, sv[hh][k]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mx2 = mx * sl2;
        *mtr[hh] = fmaxf(*mtr[hh], mx2);
        const float m_new = fmaxf(*mu[hh], mx2);
        if (m_new > *mu[hh] + thr) {
            const float corr = ex2(*mu[hh] - m_new);  // 0 while nothing was seen
            *ls[hh] *= corr;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                o[mt][nt][hh] *= corr;
                o[mt][nt][2 + hh] *= corr;
            }
            *mu[hh] = m_new;
        }
        const float mref = (*mu[hh] == -INFINITY) ? 0.0f : *mu[hh];
        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < N; ++k) {
            pv[hh][k] = ex2(fmaf(sv[hh][k], sl2, -mref));
            s += pv[hh][k];
        }
        *ls[hh] += s;
    }
}

}  // namespace fa
