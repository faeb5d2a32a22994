// kv_append.cu -- append new K/V rows to per-slot KV planes: a strided copy for
// the fp32 format, the Q4_0 quantiser with fp16 sink/ring mirroring for the
// Q4_0 format ("attention.cu", fc_attn_kv_append, fc_attn_kv_append_q4 and
// fc_attn_kv_append_slots_q4; block format from "4-bit KV cache (Q4_0 blocks)"),
// the binary16 rounding of the half-width cache ("qwen38_batched.rs", BQ_KV16)
// and the fp8 e4m3fn store with the plane's scale ("vt/ops.h",
// ReshapeAndCacheFp8: Quantize(x / scale)).
//
// All kernels are single-pass and HBM-bound: every input byte is read once
// with coalesced loads and every output byte written once.
#include <cuda_fp8.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kThreads = 256;

// One thread per 4 consecutive fp32 values of an input row.
__global__ void __launch_bounds__(kThreads)
    kv_append_f32_kernel(const float4 *__restrict__ k_new, const float4 *__restrict__ v_new,
                         uint8_t *__restrict__ k_planes, uint8_t *__restrict__ v_planes,
                         const int32_t *__restrict__ pos0, int nslots, int n, int n_kv, int hd,
                         int max_seq, size_t plane_bytes, size_t body_off, unsigned *err) {
    const int q4 = hd / 4;
    const long long total = static_cast<long long>(nslots) * n * n_kv * q4;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int e4 = static_cast<int>(i % q4);
        long long r = i / q4;
        const int h = static_cast<int>(r % n_kv);
        r /= n_kv;
        const int t = static_cast<int>(r % n);
        const int u = static_cast<int>(r / n);
        const int p0 = pos0[u];
        const long long pos = static_cast<long long>(p0) + t;
        if (p0 < 0 || pos >= max_seq) {
            if (e4 == 0) flag_error(err, FA_ERRBIT_DEVICE);
            continue;
        }
        const size_t off = static_cast<size_t>(u) * plane_bytes + body_off +
                           ((static_cast<size_t>(h) * max_seq + pos) * hd + 4 * e4) * 4;
        *reinterpret_cast<float4 *>(k_planes + off) = __ldg(k_new + i);
        *reinterpret_cast<float4 *>(v_planes + off) = __ldg(v_new + i);
    }
}

// A plane scale the fp8 store can divide by.
__device__ __forceinline__ bool good_scale(float c) { return c > 0.0f && c <= 3.402823466e38f; }

// binary16 and fp8 e4m3fn rows: one thread per 4 consecutive fp32 values of
// an input row, K and V. FP8: value / scale (IEEE division), then the
// hardware conversion to e4m3 with nearest-even rounding and saturation to
// the largest finite value (NaN stays NaN).
template <int FMT>
__global__ void __launch_bounds__(kThreads)
    kv_append_narrow_kernel(const float4 *__restrict__ k_new, const float4 *__restrict__ v_new,
                            uint8_t *__restrict__ k_planes, uint8_t *__restrict__ v_planes,
                            const int32_t *__restrict__ pos0, int nslots, int n, int n_kv,
                            int hd, int max_seq, size_t plane_bytes, size_t body_off,
                            size_t scale_off, unsigned *err) {
    constexpr int EB = FMT == kFmtF16 ? 2 : 1;  // bytes per stored value
    const int q4 = hd / 4;
    const long long total = static_cast<long long>(nslots) * n * n_kv * q4;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int e4 = static_cast<int>(i % q4);
        long long r = i / q4;
        const int h = static_cast<int>(r % n_kv);
        r /= n_kv;
        const int t = static_cast<int>(r % n);
        const int u = static_cast<int>(r / n);
        const int p0 = pos0[u];
        const long long pos = static_cast<long long>(p0) + t;
        if (p0 < 0 || pos >= max_seq) {
            if (e4 == 0) flag_error(err, FA_ERRBIT_DEVICE);
            continue;
        }
        const size_t plane = static_cast<size_t>(u) * plane_bytes;
        const size_t off =
            plane + body_off + ((static_cast<size_t>(h) * max_seq + pos) * hd + 4 * e4) * EB;
        const float4 xk = __ldg(k_new + i), xv = __ldg(v_new + i);
        if constexpr (FMT == kFmtF16) {
            *reinterpret_cast<uint2 *>(k_planes + off) =
                make_uint2(pack_half2(xk.x, xk.y), pack_half2(xk.z, xk.w));
            *reinterpret_cast<uint2 *>(v_planes + off) =
                make_uint2(pack_half2(xv.x, xv.y), pack_half2(xv.z, xv.w));
        } else {
            const float ck = *reinterpret_cast<const float *>(k_planes + plane + scale_off);
            const float cv = *reinterpret_cast<const float *>(v_planes + plane + scale_off);
            if (!good_scale(ck) || !good_scale(cv)) {
                if (e4 == 0) flag_error(err, FA_ERRBIT_DEVICE);
                continue;
            }
            *reinterpret_cast<uint32_t *>(k_planes + off) = fp8x4(xk, ck);
            *reinterpret_cast<uint32_t *>(v_planes + off) = fp8x4(xv, cv);
        }
    }
}

__global__ void kv_set_scale_kernel(uint8_t *planes, int nslots, size_t plane_bytes,
                                    size_t scale_off, float scale) {
    const int u = blockIdx.x * blockDim.x + threadIdx.x;
    if (u < nslots)
        *reinterpret_cast<float *>(planes + static_cast<size_t>(u) * plane_bytes + scale_off) =
            scale;
}

// Quantise the 32 values held by the lanes of a warp (lane j holds element j
// of the block) into the 18 bytes at blk.
__device__ __forceinline__ void q4_quant_block_warp(float x, uint8_t *blk, int lane) {
    // amax: max |x| from +0, NaN never raises it (fmaxf returns the non-NaN operand).
    float a = fmaxf(0.0f, fabsf(x));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const float d = __fdiv_rn(a, -8.0f);
    const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
    // One fp32 multiply (no contraction), a saturating round-half-even
    // conversion (NaN -> 0), a wrapping +8, then the clamp.
    const int qv = __float2int_rn(__fmul_rn(x, id));
    int c = static_cast<int>(static_cast<unsigned>(qv) + 8u);
    c = c < 0 ? 0 : (c > 15 ? 15 : c);
    const int hi = __shfl_down_sync(0xffffffffu, c, 16);
    if (lane < 16) blk[2 + lane] = static_cast<uint8_t>(c | (hi << 4));
    if (lane == 0) *reinterpret_cast<uint16_t *>(blk) = __half_as_ushort(__float2half_rn(d));
}

// One warp per Q4_0 block of an input row, K and V.
__global__ void __launch_bounds__(kThreads)
    kv_append_q4_kernel(const float *__restrict__ k_new, const float *__restrict__ v_new,
                        uint8_t *__restrict__ k_planes, uint8_t *__restrict__ v_planes,
                        const int32_t *__restrict__ pos0, int nslots, int n, int n_kv, int hd,
                        int max_seq, size_t plane_bytes, size_t body_off, size_t row_bytes,
                        size_t sink_off, size_t ring_off, int shadow_sink, int shadow_win,
                        unsigned *err) {
    const int lane = threadIdx.x & 31;
    const int nb = hd / kQ4Block;
    const long long total = static_cast<long long>(nslots) * n * n_kv * nb;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
    for (long long w = blockIdx.x * static_cast<long long>(blockDim.x / 32) + (threadIdx.x >> 5);
         w < total; w += warps) {
        const int b = static_cast<int>(w % nb);
        long long r = w / nb;
        const int h = static_cast<int>(r % n_kv);
        r /= n_kv;
        const int t = static_cast<int>(r % n);
        const int u = static_cast<int>(r / n);
        const int p0 = pos0[u];
        const long long pos = static_cast<long long>(p0) + t;
        if (p0 < 0 || pos >= max_seq) {
            if (lane == 0 && b == 0) flag_error(err, FA_ERRBIT_DEVICE);
            continue;
        }
        const float xk = __ldg(k_new + w * kQ4Block + lane);
        const float xv = __ldg(v_new + w * kQ4Block + lane);
        const size_t plane = static_cast<size_t>(u) * plane_bytes;
        const size_t blk_off =
            body_off + (static_cast<size_t>(h) * max_seq + pos) * row_bytes + b * kQ4BlockBytes;
        q4_quant_block_warp(xk, k_planes + plane + blk_off, lane);
        q4_quant_block_warp(xv, v_planes + plane + blk_off, lane);

        const int e = b * kQ4Block + lane;
        if (pos < shadow_sink) {
            const size_t so =
                plane + sink_off + ((static_cast<size_t>(h) * kSinkMax + pos) * hd + e) * 2;
            *reinterpret_cast<__half *>(k_planes + so) = __float2half_rn(xk);
            *reinterpret_cast<__half *>(v_planes + so) = __float2half_rn(xv);
        }
        // Only rows that stay among the 256 newest after this call are
        // mirrored into the ring, so no two rows of one call share a slot.
        if (shadow_win > 0 && t >= n - kRingRows) {
            const size_t ro = plane + ring_off +
                              ((static_cast<size_t>(h) * kRingRows + (pos % kRingRows)) * hd + e) * 2;
            *reinterpret_cast<__half *>(k_planes + ro) = __float2half_rn(xk);
            *reinterpret_cast<__half *>(v_planes + ro) = __float2half_rn(xv);
        }
    }
}

int grid_for(long long work_items, int items_per_block) {
    long long blocks = (work_items + items_per_block - 1) / items_per_block;
    const long long cap = static_cast<long long>(device_sm_count()) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

}  // namespace

cudaError_t launch_kv_append(const float *k_new, const float *v_new, uint8_t *k_planes,
                             uint8_t *v_planes, const int32_t *pos0, int nslots, int n,
                             const PlaneGeom &g, int shadow_sink, int shadow_win, unsigned *err,
                             cudaStream_t stream) {
    const long long items4 = static_cast<long long>(nslots) * n * g.n_kv * (g.hd / 4);
    const float4 *k4 = reinterpret_cast<const float4 *>(k_new);
    const float4 *v4 = reinterpret_cast<const float4 *>(v_new);
    if (g.fmt == kFmtF32) {
        kv_append_f32_kernel<<<grid_for(items4, kThreads), kThreads, 0, stream>>>(
            k4, v4, k_planes, v_planes, pos0, nslots, n, g.n_kv, g.hd, g.max_seq, g.bytes,
            g.body_off, err);
    } else if (g.fmt == kFmtF16) {
        kv_append_narrow_kernel<kFmtF16><<<grid_for(items4, kThreads), kThreads, 0, stream>>>(
            k4, v4, k_planes, v_planes, pos0, nslots, n, g.n_kv, g.hd, g.max_seq, g.bytes,
            g.body_off, g.scale_off, err);
    } else if (g.fmt == kFmtFp8) {
        kv_append_narrow_kernel<kFmtFp8><<<grid_for(items4, kThreads), kThreads, 0, stream>>>(
            k4, v4, k_planes, v_planes, pos0, nslots, n, g.n_kv, g.hd, g.max_seq, g.bytes,
            g.body_off, g.scale_off, err);
    } else {
        const long long items = static_cast<long long>(nslots) * n * g.n_kv * (g.hd / kQ4Block);
        kv_append_q4_kernel<<<grid_for(items, kThreads / 32), kThreads, 0, stream>>>(
            k_new, v_new, k_planes, v_planes, pos0, nslots, n, g.n_kv, g.hd, g.max_seq, g.bytes,
            g.body_off, g.row_bytes, g.sink_off, g.ring_off, shadow_sink, shadow_win, err);
    }
    return cudaGetLastError();
}

cudaError_t launch_kv_set_scale(uint8_t *planes, int nslots, size_t plane_bytes, size_t scale_off,
                                float scale, cudaStream_t stream) {
    kv_set_scale_kernel<<<(nslots + 127) / 128, 128, 0, stream>>>(planes, nslots, plane_bytes,
                                                                  scale_off, scale);
    return cudaGetLastError();
}

}  // namespace fa
