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

#include <algorithm>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kThreads = 256;

// One thread per 4 consecutive fp32 values of an input row, four independent
// coalesced loads in flight per thread. Indices are 32-bit (the host checks).
__global__ void __launch_bounds__(kThreads)
    kv_append_f32_kernel(const float4 *__restrict__ k_new, const float4 *__restrict__ v_new,
                         uint8_t *__restrict__ k_planes, uint8_t *__restrict__ v_planes,
                         const int32_t *__restrict__ pos0, int nslots, int n, int n_kv, int hd,
                         int max_seq, size_t plane_bytes, size_t body_off, unsigned *err) {
    const uint32_t q4 = static_cast<uint32_t>(hd / 4);
    const uint32_t total = static_cast<uint32_t>(nslots) * n * n_kv * q4;
    const uint32_t stride = gridDim.x * blockDim.x;
    // destination offset of element i, or ~0 if its row is out of range
    auto dst = [&](uint32_t i) -> size_t {
        const uint32_t e4 = i % q4;
        uint32_t r = i / q4;
        const uint32_t h = r % static_cast<uint32_t>(n_kv);
        r /= static_cast<uint32_t>(n_kv);
        const uint32_t t = r % static_cast<uint32_t>(n);
        const uint32_t u = r / static_cast<uint32_t>(n);
        const int p0 = pos0[u];
        const long long pos = static_cast<long long>(p0) + t;
        if (p0 < 0 || pos >= max_seq) {
            if (e4 == 0) flag_error(err, FA_ERRBIT_DEVICE);
            return ~static_cast<size_t>(0);
        }
        return static_cast<size_t>(u) * plane_bytes + body_off +
               ((static_cast<size_t>(h) * max_seq + pos) * hd + 4 * e4) * 4;
    };
    uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < total; i += 4 * stride) {
        float4 xk[4], xv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            xk[u] = __ldg(k_new + i + u * stride);
            xv[u] = __ldg(v_new + i + u * stride);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t off = dst(i + u * stride);
            if (off == ~static_cast<size_t>(0)) continue;
            *reinterpret_cast<float4 *>(k_planes + off) = xk[u];
            *reinterpret_cast<float4 *>(v_planes + off) = xv[u];
        }
    }
    for (; i < total; i += stride) {
        const size_t off = dst(i);
        if (off == ~static_cast<size_t>(0)) continue;
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

// Quantise one Q4_0 block held by an 8-lane group of the warp (lane li of the
// group holds elements 4 li .. 4 li + 3 in x) into the 18 bytes at img.
// Every lane of the warp must call it (the group reductions shuffle).
__device__ __forceinline__ void q4_quant_block8(float4 x, int li, uint8_t *img) {
    // amax: max |x| from +0; NaN never raises it (fmaxf returns the non-NaN operand)
    float a = fmaxf(fmaxf(fmaxf(0.0f, fabsf(x.x)), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
    // d = amax / -8: a scaling by a power of two, so the product by -1/8 is
    // the same correctly rounded value as the division.
    const float d = __fmul_rn(a, -0.125f);
    const float id = (d != 0.0f) ? __frcp_rn(d) : 0.0f;  // IEEE reciprocal, nearest
    // One fp32 multiply (no contraction), a saturating round-half-even
    // conversion (NaN -> 0), a wrapping +8, then the clamp to [0, 15].
    const float xs[4] = {x.x, x.y, x.z, x.w};
    uint32_t codes = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int q = __float2int_rn(__fmul_rn(xs[k], id));
        int c = static_cast<int>(static_cast<unsigned>(q) + 8u);
        c = c < 0 ? 0 : (c > 15 ? 15 : c);
        codes |= static_cast<uint32_t>(c) << (8 * k);
    }
    // byte j of the block: element j (low nibble) | element j + 16 (high)
    const uint32_t hi = __shfl_down_sync(0xffffffffu, codes, 4);
    if (li < 4) {
        const uint32_t w = codes | (hi << 4);
        uint16_t *dst = reinterpret_cast<uint16_t *>(img + 2 + 4 * li);  // 2-byte aligned
        dst[0] = static_cast<uint16_t>(w);
        dst[1] = static_cast<uint16_t>(w >> 16);
    }
    if (li == 0) *reinterpret_cast<uint16_t *>(img) = __half_as_ushort(__float2half_rn(d));
}

// One warp per 4 consecutive Q4_0 blocks of the input rows (K and V): lane l
// holds 4 values of block l / 8. The two pairs of blocks (36 bytes each, a
// 4-byte aligned run of a plane row, since rows hold an even number of
// blocks) are assembled in shared memory and leave as whole 32-bit words.
// Block indices are 32-bit (the host splits larger appends by slots) and
// blocks per row (head_dim / 32) a power of two.
constexpr int kAppendWarps = 8;

__global__ void __launch_bounds__(kAppendWarps * 32)
    kv_append_q4_kernel(const float4 *__restrict__ k_new, const float4 *__restrict__ v_new,
                        uint8_t *__restrict__ k_planes, uint8_t *__restrict__ v_planes,
                        const int32_t *__restrict__ pos0, int nslots, int n, int n_kv, int hd,
                        int max_seq, size_t plane_bytes, size_t body_off, size_t row_bytes,
                        size_t sink_off, size_t ring_off, int shadow_sink, int shadow_win,
                        unsigned *err) {
    __shared__ __align__(16) uint32_t img[kAppendWarps][2][18];  // K, V: 4 blocks each
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int gq = lane >> 3, li = lane & 7;
    const uint32_t nb_shift = hd == 64 ? 1u : (hd == 128 ? 2u : 3u);  // log2(hd / 32)
    const uint32_t total = static_cast<uint32_t>(nslots) * n * n_kv << nb_shift;  // blocks
    const uint32_t groups = (total + 3) / 4;
    uint8_t *ik = reinterpret_cast<uint8_t *>(img[wib][0]);
    uint8_t *iv = reinterpret_cast<uint8_t *>(img[wib][1]);
    const uint32_t wstep = gridDim.x * kAppendWarps;
    // the next group's values are loaded before this group is quantised
    float4 nk = make_float4(0.0f, 0.0f, 0.0f, 0.0f), nv = nk;
    uint32_t w = blockIdx.x * kAppendWarps + wib;
    if (w < groups && 4 * w + gq < total) {
        nk = __ldg(k_new + static_cast<size_t>(4 * w + gq) * 8 + li);
        nv = __ldg(v_new + static_cast<size_t>(4 * w + gq) * 8 + li);
    }
    for (; w < groups; w += wstep) {
        const uint32_t blk = 4 * w + gq;
        const bool live = blk < total;
        const float4 xk = nk, xv = nv;
        if (w + wstep < groups && 4 * (w + wstep) + gq < total) {
            nk = __ldg(k_new + static_cast<size_t>(4 * (w + wstep) + gq) * 8 + li);
            nv = __ldg(v_new + static_cast<size_t>(4 * (w + wstep) + gq) * 8 + li);
        }
        // this lane's block: row (u, t, h) and its destination
        const uint32_t row = blk >> nb_shift, b = blk & ((1u << nb_shift) - 1);
        const uint32_t r2 = row / static_cast<uint32_t>(n_kv);
        const int h = static_cast<int>(row - r2 * n_kv);
        const uint32_t uu = r2 / static_cast<uint32_t>(n);
        const int t = static_cast<int>(r2 - uu * n);
        const int p0 = live ? pos0[uu] : 0;
        const long long pos = static_cast<long long>(p0) + t;
        const bool ok = live && p0 >= 0 && pos < max_seq;
        if (live && !ok && li == 0 && b == 0) flag_error(err, FA_ERRBIT_DEVICE);
        const size_t plane = static_cast<size_t>(uu) * plane_bytes;
        const size_t dst = plane + body_off +
                           (static_cast<size_t>(h) * max_seq + (ok ? pos : 0)) * row_bytes +
                           b * kQ4BlockBytes;
        q4_quant_block8(xk, li, ik + 18 * gq);
        q4_quant_block8(xv, li, iv + 18 * gq);
        if (ok) {
            // fp16 mirrors: the shadow sink rows, and the rows that stay among
            // the 256 newest after this call (no two rows of a call share a
            // ring slot)
            const int e = static_cast<int>(b) * kQ4Block + 4 * li;
            const uint2 hk = make_uint2(pack_half2(xk.x, xk.y), pack_half2(xk.z, xk.w));
            const uint2 hv = make_uint2(pack_half2(xv.x, xv.y), pack_half2(xv.z, xv.w));
            if (pos < shadow_sink) {
                const size_t so =
                    plane + sink_off + ((static_cast<size_t>(h) * kSinkMax + pos) * hd + e) * 2;
                *reinterpret_cast<uint2 *>(k_planes + so) = hk;
                *reinterpret_cast<uint2 *>(v_planes + so) = hv;
            }
            if (shadow_win > 0 && t >= n - kRingRows) {
                const size_t ro = plane + ring_off +
                                  ((static_cast<size_t>(h) * kRingRows + (pos % kRingRows)) * hd +
                                   e) * 2;
                *reinterpret_cast<uint2 *>(k_planes + ro) = hk;
                *reinterpret_cast<uint2 *>(v_planes + ro) = hv;
            }
        }
        // word lane % 9 of pair lane / 9 goes out; the pair's first block is
        // held by the lanes of group 2 (lane / 9), which pass its destination
        const int src = 16 * (lane >= 9 ? 1 : 0);
        const size_t pdst = __shfl_sync(0xffffffffu, dst, src);
        const bool pok = __shfl_sync(0xffffffffu, ok, src);
        __syncwarp();
        if (lane < 18 && pok) {
            const size_t off = pdst + 4 * (lane % 9);
            *reinterpret_cast<uint32_t *>(k_planes + off) = img[wib][0][lane];
            *reinterpret_cast<uint32_t *>(v_planes + off) = img[wib][1][lane];
        }
        __syncwarp();
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
        if (items4 + 4LL * device_sm_count() * 16 * kThreads >= (1LL << 32))
            return cudaErrorInvalidValue;  // the kernel's indices are 32-bit
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
        // block indices stay 32-bit: slots in chunks of at most 2^30 blocks
        const long long per_slot = static_cast<long long>(n) * g.n_kv * (g.hd / kQ4Block);
        const long long chunk = per_slot > 0 ? std::max(1LL, (1LL << 30) / per_slot) : nslots;
        if (per_slot > (1LL << 30)) return cudaErrorInvalidValue;
        for (long long u0 = 0; u0 < nslots; u0 += chunk) {
            const int ns = static_cast<int>(std::min<long long>(chunk, nslots - u0));
            const size_t in_off = static_cast<size_t>(u0) * per_slot * 8;  // float4s
            const long long groups = (ns * per_slot + 3) / 4;
            kv_append_q4_kernel<<<grid_for(groups, kAppendWarps), kAppendWarps * 32, 0, stream>>>(
                k4 + in_off, v4 + in_off, k_planes + static_cast<size_t>(u0) * g.bytes,
                v_planes + static_cast<size_t>(u0) * g.bytes, pos0 + u0, ns, n, g.n_kv, g.hd,
                g.max_seq, g.bytes, g.body_off, g.row_bytes, g.sink_off, g.ring_off, shadow_sink,
                shadow_win, err);
        }
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
