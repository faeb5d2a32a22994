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
#include <mutex>

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

// Q4_0 append: one warp per input row (slot, token, kv head) of K and of V.
// The row's HD / 32 blocks are spread over the warp, L = 1024 / HD lanes per
// block, each lane holding VPL = HD / 32 consecutive values: lane l has
// elements VPL (l % L) .. of block l / L. A block's scale comes from a
// shuffle reduction over its L lanes; its 16 code bytes (byte j: element j in
// the low nibble, element j + 16 in the high one) from the lanes of its first
// half, each joined with the lane L / 2 further on. The row's 18-byte blocks
// are assembled in shared memory and leave as whole 32-bit words (row_bytes
// is a multiple of 4). Row indices are 32-bit (the host splits larger appends
// by slots).
constexpr int kAppendWarps = 8;

template <int HD>
__device__ __forceinline__ void load_vals(const float *src, float (&x)[HD / 32]) {
    constexpr int VPL = HD / 32;
    if constexpr (VPL >= 4) {
#pragma unroll
        for (int k = 0; k < VPL / 4; ++k) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(src) + k);
            x[4 * k] = v.x;
            x[4 * k + 1] = v.y;
            x[4 * k + 2] = v.z;
            x[4 * k + 3] = v.w;
        }
    } else {
        const float2 v = __ldg(reinterpret_cast<const float2 *>(src));
        x[0] = v.x;
        x[1] = v.y;
    }
}

// Quantise the block this lane shares with its L - 1 neighbours into the row
// image (block bb at byte 18 bb). Every lane of the warp must call it.
template <int HD>
__device__ __forceinline__ void q4_quant_lane(const float (&x)[HD / 32], int bb, int li,
                                              uint8_t *img) {
    constexpr int VPL = HD / 32, L = 32 / VPL;
    // amax: max |x| from +0; NaN never raises it (fmaxf returns the non-NaN operand)
    float a = 0.0f;
#pragma unroll
    for (int k = 0; k < VPL; ++k) a = fmaxf(a, fabsf(x[k]));
#pragma unroll
    for (int o = 1; o < L; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    // d = amax / -8: a scaling by a power of two, so the product by -1/8 is
    // the same correctly rounded value as the division.
    const float d = __fmul_rn(a, -0.125f);
    const float id = (d != 0.0f) ? __frcp_rn(d) : 0.0f;  // IEEE reciprocal, nearest
    // One fp32 multiply (no contraction), a saturating round-half-even
    // conversion (NaN -> 0), a wrapping +8, then the clamp to [0, 15]; four
    // codes per word, one per byte.
    uint32_t codes[(VPL + 3) / 4] = {};
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
        const int q = __float2int_rn(__fmul_rn(x[k], id));
        int c = static_cast<int>(static_cast<unsigned>(q) + 8u);
        c = c < 0 ? 0 : (c > 15 ? 15 : c);
        codes[k / 4] |= static_cast<uint32_t>(c) << (8 * (k % 4));
    }
    uint16_t *blk = reinterpret_cast<uint16_t *>(img + 18 * bb);  // 2-byte aligned
#pragma unroll
    for (int w = 0; w < (VPL + 3) / 4; ++w) {
        const uint32_t hi = __shfl_down_sync(0xffffffffu, codes[w], L / 2);
        const uint32_t bytes = codes[w] | (hi << 4);
        if (li < L / 2) {
            // VPL bytes of the block's 16 code bytes, from byte VPL li + 4 w
            uint16_t *dst = blk + 1 + (VPL * li + 4 * w) / 2;
            dst[0] = static_cast<uint16_t>(bytes);
            if (VPL >= 4) dst[1] = static_cast<uint16_t>(bytes >> 16);
        }
    }
    if (li == 0) blk[0] = __half_as_ushort(__float2half_rn(d));
}

// The lane's VPL values as fp16 at dst (a sink or ring mirror row).
template <int HD>
__device__ __forceinline__ void store_half_vals(uint8_t *dst, const float (&x)[HD / 32]) {
    constexpr int VPL = HD / 32;
    if constexpr (VPL == 8) {
        *reinterpret_cast<uint4 *>(dst) =
            make_uint4(pack_half2(x[0], x[1]), pack_half2(x[2], x[3]), pack_half2(x[4], x[5]),
                       pack_half2(x[6], x[7]));
    } else if constexpr (VPL == 4) {
        *reinterpret_cast<uint2 *>(dst) =
            make_uint2(pack_half2(x[0], x[1]), pack_half2(x[2], x[3]));
    } else {
        *reinterpret_cast<uint32_t *>(dst) = pack_half2(x[0], x[1]);
    }
}

template <int HD>
__global__ void __launch_bounds__(kAppendWarps * 32)
    kv_append_q4_kernel(const float *__restrict__ k_new, const float *__restrict__ v_new,
                        uint8_t *__restrict__ k_planes, uint8_t *__restrict__ v_planes,
                        const int32_t *__restrict__ pos0, int nslots, int n, int n_kv,
                        int max_seq, size_t plane_bytes, size_t body_off, size_t row_bytes,
                        size_t sink_off, size_t ring_off, int shadow_sink, int shadow_win,
                        unsigned *err) {
    constexpr int VPL = HD / 32, L = 32 / VPL;
    constexpr int RW = HD / 32 * kQ4BlockBytes / 4;  // 32-bit words of an output row
    __shared__ __align__(16) uint32_t img[kAppendWarps][2][RW];  // K, V rows
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int bb = lane / L, li = lane % L;
    const uint32_t rows = static_cast<uint32_t>(nslots) * n * n_kv;
    const uint32_t wstep = gridDim.x * kAppendWarps;
    uint8_t *ik = reinterpret_cast<uint8_t *>(img[wib][0]);
    uint8_t *iv = reinterpret_cast<uint8_t *>(img[wib][1]);
    const int e = VPL * lane;  // first element of the row this lane holds
    // the next row's values are loaded before this row is quantised
    float nk[VPL], nv[VPL];
    uint32_t row = blockIdx.x * kAppendWarps + wib;
    if (row < rows) {
        load_vals<HD>(k_new + static_cast<size_t>(row) * HD + e, nk);
        load_vals<HD>(v_new + static_cast<size_t>(row) * HD + e, nv);
    }
    for (; row < rows; row += wstep) {
        float xk[VPL], xv[VPL];
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            xk[k] = nk[k];
            xv[k] = nv[k];
        }
        if (row + wstep < rows) {
            load_vals<HD>(k_new + static_cast<size_t>(row + wstep) * HD + e, nk);
            load_vals<HD>(v_new + static_cast<size_t>(row + wstep) * HD + e, nv);
        }
        // the row (u, t, h) and its destination (the same for the whole warp)
        const uint32_t r2 = row / static_cast<uint32_t>(n_kv);
        const int h = static_cast<int>(row - r2 * n_kv);
        const uint32_t uu = r2 / static_cast<uint32_t>(n);
        const int t = static_cast<int>(r2 - uu * n);
        const int p0 = pos0[uu];
        const long long pos = static_cast<long long>(p0) + t;
        const bool ok = p0 >= 0 && pos < max_seq;
        if (!ok && lane == 0) flag_error(err, FA_ERRBIT_DEVICE);
        q4_quant_lane<HD>(xk, bb, li, ik);
        q4_quant_lane<HD>(xv, bb, li, iv);
        if (ok) {
            const size_t plane = static_cast<size_t>(uu) * plane_bytes;
            // fp16 mirrors: the shadow sink rows, and the rows that stay among
            // the 256 newest after this call (no two rows of a call share a
            // ring slot)
            if (pos < shadow_sink) {
                const size_t so =
                    plane + sink_off + ((static_cast<size_t>(h) * kSinkMax + pos) * HD + e) * 2;
                store_half_vals<HD>(k_planes + so, xk);
                store_half_vals<HD>(v_planes + so, xv);
            }
            if (shadow_win > 0 && t >= n - kRingRows) {
                const size_t ro =
                    plane + ring_off +
                    ((static_cast<size_t>(h) * kRingRows + (pos % kRingRows)) * HD + e) * 2;
                store_half_vals<HD>(k_planes + ro, xk);
                store_half_vals<HD>(v_planes + ro, xv);
            }
            const size_t dst =
                plane + body_off + (static_cast<size_t>(h) * max_seq + pos) * row_bytes;
            __syncwarp();
#pragma unroll
            for (int w = lane; w < RW; w += 32) {
                *reinterpret_cast<uint32_t *>(k_planes + dst + 4 * w) = img[wib][0][w];
                *reinterpret_cast<uint32_t *>(v_planes + dst + 4 * w) = img[wib][1][w];
            }
        }
        __syncwarp();  // the image is read before the next row overwrites it
    }
}

// Blocks of kernel that are resident on the device at once (one wave), per
// device and kernel; 0 if the query failed.
template <typename Kernel>
int resident_blocks(Kernel kernel, int threads, int slot) {
    constexpr int kDevs = 64, kSlots = 3;
    static int blocks[kDevs][kSlots] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs || slot < 0 ||
        slot >= kSlots) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (blocks[dev][slot] == 0) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) !=
            cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        blocks[dev][slot] = per_sm * device_sm_count();
    }
    return blocks[dev][slot];
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
            const long long rows = static_cast<long long>(ns) * n * g.n_kv;
            auto kernel = g.hd == 64    ? kv_append_q4_kernel<64>
                          : g.hd == 128 ? kv_append_q4_kernel<128>
                                        : kv_append_q4_kernel<256>;
            // one wave: every warp loops over rows with the next row's loads in flight
            const int slot = g.hd == 64 ? 0 : (g.hd == 128 ? 1 : 2);
            const int resident = resident_blocks(kernel, kAppendWarps * 32, slot);
            const long long want = (rows + kAppendWarps - 1) / kAppendWarps;
            const int grid = resident > 0 ? static_cast<int>(std::min<long long>(want, resident))
                                          : grid_for(rows, kAppendWarps);
            kernel<<<grid, kAppendWarps * 32, 0, stream>>>(
                k_new + in_off * 4, v_new + in_off * 4,
                k_planes + static_cast<size_t>(u0) * g.bytes,
                v_planes + static_cast<size_t>(u0) * g.bytes, pos0 + u0, ns, n, g.n_kv,
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
