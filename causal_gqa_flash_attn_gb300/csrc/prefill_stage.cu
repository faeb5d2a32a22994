// prefill_stage.cu -- fp16 staging for the tensor-core prefill.
//
// The prefill kernel runs its two contractions on tcgen05 tensor cores with
// fp16 operands, fed by TMA. These single-pass kernels produce those operands:
//   * Q: fp32 [n][Hq][hd] -> fp16 [n][Hq][hd], round to nearest even, for the
//     query tiles of the prefill kernel's first wave of units (the kernel
//     converts the other tiles itself, while it computes);
//   * K and V: the cache rows 0..n-1 of every kv head (n = the key rows: pos0
//     plus the chunk's queries) -> fp16 [Hkv][n][hd], the value each key has
//     for every query of the prefill. For an fp32 cache
//     that is the fp32 value rounded to fp16. For a Q4_0 cache it is the fp16
//     sink copy for s < shadow_sink, the fp16 ring copy for the 256 newest
//     rows when the shadow window is 256 wide ("attention.cu",
//     fc_kvq4_is_fp16 with the ring liveness floor of fc_attn_flash_prefill_q4,
//     which for that width depends on s alone), and otherwise the decoded
//     (c - 8) * d, exact in fp32, rounded once to fp16. For an fp8 e4m3fn cache
//     it is float(byte) * scale in fp32 (the plane's scale), rounded to fp16.
//     An fp16 cache needs no staging: the prefill reads its planes in place.
// Dequantising once here, instead of inside every prefill block that reads a
// key tile, keeps the Q4_0 ALU work O(n) instead of O(n^2 / 128).
#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kThreads = 256;
// one resident wave of blocks (2048 threads per SM): 16 per SM (two waves) made
// the 8192-token staging launch 2 us slower
constexpr int kBlocksPerSM = 8;

// Q fp32 -> fp16 over the blocks of one grid row (the rows of the prefill's
// first wave of units; its kernel converts the rest), and the prefill's
// counters and Q-ready flags zeroed. Four independent coalesced loads per
// thread are in flight at a time.
struct QStage {
    const float4 *q;
    uint2 *qh;
    long long count4;
    unsigned *counter, *stage_counter, *flags;
    int n_flags;
};

__device__ __forceinline__ void stage_q_rows(const QStage &qs) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    if (i == 0) {
        *qs.counter = 0u;
        if (qs.stage_counter) *qs.stage_counter = 0u;
    }
    for (long long f = i; f < qs.n_flags; f += stride) qs.flags[f] = 0u;
    const float4 *__restrict__ q = qs.q;
    uint2 *__restrict__ qh = qs.qh;
    for (; i + 3 * stride < qs.count4; i += 4 * stride) {
        float4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) x[u] = __ldg(q + i + u * stride);
#pragma unroll
        for (int u = 0; u < 4; ++u)
            qh[i + u * stride] = make_uint2(pack_half2(x[u].x, x[u].y), pack_half2(x[u].z, x[u].w));
    }
    for (; i < qs.count4; i += stride) {
        const float4 x = __ldg(q + i);
        qh[i] = make_uint2(pack_half2(x.x, x.y), pack_half2(x.z, x.w));
    }
}

__global__ void __launch_bounds__(kThreads) stage_q_kernel(QStage qs) { stage_q_rows(qs); }

// The K and V planes are staged by one launch: blockIdx.y picks the plane.
// When Q comes along it takes grid row 0 and K, V rows 1 and 2, so that the
// blocks that run last write K and V: those tiles, read again and again by the
// prefill, are then the freshest lines in L2.

// fp32 cache rows -> fp16, one thread per 4 values.
__global__ void __launch_bounds__(kThreads)
    stage_kv_f32_kernel(const uint8_t *__restrict__ kplane, const uint8_t *__restrict__ vplane,
                        uint2 *__restrict__ kdst, uint2 *__restrict__ vdst, int n, int n_kv,
                        int hd, int max_seq, size_t body_off, QStage qs) {
    const int prow = static_cast<int>(blockIdx.y) - (qs.q ? 1 : 0);
    if (prow < 0) {
        stage_q_rows(qs);
        return;
    }
    const uint8_t *__restrict__ plane = prow ? vplane : kplane;
    uint2 *__restrict__ dst = prow ? vdst : kdst;
    // Element i of the output (32-bit: the host checks the size) is float4
    // e4 of row s of kv head g; four independent loads in flight per thread.
    const uint32_t q4 = static_cast<uint32_t>(hd / 4);
    const uint32_t total = static_cast<uint32_t>(n_kv) * static_cast<uint32_t>(n) * q4;
    const uint32_t stride = gridDim.x * blockDim.x;
    auto src = [&](uint32_t i) {
        const uint32_t e4 = i % q4, r = i / q4;
        const uint32_t s = r % static_cast<uint32_t>(n), g = r / static_cast<uint32_t>(n);
        return reinterpret_cast<const float4 *>(
            plane + body_off + ((static_cast<size_t>(g) * max_seq + s) * hd + 4 * e4) * 4);
    };
    uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < total; i += 4 * stride) {
        float4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) x[u] = __ldg(src(i + u * stride));
#pragma unroll
        for (int u = 0; u < 4; ++u)
            dst[i + u * stride] = make_uint2(pack_half2(x[u].x, x[u].y), pack_half2(x[u].z, x[u].w));
    }
    for (; i < total; i += stride) {
        const float4 x = __ldg(src(i));
        dst[i] = make_uint2(pack_half2(x.x, x.y), pack_half2(x.z, x.w));
    }
}

// fp8 e4m3fn cache rows -> fp16, one thread per 8 values (8 bytes in, 16 out).
__global__ void __launch_bounds__(kThreads)
    stage_kv_fp8_kernel(const uint8_t *__restrict__ kplane, const uint8_t *__restrict__ vplane,
                        uint4 *__restrict__ kdst, uint4 *__restrict__ vdst, int n, int n_kv,
                        int hd, int max_seq, size_t body_off, size_t scale_off, QStage qs) {
    const int prow = static_cast<int>(blockIdx.y) - (qs.q ? 1 : 0);
    if (prow < 0) {
        stage_q_rows(qs);
        return;
    }
    const uint8_t *__restrict__ plane = prow ? vplane : kplane;
    uint4 *__restrict__ dst = prow ? vdst : kdst;
    const int q8 = hd / 8;
    const long long total = static_cast<long long>(n_kv) * n * q8;
    const float c = __ldg(reinterpret_cast<const float *>(plane + scale_off));
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int e8 = static_cast<int>(i % q8);
        const long long r = i / q8;
        const int s = static_cast<int>(r % n);
        const int g = static_cast<int>(r / n);
        const uint2 w = __ldg(reinterpret_cast<const uint2 *>(
            plane + body_off + (static_cast<size_t>(g) * max_seq + s) * hd + 8 * e8));
        dst[i] = fp8x8_to_half8_scaled(w, c);
    }
}

// Q4_0 cache rows -> fp16 value seen by every query of the prefill; one
// thread per 32-value block (4 x 16-byte stores).
__global__ void __launch_bounds__(kThreads)
    stage_kv_q4_kernel(const uint8_t *__restrict__ kplane, const uint8_t *__restrict__ vplane,
                       uint4 *__restrict__ kdst, uint4 *__restrict__ vdst, int n, int n_kv,
                       int hd, int max_seq, size_t body_off, size_t row_bytes, size_t sink_off,
                       size_t ring_off, int shadow_sink, int shadow_win, QStage qs) {
    const int prow = static_cast<int>(blockIdx.y) - (qs.q ? 1 : 0);
    if (prow < 0) {
        stage_q_rows(qs);
        return;
    }
    const uint8_t *__restrict__ plane = prow ? vplane : kplane;
    uint4 *__restrict__ dst = prow ? vdst : kdst;
    const int nb = hd / kQ4Block;
    const long long total = static_cast<long long>(n_kv) * n * nb;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int b = static_cast<int>(i % nb);
        const long long r = i / nb;
        const int s = static_cast<int>(r % n);
        const int g = static_cast<int>(r / n);
        uint4 *out = dst + i * 4;  // 32 fp16 = 4 x uint4
        const uint4 *f16 = nullptr;
        if (s < shadow_sink)
            f16 = reinterpret_cast<const uint4 *>(
                plane + sink_off + ((static_cast<size_t>(g) * kSinkMax + s) * hd + b * kQ4Block) * 2);
        else if (shadow_win >= kRingRows && s >= n - kRingRows)
            f16 = reinterpret_cast<const uint4 *>(
                plane + ring_off +
                ((static_cast<size_t>(g) * kRingRows + (s % kRingRows)) * hd + b * kQ4Block) * 2);
        if (f16) {
#pragma unroll
            for (int k = 0; k < 4; ++k) out[k] = __ldg(f16 + k);
            continue;
        }
        const uint8_t *blk =
            plane + body_off + (static_cast<size_t>(g) * max_seq + s) * row_bytes + b * kQ4BlockBytes;
        const uint16_t *w16 = reinterpret_cast<const uint16_t *>(blk);  // 2-byte aligned
        const float d = __half2float(__ushort_as_half(__ldg(w16)));
        uint32_t codes[4];  // the 16 code bytes
#pragma unroll
        for (int k = 0; k < 4; ++k)
            codes[k] = static_cast<uint32_t>(__ldg(w16 + 1 + 2 * k)) |
                       (static_cast<uint32_t>(__ldg(w16 + 2 + 2 * k)) << 16);
        uint32_t h[16];  // 32 fp16 values, element order
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
            const uint32_t bj0 = (codes[j / 4] >> (8 * (j % 4))) & 0xffu;
            const uint32_t bj1 = (codes[(j + 1) / 4] >> (8 * ((j + 1) % 4))) & 0xffu;
            // low nibbles: elements j, j+1; high nibbles: elements j+16, j+17
            h[j / 2] = pack_half2(static_cast<float>(static_cast<int>(bj0 & 15u) - 8) * d,
                                  static_cast<float>(static_cast<int>(bj1 & 15u) - 8) * d);
            h[8 + j / 2] = pack_half2(static_cast<float>(static_cast<int>(bj0 >> 4) - 8) * d,
                                      static_cast<float>(static_cast<int>(bj1 >> 4) - 8) * d);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) out[k] = make_uint4(h[4 * k], h[4 * k + 1], h[4 * k + 2], h[4 * k + 3]);
    }
}

int grid_for(long long items) {
    long long blocks = (items + kThreads - 1) / kThreads;
    const long long cap = static_cast<long long>(device_sm_count()) * kBlocksPerSM;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

QStage to_stage(const QStageArgs *a) {
    if (!a) return QStage{nullptr, nullptr, 0, nullptr, nullptr, nullptr, 0};
    return QStage{reinterpret_cast<const float4 *>(a->q), reinterpret_cast<uint2 *>(a->qh),
                  static_cast<long long>(a->count / 4), a->work_counter, a->stage_counter,
                  a->flags, a->n_flags};
}

}  // namespace

cudaError_t launch_stage_q(const QStageArgs &a, cudaStream_t stream) {
    const QStage qs = to_stage(&a);
    const long long items = qs.count4 > qs.n_flags ? qs.count4 : qs.n_flags;
    stage_q_kernel<<<grid_for(items), kThreads, 0, stream>>>(qs);
    return cudaGetLastError();
}

cudaError_t launch_stage_kv(const uint8_t *kplane, const uint8_t *vplane, __half *kdst,
                            __half *vdst, int n, const PlaneGeom &g, int shadow_sink,
                            int shadow_win, const QStageArgs *qa, cudaStream_t stream) {
    const QStage qs = to_stage(qa);
    const unsigned rows = qa ? 3u : 2u;
    auto grid = [&](long long items) {
        return dim3(grid_for(qa && qs.count4 > items ? qs.count4 : items), rows);
    };
    if (g.fmt == kFmtF32) {
        const long long items = static_cast<long long>(g.n_kv) * n * (g.hd / 4);
        if (items + 4LL * device_sm_count() * kBlocksPerSM * kThreads >= (1LL << 32))
            return cudaErrorInvalidValue;  // the kernel's indices are 32-bit
        stage_kv_f32_kernel<<<grid(items), kThreads, 0, stream>>>(
            kplane, vplane, reinterpret_cast<uint2 *>(kdst), reinterpret_cast<uint2 *>(vdst), n,
            g.n_kv, g.hd, g.max_seq, g.body_off, qs);
    } else if (g.fmt == kFmtFp8) {
        const long long items = static_cast<long long>(g.n_kv) * n * (g.hd / 8);
        stage_kv_fp8_kernel<<<grid(items), kThreads, 0, stream>>>(
            kplane, vplane, reinterpret_cast<uint4 *>(kdst), reinterpret_cast<uint4 *>(vdst), n,
            g.n_kv, g.hd, g.max_seq, g.body_off, g.scale_off, qs);
    } else if (g.fmt != kFmtQ4) {
        return cudaErrorInvalidValue;  // fp16 planes are read in place
    } else {
        const long long items = static_cast<long long>(g.n_kv) * n * (g.hd / kQ4Block);
        stage_kv_q4_kernel<<<grid(items), kThreads, 0, stream>>>(
            kplane, vplane, reinterpret_cast<uint4 *>(kdst), reinterpret_cast<uint4 *>(vdst), n,
            g.n_kv, g.hd, g.max_seq, g.body_off, g.row_bytes, g.sink_off, g.ring_off,
            shadow_sink, shadow_win, qs);
    }
    return cudaGetLastError();
}

}  // namespace fa
