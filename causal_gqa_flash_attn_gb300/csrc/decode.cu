// decode.cu -- multi-slot split-KV decode and its log-sum-exp combine
// ("attention.cu" (Foundry cuda_kernels), "Decode-mode flash attention" and
// "Multi-user decode attention": fc_attn_dec_plan, fc_attn_flash_decode_slots,
// fc_attn_flash_decode_combine).
//
// Decode reads every cached key once per (slot, kv head) and does 2 x 8 x hd
// multiply-adds per key and q head; at 288 bytes per key (K+V, Q4_0, hd 256)
// that is about 28 flop/byte, more than the CUDA cores can sustain at HBM
// speed, so both contractions run on the warp-level tensor-core path:
//   S^T (16 keys x 8 heads) = K (16 x hd) . Q^T   mma.m16n8k16, f16 -> f32
//   O^T (hd x 8 heads)     += V^T (hd x 16) . P^T  same instruction
// The 8 query heads sharing a kv head are exactly the n8 dimension, so each
// K/V row is read once for the whole group. P^T is formed in registers with
// movmatrix. tcgen05 is not used here: its smallest M is 64 and the work is
// bound by memory and dequantisation, not by MMA rate.
//
// Block = 4 warps on one (slot, kv head, entry). The entry covers a run of
// consecutive splits of the slot's plan; warps take 16-key chunks in turn,
// each with its own online softmax, and merge at the end into one partial.
#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kWarps = 4;
constexpr int kChunk = 16;  // keys per warp step

struct DecodeParams {
    const float *q;
    const uint8_t *k_planes;
    const uint8_t *v_planes;
    const int32_t *pos;
    float *ws_m, *ws_l, *ws_acc;
    uint32_t *ws_header;
    int nslots, Hq, Hkv, max_seq, sink, win, fmt, shadow_sink, shadow_win;
    int split_keys, max_splits, cpc, entries, stride;
    size_t plane_bytes, body_off, row_bytes, sink_off, ring_off;
    float sl2;  // scale * log2(e)
    unsigned *err;
};

__device__ __forceinline__ int dec_plan(int seq_len, int kps, int cap, int *split_len) {
    int ns = (seq_len + kps - 1) / kps;
    ns = ns < 1 ? 1 : (ns > cap ? cap : ns);
    int sl = (seq_len + ns - 1) / ns;
    sl = (sl + 15) & ~15;
    *split_len = sl;
    return (seq_len + sl - 1) / sl;
}

// Stage the fp16 values of keys [c0, c0+16) (clamped to kmax) of one K or V
// plane into a [16][HD+8] fp16 tile; the read rule picks the fp16 sink, the
// fp16 ring, the Q4_0 body or the fp32 body.
template <int HD>
__device__ __forceinline__ void stage_rows(const DecodeParams &P, const uint8_t *plane, int g,
                                           int p, int c0, int kmax, __half *tile, int lane) {
    constexpr int UPR = HD / 8;  // 16-byte units per row
    constexpr int STRIDE = HD + 8;
#pragma unroll 4
    for (int uu = lane; uu < kChunk * UPR; uu += 32) {
        const int k = uu / UPR;
        const int e0 = (uu % UPR) * 8;
        const int key = min(c0 + k, kmax);
        uint4 v;
        if (P.fmt == 0) {
            const float4 *src = reinterpret_cast<const float4 *>(
                plane + P.body_off + ((static_cast<size_t>(g) * P.max_seq + key) * HD + e0) * 4);
            const float4 a = __ldg(src), b = __ldg(src + 1);
            v = make_uint4(pack_half2(a.x, a.y), pack_half2(a.z, a.w), pack_half2(b.x, b.y),
                           pack_half2(b.z, b.w));
        } else if (key < P.shadow_sink) {
            v = __ldg(reinterpret_cast<const uint4 *>(
                plane + P.sink_off + ((static_cast<size_t>(g) * kSinkMax + key) * HD + e0) * 2));
        } else if (P.shadow_win > 0 && key > p - P.shadow_win) {
            v = __ldg(reinterpret_cast<const uint4 *>(
                plane + P.ring_off +
                ((static_cast<size_t>(g) * kRingRows + (key % kRingRows)) * HD + e0) * 2));
        } else {
            const uint8_t *row =
                plane + P.body_off + (static_cast<size_t>(g) * P.max_seq + key) * P.row_bytes;
            const int b = e0 / kQ4Block, j0 = e0 % kQ4Block;
            const uint8_t *blk = row + b * kQ4BlockBytes;
            const float d = __half2float(__ushort_as_half(__ldg(reinterpret_cast<const uint16_t *>(blk))));
            const uint16_t *cb = reinterpret_cast<const uint16_t *>(blk + 2 + (j0 & 15));
            const int sh = (j0 >= 16) ? 4 : 0;
            uint32_t h[4];
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
                const uint32_t w = __ldg(cb + k2);
                const int c0v = static_cast<int>((w >> sh) & 15u) - 8;
                const int c1v = static_cast<int>((w >> (8 + sh)) & 15u) - 8;
                h[k2] = pack_half2(static_cast<float>(c0v) * d, static_cast<float>(c1v) * d);
            }
            v = make_uint4(h[0], h[1], h[2], h[3]);
        }
        *reinterpret_cast<uint4 *>(tile + k * STRIDE + e0) = v;
    }
}

template <int HD, int NT>
__global__ void __launch_bounds__(kWarps * 32) decode_kernel(const DecodeParams P) {
    constexpr int STRIDE = HD + 8;
    constexpr int MT = HD / 16;
    extern __shared__ __align__(16) uint8_t dsmem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, t = lane & 3;
    const int e = blockIdx.x, g = blockIdx.y, u = blockIdx.z;
    const int G = P.Hq / P.Hkv;

    if (e == 0 && g == 0 && u == 0 && threadIdx.x == 0) {
        P.ws_header[0] = kDecodeMagic;
        P.ws_header[1] = static_cast<uint32_t>(P.nslots);
        P.ws_header[2] = static_cast<uint32_t>(P.Hq);
        P.ws_header[3] = static_cast<uint32_t>(HD);
        P.ws_header[4] = static_cast<uint32_t>(P.entries);
    }

    const int p = P.pos[u];
    int k_lo = 0, k_hi = 0;
    if (p < 0 || p >= P.max_seq) {
        if (threadIdx.x == 0 && e == 0 && g == 0) flag_error(P.err, FA_ERRBIT_DEVICE);
    } else {
        int split_len;
        const int ns = dec_plan(p + 1, P.split_keys, P.max_splits, &split_len);
        const int s_lo = e * P.cpc, s_hi = min(ns, s_lo + P.cpc);
        if (s_lo < s_hi) {
            k_lo = s_lo * split_len;
            k_hi = min(p + 1, s_hi * split_len);
        }
    }
    const size_t head0 = static_cast<size_t>(u) * P.Hq + static_cast<size_t>(g) * G;
    if (k_lo >= k_hi) {  // empty entry
        for (int hh = threadIdx.x; hh < G; hh += blockDim.x) {
            P.ws_m[(head0 + hh) * P.stride + e] = -INFINITY;
            P.ws_l[(head0 + hh) * P.stride + e] = 0.0f;
        }
        return;
    }

    __half *tk = reinterpret_cast<__half *>(dsmem) + warp * 2 * kChunk * STRIDE;
    __half *tv = tk + kChunk * STRIDE;
    const uint8_t *kplane = P.k_planes + static_cast<size_t>(u) * P.plane_bytes;
    const uint8_t *vplane = P.v_planes + static_cast<size_t>(u) * P.plane_bytes;

    // Q^T fragments (B operand): head nt*8 + r, dims 16kk + 2t + {0,1} and + {8,9}.
    uint32_t qb[NT][MT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int hh = nt * 8 + r;
        const float *qr = P.q + (head0 + (hh < G ? hh : 0)) * HD;
#pragma unroll
        for (int kk = 0; kk < MT; ++kk) {
            const int d0 = 16 * kk + 2 * t;
            if (hh < G) {
                const float2 a = *reinterpret_cast<const float2 *>(qr + d0);
                const float2 b = *reinterpret_cast<const float2 *>(qr + d0 + 8);
                qb[nt][kk][0] = pack_half2(a.x, a.y);
                qb[nt][kk][1] = pack_half2(b.x, b.y);
            } else {
                qb[nt][kk][0] = 0u;
                qb[nt][kk][1] = 0u;
            }
        }
    }

    float o[MT][NT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) o[mt][nt][k] = 0.0f;
    float m_used[NT][2], m_true[NT][2], lsum[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            m_used[nt][k] = -INFINITY;
            m_true[nt][k] = -INFINITY;
            lsum[nt][k] = 0.0f;
        }

    const uint32_t tk_s = smem_u32(tk), tv_s = smem_u32(tv);
    for (int c0 = k_lo + kChunk * warp; c0 < k_hi; c0 += kChunk * kWarps) {
        if (P.win > 0 && !(c0 < P.sink || c0 + kChunk - 1 >= p - P.win + 1)) continue;
        stage_rows<HD>(P, kplane, g, p, c0, k_hi - 1, tk, lane);
        stage_rows<HD>(P, vplane, g, p, c0, k_hi - 1, tv, lane);
        __syncwarp();

        float sacc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) sacc[nt][k] = 0.0f;
        {
            const int row = lane & 15, col = (lane >> 4) * 8;
#pragma unroll
            for (int kk = 0; kk < MT; ++kk) {
                uint32_t a[4];
                ldmatrix_x4(a, tk_s + (row * STRIDE + 16 * kk + col) * 2);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_16816(sacc[nt], a, qb[nt][kk]);
            }
        }
        const int keyA = c0 + r, keyB = c0 + r + 8;
        const bool visA = keyA < k_hi && key_visible(p, keyA, P.sink, P.win);
        const bool visB = keyB < k_hi && key_visible(p, keyB, P.sink, P.win);
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float pa[2], pbv[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float sA = visA ? sacc[nt][hh] : -INFINITY;
                const float sB = visB ? sacc[nt][2 + hh] : -INFINITY;
                float mx = fmaxf(sA, sB);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float mx2 = mx * P.sl2;
                m_true[nt][hh] = fmaxf(m_true[nt][hh], mx2);
                const float m_new = fmaxf(m_used[nt][hh], mx2);
                if (m_new > m_used[nt][hh] + 8.0f) {
                    const float corr = ex2(m_used[nt][hh] - m_new);
                    lsum[nt][hh] *= corr;
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        o[mt][nt][hh] *= corr;
                        o[mt][nt][2 + hh] *= corr;
                    }
                    m_used[nt][hh] = m_new;
                }
                const float mref = (m_used[nt][hh] == -INFINITY) ? 0.0f : m_used[nt][hh];
                pa[hh] = ex2(fmaf(sA, P.sl2, -mref));
                pbv[hh] = ex2(fmaf(sB, P.sl2, -mref));
                lsum[nt][hh] += pa[hh] + pbv[hh];
            }
            // rows = keys, cols = heads 2t, 2t+1  ->  transpose to B fragments
            pb[nt][0] = movmatrix_trans(pack_half2(pa[0], pa[1]));
            pb[nt][1] = movmatrix_trans(pack_half2(pbv[0], pbv[1]));
        }
        {
            // V^T A fragments: matrix q of ldmatrix.x4.trans reads keys
            // 8*(q>>1) .. +7 at dims 16mt + 8*(q&1).
            const int key = (lane & 7) + ((lane >> 4) << 3);
            const int col = ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t a[4];
                ldmatrix_x4_trans(a, tv_s + (key * STRIDE + 16 * mt + col) * 2);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_16816(o[mt][nt], a, pb[nt]);
            }
        }
        __syncwarp();
    }

    // per-head sums over the 8 lanes that share t
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float v = lsum[nt][hh];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            lsum[nt][hh] = v;
        }

    // ---- merge the 4 warps: per warp m_used, m_true, l [16] and O [16][HD]
    __syncthreads();
    float *sm_mu = reinterpret_cast<float *>(dsmem);      // [kWarps][16]
    float *sm_mt = sm_mu + kWarps * 16;                   // [kWarps][16]
    float *sm_l = sm_mt + kWarps * 16;                    // [kWarps][16]
    float *sm_f = sm_l + kWarps * 16;                     // [kWarps][16] weights
    float *sm_o = sm_f + kWarps * 16;                     // [kWarps][16][HD]
    if (r == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int head = nt * 8 + 2 * t + hh;
                sm_mu[warp * 16 + head] = m_used[nt][hh];
                sm_mt[warp * 16 + head] = m_true[nt][hh];
                sm_l[warp * 16 + head] = lsum[nt][hh];
            }
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int head = nt * 8 + 2 * t + (k & 1);
                const int dim = 16 * mt + r + ((k >> 1) << 3);
                sm_o[(warp * 16 + head) * HD + dim] = o[mt][nt][k];
            }
    __syncthreads();
    if (threadIdx.x < G) {
        const int head = threadIdx.x;
        float M = -INFINITY;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_mt[w * 16 + head]);
        float L = 0.0f;
        for (int w = 0; w < kWarps; ++w) {
            const float mu = sm_mu[w * 16 + head];
            const float f = (mu == -INFINITY || M == -INFINITY) ? 0.0f : ex2(mu - M);
            sm_f[w * 16 + head] = f;
            L += f * sm_l[w * 16 + head];
        }
        // natural-log reference: s * scale = (s * scale * log2 e) * ln 2
        P.ws_m[(head0 + head) * P.stride + e] = (M == -INFINITY) ? -INFINITY : M * 0.69314718055994531f;
        P.ws_l[(head0 + head) * P.stride + e] = L;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * HD; idx += blockDim.x) {
        const int head = idx / HD, dim = idx % HD;
        float a = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) a += sm_f[w * 16 + head] * sm_o[(w * 16 + head) * HD + dim];
        P.ws_acc[((head0 + head) * P.stride + e) * HD + dim] = a;
    }
}

// One warp per (slot, q head): ascending merge of the entries.
template <int HD>
__global__ void __launch_bounds__(128)
    combine_kernel(const uint32_t *__restrict__ header, const float *__restrict__ ws_m,
                   const float *__restrict__ ws_l, const float *__restrict__ ws_acc,
                   float *__restrict__ out, int nslots, int Hq, int stride, unsigned *err) {
    constexpr int PER = HD / 32;  // dims per lane
    const int lane = threadIdx.x & 31;
    const long long head = blockIdx.x * 4LL + (threadIdx.x >> 5);
    if (head >= static_cast<long long>(nslots) * Hq) return;
    if (header[0] != kDecodeMagic || header[1] != static_cast<uint32_t>(nslots) ||
        header[2] != static_cast<uint32_t>(Hq) || header[3] != static_cast<uint32_t>(HD)) {
        if (head == 0 && lane == 0) flag_error(err, FA_ERRBIT_DEVICE);
        return;
    }
    const int E = static_cast<int>(header[4]);
    if (E < 1 || E > stride) {
        if (head == 0 && lane == 0) flag_error(err, FA_ERRBIT_DEVICE);
        return;
    }
    const float *m = ws_m + head * stride;
    const float *l = ws_l + head * stride;
    float M = -INFINITY;
    for (int i = lane; i < E; i += 32) M = fmaxf(M, m[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (M == -INFINITY) {
        if (lane == 0) flag_error(err, FA_ERRBIT_DEVICE);
        return;
    }
    float acc[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) acc[k] = 0.0f;
    float L = 0.0f;
    for (int i = 0; i < E; ++i) {
        const float mi = m[i];
        if (mi == -INFINITY) continue;
        const float w = ex2((mi - M) * 1.4426950408889634f);
        L += w * l[i];
        const float *a = ws_acc + (head * stride + i) * HD + lane * PER;
#pragma unroll
        for (int k = 0; k < PER; k += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(a + k);
            acc[k] += w * v.x;
            acc[k + 1] += w * v.y;
            acc[k + 2] += w * v.z;
            acc[k + 3] += w * v.w;
        }
    }
    const float inv = 1.0f / L;
    float *dst = out + head * HD + lane * PER;
#pragma unroll
    for (int k = 0; k < PER; k += 4)
        *reinterpret_cast<float4 *>(dst + k) =
            make_float4(acc[k] * inv, acc[k + 1] * inv, acc[k + 2] * inv, acc[k + 3] * inv);
}

template <int HD, int NT>
cudaError_t launch_decode_t(const DecodeParams &P, cudaStream_t stream) {
    const size_t tiles = static_cast<size_t>(kWarps) * 2 * kChunk * (HD + 8) * 2;
    const size_t merge = static_cast<size_t>(kWarps) * 16 * (4 + HD) * 4;
    const size_t smem = tiles > merge ? tiles : merge;
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<HD, NT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(P.entries, P.Hkv, P.nslots);
    decode_kernel<HD, NT><<<grid, kWarps * 32, smem, stream>>>(P);
    return cudaGetLastError();
}

}  // namespace

size_t decode_ws_bytes(int nslots, int n_q_heads, int head_dim, int max_splits) {
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t heads = static_cast<size_t>(nslots) * n_q_heads;
    return 256 + 2 * up(heads * max_splits * 4) + up(heads * max_splits * head_dim * 4);
}

void decode_ws_carve(void *ws, int nslots, int n_q_heads, int head_dim, int max_splits,
                     DecodeWs *out) {
    (void)head_dim;
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t heads = static_cast<size_t>(nslots) * n_q_heads;
    uint8_t *b = static_cast<uint8_t *>(ws);
    out->header = reinterpret_cast<uint32_t *>(b);
    out->m = reinterpret_cast<float *>(b + 256);
    out->l = reinterpret_cast<float *>(b + 256 + up(heads * max_splits * 4));
    out->acc = reinterpret_cast<float *>(b + 256 + 2 * up(heads * max_splits * 4));
    out->stride = max_splits;
}

cudaError_t launch_decode(const DecodeArgs &a, const DecodeWs &ws, unsigned *err,
                          cudaStream_t stream) {
    DecodeParams P;
    P.q = a.q;
    P.k_planes = a.k_planes;
    P.v_planes = a.v_planes;
    P.pos = a.pos;
    P.ws_m = ws.m;
    P.ws_l = ws.l;
    P.ws_acc = ws.acc;
    P.ws_header = ws.header;
    P.nslots = a.nslots;
    P.Hq = a.n_q_heads;
    P.Hkv = a.n_kv_heads;
    P.max_seq = a.g.max_seq;
    P.sink = a.sink;
    P.win = a.win;
    P.fmt = a.g.fmt;
    P.shadow_sink = a.shadow_sink;
    P.shadow_win = a.shadow_win;
    P.split_keys = a.split_keys;
    P.max_splits = a.max_splits;
    P.cpc = ws.splits_per_cta;
    P.entries = ws.entries;
    P.stride = ws.stride;
    P.plane_bytes = a.g.bytes;
    P.body_off = a.g.body_off;
    P.row_bytes = a.g.row_bytes;
    P.sink_off = a.g.sink_off;
    P.ring_off = a.g.ring_off;
    P.sl2 = a.scale * 1.4426950408889634f;
    P.err = err;
    const int G = a.n_q_heads / a.n_kv_heads;
    const bool two = G > 8;
    switch (a.g.hd) {
        case 64: return two ? launch_decode_t<64, 2>(P, stream) : launch_decode_t<64, 1>(P, stream);
        case 128: return two ? launch_decode_t<128, 2>(P, stream) : launch_decode_t<128, 1>(P, stream);
        case 256: return two ? launch_decode_t<256, 2>(P, stream) : launch_decode_t<256, 1>(P, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_combine(const void *workspace, float *out, int nslots, int n_q_heads,
                           int head_dim, int max_splits, unsigned *err, cudaStream_t stream) {
    DecodeWs ws;
    decode_ws_carve(const_cast<void *>(workspace), nslots, n_q_heads, head_dim, max_splits, &ws);
    const long long heads = static_cast<long long>(nslots) * n_q_heads;
    const int blocks = static_cast<int>((heads + 3) / 4);
    switch (head_dim) {
        case 64:
            combine_kernel<64><<<blocks, 128, 0, stream>>>(ws.header, ws.m, ws.l, ws.acc, out,
                                                           nslots, n_q_heads, ws.stride, err);
            break;
        case 128:
            combine_kernel<128><<<blocks, 128, 0, stream>>>(ws.header, ws.m, ws.l, ws.acc, out,
                                                            nslots, n_q_heads, ws.stride, err);
            break;
        case 256:
            combine_kernel<256><<<blocks, 128, 0, stream>>>(ws.header, ws.m, ws.l, ws.acc, out,
                                                            nslots, n_q_heads, ws.stride, err);
            break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace fa
