// decode.cu -- multi-slot split-KV decode and its log-sum-exp combine
// ("attention.cu" (Foundry cuda_kernels), "Decode-mode flash attention" and
// "Multi-user decode attention": fc_attn_dec_plan, fc_attn_flash_decode_slots,
// fc_attn_flash_decode_combine).
//
// Decode reads every cached key once per (slot, kv head) and does 2 x G x hd
// multiply-adds per key; at 288 bytes per key (K+V, Q4_0, hd 256) and G = 8
// that is about 28 flop/byte, more than the CUDA cores sustain at HBM speed,
// so both contractions run on the warp-level tensor-core path
// (mma.sync.m16n8k16, fp16 in, fp32 accumulate):
//   S^T (16 keys x 8 heads) = K (16 x hd) . Q^T
//   O^T (hd x 8 heads)     += V^T (hd x 16 keys) . P^T
// The 8 query heads sharing a kv head are the n8 dimension, so each K/V row is
// read once for the group; P^T is formed in registers with movmatrix. tcgen05
// is not used here: its smallest M is 64 and this work is bound by memory and
// by the dequantisation, not by the MMA rate.
//
// Two kernels write the same partials (m, l, acc per slot, q head, entry):
//  * decode_q4_kernel (Q4_0 cache, group <= 8): 4 pairs of warps per block,
//    each pair a QK warp and a PV warp with their own rings of raw Q4_0 K and
//    V tiles (32 keys, one bulk copy each); nibbles become fp16 MMA operands in
//    registers. For K the operand is 1024 + c (one LOP3) and the
//    -1032 * sum(q) bias of each 32-element block is preloaded into a fresh
//    accumulator, then scaled by the block's d; for V the operand is 1024 + c
//    (or + 16 c) with a constant-operand MMA removing the offset, and d is
//    folded into P. Keys held as fp16 shadows (sinks, recent ring) are left to
//    one extra entry per (slot, kv head), run by the generic path.
//  * decode_kernel (fp32 caches, group 16, and that shadow entry): stages
//    16-key fp16 tiles in shared memory, reads fragments with ldmatrix.
// Each block merges its warps; fa_decode_combine merges the entries.
#include "decode_common.cuh"
#include "decode_softmax.cuh"
#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kWarps = 4;
constexpr int kChunk = 16;     // keys per step of the generic path
// Lazy rescale threshold (log2 units) of the running max: O and l keep a
// stale reference until the max grows past it. In the Q4_0 path P is
// multiplied by the block scale d in fp16, so P <= 2^2 keeps P*d finite for
// any |d| < 8192 (inputs within the fp16 range).
constexpr float kRescaleGeneric = 8.0f;
constexpr float kRescaleQ4 = 2.0f;

__device__ __forceinline__ int dec_plan(int seq_len, int kps, int cap, int *split_len) {
    int ns = (seq_len + kps - 1) / kps;
    ns = ns < 1 ? 1 : (ns > cap ? cap : ns);
    int sl = (seq_len + ns - 1) / ns;
    sl = (sl + 15) & ~15;
    *split_len = sl;
    return (seq_len + sl - 1) / sl;
}

// Is key s read from an fp16 shadow copy by the decode query at p?
__device__ __forceinline__ bool is_shadow_key(const DecodeParams &P, int p, int s) {
    return P.fmt == kFmtQ4 && (s < P.shadow_sink || (P.shadow_win > 0 && s > p - P.shadow_win));
}

__device__ __forceinline__ void write_empty(const DecodeParams &P, size_t head0, int G, int e) {
    for (int hh = threadIdx.x; hh < G; hh += blockDim.x) {
        P.ws_m[(head0 + hh) * P.stride + e] = -INFINITY;
        P.ws_l[(head0 + hh) * P.stride + e] = 0.0f;
    }
}

// Merge of a block's kWarps online-softmax states ("slots") into the block's
// partial. Slot w holds m_used, m_true, lsum of heads nt*8 + 2t + {0,1}
// (exp2 domain; lsum summed over the warp) and O^T rows r (k < 2) and r+8
// (k >= 2) of m-tile mt, heads nt*8 + 2t + (k & 1). The stats and O of a slot
// may come from different warps; merge_finish is called by every thread.
__device__ __forceinline__ float *merge_buf(uint8_t *dsmem) { return reinterpret_cast<float *>(dsmem); }

template <int NT>
__device__ __forceinline__ void merge_write_stats(uint8_t *dsmem, int slot,
                                                  const float (&m_used)[NT][2],
                                                  const float (&m_true)[NT][2],
                                                  const float (&lsum)[NT][2]) {
    const int lane = threadIdx.x & 31, r = lane >> 2, t = lane & 3;
    float *sm_mu = merge_buf(dsmem), *sm_mt = sm_mu + kWarps * 16, *sm_l = sm_mt + kWarps * 16;
    if (r == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int head = nt * 8 + 2 * t + hh;
                sm_mu[slot * 16 + head] = m_used[nt][hh];
                sm_mt[slot * 16 + head] = m_true[nt][hh];
                sm_l[slot * 16 + head] = lsum[nt][hh];
            }
    }
}

// Q4ROWS: the Q4_0 path's m-tile 2b + j rows r, r+8 hold elements 2r + j,
// 16 + 2r + j of block b; otherwise rows are in natural order.
template <int HD, int NT, bool Q4ROWS>
__device__ __forceinline__ void merge_write_o(uint8_t *dsmem, int slot,
                                              const float (&o)[HD / 16][NT][4]) {
    constexpr int MT = HD / 16;
    const int lane = threadIdx.x & 31, r = lane >> 2, t = lane & 3;
    float *sm_o = merge_buf(dsmem) + 4 * kWarps * 16;  // [kWarps][16][HD]
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int head = nt * 8 + 2 * t + (k & 1);
                const int dim = Q4ROWS ? 32 * (mt >> 1) + 16 * (k >> 1) + 2 * r + (mt & 1)
                                       : 16 * mt + r + ((k >> 1) << 3);
                sm_o[(slot * 16 + head) * HD + dim] = o[mt][nt][k];
            }
}

template <int HD>
__device__ __forceinline__ void merge_finish(const DecodeParams &P, uint8_t *dsmem, size_t head0,
                                             int G, int e) {
    float *sm_mu = merge_buf(dsmem), *sm_mt = sm_mu + kWarps * 16, *sm_l = sm_mt + kWarps * 16;
    float *sm_f = sm_l + kWarps * 16, *sm_o = sm_f + kWarps * 16;
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
        P.ws_m[(head0 + head) * P.stride + e] =
            (M == -INFINITY) ? -INFINITY : M * 0.69314718055994531f;
        P.ws_l[(head0 + head) * P.stride + e] = L;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * HD; idx += blockDim.x) {
        const int head = idx / HD, dim = idx % HD;
        bool any = false;
        for (int w = 0; w < kWarps; ++w) any |= sm_mt[w * 16 + head] != -INFINITY;
        if (!any) continue;  // empty for this head: acc is never read
        float a = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) a += sm_f[w * 16 + head] * sm_o[(w * 16 + head) * HD + dim];
        P.ws_acc[((head0 + head) * P.stride + e) * HD + dim] = a;
    }
}

// ============================================================ generic path

// Stage the fp16 values of keys [c0, c0+16) (clamped to kmax) of one K or V
// plane into a [16][HD+8] fp16 tile; the read rule picks the fp16 sink, the
// fp16 ring, the Q4_0 body, the fp32 body (rounded), the fp16 body, or the
// fp8 body times the plane's scale c (rounded).
template <int HD>
__device__ __forceinline__ void stage_rows(const DecodeParams &P, const uint8_t *plane, int g,
                                           int p, int c0, int kmax, __half *tile, int lane,
                                           float c) {
    constexpr int UPR = HD / 8;  // 16-byte units per row
    constexpr int STRIDE = HD + 8;
#pragma unroll 4
    for (int uu = lane; uu < kChunk * UPR; uu += 32) {
        const int k = uu / UPR;
        const int e0 = (uu % UPR) * 8;
        const int key = min(c0 + k, kmax);
        uint4 v;
        const size_t elem = (static_cast<size_t>(g) * P.max_seq + key) * HD + e0;
        if (P.fmt == kFmtF32) {
            const float4 *src = reinterpret_cast<const float4 *>(plane + P.body_off + elem * 4);
            const float4 a = __ldg(src), b = __ldg(src + 1);
            v = make_uint4(pack_half2(a.x, a.y), pack_half2(a.z, a.w), pack_half2(b.x, b.y),
                           pack_half2(b.z, b.w));
        } else if (P.fmt == kFmtF16) {
            v = __ldg(reinterpret_cast<const uint4 *>(plane + P.body_off + elem * 2));
        } else if (P.fmt == kFmtFp8) {
            v = fp8x8_to_half8_scaled(__ldg(reinterpret_cast<const uint2 *>(plane + P.body_off + elem)),
                                      c);
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

// Generic body: 16-key chunks of the given key ranges, round-robin over the
// warps. With shadow_only, keys that are not fp16 shadows are masked (they
// belong to the Q4_0 path).
template <int HD, int NT>
__device__ __forceinline__ void generic_body(const DecodeParams &P, uint8_t *dsmem, int e, int g,
                                             int u, int p, int lo0, int hi0, int lo1, int hi1,
                                             bool shadow_only) {
    constexpr int STRIDE = HD + 8;
    constexpr int MT = HD / 16;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, t = lane & 3;
    const int G = P.Hq / P.Hkv;
    const size_t head0 = static_cast<size_t>(u) * P.Hq + static_cast<size_t>(g) * G;

    __half *tk = reinterpret_cast<__half *>(dsmem) + warp * 2 * kChunk * STRIDE;
    __half *tv = tk + kChunk * STRIDE;
    const uint8_t *kplane = P.k_planes + static_cast<size_t>(u) * P.plane_bytes;
    const uint8_t *vplane = P.v_planes + static_cast<size_t>(u) * P.plane_bytes;
    float kscale = 1.0f, vscale = 1.0f;
    if (P.fmt == kFmtFp8) {
        kscale = __ldg(reinterpret_cast<const float *>(kplane + P.scale_off));
        vscale = __ldg(reinterpret_cast<const float *>(vplane + P.scale_off));
    }

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
    const int n0 = max(0, hi0 - lo0 + kChunk - 1) / kChunk;
    const int n1 = max(0, hi1 - lo1 + kChunk - 1) / kChunk;
    // blocks with more than kWarps warps: the extra warps only join the merge
    for (int ci = warp; warp < kWarps && ci < n0 + n1; ci += kWarps) {
        const bool first = ci < n0;
        const int c0 = first ? lo0 + kChunk * ci : lo1 + kChunk * (ci - n0);
        const int k_hi = first ? hi0 : hi1;
        if (P.win > 0 && !(c0 < P.sink || c0 + kChunk - 1 >= p - P.win + 1)) continue;
        stage_rows<HD>(P, kplane, g, p, c0, k_hi - 1, tk, lane, kscale);
        stage_rows<HD>(P, vplane, g, p, c0, k_hi - 1, tv, lane, vscale);
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
        bool visA = keyA < k_hi && key_visible(p, keyA, P.sink, P.win);
        bool visB = keyB < k_hi && key_visible(p, keyB, P.sink, P.win);
        if (shadow_only) {
            visA = visA && is_shadow_key(P, p, keyA);
            visB = visB && is_shadow_key(P, p, keyB);
        }
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float sv[2][2], pv[2][2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                sv[hh][0] = visA ? sacc[nt][hh] : -INFINITY;
                sv[hh][1] = visB ? sacc[nt][2 + hh] : -INFINITY;
            }
            fold_scores<MT, NT, 2>(sv, P.sl2, kRescaleGeneric, m_used[nt][0], m_used[nt][1],
                                   m_true[nt][0], m_true[nt][1], lsum[nt][0], lsum[nt][1], o, nt,
                                   pv);
            // rows = keys, cols = heads 2t, 2t+1  ->  transpose to B fragments
            pb[nt][0] = movmatrix_trans(pack_half2(pv[0][0], pv[1][0]));
            pb[nt][1] = movmatrix_trans(pack_half2(pv[0][1], pv[1][1]));
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
    __syncthreads();  // the merge buffer overlaps the staging tiles
    if (warp < kWarps) {
        merge_write_stats<NT>(dsmem, warp, m_used, m_true, lsum);
        merge_write_o<HD, NT, false>(dsmem, warp, o);
    }
    merge_finish<HD>(P, dsmem, head0, G, e);
}

__device__ __forceinline__ void write_header(const DecodeParams &P, int hd) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0) {
        P.ws_header[0] = kDecodeMagic;
        P.ws_header[1] = static_cast<uint32_t>(P.nslots);
        P.ws_header[2] = static_cast<uint32_t>(P.Hq);
        P.ws_header[3] = static_cast<uint32_t>(hd);
        P.ws_header[4] = static_cast<uint32_t>(P.entries);
    }
}

// Key range of body entry e of slot u: the run of plan splits [e*cpc, ...).
__device__ __forceinline__ bool entry_range(const DecodeParams &P, int e, int p, int *k_lo,
                                            int *k_hi) {
    int split_len;
    const int ns = dec_plan(p + 1, P.split_keys, P.max_splits, &split_len);
    const int s_lo = e * P.cpc, s_hi = min(ns, s_lo + P.cpc);
    if (s_lo >= s_hi) return false;
    *k_lo = s_lo * split_len;
    *k_hi = min(p + 1, s_hi * split_len);
    return *k_lo < *k_hi;
}

// Shadow entry: the fp16 sink rows and the fp16 ring rows the query reads.
template <int HD, int NT>
__device__ __forceinline__ void shadow_entry(const DecodeParams &P, uint8_t *dsmem, int e, int g,
                                             int u, int p) {
    const int G = P.Hq / P.Hkv;
    const size_t head0 = static_cast<size_t>(u) * P.Hq + static_cast<size_t>(g) * G;
    const int lo0 = 0, hi0 = min(P.shadow_sink, p + 1);
    int lo1 = 0, hi1 = 0;
    if (P.shadow_win > 0) {
        lo1 = max(hi0, p - P.shadow_win + 1);
        hi1 = p + 1;
    }
    if (hi0 <= lo0 && hi1 <= lo1) {
        write_empty(P, head0, G, e);
        return;
    }
    generic_body<HD, NT>(P, dsmem, e, g, u, p, lo0, hi0, lo1, hi1, true);
}

template <int HD, int NT>
__global__ void __launch_bounds__(kWarps * 32) decode_kernel(const DecodeParams P) {
    extern __shared__ __align__(128) uint8_t dsmem[];
    const int e = blockIdx.x, g = blockIdx.y, u = blockIdx.z;
    const int G = P.Hq / P.Hkv;
    write_header(P, HD);
    const int p = P.pos[u];
    const size_t head0 = static_cast<size_t>(u) * P.Hq + static_cast<size_t>(g) * G;
    if (p < 0 || p >= P.max_seq) {
        if (threadIdx.x == 0 && e == 0 && g == 0) flag_error(P.err, FA_ERRBIT_DEVICE);
        write_empty(P, head0, G, e);
        return;
    }
    if (e == P.shadow_entry) {
        shadow_entry<HD, NT>(P, dsmem, e, g, u, p);
        return;
    }
    int k_lo, k_hi;
    if (!entry_range(P, e, p, &k_lo, &k_hi)) {
        write_empty(P, head0, G, e);
        return;
    }
    generic_body<HD, NT>(P, dsmem, e, g, u, p, k_lo, k_hi, 0, 0, false);
}

// ============================================================== Q4_0 path
//
// The block's 8 warps form 4 pairs; pair w walks 32-key tiles w, w+4, ... of
// the entry's key range through its own rings of raw Q4_0 K tiles and V tiles
// (one bulk copy each). Warp w (QK) scores a tile, folds it into the online
// softmax and hands P^T fragments plus the O rescale factor of that tile to
// warp w+4 (PV) through a ring of P records; warp w+4 multiplies them into O.
// Each warp copies the tiles it reads (lane 0, one bulk copy per tile): the QK
// warp a K tile as soon as it has scored the tile before it in that stage, the
// PV warp a V tile as soon as it has finished the tile before it in that
// stage. So a stage frees without a barrier between the warps, and the QK
// warp, which sets the pace, does no V bookkeeping.
constexpr int kTileKeys = 32;  // keys per tile
constexpr int kPairs = 4;      // warp pairs per block
constexpr int kPRing = 2;      // P records in flight per pair
// Pipeline depths (K tiles and V tiles per pair) and residency (blocks per SM).
#ifndef FA_Q4_KSTAGES
#define FA_Q4_KSTAGES 2
#endif
#ifndef FA_Q4_VSTAGES
#define FA_Q4_VSTAGES 2
#endif
#ifndef FA_Q4_MIN_BLOCKS
#define FA_Q4_MIN_BLOCKS 2
#endif
// Unroll factor (1 or 2) of the PV warp's loop over a tile's two 16-key
// halves: 2 interleaves the halves' dependency chains, 1 keeps the registers
// and the code small. (The QK warp walks the blocks outermost and both halves
// inside, so that a block's Q fragments are read once per tile.)
#ifndef FA_Q4_PV_HALVES
#define FA_Q4_PV_HALVES 2
#endif
constexpr int kPVHalves = FA_Q4_PV_HALVES;
// Unroll factor of the QK warp's loop over pairs of 32-element blocks (an even
// and an odd block per iteration; head_dim / 64 pairs): the full unroll gives
// the scheduler the most independent work, a partial one smaller code.
#ifndef FA_Q4_QK_PAIR_UNROLL
#define FA_Q4_QK_PAIR_UNROLL 4
#endif
constexpr int kQKPairUnroll = FA_Q4_QK_PAIR_UNROLL;

template <int HD>
struct Q4Cfg {
    static constexpr int NK = FA_Q4_KSTAGES;
    static constexpr int NV = FA_Q4_VSTAGES;
    static constexpr int NB = HD / kQ4Block;                  // blocks per row
    static constexpr int MT = HD / 16;                        // m16 tiles of head_dim
    static constexpr int ROWB = NB * kQ4BlockBytes;           // bytes per row
    static constexpr int TILE = kTileKeys * ROWB;             // bytes of K (or V) per stage
    static constexpr int TILE_ALLOC = (TILE + 127) / 128 * 128;
    // P record: [32 lanes] {P^T b0, b1 of keys 0-15, b0, b1 of keys 16-31},
    // then [32 lanes] {rescale of head 2t, of head 2t+1, tile index, 0}
    static constexpr int PREC = 2 * 32 * 16;
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = NK * TILE_ALLOC;
    static constexpr int P_OFF = (NK + NV) * TILE_ALLOC;
    static constexpr int PAIR_BYTES = P_OFF + kPRing * PREC;
    // Q^T fragments [NB][32 lanes] uint4 and block biases [NB][32 lanes]
    // float4, shared by the block's QK warps (one slot, one kv head)
    static constexpr int QF_OFF = kPairs * PAIR_BYTES;
    static constexpr int QB_OFF = QF_OFF + NB * 32 * 16;
    static constexpr int BAR_OFF = QB_OFF + NB * 32 * 16;
    // per pair: kfull[NK], vfull[NV], pfull[kPRing], pempty[kPRing]
    static constexpr int BARS_PER_PAIR = NK + NV + 2 * kPRing;
    static constexpr int SMEM_PIPE = BAR_OFF + kPairs * BARS_PER_PAIR * 8 + 16;
    static constexpr int SMEM_GENERIC = kWarps * 2 * kChunk * (HD + 8) * 2;
    static constexpr int SMEM_MERGE = kWarps * 16 * (4 + HD) * 4;
    static constexpr int SMEM = SMEM_PIPE > SMEM_GENERIC
                                    ? (SMEM_PIPE > SMEM_MERGE ? SMEM_PIPE : SMEM_MERGE)
                                    : (SMEM_GENERIC > SMEM_MERGE ? SMEM_GENERIC : SMEM_MERGE);
    static_assert(NB % 2 == 0, "head_dim must be a multiple of 64");
    static_assert(NK >= 1 && NV >= 2, "pipeline depths");
    static_assert(TILE_ALLOC % 128 == 0 && PAIR_BYTES % 16 == 0 && BAR_OFF % 8 == 0, "alignment");
};

__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
    __half2 x = *reinterpret_cast<__half2 *>(&a), y = *reinterpret_cast<__half2 *>(&b);
    x = __hmul2(x, y);
    return *reinterpret_cast<uint32_t *>(&x);
}

// (x & MASK) | magic in one LOP3; magic is passed in a register so that the
// two constants need not both be encoded in the instruction.
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t x, uint32_t magic) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "n"(MASK), "r"(magic));
    return d;
}
// A value the compiler must keep in a register rather than re-materialise.
__device__ __forceinline__ uint32_t opaque(uint32_t x) {
    asm volatile("" : "+r"(x));
    return x;
}
constexpr uint32_t kMagic = 0x64006400u;     // fp16 pair (1024, 1024)
constexpr uint32_t kHNeg1032 = 0xE408E408u;  // fp16 pair (-1032, -1032)
constexpr uint32_t kHNeg1152 = 0xE480E480u;  // fp16 pair (-1152, -1152)

// Code bytes of block b that thread t (of 4 per row) turns into its K operand
// halves: a 32-bit word read at an aligned offset. Element order within the
// block is permuted per thread (and mirrored in Q): odd blocks give thread t
// bytes 4t..4t+3; even blocks, whose codes start 2 bytes off a word, give
// threads 0-2 bytes 2+4t..5+4t and thread 3 bytes 14, 15, 0, 1.
__host__ __device__ constexpr int q4k_elem(int b, int t, int i) {
    return (b & 1) ? 4 * t + i : (t < 3 ? 2 + 4 * t + i : (i < 2 ? 14 + i : i - 2));
}


// Q^T B fragments of kv head group head0 for blocks b = first, first + step,
// ... in the permuted order of q4k_elem: lo k-step of block b (elements
// 0..15) takes q, the hi k-step (16..31) q / 16, because the K operand there
// is 1024 + 16 c. bias = -(1032 sum_lo q + 1152 sum_hi q/16) over the fp16
// values, for heads 2t, 2t+1 (twice: the accumulator input of rows r and
// r + 8), so that a block's accumulator ends at sum q (c - 8). Heads >= G get
// q = 0.
template <int HD>
__device__ __forceinline__ void build_q_frags(const DecodeParams &P, size_t head0, int G,
                                              int first, int step, uint4 *qfrag, float4 *qbias) {
    constexpr int NB = HD / kQ4Block;
    const int lane = threadIdx.x & 31, r = lane >> 2, t = lane & 3;
    for (int b = first; b < NB; b += step) {
        const int hh = r;
        const float *qr = P.q + (head0 + (hh < G ? hh : 0)) * HD + 32 * b;
        const float sc = (hh < G) ? 1.0f : 0.0f;
        uint32_t w[4];
        float ps = 0.0f;
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
            const float f = hi ? 0.0625f : 1.0f;
            const float *qb0 = qr + 16 * hi;
            const __half2 x0 = __floats2half2_rn(sc * f * qb0[q4k_elem(b, t, 0)],
                                                 sc * f * qb0[q4k_elem(b, t, 2)]);
            const __half2 x1 = __floats2half2_rn(sc * f * qb0[q4k_elem(b, t, 1)],
                                                 sc * f * qb0[q4k_elem(b, t, 3)]);
            w[2 * hi] = *reinterpret_cast<const uint32_t *>(&x0);
            w[2 * hi + 1] = *reinterpret_cast<const uint32_t *>(&x1);
            const float2 f0 = __half22float2(x0), f1 = __half22float2(x1);
            ps += (hi ? -1152.0f : -1032.0f) * ((f0.x + f0.y) + (f1.x + f1.y));
        }
        ps += __shfl_xor_sync(0xffffffffu, ps, 1);
        ps += __shfl_xor_sync(0xffffffffu, ps, 2);  // head r's block bias
        const float b0 = __shfl_sync(0xffffffffu, ps, (2 * t) * 4);
        const float b1 = __shfl_sync(0xffffffffu, ps, (2 * t + 1) * 4);
        qfrag[b * 32 + lane] = make_uint4(w[0], w[1], w[2], w[3]);
        qbias[b * 32 + lane] = make_float4(b0, b1, b0, b1);
    }
}

// How far a warp pair's rings have run: K tiles and V tiles copied (and
// consumed), P records passed. A block initialises its barriers once and
// runs its pieces one after another through the same rings, so the stage and
// phase of each copy or record follow from these running counts.
struct Q4Ring {
    int k = 0, v = 0, r = 0;
};

// The barriers of every warp pair (one thread per pair) and the abort flag;
// the caller synchronises the block afterwards.
template <int HD>
__device__ __forceinline__ void q4_init(uint8_t *dsmem) {
    using C = Q4Cfg<HD>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0)
        *reinterpret_cast<volatile int *>(dsmem + C::BAR_OFF + kPairs * C::BARS_PER_PAIR * 8) = 0;
    if (warp < kPairs && lane == 0) {
        uint64_t *bars = reinterpret_cast<uint64_t *>(dsmem + C::BAR_OFF) + warp * C::BARS_PER_PAIR;
        for (int s = 0; s < C::NK + C::NV; ++s) mbar_init(&bars[s], 1);
        for (int s = 0; s < kPRing; ++s) {
            mbar_init(&bars[C::NK + C::NV + s], 1);           // pfull
            mbar_init(&bars[C::NK + C::NV + kPRing + s], 1);  // pempty
        }
        mbar_fence_init();
    }
}

// One piece of work: tiles j0 .. j1-1 of (slot u, kv head g) in the order of
// q4_tiles, written as partial entry e. rg: this warp's ring counts (the QK
// warp runs K and records, the PV warp V and records).
template <int HD>
__device__ __forceinline__ void q4_body(const DecodeParams &P, uint8_t *dsmem, int e, int g,
                                        int u, int p, const Q4Tiles &tl, int j0, int j1,
                                        Q4Ring &rg) {
    using C = Q4Cfg<HD>;
    constexpr int NB = C::NB, MT = C::MT, ROWB = C::ROWB, NK = C::NK, NV = C::NV;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, t = lane & 3;
    const int pair = warp & (kPairs - 1);
    const bool qk_role = warp < kPairs;
    const int G = P.Hq / P.Hkv;
    const size_t head0 = static_cast<size_t>(u) * P.Hq + static_cast<size_t>(g) * G;
    uint8_t *pbase = dsmem + pair * C::PAIR_BYTES;
    uint8_t *prec = pbase + C::P_OFF;  // P record ring
    uint4 *qfrag = reinterpret_cast<uint4 *>(dsmem + C::QF_OFF);
    float4 *qbias = reinterpret_cast<float4 *>(dsmem + C::QB_OFF);
    uint64_t *bars = reinterpret_cast<uint64_t *>(dsmem + C::BAR_OFF) + pair * C::BARS_PER_PAIR;
    uint64_t *kfull = bars, *vfull = bars + NK, *pfull = bars + NK + NV,
             *pempty = bars + NK + NV + kPRing;
    volatile int *abort =
        reinterpret_cast<volatile int *>(dsmem + C::BAR_OFF + kPairs * C::BARS_PER_PAIR * 8);

    build_q_frags<HD>(P, head0, G, warp, 2 * kPairs, qfrag, qbias);
    __syncthreads();

    const int ss = P.shadow_sink, sw = P.shadow_win;
    const int ntiles = j1 - j0;  // sequence index i is tile tl.kt(j0 + i)
    const int k_end = p + 1;     // keys past p are never read
    auto tile_key0 = [&](int i) -> int { return kTileKeys * tl.kt(j0 + i); };
    bool ok = true;
    // one bulk copy of tile i's rows (rounded up to 16 bytes) into dst
    auto issue = [&](const uint8_t *body, int i, uint8_t *dst, uint64_t *bar) {
        const int t0 = tile_key0(i);
        const int nk = min(kTileKeys, k_end - t0);
        const uint32_t bytes = (static_cast<uint32_t>(nk * ROWB) + 15u) & ~15u;
        mbar_arrive_expect_tx(bar, bytes);
        bulk_copy_g2s(dst, body + static_cast<size_t>(t0) * ROWB, bytes, bar);
    };
    // wait (bounded, ignoring the abort flag) for the last copy issued into
    // each of a ring's stages, so that no copy lands after the block is gone
    auto drain = [&](uint64_t *full, int nst, int issued) {
        for (int st = 0; st < nst; ++st)
            if (issued > st) {
                const long long c0 = clock64();
                while (!mbar_try_wait(&full[st], ((issued - 1 - st) / nst) & 1) &&
                       clock64() - c0 < kSpinCycles) {
                }
            }
    };

    if (qk_role) {
        // ================================================= QK + softmax warp
        const uint8_t *kbody = P.k_planes + static_cast<size_t>(u) * P.plane_bytes + P.body_off +
                               static_cast<size_t>(g) * P.max_seq * ROWB;
        float mu0 = -INFINITY, mu1 = -INFINITY, mt0 = -INFINITY, mt1 = -INFINITY;
        float ls0 = 0.0f, ls1 = 0.0f;
        // Prologue: the first NK K tiles (the PV warp copies the V tiles).
        int kt = pair;  // next tile index to copy
        int kn = 0;     // copies issued in this piece (ring count rg.k + kn)
        for (; kn < NK && kt < ntiles; ++kn) {
            const int st = (rg.k + kn) % NK;
            if (lane == 0) issue(kbody, kt, pbase + C::K_OFF + st * C::TILE_ALLOC, &kfull[st]);
            kt += kPairs;
        }
        const uint32_t magic = opaque(kMagic);
        int seq = 0;  // position of the tile in this pair's sequence
        for (int i = pair; i < ntiles; i += kPairs, ++seq) {
            const int s = (rg.k + seq) % NK;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&kfull[s], ((rg.k + seq) / NK) & 1, abort, P.err));
            if (!ok) break;
            const uint8_t *Ks = pbase + C::K_OFF + s * C::TILE_ALLOC;
            const int t0 = tile_key0(i);
            // ---- scores: half h2 holds keys t0 + 16 h2 + {r, r+8}; the
            // block's Q fragments and biases are read once for both halves
            float sc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll kQKPairUnroll
            for (int bp = 0; bp < NB / 2; ++bp)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int b = 2 * bp + j;
                const int o18 = kQ4BlockBytes * b;
                const uint4 qv = lds_v4(qfrag + b * 32 + lane);
                const float4 bv = lds_f4(qbias + b * 32 + lane);
                const float cb[4] = {bv.x, bv.y, bv.z, bv.w};
                const uint32_t qlo[2] = {qv.x, qv.y}, qhi[2] = {qv.z, qv.w};
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const uint8_t *KA = Ks + (16 * h2 + r) * ROWB;
                    const uint8_t *KB = KA + 8 * ROWB;
                    uint32_t wA, wB, dA, dB;
                    if (j == 0) {
                        const uint32_t a0 = *reinterpret_cast<const uint32_t *>(KA + o18 + 4 + 4 * t);
                        const uint32_t a1 = *reinterpret_cast<const uint32_t *>(KA + o18);
                        const uint32_t b0 = *reinterpret_cast<const uint32_t *>(KB + o18 + 4 + 4 * t);
                        const uint32_t b1 = *reinterpret_cast<const uint32_t *>(KB + o18);
                        const uint32_t sel = (t == 3) ? 0x7610u : 0x3210u;
                        wA = __byte_perm(a0, a1, sel);
                        wB = __byte_perm(b0, b1, sel);
                        dA = a1 & 0xFFFFu;
                        dB = b1 & 0xFFFFu;
                    } else {
                        wA = *reinterpret_cast<const uint32_t *>(KA + o18 + 2 + 4 * t);
                        wB = *reinterpret_cast<const uint32_t *>(KB + o18 + 2 + 4 * t);
                        dA = *reinterpret_cast<const uint16_t *>(KA + o18);
                        dB = *reinterpret_cast<const uint16_t *>(KB + o18);
                    }
                    const uint32_t wA8 = wA >> 8, wB8 = wB >> 8;
                    const uint32_t alo[4] = {and_or<0x000F000Fu>(wA, magic), and_or<0x000F000Fu>(wB, magic),
                                             and_or<0x000F000Fu>(wA8, magic), and_or<0x000F000Fu>(wB8, magic)};
                    const uint32_t ahi[4] = {and_or<0x00F000F0u>(wA, magic), and_or<0x00F000F0u>(wB, magic),
                                             and_or<0x00F000F0u>(wA8, magic), and_or<0x00F000F0u>(wB8, magic)};
                    float acc[4];
                    mma_16816_c(acc, alo, qlo, cb);
                    mma_16816(acc, ahi, qhi);
                    const float fA = __half2float(__ushort_as_half(static_cast<uint16_t>(dA)));
                    const float fB = __half2float(__ushort_as_half(static_cast<uint16_t>(dB)));
                    sc[h2][0] = fmaf(fA, acc[0], sc[h2][0]);
                    sc[h2][1] = fmaf(fA, acc[1], sc[h2][1]);
                    sc[h2][2] = fmaf(fB, acc[2], sc[h2][2]);
                    sc[h2][3] = fmaf(fB, acc[3], sc[h2][3]);
                }
            }
            const float *sc0 = sc[0], *sc1 = sc[1];
            // The scores consumed every byte this warp read from the stage, so
            // the stage can take the K tile NK places further on.
            __syncwarp();
            if (kt < ntiles) {
                if (lane == 0) {
                    fence_proxy_async_smem();  // those reads come before the copy's writes
                    issue(kbody, kt, pbase + C::K_OFF + s * C::TILE_ALLOC, &kfull[s]);
                }
                kt += kPairs;
                ++kn;
            }
            // ---- mask and fold: sv[hh][2 h2 + half] is key t0 + 16 h2 + r + 8 half.
            const int t1 = t0 + kTileKeys - 1;
            const bool whole = t1 < k_end && t0 >= ss && (sw <= 0 || t1 <= p - sw) &&
                               (P.win <= 0 || t0 >= p - P.win + 1);
            float sv[2][4], pv[2][4];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int key = t0 + 16 * h2 + r + 8 * half;
                    const bool vis = whole || (key < k_end && key_visible(p, key, P.sink, P.win) &&
                                               !(key < ss || (sw > 0 && key > p - sw)));
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
                        sv[hh][2 * h2 + half] = vis ? (h2 ? sc1 : sc0)[2 * half + hh] : -INFINITY;
                }
            const float old0 = mu0, old1 = mu1;
            float o_none[1][1][4] = {};  // O lives in the PV warp
            fold_scores<1, 1, 4>(sv, P.sl2, kRescaleQ4, mu0, mu1, mt0, mt1, ls0, ls1, o_none, 0, pv);
            // factor the PV warp applies to O before adding this tile (1: none)
            const float c0 = (mu0 != old0) ? ex2(old0 - mu0) : 1.0f;
            const float c1 = (mu1 != old1) ? ex2(old1 - mu1) : 1.0f;
            // ---- hand P^T (both halves) and the rescale to the PV warp
            const int rn = rg.r + seq;  // this record's ring count
            const int ps = rn % kPRing;
            if (rn >= kPRing) {
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&pempty[ps], ((rn / kPRing) - 1) & 1, abort, P.err));
                if (!ok) break;
            }
            uint4 *rec = reinterpret_cast<uint4 *>(prec + ps * C::PREC);
            rec[lane] = make_uint4(movmatrix_trans(pack_half2(pv[0][0], pv[1][0])),
                                   movmatrix_trans(pack_half2(pv[0][1], pv[1][1])),
                                   movmatrix_trans(pack_half2(pv[0][2], pv[1][2])),
                                   movmatrix_trans(pack_half2(pv[0][3], pv[1][3])));
            rec[32 + lane] = make_uint4(__float_as_uint(c0), __float_as_uint(c1),
                                        static_cast<uint32_t>(i), 0u);
            __syncwarp();
            if (lane == 0) mbar_arrive(&pfull[ps]);  // release: the record is visible
        }
        // end of the sequence for the PV warp
        if (ok) {
            const int rn = rg.r + seq;
            const int ps = rn % kPRing;
            if (rn >= kPRing)
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&pempty[ps], ((rn / kPRing) - 1) & 1, abort, P.err));
            if (ok) {
                uint4 *rec = reinterpret_cast<uint4 *>(prec + ps * C::PREC);
                rec[32 + lane] = make_uint4(0u, 0u, 0xFFFFFFFFu, 0u);  // tile index: none
                __syncwarp();
                if (lane == 0) mbar_arrive(&pfull[ps]);
            }
        }
        if (!ok) drain(kfull, NK, rg.k + kn);  // let this warp's copies land first
        rg.k += kn;
        rg.r += seq + 1;  // the records, and the end-of-sequence record
        float m_used[1][2] = {{mu0, mu1}}, m_true[1][2] = {{mt0, mt1}}, lsum[1][2] = {{ls0, ls1}};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float v = lsum[0][hh];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            lsum[0][hh] = v;
        }
        __syncthreads();  // both warps of every pair are done with the stages
        merge_write_stats<1>(dsmem, pair, m_used, m_true, lsum);
    } else {
        // ================================================================ PV warp
        float o[MT][1][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int k = 0; k < 4; ++k) o[mt][0][k] = 0.0f;
        const uint32_t magic = opaque(kMagic);
        const uint32_t ncorr[4] = {opaque(kHNeg1032), opaque(kHNeg1152), opaque(kHNeg1032),
                                   opaque(kHNeg1152)};
        // This warp copies the V tiles: the first NV now, then each stage again
        // as soon as it has finished the tile in it (NV tiles ahead).
        const uint8_t *vbody = P.v_planes + static_cast<size_t>(u) * P.plane_bytes + P.body_off +
                               static_cast<size_t>(g) * P.max_seq * ROWB;
        int vt = pair;  // next tile index to copy
        int vn = 0;     // copies issued in this piece (ring count rg.v + vn)
        for (; vn < NV && vt < ntiles; ++vn) {
            const int st = (rg.v + vn) % NV;
            if (lane == 0) issue(vbody, vt, pbase + C::V_OFF + st * C::TILE_ALLOC, &vfull[st]);
            vt += kPairs;
        }
        int seq = 0;
        for (;; ++seq) {
            const int rn = rg.r + seq;  // this record's ring count
            const int ps = rn % kPRing;
            ok = __all_sync(0xffffffffu, mbar_wait(&pfull[ps], (rn / kPRing) & 1, abort, P.err));
            if (!ok) break;
            const uint4 *rec = reinterpret_cast<const uint4 *>(prec + ps * C::PREC);
            const uint4 w0 = rec[lane];
            const uint4 w1 = rec[32 + lane];
            __syncwarp();
            if (lane == 0) mbar_arrive(&pempty[ps]);
            if (w1.z == 0xFFFFFFFFu) break;  // end of the sequence
            if (w1.z != static_cast<uint32_t>(pair + kPairs * seq)) {
                // not the tile this record must carry: report, stop the block
                if (lane == 0) {
                    flag_error(P.err, FA_ERRBIT_DEVICE);
                    *abort = 1;
                }
                ok = false;
                break;
            }
            const int s = (rg.v + seq) % NV;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&vfull[s], ((rg.v + seq) / NV) & 1, abort, P.err));
            if (!ok) break;
            const float c0 = __uint_as_float(w1.x), c1 = __uint_as_float(w1.y);
            if (__any_sync(0xffffffffu, c0 != 1.0f || c1 != 1.0f)) {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    o[mt][0][0] *= c0;
                    o[mt][0][2] *= c0;
                    o[mt][0][1] *= c1;
                    o[mt][0][3] *= c1;
                }
            }
            uint8_t *Vs = pbase + C::V_OFF + s * C::TILE_ALLOC;
            const int nk = k_end - tile_key0(static_cast<int>(w1.z));
            if (nk < kTileKeys) {
                // Rows past the range hold bytes of earlier tiles, bytes the copy
                // rounded up into, or nothing written yet. Their P is 0; zero
                // their scales so that 0 * d stays 0 whatever the bytes are.
                for (int idx = lane; idx < (kTileKeys - nk) * NB; idx += 32)
                    *reinterpret_cast<uint16_t *>(Vs + (nk + idx / NB) * ROWB +
                                                  (idx % NB) * kQ4BlockBytes) = 0;
                fence_proxy_async_smem();  // the next copy into this stage comes after
                __syncwarp();
            }
#pragma unroll kPVHalves
            for (int h2 = 0; h2 < 2; ++h2) {
                const uint32_t pb0 = h2 ? w0.z : w0.x;
                const uint32_t pb1 = h2 ? w0.w : w0.y;
                const uint8_t *R0 = Vs + (16 * h2 + 2 * t) * ROWB;  // key 2t
                const uint8_t *R1 = R0 + ROWB;                      // key 2t+1
                const uint8_t *R2 = R0 + 8 * ROWB;                  // key 2t+8
                const uint8_t *R3 = R2 + ROWB;                      // key 2t+9
                // The scales of block b for these four keys are the same for
                // the 8 lanes of a column group: lane (r, t) loads those of
                // block r once, and block b's come from lane 4b + t.
                const int om = kQ4BlockBytes * (r < NB ? r : 0);
                const uint32_t dm01 = __byte_perm(*reinterpret_cast<const uint16_t *>(R0 + om),
                                                  *reinterpret_cast<const uint16_t *>(R1 + om),
                                                  0x5410);
                const uint32_t dm23 = __byte_perm(*reinterpret_cast<const uint16_t *>(R2 + om),
                                                  *reinterpret_cast<const uint16_t *>(R3 + om),
                                                  0x5410);
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const int o18 = kQ4BlockBytes * b;
                    const uint32_t d01 = __shfl_sync(0xffffffffu, dm01, 4 * b + t);
                    const uint32_t d23 = __shfl_sync(0xffffffffu, dm23, 4 * b + t);
                    const uint32_t bb[2] = {hmul2u(pb0, d01), hmul2u(pb1, d23)};
                    const int oc = o18 + 2 + 2 * r;
                    const uint32_t z01 = __byte_perm(*reinterpret_cast<const uint16_t *>(R0 + oc),
                                                     *reinterpret_cast<const uint16_t *>(R1 + oc),
                                                     0x5410);
                    const uint32_t z23 = __byte_perm(*reinterpret_cast<const uint16_t *>(R2 + oc),
                                                     *reinterpret_cast<const uint16_t *>(R3 + oc),
                                                     0x5410);
                    const uint32_t y01 = z01 >> 8, y23 = z23 >> 8;
                    // m-tile 2b + j: row r is element 2r + j (operand 1024 + c),
                    // row r + 8 element 16 + 2r + j (operand 1024 + 16 c). The
                    // constant operand right after removes 1032 (row r) or 1152
                    // (row r + 8) times the sum of the block's P' from the rows.
                    const uint32_t ax[4] = {and_or<0x000F000Fu>(z01, magic), and_or<0x00F000F0u>(z01, magic),
                                            and_or<0x000F000Fu>(z23, magic), and_or<0x00F000F0u>(z23, magic)};
                    const uint32_t ay[4] = {and_or<0x000F000Fu>(y01, magic), and_or<0x00F000F0u>(y01, magic),
                                            and_or<0x000F000Fu>(y23, magic), and_or<0x00F000F0u>(y23, magic)};
                    mma_16816(o[2 * b][0], ax, bb);
                    mma_16816(o[2 * b][0], ncorr, bb);
                    mma_16816(o[2 * b + 1][0], ay, bb);
                    mma_16816(o[2 * b + 1][0], ncorr, bb);
                }
            }
            __syncwarp();  // every lane has read the stage
            if (vt < ntiles) {
                if (lane == 0) {
                    fence_proxy_async_smem();  // those reads come before the copy's writes
                    issue(vbody, vt, Vs, &vfull[s]);
                }
                vt += kPairs;
                ++vn;
            }
        }
        if (!ok) drain(vfull, NV, rg.v + vn);  // let this warp's copies land first
        rg.v += vn;
        rg.r += seq + 1;  // the records, and the end-of-sequence record
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {  // rows r + 8 carry 16 (c - 8)
            o[mt][0][2] *= 0.0625f;
            o[mt][0][3] *= 0.0625f;
        }
        __syncthreads();  // pairs with the QK warps' barrier above
        merge_write_o<HD, 1, true>(dsmem, pair, o);
    }
    merge_finish<HD>(P, dsmem, head0, G, e);
}

// Blocks [0, nslots * Hkv) are the pairs' auxiliary blocks: the fp16-shadow
// entry, the empty entries of a pair with no Q4_0 tile, and the report of a
// position out of range. The blocks after them are the body blocks.
template <int HD>
__global__ void __launch_bounds__(2 * kPairs * 32, FA_Q4_MIN_BLOCKS)
    decode_q4_kernel(const DecodeParams P) {
    extern __shared__ __align__(128) uint8_t dsmem[];
    __shared__ Q4Job sjob;
    __shared__ long long sloc[3];  // first pair's tile base, slot, kv head of the block's run
    const int G = P.Hq / P.Hkv;
    const int n_aux = P.nslots * P.Hkv;
    if (threadIdx.x < 32) {
        const Q4Job J = q4_job(P, P.q4_body_blocks);
        if (threadIdx.x == 0) {
            sjob = J;
            if (blockIdx.x == 0) {
                P.ws_header[0] = kDecodeMagic;
                P.ws_header[1] = static_cast<uint32_t>(P.nslots);
                P.ws_header[2] = static_cast<uint32_t>(P.Hq);
                P.ws_header[3] = static_cast<uint32_t>(HD);
                P.ws_header[4] = static_cast<uint32_t>(J.E);
            }
        }
    }
    __syncthreads();
    const Q4Job J = sjob;

    if (static_cast<int>(blockIdx.x) < n_aux) {
        // ---------------------------------------------------- auxiliary block
        const int u = blockIdx.x / P.Hkv, g = blockIdx.x % P.Hkv;
        const size_t head0 = static_cast<size_t>(u) * P.Hq + static_cast<size_t>(g) * G;
        const int p = P.pos[u];
        if (p < 0 || p >= P.max_seq) {
            if (threadIdx.x == 0 && g == 0) flag_error(P.err, FA_ERRBIT_DEVICE);
            write_empty_range(P, head0, G, 0, J.E);
            return;
        }
        if (q4_tiles(P, p).count() == 0) write_empty_range(P, head0, G, 0, J.Eb);
        if (J.E > J.Eb) shadow_entry<HD, 1>(P, dsmem, J.Eb, g, u, p);
        return;
    }

    // ------------------------------------------------------------ body block
    const long long bid = static_cast<long long>(blockIdx.x) - n_aux;
    const long long T0 = bid * J.C;
    const long long T1 = min(J.T, T0 + J.C);
    if (T0 >= T1) return;
    if (threadIdx.x < 32) {
        int u_hit;
        long long slot_base;
        q4_locate(P, T0, &u_hit, &slot_base);
        if (threadIdx.x == 0) {
            sloc[0] = slot_base;
            sloc[1] = u_hit;
        }
    }
    __syncthreads();
    int u = static_cast<int>(sloc[1]);
    if (u < 0) return;  // unreachable: T0 < T
    int p = P.pos[u];
    Q4Tiles tl = q4_tiles(P, p);
    const long long local = T0 - sloc[0];
    int g = static_cast<int>(local / tl.count());
    int j = static_cast<int>(local % tl.count());
    long long A = sloc[0] + static_cast<long long>(g) * tl.count();  // the pair's first tile
    volatile int *abort = reinterpret_cast<volatile int *>(
        dsmem + Q4Cfg<HD>::BAR_OFF + kPairs * Q4Cfg<HD>::BARS_PER_PAIR * 8);
    q4_init<HD>(dsmem);
    __syncthreads();
    Q4Ring rg;
    for (long long Tc = T0; Tc < T1;) {
        const int cnt = tl.count();
        const int j1 = static_cast<int>(min(static_cast<long long>(cnt), j + (T1 - Tc)));
        const int e = static_cast<int>(bid - A / J.C);
        q4_body<HD>(P, dsmem, e, g, u, p, tl, j, j1, rg);
        const size_t head0 = static_cast<size_t>(u) * P.Hq + static_cast<size_t>(g) * G;
        if (j1 == cnt) write_empty_range(P, head0, G, e + 1, J.Eb);
        Tc += j1 - j;
        // The merge wrote the stages and records with ordinary stores; the
        // next piece's copies write them through the async proxy.
        fence_proxy_async_smem();
        __syncthreads();
        if (*abort) return;
        if (Tc >= T1) break;
        // the next pair with tiles
        A = Tc;
        j = 0;
        do {
            if (++g == P.Hkv) {
                g = 0;
                ++u;
                p = P.pos[u];
                tl = q4_tiles(P, p);
            }
        } while (tl.count() == 0);
    }
}

// One warp per (slot, q head). The lanes take the entries 32 at a time to
// find the common reference M = max m_e and every entry's weight
// w_e = exp(m_e - M); then the warp accumulates sum w_e acc_e over the
// entries in ascending order (lanes split head_dim), with the loads of
// several entries in flight, and out = sum w_e acc_e / sum w_e l_e. An empty
// entry (m = -inf) has weight 0 and its acc, which was never written, is
// read but not used.
constexpr int kCombineWarps = 2;

template <int HD>
__global__ void __launch_bounds__(32 * kCombineWarps)
    combine_kernel(const uint32_t *__restrict__ header, const float *__restrict__ ws_m,
                   const float *__restrict__ ws_l, const float *__restrict__ ws_acc,
                   float *__restrict__ out, int nslots, int Hq, int stride, unsigned *err) {
    constexpr int PER = HD / 32;  // dims per lane
    const int lane = threadIdx.x & 31;
    const long long head = blockIdx.x * static_cast<long long>(kCombineWarps) + (threadIdx.x >> 5);
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
    float Lp = 0.0f;  // this lane's entries' w * l
    const float *a0 = ws_acc + head * stride * HD + lane * PER;
    for (int i0 = 0; i0 < E; i0 += 32) {
        const int i = i0 + lane;
        const float mi = i < E ? m[i] : -INFINITY;
        const float w = (mi == -INFINITY) ? 0.0f : ex2((mi - M) * 1.4426950408889634f);
        if (w != 0.0f) Lp += w * l[i];
        const int cnt = min(32, E - i0);
#pragma unroll 4
        for (int k = 0; k < cnt; ++k) {
            const float wk = __shfl_sync(0xffffffffu, w, k);
            const float *a = a0 + static_cast<long long>(i0 + k) * HD;
#pragma unroll
            for (int d = 0; d < PER; d += 4) {
                const float4 v = *reinterpret_cast<const float4 *>(a + d);
                acc[d] += wk != 0.0f ? wk * v.x : 0.0f;
                acc[d + 1] += wk != 0.0f ? wk * v.y : 0.0f;
                acc[d + 2] += wk != 0.0f ? wk * v.z : 0.0f;
                acc[d + 3] += wk != 0.0f ? wk * v.w : 0.0f;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Lp += __shfl_xor_sync(0xffffffffu, Lp, o);
    const float inv = 1.0f / Lp;
    float *dst = out + head * HD + lane * PER;
#pragma unroll
    for (int k = 0; k < PER; k += 4)
        *reinterpret_cast<float4 *>(dst + k) =
            make_float4(acc[k] * inv, acc[k + 1] * inv, acc[k + 2] * inv, acc[k + 3] * inv);
}

template <int HD, int NT>
cudaError_t launch_generic(const DecodeParams &P, cudaStream_t stream) {
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

template <int HD>
cudaError_t launch_q4(const DecodeParams &P, bool body, cudaStream_t stream) {
    using C = Q4Cfg<HD>;
    cudaError_t e = cudaFuncSetAttribute(decode_q4_kernel<HD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    // one auxiliary block per (slot, kv head), then P.q4_body_blocks body
    // blocks (none when another kernel computes the body entries)
    const long long aux = static_cast<long long>(P.nslots) * P.Hkv;
    const long long blocks = aux + (body ? P.q4_body_blocks : 0);
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    decode_q4_kernel<HD><<<static_cast<unsigned>(blocks), 2 * kPairs * 32, C::SMEM, stream>>>(P);
    return cudaGetLastError();
}

}  // namespace

DecodeShape decode_shape(int nslots, int n_q_heads, int n_kv_heads, int kv_fmt, int shadow_sink,
                         int shadow_win, int max_splits, int max_seq, size_t row_bytes) {
    DecodeShape d;
    const int G = n_q_heads / n_kv_heads;
    // The Q4_0 path bulk-copies rows of a kv head; a copy must start 16-byte
    // aligned, so every head's body must start 16-byte aligned.
    d.fast = kv_fmt == kFmtQ4 && G <= 8 && (static_cast<size_t>(max_seq) * row_bytes) % 16 == 0;
    const int hd = kv_fmt == kFmtF16 ? static_cast<int>(row_bytes / 2) : static_cast<int>(row_bytes);
    d.dense = (kv_fmt == kFmtF16 || kv_fmt == kFmtFp8) && dense_decode_supported(kv_fmt, G, hd);
    if (d.dense) {
        // persistent stream-K kernel: any entry of the workspace may be used
        d.splits_per_cta = 1;
        d.body_entries = max_splits + 1;
        d.shadow_entry = -1;
        d.entries = max_splits + 1;
        return d;
    }
    // The Q4_0 kernel cuts its work itself (stream-K) and needs two body
    // entries per head besides the shadow entry.
    const int shadow = (shadow_sink > 0 || shadow_win > 0) ? 1 : 0;
    if (d.fast && max_splits + 1 < 2 + shadow) d.fast = false;
    if (d.fast) {
        d.splits_per_cta = 1;
        d.body_entries = max_splits + 1 - shadow;
        d.shadow_entry = -1;  // decided in the kernel (entry Eb)
        d.entries = max_splits + 1;
        return d;
    }
    // Blocks to aim at for the generic path: 4 per SM.
    const long long pairs = static_cast<long long>(nslots) * n_kv_heads;
    const long long target = 4LL * device_sm_count();
    long long cpc = (pairs * max_splits + target - 1) / target;
    if (cpc < 1) cpc = 1;
    if (cpc > max_splits) cpc = max_splits;
    d.splits_per_cta = static_cast<int>(cpc);
    d.body_entries = static_cast<int>((max_splits + cpc - 1) / cpc);
    d.shadow_entry = -1;
    d.entries = d.body_entries + (d.shadow_entry >= 0 ? 1 : 0);
    return d;
}

size_t decode_ws_bytes(int nslots, int n_q_heads, int head_dim, int stride) {
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t heads = static_cast<size_t>(nslots) * n_q_heads;
    return 256 + 2 * up(heads * stride * 4) + up(heads * stride * head_dim * 4);
}

void decode_ws_carve(void *ws, int nslots, int n_q_heads, int head_dim, int stride,
                     DecodeWs *out) {
    (void)head_dim;
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t heads = static_cast<size_t>(nslots) * n_q_heads;
    uint8_t *b = static_cast<uint8_t *>(ws);
    out->header = reinterpret_cast<uint32_t *>(b);
    out->m = reinterpret_cast<float *>(b + 256);
    out->l = reinterpret_cast<float *>(b + 256 + up(heads * stride * 4));
    out->acc = reinterpret_cast<float *>(b + 256 + 2 * up(heads * stride * 4));
    out->stride = stride;
}

cudaError_t launch_decode(const DecodeArgs &a, const DecodeWs &ws, const DecodeShape &d,
                          unsigned *err, cudaStream_t stream) {
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
    P.cpc = d.splits_per_cta;
    P.entries = d.entries;
    P.stride = ws.stride;
    P.shadow_entry = d.shadow_entry;
    P.plane_bytes = a.g.bytes;
    P.body_off = a.g.body_off;
    P.row_bytes = a.g.row_bytes;
    P.sink_off = a.g.sink_off;
    P.ring_off = a.g.ring_off;
    P.scale_off = a.g.scale_off;
    P.sl2 = a.scale * 1.4426950408889634f;
    P.err = err;
    if (d.dense) return launch_decode_dense(a, ws, err, stream);
    if (d.entries > ws.stride) return cudaErrorInvalidValue;
    const int G = a.n_q_heads / a.n_kv_heads;
    if (d.fast) {
        // 32-key tiles cut over two blocks per SM (one resident wave), after
        // one auxiliary block per (slot, kv head)
        P.q4_tile_keys = kTileKeys;
        P.q4_body_blocks = FA_Q4_MIN_BLOCKS * device_sm_count();
        switch (a.g.hd) {
            case 64: return launch_q4<64>(P, true, stream);
            case 128: return launch_q4<128>(P, true, stream);
            case 256: return launch_q4<256>(P, true, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    const bool two = G > 8;
    switch (a.g.hd) {
        case 64: return two ? launch_generic<64, 2>(P, stream) : launch_generic<64, 1>(P, stream);
        case 128: return two ? launch_generic<128, 2>(P, stream) : launch_generic<128, 1>(P, stream);
        case 256: return two ? launch_generic<256, 2>(P, stream) : launch_generic<256, 1>(P, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_combine(const void *workspace, float *out, int nslots, int n_q_heads,
                           int head_dim, int stride, unsigned *err, cudaStream_t stream) {
    DecodeWs ws;
    decode_ws_carve(const_cast<void *>(workspace), nslots, n_q_heads, head_dim, stride, &ws);
    const long long heads = static_cast<long long>(nslots) * n_q_heads;
    const int blocks = static_cast<int>((heads + kCombineWarps - 1) / kCombineWarps);
    switch (head_dim) {
        case 64:
            combine_kernel<64><<<blocks, 32 * kCombineWarps, 0, stream>>>(
                ws.header, ws.m, ws.l, ws.acc, out, nslots, n_q_heads, ws.stride, err);
            break;
        case 128:
            combine_kernel<128><<<blocks, 32 * kCombineWarps, 0, stream>>>(
                ws.header, ws.m, ws.l, ws.acc, out, nslots, n_q_heads, ws.stride, err);
            break;
        case 256:
            combine_kernel<256><<<blocks, 32 * kCombineWarps, 0, stream>>>(
                ws.header, ws.m, ws.l, ws.acc, out, nslots, n_q_heads, ws.stride, err);
            break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace fa
