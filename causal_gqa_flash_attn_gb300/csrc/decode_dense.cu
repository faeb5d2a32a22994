// decode_dense.cu -- multi-slot split decode over fp16 and fp8 e4m3fn caches
// ("attention.cu", "Decode-mode flash attention" and "Multi-user decode
// attention": the same online softmax over the keys each query sees, with the
// partials {m, l, acc} merged by fa_decode_combine; the fp16 cache of
// "qwen38_batched.rs" (BQ_KV16) and the fp8 cache read of "vt/ops.h",
// PagedAttentionArgs: Dequant(byte) * k_scale | v_scale).
//
// A dense cache row is hd * 2 (fp16) or hd (fp8) bytes, so at G <= 8 query
// heads per kv head the work is a pure stream of K and V bytes: the kernel is
// bound by HBM if it keeps enough bytes in flight and reads shared memory
// without bank conflicts. Design:
//  * persistent: one block per SM, every warp an independent worker with a
//    private ring of NS stages; a stage holds a K tile and a V tile of TK
//    keys (16 for fp16, 32 for fp8, processed as 16-key MMA slices), each as
//    128-byte-wide boxes loaded by TMA with the 128-byte swizzle, so ldmatrix
//    reads them conflict-free;
//  * stream-K work split: the visible 16-key tiles of all (slot, kv head)
//    pairs, in order, are cut into equal runs, one per warp; a warp writes one
//    partial per (slot, kv head) piece it covers, as entry (warp - first warp
//    of that pair), and the warp holding a pair's last piece marks the pair's
//    remaining entries empty. Every warp streams the same number of tiles, and
//    a warp's ring runs on across piece boundaries;
//  * mma.sync m16n8k16 as in decode.cu: S^T (16 keys x 8 heads) = K Q^T and
//    O^T (hd x 8 heads) += V^T P^T, P^T formed with movmatrix;
//  * fp8: ldmatrix reads byte pairs, cvt turns each pair into an exact fp16
//    pair (every e4m3 value is an fp16 value); for K the byte order fixes
//    which head dims meet in an MMA k-step (Q's fragments use the same
//    order), for V a byte permute pairs two keys of one dim, and the output
//    rows come out in the order 16c + 2r, 16c + 2r + 1 (undone on write).
//    k_scale multiplies the score scale, v_scale the partial output: the
//    result is that of the float(byte) * scale values a reader of the cache
//    sees, up to rounding.
#include "decode_softmax.cuh"
#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr float kRescaleDense = 8.0f;  // lazy-rescale threshold (log2 units)

// Warps per block: fp16 with 16-KB stages (head_dim 256), fp16 with smaller
// stages, and fp8.
#ifndef FA_DENSE_NW_BIG
#define FA_DENSE_NW_BIG 3
#endif
#ifndef FA_DENSE_NW_SMALL
#define FA_DENSE_NW_SMALL 8
#endif
#ifndef FA_DENSE_NW_FP8
#define FA_DENSE_NW_FP8 5
#endif
// Keys per tile of the fp8 kernel (16 or 32; fp16 uses 16): a longer tile
// spreads each tile's fixed work (waits, copies, masks, the softmax step)
// over more bytes.
#ifndef FA_DENSE_TK_FP8
#define FA_DENSE_TK_FP8 32
#endif

template <int HD, int FMT>
struct DenseCfg {
    static constexpr int EB = FMT == kFmtF16 ? 2 : 1;  // bytes per element
    static constexpr int TK = FMT == kFmtF16 ? 16 : FA_DENSE_TK_FP8;  // keys per tile
    static constexpr int NSUB = TK / 16;               // 16-key MMA slices of a tile
    static constexpr int BOXB = TK * 128;              // one box: TK rows x 128 bytes
    static constexpr int NBX = HD * EB / 128;          // boxes per K (or V) tile
    static constexpr int TILE = NBX * BOXB;            // K (or V) bytes of a tile
    static constexpr int STAGE = 2 * TILE;
    // warps per block: more stages per warp keep more bytes in flight, more
    // warps cover the fp8 conversions
    static constexpr int NW = FMT == kFmtFp8      ? FA_DENSE_NW_FP8
                              : STAGE >= 16384 ? FA_DENSE_NW_BIG
                                               : FA_DENSE_NW_SMALL;
    // ring stages from a 224 KB budget (the 227 KB a block may have, less the
    // barriers and the alignment slack)
    static constexpr int NS0 = 229376 / (NW * STAGE);
    static constexpr int NS = NS0 > 8 ? 8 : NS0;       // ring stages per warp
    static constexpr int MT = HD / 16;
    static constexpr int WARP_BYTES = NS * STAGE;
    static constexpr int BAR_OFF = NW * WARP_BYTES;
    static constexpr int ABORT_OFF = BAR_OFF + NW * NS * 8;
    static constexpr int SMEM = ABORT_OFF + 16 + 1024;  // + slack to align the base to 1 KB
    static_assert(NBX >= 1 && NS >= 2 && (TK == 16 || TK == 32), "tile geometry");
};

struct DenseParams {
    const float *q;
    const int32_t *pos;
    const uint8_t *k_planes, *v_planes;  // for the fp8 scales
    float *ws_m, *ws_l, *ws_acc;
    uint32_t *ws_header;
    int nslots, Hq, Hkv, max_seq, sink, win, stride;
    size_t plane_bytes, scale_off;
    float sl2;  // scale * log2(e)
    unsigned *err;
};

// The visible TK-key tiles of the query at p (ascending): tiles 0 .. st-1
// hold the sinks; tiles wt .. p/TK the window. With win <= 0 all tiles up to
// p/TK (st covers them). nt = 0 marks a position out of range.
struct SlotTiles {
    int nt, st, wt, p;
};

template <int TK>
__device__ __forceinline__ SlotTiles slot_tiles(const DenseParams &P, int u) {
    constexpr int SH = TK == 32 ? 5 : 4;
    SlotTiles s;
    s.p = __ldg(P.pos + u);
    s.nt = 0;
    s.st = 0;
    s.wt = 0;
    if (s.p < 0 || s.p >= P.max_seq) return s;
    const int last = s.p >> SH;
    if (P.win <= 0) {
        s.st = last + 1;
        s.wt = last + 1;
        s.nt = last + 1;
        return s;
    }
    const int s_end = min(P.sink, s.p + 1);
    s.st = (s_end + TK - 1) >> SH;
    s.wt = max(max(0, s.p - P.win + 1) >> SH, s.st);
    s.nt = s.st + max(0, last - s.wt + 1);
    return s;
}

template <int TK>
__device__ __forceinline__ int tile_key(const SlotTiles &s, int j) {
    return j < s.st ? TK * j : TK * (s.wt + j - s.st);
}

// Position in the flattened tile order (slot, kv head, visible tile).
struct TileIt {
    long long A;  // flattened index of tile 0 of (u, g)
    int u, g, j;
    SlotTiles s;
};

template <int TK>
__device__ __forceinline__ void it_next(const DenseParams &P, TileIt &it) {
    if (++it.j < it.s.nt) return;
    it.j = 0;
    it.A += it.s.nt;
    if (++it.g < P.Hkv) return;
    it.g = 0;
    while (++it.u < P.nslots) {
        it.s = slot_tiles<TK>(P, it.u);
        if (it.s.nt > 0) return;
    }
}

// Four e4m3 bytes -> two fp16 pairs: bytes 0, 1 -> lo (byte 0 in the low
// half), bytes 2, 3 -> hi. Exact: every e4m3 value is an fp16 value.
__device__ __forceinline__ void e4m3x4_to_h2x2(uint32_t x, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(x));
}

// A bounded wait that ignores the abort flag: used to let this warp's own
// copies land before it leaves after an abort.
__device__ __forceinline__ void wait_drain(uint64_t *bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kSpinCycles) return;
}

template <int HD, int FMT>
__global__ void __launch_bounds__(DenseCfg<HD, FMT>::NW * 32, 1)
    decode_dense_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DenseParams P) {
    using C = DenseCfg<HD, FMT>;
    constexpr int MT = C::MT;
    extern __shared__ uint8_t dsm_raw[];
    uint8_t *dsm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, t = lane & 3;
    uint8_t *ring = dsm + warp * C::WARP_BYTES;
    uint64_t *bar = reinterpret_cast<uint64_t *>(dsm + C::BAR_OFF) + warp * C::NS;
    volatile int *abort = reinterpret_cast<volatile int *>(dsm + C::ABORT_OFF);
    if (threadIdx.x == 0) *abort = 0;
    if (lane == 0) {
        for (int s = 0; s < C::NS; ++s) mbar_init(&bar[s], 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }

    // ---- the whole job: total tiles T and the longest pair maxt
    long long T = 0;
    int maxt = 0;
    for (int u0 = 0; u0 < P.nslots; u0 += 32) {
        const int u = u0 + lane;
        const int nt = u < P.nslots ? slot_tiles<C::TK>(P, u).nt : 0;
        long long sum = nt;
        int mx = nt;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sum += __shfl_xor_sync(0xffffffffu, sum, o);
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        T += sum * P.Hkv;
        maxt = max(maxt, mx);
    }
    const long long W = static_cast<long long>(gridDim.x) * C::NW;
    long long Cw = (T + W - 1) / W;  // tiles per warp
    // at most `stride` pieces per pair: C > (maxt - 1) / (stride - 1)
    const long long cmin = maxt > 0 ? (maxt - 1) / (P.stride - 1) + 1 : 1;
    if (Cw < cmin) Cw = cmin;
    const int E = maxt > 0 ? static_cast<int>(min(static_cast<long long>(P.stride),
                                                  (maxt - 1) / Cw + 2))
                           : 1;
    const int G = P.Hq / P.Hkv;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        P.ws_header[0] = kDecodeMagic;
        P.ws_header[1] = static_cast<uint32_t>(P.nslots);
        P.ws_header[2] = static_cast<uint32_t>(P.Hq);
        P.ws_header[3] = static_cast<uint32_t>(HD);
        P.ws_header[4] = static_cast<uint32_t>(E);
    }
    const long long gw = static_cast<long long>(blockIdx.x) * C::NW + warp;
    if (gw == 0) {
        // slots whose position is out of range: all entries empty, and flagged
        for (int u = 0; u < P.nslots; ++u) {
            if (slot_tiles<C::TK>(P, u).nt > 0) continue;
            if (lane == 0) flag_error(P.err, FA_ERRBIT_DEVICE);
            for (int i = lane; i < P.Hq * E; i += 32) {
                const size_t idx = (static_cast<size_t>(u) * P.Hq + i / E) * P.stride + i % E;
                P.ws_m[idx] = -INFINITY;
                P.ws_l[idx] = 0.0f;
            }
        }
    }
    const long long T_begin = gw * Cw;
    const long long T_end = min(T, T_begin + Cw);
    if (T_begin >= T_end) return;

    // ---- locate tile T_begin
    TileIt cons;
    {
        long long base = 0;
        int u_hit = -1;
        long long slot_base = 0;
        for (int u0 = 0; u0 < P.nslots && u_hit < 0; u0 += 32) {
            const int u = u0 + lane;
            const long long cnt =
                u < P.nslots ? static_cast<long long>(slot_tiles<C::TK>(P, u).nt) * P.Hkv : 0;
            long long inc = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, base + inc > T_begin);
            if (hit) {
                const int L = __ffs(hit) - 1;
                u_hit = u0 + L;
                slot_base = base + __shfl_sync(0xffffffffu, inc - cnt, L);
            } else {
                base += __shfl_sync(0xffffffffu, inc, 31);
            }
        }
        if (u_hit < 0) return;  // unreachable: T_begin < T
        cons.u = u_hit;
        cons.s = slot_tiles<C::TK>(P, u_hit);
        const long long local = T_begin - slot_base;
        cons.g = static_cast<int>(local / cons.s.nt);
        cons.j = static_cast<int>(local % cons.s.nt);
        cons.A = slot_base + static_cast<long long>(cons.g) * cons.s.nt;
    }
    TileIt prod = cons;

    auto issue = [&](const TileIt &it, int stage) {
        uint64_t *b = &bar[stage];
        mbar_arrive_expect_tx(b, C::STAGE);
        uint8_t *dk = ring + stage * C::STAGE;
        uint8_t *dv = dk + C::TILE;
        const int c0 = tile_key<C::TK>(it.s, it.j);
#pragma unroll
        for (int bx = 0; bx < C::NBX; ++bx) {
            tma_load_4d(dk + bx * C::BOXB, &kmap, b, bx * (128 / C::EB), c0, it.g, it.u);
            tma_load_4d(dv + bx * C::BOXB, &vmap, b, bx * (128 / C::EB), c0, it.g, it.u);
        }
    };

    long long Tp = T_begin;
    for (int s = 0; s < C::NS && Tp < T_end; ++s, ++Tp) {
        if (lane == 0) issue(prod, s);
        it_next<C::TK>(P, prod);
    }

    // fragment addressing (row and swizzle phase of this lane)
    const int krow = lane & 15;
    const uint32_t koff = krow * 128;
    const int kz = (lane >> 4) ^ (krow & 7);
    const int vkey = FMT == kFmtF16 ? (lane & 7) + ((lane >> 4) << 3)
                                    : (lane & 7) + (((lane >> 3) & 1) << 3);
    const uint32_t voff = vkey * 128;
    const int vz = (FMT == kFmtF16 ? ((lane >> 3) & 1) : (lane >> 4)) ^ (vkey & 7);

    uint32_t qb[MT][2];
    float o[MT][1][4];
    float mu0 = -INFINITY, mu1 = -INFINITY, mt0 = -INFINITY, mt1 = -INFINITY, ls0 = 0.f, ls1 = 0.f;
    float sl2 = P.sl2, vscale = 1.0f;
    int e_piece = 0;
    size_t head0 = 0;

    for (long long Tc = T_begin; Tc < T_end; ++Tc) {
        const long long k = Tc - T_begin;
        const int stage = static_cast<int>(k % C::NS);
        const uint32_t parity = static_cast<uint32_t>((k / C::NS) & 1);
        if (Tc == T_begin || cons.j == 0) {
            // a new piece: (slot cons.u, kv head cons.g)
            head0 = static_cast<size_t>(cons.u) * P.Hq + static_cast<size_t>(cons.g) * G;
            e_piece = static_cast<int>(gw - cons.A / Cw);
            const int hh = r < G ? r : 0;
            const float *qr = P.q + (head0 + hh) * HD;
#pragma unroll
            for (int kk = 0; kk < MT; ++kk) {
                if (FMT == kFmtF16) {
                    const float2 a = *reinterpret_cast<const float2 *>(qr + 16 * kk + 2 * t);
                    const float2 b = *reinterpret_cast<const float2 *>(qr + 16 * kk + 2 * t + 8);
                    qb[kk][0] = pack_half2(a.x, a.y);
                    qb[kk][1] = pack_half2(b.x, b.y);
                } else {
                    const float4 a = *reinterpret_cast<const float4 *>(qr + 16 * kk + 4 * t);
                    qb[kk][0] = pack_half2(a.x, a.y);
                    qb[kk][1] = pack_half2(a.z, a.w);
                }
                if (r >= G) qb[kk][0] = qb[kk][1] = 0u;
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) o[mt][0][q4] = 0.0f;
            mu0 = mu1 = mt0 = mt1 = -INFINITY;
            ls0 = ls1 = 0.0f;
            if (FMT == kFmtFp8) {
                const size_t pl = static_cast<size_t>(cons.u) * P.plane_bytes + P.scale_off;
                sl2 = P.sl2 * __ldg(reinterpret_cast<const float *>(P.k_planes + pl));
                vscale = __ldg(reinterpret_cast<const float *>(P.v_planes + pl));
            }
        }
        if (!mbar_wait(&bar[stage], parity, abort, P.err)) {
            // let this warp's copies in flight land, then leave
            for (long long kq = Tc; kq < Tp; ++kq) {
                const long long kk2 = kq - T_begin;
                wait_drain(&bar[kk2 % C::NS], static_cast<uint32_t>((kk2 / C::NS) & 1));
            }
            return;
        }
        const int c0 = tile_key<C::TK>(cons.s, cons.j);
        const int p = cons.s.p;
        uint8_t *kt = ring + stage * C::STAGE;
        uint8_t *vt = kt + C::TILE;
        bool wrote = false;
        if (c0 + C::TK - 1 > p) {
            // rows past the slot's last key hold whatever the plane held:
            // zero them in V so that P = 0 meets finite values
            const int z0 = p - c0 + 1;
            const int nchunk = (C::TK - z0) * 8 * C::NBX;
            for (int i = lane; i < nchunk; i += 32) {
                const int bx = i / ((C::TK - z0) * 8);
                const int rem = i % ((C::TK - z0) * 8);
                *reinterpret_cast<uint4 *>(vt + bx * C::BOXB + (z0 + rem / 8) * 128 +
                                           (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            wrote = true;
            __syncwarp();
        }
        const uint32_t kb = smem_u32(kt), vb = smem_u32(vt);

        // S^T = K Q^T per 16-key slice of the tile: two accumulator chains each
        constexpr int NSUB = C::NSUB;
        float sv[2][2 * NSUB], pv[2][2 * NSUB];
#pragma unroll
        for (int sub = 0; sub < NSUB; ++sub) {
            const uint32_t kbs = kb + sub * 16 * 128 + koff;  // rows 16 sub .. of every box
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
            if (FMT == kFmtF16) {
#pragma unroll
                for (int kk = 0; kk < MT; ++kk) {
                    uint32_t a[4];
                    ldmatrix_x4(a, kbs + (kk >> 2) * C::BOXB + (((2 * (kk & 3)) ^ kz) << 4));
                    mma_16816((kk & 1) ? s1 : s0, a, qb[kk]);
                }
            } else {
#pragma unroll
                for (int kp = 0; kp < HD / 32; ++kp) {
                    uint32_t x[4];
                    ldmatrix_x4(x, kbs + (kp >> 2) * C::BOXB + (((2 * (kp & 3)) ^ kz) << 4));
                    uint32_t a0[4], a1[4];  // {row r, row r + 8} x {dims 4t..4t+1, 4t+2..4t+3}
                    e4m3x4_to_h2x2(x[0], a0[0], a0[2]);
                    e4m3x4_to_h2x2(x[1], a0[1], a0[3]);
                    e4m3x4_to_h2x2(x[2], a1[0], a1[2]);
                    e4m3x4_to_h2x2(x[3], a1[1], a1[3]);
                    mma_16816(s0, a0, qb[2 * kp]);
                    mma_16816(s1, a1, qb[2 * kp + 1]);
                }
            }
            const int keyA = c0 + 16 * sub + r, keyB = keyA + 8;
            const bool visA = key_visible(p, keyA, P.sink, P.win);
            const bool visB = key_visible(p, keyB, P.sink, P.win);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                sv[hh][2 * sub] = visA ? s0[hh] + s1[hh] : -INFINITY;
                sv[hh][2 * sub + 1] = visB ? s0[2 + hh] + s1[2 + hh] : -INFINITY;
            }
        }
        fold_scores<MT, 1, 2 * NSUB>(sv, sl2, kRescaleDense, mu0, mu1, mt0, mt1, ls0, ls1, o, 0,
                                     pv);

        // O^T += V^T P^T per slice
#pragma unroll
        for (int sub = 0; sub < NSUB; ++sub) {
            uint32_t pb[2];
            pb[0] = movmatrix_trans(pack_half2(pv[0][2 * sub], pv[1][2 * sub]));
            pb[1] = movmatrix_trans(pack_half2(pv[0][2 * sub + 1], pv[1][2 * sub + 1]));
            const uint32_t vbs = vb + sub * 16 * 128 + voff;
            if (FMT == kFmtF16) {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint32_t a[4];
                    ldmatrix_x4_trans(a, vbs + (mt >> 2) * C::BOXB + (((2 * (mt & 3)) ^ vz) << 4));
                    mma_16816(o[mt][0], a, pb);
                }
            } else {
#pragma unroll
                for (int mp = 0; mp < HD / 32; ++mp) {
                    uint32_t x[4];
                    ldmatrix_x4_trans(x, vbs + (mp >> 2) * C::BOXB + (((2 * (mp & 3)) ^ vz) << 4));
                    const uint32_t y0 = __byte_perm(x[0], 0u, 0x3120);
                    const uint32_t y1 = __byte_perm(x[1], 0u, 0x3120);
                    const uint32_t y2 = __byte_perm(x[2], 0u, 0x3120);
                    const uint32_t y3 = __byte_perm(x[3], 0u, 0x3120);
                    uint32_t a0[4], a1[4];  // {dim 2r, dim 2r + 1} x {keys 2t.., keys 2t+8..}
                    e4m3x4_to_h2x2(y0, a0[0], a0[1]);
                    e4m3x4_to_h2x2(y1, a0[2], a0[3]);
                    e4m3x4_to_h2x2(y2, a1[0], a1[1]);
                    e4m3x4_to_h2x2(y3, a1[2], a1[3]);
                    mma_16816(o[2 * mp][0], a0, pb);
                    mma_16816(o[2 * mp + 1][0], a1, pb);
                }
            }
        }

        if (cons.j == cons.s.nt - 1 || Tc == T_end - 1) {
            // end of a piece: write its partial as entry e_piece
            float l0 = ls0, l1 = ls1;
#pragma unroll
            for (int ofs = 4; ofs < 32; ofs <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, ofs);
                l1 += __shfl_xor_sync(0xffffffffu, l1, ofs);
            }
            const float f0 = (mu0 == -INFINITY || mt0 == -INFINITY) ? 0.0f : ex2(mu0 - mt0);
            const float f1 = (mu1 == -INFINITY || mt1 == -INFINITY) ? 0.0f : ex2(mu1 - mt1);
            const int h0 = 2 * t, h1 = 2 * t + 1;
            if (r == 0) {
                if (h0 < G) {
                    const size_t i0 = (head0 + h0) * P.stride + e_piece;
                    P.ws_m[i0] = mt0 == -INFINITY ? -INFINITY : mt0 * 0.69314718055994531f;
                    P.ws_l[i0] = l0 * f0;
                }
                if (h1 < G) {
                    const size_t i1 = (head0 + h1) * P.stride + e_piece;
                    P.ws_m[i1] = mt1 == -INFINITY ? -INFINITY : mt1 * 0.69314718055994531f;
                    P.ws_l[i1] = l1 * f1;
                }
            }
            const float g0 = f0 * vscale, g1 = f1 * vscale;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int h = 2 * t + (q4 & 1);
                    if (h >= G) continue;
                    const int dim = FMT == kFmtF16 ? 16 * mt + r + 8 * (q4 >> 1)
                                                   : 16 * mt + 2 * r + (q4 >> 1);
                    P.ws_acc[((head0 + h) * P.stride + e_piece) * HD + dim] =
                        o[mt][0][q4] * ((q4 & 1) ? g1 : g0);
                }
            if (cons.j == cons.s.nt - 1) {
                // this warp holds the pair's last piece: later entries are empty
                const int rest = E - e_piece - 1;
                for (int i = lane; i < rest * G; i += 32) {
                    const size_t idx = (head0 + i % G) * P.stride + e_piece + 1 + i / G;
                    P.ws_m[idx] = -INFINITY;
                    P.ws_l[idx] = 0.0f;
                }
            }
        }

        // refill this stage with the tile NS ahead
        if (wrote) fence_proxy_async_smem();
        __syncwarp();
        if (Tp < T_end) {
            if (lane == 0) issue(prod, stage);
            it_next<C::TK>(P, prod);
            ++Tp;
        }
        it_next<C::TK>(P, cons);
    }
}

template <int HD, int FMT>
cudaError_t launch_dense_hd(const DecodeArgs &a, const DecodeWs &ws, unsigned *err,
                            cudaStream_t stream) {
    using C = DenseCfg<HD, FMT>;
    const CUtensorMapDataType dt =
        FMT == kFmtF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const uint64_t dims[4] = {static_cast<uint64_t>(HD), static_cast<uint64_t>(a.g.max_seq),
                              static_cast<uint64_t>(a.n_kv_heads), static_cast<uint64_t>(a.nslots)};
    const uint64_t strides[3] = {a.g.row_bytes, a.g.row_bytes * a.g.max_seq, a.g.bytes};
    const uint32_t box[4] = {static_cast<uint32_t>(128 / C::EB), static_cast<uint32_t>(C::TK), 1,
                             1};
    CUtensorMap km, vm;
    if (!encode_tiled(&km, dt, 4, a.k_planes + a.g.body_off, dims, strides, box) ||
        !encode_tiled(&vm, dt, 4, a.v_planes + a.g.body_off, dims, strides, box))
        return cudaErrorInvalidValue;
    DenseParams P;
    P.q = a.q;
    P.pos = a.pos;
    P.k_planes = a.k_planes;
    P.v_planes = a.v_planes;
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
    P.stride = ws.stride;
    P.plane_bytes = a.g.bytes;
    P.scale_off = a.g.scale_off;
    P.sl2 = a.scale * 1.4426950408889634f;
    P.err = err;
    auto kernel = decode_dense_kernel<HD, FMT>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    kernel<<<device_sm_count(), C::NW * 32, C::SMEM, stream>>>(km, vm, P);
    return cudaGetLastError();
}

}  // namespace

bool dense_decode_supported(int kv_fmt, int G, int head_dim) {
    if (G > 8) return false;
    if (kv_fmt == kFmtF16) return head_dim == 64 || head_dim == 128 || head_dim == 256;
    if (kv_fmt == kFmtFp8) return head_dim == 128 || head_dim == 256;
    return false;
}

cudaError_t launch_decode_dense(const DecodeArgs &a, const DecodeWs &ws, unsigned *err,
                                cudaStream_t stream) {
    if (ws.stride < 2) return cudaErrorInvalidValue;
    if (a.g.fmt == kFmtF16) {
        switch (a.g.hd) {
            case 64: return launch_dense_hd<64, kFmtF16>(a, ws, err, stream);
            case 128: return launch_dense_hd<128, kFmtF16>(a, ws, err, stream);
            case 256: return launch_dense_hd<256, kFmtF16>(a, ws, err, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (a.g.hd) {
        case 128: return launch_dense_hd<128, kFmtFp8>(a, ws, err, stream);
        case 256: return launch_dense_hd<256, kFmtFp8>(a, ws, err, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
