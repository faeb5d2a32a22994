// decode_common.cuh -- what the split-KV decode kernels share: their launch
// parameters, and the stream-K cut of the Q4_0 work into equal runs of key
// tiles ("attention.cu", "Decode-mode flash attention" and "Multi-user decode
// attention": every slot's keys are cut into pieces whose partials a
// log-sum-exp combine merges).
#pragma once

#include <cstddef>
#include <cstdint>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {

struct DecodeParams {
    const float *q;
    const uint8_t *k_planes;
    const uint8_t *v_planes;
    const int32_t *pos;
    float *ws_m, *ws_l, *ws_acc;
    uint32_t *ws_header;
    int nslots, Hq, Hkv, max_seq, sink, win, fmt, shadow_sink, shadow_win;
    int split_keys, max_splits, cpc;
    int entries;       // entries written per (slot, head)
    int stride;        // entry stride of the workspace
    int shadow_entry;  // entry index of the fp16-shadow keys, or -1
    int q4_tile_keys;  // keys per tile of the Q4_0 stream-K cut
    int q4_body_blocks;  // blocks that share the Q4_0 tiles
    size_t plane_bytes, body_off, row_bytes, sink_off, ring_off, scale_off;
    float sl2;  // scale * log2(e)
    unsigned *err;
};

// The key tiles of one (slot, kv head) that a Q4_0 kernel loads, in order:
// tile kt covers keys [tk kt, tk kt + tk) clipped to [0, p], tk =
// P.q4_tile_keys. They are two runs, [a0, a0 + na) and [b0, b0 + nb): with a
// window, the tiles holding attended sinks and then the window's tiles;
// without one, a single run. Tiles whose every key is an fp16 shadow (sink
// rows below shadow_sink, recent rows above p - shadow_win) are left out: the
// shadow entry reads those.
struct Q4Tiles {
    int a0, na, b0, nb;
    __device__ __forceinline__ int count() const { return na + nb; }
    __device__ __forceinline__ int kt(int i) const { return i < na ? a0 + i : b0 + (i - na); }
};

static __device__ __forceinline__ Q4Tiles q4_tiles(const DecodeParams &P, int p) {
    const int tk = P.q4_tile_keys;
    Q4Tiles T{0, 0, 0, 0};
    if (p < 0 || p >= P.max_seq || p < P.shadow_sink) return T;
    const int nt = p / tk + 1;          // tiles holding keys 0 .. p
    const int lo = P.shadow_sink / tk;  // first tile with a key >= shadow_sink
    int hi = nt;
    if (P.shadow_win > 0) {
        const int last = p - P.shadow_win;  // the largest key read from the Q4_0 rows
        hi = last >= 0 ? min(hi, last / tk + 1) : 0;
    }
    if (P.win <= 0) {
        T.a0 = lo;
        T.na = max(0, hi - lo);
        return T;
    }
    // attended: sinks [0, min(sink, p + 1)) and the window [p - win + 1, p]
    const int ns = (min(P.sink, p + 1) + tk - 1) / tk;
    const int w0 = max(max(0, p - P.win + 1) / tk, ns);
    T.a0 = lo;
    T.na = max(0, min(ns, hi) - lo);
    T.b0 = max(w0, lo);
    T.nb = max(0, hi - T.b0);
    return T;
}

// Stream-K work split of the Q4_0 path. The loaded tiles of all (slot, kv
// head) pairs, pair after pair, are cut into equal runs of C tiles, one run
// per body block, so that every block streams the same number of bytes and
// none waits for a straggler wave. A block writes one partial per pair piece
// it covers, as entry (block - the block holding the pair's first tile); the
// block holding a pair's last piece marks the pair's later body entries empty.
// Entry Eb of every head is the fp16-shadow entry when the cache has shadows.
struct Q4Job {
    long long T;  // tiles of all pairs
    long long C;  // tiles per body block
    int Eb;       // body entries per head
    int E;        // entries per head (Eb, plus the shadow entry)
};

// Warp-wide (every lane gets the same result). nb: body blocks.
static __device__ __forceinline__ Q4Job q4_job(const DecodeParams &P, int nb) {
    const int lane = threadIdx.x & 31;
    long long T = 0;
    int maxt = 0;
    for (int u0 = 0; u0 < P.nslots; u0 += 32) {
        const int u = u0 + lane;
        const int nt = u < P.nslots ? q4_tiles(P, P.pos[u]).count() : 0;
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
    const int shadow = (P.shadow_sink > 0 || P.shadow_win > 0) ? 1 : 0;
    const int sb = P.stride - shadow;  // body entries available (>= 2)
    Q4Job J;
    J.T = T;
    J.C = nb > 0 ? (T + nb - 1) / nb : T;
    // at most sb pieces per pair: C > (maxt - 1) / (sb - 1)
    const long long cmin = maxt > 0 ? (maxt - 1) / (sb - 1) + 1 : 1;
    if (J.C < cmin) J.C = cmin;
    J.Eb = maxt > 0 ? static_cast<int>(min(static_cast<long long>(sb), (maxt - 1) / J.C + 2)) : 1;
    J.E = J.Eb + shadow;
    return J;
}

// The pair holding tile T0 of the job, found by one warp (every lane gets
// it): the slot u and the job index of that slot's first tile.
static __device__ __forceinline__ void q4_locate(const DecodeParams &P, long long T0, int *u_out,
                                                 long long *slot_base_out) {
    const int lane = threadIdx.x & 31;
    long long base = 0, slot_base = 0;
    int u_hit = -1;
    for (int u0 = 0; u0 < P.nslots && u_hit < 0; u0 += 32) {
        const int uu = u0 + lane;
        const long long cnt =
            uu < P.nslots ? static_cast<long long>(q4_tiles(P, P.pos[uu]).count()) * P.Hkv : 0;
        long long inc = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, base + inc > T0);
        if (hit) {
            const int L = __ffs(hit) - 1;
            u_hit = u0 + L;
            slot_base = base + __shfl_sync(0xffffffffu, inc - cnt, L);
        } else {
            base += __shfl_sync(0xffffffffu, inc, 31);
        }
    }
    *u_out = u_hit;
    *slot_base_out = slot_base;
}

// Entries [e0, e1) of the G heads from head0 on: empty (m = -inf, l = 0).
static __device__ __forceinline__ void write_empty_range(const DecodeParams &P, size_t head0,
                                                         int G, int e0, int e1) {
    for (int i = threadIdx.x; i < G * (e1 - e0); i += blockDim.x) {
        const size_t idx = (head0 + i % G) * P.stride + e0 + i / G;
        P.ws_m[idx] = -INFINITY;
        P.ws_l[idx] = 0.0f;
    }
}

}  // namespace fa
