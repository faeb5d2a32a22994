// decode_noalloc.cu -- fa_decode_noalloc: the multi-slot split-KV decode plus
// its combine, for callers that cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc: a plugin inside a host process
// whose allocator owns all device memory, or a latency-critical serving loop
// where cudaMalloc/cudaFree are banned because they can synchronise the
// device. fa_decode needs a caller-provided workspace for its partials; this
// entry point instead keeps them in a fixed file-scope device array, so the
// caller passes only inputs and the output.
//
// The array is kFaDecodeScratchBytes (8 MiB). Every GPU that loads the
// library holds it until the process exits. Every call shares it, so calls
// that overlap on the GPU (different streams, or different host threads on
// one device) race on it; serialise them. No part of it needs to start at
// zero: each call writes every header word, m, l and acc entry it later reads.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

constexpr size_t kFaDecodeScratchBytes = size_t(8) << 20;

__device__ __align__(256) uint8_t g_fa_decode_scratch[kFaDecodeScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of g_fa_decode_scratch, looked up per device with that
// device current. In host code the symbol itself is only a host-side
// stand-in. A successful lookup is kept for the life of the process; a failed
// one (for instance a first call made during a stream capture) is not: its
// error is taken off the runtime's last-error slot, so that it cannot be
// reported by a later unrelated check, and the next call looks again.
struct ScratchSlot {
    void *ptr = nullptr;
};
ScratchSlot g_scratch[kMaxDevices];
std::mutex g_scratch_mutex;

void *scratch_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchSlot *s = &g_scratch[dev];
    if (!s->ptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fa_decode_scratch) == cudaSuccess) {
            s->ptr = p;
        } else {
            cudaGetLastError();  // leave no sticky error behind; retry next call
        }
    }
    return s->ptr;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" fa_status fa_decode_noalloc(const float *q, const void *k_planes,
                                       const void *v_planes, const int32_t *pos, int nslots,
                                       int n_q_heads, int n_kv_heads, int head_dim, int max_seq,
                                       int sink, int win, int kv_fmt, int shadow_sink,
                                       int shadow_win, int split_keys, int max_splits,
                                       float *out, fa_stream_t stream) {
    if (n_q_heads < 1 || n_kv_heads < 1 || n_q_heads % n_kv_heads || head_dim % 32 ||
        head_dim < 32)
        return FA_ERR_INVALID;
    const int G = n_q_heads / n_kv_heads;
    if ((head_dim != 64 && head_dim != 128 && head_dim != 256) ||
        (G != 1 && G != 2 && G != 4 && G != 8 && G != 16))
        return FA_ERR_UNSUPPORTED;
    if (nslots < 0 || sink < 0 || max_seq < 1 || split_keys < 1 || max_splits < 1)
        return FA_ERR_INVALID;
    if (kv_fmt == FA_KV_F32 || kv_fmt == FA_KV_F16 || kv_fmt == FA_KV_FP8_E4M3) {
        if (shadow_sink != 0 || shadow_win != 0) return FA_ERR_INVALID;
    } else if (kv_fmt == FA_KV_Q4_0) {
        if (shadow_sink < 0 || shadow_sink > FA_Q4_SINK_MAX || shadow_win < 0 ||
            shadow_win > FA_Q4_RING_ROWS)
            return FA_ERR_INVALID;
    } else {
        return FA_ERR_INVALID;
    }
    if (nslots == 0) return FA_OK;
    if (!q || !k_planes || !v_planes || !pos || !out) return FA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k_planes) || !aligned16(v_planes) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(pos) & 3u))
        return FA_ERR_INVALID;
    fa::PlaneGeom g;
    if (!fa::plane_geom(kv_fmt, n_kv_heads, max_seq, head_dim, &g)) return FA_ERR_INVALID;

    // The same work split as fa_decode; the partials are stored with entry
    // stride equal to the number of entries (not max_splits + 1).
    const fa::DecodeShape shape = fa::decode_shape(nslots, n_q_heads, n_kv_heads, kv_fmt,
                                                   shadow_sink, shadow_win, max_splits, max_seq,
                                                   g.row_bytes);
    int entries = shape.entries;
    if (shape.dense || shape.fast) {
        // the streaming kernels adapt their work split to the entries they
        // have: at least 2, plus the Q4_0 kernel's fp16-shadow entry
        const int least = 2 + (shape.fast && (shadow_sink > 0 || shadow_win > 0) ? 1 : 0);
        while (entries > least &&
               fa::decode_ws_bytes(nslots, n_q_heads, head_dim, entries) > kFaDecodeScratchBytes)
            --entries;
    }
    if (fa::decode_ws_bytes(nslots, n_q_heads, head_dim, entries) > kFaDecodeScratchBytes)
        return FA_ERR_WORKSPACE;

    void *scratch = scratch_ptr();
    unsigned *err = fa::device_error_word();
    if (!scratch || !err) return FA_ERR_CUDA;

    fa::DecodeWs ws;
    fa::decode_ws_carve(scratch, nslots, n_q_heads, head_dim, entries, &ws);
    fa::DecodeArgs a;
    a.q = q;
    a.k_planes = static_cast<const uint8_t *>(k_planes);
    a.v_planes = static_cast<const uint8_t *>(v_planes);
    a.pos = pos;
    a.nslots = nslots;
    a.n_q_heads = n_q_heads;
    a.n_kv_heads = n_kv_heads;
    a.sink = sink;
    a.win = win;
    a.shadow_sink = kv_fmt == FA_KV_Q4_0 ? shadow_sink : 0;
    a.shadow_win = kv_fmt == FA_KV_Q4_0 ? shadow_win : 0;
    a.split_keys = split_keys;
    a.max_splits = max_splits;
    a.g = g;
    a.scale = 1.0f / sqrtf(static_cast<float>(head_dim));
    a.workspace = scratch;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = fa::launch_decode(a, ws, shape, err, s);
    // The combine carves the same array with stride `entries`.
    if (e == cudaSuccess)
        e = fa::launch_combine(scratch, out, nslots, n_q_heads, head_dim, entries, err, s);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
