// fa_api.cu -- the C ABI of libfa.so (include/fa.h): argument validation,
// plane geometry, workspace layouts, the decode split plan, and the device
// error word. Everything here runs on the host; all arithmetic of the method
// runs in the kernels of the other translation units.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

// The device error word (one per device that loads the library). Kernels set
// FA_ERRBIT_* bits with atomicOr; fa_get_device_error reads and clears it.
__device__ unsigned int g_fa_device_error;

constexpr int kMaxDevices = 64;

cudaEvent_t g_ev_start = nullptr, g_ev_stop = nullptr;  // fa_set_kernel_events

// Under stream capture the records are external event nodes, so that every
// replay of the graph records them (a plain record under capture only orders
// work); outside capture they are plain records.
cudaError_t record_event(cudaEvent_t ev, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return e;
    return cs == cudaStreamCaptureStatusActive
               ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
               : cudaEventRecord(ev, s);
}
cudaError_t record_start(cudaStream_t s) {
    return (g_ev_start && g_ev_stop) ? record_event(g_ev_start, s) : cudaSuccess;
}
cudaError_t record_stop(cudaStream_t s) {
    return (g_ev_start && g_ev_stop) ? record_event(g_ev_stop, s) : cudaSuccess;
}

struct DeviceInfo {
    std::once_flag once;
    unsigned *err = nullptr;
    int sms = 0;
};
DeviceInfo g_dev[kMaxDevices];

DeviceInfo *device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    DeviceInfo *d = &g_dev[dev];
    std::call_once(d->once, [d, dev]() {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fa_device_error) == cudaSuccess)
            d->err = static_cast<unsigned *>(p);
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
            d->sms = sms;
    });
    return d;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_hd(int hd) { return hd == 64 || hd == 128 || hd == 256; }

bool supported_group(int hq, int hkv) {
    if (hkv < 1 || hq < 1 || hq % hkv) return false;
    const int G = hq / hkv;
    return G == 1 || G == 2 || G == 4 || G == 8 || G == 16;
}

fa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Heads and shapes shared by prefill and decode.
fa_status check_heads(int n_q_heads, int n_kv_heads, int head_dim) {
    if (n_q_heads < 1 || n_kv_heads < 1 || head_dim < 1) return FA_ERR_INVALID;
    if (n_q_heads % n_kv_heads) return FA_ERR_INVALID;
    if (head_dim % 32) return FA_ERR_INVALID;
    if (!supported_hd(head_dim) || !supported_group(n_q_heads, n_kv_heads))
        return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

bool known_fmt(int kv_fmt) {
    return kv_fmt == FA_KV_F32 || kv_fmt == FA_KV_Q4_0 || kv_fmt == FA_KV_F16 ||
           kv_fmt == FA_KV_FP8_E4M3;
}

fa_status check_shadow(int kv_fmt, int shadow_sink, int shadow_win) {
    if (kv_fmt == FA_KV_F32 || kv_fmt == FA_KV_F16 || kv_fmt == FA_KV_FP8_E4M3)
        return (shadow_sink == 0 && shadow_win == 0) ? FA_OK : FA_ERR_INVALID;
    if (kv_fmt != FA_KV_Q4_0) return FA_ERR_INVALID;
    if (shadow_sink < 0 || shadow_sink > FA_Q4_SINK_MAX) return FA_ERR_INVALID;
    if (shadow_win < 0 || shadow_win > FA_Q4_RING_ROWS) return FA_ERR_INVALID;
    return FA_OK;
}

// Prefill workspace: a 256-byte header holding the kernel's work counters
// and its Q staging counter, one Q-ready flag per unit, then the fp16 staging
// of Q [n][Hq][hd], K and V [Hkv][n][hd]. A split
// prefill (Q4_0 with a shadow window narrower than the ring) adds a second
// K and V staging (the fp16 ring values) and the two parts' outputs
// [n][Hq][hd] and lses [Hq][n], fp32.
struct PrefillWs {
    size_t ctr_off, qctr_off, ctr2_off, flag_off, q_off, k_off, v_off, bytes;
    size_t k2_off, v2_off, o1_off, o2_off, l1_off, l2_off;  // split only
};
// n query rows over nk key rows
PrefillWs prefill_ws(int n, int nk, int hq, int hkv, int hd, bool split = false) {
    PrefillWs w;
    w.ctr_off = 0;
    w.qctr_off = 64;
    w.ctr2_off = 128;
    w.flag_off = 256;
    const size_t units = static_cast<size_t>((n + fa::kPrefillBQ - 1) / fa::kPrefillBQ) * hq;
    w.q_off = w.flag_off + up256(units * 4);
    w.k_off = w.q_off + up256(static_cast<size_t>(n) * hq * hd * 2);
    const size_t kv = up256(static_cast<size_t>(hkv) * nk * hd * 2);
    w.v_off = w.k_off + kv;
    w.bytes = w.v_off + kv;
    w.k2_off = w.v2_off = w.o1_off = w.o2_off = w.l1_off = w.l2_off = 0;
    if (split) {
        const size_t ob = up256(static_cast<size_t>(n) * hq * hd * 4);
        const size_t lb = up256(static_cast<size_t>(hq) * n * 4);
        w.k2_off = w.bytes;
        w.v2_off = w.k2_off + kv;
        w.o1_off = w.v2_off + kv;
        w.o2_off = w.o1_off + ob;
        w.l1_off = w.o2_off + ob;
        w.l2_off = w.l1_off + lb;
        w.bytes = w.l2_off + lb;
    }
    return w;
}

// A Q4_0 cache whose fp16 window is neither empty nor the whole ring: which
// copy of a key a query reads depends on the query, so the prefill runs as
// two parts merged by their log-sum-exps.
bool split_prefill(int kv_fmt, int shadow_win) {
    return kv_fmt == FA_KV_Q4_0 && shadow_win != 0 && shadow_win != FA_Q4_RING_ROWS;
}

}  // namespace

namespace fa {
bool plane_geom(int fmt, int n_kv, int max_seq, int hd, PlaneGeom *g);
}

namespace {

// The prefill kernel converts the Q tiles past its first wave of units
// itself: its arguments for that.
void set_q_staging(fa::PrefillArgs *a, const float *q, uint8_t *ws, const PrefillWs &w) {
    a->q = q;
    a->q_flags = reinterpret_cast<unsigned *>(ws + w.flag_off);
    a->q_stage_counter = reinterpret_cast<unsigned *>(ws + w.qctr_off);
    a->q_w0 = fa::prefill_units_staged_first(a->pos0, a->n, a->n_q_heads, a->sink, a->win);
}

// The split prefill after the Q staging and the far K/V staging: stage the
// fp16 ring values, run the far part and the near part (each with its lse)
// and merge them into out (and lse when requested).
fa_status prefill_split(const float *q, const void *k, const void *v, float *out, float *lse,
                        int pos0, int n, int hq, int hkv, int hd, int sink, int win,
                        const fa::PlaneGeom &g, int shadow_sink, int shadow_win, uint8_t *ws,
                        const PrefillWs &w, __half *qh, __half *kh, __half *vh,
                        uint8_t *tile_map, unsigned *err, cudaStream_t s) {
    (void)q;
    const int nk = pos0 + n;
    __half *kh2 = reinterpret_cast<__half *>(ws + w.k2_off);
    __half *vh2 = reinterpret_cast<__half *>(ws + w.v2_off);
    float *o1 = reinterpret_cast<float *>(ws + w.o1_off);
    float *o2 = reinterpret_cast<float *>(ws + w.o2_off);
    float *l1 = reinterpret_cast<float *>(ws + w.l1_off);
    float *l2 = reinterpret_cast<float *>(ws + w.l2_off);
    unsigned *ctr2 = reinterpret_cast<unsigned *>(ws + w.ctr2_off);
    // the ring holds the 256 newest rows (ring liveness): near keys start at F
    const int F = nk - FA_Q4_RING_ROWS > shadow_sink ? nk - FA_Q4_RING_ROWS : shadow_sink;
    cudaError_t e = fa::launch_stage_kv(static_cast<const uint8_t *>(k),
                                        static_cast<const uint8_t *>(v), kh2, vh2, nk, g,
                                        shadow_sink, FA_Q4_RING_ROWS, nullptr, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(ctr2, 0, sizeof(unsigned), s);
    fa::PrefillArgs a;
    a.qh = qh;
    a.kv_rows = nk;
    a.pos0 = pos0;
    a.n = n;
    a.n_q_heads = hq;
    a.n_kv_heads = hkv;
    a.head_dim = hd;
    a.sink = sink;
    a.win = win;
    a.scale = 1.0f / sqrtf(static_cast<float>(hd));
    a.split_f = F;
    a.split_w = shadow_win;
    // far part (the work counter was zeroed by the Q staging)
    a.kh = kh;
    a.vh = vh;
    a.out = o1;
    a.lse = l1;
    a.tile_map = tile_map;
    a.work_counter = reinterpret_cast<unsigned *>(ws + w.ctr_off);
    a.split = 1;
    set_q_staging(&a, q, ws, w);
    if (e == cudaSuccess) e = record_start(s);
    if (e == cudaSuccess) e = fa::launch_prefill_tc(a, err, s);
    // near part
    a.kh = kh2;
    a.vh = vh2;
    a.out = o2;
    a.lse = l2;
    a.tile_map = nullptr;
    a.work_counter = ctr2;
    a.split = 2;
    a.q = nullptr;  // the far part left every Q tile staged
    if (e == cudaSuccess) e = fa::launch_prefill_tc(a, err, s);
    if (e == cudaSuccess) e = record_stop(s);
    if (e == cudaSuccess)
        e = fa::launch_merge_attn_states(out, lse, o1, l1, o2, l2, n, hq, hd, -1, s);
    return from_cuda(e);
}

}  // namespace

namespace fa {

bool plane_geom(int fmt, int n_kv, int max_seq, int hd, PlaneGeom *g) {
    if (n_kv < 1 || max_seq < 1 || hd < 32 || hd % 32) return false;
    if (!known_fmt(fmt)) return false;
    g->fmt = fmt;
    g->n_kv = n_kv;
    g->max_seq = max_seq;
    g->hd = hd;
    switch (fmt) {
        case FA_KV_F32: g->row_bytes = static_cast<size_t>(hd) * 4; break;
        case FA_KV_F16: g->row_bytes = static_cast<size_t>(hd) * 2; break;
        case FA_KV_FP8_E4M3: g->row_bytes = static_cast<size_t>(hd); break;
        default: g->row_bytes = static_cast<size_t>(hd / kQ4Block) * kQ4BlockBytes; break;
    }
    g->body_off = 0;
    const size_t body = up256(static_cast<size_t>(n_kv) * max_seq * g->row_bytes);
    g->sink_off = 0;
    g->ring_off = 0;
    g->scale_off = 0;
    g->bytes = body;
    if (fmt == FA_KV_Q4_0) {
        g->sink_off = body;
        g->ring_off = body + up256(static_cast<size_t>(n_kv) * kSinkMax * hd * 2);
        g->bytes = g->ring_off + up256(static_cast<size_t>(n_kv) * kRingRows * hd * 2);
    } else if (fmt == FA_KV_FP8_E4M3) {
        g->scale_off = body;
        g->bytes = body + 256;
    }
    return true;
}

int device_sm_count() {
    DeviceInfo *d = device_info();
    return (d && d->sms > 0) ? d->sms : 148;
}

unsigned *device_error_word() {
    DeviceInfo *d = device_info();
    return d ? d->err : nullptr;
}

}  // namespace fa

extern "C" {

int fa_version(void) { return 100; }

const char *fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "ok";
        case FA_ERR_INVALID: return "invalid argument";
        case FA_ERR_UNSUPPORTED: return "unsupported shape or format";
        case FA_ERR_CUDA: return "CUDA runtime error";
        case FA_ERR_DEVICE: return "a kernel met invalid device-side data";
        case FA_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
        case FA_ERR_WORKSPACE: return "workspace too small";
    }
    return "unknown status";
}

size_t fa_kv_plane_bytes(int kv_fmt, int n_kv_heads, int max_seq, int head_dim) {
    fa::PlaneGeom g;
    if (!supported_hd(head_dim) || !fa::plane_geom(kv_fmt, n_kv_heads, max_seq, head_dim, &g))
        return 0;
    return g.bytes;
}

fa_status fa_kv_plane_layout(int kv_fmt, int n_kv_heads, int max_seq, int head_dim,
                             size_t *row_bytes, size_t *body_offset, size_t *sink_offset,
                             size_t *ring_offset) {
    fa::PlaneGeom g;
    if (!fa::plane_geom(kv_fmt, n_kv_heads, max_seq, head_dim, &g)) return FA_ERR_INVALID;
    if (!supported_hd(head_dim)) return FA_ERR_UNSUPPORTED;
    if (row_bytes) *row_bytes = g.row_bytes;
    if (body_offset) *body_offset = g.body_off;
    if (sink_offset) *sink_offset = g.sink_off;
    if (ring_offset) *ring_offset = g.ring_off;
    return FA_OK;
}

fa_status fa_kv_init(void *planes, int nslots, int kv_fmt, int n_kv_heads, int max_seq,
                     int head_dim, int shadow_sink, int shadow_win, fa_stream_t stream) {
    if (nslots < 0 || n_kv_heads < 1 || max_seq < 1 || head_dim < 32 || head_dim % 32)
        return FA_ERR_INVALID;
    if (!supported_hd(head_dim)) return FA_ERR_UNSUPPORTED;
    fa_status st = check_shadow(kv_fmt, shadow_sink, shadow_win);
    if (st != FA_OK) return st;
    fa::PlaneGeom g;
    if (!fa::plane_geom(kv_fmt, n_kv_heads, max_seq, head_dim, &g)) return FA_ERR_INVALID;
    if (nslots == 0) return FA_OK;
    if (!planes || !aligned16(planes)) return FA_ERR_INVALID;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(planes, 0, g.bytes * static_cast<size_t>(nslots), s);
    if (e == cudaSuccess && kv_fmt == FA_KV_FP8_E4M3)
        e = fa::launch_kv_set_scale(static_cast<uint8_t *>(planes), nslots, g.bytes, g.scale_off,
                                    1.0f, s);
    return from_cuda(e);
}

size_t fa_kv_scale_offset(int kv_fmt, int n_kv_heads, int max_seq, int head_dim) {
    fa::PlaneGeom g;
    if (!supported_hd(head_dim) || !fa::plane_geom(kv_fmt, n_kv_heads, max_seq, head_dim, &g))
        return 0;
    return g.scale_off;
}

fa_status fa_kv_set_scale(void *planes, int nslots, int kv_fmt, int n_kv_heads, int max_seq,
                          int head_dim, float scale, fa_stream_t stream) {
    if (kv_fmt != FA_KV_FP8_E4M3 || nslots < 0) return FA_ERR_INVALID;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return FA_ERR_INVALID;
    fa::PlaneGeom g;
    if (!fa::plane_geom(kv_fmt, n_kv_heads, max_seq, head_dim, &g)) return FA_ERR_INVALID;
    if (!supported_hd(head_dim)) return FA_ERR_UNSUPPORTED;
    if (nslots == 0) return FA_OK;
    if (!planes || !aligned16(planes)) return FA_ERR_INVALID;
    return from_cuda(fa::launch_kv_set_scale(static_cast<uint8_t *>(planes), nslots, g.bytes,
                                             g.scale_off, scale,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

fa_status fa_kv_append(const float *k_new, const float *v_new, void *k_planes, void *v_planes,
                       const int32_t *pos0, int nslots, int n, int n_kv_heads, int head_dim,
                       int max_seq, int kv_fmt, int shadow_sink, int shadow_win,
                       fa_stream_t stream) {
    if (nslots < 0 || n < 0) return FA_ERR_INVALID;
    if (n_kv_heads < 1 || max_seq < 1 || head_dim < 32 || head_dim % 32) return FA_ERR_INVALID;
    if (!supported_hd(head_dim)) return FA_ERR_UNSUPPORTED;
    fa_status st = check_shadow(kv_fmt, shadow_sink, shadow_win);
    if (st != FA_OK) return st;
    if (n > max_seq) return FA_ERR_INVALID;
    if (nslots == 0 || n == 0) return FA_OK;
    if (!k_new || !v_new || !k_planes || !v_planes || !pos0) return FA_ERR_INVALID;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_planes) || !aligned16(v_planes) ||
        (reinterpret_cast<uintptr_t>(pos0) & 3u))
        return FA_ERR_INVALID;
    fa::PlaneGeom g;
    if (!fa::plane_geom(kv_fmt, n_kv_heads, max_seq, head_dim, &g)) return FA_ERR_INVALID;
    DeviceInfo *d = device_info();
    if (!d || !d->err) return FA_ERR_CUDA;
    return from_cuda(fa::launch_kv_append(k_new, v_new, static_cast<uint8_t *>(k_planes),
                                          static_cast<uint8_t *>(v_planes), pos0, nslots, n, g,
                                          shadow_sink, shadow_win, d->err,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

size_t fa_prefill_workspace_bytes(int n, int n_q_heads, int n_kv_heads, int head_dim) {
    return fa_prefill_chunk_workspace_bytes(0, n, n_q_heads, n_kv_heads, head_dim);
}

size_t fa_prefill_chunk_workspace_bytes(int pos0, int n, int n_q_heads, int n_kv_heads,
                                        int head_dim) {
    if (pos0 < 0 || n < 0 || n_q_heads < 1 || n_kv_heads < 1 || head_dim < 1) return 0;
    return prefill_ws(n, pos0 + n, n_q_heads, n_kv_heads, head_dim).bytes;
}

size_t fa_prefill_chunk_workspace_bytes_for(int pos0, int n, int n_q_heads, int n_kv_heads,
                                            int head_dim, int kv_fmt, int shadow_win) {
    if (pos0 < 0 || n < 0 || n_q_heads < 1 || n_kv_heads < 1 || head_dim < 1) return 0;
    return prefill_ws(n, pos0 + n, n_q_heads, n_kv_heads, head_dim,
                      split_prefill(kv_fmt, shadow_win))
        .bytes;
}

fa_status fa_prefill_tile_shape(int head_dim, int *bq, int *bk) {
    if (!supported_hd(head_dim)) return FA_ERR_UNSUPPORTED;
    if (bq) *bq = fa::kPrefillBQ;
    if (bk) *bk = fa::kPrefillBK;
    return FA_OK;
}

fa_status fa_prefill(const float *q, const void *k, const void *v, float *out, int n,
                     int n_q_heads, int n_kv_heads, int head_dim, int sink, int win, int kv_fmt,
                     int max_seq, int shadow_sink, int shadow_win, void *workspace,
                     size_t workspace_bytes, uint8_t *tile_map, fa_stream_t stream) {
    return fa_prefill_lse(q, k, v, out, nullptr, n, n_q_heads, n_kv_heads, head_dim, sink, win,
                          kv_fmt, max_seq, shadow_sink, shadow_win, workspace, workspace_bytes,
                          tile_map, stream);
}

fa_status fa_prefill_lse(const float *q, const void *k, const void *v, float *out, float *lse,
                         int n, int n_q_heads, int n_kv_heads, int head_dim, int sink, int win,
                         int kv_fmt, int max_seq, int shadow_sink, int shadow_win,
                         void *workspace, size_t workspace_bytes, uint8_t *tile_map,
                         fa_stream_t stream) {
    return fa_prefill_chunk(q, k, v, out, lse, 0, n, n_q_heads, n_kv_heads, head_dim, sink, win,
                            kv_fmt, max_seq, shadow_sink, shadow_win, workspace,
                            workspace_bytes, tile_map, stream);
}

fa_status fa_prefill_chunk(const float *q, const void *k, const void *v, float *out, float *lse,
                           int pos0, int n, int n_q_heads, int n_kv_heads, int head_dim,
                           int sink, int win, int kv_fmt, int max_seq, int shadow_sink,
                           int shadow_win, void *workspace, size_t workspace_bytes,
                           uint8_t *tile_map, fa_stream_t stream) {
    fa_status st = check_heads(n_q_heads, n_kv_heads, head_dim);
    if (st != FA_OK) return st;
    if (pos0 < 0 || n < 0 || sink < 0 || max_seq < 1 || n > max_seq || pos0 > max_seq - n)
        return FA_ERR_INVALID;
    st = check_shadow(kv_fmt, shadow_sink, shadow_win);
    if (st != FA_OK) return st;
    const bool split = split_prefill(kv_fmt, shadow_win);
    if (n == 0) return FA_OK;
    if (!q || !k || !v || !out || !workspace) return FA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
        !aligned16(workspace) || (reinterpret_cast<uintptr_t>(lse) & 3u))
        return FA_ERR_INVALID;
    const int nk = pos0 + n;  // key rows 0 .. pos0+n-1
    const PrefillWs w = prefill_ws(n, nk, n_q_heads, n_kv_heads, head_dim, split);
    if (workspace_bytes < w.bytes) return FA_ERR_WORKSPACE;
    fa::PlaneGeom g;
    if (!fa::plane_geom(kv_fmt, n_kv_heads, max_seq, head_dim, &g)) return FA_ERR_INVALID;
    DeviceInfo *d = device_info();
    if (!d || !d->err) return FA_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    __half *qh = reinterpret_cast<__half *>(ws + w.q_off);
    __half *kh = reinterpret_cast<__half *>(ws + w.k_off);
    __half *vh = reinterpret_cast<__half *>(ws + w.v_off);
    unsigned *ctr = reinterpret_cast<unsigned *>(ws + w.ctr_off);
    // Q rows of the query tiles the prefill kernel's first wave covers are
    // staged here; the kernel converts the rest while it runs
    const int units = ((n + fa::kPrefillBQ - 1) / fa::kPrefillBQ) * n_q_heads;
    const int w0 = fa::prefill_units_staged_first(pos0, n, n_q_heads, sink, win);
    const size_t row0 = static_cast<size_t>(units - w0) / n_q_heads * fa::kPrefillBQ;
    const size_t row_vals = static_cast<size_t>(n_q_heads) * head_dim;
    fa::QStageArgs qs;
    qs.q = q + row0 * row_vals;
    qs.qh = qh + row0 * row_vals;
    qs.count = (static_cast<size_t>(n) - row0) * row_vals;
    qs.work_counter = ctr;
    qs.stage_counter = reinterpret_cast<unsigned *>(ws + w.qctr_off);
    qs.flags = reinterpret_cast<unsigned *>(ws + w.flag_off);
    qs.n_flags = units - w0;
    cudaError_t e = cudaSuccess;
    // An fp16 cache body is already the kernel's operand layout ([Hkv][rows]
    // [hd] binary16): the kernel's tensor maps read the planes in place.
    const bool direct = kv_fmt == FA_KV_F16;
    if (direct) {
        kh = reinterpret_cast<__half *>(static_cast<uint8_t *>(const_cast<void *>(k)) + g.body_off);
        vh = reinterpret_cast<__half *>(static_cast<uint8_t *>(const_cast<void *>(v)) + g.body_off);
        e = fa::launch_stage_q(qs, s);
    } else {
        // one launch stages Q's first rows (and zeroes the counters and
        // flags), K and V; the split's far part reads sinks and Q4_0 rows
        // (no ring), the other paths what the shadow geometry gives every query
        const int sw_stage = split ? 0 : shadow_win;
        e = fa::launch_stage_kv(static_cast<const uint8_t *>(k), static_cast<const uint8_t *>(v),
                                kh, vh, nk, g, shadow_sink, sw_stage, &qs, s);
    }
    if (e != cudaSuccess) return FA_ERR_CUDA;
    if (split) return prefill_split(q, k, v, out, lse, pos0, n, n_q_heads, n_kv_heads, head_dim,
                                    sink, win, g, shadow_sink, shadow_win, ws, w, qh, kh, vh,
                                    tile_map, d->err, s);
    fa::PrefillArgs a;
    a.qh = qh;
    a.kh = kh;
    a.vh = vh;
    a.kv_rows = direct ? max_seq : nk;
    a.out = out;
    a.tile_map = tile_map;
    a.work_counter = ctr;
    a.lse = lse;
    a.pos0 = pos0;
    a.n = n;
    a.n_q_heads = n_q_heads;
    a.n_kv_heads = n_kv_heads;
    a.head_dim = head_dim;
    a.sink = sink;
    a.win = win;
    a.scale = 1.0f / sqrtf(static_cast<float>(head_dim));
    a.prefetch_kv = direct;
    set_q_staging(&a, q, ws, w);
    e = record_start(s);
    if (e == cudaSuccess) e = fa::launch_prefill_tc(a, d->err, s);
    if (e == cudaSuccess) e = record_stop(s);
    return from_cuda(e);
}

size_t fa_decode_workspace_bytes(int nslots, int n_q_heads, int head_dim, int max_splits) {
    if (nslots < 1 || n_q_heads < 1 || head_dim < 1 || max_splits < 1) return 0;
    return fa::decode_ws_bytes(nslots, n_q_heads, head_dim, max_splits + 1);
}

fa_status fa_decode(const float *q, const void *k_planes, const void *v_planes,
                    const int32_t *pos, int nslots, int n_q_heads, int n_kv_heads, int head_dim,
                    int max_seq, int sink, int win, int kv_fmt, int shadow_sink, int shadow_win,
                    int split_keys, int max_splits, void *workspace, size_t workspace_bytes,
                    fa_stream_t stream) {
    fa_status st = check_heads(n_q_heads, n_kv_heads, head_dim);
    if (st != FA_OK) return st;
    if (nslots < 0 || sink < 0 || max_seq < 1 || split_keys < 1 || max_splits < 1)
        return FA_ERR_INVALID;
    st = check_shadow(kv_fmt, shadow_sink, shadow_win);
    if (st != FA_OK) return st;
    if (nslots == 0) return FA_OK;
    if (!q || !k_planes || !v_planes || !pos || !workspace) return FA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k_planes) || !aligned16(v_planes) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(pos) & 3u))
        return FA_ERR_INVALID;
    if (workspace_bytes < fa::decode_ws_bytes(nslots, n_q_heads, head_dim, max_splits + 1))
        return FA_ERR_WORKSPACE;
    fa::PlaneGeom g;
    if (!fa::plane_geom(kv_fmt, n_kv_heads, max_seq, head_dim, &g)) return FA_ERR_INVALID;
    DeviceInfo *d = device_info();
    if (!d || !d->err) return FA_ERR_CUDA;
    fa::DecodeWs ws;
    fa::decode_ws_carve(workspace, nslots, n_q_heads, head_dim, max_splits + 1, &ws);
    const fa::DecodeShape shape = fa::decode_shape(nslots, n_q_heads, n_kv_heads, kv_fmt,
                                                   shadow_sink, shadow_win, max_splits, max_seq,
                                                   g.row_bytes);
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
    a.workspace = workspace;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = record_start(s);
    if (e == cudaSuccess) e = fa::launch_decode(a, ws, shape, d->err, s);
    if (e == cudaSuccess) e = record_stop(s);
    return from_cuda(e);
}

fa_status fa_decode_combine(const void *workspace, float *out, int nslots, int n_q_heads,
                            int head_dim, int max_splits, fa_stream_t stream) {
    if (nslots < 0 || n_q_heads < 1 || max_splits < 1) return FA_ERR_INVALID;
    if (!supported_hd(head_dim)) return head_dim % 32 ? FA_ERR_INVALID : FA_ERR_UNSUPPORTED;
    if (nslots == 0) return FA_OK;
    if (!workspace || !out || !aligned16(workspace) || !aligned16(out)) return FA_ERR_INVALID;
    DeviceInfo *d = device_info();
    if (!d || !d->err) return FA_ERR_CUDA;
    return from_cuda(fa::launch_combine(workspace, out, nslots, n_q_heads, head_dim,
                                        max_splits + 1, d->err,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

fa_status fa_set_kernel_events(void *start, void *stop) {
    g_ev_start = static_cast<cudaEvent_t>(start);
    g_ev_stop = static_cast<cudaEvent_t>(stop);
    return FA_OK;
}

fa_status fa_get_device_error(fa_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return FA_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_fa_device_error, sizeof(v)) != cudaSuccess) return FA_ERR_CUDA;
    if (v) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_fa_device_error, &zero, sizeof(zero)) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    if (v & FA_ERRBIT_TIMEOUT) return FA_ERR_TIMEOUT;
    if (v & FA_ERRBIT_DEVICE) return FA_ERR_DEVICE;
    return FA_OK;
}

}  // extern "C"

fa_status fa_merge_attn_states(float *out, float *out_lse, const float *prefix,
                               const float *prefix_lse, const float *suffix,
                               const float *suffix_lse, int num_tokens, int n_heads, int head_dim,
                               int prefill_tokens_with_context, fa_stream_t stream) {
    if (num_tokens < 0 || n_heads < 1 || head_dim < 4 || head_dim % 4) return FA_ERR_INVALID;
    if (num_tokens == 0) return FA_OK;
    if (!out || !prefix || !prefix_lse || !suffix || !suffix_lse) return FA_ERR_INVALID;
    if (!aligned16(out) || !aligned16(prefix) || !aligned16(suffix) ||
        (reinterpret_cast<uintptr_t>(prefix_lse) & 3u) ||
        (reinterpret_cast<uintptr_t>(suffix_lse) & 3u) ||
        (reinterpret_cast<uintptr_t>(out_lse) & 3u))
        return FA_ERR_INVALID;
    return from_cuda(fa::launch_merge_attn_states(
        out, out_lse, prefix, prefix_lse, suffix, suffix_lse, num_tokens, n_heads, head_dim,
        prefill_tokens_with_context, reinterpret_cast<cudaStream_t>(stream)));
}
