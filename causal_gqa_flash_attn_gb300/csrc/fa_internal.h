// fa_internal.h -- declarations shared by the translation units of libfa.so
// (not part of the public C ABI, which is include/fa.h).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

// Bits of the device error word.
#define FA_ERRBIT_DEVICE 1u   // bad device-side data (a position out of range, header mismatch)
#define FA_ERRBIT_TIMEOUT 2u  // a bounded wait gave up

namespace fa {

constexpr int kQ4Block = 32;       // elements per Q4_0 block
constexpr int kQ4BlockBytes = 18;  // bytes per Q4_0 block
constexpr int kSinkMax = 8;        // fp16 sink rows per kv head
constexpr int kRingRows = 256;     // fp16 ring rows per kv head

// Plane geometry of one slot's K or V cache (see include/fa.h).
struct PlaneGeom {
    int fmt;
    int n_kv;
    int max_seq;
    int hd;
    size_t row_bytes;
    size_t body_off;
    size_t sink_off;   // Q4_0 only
    size_t ring_off;   // Q4_0 only
    size_t scale_off;  // FP8_E4M3 only: the plane's fp32 scale
    size_t bytes;      // whole plane, multiple of 256
};

// Format codes (include/fa.h).
constexpr int kFmtF32 = 0;
constexpr int kFmtQ4 = 1;
constexpr int kFmtF16 = 2;
constexpr int kFmtFp8 = 3;

bool plane_geom(int fmt, int n_kv, int max_seq, int hd, PlaneGeom *g);

// ---- kv_append.cu
cudaError_t launch_kv_set_scale(uint8_t *planes, int nslots, size_t plane_bytes, size_t scale_off,
                                float scale, cudaStream_t stream);
cudaError_t launch_kv_append(const float *k_new, const float *v_new, uint8_t *k_planes,
                             uint8_t *v_planes, const int32_t *pos0, int nslots, int n,
                             const PlaneGeom &g, int shadow_sink, int shadow_win,
                             unsigned *err, cudaStream_t stream);

// ---- prefill_stage.cu: fp16 staging of Q and of the K/V rows a prefill reads
// The part of Q converted before the prefill kernel (the query tiles of its
// first wave of units; the kernel converts the rest itself) and the kernel's
// counters and Q-ready flags, which the same launch zeroes.
struct QStageArgs {
    const float *q = nullptr;  // first element to convert (fp32)
    __half *qh = nullptr;      // its fp16 destination
    size_t count = 0;          // values to convert (a multiple of 4)
    unsigned *work_counter = nullptr;  // the prefill's work queue
    unsigned *stage_counter = nullptr; // the prefill's Q staging queue
    unsigned *flags = nullptr;         // the prefill's Q-ready flags
    int n_flags = 0;
};
cudaError_t launch_stage_q(const QStageArgs &qs, cudaStream_t stream);
// Stages rows 0..n-1 of the K and the V plane into kdst and vdst in one launch;
// when qs is not null the same launch also does launch_stage_q's work.
cudaError_t launch_stage_kv(const uint8_t *kplane, const uint8_t *vplane, __half *kdst,
                            __half *vdst, int n, const PlaneGeom &g, int shadow_sink,
                            int shadow_win, const QStageArgs *qs, cudaStream_t stream);

// ---- prefill_tc.cu
struct PrefillArgs {
    const __half *qh;   // [n][Hq][hd] fp16
    const __half *kh;   // [Hkv][kv_rows][hd] fp16, rows 0 .. pos0+n-1 read
    const __half *vh;   // [Hkv][kv_rows][hd] fp16
    int kv_rows;        // rows per kv head of kh, vh (>= pos0 + n)
    float *out;         // [n][Hq][hd] fp32
    uint8_t *tile_map;  // optional
    unsigned *work_counter;  // prefill work queue, zeroed by launch_stage_q
    float *lse;              // optional [Hq][n] fp32: log sum_j exp(s_j) per row
    int pos0;  // position of query row 0; keys are the cache rows 0 .. pos0+n-1
    int n, n_q_heads, n_kv_heads, head_dim, sink, win;
    float scale;
    // 0: every visible key; 1 / 2: the far / near keys of a Q4_0 cache whose
    // fp16 window split_w is narrower than the ring (near: key >= split_f and
    // key > p - split_w); 1 and 2 need lse
    int split = 0, split_f = 0, split_w = 0;
    // K/V are cache planes read in place (not staged just before): the kernel
    // asks for their rows in L2 at its start
    bool prefetch_kv = false;
    // Q staged by the kernel itself: units w >= q_w0 (heaviest first) have
    // their rows converted from q (fp32 [n][Hq][hd]) into qh by two warps of
    // the kernel, which set q_flags[w - q_w0] once a tile is there
    // (q null: all of Q was staged before the launch)
    const float *q = nullptr;
    unsigned *q_flags = nullptr;
    unsigned *q_stage_counter = nullptr;
    int q_w0 = 0;
};
constexpr int kPrefillBQ = 128;
constexpr int kPrefillBK = 128;
cudaError_t launch_prefill_tc(const PrefillArgs &a, unsigned *err, cudaStream_t stream);
// Blocks of the prefill kernel for n query rows of Hq heads (one per SM, at
// most one per unit), and the units whose Q must be staged before it: the
// whole query tiles that its first wave of units covers (its first two waves
// when those units are short).
int prefill_grid(int n, int Hq);
int prefill_units_staged_first(int pos0, int n, int Hq, int sink, int win);

// 128-byte-swizzled tiled tensor map (rank 1..5, zero fill outside the
// tensor); strides_bytes holds rank-1 entries. False if the driver refuses.
bool encode_tiled(CUtensorMap *m, CUtensorMapDataType dtype, int rank, const void *base,
                  const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box);

// ---- merge.cu
cudaError_t launch_merge_attn_states(float *out, float *out_lse, const float *prefix,
                                     const float *prefix_lse, const float *suffix,
                                     const float *suffix_lse, int T, int H, int D,
                                     int with_context, cudaStream_t stream);

// ---- decode.cu
struct DecodeArgs {
    const float *q;
    const uint8_t *k_planes;
    const uint8_t *v_planes;
    const int32_t *pos;
    int nslots, n_q_heads, n_kv_heads, sink, win, shadow_sink, shadow_win;
    int split_keys, max_splits;
    PlaneGeom g;
    float scale;
    void *workspace;
};
struct DecodeWs {
    uint32_t *header;
    float *m, *l, *acc;
    int stride;  // entry stride per (slot, head)
};
// How fa_decode splits the work: runs of splits_per_cta plan splits per block
// (body_entries blocks per (slot, kv head)), plus one entry for the fp16
// shadow keys when the Q4_0 fast path is used.
struct DecodeShape {
    bool fast;           // Q4_0 kernel (group <= 8, 16-byte aligned K/V rows per head)
    bool dense;          // fp16 / fp8 streaming kernel (decode_dense.cu)
    int splits_per_cta;
    int body_entries;
    int shadow_entry;    // -1 if none
    int entries;         // body_entries + (shadow_entry >= 0)
};
DecodeShape decode_shape(int nslots, int n_q_heads, int n_kv_heads, int kv_fmt, int shadow_sink,
                         int shadow_win, int max_splits, int max_seq, size_t row_bytes);
size_t decode_ws_bytes(int nslots, int n_q_heads, int head_dim, int stride);
// ---- decode_dense.cu: fp16 (head_dim 64..256) and fp8 (128, 256) caches, G <= 8.
// Uses up to ws.stride entries per head (>= 2) and writes the header's count.
bool dense_decode_supported(int kv_fmt, int G, int head_dim);
cudaError_t launch_decode_dense(const DecodeArgs &a, const DecodeWs &ws, unsigned *err,
                                cudaStream_t stream);
void decode_ws_carve(void *ws, int nslots, int n_q_heads, int head_dim, int stride,
                     DecodeWs *out);
cudaError_t launch_decode(const DecodeArgs &a, const DecodeWs &ws, const DecodeShape &d,
                          unsigned *err, cudaStream_t stream);
cudaError_t launch_combine(const void *workspace, float *out, int nslots, int n_q_heads,
                           int head_dim, int stride, unsigned *err, cudaStream_t stream);

constexpr uint32_t kDecodeMagic = 0x46414443u;  // "FADC"

// ---- fa_api.cu
int device_sm_count();
unsigned *device_error_word();  // this device's error word (device address)

}  // namespace fa
