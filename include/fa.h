/*
 * fa.h -- C ABI of the GB300 (sm_103a) causal grouped-query flash attention
 * library (libfa.so).
 *
 * What it computes (pages cited by title and section):
 *   "attention.cu" (Foundry cuda_kernels), file header: causal GQA attention
 *   softmax(scale * q k^T) v computed tile by tile with an online softmax
 *   (running max m, running sum l, rescaled accumulator), never materialising
 *   the n x n score matrix; q head h reads kv head h / (n_q_heads/n_kv_heads)
 *   ("vt/ops.h", vt::Attention). The attended set of the query at position p
 *   is every key j <= p when win <= 0, else [0, sink) U [p - win + 1, p].
 *
 * Conventions shared by every call:
 *   - All data pointers are DEVICE pointers, 16-byte aligned, owned by the
 *     caller. The library allocates no memory.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and never synchronises the host, except
 *     fa_get_device_error.
 *   - Argument errors are returned before anything is launched. Conditions
 *     that depend on device data (a position read from device memory out of
 *     range, a workspace header that does not match) are recorded in a device
 *     error word instead; the offending rows are skipped, never written out of
 *     bounds. fa_get_device_error reads and clears that word.
 *   - Floating-point inputs must be finite and within the binary16 range
 *     (|x| < 65504): the tensor-core path computes in fp16 with fp32
 *     accumulation. This is documented, not checked.
 *   - Supported shapes: head_dim in {64, 128, 256}; n_q_heads a multiple of
 *     n_kv_heads with group size n_q_heads/n_kv_heads in {1, 2, 4, 8, 16}.
 *     Others return FA_ERR_UNSUPPORTED.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers. */
typedef struct CUstream_st *fa_stream_t;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID = 1,     /* bad argument: null/misaligned pointer, bad size */
    FA_ERR_UNSUPPORTED = 2, /* valid but not built: head_dim, group, shadow geometry */
    FA_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed */
    FA_ERR_DEVICE = 4,      /* a kernel met bad device-side data (see fa_get_device_error) */
    FA_ERR_TIMEOUT = 5,     /* a kernel gave up a bounded wait and returned early */
    FA_ERR_WORKSPACE = 6    /* workspace too small */
} fa_status;

/* KV cache formats. */
enum {
    FA_KV_F32 = 0,     /* rows of head_dim fp32 values */
    FA_KV_Q4_0 = 1,    /* rows of head_dim/32 Q4_0 blocks of 18 bytes, plus fp16 shadows */
    FA_KV_F16 = 2,     /* rows of head_dim binary16 values */
    FA_KV_FP8_E4M3 = 3 /* rows of head_dim fp8 e4m3fn bytes, plus the plane's fp32 scale */
};

/* Q4_0 fp16 shadow capacity ("attention.cu", 4-bit KV cache section): up to 8
 * sink rows, and a ring of the 256 most recently appended rows. */
#define FA_Q4_SINK_MAX 8
#define FA_Q4_RING_ROWS 256

/* ------------------------------------------------------------------ KV planes
 *
 * A KV plane is one slot's K (or V) cache: one contiguous device buffer of
 * fa_kv_plane_bytes() bytes (a multiple of 256). Several slots are
 * consecutive planes. Layout inside a plane, offsets from
 * fa_kv_plane_layout():
 *
 *   body  [n_kv_heads][max_seq][row_bytes]   row of position s of kv head g
 *         F32:  row_bytes = head_dim * 4, fp32 values
 *         Q4_0: row_bytes = head_dim / 32 * 18. Block b of a row covers
 *               elements [32b, 32b+32): bytes 0-1 are the binary16 scale d,
 *               little-endian; byte 2+j holds the 4-bit code of element j in
 *               its low nibble and of element j+16 in its high nibble; code c
 *               decodes to (c - 8) * d ("attention.cu", 4-bit KV cache).
 *   sink  [n_kv_heads][FA_Q4_SINK_MAX][head_dim] binary16  (Q4_0 only)
 *         position s < shadow_sink, rounded to nearest even.
 *   ring  [n_kv_heads][FA_Q4_RING_ROWS][head_dim] binary16 (Q4_0 only)
 *         position s in slot s % 256 while s is among the 256 newest rows.
 *
 *   F16:  row_bytes = head_dim * 2, each value stored as binary16, rounded to
 *         nearest even (the half-width KV cache of "qwen38_batched.rs", the
 *         BQ_KV16 storage: store __float2half, read __half2float).
 *   FP8_E4M3: row_bytes = head_dim, one fp8 e4m3fn byte per value (1 sign,
 *         4 exponent bits with bias 7, 3 mantissa bits, no infinities, 0x7f
 *         and 0xff are NaN, largest finite 448). The plane holds one fp32
 *         scale at fa_kv_scale_offset() (the per-tensor k_scale / v_scale of
 *         "vt/ops.h", PagedAttentionArgs and ReshapeAndCacheFp8): the append
 *         stores byte = e4m3(x / scale), rounded to nearest even and
 *         saturated to +-448; readers see float(byte) * scale.
 *
 * The bytes are an interface: a host can read or write a plane directly
 * (a checkpoint of the cache is a copy of its planes).
 */

/* Bytes of one plane, or 0 for an invalid/unsupported geometry. */
size_t fa_kv_plane_bytes(int kv_fmt, int n_kv_heads, int max_seq, int head_dim);

/* Offsets of the parts of a plane; sink/ring offsets are 0 for every format
 * but FA_KV_Q4_0.
 * Any output pointer may be NULL. */
fa_status fa_kv_plane_layout(int kv_fmt, int n_kv_heads, int max_seq, int head_dim,
                             size_t *row_bytes, size_t *body_offset, size_t *sink_offset,
                             size_t *ring_offset);

/* Prepare nslots consecutive planes for a new sequence: every byte zero
 * (rows never appended read as 0; Q4_0 shadows empty) and, for
 * FA_KV_FP8_E4M3, the scale 1.0 (the uncalibrated default; fa_kv_set_scale
 * changes it). The planes keep no record of the geometry: every later call
 * on them passes the same (kv_fmt, n_kv_heads, max_seq, head_dim) and the
 * same shadow geometry, which this call validates (FA_ERR_INVALID /
 * FA_ERR_UNSUPPORTED as fa_kv_append). Asynchronous on stream; capturable. */
fa_status fa_kv_init(void *planes, int nslots, int kv_fmt, int n_kv_heads, int max_seq,
                     int head_dim, int shadow_sink, int shadow_win, fa_stream_t stream);

/* Offset of the fp32 scale inside an FA_KV_FP8_E4M3 plane (the body rounded
 * up to 256 bytes), or 0 for the other formats and invalid geometries. */
size_t fa_kv_scale_offset(int kv_fmt, int n_kv_heads, int max_seq, int head_dim);

/* Set the scale of nslots consecutive FA_KV_FP8_E4M3 planes (the K planes
 * take k_scale, the V planes v_scale: one call for each). Set it before the
 * first append: rows stored under one scale and read under another are
 * misread. scale must be finite and > 0, else FA_ERR_INVALID. Asynchronous
 * on stream (a kernel writes the value, so the call can be captured). */
fa_status fa_kv_set_scale(void *planes, int nslots, int kv_fmt, int n_kv_heads, int max_seq,
                          int head_dim, float scale, fa_stream_t stream);

/* Append n new K/V rows to each of nslots caches ("attention.cu",
 * fc_attn_kv_append, fc_attn_kv_append_q4, fc_attn_kv_append_slots_q4).
 *
 *   k_new, v_new  [nslots][n][n_kv_heads][head_dim] fp32 (device).
 *   k_planes,     nslots consecutive planes each (device), laid out as above.
 *   v_planes
 *   pos0          [nslots] int32 (DEVICE memory): row t of slot u lands at
 *                 position pos0[u] + t. Rows with pos0[u] < 0 or
 *                 pos0[u] + t >= max_seq are skipped and flag FA_ERR_DEVICE.
 *   kv_fmt        FA_KV_F32: rows are copied.
 *                 FA_KV_F16: each value rounded to binary16, nearest even.
 *                 FA_KV_FP8_E4M3: each value x of a plane with scale c
 *                 becomes e4m3(x / c) (IEEE fp32 division, nearest even,
 *                 saturating to +-448; NaN stays NaN). A plane whose scale
 *                 is not finite and > 0 is not written and flags
 *                 FA_ERR_DEVICE.
 *                 FA_KV_Q4_0: each 32-element block is quantised: amax =
 *                 max |x| (NaN ignored), d = amax / -8, id = d != 0 ? 1/d : 0,
 *                 code = clamp(round_half_even(x * id) + 8, 0, 15) with the
 *                 saturating float->int32 conversion (NaN -> 0) and a
 *                 wrapping +8, scale stored as binary16(d) ("attention.cu",
 *                 fc_kvq4_quant_block). Rows at positions < shadow_sink are
 *                 also written to the fp16 sink; when shadow_win > 0 the rows
 *                 of this call that remain among the 256 newest are written to
 *                 the fp16 ring.
 *   shadow_sink   0..8 (Q4_0; must be 0 for the other formats).
 *   shadow_win    0..256 (Q4_0; must be 0 for the other formats). Readers must pass the same
 *                 shadow geometry as the appends that built the cache.
 */
fa_status fa_kv_append(const float *k_new, const float *v_new, void *k_planes, void *v_planes,
                       const int32_t *pos0, int nslots, int n, int n_kv_heads, int head_dim,
                       int max_seq, int kv_fmt, int shadow_sink, int shadow_win,
                       fa_stream_t stream);

/* ------------------------------------------------------------------ prefill */

/* Workspace bytes fa_prefill needs (its work queues, one Q-ready flag per
 * (query tile, q head), the fp16 staging of Q, K and V) for every cache
 * but a Q4_0 one whose shadow window is neither 0 nor FA_Q4_RING_ROWS; that
 * case needs fa_prefill_chunk_workspace_bytes_for(). */
size_t fa_prefill_workspace_bytes(int n, int n_q_heads, int n_kv_heads, int head_dim);

/* Tile geometry of the prefill kernel for a head_dim: query rows per tile
 * (*bq) and keys per tile (*bk). Returns FA_ERR_UNSUPPORTED for other
 * head_dim. */
fa_status fa_prefill_tile_shape(int head_dim, int *bq, int *bk);

/* Causal GQA prefill of n tokens at positions 0..n-1 over the first n rows of
 * one cache ("attention.cu", fc_attn_flash_prefill / _q4; the signature
 * follows fa_prefill(q, k, v, out, n, n_q_heads, n_kv_heads, head_dim, sink,
 * win, kv_fmt) with the cache geometry, workspace and stream appended).
 *
 *   q          [n][n_q_heads][head_dim] fp32 (device).
 *   k, v       one plane each (device), rows 0..n-1 appended; the last
 *              appended row is n-1.
 *   out        [n][n_q_heads][head_dim] fp32 (device), written.
 *   sink, win  the attended set: win <= 0 full causal; else keys
 *              [0, sink) U [p - win + 1, p] for the query at p. Key tiles
 *              outside it are skipped before any load; boundary tiles are
 *              masked key by key.
 *   kv_fmt     FA_KV_F32, FA_KV_F16, FA_KV_FP8_E4M3 (the plane's scale
 *              applied on read) or FA_KV_Q4_0. A Q4_0 key s is read from its fp16
 *              copy when s < shadow_sink, or when shadow_win > 0 and s is in
 *              the shadow window of the query and still in the ring
 *              ("attention.cu", fc_kvq4_is_fp16 and the ring liveness floor
 *              of fc_attn_flash_prefill_q4). For shadow_win in {0, 256} that
 *              rule depends on s alone; for other windows it depends on the
 *              query too, and the prefill runs in two merged parts (see
 *              fa_prefill_chunk_workspace_bytes_for for the workspace).
 *   max_seq    row capacity of the planes (n <= max_seq).
 *   workspace  >= fa_prefill_workspace_bytes() bytes of device memory; its
 *              contents are scratch and need no initialisation. Calls that
 *              share a workspace must not overlap on the GPU.
 *   tile_map   NULL, or [ceil(n/bq)][ceil(n/bk)] bytes (device) the kernel sets
 *              to 1 for every (query tile, key tile) it visits. Bytes of
 *              tiles it skips are left untouched (clear them first).
 */
fa_status fa_prefill(const float *q, const void *k, const void *v, float *out, int n,
                     int n_q_heads, int n_kv_heads, int head_dim, int sink, int win,
                     int kv_fmt, int max_seq, int shadow_sink, int shadow_win,
                     void *workspace, size_t workspace_bytes, uint8_t *tile_map,
                     fa_stream_t stream);

/* fa_prefill that also writes the log-sum-exp of every query row's scores,
 * the second input of fa_merge_attn_states ("vt/ops.h" MergeAttnStates):
 *   lse[h][t] = log sum_{j in S(t)} exp(scale * q[t][h] . k[j])   (natural log)
 *   lse        [n_q_heads][n] fp32 (device, 4-byte aligned), written; NULL
 *              makes this call fa_prefill.
 * Every other argument, requirement and status is fa_prefill's. */
fa_status fa_prefill_lse(const float *q, const void *k, const void *v, float *out, float *lse,
                         int n, int n_q_heads, int n_kv_heads, int head_dim, int sink, int win,
                         int kv_fmt, int max_seq, int shadow_sink, int shadow_win,
                         void *workspace, size_t workspace_bytes, uint8_t *tile_map,
                         fa_stream_t stream);

/* Prefill of a chunk: n queries at positions pos0 .. pos0+n-1 over the cache
 * rows 0 .. pos0+n-1 (the rows of the chunk already appended at pos0..), the
 * continuation of a prefill in pieces ("attention.cu", the pos0 of
 * fc_attn_flash_prefill; no ring wrap: pos0 + n <= max_seq).
 *   q, out     [n][n_q_heads][head_dim] fp32 (device): query row t is at
 *              position pos0 + t.
 *   lse        [n_q_heads][n] fp32 or NULL, as for fa_prefill_lse.
 *   workspace  >= fa_prefill_chunk_workspace_bytes_for(pos0, n, ..., kv_fmt,
 *              shadow_win) bytes (FA_ERR_WORKSPACE otherwise).
 *   tile_map   NULL, or [ceil(n/bq)][ceil((pos0+n)/bk)] bytes, as for
 *              fa_prefill with query tiles over the chunk's rows.
 * A Q4_0 key s >= shadow_sink is read from the fp16 ring by the query at p
 * when s >= pos0 + n - 256 (it is still in the ring) and s > p - shadow_win;
 * with shadow_win = 256 that holds for every query. pos0 = 0 is
 * fa_prefill_lse. FA_ERR_INVALID if pos0 < 0 or pos0 + n > max_seq;
 * otherwise fa_prefill's checks and statuses. */
/* Workspace bytes of fa_prefill_chunk (and fa_prefill, pos0 = 0) for the given
 * cache format and shadow window. A Q4_0 cache whose shadow window is neither
 * 0 nor FA_Q4_RING_ROWS runs the prefill in two parts (keys read from the fp16
 * ring, the other keys), each with its log-sum-exp, merged as
 * fa_merge_attn_states does; this needs a second K/V staging and the parts'
 * outputs. For every other case the value equals
 * fa_prefill_chunk_workspace_bytes(). 0 for invalid sizes. */
size_t fa_prefill_chunk_workspace_bytes_for(int pos0, int n, int n_q_heads, int n_kv_heads,
                                            int head_dim, int kv_fmt, int shadow_win);

size_t fa_prefill_chunk_workspace_bytes(int pos0, int n, int n_q_heads, int n_kv_heads,
                                        int head_dim);
fa_status fa_prefill_chunk(const float *q, const void *k, const void *v, float *out, float *lse,
                           int pos0, int n, int n_q_heads, int n_kv_heads, int head_dim,
                           int sink, int win, int kv_fmt, int max_seq, int shadow_sink,
                           int shadow_win, void *workspace, size_t workspace_bytes,
                           uint8_t *tile_map, fa_stream_t stream);

/* ------------------------------------------------------- attention-state merge
 *
 * Merge of two attention results over disjoint key sets by their log-sum-exps
 * ("vt/ops.h" (vllm-cpp-sys), MergeAttnStates, after section 2.2 of the paper
 * it cites): for token t and head h, with lp = prefix_lse[h][t] and
 * ls = suffix_lse[h][t],
 *   - t >= prefill_tokens_with_context (when that is >= 0): out and out_lse
 *     are the suffix's, unchanged;
 *   - an lse of +inf counts as -inf;
 *   - lp = ls = -inf (no key on either side): out = the prefix output,
 *     out_lse = -inf;
 *   - otherwise m = max(lp, ls), wp = exp(lp - m), ws = exp(ls - m):
 *     out = prefix * wp/(wp+ws) + suffix * ws/(wp+ws), out_lse = log(wp+ws) + m.
 * Arithmetic is fp32.
 *   out, prefix, suffix   [num_tokens][n_heads][head_dim] fp32 (device,
 *                         16-byte aligned); out must not overlap the inputs.
 *   out_lse               [n_heads][num_tokens] fp32 (device) or NULL.
 *   prefix_lse, suffix_lse [n_heads][num_tokens] fp32 (device).
 *   head_dim              a multiple of 4.
 * FA_ERR_INVALID for a bad size, a NULL input or a misaligned pointer, before
 * any launch. */
fa_status fa_merge_attn_states(float *out, float *out_lse, const float *prefix,
                               const float *prefix_lse, const float *suffix,
                               const float *suffix_lse, int num_tokens, int n_heads, int head_dim,
                               int prefill_tokens_with_context, fa_stream_t stream);

/* ------------------------------------------------------------------- decode
 *
 * Multi-slot split-KV decode ("attention.cu", "Decode-mode flash attention"
 * and "Multi-user decode attention"). Slot u has one query at position
 * pos[u] and attends rows 0..pos[u] of its own cache, whose last appended row
 * must be pos[u]. Its keys are cut into pieces, and fa_decode writes one
 * partial per (slot, q head, entry) into the workspace. Over fp32 caches (and
 * for groups of 16 q heads) the pieces are runs of consecutive splits of the
 * split plan
 *     ns = clamp(ceil(L / split_keys), 1, max_splits), L = pos[u] + 1,
 *     split_len = roundup16(ceil(L / ns)).
 * Over Q4_0, fp16 and fp8 caches the visible keys of all slots are instead
 * cut into equal shares, one per thread block (or warp), so that every block
 * streams the same number of bytes; a (slot, kv head) then has as many
 * entries as shares it spans, never more than max_splits + 1. Each partial is
 *     m   = max over the entry's visible keys of s_j = scale * q . k_j
 *     l   = sum exp(s_j - m),   acc = sum exp(s_j - m) v_j      (fp32)
 * An entry with no visible key has m = -inf and l = 0 (its acc is not
 * written and never read). fa_decode_combine merges the entries of each head
 * in ascending order: M = max m_e, w_e = exp(m_e - M),
 * out = sum w_e acc_e / sum w_e l_e.
 *
 * A Q4_0 cache's fp16 shadow keys (sinks, recent ring) go to one extra entry
 * per head (the last one). Workspace layout (S = max_splits + 1): a 256-byte
 * header of uint32 words {0x46414443, nslots, n_q_heads, head_dim, E} where E <= S is the
 * number of entries fa_decode wrote per head, then m [nslots*n_q_heads][S] fp32,
 * l [nslots*n_q_heads][S] fp32 and acc [nslots*n_q_heads][S][head_dim] fp32,
 * each part starting 256-byte aligned; entry e of a head is at index e < E.
 */
size_t fa_decode_workspace_bytes(int nslots, int n_q_heads, int head_dim, int max_splits);

/*   q          [nslots][n_q_heads][head_dim] fp32 (device).
 *   k_planes,  nslots consecutive planes each (device).
 *   v_planes
 *   pos        [nslots] int32 (DEVICE memory), 0 <= pos[u] < max_seq; a slot
 *              whose position is out of range gets empty entries and flags
 *              FA_ERR_DEVICE.
 *   sink, win  attended set, as for fa_prefill.
 *   kv_fmt, shadow_sink, shadow_win   cache format and shadow geometry
 *              (shadow_win 0..256; decode reads key s from the ring when
 *              s > pos - shadow_win).
 *   split_keys keys per split of the plan (> 0); max_splits its cap (> 0).
 */
fa_status fa_decode(const float *q, const void *k_planes, const void *v_planes,
                    const int32_t *pos, int nslots, int n_q_heads, int n_kv_heads, int head_dim,
                    int max_seq, int sink, int win, int kv_fmt, int shadow_sink, int shadow_win,
                    int split_keys, int max_splits, void *workspace, size_t workspace_bytes,
                    fa_stream_t stream);

/* Merge the partials fa_decode wrote into out [nslots][n_q_heads][head_dim]
 * fp32 (device). The arguments must match the fa_decode call that filled the
 * workspace; a header mismatch flags FA_ERR_DEVICE and leaves out untouched. */
fa_status fa_decode_combine(const void *workspace, float *out, int nslots, int n_q_heads,
                            int head_dim, int max_splits, fa_stream_t stream);

/* Decode without any caller-provided device memory. The pages have no
 * counterpart to this call; it exists for callers that cannot allocate
 * device memory at all (a plugin inside a host whose allocator owns the
 * GPU's memory, or a serving loop where cudaMalloc/cudaFree are banned because
 * they can synchronise the device). It computes exactly what fa_decode
 * followed by fa_decode_combine computes, writing out [nslots][n_q_heads]
 * [head_dim] fp32 (device), with the same arguments and rules as fa_decode.
 *
 * The partials live in a fixed 8 MiB array in the library's device memory
 * (held by every GPU that loads the library until the process exits), laid
 * out as fa_decode's workspace with the entry stride equal to the number of
 * entries E (for Q4_0, fp16 and fp8 caches, whose kernels can use any number
 * of entries from 2 up (3 with fp16 shadows), E is the largest count up to
 * max_splits + 1 that fits). A problem whose partials need more than 8 MiB
 * (256 + 2*nslots*n_q_heads*E*4 + nslots*n_q_heads*E*head_dim*4 bytes, parts
 * rounded up to 256) returns FA_ERR_WORKSPACE before any launch. The call
 * allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 * Every call shares the array and it keeps the last call's contents; calls
 * that overlap on the GPU (other streams, other host threads on the device)
 * race on it, so serialise them. The first call on each device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture. If that lookup fails the
 * call returns FA_ERR_CUDA, clears the runtime's last error, and the next
 * call looks again. */
fa_status fa_decode_noalloc(const float *q, const void *k_planes, const void *v_planes,
                            const int32_t *pos, int nslots, int n_q_heads, int n_kv_heads,
                            int head_dim, int max_seq, int sink, int win, int kv_fmt,
                            int shadow_sink, int shadow_win, int split_keys, int max_splits,
                            float *out, fa_stream_t stream);

/* ---------------------------------------------------------------- profiling */

/* Optional timing hook. While both events are non-NULL (cudaEvent_t handles
 * created by the caller), every later fa_prefill records `start` on its
 * stream immediately before its tensor-core kernel and `stop` immediately
 * after it, and every fa_decode does the same around its split kernel, so
 * cudaEventElapsedTime(start, stop) is that one kernel's duration. A call
 * captured in a CUDA graph records them as external event nodes, so every
 * replay records them. Pass NULL, NULL to stop. Process-wide setting, not
 * thread-safe; never needed for correctness. */
fa_status fa_set_kernel_events(void *start, void *stop);

/* ------------------------------------------------------------------- status */

/* Synchronise `stream`, then read and clear the device error word of the
 * current device: FA_OK, FA_ERR_DEVICE or FA_ERR_TIMEOUT (or FA_ERR_CUDA if
 * the synchronisation itself failed). */
fa_status fa_get_device_error(fa_stream_t stream);

/* Static description of a status code. */
const char *fa_status_string(fa_status status);

/* Library version: major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
