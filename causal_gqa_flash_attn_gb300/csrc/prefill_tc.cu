// prefill_tc.cu -- causal GQA flash-attention prefill on sm_103a tensor cores.
//
// The method ("attention.cu" (Foundry cuda_kernels), fc_attn_flash_prefill and
// its file header): for every query row, walk the key tiles the row can see,
// score them (S = Q K^T * scale), fold them into a running max m and running
// sum l with an online softmax, and accumulate O = corr * O + P V; the n x n
// score matrix never exists. Key tiles outside [0, sink) U [p - win + 1, p]
// are skipped before anything is loaded (fc_attn_tile_in_window, extended to a
// block of query rows); tiles that straddle a boundary are masked key by key.
//
// GB300 design (one CTA per 128-query tile of one q head, 256 threads):
//   warp 0      TMA producer: Q tile once, then K and V tiles (fp16, 128-byte
//               swizzle) in the order the MMA warp consumes them.
//   warp 1      MMA issuer (one thread): S_i = Q K_i^T into a double-buffered
//               TMEM accumulator (tcgen05.mma, fp16 x fp16 -> fp32), then
//               O += P_{i-1} V_{i-1} with P read from TMEM (A operand in TMEM)
//               and V from shared memory (MN-major B).
//   warps 4-7   softmax, one thread per query row (TMEM lane): tcgen05.ld of
//               S, masking, running max in the exp2 domain (scale * log2 e
//               folded into one FMA), P packed to fp16 and tcgen05.st back over
//               S; O is rescaled in TMEM only when the max grew by more than
//               2^8 (exact: O and l always share the stale reference), and the
//               epilogue writes O / l.
// TMEM (512 columns): O [0, hd), S/P buffers 0 and 1 of 128 columns each.
// Blocks are issued heaviest query tile first so the hardware scheduler
// balances the causal triangle.
#include <cuda.h>

#include <mutex>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

template <int HD>
struct Cfg {
    static constexpr int BQ = kPrefillBQ;
    static constexpr int BK = kPrefillBK;
    static constexpr int NCHUNK = HD / 64;               // 128-byte chunks along head_dim
    static constexpr uint32_t CHUNK_BYTES = 128 * 128;   // 128 rows x 128 bytes
    static constexpr uint32_t TILE_BYTES = NCHUNK * CHUNK_BYTES;
    static constexpr int NS = (HD == 256) ? 1 : 2;       // K and V stages
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = TILE_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + NS * TILE_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_V + NS * TILE_BYTES;
    static constexpr uint32_t USED = OFF_BAR + 256;
    // at least 120 KB so that one block owns an SM (and all 512 TMEM columns)
    static constexpr uint32_t SMEM = (USED + 1024 > 120u * 1024u) ? USED + 1024 : 120u * 1024u;
    static constexpr uint32_t O_COL = 0;
    static constexpr uint32_t S_COL0 = HD;
    static constexpr uint32_t S_COL1 = HD + 128;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t IDESC_QK = idesc_f16(128, BK, 0, 0);
    static constexpr uint32_t IDESC_PV = idesc_f16(128, HD, 0, 1);
    static_assert(USED + 1024 <= 227u * 1024u, "shared memory");
};

struct Bars {
    uint64_t q_full;
    uint64_t k_full[2], k_empty[2];
    uint64_t v_full[2], v_empty[2];
    uint64_t s_full[2], p_full[2];
    uint64_t o_done;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// Key tiles a query tile [p0, p1] visits, in ascending order: the sink tiles
// [0, ns) then the window tiles [lo, hi] (lo >= ns). Visit iff
//   j0 <= p1 and (win <= 0 or j0 < min(sink, p1+1) or j0+BK-1 >= max(0, p0-win+1)).
struct TilePlan {
    int ns, lo, count;
    __device__ int kt(int i) const { return i < ns ? i : lo + (i - ns); }
};

__device__ __forceinline__ TilePlan tile_plan(int p0, int p1, int sink, int win, int bk) {
    TilePlan t;
    const int hi = p1 / bk;
    if (win <= 0) {
        t.ns = 0;
        t.lo = 0;
        t.count = hi + 1;
        return t;
    }
    const int s_end = min(sink, p1 + 1);
    t.ns = (max(s_end, 0) + bk - 1) / bk;
    const int wlo = max(0, p0 - win + 1);
    t.lo = max(wlo / bk, t.ns);
    t.count = t.ns + max(0, hi - t.lo + 1);
    return t;
}

// Every real row p in [p0, p1] sees every key of tile kt.
__device__ __forceinline__ bool tile_full(int kt, int p0, int p1, int sink, int win, int bk) {
    const int j0 = kt * bk, j1 = j0 + bk - 1;
    if (j1 > p0) return false;
    if (win <= 0) return true;
    if (j1 < sink) return true;
    return j0 >= p1 - win + 1;
}

// Wait ignoring the abort flag (still bounded): used to drain copies and MMAs
// already in flight before the block releases its TMEM and exits.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kSpinCycles) return;
}

template <int HD>
__global__ void __launch_bounds__(256, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, float *__restrict__ out,
                      uint8_t *__restrict__ tile_map, int n, int Hq, int Hkv, int sink, int win,
                      float sl2, unsigned *err) {
    using C = Cfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Bars *bars = reinterpret_cast<Bars *>(smem + C::OFF_BAR);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int nqt = (n + C::BQ - 1) / C::BQ;
    const int nkt = (n + C::BK - 1) / C::BK;
    const int qt = nqt - 1 - static_cast<int>(blockIdx.x / Hq);  // heaviest first
    const int h = static_cast<int>(blockIdx.x % Hq);
    const int g = h / (Hq / Hkv);
    const int p0 = qt * C::BQ;
    const int p1 = min(n, p0 + C::BQ) - 1;
    const TilePlan plan = tile_plan(p0, p1, sink, win, C::BK);
    const int count = plan.count;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], 1);
            mbar_init(&bars->s_full[s], 1);
            mbar_init(&bars->p_full[s], 128);
        }
        mbar_init(&bars->o_done, 1);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    volatile int *abort = &bars->abort;

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            int k_arms[2] = {0, 0}, v_arms[2] = {0, 0};
            mbar_arrive_expect_tx(&bars->q_full, C::TILE_BYTES);
            for (int c = 0; c < C::NCHUNK; ++c)
                tma_load_3d(smem + C::OFF_Q + c * C::CHUNK_BYTES, &tm_q, &bars->q_full, c * 64, h,
                            p0);
            bool ok = true;
            auto load_k = [&](int i) -> bool {
                const int st = i % C::NS;
                if (i >= C::NS &&
                    !mbar_wait(&bars->k_empty[st], ((i / C::NS) - 1) & 1, abort, err))
                    return false;
                const int kt = plan.kt(i);
                mbar_arrive_expect_tx(&bars->k_full[st], C::TILE_BYTES);
                for (int c = 0; c < C::NCHUNK; ++c)
                    tma_load_3d(smem + C::OFF_K + st * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_k,
                                &bars->k_full[st], c * 64, kt * C::BK, g);
                ++k_arms[st];
                if (tile_map) tile_map[static_cast<size_t>(qt) * nkt + kt] = 1;
                return true;
            };
            auto load_v = [&](int i) -> bool {
                const int st = i % C::NS;
                if (i >= C::NS &&
                    !mbar_wait(&bars->v_empty[st], ((i / C::NS) - 1) & 1, abort, err))
                    return false;
                const int kt = plan.kt(i);
                mbar_arrive_expect_tx(&bars->v_full[st], C::TILE_BYTES);
                for (int c = 0; c < C::NCHUNK; ++c)
                    tma_load_3d(smem + C::OFF_V + st * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_v,
                                &bars->v_full[st], c * 64, kt * C::BK, g);
                ++v_arms[st];
                return true;
            };
            // Consumption order of the MMA warp: K0, K1, V0, K2, V1, ...
            for (int i = 0; i < count && ok; ++i) {
                ok = load_k(i);
                if (ok && i >= 1) ok = load_v(i - 1);
            }
            if (ok) ok = load_v(count - 1);
            if (!ok) {  // let every copy already issued land before exit
                drain_wait(&bars->q_full, 0);
                for (int s = 0; s < 2; ++s) {
                    if (k_arms[s]) drain_wait(&bars->k_full[s], (k_arms[s] - 1) & 1);
                    if (v_arms[s]) drain_wait(&bars->v_full[s], (v_arms[s] - 1) & 1);
                }
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t sQ = smem_u32(smem + C::OFF_Q);
            const uint32_t sK = smem_u32(smem + C::OFF_K);
            const uint32_t sV = smem_u32(smem + C::OFF_V);
            auto issue_qk = [&](int i) -> bool {
                const int st = i % C::NS;
                if (!mbar_wait(&bars->k_full[st], (i / C::NS) & 1, abort, err)) return false;
                tc_fence_after();
                const uint32_t d = tmem + ((i & 1) ? C::S_COL1 : C::S_COL0);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
                    const uint64_t a = desc_sw128(sQ + off, 16, 1024);
                    const uint64_t b = desc_sw128(sK + st * C::TILE_BYTES + off, 16, 1024);
                    mma_ss(d, a, b, C::IDESC_QK, kk > 0 ? 1u : 0u);
                }
                tc_commit(&bars->k_empty[st]);
                tc_commit(&bars->s_full[i & 1]);
                return true;
            };
            auto issue_pv = [&](int j) -> bool {
                const int st = j % C::NS;
                if (!mbar_wait(&bars->p_full[j & 1], (j >> 1) & 1, abort, err)) return false;
                if (!mbar_wait(&bars->v_full[st], (j / C::NS) & 1, abort, err)) return false;
                tc_fence_after();
                const uint32_t pcol = tmem + ((j & 1) ? C::S_COL1 : C::S_COL0);
#pragma unroll
                for (int kk = 0; kk < C::BK / 16; ++kk) {
                    // V tile: [128 keys][64 dims] per 16-KB chunk; 16 keys per k-step,
                    // next 64 dims of N one chunk further (LBO), 8-key atoms 1 KB apart (SBO).
                    const uint64_t b = desc_sw128(sV + st * C::TILE_BYTES + kk * 2048,
                                                  C::CHUNK_BYTES, 1024);
                    mma_ts(tmem + C::O_COL, pcol + kk * 8, b, C::IDESC_PV,
                           (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&bars->v_empty[st]);
                tc_commit(&bars->o_done);
                return true;
            };
            bool ok = mbar_wait(&bars->q_full, 0, abort, err);
            if (ok) tc_fence_after();
            for (int i = 0; i < count && ok; ++i) {
                ok = issue_qk(i);
                if (ok && i >= 1) ok = issue_pv(i - 1);
            }
            if (ok) ok = issue_pv(count - 1);
            // every MMA issued must complete before TMEM is released
            tc_commit(&bars->drain);
            drain_wait(&bars->drain, 0);
        }
    } else if (warp >= 4) {
        // ----------------------------------------------------------- softmax
        const int r = threadIdx.x - 128;  // tile row == TMEM lane
        const int p = p0 + r;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        float m_used = -INFINITY;  // exp2-domain reference shared by O and l
        float l = 0.0f;
        bool ok = true;
        for (int i = 0; i < count; ++i) {
            const int b = i & 1;
            ok = mbar_wait(&bars->s_full[b], (i >> 1) & 1, abort, err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t scol = tmem + lane_base + (b ? C::S_COL1 : C::S_COL0);
            uint32_t s[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(scol + 32 * c, s + 32 * c);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 4; ++c) reg_fence32(s + 32 * c);

            const int kt = plan.kt(i);
            const int j0 = kt * C::BK;
            float mx = -INFINITY;
            if (tile_full(kt, p0, p1, sink, win, C::BK)) {
#pragma unroll
                for (int c = 0; c < 128; ++c) mx = fmaxf(mx, __uint_as_float(s[c]));
            } else {
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    float v = __uint_as_float(s[c]);
                    if (!key_visible(p, j0 + c, sink, win)) v = -INFINITY;
                    s[c] = __float_as_uint(v);
                    mx = fmaxf(mx, v);
                }
            }
            const float m_new = fmaxf(m_used, mx * sl2);
            float corr = 1.0f;
            bool resc = false;
            if (m_new > m_used + 8.0f) {
                if (m_used != -INFINITY) {
                    corr = ex2(m_used - m_new);
                    resc = true;
                    l *= corr;
                }
                m_used = m_new;
            }
            const float mref = (m_used == -INFINITY) ? 0.0f : m_used;
            uint32_t pk[64];
            float rs = 0.0f;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                const float a = ex2(fmaf(__uint_as_float(s[2 * c]), sl2, -mref));
                const float bq = ex2(fmaf(__uint_as_float(s[2 * c + 1]), sl2, -mref));
                rs += a + bq;
                pk[c] = pack_half2(a, bq);
            }
            l += rs;
            if (i > 0) {  // O must hold PV_{i-1} before it is rescaled and before P_i lands
                ok = mbar_wait(&bars->o_done, (i - 1) & 1, abort, err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
            }
            tc_fence_after();
            __syncwarp();
            if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
                for (int c = 0; c < HD / 32; ++c) {
                    uint32_t o[32];
                    const uint32_t oc = tmem + lane_base + C::O_COL + 32 * c;
                    tmem_ld32(oc, o);
                    tmem_wait_ld();
                    reg_fence32(o);
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * corr);
                    tmem_st32(oc, o);
                }
            }
            tmem_st32(scol, pk);
            tmem_st32(scol + 32, pk + 32);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars->p_full[b]);
        }
        if (ok) {
            ok = mbar_wait(&bars->o_done, (count - 1) & 1, abort, err);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            tc_fence_after();
            const float inv = 1.0f / l;
            float *orow = out + (static_cast<size_t>(p) * Hq + h) * HD;
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_base + C::O_COL + 32 * c, o);
                tmem_wait_ld();
                reg_fence32(o);
                if (p < n) {
#pragma unroll
                    for (int k = 0; k < 32; k += 4) {
                        float4 v;
                        v.x = __uint_as_float(o[k]) * inv;
                        v.y = __uint_as_float(o[k + 1]) * inv;
                        v.z = __uint_as_float(o[k + 2]) * inv;
                        v.w = __uint_as_float(o[k + 3]) * inv;
                        *reinterpret_cast<float4 *>(orow + 32 * c + k) = v;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// fp16 3-D tensor, 128-byte swizzle, zero fill outside the tensor.
bool encode_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1,
               uint32_t b2) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int HD>
cudaError_t launch_hd(const PrefillArgs &a, unsigned *err, cudaStream_t stream) {
    using C = Cfg<HD>;
    CUtensorMap tq, tk, tv;
    const uint64_t n = a.n, Hq = a.n_q_heads, Hkv = a.n_kv_heads;
    if (!encode_3d(&tq, a.qh, HD, Hq, n, HD * 2, Hq * HD * 2, 64, 1, C::BQ) ||
        !encode_3d(&tk, a.kh, HD, n, Hkv, HD * 2, n * HD * 2, 64, C::BK, 1) ||
        !encode_3d(&tv, a.vh, HD, n, Hkv, HD * 2, n * HD * 2, 64, C::BK, 1))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<HD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const int nqt = (a.n + C::BQ - 1) / C::BQ;
    const float sl2 = a.scale * 1.4426950408889634f;
    prefill_tc_kernel<HD><<<nqt * a.n_q_heads, 256, C::SMEM, stream>>>(
        tq, tk, tv, a.out, a.tile_map, a.n, a.n_q_heads, a.n_kv_heads, a.sink, a.win, sl2, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs &a, unsigned *err, cudaStream_t stream) {
    switch (a.head_dim) {
        case 64: return launch_hd<64>(a, err, stream);
        case 128: return launch_hd<128>(a, err, stream);
        case 256: return launch_hd<256>(a, err, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
