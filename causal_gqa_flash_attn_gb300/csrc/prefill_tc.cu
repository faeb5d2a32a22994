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
//   warps 2-3   Q staging (large prefills): the query tiles past the first
//               wave of units are converted from fp32 to fp16 here, ahead of
//               the units that need them, while the tensor cores run.
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
    // epilogue staging: per softmax warp two boxes of [32 rows][32 fp32]
    static constexpr uint32_t OFF_OST = OFF_V + NS * TILE_BYTES;
    static constexpr uint32_t OST_BYTES = 32 * 128;
    static constexpr uint32_t OFF_BAR = OFF_OST + 4 * 2 * OST_BYTES;
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

constexpr int kUnitRing = 4;

// ------------------------------------------------- flags in global memory
// A producer block publishes data for other blocks: every writing thread
// fences its stores (GPU scope, and towards the async proxy, for TMA readers),
// the writers synchronise, one thread release-stores the flag. A reader
// acquire-loads the flag and fences towards the async proxy before it issues
// TMA copies of the data.

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// After a relaxed load saw a flag set: makes that load an acquire.
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ void st_release_gpu(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Order this thread's generic-proxy global accesses with its async-proxy ones.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Wait until *flag is non-zero: bounded like mbar_wait (timeout recorded, the
// block's abort flag raised, false returned), and false as soon as *abort is.
__device__ __forceinline__ bool flag_wait(const unsigned *flag, volatile int *abort,
                                          unsigned *err) {
    if (ld_acquire_gpu(flag)) return true;
    const long long t0 = clock64();
    for (;;) {
        __nanosleep(256);
        if (ld_acquire_gpu(flag)) return true;
        if (*abort) return false;
        if (clock64() - t0 > kSpinCycles) {
            *abort = 1;
            flag_error(err, FA_ERRBIT_TIMEOUT);
            return false;
        }
    }
}


struct Bars {
    uint64_t q_full, q_empty;
    uint64_t o_free;
    uint64_t unit_full[kUnitRing], unit_empty[kUnitRing];
    int unit_id[kUnitRing];
    uint64_t k_full[2], k_empty[2];
    uint64_t v_full[2], v_empty[2];
    uint64_t s_full[2], p_full[2];
    uint64_t o_done;
    uint64_t o_last;  // the last P.V of a unit finished (one phase per unit)
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// Key tiles a query tile [p0, p1] visits, in ascending order: the sink tiles
// [0, ns) then the window tiles [lo, hi] (lo >= ns). Visit iff
//   j0 <= p1 and (win <= 0 or j0 < min(sink, p1+1) or j0+BK-1 >= max(0, p0-win+1)).
struct TilePlan {
    int ns, lo, count;
    __device__ int kt(int i) const { return i < ns ? i : lo + (i - ns); }
};

__host__ __device__ __forceinline__ TilePlan tile_plan(int p0, int p1, int sink, int win, int bk) {
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

// The tiles a unit visits: the attended set's plan, or for the near part of a
// split the tiles of the window [p - split_w + 1, p].
template <int SPLIT>
__device__ __forceinline__ TilePlan unit_plan(int p0, int p1, int sink, int win, int split_w,
                                              int bk) {
    return SPLIT == 2 ? tile_plan(p0, p1, 0, split_w, bk) : tile_plan(p0, p1, sink, win, bk);
}

// Wait ignoring the abort flag (still bounded): used to drain copies and MMAs
// already in flight before the block releases its TMEM and exits.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kSpinCycles) return;
}

// Work unit w (heaviest first): query tile nqt-1-w/Hq of q head w%Hq. Block b
// starts with unit b; afterwards its producer warp takes the next unit from a
// global counter (zeroed by the staging kernel that runs first) and hands the
// id to the MMA and softmax warps through a small ring in shared memory. Each
// unit is computed by exactly one block, so the result does not depend on the
// schedule.
struct Unit {
    int qt, h;
};

// LSE: also write each row's log-sum-exp (a separate instantiation, so that
// the plain prefill keeps its own register allocation).
// SPLIT (Q4_0 caches whose fp16 window is narrower than the ring): the keys a
// query p sees split into the "near" keys s >= F with s > p - shadow_win,
// read from the fp16 ring, and the rest ("far"), read from the sinks or the
// Q4_0 rows. SPLIT = 1 attends the far keys only (over the usual tile plan),
// SPLIT = 2 the near keys only (over the tiles of the window [p - sw + 1, p]);
// the two results are merged by their log-sum-exps. A row with no key in its
// part gets O = 0 and lse = -inf.
template <int HD, bool LSE, int SPLIT>
__global__ void __launch_bounds__(256, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_o, uint8_t *__restrict__ tile_map,
                      unsigned *__restrict__ work_counter, float *__restrict__ lse, int pos0,
                      int n, int Hq, int Hkv, int sink, int win, float sl2, unsigned *err,
                      int split_f, int split_w, const uint8_t *pf_k, const uint8_t *pf_v,
                      unsigned long long pf_head_stride, unsigned pf_head_bytes,
                      const float *__restrict__ q32, __half *__restrict__ qh,
                      unsigned *q_flags, unsigned *q_stage_ctr, int q_w0) {
    using C = Cfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Bars *bars = reinterpret_cast<Bars *>(smem + C::OFF_BAR);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int nqt = (n + C::BQ - 1) / C::BQ;
    const int nkt = (pos0 + n + C::BK - 1) / C::BK;  // keys 0 .. pos0+n-1
    const int n_units = nqt * Hq;
    const int G = gridDim.x;
    volatile int *abort_flag = nullptr;  // set below
    // j-th unit of this block, read from the ring (consumers) after the
    // producer published it; false at the end of the work (or on abort).
    auto to_unit = [&](int w, Unit *u) -> bool {
        if (w < 0 || w >= n_units) return false;
        u->qt = nqt - 1 - w / Hq;
        u->h = w % Hq;
        return true;
    };

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        mbar_init(&bars->o_free, 128);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], 1);
            mbar_init(&bars->s_full[s], 1);
            mbar_init(&bars->p_full[s], 128);
        }
        mbar_init(&bars->o_done, 1);
        mbar_init(&bars->o_last, 1);
        mbar_init(&bars->drain, 1);
        for (int k = 0; k < kUnitRing; ++k) {
            mbar_init(&bars->unit_full[k], 1);
            mbar_init(&bars->unit_empty[k], 1 + 4);  // MMA thread + 4 softmax warps
        }
        bars->abort = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_o);
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
    abort_flag = abort;
    // consumer side of the unit ring: wait for slot j and read the unit id
    auto next_unit = [&](int j, Unit *u, bool arrive_one) -> bool {
        const int slot = j % kUnitRing;
        if (!mbar_wait(&bars->unit_full[slot], (j / kUnitRing) & 1, abort_flag, err)) return false;
        const int w = *reinterpret_cast<volatile int *>(&bars->unit_id[slot]);
        if (arrive_one) mbar_arrive(&bars->unit_empty[slot]);
        return to_unit(w, u);
    };

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            // K/V rows not just written by a staging pass (an fp16 cache read in
            // place): this block asks for its share of them in L2 before its
            // first unit, so the first passes over the key tiles do not wait on
            // DRAM (pf_k null: nothing to do)
            if (pf_k) {
                constexpr unsigned kPiece = 65536;
                const unsigned per_head = (pf_head_bytes + kPiece - 1) / kPiece;
                const unsigned pieces = 2u * static_cast<unsigned>(Hkv) * per_head;
                for (unsigned i = blockIdx.x; i < pieces; i += gridDim.x) {
                    const unsigned piece = i % per_head, hv = i / per_head;
                    const unsigned off = piece * kPiece;
                    bulk_prefetch_l2(((hv & 1) ? pf_v : pf_k) + (hv >> 1) * pf_head_stride + off,
                                     min(kPiece, pf_head_bytes - off));
                }
            }
            int k_arms[2] = {0, 0}, v_arms[2] = {0, 0}, q_arms = 0;
            bool ok = true;
            // hand unit id w to the MMA and softmax warps through ring slot j
            auto publish = [&](int j, int w) -> bool {
                const int slot = j % kUnitRing;
                if (j >= kUnitRing &&
                    !mbar_wait(&bars->unit_empty[slot], ((j / kUnitRing) - 1) & 1, abort, err))
                    return false;
                bars->unit_id[slot] = w;
                mbar_arrive(&bars->unit_full[slot]);
                return true;
            };
            // key tile kt of kv head g into stage tt % NS (tt: this block's tile count)
            auto load = [&](int tt, int kt, int g, int qt, bool is_k) -> bool {
                const int st = tt % C::NS;
                uint64_t *empty = is_k ? &bars->k_empty[st] : &bars->v_empty[st];
                uint64_t *full = is_k ? &bars->k_full[st] : &bars->v_full[st];
                if (tt >= C::NS && !mbar_wait(empty, ((tt / C::NS) - 1) & 1, abort, err))
                    return false;
                mbar_arrive_expect_tx(full, C::TILE_BYTES);
                const uint32_t base = (is_k ? C::OFF_K : C::OFF_V) + st * C::TILE_BYTES;
                for (int c = 0; c < C::NCHUNK; ++c)
                    tma_load_3d(smem + base + c * C::CHUNK_BYTES, is_k ? &tm_k : &tm_v, full,
                                c * 64, kt * C::BK, g);
                if (is_k) {
                    ++k_arms[st];
                    if (tile_map) tile_map[static_cast<size_t>(qt) * nkt + kt] = 1;
                } else {
                    ++v_arms[st];
                }
                return true;
            };
            // Q tile of the j-th unit w, once the buffer is free (the previous
            // unit's last QK^T completed) and, for a unit staged by this
            // kernel, once its rows are in fp16
            auto load_q = [&](int j, int w, const Unit &u, unsigned peek) -> bool {
                if (j > 0 && !mbar_wait(&bars->q_empty, (j - 1) & 1, abort, err)) return false;
                if (w >= q_w0) {
                    if (peek)
                        fence_acq_rel_gpu();
                    else if (!flag_wait(q_flags + (w - q_w0), abort, err))
                        return false;
                    fence_proxy_async_global();
                }
#ifdef FA_TEST_SKIP_FIRST_Q
                // Test-only build: the first Q tile is never armed or loaded, so
                // the MMA warp's bounded wait on it runs out and the launch must
                // report FA_ERR_TIMEOUT and leave the context usable.
                if (j == 0) return true;
#endif
                mbar_arrive_expect_tx(&bars->q_full, C::TILE_BYTES);
                for (int c = 0; c < C::NCHUNK; ++c)
                    tma_load_3d(smem + C::OFF_Q + c * C::CHUNK_BYTES, &tm_q, &bars->q_full,
                                c * 64, u.h, u.qt * C::BQ);
                ++q_arms;
                return true;
            };
            auto plan_of = [&](const Unit &u) {
                const int q0 = u.qt * C::BQ;
                return unit_plan<SPLIT>(pos0 + q0, pos0 + min(n, q0 + C::BQ) - 1, sink, win,
                                        split_w, C::BK);
            };
            const int group = Hq / Hkv;
            int t = 0;  // tiles of this block before the current unit
            // block b starts with unit b; later units come from the global counter
            int w = static_cast<int>(blockIdx.x);
            Unit u;
            ok = publish(0, w);
            bool have = ok && to_unit(w, &u);
            if (have) ok = load_q(0, w, u, 0u);
            for (int j = 0; have && ok; ++j) {
                const int g = u.h / group;
                const TilePlan plan = plan_of(u);
                const int cnt = plan.count;
                // consumption order of the MMA warp: K0, K1, V0, K2, V1, ...,
                // V(cnt-1). The next unit is taken with the last K tile, so that
                // the counter's round trip overlaps the waits for the V stages.
                int w_next = -1;
                unsigned peek = 0;
                for (int i = 0; i < cnt && ok; ++i) {
                    ok = load(t + i, plan.kt(i), g, u.qt, true);
                    if (ok && i == cnt - 1)
                        w_next = G + static_cast<int>(atomicAdd(work_counter, 1u));
                    if (ok && i >= 1) ok = load(t + i - 1, plan.kt(i - 1), g, u.qt, false);
                }
                // a first look at the next unit's Q flag, read after the last V
                // tile is issued
                if (ok && w_next >= q_w0 && w_next < n_units)
                    peek = ld_relaxed_gpu(q_flags + (w_next - q_w0));
                if (ok) ok = load(t + cnt - 1, plan.kt(cnt - 1), g, u.qt, false);
                t += cnt;
                if (!ok) break;
                Unit un;
                ok = publish(j + 1, w_next);
                have = ok && to_unit(w_next, &un);
                if (have) ok = load_q(j + 1, w_next, un, peek);
                u = un;
            }
            if (!ok) {  // let every copy already issued land before exit
                if (q_arms) drain_wait(&bars->q_full, (q_arms - 1) & 1);
                for (int s2 = 0; s2 < 2; ++s2) {
                    if (k_arms[s2]) drain_wait(&bars->k_full[s2], (k_arms[s2] - 1) & 1);
                    if (v_arms[s2]) drain_wait(&bars->v_full[s2], (v_arms[s2] - 1) & 1);
                }
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t sQ = smem_u32(smem + C::OFF_Q);
            const uint32_t sK = smem_u32(smem + C::OFF_K);
            const uint32_t sV = smem_u32(smem + C::OFF_V);
            auto issue_qk = [&](int tt) -> bool {
                const int st = tt % C::NS;
                if (!mbar_wait(&bars->k_full[st], (tt / C::NS) & 1, abort, err)) return false;
                tc_fence_after();
                const uint32_t d = tmem + ((tt & 1) ? C::S_COL1 : C::S_COL0);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
                    const uint64_t a = desc_sw128(sQ + off, 16, 1024);
                    const uint64_t bd = desc_sw128(sK + st * C::TILE_BYTES + off, 16, 1024);
                    mma_ss(d, a, bd, C::IDESC_QK, kk > 0 ? 1u : 0u);
                }
                tc_commit(&bars->k_empty[st]);
                tc_commit(&bars->s_full[tt & 1]);
                return true;
            };
            // PV of global tile tt; `first` starts a fresh O for the unit
            auto issue_pv = [&](int tt, bool first) -> bool {
                const int st = tt % C::NS;
                if (!mbar_wait(&bars->p_full[tt & 1], (tt >> 1) & 1, abort, err)) return false;
                if (!mbar_wait(&bars->v_full[st], (tt / C::NS) & 1, abort, err)) return false;
                tc_fence_after();
                const uint32_t pcol = tmem + ((tt & 1) ? C::S_COL1 : C::S_COL0);
#pragma unroll
                for (int kk = 0; kk < C::BK / 16; ++kk) {
                    // V tile: [128 keys][64 dims] per 16-KB chunk; 16 keys per k-step,
                    // next 64 dims of N one chunk further (LBO), 8-key atoms 1 KB apart (SBO).
                    const uint64_t bd = desc_sw128(sV + st * C::TILE_BYTES + kk * 2048,
                                                   C::CHUNK_BYTES, 1024);
                    mma_ts(tmem + C::O_COL, pcol + kk * 8, bd, C::IDESC_PV,
                           (!first || kk > 0) ? 1u : 0u);
                }
                tc_commit(&bars->v_empty[st]);
                tc_commit(&bars->o_done);
                return true;
            };
            int t = 0;
            bool ok = true;
            Unit u;
            for (int j = 0; ok && next_unit(j, &u, true); ++j) {
                const int q0 = u.qt * C::BQ;
                const int p0 = pos0 + q0, p1 = pos0 + min(n, q0 + C::BQ) - 1;
                const int count = unit_plan<SPLIT>(p0, p1, sink, win, split_w, C::BK).count;
                ok = mbar_wait(&bars->q_full, j & 1, abort, err);
                if (!ok) break;
                tc_fence_after();
                for (int i = 0; i < count && ok; ++i) {
                    ok = issue_qk(t + i);
                    if (ok && i == count - 1) tc_commit(&bars->q_empty);  // Q read for the last time
                    if (ok && i >= 1) {
                        // the first P.V of a unit overwrites O: the epilogue of the
                        // previous unit must have read it
                        if (i == 1 && j > 0) {
                            ok = mbar_wait(&bars->o_free, (j - 1) & 1, abort, err);
                            if (ok) tc_fence_after();
                        }
                        if (ok) ok = issue_pv(t + i - 1, i == 1);
                    }
                }
                if (ok && count == 1 && j > 0) {
                    ok = mbar_wait(&bars->o_free, (j - 1) & 1, abort, err);
                    if (ok) tc_fence_after();
                }
                if (ok) ok = issue_pv(t + count - 1, count == 1);
                if (ok) tc_commit(&bars->o_last);
                t += count;
            }
            // every MMA issued must complete before TMEM is released
            tc_commit(&bars->drain);
            drain_wait(&bars->drain, 0);
        }
    } else if (warp < 4) {
        // ------------------------------------------------------ Q staging
        // Warps 2 and 3 each take units w >= q_w0 in order from a global
        // counter and convert the unit's Q rows (fp32 [n][Hq][hd]) to the fp16
        // rows the tensor map reads, then set the unit's flag. They wait on
        // nothing, so every claimed unit is finished by a running block, and
        // the producer warps of all blocks (this one included) only wait for
        // units some block has claimed or will claim.
        if (q32) {
            constexpr int V4 = HD / 4;         // float4 per row
            constexpr int kInFlight = 16;      // 24 or more made the kernel spill
            constexpr int LPR = V4 < 32 ? V4 : 32;  // lanes on one row in a warp-wide load
            constexpr int RPS = 32 / LPR;      // rows one warp-wide load covers
            constexpr int SPR = V4 / LPR;      // warp-wide loads per row
            constexpr int RPB = kInFlight / SPR * RPS;  // rows per batch of loads
            static_assert(kInFlight % SPR == 0, "whole rows per batch");
            const size_t rs = static_cast<size_t>(Hq) * V4;  // float4 from row to row
            const int lane_row = lane / LPR;
            const size_t lane_off = static_cast<size_t>(lane_row) * rs + lane % LPR;
            for (;;) {
                unsigned claim = 0;  // past the last unit once the block aborted
                if (lane == 0)
                    claim = *abort ? static_cast<unsigned>(n_units) : atomicAdd(q_stage_ctr, 1u);
                claim = __shfl_sync(0xffffffffu, claim, 0);
                if (claim >= static_cast<unsigned>(n_units - q_w0)) break;
                const int w = q_w0 + static_cast<int>(claim);
                const int q0 = (nqt - 1 - w / Hq) * C::BQ;
                const int rows = min(C::BQ, n - q0);
                const size_t base = (static_cast<size_t>(q0) * Hq + w % Hq) * V4 + lane_off;
                for (int r0 = 0; r0 < rows; r0 += RPB) {
                    const size_t at = base + static_cast<size_t>(r0) * rs;
                    const float4 *src = reinterpret_cast<const float4 *>(q32) + at;
                    uint2 *dst = reinterpret_cast<uint2 *>(qh) + at;
                    float4 x[kInFlight];
#pragma unroll
                    for (int k = 0; k < kInFlight; ++k) {
                        const int rr = k / SPR * RPS;  // this load's row in the batch
                        if (r0 + rr + lane_row < rows)
                            x[k] = __ldcs(src + static_cast<size_t>(rr) * rs + (k % SPR) * 32);
                    }
#pragma unroll
                    for (int k = 0; k < kInFlight; ++k) {
                        const int rr = k / SPR * RPS;
                        if (r0 + rr + lane_row < rows)
                            __stcs(dst + static_cast<size_t>(rr) * rs + (k % SPR) * 32,
                                   make_uint2(pack_half2(x[k].x, x[k].y),
                                              pack_half2(x[k].z, x[k].w)));
                    }
                }
                __threadfence();
                fence_proxy_async_global();
                __syncwarp();
                if (lane == 0) st_release_gpu(q_flags + (w - q_w0), 1u);
            }
        }
    } else {
        // ----------------------------------------------- softmax and epilogue
        const int r = threadIdx.x - 128;  // tile row == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        int t = 0;
        int stores = 0;  // TMA stores issued by this warp's lane 0
        bool ok = true;
        Unit u;
        for (int j = 0; ok; ++j) {
            const bool have = next_unit(j, &u, false);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->unit_empty[j % kUnitRing]);
            if (!__all_sync(0xffffffffu, have)) break;
            const int q0 = u.qt * C::BQ;  // query rows q0.. at positions p0..
            const int p0 = pos0 + q0, p1 = pos0 + min(n, q0 + C::BQ) - 1;
            const int p = p0 + r;
            const TilePlan plan = unit_plan<SPLIT>(p0, p1, sink, win, split_w, C::BK);
            float m_used = -INFINITY;  // exp2-domain reference shared by O and l
            float l = 0.0f;
            for (int i = 0; i < plan.count; ++i) {
                const int tt = t + i;
                const int bsel = tt & 1;
                ok = mbar_wait(&bars->s_full[bsel], (tt >> 1) & 1, abort, err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                const uint32_t scol = tmem + lane_base + (bsel ? C::S_COL1 : C::S_COL0);
                uint32_t s[128];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(scol + 32 * c, s + 32 * c);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 4; ++c) reg_fence32(s + 32 * c);

                const int kt = plan.kt(i);
                const int j0 = kt * C::BK;
                float mx = -INFINITY;
                if (tile_full(kt, p0, p1, sink, win, C::BK) &&
                    (SPLIT == 0 || (SPLIT == 1 && (j0 + C::BK - 1 < split_f ||
                                                   j0 + C::BK - 1 <= p0 - split_w)))) {
#pragma unroll
                    for (int c = 0; c < 128; ++c) mx = fmaxf(mx, __uint_as_float(s[c]));
                } else {
                    // key j0 + c is visible iff c <= hi and (c >= lo or c < sk)
                    const int hi = p - j0;
                    const int lo = win > 0 ? p - win + 1 - j0 : -1;
                    const int sk = win > 0 ? sink - j0 : -1;
                    const int fk = split_f - j0, hs = p - split_w - j0;  // near: c >= fk, c > hs
#pragma unroll
                    for (int c = 0; c < 128; ++c) {
                        bool vis = (c <= hi) & ((c >= lo) | (c < sk));
                        if (SPLIT == 1) vis &= (c < fk) | (c <= hs);
                        if (SPLIT == 2) vis &= (c >= fk) & (c > hs);
                        const float v = vis ? __uint_as_float(s[c]) : -INFINITY;
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
                // O must hold PV(tt-1) before it is rescaled. Only then is the O
                // barrier waited on: its phases cannot run ahead of this row's P
                // (PV(tt) needs it), and S(tt) ready means PV(tt-2) is done, so the
                // barrier is at phase tt-1 or tt here and the parity is unambiguous.
                // (P(tt) itself may land at once: PV(tt-2), the last reader of this
                // S buffer, is done.)
                const bool any_resc = __any_sync(0xffffffffu, resc);
                if (any_resc) {
                    ok = mbar_wait(&bars->o_done, (tt - 1) & 1, abort, err);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                }
                tc_fence_after();
                __syncwarp();
                if (any_resc) {
#pragma unroll 1
                    for (int c = 0; c < HD / 32; ++c) {
                        uint32_t o[32];
                        const uint32_t oc = tmem + lane_base + C::O_COL + 32 * c;
                        tmem_ld32(oc, o);
                        tmem_wait_ld();
                        reg_fence32(o);
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            o[k] = __float_as_uint(__uint_as_float(o[k]) * corr);
                        tmem_st32(oc, o);
                    }
                }
                tmem_st32(scol, pk);
                tmem_st32(scol + 32, pk + 32);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars->p_full[bsel]);
            }
            if (!ok) break;
            t += plan.count;
            // ---- epilogue of the unit: wait for its last P.V, then O / l leaves
            // through this warp's two staging boxes [32 rows][32 fp32] (128-byte
            // swizzle) by TMA bulk-tensor stores; rows past n are dropped.
            ok = mbar_wait(&bars->o_last, j & 1, abort, err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            // a row with no visible key (possible only in a SPLIT part) has l = 0
            const float inv = l > 0.0f ? 1.0f / l : 0.0f;
            // log sum_j exp(s_j) = ln 2 * m_used + ln l (l is relative to 2^m_used)
            if (LSE && q0 + r < n)
                lse[static_cast<size_t>(u.h) * n + q0 + r] =
                    l > 0.0f ? m_used * 0.69314718055994531f + logf(l) : -INFINITY;
            const int wr = warp & 3;  // rows 32 wr .. 32 wr + 31 of the tile
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_base + C::O_COL + 32 * c, o);
                tmem_wait_ld();
                reg_fence32(o);
                if (c == HD / 32 - 1) {  // O fully read: the next unit may overwrite it
                    tc_fence_before();
                    mbar_arrive(&bars->o_free);
                }
                // this box was last used by the store issued two chunks ago
                if (lane == 0 && stores >= 2) bulk_wait_group_read<1>();
                __syncwarp();
                uint8_t *box = smem + C::OFF_OST + (wr * 2 + (c & 1)) * C::OST_BYTES;
                uint8_t *rowp = box + lane * 128;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    float4 v;
                    v.x = __uint_as_float(o[4 * k]) * inv;
                    v.y = __uint_as_float(o[4 * k + 1]) * inv;
                    v.z = __uint_as_float(o[4 * k + 2]) * inv;
                    v.w = __uint_as_float(o[4 * k + 3]) * inv;
                    *reinterpret_cast<float4 *>(rowp + ((k ^ (lane & 7)) << 4)) = v;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && q0 + 32 * wr < n) {  // rows past n are not stored
                    tma_store_3d(&tm_o, box, 32 * c, u.h, q0 + 32 * wr);
                    bulk_commit_group();
                    ++stores;
                }
            }
        }
        if (lane == 0) bulk_wait_group_read<0>();
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

// 3-D tensor (fp16 or fp32), 128-byte swizzle, zero fill outside the tensor.
bool encode_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1,
               uint32_t b2, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_FLOAT16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dtype, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool encode_tiled(CUtensorMap *m, CUtensorMapDataType dtype, int rank, const void *base,
                  const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) st[i] = strides_bytes[i];
    }
    return fn(m, dtype, static_cast<cuuint32_t>(rank), const_cast<void *>(base), d, st, b, e,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <int HD>
cudaError_t launch_hd(const PrefillArgs &a, unsigned *err, cudaStream_t stream) {
    using C = Cfg<HD>;
    CUtensorMap tq, tk, tv, to;
    const uint64_t n = a.n, Hq = a.n_q_heads, Hkv = a.n_kv_heads;
    const uint64_t L = static_cast<uint64_t>(a.pos0) + a.n;  // key rows
    const uint64_t head_stride = static_cast<uint64_t>(a.kv_rows) * HD * 2;
    // rows L .. kv_rows-1 of a head are outside the map: a box reaching them
    // reads zeros, never the unwritten rows of a cache plane
    if (!encode_3d(&tq, a.qh, HD, Hq, n, HD * 2, Hq * HD * 2, 64, 1, C::BQ) ||
        !encode_3d(&tk, a.kh, HD, L, Hkv, HD * 2, head_stride, 64, C::BK, 1) ||
        !encode_3d(&tv, a.vh, HD, L, Hkv, HD * 2, head_stride, 64, C::BK, 1) ||
        !encode_3d(&to, a.out, HD, Hq, n, HD * 4, Hq * HD * 4, 32, 1, 32,
                   CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
        return cudaErrorInvalidValue;
    if (a.split && !a.lse) return cudaErrorInvalidValue;
    auto kernel = a.split == 1   ? prefill_tc_kernel<HD, true, 1>
                  : a.split == 2 ? prefill_tc_kernel<HD, true, 2>
                  : a.lse        ? prefill_tc_kernel<HD, true, 0>
                                 : prefill_tc_kernel<HD, false, 0>;
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const int units = ((a.n + C::BQ - 1) / C::BQ) * a.n_q_heads;
    const int grid = prefill_grid(a.n, a.n_q_heads);
    if (a.q && a.q_w0 < prefill_units_staged_first(a.pos0, a.n, a.n_q_heads, a.sink, a.win))
        return cudaErrorInvalidValue;  // a first-wave unit's Q would never be staged
    const float sl2 = a.scale * 1.4426950408889634f;
    // 32-bit byte counts per kv head (up to 8M rows at head_dim 256)
    const bool prefetch = a.prefetch_kv && L * HD * 2 < (1ull << 31);
    // units from q_w0 on have their Q converted by the kernel (all of them
    // staged before: q_w0 = units)
    const bool own_q = a.q && a.q_w0 < units;
    kernel<<<grid, 256, C::SMEM, stream>>>(
        tq, tk, tv, to, a.tile_map, a.work_counter, a.lse, a.pos0, a.n, a.n_q_heads,
        a.n_kv_heads, a.sink, a.win, sl2, err, a.split_f, a.split_w,
        prefetch ? reinterpret_cast<const uint8_t *>(a.kh) : nullptr,
        reinterpret_cast<const uint8_t *>(a.vh), static_cast<unsigned long long>(head_stride),
        static_cast<unsigned>(L * HD * 2), own_q ? a.q : nullptr, const_cast<__half *>(a.qh),
        a.q_flags, a.q_stage_counter, own_q ? a.q_w0 : units);
    return cudaGetLastError();
}

}  // namespace

int prefill_grid(int n, int Hq) {
    const int units = ((n + kPrefillBQ - 1) / kPrefillBQ) * Hq;
    return units < device_sm_count() ? units : device_sm_count();
}

int prefill_units_staged_first(int pos0, int n, int Hq, int sink, int win) {
    const int nqt = (n + kPrefillBQ - 1) / kPrefillBQ;
    // The staging warps convert one unit's rows in ~16 tile times of the
    // tensor cores (at any head_dim: both scale with it) and the blocks a wave
    // of units. When the first units are shorter than that (windows), two
    // waves are staged before the launch so that the warps start ahead.
    const TilePlan heavy =
        tile_plan(pos0 + (nqt - 1) * kPrefillBQ, pos0 + n - 1, sink, win, kPrefillBK);
    const int waves = heavy.count < 24 ? 2 : 1;
    const int w0 = (waves * prefill_grid(n, Hq) + Hq - 1) / Hq * Hq;
    return w0 < nqt * Hq ? w0 : nqt * Hq;
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, unsigned *err, cudaStream_t stream) {
    switch (a.head_dim) {
        case 64: return launch_hd<64>(a, err, stream);
        case 128: return launch_hd<128>(a, err, stream);
        case 256: return launch_hd<256>(a, err, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
