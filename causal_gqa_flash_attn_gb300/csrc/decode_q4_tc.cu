// decode_q4_tc.cu -- multi-slot split-KV decode over a Q4_0 cache on the
// tcgen05 tensor cores ("attention.cu", "Decode-mode flash attention" and
// "Multi-user decode attention": per (slot, kv head) piece of keys, the
// partial m, l, acc of the slot's query heads; "4-bit KV cache (Q4_0
// blocks)": element j of a 32-block decodes to (c_j - 8) * d).
//
// One block per SM, 288 threads, 128-key tiles (one key per TMEM lane):
//   warps 0-3 (K group, thread = key): load the key's raw Q4_0 K row from
//     global memory into registers (two tiles ahead), turn its nibbles into
//     fp16 MMA operands (1024 + c for the low nibbles, 1024 + 16 c for the
//     high ones: one LOP3 per pair) and store them in TMEM as the A operand of
//       S^T (128 keys x 16) = K' (128 x 32 per Q4_0 block) . Q'^T
//     with one 16-column accumulator per pair of blocks (block 2i in columns
//     0-7, block 2i+1 in 8-15: Q' holds the group's 8 q heads in rows 0-7 for
//     even blocks' dims and in rows 8-15 for odd blocks' dims). A third k-step
//     per block, against a constant A operand (2^10, 1, 2^-10, 0, ...), adds
//     -(1032 sum q_lo + 1152 sum q_hi / 16) as three fp16 terms, so that every
//     accumulator ends at sum (c - 8) q; the thread then scales it by its key's block
//     scale d and sums the blocks: s_h = sum_b d_b acc_b,h. It runs the
//     online softmax of its key's 8 scores (fp32, exp2, a lazy reference
//     shared by the group that moves only when some score passes it by 2^2),
//     and writes P'_b,h = p_h * dv_b (dv_b: the key's V block scales) as the
//     B operand [128 keys][64 = 8 blocks x 8 heads] of the PV MMA.
//   warps 4-7 (V group, thread = key): load the raw V row, turn it into exact
//     fp16 values c - 8 (LOP3 then one HADD2 or HFMA2 per pair) and store them
//     as the A operand V'^T (MN-major, 128-byte swizzle, [128 keys][256 dims])
//     of
//       O^T (256 dims x 64) += V'^T . P'
//     where a dim of block b only keeps column block b (its own scale): the
//     other 56 columns of the 64 are the price of folding the per-key,
//     per-block scale into the B operand. At the start of every piece the
//     group also writes Q'^T for the new (slot, kv head).
//   warp 8 (one thread): tcgen05.mma issue, TMEM allocation.
// Work split: the stream-K cut of decode_common.cuh over 128-key tiles.
// The fp16 shadow keys (sinks, recent ring) and the workspace header are left
// to decode_q4_kernel's auxiliary blocks.
#include <cuda_fp16.h>

#include "decode_common.cuh"

namespace fa {
namespace {

constexpr int kTK = 128;                  // keys per tile (TMEM lanes)
constexpr int kThreads = 288;             // K group, V group, MMA warp
constexpr float kRescale = 2.0f;          // lazy-reference threshold (log2 units)
constexpr uint32_t kMagic = 0x64006400u;  // fp16 pair (1024, 1024)

template <int HD>
struct TcCfg {
    static constexpr int NB = HD / 32;        // Q4_0 blocks per row
    static constexpr int NP = NB / 2;         // block pairs = S accumulators
    static constexpr int MT = HD / 128;       // M tiles of O^T
    static constexpr int ROWB = NB * 18;      // bytes per row
    static constexpr int ROWW = ROWB / 4;     // 32-bit words per row
    static constexpr int NKS = 3 * NB;        // k-steps of Q'^T: lo, hi of each block, then biases
    // TMEM columns
    static constexpr uint32_t KW = NB * 16;                // K': 16 per block
    static constexpr uint32_t KA0 = 0, KA1 = KW;           // two K' buffers
    static constexpr uint32_t BA = 2 * KW;                 // bias A operand: 8
    static constexpr uint32_t S = (BA + 8 + 31) / 32 * 32;   // S^T: 16 per block pair
    static constexpr uint32_t SW = NP * 16;
    static constexpr uint32_t O = (S + SW + 31) / 32 * 32;   // O^T: 64 per M tile
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(O + MT * 64 <= TMEM_COLS, "TMEM columns");
    // shared memory (offsets from a 1024-byte aligned base)
    static constexpr uint32_t VCHUNK = kTK * 128;          // [128 keys][64 dims] fp16
    static constexpr uint32_t VSTAGE = (HD / 64) * VCHUNK;
    static constexpr uint32_t OFF_V = 0;                   // 2 stages of V'
    static constexpr uint32_t OFF_P = OFF_V + 2 * VSTAGE;  // 2 stages of P' [128][64] fp16
    static constexpr uint32_t PSTAGE = kTK * 128;
    static constexpr uint32_t QCHUNK = 16 * 128;           // 16 rows x 64 k elements
    static constexpr uint32_t QBUF = NKS / 4 * QCHUNK;
    static constexpr uint32_t OFF_Q = OFF_P + 2 * PSTAGE;  // 2 buffers of Q'^T
    static constexpr uint32_t OFF_SC = OFF_Q + 2 * QBUF;   // 2 stages of V scales [128][NB] fp16
    static constexpr uint32_t SCSTAGE = kTK * NB * 2;
    static constexpr uint32_t OFF_RED = OFF_SC + 2 * SCSTAGE;  // [2][4 warps][8] fp32, [2][4] flags
    static constexpr uint32_t OFF_BAR = OFF_RED + 2 * 4 * 8 * 4 + 64;
    static constexpr uint32_t USED = OFF_BAR + 256;
    static constexpr uint32_t SMEM = USED + 1024;
    static_assert(NKS % 4 == 0, "k-steps per chunk");
    static_assert(SMEM <= 227u * 1024u, "shared memory");
    static constexpr uint32_t IDESC_S = idesc_f16(128, 16, 0, 0);
    static constexpr uint32_t IDESC_PV = idesc_f16(128, 64, 1, 1);
};

struct TcBars {
    uint64_t kp_full[2];
    uint64_t s_full, s_free;
    uint64_t v_full[2], p_full[2], pv_done[2];
    uint64_t q_full[2];
    uint64_t o_free;
    // K-group exchanges, by tile parity: the rescale flags, the maxima; and
    // the row sums of a piece's epilogue
    uint64_t xf[2], xm[2], xl;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// Element (0..31) of block b that K-order (and V') position pp of the block
// holds. Positions 0..15 are the low nibbles, 16..31 the high ones, in the
// order the words of the block are turned into fp16 pairs: word wi holds the
// code bytes J[wi][0..3] of the block, and the pairs of a word are its bytes
// (0, 2) then (1, 3). Odd blocks' code bytes start on a word; even blocks'
// start 2 bytes into one, so their first word is bytes 0, 1, 14, 15 (a
// permute of the two words that hold them) and the next three bytes 2-13.
__host__ __device__ constexpr int q4_elem(int b, int pp) {
    const int hi = pp >= 16 ? 16 : 0;
    const int kp = pp & 15;
    const int wi = kp >> 2;
    const int slot = (kp & 3) == 0 ? 0 : ((kp & 3) == 1 ? 2 : ((kp & 3) == 2 ? 1 : 3));
    int byte = 0;
    if (b & 1) {
        byte = 4 * wi + slot;
    } else if (wi == 0) {
        byte = slot == 0 ? 0 : (slot == 1 ? 1 : (slot == 2 ? 14 : 15));
    } else {
        byte = 4 * wi - 2 + slot;
    }
    return byte + hi;
}

template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t x, uint32_t magic) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "n"(MASK), "r"(magic));
    return d;
}

__device__ __forceinline__ uint32_t hadd2u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hfma2u(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// The 4 code words of block b of a row held in w[] (words of the row).
template <int ROWW>
__device__ __forceinline__ void block_words(const uint32_t (&w)[ROWW], int b, uint32_t (&x)[4]) {
    const int a = b >> 1;
    if (b & 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = w[9 * a + 5 + i];
    } else {
        x[0] = __byte_perm(w[9 * a], w[9 * a + 4], 0x5432);  // bytes 2, 3 | 4, 5 -> c0 c1 c14 c15
        x[1] = w[9 * a + 1];
        x[2] = w[9 * a + 2];
        x[3] = w[9 * a + 3];
    }
}

// fp16 bits of block b's scale d in a row held in w[].
template <int ROWW>
__device__ __forceinline__ uint32_t block_scale_bits(const uint32_t (&w)[ROWW], int b) {
    const int a = b >> 1;
    return (b & 1) ? (w[9 * a + 4] >> 16) : (w[9 * a] & 0xFFFFu);
}

__device__ __forceinline__ float h2f(uint32_t bits) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
}

// A row of ROWW words from global memory (16-byte aligned rows).
template <int ROWW>
__device__ __forceinline__ void load_row(uint32_t (&w)[ROWW], const uint8_t *src) {
    static_assert(ROWW % 4 == 0, "16-byte rows");
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int i = 0; i < ROWW / 4; ++i) {
        const uint4 v = __ldg(s4 + i);
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void reg_fence16(uint32_t *r) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

// The sequence of (piece, tile) a block walks, the same in every role: the
// pieces of its run [bid C, min(T, bid C + C)) of the job, and the tiles of
// each piece.
struct TcSeq {
    long long Tc;  // job index of the current tile
    int u, g, p, j, j1, e;
    Q4Tiles tl;
    int piece;  // pieces started so far - 1
    int i;      // tile index within the piece
    bool valid;

    __device__ void start(const DecodeParams &P, const Q4Job &J, int bid, long long slot_base,
                          int u0) {
        Tc = static_cast<long long>(bid) * J.C;
        valid = Tc < J.T && u0 >= 0;
        piece = -1;
        if (!valid) return;
        u = u0;
        p = P.pos[u];
        tl = q4_tiles(P, p);
        const long long local = Tc - slot_base;
        g = static_cast<int>(local / tl.count());
        j = static_cast<int>(local % tl.count());
        begin_piece(J, bid, slot_base + static_cast<long long>(g) * tl.count());
    }
    // a.k.a. the piece's pair starts at job index A
    __device__ void begin_piece(const Q4Job &J, int bid, long long A) {
        const long long T1 = min(J.T, static_cast<long long>(bid) * J.C + J.C);
        j1 = static_cast<int>(min(static_cast<long long>(tl.count()), j + (T1 - Tc)));
        e = static_cast<int>(bid - A / J.C);
        ++piece;
        i = 0;
    }
    __device__ bool first() const { return i == 0; }
    __device__ bool last() const { return j + i + 1 == j1; }
    __device__ int key0() const { return kTK * tl.kt(j + i); }
    // next tile; false at the end of the run
    __device__ bool next(const DecodeParams &P, const Q4Job &J, int bid) {
        ++Tc;
        const long long T1 = min(J.T, static_cast<long long>(bid) * J.C + J.C);
        if (Tc >= T1) {
            valid = false;
            return false;
        }
        if (j + i + 1 < j1) {
            ++i;
            return true;
        }
        // the next pair with tiles
        j = 0;
        do {
            if (++g == P.Hkv) {
                g = 0;
                ++u;
                p = P.pos[u];
                tl = q4_tiles(P, p);
            }
        } while (tl.count() == 0);
        begin_piece(J, bid, Tc);
        return true;
    }
};

// Bounded wait of all 128 threads of a group on a full-group exchange
// barrier: arrive, then wait for the phase. False on timeout or abort.
__device__ __forceinline__ bool group_sync(uint64_t *bar, uint32_t parity, volatile int *abort,
                                           unsigned *err) {
    mbar_arrive(bar);
    return mbar_wait(bar, parity, abort, err);
}

// Row k of the current tile of s in a K or V plane (keys past p read row p).
template <int ROWB>
__device__ __forceinline__ const uint8_t *tile_row(const DecodeParams &P, const TcSeq &s, int k,
                                                   const uint8_t *planes) {
    const int key = min(s.key0() + k, s.p);
    return planes + static_cast<size_t>(s.u) * P.plane_bytes + P.body_off +
           (static_cast<size_t>(s.g) * P.max_seq + key) * ROWB;
}

// Q'^T of (slot u, kv head g) into qbase: thread k (of 128) writes row
// n = k & 15 for block b = k >> 4, its lo, hi and bias k-steps. Rows 0-7 hold
// the group's heads for even blocks' dims, rows 8-15 for odd blocks' dims
// (zeros elsewhere and for heads >= G); the lo step holds fp16(q) and the hi
// step fp16(q / 16) in the K' element order; the bias step holds -(1032 sum
// lo + 1152 sum hi) as 2^10 t1 + t2 + 2^-10 t3. Kept out of line: it runs once
// per piece.
template <int HD>
__device__ __noinline__ void write_qt(const DecodeParams &P, uint8_t *qbase, int u, int g, int G,
                                      int k) {
    using C = TcCfg<HD>;
    constexpr int NB = C::NB;
    const int n = k & 15, b = k >> 4;
    if (b >= NB) return;
    const int h = n & 7;
    const bool act = ((n >> 3) == (b & 1)) && h < G;
    const float *qr =
        P.q + (static_cast<size_t>(u) * P.Hq + static_cast<size_t>(g) * G + h) * HD + 32 * b;
    auto put = [&](int ks, int kp, uint32_t pair) {
        const int K = ks * 16 + kp;  // even
        const int c = K >> 6, el = K & 63;
        *reinterpret_cast<uint32_t *>(qbase + c * C::QCHUNK + n * 128 +
                                      (((el >> 3) ^ (n & 7)) << 4) + (el & 7) * 2) = pair;
    };
    double bias = 0.0;
    for (int hi = 0; hi < 2; ++hi) {
        for (int kp = 0; kp < 16; kp += 2) {
            uint32_t pair = 0u;
            if (act) {
                const float f = hi ? 0.0625f : 1.0f;
                const __half a0 = __float2half_rn(qr[q4_elem(b, 16 * hi + kp)] * f);
                const __half a1 = __float2half_rn(qr[q4_elem(b, 16 * hi + kp + 1)] * f);
                bias += (hi ? 1152.0 : 1032.0) *
                        (static_cast<double>(__half2float(a0)) + __half2float(a1));
                pair = static_cast<uint32_t>(__half_as_ushort(a0)) |
                       (static_cast<uint32_t>(__half_as_ushort(a1)) << 16);
            }
            put(2 * b + hi, kp, pair);
        }
    }
    const double nb0 = -bias;
    const __half t1 = __double2half(nb0 * 0x1p-10);
    const double r1 = nb0 - 1024.0 * static_cast<double>(__half2float(t1));
    const __half t2 = __double2half(r1);
    const double r2 = r1 - static_cast<double>(__half2float(t2));
    const __half t3 = __double2half(r2 * 1024.0);
    const uint32_t p01 = act ? (static_cast<uint32_t>(__half_as_ushort(t1)) |
                                (static_cast<uint32_t>(__half_as_ushort(t2)) << 16))
                             : 0u;
    const uint32_t p23 = act ? static_cast<uint32_t>(__half_as_ushort(t3)) : 0u;
    put(2 * NB + b, 0, p01);
    put(2 * NB + b, 2, p23);
    for (int kp = 4; kp < 16; kp += 2) put(2 * NB + b, kp, 0u);
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1) decode_q4_tc_kernel(const DecodeParams P) {
    using C = TcCfg<HD>;
    constexpr int NB = C::NB, MT = C::MT, ROWB = C::ROWB, ROWW = C::ROWW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    TcBars *bars = reinterpret_cast<TcBars *>(smem + C::OFF_BAR);
    // By tile parity: the group's exchanged maxima (or row sums) [2][4 warps][8]
    // and rescale flags [2][4]. A K-group thread runs at most one tile ahead
    // of another (a tile's S^T needs every thread's K' of that tile, written
    // after the previous tile's exchanges), so two copies never collide.
    float *red2 = reinterpret_cast<float *>(smem + C::OFF_RED);
    int *flags2 = reinterpret_cast<int *>(smem + C::OFF_RED + 2 * 4 * 8 * 4);
    __shared__ Q4Job sjob;
    __shared__ long long sbase;
    __shared__ int su;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = P.Hq / P.Hkv;
    const int bid = blockIdx.x;

    if (warp == 0) {
        const Q4Job J = q4_job(P, P.q4_body_blocks);
        int u0 = -1;
        long long base = 0;
        const long long T0 = static_cast<long long>(bid) * J.C;
        if (T0 < J.T) q4_locate(P, T0, &u0, &base);
        if (lane == 0) {
            sjob = J;
            sbase = base;
            su = u0;
        }
    }
    __syncthreads();
    const Q4Job J = sjob;
    if (static_cast<long long>(bid) * J.C >= J.T || su < 0) return;  // no work for this block

    if (threadIdx.x == 0) {
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->s_free, 128);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->kp_full[s], 128);
            mbar_init(&bars->v_full[s], 128);
            mbar_init(&bars->p_full[s], 128);
            mbar_init(&bars->pv_done[s], 1);
            mbar_init(&bars->q_full[s], 128);
            mbar_init(&bars->xf[s], 128);
            mbar_init(&bars->xm[s], 128);
        }
        mbar_init(&bars->o_free, 128);
        mbar_init(&bars->xl, 128);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        mbar_fence_init();
    }
    if (warp == 8) {
        tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    volatile int *abort = &bars->abort;

    TcSeq sq;
    sq.start(P, J, bid, sbase, su);

    if (warp == 8) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t sQ = smem_u32(smem + C::OFF_Q);
            const uint32_t sV = smem_u32(smem + C::OFF_V);
            const uint32_t sP = smem_u32(smem + C::OFF_P);
            bool ok = true;
            // O^T (+)= V'^T . P' over tile t's 128 keys
            auto issue_pv = [&](int t, bool fresh, int piece) -> bool {
                const int st = t & 1;
                if (!mbar_wait(&bars->p_full[st], (t >> 1) & 1, abort, P.err)) return false;
                if (!mbar_wait(&bars->v_full[st], (t >> 1) & 1, abort, P.err)) return false;
                if (fresh && piece > 0 && !mbar_wait(&bars->o_free, (piece - 1) & 1, abort, P.err))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kTK / 16; ++kk) {
                    const uint64_t bd = desc_sw128(sP + st * C::PSTAGE + kk * 2048, C::PSTAGE, 1024);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        const uint64_t ad = desc_sw128(
                            sV + st * C::VSTAGE + 2 * mt * C::VCHUNK + kk * 2048, C::VCHUNK, 1024);
                        mma_ss(tmem + C::O + 64 * mt, ad, bd, C::IDESC_PV,
                               (fresh && kk == 0) ? 0u : 1u);
                    }
                }
                tc_commit(&bars->pv_done[st]);
                return true;
            };
            // S^T(t) = K'(t) . Q'^T: per block pair, the lo, hi and bias k-steps
            // of both blocks. sp: the sequence positioned at tile t.
            auto issue_s = [&](int t, const TcSeq &sp) -> bool {
                if (sp.first() &&
                    !mbar_wait(&bars->q_full[sp.piece & 1], (sp.piece >> 1) & 1, abort, P.err))
                    return false;
                if (!mbar_wait(&bars->kp_full[t & 1], (t >> 1) & 1, abort, P.err)) return false;
                if (t >= 1 && !mbar_wait(&bars->s_free, (t - 1) & 1, abort, P.err)) return false;
                tc_fence_after();
                const uint32_t qb = sQ + (sp.piece & 1) * C::QBUF;
                const uint32_t ka = (t & 1) ? C::KA1 : C::KA0;
#pragma unroll
                for (int b = 0; b < NB; ++b) {
#pragma unroll
                    for (int k3 = 0; k3 < 3; ++k3) {
                        const int ks = k3 < 2 ? 2 * b + k3 : 2 * NB + b;
                        const uint64_t bd =
                            desc_sw128(qb + (ks >> 2) * C::QCHUNK + (ks & 3) * 32, 16, 1024);
                        const uint32_t a = tmem + (k3 < 2 ? ka + 16 * b + 8 * k3 : C::BA);
                        mma_ts(tmem + C::S + 16 * (b >> 1), a, bd, C::IDESC_S,
                               ((b & 1) == 0 && k3 == 0) ? 0u : 1u);
                    }
                }
                tc_commit(&bars->s_full);
                return true;
            };
            // S(t + 1) is issued before PV(t), so that it runs while the K
            // group does the softmax of tile t.
            TcSeq nx = sq;  // positioned at tile t + 1
            int t = 0;
            ok = issue_s(0, sq);
            bool more = ok && nx.next(P, J, bid);
            for (; ok; ++t) {
                if (more) {
                    ok = issue_s(t + 1, nx);
                    if (!ok) break;
                }
                ok = issue_pv(t, sq.first(), sq.piece);
                if (!ok || !more) break;
                sq.next(P, J, bid);
                more = nx.next(P, J, bid);
            }
            // every MMA issued must complete before TMEM is released
            tc_commit(&bars->drain);
            const long long c0 = clock64();
            while (!mbar_try_wait(&bars->drain, 0) && clock64() - c0 < kSpinCycles) {
            }
        }
    } else if (warp < 4) {
        // ------------------------------------------- K group: K', softmax, P'
        const int k = threadIdx.x;  // key of the tile, TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        {   // the bias operand: k elements 0-2 are 2^10, 1, 2^-10, the rest 0
            const uint32_t bias_a[8] = {0x3C006400u, 0x00001400u, 0u, 0u, 0u, 0u, 0u, 0u};
            tmem_st8(tmem + lane_base + C::BA, bias_a);
        }
        const uint32_t magic = kMagic;
        uint32_t w[ROWW];  // raw K row of the next tile to turn into K'
        uint32_t dk[NB / 2], dk_next[NB / 2];  // K block scales (fp16 pairs): tiles t, t + 1
        TcSeq pf = sq;     // the tile whose row is in w
        // K' of the tile in w into buffer kb (its S^T MMAs must be done with it)
        auto write_kprime = [&](int kb, uint32_t (&dks)[NB / 2]) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                uint32_t x[4];
                block_words<ROWW>(w, b, x);
                if (b & 1)
                    dks[b >> 1] |= block_scale_bits<ROWW>(w, b) << 16;
                else
                    dks[b >> 1] = block_scale_bits<ROWW>(w, b);
                uint32_t col[16];
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
                    const uint32_t y = x[wi] >> 8;
                    col[2 * wi] = and_or<0x000F000Fu>(x[wi], magic);
                    col[2 * wi + 1] = and_or<0x000F000Fu>(y, magic);
                    col[8 + 2 * wi] = and_or<0x00F000F0u>(x[wi], magic);
                    col[8 + 2 * wi + 1] = and_or<0x00F000F0u>(y, magic);
                }
                tmem_st16(tmem + lane_base + (kb ? C::KA1 : C::KA0) + 16 * b, col);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars->kp_full[kb]);
        };
        load_row<ROWW>(w, tile_row<ROWB>(P, pf, k, P.k_planes));
        write_kprime(0, dk);
        if (pf.next(P, J, bid)) load_row<ROWW>(w, tile_row<ROWB>(P, pf, k, P.k_planes));
        float m_ref[8], l_acc[8];
        int xm_uses0 = 0, xm_uses1 = 0, xl_uses = 0;
        bool ok = true;
        int t = 0;
        for (; ok && sq.valid; ++t) {
            const int cur = t & 1;  // K' buffer of tile t
            if (sq.first()) {
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    m_ref[h] = -INFINITY;
                    l_acc[h] = 0.0f;
                }
            }
            // ---- S^T(t): s_h = sum_b d_b acc_b,h, 32 columns (4 blocks) at a time
            ok = mbar_wait(&bars->s_full, t & 1, abort, P.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            float s[8];
#pragma unroll
            for (int h = 0; h < 8; ++h) s[h] = 0.0f;
#pragma unroll
            for (int pp = 0; pp < static_cast<int>(C::NP); ++pp) {
                uint32_t sr[16];  // blocks 2 pp (columns 0-7) and 2 pp + 1 (8-15)
                tmem_ld16(tmem + lane_base + C::S + 16 * pp, sr);
                tmem_wait_ld();
                reg_fence16(sr);
                const float d0 = h2f(dk[pp] & 0xFFFFu), d1 = h2f(dk[pp] >> 16);
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    s[h] = fmaf(d0, __uint_as_float(sr[h]), s[h]);
                    s[h] = fmaf(d1, __uint_as_float(sr[8 + h]), s[h]);
                }
            }
            tc_fence_before();
            mbar_arrive(&bars->s_free);
            // ---- K'(t + 1) into the other buffer (S^T(t - 1), its last
            // reader, is done), so that S^T(t + 1) runs during this softmax
            if (pf.valid) {
                write_kprime(cur ^ 1, dk_next);
                if (pf.next(P, J, bid)) load_row<ROWW>(w, tile_row<ROWB>(P, pf, k, P.k_planes));
            }
            const int key = sq.key0() + k;
            const int p = sq.p;
            const bool vis = key <= p && key_visible(p, key, P.sink, P.win) &&
                             !(key < P.shadow_sink || (P.shadow_win > 0 && key > p - P.shadow_win));
#pragma unroll
            for (int h = 0; h < 8; ++h) s[h] = vis ? s[h] * P.sl2 : -INFINITY;
            // ---- lazy reference: moves only when a score passes it by 2^2
            bool need = false;
#pragma unroll
            for (int h = 0; h < 8; ++h) need |= s[h] > m_ref[h] + kRescale;
            float *red = red2 + (t & 1) * 32;
            int *flags = flags2 + (t & 1) * 4;
            const unsigned nb_ = __ballot_sync(0xffffffffu, need);
            if (lane == 0) flags[warp] = nb_ != 0;
            ok = group_sync(&bars->xf[t & 1], (t >> 1) & 1, abort, P.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const bool any = flags[0] | flags[1] | flags[2] | flags[3];
            if (any) {
                float mx[8];
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    float v = s[h];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                    mx[h] = v;
                }
                if (lane < 8) {
                    float v = mx[0];
#pragma unroll
                    for (int h = 1; h < 8; ++h)
                        if (lane == h) v = mx[h];
                    red[warp * 8 + lane] = v;
                }
                ok = group_sync(&bars->xm[t & 1], (cur ? xm_uses1 : xm_uses0) & 1, abort, P.err);
                if (cur) ++xm_uses1; else ++xm_uses0;
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                float corr[8];
                bool resc = false;
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const float tmax = fmaxf(fmaxf(red[h], red[8 + h]), fmaxf(red[16 + h], red[24 + h]));
                    corr[h] = 1.0f;
                    if (tmax > m_ref[h] + kRescale) {
                        if (m_ref[h] != -INFINITY) {
                            corr[h] = ex2(m_ref[h] - tmax);
                            resc = true;
                        }
                        l_acc[h] *= corr[h];
                        m_ref[h] = tmax;
                    }
                }
                if (resc && !sq.first()) {
                    // O holds P'V of tiles before t: rescale it after PV(t - 1)
                    ok = mbar_wait(&bars->pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, abort, P.err);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll 1
                        for (int c2 = 0; c2 < 2; ++c2) {
                            uint32_t o[32];
                            const uint32_t oc = tmem + lane_base + C::O + 64 * mt + 32 * c2;
                            tmem_ld32(oc, o);
                            tmem_wait_ld();
                            reg_fence32(o);
#pragma unroll
                            for (int c = 0; c < 32; ++c)
                                o[c] = __float_as_uint(__uint_as_float(o[c]) * corr[c & 7]);
                            tmem_st32(oc, o);
                        }
                    }
                    tmem_wait_st();
                }
            }
            float (&pr)[8] = s;  // the weights replace the scores
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                pr[h] = vis ? ex2(s[h] - m_ref[h]) : 0.0f;
                l_acc[h] += pr[h];
            }
            // ---- P' of tile t: p_h * dv_b as fp16, [key][block][head]; the V
            // scales come from the V group with V'(t), the stage is free once
            // PV(t - 2) is done
            ok = mbar_wait(&bars->v_full[t & 1], (t >> 1) & 1, abort, P.err);
            if (ok && t >= 2)
                ok = mbar_wait(&bars->pv_done[t & 1], ((t - 2) >> 1) & 1, abort, P.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const uint4 dvw = *reinterpret_cast<const uint4 *>(smem + C::OFF_SC + (t & 1) * C::SCSTAGE + k * 16);
            const uint32_t dvp[4] = {dvw.x, dvw.y, dvw.z, dvw.w};  // blocks (0,1), (2,3), ...
            const uint32_t ph[4] = {pack_half2(pr[0], pr[1]), pack_half2(pr[2], pr[3]),
                                    pack_half2(pr[4], pr[5]), pack_half2(pr[6], pr[7])};
            uint8_t *prow = smem + C::OFF_P + (t & 1) * C::PSTAGE + k * 128;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const uint32_t dv = (b & 1) ? (dvp[b >> 1] >> 16) : (dvp[b >> 1] & 0xFFFFu);
                const uint32_t d2 = vis ? (dv | (dv << 16)) : 0u;
                uint4 v;
                v.x = hmul2u(ph[0], d2);
                v.y = hmul2u(ph[1], d2);
                v.z = hmul2u(ph[2], d2);
                v.w = hmul2u(ph[3], d2);
                *reinterpret_cast<uint4 *>(prow + ((b ^ (k & 7)) << 4)) = v;
            }
            fence_proxy_async_smem();
            tc_fence_before();  // a rescale's TMEM stores come before the PV MMAs
            mbar_arrive(&bars->p_full[t & 1]);

            if (sq.last()) {
                // ---- epilogue of the piece: l over the group's keys, then the
                // O^T rows of this lane (relative to 2^m_ref, like l), m. Every
                // thread of the group read red[] (the maxima) before its p_full
                // arrival, so once PV(t) is done red[] may take the sums.
                ok = mbar_wait(&bars->pv_done[t & 1], (t >> 1) & 1, abort, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    float v = l_acc[h];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == h) red[warp * 8 + h] = v;
                }
                ok = group_sync(&bars->xl, xl_uses & 1, abort, P.err);
                ++xl_uses;
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                const size_t head0 = static_cast<size_t>(sq.u) * P.Hq + static_cast<size_t>(sq.g) * G;
                const int e = sq.e;
#pragma unroll 1
                for (int mt = 0; mt < MT; ++mt) {
                    // V' position 128 mt + k of this lane: its block b keeps
                    // O^T columns 8 b .. 8 b + 7 (its own scale)
                    const int P0 = 128 * mt + k;
                    const int b = P0 >> 5;
                    const int dim = 32 * b + q4_elem(b, P0 & 31);
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_base + C::O + 64 * mt + 32 * (b >> 2), o);
                    tmem_wait_ld();
                    reg_fence32(o);
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        const float L = (red[h] + red[8 + h]) + (red[16 + h] + red[24 + h]);
                        if (h < G && L > 0.0f)
                            P.ws_acc[((head0 + h) * P.stride + e) * HD + dim] =
                                __uint_as_float(o[8 * (b & 3) + h]);
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars->o_free);
                if (k < G) {
                    const float L = (red[k] + red[8 + k]) + (red[16 + k] + red[24 + k]);
                    const size_t row = (head0 + k) * P.stride + e;
                    float mk = m_ref[0];
#pragma unroll
                    for (int h = 1; h < 8; ++h)
                        if (k == h) mk = m_ref[h];
                    P.ws_m[row] = (L > 0.0f) ? mk * 0.69314718055994531f : -INFINITY;
                    P.ws_l[row] = L;
                }
                if (sq.j1 == sq.tl.count()) {
                    // later body entries of the pair: empty
                    for (int i = k; i < G * (J.Eb - e - 1); i += 128) {
                        const size_t idx = (head0 + i % G) * P.stride + e + 1 + i / G;
                        P.ws_m[idx] = -INFINITY;
                        P.ws_l[idx] = 0.0f;
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < NB / 2; ++i) dk[i] = dk_next[i];
            sq.next(P, J, bid);
        }
    } else {
        // ------------------------------------------------ V group: V', Q'^T
        const int k = threadIdx.x - 128;
        uint32_t w[ROWW];  // raw V row of tile t (then of tile t + 1)
        TcSeq pf = sq;
        load_row<ROWW>(w, tile_row<ROWB>(P, pf, k, P.v_planes));
        const uint32_t magic = kMagic;
        const uint32_t neg1032 = 0xE408E408u;    // (-1032, -1032)
        const uint32_t sixteenth = 0x2C002C00u;  // (1/16, 1/16)
        const uint32_t neg72 = 0xD480D480u;      // (-72, -72)
        bool ok = true;
        for (int t = 0; ok && sq.valid; ++t) {
            if (t >= 2) {  // V'(t - 2), P'(t - 2) and the scales of t - 2 are read
                ok = mbar_wait(&bars->pv_done[t & 1], ((t - 2) >> 1) & 1, abort, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
            }
            if (sq.first()) {
                write_qt<HD>(P, smem + C::OFF_Q + (sq.piece & 1) * C::QBUF, sq.u, sq.g, G, k);
                fence_proxy_async_smem();
                mbar_arrive(&bars->q_full[sq.piece & 1]);
            }
            // ---- V' of tile t: exact c - 8 as fp16, MN-major with the 128-byte swizzle
            uint8_t *vs = smem + C::OFF_V + (t & 1) * C::VSTAGE;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                uint32_t x[4];
                block_words<ROWW>(w, b, x);
                uint32_t lo[8], hi[8];
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
                    const uint32_t y = x[wi] >> 8;
                    lo[2 * wi] = hadd2u(and_or<0x000F000Fu>(x[wi], magic), neg1032);
                    lo[2 * wi + 1] = hadd2u(and_or<0x000F000Fu>(y, magic), neg1032);
                    hi[2 * wi] = hfma2u(and_or<0x00F000F0u>(x[wi], magic), sixteenth, neg72);
                    hi[2 * wi + 1] = hfma2u(and_or<0x00F000F0u>(y, magic), sixteenth, neg72);
                }
                // positions 32 b .. 32 b + 31: units of 8 fp16 (lo 0-1, hi 2-3)
#pragma unroll
                for (int un = 0; un < 4; ++un) {
                    const int P0 = 32 * b + 8 * un;
                    const int c = P0 >> 6, unit = (P0 & 63) >> 3;
                    const uint32_t *src = un < 2 ? lo + 4 * un : hi + 4 * (un - 2);
                    *reinterpret_cast<uint4 *>(vs + c * C::VCHUNK + k * 128 + ((unit ^ (k & 7)) << 4)) =
                        make_uint4(src[0], src[1], src[2], src[3]);
                }
            }
            {   // the key's V block scales, for the K group's P'
                uint32_t sc[NB / 2];
#pragma unroll
                for (int b2 = 0; b2 < NB / 2; ++b2)
                    sc[b2] = block_scale_bits<ROWW>(w, 2 * b2) |
                             (block_scale_bits<ROWW>(w, 2 * b2 + 1) << 16);
                *reinterpret_cast<uint4 *>(smem + C::OFF_SC + (t & 1) * C::SCSTAGE + k * 16) =
                    make_uint4(sc[0], sc[1], sc[2], sc[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars->v_full[t & 1]);
            // the raw row of tile t + 1: it lands while the K group scores tile t
            if (pf.valid && pf.next(P, J, bid)) load_row<ROWW>(w, tile_row<ROWB>(P, pf, k, P.v_planes));
            sq.next(P, J, bid);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace

bool q4_tc_supported(int head_dim, int G) { return head_dim == 256 && G <= 8; }

int q4_tc_tile_keys() { return kTK; }

cudaError_t launch_q4_tc(const DecodeParams &P, int head_dim, cudaStream_t stream) {
    if (head_dim != 256) return cudaErrorInvalidValue;
    using C = TcCfg<256>;
    cudaError_t e = cudaFuncSetAttribute(decode_q4_tc_kernel<256>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    decode_q4_tc_kernel<256><<<P.q4_body_blocks, kThreads, C::SMEM, stream>>>(P);
    return cudaGetLastError();
}

}  // namespace fa
