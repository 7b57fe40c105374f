// bwd_sm103.cu -- FlashAttention-2 backward main kernel for GB300 (sm_103a),
// f16 / bf16 inputs, head dim 64 or 128 (32 and 96 run these with zero-filled columns).
//
// Math (the chain rule of O = softmax(scale Q K^T) V, with the saved LSE as
// the softmax normaliser and D from the preprocess step; boostr
// flash_bwd.rs, doc comment "Two-step process", step 2 "compute dQ
// (atomicAdd), dK, dV"):
//   S^T  = K Q^T            P^T  = exp2(S^T * scale*log2e - LSE*log2e)
//   dP^T = V dO^T           dS^T = P^T * (dP^T - D)
//   dV  += P^T dO           dK  += dS^T Q        dQacc += dS K  (fp32 reduction)
//
// Design (Blackwell-native, not the pages' one-thread-per-key-row design):
//   * one CTA owns a 128-row key/value tile of one (batch, kv head) and walks
//     every 128-row query tile of every query head of the group, so dK and dV
//     of the group are summed in tensor memory without atomics.  Causal calls
//     start the heaviest key tiles first; non-causal and windowed calls run the
//     groups in blocks of 4 (L2 locality of the dQ adds and the Q / dO reads);
//   * the five per-tile products run on the 5th-generation tensor cores
//     (tcgen05.mma, M = 128, fp32 accumulation in TMEM).  S^T and dP^T are
//     computed "key-major" (TMEM lane = key row), so the softmax-gradient
//     threads own one key row each and write P^T / dS^T back into TMEM, packed
//     to 16 bits, as the A operand of the dV / dK products;
//   * TMA (cp.async.bulk.tensor, 128-byte swizzle) stages K, V once and Q, dO
//     in a multi-stage ring; tiles that no query can see are skipped;
//   * the dQ tile (dS K) is drained from TMEM and added to the fp32
//     accumulator in global memory with TMA bulk reduce-adds, staged through
//     the dS shared-memory tile (free once the dQ product ran) and, for d = 128,
//     the iteration's dO tile (free once the dV product ran);
//   * warp roles: warps 0-3 drain dQ; warps 4-11 compute P and dS and run the
//     dK / dV epilogue, two warps per TMEM lane quadrant (one per 64-query half,
//     so each SM sub-partition has two of them to hide TMEM / shared latency);
//     warp 12 issues TMA; warp 13 owns TMEM and issues MMAs (at d = 64 the S and
//     dP products, warp 14 the dV, dQ and dK products); the deterministic
//     instance adds one warp that takes the dQ turns and issues the reduce-adds;
//   * 128-column TMEM buffers take the roles X(i): S(i) -> P(i) (packed) -> dQ(i)
//     and Y(i): dP(i) -> dS(i) (packed in place), where "packed" puts queries
//     [0,64) in columns [0,32) and queries [64,128) in columns [64,96).  Two
//     buffers at d = 128 (Y(i) becomes X(i+1): S(i+1) waits for the dK product
//     of iteration i); three at d = 64, where S(i+1) goes into Y(i-1) and runs
//     while the softmax warps still work on iteration i.  dP(i+1) always goes
//     into X(i) once dQ(i) has been drained; the dQ product is issued first once
//     dS(i) is ready, so its drain starts as early as possible;
//   * every mbarrier wait is bounded: on timeout the kernel records an error
//     word, lets the other roles drop out, waits for its own copies / MMAs in
//     flight, frees TMEM and returns.
//
// TMEM columns (512 allocated): dV [0, D), dK [D, 2D), buffers from 2D, 128
// columns each (two at D = 128, three at D = 64).
#include <math.h>

#include "bounded_wait.cuh"
#include "fa_internal.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int BM = kTileQ;  // 128 query rows per iteration
constexpr int BN = kTileK;  // 128 key rows per CTA
static_assert(BM == 128, "the packed P / dS column layout assumes two 64-query halves");
// 14 warps; d = 64 adds a second MMA-issuing warp (kWarpMma2) and deterministic mode a warp for
// the dQ turns (red_warp)
__host__ __device__ constexpr int threads_for(bool det, int D) { return 32 * (14 + (D == 64) + det); }
__host__ __device__ constexpr int red_warp(int D) { return D == 64 ? 15 : 14; }
// warps 0-3 drain dQ; warps 4-11 compute P / dS (two warps per TMEM lane quadrant, one
// per half of the query columns); warp 12 issues TMA; warp 13 owns TMEM and issues MMAs;
// warp 14, in deterministic mode, takes the dQ turns and issues the dQ reduce-adds
constexpr int kWarpDrain0 = 0, kWarpSoft0 = 4, kNumSoftWarps = 8, kWarpTma = 12, kWarpMma = 13,
              kWarpMma2 = 14;
constexpr int kHalfQ = BM / 2;  // query columns per softmax warp
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDrainBarrier = 1;                           // named barrier of the drain warps

template <int D>
struct Cfg {
    static constexpr int STAGES = D == 128 ? 2 : 3;
    // d = 64 leaves TMEM room for a third S / dP buffer (dV, dK take 64 columns each) and
    // shared memory for a second dS tile, so S(i+1) need not wait for the dK product of
    // iteration i, nor dS(i+1) for the dQ(i) reduce to read the dS tile
    static constexpr int NBUF = D == 64 ? 3 : 2;  // 128-column TMEM buffers
    static constexpr int NDS = D == 64 ? 2 : 1;   // shared dS tiles
    static constexpr int BOXES = D / 64;                 // 64-column boxes per tile row
    static constexpr uint32_t kTileK_B = BN * D * 2;     // K or V tile bytes
    static constexpr uint32_t kTileQ_B = BM * D * 2;     // Q or dO tile bytes
    static constexpr uint32_t kBoxK_B = BN * 128;        // one 64-column box of K / V
    static constexpr uint32_t kBoxQ_B = BM * 128;        // one 64-column box of Q / dO
    static constexpr uint32_t kdS_B = BN * BM * 2;       // dS tile; also the dQ staging area
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = OFF_K + kTileK_B;
    static constexpr uint32_t OFF_Q = OFF_V + kTileK_B;
    static constexpr uint32_t OFF_DO = OFF_Q + STAGES * kTileQ_B;
    static constexpr uint32_t OFF_DS = OFF_DO + STAGES * kTileQ_B;
    static constexpr uint32_t OFF_LSE = OFF_DS + NDS * kdS_B;
    static constexpr uint32_t OFF_DD = OFF_LSE + STAGES * BM * 4;
    static constexpr uint32_t OFF_BAR = OFF_DD + STAGES * BM * 4;
    static constexpr uint32_t kNumBars = 23 + 4 * STAGES;  // B_STAGE0 + 4 * STAGES
    static constexpr uint32_t OFF_MISC = OFF_BAR + kNumBars * 8;
    static constexpr uint32_t SMEM = OFF_MISC + 16;
    static constexpr uint32_t TM_DV = 0, TM_DK = D, TM_BUF0 = 2 * D;
    static_assert(TM_BUF0 + 128 * NBUF <= kTmemCols, "TMEM columns");
    static_assert(kdS_B == 2 * BM * 128, "the dS tile doubles as two 128-row x 32-fp32 dQ staging boxes");
};

// Barrier slots.
enum {
    B_KV = 0,      // K, V landed (TMA)
    B_S_FULL,      // S(i) in TMEM (MMA commit); one per TMEM buffer when there are 3
    B_DP_FULL = B_S_FULL + 3,  // dP(i) in TMEM (MMA commit)
    B_P_READY,     // P(i) packed in TMEM (8 softmax warps); one per TMEM buffer when there are 3
    B_DS_READY = B_P_READY + 3,  // dS(i) packed in TMEM and in shared memory (8 softmax warps)
    B_DS_EMPTY,    // a shared dS tile free again: dQ(i) staged out of it and read by TMA; one per tile
    B_DQ_FULL = B_DS_EMPTY + 2,  // dQ(i) in TMEM (MMA commit)
    B_DQ_EMPTY,    // dQ(i) copied out of TMEM (4 drain warps)
    B_DQ_STAGED,   // dQ(i) staged in dS tile dt(i) for the deterministic adds (4 drain warps); one per tile
    B_G3 = B_DQ_STAGED + 2,          // dV product of iteration i done (MMA commit)
    B_G4,          // dK product of iteration i done (MMA commit)
    B_ACC,         // every product done: dK / dV final (MMA commit)
    B_FINAL,       // MMA shutdown
    B_FINAL_A,     // S / dP issuer shutdown (two issuers)
    B_YFREE,       // two issuers: the dK product of the iteration that used buffer k as Y is done
    B_STAGE0 = B_YFREE + 3  // then the stage ring: STAGES "full" and STAGES "empty" barriers for
                            // the Q tiles (with the LSE rows), then the same for the dO tiles (with D)
};

struct Params {
    const float* lse2;
    const float* Dws;
    void* dK;
    void* dV;
    unsigned int* err;
    unsigned int* dq_sem;  // deterministic dQ: [B*H][query tiles] turn counters, else nullptr
    unsigned int* ticket;  // deterministic dQ: counter handing out logical CTA indices, else nullptr
    int B, H, H_kv, S_q, S_k, S_q_pad;
    int d;  // head dim of the tensors (<= D: columns d..D-1 are zero-filled by TMA, never stored)
    float scale, scale_log2;
    int causal, window;
    int group_chunk;  // (b, kv head) groups per block of the CTA order (divides B * H_kv)
};

// TMEM column (relative to a buffer) of the packed 16-bit A operand for MMA k-step k
// (queries [16k, 16k+16)): each 64-query half is packed into the first 32 columns of
// the 64 fp32 columns it was read from.
__device__ __forceinline__ uint32_t packed_col(int k) { return (uint32_t)((k / 4) * 64 + (k % 4) * 8); }

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack2_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    return kBF16 ? pack2_bf16(lo, hi) : pack2_f16(lo, hi);
}
template <bool kBF16>
__device__ __forceinline__ float2 unpack2(uint32_t v) {
    if (kBF16) return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
    return __half22float2(*reinterpret_cast<__half2*>(&v));
}

// tcgen05.wait::ld that also names the 32 registers a tcgen05.ld filled as operands, so the
// compiler cannot move a use of them above the wait (they are written asynchronously).
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t* r) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                   "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
                   "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
                   "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
                   "+r"(r[31])
                 :
                 : "memory");
}

static_assert(B_STAGE0 == 23, "Cfg::kNumBars counts 23 named barriers before the stage ring");

template <typename T, int D, bool kDet, int kSplit>
__global__ void __launch_bounds__(threads_for(kDet, D), 1)
    bwd_sm103_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                     const __grid_constant__ CUtensorMap tmdQ, const Params p) {
    using C = Cfg<D>;
    constexpr bool kBF16 = TypeTraits<T>::kId == FA_BF16;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // the dQ finalisation (launched as a programmatic dependent) may be scheduled once every
    // CTA of this grid has started; it waits for this grid to complete
    ptx::griddep_launch_dependents();
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 4);
    uint32_t* ticket_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 8);
    auto bar = [&](int i) { return sbase + C::OFF_BAR + 8u * (uint32_t)i; };
    // At d = 128 the Q and dO stages are loaded and released separately: the drain stages half
    // of dQ(i) in the dO tile, and the Q tile of iteration i+2 (for S(i+2) and the P pass) need
    // not wait until TMA has read that out.  At d = 64 both tiles of an iteration share one
    // full and one empty barrier (measured 3 % faster there).
    constexpr bool kSplitRing = D == 128;
    constexpr bool kPipeLd = D == 128;  // softmax passes: TMEM loads in two halves, overlapped
    auto full_q = [&](int s) { return bar(B_STAGE0 + s); };
    auto empty_q = [&](int s) { return bar(B_STAGE0 + C::STAGES + s); };
    auto full_do = [&](int s) { return kSplitRing ? bar(B_STAGE0 + 2 * C::STAGES + s) : full_q(s); };
    auto empty_do = [&](int s) { return kSplitRing ? bar(B_STAGE0 + 3 * C::STAGES + s) : empty_q(s); };

    if (threadIdx.x == 0) {
        if ((sbase & 1023u) != 0) atomicOr(p.err, kErrSmemAlign);
        *abort_flag = (sbase & 1023u) != 0;
        for (int i = 0; i < (int)C::kNumBars; ++i) {
            uint32_t count = ((i >= B_P_READY && i < B_P_READY + 3) || i == B_DS_READY) ? (uint32_t)kNumSoftWarps
                             : (i == B_DQ_EMPTY || i == B_DQ_STAGED || i == B_DQ_STAGED + 1) ? 4u
                                                               : 1u;
            if (D == 128 && i >= B_STAGE0 + 3 * C::STAGES) count = 2;  // dO stage "empty": MMA + drain
            ptx::mbar_init(bar(i), count);
        }
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
        if (kDet) *ticket_slot = atomicAdd(p.ticket, 1u);
    }
    if (warp == kWarpMma) {
        ptx::tmem_alloc(sbase + C::OFF_MISC + 4, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tm_buf0 = tmem + C::TM_BUF0;  // buffer x at tm_buf0 + 128 * x

    // ---- work assignment: logical index blk = (block of group_chunk (b, kv head) groups) x
    // key tile x (group within the block).  blk is blockIdx.x, except in deterministic mode,
    // where each CTA takes it from a ticket counter in the order the CTAs start: a CTA then
    // only waits (for dQ turns) on CTAs of lower logical index, which have all started,
    // whatever order the hardware dispatches blocks in.  With one block of every group
    // (causal) the heaviest key tiles (most query tiles) start first.  When every key tile
    // sees about as many query tiles (no causal mask, or a sliding window) blocks of a few
    // groups run one after the other instead, so that all key-tile CTAs of a group run side
    // by side.  Each CTA walks its query tiles from the last one down, heads innermost: CTAs
    // running side by side reduce into and read the same dQ / Q / dO tiles at about the
    // same time.  Within a group a lower key tile always has a lower logical index.
    const int n_key_tiles = (p.S_k + BN - 1) / BN;
    // With split = 2 (default mode only) the two CTAs of a cluster share one logical index,
    // each taking one contiguous half of its query tiles, and add their dK / dV partials
    // through distributed shared memory at the end (small grids, long causal key tiles).
    const int rank = kSplit > 1 ? (int)(blockIdx.x % kSplit) : 0;  // rank within the 1-D cluster
    const int blk = kDet ? (int)*ticket_slot : (int)(blockIdx.x / kSplit);
    const int chunk = blk / (n_key_tiles * p.group_chunk);
    const int in_chunk = blk % (n_key_tiles * p.group_chunk);
    const int n_tile = in_chunk / p.group_chunk;
    const int bkv = chunk * p.group_chunk + in_chunk % p.group_chunk;
    const int b = bkv / p.H_kv, hk = bkv % p.H_kv;
    const int g = p.H / p.H_kv;
    const int n0 = n_tile * BN;
    const int off = p.S_k - p.S_q;  // query i sits at key position i + off
    // query tiles [m_start, m_end) hold every row that sees a key of this tile (causal
    // edge below, sliding-window band edges on either side)
    Shape sh;  // the fields the range helpers read
    sh.S_q = p.S_q;
    sh.S_k = p.S_k;
    sh.causal = p.causal;
    sh.window = p.window;
    int q_lo, q_hi;
    query_range(sh, n0, min(n0 + BN, p.S_k), q_lo, q_hi);
    const int m_tiles = (p.S_q + BM - 1) / BM;
    const int m_first = q_lo / BM;
    const int m_last = q_hi > q_lo ? (q_hi + BM - 1) / BM : m_first;
    // this CTA's query tiles [m_start, m_end)
    const int m_start = kSplit > 1 ? m_first + (m_last - m_first) * rank / kSplit : m_first;
    const int m_end = kSplit > 1 ? m_first + (m_last - m_first) * (rank + 1) / kSplit : m_last;
    const int nm = m_end - m_start;
    const int n_it = g * nm;

    // Buffer roles.  Iteration i computes S(i) -> P(i) -> dQ(i) in buffer xb(i) and
    // dP(i) -> dS(i) in buffer yb(i); dP(i+1) always goes into xb(i) once dQ(i) left it.
    // Two buffers: S(i+1) goes into yb(i) once the dK product of iteration i has read dS(i).
    // Three: buffer k serves as xb(i), yb(i+1), xb(i+3), ..., so S(i+1) goes into yb(i-1),
    // free once the dK product of iteration i-1 is done, and runs while the softmax still
    // works on iteration i.  Each buffer then has its own S / P barriers (its uses are three
    // iterations apart, so no parity wait can see a phase two ahead).  dS(i) is staged in
    // shared dS tile dt(i).
    constexpr int NBUF = C::NBUF, NDS = C::NDS;
    auto xb = [](int i) { return NBUF == 3 ? (2 * i) % 3 : (i & 1); };
    auto yb = [](int i) { return NBUF == 3 ? (2 * i + 1) % 3 : ((i & 1) ^ 1); };
    auto sp_slot = [](int i) { return NBUF == 3 ? (2 * i) % 3 : 0; };  // S / P barrier of iteration i
    auto sp_par = [](int i) { return NBUF == 3 ? (i / 3) & 1 : i & 1; };
    auto dt = [](int i) { return NDS == 2 ? (i & 1) : 0; };

    auto iter_coords = [&](int it, int& bh, int& m0) {
        const int hh = it % g;
        m0 = (m_end - 1 - it / g) * BM;
        bh = b * p.H + hk * g + hh;
    };
    // Bulk reduce-adds of the dQ tile staged for iteration it (one thread), then the
    // releases once TMA has read each staging area: the dS tile (B_DS_EMPTY) and, at
    // d = 128, the dO stage, whose second arrival (after the MMA warp's, once the dK
    // product is done) lets the next dO load in.
    auto reduce_staged = [&](int s, int tile, int bh, int m0, bool add) {
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {  // one bulk group per staging area, dS tile first
            const uint32_t area =
                sbase + (h == 0 ? C::OFF_DS + tile * C::kdS_B : C::OFF_DO + s * C::kTileQ_B);
            if (add) {  // 32-column boxes past the head dim hold zeros and are not added
                // the accumulator lines stay in L2 ahead of the Q / dO stream: the
                // finalise pass then reads much of dQacc from L2
                const uint64_t pol = ptx::policy_evict_last();
                if (h * 64 < p.d) ptx::tma_reduce_add_3d_hint(&tmdQ, area, h * 64, m0, bh, pol);
                if (h * 64 + 32 < p.d) ptx::tma_reduce_add_3d_hint(&tmdQ, area + BM * 128, h * 64 + 32, m0, bh, pol);
            }
            ptx::bulk_commit_group();
        }
        if (D == 128) {
            ptx::bulk_wait_read_1();  // the dS-tile group (the older one) was read
            ptx::mbar_arrive(bar(B_DS_EMPTY + tile));
            ptx::bulk_wait_read_all();
            ptx::mbar_arrive(empty_do(s));  // second of two arrivals (MMA commit after dK)
        } else {
            ptx::bulk_wait_read_all();
            ptx::mbar_arrive(bar(B_DS_EMPTY + tile));
        }
    };
    constexpr bool det = kDet;  // p.dq_sem holds the turn counters

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ producer
        // One thread loads K, V, then the Q tiles (with the LSE rows) and the dO tiles (with
        // D) of the stage ring, each as soon as its own slot is free, polling both "empty"
        // barriers without blocking on either.
        if (lane == 0 && !*abort_flag) {
            // K and V are read by this CTA alone: their lines go first when L2 needs room (the dQ
            // accumulator lines the reduce-adds update stay; measured 0.6 % faster)
            const uint64_t kv_pol = ptx::policy_evict_first();
            ptx::mbar_arrive_expect_tx(bar(B_KV), 2 * C::kTileK_B);
            for (int x = 0; x < C::BOXES; ++x) {
                ptx::tma_load_3d_hint(sbase + C::OFF_K + x * C::kBoxK_B, &tmK, x * 64, n0, bkv, bar(B_KV), kv_pol);
                ptx::tma_load_3d_hint(sbase + C::OFF_V + x * C::kBoxK_B, &tmV, x * 64, n0, bkv, bar(B_KV), kv_pol);
            }
            // launched as a programmatic dependent of the preprocess pass: the LSE copy and D it
            // writes are read from here on
            ptx::griddep_wait();
            ptx::fence_proxy_async_global();
            // the lse2 and D rows travel with the Q tile (the P pass waits for it; the dS pass
            // comes later in the same iteration and the Q stage is released after the dK product)
            auto load = [&](bool is_q, int it) {
                const int s = it % C::STAGES;
                int bh, m0;
                iter_coords(it, bh, m0);
                const uint32_t full = is_q ? full_q(s) : full_do(s);
                const uint32_t bytes = is_q ? C::kTileQ_B * (kSplitRing ? 1 : 2) + 2 * BM * 4 : C::kTileQ_B;
                if (is_q || kSplitRing) ptx::mbar_arrive_expect_tx(full, bytes);
                for (int x = 0; x < C::BOXES; ++x)
                    ptx::tma_load_3d(sbase + (is_q ? C::OFF_Q : C::OFF_DO) + s * C::kTileQ_B + x * C::kBoxQ_B,
                                     is_q ? &tmQ : &tmdO, x * 64, m0, bh, full);
                if (is_q) {
                    const size_t row0 = (size_t)bh * p.S_q_pad + m0;
                    ptx::bulk_load(sbase + C::OFF_LSE + s * BM * 4, p.lse2 + row0, BM * 4, full);
                    ptx::bulk_load(sbase + C::OFF_DD + s * BM * 4, p.Dws + row0, BM * 4, full);
                }
            };
            int iq = 0, id = 0;  // loads issued
            uint64_t t0 = ptx::globaltimer();
            uint32_t spins = 0;
            while (iq < n_it || id < n_it) {
                bool progress = false;
                if (iq < n_it && (iq < C::STAGES || ptx::mbar_test_wait(empty_q(iq % C::STAGES),
                                                                        ((iq / C::STAGES) - 1) & 1))) {
                    load(true, iq);
                    if (!kSplitRing) load(false, id++);  // one shared barrier: both tiles at once
                    ++iq;
                    progress = true;
                }
                if (kSplitRing && id < n_it &&
                    (id < C::STAGES || ptx::mbar_test_wait(empty_do(id % C::STAGES), ((id / C::STAGES) - 1) & 1))) {
                    load(false, id++);
                    progress = true;
                }
                if (progress) {
                    t0 = ptx::globaltimer();
                } else if (++spins % 64 == 0) {
                    if (*abort_flag) break;
                    if (ptx::globaltimer() - t0 > kWaitLimitNs) {
                        *abort_flag = 1;
                        atomicOr(p.err, kErrTimeout);
                        break;
                    }
                }
            }
            // never leave copies in flight into shared memory that is about to be released
            drain_wait(bar(B_KV), 0);
            for (int it = iq - C::STAGES < 0 ? 0 : iq - C::STAGES; it < iq; ++it)
                drain_wait(full_q(it % C::STAGES), (it / C::STAGES) & 1);
            if (kSplitRing)
                for (int it = id - C::STAGES < 0 ? 0 : id - C::STAGES; it < id; ++it)
                    drain_wait(full_do(it % C::STAGES), (it / C::STAGES) & 1);
        }
    } else if (warp == kWarpMma || (NBUF == 3 && warp == kWarpMma2)) {
        // ------------------------------------------------------------ MMA issuers
        // With two TMEM buffers warp 13 issues every product.  With three (d = 64) warp 13
        // issues S and dP and warp 14 dV, dQ and dK, so that no product waits behind another's
        // inputs in one thread's program order (measured with clock64 stamps: one issuer
        // waiting for the dK product of iteration i-1 before S(i+1) saw P(i) ~2.4K cycles
        // late).  Every hazard between the two is on a barrier: S(i+1) into yb(i-1) waits for
        // that buffer's Y-free barrier (the dK product of iteration i-1, one barrier per
        // buffer, so no wait can see a phase two ahead), dP(i+1) into xb(i) for the drain's
        // B_DQ_EMPTY; the dV, dQ and dK products follow the softmax's P and dS barriers, which
        // imply S(i) and dP(i) are complete.
        const bool issue_sd = NBUF == 2 || warp == kWarpMma;  // S and dP products
        const bool issue_g = NBUF == 2 || warp == kWarpMma2;  // dV, dQ and dK products
        if (lane == 0 && !*abort_flag && n_it > 0) {
            constexpr uint32_t ID_SD = ptx::idesc_f16(BN, BM, kBF16, false, false);  // S^T, dP^T
            constexpr uint32_t ID_KV = ptx::idesc_f16(BN, D, kBF16, false, true);    // dV, dK (A in TMEM)
            constexpr uint32_t ID_Q = ptx::idesc_f16(BM, D, kBF16, true, true);      // dQ
            const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
            // S^T = K Q^T or dP^T = V dO^T into a TMEM buffer; both operands K-major.
            auto gemm_sd = [&](uint32_t d_tmem, uint32_t a_base, uint32_t b_base) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t koff = (k / 4) * C::kBoxK_B + (k % 4) * 32;
                    const uint32_t koffb = (k / 4) * C::kBoxQ_B + (k % 4) * 32;
                    ptx::mma_ss(d_tmem, ptx::sw128_desc(a_base + koff, 16, 1024),
                                ptx::sw128_desc(b_base + koffb, 16, 1024), ID_SD, k > 0);
                }
            };
            bool ok = true;
            if (issue_sd) {
                ok = wait_bar(bar(B_KV), 0, abort_flag, p.err);
                if (ok) ok = wait_bar(full_q(0), 0, abort_flag, p.err);
                if (ok) {
                    ptx::tc_fence_after();
                    gemm_sd(tm_buf0 + 128 * xb(0), sK, sbase + C::OFF_Q);
                    ptx::mma_commit(bar(B_S_FULL + sp_slot(0)));
                }
                if (ok) ok = wait_bar(full_do(0), 0, abort_flag, p.err);
                if (ok) {
                    ptx::tc_fence_after();
                    gemm_sd(tm_buf0 + 128 * yb(0), sV, sbase + C::OFF_DO);
                    ptx::mma_commit(bar(B_DP_FULL));
                }
            }
            for (int it = 0; ok && it < n_it; ++it) {
                const int s = it % C::STAGES;
                const int s1 = (it + 1) % C::STAGES;
                const uint32_t X = tm_buf0 + 128 * xb(it);  // S -> P -> dQ of this iteration
                const uint32_t Y = tm_buf0 + 128 * yb(it);  // dP -> dS of this iteration
                const uint32_t sQ = sbase + C::OFF_Q + s * C::kTileQ_B;
                const uint32_t sdO = sbase + C::OFF_DO + s * C::kTileQ_B;
                const uint32_t sdS = sbase + C::OFF_DS + dt(it) * C::kdS_B;
                if (NBUF == 3 && issue_sd) {
                    if (it + 1 < n_it) {
                        // S(i+1) into yb(i-1) once Q(i+1) is in and the dK product of iteration
                        // i-1 stopped reading dS(i-1) from it (the first iteration's is unused)
                        if (!(ok = wait_bar(full_q(s1), ((it + 1) / C::STAGES) & 1, abort_flag, p.err))) break;
                        if (it > 0 &&
                            !(ok = wait_bar(bar(B_YFREE + yb(it - 1)), ((it - 1) / 3) & 1, abort_flag, p.err)))
                            break;
                        ptx::tc_fence_after();
                        gemm_sd(tm_buf0 + 128 * xb(it + 1), sK, sbase + C::OFF_Q + s1 * C::kTileQ_B);
                        ptx::mma_commit(bar(B_S_FULL + sp_slot(it + 1)));
                        // dP(i+1) into xb(i) once dQ(i) left it
                        if (!(ok = wait_bar(bar(B_DQ_EMPTY), it & 1, abort_flag, p.err))) break;
                        if (!(ok = wait_bar(full_do(s1), ((it + 1) / C::STAGES) & 1, abort_flag, p.err))) break;
                        ptx::tc_fence_after();
                        gemm_sd(X, sV, sbase + C::OFF_DO + s1 * C::kTileQ_B);
                        ptx::mma_commit(bar(B_DP_FULL));
                    }
                    continue;
                }
                // dV += P^T dO.  A = P^T in TMEM: queries [0,64) packed in X[0,32), queries
                // [64,128) in X[64,96); 16 queries = 8 packed columns per step.
                if (!(ok = wait_bar(bar(B_P_READY + sp_slot(it)), sp_par(it), abort_flag, p.err))) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int k = 0; k < BM / 16; ++k)
                    ptx::mma_ts(tmem + C::TM_DV, X + packed_col(k), ptx::sw128_desc(sdO + k * 2048, C::kBoxQ_B, 1024),
                                ID_KV, (it > 0 || k > 0) ? 1u : 0u);
                ptx::mma_commit(bar(B_G3));
                // dQ = dS K first (its drain is the longest chain), into X once the dV
                // product stopped reading P from it
                if (!(ok = wait_bar(bar(B_DS_READY), it & 1, abort_flag, p.err))) break;
                if (!(ok = wait_bar(bar(B_G3), it & 1, abort_flag, p.err))) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                    ptx::mma_ss(X, ptx::sw128_desc(sdS + k * 2048, BN * 128, 1024),
                                ptx::sw128_desc(sK + k * 2048, C::kBoxK_B, 1024), ID_Q, k > 0);
                ptx::mma_commit(bar(B_DQ_FULL));
                // dK += dS^T Q   (A = dS^T in TMEM, packed like P^T, in Y)
#pragma unroll
                for (int k = 0; k < BM / 16; ++k)
                    ptx::mma_ts(tmem + C::TM_DK, Y + packed_col(k), ptx::sw128_desc(sQ + k * 2048, C::kBoxQ_B, 1024),
                                ID_KV, (it > 0 || k > 0) ? 1u : 0u);
                ptx::mma_commit(bar(NBUF == 3 ? B_YFREE + yb(it) : B_G4));
                // Q(i), dO(i) no longer read by MMAs (S(i) and dP(i) completed before dS(i);
                // for d = 128 the dO stage is free only once the drain also arrived: it stages
                // half of dQ(i) in the dO tile)
                ptx::mma_commit(empty_q(s));
                if (kSplitRing) ptx::mma_commit(empty_do(s));
                if (NBUF == 2 && it + 1 < n_it) {
                    // S(i+1) into Y once the dK product stopped reading dS(i) from it
                    if (!(ok = wait_bar(full_q(s1), ((it + 1) / C::STAGES) & 1, abort_flag, p.err))) break;
                    if (!(ok = wait_bar(bar(B_G4), it & 1, abort_flag, p.err))) break;
                    ptx::tc_fence_after();
                    gemm_sd(Y, sK, sbase + C::OFF_Q + s1 * C::kTileQ_B);
                    ptx::mma_commit(bar(B_S_FULL + sp_slot(it + 1)));
                    // dP(i+1) into X once dQ(i) left it
                    if (!(ok = wait_bar(bar(B_DQ_EMPTY), it & 1, abort_flag, p.err))) break;
                    if (!(ok = wait_bar(full_do(s1), ((it + 1) / C::STAGES) & 1, abort_flag, p.err))) break;
                    ptx::tc_fence_after();
                    gemm_sd(X, sV, sbase + C::OFF_DO + s1 * C::kTileQ_B);
                    ptx::mma_commit(bar(B_DP_FULL));
                }
            }
            if (issue_g) ptx::mma_commit(bar(B_ACC));
            // no MMA of this thread may still write TMEM when it is released
            const int fin = issue_g ? B_FINAL : B_FINAL_A;
            ptx::mma_commit(bar(fin));
            drain_wait(bar(fin), 0);
        }
        __syncwarp();
    } else if (warp >= kWarpSoft0 && warp < kWarpSoft0 + kNumSoftWarps) {
        // ------------------------------------------------------------ P / dS
        // One key row per thread (TMEM lane), two warps per lane quadrant: warp half hf
        // owns query columns [hf*64, hf*64+64) of S / dP and packs its P / dS into the
        // first 32 of those columns, so the two warps of a quadrant never touch each
        // other's TMEM columns.
        const int qd = warp & 3;                          // TMEM lane quadrant
        const int hf = (warp - kWarpSoft0) >> 2;          // query half
        const int qh = hf * kHalfQ;                       // first query column of this warp
        const int t = qd * 32 + lane;                     // key row within the tile
        const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
        const int j = n0 + t;
        const bool row_valid = j < p.S_k;
        // key-major rows of the shared dS tile, 128-byte swizzled MN-major; one 64-query block per half
        uint8_t* sdS_row = smem + C::OFF_DS + hf * (BN * 128) + (t >> 3) * 1024 + (t & 7) * 128;
        bool ok = !*abort_flag;
        for (int it = 0; ok && it < n_it; ++it) {
            const int s = it % C::STAGES;
            const uint32_t X = tm_buf0 + 128 * xb(it) + lane_off + qh;
            const uint32_t Y = tm_buf0 + 128 * yb(it) + lane_off + qh;
            int bh, m0;
            iter_coords(it, bh, m0);
            const int i_lo = m0 + qh;  // first query row of this warp's columns
            // Columns q of this warp (query i_lo + q, key position i_lo + off + q) that see
            // this lane's key j form one interval (visible_queries); a padding key row sees
            // nothing.  Only qa stays live across the waits: the bounds are cheap to redo.
            const int qa = j - i_lo - off;
            // warp-uniform: the chosen path holds .sync.aligned TMEM accesses; the per-element
            // selects inside the masked path handle each lane's own row
            bool full;
            {
                int lo, hi;
                visible_queries(qa, p.causal, p.window, lo, hi);
                full = row_valid && lo <= 0 && hi >= kHalfQ;
            }
            const bool mask_tile = __any_sync(0xffffffffu, !full);
            const float* sl = reinterpret_cast<const float*>(smem + C::OFF_LSE + s * BM * 4) + qh;
            const float* sd = reinterpret_cast<const float*>(smem + C::OFF_DD + s * BM * 4) + qh;
            if (!(ok = wait_bar_warp(full_q(s), (it / C::STAGES) & 1, abort_flag, p.err))) break;
            if (!(ok = wait_bar_warp(bar(B_S_FULL + sp_slot(it)), sp_par(it), abort_flag, p.err))) break;
            ptx::tc_fence_after();
            // P = exp2(S * scale*log2e - LSE*log2e), packed to 16 bits in place.  Masking is
            // decided once per warp, outside the unrolled loop, so the 64 independent exp
            // chains stay one basic block.
            uint32_t Pp[kHalfQ / 2];
            auto p_block = [&](bool masked) {
                // d = 128: the second 32 columns load while the first 32 are computed (bench
                // shape 331 -> 329 us; at d = 64 it measured 241 -> 243 us and is not used)
                uint32_t r[kHalfQ];
                ptx::tmem_ld32p(X, r);
                if constexpr (kPipeLd) {
                    tmem_wait_ld_regs(r);
                    ptx::tmem_ld32p(X + 32, r + 32);
                } else {
                    ptx::tmem_ld32p(X + 32, r + 32);
                    ptx::tmem_wait_ld();
                }
                const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
                for (int q = 0; q < kHalfQ; q += 4) {
                    if (kPipeLd && q == 32) tmem_wait_ld_regs(r + 32);
                    const float4 l4 = *reinterpret_cast<const float4*>(sl + q);
                    float2 a = __ffma2_rn(make_float2(__uint_as_float(r[q]), __uint_as_float(r[q + 1])), sc2,
                                          make_float2(-l4.x, -l4.y));
                    float2 b = __ffma2_rn(make_float2(__uint_as_float(r[q + 2]), __uint_as_float(r[q + 3])), sc2,
                                          make_float2(-l4.z, -l4.w));
                    a = make_float2(ptx::ex2(a.x), ptx::ex2(a.y));
                    b = make_float2(ptx::ex2(b.x), ptx::ex2(b.y));
                    if (masked) {
                        int q_lo, q_hi;
                        visible_queries(qa, p.causal, p.window, q_lo, q_hi);
                        const unsigned q_span = row_valid ? (unsigned)(q_hi - q_lo) : 0u;
                        a.x = (unsigned)(q + 0 - q_lo) < q_span ? a.x : 0.f;
                        a.y = (unsigned)(q + 1 - q_lo) < q_span ? a.y : 0.f;
                        b.x = (unsigned)(q + 2 - q_lo) < q_span ? b.x : 0.f;
                        b.y = (unsigned)(q + 3 - q_lo) < q_span ? b.y : 0.f;
                    }
                    Pp[q / 2] = pack2<kBF16>(a.x, a.y);
                    Pp[q / 2 + 1] = pack2<kBF16>(b.x, b.y);
                }
                ptx::tmem_st32(X, Pp);
            };
            if (mask_tile)
                p_block(true);
            else
                p_block(false);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(B_P_READY + sp_slot(it)));

            // dS = P * (dP - D): packed in place into this warp's first 32 columns of Y for
            // the dK product, and into the shared dS tile for dQ.
            if (!(ok = wait_bar_warp(bar(B_DP_FULL), it & 1, abort_flag, p.err))) break;
            // The dS tile of this iteration was last used NDS iterations ago.  At d = 128 its
            // release is waited for only just before the stores below, so the dP load and the
            // arithmetic overlap the wait (measured 335 -> 331 us on the bench shape, 1193 ->
            // 1165 us on fp16 S = 8192; at d = 64 it made no gain and stays here).
            if (D != 128 && it >= NDS &&
                !(ok = wait_bar_warp(bar(B_DS_EMPTY + dt(it)), ((it - NDS) / NDS) & 1, abort_flag, p.err)))
                break;
            ptx::tc_fence_after();
            {
                // as in the P pass (d = 128)
                uint32_t r[kHalfQ];
                ptx::tmem_ld32p(Y, r);
                if constexpr (kPipeLd) {
                    tmem_wait_ld_regs(r);
                    ptx::tmem_ld32p(Y + 32, r + 32);
                } else {
                    ptx::tmem_ld32p(Y + 32, r + 32);
                    ptx::tmem_wait_ld();
                }
                uint32_t pk[kHalfQ / 2];
#pragma unroll
                for (int q = 0; q < kHalfQ; q += 4) {
                    if (kPipeLd && q == 32) tmem_wait_ld_regs(r + 32);
                    const float4 d4 = *reinterpret_cast<const float4*>(sd + q);
                    const float2 p01 = unpack2<kBF16>(Pp[q / 2]);
                    const float2 p23 = unpack2<kBF16>(Pp[q / 2 + 1]);
                    // dP - D (one rounding, as fp32 subtraction), then times P
                    const float2 t01 = __ffma2_rn(make_float2(d4.x, d4.y), make_float2(-1.f, -1.f),
                                                  make_float2(__uint_as_float(r[q]), __uint_as_float(r[q + 1])));
                    const float2 t23 = __ffma2_rn(make_float2(d4.z, d4.w), make_float2(-1.f, -1.f),
                                                  make_float2(__uint_as_float(r[q + 2]), __uint_as_float(r[q + 3])));
                    const float2 s01 = __fmul2_rn(p01, t01);
                    const float2 s23 = __fmul2_rn(p23, t23);
                    pk[q / 2] = pack2<kBF16>(s01.x, s01.y);
                    pk[q / 2 + 1] = pack2<kBF16>(s23.x, s23.y);
                }
                ptx::tmem_st32(Y, pk);  // columns already read
                if (D == 128 && it >= NDS &&
                    !(ok = wait_bar_warp(bar(B_DS_EMPTY + dt(it)), ((it - NDS) / NDS) & 1, abort_flag, p.err))) {
                    ptx::tmem_wait_st();  // no TMEM store in flight at the release
                    break;
                }
#pragma unroll
                for (int u = 0; u < kHalfQ / 8; ++u)  // 8 queries = one 16-byte chunk
                    *reinterpret_cast<uint4*>(sdS_row + dt(it) * C::kdS_B + ((u ^ (t & 7)) << 4)) =
                        make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(B_DS_READY));
        }
        // ---- epilogue: dV and scale * dK rows to global, columns [hf*D/2, hf*D/2 + D/2).  In a
        // split pair the rows are written after the CTA barrier at the end instead (below).
        if (ok && n_it > 0) ok = wait_bar_warp(bar(B_ACC), 0, abort_flag, p.err);
        if (ok && kSplit == 1) {
            ptx::tc_fence_after();
            T* dVrow = static_cast<T*>(p.dV) + ((size_t)bkv * p.S_k + j) * p.d;
            T* dKrow = static_cast<T*>(p.dK) + ((size_t)bkv * p.S_k + j) * p.d;
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                const int c = hf * (D / 64) + cc;  // 32-column chunk
                uint32_t rv[32], rk[32];
                if (n_it > 0) {
                    ptx::tmem_ld32p(tmem + C::TM_DV + lane_off + c * 32, rv);
                    ptx::tmem_ld32p(tmem + C::TM_DK + lane_off + c * 32, rk);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) rv[k] = rk[k] = 0u;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint32_t ov[4], ok4[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int e = u * 8 + 2 * k;
                        ov[k] = pack2<kBF16>(__uint_as_float(rv[e]), __uint_as_float(rv[e + 1]));
                        ok4[k] = pack2<kBF16>(__uint_as_float(rk[e]) * p.scale, __uint_as_float(rk[e + 1]) * p.scale);
                    }
                    if (row_valid && c * 32 + u * 8 < p.d) {
                        *reinterpret_cast<uint4*>(dVrow + c * 32 + u * 8) = make_uint4(ov[0], ov[1], ov[2], ov[3]);
                        *reinterpret_cast<uint4*>(dKrow + c * 32 + u * 8) = make_uint4(ok4[0], ok4[1], ok4[2], ok4[3]);
                    }
                }
            }
        }
    } else if (warp >= kWarpDrain0 && warp < kWarpDrain0 + 4) {
        // ------------------------------------------------------------ dQ drain (one query row per thread)
        // dQ(i) rows -> registers -> shared memory as 128 x 32 fp32 boxes (128-byte
        // swizzle) -> TMA reduce-add into the fp32 accumulator, issued by the drain's first
        // thread (or, deterministic, by the reduce warp, so that waiting for a turn or for
        // a reduce to complete never holds up the drain).  Columns [0, 64) are staged in
        // the dS tile (free once the dQ product ran), columns [64, 128) in the dO tile of
        // the same iteration (free once the dV product ran), so both bulk reductions are in
        // flight together.  Only bulk reductions are used: per-thread red.global
        // instructions would crowd the SM's memory-instruction path the MMA warp issues
        // through.  Staging dQ(i+1) never overwrites data a reduce has yet to read: it needs
        // dS(i+1) consumed (B_DQ_FULL), and the softmax wrote dS(i+1) only after the dS tile
        // was released (B_DS_EMPTY), while the dO tile of iteration i+1 was loaded only
        // after the stage's previous reduce had read it.
        const int t = (warp - kWarpDrain0) * 32 + lane;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        ptx::griddep_wait();  // the accumulator was zeroed by the preprocess pass
        ptx::fence_proxy_async_global();
        bool ok = !*abort_flag;
        for (int it = 0; ok && it < n_it; ++it) {
            const int s = it % C::STAGES;
            const uint32_t X = tm_buf0 + 128 * xb(it) + lane_off;
            int bh, m0;
            iter_coords(it, bh, m0);
            // all four drain warps take the same decision (each arrives on B_DQ_STAGED below)
            ok = ptx::named_bar_and(kDrainBarrier, 128, wait_bar(bar(B_DQ_FULL), it & 1, abort_flag, p.err));
            if (!ok) break;
            ptx::tc_fence_after();
            // Both staging areas are free: the dQ product (reads dS) and, before it, the dV
            // product (reads dO) are complete (B_DQ_FULL); the previous bulk reduce out of the
            // dS tile was read before B_DS_EMPTY let the next dS in.  64 columns at a time
            // (register budget); the TMEM buffer is released after the last load, which still
            // precedes the end of the dK and next-S products the MMA warp has queued.
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                uint32_t r[64];
                ptx::tmem_ld32p(X + h * 64, r);
                ptx::tmem_ld32p(X + h * 64 + 32, r + 32);
                ptx::tmem_wait_ld();
                if (h == D / 64 - 1) {
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bar(B_DQ_EMPTY));
                }
                uint8_t* area = smem + (h == 0 ? C::OFF_DS + dt(it) * C::kdS_B : C::OFF_DO + s * C::kTileQ_B);
#pragma unroll
                for (int bx = 0; bx < 2; ++bx)
#pragma unroll
                    for (int cq = 0; cq < 8; ++cq) {
                        const int e = bx * 32 + cq * 4;
                        *reinterpret_cast<uint4*>(area + bx * (BM * 128) + t * 128 + ((cq ^ (t & 7)) << 4)) =
                            make_uint4(r[e], r[e + 1], r[e + 2], r[e + 3]);
                    }
            }
            ptx::fence_proxy_async_smem();  // the staged dQ before the bulk reads
            if (det) {  // the reduce warp takes the turn and issues the adds
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(B_DQ_STAGED + dt(it)));
            } else {
                ptx::named_bar_sync(kDrainBarrier, 128);
                if (t == 0) reduce_staged(s, dt(it), bh, m0, true);
            }
        }
        if (!det && t == 0) ptx::bulk_wait_all();
    } else if (warp == red_warp(D)) {
        // ------------------------------------------------------------ deterministic dQ adds
        // One thread waits for each staged dQ(i), takes the tile's turn, issues the
        // reduce-adds and passes the turn on once they are complete, so none of these waits
        // holds up the drain (measured 9 % faster in deterministic mode than in the drain's
        // issuer; the default mode keeps the issuer, 2-4 % faster there).
        if (lane == 0 && det) {
            ptx::griddep_wait();
            ptx::fence_proxy_async_global();
            bool ok = !*abort_flag;
            unsigned int* prev_sem = nullptr;  // turn to pass on once complete
            unsigned int prev_turn = 0;
            for (int it = 0; ok && it < n_it; ++it) {
                const int s = it % C::STAGES;
                int bh, m0;
                iter_coords(it, bh, m0);
                // one barrier per dS tile: with two tiles the drain may stage dQ(i+1) before
                // this thread waits for dQ(i), so a shared barrier could run two phases ahead
                if (!(ok = wait_bar(bar(B_DQ_STAGED + dt(it)), (it / NDS) & 1, abort_flag, p.err))) break;
                // Deterministic dQ: the key tiles that touch this query tile add into it in
                // key-tile order.  Turn t of the tile's counter belongs to its t-th such key
                // tile (they are consecutive: the first is where key_range of the query tile
                // starts).  Wait for the turn, add, and pass it on once the adds are complete:
                // one iteration later, so this thread never waits for its newest reduce.  Holding
                // that turn meanwhile cannot deadlock: only CTAs of higher logical index wait
                // for it, and this CTA never waits for one of those.
                int k_lo, k_hi;
                key_range(sh, m0, min(m0 + BM, p.S_q), k_lo, k_hi);
                const unsigned int turn = (unsigned int)(n_tile - k_lo / BN);
                unsigned int* sem = p.dq_sem + (size_t)bh * m_tiles + m0 / BM;
                const bool go = wait_counter(sem, turn, abort_flag, p.err);
                ptx::fence_proxy_async_global();  // the earlier turns' adds before ours
                reduce_staged(s, dt(it), bh, m0, go);
                if (prev_sem != nullptr) {
                    // the previous tile's groups are complete once at most this tile's are pending
                    ptx::bulk_wait_pending<D / 64>();
                    ptx::fence_proxy_async_global();  // its adds before the next turn's
                    ptx::st_release_gpu(prev_sem, prev_turn + 1);
                }
                prev_sem = go ? sem : nullptr;
                prev_turn = turn;
            }
            ptx::bulk_wait_all();
            if (prev_sem != nullptr) {
                ptx::fence_proxy_async_global();
                ptx::st_release_gpu(prev_sem, prev_turn + 1);
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (kSplit > 1) {
        // Rank 1 parks its fp32 dK / dV partial sums in its shared memory (over the Q / dO / dS
        // tiles, rows padded by four words): only after the barrier above, which the drain's
        // issuing thread reaches once its bulk reduce-adds (which read the dS and dO tiles)
        // are complete.  Rank 0 adds them after the cluster barrier.
        if (rank == 1 && warp >= kWarpSoft0 && warp < kWarpSoft0 + kNumSoftWarps && !*abort_flag) {
            const int qd = warp & 3, hf = (warp - kWarpSoft0) >> 2;
            const int t = qd * 32 + lane;
            const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
            ptx::tc_fence_after();
            float* park = reinterpret_cast<float*>(smem + C::OFF_Q);  // dV part, then dK part
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                const int c = hf * (D / 64) + cc;  // 32-column chunk
                uint32_t rv[32], rk[32];
                if (n_it > 0) {
                    ptx::tmem_ld32p(tmem + C::TM_DV + lane_off + c * 32, rv);
                    ptx::tmem_ld32p(tmem + C::TM_DK + lane_off + c * 32, rk);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) rv[k] = rk[k] = 0u;
                }
#pragma unroll
                for (int k = 0; k < 32; k += 4) {
                    *reinterpret_cast<uint4*>(park + t * (D + 4) + c * 32 + k) =
                        make_uint4(rv[k], rv[k + 1], rv[k + 2], rv[k + 3]);
                    *reinterpret_cast<uint4*>(park + BN * (D + 4) + t * (D + 4) + c * 32 + k) =
                        make_uint4(rk[k], rk[k + 1], rk[k + 2], rk[k + 3]);
                }
            }
        }
        // every thread of both CTAs: rank 1's partial sums are in its shared memory
        ptx::cluster_sync();
        if (rank == 0 && warp >= kWarpSoft0 && warp < kWarpSoft0 + kNumSoftWarps && !*abort_flag) {
            const int qd = warp & 3, hf = (warp - kWarpSoft0) >> 2;
            const int t = qd * 32 + lane;
            const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
            const int j = n0 + t;
            const uint32_t park = ptx::mapa_shared(sbase + C::OFF_Q, 1);
            T* dVrow = static_cast<T*>(p.dV) + ((size_t)bkv * p.S_k + j) * p.d;
            T* dKrow = static_cast<T*>(p.dK) + ((size_t)bkv * p.S_k + j) * p.d;
#pragma unroll 1
            for (int cc = 0; cc < D / 64; ++cc) {
                const int c = hf * (D / 64) + cc;
                uint32_t rv[32], rk[32];
                if (n_it > 0) {
                    ptx::tmem_ld32p(tmem + C::TM_DV + lane_off + c * 32, rv);
                    ptx::tmem_ld32p(tmem + C::TM_DK + lane_off + c * 32, rk);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) rv[k] = rk[k] = 0u;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint32_t ov[4], ok4[4];
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const uint32_t o = (uint32_t)((t * (D + 4) + c * 32 + u * 8 + 4 * h2) * 4);
                        const float4 pv = ptx::ld_shared_cluster_v4(park + o);
                        const float4 pk = ptx::ld_shared_cluster_v4(park + BN * (D + 4) * 4 + o);
                        const int e = u * 8 + 4 * h2;
                        ov[2 * h2] = pack2<kBF16>(__uint_as_float(rv[e]) + pv.x, __uint_as_float(rv[e + 1]) + pv.y);
                        ov[2 * h2 + 1] = pack2<kBF16>(__uint_as_float(rv[e + 2]) + pv.z, __uint_as_float(rv[e + 3]) + pv.w);
                        ok4[2 * h2] = pack2<kBF16>((__uint_as_float(rk[e]) + pk.x) * p.scale,
                                                   (__uint_as_float(rk[e + 1]) + pk.y) * p.scale);
                        ok4[2 * h2 + 1] = pack2<kBF16>((__uint_as_float(rk[e + 2]) + pk.z) * p.scale,
                                                       (__uint_as_float(rk[e + 3]) + pk.w) * p.scale);
                    }
                    if (j < p.S_k && c * 32 + u * 8 < p.d) {
                        *reinterpret_cast<uint4*>(dVrow + c * 32 + u * 8) = make_uint4(ov[0], ov[1], ov[2], ov[3]);
                        *reinterpret_cast<uint4*>(dKrow + c * 32 + u * 8) = make_uint4(ok4[0], ok4[1], ok4[2], ok4[3]);
                    }
                }
            }
        }
        ptx::tc_fence_before();
        ptx::cluster_sync();  // rank 0 has read rank 1's shared memory: both may exit
        ptx::tc_fence_after();
    }
    if (warp == kWarpMma) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// 3-D view [heads][rows][D] of a [B, heads, rows, D] tensor with a 128-byte-wide,
// 128-row box (64 16-bit or 32 fp32 columns) and 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, int heads, int rows,
              int D) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)heads};
    const cuuint64_t strides[2] = {(cuuint64_t)D * esize, (cuuint64_t)rows * D * esize};
    const cuuint32_t box[3] = {(cuuint32_t)(128 / esize), 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int D>
cudaError_t launch_t(const void* Q, const void* K, const void* V, const void* dO,
                     const Workspace& ws, void* dK, void* dV, const Shape& s, cudaStream_t st) {
    using C = Cfg<D>;
    static_assert(C::SMEM <= 232448, "shared memory budget");
    CUtensorMap tq, tk, tv, tdo, tdq;
    const CUtensorMapDataType dt =
        TypeTraits<T>::kId == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // global extents and strides use the tensors' head dim s.d; the kernel reads D columns
    // (boxes past s.d come back zero-filled)
    if (s.d > D || s.d % 32 != 0 || !make_map(&tq, Q, dt, 2, s.B * s.H, s.S_q, s.d) ||
        !make_map(&tk, K, dt, 2, s.B * s.H_kv, s.S_k, s.d) || !make_map(&tv, V, dt, 2, s.B * s.H_kv, s.S_k, s.d) ||
        !make_map(&tdo, dO, dt, 2, s.B * s.H, s.S_q, s.d) ||
        !make_map(&tdq, ws.dqacc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, s.B * s.H, s.S_q, s.d))
        return cudaErrorInvalidValue;
    Params p;
    p.lse2 = ws.lse2;
    p.Dws = ws.Dws;
    p.dK = dK;
    p.dV = dV;
    p.err = ws.err;
    p.dq_sem = ws.dq_sem;
    p.ticket = ws.dq_ticket;
    p.B = s.B;
    p.H = s.H;
    p.H_kv = s.H_kv;
    p.S_q = s.S_q;
    p.S_k = s.S_k;
    p.S_q_pad = s.S_q_pad;
    p.d = s.d;
    p.scale = s.scale;
    p.scale_log2 = s.scale * 1.4426950408889634f;
    p.causal = s.causal;
    p.window = s.window;
    // blocks of 4 groups when the key tiles carry about equal work (measured 1-4 % faster on
    // non-causal and windowed shapes: L2 locality of the dQ reduce-adds and Q / dO reads);
    // causal keeps one block so the heaviest key tiles start first (4-group blocks left the
    // heaviest tiles of the last block running alone at the end: 18 % slower)
    // (and deterministic calls keep one block: with a group's key-tile CTAs side by side
    // each waits for its predecessor's turn on every tile, 1706 -> 2154 us on fp16 S=8192)
    const int groups = s.B * s.H_kv;
    p.group_chunk = groups;
    if ((!s.causal || s.window > 0) && ws.dq_sem == nullptr)
        p.group_chunk = groups % 4 == 0 ? 4 : (groups % 2 == 0 ? 2 : groups);
    // a cluster of two CTAs per key tile for small grids and long causal key tiles (the
    // deterministic mode takes its CTA indices from a start-order ticket, which cannot pair
    // cluster ranks: one CTA per key tile there)
    const int split = ws.dq_sem != nullptr ? 1 : key_tile_split(s, BN, BM);
    auto kern = ws.dq_sem != nullptr ? bwd_sm103_kernel<T, D, true, 1>
                                     : (split == 2 ? bwd_sm103_kernel<T, D, false, 2> : bwd_sm103_kernel<T, D, false, 1>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    const long grid = (long)((s.S_k + BN - 1) / BN) * s.B * s.H_kv * split;
    const int threads = threads_for(ws.dq_sem != nullptr, D);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (split > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)split;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (ws.dq_sem == nullptr) {
        // programmatic dependent launch: the set-up (barriers, TMEM, K / V loads) overlaps the
        // end of the preprocess pass; the roles that read what it wrote wait for it
        // (deterministic calls keep the full dependency: their turn counters and ticket are
        // reset by a memset ahead of the preprocess pass)
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = (unsigned)na;
    return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tdo, tdq, p);
}

}  // namespace

cudaError_t launch_bwd_sm103(int dtype, const void* Q, const void* K, const void* V,
                             const void* dO, const Workspace& ws, void* dK, void* dV,
                             const Shape& s, cudaStream_t st) {
    const int D = tc_head_dim(s.d);  // d = 32 / 96 run the 64 / 128 kernels
    if (D == 64) {
        if (dtype == FA_F16) return launch_t<__half, 64>(Q, K, V, dO, ws, dK, dV, s, st);
        if (dtype == FA_BF16) return launch_t<__nv_bfloat16, 64>(Q, K, V, dO, ws, dK, dV, s, st);
    } else if (D == 128) {
        if (dtype == FA_F16) return launch_t<__half, 128>(Q, K, V, dO, ws, dK, dV, s, st);
        if (dtype == FA_BF16) return launch_t<__nv_bfloat16, 128>(Q, K, V, dO, ws, dK, dV, s, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace fa
