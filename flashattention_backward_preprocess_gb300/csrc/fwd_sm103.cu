// fwd_sm103.cu -- attention forward for GB300 (sm_103a), f16 / bf16, head dim 64,
// 128 or 256 (32 and 96 run the 64 / 128 kernels with zero-filled columns): the O
// and LSE the backward consumes (boostr autograd_attention.rs: the
// forward saves q, k, v, output and lse for FlashAttentionBackward).
//
//   s_ij = scale <Q_i, K_j> over the visible keys j (key_visible: causal keeps
//          j <= i + S_k - S_q, a sliding window a band around that position)
//   O_i  = sum_j exp(s_ij) V_j / sum_j exp(s_ij),   LSE_i = log sum_j exp(s_ij)
// computed with the online softmax over 128-key tiles (64-key at d = 256); a row that sees no key
// gets O = 0 and LSE = -inf.
//
// Design:
//   * the (128-row query tile, query head) items are walked the query tiles with the most
//     visible key tiles first, by a persistent grid (one CTA per SM) for causal and windowed
//     calls at d <= 128, where the next item's Q load and S products overlap the current
//     item's epilogue, and one CTA per item otherwise;
//   * S = Q K^T for key tile j runs on the 5th-generation tensor cores into one of
//     three 128-column TMEM buffers (two at d = 256, whose O takes columns
//     [256, 512)), so S(j+1) and S(j+2) are computed while the softmax warps work
//     on S(j); P = exp2(x - m) is packed to 16 bits in place and
//     is the TMEM A operand of O += P V (O accumulates in TMEM, fp32);
//   * one softmax thread per query row (TMEM lane), logits handled in log2 units
//     x = s * log2(e).  The running max m moves only when a tile's max exceeds it
//     by more than 8 (P then stays <= 2^8); only then is the O row rescaled in
//     TMEM, after the previous P V product has finished;
//   * TMA (128-byte swizzle) loads the Q tile once and K / V through a ring;
//     the epilogue divides O by the row sum and writes O and LSE;
//   * warp roles: warps 0-3 softmax and epilogue, warp 4 TMA, warp 5 TMEM owner and
//     issuer of the S products, warp 6 issuer of the P V products; every mbarrier wait
//     is bounded (a timeout records an error word, the other roles drop out, TMEM is
//     freed and the kernel returns).
#include <math.h>

#include "bounded_wait.cuh"
#include "fa_internal.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int BM = 128;  // query rows per CTA
constexpr int kThreads = 224;
constexpr int kWarpTma = 4, kWarpMma = 5, kWarpPv = 6;  // MMA issuers: S products (5), P V products (6)
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;  // move the running max only past this margin

template <int D>
struct FCfg {
    // key rows per step: 128, or 64 at d = 256 so that Q, two K / V stages and the 256-column O
    // accumulator fit shared memory and TMEM
    static constexpr int BN = D <= 128 ? 128 : 64;
    static constexpr int STAGES = D == 64 ? 4 : (D == 128 ? 3 : 2);
    static constexpr int NBUF = D <= 128 ? 3 : 2;          // S buffers in TMEM, 128 columns apart
    static constexpr int BOXES = D / 64;                    // 64-column boxes per tile row
    static constexpr uint32_t kTileQ_B = BM * D * 2;        // Q tile
    static constexpr uint32_t kTileKV_B = BN * D * 2;       // K or V tile
    static constexpr uint32_t kBoxQ_B = BM * 128;           // one 64-column box of the Q tile
    static constexpr uint32_t kBoxKV_B = BN * 128;          // one 64-column box of a K / V tile
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + kTileQ_B;
    static constexpr uint32_t OFF_V = OFF_K + STAGES * kTileKV_B;
    static constexpr uint32_t OFF_BAR = OFF_V + STAGES * kTileKV_B;
    // S buffer b at column 128 b (BN columns used); O after them: [384, 384+D) or [256, 512)
    static constexpr uint32_t TM_S = 0, TM_O = 128 * NBUF;
    static_assert(TM_O + D <= 512, "TMEM columns");
};

enum {
    F_Q = 0,      // Q tile landed (TMA)
    F_S0,             // S(j) in buffer j % NBUF (MMA commit), one slot per buffer (up to 3)
    F_P0 = F_S0 + 3,  // P(j) packed in buffer j % NBUF (4 softmax warps), one slot per buffer
    F_PV0 = F_P0 + 3, // O += P(j) V(j) done (MMA commit), one slot per buffer
    F_FINAL = F_PV0 + 3,  // every product done (P V issuer's last commit)
    F_QE,         // the Q tile may be reloaded: the S products of an item completed (MMA commit)
    F_OFULL,      // O of an item complete (P V issuer's commit after the item's last product)
    F_OFREE,      // O of an item read by the epilogue (4 softmax warps)
    F_STAGE0      // then STAGES "full" barriers, then STAGES "empty" barriers
};

struct FParams {
    void* O;
    float* LSE;
    unsigned int* err;
    int B, H, H_kv, S_q, S_k;
    int d;  // head dim of the tensors (<= D: columns d..D-1 are zero-filled by TMA, never stored)
    float scale_log2;
    int window;  // sliding-window size, 0 = none
};

// max(a, b, c) in one instruction (three-input max.f32, sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if (kBF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// One CTA per item (non-causal calls, d = 256, grids that fit one wave).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_sm103_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const FParams p, int causal) {
    using C = FCfg<D>;
    constexpr int BN = C::BN, NB = C::NBUF;
    constexpr bool kBF16 = TypeTraits<T>::kId == FA_BF16;
    constexpr int kNumBars = F_STAGE0 + 2 * C::STAGES;
    constexpr uint32_t OFF_MISC = C::OFF_BAR + kNumBars * 8;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 4);
    auto bar = [&](int i) { return sbase + C::OFF_BAR + 8u * (uint32_t)i; };
    auto bar_full = [&](int s) { return bar(F_STAGE0 + s); };
    auto bar_empty = [&](int s) { return bar(F_STAGE0 + C::STAGES + s); };

    // ---- work: the query tiles that see the most key tiles first, heads innermost
    const int BH = p.B * p.H;
    const int m_tiles = (p.S_q + BM - 1) / BM;
    const int n_tiles = (p.S_k + BN - 1) / BN;
    const int mt = m_tiles - 1 - (int)(blockIdx.x / BH);
    const int bh = (int)(blockIdx.x % BH);
    const int b = bh / p.H, h = bh % p.H;
    const int bkv = b * p.H_kv + h / (p.H / p.H_kv);
    const int m0 = mt * BM;
    const int off = p.S_k - p.S_q;  // query i sits at key position i + off
    // key tiles [n_first, n_first + n_cnt) hold every key a row of this tile sees
    int n_first = 0, n_cnt = 0;
    {
        Shape sh;
        sh.S_q = p.S_q;
        sh.S_k = p.S_k;
        sh.causal = causal;
        sh.window = p.window;
        int k_lo, k_hi;
        key_range(sh, m0, min(m0 + BM, p.S_q), k_lo, k_hi);
        if (k_hi > k_lo) {
            n_first = k_lo / BN;
            n_cnt = min((k_hi + BN - 1) / BN, n_tiles) - n_first;
        }
    }

    if (threadIdx.x == 0) {
        if ((sbase & 1023u) != 0) atomicOr(p.err, kErrSmemAlign);
        *abort_flag = (sbase & 1023u) != 0;
        for (int i = 0; i < kNumBars; ++i) ptx::mbar_init(bar(i), (i >= F_P0 && i < F_P0 + 3) ? 4u : 1u);
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == kWarpMma) {
        ptx::tmem_alloc(sbase + OFF_MISC + 4, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && !*abort_flag && n_cnt > 0) {
            ptx::mbar_arrive_expect_tx(bar(F_Q), C::kTileQ_B);
            for (int x = 0; x < C::BOXES; ++x)
                ptx::tma_load_3d(sbase + C::OFF_Q + x * C::kBoxQ_B, &tmQ, x * 64, m0, bh, bar(F_Q));
            int issued = 0;
            for (int j = 0; j < n_cnt; ++j) {
                const int s = j % C::STAGES;
                if (j >= C::STAGES && !wait_bar(bar_empty(s), ((j / C::STAGES) - 1) & 1, abort_flag, p.err)) break;
                ptx::mbar_arrive_expect_tx(bar_full(s), 2 * C::kTileKV_B);
                for (int x = 0; x < C::BOXES; ++x) {
                    ptx::tma_load_3d(sbase + C::OFF_K + s * C::kTileKV_B + x * C::kBoxKV_B, &tmK, x * 64,
                                     (n_first + j) * BN, bkv,
                                     bar_full(s));
                    ptx::tma_load_3d(sbase + C::OFF_V + s * C::kTileKV_B + x * C::kBoxKV_B, &tmV, x * 64,
                                     (n_first + j) * BN, bkv,
                                     bar_full(s));
                }
                issued = j + 1;
            }
            // never leave copies in flight into shared memory that is about to be released
            drain_wait(bar(F_Q), 0);
            for (int j = issued - C::STAGES < 0 ? 0 : issued - C::STAGES; j < issued; ++j)
                drain_wait(bar_full(j % C::STAGES), (j / C::STAGES) & 1);
        }
    } else if (warp == kWarpMma || warp == kWarpPv) {
        // ------------------------------------------------------------ MMA issuers
        // tcgen05.mma issue stalls while the tensor pipe's short queue is full, so one thread
        // can run only about one product ahead of the pipe and every commit, barrier wait and
        // fence it executes leaves the pipe idle.  Two issuers hide each other's bookkeeping:
        // warp 5 issues S = Q K^T, warp 6 issues O += P V.  Products of different threads are
        // not ordered with each other, so every hazard between them goes through a barrier:
        // S(j) into buffer j % NBUF waits until P V(j-NBUF) has read P out of it (one P V barrier per
        // buffer, so that wait can never see a phase two ahead), and P V(j) runs only once the
        // softmax has turned S(j) into P(j), which implies S(j) is complete.  Three S buffers
        // (d <= 128) let S(j+2) run while the softmax still works on S(j) and S(j+1).
        if (lane == 0 && !*abort_flag && n_cnt > 0) {
            constexpr uint32_t ID_S = ptx::idesc_f16(BM, BN, kBF16, false, false);  // S = Q K^T
            constexpr uint32_t ID_PV = ptx::idesc_f16(BM, D, kBF16, false, true);   // O += P V (A in TMEM)
            auto desc_add = [](uint64_t d, uint32_t bytes) { return d + (bytes >> 4); };
            bool ok = true;
            if (warp == kWarpMma) {
                const uint64_t dQ_k = ptx::sw128_desc(sbase + C::OFF_Q, 16, 1024);
                const uint64_t dK_k = ptx::sw128_desc(sbase + C::OFF_K, 16, 1024);  // + stage offset
                ok = wait_bar(bar(F_Q), 0, abort_flag, p.err);
                for (int j = 0; ok && j < n_cnt; ++j) {
                    const int s = j % C::STAGES;
                    if (!(ok = wait_bar(bar_full(s), (j / C::STAGES) & 1, abort_flag, p.err))) break;
                    if (j >= NB && !(ok = wait_bar(bar(F_PV0 + j % NB), (j / NB - 1) & 1, abort_flag, p.err))) break;
                    ptx::tc_fence_after();
                    const uint32_t so = (uint32_t)s * C::kTileKV_B;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t kq = (k / 4) * C::kBoxQ_B + (k % 4) * 32;
                        const uint32_t kk = (k / 4) * C::kBoxKV_B + (k % 4) * 32;
                        ptx::mma_ss(tmem + C::TM_S + (j % NB) * 128, desc_add(dQ_k, kq), desc_add(dK_k, so + kk),
                                    ID_S, k > 0);
                    }
                    ptx::mma_commit(bar(F_S0 + j % NB));
                }
                // this thread's products must be complete before TMEM is released; every S it
                // issued is read by a P V product, so they are, once the P V issuer drained
            } else {
                const uint64_t dV_mn = ptx::sw128_desc(sbase + C::OFF_V, C::kBoxKV_B, 1024);  // + stage offset
                for (int j = 0; ok && j < n_cnt; ++j) {
                    const int s = j % C::STAGES;
                    // O += P(j) V(j)   (A = P packed in buffer j % NBUF: 16 keys = 8 packed columns per step)
                    if (!(ok = wait_bar(bar(F_P0 + j % NB), (j / NB) & 1, abort_flag, p.err))) break;
                    ptx::tc_fence_after();
#pragma unroll
                    for (int k = 0; k < BN / 16; ++k)
                        ptx::mma_ts(tmem + C::TM_O, tmem + C::TM_S + (j % NB) * 128 + k * 8,
                                    desc_add(dV_mn, (uint32_t)s * C::kTileKV_B + k * 2048), ID_PV,
                                    (j > 0 || k > 0) ? 1u : 0u);
                    ptx::mma_commit(bar(F_PV0 + j % NB));
                    ptx::mma_commit(bar_empty(s));  // K(j), V(j) no longer read (S(j) completed before P(j))
                }
                // no MMA may still write TMEM when it is released
                ptx::mma_commit(bar(F_FINAL));
                drain_wait(bar(F_FINAL), 0);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int t = warp * 32 + lane;  // TMEM lane == query row within the tile
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const int i = m0 + t;
        const bool row_valid = i < p.S_q;
        float m_run = -INFINITY;  // running max of x = s * log2(e), moved lazily
        float l_run = 0.f;        // sum of exp2(x - m_run)
        bool ok = !*abort_flag;
        for (int j = 0; ok && j < n_cnt; ++j) {
            const uint32_t buf = tmem + C::TM_S + (j % NB) * 128 + lane_off;
            const int n0 = (n_first + j) * BN;
            // Key columns c of this tile (key n0 + c) that the row sees form one interval
            // (visible_keys of the row's key position i + off), cut to the keys that exist.
            int c_lo, c_hi;
            visible_keys(i + off - n0, causal, p.window, c_lo, c_hi);
            c_lo = max(c_lo, 0);
            c_hi = min(c_hi, p.S_k - n0);
            const unsigned c_span = c_hi > c_lo ? (unsigned)(c_hi - c_lo) : 0u;
            // warp-uniform: the chosen path holds .sync.aligned TMEM accesses
            const bool masked = __any_sync(0xffffffffu, !(c_lo <= 0 && c_hi >= BN));
            if (!(ok = wait_bar_warp(bar(F_S0 + j % NB), (j / NB) & 1, abort_flag, p.err))) break;
            ptx::tc_fence_after();
            uint32_t r[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) ptx::tmem_ld32p(buf + c * 32, r + c * 32);
            ptx::tmem_wait_ld();
            // masked scores become -inf in place; row max over eight independent chains of
            // three-input maxima (one instruction per two scores)
            if (masked) {
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    r[c] = (unsigned)(c - c_lo) < c_span ? r[c] : __float_as_uint(-INFINITY);
            }
            float mx8[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) mx8[q] = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN; c += 2)
                mx8[(c >> 1) & 7] = fmax3(mx8[(c >> 1) & 7], __uint_as_float(r[c]), __uint_as_float(r[c + 1]));
            float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            mx = mx == -INFINITY ? -INFINITY : mx * p.scale_log2;
            // lazy running max: move it only when this tile exceeds it by more than the margin
            float alpha = 1.f;
            const bool rescale = mx > m_run + kRescaleLog2;
            if (rescale) {
                alpha = m_run == -INFINITY ? 0.f : ptx::ex2(m_run - mx);
                m_run = mx;
            }
            const float m_use = m_run == -INFINITY ? 0.f : m_run;  // rows with nothing visible yet: P = 0
            // scale-and-shift and the row sum on packed fp32 pairs (one instruction per two
            // scores); -inf scores give P = 0
            const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
            const float2 nm2 = make_float2(-m_use, -m_use);
            float2 sum2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                              make_float2(0.f, 0.f)};
            uint32_t Pp[BN / 2];
#pragma unroll
            for (int c = 0; c < BN; c += 2) {
                const float2 x = __ffma2_rn(make_float2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), sc2, nm2);
                const float2 pp = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
                sum2[(c >> 1) & 3] = __fadd2_rn(sum2[(c >> 1) & 3], pp);
                Pp[c / 2] = pack2<kBF16>(pp.x, pp.y);
            }
            const float2 s2 = __fadd2_rn(__fadd2_rn(sum2[0], sum2[1]), __fadd2_rn(sum2[2], sum2[3]));
            const float sum = s2.x + s2.y;
            l_run = l_run * alpha + sum;
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)  // packed P into columns [0, BN/2): already read
                ptx::tmem_st32(buf + c * 32, Pp + c * 32);
            // rescale the O row before the next P V product accumulates into it
            if (j > 0 && __any_sync(0xffffffffu, rescale)) {
                if (!(ok = wait_bar_warp(bar(F_PV0 + (j - 1) % NB), ((j - 1) / NB) & 1, abort_flag, p.err))) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    ptx::tmem_ld32p(tmem + C::TM_O + lane_off + c * 32, o);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                    ptx::tmem_st32(tmem + C::TM_O + lane_off + c * 32, o);
                }
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(F_P0 + j % NB));
        }
        // ---- epilogue: O = acc / l, LSE = (m + log2 l) * ln 2.  Wait for the MMA issuer's
        // final commit (every product done), not for a parity of the shared P V barrier:
        // after the last tile that barrier may still be in the phase of the product before
        // last, whose parity is the opposite one, and a parity wait would pass at once.
        if (ok && n_cnt > 0) ok = wait_bar_warp(bar(F_FINAL), 0, abort_flag, p.err);
        if (ok) {
            ptx::tc_fence_after();
            const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
            T* Orow = static_cast<T*>(p.O) + ((size_t)bh * p.S_q + i) * p.d;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                if (n_cnt > 0) {
                    ptx::tmem_ld32p(tmem + C::TM_O + lane_off + c * 32, o);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = 0u;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint32_t w4[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        w4[k] = pack2<kBF16>(__uint_as_float(o[u * 8 + 2 * k]) * inv_l,
                                             __uint_as_float(o[u * 8 + 2 * k + 1]) * inv_l);
                    if (row_valid && c * 32 + u * 8 < p.d)
                        *reinterpret_cast<uint4*>(Orow + c * 32 + u * 8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
            }
            if (row_valid)
                p.LSE[(size_t)bh * p.S_q + i] = l_run > 0.f ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == kWarpMma) ptx::tmem_dealloc(tmem, kTmemCols);
}

// Persistent variant for causal and windowed calls at d <= 128: one CTA per SM walks its
// share of the items, and the next item's loads and S products overlap this item's
// epilogue.  The per-tile work is the same as in fwd_sm103_kernel; the two are kept
// separate because the cross-item bookkeeping (item loop, polling producer, per-item
// barriers) measured 2-4 % slower on the shapes the one-item kernel serves.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_sm103_persistent_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const FParams p, int causal) {
    using C = FCfg<D>;
    constexpr int BN = C::BN, NB = C::NBUF;
    constexpr bool kBF16 = TypeTraits<T>::kId == FA_BF16;
    constexpr int kNumBars = F_STAGE0 + 2 * C::STAGES;
    constexpr uint32_t OFF_MISC = C::OFF_BAR + kNumBars * 8;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 4);
    auto bar = [&](int i) { return sbase + C::OFF_BAR + 8u * (uint32_t)i; };
    auto bar_full = [&](int s) { return bar(F_STAGE0 + s); };
    auto bar_empty = [&](int s) { return bar(F_STAGE0 + C::STAGES + s); };

    // ---- work items: (query tile, query head), the query tiles that see the most key tiles
    // first, heads innermost.  The grid is persistent (at most one CTA per SM); CTA c takes the
    // items of round r in snake order (c, then G-1-c, ...), which evens out the rounds'
    // decreasing weights.  Every role walks the same item sequence and skips the items whose
    // rows see no key in the same way, so the per-item barrier phases (counted over the items
    // with work) and the per-tile ones (counted over all key tiles of this CTA) agree.
    const int BH = p.B * p.H;
    const int m_tiles = (p.S_q + BM - 1) / BM;
    const int n_tiles = (p.S_k + BN - 1) / BN;
    const int n_items = m_tiles * BH;
    const int G = (int)gridDim.x;
    const int off = p.S_k - p.S_q;  // query i sits at key position i + off
    struct Item {
        int bh, bkv, m0, n_first, n_cnt;
    };
    auto item = [&](int k, Item& it) -> bool {  // this CTA's k-th item; false past the end
        const int r = k, c = (int)blockIdx.x;
        const int w = r * G + ((r & 1) ? G - 1 - c : c);
        if (w >= n_items) return false;
        const int mt = m_tiles - 1 - w / BH;
        it.bh = w % BH;
        const int b = it.bh / p.H, h = it.bh % p.H;
        it.bkv = b * p.H_kv + h / (p.H / p.H_kv);
        it.m0 = mt * BM;
        // key tiles [n_first, n_first + n_cnt) hold every key a row of this tile sees
        it.n_first = 0;
        it.n_cnt = 0;
        Shape sh;
        sh.S_q = p.S_q;
        sh.S_k = p.S_k;
        sh.causal = causal;
        sh.window = p.window;
        int k_lo, k_hi;
        key_range(sh, it.m0, min(it.m0 + BM, p.S_q), k_lo, k_hi);
        if (k_hi > k_lo) {
            it.n_first = k_lo / BN;
            it.n_cnt = min((k_hi + BN - 1) / BN, n_tiles) - it.n_first;
        }
        return true;
    };
    // rounds with a full item for this CTA (the last round may leave it without one)
    const int n_rounds = (n_items + G - 1) / G;

    if (threadIdx.x == 0) {
        if ((sbase & 1023u) != 0) atomicOr(p.err, kErrSmemAlign);
        *abort_flag = (sbase & 1023u) != 0;
        for (int i = 0; i < kNumBars; ++i)
            ptx::mbar_init(bar(i), ((i >= F_P0 && i < F_P0 + 3) || i == F_OFREE) ? 4u : 1u);
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == kWarpMma) {
        ptx::tmem_alloc(sbase + OFF_MISC + 4, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ producer
        // One thread, two streams walking the same item sequence: the Q tile of each item with
        // work (once every S product of the previous one completed) and the K / V tiles of the
        // ring (each as soon as its slot is free), polling both without blocking on either, so
        // the next item's first K / V tiles load while this item's last S products still run.
        if (lane == 0 && !*abort_flag) {
            int q_k = 0, q_act = 0;             // Q stream: next item, Q tiles loaded
            int kv_k = 0, kv_j = 0, jg = 0;     // K / V stream: item, tile within it, tiles loaded
            Item q_it, kv_it;
            bool q_more = true, kv_more = true;
            auto next_active = [&](int& k, Item& it) -> bool {  // first item with work from k on
                for (; k < n_rounds; ++k)
                    if (!item(k, it)) return false;
                    else if (it.n_cnt > 0) return true;
                return false;
            };
            q_more = next_active(q_k, q_it);
            kv_more = next_active(kv_k, kv_it);
            uint64_t t0 = ptx::globaltimer();
            uint32_t spins = 0;
            while (q_more || kv_more) {
                bool progress = false;
                if (q_more && (q_act == 0 || ptx::mbar_test_wait(bar(F_QE), (q_act - 1) & 1))) {
                    ptx::mbar_arrive_expect_tx(bar(F_Q), C::kTileQ_B);
                    for (int x = 0; x < C::BOXES; ++x)
                        ptx::tma_load_3d(sbase + C::OFF_Q + x * C::kBoxQ_B, &tmQ, x * 64, q_it.m0, q_it.bh, bar(F_Q));
                    ++q_act;
                    ++q_k;
                    q_more = next_active(q_k, q_it);
                    progress = true;
                }
                if (kv_more &&
                    (jg < C::STAGES || ptx::mbar_test_wait(bar_empty(jg % C::STAGES), ((jg / C::STAGES) - 1) & 1))) {
                    const int s = jg % C::STAGES;
                    ptx::mbar_arrive_expect_tx(bar_full(s), 2 * C::kTileKV_B);
                    for (int x = 0; x < C::BOXES; ++x) {
                        ptx::tma_load_3d(sbase + C::OFF_K + s * C::kTileKV_B + x * C::kBoxKV_B, &tmK, x * 64,
                                         (kv_it.n_first + kv_j) * BN, kv_it.bkv, bar_full(s));
                        ptx::tma_load_3d(sbase + C::OFF_V + s * C::kTileKV_B + x * C::kBoxKV_B, &tmV, x * 64,
                                         (kv_it.n_first + kv_j) * BN, kv_it.bkv, bar_full(s));
                    }
                    ++jg;
                    if (++kv_j == kv_it.n_cnt) {
                        kv_j = 0;
                        ++kv_k;
                        kv_more = next_active(kv_k, kv_it);
                    }
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
            // never leave copies in flight into shared memory that is about to be released: the
            // last Q load and the last STAGES K / V loads issued
            if (q_act > 0) drain_wait(bar(F_Q), (q_act - 1) & 1);
            for (int j = jg - C::STAGES < 0 ? 0 : jg - C::STAGES; j < jg; ++j)
                drain_wait(bar_full(j % C::STAGES), (j / C::STAGES) & 1);
        }
    } else if (warp == kWarpMma || warp == kWarpPv) {
        // ------------------------------------------------------------ MMA issuers
        // tcgen05.mma issue stalls while the tensor pipe's short queue is full, so one thread
        // can run only about one product ahead of the pipe and every commit, barrier wait and
        // fence it executes leaves the pipe idle.  Two issuers hide each other's bookkeeping:
        // warp 5 issues S = Q K^T, warp 6 issues O += P V.  Products of different threads are
        // not ordered with each other, so every hazard between them goes through a barrier:
        // S(j) into buffer j % NBUF waits until P V(j-NBUF) has read P out of it (one P V barrier per
        // buffer, so that wait can never see a phase two ahead), and P V(j) runs only once the
        // softmax has turned S(j) into P(j), which implies S(j) is complete.  Three S buffers
        // (d <= 128) let S(j+2) run while the softmax still works on S(j) and S(j+1).  Across
        // items: the S products of the next item start while the softmax warps run this item's
        // epilogue; its first P V product (which overwrites O) waits until they have read O.
        if (lane == 0 && !*abort_flag) {
            constexpr uint32_t ID_S = ptx::idesc_f16(BM, BN, kBF16, false, false);  // S = Q K^T
            constexpr uint32_t ID_PV = ptx::idesc_f16(BM, D, kBF16, false, true);   // O += P V (A in TMEM)
            auto desc_add = [](uint64_t d, uint32_t bytes) { return d + (bytes >> 4); };
            bool ok = true;
            int jg = 0, ka = 0;
            if (warp == kWarpMma) {
                const uint64_t dQ_k = ptx::sw128_desc(sbase + C::OFF_Q, 16, 1024);
                const uint64_t dK_k = ptx::sw128_desc(sbase + C::OFF_K, 16, 1024);  // + stage offset
                for (int k = 0; ok && k < n_rounds; ++k) {
                    Item it;
                    if (!item(k, it)) break;
                    if (it.n_cnt == 0) continue;
                    if (!(ok = wait_bar(bar(F_Q), ka & 1, abort_flag, p.err))) break;
                    for (int j = 0; j < it.n_cnt; ++j, ++jg) {
                        const int s = jg % C::STAGES;
                        if (!(ok = wait_bar(bar_full(s), (jg / C::STAGES) & 1, abort_flag, p.err))) break;
                        if (jg >= NB && !(ok = wait_bar(bar(F_PV0 + jg % NB), (jg / NB - 1) & 1, abort_flag, p.err)))
                            break;
                        ptx::tc_fence_after();
                        const uint32_t so = (uint32_t)s * C::kTileKV_B;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t kq = (kk / 4) * C::kBoxQ_B + (kk % 4) * 32;
                            const uint32_t kv = (kk / 4) * C::kBoxKV_B + (kk % 4) * 32;
                            ptx::mma_ss(tmem + C::TM_S + (jg % NB) * 128, desc_add(dQ_k, kq), desc_add(dK_k, so + kv),
                                        ID_S, kk > 0);
                        }
                        ptx::mma_commit(bar(F_S0 + jg % NB));
                    }
                    if (!ok) break;
                    ptx::mma_commit(bar(F_QE));  // the Q tile is free once these S products completed
                    ++ka;
                }
                // this thread's products must be complete before TMEM is released; every S it
                // issued is read by a P V product, so they are, once the P V issuer drained
            } else {
                const uint64_t dV_mn = ptx::sw128_desc(sbase + C::OFF_V, C::kBoxKV_B, 1024);  // + stage offset
                for (int k = 0; ok && k < n_rounds; ++k) {
                    Item it;
                    if (!item(k, it)) break;
                    if (it.n_cnt == 0) continue;
                    for (int j = 0; j < it.n_cnt; ++j, ++jg) {
                        const int s = jg % C::STAGES;
                        // O += P(j) V(j)   (A = P packed in buffer j % NBUF: 16 keys = 8 packed columns per step)
                        if (!(ok = wait_bar(bar(F_P0 + jg % NB), (jg / NB) & 1, abort_flag, p.err))) break;
                        // the first product of an item overwrites O: the epilogue of the previous
                        // item must have read it
                        if (j == 0 && ka > 0 && !(ok = wait_bar(bar(F_OFREE), (ka - 1) & 1, abort_flag, p.err)))
                            break;
                        ptx::tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk)
                            ptx::mma_ts(tmem + C::TM_O, tmem + C::TM_S + (jg % NB) * 128 + kk * 8,
                                        desc_add(dV_mn, (uint32_t)s * C::kTileKV_B + kk * 2048), ID_PV,
                                        (j > 0 || kk > 0) ? 1u : 0u);
                        ptx::mma_commit(bar(F_PV0 + jg % NB));
                        ptx::mma_commit(bar_empty(s));  // K(j), V(j) no longer read (S(j) completed before P(j))
                    }
                    if (!ok) break;
                    ptx::mma_commit(bar(F_OFULL));  // O of this item complete
                    ++ka;
                }
                // no MMA may still write TMEM when it is released
                ptx::mma_commit(bar(F_FINAL));
                drain_wait(bar(F_FINAL), 0);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int t = warp * 32 + lane;  // TMEM lane == query row within the tile
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        bool ok = !*abort_flag;
        int jg = 0, ka = 0;
        for (int k = 0; ok && k < n_rounds; ++k) {
            Item it;
            if (!item(k, it)) break;
            const int i = it.m0 + t;
            const bool row_valid = i < p.S_q;
            float m_run = -INFINITY;  // running max of x = s * log2(e), moved lazily
            float l_run = 0.f;        // sum of exp2(x - m_run)
            for (int j = 0; ok && j < it.n_cnt; ++j, ++jg) {
                const uint32_t buf = tmem + C::TM_S + (jg % NB) * 128 + lane_off;
                const int n0 = (it.n_first + j) * BN;
                // Key columns c of this tile (key n0 + c) that the row sees form one interval
                // (visible_keys of the row's key position i + off), cut to the keys that exist.
                int c_lo, c_hi;
                visible_keys(i + off - n0, causal, p.window, c_lo, c_hi);
                c_lo = max(c_lo, 0);
                c_hi = min(c_hi, p.S_k - n0);
                const unsigned c_span = c_hi > c_lo ? (unsigned)(c_hi - c_lo) : 0u;
                // warp-uniform: the chosen path holds .sync.aligned TMEM accesses
                const bool masked = __any_sync(0xffffffffu, !(c_lo <= 0 && c_hi >= BN));
                if (!(ok = wait_bar_warp(bar(F_S0 + jg % NB), (jg / NB) & 1, abort_flag, p.err))) break;
                ptx::tc_fence_after();
                uint32_t r[BN];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) ptx::tmem_ld32p(buf + c * 32, r + c * 32);
                ptx::tmem_wait_ld();
                // masked scores become -inf in place; row max over eight independent chains of
                // three-input maxima (one instruction per two scores)
                if (masked) {
#pragma unroll
                    for (int c = 0; c < BN; ++c)
                        r[c] = (unsigned)(c - c_lo) < c_span ? r[c] : __float_as_uint(-INFINITY);
                }
                float mx8[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) mx8[q] = -INFINITY;
#pragma unroll
                for (int c = 0; c < BN; c += 2)
                    mx8[(c >> 1) & 7] = fmax3(mx8[(c >> 1) & 7], __uint_as_float(r[c]), __uint_as_float(r[c + 1]));
                float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                 fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                mx = mx == -INFINITY ? -INFINITY : mx * p.scale_log2;
                // lazy running max: move it only when this tile exceeds it by more than the margin
                float alpha = 1.f;
                const bool rescale = mx > m_run + kRescaleLog2;
                if (rescale) {
                    alpha = m_run == -INFINITY ? 0.f : ptx::ex2(m_run - mx);
                    m_run = mx;
                }
                const float m_use = m_run == -INFINITY ? 0.f : m_run;  // rows with nothing visible yet: P = 0
                // scale-and-shift and the row sum on packed fp32 pairs (one instruction per two
                // scores); -inf scores give P = 0
                const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
                const float2 nm2 = make_float2(-m_use, -m_use);
                float2 sum2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                  make_float2(0.f, 0.f)};
                uint32_t Pp[BN / 2];
#pragma unroll
                for (int c = 0; c < BN; c += 2) {
                    const float2 x = __ffma2_rn(make_float2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), sc2, nm2);
                    const float2 pp = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
                    sum2[(c >> 1) & 3] = __fadd2_rn(sum2[(c >> 1) & 3], pp);
                    Pp[c / 2] = pack2<kBF16>(pp.x, pp.y);
                }
                const float2 s2 = __fadd2_rn(__fadd2_rn(sum2[0], sum2[1]), __fadd2_rn(sum2[2], sum2[3]));
                const float sum = s2.x + s2.y;
                l_run = l_run * alpha + sum;
#pragma unroll
                for (int c = 0; c < BN / 64; ++c)  // packed P into columns [0, BN/2): already read
                    ptx::tmem_st32(buf + c * 32, Pp + c * 32);
                // rescale the O row before the next P V product accumulates into it
                if (j > 0 && __any_sync(0xffffffffu, rescale)) {
                    if (!(ok = wait_bar_warp(bar(F_PV0 + (jg - 1) % NB), ((jg - 1) / NB) & 1, abort_flag, p.err)))
                        break;
                    ptx::tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        ptx::tmem_ld32p(tmem + C::TM_O + lane_off + c * 32, o);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int kk = 0; kk < 32; ++kk) o[kk] = __float_as_uint(__uint_as_float(o[kk]) * alpha);
                        ptx::tmem_st32(tmem + C::TM_O + lane_off + c * 32, o);
                    }
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(F_P0 + jg % NB));
            }
            if (!ok) break;
            // ---- epilogue: O = acc / l, LSE = (m + log2 l) * ln 2.  Wait for the P V issuer's
            // commit after this item's last product (every product of the item done), not for a
            // parity of a shared P V barrier, which may still be in the phase of an earlier product.
            const bool has = it.n_cnt > 0;
            if (has && !(ok = wait_bar_warp(bar(F_OFULL), ka & 1, abort_flag, p.err))) break;
            ptx::tc_fence_after();
            const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
            T* Orow = static_cast<T*>(p.O) + ((size_t)it.bh * p.S_q + i) * p.d;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                if (has) {
                    ptx::tmem_ld32p(tmem + C::TM_O + lane_off + c * 32, o);
                    ptx::tmem_wait_ld();
                    if (c == D / 32 - 1) {  // O read: the next item's first P V product may overwrite it
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(bar(F_OFREE));
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 32; ++kk) o[kk] = 0u;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint32_t w4[4];
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        w4[kk] = pack2<kBF16>(__uint_as_float(o[u * 8 + 2 * kk]) * inv_l,
                                              __uint_as_float(o[u * 8 + 2 * kk + 1]) * inv_l);
                    if (row_valid && c * 32 + u * 8 < p.d)
                        *reinterpret_cast<uint4*>(Orow + c * 32 + u * 8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
            }
            if (row_valid)
                p.LSE[(size_t)it.bh * p.S_q + i] =
                    l_run > 0.f ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
            if (has) ++ka;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
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

// 3-D view [heads][rows][D] of a [B, heads, rows, D] 16-bit tensor: 64-column x box_rows-row
// boxes with 128-byte swizzle (rows and columns past the end read as zeros).
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int heads, int rows, int D,
              int box_rows) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)heads};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)rows * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int D>
cudaError_t launch_t(const void* Q, const void* K, const void* V, void* O, float* LSE, unsigned int* err,
                     const Shape& s, cudaStream_t st) {
    using C = FCfg<D>;
    constexpr uint32_t kSmem = C::OFF_BAR + (F_STAGE0 + 2 * C::STAGES) * 8 + 16;
    static_assert(kSmem <= 232448, "shared memory budget");
    const CUtensorMapDataType dt =
        TypeTraits<T>::kId == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tq, tk, tv;
    // global extents and strides use the tensors' head dim s.d; the kernel reads D columns
    if (s.d > D || s.d % 32 != 0 || !make_map(&tq, Q, dt, s.B * s.H, s.S_q, s.d, BM) ||
        !make_map(&tk, K, dt, s.B * s.H_kv, s.S_k, s.d, C::BN) ||
        !make_map(&tv, V, dt, s.B * s.H_kv, s.S_k, s.d, C::BN))
        return cudaErrorInvalidValue;
    FParams p;
    p.O = O;
    p.LSE = LSE;
    p.err = err;
    p.B = s.B;
    p.H = s.H;
    p.H_kv = s.H_kv;
    p.S_q = s.S_q;
    p.S_k = s.S_k;
    p.d = s.d;
    p.scale_log2 = s.scale * 1.4426950408889634f;
    p.window = s.window;
    // Causal and windowed calls at d <= 128 run persistent (one CTA per SM, shared memory
    // allows no second), each CTA walking its share of the (query tile, head) items: their items
    // are short and uneven, and overlapping one item's epilogue with the next one's start took
    // the causal bf16 B=4 H=32 S=2048 shape from 177 to 154-159 us.  Other calls keep one CTA
    // per item in the one-item kernel: measured in one run, the persistent kernel was 3-4.5 %
    // slower there (non-causal S = 8192, causal d = 256).
    const long items = (long)((s.S_q + BM - 1) / BM) * s.B * s.H;
    long grid = items;
    bool persist = false;
    if (D <= 128 && (s.causal || s.window > 0)) {
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms > 0 && items > sms) {
            grid = sms;
            persist = true;
        }
    }
    if constexpr (D <= 128) {
        if (persist) {
            auto kern = fwd_sm103_persistent_kernel<T, D>;
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
            if (e != cudaSuccess) return e;
            kern<<<(unsigned)grid, kThreads, kSmem, st>>>(tq, tk, tv, p, s.causal);
            return cudaGetLastError();
        }
    }
    auto kern = fwd_sm103_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, kThreads, kSmem, st>>>(tq, tk, tv, p, s.causal);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_sm103(int dtype, const void* Q, const void* K, const void* V, void* O, float* LSE,
                            unsigned int* err, const Shape& s, cudaStream_t st) {
    // every head dim the library takes: d = 32 / 96 run the 64 / 128 kernels, d = 256 its own
    const int D = s.d == 256 ? 256 : tc_head_dim(s.d);
    if (D == 256) {
        if (dtype == FA_F16) return launch_t<__half, 256>(Q, K, V, O, LSE, err, s, st);
        if (dtype == FA_BF16) return launch_t<__nv_bfloat16, 256>(Q, K, V, O, LSE, err, s, st);
    } else if (D == 64) {
        if (dtype == FA_F16) return launch_t<__half, 64>(Q, K, V, O, LSE, err, s, st);
        if (dtype == FA_BF16) return launch_t<__nv_bfloat16, 64>(Q, K, V, O, LSE, err, s, st);
    } else if (D == 128) {
        if (dtype == FA_F16) return launch_t<__half, 128>(Q, K, V, O, LSE, err, s, st);
        if (dtype == FA_BF16) return launch_t<__nv_bfloat16, 128>(Q, K, V, O, LSE, err, s, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace fa
