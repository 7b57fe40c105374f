// bwd_sm103.cu -- FlashAttention-2 backward main kernel for GB300 (sm_103a),
// f16 / bf16 inputs, head dim 64 or 128.
//
// Math (the chain rule of O = softmax(scale Q K^T) V, with the saved LSE as
// the softmax normaliser and D from the preprocess step; boostr
// flash_bwd.rs, doc comment "Two-step process", step 2 "compute dQ
// (atomicAdd), dK, dV"):
//   S^T  = K Q^T            P^T  = exp2(S^T * scale*log2e - LSE*log2e)
//   dP^T = V dO^T           dS^T = P^T * (dP^T - D)
//   dV  += P^T dO           dK  += dS^T Q        dQacc += dS K  (fp32 atomics)
//
// Design (Blackwell-native, not the pages' one-thread-per-key-row design):
//   * one CTA owns a 128-row key/value tile of one (batch, kv head) and walks
//     every 128-row query tile of every query head of the group, so dK and dV
//     of the group are summed in tensor memory without atomics;
//   * the five per-tile products run on the 5th-generation tensor cores
//     (tcgen05.mma, M = 128, fp32 accumulation in TMEM).  S^T and dP^T are
//     computed "key-major" (TMEM lane = key row), so the softmax-gradient
//     threads own one key row each and write P^T / dS^T back into TMEM as the
//     A operand of the dV / dK products;
//   * TMA (cp.async.bulk.tensor, 128-byte swizzle) stages K, V once and Q, dO
//     in a multi-stage ring; causal tiles that no query can see are skipped;
//   * warp roles: warps 0-3 drain the dQ tile from TMEM and add it to the
//     fp32 accumulator in global memory (red.global.add.v4.f32), warps 4-7
//     compute P and dS and run the dK / dV epilogue, warp 8 issues TMA,
//     warp 9 owns TMEM and issues the MMAs;
//   * two 128-column TMEM buffers alternate roles each iteration: S(i) and
//     later dQ(i) live in one, dP(i) / dS(i) in the other, so the next S can
//     be computed while dQ(i) is drained.
//   * every mbarrier wait is bounded: on timeout the kernel records an error
//     word, lets the other roles drop out, waits for its own copies / MMAs in
//     flight, frees TMEM and returns.
//
// TMEM columns (512 allocated): dV [0, D), dK [D, 2D), buffer 0 [2D, 2D+128),
// buffer 1 [2D+128, 2D+256).
#include <math.h>

#include "fa_internal.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int BM = kTileQ;  // 128 query rows per iteration
constexpr int BN = kTileK;  // 128 key rows per CTA
constexpr int kThreads = 320;
constexpr int kWarpDrain0 = 0, kWarpSoft0 = 4, kWarpTma = 8, kWarpMma = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 10ull * 1000 * 1000 * 1000;  // 10 s

template <int D>
struct Cfg {
    static constexpr int STAGES = D == 128 ? 2 : 3;
    static constexpr int BOXES = D / 64;                 // 64-column boxes per tile row
    static constexpr uint32_t kTileK_B = BN * D * 2;     // K or V tile bytes
    static constexpr uint32_t kTileQ_B = BM * D * 2;     // Q or dO tile bytes
    static constexpr uint32_t kBoxK_B = BN * 128;        // one 64-column box of K / V
    static constexpr uint32_t kBoxQ_B = BM * 128;        // one 64-column box of Q / dO
    static constexpr uint32_t kdS_B = BN * BM * 2;
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = OFF_K + kTileK_B;
    static constexpr uint32_t OFF_Q = OFF_V + kTileK_B;
    static constexpr uint32_t OFF_DO = OFF_Q + STAGES * kTileQ_B;
    static constexpr uint32_t OFF_DS = OFF_DO + STAGES * kTileQ_B;
    static constexpr uint32_t OFF_LSE = OFF_DS + kdS_B;
    static constexpr uint32_t OFF_DD = OFF_LSE + STAGES * BM * 4;
    static constexpr uint32_t OFF_BAR = OFF_DD + STAGES * BM * 4;
    static constexpr uint32_t kNumBars = 16 + 2 * STAGES;
    static constexpr uint32_t OFF_MISC = OFF_BAR + kNumBars * 8;
    static constexpr uint32_t SMEM = OFF_MISC + 16;
    static constexpr uint32_t TM_DV = 0, TM_DK = D, TM_BUF0 = 2 * D;
};

// Barrier slots.
enum {
    B_KV = 0,
    B_S_FULL,
    B_DP_FULL,
    B_P_READY,
    B_DS_READY,
    B_DS_EMPTY,
    B_DQ_FULL,
    B_DQ_EMPTY,
    B_G3,
    B_G4,
    B_ACC,
    B_FINAL,
    B_STAGE0  // then STAGES "full" barriers, then STAGES "empty" barriers
};

struct Params {
    const float* lse2;
    const float* Dws;
    float* dqacc;
    void* dK;
    void* dV;
    unsigned int* err;
    int B, H, H_kv, S_q, S_k, S_q_pad;
    float scale, scale_log2;
    int causal;
    int n_kv_tiles;
};

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack2_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Bounded wait.  Returns false (and raises the CTA abort flag and the device
// error word) if the phase did not complete in time or another role aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned int* err) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    uint32_t spins = 0;
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (++spins % 64 == 0) {
            if (*abort_flag) return false;
            if (ptx::globaltimer() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicOr(err, kErrTimeout);
                return false;
            }
        }
    }
}

// Warp-uniform bounded wait: every lane waits (each gets the acquire), the
// warp then agrees, so a timeout seen by one lane makes the whole warp leave.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              unsigned int* err) {
    const bool ok = wait_bar(bar, parity, abort_flag, err);
    return __all_sync(0xffffffffu, ok);
}

// Wait used while shutting down after an abort: bounded, no flag checks.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer() - t0 > kWaitLimitNs) return;
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_sm103_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                     const Params p) {
    using C = Cfg<D>;
    constexpr bool kBF16 = sizeof(T) == 2 && TypeTraits<T>::kId == FA_BF16;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 4);
    auto bar = [&](int i) { return sbase + C::OFF_BAR + 8u * (uint32_t)i; };
    auto bar_full = [&](int s) { return bar(B_STAGE0 + s); };
    auto bar_empty = [&](int s) { return bar(B_STAGE0 + C::STAGES + s); };

    // ---- work assignment: blockIdx.x = key tile (heaviest causal tiles first) x (b, kv head)
    const int bhkv_count = p.B * p.H_kv;
    const int n_tile = blockIdx.x / bhkv_count;
    const int bkv = blockIdx.x % bhkv_count;
    const int b = bkv / p.H_kv, hk = bkv % p.H_kv;
    const int g = p.H / p.H_kv;
    const int n0 = n_tile * BN;
    const int off = p.S_k - p.S_q;  // key j visible to query i iff j <= i + off (causal)
    const int m_tiles = (p.S_q + BM - 1) / BM;
    int m_start = 0;
    if (p.causal) {
        const int first_q = n0 - off;  // first query row that can see key n0
        m_start = first_q <= 0 ? 0 : first_q / BM;
    }
    const int nm = m_tiles > m_start ? m_tiles - m_start : 0;
    const int n_it = g * nm;

    if (threadIdx.x == 0) {
        if ((sbase & 1023u) != 0) atomicOr(p.err, kErrSmemAlign);
        *abort_flag = (sbase & 1023u) != 0;
        for (int i = 0; i < (int)C::kNumBars; ++i)
            ptx::mbar_init(bar(i), (i == B_P_READY || i == B_DS_READY || i == B_DQ_EMPTY) ? 4u : 1u);
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
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

    auto iter_coords = [&](int it, int& bh, int& m0) {
        const int hh = it / nm;
        m0 = (m_start + it % nm) * BM;
        bh = b * p.H + hk * g + hh;
    };

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && !*abort_flag) {
            ptx::mbar_arrive_expect_tx(bar(B_KV), 2 * C::kTileK_B);
            for (int x = 0; x < C::BOXES; ++x) {
                ptx::tma_load_3d(sbase + C::OFF_K + x * C::kBoxK_B, &tmK, x * 64, n0, bkv, bar(B_KV));
                ptx::tma_load_3d(sbase + C::OFF_V + x * C::kBoxK_B, &tmV, x * 64, n0, bkv, bar(B_KV));
            }
            int issued = 0;
            for (int it = 0; it < n_it; ++it) {
                const int s = it % C::STAGES;
                if (it >= C::STAGES &&
                    !wait_bar(bar_empty(s), ((it / C::STAGES) - 1) & 1, abort_flag, p.err))
                    break;
                int bh, m0;
                iter_coords(it, bh, m0);
                ptx::mbar_arrive_expect_tx(bar_full(s), 2 * C::kTileQ_B + 2 * BM * 4);
                for (int x = 0; x < C::BOXES; ++x) {
                    ptx::tma_load_3d(sbase + C::OFF_Q + s * C::kTileQ_B + x * C::kBoxQ_B, &tmQ, x * 64,
                                     m0, bh, bar_full(s));
                    ptx::tma_load_3d(sbase + C::OFF_DO + s * C::kTileQ_B + x * C::kBoxQ_B, &tmdO,
                                     x * 64, m0, bh, bar_full(s));
                }
                const size_t row0 = (size_t)bh * p.S_q_pad + m0;
                ptx::bulk_load(sbase + C::OFF_LSE + s * BM * 4, p.lse2 + row0, BM * 4, bar_full(s));
                ptx::bulk_load(sbase + C::OFF_DD + s * BM * 4, p.Dws + row0, BM * 4, bar_full(s));
                issued = it + 1;
            }
            // never leave copies in flight into shared memory that is about to be released
            drain_wait(bar(B_KV), 0);
            for (int it = issued - C::STAGES < 0 ? 0 : issued - C::STAGES; it < issued; ++it)
                drain_wait(bar_full(it % C::STAGES), (it / C::STAGES) & 1);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && !*abort_flag && n_it > 0) {
            constexpr uint32_t ID_SD = ptx::idesc_f16(BN, BM, kBF16, false, false);  // S^T, dP^T
            constexpr uint32_t ID_KV = ptx::idesc_f16(BN, D, kBF16, false, true);    // dV, dK (A in TMEM)
            constexpr uint32_t ID_Q = ptx::idesc_f16(BM, D, kBF16, true, true);      // dQ
            const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sdS = sbase + C::OFF_DS;
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
            bool ok = wait_bar(bar(B_KV), 0, abort_flag, p.err);
            if (ok) ok = wait_bar(bar_full(0), 0, abort_flag, p.err);
            if (ok) {
                ptx::tc_fence_after();
                gemm_sd(tm_buf0, sK, sbase + C::OFF_Q);
                ptx::mma_commit(bar(B_S_FULL));
                gemm_sd((tm_buf0 + 128), sV, sbase + C::OFF_DO);
                ptx::mma_commit(bar(B_DP_FULL));
            }
            for (int it = 0; ok && it < n_it; ++it) {
                const int s = it % C::STAGES;
                const int bs = it & 1;
                const uint32_t sQ = sbase + C::OFF_Q + s * C::kTileQ_B;
                const uint32_t sdO = sbase + C::OFF_DO + s * C::kTileQ_B;
                // dV += P^T dO   (A = P^T in TMEM, 16 query columns = 8 packed columns per step)
                if (!(ok = wait_bar(bar(B_P_READY), it & 1, abort_flag, p.err))) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int k = 0; k < BM / 16; ++k)
                    ptx::mma_ts(tmem + C::TM_DV, (tm_buf0 + 128 * bs) + k * 8,
                                ptx::sw128_desc(sdO + k * 2048, C::kBoxQ_B, 1024), ID_KV,
                                (it > 0 || k > 0) ? 1u : 0u);
                ptx::mma_commit(bar(B_G3));
                // dK += dS^T Q
                if (!(ok = wait_bar(bar(B_DS_READY), it & 1, abort_flag, p.err))) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int k = 0; k < BM / 16; ++k)
                    ptx::mma_ts(tmem + C::TM_DK, (tm_buf0 + 128 * (bs ^ 1)) + k * 8,
                                ptx::sw128_desc(sQ + k * 2048, C::kBoxQ_B, 1024), ID_KV,
                                (it > 0 || k > 0) ? 1u : 0u);
                ptx::mma_commit(bar(B_G4));
                // dQ = dS K into the S buffer once the dV product stopped reading P from it
                if (!(ok = wait_bar(bar(B_G3), it & 1, abort_flag, p.err))) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                    ptx::mma_ss((tm_buf0 + 128 * bs), ptx::sw128_desc(sdS + k * 2048, BN * 128, 1024),
                                ptx::sw128_desc(sK + k * 2048, C::kBoxK_B, 1024), ID_Q, k > 0);
                ptx::mma_commit(bar(B_DQ_FULL));
                ptx::mma_commit(bar_empty(s));
                ptx::mma_commit(bar(B_DS_EMPTY));
                if (it + 1 < n_it) {
                    const int s1 = (it + 1) % C::STAGES;
                    if (!(ok = wait_bar(bar_full(s1), ((it + 1) / C::STAGES) & 1, abort_flag, p.err))) break;
                    if (!(ok = wait_bar(bar(B_G4), it & 1, abort_flag, p.err))) break;
                    ptx::tc_fence_after();
                    gemm_sd((tm_buf0 + 128 * (bs ^ 1)), sK, sbase + C::OFF_Q + s1 * C::kTileQ_B);
                    ptx::mma_commit(bar(B_S_FULL));
                    if (!(ok = wait_bar(bar(B_DQ_EMPTY), it & 1, abort_flag, p.err))) break;
                    ptx::tc_fence_after();
                    gemm_sd((tm_buf0 + 128 * bs), sV, sbase + C::OFF_DO + s1 * C::kTileQ_B);
                    ptx::mma_commit(bar(B_DP_FULL));
                }
            }
            ptx::mma_commit(bar(B_ACC));
            // no MMA may still write TMEM when it is released
            ptx::mma_commit(bar(B_FINAL));
            drain_wait(bar(B_FINAL), 0);
        }
        __syncwarp();
    } else if (warp >= kWarpSoft0 && warp < kWarpSoft0 + 4) {
        // ------------------------------------------------------------ P / dS (one key row per thread)
        const int t = (warp - kWarpSoft0) * 32 + lane;  // TMEM lane == key row within the tile
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const int j = n0 + t;
        const bool row_valid = j < p.S_k;
        bool ok = !*abort_flag;
        for (int it = 0; ok && it < n_it; ++it) {
            const int s = it % C::STAGES;
            const int bs = it & 1;
            int bh, m0;
            iter_coords(it, bh, m0);
            const bool mask_tile = !row_valid ? true : (p.causal && (n0 + BN - 1 > m0 + off));
            const float* sl = reinterpret_cast<const float*>(smem + C::OFF_LSE + s * BM * 4);
            const float* sd = reinterpret_cast<const float*>(smem + C::OFF_DD + s * BM * 4);
            if (!(ok = wait_bar_warp(bar_full(s), (it / C::STAGES) & 1, abort_flag, p.err))) break;
            if (!(ok = wait_bar_warp(bar(B_S_FULL), it & 1, abort_flag, p.err))) break;
            ptx::tc_fence_after();
            float P[BM];
#pragma unroll
            for (int c = 0; c < BM / 32; ++c) {
                uint32_t r[32];
                ptx::tmem_ld32((tm_buf0 + 128 * bs) + lane_off + c * 32, r);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const int q = c * 32 + k;
                    float x = ptx::ex2(fmaf(__uint_as_float(r[k]), p.scale_log2, -sl[q]));
                    if (mask_tile) {
                        const bool vis = row_valid && (!p.causal || j <= m0 + q + off);
                        x = vis ? x : 0.f;
                    }
                    P[q] = x;
                }
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    pk[k] = kBF16 ? pack2_bf16(P[c * 32 + 2 * k], P[c * 32 + 2 * k + 1])
                                  : pack2_f16(P[c * 32 + 2 * k], P[c * 32 + 2 * k + 1]);
                ptx::tmem_st16((tm_buf0 + 128 * bs) + lane_off + c * 16, pk);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(B_P_READY));

            if (!(ok = wait_bar_warp(bar(B_DP_FULL), it & 1, abort_flag, p.err))) break;
            if (it > 0 && !(ok = wait_bar_warp(bar(B_DS_EMPTY), (it - 1) & 1, abort_flag, p.err))) break;
            ptx::tc_fence_after();
            uint8_t* sdS_row = smem + C::OFF_DS + (t >> 3) * 1024 + (t & 7) * 128;
#pragma unroll
            for (int c = 0; c < BM / 32; ++c) {
                uint32_t r[32];
                ptx::tmem_ld32((tm_buf0 + 128 * (bs ^ 1)) + lane_off + c * 32, r);
                ptx::tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int q = c * 32 + 2 * k;
                    const float d0 = P[q] * (__uint_as_float(r[2 * k]) - sd[q]);
                    const float d1 = P[q + 1] * (__uint_as_float(r[2 * k + 1]) - sd[q + 1]);
                    pk[k] = kBF16 ? pack2_bf16(d0, d1) : pack2_f16(d0, d1);
                }
                ptx::tmem_st16((tm_buf0 + 128 * (bs ^ 1)) + lane_off + c * 16, pk);
                // dS (key-major rows, query-contiguous) for the dQ product:
                // 128-byte swizzled MN-major layout, 8-query chunks.
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int q0 = c * 32 + u * 8;
                    const int blk = q0 >> 6, chunk = (q0 & 63) >> 3;
                    uint4 v = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                    *reinterpret_cast<uint4*>(sdS_row + blk * (BN * 128) + ((chunk ^ (t & 7)) << 4)) = v;
                }
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(B_DS_READY));
        }
        // ---- epilogue: dV and scale * dK rows to global
        if (ok && n_it > 0) ok = wait_bar_warp(bar(B_ACC), 0, abort_flag, p.err);
        if (ok) {
            ptx::tc_fence_after();
            T* dVrow = static_cast<T*>(p.dV) + ((size_t)bkv * p.S_k + j) * D;
            T* dKrow = static_cast<T*>(p.dK) + ((size_t)bkv * p.S_k + j) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t rv[32], rk[32];
                if (n_it > 0) {
                    ptx::tmem_ld32(tmem + C::TM_DV + lane_off + c * 32, rv);
                    ptx::tmem_ld32(tmem + C::TM_DK + lane_off + c * 32, rk);
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
                        const float v0 = __uint_as_float(rv[e]), v1 = __uint_as_float(rv[e + 1]);
                        const float k0 = __uint_as_float(rk[e]) * p.scale, k1 = __uint_as_float(rk[e + 1]) * p.scale;
                        ov[k] = kBF16 ? pack2_bf16(v0, v1) : pack2_f16(v0, v1);
                        ok4[k] = kBF16 ? pack2_bf16(k0, k1) : pack2_f16(k0, k1);
                    }
                    if (row_valid) {
                        *reinterpret_cast<uint4*>(dVrow + c * 32 + u * 8) = make_uint4(ov[0], ov[1], ov[2], ov[3]);
                        *reinterpret_cast<uint4*>(dKrow + c * 32 + u * 8) = make_uint4(ok4[0], ok4[1], ok4[2], ok4[3]);
                    }
                }
            }
        }
    } else if (warp >= kWarpDrain0 && warp < kWarpDrain0 + 4) {
        // ------------------------------------------------------------ dQ drain (one query row per thread)
        const int t = (warp - kWarpDrain0) * 32 + lane;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        bool ok = !*abort_flag;
        for (int it = 0; ok && it < n_it; ++it) {
            const int bs = it & 1;
            int bh, m0;
            iter_coords(it, bh, m0);
            if (!(ok = wait_bar_warp(bar(B_DQ_FULL), it & 1, abort_flag, p.err))) break;
            ptx::tc_fence_after();
            uint32_t r[D / 32][32];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) ptx::tmem_ld32((tm_buf0 + 128 * bs) + lane_off + c * 32, r[c]);
            ptx::tmem_wait_ld();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(B_DQ_EMPTY));
            const int row = m0 + t;
            if (row < p.S_q) {
                float* dst = p.dqacc + ((size_t)bh * p.S_q + row) * D;
#pragma unroll
                for (int c = 0; c < D / 4; ++c)
                    ptx::red_add_v4(dst + 4 * c, __uint_as_float(r[c / 8][(4 * c) % 32]),
                                    __uint_as_float(r[c / 8][(4 * c + 1) % 32]),
                                    __uint_as_float(r[c / 8][(4 * c + 2) % 32]),
                                    __uint_as_float(r[c / 8][(4 * c + 3) % 32]));
            }
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

// 3-D view [heads][rows][D] of a [B, heads, rows, D] tensor, box = 64 columns x 128 rows.
bool make_map(CUtensorMap* m, const void* base, int dtype, int heads, int rows, int D) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)heads};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)rows * D * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt =
        dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int D>
cudaError_t launch_t(const void* Q, const void* K, const void* V, const void* dO,
                     const Workspace& ws, void* dK, void* dV, const Shape& s, cudaStream_t st) {
    using C = Cfg<D>;
    static_assert(C::SMEM <= 232448, "shared memory budget");
    CUtensorMap tq, tk, tv, tdo;
    const int dt = TypeTraits<T>::kId;
    if (!make_map(&tq, Q, dt, s.B * s.H, s.S_q, D) || !make_map(&tk, K, dt, s.B * s.H_kv, s.S_k, D) ||
        !make_map(&tv, V, dt, s.B * s.H_kv, s.S_k, D) || !make_map(&tdo, dO, dt, s.B * s.H, s.S_q, D))
        return cudaErrorInvalidValue;
    Params p;
    p.lse2 = ws.lse2;
    p.Dws = ws.Dws;
    p.dqacc = ws.dqacc;
    p.dK = dK;
    p.dV = dV;
    p.err = ws.err;
    p.B = s.B;
    p.H = s.H;
    p.H_kv = s.H_kv;
    p.S_q = s.S_q;
    p.S_k = s.S_k;
    p.S_q_pad = s.S_q_pad;
    p.scale = s.scale;
    p.scale_log2 = s.scale * 1.4426950408889634f;
    p.causal = s.causal;
    p.n_kv_tiles = (s.S_k + BN - 1) / BN;
    auto kern = bwd_sm103_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    const long grid = (long)p.n_kv_tiles * s.B * s.H_kv;
    kern<<<(unsigned)grid, kThreads, C::SMEM, st>>>(tq, tk, tv, tdo, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_sm103(int dtype, const void* Q, const void* K, const void* V,
                             const void* dO, const Workspace& ws, void* dK, void* dV,
                             const Shape& s, cudaStream_t st) {
    if (s.d == 64) {
        if (dtype == FA_F16) return launch_t<__half, 64>(Q, K, V, dO, ws, dK, dV, s, st);
        if (dtype == FA_BF16) return launch_t<__nv_bfloat16, 64>(Q, K, V, dO, ws, dK, dV, s, st);
    } else if (s.d == 128) {
        if (dtype == FA_F16) return launch_t<__half, 128>(Q, K, V, dO, ws, dK, dV, s, st);
        if (dtype == FA_BF16) return launch_t<__nv_bfloat16, 128>(Q, K, V, dO, ws, dK, dV, s, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace fa
