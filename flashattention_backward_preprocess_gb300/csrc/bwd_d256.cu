// bwd_d256.cu -- FlashAttention-2 backward main kernel for head dim 256 on GB300
// (sm_103a), f16 / bf16, on the 5th-generation tensor cores.
//
// Same mathematics as the d <= 128 kernel (boostr flash_bwd.rs, doc comment "Two-step
// process", step 2 "compute dQ (atomicAdd), dK, dV"), with the per-tile products
//   S    = Q K^T            P    = exp2(S * scale*log2e - LSE*log2e)
//   dP   = dO V^T           dS   = P * (dP - D)
//   dV^T += dO^T P          dK^T += Q^T dS          dQacc += dS K  (fp32 reduction)
// but a layout of its own: at d = 256 the dK and dV of a 128-key tile alone would fill the
// 512 TMEM columns, and a 128-row Q or dO tile is 64 KB, so
//   * one CTA owns 64 keys of one (batch, kv head) and walks every 64-row query tile of
//     every query head of the group (heads innermost), so dK and dV of the group are
//     summed in TMEM without atomics;
//   * dK and dV accumulate transposed (dK^T, dV^T: TMEM lane = head-dim row), as two
//     M = 128 halves of d, 64 columns each (one per key);
//   * S, dP and dQ are "query-major" M = 64 products (TMEM lanes 16q .. 16q + 15 of each
//     lane quadrant q hold query rows 16q .. 16q + 15); dQ (64 x 256) is computed in two
//     128-column halves that share one TMEM buffer;
//   * the softmax-gradient warps write P and dS to shared memory, 16-bit, as the B operand
//     of the dV^T / dK^T products and (dS) the A operand of the dQ product;
//   * TMA stages K, V once and Q, dO (64 rows, 32 KB each) through a 2-stage ring; a stage
//     is free for the load two iterations ahead as soon as the dK^T product, the last one
//     reading it, is done;
//   * the dQ halves are drained TMEM -> registers -> fp32 vector reductions
//     (red.global.add.v2.f32, all 32 lanes of each drain warp) into the accumulator.  dQ is
//     not staged through shared memory for bulk reduce-adds as it is at d <= 128: that
//     holds the stage until TMA has read it, and the products (~270 KB of shared-memory
//     operands per iteration) compete with the staging traffic; measured 36 % slower.
//     The reductions bound the kernel: 64 KB of fp32 adds per 10.5 MFLOP iteration.
// TMEM (512 columns): dV^T [0, 128), dK^T [128, 256), S [256, 320), dP [320, 384), dQ half
// [384, 512).  Shared memory: K, V 32 KB each, 2 x (Q 32 KB + dO 32 KB), P and dS tiles
// 2 x 8 KB each, LSE / D rows: 230 KB.
// Warp roles: 0-3 drain dQ (one per lane quadrant); 4-11 P / dS and the dK / dV epilogue
// (two per quadrant, one per 32-key half); 12 TMA; 13 TMEM owner and MMA issuer.
// Every mbarrier wait is bounded; on timeout the kernel records an error word, the other
// roles drop out, TMEM is freed and the kernel returns.
#include <math.h>

#include "bounded_wait.cuh"
#include "fa_internal.cuh"
#include "sm103_ptx.cuh"
#include "tma_map.cuh"

namespace fa {
namespace {

constexpr int D = 256;
constexpr int BM = 64;  // query rows per iteration
constexpr int BN = 64;  // key rows per CTA
constexpr int STAGES = 2;
constexpr int kThreads = 14 * 32;
constexpr int kWarpDrain0 = 0, kWarpSoft0 = 4, kNumSoftWarps = 8, kWarpTma = 12, kWarpMma = 13;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_DV = 0, TM_DK = 128, TM_S = 256, TM_DP = 320, TM_DQ = 384;

constexpr uint32_t kBox = 64 * 128;                 // one 64-column box of a 64-row tile (8 KB)
constexpr uint32_t kTile = 4 * kBox;                // a 64 x 256 16-bit tile (32 KB)
constexpr uint32_t kPT = BM * 128;                  // a P or dS tile: 64 queries x 64 keys, 16-bit
constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_V = OFF_K + kTile;
constexpr uint32_t OFF_Q = OFF_V + kTile;
constexpr uint32_t OFF_DO = OFF_Q + STAGES * kTile;
constexpr uint32_t OFF_P = OFF_DO + STAGES * kTile;
constexpr uint32_t OFF_DS = OFF_P + 2 * kPT;
constexpr uint32_t OFF_LSE = OFF_DS + 2 * kPT;
constexpr uint32_t OFF_DD = OFF_LSE + STAGES * BM * 4;
constexpr uint32_t OFF_BAR = OFF_DD + STAGES * BM * 4;

// Barrier slots.
enum {
    B_KV = 0,    // K, V landed (TMA)
    B_S_FULL,    // S(i) in TMEM (MMA commit)
    B_DP_FULL,   // dP(i) in TMEM (MMA commit)
    B_P_READY,   // P(i) in its shared tile, S read out of TMEM (8 softmax warps)
    B_DS_READY,  // dS(i) in its shared tile, dP read out of TMEM (8 softmax warps)
    B_DQ_FULL,   // a dQ half in TMEM (MMA commit; two phases per iteration)
    B_DQ_EMPTY,  // that half read out of TMEM (4 drain warps)
    B_PT_FREE,   // P tile k no longer read (MMA commit after the dV^T product); 2 slots
    B_DT_FREE = B_PT_FREE + 2,  // dS tile k no longer read (commit after the dQ products); 2 slots
    B_ACC = B_DT_FREE + 2,       // every product done (MMA commit)
    B_FINAL,     // MMA shutdown
    B_STAGE0     // STAGES "full" barriers, then STAGES "empty" barriers
};
constexpr uint32_t kNumBars = B_STAGE0 + 2 * STAGES;
constexpr uint32_t OFF_MISC = OFF_BAR + kNumBars * 8;
constexpr uint32_t SMEM = OFF_MISC + 16;
static_assert(SMEM <= 232448, "shared memory budget");

struct Params {
    const float* lse2;
    const float* Dws;
    void* dK;
    void* dV;
    float* dqacc;  // fp32 dQ accumulator [B*H][S_q][256]
    unsigned int* err;
    int B, H, H_kv, S_q, S_k, S_q_pad;
    float scale, scale_log2;
    int causal, window;
    int group_chunk;  // (b, kv head) groups per block of the CTA order (divides B * H_kv)
    int skip_dq;      // 1: leave dQ alone (deterministic mode computes it in a kernel of its own)
    int split;        // CTAs per key tile (1, or 2 = a cluster splitting the query tiles, see below)
};

template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if (kBF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// 16 TMEM lanes x 32 columns starting at taddr (lane field = the quadrant's first lane):
// register 4j + 0/1 of thread t holds row t/4, columns 8j + 2(t%4) + 0/1; registers
// 4j + 2/3 hold row t/4 + 8, the same columns.
__device__ __forceinline__ void tmem_ld16x256_x4(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// 16 TMEM lanes x 128 columns: register 4j + 0/1 of thread t holds row t/4, columns
// 8j + 2(t%4) + 0/1; registers 4j + 2/3 row t/4 + 8 (j = 0..15).
__device__ __forceinline__ void tmem_ld16x256_x16(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
        "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr));
}

// Byte offset of element (row, col) of a 128-byte-swizzled tile with 128-byte rows
// (64 16-bit or 32 fp32 columns): 8-row atoms of 1024 bytes, 16-byte chunks XOR row % 8.
__device__ __forceinline__ uint32_t sw128_off(int row, int byte_in_row) {
    return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((((byte_in_row >> 4) ^ (row & 7))) << 4) +
                      (byte_in_row & 15));
}

// dV and scale * dK for keys j0 .. j0 + 31 (those below S_k) at head-dim index dcol
template <typename T>
__device__ __forceinline__ void write_dkv(const Params& p, int bkv, int j0, int dcol, const uint32_t (&rv)[32],
                                          const uint32_t (&rk)[32]) {
    T* dVb = static_cast<T*>(p.dV) + (size_t)bkv * p.S_k * D + dcol;
    T* dKb = static_cast<T*>(p.dK) + (size_t)bkv * p.S_k * D + dcol;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        const int j = j0 + k;
        if (j < p.S_k) {
            dVb[(size_t)j * D] = TypeTraits<T>::from_f32(__uint_as_float(rv[k]));
            dKb[(size_t)j * D] = TypeTraits<T>::from_f32(__uint_as_float(rk[k]) * p.scale);
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_d256_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const Params p) {
    constexpr bool kBF16 = TypeTraits<T>::kId == FA_BF16;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 4);
    auto bar = [&](int i) { return sbase + OFF_BAR + 8u * (uint32_t)i; };
    auto bar_full = [&](int s) { return bar(B_STAGE0 + s); };
    auto bar_empty = [&](int s) { return bar(B_STAGE0 + STAGES + s); };

    // ---- work assignment (as the d <= 128 kernel): item = (block of group_chunk (b, kv head)
    // groups) x key tile x (group within the block); each CTA walks its query tiles from the
    // last one down, the group's heads innermost.  With split = 2 the two CTAs of a cluster
    // share one item, each taking one contiguous half of its query tiles (a long causal key
    // tile would otherwise set the kernel's time alone), and add their dK / dV partials
    // through distributed shared memory at the end.
    const int n_key_tiles = (p.S_k + BN - 1) / BN;
    const int rank = (int)(blockIdx.x % (unsigned)p.split);  // rank within the cluster (1-D)
    const int item = (int)(blockIdx.x / (unsigned)p.split);
    const int chunk = item / (n_key_tiles * p.group_chunk);
    const int in_chunk = item % (n_key_tiles * p.group_chunk);
    const int n_tile = in_chunk / p.group_chunk;
    const int bkv = chunk * p.group_chunk + in_chunk % p.group_chunk;
    const int b = bkv / p.H_kv, hk = bkv % p.H_kv;
    const int g = p.H / p.H_kv;
    const int n0 = n_tile * BN;
    const int off = p.S_k - p.S_q;  // query i sits at key position i + off
    Shape sh;                       // the fields the range helpers read
    sh.S_q = p.S_q;
    sh.S_k = p.S_k;
    sh.causal = p.causal;
    sh.window = p.window;
    int q_lo, q_hi;
    query_range(sh, n0, min(n0 + BN, p.S_k), q_lo, q_hi);
    const int m_first = q_lo / BM;
    const int m_last = q_hi > q_lo ? (q_hi + BM - 1) / BM : m_first;
    // this CTA's query tiles [m_start, m_end)
    const int m_start = m_first + (m_last - m_first) * rank / p.split;
    const int m_end = m_first + (m_last - m_first) * (rank + 1) / p.split;
    const int n_it = g * (m_end - m_start);
    auto iter_coords = [&](int it, int& bh, int& m0) {
        m0 = (m_end - 1 - it / g) * BM;
        bh = b * p.H + hk * g + it % g;
    };

    if (threadIdx.x == 0) {
        if ((sbase & 1023u) != 0) atomicOr(p.err, kErrSmemAlign);
        *abort_flag = (sbase & 1023u) != 0;
        for (int i = 0; i < (int)kNumBars; ++i) {
            uint32_t count = 1;
            if (i == B_P_READY || i == B_DS_READY) count = kNumSoftWarps;
            if (i == B_DQ_EMPTY) count = 4;
            ptx::mbar_init(bar(i), count);
        }
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
        if (lane == 0 && !*abort_flag) {
            ptx::mbar_arrive_expect_tx(bar(B_KV), 2 * kTile);
            for (int x = 0; x < 4; ++x) {
                ptx::tma_load_3d(sbase + OFF_K + x * kBox, &tmK, x * 64, n0, bkv, bar(B_KV));
                ptx::tma_load_3d(sbase + OFF_V + x * kBox, &tmV, x * 64, n0, bkv, bar(B_KV));
            }
            auto load_stage = [&](int it) {
                const int s = it % STAGES;
                int bh, m0;
                iter_coords(it, bh, m0);
                ptx::mbar_arrive_expect_tx(bar_full(s), 2 * kTile + 2 * BM * 4);
                for (int x = 0; x < 4; ++x) {
                    ptx::tma_load_3d(sbase + OFF_Q + s * kTile + x * kBox, &tmQ, x * 64, m0, bh, bar_full(s));
                    ptx::tma_load_3d(sbase + OFF_DO + s * kTile + x * kBox, &tmdO, x * 64, m0, bh, bar_full(s));
                }
                const size_t row0 = (size_t)bh * p.S_q_pad + m0;
                ptx::bulk_load(sbase + OFF_LSE + s * BM * 4, p.lse2 + row0, BM * 4, bar_full(s));
                ptx::bulk_load(sbase + OFF_DD + s * BM * 4, p.Dws + row0, BM * 4, bar_full(s));
            };
            int issued = 0;
            for (int it = 0; it < n_it; ++it) {
                const int s = it % STAGES;
                // stage s was last read by the dK^T product of iteration it - 2 (MMA commit)
                if (it >= STAGES && !wait_bar(bar_empty(s), ((it / STAGES) - 1) & 1, abort_flag, p.err)) break;
                load_stage(it);
                issued = it + 1;
            }
            // never leave copies in flight into shared memory that is about to be released
            drain_wait(bar(B_KV), 0);
            for (int it = issued - STAGES < 0 ? 0 : issued - STAGES; it < issued; ++it)
                drain_wait(bar_full(it % STAGES), (it / STAGES) & 1);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && !*abort_flag && n_it > 0) {
            constexpr uint32_t ID_S = ptx::idesc_f16(64, 64, kBF16, false, false);   // S, dP
            constexpr uint32_t ID_T = ptx::idesc_f16(128, 64, kBF16, true, true);    // dV^T, dK^T
            constexpr uint32_t ID_Q = ptx::idesc_f16(64, 128, kBF16, false, true);   // dQ halves
            const uint32_t sK = sbase + OFF_K, sV = sbase + OFF_V;
            // S = Q K^T or dP = dO V^T (M = 64 queries, N = 64 keys, 16 K-steps over d; both
            // operands K-major)
            auto gemm_s = [&](uint32_t d_tmem, uint32_t a_base, uint32_t b_base) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t koff = (k / 4) * kBox + (k % 4) * 32;
                    ptx::mma_ss(d_tmem, ptx::sw128_desc(a_base + koff, 16, 1024),
                                ptx::sw128_desc(b_base + koff, 16, 1024), ID_S, k > 0);
                }
            };
            // acc^T += X^T Y for the two 128-row halves of d: A = X^T (MN-major: the 16-bit
            // [64 x 256] tile, two 64-column boxes per half), B = Y (the [64 x 64] P or dS
            // tile, MN-major); K = the 64 queries in 4 steps
            auto gemm_t = [&](uint32_t d_tmem, uint32_t x_base, uint32_t y_base, bool acc) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int k = 0; k < BM / 16; ++k)
                        ptx::mma_ss(d_tmem + 64 * h, ptx::sw128_desc(x_base + 2 * h * kBox + k * 2048, kBox, 1024),
                                    ptx::sw128_desc(y_base + k * 2048, kPT, 1024), ID_T, (acc || k > 0) ? 1u : 0u);
            };
            // dQ half h = dS K[:, 128h, 128h + 128): A = dS (K-major over the 64 keys), B = K
            // (MN-major, two 64-column boxes)
            auto gemm_q = [&](uint32_t ds_base, int h) {
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                    ptx::mma_ss(tmem + TM_DQ, ptx::sw128_desc(ds_base + k * 32, 16, 1024),
                                ptx::sw128_desc(sK + 2 * h * kBox + k * 2048, kBox, 1024), ID_Q, k > 0);
            };
            bool ok = wait_bar(bar(B_KV), 0, abort_flag, p.err);
            if (ok) ok = wait_bar(bar_full(0), 0, abort_flag, p.err);
            if (ok) {
                ptx::tc_fence_after();
                gemm_s(tmem + TM_S, sbase + OFF_Q, sK);
                ptx::mma_commit(bar(B_S_FULL));
                gemm_s(tmem + TM_DP, sbase + OFF_DO, sV);
                ptx::mma_commit(bar(B_DP_FULL));
            }
            for (int it = 0; ok && it < n_it; ++it) {
                const int s = it % STAGES, s1 = (it + 1) % STAGES;
                const uint32_t sQ = sbase + OFF_Q + s * kTile, sdO = sbase + OFF_DO + s * kTile;
                const uint32_t sP = sbase + OFF_P + (it & 1) * kPT, sdS = sbase + OFF_DS + (it & 1) * kPT;
                // dV^T += dO^T P once P(i) is in its tile (the softmax read S(i) before)
                if (!(ok = wait_bar(bar(B_P_READY), it & 1, abort_flag, p.err))) break;
                ptx::tc_fence_after();
                gemm_t(tmem + TM_DV, sdO, sP, it > 0);
                ptx::mma_commit(bar(B_PT_FREE + (it & 1)));
                // S(i+1) into the S buffer (read out already)
                if (it + 1 < n_it) {
                    if (!(ok = wait_bar(bar_full(s1), ((it + 1) / STAGES) & 1, abort_flag, p.err))) break;
                    ptx::tc_fence_after();
                    gemm_s(tmem + TM_S, sbase + OFF_Q + s1 * kTile, sK);
                    ptx::mma_commit(bar(B_S_FULL));
                }
                // dK^T += Q^T dS once dS(i) is in its tile (the softmax read dP(i) before)
                if (!(ok = wait_bar(bar(B_DS_READY), it & 1, abort_flag, p.err))) break;
                ptx::tc_fence_after();
                gemm_t(tmem + TM_DK, sQ, sdS, it > 0);
                ptx::mma_commit(bar_empty(s));  // Q(i), dO(i) read for the last time
                if (!p.skip_dq) {
                    // dQ low half into the dQ buffer once the drain read the previous high half
                    if (it > 0 && !(ok = wait_bar(bar(B_DQ_EMPTY), 1, abort_flag, p.err))) break;
                    ptx::tc_fence_after();
                    gemm_q(sdS, 0);
                    ptx::mma_commit(bar(B_DQ_FULL));
                }
                // dP(i+1) while the drain reads the low half (the dP buffer was read out already)
                if (it + 1 < n_it) {
                    gemm_s(tmem + TM_DP, sbase + OFF_DO + s1 * kTile, sV);
                    ptx::mma_commit(bar(B_DP_FULL));
                }
                if (!p.skip_dq) {
                    if (!(ok = wait_bar(bar(B_DQ_EMPTY), 0, abort_flag, p.err))) break;
                    ptx::tc_fence_after();
                    gemm_q(sdS, 1);
                    ptx::mma_commit(bar(B_DQ_FULL));
                }
                ptx::mma_commit(bar(B_DT_FREE + (it & 1)));
            }
            ptx::mma_commit(bar(B_ACC));
            // no MMA may still write TMEM when it is released
            ptx::mma_commit(bar(B_FINAL));
            drain_wait(bar(B_FINAL), 0);
        }
        __syncwarp();
    } else if (warp >= kWarpSoft0 && warp < kWarpSoft0 + kNumSoftWarps) {
        // ------------------------------------------------------------ P / dS
        // Warp (quadrant qd, key half hc): query rows 16 qd + t/4 and 16 qd + t/4 + 8 of the
        // tile, keys 32 hc + 8j + 2(t%4) + 0/1 (j = 0..3), from TMEM lanes 32 qd ...
        const int qd = warp & 3;
        const int hc = (warp - kWarpSoft0) >> 2;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        const int ra = 16 * qd + (lane >> 2), rb = ra + 8;  // the thread's two query rows
        const int c0 = 32 * hc + 2 * (lane & 3);             // its first key column
        bool ok = !*abort_flag;
        for (int it = 0; ok && it < n_it; ++it) {
            const int s = it % STAGES;
            int bh, m0;
            iter_coords(it, bh, m0);
            const float* sl = reinterpret_cast<const float*>(smem + OFF_LSE + s * BM * 4);
            const float* sd = reinterpret_cast<const float*>(smem + OFF_DD + s * BM * 4);
            // every element of the tile visible (no mask needed): the extreme query-key
            // offsets of the tile satisfy the causal and window conditions, no key past S_k
            const int pk_min = m0 + off - (n0 + BN - 1), pk_max = m0 + BM - 1 + off - n0;
            const bool full = n0 + BN <= p.S_k && (!p.causal || pk_min >= 0) &&
                              (p.window <= 0 || (pk_max < p.window && (p.causal || -pk_min < p.window)));
            if (!(ok = wait_bar_warp(bar_full(s), (it / STAGES) & 1, abort_flag, p.err))) break;
            if (!(ok = wait_bar_warp(bar(B_S_FULL), it & 1, abort_flag, p.err))) break;
            ptx::tc_fence_after();
            uint32_t r[16];
            tmem_ld16x256_x4(tmem + TM_S + lane_base + 32 * hc, r);
            ptx::tmem_wait_ld();
            const float la = sl[ra], lb = sl[rb];
            float pv[16];  // P at (row, col) in the register layout of r
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int row = (e & 2) ? rb : ra;
                const int col = c0 + 8 * (e >> 2) + (e & 1);
                float x = ptx::ex2(fmaf(__uint_as_float(r[e]), p.scale_log2, -((e & 2) ? lb : la)));
                if (!full) {
                    const int j = n0 + col;
                    x = (j < p.S_k && key_visible(m0 + row + off, j, p.causal, p.window)) ? x : 0.f;
                }
                pv[e] = x;
            }
            // the P tile of this parity was last read by the dV^T product two iterations ago
            if (it >= 2 && !(ok = wait_bar_warp(bar(B_PT_FREE + (it & 1)), ((it >> 1) - 1) & 1, abort_flag, p.err)))
                break;
            uint8_t* tP = smem + OFF_P + (it & 1) * kPT;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int cb = 2 * (c0 + 8 * j);  // byte of the column pair within the row
                *reinterpret_cast<uint32_t*>(tP + sw128_off(ra, cb)) = pack2<kBF16>(pv[4 * j], pv[4 * j + 1]);
                *reinterpret_cast<uint32_t*>(tP + sw128_off(rb, cb)) = pack2<kBF16>(pv[4 * j + 2], pv[4 * j + 3]);
            }
            ptx::tc_fence_before();
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(B_P_READY));

            // dS = P * (dP - D), with P rounded as the dV^T product saw it
            if (!(ok = wait_bar_warp(bar(B_DP_FULL), it & 1, abort_flag, p.err))) break;
            if (it >= 2 && !(ok = wait_bar_warp(bar(B_DT_FREE + (it & 1)), ((it >> 1) - 1) & 1, abort_flag, p.err)))
                break;
            ptx::tc_fence_after();
            tmem_ld16x256_x4(tmem + TM_DP + lane_base + 32 * hc, r);
            ptx::tmem_wait_ld();
            const float da = sd[ra], db = sd[rb];
            uint8_t* tS = smem + OFF_DS + (it & 1) * kPT;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float ds[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int e = 4 * j + u;
                    const uint32_t pr = pack2<kBF16>(pv[e], 0.f);
                    const float pq = kBF16 ? __uint_as_float(pr << 16) : __half2float(*reinterpret_cast<const __half*>(&pr));
                    ds[u] = pq * (__uint_as_float(r[e]) - ((u & 2) ? db : da));
                }
                const int cb = 2 * (c0 + 8 * j);
                *reinterpret_cast<uint32_t*>(tS + sw128_off(ra, cb)) = pack2<kBF16>(ds[0], ds[1]);
                *reinterpret_cast<uint32_t*>(tS + sw128_off(rb, cb)) = pack2<kBF16>(ds[2], ds[3]);
            }
            ptx::tc_fence_before();
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(B_DS_READY));
        }
        // ---- epilogue: dV^T and scale * dK^T rows (one head-dim index per thread) to dV, dK.
        // In a split pair the rows are written after the CTA barrier at the end instead.
        if (ok && n_it > 0) ok = wait_bar_warp(bar(B_ACC), 0, abort_flag, p.err);
        if (ok && p.split == 1) {
            ptx::tc_fence_after();
            const int dcol = 128 * hc + 32 * qd + lane;  // head-dim index of this thread
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t rv[32], rk[32];
                if (n_it > 0) {
                    ptx::tmem_ld32p(tmem + TM_DV + 64 * hc + lane_base + 32 * c, rv);
                    ptx::tmem_ld32p(tmem + TM_DK + 64 * hc + lane_base + 32 * c, rk);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) rv[k] = rk[k] = 0u;
                }
                write_dkv<T>(p, bkv, n0 + 32 * c, dcol, rv, rk);
            }
        }
    } else if (warp >= kWarpDrain0 && warp < kWarpDrain0 + 4) {
        // ------------------------------------------------------------ dQ drain
        // Warp qd reads the 16 query rows of its lane quadrant, a whole 128-column half at a
        // time, with all 32 threads (rows t/4 and t/4 + 8, column pairs), releases the TMEM
        // buffer, then adds the values into the accumulator rows with fp32 vector reductions.
        const int qd = warp;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        const int ra = 16 * qd + (lane >> 2), rb = ra + 8;
        const int c0 = 2 * (lane & 3);
        bool ok = !*abort_flag && !p.skip_dq;
        for (int it = 0; ok && it < n_it; ++it) {
            int bh, m0;
            iter_coords(it, bh, m0);
            const bool a_ok = m0 + ra < p.S_q, b_ok = m0 + rb < p.S_q;
            float* ga = p.dqacc + ((size_t)bh * p.S_q + m0 + ra) * D + c0;
            float* gb = ga + 8 * D;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                if (!(ok = wait_bar_warp(bar(B_DQ_FULL), h, abort_flag, p.err))) break;
                ptx::tc_fence_after();
                uint32_t r[64];
                tmem_ld16x256_x16(tmem + TM_DQ + lane_base, r);
                ptx::tmem_wait_ld();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(B_DQ_EMPTY));
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int col = 128 * h + 8 * j;
                    if (a_ok) ptx::red_add_v2(ga + col, __uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]));
                    if (b_ok) ptx::red_add_v2(gb + col, __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (p.split > 1) {
        // Rank 1 parks its fp32 dK / dV partial sums in its shared memory (fp32, [key][d], over
        // the Q and dO stages, whose loads have all landed and been read) after the barrier
        // above; rank 0 adds them after the cluster barrier.
        if (rank == 1 && warp >= kWarpSoft0 && warp < kWarpSoft0 + kNumSoftWarps && !*abort_flag) {
            const int qd = warp & 3, hc = (warp - kWarpSoft0) >> 2;
            const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
            const int dcol = 128 * hc + 32 * qd + lane;
            float* park = reinterpret_cast<float*>(smem + OFF_Q);  // dV part, then dK part
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t rv[32], rk[32];
                if (n_it > 0) {
                    ptx::tmem_ld32p(tmem + TM_DV + 64 * hc + lane_base + 32 * c, rv);
                    ptx::tmem_ld32p(tmem + TM_DK + 64 * hc + lane_base + 32 * c, rk);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) rv[k] = rk[k] = 0u;
                }
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    park[(32 * c + k) * D + dcol] = __uint_as_float(rv[k]);
                    park[BN * D + (32 * c + k) * D + dcol] = __uint_as_float(rk[k]);
                }
            }
        }
        // every thread of both CTAs: rank 1's partial sums are in its shared memory
        ptx::cluster_sync();
        if (rank == 0 && warp >= kWarpSoft0 && warp < kWarpSoft0 + kNumSoftWarps && !*abort_flag) {
            const int qd = warp & 3, hc = (warp - kWarpSoft0) >> 2;
            const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
            const int dcol = 128 * hc + 32 * qd + lane;
            const uint32_t park = ptx::mapa_shared(sbase + OFF_Q, 1);
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t rv[32], rk[32];
                if (n_it > 0) {
                    ptx::tmem_ld32p(tmem + TM_DV + 64 * hc + lane_base + 32 * c, rv);
                    ptx::tmem_ld32p(tmem + TM_DK + 64 * hc + lane_base + 32 * c, rk);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) rv[k] = rk[k] = 0u;
                }
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const uint32_t o = (uint32_t)(((32 * c + k) * D + dcol) * 4);
                    rv[k] = __float_as_uint(__uint_as_float(rv[k]) + ptx::ld_shared_cluster_f32(park + o));
                    rk[k] = __float_as_uint(__uint_as_float(rk[k]) + ptx::ld_shared_cluster_f32(park + BN * D * 4 + o));
                }
                write_dkv<T>(p, bkv, n0 + 32 * c, dcol, rv, rk);
            }
        }
        ptx::tc_fence_before();
        ptx::cluster_sync();  // rank 0 has read rank 1's shared memory: both may exit
        ptx::tc_fence_after();
    }
    if (warp == kWarpMma) ptx::tmem_dealloc(tmem, kTmemCols);
}

template <typename T>
cudaError_t launch_t(const void* Q, const void* K, const void* V, const void* dO, const Workspace& ws, void* dK,
                     void* dV, const Shape& s, bool skip_dq, cudaStream_t st) {
    CUtensorMap tq, tk, tv, tdo;
    const CUtensorMapDataType dt =
        TypeTraits<T>::kId == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (s.d != D || !tma_map_3d(&tq, Q, dt, 2, s.B * s.H, s.S_q, D, BM) ||
        !tma_map_3d(&tk, K, dt, 2, s.B * s.H_kv, s.S_k, D, BN) || !tma_map_3d(&tv, V, dt, 2, s.B * s.H_kv, s.S_k, D, BN) ||
        !tma_map_3d(&tdo, dO, dt, 2, s.B * s.H, s.S_q, D, BM))
        return cudaErrorInvalidValue;
    Params p;
    p.lse2 = ws.lse2;
    p.Dws = ws.Dws;
    p.dK = dK;
    p.dV = dV;
    p.dqacc = ws.dqacc;
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
    p.window = s.window;
    p.skip_dq = skip_dq ? 1 : 0;
    // the block order of the d <= 128 kernel: one block of every group for causal calls
    // (heaviest key tiles first), blocks of 4 groups otherwise
    const int groups = s.B * s.H_kv;
    p.group_chunk = groups;
    if (!s.causal || s.window > 0) p.group_chunk = groups % 4 == 0 ? 4 : (groups % 2 == 0 ? 2 : groups);
    cudaError_t e = cudaFuncSetAttribute(bwd_d256_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
    if (e != cudaSuccess) return e;
    p.split = key_tile_split(s, BN, BM);
    const long grid = (long)((s.S_k + BN - 1) / BN) * s.B * s.H_kv * p.split;
    if (p.split == 1) {
        bwd_d256_kernel<T><<<(unsigned)grid, kThreads, SMEM, st>>>(tq, tk, tv, tdo, p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, bwd_d256_kernel<T>, tq, tk, tv, tdo, p);
}

}  // namespace

cudaError_t launch_bwd_d256(int dtype, const void* Q, const void* K, const void* V, const void* dO,
                            const Workspace& ws, void* dK, void* dV, const Shape& s, bool skip_dq,
                            cudaStream_t st) {
    if (dtype == FA_F16) return launch_t<__half>(Q, K, V, dO, ws, dK, dV, s, skip_dq, st);
    if (dtype == FA_BF16) return launch_t<__nv_bfloat16>(Q, K, V, dO, ws, dK, dV, s, skip_dq, st);
    return cudaErrorInvalidValue;
}

}  // namespace fa
