// bwd_simt.cu -- CUDA-core (FFMA) main backward kernel, used for fp32 inputs (and
// for f16 / bf16 when FA_BWD_KERNEL=simt).  fp32 needs the 1e-4 relative tolerance,
// which tf32 tensor-core operands (10-bit mantissa) do not meet, so the five products run
// on the FMA pipe, in fp32.
//
// Work split (same math as the tensor-core kernels): one CTA owns a tile of BN key/value
// rows of one (batch, kv head), keeps its dK / dV rows in registers, and walks BM-row query
// tiles of every query head in the group:
//   S  = Q K^T,  P = exp(scale * S - LSE)  (masked -> 0)    dP = dO V^T
//   dS = P * (dP - D)
//   dV += P^T dO,   dK += dS^T Q,   dQacc += dS K   (vector fp32 reductions into global)
// Every product is a register-tiled block product from shared memory (fp32 rows padded by
// four words, so the 16-byte accesses of a quarter warp fall in distinct banks): thread
// (ty, tx) of the 16 x 16 grid owns rows ty + 16r and columns tx + 16c of S / dP, key rows
// ty + 16r and 4-column groups tx + 16g of dK / dV, query rows ty + 16r and the same column
// groups of dQ.  scale is applied to dK here and to dQ in the finalisation kernel.
// For fp32 outputs a key tile can be split over two CTAs (small grids, long causal key
// tiles): each takes one half of the tile's (head, query tile) iterations and adds its dK / dV
// partial sums into the zeroed outputs with fp32 reductions.  Two addends onto zero give the
// same bits in either order, so dK and dV stay reproducible.
#include <math.h>

#include "fa_internal.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 256;  // 16 x 16

template <int D>
struct SCfg {
    static constexpr int BN = D <= 128 ? 64 : 32;  // key rows per CTA (shared memory at d = 256)
    static constexpr int BM = BN;                  // query rows per step
    static constexpr int LD = D + 4;               // padded fp32 row of a Q / K / V / dO tile
    static constexpr int LP = BN + 4;              // padded fp32 row of the P / dS tiles
    static constexpr int TR = BM / 16;             // rows per thread (S, dP, dQ)
    static constexpr int TC = BN / 16;             // key columns per thread (S, dP) = key rows (dK, dV)
    static constexpr int NG = (D / 4 + 15) / 16;   // 4-column groups per thread (dK, dV, dQ)
    static constexpr size_t SMEM = sizeof(float) * ((size_t)(2 * BN + 2 * BM) * LD + 2 * BM * LP + 2 * BM);
};

template <typename T>
__device__ __forceinline__ float4 load4(const T* p) {
    if constexpr (sizeof(T) == 4) {
        return *reinterpret_cast<const float4*>(p);
    } else {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        const T* t = reinterpret_cast<const T*>(&u);
        return make_float4(TypeTraits<T>::to_f32(t[0]), TypeTraits<T>::to_f32(t[1]), TypeTraits<T>::to_f32(t[2]),
                           TypeTraits<T>::to_f32(t[3]));
    }
}

// rows [0, n) of a [rows][D] global tile into a padded fp32 shared tile; rows n.. get zeros
template <typename T, int D>
__device__ __forceinline__ void stage_rows(float* dst, const T* src, int n, int rows) {
    constexpr int LD = D + 4;
    for (int e = threadIdx.x; e < rows * (D / 4); e += kThreads) {
        const int r = e / (D / 4), c4 = e % (D / 4);
        const float4 v = r < n ? load4(src + (size_t)r * D + 4 * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(dst + r * LD + 4 * c4) = v;
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) bwd_simt_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
    const T* __restrict__ dO, const float* __restrict__ lse2, const float* __restrict__ Dws,
    float* __restrict__ dqacc, T* __restrict__ dK, T* __restrict__ dV, Shape s, int split) {
    using C = SCfg<D>;
    constexpr int BN = C::BN, BM = C::BM, LD = C::LD, LP = C::LP, TR = C::TR, TC = C::TC, NG = C::NG;
    extern __shared__ float4 smem4[];
    float* smem = reinterpret_cast<float*>(smem4);
    float* sK = smem;               // [BN][LD]
    float* sV = sK + BN * LD;       // [BN][LD]
    float* sQ = sV + BN * LD;       // [BM][LD]
    float* sdO = sQ + BM * LD;      // [BM][LD]
    float* sP = sdO + BM * LD;      // [BM][LP]
    float* sdS = sP + BM * LP;      // [BM][LP]
    float* sL = sdS + BM * LP;      // [BM] LSE * log2 e
    float* sDd = sL + BM;           // [BM] D

    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    // blockIdx.x = (key tile x (batch, kv head), key tile outer: with causal masking the key
    // tiles with the most query rows start first) x the split rank
    const int groups = s.B * s.H_kv;
    const int rank = (int)(blockIdx.x % (unsigned)split);
    const int item = (int)(blockIdx.x / (unsigned)split);
    const int n0 = (item / groups) * BN;
    const int bkv = item % groups;
    const int b = bkv / s.H_kv, hk = bkv % s.H_kv;
    const int g = s.H / s.H_kv;
    const int off = s.S_k - s.S_q;  // query i sits at key position i + off
    const float kLog2e = 1.4426950408889634f;
    const float sc2 = s.scale * kLog2e;

    stage_rows<T, D>(sK, K + ((size_t)bkv * s.S_k + n0) * D, min(BN, s.S_k - n0), BN);
    stage_rows<T, D>(sV, V + ((size_t)bkv * s.S_k + n0) * D, min(BN, s.S_k - n0), BN);

    float accV[TC][NG][4], accK[TC][NG][4];
#pragma unroll
    for (int r = 0; r < TC; ++r)
#pragma unroll
        for (int q = 0; q < NG; ++q)
#pragma unroll
            for (int u = 0; u < 4; ++u) accV[r][q][u] = accK[r][q][u] = 0.f;

    // query rows [i_begin, i_end) see a key of this tile: nq query tiles per head, this CTA's
    // share of the g * nq (head, query tile) iterations is [it_lo, it_hi)
    int i_begin, i_end;
    query_range(s, n0, min(n0 + BN, s.S_k), i_begin, i_end);
    const int m_first = i_begin / BM * BM;
    const int nq = i_end > i_begin ? (i_end - m_first + BM - 1) / BM : 0;
    const int it_lo = g * nq * rank / split, it_hi = g * nq * (rank + 1) / split;

    {
        for (int it = it_lo; it < it_hi; ++it) {
            const int hh = it / nq;
            const int bh = b * s.H + hk * g + hh;
            const int m0 = m_first + (it % nq) * BM;
            const int rows = min(BM, s.S_q - m0);
            __syncthreads();  // the previous step's reads of sQ, sdO, sP, sdS are done
            stage_rows<T, D>(sQ, Q + ((size_t)bh * s.S_q + m0) * D, rows, BM);
            stage_rows<T, D>(sdO, dO + ((size_t)bh * s.S_q + m0) * D, rows, BM);
            for (int r = tid; r < BM; r += kThreads) {
                sL[r] = lse2[(size_t)bh * s.S_q_pad + m0 + r];  // +inf on padding rows: P = 0
                sDd[r] = Dws[(size_t)bh * s.S_q_pad + m0 + r];
            }
            __syncthreads();
            // ---- S and dP blocks (rows ty + 16r, keys tx + 16c), 4 head-dim columns a step
            float accS[TR][TC], accP[TR][TC];
#pragma unroll
            for (int r = 0; r < TR; ++r)
#pragma unroll
                for (int c = 0; c < TC; ++c) accS[r][c] = accP[r][c] = 0.f;
#pragma unroll 4
            for (int k = 0; k < D; k += 4) {
                float4 q[TR], o[TR], kk[TC], v[TC];
#pragma unroll
                for (int r = 0; r < TR; ++r) {
                    q[r] = *reinterpret_cast<const float4*>(sQ + (ty + 16 * r) * LD + k);
                    o[r] = *reinterpret_cast<const float4*>(sdO + (ty + 16 * r) * LD + k);
                }
#pragma unroll
                for (int c = 0; c < TC; ++c) {
                    kk[c] = *reinterpret_cast<const float4*>(sK + (tx + 16 * c) * LD + k);
                    v[c] = *reinterpret_cast<const float4*>(sV + (tx + 16 * c) * LD + k);
                }
#pragma unroll
                for (int r = 0; r < TR; ++r)
#pragma unroll
                    for (int c = 0; c < TC; ++c) {
                        accS[r][c] = fmaf(q[r].x, kk[c].x, accS[r][c]);
                        accS[r][c] = fmaf(q[r].y, kk[c].y, accS[r][c]);
                        accS[r][c] = fmaf(q[r].z, kk[c].z, accS[r][c]);
                        accS[r][c] = fmaf(q[r].w, kk[c].w, accS[r][c]);
                        accP[r][c] = fmaf(o[r].x, v[c].x, accP[r][c]);
                        accP[r][c] = fmaf(o[r].y, v[c].y, accP[r][c]);
                        accP[r][c] = fmaf(o[r].z, v[c].z, accP[r][c]);
                        accP[r][c] = fmaf(o[r].w, v[c].w, accP[r][c]);
                    }
            }
            // ---- P = exp(scale S - LSE) (visible pairs only), dS = P (dP - D)
#pragma unroll
            for (int r = 0; r < TR; ++r) {
                const int ri = ty + 16 * r, i = m0 + ri;
                const float l2 = sL[ri], Di = sDd[ri];
#pragma unroll
                for (int c = 0; c < TC; ++c) {
                    const int j = n0 + tx + 16 * c;
                    const bool vis = i < s.S_q && j < s.S_k && key_visible(i + off, j, s.causal, s.window);
                    const float pv = vis ? exp2f(fmaf(accS[r][c], sc2, -l2)) : 0.f;
                    sP[ri * LP + tx + 16 * c] = pv;
                    sdS[ri * LP + tx + 16 * c] = pv * (accP[r][c] - Di);
                }
            }
            __syncthreads();
            // ---- dV += P^T dO and dK += dS^T Q (key rows ty + 16r, column groups tx + 16q)
#pragma unroll 2
            for (int i = 0; i < BM; ++i) {
                float pk[TC], dk[TC];
#pragma unroll
                for (int r = 0; r < TC; ++r) {
                    pk[r] = sP[i * LP + ty + 16 * r];
                    dk[r] = sdS[i * LP + ty + 16 * r];
                }
#pragma unroll
                for (int q = 0; q < NG; ++q) {
                    const int f = tx + 16 * q;
                    if (NG * 16 * 4 == D || f < D / 4) {
                        const float4 o = *reinterpret_cast<const float4*>(sdO + i * LD + 4 * f);
                        const float4 x = *reinterpret_cast<const float4*>(sQ + i * LD + 4 * f);
#pragma unroll
                        for (int r = 0; r < TC; ++r) {
                            accV[r][q][0] = fmaf(pk[r], o.x, accV[r][q][0]);
                            accV[r][q][1] = fmaf(pk[r], o.y, accV[r][q][1]);
                            accV[r][q][2] = fmaf(pk[r], o.z, accV[r][q][2]);
                            accV[r][q][3] = fmaf(pk[r], o.w, accV[r][q][3]);
                            accK[r][q][0] = fmaf(dk[r], x.x, accK[r][q][0]);
                            accK[r][q][1] = fmaf(dk[r], x.y, accK[r][q][1]);
                            accK[r][q][2] = fmaf(dk[r], x.z, accK[r][q][2]);
                            accK[r][q][3] = fmaf(dk[r], x.w, accK[r][q][3]);
                        }
                    }
                }
            }
            // ---- dQacc += dS K (query rows ty + 16r, column groups tx + 16q)
            if (dqacc != nullptr) {
                float accQ[TR][NG][4];
#pragma unroll
                for (int r = 0; r < TR; ++r)
#pragma unroll
                    for (int q = 0; q < NG; ++q)
#pragma unroll
                        for (int u = 0; u < 4; ++u) accQ[r][q][u] = 0.f;
#pragma unroll 2
                for (int jj = 0; jj < BN; ++jj) {
                    float ds[TR];
#pragma unroll
                    for (int r = 0; r < TR; ++r) ds[r] = sdS[(ty + 16 * r) * LP + jj];
#pragma unroll
                    for (int q = 0; q < NG; ++q) {
                        const int f = tx + 16 * q;
                        if (NG * 16 * 4 == D || f < D / 4) {
                            const float4 kv = *reinterpret_cast<const float4*>(sK + jj * LD + 4 * f);
#pragma unroll
                            for (int r = 0; r < TR; ++r) {
                                accQ[r][q][0] = fmaf(ds[r], kv.x, accQ[r][q][0]);
                                accQ[r][q][1] = fmaf(ds[r], kv.y, accQ[r][q][1]);
                                accQ[r][q][2] = fmaf(ds[r], kv.z, accQ[r][q][2]);
                                accQ[r][q][3] = fmaf(ds[r], kv.w, accQ[r][q][3]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < TR; ++r) {
                    const int ri = ty + 16 * r;
                    if (ri < rows) {
#pragma unroll
                        for (int q = 0; q < NG; ++q) {
                            const int f = tx + 16 * q;
                            if (NG * 16 * 4 == D || f < D / 4)
                                ptx::red_add_v4(dqacc + ((size_t)bh * s.S_q + m0 + ri) * D + 4 * f, accQ[r][q][0],
                                                accQ[r][q][1], accQ[r][q][2], accQ[r][q][3]);
                        }
                    }
                }
            }
        }
    }
    // ---- dK (scaled) and dV rows of this tile (added into the zeroed fp32 outputs when split)
#pragma unroll
    for (int r = 0; r < TC; ++r) {
        const int j = n0 + ty + 16 * r;
        if (j >= s.S_k) continue;
#pragma unroll
        for (int q = 0; q < NG; ++q) {
            const int f = tx + 16 * q;
            if (!(NG * 16 * 4 == D || f < D / 4)) continue;
            T* pv = dV + ((size_t)bkv * s.S_k + j) * D + 4 * f;
            T* pk = dK + ((size_t)bkv * s.S_k + j) * D + 4 * f;
            if constexpr (sizeof(T) == 4) {
                if (split > 1) {
                    ptx::red_add_v4(reinterpret_cast<float*>(pv), accV[r][q][0], accV[r][q][1], accV[r][q][2],
                                    accV[r][q][3]);
                    ptx::red_add_v4(reinterpret_cast<float*>(pk), accK[r][q][0] * s.scale, accK[r][q][1] * s.scale,
                                    accK[r][q][2] * s.scale, accK[r][q][3] * s.scale);
                    continue;
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                pv[u] = TypeTraits<T>::from_f32(accV[r][q][u]);
                pk[u] = TypeTraits<T>::from_f32(accK[r][q][u] * s.scale);
            }
        }
    }
}

// Deterministic dQ on CUDA cores: one CTA per (kDqRows-row query block, query head) forms
//   dQacc_i = sum_j dS_ij K_j,  dS_ij = P_ij (<dO_i, V_j> - D_i),  P_ij = exp(scale <Q_i, K_j> - LSE_i)
// itself, visiting the visible keys in increasing index order, so every row is one fixed
// sequence of fp32 additions (no atomics).  S and dP are recomputed from Q, K, V, dO.
constexpr int kDqRows = 16;  // query rows per CTA
constexpr int kDqKeys = 32;  // keys per step
constexpr int kDqThreads = 128;

template <typename T, int D>
__global__ void __launch_bounds__(kDqThreads) dq_simt_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
    const T* __restrict__ dO, const float* __restrict__ lse2, const float* __restrict__ Dws,
    float* __restrict__ dqacc, Shape s) {
    extern __shared__ float smem[];
    float* sQ = smem;                     // [kDqRows][D]
    float* sdO = sQ + kDqRows * D;        // [kDqRows][D]
    float* sK = sdO + kDqRows * D;        // [kDqKeys][D]
    float* sV = sK + kDqKeys * D;         // [kDqKeys][D]
    float* sdS = sV + kDqKeys * D;        // [kDqRows][kDqKeys]
    constexpr int kPerThread = kDqRows * D / kDqThreads;  // dQ elements a thread accumulates
    static_assert(kPerThread * kDqThreads == kDqRows * D, "thread split of the dQ block");

    const int tid = threadIdx.x;
    const int m0 = blockIdx.x * kDqRows;
    const int bh = blockIdx.y;
    const int b = bh / s.H, h = bh % s.H;
    const int bkv = b * s.H_kv + h / (s.H / s.H_kv);
    const int off = s.S_k - s.S_q;
    const float kLog2e = 1.4426950408889634f;
    const int rows = min(kDqRows, s.S_q - m0);

    for (int e = tid; e < kDqRows * D; e += kDqThreads) {
        const int r = e / D, c = e % D;
        const size_t gi = ((size_t)bh * s.S_q + m0 + r) * D + c;
        sQ[e] = r < rows ? TypeTraits<T>::to_f32(Q[gi]) : 0.f;
        sdO[e] = r < rows ? TypeTraits<T>::to_f32(dO[gi]) : 0.f;
    }
    // thread tid owns block elements e = tid + a * kDqThreads: row e / D, column e % D
    float acc[kPerThread];
#pragma unroll
    for (int a = 0; a < kPerThread; ++a) acc[a] = 0.f;

    int k_lo, k_hi;
    key_range(s, m0, m0 + rows, k_lo, k_hi);
    for (int n0 = k_lo - k_lo % kDqKeys; n0 < k_hi; n0 += kDqKeys) {
        __syncthreads();  // previous step's sK / sdS reads are done
        for (int e = tid; e < kDqKeys * D; e += kDqThreads) {
            const int j = n0 + e / D;
            const size_t gi = ((size_t)bkv * s.S_k + j) * D + e % D;
            sK[e] = j < s.S_k ? TypeTraits<T>::to_f32(K[gi]) : 0.f;
            sV[e] = j < s.S_k ? TypeTraits<T>::to_f32(V[gi]) : 0.f;
        }
        __syncthreads();
        for (int pr = tid; pr < kDqRows * kDqKeys; pr += kDqThreads) {
            const int r = pr / kDqKeys, jj = pr % kDqKeys;
            const int i = m0 + r, j = n0 + jj;
            float ds = 0.f;
            if (r < rows && j < s.S_k && key_visible(i + off, j, s.causal, s.window)) {
                float sc = 0.f, dp = 0.f;
                for (int c = 0; c < D; ++c) {
                    sc = fmaf(sQ[r * D + c], sK[jj * D + c], sc);
                    dp = fmaf(sdO[r * D + c], sV[jj * D + c], dp);
                }
                const size_t row = (size_t)bh * s.S_q_pad + i;
                const float p = exp2f(fmaf(sc, s.scale * kLog2e, -lse2[row]));
                ds = p * (dp - Dws[row]);
            }
            sdS[pr] = ds;
        }
        __syncthreads();
#pragma unroll
        for (int a = 0; a < kPerThread; ++a) {
            const int e = tid + a * kDqThreads, r = e / D, c = e % D;
            for (int jj = 0; jj < kDqKeys; ++jj) acc[a] = fmaf(sdS[r * kDqKeys + jj], sK[jj * D + c], acc[a]);
        }
    }
#pragma unroll
    for (int a = 0; a < kPerThread; ++a) {
        const int e = tid + a * kDqThreads, r = e / D, c = e % D;
        if (r < rows) dqacc[((size_t)bh * s.S_q + m0 + r) * D + c] = acc[a];
    }
}

template <typename T, int D>
cudaError_t launch_t(const void* Q, const void* K, const void* V, const void* dO,
                     const Workspace& ws, void* dK, void* dV, const Shape& s, bool skip_dq,
                     cudaStream_t st) {
    using C = SCfg<D>;
    auto kern = bwd_simt_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    // fp32 outputs: two CTAs per key tile when the grid would not fill the SMs or its heaviest
    // causal CTA outlasts the per-SM share (in both modes, so that dK and dV do not depend on
    // the mode: two partial sums added onto zero give the same bits in either order)
    int split = 1;
    if (sizeof(T) == 4) {
        const long ctas = (long)((s.S_k + C::BN - 1) / C::BN) * s.B * s.H_kv;
        static int sms = 0;
        if (sms == 0) {
            int dev = 0;
            if (cudaGetDevice(&dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
                sms = 148;
        }
        if (ctas < sms || key_tile_split(s, C::BN, C::BM) == 2) split = 2;
    }
    if (split > 1) {
        const size_t bytes = (size_t)s.B * s.H_kv * s.S_k * D * sizeof(T);
        if ((e = cudaMemsetAsync(dK, 0, bytes, st)) != cudaSuccess) return e;
        if ((e = cudaMemsetAsync(dV, 0, bytes, st)) != cudaSuccess) return e;
    }
    const long grid = (long)((s.S_k + C::BN - 1) / C::BN) * s.B * s.H_kv * split;
    kern<<<(unsigned)grid, kThreads, C::SMEM, st>>>(static_cast<const T*>(Q), static_cast<const T*>(K),
                                                    static_cast<const T*>(V), static_cast<const T*>(dO),
                                                    ws.lse2, ws.Dws, skip_dq ? nullptr : ws.dqacc,
                                                    static_cast<T*>(dK), static_cast<T*>(dV), s, split);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_dq_t(const void* Q, const void* K, const void* V, const void* dO, const Workspace& ws,
                        const Shape& s, cudaStream_t st) {
    const size_t smem = sizeof(float) * (2 * kDqRows * D + 2 * kDqKeys * D + kDqRows * kDqKeys);
    auto kern = dq_simt_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((s.S_q + kDqRows - 1) / kDqRows, s.B * s.H);
    kern<<<grid, kDqThreads, smem, st>>>(static_cast<const T*>(Q), static_cast<const T*>(K),
                                         static_cast<const T*>(V), static_cast<const T*>(dO), ws.lse2, ws.Dws,
                                         ws.dqacc, s);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dq_simt(int dtype, const void* Q, const void* K, const void* V, const void* dO,
                           const Workspace& ws, const Shape& s, cudaStream_t st) {
#define FA_L(T, DD) return launch_dq_t<T, DD>(Q, K, V, dO, ws, s, st)
    FA_DISPATCH_HEAD_DIM(dtype, s.d, FA_L);
#undef FA_L
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_simt(int dtype, const void* Q, const void* K, const void* V,
                            const void* dO, const Workspace& ws, void* dK, void* dV,
                            const Shape& s, bool skip_dq, cudaStream_t st) {
#define FA_L(T, DD) return launch_t<T, DD>(Q, K, V, dO, ws, dK, dV, s, skip_dq, st)
    FA_DISPATCH_HEAD_DIM(dtype, s.d, FA_L);
#undef FA_L
    return cudaErrorInvalidValue;
}

}  // namespace fa
