// bwd_simt.cu -- CUDA-core (FFMA) main backward kernel, used for fp32
// inputs.  fp32 needs the 1e-4 relative tolerance, which tf32 tensor-core
// operands (10-bit mantissa) would not meet, and the fp32 workloads are small,
// so this kernel favours plain, checkable arithmetic over speed.
//
// Work split (same math as the tensor-core kernel): one CTA owns a tile of
// kTile key/value rows of one (batch, kv head), keeps its dK / dV rows in
// shared memory, and walks every query row of every query head in the group:
//   S_ij = <Q_i, K_j>,  P_ij = exp(scale * S_ij - LSE_i)   (masked -> 0)
//   dP_ij = <dO_i, V_j>, dS_ij = P_ij * (dP_ij - D_i)
//   dV_j += P_ij dO_i,   dK_j += dS_ij Q_i,   dQacc_i += sum_j dS_ij K_j (atomic)
// scale is applied to dK here and to dQ in the finalisation kernel.
#include <math.h>

#include "fa_internal.cuh"

namespace fa {
namespace {

constexpr int kTile = 32;      // key rows per CTA
constexpr int kThreads = 128;  // 4 warps

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) bwd_simt_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
    const T* __restrict__ dO, const float* __restrict__ lse2, const float* __restrict__ Dws,
    float* __restrict__ dqacc, T* __restrict__ dK, T* __restrict__ dV, Shape s) {
    extern __shared__ float smem[];
    float* sK = smem;                 // [kTile][D]
    float* sV = sK + kTile * D;       // [kTile][D]
    float* sdK = sV + kTile * D;      // [kTile][D]
    float* sdV = sdK + kTile * D;     // [kTile][D]
    float* sq = sdV + kTile * D;      // [D]
    float* sdo = sq + D;              // [D]
    float* sp = sdo + D;              // [kTile]
    float* sds = sp + kTile;          // [kTile]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * kTile;
    const int bkv = blockIdx.y;  // b * H_kv + hk
    const int b = bkv / s.H_kv, hk = bkv % s.H_kv;
    const int g = s.H / s.H_kv;
    const int off = s.S_k - s.S_q;  // query i sits at key position i + off
    const float kLog2e = 1.4426950408889634f;

    for (int e = tid; e < kTile * D; e += kThreads) {
        const int j = e / D, c = e % D;
        const int jj = n0 + j;
        const size_t gi = ((size_t)bkv * s.S_k + jj) * D + c;
        sK[e] = jj < s.S_k ? TypeTraits<T>::to_f32(K[gi]) : 0.f;
        sV[e] = jj < s.S_k ? TypeTraits<T>::to_f32(V[gi]) : 0.f;
        sdK[e] = 0.f;
        sdV[e] = 0.f;
    }
    __syncthreads();

    // query rows [i_begin, i_end) see a key of this tile
    int i_begin, i_end;
    query_range(s, n0, min(n0 + kTile, s.S_k), i_begin, i_end);

    for (int h = hk * g; h < (hk + 1) * g; ++h) {
        const int bh = b * s.H + h;
        for (int i = i_begin; i < i_end; ++i) {
            const size_t qi = ((size_t)bh * s.S_q + i) * D;
            for (int c = tid; c < D; c += kThreads) {
                sq[c] = TypeTraits<T>::to_f32(Q[qi + c]);
                sdo[c] = TypeTraits<T>::to_f32(dO[qi + c]);
            }
            __syncthreads();
            const float l2 = lse2[(size_t)bh * s.S_q_pad + i];
            const float Di = Dws[(size_t)bh * s.S_q_pad + i];
            for (int r = 0; r < kTile / 4; ++r) {
                const int j = warp * (kTile / 4) + r;
                float sd = 0.f, dp = 0.f;
                for (int c = lane; c < D; c += 32) {
                    sd = fmaf(sq[c], sK[j * D + c], sd);
                    dp = fmaf(sdo[c], sV[j * D + c], dp);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    sd += __shfl_xor_sync(0xffffffffu, sd, o);
                    dp += __shfl_xor_sync(0xffffffffu, dp, o);
                }
                if (lane == 0) {
                    const int jj = n0 + j;
                    const bool vis = jj < s.S_k && key_visible(i + off, jj, s.causal, s.window);
                    // exp(scale*S - LSE) = exp2(scale*log2e*S - LSE*log2e)
                    const float p = vis ? exp2f(fmaf(sd, s.scale * kLog2e, -l2)) : 0.f;
                    sp[j] = p;
                    sds[j] = p * (dp - Di);
                }
            }
            __syncthreads();
            for (int c = tid; c < D; c += kThreads) {
                float acc = 0.f;
                const float qc = sq[c], doc = sdo[c];
#pragma unroll 8
                for (int j = 0; j < kTile; ++j) {
                    sdV[j * D + c] = fmaf(sp[j], doc, sdV[j * D + c]);
                    sdK[j * D + c] = fmaf(sds[j], qc, sdK[j * D + c]);
                    acc = fmaf(sds[j], sK[j * D + c], acc);
                }
                if (dqacc != nullptr) atomicAdd(dqacc + qi + c, acc);  // null: dQ by dq_simt_kernel
            }
            __syncthreads();
        }
    }
    for (int e = tid; e < kTile * D; e += kThreads) {
        const int j = e / D, c = e % D;
        const int jj = n0 + j;
        if (jj < s.S_k) {
            const size_t gi = ((size_t)bkv * s.S_k + jj) * D + c;
            dK[gi] = TypeTraits<T>::from_f32(sdK[e] * s.scale);
            dV[gi] = TypeTraits<T>::from_f32(sdV[e]);
        }
    }
}

// Deterministic dQ on CUDA cores: one CTA per (kDqRows-row query block, query head) forms
//   dQacc_i = sum_j dS_ij K_j,  dS_ij = P_ij (<dO_i, V_j> - D_i),  P_ij = exp(scale <Q_i, K_j> - LSE_i)
// itself, visiting the visible keys in increasing index order, so every row is one fixed
// sequence of fp32 additions (no atomics).  S and dP are recomputed from Q, K, V, dO.
constexpr int kDqRows = 16;  // query rows per CTA
constexpr int kDqKeys = 32;  // keys per step

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) dq_simt_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
    const T* __restrict__ dO, const float* __restrict__ lse2, const float* __restrict__ Dws,
    float* __restrict__ dqacc, Shape s) {
    extern __shared__ float smem[];
    float* sQ = smem;                     // [kDqRows][D]
    float* sdO = sQ + kDqRows * D;        // [kDqRows][D]
    float* sK = sdO + kDqRows * D;        // [kDqKeys][D]
    float* sV = sK + kDqKeys * D;         // [kDqKeys][D]
    float* sdS = sV + kDqKeys * D;        // [kDqRows][kDqKeys]
    constexpr int kPerThread = kDqRows * D / kThreads;  // dQ elements a thread accumulates
    static_assert(kPerThread * kThreads == kDqRows * D, "thread split of the dQ block");

    const int tid = threadIdx.x;
    const int m0 = blockIdx.x * kDqRows;
    const int bh = blockIdx.y;
    const int b = bh / s.H, h = bh % s.H;
    const int bkv = b * s.H_kv + h / (s.H / s.H_kv);
    const int off = s.S_k - s.S_q;
    const float kLog2e = 1.4426950408889634f;
    const int rows = min(kDqRows, s.S_q - m0);

    for (int e = tid; e < kDqRows * D; e += kThreads) {
        const int r = e / D, c = e % D;
        const size_t gi = ((size_t)bh * s.S_q + m0 + r) * D + c;
        sQ[e] = r < rows ? TypeTraits<T>::to_f32(Q[gi]) : 0.f;
        sdO[e] = r < rows ? TypeTraits<T>::to_f32(dO[gi]) : 0.f;
    }
    // thread tid owns block elements e = tid + a * kThreads: row e / D, column e % D
    float acc[kPerThread];
#pragma unroll
    for (int a = 0; a < kPerThread; ++a) acc[a] = 0.f;

    int k_lo, k_hi;
    key_range(s, m0, m0 + rows, k_lo, k_hi);
    for (int n0 = k_lo - k_lo % kDqKeys; n0 < k_hi; n0 += kDqKeys) {
        __syncthreads();  // previous step's sK / sdS reads are done
        for (int e = tid; e < kDqKeys * D; e += kThreads) {
            const int j = n0 + e / D;
            const size_t gi = ((size_t)bkv * s.S_k + j) * D + e % D;
            sK[e] = j < s.S_k ? TypeTraits<T>::to_f32(K[gi]) : 0.f;
            sV[e] = j < s.S_k ? TypeTraits<T>::to_f32(V[gi]) : 0.f;
        }
        __syncthreads();
        for (int pr = tid; pr < kDqRows * kDqKeys; pr += kThreads) {
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
            const int e = tid + a * kThreads, r = e / D, c = e % D;
            for (int jj = 0; jj < kDqKeys; ++jj) acc[a] = fmaf(sdS[r * kDqKeys + jj], sK[jj * D + c], acc[a]);
        }
    }
#pragma unroll
    for (int a = 0; a < kPerThread; ++a) {
        const int e = tid + a * kThreads, r = e / D, c = e % D;
        if (r < rows) dqacc[((size_t)bh * s.S_q + m0 + r) * D + c] = acc[a];
    }
}

template <typename T, int D>
cudaError_t launch_t(const void* Q, const void* K, const void* V, const void* dO,
                     const Workspace& ws, void* dK, void* dV, const Shape& s, bool skip_dq,
                     cudaStream_t st) {
    const size_t smem = sizeof(float) * (4 * kTile * D + 2 * D + 2 * kTile);
    auto kern = bwd_simt_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((s.S_k + kTile - 1) / kTile, s.B * s.H_kv);
    kern<<<grid, kThreads, smem, st>>>(static_cast<const T*>(Q), static_cast<const T*>(K),
                                       static_cast<const T*>(V), static_cast<const T*>(dO),
                                       ws.lse2, ws.Dws, skip_dq ? nullptr : ws.dqacc, static_cast<T*>(dK),
                                       static_cast<T*>(dV), s);
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
    kern<<<grid, kThreads, smem, st>>>(static_cast<const T*>(Q), static_cast<const T*>(K),
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
