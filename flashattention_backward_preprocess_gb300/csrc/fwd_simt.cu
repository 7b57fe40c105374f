// fwd_simt.cu -- attention forward helper: produces the O and LSE that the
// backward consumes (boostr autograd_attention.rs: the forward saves
// q, k, v, output and lse for FlashAttentionBackward).  Correctness helper on
// CUDA cores in fp32 with the usual online softmax over key tiles:
//   m_i  = running max of scale * <Q_i, K_j>,  l_i = sum_j exp(s_ij - m_i)
//   O_i  = sum_j exp(s_ij - m_i) V_j / l_i,     LSE_i = m_i + log(l_i)
// A row that sees no key gets O = 0 and LSE = -inf.
#include <math.h>

#include "fa_internal.cuh"

namespace fa {
namespace {

constexpr int BM = 64;        // query rows per CTA
constexpr int BN = 64;        // key rows per step
constexpr int kThreads = 256; // 16 x 16 threads, each owns a 4 x 4 block of S
constexpr int KT_LD = BN + 4; // padded row length of the transposed K tile

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(const T* __restrict__ Q,
                                                            const T* __restrict__ K,
                                                            const T* __restrict__ V,
                                                            T* __restrict__ O,
                                                            float* __restrict__ LSE, Shape s) {
    extern __shared__ float smem[];
    float* sQ = smem;              // [BM][D]
    float* sKt = sQ + BM * D;      // [D][KT_LD]   K tile transposed
    float* sV = sKt + D * KT_LD;   // [BN][D]
    float* sP = sV + BN * D;       // [BM][BN]

    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int m0 = blockIdx.x * BM;
    const int bh = blockIdx.y;
    const int b = bh / s.H, h = bh % s.H;
    const int hk = h / (s.H / s.H_kv);
    const size_t kv_base = ((size_t)b * s.H_kv + hk) * s.S_k;
    const int off = s.S_k - s.S_q;
    constexpr int CPT = D / 16;  // output columns per thread: c = tx + 16 * cc

    for (int e = tid; e < BM * D; e += kThreads) {
        const int r = e / D, c = e % D;
        const int i = m0 + r;
        sQ[e] = i < s.S_q ? TypeTraits<T>::to_f32(Q[((size_t)bh * s.S_q + i) * D + c]) : 0.f;
    }

    float m[4], l[4], acc[4][CPT];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        m[a] = -INFINITY;
        l[a] = 0.f;
#pragma unroll
        for (int cc = 0; cc < CPT; ++cc) acc[a][cc] = 0.f;
    }

    // key columns [n_lo, n_end) hold every key a row of this tile sees
    int n_lo, n_end;
    key_range(s, m0, min(m0 + BM, s.S_q), n_lo, n_end);
    for (int n0 = n_lo - n_lo % BN; n0 < n_end; n0 += BN) {
        __syncthreads();
        for (int e = tid; e < BN * D; e += kThreads) {
            const int r = e / D, c = e % D;
            const int j = n0 + r;
            const bool ok = j < s.S_k;
            sKt[c * KT_LD + r] = ok ? TypeTraits<T>::to_f32(K[(kv_base + j) * D + c]) : 0.f;
            sV[e] = ok ? TypeTraits<T>::to_f32(V[(kv_base + j) * D + c]) : 0.f;
        }
        __syncthreads();
        float sc[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) sc[a][bb] = 0.f;
        for (int c = 0; c < D; ++c) {
            const float4 k4 = *reinterpret_cast<const float4*>(sKt + c * KT_LD + tx * 4);
            const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const float qv = sQ[(ty * 4 + a) * D + c];
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) sc[a][bb] = fmaf(qv, kv[bb], sc[a][bb]);
            }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = m0 + ty * 4 + a;
            float rmax = -INFINITY;
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
                const int j = n0 + tx * 4 + bb;
                const bool vis = j < s.S_k && key_visible(i + off, j, s.causal, s.window);
                sc[a][bb] = vis ? sc[a][bb] * s.scale : -INFINITY;
                rmax = fmaxf(rmax, sc[a][bb]);
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) rmax = fmaxf(rmax, __shfl_xor_sync(0xffffffffu, rmax, o, 16));
            const float mn = fmaxf(m[a], rmax);
            const float alpha = (mn == -INFINITY) ? 1.f : expf(m[a] - mn);
            float rs = 0.f;
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
                const float p = (mn == -INFINITY) ? 0.f : expf(sc[a][bb] - mn);
                sP[(ty * 4 + a) * BN + tx * 4 + bb] = p;
                rs += p;
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o, 16);
            l[a] = l[a] * alpha + rs;
            m[a] = mn;
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) acc[a][cc] *= alpha;
        }
        __syncthreads();
        for (int j = 0; j < BN; ++j) {
            float vv[CPT];
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) vv[cc] = sV[j * D + tx + 16 * cc];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const float p = sP[(ty * 4 + a) * BN + j];
#pragma unroll
                for (int cc = 0; cc < CPT; ++cc) acc[a][cc] = fmaf(p, vv[cc], acc[a][cc]);
            }
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int i = m0 + ty * 4 + a;
        if (i >= s.S_q) continue;
        const float inv = l[a] > 0.f ? 1.f / l[a] : 0.f;
        const size_t oi = ((size_t)bh * s.S_q + i) * D;
#pragma unroll
        for (int cc = 0; cc < CPT; ++cc) O[oi + tx + 16 * cc] = TypeTraits<T>::from_f32(acc[a][cc] * inv);
        if (tx == 0) LSE[(size_t)bh * s.S_q + i] = l[a] > 0.f ? m[a] + logf(l[a]) : -INFINITY;
    }
}

template <typename T, int D>
cudaError_t launch_t(const void* Q, const void* K, const void* V, void* O, float* LSE,
                     const Shape& s, cudaStream_t st) {
    const size_t smem = sizeof(float) * (BM * D + D * KT_LD + BN * D + BM * BN);
    auto kern = fwd_simt_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((s.S_q + BM - 1) / BM, s.B * s.H);
    kern<<<grid, kThreads, smem, st>>>(static_cast<const T*>(Q), static_cast<const T*>(K),
                                       static_cast<const T*>(V), static_cast<T*>(O), LSE, s);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(int dtype, const void* Q, const void* K, const void* V, void* O,
                            float* LSE, const Shape& s, cudaStream_t st) {
#define FA_L(T, DD) return launch_t<T, DD>(Q, K, V, O, LSE, s, st)
    FA_DISPATCH_HEAD_DIM(dtype, s.d, FA_L);
#undef FA_L
    return cudaErrorInvalidValue;
}

}  // namespace fa
