// preprocess.cu -- step 1 of the FlashAttention-2 backward and the dQ
// finalisation.
//
// Step 1 (boostr flash_bwd.rs, "Step 1: Preprocessing -- compute
// D = rowsum(dO (.) O) per query position"): one fp32 dot product per query
// row.  It is HBM-bound (2 * d * sizeof(T) bytes read per row), so the kernel
// is a plain streaming row reduction: a group of LPR lanes (the row's 16-byte
// chunks rounded up to a power of two, at most 32) loads the row's chunks of
// dO and O, one or more per lane, and reduces with shuffles.
// In the fused form used by fa_bwd the same pass also
//   * writes LSE * log2(e) into a row-padded copy (so the main kernel can use
//     exp2 and read whole 128-row tiles with one bulk copy; padding rows and
//     rows that see no key get +inf, which makes their P exactly 0), and
//   * zeroes the fp32 dQ accumulator rows (flash_bwd.rs allocates dQ zeroed
//     because the main kernel adds into it atomically).
//
// dQ finalisation: dQ = scale * dQacc cast to the element type (round to
// nearest even).
#include <math.h>

#include "fa_internal.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

// Lanes per row: the row's chunk count rounded up to a power of two, at most a warp.
constexpr int lanes_per_row(int chunks) {
    int l = 1;
    while (l < chunks && l < 32) l *= 2;
    return l;
}

template <typename T, int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const T* __restrict__ dO,
                                                         const T* __restrict__ O,
                                                         const float* __restrict__ LSE,
                                                         float* __restrict__ Dout,
                                                         float* __restrict__ lse2,
                                                         float* __restrict__ dqacc, int BH,
                                                         int S_q, int rows_stride) {
    // the main kernel may start its set-up while the last blocks of this pass run (it waits
    // for this grid before it reads D, the LSE copy or the accumulator)
    ptx::griddep_launch_dependents();
    constexpr int VEC = 16 / sizeof(T);  // elements per 16-byte chunk
    constexpr int CPR = D / VEC;         // 16-byte chunks per row
    constexpr int LPR = lanes_per_row(CPR);
    static_assert(CPR * VEC == D && LPR >= 1 && LPR <= 32 && (32 % LPR) == 0, "row split");
    const long total_rows = (long)BH * rows_stride;
    const long gtid = (long)blockIdx.x * blockDim.x + threadIdx.x;
    const long row = gtid / LPR;        // padded row index (bh * rows_stride + i)
    const int lane_in_row = (int)(gtid % LPR);
    const bool in_range = row < total_rows;
    const int bh = in_range ? (int)(row / rows_stride) : 0;
    const int i = in_range ? (int)(row % rows_stride) : 0;
    const bool valid = in_range && i < S_q;

    float acc = 0.f;
    if (valid) {
#pragma unroll
        for (int ch = lane_in_row; ch < CPR; ch += LPR) {
            const size_t off = ((size_t)bh * S_q + i) * D + (size_t)ch * VEC;
            // streaming loads (evict first): dO and O are read once here
            const int4 a = __ldcs(reinterpret_cast<const int4*>(dO + off));
            const int4 b = __ldcs(reinterpret_cast<const int4*>(O + off));
            const T* ta = reinterpret_cast<const T*>(&a);
            const T* tb = reinterpret_cast<const T*>(&b);
#pragma unroll
            for (int k = 0; k < VEC; ++k)
                acc = fmaf(TypeTraits<T>::to_f32(ta[k]), TypeTraits<T>::to_f32(tb[k]), acc);
            if (dqacc != nullptr) {
                float4* z = reinterpret_cast<float4*>(dqacc + off);
#pragma unroll
                for (int k = 0; k < VEC / 4; ++k) z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    }
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, LPR);
    if (in_range && lane_in_row == 0) {
        Dout[row] = valid ? acc : 0.f;
        if (lse2 != nullptr) {
            float l = valid ? LSE[(size_t)bh * S_q + i] : -INFINITY;
            // exp2(s * scale * log2e - lse2) == exp(scale * s - LSE); a row with
            // LSE = -inf (no visible key) or a padding row must give P = 0.
            lse2[row] = (l == -INFINITY || isnan(l)) ? INFINITY : l * 1.4426950408889634f;
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(256) dq_finalize_kernel(const float* __restrict__ acc,
                                                          T* __restrict__ dQ, size_t n8,
                                                          float scale) {
    // n8 = number of 8-element groups; d is a multiple of 8 so rows never split.  Launched
    // as a programmatic dependent of the main kernel: wait until it has completed.
    ptx::griddep_wait();
    for (size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x; g < n8;
         g += (size_t)gridDim.x * blockDim.x) {
        // streaming loads and stores (evict first): the lines of the accumulator the main
        // kernel's reduce-adds left in L2 are not pushed out by the ones read from DRAM
        const float4 a = __ldcs(reinterpret_cast<const float4*>(acc) + 2 * g);
        const float4 b = __ldcs(reinterpret_cast<const float4*>(acc) + 2 * g + 1);
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        if constexpr (sizeof(T) == 4) {
            float4* o = reinterpret_cast<float4*>(dQ) + 2 * g;
            o[0] = make_float4(v[0] * scale, v[1] * scale, v[2] * scale, v[3] * scale);
            o[1] = make_float4(v[4] * scale, v[5] * scale, v[6] * scale, v[7] * scale);
        } else {
            alignas(16) T t[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) t[k] = TypeTraits<T>::from_f32(v[k] * scale);
            __stcs(reinterpret_cast<int4*>(dQ) + g, *reinterpret_cast<const int4*>(t));
        }
    }
}

template <typename T, int D>
cudaError_t launch_pre_t(const void* dO, const void* O, const float* LSE, float* Dout,
                         float* lse2, float* dqacc, const Shape& s, int rows_stride,
                         cudaStream_t st) {
    constexpr int LPR = lanes_per_row(D / (16 / (int)sizeof(T)));
    const long threads = (long)s.B * s.H * rows_stride * LPR;
    const int block = 256;
    const long grid = (threads + block - 1) / block;
    preprocess_kernel<T, D><<<(unsigned)grid, block, 0, st>>>(
        static_cast<const T*>(dO), static_cast<const T*>(O), LSE, Dout, lse2, dqacc,
        s.B * s.H, s.S_q, rows_stride);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_fin_t(const float* acc, void* dQ, const Shape& s, cudaStream_t st) {
    const size_t n8 = (size_t)s.B * s.H * s.S_q * s.d / 8;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    size_t grid = (n8 + 255) / 256;
    const size_t cap = (size_t)sms * 8;
    if (grid > cap) grid = cap;
    if (grid == 0) grid = 1;
    // programmatic dependent launch: the blocks are scheduled while the main kernel's last
    // CTAs finish and start converting as soon as it has completed
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dq_finalize_kernel<T>, acc, static_cast<T*>(dQ), n8, s.scale);
}

}  // namespace

cudaError_t launch_preprocess(int dtype, const void* dO, const void* O, const float* LSE,
                              float* D, float* lse2, float* dqacc, const Shape& s,
                              int rows_stride, cudaStream_t st) {
#define FA_PRE(T, DD) return launch_pre_t<T, DD>(dO, O, LSE, D, lse2, dqacc, s, rows_stride, st)
    FA_DISPATCH_HEAD_DIM(dtype, s.d, FA_PRE);
#undef FA_PRE
    return cudaErrorInvalidValue;
}

cudaError_t launch_dq_finalize(int dtype, const float* dqacc, void* dQ, const Shape& s,
                               cudaStream_t st) {
    if (dtype == FA_F32) return launch_fin_t<float>(dqacc, dQ, s, st);
    if (dtype == FA_F16) return launch_fin_t<__half>(dqacc, dQ, s, st);
    if (dtype == FA_BF16) return launch_fin_t<__nv_bfloat16>(dqacc, dQ, s, st);
    return cudaErrorInvalidValue;
}

}  // namespace fa
