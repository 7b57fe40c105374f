// fa_internal.cuh -- shared definitions of the CUDA library (not part of the
// C ABI).  Element-type helpers, the workspace view the launchers receive and
// the launcher prototypes each .cu file implements.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fa.h"  // include/fa.h (nvcc -I include)

namespace fa {

// Element types: float, __half, __nv_bfloat16.
template <typename T> struct TypeTraits;
template <> struct TypeTraits<float> {
    static constexpr int kId = FA_F32;
    __device__ __forceinline__ static float to_f32(float x) { return x; }
    __device__ __forceinline__ static float from_f32(float x) { return x; }
};
template <> struct TypeTraits<__half> {
    static constexpr int kId = FA_F16;
    __device__ __forceinline__ static float to_f32(__half x) { return __half2float(x); }
    __device__ __forceinline__ static __half from_f32(float x) { return __float2half_rn(x); }
};
template <> struct TypeTraits<__nv_bfloat16> {
    static constexpr int kId = FA_BF16;
    __device__ __forceinline__ static float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
    __device__ __forceinline__ static __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};

// Problem shape shared by every launcher.
struct Shape {
    int B, H, H_kv, S_q, S_k, d;
    float scale;
    int causal;
    int S_q_pad;  // S_q rounded up to the main kernel's query tile (128)
};

// Device error word codes (bit set by a kernel whose bounded wait ran out).
enum : unsigned int {
    kErrTimeout = 1u,
    kErrSmemAlign = 2u,
};

// Library-owned scratch for one fa_bwd call (device memory).
struct Workspace {
    unsigned int* err;  // [4] error words
    float* lse2;        // [B*H][S_q_pad] LSE * log2(e), +inf on padding / empty rows
    float* Dws;         // [B*H][S_q_pad] D = rowsum(dO * O), 0 on padding
    float* dqacc;       // [B*H][S_q][d] fp32 dQ accumulator (unscaled)
};

constexpr int kTileQ = 128;  // query rows per main-kernel iteration
constexpr int kTileK = 128;  // key rows per main-kernel CTA

// preprocess.cu
cudaError_t launch_preprocess(int dtype, const void* dO, const void* O, const float* LSE,
                              float* D, float* lse2, float* dqacc, const Shape& s,
                              int rows_stride, cudaStream_t st);
cudaError_t launch_dq_finalize(int dtype, const float* dqacc, void* dQ, const Shape& s,
                               cudaStream_t st);
// bwd_simt.cu (fp32 path)
cudaError_t launch_bwd_simt(int dtype, const void* Q, const void* K, const void* V,
                            const void* dO, const Workspace& ws, void* dK, void* dV,
                            const Shape& s, cudaStream_t st);
// fwd_simt.cu
cudaError_t launch_fwd_simt(int dtype, const void* Q, const void* K, const void* V, void* O,
                            float* LSE, const Shape& s, cudaStream_t st);
// bwd_sm103.cu (tcgen05 path for f16 / bf16)
cudaError_t launch_bwd_sm103(int dtype, const void* Q, const void* K, const void* V,
                             const void* dO, const Workspace& ws, void* dK, void* dV,
                             const Shape& s, cudaStream_t st);

// fwd_sm103.cu (tcgen05 forward for f16 / bf16, head dim 64 or 128)
cudaError_t launch_fwd_sm103(int dtype, const void* Q, const void* K, const void* V, void* O,
                             float* LSE, unsigned int* err, const Shape& s, cudaStream_t st);
// selftest.cu
cudaError_t launch_wait_selftest(unsigned int* err, uint64_t limit_ns, cudaStream_t st);

// api.cu: argument checks and error text shared by the entry points.
int validate_bwd_args(const void* dO, const void* Q, const void* K, const void* V, const void* O,
                      const float* LSE, const void* dQ, const void* dK, const void* dV, int B, int H,
                      int H_kv, int S_q, int S_k, int d, float scale, int causal, int dtype);
int set_error(int status, const char* arg, const char* reason);
void clear_error();

}  // namespace fa
