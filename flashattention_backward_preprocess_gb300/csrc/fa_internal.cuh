// fa_internal.cuh -- shared definitions of the CUDA library (not part of the
// C ABI).  Element-type helpers, the workspace view the launchers receive and
// the launcher prototypes each .cu file implements.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "error_words.h"
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
    int window;   // sliding-window size, 0 = none
    int S_q_pad;  // S_q rounded up to the main kernel's query tile (128)
};

// Visibility of key j to query i.  Query i sits at key position p = i + S_k - S_q
// (bottom-right alignment).  Causal hides keys after p.  A sliding window w > 0
// (boostr autograd_attention.rs, window_size of FlashAttentionConfig; 0 = none)
// hides keys w or more positions before p and, when not causal, w or more after.
__host__ __device__ __forceinline__ bool key_visible(int p, int j, int causal, int window) {
    if (causal && j > p) return false;
    if (window > 0 && (p - j >= window || (!causal && j - p >= window))) return false;
    return true;
}

// The same test for a run of positions, as one interval (kernels compare each element
// against it with a single unsigned comparison; kOpen stands for "no bound").
constexpr int kOpen = 1 << 29;

// Offsets q whose query (key position base + q) sees key j = base + dj: q in [lo, hi).
__host__ __device__ __forceinline__ void visible_queries(int dj, int causal, int window, int& lo, int& hi) {
    lo = causal ? dj : (window > 0 ? dj - window + 1 : -kOpen);
    hi = window > 0 ? dj + window : kOpen;
}

// Offsets c whose key (base + c) the query at key position base + dp sees: c in [lo, hi).
__host__ __device__ __forceinline__ void visible_keys(int dp, int causal, int window, int& lo, int& hi) {
    lo = window > 0 ? dp - window + 1 : -kOpen;
    hi = causal ? dp + 1 : (window > 0 ? dp + window : kOpen);
}

// Query rows [lo, hi) that see at least one key of [j0, j1) (j0 < j1 <= S_k);
// empty when hi <= lo.  Exact for a band: the first such row sees key j0 or is
// the first past the causal edge, the last one sees key j1 - 1.
__host__ __device__ __forceinline__ void query_range(const Shape& s, int j0, int j1, int& lo, int& hi) {
    const int off = s.S_k - s.S_q;
    lo = 0;
    hi = s.S_q;
    if (s.causal) lo = j0 - off > lo ? j0 - off : lo;  // p >= j0
    if (s.window > 0) {
        const int h = j1 - 1 + s.window - off;  // p - (j1 - 1) < w
        hi = h < hi ? h : hi;
        if (!s.causal) lo = j0 - s.window + 1 - off > lo ? j0 - s.window + 1 - off : lo;  // j0 - p < w
    }
}

// Key columns [lo, hi) visible to at least one query row of [i0, i1) (i0 < i1 <= S_q);
// empty when hi <= lo.
__host__ __device__ __forceinline__ void key_range(const Shape& s, int i0, int i1, int& lo, int& hi) {
    const int off = s.S_k - s.S_q;
    lo = 0;
    hi = s.S_k;
    if (s.causal) hi = i1 + off < hi ? i1 + off : hi;  // j <= p of the last row
    if (s.window > 0) {
        lo = i0 + off - s.window + 1 > lo ? i0 + off - s.window + 1 : lo;  // p_first - j < w
        if (!s.causal) hi = i1 - 1 + off + s.window < hi ? i1 - 1 + off + s.window : hi;  // j - p_last < w
    }
}

// Head dims the library takes.  The CUDA-core kernels and the preprocess are instantiated
// for each; the tensor-core kernels run d = 32 and 96 as d = 64 and 128 with the missing
// columns zero-filled by TMA (their global extents and strides stay d); at d = 256 the
// forward has a tensor-core instance of its own and the backward a kernel of its own
// (bwd_d256.cu).
#define FA_FOR_DTYPE(dtype, DD, CALL)              \
    do {                                           \
        if ((dtype) == FA_F32) CALL(float, DD);    \
        if ((dtype) == FA_F16) CALL(__half, DD);   \
        if ((dtype) == FA_BF16) CALL(__nv_bfloat16, DD); \
    } while (0)
#define FA_DISPATCH_HEAD_DIM(dtype, d, CALL)                      \
    do {                                                          \
        switch (d) {                                              \
            case 32: FA_FOR_DTYPE(dtype, 32, CALL); break;        \
            case 64: FA_FOR_DTYPE(dtype, 64, CALL); break;        \
            case 96: FA_FOR_DTYPE(dtype, 96, CALL); break;        \
            case 128: FA_FOR_DTYPE(dtype, 128, CALL); break;      \
            case 256: FA_FOR_DTYPE(dtype, 256, CALL); break;      \
            default: break;                                       \
        }                                                         \
    } while (0)
inline bool head_dim_supported(int d) { return d == 32 || d == 64 || d == 96 || d == 128 || d == 256; }
// The tensor-core backward's compiled head dim for a call's d (0: none, CUDA cores instead);
// the forward adds d = 256.
inline int tc_head_dim(int d) { return d == 32 || d == 64 ? 64 : (d == 96 || d == 128 ? 128 : 0); }

// Library-owned scratch for one fa_bwd call (device memory).
struct Workspace {
    unsigned int* err;  // [4] error words
    float* lse2;        // [B*H][S_q_pad] LSE * log2(e), +inf on padding / empty rows
    float* Dws;         // [B*H][S_q_pad] D = rowsum(dO * O), 0 on padding
    float* dqacc;       // [B*H][S_q][d] fp32 dQ accumulator (unscaled)
    // [B*H][ceil(S_q / 128)] turn counters of the deterministic dQ reduction (zeroed per
    // call), or nullptr: then dQ tiles are reduced in whatever order the CTAs reach them
    unsigned int* dq_sem;
    // deterministic dQ: the counter (zeroed with dq_sem) from which the CTAs take their
    // logical indices in start order; nullptr otherwise
    unsigned int* dq_ticket;
};

constexpr int kTileQ = 128;  // query rows per main-kernel iteration
constexpr int kTileK = 128;  // key rows per main-kernel CTA

// preprocess.cu
cudaError_t launch_preprocess(int dtype, const void* dO, const void* O, const float* LSE,
                              float* D, float* lse2, float* dqacc, const Shape& s,
                              int rows_stride, cudaStream_t st);
cudaError_t launch_dq_finalize(int dtype, const float* dqacc, void* dQ, const Shape& s,
                               cudaStream_t st);
// bwd_simt.cu (fp32 path).  skip_dq: leave the dQ accumulator alone (launch_dq_simt fills it).
cudaError_t launch_bwd_simt(int dtype, const void* Q, const void* K, const void* V,
                            const void* dO, const Workspace& ws, void* dK, void* dV,
                            const Shape& s, bool skip_dq, cudaStream_t st);
// Deterministic dQ accumulator rows on CUDA cores (each row summed over keys in index order).
cudaError_t launch_dq_simt(int dtype, const void* Q, const void* K, const void* V, const void* dO,
                           const Workspace& ws, const Shape& s, cudaStream_t st);
// fwd_simt.cu
cudaError_t launch_fwd_simt(int dtype, const void* Q, const void* K, const void* V, void* O,
                            float* LSE, const Shape& s, cudaStream_t st);
// bwd_d256.cu (tcgen05 path for f16 / bf16 at head dim 256; skip_dq: dK, dV only)
cudaError_t launch_bwd_d256(int dtype, const void* Q, const void* K, const void* V, const void* dO,
                            const Workspace& ws, void* dK, void* dV, const Shape& s, bool skip_dq,
                            cudaStream_t st);
// bwd_sm103.cu (tcgen05 path for f16 / bf16)
cudaError_t launch_bwd_sm103(int dtype, const void* Q, const void* K, const void* V,
                             const void* dO, const Workspace& ws, void* dK, void* dV,
                             const Shape& s, cudaStream_t st);

// fwd_sm103.cu (tcgen05 forward for f16 / bf16, head dim 64 or 128)
cudaError_t launch_fwd_sm103(int dtype, const void* Q, const void* K, const void* V, void* O,
                             float* LSE, unsigned int* err, const Shape& s, cudaStream_t st);
// selftest.cu
cudaError_t launch_wait_selftest(unsigned int* err, uint64_t limit_ns, cudaStream_t st);

// api.cu: CTAs per key tile for a tensor-core backward launch with bn-key CTAs walking
// bm-row query tiles: 2 (a cluster that splits each key tile's query tiles in halves) when
// the CTA with the most iterations would outlast an even share of the whole over the SMs
// (long causal problems), else 1.
int key_tile_split(const Shape& s, int bn, int bm);

// api.cu: argument checks and error text shared by the entry points.
int validate_bwd_args(const void* dO, const void* Q, const void* K, const void* V, const void* O,
                      const float* LSE, const void* dQ, const void* dK, const void* dV, int B, int H,
                      int H_kv, int S_q, int S_k, int d, float scale, int causal, int dtype);
int set_error(int status, const char* arg, const char* reason);
void clear_error();
// The main backward kernel fa_bwd runs for a dtype and head dim; every backward entry point
// picks it with this one function.  f16 / bf16 run a tcgen05 kernel (head dims up to 128, or
// the d = 256 one) unless FA_BWD_KERNEL=simt; f32 runs on CUDA cores.
enum BwdKernel { kBwdSimt = 0, kBwdSm103 = 1, kBwdD256 = 2 };
int bwd_kernel_for(int dtype, int d);

// noalloc.cu: reads the error word of the no-allocation scratch on the current device
// into *word and clears it (0 if fa_bwd_noalloc never ran on this device).  Returns an
// fa_status.
int noalloc_take_error_word(unsigned int* word);

}  // namespace fa
