// noalloc.cu -- fa_bwd_noalloc: the full backward (preprocess, main kernel,
// dQ finalise) for callers that must not allocate device memory.
//
// fa_bwd keeps its scratch (fp32 dQ accumulator, D, padded LSE copy, error
// words) in a workspace it allocates with cudaMalloc on first use.  Some
// callers cannot allow that: code running under a memory pool or allocator
// that owns all device memory, hosts whose allocation calls would
// synchronize the device at a bad moment, or runtimes that forbid the library
// from allocating on its own.  This entry point instead uses one fixed
// scratch array compiled into the library (g_fa_noalloc_scratch below), so a
// call only launches kernels.
//
// Rules for users:
//   * The array is kFaNoallocScratchBytes (32 MiB) on every GPU that loads the
//     library, held until the process exits.  A shape needs
//       256 + 2 * 4 * B*H*ceil(S_q/128)*128 + 4 * B*H*S_q*d   bytes
//     (each part rounded up to 256); larger shapes are rejected with
//     FA_ERR_INVALID_ARG ("scratch: ...") and nothing is launched.
//   * The first call on a device looks up the array's device address
//     (cudaGetSymbolAddress, which may load the library's device code) and
//     enqueues the clearing of its error words on the caller's stream; make
//     that first call before any stream capture.
//   * All calls share the one array and it keeps the last call's contents;
//     every call re-zeroes the parts that must start at zero.  Calls whose GPU
//     work overlaps (other streams, other host threads) race on it: order them
//     on one stream.
//   * Device-side bounded-wait timeouts of this variant are recorded in the
//     array's first word; fa_check_device reads and clears it (after
//     synchronizing the stream it is given, so pass the stream of the calls).
//   * The main kernel is chosen as fa_bwd chooses it (FA_BWD_KERNEL=simt
//     included).
#include <stdio.h>

#include <mutex>

#include "fa_internal.cuh"

namespace {
constexpr size_t kFaNoallocScratchBytes = 32u << 20;
constexpr int kFaMaxDevices = 64;
}  // namespace

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol: never pass it to a kernel, use the address looked up below.
static __device__ __align__(256) unsigned char g_fa_noalloc_scratch[kFaNoallocScratchBytes];

namespace fa {
namespace {

std::mutex g_na_mu;
void* g_na_ptr[kFaMaxDevices] = {};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Device address of the scratch array on the current device (set-up once per device: the
// address lookup, then the clearing of the error words enqueued on `st`; the address is
// published only once that clear is enqueued, so every later call finds clean words).
int scratch_address(cudaStream_t st, void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(FA_ERR_CUDA, "cudaGetDevice", cudaGetErrorString(e));
    if (dev < 0 || dev >= kFaMaxDevices) return set_error(FA_ERR_UNSUPPORTED, "device", "device index too large");
    std::lock_guard<std::mutex> lk(g_na_mu);
    if (g_na_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fa_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return set_error(FA_ERR_CUDA, "cudaGetSymbolAddress", cudaGetErrorString(e));
        e = cudaMemsetAsync(p, 0, 256, st);  // error words
        if (e != cudaSuccess) return set_error(FA_ERR_CUDA, "cudaMemsetAsync", cudaGetErrorString(e));
        g_na_ptr[dev] = p;
    }
    *out = g_na_ptr[dev];
    return FA_OK;
}

}  // namespace

int noalloc_take_error_word(unsigned int* word) {
    *word = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(FA_ERR_CUDA, "cudaGetDevice", cudaGetErrorString(e));
    if (dev < 0 || dev >= kFaMaxDevices) return FA_OK;
    std::lock_guard<std::mutex> lk(g_na_mu);
    if (g_na_ptr[dev] == nullptr) return FA_OK;  // never used on this device
    e = cudaMemcpy(word, g_na_ptr[dev], sizeof(unsigned int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return set_error(FA_ERR_CUDA, "cudaMemcpy", cudaGetErrorString(e));
    if (*word != 0) {
        e = cudaMemset(g_na_ptr[dev], 0, sizeof(unsigned int));
        if (e != cudaSuccess) return set_error(FA_ERR_CUDA, "cudaMemset", cudaGetErrorString(e));
    }
    return FA_OK;
}

}  // namespace fa

using namespace fa;

extern "C" int fa_bwd_noalloc(const void* dO, const void* Q, const void* K, const void* V,
                              const void* O, const float* LSE, void* dQ, void* dK, void* dV, int B,
                              int H, int H_kv, int S_q, int S_k, int d, float scale, int causal,
                              int dtype, void* stream) {
    clear_error();
    int rc = validate_bwd_args(dO, Q, K, V, O, LSE, dQ, dK, dV, B, H, H_kv, S_q, S_k, d, scale, causal,
                               dtype);
    if (rc != FA_OK) return rc;
    const int S_q_pad = (S_q + kTileQ - 1) / kTileQ * kTileQ;
    const size_t rows_pad = (size_t)B * H * S_q_pad;
    const size_t off_lse2 = 256;
    const size_t off_D = off_lse2 + up256(rows_pad * 4);
    const size_t off_dq = off_D + up256(rows_pad * 4);
    const size_t total = off_dq + up256((size_t)B * H * S_q * d * 4);
    if (total > kFaNoallocScratchBytes) {
        char msg[160];
        snprintf(msg, sizeof msg, "this shape needs %zu bytes of scratch, fa_bwd_noalloc has %zu (use fa_bwd)",
                 total, kFaNoallocScratchBytes);
        return set_error(FA_ERR_INVALID_ARG, "scratch", msg);
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void* base = nullptr;
    if ((rc = scratch_address(st, &base)) != FA_OK) return rc;
    char* b = static_cast<char*>(base);
    Workspace ws;
    ws.err = reinterpret_cast<unsigned int*>(b);
    ws.lse2 = reinterpret_cast<float*>(b + off_lse2);
    ws.Dws = reinterpret_cast<float*>(b + off_D);
    ws.dqacc = reinterpret_cast<float*>(b + off_dq);
    ws.dq_sem = nullptr;
    ws.dq_ticket = nullptr;
    Shape s;
    s.B = B;
    s.H = H;
    s.H_kv = H_kv;
    s.S_q = S_q;
    s.S_k = S_k;
    s.d = d;
    s.scale = scale;
    s.causal = causal;
    s.window = 0;
    s.S_q_pad = S_q_pad;
    // the preprocess pass also zeroes the dQ accumulator rows this call uses
    cudaError_t e = launch_preprocess(dtype, dO, O, LSE, ws.Dws, ws.lse2, ws.dqacc, s, S_q_pad, st);
    if (e != cudaSuccess) return set_error(FA_ERR_CUDA, "preprocess launch", cudaGetErrorString(e));
    const int kind = bwd_kernel_for(dtype, d);
    e = kind == kBwdSm103 ? launch_bwd_sm103(dtype, Q, K, V, dO, ws, dK, dV, s, st)
        : kind == kBwdD256 ? launch_bwd_d256(dtype, Q, K, V, dO, ws, dK, dV, s, false, st)
                           : launch_bwd_simt(dtype, Q, K, V, dO, ws, dK, dV, s, false, st);
    if (e != cudaSuccess) return set_error(FA_ERR_CUDA, "main kernel launch", cudaGetErrorString(e));
    e = launch_dq_finalize(dtype, ws.dqacc, dQ, s, st);
    if (e != cudaSuccess) return set_error(FA_ERR_CUDA, "dq finalize launch", cudaGetErrorString(e));
    return FA_OK;
}
