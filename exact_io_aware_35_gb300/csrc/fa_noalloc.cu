// fa_noalloc.cu -- fa_bwd_noalloc: the backward pass for callers that cannot
// allocate device memory.
//
// fa_bwd needs a caller-supplied workspace for D (one fp32 per query row and
// head).  Some callers have no way to get one: a plug-in running inside a host
// application that owns every device allocation, or a loop that must never
// call cudaMalloc mid-step (an allocation can stall or fail there).  This
// entry point keeps D in a fixed array compiled into the library instead, so
// the caller passes only its inputs and outputs.
#include <mutex>
#include <stdio.h>

#include "fa.h"
#include "fa_internal.h"

namespace fa {

// Capacity of the built-in D scratch: B * H * N rows, 4 bytes each (8 MiB).
// Every GPU that loads the library keeps this array until the process exits.
constexpr long long kNoallocMaxRows = 1LL << 21;

namespace {

// The scratch itself.  In host code this name is only a stand-in for the
// symbol, not a device address: the device address is fetched with
// cudaGetSymbolAddress below, once per device.
static __device__ __align__(256) float g_noalloc_dsum[kNoallocMaxRows];

constexpr int kMaxDev = 64;
float* g_noalloc_ptr[kMaxDev] = {};
std::mutex g_noalloc_mu;

// Device address of the scratch on the current device, looked up on the first
// call made on that device.
fa_status noalloc_scratch(float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_dsum) != cudaSuccess || !p) return FA_ERR_CUDA;
        g_noalloc_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                    const void* dout, const float* lse, void* dq, void* dk,
                                    void* dv, const void* o_lo, int B, int H, int Hkv, int N,
                                    int d, int causal, float scale, void* stream) {
    if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
    const long long rows = static_cast<long long>(B) * H * N;
    if (rows > fa::kNoallocMaxRows) {
        fprintf(stderr,
                "fa_bwd_noalloc: B*H*N = %lld exceeds the built-in scratch of %lld rows; "
                "use fa_bwd with a workspace\n",
                rows, fa::kNoallocMaxRows);
        return FA_ERR_INVALID_ARG;
    }
    float* scratch = nullptr;
    const fa_status st = fa::noalloc_scratch(&scratch);
    if (st != FA_OK) return st;
    // D needs no clearing: the first stage writes every entry the later two read.
    // No fp16 operand copies (they would need B*N*(2H + 2Hkv)*d*2 more bytes):
    // the bf16 operand path.
    return fa::bwd_run(FA_BWD_DSUM | FA_BWD_DKDV | FA_BWD_DQ, q, k, v, o, dout, lse, dq, dk, dv,
                       scratch, nullptr, o_lo, B, H, Hkv, N, d, causal, scale, stream);
}
