// fa_internal.h -- parameters and launchers shared by libfa's translation
// units (the C ABI in fa_api.cu, the kernels in fa_fwd.cu / fa_bwd.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// Default bound on any single in-kernel wait (ns).  No legitimate wait comes
// within orders of magnitude of it.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// Tile sizes of the tcgen05 kernels: 128-row M tiles (one accumulator row per
// TMEM lane), 128-key tiles.
constexpr int kBM = 128;
constexpr int kBN = 128;

struct FwdArgs {
    float* lse;          // [B, Hq, N]
    uint16_t* o_lo;      // [B, N, Hq, d] bf16 low half of O, or null
    uint32_t* status;    // device status word
    int B, Hq, Hkv, N, g;
    int causal;
    float scale_log2;    // scale * log2(e)
    int n_qblk;          // ceil(N / 256): CTA query blocks (two 128-row tiles each)
    uint64_t timeout_ns;
};

struct BwdArgs {
    const float* lse;    // [B, Hq, N] natural-log lse of the scaled scores
    float* dsum;         // [B, Hq, N] workspace: D_i = sum_c dO_ic O_ic
    const uint16_t* o;   // [B, N, Hq, d] bf16
    const uint16_t* dout;
    const uint16_t* o_lo;  // optional low half of O (null: D from o alone)
    uint32_t* status;
    int B, Hq, Hkv, N, d, g;
    int causal;
    float scale;         // softmax scale
    float scale_log2;    // scale * log2(e)
    uint64_t timeout_ns;
};

// Tensor maps of one call (all 4-D: d, H, N, B; box 64 x 1 x 128 x 1).
struct FwdMaps {
    CUtensorMap q, k, v, o;
};

struct BwdMaps {
    CUtensorMap q, k, v, dout, dq, dk, dv;
};

cudaError_t launch_fwd(const FwdMaps& maps, const FwdArgs& args, int d, cudaStream_t stream);
// The backward's kernels, one per file (d = 64 or 128).
template <int D>
cudaError_t launch_bwd_dkdv(const BwdMaps& maps, const BwdArgs& args, cudaStream_t stream);
template <int D>
cudaError_t launch_bwd_dq(const BwdMaps& maps, const BwdArgs& args, cudaStream_t stream);

// stages: bit 0 dsum, bit 1 dK/dV, bit 2 dQ (run in that order)
cudaError_t launch_bwd(const BwdMaps& maps, const BwdArgs& args, int stages, cudaStream_t stream);

}  // namespace fa
