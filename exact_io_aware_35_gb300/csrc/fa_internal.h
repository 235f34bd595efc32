// fa_internal.h -- parameters and launchers shared by libfa's translation
// units (the C ABI in fa_api.cu, the kernels in fa_fwd.cu / fa_bwd.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fa.h"
#include "sm103_ptx.cuh"

namespace fa {

// Default bound on any single in-kernel wait (ns).  No legitimate wait comes
// within orders of magnitude of it.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// Tile sizes of the tcgen05 kernels: 128-row M tiles (one accumulator row per
// TMEM lane), 128-key tiles.
constexpr int kBM = 128;
constexpr int kBN = 128;

// Block-sparse forward: the longest mask row a thread block keeps in shared
// memory (bits), so N <= 7,168 x 128 = 917,504.
constexpr int kSparseMaxBlocks = 7168;

// fp16 operand path.  bf16 inputs are copied to fp16 after a power-of-two
// scaling (f16_scales_from), exact for all but the tiniest elements (bf16
// carries 8 significant bits, fp16 11); P, P^T (at most 2^8) and dS, dS^T
// (scaled so that the bound 2 d max|dO| max|V| lands under 2^15) are then
// rounded to fp16 instead of bf16 before they feed an MMA: 3 more bits on the
// operands whose rounding the outputs amplify.  The scalings are undone
// exactly in the kernels' epilogues (or folded into scale * log2 e).
struct F16Scales {
    int q, k, v, dout;  // x16 = fp16(x * 2^s) for the four operand tensors
    int ds;             // dS16 = fp16(dS * 2^ds)
};

// One fp16-copy job: up to four tensors (slots q, k, v, dout; n = 0 skips a
// slot).  absmax (4 words, zeroed before the job) and scales live in device
// memory.
struct F16Prep {
    const uint16_t* src[4];
    uint16_t* dst[4];
    size_t n[4];  // elements, multiples of 8
    uint32_t* absmax;
    F16Scales* scales;
    int d;
    int convert_mask;  // slots to copy (the maxima are taken for every slot with n > 0);
                       // 0: maxima only, a later kernel copies and writes the scales
};

cudaError_t launch_f16_prep(const F16Prep& p, cudaStream_t stream);

// target - ceil(log2 a) for a > 0 given as float bits, clamped to [-40, 40];
// 0 for a == 0 or a non-finite maximum (the copy then carries the inf/NaN
// just as the bf16 path would).  So max * 2^s lands in (2^(target-1),
// 2^target], and the exponent sums the kernels form stay normal powers of two.
__device__ __forceinline__ int f16_exp_to(uint32_t bits, int target) {
    if (bits == 0u || bits >= 0x7f800000u) return 0;
    const int E = static_cast<int>(bits >> 23);
    const int e = (E == 0) ? -126 : (E - 127 + ((bits & 0x7fffffu) ? 1 : 0));
    return max(-40, min(40, target - e));
}

// The scales from the maxima of q, k, v, dout (float bits).  q, k go to just
// under 2^15.  dS is bounded by 2 d max|dO| max|V| and goes under 2^15.  V
// goes under 2^4 and dO gets ds - v, so that V dO^T (fp16 copies) carries
// exactly 2^ds, the scale dS needs, with no extra multiply; that puts the
// copy of dO under 2^(12 - log2(2d)) (16 at d = 128).  A bf16 value converts
// to fp16 exactly when its exponent lies in [-17, 15], so the copies of q, k
// are exact for elements above 2^-31 of the maximum and those of v, dO above
// 2^-19 (smaller ones round at an absolute 2^-24 of the scaled values).
__device__ __forceinline__ F16Scales f16_scales_from(const uint32_t* absmax, int d) {
    F16Scales s;
    s.q = f16_exp_to(absmax[0], 15);
    s.k = f16_exp_to(absmax[1], 15);
    s.v = f16_exp_to(absmax[2], 4);
    // |dS| = |P (dP - D)| <= 2 max|dP| <= 2 d max|dO| max|V|
    const float bound = 2.f * static_cast<float>(d) * __uint_as_float(absmax[3]) *
                        __uint_as_float(absmax[2]);
    s.ds = f16_exp_to(__float_as_uint(bound), 15);
    s.dout = s.ds - s.v;
    return s;
}

struct FwdArgs {
    uint16_t* o;         // [B, N, Hq, d] bf16
    float* lse;          // [B, Hq, N]
    uint16_t* o_lo;      // [B, N, Hq, d] bf16 low half of O, or null
    const F16Scales* f16s;  // non-null: P and V enter O += P V in fp16 (V map = fp16 copy)
    uint16_t* q16;       // non-null (with f16s): the kernel writes fp16(q * 2^s.q) here
    int B, Hq, Hkv, N, g;
    int causal;
    float scale_log2;    // scale * log2(e)
    int n_qblk;          // ceil(N / 256): query blocks (two 128-row tiles each)
    int num_ctas;        // persistent CTAs to launch at most (the device's SM count)
    // block-sparse: [Hq, nb, nb] bytes (nb = ceil(N / 128)), nonzero = the
    // 128 x 128 block is computed; null: every block (up to the causal limit)
    const uint8_t* block_mask;
    Watch watch;         // status words, time limit and id of the launch
};

struct BwdArgs {
    const float* lse;    // [B, Hq, N] natural-log lse of the scaled scores
    float* dsum;         // [B, Hq, N] workspace: D_i = sum_c dO_ic O_ic
    const uint16_t* o;   // [B, N, Hq, d] bf16
    const uint16_t* dout;
    const uint16_t* o_lo;  // optional low half of O (null: D from o alone)
    const F16Scales* f16s;  // non-null: fp16 operand path (maps *16 are the fp16 copies)
    // fp16 operand path: absmax holds max|q|, max|k|, max|v|, max|dout| as float
    // bits; the dQ kernel forms the scales from it, writes them to scales_w (for
    // the dK/dV kernel) and writes dout16 = fp16(dout * 2^s) from the dout tiles
    // it loads anyway
    uint16_t* dout16;
    const uint32_t* absmax;
    F16Scales* scales_w;
    uint32_t* dout_max;  // non-null: the dsum kernel also takes max|dout| into it
    int B, Hq, Hkv, N, d, g;
    int causal;
    float scale;         // softmax scale
    float scale_log2;    // scale * log2(e)
    int num_ctas;        // persistent CTAs to launch at most (the device's SM count)
    Watch watch;         // status words, time limit and id of the launch
};

// Split-KV forward (fa_decode.cu): Nq queries of gp heads sharing a KV head
// per 128-row tile (qpt queries x gp heads), the key blocks cut into `splits`
// ranges of blocks_per_split blocks.
struct DecodeArgs {
    uint16_t* o;        // [B, Nq, Hq, d] bf16
    float* lse;         // [B, Hq, Nq]
    float* part_o;      // splits > 1: [splits, B, Hq, Nq, d] fp32 workspace
    float* part_lse;    // splits > 1: [splits, B, Hq, Nq]
    int B, Hq, Hkv, Nq, Nk, g;
    int causal;         // query i sees keys j <= i + Nk - Nq
    float scale_log2;
    int gp;             // query heads per tile
    int qpt, n_qt;      // queries per tile (128 / gp), query tiles
    int splits, blocks_per_split;
    Watch watch;         // status words, time limit and id of the launch
};

struct DecodeMaps {
    CUtensorMap q;      // box 64 x g x qpt x 1
    CUtensorMap k, v;   // box 64 x 1 x 128 x 1
};

cudaError_t launch_decode(const DecodeMaps& maps, const DecodeArgs& args, int d,
                          cudaStream_t stream);

// FP8 (e4m3) forward (fa_fp8.cu), d = 128.  q8, k8: [B, N, H, 128] bytes, one
// scale per (batch, head, 128-row block) (sq, sk: [B, H, nb]); vt8: V^T per
// head, [B, Hkv, 128, ldv] bytes (ldv = N rounded up to 16, padding zero),
// one scale per (batch, kv head) (sv: [B, Hkv]).  Element = byte * scale.
struct Fp8Args {
    // inputs of the quantisation (bf16) and its outputs
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    uint8_t* q8;
    uint8_t* k8;
    uint8_t* vt8;
    float* sq;
    float* sk;
    float* sv;
    uint32_t* vmax;     // [B, Hkv] max |v| as float bits (zeroed before the prep)
    // the forward
    uint16_t* o;        // [B, N, Hq, 128] bf16
    float* lse;         // [B, Hq, N]
    int B, Hq, Hkv, N, g, ldv, nb;
    int causal;
    int rotate;         // q, k rows multiplied by diag(signs) H_128 before quantising
    int quantize, attend;  // which of the two steps to run
    int num_ctas;       // persistent CTAs to launch at most (the device's SM count)
    float scale_log2;   // scale * log2(e), / 128 when rotated (H_128 H_128^T = 128 I)
    Watch watch;         // status words, time limit and id of the launch
};

struct Fp8Maps {
    CUtensorMap q8, k8;  // dims (128, H, N, B) bytes, box 128 x 1 x 128 x 1
    CUtensorMap vt8;     // dims (ldv, 128, Hkv, B) bytes, box 128 x 128 x 1 x 1
};

// Quantisation of q, k, v into the fp8 buffers of `args` (three kernels and a
// memset), then the forward kernel.
cudaError_t launch_fp8(const Fp8Maps& maps, const Fp8Args& args, cudaStream_t stream);

// Tensor maps of one call (all 4-D: d, H, N, B; box 64 x 1 x 128 x 1); o is
// set for the block-sparse forward only (its epilogue stores through it).
struct FwdMaps {
    CUtensorMap q, k, v, o;
};

struct BwdMaps {
    CUtensorMap q, k, v, dout, dq, dk, dv;
    CUtensorMap q16, k16, v16, dout16;  // fp16 copies (fp16 operand path only)
};

cudaError_t launch_fwd(const FwdMaps& maps, const FwdArgs& args, int d, cudaStream_t stream);
// The backward's kernels, one per file (d = 64 or 128).
template <int D>
cudaError_t launch_bwd_dkdv(const BwdMaps& maps, const BwdArgs& args, cudaStream_t stream);
template <int D>
cudaError_t launch_bwd_dq(const BwdMaps& maps, const BwdArgs& args, cudaStream_t stream);

// The backward behind fa_bwd_stage and fa_bwd_noalloc.  dsum: D workspace;
// f16_ws: a workspace laid out as fa_bwd_workspace_size describes (fp16
// operand path), or null for the bf16 path.  stages: FA_BWD_* bits.
fa_status bwd_run(int stages, const void* q, const void* k, const void* v, const void* o,
                  const void* dout, const float* lse, void* dq, void* dk, void* dv, float* dsum,
                  void* f16_ws, const void* o_lo, int B, int H, int Hkv, int N, int d, int causal,
                  float scale, void* stream);

// stages: bit 0 dsum, bit 1 dK/dV, bit 2 dQ (run in that order)
cudaError_t launch_bwd(const BwdMaps& maps, const BwdArgs& args, int stages, cudaStream_t stream);

}  // namespace fa
