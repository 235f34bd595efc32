// fa_bwd.cu -- exact attention backward for sm_103a (tcgen05 + TMEM + TMA).
//
// The pages say only that the backward pass recomputes the attention matrix
// from Q, K, V and the stored row statistics instead of reading a stored P
// ("FlashAttention Kernel", the recomputation bullets; "FlashAttention", the
// recomputation paragraph).  The gradients themselves are the derivative of
// O = softmax(scale Q K^T) V for a loss with dL/dO = dO:
//     P_ij = exp(scale q_i.k_j - lse_i)          (recomputed, never stored)
//     dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic = sum_j P_ij dP_ij
//     dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q
// summed over the query heads of a GQA group for dK and dV.
//
// Three kernels on the caller's stream, no atomics (every output element is
// owned by one CTA, so results are bitwise reproducible):
//   1. dsum (this file): D = rowsum(dO o O) in fp32, HBM-bound (on the fp16
//      operand path it also writes the fp16 copy of dO).
//   2. dK, dV (fa_bwd_dkdv.cu): one CTA per (batch, kv head, 128-key block).
//   3. dQ (fa_bwd_dq.cu): one CTA per (batch, q head, 128-query block).
#include "fa_bwd_common.cuh"

namespace fa {
namespace {

using namespace bwd;

// D_i = sum_c dO_ic * O_ic.  d/8 threads per row, 8 bf16 (16 bytes) each,
// reduced with shuffles.  o_lo (optional) is the low bf16 half of O written by
// the training forward; D then uses o + o_lo, i.e. O to about 16 significant
// bits.
// F16 (fp16 operand path, fused with the copy of dout): the thread also
// writes its 8 elements of dout16 = fp16(dout * 2^s), s from the maxima an
// earlier kernel left in absmax, and one thread writes the scales.
template <bool F16>
__global__ void __launch_bounds__(256) fa_bwd_dsum_kernel(const uint16_t* __restrict__ o,
                                                          const uint16_t* __restrict__ o_lo,
                                                          const uint16_t* __restrict__ dout,
                                                          float* __restrict__ dsum, int B, int N,
                                                          int Hq, int d,
                                                          uint16_t* __restrict__ dout16,
                                                          const uint32_t* __restrict__ absmax,
                                                          F16Scales* __restrict__ scales_w) {
    const int tpr = d >> 3;
    const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long rows = static_cast<long long>(B) * N * Hq;
    const long long row = gid / tpr;
    const int part = static_cast<int>(gid % tpr);
    float acc = 0.f;
    float mul = 1.f;
    if (F16) {
        const F16Scales sc = f16_scales_from(absmax, d);
        if (gid == 0) *scales_w = sc;
        mul = pow2f(sc.dout);
    }
    if (row < rows) {
        const uint4 x = *reinterpret_cast<const uint4*>(o + row * d + part * 8);
        const uint4 g = *reinterpret_cast<const uint4*>(dout + row * d + part * 8);
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
        const uint32_t gs[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc = fmaf(bf16lo(xs[i]), bf16lo(gs[i]), acc);
            acc = fmaf(bf16hi(xs[i]), bf16hi(gs[i]), acc);
        }
        if (F16) {
            uint32_t h[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) h[i] = pack_f16(bf16lo(gs[i]) * mul, bf16hi(gs[i]) * mul);
            *reinterpret_cast<uint4*>(dout16 + row * d + part * 8) = make_uint4(h[0], h[1], h[2], h[3]);
        }
        if (o_lo) {
            const uint4 y = *reinterpret_cast<const uint4*>(o_lo + row * d + part * 8);
            const uint32_t ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc = fmaf(bf16lo(ys[i]), bf16lo(gs[i]), acc);
                acc = fmaf(bf16hi(ys[i]), bf16hi(gs[i]), acc);
            }
        }
    }
    // tpr is 8 or 16 and divides 32, so a row's threads sit in one warp
    for (int m = tpr >> 1; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (row < rows && part == 0) {
        const int h = static_cast<int>(row % Hq);
        const long long bn = row / Hq;
        const int n = static_cast<int>(bn % N);
        const int b = static_cast<int>(bn / N);
        dsum[(static_cast<long long>(b) * Hq + h) * N + n] = acc;
    }
}

template <int D>
cudaError_t launch_bwd_d(const BwdMaps& m, const BwdArgs& a, int stages, cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    if (stages & 1) {  // D = rowsum(dO o O)
        const long long threads = static_cast<long long>(a.B) * a.N * a.Hq * (D / 8);
        const long long blocks = (threads + 255) / 256;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        if (a.dout16)
            fa_bwd_dsum_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
                a.o, a.o_lo, a.dout, a.dsum, a.B, a.N, a.Hq, D, a.dout16, a.absmax, a.scales_w);
        else
            fa_bwd_dsum_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
                a.o, a.o_lo, a.dout, a.dsum, a.B, a.N, a.Hq, D, nullptr, nullptr, nullptr);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (stages & 2)
        if ((e = launch_bwd_dkdv<D>(m, a, st)) != cudaSuccess) return e;
    if (stages & 4)
        if ((e = launch_bwd_dq<D>(m, a, st)) != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd(const BwdMaps& maps, const BwdArgs& args, int stages, cudaStream_t stream) {
    if (args.d == 64) return launch_bwd_d<64>(maps, args, stages, stream);
    if (args.d == 128) return launch_bwd_d<128>(maps, args, stages, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa
