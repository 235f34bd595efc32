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
//      operand path it also takes max |dO|).
//   2. dQ (fa_bwd_dq.cu): one CTA per (batch, q head, 128-query block); on
//      the fp16 operand path it also writes the fp16 copy of dO.
//   3. dK, dV (fa_bwd_dkdv.cu): one CTA per (batch, kv head, 128-key block).
#include "fa_bwd_common.cuh"

namespace fa {
namespace {

using namespace bwd;

// D_i = sum_c dO_ic * O_ic.  d/8 threads per row, 8 bf16 (16 bytes) each,
// reduced with shuffles; a grid-stride loop over (row, part) units with two
// units (six 16-byte streaming loads) in flight per thread.  o_lo (optional)
// is the low bf16 half of O written by the training forward; D then uses
// o + o_lo, i.e. O to about 16 significant bits.
// MAX (fp16 operand path): the kernel also takes max |dout| (as the bits of
// a non-negative float, which order like integers) into *dout_max, one
// atomicMax per block.
template <int D, bool MAX>
__global__ void __launch_bounds__(256) fa_bwd_dsum_kernel(const uint16_t* __restrict__ o,
                                                          const uint16_t* __restrict__ o_lo,
                                                          const uint16_t* __restrict__ dout,
                                                          float* __restrict__ dsum, int B, int N,
                                                          int Hq,
                                                          uint32_t* __restrict__ dout_max) {
    constexpr int TPR = D / 8;  // 8 or 16: divides 32, so a row's threads share a warp
    __shared__ uint32_t wmax[8];
    const long long units = static_cast<long long>(B) * N * Hq * TPR;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const int lane = threadIdx.x & 31;
    uint32_t m = 0;
    auto row_sum = [&](uint4 x, uint4 g, uint4 y) {
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
        const uint32_t gs[4] = {g.x, g.y, g.z, g.w};
        const uint32_t ys[4] = {y.x, y.y, y.z, y.w};
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc = fmaf(bf16lo(xs[i]), bf16lo(gs[i]), acc);
            acc = fmaf(bf16hi(xs[i]), bf16hi(gs[i]), acc);
            if (MAX) {
                m = max(m, (gs[i] & 0x7fffu) << 16);
                m = max(m, gs[i] & 0x7fff0000u);
            }
        }
        if (o_lo) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc = fmaf(bf16lo(ys[i]), bf16lo(gs[i]), acc);
                acc = fmaf(bf16hi(ys[i]), bf16hi(gs[i]), acc);
            }
        }
        return acc;
    };
    // unit u = (row u / TPR, part u % TPR); rows are (b, n, h) in memory
    // order, D is stored [b, h, n]; B * N * Hq < 2^31
    auto finish = [&](long long u, float acc) {
#pragma unroll
        for (int s = TPR / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
        if (u < units && (u & (TPR - 1)) == 0) {
            const uint32_t row = static_cast<uint32_t>(u / TPR);
            const uint32_t h = row % static_cast<uint32_t>(Hq);
            const uint32_t bn = row / static_cast<uint32_t>(Hq);
            const uint32_t n = bn % static_cast<uint32_t>(N);
            const uint32_t b = bn / static_cast<uint32_t>(N);
            dsum[(static_cast<size_t>(b) * Hq + h) * N + n] = acc;
        }
    };
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    auto ld = [&](const uint16_t* base, long long u) {
        return u < units ? ld_stream_v4(base + u * 8) : zero;
    };
    // warp-uniform trip counts (u0 is the warp's first unit; stride is a
    // multiple of 32 and units a multiple of TPR)
    long long u0 = static_cast<long long>(blockIdx.x) * blockDim.x + (threadIdx.x - lane);
    for (; u0 + stride < units; u0 += 2 * stride) {
        const long long ua = u0 + lane, ub = ua + stride;
        const uint4 xa = ld(o, ua), ga = ld(dout, ua), xb = ld(o, ub), gb = ld(dout, ub);
        const uint4 ya = o_lo ? ld(o_lo, ua) : zero, yb = o_lo ? ld(o_lo, ub) : zero;
        const float sa = row_sum(xa, ga, ya);
        const float sb = row_sum(xb, gb, yb);
        finish(ua, sa);
        finish(ub, sb);
    }
    for (; u0 < units; u0 += stride) {
        const long long ua = u0 + lane;
        const uint4 xa = ld(o, ua), ga = ld(dout, ua);
        const uint4 ya = o_lo ? ld(o_lo, ua) : zero;
        finish(ua, row_sum(xa, ga, ya));
    }
    if (MAX) {
        m = __reduce_max_sync(0xffffffffu, m);
        if (lane == 0) wmax[threadIdx.x >> 5] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int w = 1; w < 8; ++w) m = max(m, wmax[w]);
            if (m != 0) atomicMax(dout_max, m);
        }
    }
}

template <int D>
cudaError_t launch_bwd_d(const BwdMaps& m, const BwdArgs& a, int stages, cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    if (stages & 1) {  // D = rowsum(dO o O)
        const long long units = static_cast<long long>(a.B) * a.N * a.Hq * (D / 8);
        const long long want = (units + 255) / 256;
        // two waves of 8 blocks of 256 threads per SM of this GPU's 152 (the
        // second evens out the finish); the loop covers the rest
        const unsigned blocks = static_cast<unsigned>(want > 2432 ? 2432 : want);
        if (a.dout_max)
            fa_bwd_dsum_kernel<D, true><<<blocks, 256, 0, st>>>(a.o, a.o_lo, a.dout, a.dsum, a.B,
                                                                a.N, a.Hq, a.dout_max);
        else
            fa_bwd_dsum_kernel<D, false><<<blocks, 256, 0, st>>>(a.o, a.o_lo, a.dout, a.dsum,
                                                                 a.B, a.N, a.Hq, nullptr);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // dQ before dK, dV: on the fp16 operand path the dQ kernel writes the copy
    // of dout that the dK/dV kernel reads
    if (stages & 4)
        if ((e = launch_bwd_dq<D>(m, a, st)) != cudaSuccess) return e;
    if (stages & 2)
        if ((e = launch_bwd_dkdv<D>(m, a, st)) != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd(const BwdMaps& maps, const BwdArgs& args, int stages, cudaStream_t stream) {
    if (args.d == 64) return launch_bwd_d<64>(maps, args, stages, stream);
    if (args.d == 128) return launch_bwd_d<128>(maps, args, stages, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa
