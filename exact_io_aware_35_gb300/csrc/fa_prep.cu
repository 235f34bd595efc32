// fa_prep.cu -- fp16 copies of the MMA operand tensors, scaled by powers of two.
//
// Two launches per job (up to four tensors, blockIdx.y picks one): the first
// takes max |x| of each tensor (atomicMax on the float bit pattern, which
// orders non-negative floats like integers), the second turns the maxima into
// F16Scales and writes fp16(x * 2^s).  Both are HBM-bound grid-stride loops
// over 16-byte vectors (8 elements).  The exponents (f16_scales_from) put
// the scaled maxima well inside fp16's range, which keeps the copies exact
// for all but elements many orders of magnitude below the maximum.
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kPrepThreads = 256;

__device__ __forceinline__ uint32_t absmax8(uint4 v, uint32_t m) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        // |x| of each bf16 half as the bits of an fp32 value
        m = max(m, (w[j] & 0x7fffu) << 16);
        m = max(m, w[j] & 0x7fff0000u);
    }
    return m;
}

__global__ void __launch_bounds__(kPrepThreads) f16_absmax_kernel(const F16Prep p) {
    const int t = blockIdx.y;
    const size_t n8 = p.n[t] / 8;
    const uint4* src = reinterpret_cast<const uint4*>(p.src[t]);
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    uint32_t m = 0;
    // Back to front (element n8-1-i), four independent 16-byte loads in flight
    // per thread: the front of the tensor is then what L2 holds when the copy
    // (or the D kernel) reads it front to back right after.
    const uint4* end = src + n8 - 1;
    for (; i + 3 * stride < n8; i += 4 * stride) {
        const uint4 a = *(end - i), b = *(end - i - stride), c = *(end - i - 2 * stride),
                    d = *(end - i - 3 * stride);
        m = absmax8(d, absmax8(c, absmax8(b, absmax8(a, m))));
    }
    for (; i < n8; i += stride) m = absmax8(*(end - i), m);
    m = __reduce_max_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0 && m != 0) atomicMax(p.absmax + t, m);
}

__global__ void __launch_bounds__(kPrepThreads) f16_convert_kernel(const F16Prep p) {
    const int t = blockIdx.y;
    const F16Scales s = f16_scales_from(p.absmax, p.d);
    if (blockIdx.x == 0 && t == 0 && threadIdx.x == 0) *p.scales = s;
    const int e = (t == 0) ? s.q : (t == 1) ? s.k : (t == 2) ? s.v : s.dout;
    const float mul = pow2f(e);
    const size_t n8 = ((p.convert_mask >> t) & 1) ? p.n[t] / 8 : 0;
    const uint4* src = reinterpret_cast<const uint4*>(p.src[t]);
    uint4* dst = reinterpret_cast<uint4*>(p.dst[t]);
    auto cvt8 = [&](uint4 v) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            o[j] = pack_f16(__uint_as_float(w[j] << 16) * mul,
                            __uint_as_float(w[j] & 0xffff0000u) * mul);
        return make_uint4(o[0], o[1], o[2], o[3]);
    };
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    // two independent 16-byte loads in flight per thread
    for (; i + stride < n8; i += 2 * stride) {
        const uint4 a = src[i], b = src[i + stride];
        dst[i] = cvt8(a);
        dst[i + stride] = cvt8(b);
    }
    for (; i < n8; i += stride) dst[i] = cvt8(src[i]);
}

}  // namespace

cudaError_t launch_f16_prep(const F16Prep& p, cudaStream_t st) {
    size_t nmax = 0;
    for (int t = 0; t < 4; ++t) nmax = p.n[t] > nmax ? p.n[t] : nmax;
    // up to 8 blocks per SM of this GPU's 152 (grid-stride loops cover the rest)
    const size_t want = (nmax / 8 + kPrepThreads - 1) / kPrepThreads;
    const unsigned gx = static_cast<unsigned>(want < 1 ? 1 : (want > 1216 ? 1216 : want));
    // only the maxima of the tensors in this job start over: a job that copies
    // dout alone keeps the q, k, v maxima an earlier job left (the scales are
    // always recomputed from all four)
    cudaError_t e = cudaSuccess;
    for (int t = 0; t < 4 && e == cudaSuccess; ++t)
        if (p.n[t] > 0) e = cudaMemsetAsync(p.absmax + t, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    f16_absmax_kernel<<<dim3(gx, 4), kPrepThreads, 0, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (p.convert_mask == 0) return cudaSuccess;  // the maxima alone (the dQ kernel copies dO)
    f16_convert_kernel<<<dim3(gx, 4), kPrepThreads, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace fa
