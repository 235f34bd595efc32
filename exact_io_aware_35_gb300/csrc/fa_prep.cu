// fa_prep.cu -- fp16 copies of the MMA operand tensors, scaled by powers of two.
//
// Two launches per job (up to four tensors): the first takes max |x| of each
// tensor (atomicMax on the float bit pattern, which orders non-negative
// floats like integers), the second turns the maxima into F16Scales and
// writes fp16(x * 2^s).  Both are HBM-bound loops over chunks of 16-byte
// vectors (8 elements), eight loads in flight per thread; the copy walks
// the chunks in the reverse of the maxima's order, so it starts on what L2
// still holds.  The exponents (f16_scales_from) put
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

// The job's tensors as one sequence of chunks of kChunkVec 16-byte vectors
// (each chunk inside one tensor): q's chunks, then k's, v's, dout's.  A
// thread takes kVecPerThread vectors of a chunk, all loads in flight at once.
constexpr int kVecPerThread = 8;
constexpr int kChunkVec = kPrepThreads * kVecPerThread;

struct ChunkMap {
    size_t n8[4];
    size_t first[5];  // first chunk of each tensor; first[4] = total
    __device__ __forceinline__ ChunkMap(const F16Prep& p, int mask) {
        first[0] = 0;
        for (int t = 0; t < 4; ++t) {
            n8[t] = ((mask >> t) & 1) ? p.n[t] / 8 : 0;
            first[t + 1] = first[t] + (n8[t] + kChunkVec - 1) / kChunkVec;
        }
    }
    __device__ __forceinline__ int tensor_of(size_t c) const {
        return (c >= first[1]) + (c >= first[2]) + (c >= first[3]);
    }
};

// a[t] for a runtime t without local-memory indexing
template <typename T>
__device__ __forceinline__ T pick(const T (&a)[4], int t) {
    return t == 0 ? a[0] : t == 1 ? a[1] : t == 2 ? a[2] : a[3];
}
template <typename T>
__device__ __forceinline__ T pick(const T (&a)[5], int t) {
    return t == 0 ? a[0] : t == 1 ? a[1] : t == 2 ? a[2] : t == 3 ? a[3] : a[4];
}

__global__ void __launch_bounds__(kPrepThreads) f16_absmax_kernel(const F16Prep p) {
    int present = 0;
    for (int t = 0; t < 4; ++t) present |= (p.n[t] > 0) << t;
    const ChunkMap cm(p, present);
    uint32_t m[4] = {0, 0, 0, 0};
    // front to back in tensor order, so that the last tensors read (k, v) are
    // what L2 holds when the copy kernel reads them back to front right after
    for (size_t c = blockIdx.x; c < cm.first[4]; c += gridDim.x) {
        const int t = cm.tensor_of(c);
        const uint4* src = reinterpret_cast<const uint4*>(pick(p.src, t));
        const size_t n8 = pick(cm.n8, t);
        const size_t base = (c - pick(cm.first, t)) * kChunkVec + threadIdx.x;
        uint4 v[kVecPerThread];
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) {
            const size_t j = base + static_cast<size_t>(i) * kPrepThreads;
            v[i] = j < n8 ? src[j] : make_uint4(0, 0, 0, 0);
        }
        uint32_t mm = 0;
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) mm = absmax8(v[i], mm);
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (u == t) m[u] = max(m[u], mm);
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint32_t r = __reduce_max_sync(0xffffffffu, m[t]);
        if ((threadIdx.x & 31) == 0 && r != 0) atomicMax(p.absmax + t, r);
    }
}

__global__ void __launch_bounds__(kPrepThreads) f16_convert_kernel(const F16Prep p) {
    const F16Scales s = f16_scales_from(p.absmax, p.d);
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.scales = s;
    const ChunkMap cm(p, p.convert_mask);
    const float mul[4] = {pow2f(s.q), pow2f(s.k), pow2f(s.v), pow2f(s.dout)};
    // back to front over the chunks: the most recently read ones first
    const size_t total = cm.first[4];
    for (size_t cc = blockIdx.x; cc < total; cc += gridDim.x) {
        const size_t c = total - 1 - cc;
        const int t = cm.tensor_of(c);
        const uint4* src = reinterpret_cast<const uint4*>(pick(p.src, t));
        uint4* dst = reinterpret_cast<uint4*>(pick(p.dst, t));
        const float f = pick(mul, t);
        const size_t n8 = pick(cm.n8, t);
        const size_t base = (c - pick(cm.first, t)) * kChunkVec + threadIdx.x;
        uint4 v[kVecPerThread];
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) {
            const size_t j = base + static_cast<size_t>(i) * kPrepThreads;
            if (j < n8) v[i] = src[j];
        }
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) {
            const size_t j = base + static_cast<size_t>(i) * kPrepThreads;
            if (j < n8) {
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                uint32_t o[4];
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    o[h] = pack_f16(__uint_as_float(w[h] << 16) * f,
                                    __uint_as_float(w[h] & 0xffff0000u) * f);
                dst[j] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

}  // namespace

cudaError_t launch_f16_prep(const F16Prep& p, cudaStream_t st) {
    size_t chunks = 0;
    for (int t = 0; t < 4; ++t) chunks += (p.n[t] / 8 + kChunkVec - 1) / kChunkVec;
    // up to 8 blocks per SM of this GPU's 152, each looping over chunks
    const unsigned gx = static_cast<unsigned>(chunks < 1 ? 1 : (chunks > 1216 ? 1216 : chunks));
    // only the maxima of the tensors in this job start over: a job that copies
    // dout alone keeps the q, k, v maxima an earlier job left (the scales are
    // always recomputed from all four)
    cudaError_t e = cudaSuccess;
    for (int t = 0; t < 4 && e == cudaSuccess; ++t)
        if (p.n[t] > 0) e = cudaMemsetAsync(p.absmax + t, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    f16_absmax_kernel<<<gx, kPrepThreads, 0, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (p.convert_mask == 0) return cudaSuccess;  // the maxima alone (the dQ kernel copies dO)
    f16_convert_kernel<<<gx, kPrepThreads, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace fa
