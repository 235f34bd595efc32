// fa_bwd_common.cuh -- pieces shared by the backward kernels (fa_bwd.cu,
// fa_bwd_dkdv.cu, fa_bwd_dq.cu).
#pragma once

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace bwd {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kWarpMma = 8;
constexpr int kWarpLoad = 9;
constexpr int kWarpGate = 10;  // dQ kernel: loads landed -> the MMA thread's LD barrier
constexpr int kWarpCopy = 11;  // dQ kernel: the fp16 copy of the dO tile
constexpr int kThreads = 384;  // WG0, WG1 compute; warp 8 MMA; warp 9 TMA; 10 gate; 11 copy

template <int D>
struct Tiles {
    static constexpr int CHUNK = kBM * 128;     // one 64-column chunk of a 128-row tile
    static constexpr int NCH = D / 64;
    static constexpr int TILE = NCH * CHUNK;    // 128 x D bf16
    static constexpr int HALF_ROWS = 64 * 128;  // byte offset of row 64 inside a chunk
};

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Writes a 128-row x (cols [c_lo, c_hi)) slab of fp32 TMEM values (scaled by
// `mul`) as bf16 into a TMA staging tile laid out as 64-column chunks of
// 128-byte swizzled rows.  The thread owns TMEM lane / tile row r.
template <int CHUNK>
__device__ __forceinline__ void stage_rows_bf16(uint32_t t_row, uint32_t stage, int r, int c_lo,
                                                int c_hi, float mul) {
    for (int cb = c_lo; cb < c_hi; cb += 32) {
        uint32_t v[32];
        tmem_ld32(t_row + cb, v);
        tmem_wait_ld();
        reg_fence<32>(v);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
        const uint32_t rowbase = stage + (cb >> 6) * CHUNK + r * 128;
#pragma unroll
        for (int p4 = 0; p4 < 4; ++p4) {
            const int piece = ((cb & 63) >> 3) + p4;
            st_shared_v4(rowbase + ((piece ^ (r & 7)) << 4), w[4 * p4], w[4 * p4 + 1],
                         w[4 * p4 + 2], w[4 * p4 + 3]);
        }
    }
}

// Copies row r of a 128 x D bf16 tile (TMA layout: 64-column chunks of
// 128-byte swizzled rows) into TMEM as an MMA A operand: lane r, column c
// holds elements 2c (low half) and 2c+1.
template <int D>
__device__ __forceinline__ void tile_row_to_tmem(uint32_t tile, uint32_t t_row, int r) {
    using T = Tiles<D>;
#pragma unroll
    for (int c = 0; c < T::NCH; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const uint32_t addr = tile + c * T::CHUNK + r * 128 + ((p ^ (r & 7)) << 4);
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v[4 * p]), "=r"(v[4 * p + 1]), "=r"(v[4 * p + 2]), "=r"(v[4 * p + 3])
                         : "r"(addr)
                         : "memory");
        }
        tmem_st32(t_row + c * 32, v);
    }
}

}  // namespace bwd
}  // namespace fa
