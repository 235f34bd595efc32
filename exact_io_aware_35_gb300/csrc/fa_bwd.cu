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
//   1. dsum:  D = rowsum(dO o O) in fp32 (HBM-bound, coalesced 16-byte loads).
//   2. dkdv:  one CTA per (batch, kv head, 128-key block).  K and V stay in
//             shared memory; Q_i and dO_i stream through a 2-stage TMA ring
//             for every query head of the group and every query block that
//             sees the key block.  S^T = K Q_i^T and dP^T = V dO_i^T go to
//             TMEM; two warpgroups (one per 64-query half) turn them into P^T
//             and dS^T (bf16) in place; dV += P^T dO_i and dK += dS^T Q_i then
//             take P^T / dS^T straight from TMEM as the A operand.
//   3. dq:    one CTA per (batch, q head, 128-query block); K_j, V_j stream
//             through a 2-stage ring; S = Q K_j^T and dP = dO V_j^T in TMEM,
//             dS in place, dQ += dS K_j accumulated in TMEM.
// Computing S^T directly (keys on the TMEM lanes) is what lets the key-side
// gradients take their A operand from TMEM without a transpose.
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
    static constexpr int CHUNK = kBM * 128;   // one 64-column chunk of a 128-row tile
    static constexpr int NCH = D / 64;
    static constexpr int TILE = NCH * CHUNK;  // 128 x D bf16
    static constexpr int NST = 2;             // ring stages
    static constexpr int THREADS = 384;       // WG0, WG1 compute; warp 8 MMA; warp 9 TMA
    // TMEM columns
    static constexpr uint32_t TM_S = 0;       // S or S^T (fp32, 128 cols); P/dS bf16 in place
    static constexpr uint32_t TM_DP = 128;    // dP or dP^T (fp32, 128 cols)
    static constexpr uint32_t TM_ACC = 256;   // dQ | dV, dK accumulators
    static constexpr uint32_t TM_COLS = 512;
};

constexpr int kWarpMma = 8;
constexpr int kWarpLoad = 9;

// ----------------------------------------------------------------------------
// 1. D_i = sum_c dO_ic * O_ic
// ----------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__global__ void __launch_bounds__(256) fa_bwd_dsum_kernel(const uint16_t* __restrict__ o,
                                                          const uint16_t* __restrict__ dout,
                                                          float* __restrict__ dsum, int B, int N,
                                                          int Hq, int d) {
    const int tpr = d >> 3;  // threads per row, 8 bf16 (16 bytes) each
    const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long rows = static_cast<long long>(B) * N * Hq;
    const long long row = gid / tpr;
    const int part = static_cast<int>(gid % tpr);
    float acc = 0.f;
    if (row < rows) {
        const uint4 a = *reinterpret_cast<const uint4*>(o + row * d + part * 8);
        const uint4 g = *reinterpret_cast<const uint4*>(dout + row * d + part * 8);
        acc = bf16lo(a.x) * bf16lo(g.x) + bf16hi(a.x) * bf16hi(g.x);
        acc = fmaf(bf16lo(a.y), bf16lo(g.y), acc);
        acc = fmaf(bf16hi(a.y), bf16hi(g.y), acc);
        acc = fmaf(bf16lo(a.z), bf16lo(g.z), acc);
        acc = fmaf(bf16hi(a.z), bf16hi(g.z), acc);
        acc = fmaf(bf16lo(a.w), bf16lo(g.w), acc);
        acc = fmaf(bf16hi(a.w), bf16hi(g.w), acc);
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

// Writes a 128-row x (cols [c_lo, c_hi)) slab of fp32 TMEM values (scaled by
// `mul`) as bf16 into a TMA staging tile laid out as 64-column chunks of
// 128-byte swizzled rows.  Thread owns TMEM lane / tile row r.
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

// ----------------------------------------------------------------------------
// 3. dQ: one CTA per (b, q head, 128-query block)
// ----------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(384, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmDO,
                     const __grid_constant__ CUtensorMap tmDQ, const BwdArgs a) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sDO = sQ + C::TILE;
    const uint32_t sKV = sDO + C::TILE;  // stage s: K at sKV + 2s*TILE, V after it
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (2 + 2 * C::NST) * C::TILE);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t BAR_QDO = bar0;
    auto BAR_KVF = [&](int s) { return bar0 + 8u * (1 + s); };
    auto BAR_KVE = [&](int s) { return bar0 + 8u * (1 + C::NST + s); };
    const uint32_t BAR_SF = bar0 + 8u * (1 + 2 * C::NST);
    const uint32_t BAR_PF = BAR_SF + 8;
    const uint32_t BAR_ACC = BAR_SF + 16;

    const int warp = warp_id();
    const int lane = lane_id();
    const int nqb = (a.N + kBM - 1) / kBM;
    const int per = a.B * a.Hq;
    const int qi = nqb - 1 - static_cast<int>(blockIdx.x) / per;  // longest first
    const int bh = static_cast<int>(blockIdx.x) % per;
    const int b = bh / a.Hq;
    const int h = bh % a.Hq;
    const int hk = h / a.g;
    const int nkv_all = (a.N + kBN - 1) / kBN;
    const int nj = a.causal ? min(qi + 1, nkv_all) : nkv_all;

    if (warp == 0 && lane == 0) {
        mbar_init(BAR_QDO, 1);
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(BAR_KVF(s), 1);
            mbar_init(BAR_KVE(s), 1);
        }
        mbar_init(BAR_SF, 1);
        mbar_init(BAR_PF, 256);
        mbar_init(BAR_ACC, 1);
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    if (warp == kWarpLoad) {
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmDO);
            tma_prefetch_desc(&tmDQ);
            const uint64_t pol_kv = l2_policy_evict_last();
            mbar_arrive_expect_tx(BAR_QDO, 2 * C::TILE);
            for (int c = 0; c < C::NCH; ++c) {
                tma_load_4d(sQ + c * C::CHUNK, &tmQ, BAR_QDO, c * 64, h, qi * kBM, b);
                tma_load_4d(sDO + c * C::CHUNK, &tmDO, BAR_QDO, c * 64, h, qi * kBM, b);
            }
            int last_j[C::NST] = {-1, -1};
            for (int j = 0; j < nj; ++j) {
                const int s = j % C::NST;
                if (!mbar_wait(BAR_KVE(s), ((j / C::NST) & 1) ^ 1u, a.status, a.timeout_ns, 20))
                    break;
                mbar_arrive_expect_tx(BAR_KVF(s), 2 * C::TILE);
                const uint32_t dst = sKV + 2 * s * C::TILE;
                for (int c = 0; c < C::NCH; ++c) {
                    tma_load_4d_hint(dst + c * C::CHUNK, &tmK, BAR_KVF(s), c * 64, hk, j * kBN, b,
                                     pol_kv);
                    tma_load_4d_hint(dst + C::TILE + c * C::CHUNK, &tmV, BAR_KVF(s), c * 64, hk,
                                     j * kBN, b, pol_kv);
                }
                last_j[s] = j;
            }
            mbar_wait(BAR_QDO, 0, a.status, a.timeout_ns, 21);
            for (int s = 0; s < C::NST; ++s)
                if (last_j[s] >= 0)
                    mbar_wait(BAR_KVF(s), (last_j[s] / C::NST) & 1, a.status, a.timeout_ns, 21);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            constexpr uint32_t IDESC_SS = idesc_bf16(kBM, kBN, false, false);  // S, dP
            constexpr uint32_t IDESC_DQ = idesc_bf16(kBM, D, false, true);     // dQ += dS K
            const uint32_t tS = tbase + C::TM_S, tDP = tbase + C::TM_DP, tDQ = tbase + C::TM_ACC;
            bool ok = mbar_wait(BAR_QDO, 0, a.status, a.timeout_ns, 22);
            for (int j = 0; j < nj && ok; ++j) {
                const int s = j % C::NST;
                if (!(ok = mbar_wait(BAR_KVF(s), (j / C::NST) & 1, a.status, a.timeout_ns, 23)))
                    break;
                tc_fence_after();
                const uint32_t sK = sKV + 2 * s * C::TILE, sV = sK + C::TILE;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
                    mma_bf16_ss(tS, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024),
                                IDESC_SS, ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
                    mma_bf16_ss(tDP, sdesc_sw128(sDO + off, 16, 1024),
                                sdesc_sw128(sV + off, 16, 1024), IDESC_SS, ks > 0);
                }
                mma_commit(BAR_SF);
                if (!(ok = mbar_wait(BAR_PF, j & 1, a.status, a.timeout_ns, 24))) break;
                tc_fence_after();
                // dS (bf16) lies at columns [0,32) (keys 0-63) and [64,96) (keys 64-127)
#pragma unroll
                for (int ks = 0; ks < kBN / 16; ++ks) {
                    const uint32_t acol = (ks < 4) ? ks * 8 : 64 + (ks - 4) * 8;
                    mma_bf16_ts(tDQ, tS + acol, sdesc_sw128(sK + ks * 2048, C::CHUNK, 1024),
                                IDESC_DQ, (j > 0 || ks > 0) ? 1u : 0u);
                }
                mma_commit(BAR_KVE(s));
            }
            mma_commit(BAR_ACC);
            mbar_wait(BAR_ACC, 0, a.status, a.timeout_ns, 25);
        }
        __syncwarp();
    } else if (warp < 8) {
        const int wg = warp >> 2;            // 0: keys 0-63 of each block, 1: keys 64-127
        const int r = (warp & 3) * 32 + lane;
        const int grow = qi * kBM + r;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tbase + C::TM_S + lane_off;
        const uint32_t tDP = tbase + C::TM_DP + lane_off;
        const int c0 = wg * 64;
        const bool valid = grow < a.N;
        const size_t st_idx = (static_cast<size_t>(b) * a.Hq + h) * a.N + (valid ? grow : 0);
        const float nlse2 = valid ? -a.lse[st_idx] * kLog2e : 0.f;
        const float dval = valid ? a.dsum[st_idx] : 0.f;
        const float sl2 = a.scale_log2;
        const int lim = a.causal ? min(grow, a.N - 1) : a.N - 1;
        bool ok = true;
        for (int j = 0; j < nj; ++j) {
            if (!(ok = mbar_wait(BAR_SF, j & 1, a.status, a.timeout_ns, 26))) break;
            tc_fence_after();
            uint32_t sv[64], dp[64];
            tmem_ld32(tS + c0, sv);
            tmem_ld32(tS + c0 + 32, sv + 32);
            tmem_ld32(tDP + c0, dp);
            tmem_ld32(tDP + c0 + 32, dp + 32);
            tmem_wait_ld();
            reg_fence<64>(sv);
            reg_fence<64>(dp);
            const int kbase = j * kBN + c0;
            const bool need_mask = kbase + 63 > lim;
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
                float p0 = ex2(fmaf(__uint_as_float(sv[c]), sl2, nlse2));
                float p1 = ex2(fmaf(__uint_as_float(sv[c + 1]), sl2, nlse2));
                if (need_mask) {
                    p0 = (kbase + c > lim) ? 0.f : p0;
                    p1 = (kbase + c + 1 > lim) ? 0.f : p1;
                }
                const float ds0 = p0 * (__uint_as_float(dp[c]) - dval);
                const float ds1 = p1 * (__uint_as_float(dp[c + 1]) - dval);
                pk[c >> 1] = pack_bf16(ds0, ds1);
            }
            tmem_st32(tS + c0, pk);  // inside this warpgroup's own S columns
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR_PF);
        }
        const bool ok_e = ok && mbar_wait(BAR_ACC, 0, a.status, a.timeout_ns, 27);
        if (ok_e) {
            tc_fence_after();
            // dQ = scale * (dS K): each warpgroup stages half of the d columns
            stage_rows_bf16<C::CHUNK>(tbase + C::TM_ACC + lane_off, sQ, r, wg * (D / 2),
                                      (wg + 1) * (D / 2), a.scale);
            fence_proxy_async_smem();
        }
        named_bar_sync(1, 256);
        if (ok_e && warp == 0 && lane == 0) {
            for (int c = 0; c < C::NCH; ++c)
                tma_store_4d(&tmDQ, sQ + c * C::CHUNK, c * 64, h, qi * kBM, b);
            tma_store_commit();
            tma_store_wait_read_all();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tbase, C::TM_COLS);
    }
}

// BWD_DKDV_KERNEL

}  // namespace

// BWD_LAUNCH

}  // namespace fa
