// fa_bwd_dq.cu -- dQ = scale * dS K for exact attention, sm_103a.
//
// One CTA per (batch, query head, 128-query block).  Recomputes, for every key
// block j the block sees, S = Q K_j^T and dP = dO V_j^T, then
// P = exp2(S * scale * log2(e) - lse * log2(e)) and dS = P o (dP - D), and
// accumulates dQ += dS K_j in tensor memory (the recomputation the pages
// describe for the backward pass: "FlashAttention Kernel", recomputation
// bullet; the gradient formulas are the derivative of the forward definition).
//
// Pipelining: each 128-key block is split into two 64-key halves with their
// own barriers.  Warpgroup 0 turns half a into dS while the tensor core
// computes half b's scores and the previous half's dQ update, and vice
// versa, so the elementwise work hides behind MMAs.  Q and dO are copied into
// TMEM once and used as the A operand of the score MMAs, so those MMAs read
// only K_j / V_j from shared memory.
//
// TMEM (512 columns): S [0,128) (half a: [0,64), half b: [64,128)),
// dP [128,256), dQ [256,256+D), Q [384,384+D/2), dO [448,448+D/2).
#include "fa_bwd_common.cuh"

namespace fa {
namespace {

using namespace bwd;

template <int D>
struct DqCfg : Tiles<D> {
    using T = Tiles<D>;
    static constexpr int NST = 2;  // K/V ring stages
    static constexpr int OFF_KV = 2 * T::TILE;  // after Q, dO
    static constexpr int OFF_BAR = OFF_KV + NST * 2 * T::TILE;
    static constexpr int NBAR = 1 + 2 * NST + 1 + 2 + 2 + 1;
    static constexpr int SMEM_BYTES = 1024 + OFF_BAR + NBAR * 8 + 16;
    static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DQ = 256, TM_Q = 384, TM_DO = 448;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmDO,
                     const __grid_constant__ CUtensorMap tmDQ, const BwdArgs a) {
    using C = DqCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sDO = sQ + C::TILE;
    const uint32_t sKV = sQ + C::OFF_KV;  // stage s: K at sKV + 2s*TILE, V after it
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t BAR_QDO = bar0;  // Q, dO tiles landed
    auto BAR_KVF = [&](int s) { return bar0 + 8u * (1 + s); };
    auto BAR_KVE = [&](int s) { return bar0 + 8u * (1 + C::NST + s); };
    const uint32_t BAR_QT = bar0 + 8u * (1 + 2 * C::NST);          // Q, dO copied to TMEM
    auto BAR_SF = [&](int hf) { return BAR_QT + 8u * (1 + hf); };  // half's S, dP ready
    auto BAR_PF = [&](int hf) { return BAR_QT + 8u * (3 + hf); };  // half's dS written
    const uint32_t BAR_ACC = BAR_QT + 8u * 5;

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
        mbar_init(BAR_QT, 256);
        for (int hf = 0; hf < 2; ++hf) {
            mbar_init(BAR_SF(hf), 1);
            mbar_init(BAR_PF(hf), 128);
        }
        mbar_init(BAR_ACC, 1);
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), 512);
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
            // no copies in flight at exit: wait (bounded) for the last load of each stage
            mbar_wait(BAR_QDO, 0, a.status, a.timeout_ns, 21);
            for (int s = 0; s < C::NST; ++s)
                if (last_j[s] >= 0)
                    mbar_wait(BAR_KVF(s), (last_j[s] / C::NST) & 1, a.status, a.timeout_ns, 21);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(kBM, 64, false, false);  // S, dP halves
            constexpr uint32_t IDESC_DQ = idesc_bf16(kBM, D, false, true);   // dQ += dS K
            const uint32_t tS = tbase + C::TM_S, tDP = tbase + C::TM_DP, tDQ = tbase + C::TM_DQ;
            const uint32_t tQ = tbase + C::TM_Q, tDO = tbase + C::TM_DO;
            // scores of key half hf of the block in stage s: A = Q / dO from TMEM,
            // B = rows 64*hf.. of K_j / V_j (K-major)
            auto issue_s = [&](int hf, int s) {
                const uint32_t sK = sKV + 2 * s * C::TILE, sV = sK + C::TILE;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32 + hf * C::HALF_ROWS;
                    mma_bf16_ts(tS + hf * 64, tQ + ks * 8, sdesc_sw128(sK + off, 16, 1024), IDESC_S,
                                ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32 + hf * C::HALF_ROWS;
                    mma_bf16_ts(tDP + hf * 64, tDO + ks * 8, sdesc_sw128(sV + off, 16, 1024),
                                IDESC_S, ks > 0);
                }
                mma_commit(BAR_SF(hf));
            };
            // dQ += dS_half K_half: dS (bf16) at columns [64*hf, 64*hf+32), K rows
            // 64*hf.. read MN-major
            auto issue_dq = [&](int hf, int s, bool first) {
                const uint32_t sK = sKV + 2 * s * C::TILE;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_ts(tDQ, tS + hf * 64 + ks * 8,
                                sdesc_sw128(sK + hf * C::HALF_ROWS + ks * 2048, C::CHUNK, 1024),
                                IDESC_DQ, (first && ks == 0) ? 0u : 1u);
            };
            bool ok = mbar_wait(BAR_QT, 0, a.status, a.timeout_ns, 22) &&
                      mbar_wait(BAR_KVF(0), 0, a.status, a.timeout_ns, 23);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                issue_s(1, 0);
            }
            for (int j = 0; j < nj && ok; ++j) {
                const int s = j % C::NST;
                const int s2 = (j + 1) % C::NST;
                if (!(ok = mbar_wait(BAR_PF(0), j & 1, a.status, a.timeout_ns, 24))) break;
                tc_fence_after();
                issue_dq(0, s, j == 0);
                if (j + 1 < nj) {
                    if (!(ok = mbar_wait(BAR_KVF(s2), ((j + 1) / C::NST) & 1, a.status,
                                         a.timeout_ns, 23)))
                        break;
                    tc_fence_after();
                    issue_s(0, s2);
                }
                if (!(ok = mbar_wait(BAR_PF(1), j & 1, a.status, a.timeout_ns, 24))) break;
                tc_fence_after();
                issue_dq(1, s, false);
                mma_commit(BAR_KVE(s));
                if (j + 1 < nj) issue_s(1, s2);
            }
            // every issued MMA has finished before TMEM is released
            mma_commit(BAR_ACC);
            mbar_wait(BAR_ACC, 0, a.status, a.timeout_ns, 25);
        }
        __syncwarp();
    } else if (warp < 8) {
        const int hf = warp >> 2;  // key half of every block this warpgroup handles
        const int r = (warp & 3) * 32 + lane;
        const int grow = qi * kBM + r;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tbase + C::TM_S + lane_off + hf * 64;
        const uint32_t tDP = tbase + C::TM_DP + lane_off + hf * 64;
        const bool valid = grow < a.N;
        const size_t st_idx = (static_cast<size_t>(b) * a.Hq + h) * a.N + (valid ? grow : 0);
        const float nlse2 = valid ? -a.lse[st_idx] * kLog2e : 0.f;
        const float dval = valid ? a.dsum[st_idx] : 0.f;
        const float sl2 = a.scale_log2;
        const int lim = a.causal ? min(grow, a.N - 1) : a.N - 1;
        // Q (warpgroup 0) and dO (warpgroup 1) rows into TMEM as MMA A operands
        bool ok = mbar_wait(BAR_QDO, 0, a.status, a.timeout_ns, 26);
        if (ok) {
            tile_row_to_tmem<D>(hf ? sDO : sQ, tbase + (hf ? C::TM_DO : C::TM_Q) + lane_off, r);
            tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(BAR_QT);
        for (int j = 0; j < nj && ok; ++j) {
            if (!(ok = mbar_wait(BAR_SF(hf), j & 1, a.status, a.timeout_ns, 26))) break;
            tc_fence_after();
            uint32_t sv[64], dp[64];
            tmem_ld32(tS, sv);
            tmem_ld32(tS + 32, sv + 32);
            tmem_ld32(tDP, dp);
            tmem_ld32(tDP + 32, dp + 32);
            tmem_wait_ld();
            reg_fence<64>(sv);
            reg_fence<64>(dp);
            const int kbase = j * kBN + hf * 64;
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
                pk[c >> 1] = pack_bf16(p0 * (__uint_as_float(dp[c]) - dval),
                                       p1 * (__uint_as_float(dp[c + 1]) - dval));
            }
            tmem_st32(tS, pk);  // dS over this half's S columns
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR_PF(hf));
        }
        const bool ok_e = ok && mbar_wait(BAR_ACC, 0, a.status, a.timeout_ns, 27);
        if (ok_e) {
            tc_fence_after();
            // dQ = scale * (dS K): each warpgroup stages half of the d columns into
            // the Q tile's shared memory (Q now lives in TMEM)
            stage_rows_bf16<C::CHUNK>(tbase + C::TM_DQ + lane_off, sQ, r, hf * (D / 2),
                                      (hf + 1) * (D / 2), a.scale);
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
        tmem_dealloc(tbase, 512);
    }
}

}  // namespace

template <int D>
cudaError_t launch_bwd_dq(const BwdMaps& m, const BwdArgs& a, cudaStream_t st) {
    auto kern = fa_bwd_dq_kernel<D>;
    constexpr int smem = DqCfg<D>::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long nblk = static_cast<long long>((a.N + kBM - 1) / kBM) * a.B * a.Hq;
    if (nblk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<static_cast<unsigned>(nblk), kThreads, smem, st>>>(m.q, m.k, m.v, m.dout, m.dq, a);
    return cudaGetLastError();
}

template cudaError_t launch_bwd_dq<64>(const BwdMaps&, const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_dq<128>(const BwdMaps&, const BwdArgs&, cudaStream_t);

}  // namespace fa
