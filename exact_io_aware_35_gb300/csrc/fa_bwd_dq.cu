// fa_bwd_dq.cu -- dQ = scale * dS K for exact attention, sm_103a.
//
// One CTA per (batch, query head, 128-query block).  Recomputes, for every key
// block j the block sees, S = Q K_j^T and dP = dO V_j^T, then
// P = exp2(S * scale * log2(e) - lse * log2(e)) and dS = P o (dP - D), and
// accumulates dQ += dS K_j in tensor memory (the recomputation the pages
// describe for the backward pass: "FlashAttention Kernel", recomputation
// bullet; the gradient formulas are the derivative of the forward definition).
//
// Pipelining.  Every MMA is 128 wide (a tcgen05.mma of N = 64 cannot be issued
// faster than ~46 cycles, a third more than its math takes; N = 128 runs at the
// math rate).  S is double-buffered in TMEM, so S(j+2) is computed while the
// two warpgroups turn block j+1 into dS (warpgroup h takes keys 64h..64h+63);
// dQ += dS_h K_h is issued as soon as warpgroup h is done, then dP(j+2) into
// the single dP buffer.  K and V stream through a 5-slot TMA ring.
//
// TMEM (512 columns): S0 [0,128), S1 [128,256), dP [256,384), dQ [384,384+D).
#include "fa_bwd_common.cuh"

namespace fa {
namespace {

using namespace bwd;

template <int D>
struct DqCfg : Tiles<D> {
    using T = Tiles<D>;
    static constexpr int NSLOT = (D == 128) ? 5 : 8;  // K / V ring slots, one tile each
    static constexpr int OFF_KV = 2 * T::TILE;          // after Q, dO
    static constexpr int OFF_BAR = OFF_KV + NSLOT * T::TILE;
    static constexpr int NBAR = 1 + 2 * NSLOT + 1 + 2 + 1;
    static constexpr int SMEM_BYTES = 1024 + OFF_BAR + NBAR * 8 + 16;
    static constexpr uint32_t TM_S = 0, TM_DP = 256, TM_DQ = 384;
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
    const uint32_t sKV = sQ + C::OFF_KV;  // slot t at sKV + t*TILE; K_j is tile 2j, V_j tile 2j+1
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t BAR_QDO = bar0;  // Q, dO tiles landed
    auto BAR_KVF = [&](int t) { return bar0 + 8u * (1 + t); };
    auto BAR_KVE = [&](int t) { return bar0 + 8u * (1 + C::NSLOT + t); };
    const uint32_t BAR_SDF = bar0 + 8u * (1 + 2 * C::NSLOT);       // block's S and dP ready
    auto BAR_PF = [&](int hf) { return BAR_SDF + 8u * (1 + hf); };  // half's dS written
    const uint32_t BAR_ACC = BAR_SDF + 8u * 3;

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
        for (int t = 0; t < C::NSLOT; ++t) {
            mbar_init(BAR_KVF(t), 1);
            mbar_init(BAR_KVE(t), 1);
        }
        mbar_init(BAR_SDF, 1);
        for (int hf = 0; hf < 2; ++hf) mbar_init(BAR_PF(hf), 128);
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
            int last_idx[C::NSLOT];
            for (int t = 0; t < C::NSLOT; ++t) last_idx[t] = -1;
            bool ok = true;
            for (int idx = 0; idx < 2 * nj && ok; ++idx) {
                const int t = idx % C::NSLOT;
                if (!(ok = mbar_wait(BAR_KVE(t), ((idx / C::NSLOT) & 1) ^ 1u, a.status,
                                     a.timeout_ns, 20)))
                    break;
                mbar_arrive_expect_tx(BAR_KVF(t), C::TILE);
                const CUtensorMap* tm = (idx & 1) ? &tmV : &tmK;
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_4d_hint(sKV + t * C::TILE + c * C::CHUNK, tm, BAR_KVF(t), c * 64, hk,
                                     (idx >> 1) * kBN, b, pol_kv);
                last_idx[t] = idx;
            }
            // no copies in flight at exit: wait (bounded) for the last load of each slot
            mbar_wait(BAR_QDO, 0, a.status, a.timeout_ns, 21);
            for (int t = 0; t < C::NSLOT; ++t)
                if (last_idx[t] >= 0)
                    mbar_wait(BAR_KVF(t), (last_idx[t] / C::NSLOT) & 1, a.status, a.timeout_ns, 21);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(kBM, kBN, false, false);  // S, dP
            constexpr uint32_t IDESC_DQ = idesc_bf16(kBM, D, false, true);     // dQ += dS K
            const uint32_t tDP = tbase + C::TM_DP, tDQ = tbase + C::TM_DQ;
            auto kslot = [&](int jj) { return (2 * jj) % C::NSLOT; };
            auto vslot = [&](int jj) { return (2 * jj + 1) % C::NSLOT; };
            auto ready = [&](int tile) {  // wait for ring tile `tile` (K_j = 2j, V_j = 2j+1)
                const bool r = mbar_wait(BAR_KVF(tile % C::NSLOT), (tile / C::NSLOT) & 1,
                                         a.status, a.timeout_ns, 23);
                tc_fence_after();
                return r;
            };
            // S(jj) = Q K_jj^T into S buffer jj & 1 (A = Q, B = K_jj, both K-major)
            auto issue_s = [&](int jj) {
                const uint32_t sK = sKV + kslot(jj) * C::TILE;
                const uint32_t dS = tbase + C::TM_S + (jj & 1) * kBN;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
                    mma_bf16_ss(dS, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024),
                                IDESC_S, ks > 0);
                }
            };
            // dP(jj) = dO V_jj^T into the dP buffer; the commit also covers S(jj)
            auto issue_dp = [&](int jj) {
                const uint32_t sV = sKV + vslot(jj) * C::TILE;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
                    mma_bf16_ss(tDP, sdesc_sw128(sDO + off, 16, 1024),
                                sdesc_sw128(sV + off, 16, 1024), IDESC_S, ks > 0);
                }
                mma_commit(BAR_SDF);
            };
            // dQ += dS_h K_h: dS (bf16) of keys 64h.. at columns [64h, 64h+32) of S
            // buffer jj & 1; K rows 64h.. read MN-major
            auto issue_dq = [&](int jj, int hf) {
                const uint32_t sK = sKV + kslot(jj) * C::TILE;
                const uint32_t aS = tbase + C::TM_S + (jj & 1) * kBN + hf * 64;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_ts(tDQ, aS + ks * 8,
                                sdesc_sw128(sK + hf * C::HALF_ROWS + ks * 2048, C::CHUNK, 1024),
                                IDESC_DQ, (jj == 0 && hf == 0 && ks == 0) ? 0u : 1u);
            };
            bool ok = mbar_wait(BAR_QDO, 0, a.status, a.timeout_ns, 22) && ready(0);
            if (ok) issue_s(0);
            if (ok && (ok = ready(1))) issue_dp(0);
            if (ok && nj > 1 && (ok = ready(2))) issue_s(1);
            for (int j = 0; j < nj && ok; ++j) {
                if (!(ok = mbar_wait(BAR_PF(0), j & 1, a.status, a.timeout_ns, 24))) break;
                tc_fence_after();
                issue_dq(j, 0);
                if (!(ok = mbar_wait(BAR_PF(1), j & 1, a.status, a.timeout_ns, 24))) break;
                tc_fence_after();
                issue_dq(j, 1);
                // K_j and V_j are free once these MMAs complete
                mma_commit(BAR_KVE(kslot(j)));
                mma_commit(BAR_KVE(vslot(j)));
                // both warpgroups have read dP(j): the dP buffer may be overwritten
                if (j + 1 < nj) {
                    if (!(ok = ready(2 * (j + 1) + 1))) break;
                    issue_dp(j + 1);
                }
                // S buffer j & 1 is read by dQ(j) above before S(j+2) lands in it
                if (j + 2 < nj) {
                    if (!(ok = ready(2 * (j + 2)))) break;
                    issue_s(j + 2);
                }
            }
            // every issued MMA has finished before TMEM is released
            mma_commit(BAR_ACC);
            mbar_wait(BAR_ACC, 0, a.status, a.timeout_ns, 25);
        }
        __syncwarp();
    } else if (warp < 8) {
        const int hf = warp >> 2;  // keys 64*hf..64*hf+63 of every block
        const int r = (warp & 3) * 32 + lane;
        const int grow = qi * kBM + r;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tDP = tbase + C::TM_DP + lane_off + hf * 64;
        const bool valid = grow < a.N;
        const size_t st_idx = (static_cast<size_t>(b) * a.Hq + h) * a.N + (valid ? grow : 0);
        const float nlse2 = valid ? -a.lse[st_idx] * kLog2e : 0.f;
        const float dval = valid ? a.dsum[st_idx] : 0.f;
        const float sl2 = a.scale_log2;
        const int lim = a.causal ? min(grow, a.N - 1) : a.N - 1;
        bool ok = true;
        for (int j = 0; j < nj && ok; ++j) {
            if (!(ok = mbar_wait(BAR_SDF, j & 1, a.status, a.timeout_ns, 26))) break;
            tc_fence_after();
            const uint32_t tS = tbase + C::TM_S + (j & 1) * kBN + lane_off + hf * 64;
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
            const uint64_t sl2x2 = f2(sl2, sl2), nlse2x2 = f2(nlse2, nlse2);
            const uint64_t ndx2 = f2(-dval, -dval);
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
                // two columns per packed f32x2 FMA / ADD / MUL
                float x0, x1;
                f2_split(fma2(f2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2, nlse2x2),
                         x0, x1);
                float p0 = ex2(x0), p1 = ex2(x1);
                if (need_mask) {
                    p0 = (kbase + c > lim) ? 0.f : p0;
                    p1 = (kbase + c + 1 > lim) ? 0.f : p1;
                }
                const uint64_t t = add2(f2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])), ndx2);
                float d0, d1;
                f2_split(mul2(f2(p0, p1), t), d0, d1);
                pk[c >> 1] = pack_bf16(d0, d1);
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
            // the Q tile's shared memory (no MMA reads Q any more)
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
