// fa_bwd_dkdv.cu -- dK and dV for exact attention, sm_103a.
//
// One CTA per (batch, kv head, 128-key block).  K and V stay in shared
// memory; Q_i and dO_i of every query head of the GQA group and every query
// block that sees the key block stream through a 2-stage TMA ring, with
// lse * log2(e) and D for the block's queries staged by the TMA warp.  For
// each, S^T = K Q_i^T and dP^T = V dO_i^T are recomputed into TMEM (keys on
// the TMEM lanes), turned into P^T = exp2(S^T * scale * log2(e) - lse2) and
// dS^T = P^T o (dP^T - D) in place (bf16), and dV += P^T dO_i,
// dK += dS^T Q_i take P^T / dS^T straight from TMEM as the A operand -- so no
// transpose is ever materialised.  The group's query heads are summed inside
// the CTA: no atomics.
//
// Pipelining: each 128-query block is split into two 64-query halves with
// their own barriers; warpgroup hf computes half hf while the tensor core
// works on the other half (the dV/dK update of one, the scores of the other).
//
// TMEM (512 columns): S^T [0,128) | dP^T [128,256) | dV [256,256+D) |
// dK [256+D, 256+2D).
#include "fa_bwd_common.cuh"

namespace fa {
namespace {

using namespace bwd;

template <int D>
struct DkdvCfg : Tiles<D> {
    using T = Tiles<D>;
    static constexpr int NST = 2;  // {Q_i, dO_i} ring stages
    // smem: K, V, then NST stages of {Q_i, dO_i}, then per-stage lse2 / D vectors
    static constexpr int OFF_STAGE = 2 * T::TILE;
    static constexpr int OFF_VEC = OFF_STAGE + NST * 2 * T::TILE;
    static constexpr int VEC_BYTES = 2 * kBM * 4;  // lse2[128], D[128]
    static constexpr int OFF_BAR = OFF_VEC + NST * VEC_BYTES;
    static constexpr int NBAR = 1 + 2 * NST + 2 + 2 + 1;
    static constexpr int SMEM_BYTES = 1024 + OFF_BAR + NBAR * 8 + 16;
    static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_ACC = 256;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmDO,
                       const __grid_constant__ CUtensorMap tmDK,
                       const __grid_constant__ CUtensorMap tmDV, const BwdArgs a) {
    using C = DkdvCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sK = smem_u32(smem);
    const uint32_t sV = sK + C::TILE;
    const uint32_t sStage = sK + C::OFF_STAGE;  // stage s: Q at +2s*TILE, dO after it
    float* vec = reinterpret_cast<float*>(smem + C::OFF_VEC);  // stage s: lse2 at s*256, D at +128
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t BAR_KV = bar0;
    auto BAR_STF = [&](int s) { return bar0 + 8u * (1 + s); };
    auto BAR_STE = [&](int s) { return bar0 + 8u * (1 + C::NST + s); };
    const uint32_t BAR_SF0 = bar0 + 8u * (1 + 2 * C::NST);
    auto BAR_SF = [&](int hf) { return BAR_SF0 + 8u * hf; };        // half's S^T, dP^T ready
    auto BAR_PF = [&](int hf) { return BAR_SF0 + 8u * (2 + hf); };  // half's P^T, dS^T written
    const uint32_t BAR_ACC = BAR_SF0 + 8u * 4;

    const int warp = warp_id();
    const int lane = lane_id();
    const int nqb = (a.N + kBM - 1) / kBM;
    const int per = a.B * a.Hkv;
    const int jb = static_cast<int>(blockIdx.x) / per;  // causal: low key blocks have most work
    const int bh = static_cast<int>(blockIdx.x) % per;
    const int b = bh / a.Hkv;
    const int hk = bh % a.Hkv;
    const int qi0 = a.causal ? jb : 0;  // first query block that sees this key block
    const int nqi = nqb - qi0;
    const int n_it = a.g * nqi;         // (query head of the group, query block) pairs

    if (warp == 0 && lane == 0) {
        mbar_init(BAR_KV, 1);
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(BAR_STF(s), 1 + 32);  // TMA transaction arrive + 32 lanes' vector writes
            mbar_init(BAR_STE(s), 1);
        }
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
        // TMA for tiles (lane 0); all 32 lanes fill the per-query lse2 / D vectors
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmDO);
            tma_prefetch_desc(&tmDK);
            tma_prefetch_desc(&tmDV);
            mbar_arrive_expect_tx(BAR_KV, 2 * C::TILE);
            for (int c = 0; c < C::NCH; ++c) {
                tma_load_4d(sK + c * C::CHUNK, &tmK, BAR_KV, c * 64, hk, jb * kBN, b);
                tma_load_4d(sV + c * C::CHUNK, &tmV, BAR_KV, c * 64, hk, jb * kBN, b);
            }
        }
        const uint64_t pol_q = l2_policy_evict_last();
        int last_it[C::NST] = {-1, -1};
        for (int it = 0; it < n_it; ++it) {
            const int s = it % C::NST;
            const int hq = hk * a.g + it / nqi;
            const int qi = qi0 + it % nqi;
            if (!mbar_wait(BAR_STE(s), ((it / C::NST) & 1) ^ 1u, a.status, a.timeout_ns, 30)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(BAR_STF(s), 2 * C::TILE);
                const uint32_t dst = sStage + 2 * s * C::TILE;
                for (int c = 0; c < C::NCH; ++c) {
                    tma_load_4d_hint(dst + c * C::CHUNK, &tmQ, BAR_STF(s), c * 64, hq, qi * kBM, b,
                                     pol_q);
                    tma_load_4d_hint(dst + C::TILE + c * C::CHUNK, &tmDO, BAR_STF(s), c * 64, hq,
                                     qi * kBM, b, pol_q);
                }
            }
            float* lse2 = vec + s * 2 * kBM;
            float* dv = lse2 + kBM;
            const size_t base = (static_cast<size_t>(b) * a.Hq + hq) * a.N;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = lane * 4 + u;
                const int q = qi * kBM + c;
                // a query row past N contributes nothing: P = exp2(-inf) = 0
                lse2[c] = (q < a.N) ? a.lse[base + q] * kLog2e : INFINITY;
                dv[c] = (q < a.N) ? a.dsum[base + q] : 0.f;
            }
            mbar_arrive(BAR_STF(s));
            last_it[s] = it;
        }
        if (lane == 0) {  // no copies in flight at exit
            mbar_wait(BAR_KV, 0, a.status, a.timeout_ns, 31);
            for (int s = 0; s < C::NST; ++s)
                if (last_it[s] >= 0)
                    mbar_wait(BAR_STF(s), (last_it[s] / C::NST) & 1, a.status, a.timeout_ns, 31);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(kBN, 64, false, false);  // S^T, dP^T halves
            constexpr uint32_t IDESC_ACC = idesc_bf16(kBN, D, false, true);  // dV, dK
            const uint32_t tS = tbase + C::TM_S, tDP = tbase + C::TM_DP;
            const uint32_t tDV = tbase + C::TM_ACC, tDK = tbase + C::TM_ACC + D;
            // S^T, dP^T for query half hf of stage s: B = rows 64*hf.. of Q_i / dO_i
            auto issue_s = [&](int hf, int s) {
                const uint32_t sQ = sStage + 2 * s * C::TILE, sDO = sQ + C::TILE;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
                    mma_bf16_ss(tS + hf * 64, sdesc_sw128(sK + off, 16, 1024),
                                sdesc_sw128(sQ + off + hf * C::HALF_ROWS, 16, 1024), IDESC_S, ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
                    mma_bf16_ss(tDP + hf * 64, sdesc_sw128(sV + off, 16, 1024),
                                sdesc_sw128(sDO + off + hf * C::HALF_ROWS, 16, 1024), IDESC_S,
                                ks > 0);
                }
                mma_commit(BAR_SF(hf));
            };
            // dV += P^T_h dO_h, dK += dS^T_h Q_h: P^T / dS^T (bf16) at columns
            // [64*hf, 64*hf+32) of S^T / dP^T; dO, Q rows 64*hf.. read MN-major
            auto issue_acc = [&](int hf, int s, bool first) {
                const uint32_t sQ = sStage + 2 * s * C::TILE, sDO = sQ + C::TILE;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t acc = (first && ks == 0) ? 0u : 1u;
                    const uint32_t boff = hf * C::HALF_ROWS + ks * 2048;
                    mma_bf16_ts(tDV, tS + hf * 64 + ks * 8, sdesc_sw128(sDO + boff, C::CHUNK, 1024),
                                IDESC_ACC, acc);
                    mma_bf16_ts(tDK, tDP + hf * 64 + ks * 8, sdesc_sw128(sQ + boff, C::CHUNK, 1024),
                                IDESC_ACC, acc);
                }
            };
            bool ok = mbar_wait(BAR_KV, 0, a.status, a.timeout_ns, 32) &&
                      mbar_wait(BAR_STF(0), 0, a.status, a.timeout_ns, 33);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                issue_s(1, 0);
            }
            for (int it = 0; it < n_it && ok; ++it) {
                const int s = it % C::NST;
                const int s2 = (it + 1) % C::NST;
                if (!(ok = mbar_wait(BAR_PF(0), it & 1, a.status, a.timeout_ns, 34))) break;
                tc_fence_after();
                issue_acc(0, s, it == 0);
                if (it + 1 < n_it) {
                    if (!(ok = mbar_wait(BAR_STF(s2), ((it + 1) / C::NST) & 1, a.status,
                                         a.timeout_ns, 33)))
                        break;
                    tc_fence_after();
                    issue_s(0, s2);
                }
                if (!(ok = mbar_wait(BAR_PF(1), it & 1, a.status, a.timeout_ns, 34))) break;
                tc_fence_after();
                issue_acc(1, s, false);
                mma_commit(BAR_STE(s));
                if (it + 1 < n_it) issue_s(1, s2);
            }
            // every issued MMA has finished before TMEM is released
            mma_commit(BAR_ACC);
            mbar_wait(BAR_ACC, 0, a.status, a.timeout_ns, 35);
        }
        __syncwarp();
    } else if (warp < 8) {
        const int hf = warp >> 2;  // query half (0: queries 0-63, 1: 64-127) of each block
        const int r = (warp & 3) * 32 + lane;
        const int key = jb * kBN + r;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tbase + C::TM_S + lane_off + hf * 64;
        const uint32_t tDP = tbase + C::TM_DP + lane_off + hf * 64;
        const float sl2 = a.scale_log2;
        bool ok = true;
        for (int it = 0; it < n_it; ++it) {
            const int s = it % C::NST;
            const int qi = qi0 + it % nqi;
            if (!(ok = mbar_wait(BAR_SF(hf), it & 1, a.status, a.timeout_ns, 36))) break;
            tc_fence_after();
            uint32_t sv[64], dp[64];
            tmem_ld32(tS, sv);
            tmem_ld32(tS + 32, sv + 32);
            tmem_ld32(tDP, dp);
            tmem_ld32(tDP + 32, dp + 32);
            tmem_wait_ld();
            reg_fence<64>(sv);
            reg_fence<64>(dp);
            const float* lse2 = vec + s * 2 * kBM + hf * 64;
            const float* dvec = vec + s * 2 * kBM + kBM + hf * 64;
            const int qbase = qi * kBM + hf * 64;
            // causal: key r is hidden from query q when key > q
            const bool need_mask = a.causal && key > qbase;
            const uint64_t sl2x2 = f2(sl2, sl2);
            uint32_t pk[32], dk[32];
#pragma unroll
            for (int c = 0; c < 64; c += 4) {
                const float4 l4 = *reinterpret_cast<const float4*>(lse2 + c);
                const float4 d4 = *reinterpret_cast<const float4*>(dvec + c);
                // two columns per packed f32x2 FMA / ADD / MUL
                float x[4], p[4], e[4];
                f2_split(fma2(f2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2,
                              f2(-l4.x, -l4.y)), x[0], x[1]);
                f2_split(fma2(f2(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), sl2x2,
                              f2(-l4.z, -l4.w)), x[2], x[3]);
#pragma unroll
                for (int u = 0; u < 4; ++u) p[u] = ex2(x[u]);
                if (need_mask) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) p[u] = (key > qbase + c + u) ? 0.f : p[u];
                }
                f2_split(mul2(f2(p[0], p[1]),
                              add2(f2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])),
                                   f2(-d4.x, -d4.y))), e[0], e[1]);
                f2_split(mul2(f2(p[2], p[3]),
                              add2(f2(__uint_as_float(dp[c + 2]), __uint_as_float(dp[c + 3])),
                                   f2(-d4.z, -d4.w))), e[2], e[3]);
                pk[c >> 1] = pack_bf16(p[0], p[1]);
                pk[(c >> 1) + 1] = pack_bf16(p[2], p[3]);
                dk[c >> 1] = pack_bf16(e[0], e[1]);
                dk[(c >> 1) + 1] = pack_bf16(e[2], e[3]);
            }
            tmem_st32(tS, pk);   // P^T over this half's S^T columns
            tmem_st32(tDP, dk);  // dS^T over this half's dP^T columns
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR_PF(hf));
        }
        const bool ok_e = ok && mbar_wait(BAR_ACC, 0, a.status, a.timeout_ns, 37);
        // warpgroup 0 writes dV, warpgroup 1 writes dK = scale * (dS^T Q); staging
        // reuses stage 0's Q (dV) and dO (dK) buffers, idle once all MMAs are done
        const uint32_t stage = sStage + hf * C::TILE;
        if (ok_e) {
            tc_fence_after();
            stage_rows_bf16<C::CHUNK>(tbase + C::TM_ACC + hf * D + lane_off, stage, r, 0, D,
                                      hf ? a.scale : 1.f);
            fence_proxy_async_smem();
        }
        named_bar_sync(1 + hf, 128);
        if (ok_e && r == 0) {
            const CUtensorMap* tm = hf ? &tmDK : &tmDV;
            for (int c = 0; c < C::NCH; ++c)
                tma_store_4d(tm, stage + c * C::CHUNK, c * 64, hk, jb * kBN, b);
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
cudaError_t launch_bwd_dkdv(const BwdMaps& m, const BwdArgs& a, cudaStream_t st) {
    auto kern = fa_bwd_dkdv_kernel<D>;
    constexpr int smem = DkdvCfg<D>::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long nblk = static_cast<long long>((a.N + kBN - 1) / kBN) * a.B * a.Hkv;
    if (nblk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<static_cast<unsigned>(nblk), kThreads, smem, st>>>(m.q, m.k, m.v, m.dout, m.dk, m.dv,
                                                              a);
    return cudaGetLastError();
}

template cudaError_t launch_bwd_dkdv<64>(const BwdMaps&, const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_dkdv<128>(const BwdMaps&, const BwdArgs&, cudaStream_t);

}  // namespace fa
