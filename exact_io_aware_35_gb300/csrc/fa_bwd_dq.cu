// fa_bwd_dq.cu -- dQ = scale * dS K for exact attention, sm_103a.
//
// One CTA per (batch, query head, 128-query block).  Recomputes, for every key
// block j the block sees, S = Q K_j^T and dP = dO V_j^T, then
// P = exp2(S * scale * log2(e) - lse * log2(e)) and dS = P o (dP - D), and
// accumulates dQ += dS K_j in tensor memory (the recomputation the pages
// describe for the backward pass: "FlashAttention Kernel", recomputation
// bullet; the gradient formulas are the derivative of the forward definition).
//
// Pipelining.  Every MMA is 128 wide.  dP is double-buffered in TMEM and S is
// not: as soon as both warpgroups have copied S(j) and dP(j) into registers
// (barrier LD), the tensor core computes S(j+1) into the S buffer, while the
// warpgroups write dS(j) (bf16 or fp16) over the dP(j) columns they read.
// dQ += dS(j) K_j then reads it from there (barrier PF), and dP(j+2) follows
// dQ(j) at once into that buffer: it waits for nothing the warps do, so it is
// done long before they reach block j+2.  The tensor core's order per block is
// S(j+1), dQ(j), dP(j+2); the warpgroups find S and dP ready at every block.
// Four compute warpgroups: warpgroup h takes keys 32h..32h+31 of every block
// and writes their dS into the first 16 of its own 32 dP columns, which keeps
// the chain of loads, exponentials and stores per block short.  K and V stream through
// separate TMA rings, loaded in the products' first-use order (K_0, V_0, V_1,
// K_1, V_2, K_2, ...); a gate warp adds one arrival to LD(j) once K_{j+1} has
// landed, so S(j+1) needs one wait in the issuing thread (every wait there
// costs tensor-core time); V_{j+2}, loaded two blocks ahead, is checked by the
// MMA thread itself before dP(j+2).  Only LD carries the gate:
// the warpgroups reach LD(j+1) only after S(j+1), which waits for LD(j), so no
// arrival can land in the wrong phase.  PF needs one more step, because S(j+1)
// is committed before the MMA thread waits for PF(j): the MMA thread arrives
// on PFS once it has seen PF(j) complete, and a warp waits for that before its
// PF(j+1) arrival.  Without it a warp that ran a block ahead could arrive in
// PF(j)'s phase, or PF could complete twice under the MMA thread's parity wait.
//
// TMEM (512 columns): S [0,128), dP0 [128,256), dP1 [256,384), dQ [384,384+D).
#include "fa_bwd_common.cuh"

namespace fa {
namespace {

using namespace bwd;

// 16 compute warps (four warpgroups), then the MMA, TMA, gate and copy warps
constexpr int kDqCompute = 512;
constexpr int kDqWarpMma = 16;
constexpr int kDqWarpLoad = 17;
constexpr int kDqWarpGate = 18;
constexpr int kDqWarpCopy = 19;
constexpr int kDqThreads = 640;

template <int D>
struct DqCfg : Tiles<D> {
    using T = Tiles<D>;
    // K ring: K_j (dQ), K_{j+1} (S), loads ahead; V ring: V_{j+2} (dP), loads
    // ahead.  A tile lands about a block's time after its load starts, and at
    // d = 128 (32 KB tiles) shared memory holds only one slot ahead of each;
    // at d = 64 (16 KB) each ring gets one more.
    static constexpr int KS = (D == 64) ? 4 : 3;
    static constexpr int VS = (D == 64) ? 3 : 2;
    static constexpr int OFF_K = 2 * T::TILE;  // after Q, dO
    static constexpr int OFF_V = OFF_K + KS * T::TILE;
    static constexpr int OFF_BAR = OFF_V + VS * T::TILE;
    // barriers: Q/dO, K full/empty[KS], V full/empty[VS], S+dP ready, copied to
    // registers, dS written, all MMAs done, dS written seen by the MMA thread
    static constexpr int NBAR = 1 + 2 * KS + 2 * VS + 5;
    static constexpr int SMEM_BYTES = 1024 + OFF_BAR + NBAR * 8 + 16;
    static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DQ = 384;
};

// The fp16 operand scales from the four maxima in absmax (one 16-byte load).
template <int D>
__device__ __forceinline__ F16Scales scales_of(const uint32_t* absmax) {
    int m[4];
    ld_once_v4(reinterpret_cast<const int*>(absmax), m[0], m[1], m[2], m[3]);
    const uint32_t u[4] = {static_cast<uint32_t>(m[0]), static_cast<uint32_t>(m[1]),
                           static_cast<uint32_t>(m[2]), static_cast<uint32_t>(m[3])};
    return f16_scales_from(u, D);
}

// F16: Q and K tiles are the fp16 copies (scaled by 2^q, 2^k; S carries
// 2^(q+k), folded into scale * log2 e) and dS * 2^ds is rounded to fp16, so
// dQ carries 2^(ds+k), undone in the epilogue.  dO and V stay bf16: dP is
// not rounded before use.
template <int D, bool F16>
__global__ void __launch_bounds__(kDqThreads, 1)
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
    const uint32_t sK = sQ + C::OFF_K;  // K_j in slot j % KS
    const uint32_t sV = sQ + C::OFF_V;  // V_j in slot j % VS
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t BAR_QDO = bar0;  // Q, dO tiles landed
    auto BAR_KF = [&](int s) { return bar0 + 8u * (1 + s); };
    auto BAR_KE = [&](int s) { return bar0 + 8u * (1 + C::KS + s); };
    auto BAR_VF = [&](int s) { return bar0 + 8u * (1 + 2 * C::KS + s); };
    auto BAR_VE = [&](int s) { return bar0 + 8u * (1 + 2 * C::KS + C::VS + s); };
    const uint32_t BAR_SDF = bar0 + 8u * (1 + 2 * C::KS + 2 * C::VS);  // S(j), dP(j) ready
    const uint32_t BAR_LD = BAR_SDF + 8u;   // S(j), dP(j) copied to registers
    const uint32_t BAR_PF = BAR_SDF + 16u;  // dS(j) written
    const uint32_t BAR_ACC = BAR_SDF + 24u;
    const uint32_t BAR_PFS = BAR_SDF + 32u;  // the MMA thread has seen PF(j) complete

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
        for (int s = 0; s < C::KS; ++s) {
            mbar_init(BAR_KF(s), 1);
            mbar_init(BAR_KE(s), 1);
        }
        for (int s = 0; s < C::VS; ++s) {
            mbar_init(BAR_VF(s), 1);
            mbar_init(BAR_VE(s), 1);
        }
        mbar_init(BAR_SDF, 1);
        mbar_init(BAR_LD, kDqCompute + 1);  // compute threads and the gate
        mbar_init(BAR_PF, kDqCompute);
        mbar_init(BAR_ACC, 1);
        mbar_init(BAR_PFS, 1);
        fence_barrier_init();
    }
    if (warp == kDqWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    // Registers: 640 threads launch with 96 each (61,440); the compute
    // warpgroups take 104 and the issue warpgroup keeps 64
    // (512 x 104 + 128 x 64 = 61,440).

    if (warp == kDqWarpLoad) {
        setmaxnreg_dec<64>();
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
            int last_k[C::KS], last_v[C::VS];
            for (int s = 0; s < C::KS; ++s) last_k[s] = -1;
            for (int s = 0; s < C::VS; ++s) last_v[s] = -1;
            // key block jj of K (isv = 0) or V (isv = 1) into its ring; the first
            // use of a slot waits on parity 1, which a fresh barrier reports complete
            auto load = [&](int jj, bool isv) {
                const int ns = isv ? C::VS : C::KS;
                const int slot = jj % ns;
                const uint32_t ph = ((jj / ns) & 1) ^ 1u;
                if (!mbar_wait(isv ? BAR_VE(slot) : BAR_KE(slot), ph, a.watch, 20))
                    return false;
                const uint32_t full = isv ? BAR_VF(slot) : BAR_KF(slot);
                const uint32_t dst = (isv ? sV : sK) + slot * C::TILE;
                mbar_arrive_expect_tx(full, C::TILE);
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_4d_hint(dst + c * C::CHUNK, isv ? &tmV : &tmK, full, c * 64, hk,
                                     jj * kBN, b, pol_kv);
                if (isv)
                    last_v[slot] = jj;
                else
                    last_k[slot] = jj;
                return true;
            };
            // first-use order of the MMAs: K_0, V_0, V_1, K_1, V_2, K_2, ...
            bool ok = load(0, false) && load(0, true);
            for (int i = 1; i < nj && ok; ++i) ok = load(i, true) && load(i, false);
            // no copies in flight at exit: wait (bounded) for the last load of each slot
            mbar_drain(BAR_QDO, 0, a.watch, 21);
            for (int s = 0; s < C::KS; ++s)
                if (last_k[s] >= 0)
                    mbar_drain(BAR_KF(s), (last_k[s] / C::KS) & 1, a.watch, 21);
            for (int s = 0; s < C::VS; ++s)
                if (last_v[s] >= 0)
                    mbar_drain(BAR_VF(s), (last_v[s] / C::VS) & 1, a.watch, 21);
        }
        __syncwarp();
    } else if (warp == kDqWarpGate) {
        // ================= gate: K_{j+1} landed -> LD(j) =================
        // Its arrival on LD(j) comes only after LD's previous phase is over.
        setmaxnreg_dec<64>();
        if (lane == 0) {
            bool ok = true;
            for (int j = 0; j < nj && ok; ++j) {
                if (j + 1 < nj)
                    ok = mbar_wait(BAR_KF((j + 1) % C::KS), ((j + 1) / C::KS) & 1, a.watch, 28);
                if (ok && j > 0) ok = mbar_wait(BAR_LD, (j - 1) & 1, a.watch, 28);
                if (ok) mbar_arrive(BAR_LD);
            }
        }
        __syncwarp();
    } else if (warp == kDqWarpCopy) {
        // ============ copy: dO tile -> fp16(dO * 2^s) (fp16 operand path) ============
        // The scales come from the maxima in absmax (taken before this kernel);
        // block 0 stores them for the dK/dV kernel, which also reads the copy.
        setmaxnreg_dec<64>();
        if (F16) {
            const F16Scales sc = scales_of<D>(a.absmax);
            if (blockIdx.x == 0 && lane == 0) *a.scales_w = sc;
            const float mul = pow2f(sc.dout);
            const size_t row_el = static_cast<size_t>(a.Hq) * D;  // elements per token
            uint16_t* dst = a.dout16 + (static_cast<size_t>(b) * a.N + qi * kBM) * row_el + h * D;
            if (mbar_wait_warp(BAR_QDO, 0, a.watch, 29))
                warp_tile_to_f16<D>(sDO, dst, row_el, a.N - qi * kBM, mul, lane);
        }
        __syncwarp();
    } else if (warp == kDqWarpMma) {
        // ================= MMA issuer (the whole warp; the leader lane issues) =================
        setmaxnreg_dec<64>();
        {
            const uint32_t leader = elect_one();
            constexpr uint32_t IDESC_S = idesc_16(kBM, kBN, false, false, F16);  // S = Q K^T
            constexpr uint32_t IDESC_DP = idesc_bf16(kBM, kBN, false, false);    // dP = dO V^T
            constexpr uint32_t IDESC_DQ = idesc_16(kBM, D, false, true, F16);    // dQ += dS K
            const uint32_t tS = tbase + C::TM_S, tDQ = tbase + C::TM_DQ;
            auto tDP = [&](int jj) { return tbase + C::TM_DP + (jj & 1) * 128; };
            auto k_ready = [&](int jj) {
                const bool r = mbar_wait_warp(BAR_KF(jj % C::KS), (jj / C::KS) & 1, a.watch, 23);
                tc_fence_after();
                return r;
            };
            auto v_ready = [&](int jj) {
                const bool r = mbar_wait_warp(BAR_VF(jj % C::VS), (jj / C::VS) & 1, a.watch, 23);
                tc_fence_after();
                return r;
            };
            // descriptors: K-major tiles (S, dP operands) and the MN-major K tile
            // (dQ), built once; each MMA only moves the start address
            constexpr uint32_t HI = sdesc_hi(1024);
            const uint32_t q_lo = sdesc_lo(sQ, 16), do_lo = sdesc_lo(sDO, 16);
            // dst = A B^T over the head dimension (both K-major): S = Q K^T, dP = dO V^T
            auto issue_t = [&](uint32_t dst, uint32_t a_lo, uint32_t sB, uint32_t idesc) {
                const uint32_t b_lo = sdesc_lo(sB, 16);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
                    mma_bf16_ss_w(leader, dst, sdesc_at(a_lo, HI, off), sdesc_at(b_lo, HI, off), idesc, ks > 0);
                }
            };
            // dP(jj) = dO V_jj^T; V_jj's slot is free once it has run
            auto issue_dp = [&](int jj) {
                issue_t(tDP(jj), do_lo, sV + (jj % C::VS) * C::TILE, IDESC_DP);
                mma_commit_w(leader, BAR_VE(jj % C::VS));
            };
            // dQ += dS(jj) K_jj: dS (packed pairs) of keys 16ks.. at columns
            // 32(ks/2) + (ks%2)*8 of dP buffer jj & 1; K rows 16ks.. read MN-major.
            // The caller commits K_jj's slot free (after the next dP, so that
            // the two batches go to the tensor core back to back).
            auto issue_dq = [&](int jj) {
                const uint32_t k_lo = sdesc_lo(sK + (jj % C::KS) * C::TILE, C::CHUNK), aS = tDP(jj);
#pragma unroll
                for (int ks = 0; ks < kBN / 16; ++ks)
                    mma_bf16_ts_w(leader, tDQ, aS + (ks >> 1) * 32 + (ks & 1) * 8,
                                  sdesc_at(k_lo, HI, ks * 2048), IDESC_DQ,
                                  (jj == 0 && ks == 0) ? 0u : 1u);
            };
            bool ok = mbar_wait_warp(BAR_QDO, 0, a.watch, 22) && k_ready(0);
            if (ok) issue_t(tS, q_lo, sK, IDESC_S);
            if (ok && (ok = v_ready(0))) {
                issue_dp(0);
                mma_commit_w(leader, BAR_SDF);
            }
            if (ok && nj > 1 && (ok = v_ready(1))) issue_dp(1);  // into the other dP buffer
            for (int j = 0; j < nj && ok; ++j) {
                // S(j+1) into the S buffer once both warpgroups hold S(j), dP(j)
                // and K_{j+1} has landed (the gate's arrival on LD); its commit
                // also covers dP(j+1), issued a block earlier
                if (j + 1 < nj) {
                    if (!(ok = mbar_wait_warp(BAR_LD, j & 1, a.watch, 24))) break;
                    tc_fence_after();
                    issue_t(tS, q_lo, sK + ((j + 1) % C::KS) * C::TILE, IDESC_S);
                    mma_commit_w(leader, BAR_SDF);
                }
                if (!(ok = mbar_wait_warp(BAR_PF, j & 1, a.watch, 24))) break;
                if (leader) mbar_arrive(BAR_PFS);  // the warps may now arrive on PF(j+1)
                tc_fence_after();
                issue_dq(j);
                // dP(j+2) over dS(j), which dQ(j), issued just before by this
                // thread, reads first
                if (j + 2 < nj) {
                    if (!(ok = v_ready(j + 2))) break;
                    issue_dp(j + 2);
                }
                mma_commit_w(leader, BAR_KE(j % C::KS));  // dQ(j) was K_j's last reader
            }
            // every issued MMA has finished before TMEM is released
            mma_commit_w(leader, BAR_ACC);
            mbar_drain(BAR_ACC, 0, a.watch, 25);
        }
        __syncwarp();
    } else if (warp < 16) {
        setmaxnreg_inc<104>();
        const int hf = warp >> 2;  // keys 32*hf..32*hf+31 of every block
        const int r = (warp & 3) * 32 + lane;
        const int grow = qi * kBM + r;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tbase + C::TM_S + lane_off + hf * 32;
        const bool valid = grow < a.N;
        const size_t st_idx = (static_cast<size_t>(b) * a.Hq + h) * a.N + (valid ? grow : 0);
        const float nlse2 = valid ? -a.lse[st_idx] * kLog2e : 0.f;
        const float dval = valid ? a.dsum[st_idx] : 0.f;
        // fp16 path: undo 2^(q+k) on S; dS = P (dP - D) carries 2^ds
        int eq = 0, ek = 0, eds = 0;
        if (F16) {
            const F16Scales sc = scales_of<D>(a.absmax);
            eq = sc.q;
            ek = sc.k;
            eds = sc.ds;
        }
        const float sl2 = a.scale_log2 * pow2f(-(eq + ek));
        const float dsc = pow2f(eds);
        const int lim = a.causal ? min(grow, a.N - 1) : a.N - 1;
        const uint64_t sl2x2 = f2(sl2, sl2), nlse2x2 = f2(nlse2, nlse2);
        const uint64_t ndx2 = f2(-dval * dsc, -dval * dsc), dsc2 = f2(dsc, dsc);
        bool ok = true;
        for (int j = 0; j < nj && ok; ++j) {
            if (!(ok = mbar_wait_warp(BAR_SDF, j & 1, a.watch, 26))) break;
            tc_fence_after();
            const uint32_t tDP = tbase + C::TM_DP + (j & 1) * 128 + lane_off + hf * 32;
            uint32_t sv[32], dp[32];
            tmem_ld32(tS, sv);
            tmem_ld32(tDP, dp);
            tmem_wait_ld();
            reg_fence<32>(sv);
            reg_fence<32>(dp);
            // both buffers are in registers: S(j+1) may now overwrite S(j)
            tc_fence_before();
            mbar_arrive(BAR_LD);
            const int kbase = j * kBN + hf * 32;
            const bool need_mask = kbase + 31 > lim;
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
                // two columns per packed f32x2 FMA / ADD / MUL
                float x0, x1;
                f2_split(fma2(f2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2, nlse2x2),
                         x0, x1);
                float p0 = ex2(x0), p1 = ex2(x1);
                if (need_mask) {
                    p0 = (kbase + c > lim) ? 0.f : p0;
                    p1 = (kbase + c + 1 > lim) ? 0.f : p1;
                }
                const uint64_t t =
                    fma2(f2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])), dsc2, ndx2);
                float d0, d1;
                f2_split(mul2(f2(p0, p1), t), d0, d1);
                pk[c >> 1] = pack_op<F16>(d0, d1);
            }
            tmem_st16(tDP, pk);  // dS over the first 16 of this quarter's dP columns
            tmem_wait_st();
            tc_fence_before();
            // S(j), dP(j) were issued before the MMA thread waits for PF(j-1):
            // arriving on PF(j) only once that thread has seen PF(j-1) keeps a
            // fast warp's arrival out of PF(j-1)'s phase and PF from running
            // two phases ahead of the thread's parity wait
            if (j > 0 && !(ok = mbar_wait_warp(BAR_PFS, (j - 1) & 1, a.watch, 39))) break;
            mbar_arrive(BAR_PF);
        }
        const bool ok_e = ok && mbar_wait_warp(BAR_ACC, 0, a.watch, 27);
        if (ok_e) {
            tc_fence_after();
            // dQ = scale * (dS K): the warpgroups stage 32-column slices of it
            // into the Q tile's shared memory (no MMA reads Q any more)
            if (hf * 32 < D)
                stage_rows_bf16<C::CHUNK>(tbase + C::TM_DQ + lane_off, sQ, r, hf * 32, hf * 32 + 32,
                                          a.scale * pow2f(-(eds + ek)));
            fence_proxy_async_smem();
        }
        named_bar_sync(1, kDqCompute);
        if (ok_e && warp == 0 && lane == 0) {
            for (int c = 0; c < C::NCH; ++c)
                tma_store_4d(&tmDQ, sQ + c * C::CHUNK, c * 64, h, qi * kBM, b);
            tma_store_commit();
            tma_store_wait_read_all();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kDqWarpMma) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

}  // namespace

template <int D, bool F16>
cudaError_t launch_dq(const BwdMaps& m, const BwdArgs& a, cudaStream_t st) {
    auto kern = fa_bwd_dq_kernel<D, F16>;
    constexpr int smem = DqCfg<D>::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long nblk = static_cast<long long>((a.N + kBM - 1) / kBM) * a.B * a.Hq;
    if (nblk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<static_cast<unsigned>(nblk), kDqThreads, smem, st>>>(F16 ? m.q16 : m.q, F16 ? m.k16 : m.k,
                                                            m.v, m.dout, m.dq, a);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_dq(const BwdMaps& m, const BwdArgs& a, cudaStream_t st) {
    return a.f16s ? launch_dq<D, true>(m, a, st) : launch_dq<D, false>(m, a, st);
}

template cudaError_t launch_bwd_dq<64>(const BwdMaps&, const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_dq<128>(const BwdMaps&, const BwdArgs&, cudaStream_t);

}  // namespace fa
