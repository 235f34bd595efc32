// fa_bwd_dq.cu -- dQ = scale * dS K for exact attention, sm_103a.
//
// Work items are (batch, query head, 128-query block).  Recomputes, for every key
// block j an item sees, S = Q K_j^T and dP = dO V_j^T, then
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
// Items.  At d = 64 the CTAs are persistent (one per SM, items dealt longest
// first) and blocks carry global indices across a CTA's items, so the rings,
// the dP buffers and the per-block barriers run on: the next item's Q and dO
// load once its predecessor's last S and dP are done and the copy warp has
// read dO (barrier QE), and its first S and dP run while the warps finish the
// previous item's blocks and epilogue.  The warps stage dQ in a buffer of its
// own (barrier EPF) and the copy warp stores it from there (EPE frees it
// again).  At d = 128 shared memory has no room for that buffer: one item per
// CTA, dQ staged in the Q tile.
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
    // d = 64: persistent CTAs, one per SM, dealt items longest first; dQ is
    // staged for its TMA store in a buffer of its own, so the next item's Q
    // tile can land meanwhile.  d = 128 has no room for that buffer: one item
    // per CTA, dQ staged in the Q tile once no score product reads it.
    static constexpr bool PERSIST = (D == 64);
    static constexpr int OFF_K = 2 * T::TILE;  // after Q, dO
    static constexpr int OFF_V = OFF_K + KS * T::TILE;
    static constexpr int OFF_ST = OFF_V + VS * T::TILE;
    static constexpr int OFF_BAR = OFF_ST + (PERSIST ? T::TILE : 0);
    // barriers: Q/dO full, K full/empty[KS], V full/empty[VS], S+dP ready,
    // copied to registers, dS written, an item's MMAs done, dS written seen by
    // the MMA thread, Q/dO free, dQ staged, staging free, all MMAs done
    static constexpr int NBAR = 1 + 2 * KS + 2 * VS + 5 + 4;
    static constexpr int SMEM_BYTES = 1024 + OFF_BAR + NBAR * 8 + 16;
    static_assert(SMEM_BYTES <= 232448, "dynamic shared memory above the 227 KB a block may use");
    static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DQ = 384;
};

// One work item: (batch, query head, 128-query block), longest first.
struct DqItem {
    int b, h, hk, qi, nj;
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
    const uint32_t sK = sQ + C::OFF_K;  // global block g's K in slot g % KS
    const uint32_t sV = sQ + C::OFF_V;  // global block g's V in slot g % VS
    const uint32_t sST = C::PERSIST ? sQ + C::OFF_ST : sQ;  // dQ staged for its TMA store
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t BAR_QDO = bar0;  // the item's Q, dO tiles landed
    auto BAR_KF = [&](int s) { return bar0 + 8u * (1 + s); };
    auto BAR_KE = [&](int s) { return bar0 + 8u * (1 + C::KS + s); };
    auto BAR_VF = [&](int s) { return bar0 + 8u * (1 + 2 * C::KS + s); };
    auto BAR_VE = [&](int s) { return bar0 + 8u * (1 + 2 * C::KS + C::VS + s); };
    const uint32_t BAR_SDF = bar0 + 8u * (1 + 2 * C::KS + 2 * C::VS);  // S(g), dP(g) ready
    const uint32_t BAR_LD = BAR_SDF + 8u;    // S(g), dP(g) copied to registers
    const uint32_t BAR_PF = BAR_SDF + 16u;   // dS(g) written
    const uint32_t BAR_ACC = BAR_SDF + 24u;  // the item's dQ complete in TMEM
    const uint32_t BAR_PFS = BAR_SDF + 32u;  // the MMA thread has seen PF(g) complete
    const uint32_t BAR_QE = BAR_SDF + 40u;   // the item's Q, dO no longer read
    const uint32_t BAR_EPF = BAR_SDF + 48u;  // the item's dQ staged
    const uint32_t BAR_EPE = BAR_SDF + 56u;  // the staging buffer stored (free again)
    const uint32_t BAR_DONE = BAR_SDF + 64u;

    const int warp = warp_id();
    const int lane = lane_id();
    const int nqb = (a.N + kBM - 1) / kBM;
    const int per = a.B * a.Hq;
    const int n_items = nqb * per;
    const int nkv_all = (a.N + kBN - 1) / kBN;
    // Blocks carry global indices g across the CTA's items, so the K/V rings,
    // the dP buffers (g % 2) and the per-block barriers run on from one item
    // to the next.
    auto item = [&](int w) {
        DqItem I;
        I.qi = nqb - 1 - w / per;  // longest first
        const int bh = w % per;
        I.b = bh / a.Hq;
        I.h = bh % a.Hq;
        I.hk = I.h / a.g;
        I.nj = a.causal ? min(I.qi + 1, nkv_all) : nkv_all;
        return I;
    };

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
        mbar_init(BAR_QE, F16 ? 2 : 1);  // the MMA thread's commit, the copy warp
        mbar_init(BAR_EPF, kDqCompute);
        mbar_init(BAR_EPE, 1);
        mbar_init(BAR_DONE, 1);
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
            int last_k[C::KS], last_v[C::VS];
            for (int s = 0; s < C::KS; ++s) last_k[s] = -1;
            for (int s = 0; s < C::VS; ++s) last_v[s] = -1;
            // global block g (key block kb of item I) of K (isv = 0) or V (isv =
            // 1) into its ring; the first use of a slot waits on parity 1, which
            // a fresh barrier reports complete
            auto load = [&](int g, int kb, const DqItem& I, bool isv) {
                const int ns = isv ? C::VS : C::KS;
                const int slot = g % ns;
                const uint32_t ph = ((g / ns) & 1) ^ 1u;
                if (!mbar_wait(isv ? BAR_VE(slot) : BAR_KE(slot), ph, a.watch, 20))
                    return false;
                const uint32_t full = isv ? BAR_VF(slot) : BAR_KF(slot);
                const uint32_t dst = (isv ? sV : sK) + slot * C::TILE;
                mbar_arrive_expect_tx(full, C::TILE);
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_4d_hint(dst + c * C::CHUNK, isv ? &tmV : &tmK, full, c * 64, I.hk,
                                     kb * kBN, I.b, pol_kv);
                if (isv)
                    last_v[slot] = g;
                else
                    last_k[slot] = g;
                return true;
            };
            bool ok = true;
            int g0 = 0, it = 0;
            for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++it) {
                const DqItem I = item(w);
                // the previous item's last S and dP (and the dO copy) are done with Q, dO
                if (it > 0 && !(ok = mbar_wait(BAR_QE, (it - 1) & 1, a.watch, 41))) break;
                mbar_arrive_expect_tx(BAR_QDO, 2 * C::TILE);
                for (int c = 0; c < C::NCH; ++c) {
                    tma_load_4d(sQ + c * C::CHUNK, &tmQ, BAR_QDO, c * 64, I.h, I.qi * kBM, I.b);
                    tma_load_4d(sDO + c * C::CHUNK, &tmDO, BAR_QDO, c * 64, I.h, I.qi * kBM, I.b);
                }
                // first-use order of the MMAs: K_0, V_0, V_1, K_1, V_2, K_2, ...
                ok = load(g0, 0, I, false) && load(g0, 0, I, true);
                for (int i = 1; i < I.nj && ok; ++i)
                    ok = load(g0 + i, i, I, true) && load(g0 + i, i, I, false);
                g0 += I.nj;
            }
            // no copies in flight at exit: wait (bounded) for the last Q, dO and
            // the last load of each slot
            if (it > 0) mbar_drain(BAR_QDO, (it - 1) & 1, a.watch, 21);
            for (int s = 0; s < C::KS; ++s)
                if (last_k[s] >= 0)
                    mbar_drain(BAR_KF(s), (last_k[s] / C::KS) & 1, a.watch, 21);
            for (int s = 0; s < C::VS; ++s)
                if (last_v[s] >= 0)
                    mbar_drain(BAR_VF(s), (last_v[s] / C::VS) & 1, a.watch, 21);
        }
        __syncwarp();
    } else if (warp == kDqWarpGate) {
        // ================= gate: K_{g+1} landed -> LD(g) =================
        // Its arrival on LD(g) comes only after LD's previous phase is over.
        // K_{g+1} is the next item's first K at an item's last block.
        setmaxnreg_dec<64>();
        if (lane == 0) {
            bool ok = true;
            int g = 0;
            for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
                const DqItem I = item(w);
                const bool more_items = w + static_cast<int>(gridDim.x) < n_items;
                for (int j = 0; j < I.nj && ok; ++j, ++g) {
                    if (j + 1 < I.nj || more_items)
                        ok = mbar_wait(BAR_KF((g + 1) % C::KS), ((g + 1) / C::KS) & 1, a.watch, 28);
                    if (ok && g > 0) ok = mbar_wait(BAR_LD, (g - 1) & 1, a.watch, 28);
                    if (ok) mbar_arrive(BAR_LD);
                }
            }
        }
        __syncwarp();
    } else if (warp == kDqWarpCopy) {
        // ====== copy and store: each item's dO tile -> fp16(dO * 2^s) (fp16
        // operand path), then its staged dQ -> global memory (TMA store) ======
        // The scales come from the maxima in absmax (taken before this kernel);
        // block 0 stores them for the dK/dV kernel, which also reads the copy.
        setmaxnreg_dec<64>();
        float mul = 1.f;
        if (F16) {
            const F16Scales sc = scales_of<D>(a.absmax);
            if (blockIdx.x == 0 && lane == 0) *a.scales_w = sc;
            mul = pow2f(sc.dout);
        }
        const size_t row_el = static_cast<size_t>(a.Hq) * D;  // elements per token
        bool ok = true;
        int it = 0;
        for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++it) {
            const DqItem I = item(w);
            if (F16) {
                if (!(ok = mbar_wait_warp(BAR_QDO, it & 1, a.watch, 29))) break;
                uint16_t* dst =
                    a.dout16 + (static_cast<size_t>(I.b) * a.N + I.qi * kBM) * row_el + I.h * D;
                warp_tile_to_f16<D>(sDO, dst, row_el, a.N - I.qi * kBM, mul, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR_QE);
            }
            if (!(ok = mbar_wait_warp(BAR_EPF, it & 1, a.watch, 42))) break;
            if (lane == 0) {
                for (int c = 0; c < C::NCH; ++c)
                    tma_store_4d(&tmDQ, sST + c * C::CHUNK, c * 64, I.h, I.qi * kBM, I.b);
                tma_store_commit();
                tma_store_wait_read_all();
                mbar_arrive(BAR_EPE);  // the staging buffer may be written again
            }
            __syncwarp();
        }
    } else if (warp == kDqWarpMma) {
        // ================= MMA issuer (the whole warp; the leader lane issues) =================
        setmaxnreg_dec<64>();
        {
            const uint32_t leader = elect_one();
            constexpr uint32_t IDESC_S = idesc_16(kBM, kBN, false, false, F16);  // S = Q K^T
            constexpr uint32_t IDESC_DP = idesc_bf16(kBM, kBN, false, false);    // dP = dO V^T
            constexpr uint32_t IDESC_DQ = idesc_16(kBM, D, false, true, F16);    // dQ += dS K
            const uint32_t tS = tbase + C::TM_S, tDQ = tbase + C::TM_DQ;
            auto tDP = [&](int g) { return tbase + C::TM_DP + (g & 1) * 128; };
            auto k_ready = [&](int g) {
                const bool r = mbar_wait_warp(BAR_KF(g % C::KS), (g / C::KS) & 1, a.watch, 23);
                tc_fence_after();
                return r;
            };
            auto v_ready = [&](int g) {
                const bool r = mbar_wait_warp(BAR_VF(g % C::VS), (g / C::VS) & 1, a.watch, 23);
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
            // dP(g) = dO V_g^T; V_g's slot is free once it has run
            auto issue_dp = [&](int g) {
                issue_t(tDP(g), do_lo, sV + (g % C::VS) * C::TILE, IDESC_DP);
                mma_commit_w(leader, BAR_VE(g % C::VS));
            };
            // dQ += dS(g) K_g (first: the item's first block starts it afresh):
            // dS (packed pairs) of keys 16ks.. at columns 32(ks/2) + (ks%2)*8 of
            // dP buffer g & 1; K rows 16ks.. read MN-major.  The caller commits
            // K_g's slot free (after the next dP, so that the two batches reach
            // the tensor core back to back).
            auto issue_dq = [&](int g, bool first) {
                const uint32_t k_lo = sdesc_lo(sK + (g % C::KS) * C::TILE, C::CHUNK), aS = tDP(g);
#pragma unroll
                for (int ks = 0; ks < kBN / 16; ++ks)
                    mma_bf16_ts_w(leader, tDQ, aS + (ks >> 1) * 32 + (ks & 1) * 8,
                                  sdesc_at(k_lo, HI, ks * 2048), IDESC_DQ,
                                  (first && ks == 0) ? 0u : 1u);
            };
            bool ok = true;
            int g0 = 0, it = 0;
            for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++it) {
                const DqItem I = item(w);
                const int nj = I.nj;
                if (!(ok = mbar_wait_warp(BAR_QDO, it & 1, a.watch, 22))) break;
                // S(g0) overwrites S of the previous item's last block: every warp
                // holds that one (LD; waiting it also keeps the parity waits on LD
                // in order)
                if (it > 0 && !(ok = mbar_wait_warp(BAR_LD, (g0 - 1) & 1, a.watch, 24))) break;
                if (!(ok = k_ready(g0))) break;
                issue_t(tS, q_lo, sK + (g0 % C::KS) * C::TILE, IDESC_S);
                if (!(ok = v_ready(g0))) break;
                issue_dp(g0);
                mma_commit_w(leader, BAR_SDF);
                if (nj == 1) mma_commit_w(leader, BAR_QE);  // the item's last S and dP
                if (nj > 1) {  // into the other dP buffer
                    if (!(ok = v_ready(g0 + 1))) break;
                    issue_dp(g0 + 1);
                }
                for (int j = 0; j < nj && ok; ++j) {
                    const int g = g0 + j;
                    // S(g+1) into the S buffer once both warpgroups hold S(g), dP(g)
                    // and K_{g+1} has landed (the gate's arrival on LD); its commit
                    // also covers dP(g+1), issued a block earlier
                    if (j + 1 < nj) {
                        if (!(ok = mbar_wait_warp(BAR_LD, g & 1, a.watch, 24))) break;
                        tc_fence_after();
                        issue_t(tS, q_lo, sK + ((g + 1) % C::KS) * C::TILE, IDESC_S);
                        mma_commit_w(leader, BAR_SDF);
                        if (j + 2 == nj) mma_commit_w(leader, BAR_QE);  // the item's last S, dP
                    }
                    if (!(ok = mbar_wait_warp(BAR_PF, g & 1, a.watch, 24))) break;
                    if (leader) mbar_arrive(BAR_PFS);  // the warps may now arrive on PF(g+1)
                    tc_fence_after();
                    issue_dq(g, j == 0);
                    // dP(g+2) over dS(g), which dQ(g), issued just before by this
                    // thread, reads first
                    if (j + 2 < nj) {
                        if (!(ok = v_ready(g + 2))) break;
                        issue_dp(g + 2);
                    }
                    mma_commit_w(leader, BAR_KE(g % C::KS));  // dQ(g) was K_g's last reader
                }
                if (!ok) break;
                mma_commit_w(leader, BAR_ACC);  // the item's dQ is complete
                g0 += nj;
            }
            // every issued MMA has finished before TMEM is released
            mma_commit_w(leader, BAR_DONE);
            mbar_drain(BAR_DONE, 0, a.watch, 25);
        }
        __syncwarp();
    } else if (warp < 16) {
        setmaxnreg_inc<104>();
        const int hf = warp >> 2;  // keys 32*hf..32*hf+31 of every block
        const int r = (warp & 3) * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tbase + C::TM_S + lane_off + hf * 32;
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
        const float out_mul = a.scale * pow2f(-(eds + ek));  // dQ carries 2^(ds+k)
        const uint64_t sl2x2 = f2(sl2, sl2), dsc2 = f2(dsc, dsc);
        // this thread's row's lse and D, read one item ahead
        auto row_vals = [&](int w, float& nl, float& dv) {
            const DqItem I = item(w);
            const int grow = I.qi * kBM + r;
            const bool valid = grow < a.N;
            const size_t idx = (static_cast<size_t>(I.b) * a.Hq + I.h) * a.N + (valid ? grow : 0);
            nl = valid ? -a.lse[idx] * kLog2e : 0.f;
            dv = valid ? a.dsum[idx] : 0.f;
        };
        float nlse2_next = 0.f, dval_next = 0.f;
        if (static_cast<int>(blockIdx.x) < n_items) row_vals(blockIdx.x, nlse2_next, dval_next);
        bool ok = true;
        int g0 = 0, it = 0;
        for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++it) {
            const DqItem I = item(w);
            const int nj = I.nj;
            const int grow = I.qi * kBM + r;
            const int lim = a.causal ? min(grow, a.N - 1) : a.N - 1;
            const float nlse2 = nlse2_next, dval = dval_next;
            if (w + static_cast<int>(gridDim.x) < n_items)
                row_vals(w + gridDim.x, nlse2_next, dval_next);
            const uint64_t nlse2x2 = f2(nlse2, nlse2);
            const uint64_t ndx2 = f2(-dval * dsc, -dval * dsc);
            for (int j = 0; j < nj && ok; ++j) {
                const int g = g0 + j;
                if (!(ok = mbar_wait_warp(BAR_SDF, g & 1, a.watch, 26))) break;
                tc_fence_after();
                const uint32_t tDP = tbase + C::TM_DP + (g & 1) * 128 + lane_off + hf * 32;
                uint32_t sv[32], dp[32];
                tmem_ld32(tS, sv);
                tmem_ld32(tDP, dp);
                tmem_wait_ld();
                reg_fence<32>(sv);
                reg_fence<32>(dp);
                // both buffers are in registers: S(g+1) may now overwrite S(g)
                tc_fence_before();
                mbar_arrive(BAR_LD);
                const int kbase = j * kBN + hf * 32;
                const bool need_mask = kbase + 31 > lim;
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    // two columns per packed f32x2 FMA / ADD / MUL
                    float x0, x1;
                    f2_split(fma2(f2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2,
                                  nlse2x2),
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
                // S(g), dP(g) were issued before the MMA thread waits for PF(g-1):
                // arriving on PF(g) only once that thread has seen PF(g-1) keeps a
                // fast warp's arrival out of PF(g-1)'s phase and PF from running
                // two phases ahead of the thread's parity wait
                if (g > 0 && !(ok = mbar_wait_warp(BAR_PFS, (g - 1) & 1, a.watch, 39))) break;
                mbar_arrive(BAR_PF);
            }
            if (!ok) break;
            g0 += nj;
            // ---- epilogue: dQ = scale * (dS K) -> bf16, staged for the copy
            // warp's TMA store.  The next item's first dQ product starts the
            // accumulator afresh only after PF of its first block, which every
            // warp arrives on after these TMEM loads.
            if (!(ok = mbar_wait_warp(BAR_ACC, it & 1, a.watch, 27))) break;
            tc_fence_after();
            // the staging buffer is free once the previous item's store has read it
            if (C::PERSIST && it > 0 && !(ok = mbar_wait_warp(BAR_EPE, (it - 1) & 1, a.watch, 43)))
                break;
            if (hf * 32 < D)
                stage_rows_bf16<C::CHUNK>(tbase + C::TM_DQ + lane_off, sST, r, hf * 32, hf * 32 + 32,
                                          out_mul);
            fence_proxy_async_smem();
            mbar_arrive(BAR_EPF);
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
    const long long items = static_cast<long long>((a.N + kBM - 1) / kBM) * a.B * a.Hq;
    if (items <= 0 || items > 0x7fffffffLL || a.num_ctas <= 0) return cudaErrorInvalidConfiguration;
    // d = 64: persistent, one CTA per SM; d = 128: one CTA per item
    const long long ctas = DqCfg<D>::PERSIST ? (items < a.num_ctas ? items : a.num_ctas) : items;
    kern<<<static_cast<unsigned>(ctas), kDqThreads, smem, st>>>(F16 ? m.q16 : m.q, F16 ? m.k16 : m.k,
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
