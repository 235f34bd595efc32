// fa_fwd.cu -- exact attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes: O = softmax(scale * Q K^T [+ causal mask]) V and the
// per-row log-sum-exp, one (batch, head, 256-query block) per thread block,
// streaming 128-key blocks of K and V and folding each block into running
// row statistics with the online-softmax update of "FlashAttention and the
// Kernel Era", section "The Mathematics" (m_new = max(m, max S_j),
// l_new = l * e^{m - m_new} + sum e^{S_j - m_new}) and the output update of
// "FlashAttention 1, 2, and 3 Explained", section 2
// (O_new = diag(e^{m_old - m_new}) O_old + P_j V_j).  The N x N score matrix
// only ever exists one 128 x 128 tile at a time, in tensor memory.
//
// How it maps to sm_103a (a redesign for Blackwell, not the pages' A100/H100
// kernels):
//   * each CTA holds two 128-row query tiles (Q0, Q1) in shared memory and
//     streams K_j, V_j through a ring of TMA-filled shared-memory slots;
//   * one thread issues every tcgen05.mma: S_t = Q_t K_j^T into TMEM, then
//     O_t += P_t V_j with P_t read straight from TMEM (bf16, written over S_t);
//   * two softmax warpgroups, one per query tile, each thread owning one
//     query row (one TMEM lane): load S, mask, row max, exp2, row sum, write P
//     back to TMEM; while one warpgroup does its softmax the tensor core works
//     on the other tile, which is the overlap of matmul and softmax that
//     "FlashAttention and the Kernel Era" describes for FlashAttention-3;
//   * exp2 with scale*log2(e) folded into one FMA; the running max is only
//     moved (and O rescaled in TMEM) when the block max exceeds it by more
//     than 2^8, which keeps l and O consistent with the same reference and is
//     exact (only the headroom of fp32 changes);
//   * causal: blocks above the diagonal are never loaded or multiplied;
//     only the diagonal block is masked element by element;
//   * the epilogue divides O by l, rounds to bf16, stages the tile in the
//     (now free) Q buffer with the 128-byte swizzle and writes it with one TMA
//     store; lse = (m + log2 l) * ln 2.  The training forward also writes
//     o_lo = bf16(O32 - O), the rounding residual of O, with plain stores.
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

template <int D>
struct FwdCfg {
    static constexpr int CHUNK = kBM * 128;          // one 64-column chunk of a 128-row tile
    static constexpr int NCH = D / 64;               // chunks per tile
    static constexpr int TILE = NCH * CHUNK;         // bytes of a 128 x D bf16 tile
    static constexpr int NSLOT = (D == 128) ? 4 : 8; // K/V ring slots
    static constexpr int SMEM_Q = 2 * TILE;
    static constexpr int SMEM_KV = NSLOT * TILE;
    // barriers: q_full, kv_full[NSLOT], kv_empty[NSLOT], s_full[2], p_full[2],
    // o_final[2], mma_done, q_copied, s_empty[2], pv_done[2]
    static constexpr int NBAR = 1 + 2 * NSLOT + 2 + 2 + 2 + 1 + 1 + 2 + 2;
    static constexpr int SMEM_BYTES = 1024 /*align slack*/ + SMEM_Q + SMEM_KV + NBAR * 8 + 16;
    // TMEM columns: S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D, 256+2D)
    // and, at D = 64, P0 [384,448) P1 [448,512): P (fp16 or bf16 pairs) gets
    // columns of its own instead of overwriting S_t (SPLITP), so the next
    // score product of a tile need not wait for the P V product before it.
    static constexpr uint32_t TM_S = 0;
    static constexpr uint32_t TM_O = 256;
    static constexpr bool SPLITP = (D == 64);
    static constexpr uint32_t TM_P = 256 + 2 * D;
    static constexpr uint32_t TM_COLS = 512;
    static constexpr int THREADS = 384;              // softmax WG0, WG1, WG2 = {MMA, TMA, gate, copy}
};

constexpr int kWarpMma = 8;
constexpr int kWarpLoad = 9;
// The gate warp folds "K/V tiles landed" into the p_full barriers, so the MMA
// thread waits on two barriers per key block instead of four: every mbarrier
// wait in the issuing thread costs tensor-core time.
constexpr int kWarpGate = 10;
// The training forward's copy warp writes the fp16 copy of the CTA's Q tiles
// (for the backward) while the tiles sit in shared memory anyway.
constexpr int kWarpCopy = 11;

// Row-max and exp threshold for the lazy rescale: the reference max is only
// moved when the new block maximum exceeds it by more than 2^8 (in log2
// units), so unnormalised P values stay below 256.
constexpr float kRescaleThreshold = 8.0f;

// The key blocks the CTA's two query tiles multiply.  Tile t takes the
// blocks below n[t] (the causal diagonal or the ragged end), and, with a block
// mask (SPARSE), only those whose mask byte is set.  Every role walks the
// union of the two tiles' blocks in increasing order, the i-th union block
// occupying ring entries 2i (K) and 2i + 1 (V); without a mask the union is
// 0 .. n[1] - 1 and tile 0 just stops one block early on the diagonal.
template <bool SPARSE>
struct TileBlocks {
    int n[2];
    const uint8_t* row[2];  // SPARSE: the tiles' mask rows (null: the tile has no block)
    __device__ __forceinline__ bool has(int t, int u) const {
        if (u >= n[t]) return false;
        return SPARSE ? (row[t] != nullptr && row[t][u] != 0) : true;
    }
    __device__ __forceinline__ int next(int u) const {  // next union block after u, or -1
        if constexpr (!SPARSE) {
            return u + 1 < n[1] ? u + 1 : -1;
        } else {
            const int hi = max(n[0], n[1]);
            for (++u; u < hi; ++u)
                if (has(0, u) || has(1, u)) return u;
            return -1;
        }
    }
    __device__ __forceinline__ int next_of(int t, int u) const {  // tile t's next block, or -1
        if constexpr (!SPARSE) {
            return u + 1 < n[t] ? u + 1 : -1;
        } else {
            for (++u; u < n[t]; ++u)
                if (has(t, u)) return u;
            return -1;
        }
    }
};

// F16: P is rounded to fp16 (not bf16) and multiplies the fp16 copy of V,
// scaled by 2^v (the training forward, whose O feeds the backward's D).
// SPARSE: the tiles multiply only the key blocks a.block_mask selects.
template <int D, bool F16, bool SPARSE>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const FwdArgs a) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sKV = sQ + C::SMEM_Q;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::SMEM_Q + C::SMEM_KV);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
    const uint32_t bar0 = smem_u32(bars);
    auto BAR_Q = [&]() { return bar0; };
    auto BAR_KVF = [&](int s) { return bar0 + 8u * (1 + s); };
    auto BAR_KVE = [&](int s) { return bar0 + 8u * (1 + C::NSLOT + s); };
    auto BAR_SF = [&](int t) { return bar0 + 8u * (1 + 2 * C::NSLOT + t); };
    auto BAR_PF = [&](int t) { return bar0 + 8u * (3 + 2 * C::NSLOT + t); };
    auto BAR_OF = [&](int t) { return bar0 + 8u * (5 + 2 * C::NSLOT + t); };
    const uint32_t BAR_DONE = bar0 + 8u * (7 + 2 * C::NSLOT);
    const uint32_t BAR_QC = bar0 + 8u * (8 + 2 * C::NSLOT);  // Q tiles read by the copy warp
    // SPLITP only: S_t is in the softmax's registers / PV_t has finished
    auto BAR_SE = [&](int t) { return bar0 + 8u * (9 + 2 * C::NSLOT + t); };
    auto BAR_PVD = [&](int t) { return bar0 + 8u * (11 + 2 * C::NSLOT + t); };

    const int warp = warp_id();
    const int lane = lane_id();

    // ---- work decode: longest query blocks first, heads of one KV group adjacent
    const int per = a.B * a.Hq;
    const int qb = a.n_qblk - 1 - static_cast<int>(blockIdx.x) / per;
    const int bh = static_cast<int>(blockIdx.x) % per;
    const int b = bh / a.Hq;
    const int h = bh % a.Hq;
    const int hk = h / a.g;
    const int row0 = qb * 2 * kBM;
    const int nkv_all = (a.N + kBN - 1) / kBN;
    // key blocks below each query tile's limit (causal: up to and including its
    // diagonal), and with a mask only those it selects
    TileBlocks<SPARSE> blk;
    blk.n[0] = a.causal ? min(row0 / kBN + 1, nkv_all) : nkv_all;
    blk.n[1] = a.causal ? min((row0 + kBM) / kBN + 1, nkv_all) : nkv_all;
    blk.row[0] = blk.row[1] = nullptr;
    if (SPARSE)
        for (int t = 0; t < 2; ++t)
            if (2 * qb + t < nkv_all)
                blk.row[t] = a.block_mask + (static_cast<size_t>(h) * nkv_all + 2 * qb + t) * nkv_all;
    const int u_first = SPARSE ? blk.next(-1) : 0;  // first union block (-1: none)

    // ---- set-up
    if (warp == 0 && lane == 0) {
        mbar_init(BAR_Q(), 1);
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(BAR_KVF(s), 1);
            mbar_init(BAR_KVE(s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(BAR_SF(t), 1);
            mbar_init(BAR_PF(t), 128 + 1);  // the tile's softmax threads and the gate
            mbar_init(BAR_OF(t), 1);
            mbar_init(BAR_SE(t), 4);  // one arrival per softmax warp of the tile
            mbar_init(BAR_PVD(t), 1);
        }
        mbar_init(BAR_DONE, 1);
        mbar_init(BAR_QC, 1);
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
        // ================= TMA producer =================
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmO);
            const uint64_t pol_kv = l2_policy_evict_last();
            const uint64_t pol_q = l2_policy_evict_first();
            mbar_arrive_expect_tx(BAR_Q(), 2 * C::TILE);
            for (int t = 0; t < 2; ++t)
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_4d_hint(sQ + t * C::TILE + c * C::CHUNK, &tmQ, BAR_Q(), c * 64, h,
                                     row0 + t * kBM, b, pol_q);
            int last_idx[C::NSLOT];
            for (int s = 0; s < C::NSLOT; ++s) last_idx[s] = -1;
            bool ok = true;
            for (int i = 0, u = u_first; u >= 0 && ok; ++i, u = blk.next(u)) {
                for (int w = 0; w < 2; ++w) {
                    const int idx = 2 * i + w;
                    const int slot = idx % C::NSLOT;
                    const uint32_t ph = (idx / C::NSLOT) & 1;
                    if (!mbar_wait(BAR_KVE(slot), ph ^ 1u, a.watch, 1)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(BAR_KVF(slot), C::TILE);
                    const CUtensorMap* tm = w ? &tmV : &tmK;
                    for (int c = 0; c < C::NCH; ++c)
                        tma_load_4d_hint(sKV + slot * C::TILE + c * C::CHUNK, tm, BAR_KVF(slot),
                                         c * 64, hk, u * kBN, b, pol_kv);
                    last_idx[slot] = idx;
                }
            }
            // Never leave the CTA with copies in flight: wait (bounded) for the
            // last load issued into every slot, and for Q.
            mbar_drain(BAR_Q(), 0, a.watch, 2);
            for (int s = 0; s < C::NSLOT; ++s)
                if (last_idx[s] >= 0)
                    mbar_drain(BAR_KVF(s), (last_idx[s] / C::NSLOT) & 1, a.watch, 2);
        }
        __syncwarp();
    } else if (warp == kWarpGate) {
        // ================= gate: loads -> p_full =================
        // For key block j it waits for V_j and K_{j+1}, then adds one arrival
        // to p_full(t) for each tile t that multiplies block j, but only once
        // that barrier's previous phase has completed, so the arrival can
        // never be counted in the wrong phase.
        if (lane == 0) {
            bool ok = true;
            int cnt[2] = {0, 0};  // blocks each tile has multiplied so far
            for (int i = 0, u = u_first; u >= 0 && ok; ++i) {
                const int un = blk.next(u);
                const int vidx = 2 * i + 1, kidx = 2 * i + 2;
                ok = mbar_wait(BAR_KVF(vidx % C::NSLOT), (vidx / C::NSLOT) & 1, a.watch, 5);
                if (ok && un >= 0)
                    ok = mbar_wait(BAR_KVF(kidx % C::NSLOT), (kidx / C::NSLOT) & 1, a.watch, 5);
                for (int t = 0; t < 2 && ok; ++t) {
                    if (!blk.has(t, u)) continue;
                    if (cnt[t] > 0) ok = mbar_wait(BAR_PF(t), (cnt[t] - 1) & 1, a.watch, 7);
                    if (ok) mbar_arrive(BAR_PF(t));
                    ++cnt[t];
                }
                u = un;
            }
        }
        __syncwarp();
    } else if (warp == kWarpCopy) {
        // ================= copy: Q tiles -> fp16(q * 2^s) =================
        // Only the training forward (F16 with q16 set); the epilogues, which
        // stage O in the Q buffers, wait for BAR_QC.
        if (F16 && a.q16 != nullptr) {
            const float mul = pow2f(ld_once(&a.f16s->q));
            const size_t row_el = static_cast<size_t>(a.Hq) * D;  // elements per token
            if (mbar_wait_warp(BAR_Q(), 0, a.watch, 15)) {
                for (int t = 0; t < 2; ++t)
                    warp_tile_to_f16<D>(sQ + t * C::TILE,
                                        a.q16 + (static_cast<size_t>(b) * a.N + row0 + t * kBM) *
                                                    row_el + h * D,
                                        row_el, a.N - (row0 + t * kBM), mul, lane);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR_QC);  // also after a failed wait: never blocks the epilogue
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ================= MMA issuer (the whole warp; the leader lane issues) =================
        {
            const uint32_t leader = elect_one();
            constexpr uint32_t IDESC_QK = idesc_bf16(kBM, kBN, false, false);
            constexpr uint32_t IDESC_PV = idesc_16(kBM, D, false, true, F16);
            // descriptors built once per tile; each MMA only moves the start address
            constexpr uint32_t HI = sdesc_hi(1024);
            const uint32_t q_lo = sdesc_lo(sQ, 16);
            auto issue_qk = [&](int t, int slot) {
                const uint32_t dS = tbase + C::TM_S + t * kBN;
                const uint32_t a_lo = q_lo + ((t * C::TILE) >> 4);
                const uint32_t b_lo = sdesc_lo(sKV + slot * C::TILE, 16);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
                    mma_bf16_ss_w(leader, dS, sdesc_at(a_lo, HI, off), sdesc_at(b_lo, HI, off), IDESC_QK, ks > 0);
                }
            };
            auto issue_pv = [&](int t, int slot, bool acc) {
                const uint32_t dO = tbase + C::TM_O + t * D;
                // P: its own columns (SPLITP), else over S_t
                const uint32_t aP = tbase + (C::SPLITP ? C::TM_P + t * (kBN / 2) : C::TM_S + t * kBN);
                const uint32_t b_lo = sdesc_lo(sKV + slot * C::TILE, C::CHUNK);
#pragma unroll
                for (int ks = 0; ks < kBN / 16; ++ks)
                    mma_bf16_ts_w(leader, dO, aP + ks * 8, sdesc_at(b_lo, HI, ks * 2048), IDESC_PV,
                                (acc || ks > 0) ? 1u : 0u);
            };
            bool ok = mbar_wait_warp(BAR_Q(), 0, a.watch, 3);
            if constexpr (C::SPLITP) {
                // Per union block u (ring entries 2i, 2i + 1) with next union
                // block un, tile by tile: S_t(un) once the tile's softmax holds
                // S_t(u) in registers (s_empty) and K(un) has landed, then
                // PV_t(u) on p_full(t) (which also says V(u) has landed, the
                // gate), committed to pv_done(t): the softmax writes P_t and
                // rescales O_t only after it.
                int nqk[2] = {0, 0}, cnt[2] = {0, 0};
                if (ok && u_first >= 0) {
                    ok = mbar_wait_warp(BAR_KVF(0), 0, a.watch, 4);
                    if (ok) {
                        tc_fence_after();
                        for (int t = 0; t < 2; ++t)
                            if (blk.has(t, u_first)) {
                                issue_qk(t, 0);
                                mma_commit_w(leader, BAR_SF(t));
                                ++nqk[t];
                            }
                        mma_commit_w(leader, BAR_KVE(0));
                    }
                }
                for (int i = 0, u = u_first; u >= 0 && ok; ++i) {
                    const int un = blk.next(u);
                    const int vslot = (2 * i + 1) % C::NSLOT;
                    const int kidx = 2 * i + 2;
                    const int kslot = kidx % C::NSLOT;
                    bool k_ready = false;
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (un >= 0 && blk.has(t, un)) {
                            if (nqk[t] > 0 &&
                                !(ok = mbar_wait_warp(BAR_SE(t), (nqk[t] - 1) & 1, a.watch, 17 + t)))
                                break;
                            if (!k_ready) {
                                if (!(ok = mbar_wait_warp(BAR_KVF(kslot), (kidx / C::NSLOT) & 1,
                                                          a.watch, 19)))
                                    break;
                                k_ready = true;
                            }
                            tc_fence_after();
                            issue_qk(t, kslot);
                            mma_commit_w(leader, BAR_SF(t));
                            ++nqk[t];
                        }
                        if (blk.has(t, u)) {
                            if (!(ok = mbar_wait_warp(BAR_PF(t), cnt[t] & 1, a.watch, 6 + 2 * t)))
                                break;
                            tc_fence_after();
                            issue_pv(t, vslot, cnt[t] > 0);
                            mma_commit_w(leader, BAR_PVD(t));
                            ++cnt[t];
                            if (blk.next_of(t, u) < 0) mma_commit_w(leader, BAR_OF(t));
                        }
                    }
                    if (!ok) break;
                    mma_commit_w(leader, BAR_KVE(vslot));
                    if (un >= 0) mma_commit_w(leader, BAR_KVE(kslot));
                    u = un;
                }
            } else {
            if (ok && u_first >= 0) {
                // first union block: the score tiles of the tiles that have it
                ok = mbar_wait_warp(BAR_KVF(0), 0, a.watch, 4);
                if (ok) {
                    tc_fence_after();
                    for (int t = 0; t < 2; ++t)
                        if (blk.has(t, u_first)) {
                            issue_qk(t, 0);
                            mma_commit_w(leader, BAR_SF(t));
                        }
                    mma_commit_w(leader, BAR_KVE(0));
                }
            }
            // Per union block u (ring entries 2i, 2i + 1), with un the next one:
            // PV0(u), S0(un), PV1(u), S1(un) for the tiles that have them.  p_full(t)
            // for u also means V(u) and K(un) have landed (the gate), and at
            // least one tile has u, so no S(un) is issued before one such wait;
            // S_t(un) follows PV_t of the tile's last block, which read P_t.
            int cnt[2] = {0, 0};
            for (int i = 0, u = u_first; u >= 0 && ok; ++i) {
                const int un = blk.next(u);
                const int vslot = (2 * i + 1) % C::NSLOT;
                const int kslot = (2 * i + 2) % C::NSLOT;
                const bool h0 = blk.has(0, u), h0n = un >= 0 && blk.has(0, un);
                if (h0) {
                    if (!(ok = mbar_wait_warp(BAR_PF(0), cnt[0] & 1, a.watch, 6))) break;
                    tc_fence_after();
                    issue_pv(0, vslot, cnt[0] > 0);
                    ++cnt[0];
                    if (blk.next_of(0, u) < 0) mma_commit_w(leader, BAR_OF(0));
                    if (h0n) {
                        issue_qk(0, kslot);
                        mma_commit_w(leader, BAR_SF(0));
                    }
                }
                if (blk.has(1, u)) {
                    if (!(ok = mbar_wait_warp(BAR_PF(1), cnt[1] & 1, a.watch, 8))) break;
                    tc_fence_after();
                    issue_pv(1, vslot, cnt[1] > 0);
                    ++cnt[1];
                }
                mma_commit_w(leader, BAR_KVE(vslot));
                if (blk.has(1, u) && blk.next_of(1, u) < 0) mma_commit_w(leader, BAR_OF(1));
                if (un >= 0) {
                    if (blk.has(1, un)) {
                        issue_qk(1, kslot);
                        mma_commit_w(leader, BAR_SF(1));
                    }
                    if (!h0 && h0n) {
                        issue_qk(0, kslot);
                        mma_commit_w(leader, BAR_SF(0));
                    }
                    mma_commit_w(leader, BAR_KVE(kslot));
                }
                u = un;
            }
            }  // SPLITP
            // all issued MMAs have finished before TMEM can be released
            mma_commit_w(leader, BAR_DONE);
            mbar_drain(BAR_DONE, 0, a.watch, 9);
        }
        __syncwarp();
    } else if (warp < 8) {
        // ================= softmax warpgroups (warps 0-3: tile 0, 4-7: tile 1)
        const int t = warp >> 2;               // query tile of this warpgroup
        const int wq = warp & 3;               // its warp owns TMEM lanes 32*wq..32*wq+31
        const int r = wq * 32 + lane;          // row within the tile
        const int grow = row0 + t * kBM + r;   // query index
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tbase + C::TM_S + t * kBN + lane_off;
        const uint32_t tO = tbase + C::TM_O + t * D + lane_off;
        // where P goes: its own columns (SPLITP), else over S_t
        const uint32_t tP = C::SPLITP ? tbase + C::TM_P + t * (kBN / 2) + lane_off : tS;
        const float sl2 = a.scale_log2;
        int eq = 0, ek = 0, ev = 0, edo = 0;  // fp16 path: O carries 2^ev
        if (F16) ld_once_v4(&a.f16s->q, eq, ek, ev, edo);
        // last key index this row may see
        const int lim = a.causal ? min(grow, a.N - 1) : a.N - 1;
        float m_ref = -INFINITY;  // reference max of the exponentials (log2 units)
        float l = 0.f;            // running sum, relative to m_ref
        bool ok = true;
        const int u0 = blk.has(t, 0) ? 0 : blk.next_of(t, 0);  // the tile's first block
        int j = 0;                                               // blocks done so far
        for (int u = u0; u >= 0; u = blk.next_of(t, u), ++j) {
            if (!(ok = mbar_wait_warp(BAR_SF(t), j & 1, a.watch, 10 + t))) break;
            tc_fence_after();
            uint32_t s[kBN];
            tmem_ld32(tS + 0, s);
            tmem_ld32(tS + 32, s + 32);
            tmem_ld32(tS + 64, s + 64);
            tmem_ld32(tS + 96, s + 96);
            tmem_wait_ld();
            reg_fence<kBN>(s);
            if constexpr (C::SPLITP) {  // S_t may now be overwritten by the next score product
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR_SE(t));
            }
            float x[kBN];
#pragma unroll
            for (int c = 0; c < kBN; ++c) x[c] = __uint_as_float(s[c]);
            const int kbase = u * kBN;
            if (kbase + kBN - 1 > lim) {  // diagonal block or ragged tail: mask
#pragma unroll
                for (int c = 0; c < kBN; ++c) x[c] = (kbase + c > lim) ? -INFINITY : x[c];
            }
            // row max: eight running maxima, three-input max instructions
            float mk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mk[i] = fmaxf(x[i], x[i + 8]);
#pragma unroll
            for (int c = 16; c < kBN; c += 16)
#pragma unroll
                for (int i = 0; i < 8; ++i) mk[i] = fmax3(mk[i], x[c + i], x[c + 8 + i]);
            const float mx = fmax3(fmax3(mk[0], mk[1], mk[2]), fmax3(mk[3], mk[4], mk[5]),
                                   fmaxf(mk[6], mk[7]));
            const float m_new = fmaxf(m_ref, mx * sl2);
            const bool need = m_new > m_ref + kRescaleThreshold;
            float alpha = 1.f;
            if (need) {
                alpha = ex2(m_ref - m_new);
                l *= alpha;
                m_ref = m_new;
            }
            if (C::SPLITP && j > 0) {  // PV_t of the previous block still reads P_t, writes O_t
                if (!(ok = mbar_wait_warp(BAR_PVD(t), (j - 1) & 1, a.watch, 20 + t))) break;
                tc_fence_after();
            }
            const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
            const uint64_t sl2x2 = f2(sl2, sl2), negx2 = f2(neg, neg);
            uint64_t ls2[4] = {0, 0, 0, 0};  // packed partial row sums
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 64; c += 2) {
                    float e0, e1;
                    f2_split(fma2(f2(x[half * 64 + c], x[half * 64 + c + 1]), sl2x2, negx2), e0, e1);
                    const float p0 = ex2(e0), p1 = ex2(e1);
                    ls2[(c >> 1) & 3] = add2(ls2[(c >> 1) & 3], f2(p0, p1));
                    pk[c >> 1] = pack_op<F16>(p0, p1);
                }
                tmem_st32(tP + half * 32, pk);
            }
            {
                const uint64_t t = add2(add2(ls2[0], ls2[1]), add2(ls2[2], ls2[3]));
                float a0, a1;
                f2_split(t, a0, a1);
                l += a0 + a1;
            }
            // O_t was last written by the P V product of block j-1, which
            // completed before this block's scores were committed (SPLITP:
            // before pv_done, waited for above).
            if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int cb = 0; cb < D; cb += 32) {
                    uint32_t o[32];
                    tmem_ld32(tO + cb, o);
                    tmem_wait_ld();
                    reg_fence<32>(o);
                    const uint64_t ax2 = f2(alpha, alpha);
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        float u0, u1;
                        f2_split(mul2(f2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), ax2), u0, u1);
                        o[i] = __float_as_uint(u0);
                        o[i + 1] = __float_as_uint(u1);
                    }
                    tmem_st32(tO + cb, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR_PF(t));
        }
        // ---- epilogue: O / l -> bf16 -> swizzled staging in Q_t's buffer -> TMA store
        // (a tile with no key block -- block-sparse only -- writes O = 0 and
        // lse = -inf: no MMA ever wrote its O, and only the Q load, which must
        // land before the buffer is reused, touched its staging buffer)
        const bool any = u0 >= 0;
        bool ok_e = ok && (any ? mbar_wait_warp(BAR_OF(t), 0, a.watch, 12 + t)
                               : mbar_wait_warp(BAR_Q(), 0, a.watch, 16));
        if (F16 && a.q16 != nullptr)  // the copy warp is done with the Q buffers
            ok_e = ok_e && mbar_wait_warp(BAR_QC, 0, a.watch, 14);
        const uint32_t stage = sQ + t * C::TILE;
        if (ok_e) {
            tc_fence_after();
            // O was accumulated against V * 2^v on the fp16 path
            const float inv_l = (l > 0.f) ? pow2f(-ev) / l : 0.f;
#pragma unroll
            for (int cb = 0; cb < D; cb += 32) {
                uint32_t o[32];
                tmem_ld32(tO + cb, o);
                tmem_wait_ld();
                reg_fence<32>(o);
                if (SPARSE && !any)
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                uint32_t w[16], wl[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float f0 = __uint_as_float(o[2 * i]) * inv_l;
                    const float f1 = __uint_as_float(o[2 * i + 1]) * inv_l;
                    w[i] = pack_bf16(f0, f1);
                    // rounding residual for the training forward's o_lo
                    wl[i] = pack_bf16(f0 - __uint_as_float(w[i] << 16),
                                      f1 - __uint_as_float(w[i] & 0xFFFF0000u));
                }
                if (a.o_lo != nullptr && grow < a.N) {
                    uint4* dst = reinterpret_cast<uint4*>(
                        a.o_lo + ((static_cast<size_t>(b) * a.N + grow) * a.Hq + h) * D + cb);
#pragma unroll
                    for (int p4 = 0; p4 < 4; ++p4)
                        dst[p4] = make_uint4(wl[4 * p4], wl[4 * p4 + 1], wl[4 * p4 + 2],
                                             wl[4 * p4 + 3]);
                }
                const uint32_t rowbase = stage + (cb >> 6) * C::CHUNK + r * 128;
#pragma unroll
                for (int p4 = 0; p4 < 4; ++p4) {
                    const int piece = ((cb & 63) >> 3) + p4;  // 16-byte piece within the row
                    st_shared_v4(rowbase + ((piece ^ (r & 7)) << 4), w[4 * p4], w[4 * p4 + 1],
                                 w[4 * p4 + 2], w[4 * p4 + 3]);
                }
            }
            if (grow < a.N)
                a.lse[(static_cast<size_t>(b) * a.Hq + h) * a.N + grow] =
                    (m_ref + log2f(l)) * 0.6931471805599453f;
            fence_proxy_async_smem();
        }
        named_bar_sync(1 + t, 128);
        if (ok_e && r == 0) {
            for (int c = 0; c < C::NCH; ++c)
                tma_store_4d(&tmO, stage + c * C::CHUNK, c * 64, h, row0 + t * kBM, b);
            tma_store_commit();
            tma_store_wait_read_all();
        }
    }

    // ---- tear-down
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tbase, C::TM_COLS);
    }
}

template <int D, bool F16, bool SPARSE>
cudaError_t launch_fwd_d(const FwdMaps& m, const FwdArgs& a, cudaStream_t st) {
    using C = FwdCfg<D>;
    auto kern = fa_fwd_kernel<D, F16, SPARSE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long nblk = static_cast<long long>(a.n_qblk) * a.B * a.Hq;
    if (nblk <= 0 || nblk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<static_cast<unsigned>(nblk), C::THREADS, C::SMEM_BYTES, st>>>(m.q, m.k, m.v, m.o, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdMaps& maps, const FwdArgs& args, int d, cudaStream_t stream) {
    const bool f16 = args.f16s != nullptr;
    if (args.block_mask != nullptr) {  // block-sparse: the inference forward's arithmetic
        if (f16) return cudaErrorInvalidValue;
        if (d == 64) return launch_fwd_d<64, false, true>(maps, args, stream);
        if (d == 128) return launch_fwd_d<128, false, true>(maps, args, stream);
        return cudaErrorInvalidValue;
    }
    if (d == 64) return f16 ? launch_fwd_d<64, true, false>(maps, args, stream)
                            : launch_fwd_d<64, false, false>(maps, args, stream);
    if (d == 128) return f16 ? launch_fwd_d<128, true, false>(maps, args, stream)
                             : launch_fwd_d<128, false, false>(maps, args, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa
