// fa_bwd_dkdv.cu -- dK and dV for exact attention, sm_103a.
//
// One work item per (batch, kv head, 128-key block): one CTA each at d = 128,
// persistent CTAs walking several at d = 64.  An item's K and V stay in shared
// memory (at d = 64 in one of two buffers, so that the next item's land while
// the current one runs); Q_i and dO_i of every query head of the GQA group and
// every query block that sees the key block stream through a TMA ring (2
// stages, 3 at d = 64), with lse * log2(e) and D for the block's queries
// staged by the TMA warp, which reads them a step ahead.  For
// each, S^T = K Q_i^T and dP^T = V dO_i^T are recomputed into TMEM (keys on
// the TMEM lanes), turned into P^T = exp2(S^T * scale * log2(e) - lse2) and
// dS^T = P^T o (dP^T - D) in place (16-bit pairs), and dV += P^T dO_i,
// dK += dS^T Q_i take P^T / dS^T straight from TMEM as the A operand -- so no
// transpose is ever materialised.  The group's query heads are summed inside
// the CTA: no atomics.
//
// Pipelining.  Every MMA is 128 wide: a tcgen05.mma with N = 64 costs its
// issuing thread about as long as one with N = 128 and reads more shared
// memory per flop.  Two 128-column TMEM regions X and Y swap roles every
// block: S^T(i) and then P^T(i), dS^T(i) live in one, dP^T(i) in the other.
// The warps' work on a block comes in two steps, so that its exponentials
// run while the tensor core is busy with the block before: P^T(i) as soon as
// S^T(i) is in TMEM (then dV += P^T dO of block i starts), and dS^T(i) =
// P^T(i) (dP^T(i) - D) once dP^T(i) is (P^T kept in registers, rounded as it
// entered the product).  As soon as all warpgroups have copied dP^T(i) into
// registers, the tensor core computes S^T(i+1) over it; dK += dS^T Q follows
// dS^T(i), and dP^T(i+1) is then written over P^T(i), dS^T(i).  The tensor
// core's order per block: dV(i), S^T(i+1), dK(i), dP^T(i+1).  Warpgroup w owns queries
// 32w..32w+31 of each block and writes its P^T and dS^T (16-bit pairs) over
// the S^T columns it read.  (Tried and dropped: 64-query sub-blocks with two
// TMEM buffers of 64-wide S^T and dP^T, which would hide the hand-off
// entirely; the 64-wide products ran at about 100 cycles per MMA in the
// kernel, and the whole was 24% slower.)
//
// TMEM (512 columns): X [0,128) | Y [128,256) | dV [256,256+D) | dK [256+D, 256+2D).
#include "fa_bwd_common.cuh"

namespace fa {
namespace {

// Elementwise product of two fp16 pairs, rounded once to fp16 (nearest even).
__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

using namespace bwd;

// Warp roles: warps 0-15 are four compute warpgroups (warpgroup w takes
// queries 32w..32w+31 of every block: four warps per SM sub-partition keep the
// exp2 and FMA pipes busy through each other's latencies), warp 16 issues the
// MMAs, warp 17 loads, warp 18 stores each item's dV and dK.
constexpr int kDkWarpMma = 16;
constexpr int kDkWarpLoad = 17;
constexpr int kDkWarpStore = 18;
constexpr int kDkThreads = 19 * 32;
constexpr int kDkCompute = 512;  // compute threads

template <int D>
struct DkdvCfg : Tiles<D> {
    using T = Tiles<D>;
    // {Q_i, dO_i} ring stages: a stage's next load starts when dK of its last
    // step is done; at d = 64 (32 KB stages) shared memory has room for a third
    static constexpr int NST = (D == 64) ? 3 : 2;
    // d = 64: persistent CTAs, one per SM, dealt items longest first; dV and
    // dK are staged for their TMA stores in a buffer of their own, so the next
    // item's first stages can land meanwhile.  d = 128 has no room for that
    // buffer: one item per CTA, dV and dK staged in stage 0's tiles.
    static constexpr bool PERSIST = (D == 64);
    // K/V buffers: at d = 64 item it's K, V go to buffer it % 2, loaded while
    // item it - 1 runs (once item it - 2 is done with the buffer)
    static constexpr int KVB = PERSIST ? 2 : 1;
    // smem: K, V, then NST stages of {Q_i, dO_i}, then per-stage lse2 / D
    // vectors, then (d = 64) the dV, dK staging tiles and the second K, V
    static constexpr int OFF_STAGE = 2 * T::TILE;
    static constexpr int OFF_VEC = OFF_STAGE + NST * 2 * T::TILE;
    static constexpr int VEC_BYTES = 2 * kBM * 4;  // lse2[128], D[128]
    static constexpr int OFF_ST = OFF_VEC + NST * VEC_BYTES;  // a multiple of 1024
    static constexpr int OFF_KV2 = OFF_ST + (PERSIST ? 2 * T::TILE : 0);
    static constexpr int OFF_BAR = OFF_KV2 + (KVB - 1) * 2 * T::TILE;
    // barriers: K/V full, stage full[NST], stage empty[NST], dP^T ready, dP^T
    // copied to registers, P^T written, dS^T written, an item's MMAs done, S^T
    // ready, K/V free, dV/dK staged, staging free, all MMAs done, then K/V full
    // and free of the second buffer
    static constexpr int NBAR = 1 + 2 * NST + 6 + 4 + 2 * (KVB - 1);
    static constexpr int SMEM_BYTES = 1024 + OFF_BAR + NBAR * 8 + 16;
    static_assert(SMEM_BYTES <= 232448, "dynamic shared memory above the 227 KB a block may use");
    static constexpr uint32_t TM_X = 0, TM_Y = 128, TM_ACC = 256;
};

// One work item: (batch, kv head, 128-key block), low key blocks (the most
// query blocks under the causal mask) first; its steps are (query head of the
// group, query block) pairs.
struct DkItem {
    int b, hk, jb, qi0, nqi, n_it;
};

// F16: every operand tile is the fp16 copy (Q, K, V, dO scaled by 2^q, 2^k,
// 2^v, 2^dout); P^T and dS^T * 2^ds are rounded to fp16.  S^T then carries
// 2^(q+k) (folded into scale * log2 e), dP^T 2^(v+dout), dV 2^dout and dK
// 2^(ds+q), all undone exactly.
template <int D, bool F16>
__global__ void __launch_bounds__(kDkThreads, 1)
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
    // K, V of buffer b (V follows K)
    auto sK_of = [&](int b) { return b ? sK + C::OFF_KV2 : sK; };
    const uint32_t sStage = sK + C::OFF_STAGE;  // stage s: Q at +2s*TILE, dO after it
    // where dV (which = 0) and dK (which = 1) are staged for their stores
    const uint32_t sST = C::PERSIST ? sK + C::OFF_ST : sStage;
    float* vec = reinterpret_cast<float*>(smem + C::OFF_VEC);  // stage s: lse2 at s*256, D at +128
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
    const uint32_t bar0 = smem_u32(bars);
    auto BAR_KV = [&](int b) { return b ? bar0 + 8u * (1 + 2 * C::NST + 10) : bar0; };
    auto BAR_STF = [&](int s) { return bar0 + 8u * (1 + s); };
    auto BAR_STE = [&](int s) { return bar0 + 8u * (1 + C::NST + s); };
    const uint32_t BAR_SDF = bar0 + 8u * (1 + 2 * C::NST);  // step's dP^T ready
    const uint32_t BAR_LD = BAR_SDF + 8u;                   // dP^T copied to registers
    const uint32_t BAR_PF = BAR_SDF + 16u;                  // P^T written
    const uint32_t BAR_DSF = BAR_SDF + 24u;                 // dS^T written
    const uint32_t BAR_ACC = BAR_SDF + 32u;                 // the item's dV, dK complete
    const uint32_t BAR_STR = BAR_SDF + 40u;                 // step's S^T ready
    auto BAR_KVE = [&](int b) {  // the item's K, V no longer read
        return b ? BAR_SDF + 88u : BAR_SDF + 48u;
    };
    const uint32_t BAR_EPF = BAR_SDF + 56u;                 // the item's dV, dK staged
    const uint32_t BAR_EPE = BAR_SDF + 64u;                 // the staging stored (free again)
    const uint32_t BAR_DONE = BAR_SDF + 72u;

    const int warp = warp_id();
    const int lane = lane_id();
    const int nqb = (a.N + kBM - 1) / kBM;
    const int per = a.B * a.Hkv;
    const int n_items = nqb * per;
    // Steps carry global indices g across a CTA's items, so the stage ring,
    // the TMEM regions (X/Y by g's parity) and the per-step barriers run on
    // from one item to the next.
    auto item = [&](int w) {
        DkItem I;
        I.jb = w / per;  // causal: low key blocks have most work
        const int bh = w % per;
        I.b = bh / a.Hkv;
        I.hk = bh % a.Hkv;
        I.qi0 = a.causal ? I.jb : 0;  // first query block that sees this key block
        I.nqi = nqb - I.qi0;
        I.n_it = a.g * I.nqi;         // (query head of the group, query block) pairs
        return I;
    };

    if (warp == 0 && lane == 0) {
        for (int b = 0; b < C::KVB; ++b) {
            mbar_init(BAR_KV(b), 1);
            mbar_init(BAR_KVE(b), 1);
        }
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(BAR_STF(s), 1 + 32);  // TMA transaction arrive + 32 lanes' vector writes
            mbar_init(BAR_STE(s), 1);
        }
        mbar_init(BAR_SDF, 1);
        mbar_init(BAR_LD, kDkCompute);
        mbar_init(BAR_PF, kDkCompute);
        mbar_init(BAR_DSF, kDkCompute);
        mbar_init(BAR_ACC, 1);
        mbar_init(BAR_STR, 1);
        mbar_init(BAR_EPF, kDkCompute);
        mbar_init(BAR_EPE, 1);
        mbar_init(BAR_DONE, 1);
        fence_barrier_init();
    }
    if (warp == kDkWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    // region of S^T(g) (then P^T, dS^T), and of dP^T(g)
    auto reg_s = [&](int g) { return tbase + ((g & 1) ? C::TM_Y : C::TM_X); };
    auto reg_d = [&](int g) { return tbase + ((g & 1) ? C::TM_X : C::TM_Y); };

    if (warp == kDkWarpLoad) {
        // TMA for tiles (lane 0); all 32 lanes fill the per-query lse2 / D vectors
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmDO);
            tma_prefetch_desc(&tmDK);
            tma_prefetch_desc(&tmDV);
        }
        const uint64_t pol_q = l2_policy_evict_last();
        int last_it[C::NST];
        for (int s = 0; s < C::NST; ++s) last_it[s] = -1;
        // fp16 path: D is staged times 2^ds, the scale of dP^T (V dO^T of the
        // copies carries exactly 2^ds: the copy of dO is scaled by ds - v)
        const float dsc = F16 ? pow2f(ld_once(&a.f16s->ds)) : 1.f;
        // A step's lse and D values (4 queries a lane) are read from global
        // memory one step before the step that stages them and are first used
        // there, so their latency never holds up the producer: two register sets,
        // picked by the parity of the global step index (no copy between them,
        // which would wait for the loads).  Rows past N read row N - 1 and are
        // replaced when staged.
        auto raw_vals = [&](const DkItem& It, int j, float (&r)[8]) {
            const int hq = It.hk * a.g + j / It.nqi;
            const int qi = It.qi0 + j % It.nqi;
            const size_t base = (static_cast<size_t>(It.b) * a.Hq + hq) * a.N;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int q = min(qi * kBM + lane * 4 + u, a.N - 1);
                r[u] = a.lse[base + q];
                r[4 + u] = a.dsum[base + q];
            }
        };
        float ra[8], rb[8];
        bool ok = true;
        int g0 = 0, it = 0;
        if (static_cast<int>(blockIdx.x) < n_items) raw_vals(item(blockIdx.x), 0, ra);
        for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++it) {
            const DkItem I = item(w);
            // the buffer's previous item's last S^T and dP^T are done with K, V
            const int kb = it % C::KVB;
            if (it >= C::KVB &&
                !(ok = mbar_wait_warp(BAR_KVE(kb), ((it - C::KVB) / C::KVB) & 1, a.watch, 44)))
                break;
            if (lane == 0) {
                const uint32_t dK = sK_of(kb), dV = dK + C::TILE;
                mbar_arrive_expect_tx(BAR_KV(kb), 2 * C::TILE);
                for (int c = 0; c < C::NCH; ++c) {
                    tma_load_4d(dK + c * C::CHUNK, &tmK, BAR_KV(kb), c * 64, I.hk, I.jb * kBN, I.b);
                    tma_load_4d(dV + c * C::CHUNK, &tmV, BAR_KV(kb), c * 64, I.hk, I.jb * kBN, I.b);
                }
            }
            for (int j = 0; j < I.n_it; ++j) {
                const int g = g0 + j;
                const int s = g % C::NST;
                const int hq = I.hk * a.g + j / I.nqi;
                const int qi = I.qi0 + j % I.nqi;
                auto step = [&](const float (&cur)[8], float (&nxt)[8]) -> bool {
                    // the next step's values (the next item's first step after the last)
                    if (j + 1 < I.n_it)
                        raw_vals(I, j + 1, nxt);
                    else if (w + static_cast<int>(gridDim.x) < n_items)
                        raw_vals(item(w + gridDim.x), 0, nxt);
                    // L2 prefetch of the Q, dO tiles two steps ahead (no slot needed)
                    if (lane == 0 && j + 2 < I.n_it) {
                        const int j2 = j + 2;
                        const int hq2 = I.hk * a.g + j2 / I.nqi, q2 = (I.qi0 + j2 % I.nqi) * kBM;
                        for (int c = 0; c < C::NCH; ++c) {
                            tma_prefetch_4d(&tmQ, c * 64, hq2, q2, I.b, pol_q);
                            tma_prefetch_4d(&tmDO, c * 64, hq2, q2, I.b, pol_q);
                        }
                    }
                    if (!mbar_wait_warp(BAR_STE(s), ((g / C::NST) & 1) ^ 1u, a.watch, 30)) return false;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(BAR_STF(s), 2 * C::TILE);
                        const uint32_t dst = sStage + 2 * s * C::TILE;
                        for (int c = 0; c < C::NCH; ++c) {
                            tma_load_4d_hint(dst + c * C::CHUNK, &tmQ, BAR_STF(s), c * 64, hq, qi * kBM,
                                             I.b, pol_q);
                            tma_load_4d_hint(dst + C::TILE + c * C::CHUNK, &tmDO, BAR_STF(s), c * 64, hq,
                                             qi * kBM, I.b, pol_q);
                        }
                    }
                    float lv[4], dv4[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        // a query row past N contributes nothing: P = exp2(-inf) = 0
                        const bool in = qi * kBM + lane * 4 + u < a.N;
                        lv[u] = in ? cur[u] * kLog2e : INFINITY;
                        dv4[u] = in ? cur[4 + u] * dsc : 0.f;
                    }
                    float* lse2 = vec + s * 2 * kBM;
                    *reinterpret_cast<float4*>(lse2 + lane * 4) = make_float4(lv[0], lv[1], lv[2], lv[3]);
                    *reinterpret_cast<float4*>(lse2 + kBM + lane * 4) =
                        make_float4(dv4[0], dv4[1], dv4[2], dv4[3]);
                    mbar_arrive(BAR_STF(s));
                    return true;
                };
                if (!(ok = (g & 1) ? step(rb, ra) : step(ra, rb))) break;
                last_it[s] = g;
            }
            g0 += I.n_it;
        }
        if (lane == 0) {  // no copies in flight at exit
            for (int b = 0; b < C::KVB; ++b)
                if (it > b) {  // the buffer's last load
                    const int last = b + ((it - 1 - b) / C::KVB) * C::KVB;
                    mbar_drain(BAR_KV(b), (last / C::KVB) & 1, a.watch, 31);
                }
            for (int s = 0; s < C::NST; ++s)
                if (last_it[s] >= 0)
                    mbar_drain(BAR_STF(s), (last_it[s] / C::NST) & 1, a.watch, 31);
        }
        __syncwarp();
    } else if (warp == kDkWarpStore) {
        // ================= store: each item's staged dV and dK -> global memory =================
        bool ok = true;
        int it = 0;
        for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++it) {
            const DkItem I = item(w);
            if (!(ok = mbar_wait_warp(BAR_EPF, it & 1, a.watch, 45))) break;
            if (lane == 0) {
                for (int which = 0; which < 2; ++which) {
                    const CUtensorMap* tm = which ? &tmDK : &tmDV;
                    for (int c = 0; c < C::NCH; ++c)
                        tma_store_4d(tm, sST + which * C::TILE + c * C::CHUNK, c * 64, I.hk,
                                     I.jb * kBN, I.b);
                }
                tma_store_commit();
                tma_store_wait_read_all();
                mbar_arrive(BAR_EPE);  // the staging may be written again
            }
            __syncwarp();
        }
    } else if (warp == kDkWarpMma) {
        {
            const uint32_t leader = elect_one();
            constexpr uint32_t IDESC_S = idesc_16(kBN, kBM, false, false, F16);  // S^T, dP^T
            constexpr uint32_t IDESC_ACC = idesc_16(kBN, D, false, true, F16);  // dV, dK
            const uint32_t tDV = tbase + C::TM_ACC, tDK = tbase + C::TM_ACC + D;
            auto stage_q = [&](int s) { return sStage + 2 * s * C::TILE; };
            // descriptors built once per tile; each MMA only moves the start address
            constexpr uint32_t HI = sdesc_hi(1024);
            // dst = A B^T over the head dimension: S^T = K Q^T or dP^T = V dO^T
            auto issue_t = [&](uint32_t dst, uint32_t a_lo, uint32_t sB) {
                const uint32_t b_lo = sdesc_lo(sB, 16);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
                    mma_bf16_ss_w(leader, dst, sdesc_at(a_lo, HI, off), sdesc_at(b_lo, HI, off), IDESC_S, ks > 0);
                }
            };
            // dV += P^T dO (dk = false) or dK += dS^T Q (dk = true), starting afresh
            // at an item's first step: for queries 16ks.., P^T / dS^T (16-bit
            // pairs) sit in columns 32w + (ks%2)*8 / 32w + 16 + (ks%2)*8 of S^T's
            // region (w = ks/2); dO, Q rows 16ks.. are read MN-major
            auto issue_acc = [&](int g, int s, bool dk, bool first) {
                const uint32_t b_lo = sdesc_lo(stage_q(s) + (dk ? 0 : C::TILE), C::CHUNK);
                const uint32_t rs = reg_s(g) + (dk ? 16 : 0);
#pragma unroll
                for (int ks = 0; ks < kBM / 16; ++ks)
                    mma_bf16_ts_w(leader, dk ? tDK : tDV, rs + (ks >> 1) * 32 + (ks & 1) * 8,
                                sdesc_at(b_lo, HI, ks * 2048), IDESC_ACC, (first && ks == 0) ? 0u : 1u);
            };
            // per step: dV(g) once P^T(g) is written; S^T(g+1) over dP^T(g)
            // once every warp holds dP^T(g); dK(g) once dS^T(g) is written;
            // dP^T(g+1) over P^T(g), dS^T(g), which the two products above
            // read first.  The warps form P^T(g+1) from S^T(g+1) while the
            // tensor core runs dK(g) and dP^T(g+1).
            bool ok = true;
            int g0 = 0, it = 0;
            for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++it) {
                const DkItem I = item(w);
                const int n = I.n_it;
                const int kb = it % C::KVB;
                const uint32_t k_lo = sdesc_lo(sK_of(kb), 16), v_lo = sdesc_lo(sK_of(kb) + C::TILE, 16);
                if (!(ok = mbar_wait_warp(BAR_KV(kb), (it / C::KVB) & 1, a.watch, 32) &&
                           mbar_wait_warp(BAR_STF(g0 % C::NST), (g0 / C::NST) & 1, a.watch, 33)))
                    break;
                // S^T(g0) goes over dP^T of the previous item's last step, which
                // every warp holds (implied by its DSF, waited below; kept so that
                // the parity waits on LD stay in order)
                if (it > 0 && !(ok = mbar_wait_warp(BAR_LD, (g0 - 1) & 1, a.watch, 34))) break;
                tc_fence_after();
                issue_t(reg_s(g0), k_lo, stage_q(g0 % C::NST));
                mma_commit_w(leader, BAR_STR);
                issue_t(reg_d(g0), v_lo, stage_q(g0 % C::NST) + C::TILE);
                mma_commit_w(leader, BAR_SDF);
                if (n == 1) mma_commit_w(leader, BAR_KVE(kb));  // the item's last S^T and dP^T
                for (int j = 0; j < n && ok; ++j) {
                    const int g = g0 + j;
                    const int s = g % C::NST;
                    const int s2 = (g + 1) % C::NST;
                    const bool more = j + 1 < n;
                    if (!(ok = mbar_wait_warp(BAR_PF, g & 1, a.watch, 34))) break;
                    tc_fence_after();
                    issue_acc(g, s, false, j == 0);
                    if (more) {
                        if (!(ok = mbar_wait_warp(BAR_STF(s2), ((g + 1) / C::NST) & 1, a.watch, 33)))
                            break;
                        if (!(ok = mbar_wait_warp(BAR_LD, g & 1, a.watch, 34))) break;
                        tc_fence_after();
                        issue_t(reg_s(g + 1), k_lo, stage_q(s2));  // over dP^T(g)
                        mma_commit_w(leader, BAR_STR);
                    }
                    if (!(ok = mbar_wait_warp(BAR_DSF, g & 1, a.watch, 38))) break;
                    tc_fence_after();
                    issue_acc(g, s, true, j == 0);
                    mma_commit_w(leader, BAR_STE(s));
                    if (more) {
                        issue_t(reg_d(g + 1), v_lo, stage_q(s2) + C::TILE);  // over P^T(g), dS^T(g)
                        mma_commit_w(leader, BAR_SDF);
                        if (j + 2 == n) mma_commit_w(leader, BAR_KVE(kb));  // the item's last S^T, dP^T
                    }
                }
                if (!ok) break;
                mma_commit_w(leader, BAR_ACC);  // the item's dV and dK are complete
                g0 += n;
            }
            // every issued MMA has finished before TMEM is released
            mma_commit_w(leader, BAR_DONE);
            mbar_drain(BAR_DONE, 0, a.watch, 35);
        }
        __syncwarp();
    } else if (warp < 16) {
        const int wg = warp >> 2;  // queries 32*wg..32*wg+31 of each block
        const int r = (warp & 3) * 32 + lane;
        const int t4 = lane & 3;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        // fp16 path: undo 2^(q+k) on S^T; dP^T and the staged D both carry
        // 2^ds, so dS^T = P^T (dP^T - D) does too
        int eq = 0, ek = 0, ev = 0, edo = 0;
        if (F16) ld_once_v4(&a.f16s->q, eq, ek, ev, edo);
        const int eds = F16 ? ld_once(&a.f16s->ds) : 0;
        const float sl2 = a.scale_log2 * pow2f(-(eq + ek));
        // the epilogue factor, formed here so the exponents die before the loop:
        // dV carries 2^dout, dK scale * 2^(ds+q) on the fp16 path
        const int which = wg >> 1, half = wg & 1;
        const float mul_e = which ? a.scale * pow2f(-(eds + eq)) : pow2f(-edo);
        const uint64_t sl2x2 = f2(sl2, sl2);
        bool ok = true;
        int g0 = 0, it = 0;
        for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++it) {
            const DkItem I = item(w);
            // In the 16x256b TMEM shape a thread holds, of each 16-lane block of
            // its warp's 32 lanes, rows lane/4 and lane/4 + 8 and the 8 columns
            // 8j + 2(lane%4) + {0,1} of the warpgroup's 32: so it needs only 8
            // entries of the query-indexed vectors lse2 and D.
            const int key0 = I.jb * kBN + (warp & 3) * 32 + (lane >> 2);
            for (int j = 0; j < I.n_it; ++j) {
                const int g = g0 + j;
                const int s = g % C::NST;
                const int qi = I.qi0 + j % I.nqi;
                const uint32_t rs = reg_s(g) + wg * 32 + lane_off;
                const uint32_t rd = reg_d(g) + wg * 32 + lane_off;
                const float* lse2 = vec + s * 2 * kBM + wg * 32;
                const float* dvec = vec + s * 2 * kBM + kBM + wg * 32;
                const int qbase = qi * kBM + wg * 32 + 2 * t4;  // query of the thread's column 0
                // ---- P^T = exp2(S^T scale log2 e - lse2), as soon as S^T is in TMEM
                if (!(ok = mbar_wait_warp(BAR_STR, g & 1, a.watch, 36))) break;
                tc_fence_after();
                uint64_t nl[4];  // -lse2 of the thread's column pairs
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float2 l2 = *reinterpret_cast<const float2*>(lse2 + 8 * jj + 2 * t4);
                    nl[jj] = f2(-l2.x, -l2.y);
                }
                uint32_t pk[2][8];  // P^T (16-bit pairs), kept for dS^T
#pragma unroll
                for (int lb = 0; lb < 2; ++lb) {  // TMEM lanes 16*lb.. of the warp's 32
                    const uint32_t lo = static_cast<uint32_t>(lb * 16) << 16;
                    uint32_t sv[16];
                    tmem_ld16x256_x4(rs + lo, sv);
                    tmem_wait_ld();
                    reg_fence<16>(sv);
                    const int key = key0 + 16 * lb;  // key of the thread's first row (+8: second)
                    // causal: key k is hidden from query q when k > q
                    const bool need_mask = a.causal && key + 8 > qbase;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
                        for (int rsel = 0; rsel < 2; ++rsel) {
                            const int i = 4 * jj + 2 * rsel;
                            float x0, x1;
                            f2_split(fma2(f2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), sl2x2,
                                          nl[jj]), x0, x1);
                            float p0 = ex2(x0), p1 = ex2(x1);
                            if (need_mask) {
                                const int q = qbase + 8 * jj, k = key + 8 * rsel;
                                p0 = (k > q) ? 0.f : p0;
                                p1 = (k > q + 1) ? 0.f : p1;
                            }
                            pk[lb][2 * jj + rsel] = pack_op<F16>(p0, p1);
                        }
                    }
                    tmem_st16x128_x4(rs + lo, pk[lb]);  // P^T over the first 16 S^T columns read
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(BAR_PF);
                // ---- dS^T = P^T (dP^T - D), once dP^T is in TMEM (from the rounded P^T)
                if (!(ok = mbar_wait_warp(BAR_SDF, g & 1, a.watch, 40))) break;
                tc_fence_after();
                uint32_t dp[2][16];
                tmem_ld16x256_x4(rd, dp[0]);
                tmem_ld16x256_x4(rd + (16u << 16), dp[1]);
                uint64_t nd[4];  // -D of the thread's column pairs
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float2 d2 = *reinterpret_cast<const float2*>(dvec + 8 * jj + 2 * t4);
                    nd[jj] = f2(-d2.x, -d2.y);
                }
                tmem_wait_ld();
                reg_fence<16>(dp[0]);
                reg_fence<16>(dp[1]);
                // every warp holds dP^T: S^T(g+1) may overwrite it
                tc_fence_before();
                mbar_arrive(BAR_LD);
                uint32_t dk[2][8];
#pragma unroll
                for (int lb = 0; lb < 2; ++lb)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                        for (int rsel = 0; rsel < 2; ++rsel) {
                            const int i = 4 * jj + 2 * rsel;
                            const uint64_t t = add2(
                                f2(__uint_as_float(dp[lb][i]), __uint_as_float(dp[lb][i + 1])), nd[jj]);
                            if constexpr (F16) {
                                // fp16 path: dP^T - D rounded to fp16, then one packed
                                // fp16 product with the rounded P^T (two roundings of
                                // 2^-11 each, three instructions a pair)
                                float t0, t1;
                                f2_split(t, t0, t1);
                                dk[lb][2 * jj + rsel] = mul_f16x2(pk[lb][2 * jj + rsel], pack_f16(t0, t1));
                            } else {
                                float p0, p1, e0, e1;
                                unpack_op<F16>(pk[lb][2 * jj + rsel], p0, p1);
                                f2_split(mul2(f2(p0, p1), t), e0, e1);
                                dk[lb][2 * jj + rsel] = pack_op<F16>(e0, e1);
                            }
                        }
                tmem_st16x128_x4(rs + 16, dk[0]);  // dS^T over the other 16
                tmem_st16x128_x4(rs + (16u << 16) + 16, dk[1]);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(BAR_DSF);
            }
            if (!ok) break;
            g0 += I.n_it;
            // ---- epilogue: warpgroups 0, 1 write the two column halves of dV,
            // warpgroups 2, 3 those of dK = scale * (dS^T Q), into the staging
            // for the store warp.  The next item's dV, dK products start the
            // accumulators afresh only after PF / DSF of its first step, which
            // every warp arrives on after these TMEM loads.
            if (!(ok = mbar_wait_warp(BAR_ACC, it & 1, a.watch, 37))) break;
            tc_fence_after();
            // the staging is free once the previous item's stores have read it
            if (C::PERSIST && it > 0 && !(ok = mbar_wait_warp(BAR_EPE, (it - 1) & 1, a.watch, 46)))
                break;
            // dV carries 2^dout, dK 2^(ds+q) on the fp16 path
            stage_rows_bf16<C::CHUNK>(tbase + C::TM_ACC + which * D + lane_off, sST + which * C::TILE,
                                      r, half * (D / 2), (half + 1) * (D / 2), mul_e);
            fence_proxy_async_smem();
            mbar_arrive(BAR_EPF);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kDkWarpMma) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

}  // namespace

template <int D, bool F16>
cudaError_t launch_dkdv(const BwdMaps& m, const BwdArgs& a, cudaStream_t st) {
    auto kern = fa_bwd_dkdv_kernel<D, F16>;
    constexpr int smem = DkdvCfg<D>::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long items = static_cast<long long>((a.N + kBN - 1) / kBN) * a.B * a.Hkv;
    if (items <= 0 || items > 0x7fffffffLL || a.num_ctas <= 0) return cudaErrorInvalidConfiguration;
    // d = 64: persistent, one CTA per SM; d = 128: one CTA per item
    const long long ctas = DkdvCfg<D>::PERSIST ? (items < a.num_ctas ? items : a.num_ctas) : items;
    const unsigned grid = static_cast<unsigned>(ctas);
    if (F16)
        kern<<<grid, kDkThreads, smem, st>>>(m.q16, m.k16, m.v16, m.dout16, m.dk, m.dv, a);
    else
        kern<<<grid, kDkThreads, smem, st>>>(m.q, m.k, m.v, m.dout, m.dk, m.dv, a);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_dkdv(const BwdMaps& m, const BwdArgs& a, cudaStream_t st) {
    return a.f16s ? launch_dkdv<D, true>(m, a, st) : launch_dkdv<D, false>(m, a, st);
}

template cudaError_t launch_bwd_dkdv<64>(const BwdMaps&, const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_dkdv<128>(const BwdMaps&, const BwdArgs&, cudaStream_t);

}  // namespace fa
