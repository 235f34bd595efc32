// fa_decode.cu -- split-KV forward (FlashDecoding) for sm_103a: Nq queries
// against a long key/value sequence of Nk, the key range cut into splits that
// run as separate CTAs, then an exact combine.
//
// What it computes: the same O = softmax(scale * Q K^T [+ causal]) V and lse as
// fa_fwd, for queries that are the last Nq positions of a sequence of Nk
// (causal: query i sees keys j <= i + Nk - Nq).  The pages describe
// FlashDecoding as parallelising decoding over the key/value length and then
// combining ("FlashAttention Kernel", the FlashDecoding mentions); the combine
// is the online-softmax merge of two blocks ("FlashAttention 1, 2, and 3
// Explained", section 2: l = e^{m1-m} l1 + e^{m2-m} l2, O likewise), applied to
// the splits' (O_s, lse_s).
//
// Decode is bound by reading K and V from HBM once, so the design serves that:
//   * the g query heads of a KV group share one CTA: its 128-row query tile
//     holds (query, head) pairs -- QPT = 128 / g queries of all g heads, one
//     TMA box of g heads x QPT queries -- so K and V are read once per group,
//     not once per head;
//   * every CTA streams its split's K/V blocks through a 6-slot TMA ring (three
//     blocks of K and V in flight); S is double-buffered in TMEM so S(j+1)
//     and O += P(j-1) V run on the tensor core while the softmax of block j
//     runs; the grid is sized to fill the GPU's 152 SMs at least twice;
//   * one softmax thread per tile row (= TMEM lane), exp2 with scale * log2 e
//     folded in, the lazy rescale of the forward kernel (the reference max
//     moves only by more than 2^8; O is rescaled in TMEM after the product
//     that last wrote it has finished);
//   * with one split the kernel writes bf16 O and lse itself; with several,
//     fp32 (O_s, lse_s) per split go to the caller's workspace and
//     fa_decode_combine_kernel merges them.
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

template <int D>
struct DecCfg {
    static constexpr int CHUNK = kBM * 128;           // one 64-column chunk of a 128-row tile
    static constexpr int NCH = D / 64;
    static constexpr int TILE = NCH * CHUNK;          // 128 x D bf16
    static constexpr int NSLOT = (D == 128) ? 6 : 12;  // K/V ring slots
    // barriers: q_full, kv_full[NSLOT], kv_empty[NSLOT], s_full[2], p_full[2],
    // pv_done, o_final
    static constexpr int NBAR = 1 + 2 * NSLOT + 2 + 2 + 1 + 1;
    static constexpr int SMEM_BYTES = 1024 + TILE + NSLOT * TILE + NBAR * 8 + 16;
    static constexpr uint32_t TM_S = 0, TM_O = 256;   // S0 [0,128), S1 [128,256), O [256, 256+D)
    static constexpr int THREADS = 192;               // softmax warps 0-3, MMA warp 4, TMA warp 5
};

// The key blocks a CTA visits: every block of [lo, hi).  Every role walks
// the same sequence.
struct KeyBlocks {
    int lo, hi;
    __device__ int next(int kb) const { return kb + 1; }
    __device__ int first() const { return lo; }
    __device__ int count() const { return hi > lo ? hi - lo : 0; }
};

constexpr int kDecWarpMma = 4;
constexpr int kDecWarpLoad = 5;
constexpr float kDecRescale = 8.0f;  // lazy rescale threshold (log2 units)

template <int D>
__global__ void __launch_bounds__(DecCfg<D>::THREADS, 1)
    fa_decode_split_kernel(const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const DecodeArgs a) {
    using C = DecCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sKV = sQ + C::TILE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::TILE + C::NSLOT * C::TILE);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t BAR_Q = bar0;
    auto BAR_KVF = [&](int s) { return bar0 + 8u * (1 + s); };
    auto BAR_KVE = [&](int s) { return bar0 + 8u * (1 + C::NSLOT + s); };
    auto BAR_SF = [&](int t) { return bar0 + 8u * (1 + 2 * C::NSLOT + t); };
    auto BAR_PF = [&](int t) { return bar0 + 8u * (3 + 2 * C::NSLOT + t); };
    const uint32_t BAR_PVD = bar0 + 8u * (5 + 2 * C::NSLOT);  // O += P(j) V_j done
    const uint32_t BAR_OF = bar0 + 8u * (6 + 2 * C::NSLOT);   // all products done

    const int warp = warp_id();
    const int lane = lane_id();

    // ---- work decode: split fastest, then query tile, then (batch, head group)
    int t = static_cast<int>(blockIdx.x);
    const int split = t % a.splits;
    t /= a.splits;
    const int qt = t % a.n_qt;
    t /= a.n_qt;
    const int n_hg = a.Hq / a.gp;
    const int b = t / n_hg;
    const int h0 = (t % n_hg) * a.gp;                  // first query head of the tile
    const int hk = h0 / a.g;                           // the key/value head they share
    const int q0 = qt * a.qpt;                         // first query of the tile
    const int nq_tile = min(a.qpt, a.Nq - q0);         // queries in this tile
    const int rows = nq_tile * a.gp;                   // valid tile rows
    const int nkv_all = (a.Nk + kBN - 1) / kBN;
    const int jb0 = split * a.blocks_per_split;
    int jb1 = min(jb0 + a.blocks_per_split, nkv_all);
    if (a.causal) jb1 = min(jb1, (q0 + nq_tile - 1 + a.Nk - a.Nq) / kBN + 1);
    const KeyBlocks blocks{jb0, jb1};
    const int nkv = blocks.count();

    if (warp == 0 && lane == 0) {
        mbar_init(BAR_Q, 1);
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(BAR_KVF(s), 1);
            mbar_init(BAR_KVE(s), 1);
        }
        for (int u = 0; u < 2; ++u) {
            mbar_init(BAR_SF(u), 1);
            mbar_init(BAR_PF(u), 128);
        }
        mbar_init(BAR_PVD, 1);
        mbar_init(BAR_OF, 1);
        fence_barrier_init();
    }
    // tile rows the TMA box does not cover start at zero (the MMA reads all 128)
    if (warp < 4) {
        const int r = threadIdx.x;
        if (r >= a.gp * a.qpt) {
            for (int c = 0; c < C::NCH; ++c)
                for (int p = 0; p < 8; ++p)
                    st_shared_v4(sQ + c * C::CHUNK + r * 128 + p * 16, 0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
    }
    if (warp == kDecWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    if (warp == kDecWarpLoad) {
        // ================= TMA producer =================
        if (lane == 0 && nkv > 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            const uint64_t pol = l2_policy_evict_first();  // K, V are read once
            mbar_arrive_expect_tx(BAR_Q, C::NCH * a.gp * a.qpt * 128);
            for (int c = 0; c < C::NCH; ++c)
                tma_load_4d(sQ + c * C::CHUNK, &tmQ, BAR_Q, c * 64, h0, q0, b);
            int last_idx[C::NSLOT];
            for (int s = 0; s < C::NSLOT; ++s) last_idx[s] = -1;
            bool ok = true;
            int kb = blocks.first();
            for (int j = 0; j < nkv && ok; ++j, kb = blocks.next(kb)) {
                for (int w = 0; w < 2; ++w) {  // K_j then V_j
                    const int idx = 2 * j + w;
                    const int slot = idx % C::NSLOT;
                    if (!(ok = mbar_wait(BAR_KVE(slot), ((idx / C::NSLOT) & 1) ^ 1u, a.watch, 40)))
                        break;
                    mbar_arrive_expect_tx(BAR_KVF(slot), C::TILE);
                    for (int c = 0; c < C::NCH; ++c)
                        tma_load_4d_hint(sKV + slot * C::TILE + c * C::CHUNK, w ? &tmV : &tmK,
                                         BAR_KVF(slot), c * 64, hk, kb * kBN, b, pol);
                    last_idx[slot] = idx;
                }
            }
            // no copies in flight at exit
            mbar_drain(BAR_Q, 0, a.watch, 41);
            for (int s = 0; s < C::NSLOT; ++s)
                if (last_idx[s] >= 0)
                    mbar_drain(BAR_KVF(s), (last_idx[s] / C::NSLOT) & 1, a.watch,
                              41);
        }
        __syncwarp();
    } else if (warp == kDecWarpMma) {
        // ================= MMA issuer (one thread) =================
        // order: S(0), S(1), PV(0), S(2), PV(1), ...: the softmax of block j
        // overlaps S(j+1) and PV(j-1)
        if (lane == 0 && nkv > 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(kBM, kBN, false, false);
            constexpr uint32_t IDESC_PV = idesc_bf16(kBM, D, false, true);
            constexpr uint32_t HI = sdesc_hi(1024);
            const uint32_t q_lo = sdesc_lo(sQ, 16);
            const uint32_t tO = tbase + C::TM_O;
            auto slot_of = [&](int j, int w) { return (2 * j + w) % C::NSLOT; };
            auto landed = [&](int j, int w) {
                const int idx = 2 * j + w;
                const bool r = mbar_wait(BAR_KVF(idx % C::NSLOT), (idx / C::NSLOT) & 1, a.watch, 42);
                tc_fence_after();
                return r;
            };
            auto issue_s = [&](int j) {  // S(j) = Q K_j^T into buffer j & 1
                const uint32_t k_lo = sdesc_lo(sKV + slot_of(j, 0) * C::TILE, 16);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
                    mma_bf16_ss(tbase + C::TM_S + (j & 1) * kBN, sdesc_at(q_lo, HI, off),
                                sdesc_at(k_lo, HI, off), IDESC_S, ks > 0);
                }
                mma_commit(BAR_SF(j & 1));
                mma_commit(BAR_KVE(slot_of(j, 0)));
            };
            auto issue_pv = [&](int j) {  // O += P(j) V_j, P (bf16) over S buffer j & 1
                const uint32_t v_lo = sdesc_lo(sKV + slot_of(j, 1) * C::TILE, C::CHUNK);
                const uint32_t aP = tbase + C::TM_S + (j & 1) * kBN;
#pragma unroll
                for (int ks = 0; ks < kBN / 16; ++ks)
                    mma_bf16_ts(tO, aP + ks * 8, sdesc_at(v_lo, HI, ks * 2048), IDESC_PV,
                                (j > 0 || ks > 0) ? 1u : 0u);
                mma_commit(BAR_KVE(slot_of(j, 1)));
                mma_commit(BAR_PVD);
            };
            bool ok = mbar_wait(BAR_Q, 0, a.watch, 43);
            if (ok && (ok = landed(0, 0))) issue_s(0);
            for (int j = 0; j < nkv && ok; ++j) {
                // S(j+1) into the other buffer: its previous content, P(j-1), was
                // read by PV(j-1), issued earlier by this thread
                if (j + 1 < nkv) {
                    if (!(ok = landed(j + 1, 0))) break;
                    issue_s(j + 1);
                }
                if (!(ok = mbar_wait(BAR_PF(j & 1), (j >> 1) & 1, a.watch, 44)))
                    break;
                tc_fence_after();
                if (!(ok = landed(j, 1))) break;
                issue_pv(j);
            }
            mma_commit(BAR_OF);
            mbar_drain(BAR_OF, 0, a.watch, 45);
        }
        __syncwarp();
    } else {
        // ================= softmax: one tile row per thread =================
        const int r = threadIdx.x;  // tile row = TMEM lane
        const bool valid = r < rows;
        const int qn = q0 + (valid ? r / a.gp : 0);  // query index
        const int h = h0 + (valid ? r % a.gp : 0);   // query head
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t tO = tbase + C::TM_O + lane_off;
        const float sl2 = a.scale_log2;
        const int lim = a.causal ? min(qn + a.Nk - a.Nq, a.Nk - 1) : a.Nk - 1;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        int kb = blocks.first();
        for (int j = 0; j < nkv; ++j, kb = blocks.next(kb)) {
            if (!(ok = mbar_wait_warp(BAR_SF(j & 1), (j >> 1) & 1, a.watch, 46))) break;
            tc_fence_after();
            const uint32_t tS = tbase + C::TM_S + (j & 1) * kBN + lane_off;
            uint32_t s[kBN];
            tmem_ld32(tS + 0, s);
            tmem_ld32(tS + 32, s + 32);
            tmem_ld32(tS + 64, s + 64);
            tmem_ld32(tS + 96, s + 96);
            tmem_wait_ld();
            reg_fence<kBN>(s);
            float x[kBN];
#pragma unroll
            for (int c = 0; c < kBN; ++c) x[c] = __uint_as_float(s[c]);
            const int kbase = kb * kBN;
            if (kbase + kBN - 1 > lim) {  // causal edge or ragged tail
#pragma unroll
                for (int c = 0; c < kBN; ++c) x[c] = (kbase + c > lim) ? -INFINITY : x[c];
            }
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
            const bool need = m_new > m_ref + kDecRescale;
            float alpha = 1.f;
            if (need) {
                alpha = ex2(m_ref - m_new);
                l *= alpha;
                m_ref = m_new;
            }
            const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
            const uint64_t sl2x2 = f2(sl2, sl2), negx2 = f2(neg, neg);
            uint64_t ls2[4] = {0, 0, 0, 0};
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 64; c += 2) {
                    float e0, e1;
                    f2_split(fma2(f2(x[half * 64 + c], x[half * 64 + c + 1]), sl2x2, negx2), e0,
                             e1);
                    const float p0 = ex2(e0), p1 = ex2(e1);
                    ls2[(c >> 1) & 3] = add2(ls2[(c >> 1) & 3], f2(p0, p1));
                    pk[c >> 1] = pack_bf16(p0, p1);
                }
                tmem_st32(tS + half * 32, pk);
            }
            {
                const uint64_t tt = add2(add2(ls2[0], ls2[1]), add2(ls2[2], ls2[3]));
                float a0, a1;
                f2_split(tt, a0, a1);
                l += a0 + a1;
            }
            // O was last written by PV(j-1), which may still be running: wait
            // for it before rescaling (rare: only when the reference max moves)
            if (j > 0 && __any_sync(0xffffffffu, need)) {
                if (!(ok = mbar_wait_warp(BAR_PVD, (j - 1) & 1, a.watch, 47))) break;
                tc_fence_after();
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
                        f2_split(mul2(f2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), ax2),
                                 u0, u1);
                        o[i] = __float_as_uint(u0);
                        o[i + 1] = __float_as_uint(u1);
                    }
                    tmem_st32(tO + cb, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR_PF(j & 1));
        }
        // ---- epilogue: O / l and lse, straight to the output (one split) or
        // to this split's fp32 slot of the workspace
        const bool ok_e = ok && (nkv == 0 || mbar_wait_warp(BAR_OF, 0, a.watch, 48));
        if (ok_e) {
            if (nkv > 0) tc_fence_after();
            const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
            const float lse = (l > 0.f) ? (m_ref + log2f(l)) * 0.6931471805599453f : -INFINITY;
            const size_t row = (static_cast<size_t>(b) * a.Hq + h) * a.Nq + qn;  // [B, Hq, Nq]
            if (a.splits == 1) {
                uint16_t* dst = a.o + ((static_cast<size_t>(b) * a.Nq + qn) * a.Hq + h) * D;
#pragma unroll
                for (int cb = 0; cb < D; cb += 32) {
                    uint32_t o[32];
                    if (nkv > 0) {
                        tmem_ld32(tO + cb, o);
                        tmem_wait_ld();
                        reg_fence<32>(o);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = 0u;
                    }
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv_l,
                                         __uint_as_float(o[2 * i + 1]) * inv_l);
                    if (valid)
#pragma unroll
                        for (int p4 = 0; p4 < 4; ++p4)
                            reinterpret_cast<uint4*>(dst + cb)[p4] =
                                make_uint4(w[4 * p4], w[4 * p4 + 1], w[4 * p4 + 2], w[4 * p4 + 3]);
                }
                if (valid) a.lse[row] = lse;
            } else {
                const size_t srow = static_cast<size_t>(split) * a.B * a.Hq * a.Nq + row;
                float* dst = a.part_o + srow * D;
#pragma unroll
                for (int cb = 0; cb < D; cb += 32) {
                    uint32_t o[32];
                    if (nkv > 0) {
                        tmem_ld32(tO + cb, o);
                        tmem_wait_ld();
                        reg_fence<32>(o);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = 0u;
                    }
                    if (valid)
#pragma unroll
                        for (int p4 = 0; p4 < 8; ++p4)
                            reinterpret_cast<float4*>(dst + cb)[p4] =
                                make_float4(__uint_as_float(o[4 * p4]) * inv_l,
                                            __uint_as_float(o[4 * p4 + 1]) * inv_l,
                                            __uint_as_float(o[4 * p4 + 2]) * inv_l,
                                            __uint_as_float(o[4 * p4 + 3]) * inv_l);
                }
                if (valid) a.part_lse[srow] = lse;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kDecWarpMma) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// Merges the splits of every (batch, head, query) row: with m = max_s lse_s
// and w_s = e^{lse_s - m}, O = sum_s w_s O_s / sum_s w_s and
// lse = m + ln sum_s w_s (the two-block online-softmax update applied across
// the splits).  One block of 256 threads per row: all threads take the
// maximum over the splits together, then thread (group, column) sums the
// splits s = group (mod 256 / D) of one column, and the groups are added in
// shared memory.
template <int D>
__global__ void __launch_bounds__(256) fa_decode_combine_kernel(const DecodeArgs a) {
    constexpr int G = 256 / D;  // split groups
    __shared__ float red[8];
    __shared__ float part[G][D + 1];
    __shared__ float wpart[G];
    const size_t rows = static_cast<size_t>(a.B) * a.Hq * a.Nq;
    const size_t row = blockIdx.x;
    const int t = threadIdx.x;
    float m = -INFINITY;
    for (int s = t; s < a.splits; s += 256) m = fmaxf(m, a.part_lse[s * rows + row]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((t & 31) == 0) red[t >> 5] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
    const int grp = t / D, c = t % D;
    float acc = 0.f, wsum = 0.f;
#pragma unroll 4
    for (int s = grp; s < a.splits; s += G) {
        const float ls = a.part_lse[s * rows + row];
        // a split that no key of this query reaches has lse = -inf, weight 0
        const float w = (ls == -INFINITY) ? 0.f : expf(ls - m);
        wsum += w;
        acc = fmaf(w, a.part_o[(s * rows + row) * D + c], acc);
    }
    part[grp][c] = acc;
    if (c == 0) wpart[grp] = wsum;
    __syncthreads();
    if (grp == 0) {
        float tot = 0.f, wt = 0.f;
#pragma unroll
        for (int g2 = 0; g2 < G; ++g2) {
            tot += part[g2][c];
            wt += wpart[g2];
        }
        const float inv = wt > 0.f ? 1.f / wt : 0.f;
        // row = (b, h, n) -> output [B, Nq, Hq, D]
        const int n = static_cast<int>(row % a.Nq);
        const size_t bh = row / a.Nq;
        const int h = static_cast<int>(bh % a.Hq);
        const int b = static_cast<int>(bh / a.Hq);
        const float val = tot * inv;
        uint16_t* dst = a.o + ((static_cast<size_t>(b) * a.Nq + n) * a.Hq + h) * D + c;
        *dst = static_cast<uint16_t>(pack_bf16(val, 0.f) & 0xffffu);
        if (c == 0) a.lse[row] = m + logf(wt);
    }
}

template <int D>
cudaError_t launch_decode_d(const DecodeMaps& mp, const DecodeArgs& a, cudaStream_t st) {
    using C = DecCfg<D>;
    auto kern = fa_decode_split_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long nblk = static_cast<long long>(a.B) * (a.Hq / a.gp) * a.n_qt * a.splits;
    if (nblk <= 0 || nblk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<static_cast<unsigned>(nblk), C::THREADS, C::SMEM_BYTES, st>>>(mp.q, mp.k, mp.v, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (a.splits > 1) {
        const long long rows = static_cast<long long>(a.B) * a.Hq * a.Nq;
        if (rows > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        fa_decode_combine_kernel<D><<<static_cast<unsigned>(rows), 256, 0, st>>>(a);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace

cudaError_t launch_decode(const DecodeMaps& maps, const DecodeArgs& args, int d,
                          cudaStream_t stream) {
    if (d == 64) return launch_decode_d<64>(maps, args, stream);
    if (d == 128) return launch_decode_d<128>(maps, args, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa
