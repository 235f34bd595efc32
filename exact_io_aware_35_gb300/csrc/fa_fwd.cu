// fa_fwd.cu -- exact attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes: O = softmax(scale * Q K^T [+ causal mask]) V and the
// per-row log-sum-exp, one (batch, head, 256-query block) work item at a
// time, streaming 128-key blocks of K and V and folding each block into
// running row statistics with the online-softmax update of "FlashAttention
// and the Kernel Era", section "The Mathematics" (m_new = max(m, max S_j),
// l_new = l * e^{m - m_new} + sum e^{S_j - m_new}) and the output update of
// "FlashAttention 1, 2, and 3 Explained", section 2
// (O_new = diag(e^{m_old - m_new}) O_old + P_j V_j).  The N x N score matrix
// only ever exists one 128 x 128 tile at a time, in tensor memory.
//
// How it maps to sm_103a (a redesign for Blackwell, not the pages' A100/H100
// kernels):
//   * persistent CTAs, one per SM, each walking work items (longest first);
//     the K/V ring, the barrier phases and TMEM run on from one item to the
//     next, so an item's Q and first K/V loads and first score product
//     overlap the previous item's last blocks and epilogue;
//   * each item is two 128-row query tiles (Q0, Q1) in shared memory; K_j,
//     V_j stream through a ring of TMA-filled shared-memory slots;
//   * S_t = Q_t K_j^T and O_t += P_t V_j on the tensor core, accumulators and
//     P in TMEM.  At d = 128 one thread issues every product, P overwrites
//     S_t, and S_t(j+1) follows PV_t(j); at d = 64 P has TMEM columns of its
//     own and each tile has its own issuing thread, which issues S_t(j+1) as
//     soon as the softmax holds S_t(j) in registers;
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
//   * the epilogue divides O by l, rounds to bf16 and writes each row from
//     its thread's registers straight to global memory (no staging, so the
//     Q buffers are free for the next item); lse = (m + log2 l) * ln 2.  The
//     training forward also writes o_lo = bf16(O32 - O), the rounding
//     residual of O, and the fp16 copy of Q for the backward.
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

// Block-sparse: words of the per-tile mask bitmask in shared memory; rows of
// up to 32 x 224 = 7,168 key blocks (N <= 917,504) fit beside the K/V ring.
constexpr int kSparseMaskWords = kSparseMaxBlocks / 32;

template <int D, bool SPARSE>
struct FwdCfg {
    static constexpr int CHUNK = kBM * 128;          // one 64-column chunk of a 128-row tile
    static constexpr int NCH = D / 64;               // chunks per tile
    static constexpr int TILE = NCH * CHUNK;         // bytes of a 128 x D bf16 tile
    // K/V ring slots: the block-sparse kernel streams each tile's K and V on
    // its own (four ring entries per step) and takes one slot more at D = 128
    static constexpr int NSLOT = (D == 128) ? (SPARSE ? 5 : 4) : 8;
    static constexpr int SMEM_Q = 2 * TILE;
    static constexpr int SMEM_KV = NSLOT * TILE;
    // the epilogue's per-warp transpose buffers, 32 rows x 64 bytes per softmax
    // warp; block-sparse CTAs run one item each and use their tile's Q buffer
    static constexpr int SMEM_STAGE = SPARSE ? 0 : 8 * 2048;
    // barriers: q_full, q_empty, kv_full[NSLOT], kv_empty[NSLOT], s_full[2],
    // p_full[2], o_final[2], s_empty[2], pv_done[2], mma_done, for
    // block-sparse epi[2] (a tile's O staged for its TMA store), and g1 (the
    // gate has seen the item's first K entries land)
    static constexpr int NBAR = 2 + 2 * NSLOT + 10 + 1 + (SPARSE ? 2 : 0) + 1;
    // block-sparse: the item's two mask rows as bitmasks (one bit per key
    // block), read from global memory once when the CTA starts
    static constexpr int SMEM_MASK = SPARSE ? (8 + 2 * kSparseMaskWords) * 4 : 0;
    static constexpr int SMEM_BYTES =
        1024 /*align slack*/ + SMEM_Q + SMEM_KV + SMEM_STAGE + NBAR * 8 + 16 + SMEM_MASK;
    static_assert(SMEM_BYTES <= 232448, "dynamic shared memory above the 227 KB a block may use");
    // TMEM columns: S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D, 256+2D)
    // and, at D = 64, P0 [384,448) P1 [448,512): P (fp16 or bf16 pairs) gets
    // columns of its own instead of overwriting S_t (SPLITP).
    static constexpr uint32_t TM_S = 0;
    static constexpr uint32_t TM_O = 256;
    static constexpr bool SPLITP = (D == 64);
    static constexpr uint32_t TM_P = 256 + 2 * D;
    static constexpr uint32_t TM_COLS = 512;
    static constexpr int THREADS = 384;  // softmax WG0, WG1, WG2 = {MMA, TMA, gate/MMA 1, copy}
    // dense SPLITP: both tiles' issuers release every shared ring entry
    static constexpr uint32_t KVE_COUNT = (SPLITP && !SPARSE) ? 2u : 1u;
};

constexpr int kWarpMma = 8;   // the MMA issuer (tile 0's at d = 64); allocates TMEM
constexpr int kWarpLoad = 9;
// d = 128: the gate warp folds "K/V tiles landed" into the p_full barriers,
// so the MMA thread waits on two barriers per key block instead of four.
// d = 64: tile 1's MMA issuer.
constexpr int kWarpGate = 10;
// The training forward's copy warp writes the fp16 copy of the item's Q
// tiles (for the backward) while the tiles sit in shared memory anyway.
constexpr int kWarpCopy = 11;

// Row-max and exp threshold for the lazy rescale: the reference max is only
// moved when the new block maximum exceeds it by more than 2^8 (in log2
// units), so unnormalised P values stay below 256.
constexpr float kRescaleThreshold = 8.0f;

// The key blocks an item's two query tiles multiply.  Tile t takes the
// blocks below n[t] (the causal diagonal or the ragged end), and, with a block
// mask (SPARSE), only those whose mask byte is set: count[t] blocks, the
// highest of them last[t].  Blocks are taken in increasing order, so only a
// tile's last block can need the element mask (only block n[t] - 1 reaches
// past the diagonal or the ragged end).
//   Dense: the tiles share K_j, V_j; every role walks j = 0 .. n[1] - 1, block
//   j in the item's ring entries 2j (K) and 2j + 1 (V), and tile 0 just stops
//   one block early on the diagonal.
//   SPARSE: each tile streams the K and V of its own blocks (the two mask
//   rows differ, and a shared walk would idle one tile on every block only
//   the other has).  The tiles advance by step k, the k-th block of each; the
//   ring holds K_0(0), K_1(0), then per step, tile by tile, V_t(k) and
//   K_t(k+1) of the tiles that still have blocks.  That order depends only on
//   the counts, so the issuers, the gate and the softmax run counted loops;
//   only the producer needs the block indices, which it takes from the rows'
//   bitmasks in shared memory (BlockCursor).
template <bool SPARSE>
struct TileBlocks {
    int n[2];
    int count[2];
    int last[2];  // -1 for a tile with no block
};

// The set bits of a tile's bitmask in increasing order (bit u of word u / 32:
// block u is selected and below n[t]); `base` is the bitmask's shared-memory
// address (32-bit state throughout: the producer that walks it runs on few
// registers).
struct BlockCursor {
    uint32_t base;
    int wd, nw;
    uint32_t cur;
    __device__ __forceinline__ BlockCursor(uint32_t b, int n)
        : base(b), wd(0), nw((n + 31) >> 5), cur(nw > 0 ? ld_shared_u32(b) : 0u) {}
    __device__ __forceinline__ int next() {  // the next block, or -1
        while (cur == 0u) {
            if (++wd >= nw) return -1;
            cur = ld_shared_u32(base + 4u * wd);
        }
        const int u = wd * 32 + __ffs(static_cast<int>(cur)) - 1;
        cur &= cur - 1u;
        return u;
    }
};

// Block-sparse shared memory beside the ring: eight words of per-warp partial
// counts (build_mask_bits), then each tile's bitmask.
constexpr int kSparseMaskHead = 8;

// One work item: (batch, head, 256-query block).  Dense: longest blocks
// first over the whole launch, the heads of one KV group adjacent.  SPARSE:
// the items of one (batch, KV head) adjacent (longest first within it), so
// that the CTAs running at one time read the scattered K/V blocks of one or
// two KV heads.
// SPARSE: `mk` is the CTA's shared-memory copy of the item's mask rows
// (build_mask_bits; a block-sparse CTA runs exactly one item), or null while
// it is being built.
template <bool SPARSE>
struct Item {
    int b, h, hk, row0, qb;
    TileBlocks<SPARSE> blk;
    __device__ __forceinline__ Item(int w, const FwdArgs& a, const uint32_t* mk) {
        if constexpr (SPARSE) {
            const int per_kv = a.n_qblk * a.g;
            const int bk = w / per_kv, r = w % per_kv;
            b = bk / a.Hkv;
            hk = bk % a.Hkv;
            qb = a.n_qblk - 1 - r / a.g;
            h = hk * a.g + r % a.g;
        } else {
            const int per = a.B * a.Hq;
            qb = a.n_qblk - 1 - w / per;
            const int bh = w % per;
            b = bh / a.Hq;
            h = bh % a.Hq;
            hk = h / a.g;
        }
        row0 = qb * 2 * kBM;
        const int nkv_all = (a.N + kBN - 1) / kBN;
        blk.n[0] = a.causal ? min(row0 / kBN + 1, nkv_all) : nkv_all;
        blk.n[1] = a.causal ? min((row0 + kBM) / kBN + 1, nkv_all) : nkv_all;
        for (int t = 0; t < 2; ++t) {
            blk.count[t] = blk.n[t];
            blk.last[t] = blk.n[t] - 1;
        }
        if (SPARSE && mk != nullptr)
            for (int t = 0; t < 2; ++t) {
                // warps t, t + 2, t + 4, t + 6 built tile t: (count << 16) | (last + 1)
                int c = 0, l1 = 0;
                for (int i = t; i < 8; i += 2) {
                    const uint32_t p = mk[i];
                    c += static_cast<int>(p >> 16);
                    l1 = max(l1, static_cast<int>(p & 0xffffu));
                }
                blk.count[t] = c;
                blk.last[t] = l1 - 1;
            }
    }
    // tile t's row of the global block mask (null past the last query block)
    __device__ __forceinline__ const uint8_t* mask_row(const FwdArgs& a, int t) const {
        const int nkv_all = (a.N + kBN - 1) / kBN;
        if (2 * qb + t >= nkv_all) return nullptr;
        return a.block_mask + (static_cast<size_t>(h) * nkv_all + 2 * qb + t) * nkv_all;
    }
    // SPARSE: tile t's bitmask in the shared-memory copy at address mk
    __device__ __forceinline__ BlockCursor cursor(uint32_t mk, int t) const {
        return BlockCursor(mk + 4u * (kSparseMaskHead + t * kSparseMaskWords), blk.n[t]);
    }
};

// Block-sparse: warps 0-7 turn the item's two mask rows into bitmasks (warp
// w takes tile w & 1 and every fourth word from w >> 1): 32 coalesced byte
// loads and a ballot per word, bits at or past the tile's limit n[t] left
// clear (a row past the last query block has none).  Each warp also leaves
// its words' block count and highest block + 1 in its head word.
template <bool SPARSE>
__device__ __forceinline__ void build_mask_bits(const Item<SPARSE>& I, const FwdArgs& a,
                                                uint32_t* mk, int warp, int lane) {
    const int t = warp & 1;
    const uint8_t* row = I.mask_row(a, t);
    const int n = I.blk.n[t];
    int c = 0, l1 = 0;
    for (int wd = warp >> 1; wd * 32 < n; wd += 4) {
        const int u = wd * 32 + lane;
        const bool on = row != nullptr && u < n && row[u] != 0;
        const uint32_t word = __ballot_sync(0xffffffffu, on);
        if (lane == 0) mk[kSparseMaskHead + t * kSparseMaskWords + wd] = word;
        c += __popc(word);
        if (word != 0u) l1 = wd * 32 + 32 - __clz(static_cast<int>(word));
    }
    if (lane == 0) mk[warp] = (static_cast<uint32_t>(c) << 16) | static_cast<uint32_t>(l1);
}

// F16: P is rounded to fp16 (not bf16) and multiplies the fp16 copy of V,
// scaled by 2^v (the training forward, whose O feeds the backward's D).
// SPARSE: the tiles multiply only the key blocks a.block_mask selects.
template <int D, bool F16, bool SPARSE>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const FwdArgs a) {
    using C = FwdCfg<D, SPARSE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sKV = sQ + C::SMEM_Q;
    const uint32_t sStage = sKV + C::SMEM_KV;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::SMEM_Q + C::SMEM_KV + C::SMEM_STAGE);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
    uint32_t* mbits = tmem_slot + 4;  // block-sparse bitmasks (SMEM_MASK bytes)
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t BAR_Q = bar0;        // the item's Q tiles landed
    const uint32_t BAR_QE = bar0 + 8u;  // the item's Q tiles no longer read
    auto BAR_KVF = [&](int s) { return bar0 + 8u * (2 + s); };
    auto BAR_KVE = [&](int s) { return bar0 + 8u * (2 + C::NSLOT + s); };
    auto BAR_SF = [&](int t) { return bar0 + 8u * (2 + 2 * C::NSLOT + t); };
    auto BAR_PF = [&](int t) { return bar0 + 8u * (4 + 2 * C::NSLOT + t); };
    auto BAR_OF = [&](int t) { return bar0 + 8u * (6 + 2 * C::NSLOT + t); };
    // SPLITP only: S_t is in the softmax's registers / PV_t has finished
    auto BAR_SE = [&](int t) { return bar0 + 8u * (8 + 2 * C::NSLOT + t); };
    auto BAR_PVD = [&](int t) { return bar0 + 8u * (10 + 2 * C::NSLOT + t); };
    const uint32_t BAR_DONE = bar0 + 8u * (12 + 2 * C::NSLOT);
    auto BAR_EPI = [&](int t) { return bar0 + 8u * (13 + 2 * C::NSLOT + t); };
    const uint32_t BAR_G1 = bar0 + 8u * (C::NBAR - 1);

    const int warp = warp_id();
    const int lane = lane_id();
    const int n_items = a.n_qblk * a.B * a.Hq;
    const bool copy_q = F16 && a.q16 != nullptr;
    constexpr int kIssuers = C::SPLITP ? 2 : 1;

    // ---- set-up
    if (warp == 0 && lane == 0) {
        mbar_init(BAR_Q, 1);
        mbar_init(BAR_QE, kIssuers + (copy_q ? 1 : 0));
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(BAR_KVF(s), 1);
            mbar_init(BAR_KVE(s), C::KVE_COUNT);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(BAR_SF(t), 1);
            // the tile's softmax threads, and at d = 128 the gate
            mbar_init(BAR_PF(t), C::SPLITP ? 128 : 128 + 1);
            mbar_init(BAR_OF(t), 1);
            mbar_init(BAR_SE(t), 4);  // one arrival per softmax warp of the tile
            mbar_init(BAR_PVD(t), 1);
            if (SPARSE) mbar_init(BAR_EPI(t), 4);  // likewise
        }
        mbar_init(BAR_DONE, kIssuers);
        mbar_init(BAR_G1, 1);
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
        tmem_relinquish();
    }
    if constexpr (SPARSE)
        if (warp < 8) build_mask_bits(Item<SPARSE>(blockIdx.x, a, nullptr), a, mbits, warp, lane);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    // Registers: the launch gives every thread 168 (384 x 168 = 64,512); each
    // role below starts by moving its warpgroup's share: the softmax
    // warpgroups, which hold a 128-column row each, take 208 and the issue /
    // copy warpgroup keeps 88 (2 x 128 x 208 + 128 x 88 = 64,512, the whole
    // launch pool).

    constexpr uint32_t IDESC_QK = idesc_bf16(kBM, kBN, false, false);
    constexpr uint32_t IDESC_PV = idesc_16(kBM, D, false, true, F16);
    constexpr uint32_t HI = sdesc_hi(1024);
    // S_t = Q_t K^T from the K tile in ring slot `slot`
    auto issue_qk = [&](uint32_t leader, int t, int slot) {
        const uint32_t dS = tbase + C::TM_S + t * kBN;
        const uint32_t a_lo = sdesc_lo(sQ + t * C::TILE, 16);
        const uint32_t b_lo = sdesc_lo(sKV + slot * C::TILE, 16);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
            mma_bf16_ss_w(leader, dS, sdesc_at(a_lo, HI, off), sdesc_at(b_lo, HI, off), IDESC_QK,
                          ks > 0);
        }
    };
    // O_t (+)= P_t V from the V tile in ring slot `slot`
    auto issue_pv = [&](uint32_t leader, int t, int slot, bool acc) {
        const uint32_t dO = tbase + C::TM_O + t * D;
        const uint32_t aP = tbase + (C::SPLITP ? C::TM_P + t * (kBN / 2) : C::TM_S + t * kBN);
        const uint32_t b_lo = sdesc_lo(sKV + slot * C::TILE, C::CHUNK);
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks)
            mma_bf16_ts_w(leader, dO, aP + ks * 8, sdesc_at(b_lo, HI, ks * 2048), IDESC_PV,
                          (acc || ks > 0) ? 1u : 0u);
    };

    if (warp == kWarpLoad) {
        // ================= TMA producer =================
        setmaxnreg_dec<88>();
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            const uint64_t pol_kv = l2_policy_evict_last();
            const uint64_t pol_q = l2_policy_evict_first();
            int last_idx[C::NSLOT];
            for (int s = 0; s < C::NSLOT; ++s) last_idx[s] = -1;
            bool ok = true;
            int e = 0;   // ring entry, running over the items
            int it = 0;  // items started
            for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++it) {
                const Item<SPARSE> I(w, a, mbits);
                // the previous item's score products and q copy are done with Q
                if (it > 0 && !(ok = mbar_wait(BAR_QE, (it - 1) & 1, a.watch, 22))) break;
                mbar_arrive_expect_tx(BAR_Q, 2 * C::TILE);
                for (int t = 0; t < 2; ++t)
                    for (int c = 0; c < C::NCH; ++c)
                        tma_load_4d_hint(sQ + t * C::TILE + c * C::CHUNK, &tmQ, BAR_Q, c * 64, I.h,
                                         I.row0 + t * kBM, I.b, pol_q);
                auto load = [&](const CUtensorMap* tm, int u) {
                    const int slot = e % C::NSLOT;
                    const uint32_t ph = (e / C::NSLOT) & 1;
                    if (!(ok = mbar_wait(BAR_KVE(slot), ph ^ 1u, a.watch, 1))) return;
                    mbar_arrive_expect_tx(BAR_KVF(slot), C::TILE);
                    for (int c = 0; c < C::NCH; ++c)
                        tma_load_4d_hint(sKV + slot * C::TILE + c * C::CHUNK, tm, BAR_KVF(slot),
                                         c * 64, I.hk, u * kBN, I.b, pol_kv);
                    last_idx[slot] = e++;
                };
                if constexpr (SPARSE) {
                    BlockCursor cur[2] = {I.cursor(smem_u32(mbits), 0), I.cursor(smem_u32(mbits), 1)};
                    int u[2] = {cur[0].next(), cur[1].next()};
                    for (int t = 0; t < 2 && ok; ++t)
                        if (u[t] >= 0) load(&tmK, u[t]);
                    while (ok && (u[0] >= 0 || u[1] >= 0)) {
                        for (int t = 0; t < 2 && ok; ++t) {
                            if (u[t] < 0) continue;
                            load(&tmV, u[t]);
                            const int un = cur[t].next();
                            if (ok && un >= 0) load(&tmK, un);
                            u[t] = un;
                        }
                    }
                } else {
                    for (int u = 0; u < I.blk.n[1] && ok; ++u) {
                        load(&tmK, u);
                        if (ok) load(&tmV, u);
                    }
                }
            }
            // Never leave the CTA with copies in flight: wait (bounded) for the
            // last load issued into every slot, and for the last Q.
            if (it > 0) mbar_drain(BAR_Q, (it - 1) & 1, a.watch, 2);
            for (int s = 0; s < C::NSLOT; ++s)
                if (last_idx[s] >= 0)
                    mbar_drain(BAR_KVF(s), (last_idx[s] / C::NSLOT) & 1, a.watch, 2);
        }
        __syncwarp();
    } else if ((warp == kWarpMma || warp == kWarpGate) && C::SPLITP) {
        // ================= d = 64: tile t's MMA issuer (warp-wide; the leader issues) ======
        // Per block k of the tile: S_t(k+1) once the softmax holds S_t(k) in
        // registers (s_empty) and K(k+1) has landed, then PV_t(k) on p_full(t)
        // once V(k) has landed, committed to pv_done(t): the softmax writes
        // P_t and rescales O_t only after it.  Each ring entry is released
        // right after the product that reads it (dense entries by both
        // issuers).
        setmaxnreg_dec<88>();
        const int t = (warp == kWarpMma) ? 0 : 1;
        const uint32_t leader = elect_one();
        bool ok = true;
        int e = 0, it = 0, nqk = 0, npv = 0;
        auto qk = [&](int ek) {  // S_t from ring entry ek
            if (nqk > 0 && !(ok = mbar_wait_warp(BAR_SE(t), (nqk - 1) & 1, a.watch, 17 + t))) return;
            if (!(ok = mbar_wait_warp(BAR_KVF(ek % C::NSLOT), (ek / C::NSLOT) & 1, a.watch, 19)))
                return;
            tc_fence_after();
            issue_qk(leader, t, ek % C::NSLOT);
            mma_commit_w(leader, BAR_SF(t));
            mma_commit_w(leader, BAR_KVE(ek % C::NSLOT));
            ++nqk;
        };
        auto pv = [&](int ev, bool acc, bool last) {  // O_t (+)= P_t V from ring entry ev
            if (!(ok = mbar_wait_warp(BAR_KVF(ev % C::NSLOT), (ev / C::NSLOT) & 1, a.watch, 23 + t)))
                return;
            if (!(ok = mbar_wait_warp(BAR_PF(t), npv & 1, a.watch, 6 + 2 * t))) return;
            tc_fence_after();
            issue_pv(leader, t, ev % C::NSLOT, acc);
            mma_commit_w(leader, BAR_PVD(t));
            mma_commit_w(leader, BAR_KVE(ev % C::NSLOT));
            if (last) mma_commit_w(leader, BAR_OF(t));
            ++npv;
        };
        for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++it) {
            const Item<SPARSE> I(w, a, mbits);
            if (!(ok = mbar_wait_warp(BAR_Q, it & 1, a.watch, 3))) break;
            if constexpr (SPARSE) {
                // count both tiles' streams to find this tile's ring entries
                const int c0 = I.blk.count[0], c1 = I.blk.count[1];
                const int ek0 = (t == 0 || c0 == 0) ? e : e + 1;
                e += (c0 > 0) + (c1 > 0);
                if (I.blk.count[t] > 0) qk(ek0);
                for (int k = 0; k < max(c0, c1) && ok; ++k)
                    for (int tt = 0; tt < 2 && ok; ++tt) {
                        const int c = tt == 0 ? c0 : c1;
                        if (k >= c) continue;
                        const int ev = e++;
                        const bool more = k + 1 < c;
                        const int ek = more ? e++ : -1;
                        if (tt == t) {
                            if (more) qk(ek);
                            if (ok) pv(ev, k > 0, !more);
                        }
                    }
            } else {
                const int n = I.blk.n[t], n1 = I.blk.n[1];
                for (int k = 0; k <= n && ok; ++k) {
                    if (k < n) qk(e + 2 * k);
                    if (ok && k > 0) pv(e + 2 * (k - 1) + 1, k > 1, k == n);
                }
                // tile 0 stops short of tile 1 on the causal diagonal: release
                // the entries of the blocks past its limit, each once its
                // slot's previous use has been released (so the arrival
                // lands in the right phase)
                if (t == 0)
                    for (int ee = e + 2 * n; ee < e + 2 * n1 && ok; ++ee) {
                        const int s = ee % C::NSLOT, ph = ee / C::NSLOT;
                        if (ph > 0) ok = mbar_wait_warp(BAR_KVE(s), (ph - 1) & 1, a.watch, 25);
                        if (ok && leader) mbar_arrive(BAR_KVE(s));
                        __syncwarp();
                    }
                e += 2 * n1;
            }
            // the item's score products read Q; q_empty lets the producer reload it
            mma_commit_w(leader, BAR_QE);
        }
        // all issued MMAs have finished before TMEM can be released
        mma_commit_w(leader, BAR_DONE);
        if (t == 0) mbar_drain(BAR_DONE, 0, a.watch, 9);
        __syncwarp();
    } else if (warp == kWarpGate) {
        // ================= d = 128 gate: loads -> p_full =================
        // For block k of tile t it waits for V(k) and K(k+1), then adds one
        // arrival to p_full(t), but only once that barrier's previous phase
        // has completed, so the arrival can never be counted in the wrong
        // phase.  It is the only thread that waits on the ring's kv_full
        // barriers, every entry in ring order: an item's first K entries too,
        // which it passes on to the MMA thread on g1.  A slot's parity wait
        // answers right only at the awaited phase or the one after it; seeing
        // every phase of a slot, and letting no entry be used before it has
        // seen it land, keeps every wait there.
        setmaxnreg_dec<88>();
        if (lane == 0) {
            bool ok = true;
            int e = 0;
            int cnt[2] = {0, 0};  // blocks each tile has multiplied so far
            auto arrive = [&](int t) {
                if (ok && cnt[t] > 0) ok = mbar_wait(BAR_PF(t), (cnt[t] - 1) & 1, a.watch, 7);
                if (ok) mbar_arrive(BAR_PF(t));
                ++cnt[t];
            };
            auto landed = [&](int ee) {
                if (ok) ok = mbar_wait(BAR_KVF(ee % C::NSLOT), (ee / C::NSLOT) & 1, a.watch, 5);
            };
            for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
                const Item<SPARSE> I(w, a, mbits);
                if constexpr (SPARSE) {
                    const int c0 = I.blk.count[0], c1 = I.blk.count[1];
                    if (c0 > 0) landed(e++);  // the K_t(0)
                    if (c1 > 0) landed(e++);
                    if (ok && (c0 > 0 || c1 > 0)) mbar_arrive(BAR_G1);
                    for (int k = 0; k < max(c0, c1) && ok; ++k)
                        for (int t = 0; t < 2 && ok; ++t) {
                            const int c = t == 0 ? c0 : c1;
                            if (k >= c) continue;
                            landed(e++);
                            if (k + 1 < c) landed(e++);
                            arrive(t);
                        }
                } else {
                    const int n1 = I.blk.n[1];
                    landed(e);  // K(0)
                    if (ok) mbar_arrive(BAR_G1);
                    for (int u = 0; u < n1 && ok; ++u) {
                        landed(e + 2 * u + 1);
                        if (u + 1 < n1) landed(e + 2 * u + 2);
                        for (int t = 0; t < 2; ++t)
                            if (u < I.blk.n[t]) arrive(t);
                    }
                    e += 2 * n1;
                }
            }
        }
        __syncwarp();
    } else if (warp == kWarpCopy) {
        // ================= copy: Q tiles -> fp16(q * 2^s) =================
        // Only the training forward (F16 with q16 set); then q_empty also
        // waits for this warp.
        setmaxnreg_dec<88>();
        if (copy_q) {
            const float mul = pow2f(ld_once(&a.f16s->q));
            const size_t row_el = static_cast<size_t>(a.Hq) * D;  // elements per token
            int it = 0;
            for (int w = blockIdx.x; w < n_items; w += gridDim.x, ++it) {
                const Item<SPARSE> I(w, a, mbits);
                if (!mbar_wait_warp(BAR_Q, it & 1, a.watch, 15)) break;
                for (int t = 0; t < 2; ++t)
                    warp_tile_to_f16<D>(
                        sQ + t * C::TILE,
                        a.q16 + (static_cast<size_t>(I.b) * a.N + I.row0 + t * kBM) * row_el + I.h * D,
                        row_el, a.N - (I.row0 + t * kBM), mul, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR_QE);
            }
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ================= d = 128 MMA issuer (the whole warp; the leader lane issues) ======
        setmaxnreg_dec<88>();
        const uint32_t leader = elect_one();
        bool ok = true;
        int e = 0, it = 0, ng1 = 0;
        int cnt[2] = {0, 0};  // p_full phases waited, per tile
        for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++it) {
            const Item<SPARSE> I(w, a, mbits);
            if (!(ok = mbar_wait_warp(BAR_Q, it & 1, a.watch, 3))) break;
            if constexpr (SPARSE) {
                // Per step k, tile by tile: PV_t(k) on p_full(t) (V_t(k) and
                // K_t(k+1) landed, the gate), then S_t(k+1).  Every ring entry is
                // released right after the product that reads it.
                const int c0 = I.blk.count[0], c1 = I.blk.count[1];
                // the gate has seen the item's first K entries land (g1)
                if ((c0 > 0 || c1 > 0) && !(ok = mbar_wait_warp(BAR_G1, ng1++ & 1, a.watch, 4)))
                    break;
                for (int t = 0; t < 2 && ok; ++t) {
                    if ((t == 0 ? c0 : c1) == 0) continue;
                    const int ek = e++;
                    tc_fence_after();
                    issue_qk(leader, t, ek % C::NSLOT);
                    mma_commit_w(leader, BAR_SF(t));
                    mma_commit_w(leader, BAR_KVE(ek % C::NSLOT));
                }
                for (int k = 0; k < max(c0, c1) && ok; ++k)
                    for (int t = 0; t < 2 && ok; ++t) {
                        const int c = t == 0 ? c0 : c1;
                        if (k >= c) continue;
                        const int ev = e++;
                        const bool more = k + 1 < c;
                        const int ek = more ? e++ : -1;
                        if (!(ok = mbar_wait_warp(BAR_PF(t), cnt[t] & 1, a.watch, 6 + 2 * t))) break;
                        tc_fence_after();
                        issue_pv(leader, t, ev % C::NSLOT, k > 0);
                        mma_commit_w(leader, BAR_KVE(ev % C::NSLOT));
                        ++cnt[t];
                        if (!more) mma_commit_w(leader, BAR_OF(t));
                        if (more) {
                            issue_qk(leader, t, ek % C::NSLOT);
                            mma_commit_w(leader, BAR_SF(t));
                            mma_commit_w(leader, BAR_KVE(ek % C::NSLOT));
                        }
                    }
            } else {
                // Per key block u (item entries 2u, 2u + 1): PV0(u) and S0(u + 1)
                // while tile 0 has them, PV1(u), S1(u + 1).  p_full(t) for u also
                // means V(u) and K(u + 1) have landed (the gate); S_t(u + 1)
                // follows PV_t(u), which read P_t over S_t.  The item's first
                // S_t follows the previous item's last PV_t the same way.
                const int n0 = I.blk.n[0], n1 = I.blk.n[1];
                // K(0) has landed: the gate has seen it (g1)
                if (!(ok = mbar_wait_warp(BAR_G1, ng1++ & 1, a.watch, 4))) break;
                tc_fence_after();
                for (int t = 0; t < 2; ++t) {
                    issue_qk(leader, t, e % C::NSLOT);
                    mma_commit_w(leader, BAR_SF(t));
                }
                mma_commit_w(leader, BAR_KVE(e % C::NSLOT));
                for (int u = 0; u < n1 && ok; ++u) {
                    const int vslot = (e + 2 * u + 1) % C::NSLOT;
                    const int kslot = (e + 2 * u + 2) % C::NSLOT;
                    if (u < n0) {
                        if (!(ok = mbar_wait_warp(BAR_PF(0), cnt[0] & 1, a.watch, 6))) break;
                        tc_fence_after();
                        issue_pv(leader, 0, vslot, u > 0);
                        ++cnt[0];
                        if (u == n0 - 1) mma_commit_w(leader, BAR_OF(0));
                        if (u + 1 < n0) {
                            issue_qk(leader, 0, kslot);
                            mma_commit_w(leader, BAR_SF(0));
                        }
                    }
                    if (!(ok = mbar_wait_warp(BAR_PF(1), cnt[1] & 1, a.watch, 8))) break;
                    tc_fence_after();
                    issue_pv(leader, 1, vslot, u > 0);
                    ++cnt[1];
                    mma_commit_w(leader, BAR_KVE(vslot));
                    if (u == n1 - 1) mma_commit_w(leader, BAR_OF(1));
                    if (u + 1 < n1) {
                        issue_qk(leader, 1, kslot);
                        mma_commit_w(leader, BAR_SF(1));
                        mma_commit_w(leader, BAR_KVE(kslot));
                    }
                }
                e += 2 * n1;
            }
            // the item's score products read Q; q_empty lets the producer reload it
            mma_commit_w(leader, BAR_QE);
        }
        // all issued MMAs have finished before TMEM can be released
        mma_commit_w(leader, BAR_DONE);
        mbar_drain(BAR_DONE, 0, a.watch, 9);
        __syncwarp();
    } else if (warp < 8) {
        // ================= softmax warpgroups (warps 0-3: tile 0, 4-7: tile 1)
        setmaxnreg_inc<208>();
        const int t = warp >> 2;               // query tile of this warpgroup
        const int wq = warp & 3;               // its warp owns TMEM lanes 32*wq..32*wq+31
        const int r = wq * 32 + lane;          // row within the tile
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tbase + C::TM_S + t * kBN + lane_off;
        const uint32_t tO = tbase + C::TM_O + t * D + lane_off;
        // where P goes: its own columns (SPLITP), else over S_t
        const uint32_t tP = C::SPLITP ? tbase + C::TM_P + t * (kBN / 2) + lane_off : tS;
        const float sl2 = a.scale_log2;
        int eq = 0, ek = 0, ev = 0, edo = 0;  // fp16 path: O carries 2^ev
        if (F16) ld_once_v4(&a.f16s->q, eq, ek, ev, edo);
        bool ok = true;
        int nsf = 0, npf = 0, nof = 0;  // phases of s_full, p_full, o_final so far
        for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
            const Item<SPARSE> I(w, a, mbits);
            const int grow = I.row0 + t * kBM + r;  // query index
            // last key index this row may see
            const int lim = a.causal ? min(grow, a.N - 1) : a.N - 1;
            float m_ref = -INFINITY;  // reference max of the exponentials (log2 units)
            float l = 0.f;            // running sum, relative to m_ref
            // per-item values, read once here: inside the loop every barrier
            // wait would force a fresh read of the item from local memory
            const int nblk = I.blk.count[t];
            // only the tile's last block can reach past the diagonal or the
            // ragged end
            const int klast = I.blk.last[t] * kBN;
            const bool mask_last = klast + kBN - 1 > lim;
            for (int j = 0; j < nblk; ++j) {  // the tile's j-th block
                if (!(ok = mbar_wait_warp(BAR_SF(t), nsf & 1, a.watch, 10 + t))) break;
                ++nsf;
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
                if (mask_last && j == nblk - 1) {  // diagonal block or ragged tail: mask
#pragma unroll
                    for (int c = 0; c < kBN; ++c) x[c] = (klast + c > lim) ? -INFINITY : x[c];
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
                // SPLITP: PV_t of the previous block still reads P_t and writes
                // O_t (the item's first block: the epilogue already waited for
                // the previous item's last one)
                if (C::SPLITP && j > 0) {
                    if (!(ok = mbar_wait_warp(BAR_PVD(t), (npf - 1) & 1, a.watch, 20 + t))) break;
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
                        f2_split(fma2(f2(x[half * 64 + c], x[half * 64 + c + 1]), sl2x2, negx2), e0,
                                 e1);
                        const float p0 = ex2(e0), p1 = ex2(e1);
                        ls2[(c >> 1) & 3] = add2(ls2[(c >> 1) & 3], f2(p0, p1));
                        pk[c >> 1] = pack_op<F16>(p0, p1);
                    }
                    tmem_st32(tP + half * 32, pk);
                }
                {
                    const uint64_t sum2 = add2(add2(ls2[0], ls2[1]), add2(ls2[2], ls2[3]));
                    float a0, a1;
                    f2_split(sum2, a0, a1);
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
                            float v0, v1;
                            f2_split(mul2(f2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), ax2),
                                     v0, v1);
                            o[i] = __float_as_uint(v0);
                            o[i + 1] = __float_as_uint(v1);
                        }
                        tmem_st32(tO + cb, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(BAR_PF(t));
                ++npf;
            }
            if (!ok) break;
            if constexpr (SPARSE) {
                // ---- block-sparse epilogue: O / l -> bf16 rows in the tile's
                // own Q buffer (the 128-byte swizzle of the TMA maps), then one
                // TMA store, which also drops the rows past N.  One item per
                // CTA: Q_t is idle once o_final(t) says the tile's last
                // product, and so its last score product, is done; a tile with
                // no key block (O = 0, lse = -inf) waits for its Q load, the
                // buffer's only other writer, instead.
                const bool any = nblk > 0;
                if (!(ok = any ? mbar_wait_warp(BAR_OF(t), nof & 1, a.watch, 12 + t)
                               : mbar_wait_warp(BAR_Q, 0, a.watch, 26)))
                    break;
                nof += any ? 1 : 0;
                tc_fence_after();
                const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
                const uint32_t stage = sQ + t * C::TILE;
#pragma unroll
                for (int ch = 0; ch < C::NCH; ++ch) {  // 64-column chunks: one TMEM wait each
                    uint32_t o[64];
                    if (any) {
                        tmem_ld32(tO + ch * 64, o);
                        tmem_ld32(tO + ch * 64 + 32, o + 32);
                        tmem_wait_ld();
                        reg_fence<64>(o);
                    } else {
#pragma unroll
                        for (int i = 0; i < 64; ++i) o[i] = 0u;
                    }
                    const uint32_t rowbase = stage + ch * C::CHUNK + r * 128;
#pragma unroll
                    for (int p8 = 0; p8 < 8; ++p8) {  // 16-byte pieces of the row's 128 bytes
                        uint32_t wv[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            wv[i] = pack_bf16(__uint_as_float(o[8 * p8 + 2 * i]) * inv_l,
                                              __uint_as_float(o[8 * p8 + 2 * i + 1]) * inv_l);
                        st_shared_v4(rowbase + ((p8 ^ (r & 7)) << 4), wv[0], wv[1], wv[2], wv[3]);
                    }
                }
                if (grow < a.N)
                    a.lse[(static_cast<size_t>(I.b) * a.Hq + I.h) * a.N + grow] =
                        (m_ref + log2f(l)) * 0.6931471805599453f;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR_EPI(t));
                if (wq == 0) {  // the tile's first warp waits for all four, one lane stores
                    if (!(ok = mbar_wait_warp(BAR_EPI(t), 0, a.watch, 27))) break;
                    if (lane == 0) {
                        for (int c = 0; c < C::NCH; ++c)
                            tma_store_4d(&tmO, stage + c * C::CHUNK, c * 64, I.h, I.row0 + t * kBM,
                                         I.b);
                        tma_store_commit();
                        tma_store_wait_read_all();
                    }
                    __syncwarp();
                }
                continue;
            }
            // ---- epilogue: O / l -> bf16, each row from its thread straight to
            // global memory.  The next item's first P V product overwrites
            // O_t only after this tile's next p_full arrival, which follows the
            // loads below.
            const bool any = nblk > 0;
            if (any) {
                if (!(ok = mbar_wait_warp(BAR_OF(t), nof & 1, a.watch, 12 + t))) break;
                ++nof;
                tc_fence_after();
            }
            // O was accumulated against V * 2^v on the fp16 path
            const float inv_l = (l > 0.f) ? pow2f(-ev) / l : 0.f;
            // Rows reach global memory through this warp's transpose buffer: a
            // thread writes its row's 64-byte piece of a 32-column chunk, then
            // each store instruction writes whole pieces of eight rows (the
            // 16-byte quarters of row R at R * 64 + 16 * (q ^ ((R >> 1) & 3)),
            // which keeps both sides free of bank conflicts).
            const uint32_t stg = sStage + warp * 2048;
            const int wrow0 = I.row0 + t * kBM + wq * 32;  // the warp's first query
            auto store_chunk = [&](uint16_t* dstT, const uint32_t (&wv)[16], int cb) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    st_shared_v4(stg + lane * 64 + ((q4 ^ ((lane >> 1) & 3)) << 4), wv[4 * q4],
                                 wv[4 * q4 + 1], wv[4 * q4 + 2], wv[4 * q4 + 3]);
                __syncwarp();
#pragma unroll
                for (int s8 = 0; s8 < 4; ++s8) {
                    const int R = 8 * s8 + (lane >> 2), q4 = lane & 3;
                    uint32_t v[4];
                    ld_shared_v4(stg + R * 64 + ((q4 ^ ((R >> 1) & 3)) << 4), v);
                    if (wrow0 + R < a.N)
                        *reinterpret_cast<uint4*>(
                            dstT + ((static_cast<size_t>(I.b) * a.N + wrow0 + R) * a.Hq + I.h) * D +
                            cb + q4 * 8) = make_uint4(v[0], v[1], v[2], v[3]);
                }
                __syncwarp();
            };
#pragma unroll
            for (int cb = 0; cb < D; cb += 32) {
                uint32_t o[32];
                if (any) {
                    tmem_ld32(tO + cb, o);
                    tmem_wait_ld();
                    reg_fence<32>(o);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                uint32_t wv[16], wl[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float f0 = __uint_as_float(o[2 * i]) * inv_l;
                    const float f1 = __uint_as_float(o[2 * i + 1]) * inv_l;
                    wv[i] = pack_bf16(f0, f1);
                    // rounding residual for the training forward's o_lo
                    wl[i] = pack_bf16(f0 - __uint_as_float(wv[i] << 16),
                                      f1 - __uint_as_float(wv[i] & 0xFFFF0000u));
                }
                store_chunk(a.o, wv, cb);
                if (a.o_lo != nullptr) store_chunk(a.o_lo, wl, cb);
            }
            if (grow < a.N)
                a.lse[(static_cast<size_t>(I.b) * a.Hq + I.h) * a.N + grow] =
                    (m_ref + log2f(l)) * 0.6931471805599453f;
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
    using C = FwdCfg<D, SPARSE>;
    auto kern = fa_fwd_kernel<D, F16, SPARSE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long items = static_cast<long long>(a.n_qblk) * a.B * a.Hq;
    if (items <= 0 || items > 0x7fffffffLL || a.num_ctas <= 0) return cudaErrorInvalidConfiguration;
    // Dense: persistent, one CTA per SM (shared memory and registers allow no
    // more), items dealt out round robin, longest query blocks first.
    // Block-sparse: one CTA per item, balanced by the hardware's block
    // scheduler (measured faster than the fixed deal on the synthetic masks,
    // whose items differ in length with the mask).
    const long long ctas = SPARSE ? items : (items < a.num_ctas ? items : a.num_ctas);
    const unsigned grid = static_cast<unsigned>(ctas);
    // the O map is read by the block-sparse epilogue only
    kern<<<grid, C::THREADS, C::SMEM_BYTES, st>>>(m.q, m.k, m.v, SPARSE ? m.o : m.q, a);
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
