// fa_fp8.cu -- FP8 (e4m3) attention forward for sm_103a, head dimension 128.
//
// What it computes: O = softmax(scale * Q K^T [+ causal]) V and lse, as
// fa_fwd, with Q, K, V and P entering the products as e4m3 values -- the
// low-precision forward the pages describe for FlashAttention-3: block
// quantisation (one scale per block instead of per tensor) and "incoherent
// processing", a random orthogonal rotation of Q and K that spreads outliers
// before they are quantised ("FlashAttention and the Kernel Era", the FP8
// paragraph; "FlashAttention 1, 2, and 3 Explained", section 4).
//
//   * Quantisation (three small kernels): every 128-row block of each head of
//     Q and of K gets its own scale amax / 448 (448 = the largest e4m3); with
//     rotation on, the rows are first multiplied by diag(s) H, H the 128-point
//     Walsh-Hadamard matrix (unnormalised, so H H^T = 128 I, folded into the
//     softmax scale) and s fixed random signs, which leaves Q K^T unchanged.
//     V gets one scale per head and is stored transposed (d rows x keys), the
//     K-major layout the P V product needs as its B operand.
//   * Forward: two 128-query tiles of one head per CTA (16 KB e4m3 tiles, all
//     512 TMEM columns: S0, S1, O0, O1), the products of one tile overlapping
//     the softmax of the other as in the bf16 forward.  S = Q8 K8^T and
//     O += P8 V8 are tcgen05.mma kind::f8f6f4 (K = 32 per instruction); S is
//     scaled by scale * log2 e * sq * sk_j in the softmax; P (at most 2^8
//     under the lazy rescale, inside e4m3's range) is rounded to e4m3 and
//     written back to TMEM as the A operand of P V; O is multiplied by sv / l
//     at the end.
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kF8Tile = 128 * 128;  // bytes of a 128 x 128 e4m3 tile
constexpr int kF8Slots = 8;         // K / V^T ring slots (four key blocks)
// softmax warps 0-7 (two tiles), MMA 8, TMA 9, gate 10, warp 11 idle (a whole
// issue warpgroup for setmaxnreg)
constexpr int kF8Threads = 384;
constexpr int kF8WarpMma = 8;
constexpr int kF8WarpLoad = 9;
constexpr int kF8WarpGate = 10;
// barriers: Q, K/V full[slots], empty[slots], s_full[2], p_full[2], o_final[2], done,
// q_empty
constexpr int kF8Bars = 1 + 2 * kF8Slots + 2 + 2 + 2 + 1 + 1 + 1;
constexpr int kF8Stage = 8 * 2048;  // the epilogue's per-warp transpose buffers
constexpr float kE4m3Max = 448.f;

// The fixed sign of column c in the rotation diag(s) H: the top bit of
// c * 2654435761 (mod 2^32) -- a multiplicative hash, the same on every call.
__device__ __forceinline__ float rot_sign(int c) {
    return ((static_cast<uint32_t>(c) * 2654435761u) >> 31) ? -1.f : 1.f;
}

// x[i] = element 32 * q + i of a 128-element row spread over the four lanes
// of a lane quad (q = lane & 3).  In place: y[k] = sum_c (-1)^popcount(k & c)
// x[c] (the Walsh-Hadamard transform in natural order): butterflies over
// element strides 1..16 inside the lane, 32 and 64 across the quad.  (A
// whole warp on one row, four elements a lane, needed five shuffle stages,
// and the shuffles set the pace of the quantisation.)
__device__ __forceinline__ void hadamard128_quad(float (&x)[32], int q) {
#pragma unroll
    for (int s = 1; s < 32; s <<= 1)
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if ((i & s) == 0) {
                const float a = x[i], b = x[i + s];
                x[i] = a + b;
                x[i + s] = a - b;
            }
#pragma unroll
    for (int s = 1; s < 4; s <<= 1)  // lane strides 1, 2: element strides 32, 64
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float y = __shfl_xor_sync(0xffffffffu, x[i], s);
            x[i] = (q & s) ? (y - x[i]) : (x[i] + y);
        }
}

// One 128-row block of one head of q or k, in one pass: each warp holds 16
// rows in registers, 8 at a time across its lane quads (lane 4r + q holds
// elements 32q..32q+31 of row r), all of a lane's 16-byte loads in flight at
// once, while the block's max |x| is reduced; then it writes the bytes.
__global__ void __launch_bounds__(256) fp8_rows_kernel(const uint16_t* __restrict__ x,
                                                       uint8_t* __restrict__ x8,
                                                       float* __restrict__ sx, int N, int H,
                                                       int nb, int rotate) {
    constexpr int PASSES = 2;  // 8 rows a warp per pass
    __shared__ float red[8];
    const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = lane & 3, rq = lane >> 2;
    float v[PASSES][32];
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int n = blk * 128 + warp * 16 + p * 8 + rq;
        uint4 u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) u[i] = make_uint4(0u, 0u, 0u, 0u);
        if (n < N) {
            const uint4* src = reinterpret_cast<const uint4*>(
                x + ((static_cast<size_t>(b) * N + n) * H + h) * 128 + 32 * q);
#pragma unroll
            for (int i = 0; i < 4; ++i) u[i] = src[i];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t w4[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[p][8 * i + 2 * j] = __uint_as_float(w4[j] << 16);
                v[p][8 * i + 2 * j + 1] = __uint_as_float(w4[j] & 0xffff0000u);
            }
        }
    }
    float m = 0.f;
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        if (rotate) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[p][i] *= rot_sign(32 * q + i);
            hadamard128_quad(v[p], q);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(v[p][i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
    const float inv = m > 0.f ? kE4m3Max / m : 1.f;
    if (threadIdx.x == 0)
        sx[(static_cast<size_t>(b) * H + h) * nb + blk] = m > 0.f ? m / kE4m3Max : 1.f;
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int n = blk * 128 + warp * 16 + p * 8 + rq;
        if (n < N) {
            uint32_t w8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                w8[i] = pack_e4m3x4(v[p][4 * i] * inv, v[p][4 * i + 1] * inv, v[p][4 * i + 2] * inv,
                                    v[p][4 * i + 3] * inv);
            uint4* dst = reinterpret_cast<uint4*>(
                x8 + ((static_cast<size_t>(b) * N + n) * H + h) * 128 + 32 * q);
            dst[0] = make_uint4(w8[0], w8[1], w8[2], w8[3]);
            dst[1] = make_uint4(w8[4], w8[5], w8[6], w8[7]);
        }
    }
}

// max |v| of each 128-key block of each (batch, kv head) into vmax (float bits,
// atomicMax: non-negative floats order like their bits).
__global__ void __launch_bounds__(128) fp8_vmax_kernel(const uint16_t* __restrict__ v,
                                                       uint32_t* __restrict__ vmax, int N,
                                                       int Hkv) {
    const int blk = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    uint32_t m = 0;
    // the block's 16-byte pieces, all of a thread's sixteen loads in flight at once
    uint4 u[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const int i = threadIdx.x + 128 * k;
        const int n = blk * 128 + i / 16;
        u[k] = (n < N) ? *reinterpret_cast<const uint4*>(
                             v + ((static_cast<size_t>(b) * N + n) * Hkv + hk) * 128 + (i % 16) * 8)
                       : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const uint32_t w[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            m = max(m, (w[j] & 0x7fffu) << 16);
            m = max(m, w[j] & 0x7fff0000u);
        }
    }
    m = __reduce_max_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0 && m != 0) atomicMax(vmax + static_cast<size_t>(b) * Hkv + hk, m);
}

// V^T in e4m3 with one scale per head: each CTA turns a 128-key block into
// 128 rows (one per head-dimension column) of 128 bytes; keys past N are 0.
__global__ void __launch_bounds__(128) fp8_vt_kernel(const uint16_t* __restrict__ v,
                                                     const uint32_t* __restrict__ vmax,
                                                     uint8_t* __restrict__ vt8,
                                                     float* __restrict__ sv, int N, int Hkv,
                                                     int ldv) {
    __shared__ uint16_t tile[128][128 + 8];  // [key][column]
    const int blk = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const float m = __uint_as_float(vmax[static_cast<size_t>(b) * Hkv + hk]);
    const float inv = m > 0.f ? kE4m3Max / m : 1.f;
    if (blk == 0 && threadIdx.x == 0) sv[static_cast<size_t>(b) * Hkv + hk] = m > 0.f ? m / kE4m3Max : 1.f;
    {
        uint4 u[16];  // all of a thread's sixteen loads in flight at once
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int i = threadIdx.x + 128 * k;
            const int n = blk * 128 + i / 16;
            u[k] = (n < N) ? *reinterpret_cast<const uint4*>(
                                 v + ((static_cast<size_t>(b) * N + n) * Hkv + hk) * 128 + (i % 16) * 8)
                           : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int i = threadIdx.x + 128 * k;
            *reinterpret_cast<uint4*>(&tile[i / 16][(i % 16) * 8]) = u[k];
        }
    }
    __syncthreads();
    const int c = threadIdx.x;  // head-dimension column = output row
    uint8_t* dst = vt8 + ((static_cast<size_t>(b) * Hkv + hk) * 128 + c) * ldv + blk * 128;
    for (int k16 = 0; k16 < 128; k16 += 16) {
        if (blk * 128 + k16 >= ldv) break;
        uint32_t w[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            float f[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                f[e] = __uint_as_float(static_cast<uint32_t>(tile[k16 + 4 * q4 + e][c]) << 16) * inv;
            w[q4] = pack_e4m3x4(f[0], f[1], f[2], f[3]);
        }
        *reinterpret_cast<uint4*>(dst + k16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// The forward: persistent CTAs, one per SM, walking (batch, head, 256-query
// block) work items longest first, as the bf16 forward does; the K/V^T ring,
// the barrier phases and TMEM run on from one item to the next, and the
// producer loads an item's Q tiles once the previous item's score products
// are done with them (q_empty).  Per item: two 128-row query tiles, K_j and
// V^T_j streamed through one ring, and the matmul/softmax interleave of the
// bf16 forward -- the tensor core runs one tile's products while the other
// tile's softmax runs -- with every product a kind::f8f6f4 MMA (K = 32 per
// instruction).  TMEM: S0 | S1 | O0 | O1, 128 columns each; P (e4m3, four per
// 32-bit column) goes over the first 32 columns of its S and feeds P V from
// TMEM.  Warps 0-3 do the softmax of tile 0, 4-7 of tile 1 (one query row
// per thread, 208 registers by setmaxnreg), warp 8 issues MMAs, warp 9
// loads, warp 10 is the gate: it folds "V_j and K_{j+1} landed" into the
// p_full barriers, so the MMA thread waits on two barriers per key block;
// warp 11 only completes the issue warpgroup (80 registers each).
__global__ void __launch_bounds__(kF8Threads, 1)
    fa_fp8_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmVt, const Fp8Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sQ = smem_u32(smem);  // Q0, Q1
    const uint32_t sKV = sQ + 2 * kF8Tile;  // slot s at s * kF8Tile
    const uint32_t sStage = sKV + kF8Slots * kF8Tile;  // the epilogue's per-warp buffers
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kF8Tile + kF8Slots * kF8Tile + kF8Stage);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kF8Bars);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t BAR_Q = bar0;
    auto BAR_KVF = [&](int s) { return bar0 + 8u * (1 + s); };
    auto BAR_KVE = [&](int s) { return bar0 + 8u * (1 + kF8Slots + s); };
    auto BAR_SF = [&](int t) { return bar0 + 8u * (1 + 2 * kF8Slots + t); };  // S_t(j) ready
    auto BAR_PF = [&](int t) { return bar0 + 8u * (3 + 2 * kF8Slots + t); };  // P_t(j) written
    auto BAR_OF = [&](int t) { return bar0 + 8u * (5 + 2 * kF8Slots + t); };  // O_t final
    const uint32_t BAR_DONE = bar0 + 8u * (7 + 2 * kF8Slots);
    const uint32_t BAR_QE = bar0 + 8u * (8 + 2 * kF8Slots);  // the item's Q tiles no longer read
    const uint32_t BAR_G1 = bar0 + 8u * (9 + 2 * kF8Slots);  // the gate has seen the item's K_0 land

    const int warp = warp_id();
    const int lane = lane_id();
    const int per = a.B * a.Hq;
    const int n_qblk = (a.nb + 1) / 2;
    const int n_items = n_qblk * per;
    // work item w: longest query blocks first, heads of one KV group adjacent
    struct Item {
        int qb, b, h, hk, nkv0, nkv;  // key blocks tile t = 0, 1 (query blocks 2qb, 2qb + 1) multiplies
    };
    auto item = [&](int w) {
        Item I;
        I.qb = n_qblk - 1 - w / per;
        const int bh = w % per;
        I.b = bh / a.Hq;
        I.h = bh % a.Hq;
        I.hk = I.h / a.g;
        I.nkv0 = a.causal ? min(2 * I.qb + 1, a.nb) : a.nb;
        I.nkv = a.causal ? min(2 * I.qb + 2, a.nb) : a.nb;
        return I;
    };

    if (warp == 0 && lane == 0) {
        mbar_init(BAR_Q, 1);
        for (int s = 0; s < kF8Slots; ++s) {
            mbar_init(BAR_KVF(s), 1);
            mbar_init(BAR_KVE(s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(BAR_SF(t), 1);
            mbar_init(BAR_PF(t), 128 + 1);  // the tile's softmax threads and the gate
            mbar_init(BAR_OF(t), 1);
        }
        mbar_init(BAR_DONE, 1);
        mbar_init(BAR_QE, 1);
        mbar_init(BAR_G1, 1);
        fence_barrier_init();
    }
    if (warp == kF8WarpMma) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;  // S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512)
    // Registers: 384 threads launch with 168 each (64,512); each role first
    // moves its warpgroup's share: 208 for the softmax warpgroups, 80 for the
    // issue warpgroup (2 x 128 x 208 + 128 x 80 = 63,488).

    if (warp == kF8WarpLoad) {
        // ================= TMA producer: per item Q0, Q1, then K_j, V^T_j alternately ======
        setmaxnreg_dec<80>();
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmVt);
            const uint64_t pol = l2_policy_evict_last();  // re-read by every query block
            int last_idx[kF8Slots];
            for (int s = 0; s < kF8Slots; ++s) last_idx[s] = -1;
            bool ok = true;
            int e = 0, it = 0;  // ring entry and items started, running over the items
            for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++it) {
                const Item I = item(w);
                // the previous item's score products are done with Q
                if (it > 0 && !(ok = mbar_wait(BAR_QE, (it - 1) & 1, a.watch, 64))) break;
                mbar_arrive_expect_tx(BAR_Q, 2 * kF8Tile);  // rows past N read as zero
                for (int t = 0; t < 2; ++t)
                    tma_load_4d(sQ + t * kF8Tile, &tmQ, BAR_Q, 0, I.h, (2 * I.qb + t) * 128, I.b);
                for (int j = 0; j < I.nkv && ok; ++j)
                    for (int wv = 0; wv < 2 && ok; ++wv, ++e) {
                        const int slot = e % kF8Slots;
                        if (!(ok = mbar_wait(BAR_KVE(slot), ((e / kF8Slots) & 1) ^ 1u, a.watch, 50)))
                            break;
                        mbar_arrive_expect_tx(BAR_KVF(slot), kF8Tile);
                        if (wv == 0)
                            tma_load_4d_hint(sKV + slot * kF8Tile, &tmK, BAR_KVF(slot), 0, I.hk,
                                             j * 128, I.b, pol);
                        else
                            tma_load_4d_hint(sKV + slot * kF8Tile, &tmVt, BAR_KVF(slot), j * 128, 0,
                                             I.hk, I.b, pol);
                        last_idx[slot] = e;
                    }
            }
            // no copies in flight at exit: the last Q, the last load into each slot
            if (it > 0) mbar_drain(BAR_Q, (it - 1) & 1, a.watch, 51);
            for (int s = 0; s < kF8Slots; ++s)
                if (last_idx[s] >= 0)
                    mbar_drain(BAR_KVF(s), (last_idx[s] / kF8Slots) & 1, a.watch, 51);
        }
        __syncwarp();
    } else if (warp == kF8WarpGate) {
        // ================= gate: V_j and K_{j+1} landed -> p_full(t) =================
        // one arrival per tile that multiplies block j, made only after that
        // barrier's previous phase is over, so it can never count in the wrong
        // one.  It alone waits on the ring's kv_full barriers, every entry in
        // order (each item's K_0 too, passed on to the MMA thread on g1), so
        // that its parity waits always find their slot at the awaited phase
        // or the one after.
        setmaxnreg_dec<80>();
        if (lane == 0) {
            bool ok = true;
            int e = 0, cnt[2] = {0, 0};
            for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
                const Item I = item(w);
                ok = mbar_wait(BAR_KVF(e % kF8Slots), (e / kF8Slots) & 1, a.watch, 58);  // K_0
                if (ok) mbar_arrive(BAR_G1);
                for (int j = 0; j < I.nkv && ok; ++j) {
                    const int vidx = e + 2 * j + 1, kidx = e + 2 * j + 2;
                    ok = mbar_wait(BAR_KVF(vidx % kF8Slots), (vidx / kF8Slots) & 1, a.watch, 58);
                    if (ok && j + 1 < I.nkv)
                        ok = mbar_wait(BAR_KVF(kidx % kF8Slots), (kidx / kF8Slots) & 1, a.watch, 58);
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (t == 0 && j >= I.nkv0) continue;
                        if (cnt[t] > 0) ok = mbar_wait(BAR_PF(t), (cnt[t] - 1) & 1, a.watch, 59);
                        if (ok) mbar_arrive(BAR_PF(t));
                        ++cnt[t];
                    }
                }
                e += 2 * I.nkv;
            }
        }
        __syncwarp();
    } else if (warp == kF8WarpMma) {
        // ================= MMA issuer: PV0(j), S0(j+1), PV1(j), S1(j+1) =================
        // S_t and P_t share TMEM columns: S_t(j+1) is issued after PV_t(j),
        // which reads P_t(j), and the tensor core runs one thread's MMAs in
        // order; an item's first S_t follows the previous item's last PV_t
        // the same way
        setmaxnreg_dec<80>();
        if (lane == 0) {
            constexpr uint32_t ID = idesc_e4m3(128, 128);
            constexpr uint32_t HI = sdesc_hi(1024);
            const uint32_t q_lo = sdesc_lo(sQ, 16);
            auto issue_s = [&](int t, int slot) {
                const uint32_t k_lo = sdesc_lo(sKV + slot * kF8Tile, 16);
                const uint32_t a_lo = q_lo + ((t * kF8Tile) >> 4);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)  // 32 e4m3 = 32 bytes of the 128-byte rows
                    mma_f8_ss(tbase + t * 128, sdesc_at(a_lo, HI, ks * 32), sdesc_at(k_lo, HI, ks * 32),
                              ID, ks > 0);
            };
            auto issue_pv = [&](int t, int slot, bool acc) {
                const uint32_t v_lo = sdesc_lo(sKV + slot * kF8Tile, 16);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)  // 32 keys = 8 TMEM columns of P
                    mma_f8_ts(tbase + 256 + t * 128, tbase + t * 128 + ks * 8,
                              sdesc_at(v_lo, HI, ks * 32), ID, (acc || ks > 0) ? 1u : 0u);
            };
            bool ok = true;
            int e = 0, it = 0, cnt[2] = {0, 0};
            for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x, ++it) {
                const Item I = item(w);
                if (!(ok = mbar_wait(BAR_Q, it & 1, a.watch, 53))) break;
                // K_0 has landed: the gate has seen it (g1)
                if (!(ok = mbar_wait(BAR_G1, it & 1, a.watch, 53))) break;
                tc_fence_after();
                issue_s(0, e % kF8Slots);
                mma_commit(BAR_SF(0));
                issue_s(1, e % kF8Slots);
                mma_commit(BAR_SF(1));
                mma_commit(BAR_KVE(e % kF8Slots));
                // p_full(t) for block j also means V_j and K_{j+1} have landed
                for (int j = 0; j < I.nkv && ok; ++j) {
                    const int vslot = (e + 2 * j + 1) % kF8Slots, kslot = (e + 2 * j + 2) % kF8Slots;
                    if (j < I.nkv0) {
                        if (!(ok = mbar_wait(BAR_PF(0), cnt[0] & 1, a.watch, 54))) break;
                        ++cnt[0];
                        tc_fence_after();
                        issue_pv(0, vslot, j > 0);
                        if (j == I.nkv0 - 1) mma_commit(BAR_OF(0));
                    }
                    if (j + 1 < I.nkv0) {
                        issue_s(0, kslot);
                        mma_commit(BAR_SF(0));
                    }
                    if (!(ok = mbar_wait(BAR_PF(1), cnt[1] & 1, a.watch, 54))) break;
                    ++cnt[1];
                    tc_fence_after();
                    issue_pv(1, vslot, j > 0);
                    mma_commit(BAR_KVE(vslot));
                    if (j == I.nkv - 1) mma_commit(BAR_OF(1));
                    if (j + 1 < I.nkv) {
                        issue_s(1, kslot);
                        mma_commit(BAR_SF(1));
                        mma_commit(BAR_KVE(kslot));
                    }
                }
                if (!ok) break;
                e += 2 * I.nkv;
                mma_commit(BAR_QE);  // the item's score products have read Q
            }
            mma_commit(BAR_DONE);
            mbar_drain(BAR_DONE, 0, a.watch, 55);
        }
        __syncwarp();
    } else if (warp == kF8WarpMma + 3) {
        setmaxnreg_dec<80>();  // idle: completes the issue warpgroup
    } else {
        // ================= softmax: one query row per thread =================
        setmaxnreg_inc<208>();
        const int t = warp >> 2;   // query tile
        const int wq = warp & 3;   // TMEM lanes 32 wq ..
        const int r = wq * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tbase + t * 128 + lane_off, tO = tbase + 256 + t * 128 + lane_off;
        const uint32_t stg = sStage + warp * 2048;
        bool ok = true;
        int nsf = 0, nof = 0;  // phases of s_full and o_final so far
        // the tile's query-block scale, read one item ahead (and first used
        // there, in the item's first block)
        auto q_scale = [&](int w) {
            const Item J = item(w);
            const int qt = 2 * J.qb + t;
            return qt < a.nb ? a.sq[(static_cast<size_t>(J.b) * a.Hq + J.h) * a.nb + qt] : 0.f;
        };
        float sq_next = static_cast<int>(blockIdx.x) < n_items ? q_scale(blockIdx.x) : 0.f;
        for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
            const Item I = item(w);
            const int qt = 2 * I.qb + t;  // 128-row query block of the tile
            const int grow = qt * 128 + r;
            const float sq = sq_next;
            if (w + static_cast<int>(gridDim.x) < n_items) sq_next = q_scale(w + gridDim.x);
            const float* skrow = a.sk + (static_cast<size_t>(I.b) * a.Hkv + I.hk) * a.nb;
            // V's scale, read now and first used by the epilogue
            const float sv = a.sv[static_cast<size_t>(I.b) * a.Hkv + I.hk];
            const int lim = a.causal ? min(grow, a.N - 1) : a.N - 1;
            const int nkv_mine = t ? I.nkv : I.nkv0;
            float m_ref = -INFINITY, l = 0.f;
            // key block j's scale, read a block ahead so that its load has a
            // whole block to land before the maximum needs it
            float sk_next = nkv_mine > 0 ? skrow[0] : 0.f;
            for (int j = 0; j < nkv_mine; ++j) {
                const float sk_j = sk_next;
                if (j + 1 < nkv_mine) sk_next = skrow[j + 1];
                if (!(ok = mbar_wait_warp(BAR_SF(t), nsf & 1, a.watch, 56))) break;
                ++nsf;
                tc_fence_after();
                // x = S * sl2 in log2 units; the maximum is taken on S itself (sl2 > 0)
                // and every exponent is one FMA, two columns per packed f32x2 op
                const float sl2 = a.scale_log2 * sq * sk_j;
                uint32_t s[128];
                tmem_ld32(tS + 0, s);
                tmem_ld32(tS + 32, s + 32);
                tmem_ld32(tS + 64, s + 64);
                tmem_ld32(tS + 96, s + 96);
                tmem_wait_ld();
                reg_fence<128>(s);
                const int kbase = j * 128;
                if (kbase + 127 > lim) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        s[c] = (kbase + c > lim) ? __float_as_uint(-INFINITY) : s[c];
                }
                float mk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    mk[i] = fmaxf(__uint_as_float(s[i]), __uint_as_float(s[i + 8]));
#pragma unroll
                for (int c = 16; c < 128; c += 16)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        mk[i] = fmax3(mk[i], __uint_as_float(s[c + i]), __uint_as_float(s[c + 8 + i]));
                const float mx = fmax3(fmax3(mk[0], mk[1], mk[2]), fmax3(mk[3], mk[4], mk[5]),
                                       fmaxf(mk[6], mk[7])) * sl2;
                const float m_new = fmaxf(m_ref, mx);
                const bool need = m_new > m_ref + 8.f;  // lazy rescale: P stays <= 2^8 < 448
                float alpha = 1.f;
                if (need) {
                    alpha = ex2(m_ref - m_new);
                    l *= alpha;
                    m_ref = m_new;
                }
                const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
                const uint64_t sl2x2 = f2(sl2, sl2), negx2 = f2(neg, neg);
                uint64_t ls2[2] = {0, 0};
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 128; c += 4) {
                    float e0, e1, e2, e3;
                    f2_split(fma2(f2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2x2, negx2),
                             e0, e1);
                    f2_split(fma2(f2(__uint_as_float(s[c + 2]), __uint_as_float(s[c + 3])), sl2x2,
                                  negx2), e2, e3);
                    const float p0 = ex2(e0), p1 = ex2(e1), p2 = ex2(e2), p3 = ex2(e3);
                    ls2[0] = add2(ls2[0], f2(p0, p1));
                    ls2[1] = add2(ls2[1], f2(p2, p3));
                    pk[c >> 2] = pack_e4m3x4(p0, p1, p2, p3);
                }
                {
                    float a0, a1;
                    f2_split(add2(ls2[0], ls2[1]), a0, a1);
                    l += a0 + a1;
                }
                tmem_st32(tS, pk);  // P (e4m3) over the first 32 columns of S_t
                // O_t was last written by PV_t(j-1), which finished before S_t(j)
                if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                    for (int cb = 0; cb < 128; cb += 32) {
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
                mbar_arrive(BAR_PF(t));
            }
            if (!ok) break;
            // ---- epilogue: O * sv / l -> bf16; lse.  Rows reach global memory
            // through this warp's transpose buffer: a thread writes its row's
            // 64-byte piece of a 32-column chunk, then each store instruction
            // writes whole pieces of eight rows (16-byte quarters of row R at
            // R * 64 + 16 * (q ^ ((R >> 1) & 3)), free of bank conflicts).  The
            // next item's first P V product overwrites O_t only after this
            // tile's next p_full arrival, which follows the loads below.
            if (!(ok = mbar_wait_warp(BAR_OF(t), nof & 1, a.watch, 57))) break;
            ++nof;
            tc_fence_after();
            const float f = (l > 0.f) ? sv / l : 0.f;
            const int wrow0 = qt * 128 + wq * 32;  // the warp's first query
#pragma unroll
            for (int cb = 0; cb < 128; cb += 32) {
                uint32_t o[32];
                tmem_ld32(tO + cb, o);
                tmem_wait_ld();
                reg_fence<32>(o);
                uint32_t wv[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    wv[i] = pack_bf16(__uint_as_float(o[2 * i]) * f, __uint_as_float(o[2 * i + 1]) * f);
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
                            a.o + ((static_cast<size_t>(I.b) * a.N + wrow0 + R) * a.Hq + I.h) * 128 +
                            cb + q4 * 8) = make_uint4(v[0], v[1], v[2], v[3]);
                }
                __syncwarp();
            }
            if (grow < a.N)
                a.lse[(static_cast<size_t>(I.b) * a.Hq + I.h) * a.N + grow] =
                    (m_ref + log2f(l)) * 0.6931471805599453f;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kF8WarpMma) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

constexpr int kF8Smem = 1024 + 2 * kF8Tile + kF8Slots * kF8Tile + kF8Stage + kF8Bars * 8 + 16;

}  // namespace

cudaError_t launch_fp8(const Fp8Maps& m, const Fp8Args& a, cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    if (a.quantize) {
    if ((e = cudaMemsetAsync(a.vmax, 0, sizeof(uint32_t) * a.B * a.Hkv, st)) != cudaSuccess)
        return e;
    fp8_rows_kernel<<<dim3(a.nb, a.Hq, a.B), 256, 0, st>>>(a.q, a.q8, a.sq, a.N, a.Hq, a.nb,
                                                           a.rotate);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    fp8_rows_kernel<<<dim3(a.nb, a.Hkv, a.B), 256, 0, st>>>(a.k, a.k8, a.sk, a.N, a.Hkv, a.nb,
                                                            a.rotate);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    fp8_vmax_kernel<<<dim3(a.nb, a.Hkv, a.B), 128, 0, st>>>(a.v, a.vmax, a.N, a.Hkv);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    fp8_vt_kernel<<<dim3(a.nb, a.Hkv, a.B), 128, 0, st>>>(a.v, a.vmax, a.vt8, a.sv, a.N, a.Hkv,
                                                          a.ldv);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (!a.attend) return cudaSuccess;
    if ((e = cudaFuncSetAttribute(fa_fp8_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kF8Smem)) != cudaSuccess)
        return e;
    const long long items = static_cast<long long>((a.nb + 1) / 2) * a.B * a.Hq;
    if (items <= 0 || items > 0x7fffffffLL || a.num_ctas <= 0) return cudaErrorInvalidConfiguration;
    // persistent: one CTA per SM (shared memory and registers allow no more)
    const unsigned grid = static_cast<unsigned>(items < a.num_ctas ? items : a.num_ctas);
    fa_fp8_fwd_kernel<<<grid, kF8Threads, kF8Smem, st>>>(m.q8, m.k8, m.vt8, a);
    return cudaGetLastError();
}

}  // namespace fa
