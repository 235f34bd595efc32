// fa_api.cu -- the C ABI of libfa (declared in include/fa.h): argument
// checks, TMA tensor maps, the device status word, and launches on the
// caller's stream.  No device memory is allocated here.
#include <stdio.h>
#include <string.h>

#include <atomic>

#include <cudaTypedefs.h>

#include "fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

// Status words written by bounded waits that run out (one pair per device: a
// __device__ variable exists once per device context): [0] the first failure
// since the host last read it, [1] the id of the last launch that failed.
__device__ uint32_t g_status_word[2];

namespace {

thread_local char t_last_error[256] = "";

// Launch ids for the bounded waits: every launch gets its own nonzero id, so
// that its thread blocks can tell a failure of their own launch (stop at
// once) from one an earlier launch left in the status words.
std::atomic<uint32_t> g_launch_counter{0};

Watch make_watch(uint32_t* status, uint64_t timeout_ns = kWaitTimeoutNs) {
    uint32_t id = 0;
    while (id == 0) id = g_launch_counter.fetch_add(1, std::memory_order_relaxed) + 1;
    Watch w;
    w.status = status;
    w.timeout_ns = timeout_ns;
    w.launch = id;
    return w;
}

fa_status cuda_fail(cudaError_t e, const char* where) {
    snprintf(t_last_error, sizeof(t_last_error), "%s: %s (%d)", where, cudaGetErrorString(e),
             static_cast<int>(e));
    return FA_ERR_CUDA;
}

constexpr int kMaxDevices = 64;
struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    uint32_t* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Per-device set-up: checks for an sm_103 device and fetches the device
// address of the status word (no allocation).
fa_status device_ready(DeviceInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    DeviceInfo& di = g_dev[dev];
    if (!di.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        di.supported = (major == 10 && minor == 3);
        if ((e = cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (di.supported) {
            void* p = nullptr;
            if ((e = cudaGetSymbolAddress(&p, g_status_word)) != cudaSuccess)
                return cuda_fail(e, "cudaGetSymbolAddress(status)");
            di.status = static_cast<uint32_t*>(p);
        }
        if (!g_encode) {
            cudaDriverEntryPointQueryResult q;
            void* fn = nullptr;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                return cuda_fail(e == cudaSuccess ? cudaErrorSymbolNotFound : e,
                                 "cuTensorMapEncodeTiled entry point");
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        di.ready = true;
    }
    if (!di.supported) {
        snprintf(t_last_error, sizeof(t_last_error), "device %d is not an sm_103 GPU", dev);
        return FA_ERR_UNSUPPORTED;
    }
    *out = &di;
    return FA_OK;
}

// Tensor map of a [B, N, H, d] bf16 (or, f16 = true, fp16) tensor: dims
// (d, H, N, B), box (64, heads, rows, 1), 128-byte swizzle; rows past N read
// as zero and are never written.
fa_status make_map(CUtensorMap* m, const void* ptr, int B, int N, int H, int d, bool f16 = false,
                   int rows = kBM, int heads = 1) {
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(H) * d * 2,
                             static_cast<cuuint64_t>(N) * H * d * 2};
    cuuint32_t box[4] = {64, static_cast<cuuint32_t>(heads), static_cast<cuuint32_t>(rows), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          4, const_cast<void*>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(t_last_error, sizeof(t_last_error), "cuTensorMapEncodeTiled failed (%d)",
                 static_cast<int>(r));
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Byte offsets inside the training workspace (each 256-aligned), shared by
// fa_fwd_train and fa_bwd: D, the fp16 copies of Q, K, V, dO, the absmax
// words and the scales.
struct WsLayout {
    size_t d, q16, k16, v16, do16, absmax, scales, total;
};

WsLayout bwd_layout(int B, int H, int Hkv, int N, int d) {
    const size_t q_el = static_cast<size_t>(B) * N * H * d, kv_el = static_cast<size_t>(B) * N * Hkv * d;
    WsLayout w{};
    w.d = 0;
    w.q16 = up256(4ull * static_cast<size_t>(B) * H * N);
    w.k16 = w.q16 + up256(2 * q_el);
    w.v16 = w.k16 + up256(2 * kv_el);
    w.do16 = w.v16 + up256(2 * kv_el);
    w.absmax = w.do16 + up256(2 * q_el);
    w.scales = w.absmax + 256;
    w.total = w.scales + 256;
    return w;
}

template <typename T>
T* at(void* base, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

// A job that copies the listed tensors (q, k, v, dout; null = skip) into the
// workspace's fp16 slots.
F16Prep prep_job(void* ws, const WsLayout& wl, const void* q, const void* k, const void* v,
                 const void* dout, int B, int H, int Hkv, int N, int d) {
    F16Prep p{};
    const void* src[4] = {q, k, v, dout};
    const size_t off[4] = {wl.q16, wl.k16, wl.v16, wl.do16};
    const size_t nq = static_cast<size_t>(B) * N * H * d, nkv = static_cast<size_t>(B) * N * Hkv * d;
    const size_t n[4] = {nq, nkv, nkv, nq};
    for (int t = 0; t < 4; ++t) {
        p.src[t] = static_cast<const uint16_t*>(src[t]);
        p.dst[t] = at<uint16_t>(ws, off[t]);
        p.n[t] = src[t] ? n[t] : 0;
    }
    p.absmax = at<uint32_t>(ws, wl.absmax);
    p.scales = at<F16Scales>(ws, wl.scales);
    p.d = d;
    p.convert_mask = (q ? 1 : 0) | (k ? 2 : 0) | (v ? 4 : 0) | (dout ? 8 : 0);
    return p;
}


fa_status check_sizes(int B, int H, int Hkv, int N, int d, float scale) {
    if (B < 1 || H < 1 || Hkv < 1 || N < 1) return FA_ERR_INVALID_ARG;
    if (H % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !(scale < 3.0e38f)) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    // every element offset and every TMA coordinate must fit in 32-bit ints
    const long long qel = static_cast<long long>(B) * N * H * d;
    if (qel >= (1LL << 40) || N > (1 << 30) || static_cast<long long>(B) * H * N >= (1LL << 31))
        return FA_ERR_INVALID_ARG;
    return FA_OK;
}

__global__ void watchdog_probe_kernel(const Watch w) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(b, 0, w, 0xFE);  // nothing ever arrives
    __syncthreads();
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

const char* fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT";
    }
    return "FA_ERR_UNKNOWN";
}

const char* fa_last_cuda_error(void) { return t_last_error; }

size_t fa_bwd_workspace_size(int B, int H, int Hkv, int N, int d) {
    if (check_sizes(B, H, Hkv, N, d, 1.f) != FA_OK) return 0;
    return bwd_layout(B, H, Hkv, N, d).total;
}



fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int Hkv, int N, int d, int causal, float scale, void* stream) {
    return fa_fwd_train(q, k, v, o, nullptr, lse, nullptr, B, H, Hkv, N, d, causal, scale,
                        stream);
}

fa_status fa_fwd_train(const void* q, const void* k, const void* v, void* o, void* o_lo,
                       float* lse, void* workspace, int B, int H, int Hkv, int N, int d,
                       int causal, float scale, void* stream) {
    t_last_error[0] = 0;
    fa_status st = check_sizes(B, H, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_INVALID_ARG;
    if (o_lo && !aligned16(o_lo)) return FA_ERR_INVALID_ARG;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID_ARG;
    DeviceInfo* di = nullptr;
    if ((st = device_ready(&di)) != FA_OK) return st;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const WsLayout wl = bwd_layout(B, H, Hkv, N, d);
    FwdMaps maps;
    if ((st = make_map(&maps.q, q, B, N, H, d)) != FA_OK) return st;
    if ((st = make_map(&maps.k, k, B, N, Hkv, d)) != FA_OK) return st;
    if (workspace) {
        // fp16 copies of Q, K, V: V for the P V product (P then in fp16), Q and
        // K left for a backward that runs with FA_BWD_PREP_DOUT on this workspace.
        // The prep kernels take the three maxima and copy K and V; the forward
        // kernel copies the Q tiles it loads anyway.
        if ((st = make_map(&maps.v, at<void>(workspace, wl.v16), B, N, Hkv, d, true)) != FA_OK)
            return st;
        F16Prep p = prep_job(workspace, wl, q, k, v, nullptr, B, H, Hkv, N, d);
        p.convert_mask &= ~1;
        const cudaError_t e = launch_f16_prep(p, cs);
        if (e != cudaSuccess) return cuda_fail(e, "fp16 copies of Q, K, V");
    } else if ((st = make_map(&maps.v, v, B, N, Hkv, d)) != FA_OK) {
        return st;
    }
    FwdArgs a;
    a.o = static_cast<uint16_t*>(o);
    a.lse = lse;
    a.o_lo = static_cast<uint16_t*>(o_lo);
    a.f16s = workspace ? at<const F16Scales>(workspace, wl.scales) : nullptr;
    a.q16 = workspace ? at<uint16_t>(workspace, wl.q16) : nullptr;
    a.B = B;
    a.Hq = H;
    a.Hkv = Hkv;
    a.N = N;
    a.g = H / Hkv;
    a.causal = causal ? 1 : 0;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.n_qblk = (N + 2 * kBM - 1) / (2 * kBM);
    a.num_ctas = di->num_sms;
    a.block_mask = nullptr;
    a.watch = make_watch(di->status);
    cudaError_t e = launch_fwd(maps, a, d, cs);
    if (e != cudaSuccess) return cuda_fail(e, "fa_fwd launch");
    return FA_OK;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, void* workspace,
                 const void* o_lo, int B, int H, int Hkv, int N, int d, int causal, float scale,
                 void* stream) {
    return fa_bwd_stage(FA_BWD_PREP | FA_BWD_DSUM | FA_BWD_DKDV | FA_BWD_DQ, q, k, v, o, dout, lse,
                        dq, dk, dv, workspace, o_lo, B, H, Hkv, N, d, causal, scale, stream);
}

fa_status fa_bwd_stage(int stages, const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv,
                       void* workspace, const void* o_lo, int B, int H, int Hkv, int N, int d,
                       int causal, float scale, void* stream) {
    t_last_error[0] = 0;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return FA_ERR_INVALID_ARG;
    return fa::bwd_run(stages, q, k, v, o, dout, lse, dq, dk, dv, static_cast<float*>(workspace),
                       workspace, o_lo, B, H, Hkv, N, d, causal, scale, stream);
}

}  // extern "C"

namespace fa {

fa_status bwd_run(int stages, const void* q, const void* k, const void* v, const void* o,
                  const void* dout, const float* lse, void* dq, void* dk, void* dv, float* dsum,
                  void* f16_ws, const void* o_lo, int B, int H, int Hkv, int N, int d, int causal,
                  float scale, void* stream) {
    t_last_error[0] = 0;
    if (stages <= 0 || stages > 31) return FA_ERR_INVALID_ARG;
    fa_status st = check_sizes(B, H, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
        !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(dsum))
        return FA_ERR_INVALID_ARG;
    if (o_lo && !aligned16(o_lo)) return FA_ERR_INVALID_ARG;
    DeviceInfo* di = nullptr;
    if ((st = device_ready(&di)) != FA_OK) return st;
    BwdMaps maps;
    if ((st = make_map(&maps.q, q, B, N, H, d)) != FA_OK) return st;
    if ((st = make_map(&maps.k, k, B, N, Hkv, d)) != FA_OK) return st;
    if ((st = make_map(&maps.v, v, B, N, Hkv, d)) != FA_OK) return st;
    if ((st = make_map(&maps.dout, dout, B, N, H, d)) != FA_OK) return st;
    if ((st = make_map(&maps.dq, dq, B, N, H, d)) != FA_OK) return st;
    if ((st = make_map(&maps.dk, dk, B, N, Hkv, d)) != FA_OK) return st;
    if ((st = make_map(&maps.dv, dv, B, N, Hkv, d)) != FA_OK) return st;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const WsLayout wl = bwd_layout(B, H, Hkv, N, d);
    if (f16_ws) {
        if ((st = make_map(&maps.q16, at<void>(f16_ws, wl.q16), B, N, H, d, true)) != FA_OK)
            return st;
        if ((st = make_map(&maps.k16, at<void>(f16_ws, wl.k16), B, N, Hkv, d, true)) != FA_OK)
            return st;
        if ((st = make_map(&maps.v16, at<void>(f16_ws, wl.v16), B, N, Hkv, d, true)) != FA_OK)
            return st;
        if ((st = make_map(&maps.dout16, at<void>(f16_ws, wl.do16), B, N, H, d, true)) != FA_OK)
            return st;
        if (stages & (FA_BWD_PREP | FA_BWD_PREP_DOUT)) {
            const bool all = (stages & FA_BWD_PREP) != 0;
            // max |dO| comes from the dsum kernel when D is formed in the same
            // call (it reads dO anyway), else from the prep kernels
            const bool max_in_dsum = (stages & FA_BWD_DSUM) != 0;
            F16Prep p = prep_job(f16_ws, wl, all ? q : nullptr, all ? k : nullptr,
                                 all ? v : nullptr, max_in_dsum ? nullptr : dout, B, H, Hkv, N, d);
            p.convert_mask &= ~8;  // the dQ kernel writes the copy of dO
            cudaError_t e = cudaSuccess;
            if (max_in_dsum)
                e = cudaMemsetAsync(at<uint32_t>(f16_ws, wl.absmax) + 3, 0, sizeof(uint32_t), cs);
            if (e == cudaSuccess && (p.n[0] | p.n[1] | p.n[2] | p.n[3]) != 0)
                e = launch_f16_prep(p, cs);
            if (e != cudaSuccess) return cuda_fail(e, "fp16 operand copies");
        }
    }
    BwdArgs a;
    a.lse = lse;
    a.dsum = dsum;
    a.f16s = f16_ws ? at<const F16Scales>(f16_ws, wl.scales) : nullptr;
    a.dout16 = f16_ws ? at<uint16_t>(f16_ws, wl.do16) : nullptr;
    a.absmax = f16_ws ? at<uint32_t>(f16_ws, wl.absmax) : nullptr;
    a.scales_w = f16_ws ? at<F16Scales>(f16_ws, wl.scales) : nullptr;
    a.dout_max = f16_ws && (stages & (FA_BWD_PREP | FA_BWD_PREP_DOUT)) && (stages & FA_BWD_DSUM)
                     ? at<uint32_t>(f16_ws, wl.absmax) + 3
                     : nullptr;
    a.o = static_cast<const uint16_t*>(o);
    a.dout = static_cast<const uint16_t*>(dout);
    a.o_lo = static_cast<const uint16_t*>(o_lo);
    a.B = B;
    a.Hq = H;
    a.Hkv = Hkv;
    a.N = N;
    a.d = d;
    a.g = H / Hkv;
    a.causal = causal ? 1 : 0;
    a.scale = scale;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.num_ctas = di->num_sms;
    a.watch = make_watch(di->status);
    if ((stages & 7) == 0) return FA_OK;
    cudaError_t e = launch_bwd(maps, a, stages & 7, cs);
    if (e != cudaSuccess) return cuda_fail(e, "fa_bwd launch");
    return FA_OK;
}

}  // namespace fa

namespace fa {
namespace {

// How a split-KV call is cut: qpt queries of all g heads per 128-row tile,
// and the key blocks into splits of blocks_per_split blocks.  num_splits <= 0
// picks the count with the shortest estimated time on this GPU's 152 SMs.
struct DecodePlan {
    int g, qpt, n_qt, splits, blocks_per_split;
};

fa_status decode_plan(int B, int H, int Hkv, int Nq, int Nk, int d, int causal, int num_splits,
                      DecodePlan* pl) {
    if (B < 1 || H < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (causal && Nq > Nk) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    const int g = H / Hkv;
    if (g > kBM) return FA_ERR_UNSUPPORTED;
    const long long qel = static_cast<long long>(B) * Nq * H * d;
    const long long kel = static_cast<long long>(B) * Nk * Hkv * d;
    if (qel >= (1LL << 40) || kel >= (1LL << 40) || Nq > (1 << 30) || Nk > (1 << 30) ||
        static_cast<long long>(B) * H * Nq >= (1LL << 31))
        return FA_ERR_INVALID_ARG;
    pl->g = g;
    pl->qpt = kBM / g;
    pl->n_qt = (Nq + pl->qpt - 1) / pl->qpt;
    const int nblk = (Nk + kBN - 1) / kBN;
    const long long units = static_cast<long long>(B) * Hkv * pl->n_qt;
    int splits = num_splits;
    if (splits <= 0) {
        // One CTA per SM (the K/V ring takes the shared memory), so the time
        // is about waves x (blocks per split + ~3 blocks of set-up); take the
        // count that minimises it (the smallest on ties).
        const int cap = nblk < 1024 ? nblk : 1024;
        long long best = -1;
        for (int s2 = 1; s2 <= cap; ++s2) {
            const int bps = (nblk + s2 - 1) / s2;
            const long long ctas = units * ((nblk + bps - 1) / bps);
            const long long cost = ((ctas + 151) / 152) * (bps + 3);
            if (best < 0 || cost < best) {
                best = cost;
                splits = s2;
            }
        }
    }
    if (splits > nblk) splits = nblk;
    if (splits < 1) splits = 1;
    pl->blocks_per_split = (nblk + splits - 1) / splits;
    pl->splits = (nblk + pl->blocks_per_split - 1) / pl->blocks_per_split;  // none empty
    if (units * pl->splits > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    return FA_OK;
}

// Workspace of a call with `splits` > 1: fp32 O_s [splits, B, H, Nq, d], then
// lse_s [splits, B, H, Nq], each part rounded up to 256 bytes.
size_t decode_part_bytes(int B, int H, int Nq, int d, int splits, size_t* lse_off) {
    const size_t rows = static_cast<size_t>(splits) * B * H * Nq;
    *lse_off = up256(rows * d * 4);
    return *lse_off + up256(rows * 4);
}

}  // namespace
}  // namespace fa

extern "C" {

int fa_fwd_splitkv_num_splits(int B, int H, int Hkv, int Nq, int Nk, int d, int causal,
                              int num_splits) {
    fa::DecodePlan pl;
    if (fa::decode_plan(B, H, Hkv, Nq, Nk, d, causal, num_splits, &pl) != FA_OK) return 0;
    return pl.splits;
}

size_t fa_fwd_splitkv_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d, int causal,
                                     int num_splits) {
    fa::DecodePlan pl;
    if (fa::decode_plan(B, H, Hkv, Nq, Nk, d, causal, num_splits, &pl) != FA_OK) return 0;
    if (pl.splits == 1) return 0;
    size_t off = 0;
    return fa::decode_part_bytes(B, H, Nq, d, pl.splits, &off);
}

fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                         void* workspace, int B, int H, int Hkv, int Nq, int Nk, int d,
                         int causal, float scale, int num_splits, void* stream) {
    t_last_error[0] = 0;
    fa::DecodePlan pl;
    fa_status st = fa::decode_plan(B, H, Hkv, Nq, Nk, d, causal, num_splits, &pl);
    if (st != FA_OK) return st;
    if (!(scale > 0.f) || !(scale < 3.0e38f)) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_INVALID_ARG;
    if (pl.splits > 1 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return FA_ERR_INVALID_ARG;
    DeviceInfo* di = nullptr;
    if ((st = device_ready(&di)) != FA_OK) return st;
    DecodeMaps maps;
    if ((st = make_map(&maps.q, q, B, Nq, H, d, false, pl.qpt, pl.g)) != FA_OK) return st;
    if ((st = make_map(&maps.k, k, B, Nk, Hkv, d)) != FA_OK) return st;
    if ((st = make_map(&maps.v, v, B, Nk, Hkv, d)) != FA_OK) return st;
    DecodeArgs a;
    a.o = static_cast<uint16_t*>(o);
    a.lse = lse;
    a.part_o = nullptr;
    a.part_lse = nullptr;
    if (pl.splits > 1) {
        size_t lse_off = 0;
        fa::decode_part_bytes(B, H, Nq, d, pl.splits, &lse_off);
        a.part_o = static_cast<float*>(workspace);
        a.part_lse = at<float>(workspace, lse_off);
    }
    a.B = B;
    a.Hq = H;
    a.Hkv = Hkv;
    a.Nq = Nq;
    a.Nk = Nk;
    a.g = pl.g;
    a.gp = pl.g;
    a.causal = causal ? 1 : 0;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.qpt = pl.qpt;
    a.n_qt = pl.n_qt;
    a.splits = pl.splits;
    a.blocks_per_split = pl.blocks_per_split;
    a.watch = make_watch(di->status);
    const cudaError_t e = launch_decode(maps, a, d, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fa_fwd_splitkv launch");
    return FA_OK;
}

fa_status fa_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse,
                             const uint8_t* block_mask, int B, int H, int Hkv, int N, int d,
                             int causal, float scale, void* stream) {
    t_last_error[0] = 0;
    fa_status st = check_sizes(B, H, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        !block_mask)
        return FA_ERR_INVALID_ARG;
    const int nb = (N + kBM - 1) / kBM;
    if (static_cast<long long>(B) * H * nb > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    if (nb > kSparseMaxBlocks) return FA_ERR_UNSUPPORTED;
    DeviceInfo* di = nullptr;
    if ((st = device_ready(&di)) != FA_OK) return st;
    FwdMaps maps;
    if ((st = make_map(&maps.q, q, B, N, H, d)) != FA_OK) return st;
    if ((st = make_map(&maps.k, k, B, N, Hkv, d)) != FA_OK) return st;
    if ((st = make_map(&maps.v, v, B, N, Hkv, d)) != FA_OK) return st;
    if ((st = make_map(&maps.o, o, B, N, H, d)) != FA_OK) return st;
    // the forward kernel, each of its two query tiles walking its own mask row
    FwdArgs a;
    a.o = static_cast<uint16_t*>(o);
    a.lse = lse;
    a.o_lo = nullptr;
    a.f16s = nullptr;
    a.q16 = nullptr;
    a.B = B;
    a.Hq = H;
    a.Hkv = Hkv;
    a.N = N;
    a.g = H / Hkv;
    a.causal = causal ? 1 : 0;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.n_qblk = (N + 2 * kBM - 1) / (2 * kBM);
    a.num_ctas = di->num_sms;
    a.block_mask = block_mask;
    a.watch = make_watch(di->status);
    const cudaError_t e = launch_fwd(maps, a, d, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fa_fwd_blocksparse launch");
    return FA_OK;
}

}  // extern "C"

namespace fa {
namespace {

// A tiled 4-D tensor map over bytes (e4m3), 128-byte swizzle.
fa_status make_map_u8(CUtensorMap* m, const void* ptr, const cuuint64_t (&dims)[4],
                      const cuuint64_t (&strides)[3], const cuuint32_t (&box)[4]) {
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr),
                          const_cast<cuuint64_t*>(dims), const_cast<cuuint64_t*>(strides),
                          const_cast<cuuint32_t*>(box), estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(t_last_error, sizeof(t_last_error), "cuTensorMapEncodeTiled failed (%d)",
                 static_cast<int>(r));
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

// Byte offsets of the FP8 workspace: q8, k8, vt8, sq, sk, sv, vmax (each
// 256-aligned).
struct Fp8Layout {
    size_t q8, k8, vt8, sq, sk, sv, vmax, total;
    int nb, ldv;
};

Fp8Layout fp8_layout(int B, int H, int Hkv, int N) {
    Fp8Layout L{};
    L.nb = (N + 127) / 128;
    L.ldv = (N + 15) / 16 * 16;
    L.q8 = 0;
    L.k8 = L.q8 + up256(static_cast<size_t>(B) * N * H * 128);
    L.vt8 = L.k8 + up256(static_cast<size_t>(B) * N * Hkv * 128);
    L.sq = L.vt8 + up256(static_cast<size_t>(B) * Hkv * 128 * L.ldv);
    L.sk = L.sq + up256(static_cast<size_t>(B) * H * L.nb * 4);
    L.sv = L.sk + up256(static_cast<size_t>(B) * Hkv * L.nb * 4);
    L.vmax = L.sv + up256(static_cast<size_t>(B) * Hkv * 4);
    L.total = L.vmax + up256(static_cast<size_t>(B) * Hkv * 4);
    return L;
}

}  // namespace
}  // namespace fa

extern "C" {

size_t fa_fwd_fp8_workspace_size(int B, int H, int Hkv, int N, int d) {
    if (check_sizes(B, H, Hkv, N, d, 1.f) != FA_OK || d != 128) return 0;
    return fa::fp8_layout(B, H, Hkv, N).total;
}

fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                     void* workspace, int B, int H, int Hkv, int N, int d, int causal,
                     float scale, int flags, void* stream) {
    t_last_error[0] = 0;
    fa_status st = check_sizes(B, H, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    if (flags & ~(FA_FP8_ROTATE | FA_FP8_QUANTIZE_ONLY | FA_FP8_ATTEND_ONLY)) return FA_ERR_INVALID_ARG;
    if ((flags & FA_FP8_QUANTIZE_ONLY) && (flags & FA_FP8_ATTEND_ONLY)) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        !workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return FA_ERR_INVALID_ARG;
    DeviceInfo* di = nullptr;
    if ((st = device_ready(&di)) != FA_OK) return st;
    const fa::Fp8Layout L = fa::fp8_layout(B, H, Hkv, N);
    Fp8Maps maps;
    {
        const cuuint64_t dq[4] = {128, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(N),
                                  static_cast<cuuint64_t>(B)};
        const cuuint64_t sq[3] = {128, static_cast<cuuint64_t>(H) * 128,
                                  static_cast<cuuint64_t>(N) * H * 128};
        const cuuint64_t dk[4] = {128, static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(N),
                                  static_cast<cuuint64_t>(B)};
        const cuuint64_t sk[3] = {128, static_cast<cuuint64_t>(Hkv) * 128,
                                  static_cast<cuuint64_t>(N) * Hkv * 128};
        const cuuint64_t dv[4] = {static_cast<cuuint64_t>(L.ldv), 128,
                                  static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(B)};
        const cuuint64_t sv[3] = {static_cast<cuuint64_t>(L.ldv),
                                  static_cast<cuuint64_t>(L.ldv) * 128,
                                  static_cast<cuuint64_t>(L.ldv) * 128 * Hkv};
        const cuuint32_t box_rows[4] = {128, 1, 128, 1};
        const cuuint32_t box_vt[4] = {128, 128, 1, 1};
        if ((st = fa::make_map_u8(&maps.q8, at<void>(workspace, L.q8), dq, sq, box_rows)) != FA_OK)
            return st;
        if ((st = fa::make_map_u8(&maps.k8, at<void>(workspace, L.k8), dk, sk, box_rows)) != FA_OK)
            return st;
        if ((st = fa::make_map_u8(&maps.vt8, at<void>(workspace, L.vt8), dv, sv, box_vt)) != FA_OK)
            return st;
    }
    Fp8Args a;
    a.q = static_cast<const uint16_t*>(q);
    a.k = static_cast<const uint16_t*>(k);
    a.v = static_cast<const uint16_t*>(v);
    a.q8 = at<uint8_t>(workspace, L.q8);
    a.k8 = at<uint8_t>(workspace, L.k8);
    a.vt8 = at<uint8_t>(workspace, L.vt8);
    a.sq = at<float>(workspace, L.sq);
    a.sk = at<float>(workspace, L.sk);
    a.sv = at<float>(workspace, L.sv);
    a.vmax = at<uint32_t>(workspace, L.vmax);
    a.o = static_cast<uint16_t*>(o);
    a.lse = lse;
    a.B = B;
    a.Hq = H;
    a.Hkv = Hkv;
    a.N = N;
    a.g = H / Hkv;
    a.ldv = L.ldv;
    a.nb = L.nb;
    a.causal = causal ? 1 : 0;
    a.rotate = (flags & FA_FP8_ROTATE) ? 1 : 0;
    a.quantize = (flags & FA_FP8_ATTEND_ONLY) ? 0 : 1;
    a.attend = (flags & FA_FP8_QUANTIZE_ONLY) ? 0 : 1;
    a.num_ctas = di->num_sms;
    a.scale_log2 = scale * 1.4426950408889634f * (a.rotate ? 1.f / 128.f : 1.f);
    a.watch = make_watch(di->status);
    const cudaError_t e = launch_fp8(maps, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fa_fwd_fp8 launch");
    return FA_OK;
}

}  // extern "C"

extern "C" {

fa_status fa_get_device_error(void* stream) {
    t_last_error[0] = 0;
    DeviceInfo* di = nullptr;
    fa_status st = device_ready(&di);
    if (st != FA_OK) return st;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    uint32_t word = 0;
    if ((e = cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word))) != cudaSuccess)
        return cuda_fail(e, "read status word");
    if (word != 0) {
        // word [1] (the failed launch's id) stays: ids are never reused
        const uint32_t zero = 0;
        if ((e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero))) != cudaSuccess)
            return cuda_fail(e, "clear status word");
        snprintf(t_last_error, sizeof(t_last_error), "device status 0x%x (site %u)", word,
                 word >> 8);
        return (word & 0xFF) == kDevTimeout ? FA_ERR_DEVICE_TIMEOUT : FA_ERR_CUDA;
    }
    return FA_OK;
}

fa_status fa_debug_watchdog_probe(uint64_t timeout_ns, int num_blocks, void* stream) {
    t_last_error[0] = 0;
    DeviceInfo* di = nullptr;
    fa_status st = device_ready(&di);
    if (st != FA_OK) return st;
    if (timeout_ns < 1000ull) timeout_ns = 1000ull;
    if (timeout_ns > 5000000000ull) timeout_ns = 5000000000ull;
    if (num_blocks < 1) num_blocks = 1;
    if (num_blocks > (1 << 20)) num_blocks = 1 << 20;
    watchdog_probe_kernel<<<num_blocks, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        make_watch(di->status, timeout_ns));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "watchdog probe launch");
    return FA_OK;
}

}  // extern "C"
