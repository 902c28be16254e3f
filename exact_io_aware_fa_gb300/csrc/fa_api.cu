// fa_api.cu -- the C ABI declared in include/fa.h: argument checks, TMA tensor-map
// encoding, workspace handling and kernel launches. No compute happens here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "fa_common.cuh"
#include "fa_launch.h"

static_assert(FA_MAX_SPLITS <= 64, "the split merge holds at most two LSEs per lane");

namespace {

thread_local int t_last_cuda_error = 0;

// The device error word the kernels write when a wait gives up (one per device).
__device__ int g_fa_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

fa_status cuda_fail(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return FA_ERR_CUDA;
}

// Make the current device's primary context current on the calling thread before any driver
// call (tensor-map encoding needs one). A thread that only ever selected a device -- e.g. a
// framework's worker thread for the default device -- may have none bound yet.
thread_local int t_bound_dev = -1;
fa_status bind_context() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev != t_bound_dev) {
        e = cudaSetDevice(dev);
        if (e != cudaSuccess) return cuda_fail(e);
        t_bound_dev = dev;
    }
    return FA_OK;
}

// Driver entry point for cuTensorMapEncodeTiled, resolved through the runtime so the
// library does not link libcuda directly.
fa_status get_encode(EncodeTiledFn* out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess) return cuda_fail(e);
        if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cuda_fail(cudaErrorNotSupported);
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    *out = g_encode;
    return FA_OK;
}

// Address of this device's error word (looked up once per device, with that device current).
fa_status get_err_ptr(int** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fa_error_word);
        if (e != cudaSuccess) return cuda_fail(e);
        g_err_ptr[dev] = static_cast<int*>(p);
    }
    *out = g_err_ptr[dev];
    return FA_OK;
}

// Streaming-multiprocessor count of the current device (looked up once per device).
fa_status get_num_sms(int* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_num_sms[dev] == 0) {
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        g_num_sms[dev] = n > 0 ? n : 1;
    }
    *out = g_num_sms[dev];
    return FA_OK;
}

// 3-D tiled map over a contiguous [BH, N, d] tensor of bf16 (or fp32): dims {d, N, BH}, box
// {128 bytes of columns, box_rows, 1}, 128-byte swizzle. Rows past N inside a box read as zero
// and are not written by stores or reductions.
fa_status make_map(CUtensorMap* m, const void* base, int BH, int N, int d, int box_rows,
                   bool fp32 = false) {
    EncodeTiledFn enc = nullptr;
    fa_status st = get_encode(&enc);
    if (st != FA_OK) return st;
    const cuuint64_t esz = fp32 ? 4u : 2u;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * esz, (cuuint64_t)N * (cuuint64_t)d * esz};
    cuuint32_t box[3] = {(cuuint32_t)(128u / esz), (cuuint32_t)box_rows, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                     const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = (int)r;
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Problem shape after the host checks.
struct Shape {
    int B, Hq, Hkv, Tq, Tk, d, causal, window;
    int BHq, BHkv;
};

// Checks shared by every entry point. Sets *empty when there is nothing to compute (no query
// rows; the backward still owes zero dK/dV when there are keys).
fa_status check_shape(int B, int Hq, int Hkv, int Tq, int Tk, int d, int causal, int window,
                      float scale, Shape* sh, bool* empty) {
    if (B < 0 || Hq < 0 || Hkv < 0 || Tq < 0 || Tk < 0) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (window < -1) return FA_ERR_INVALID_ARG;
    if (window >= 0 && !causal) return FA_ERR_INVALID_ARG;  // the window hangs off the diagonal
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if ((Hq == 0) != (Hkv == 0)) return FA_ERR_INVALID_ARG;
    if (Hkv > 0 && Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
    const long long bhq = (long long)B * (long long)Hq;
    const long long bhkv = (long long)B * (long long)Hkv;
    *empty = (bhq == 0 || Tq == 0);
    if (bhq > 0 && Tq > 0) {
        // every query row must see at least one key
        if (Tk == 0) return FA_ERR_INVALID_ARG;
        if (causal && Tq > Tk) return FA_ERR_INVALID_ARG;
    }
    if (bhq > INT_MAX || bhkv > INT_MAX) return FA_ERR_UNSUPPORTED;
    if ((long long)Tq + 256 > INT_MAX || (long long)Tk + 256 > INT_MAX) return FA_ERR_UNSUPPORTED;
    if (((long long)Tq + 255) / 256 * bhq > INT_MAX) return FA_ERR_UNSUPPORTED;
    if (((long long)Tk + 127) / 128 * bhkv > INT_MAX) return FA_ERR_UNSUPPORTED;
    sh->B = B;
    sh->Hq = Hq;
    sh->Hkv = Hkv;
    sh->Tq = Tq;
    sh->Tk = Tk;
    sh->d = d;
    sh->causal = causal;
    sh->window = window;
    sh->BHq = (int)bhq;
    sh->BHkv = (int)bhkv;
    return FA_OK;
}

// Backward workspace: two 16-byte fold records per (padded) query row, the fp32 dQ
// accumulator, then a 256-byte tail holding the main kernel's unit counter.
constexpr size_t kSchedBytes = 256;
size_t workspace_bytes(long long bhq, long long tq, int d) {
    const size_t npad = ((size_t)tq + 127) / 128 * 128;
    return 2 * (size_t)bhq * npad * 16u + (size_t)bhq * npad * (size_t)d * sizeof(float) +
           kSchedBytes;
}

constexpr float kLog2e = 1.4426950408889634074f;

// Workspace of fa_backward_noalloc: one array per device that loads the library, kept for
// the life of the process. Host code must not use its name as an address (it is a host-side
// stand-in); the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device, looked up once per device.
fa_status get_noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e);
        if (p == nullptr) return cuda_fail(cudaErrorInvalidSymbol);
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return FA_OK;
}

// Diagnostic: one warp waits, through the attention kernels' bounded wait, on an mbarrier that
// nothing ever arrives on; the wait gives up after limit_ns, records kDevTimeoutLoad in the error
// word and the kernel returns.
__global__ void fa_wait_selftest_kernel(int* err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        fa::ptx::mbar_init(fa::ptx::smem_addr(&bar), 1);
        abort_flag = 0;
        fa::ptx::fence_barrier_init();
    }
    __syncthreads();
    fa::warp_wait(fa::ptx::smem_addr(&bar), 0, &abort_flag, err, fa::kDevTimeoutLoad, limit_ns);
}

// Query heads of a KV head packed into one block of group * Tq query rows (forward only): for
// short query blocks (decode, short chunks) a 128-row tile would otherwise carry at most Tq
// live rows, and every query head would stream its KV head's K and V on its own.
constexpr int kPackMaxTq = 64;
bool pack_heads(int Hq, int Hkv, int Tq) { return Hkv > 0 && Hq > Hkv && Tq <= kPackMaxTq; }

// ---- host-buffer step (fa_forward_backward_host) ----------------------------------------

// Streams and events of the host-buffer step, created once per device and reused; g_host_mu is
// held while a step is enqueued, so reusing the events is safe (a stream wait takes the state of
// the event's latest record at the time of the wait call).
struct HostStepRes {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr, comp[2] = {nullptr, nullptr};
    cudaEvent_t entry = nullptr, done = nullptr;
    cudaEvent_t in_fwd[FA_MAX_HOST_CHUNKS] = {};   // a chunk's Q, K, V landed
    cudaEvent_t in_done[FA_MAX_HOST_CHUNKS] = {};  // and its dO
    cudaEvent_t fwd_done[FA_MAX_HOST_CHUNKS] = {};
    cudaEvent_t comp_done[FA_MAX_HOST_CHUNKS] = {};
};
std::mutex g_host_mu;
HostStepRes g_host_res[kMaxDevices];

fa_status host_step_resources(HostStepRes** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    HostStepRes& r = g_host_res[dev];
    if (!r.ready) {
        cudaStream_t* ss[4] = {&r.in, &r.out, &r.comp[0], &r.comp[1]};
        for (cudaStream_t* sp : ss)
            if ((e = cudaStreamCreateWithFlags(sp, cudaStreamNonBlocking)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaEventCreateWithFlags(&r.entry, cudaEventDisableTiming)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaEventCreateWithFlags(&r.done, cudaEventDisableTiming)) != cudaSuccess) return cuda_fail(e);
        for (int c = 0; c < FA_MAX_HOST_CHUNKS; ++c) {
            if ((e = cudaEventCreateWithFlags(&r.in_fwd[c], cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail(e);
            if ((e = cudaEventCreateWithFlags(&r.in_done[c], cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail(e);
            if ((e = cudaEventCreateWithFlags(&r.fwd_done[c], cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail(e);
            if ((e = cudaEventCreateWithFlags(&r.comp_done[c], cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail(e);
        }
        r.ready = true;
    }
    *out = &r;
    return FA_OK;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// First KV head of chunk c (of nch, nearly equal shares) over nkv heads.
int chunk_start(int c, int nch, int nkv) { return (int)((long long)nkv * c / nch); }

// Chunks of the host-buffer step and its device layout: the device copies of every tensor at
// full size, then one backward workspace per compute stream, sized for the largest chunk.
struct HostPlan {
    int nch, group, kv_per_chunk_max;
    size_t q_bytes, kv_bytes, lse_bytes, ws_bytes;
    size_t off_q, off_k, off_v, off_do, off_o, off_lse, off_dq, off_dk, off_dv, off_ws, total;
};

HostPlan host_plan(const Shape& sh, int nchunks) {
    HostPlan p;
    const int nkv = sh.BHkv;
    int n = nchunks == 0 ? 4 : nchunks;
    p.nch = std::max(1, std::min(n, std::max(1, nkv)));
    p.group = sh.Hkv > 0 ? sh.Hq / sh.Hkv : 1;
    p.kv_per_chunk_max = 0;
    for (int c = 0; c < p.nch; ++c)
        p.kv_per_chunk_max = std::max(p.kv_per_chunk_max, chunk_start(c + 1, p.nch, nkv) - chunk_start(c, p.nch, nkv));
    p.q_bytes = (size_t)sh.BHq * (size_t)sh.Tq * (size_t)sh.d * 2u;
    p.kv_bytes = (size_t)sh.BHkv * (size_t)sh.Tk * (size_t)sh.d * 2u;
    p.lse_bytes = (size_t)sh.BHq * (size_t)sh.Tq * sizeof(float);
    p.ws_bytes = workspace_bytes((long long)p.kv_per_chunk_max * p.group, sh.Tq, sh.d);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += round256(bytes);
        return o;
    };
    p.off_q = take(p.q_bytes);
    p.off_k = take(p.kv_bytes);
    p.off_v = take(p.kv_bytes);
    p.off_do = take(p.q_bytes);
    p.off_o = take(p.q_bytes);
    p.off_lse = take(p.lse_bytes);
    p.off_dq = take(p.q_bytes);
    p.off_dk = take(p.kv_bytes);
    p.off_dv = take(p.kv_bytes);
    p.off_ws = take(2 * round256(p.ws_bytes));
    p.total = off;
    return p;
}

}  // namespace

extern "C" {

const char* fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_ALIGNMENT: return "FA_ERR_ALIGNMENT";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    }
    return "FA_ERR_UNKNOWN";
}

int fa_last_cuda_error(void) { return t_last_cuda_error; }

// Split-KV workspace: nsplit partial O (fp32 [B*Hq, Tq, d]) then nsplit partial LSE
// (fp32 [B*Hq, Tq]), each part 256-byte aligned.
static size_t splitkv_bytes(long long bhq, long long tq, int d, int nsplit, size_t* lse_off) {
    const size_t rows = (size_t)bhq * (size_t)tq * (size_t)nsplit;
    const size_t o_bytes = (rows * (size_t)d * sizeof(float) + 255) / 256 * 256;
    if (lse_off) *lse_off = o_bytes;
    return o_bytes + (rows * sizeof(float) + 255) / 256 * 256;
}

size_t fa_forward_splitkv_workspace_bytes(int B, int Hq, int Tq, int d, int nsplit) {
    if (B <= 0 || Hq <= 0 || Tq <= 0 || (d != 64 && d != 128) || nsplit < 2 ||
        nsplit > FA_MAX_SPLITS)
        return 0;
    return splitkv_bytes((long long)B * Hq, Tq, d, nsplit, nullptr);
}

int fa_forward_choose_splits(int B, int Hq, int Hkv, int Tq, int Tk, int num_sms) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Tq <= 0 || Tk <= 0 || num_sms <= 0 || Hq % Hkv != 0)
        return 1;
    // Cost model in 128-key tile steps (fitted to GB300 timings of decode and chunked-prefill
    // shapes): n splits run ceil(units * n / SMs) rounds of units costing ceil(tiles / n)
    // steps plus a fixed cost per unit (Q load, epilogue, partial writes: ~2 steps for a
    // single live query row, ~5.5 for a full 256-row block), and the merge adds ~2. A split is
    // taken only when it beats the unsplit launch by 10 %; among equal costs the fewest win.
    // Rounds are counted against 85 % of the SMs: on decode shapes the fastest split launch
    // had ~128 units for 152 SMs (8 packed blocks: 16 splits 31 us, 19 splits 36 us).
    const long long sms = std::max(1LL, (long long)num_sms * 85 / 100);
    const bool packed = pack_heads(Hq, Hkv, Tq);
    const long long rows = packed ? (long long)(Hq / Hkv) * Tq : Tq;
    const long long units = (rows + 255) / 256 * (long long)B * (packed ? Hkv : Hq);
    const long long tiles = ((long long)Tk + 127) / 128;
    if (tiles <= 1) return 1;
    const double fixed = 2.0 + 3.5 * (double)std::min<long long>(rows, 256) / 256.0;
    const double merge = 2.0;
    const double unsplit = (double)((units + sms - 1) / sms) * ((double)tiles + fixed);
    int best_n = 1;
    double best = 0.0;
    for (int n = 2; n <= FA_MAX_SPLITS && n <= tiles; ++n) {
        const double rounds = (double)((units * n + sms - 1) / sms);
        const double c = rounds * ((double)((tiles + n - 1) / n) + fixed) + merge;
        if (best_n == 1 || c < best) {
            best_n = n;
            best = c;
        }
    }
    return (best_n > 1 && best < 0.9 * unsplit) ? best_n : 1;
}

fa_status fa_forward_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int Hq, int Hkv, int Tq, int Tk, int d, int causal,
                             int window, float scale, int nsplit, void* workspace,
                             struct CUstream_st* stream) {
    if (nsplit < 1 || nsplit > FA_MAX_SPLITS) return FA_ERR_INVALID_ARG;
    Shape sh;
    bool empty = false;
    fa_status st = check_shape(B, Hq, Hkv, Tq, Tk, d, causal, window, scale, &sh, &empty);
    if (st != FA_OK || empty) return st;
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
        return FA_ERR_ALIGNMENT;
    if (nsplit > 1 && workspace && !aligned(workspace, 256)) return FA_ERR_ALIGNMENT;
    // With packed heads the kernel sees B*Hkv heads of group*Tq rows each: the same memory,
    // since a KV head's query heads are adjacent in [B*Hq, Tq, d] (and in LSE [B*Hq, Tq]).
    const bool packed = pack_heads(Hq, Hkv, Tq);
    const int rows = packed ? (Hq / Hkv) * Tq : Tq;
    const int heads = packed ? sh.BHkv : sh.BHq;
    if (((long long)rows + 255) / 256 * heads * nsplit > INT_MAX) return FA_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = bind_context()) != FA_OK) return st;
    fa::FwdLaunch a;
    std::memset(&a, 0, sizeof a);
    if ((st = make_map(&a.tm_q, q, heads, rows, d, 128)) != FA_OK) return st;
    if ((st = make_map(&a.tm_o, o, heads, rows, d, 128)) != FA_OK) return st;
    if ((st = make_map(&a.tm_k, k, sh.BHkv, Tk, d, 128)) != FA_OK) return st;
    if ((st = make_map(&a.tm_v, v, sh.BHkv, Tk, d, 128)) != FA_OK) return st;
    if ((st = get_err_ptr(&a.err)) != FA_OK) return st;
    if ((st = get_num_sms(&a.num_sms)) != FA_OK) return st;
    a.Tq = rows;
    a.tq_pos = Tq;
    a.Tk = Tk;
    a.Hq = packed ? Hkv : Hq;
    a.Hkv = Hkv;
    a.BHq = heads;
    a.window = window;
    a.c = scale * kLog2e;
    a.lse = lse;
    a.o = o;
    a.nsplit = nsplit;
    void* ws = workspace;
    bool owned = false;
    if (nsplit > 1) {
        size_t lse_off = 0;
        const size_t bytes = splitkv_bytes(sh.BHq, Tq, d, nsplit, &lse_off);
        if (!ws) {
            cudaError_t e = cudaMallocAsync(&ws, bytes, s);
            if (e != cudaSuccess) return cuda_fail(e);
            owned = true;
        }
        a.part_o = static_cast<float*>(ws);
        a.part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + lse_off);
    }
    cudaError_t e = fa::launch_forward(a, d, causal != 0, s);
    if (owned) {
        cudaError_t e2 = cudaFreeAsync(ws, s);
        if (e == cudaSuccess) e = e2;
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
}

fa_status fa_forward_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int Hq, int Hkv, int Tq, int Tk, int d, int causal, int window,
                        float scale, struct CUstream_st* stream) {
    return fa_forward_splitkv(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, causal, window, scale, 1,
                              nullptr, stream);
}

fa_status fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int d, int causal, float scale, struct CUstream_st* stream) {
    return fa_forward_ex(q, k, v, o, lse, B, H, H, N, N, d, causal, -1, scale, stream);
}

size_t fa_backward_workspace_bytes(int B, int H, int N, int d) {
    if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128)) return 0;
    return workspace_bytes((long long)B * H, N, d);
}

fa_status fa_backward_ex(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                         int Hq, int Hkv, int Tq, int Tk, int d, int causal, int window,
                         float scale, void* workspace, struct CUstream_st* stream) {
    Shape sh;
    bool empty = false;
    fa_status st = check_shape(B, Hq, Hkv, Tq, Tk, d, causal, window, scale, &sh, &empty);
    if (st != FA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (empty) {
        // No query rows: every key gets zero gradient.
        const size_t kv_bytes = (size_t)sh.BHkv * (size_t)Tk * (size_t)d * 2u;
        if (kv_bytes == 0) return FA_OK;
        if (!dk || !dv) return FA_ERR_INVALID_ARG;
        cudaError_t e = cudaMemsetAsync(dk, 0, kv_bytes, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, kv_bytes, s);
        if (e != cudaSuccess) return cuda_fail(e);
        return FA_OK;
    }
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
        !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
        !aligned(lse, 4))
        return FA_ERR_ALIGNMENT;
    if (workspace && !aligned(workspace, 256)) return FA_ERR_ALIGNMENT;
    const int Npad = (Tq + 127) / 128 * 128;
    if ((st = bind_context()) != FA_OK) return st;
    fa::BwdLaunch a;
    std::memset(&a, 0, sizeof a);
    const int q_rows = (d == 128) ? 64 : 128;  // query rows per backward step
    if ((st = make_map(&a.tm_q, q, sh.BHq, Tq, d, q_rows)) != FA_OK) return st;
    if ((st = make_map(&a.tm_do, dout, sh.BHq, Tq, d, q_rows)) != FA_OK) return st;
    if ((st = make_map(&a.tm_k, k, sh.BHkv, Tk, d, 128)) != FA_OK) return st;
    if ((st = make_map(&a.tm_v, v, sh.BHkv, Tk, d, 128)) != FA_OK) return st;
    if ((st = make_map(&a.tm_dk, dk, sh.BHkv, Tk, d, 128)) != FA_OK) return st;
    if ((st = make_map(&a.tm_dv, dv, sh.BHkv, Tk, d, 128)) != FA_OK) return st;
    if ((st = get_err_ptr(&a.err)) != FA_OK) return st;
    if ((st = get_num_sms(&a.num_sms)) != FA_OK) return st;
    const size_t ws_bytes = workspace_bytes(sh.BHq, Tq, d);
    void* ws = workspace;
    bool owned = false;
    if (!ws) {
        cudaError_t e = cudaMallocAsync(&ws, ws_bytes, s);
        if (e != cudaSuccess) return cuda_fail(e);
        owned = true;
    }
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    a.dq = dq;
    a.folds = ws;
    a.dq_acc = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + 2 * (size_t)sh.BHq * (size_t)Npad * 16u);
    a.sched = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(ws) + ws_bytes - kSchedBytes);
    // dQ accumulator: [B*Hq, Npad, d] at d = 64; at d = 128 the main kernel computes dQ
    // transposed and accumulates it as [B*Hq, d, Npad] (boxes of 32 queries x 128 rows).
    st = (d == 128) ? make_map(&a.tm_dqacc, a.dq_acc, sh.BHq, d, Npad, 128, true)
                    : make_map(&a.tm_dqacc, a.dq_acc, sh.BHq, Npad, d, q_rows, true);
    if (st != FA_OK) {
        if (owned) cudaFreeAsync(ws, s);
        return st;
    }
    a.Tq = Tq;
    a.Tk = Tk;
    a.Npad = Npad;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.BHq = sh.BHq;
    a.BHkv = sh.BHkv;
    a.d = d;
    a.window = window;
    a.scale = scale;
    a.c = scale * kLog2e;
    cudaError_t e = fa::launch_backward(a, causal != 0, s);
    if (owned) {
        cudaError_t e2 = cudaFreeAsync(ws, s);
        if (e == cudaSuccess) e = e2;
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
}

fa_status fa_backward(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                      int H, int N, int d, int causal, float scale, void* workspace,
                      struct CUstream_st* stream) {
    return fa_backward_ex(q, k, v, o, lse, dout, dq, dk, dv, B, H, H, N, N, d, causal, -1, scale,
                          workspace, stream);
}

fa_status fa_backward_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, int causal, float scale,
                              struct CUstream_st* stream) {
    Shape sh;
    bool empty = false;
    fa_status st = check_shape(B, H, H, N, N, d, causal, -1, scale, &sh, &empty);
    if (st != FA_OK || empty) return st;
    if (fa_backward_workspace_bytes(B, H, N, d) > (size_t)FA_NOALLOC_SCRATCH_BYTES)
        return FA_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if ((st = get_noalloc_scratch(&scratch)) != FA_OK) return st;
    return fa_backward(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, causal, scale, scratch,
                       stream);
}

size_t fa_noalloc_scratch_bytes(void) { return (size_t)FA_NOALLOC_SCRATCH_BYTES; }

fa_status fa_naive_softmax(const float* s, void* p, float* lse, long long rows, int N, int causal,
                           float scale, struct CUstream_st* stream) {
    if (rows < 0 || N < 0 || (causal != 0 && causal != 1)) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (rows == 0 || N == 0) return FA_OK;
    if (!s || !p || !lse) return FA_ERR_INVALID_ARG;
    if (!aligned(s, 4) || !aligned(p, 2) || !aligned(lse, 4)) return FA_ERR_ALIGNMENT;
    fa_status st = bind_context();
    if (st != FA_OK) return st;
    cudaError_t e = fa::launch_naive_softmax(s, p, lse, rows, N, causal, scale,
                                             reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

fa_status fa_selftest_wait_timeout(unsigned int limit_us, struct CUstream_st* stream) {
    if (limit_us == 0 || limit_us > 1000000u) return FA_ERR_INVALID_ARG;
    int* err = nullptr;
    fa_status st = get_err_ptr(&err);
    if (st != FA_OK) return st;
    fa_wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        err, (unsigned long long)limit_us * 1000ull);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
}

size_t fa_forward_backward_host_device_bytes(int B, int Hq, int Hkv, int Tq, int Tk, int d,
                                             int nchunks) {
    if (nchunks < 0 || nchunks > FA_MAX_HOST_CHUNKS) return 0;
    Shape sh;
    bool empty = false;
    // the shape rules of the device calls (causal = 0 accepts every Tq / Tk pairing)
    if (check_shape(B, Hq, Hkv, Tq, Tk, d, 0, -1, 1.0f, &sh, &empty) != FA_OK) return 0;
    return host_plan(sh, nchunks).total;
}

fa_status fa_forward_backward_host(const void* q, const void* k, const void* v, const void* dout,
                                   void* o, float* lse, void* dq, void* dk, void* dv, int B,
                                   int Hq, int Hkv, int Tq, int Tk, int d, int causal, int window,
                                   float scale, int nchunks, void* device_buffer,
                                   struct CUstream_st* stream) {
    if (nchunks < 0 || nchunks > FA_MAX_HOST_CHUNKS) return FA_ERR_INVALID_ARG;
    Shape sh;
    bool empty = false;
    fa_status st = check_shape(B, Hq, Hkv, Tq, Tk, d, causal, window, scale, &sh, &empty);
    if (st != FA_OK) return st;
    const HostPlan p = host_plan(sh, nchunks);
    if (p.q_bytes > 0 && (!q || !dout || !o || !lse || !dq)) return FA_ERR_INVALID_ARG;
    if (p.kv_bytes > 0 && (!k || !v || !dk || !dv)) return FA_ERR_INVALID_ARG;
    if (p.q_bytes == 0 && p.kv_bytes == 0) return FA_OK;
    if (device_buffer && !aligned(device_buffer, 256)) return FA_ERR_INVALID_ARG;
    if ((st = bind_context()) != FA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lk(g_host_mu);
    HostStepRes* r = nullptr;
    if ((st = host_step_resources(&r)) != FA_OK) return st;
    uint8_t* buf = static_cast<uint8_t*>(device_buffer);
    bool owned = false;
    cudaError_t e = cudaSuccess;
    if (!buf) {
        void* m = nullptr;
        if ((e = cudaMallocAsync(&m, p.total, s)) != cudaSuccess) return cuda_fail(e);
        buf = static_cast<uint8_t*>(m);
        owned = true;
    }
    // Every failure past this point still joins the internal streams back into `stream`, so
    // that nothing queued here outlives a buffer the caller or the library frees afterwards.
    fa_status result = FA_OK;
    auto fail = [&](cudaError_t err) {
        if (result == FA_OK) result = cuda_fail(err);
    };
    if ((e = cudaEventRecord(r->entry, s)) != cudaSuccess) {
        if (owned) cudaFreeAsync(buf, s);
        return cuda_fail(e);
    }
    cudaStream_t all[4] = {r->in, r->out, r->comp[0], r->comp[1]};
    for (cudaStream_t x : all)
        if ((e = cudaStreamWaitEvent(x, r->entry, 0)) != cudaSuccess) fail(e);

    const size_t qrow = (size_t)Tq * d * 2u, krow = (size_t)Tk * d * 2u, lrow = (size_t)Tq * 4u;
    const uint8_t* hq = static_cast<const uint8_t*>(q);
    const uint8_t* hk = static_cast<const uint8_t*>(k);
    const uint8_t* hv = static_cast<const uint8_t*>(v);
    const uint8_t* hdo = static_cast<const uint8_t*>(dout);
    auto kv0_of = [&](int c) { return chunk_start(c, p.nch, sh.BHkv); };
    // copies in
    for (int c = 0; c < p.nch && result == FA_OK; ++c) {
        const size_t h0 = (size_t)kv0_of(c), h1 = (size_t)kv0_of(c + 1);
        const size_t g0 = h0 * p.group, g1 = h1 * p.group;
        const struct { size_t off; const uint8_t* src; size_t row, a, b; } cp[4] = {
            {p.off_q, hq, qrow, g0, g1}, {p.off_k, hk, krow, h0, h1},
            {p.off_v, hv, krow, h0, h1}, {p.off_do, hdo, qrow, g0, g1}};
        for (int i = 0; i < 4; ++i) {
            const auto& x = cp[i];
            const size_t bytes = (x.b - x.a) * x.row;
            if (bytes > 0) {
                e = cudaMemcpyAsync(buf + x.off + x.a * x.row, x.src + x.a * x.row, bytes,
                                    cudaMemcpyHostToDevice, r->in);
                if (e != cudaSuccess) fail(e);
            }
            // the forward needs Q, K, V only; dO (last) is for the backward
            if (i == 2 && (e = cudaEventRecord(r->in_fwd[c], r->in)) != cudaSuccess) fail(e);
        }
        if ((e = cudaEventRecord(r->in_done[c], r->in)) != cudaSuccess) fail(e);
    }
    // kernels: chunk c on compute stream c % 2, with that stream's workspace
    for (int c = 0; c < p.nch && result == FA_OK; ++c) {
        const int h0 = kv0_of(c), h1 = kv0_of(c + 1);
        const int nkv = h1 - h0, nq = nkv * p.group;
        cudaStream_t cs = r->comp[c & 1];
        if ((e = cudaStreamWaitEvent(cs, r->in_fwd[c], 0)) != cudaSuccess) {
            fail(e);
            break;
        }
        const size_t g0 = (size_t)h0 * p.group;
        uint8_t* ws = buf + p.off_ws + (size_t)(c & 1) * round256(p.ws_bytes);
        CUstream_st* csx = reinterpret_cast<CUstream_st*>(cs);
        // A chunk is the flattened [B*H] layout cut along heads: batch 1 with nq query heads
        // over nkv KV heads keeps query head j on KV head j / group.
        fa_status st2 = fa_forward_ex(buf + p.off_q + g0 * qrow, buf + p.off_k + h0 * krow,
                                      buf + p.off_v + h0 * krow, buf + p.off_o + g0 * qrow,
                                      reinterpret_cast<float*>(buf + p.off_lse + g0 * lrow), 1, nq,
                                      nkv, Tq, Tk, d, causal, window, scale, csx);
        if (st2 == FA_OK && (e = cudaEventRecord(r->fwd_done[c], cs)) != cudaSuccess) fail(e);
        if (st2 == FA_OK && (e = cudaStreamWaitEvent(cs, r->in_done[c], 0)) != cudaSuccess) fail(e);
        if (st2 == FA_OK && result == FA_OK)
            st2 = fa_backward_ex(buf + p.off_q + g0 * qrow, buf + p.off_k + h0 * krow,
                                 buf + p.off_v + h0 * krow, buf + p.off_o + g0 * qrow,
                                 reinterpret_cast<const float*>(buf + p.off_lse + g0 * lrow),
                                 buf + p.off_do + g0 * qrow, buf + p.off_dq + g0 * qrow,
                                 buf + p.off_dk + h0 * krow, buf + p.off_dv + h0 * krow, 1, nq, nkv,
                                 Tq, Tk, d, causal, window, scale, ws, csx);
        if (st2 != FA_OK) {
            result = st2;
            break;
        }
        if ((e = cudaEventRecord(r->comp_done[c], cs)) != cudaSuccess) fail(e);
    }
    // copies out: O and LSE once the chunk's forward is done, the gradients after its backward
    uint8_t* ho = static_cast<uint8_t*>(o);
    uint8_t* hl = reinterpret_cast<uint8_t*>(lse);
    uint8_t* hdq = static_cast<uint8_t*>(dq);
    uint8_t* hdk = static_cast<uint8_t*>(dk);
    uint8_t* hdv = static_cast<uint8_t*>(dv);
    for (int c = 0; c < p.nch && result == FA_OK; ++c) {
        const size_t h0 = (size_t)kv0_of(c), h1 = (size_t)kv0_of(c + 1);
        const size_t g0 = h0 * p.group, g1 = h1 * p.group;
        const struct { size_t off; uint8_t* dst; size_t row, a, b; } cp[5] = {
            {p.off_o, ho, qrow, g0, g1}, {p.off_lse, hl, lrow, g0, g1}, {p.off_dq, hdq, qrow, g0, g1},
            {p.off_dk, hdk, krow, h0, h1}, {p.off_dv, hdv, krow, h0, h1}};
        for (int i = 0; i < 5 && result == FA_OK; ++i) {
            if (i == 0 || i == 2) {
                cudaEvent_t ev = (i == 0) ? r->fwd_done[c] : r->comp_done[c];
                if ((e = cudaStreamWaitEvent(r->out, ev, 0)) != cudaSuccess) {
                    fail(e);
                    break;
                }
            }
            const auto& x = cp[i];
            const size_t bytes = (x.b - x.a) * x.row;
            if (bytes == 0) continue;
            e = cudaMemcpyAsync(x.dst + x.a * x.row, buf + x.off + x.a * x.row, bytes,
                                cudaMemcpyDeviceToHost, r->out);
            if (e != cudaSuccess) fail(e);
        }
    }
    // join: every internal stream's work is done before later work on `stream`
    for (cudaStream_t x : all) {
        if ((e = cudaEventRecord(r->done, x)) != cudaSuccess) fail(e);
        if ((e = cudaStreamWaitEvent(s, r->done, 0)) != cudaSuccess) fail(e);
    }
    if (owned && (e = cudaFreeAsync(buf, s)) != cudaSuccess) fail(e);
    return result;
}

fa_status fa_device_error(struct CUstream_st* stream, int* code) {
    if (!code) return FA_ERR_INVALID_ARG;
    *code = 0;
    int* p = nullptr;
    fa_status st = get_err_ptr(&p);
    if (st != FA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    int h = 0;
    e = cudaMemcpy(&h, p, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    if (h != 0) {
        const int zero = 0;
        e = cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    *code = h;
    return h ? FA_ERR_TIMEOUT : FA_OK;
}

}  // extern "C"
