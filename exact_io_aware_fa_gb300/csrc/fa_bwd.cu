// fa_bwd.cu -- exact attention backward for sm_103a, by recomputation from the saved LSE.
//
// Method ("FlashAttention: from IO-Aware Attention to GPU work partitioning",
// blog.euler0525.cn, sections "Tiling、Fusion 与 Backward Recomputation",
// "FlashAttention-2" and "Sequence Parallelism"):
//   P_ij = exp(S_ij - L_i) rebuilt tile by tile from Q, K and the saved L = LSE;
//   dV = P^T dO,  dP = dO V^T,  D_i = O_i . dO_i,  dS = P (.) (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q  (the scale factors follow from S = scale Q K^T).
//   Work is partitioned over key tiles (column-oriented): a work unit is one 128-key tile
//   K_j, V_j of one KV head and its dK_j, dV_j, summed over every query head that reads the
//   KV head (grouped heads) and over the query steps that can see the tile (query offset,
//   causal diagonal, sliding window); contributions to dQ from different key tiles are added
//   in fp32 with (bulk) atomic reductions. The main kernel is persistent: one CTA per SM
//   takes units from an atomic counter until none are left.
//
// Three kernels:
//   fa_bwd_pre_kernel   D_i = sum_e dO_ie O_ie; per query row the fold records of -LSE/scale
//                       and -D (exact three-part bf16 sums); dQ accumulator zeroed.
//   fa_bwd_kernel<D>    per unit (key tile): loop over query steps:
//                       S'^T = K Q_i^T + fold and dP'^T = V dO_i^T + fold (tcgen05, TMEM; the
//                       fold MMA against a ones tile subtracts LSE and D inside the MMA);
//                       P^T = exp2(c S'^T) (to TMEM) and dS^T = P^T (.) dP'^T (to smem) by two
//                       compute warpgroups, one thread per key row; dV += P^T dO_i (A from
//                       TMEM), dK += dS^T Q_i (A from smem), the dQ_i partial (A/B from smem)
//                       drained from TMEM by a third warpgroup and added into the fp32 dQ
//                       accumulator with a TMA bulk reduce-add. The next step's S'^T/dP'^T
//                       are issued as soon as the compute warps have read the current ones, so
//                       they overlap dV/dK/dQ of this step; Q/dO ring 3 deep. dV and scale*dK
//                       leave through the drain warps while the next unit starts.
//   fa_bwd_dq_kernel    dQ = bf16(scale * dQacc).
//
// d = 128: query steps of 64 rows, the dQ partial computed transposed (dQ^T = K^T dS^T,
//          M = d = 128) so its TMEM lanes are head-dim columns.
// d = 64:  query steps of 128 rows, dQ = dS K with M = 128 query rows.
#include <algorithm>

#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {
namespace {

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
}

// ----------------------------------------------------------------------------------------
// Preprocess: D/8 threads per row, 16-byte loads; 256 threads cover 2048/D rows.
//
// Per query row it writes two "fold" records that let the main kernel's MMAs subtract the row
// statistics themselves: S'^T = K Q^T + 1 * (-LSE/scale) and dP'^T = V dO^T + 1 * (-D), added as
// one more K=16 MMA against a constant tile of ones. A record is 8 bf16 (16 bytes): the value
// split exactly into three bf16 parts (hi + mid + lo) at k = 0, 1, 2, zeros at k = 3..7.
// Consecutive rows' records are 16 bytes apart, which is the tcgen05 no-swizzle K-major layout
// of an 8-wide K slice (8-row core matrices of 16-byte rows, 8-row groups 128 bytes apart), so
// one bulk copy of a query block's records lands in shared memory ready for the MMA.
// ----------------------------------------------------------------------------------------
// Exact three-part bf16 split of v: hi = bf16(v), mid = bf16(v - hi), lo = v - hi - mid (each
// difference is exact in fp32, and lo has at most 8 significant bits).
__device__ __forceinline__ uint4 fold_record(float v) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
    uint4 w;
    w.x = (uint32_t)__bfloat16_as_ushort(hi) | ((uint32_t)__bfloat16_as_ushort(mid) << 16);
    w.y = (uint32_t)__bfloat16_as_ushort(lo);
    w.z = 0u;
    w.w = 0u;
    return w;
}

// Byte offset of row n's record in a fold array: 16 bytes per row, rows contiguous.
__device__ __forceinline__ size_t fold_offset(size_t bh, int Npad, int n) {
    return (bh * (size_t)Npad + (size_t)n) * 16u;
}

template <int D>
__global__ void __launch_bounds__(256)
fa_bwd_pre_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                  const float* __restrict__ lse, uint8_t* __restrict__ folds,
                  float* __restrict__ dq_acc, unsigned* __restrict__ sched, int N, int Npad, int BH,
                  float inv_scale) {
    constexpr int TPR = D / 8;            // threads per row
    constexpr int RPB = 256 / TPR;        // rows per block
    // Launched as a dependent of whatever kernel precedes it (typically the forward): wait for
    // it before reading O, LSE, dO or touching the workspace. The main kernel may launch (and
    // run its prologue) once every block of this one has started; it waits for this kernel's
    // completion before reading anything it writes.
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    if (blockIdx.x == 0 && threadIdx.x == 0) *sched = 0u;  // the main kernel's unit counter
    const int sub = threadIdx.x % TPR;
    const long long row_global = (long long)blockIdx.x * RPB + threadIdx.x / TPR;  // over BH*Npad
    const bool valid_row = row_global < (long long)BH * Npad;
    const int bh = valid_row ? (int)(row_global / Npad) : 0;
    const int n = valid_row ? (int)(row_global % Npad) : 0;
    float dot = 0.f;
    if (valid_row && n < N) {
        const size_t base = ((size_t)bh * N + n) * D + sub * 8;
        const uint4 a = *reinterpret_cast<const uint4*>(o + base);
        const uint4 b = *reinterpret_cast<const uint4*>(dout + base);
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 fa = __bfloat1622float2(pa[i]);
            const float2 fb = __bfloat1622float2(pb[i]);
            dot = fmaf(fa.x, fb.x, dot);
            dot = fmaf(fa.y, fb.y, dot);
        }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    if (!valid_row) return;
    if (sub == 0) {
        // Padded rows get a large finite negative shift (their P must be 0; a finite value keeps
        // the zero products of the fold MMA free of 0 * inf).
        const float v = (n < N) ? -lse[(size_t)bh * N + n] * inv_scale : -0x1.0p100f;
        const size_t off = fold_offset((size_t)bh, Npad, n);
        uint8_t* lf = folds + off;
        uint8_t* df = folds + (size_t)BH * Npad * 16u + off;
        *reinterpret_cast<uint4*>(lf) = fold_record(v);
        *reinterpret_cast<uint4*>(df) = fold_record((n < N) ? -dot : 0.f);
    }
    float4* acc = reinterpret_cast<float4*>(dq_acc + ((size_t)bh * Npad + n) * D + sub * 8);
    acc[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ----------------------------------------------------------------------------------------
// dQ convert.
// ----------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256)
fa_bwd_dq_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq, int N, int Npad,
                 int BH, float scale) {
    ptx::griddep_wait();  // the main kernel's dQ sums (this kernel may launch during its tail)
    const long long idx8 = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // 8 elements each
    const long long total8 = (long long)BH * N * (D / 8);
    if (idx8 >= total8) return;
    const long long row = idx8 / (D / 8);
    const int col8 = (int)(idx8 % (D / 8));
    const int bh = (int)(row / N);
    const int n = (int)(row % N);
    const float4* src = reinterpret_cast<const float4*>(dq_acc + ((size_t)bh * Npad + n) * D + col8 * 8);
    const float4 a = src[0], b = src[1];
    uint4 w;
    w.x = ptx::pack_bf16x2(a.x * scale, a.y * scale);
    w.y = ptx::pack_bf16x2(a.z * scale, a.w * scale);
    w.z = ptx::pack_bf16x2(b.x * scale, b.y * scale);
    w.w = ptx::pack_bf16x2(b.z * scale, b.w * scale);
    *reinterpret_cast<uint4*>(dq + ((size_t)bh * N + n) * D + col8 * 8) = w;
}

// dQ convert for d = 128, whose main kernel accumulates dQ transposed, [B*H][d][Npad] (each
// drain thread then owns a contiguous row). A block transposes a tile of 64 queries x 128
// head-dim columns through shared memory: reads along the queries, writes bf16 rows.
__global__ void __launch_bounds__(256)
fa_bwd_dqt_kernel(const float* __restrict__ dq_acc_t, __nv_bfloat16* __restrict__ dq, int N,
                  int Npad, int tiles, float scale) {
    constexpr int D = 128, TQ = 64;
    __shared__ float tile[D][TQ + 1];
    ptx::griddep_wait();  // the main kernel's dQ sums (this kernel may launch during its tail)
    const int bh = (int)(blockIdx.x / (unsigned)tiles);
    const int n0 = (int)(blockIdx.x % (unsigned)tiles) * TQ;
    const float* src = dq_acc_t + (size_t)bh * D * Npad + n0;
#pragma unroll 4
    for (int i = 0; i < D * TQ / 256; ++i) {
        const int idx = i * 256 + (int)threadIdx.x;
        const int e = idx / TQ, q = idx % TQ;
        tile[e][q] = src[(size_t)e * Npad + q];  // n0 + q < Npad (Npad is a multiple of 128)
    }
    __syncthreads();
#pragma unroll 4
    for (int i = 0; i < D * TQ / 512; ++i) {
        const int idx = i * 256 + (int)threadIdx.x;
        const int q = idx / (D / 2), e = 2 * (idx % (D / 2));
        if (n0 + q < N)
            *reinterpret_cast<uint32_t*>(dq + ((size_t)bh * N + n0 + q) * D + e) =
                ptx::pack_bf16x2(tile[e][q] * scale, tile[e + 1][q] * scale);
    }
}

// ----------------------------------------------------------------------------------------
// Main backward kernel.
// ----------------------------------------------------------------------------------------
// Problem shape of the backward: as the forward (query head bh_q reads KV head bh_q / group,
// query row i at key position offset + i, optional window), seen from a key tile.
struct BwdShape {
    int Tq, Tk, Npad, Hq, Hkv, group, offset, window, BHq, BHkv, nkb;
    int kv_chunk;  // KV heads per chunk of the unit order (1: head by head)
};

template <int D>
struct BwdCfg {
    static constexpr int KT = 128;                    // keys per CTA
    static constexpr int BMQ = (D == 128) ? 64 : 128; // query rows per step
    static constexpr int NQS = 3;                     // Q/dO ring depth
    static constexpr int NDS = (D == 64) ? 2 : 1;     // dS buffers (shared memory allowing)
    static constexpr uint32_t KTILE = 128u * D * 2u;  // K or V tile bytes
    static constexpr uint32_t KCHUNK = 128u * 128u;   // 128 rows x 64 cols
    static constexpr uint32_t QTILE = (uint32_t)BMQ * D * 2u;
    static constexpr uint32_t QCHUNK = (uint32_t)BMQ * 128u;  // BMQ rows x 64 cols
    static constexpr uint32_t FOLD_BYTES = (uint32_t)BMQ * 16u;  // fold records of a query block
    // stage: [Q][dO][-LSE/scale fold][-D fold], padded to 1024
    static constexpr uint32_t STAGE_BYTES = ((2 * QTILE + 2 * FOLD_BYTES) + 1023u) / 1024u * 1024u;
    // dS tile: 128 key rows, BMQ queries contiguous per row, in 64-query (128-byte) regions
    static constexpr uint32_t DS_BYTES = (uint32_t)BMQ * 128u * 2u;
    static constexpr uint32_t DSREG = 128u * 128u;           // one 64-query region
    static constexpr uint32_t DQBOX = (uint32_t)BMQ * 128u;  // one 32-column fp32 box
    static constexpr uint32_t DQBOX_T = 128u * 128u;         // d = 128: 32 queries x 128 e rows
    // fp32 dQ staging: d=64 drains one box at a time through one box of staging (the shared
    // memory goes to the second dS buffer); d=128 stages all four boxes at once.
    static constexpr uint32_t DQS_BYTES = (D == 64) ? DQBOX : 2u * DQBOX_T;
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = OFF_K + KTILE;
    static constexpr uint32_t OFF_ST = OFF_V + KTILE;
    static constexpr uint32_t OFF_DS = OFF_ST + NQS * STAGE_BYTES;
    static constexpr uint32_t OFF_DQS = OFF_DS + NDS * DS_BYTES;
    static constexpr uint32_t OFF_ONES = OFF_DQS + DQS_BYTES;  // ones tile [128 keys x 16]
    static constexpr uint32_t OFF_BAR = OFF_ONES + 128u * 32u;
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + 512 + 1024;
    static_assert(NQS <= 3 && NDS >= 1 && NDS <= 2, "barrier arrays");
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
    static_assert(DQS_BYTES >= (uint32_t)(D / 64) * KCHUNK, "dV / dK epilogue staged in the dQ staging");
    static constexpr int THREADS = 512;
    // TMEM columns. d=128: dV[0,128) dK[128,256) S^T[256,320) dP^T[320,384) dQ^T[384,448)
    // P^T[448,480). d=64: dV[0,64) dK[64,128) S^T[128,256) dP^T[256,384) dQ[384,448) P^T[448,512).
    static constexpr uint32_t DV_COL = 0;
    static constexpr uint32_t DK_COL = (uint32_t)D;
    static constexpr uint32_t S_COL = 2u * D;
    static constexpr uint32_t DP_COL = S_COL + BMQ;
    static constexpr uint32_t DQ_COL = 384;
    static constexpr uint32_t PT_COL = 448;
};

struct BwdBars {
    uint64_t kv_full, kv_empty;       // per unit: K/V landed / every MMA reading them done
    uint64_t dkv_full, dkv_free;      // per unit: dV/dK final in TMEM / read by the epilogue
    uint64_t q_full[3], q_empty[3];
    uint64_t s_full, s_free, p_ready, mma_done;
    uint64_t ds_free[2];  // one per dS buffer (NDS <= 2)
    uint64_t dq_full, dq_free;
    uint64_t final_bar;
    uint64_t uid_full[4], uid_empty[4];  // unit-id ring: published by the producer, read by all
    int uid[4];
    uint32_t tmem_base;
    int abort_flag;
};

// One work unit: KV head bh_kv, keys [key0, key0 + 128). It visits every query head of the
// group and, for each, the query steps whose rows can see some key of the tile: from the causal
// diagonal (query position offset + q >= key) to the window's reach (position - window <= key).
// A tile no query sees has no steps and stores zero gradients. Unit order: the KV heads are cut
// into chunks of kv_chunk heads; chunk by chunk, and inside a chunk key tile by key tile. With
// one head per chunk the walk is head by head (neighbouring units share their query heads' Q/dO
// in L2, the best order when every unit costs the same); under a causal mask larger chunks put
// each chunk's costliest tiles (whose queries reach back to the diagonal) first and its cheapest
// last, so that the launch ends on short units, while a chunk's Q/dO still fits in L2.
struct BwdUnit {
    int bh_kv, key0, i0, i1, nsteps_g, nsteps, bhq_base;
};

template <int D, bool CAUSAL, bool WINDOW>
__device__ __forceinline__ BwdUnit bwd_unit(int u, const BwdShape& sh) {
    using C = BwdCfg<D>;
    BwdUnit w;
    const uint32_t per_chunk = (uint32_t)sh.kv_chunk * (uint32_t)sh.nkb;
    const uint32_t chunk = (uint32_t)u / per_chunk;
    const uint32_t r = (uint32_t)u - chunk * per_chunk;
    const uint32_t h0 = chunk * (uint32_t)sh.kv_chunk;
    const uint32_t hc = min((uint32_t)sh.kv_chunk, (uint32_t)sh.BHkv - h0);  // last chunk: fewer
    w.bh_kv = (int)(h0 + r % hc);
    const int kb = (int)(r / hc);
    w.key0 = kb * C::KT;
    const int nq_total = (sh.Tq + C::BMQ - 1) / C::BMQ;
    w.i0 = CAUSAL ? max(0, w.key0 - sh.offset) / C::BMQ : 0;
    w.i1 = nq_total - 1;
    if (WINDOW) {
        const int reach = w.key0 + C::KT - 1 + sh.window - sh.offset;  // last query seeing a key
        w.i1 = (reach < 0) ? -1 : min(w.i1, reach / C::BMQ);
    }
    w.nsteps_g = max(0, w.i1 - w.i0 + 1);
    w.nsteps = w.nsteps_g * sh.group;
    w.bhq_base = (w.bh_kv / sh.Hkv) * sh.Hq + (w.bh_kv % sh.Hkv) * sh.group;
    return w;
}

// Walks a unit's steps query head by query head of the group, each over query blocks i0 .. i1
// (no division per step).
struct StepCursor {
    int bhq, qi;
    __device__ __forceinline__ StepCursor(const BwdUnit& w) : bhq(w.bhq_base), qi(w.i0) {}
    __device__ __forceinline__ void next(const BwdUnit& w) {
        if (++qi > w.i1) {
            qi = w.i0;
            ++bhq;
        }
    }
};

// WINDOW (causal only): queries more than `window` positions past a key do not see it.
// Persistent: one CTA per SM walks units taken from a launch-wide counter; every step barrier
// counts steps over all of the CTA's units, so one unit's tail (last dQ drain, dV/dK epilogue)
// overlaps the next unit's first steps.
template <int D, bool CAUSAL, bool WINDOW>
__global__ void __launch_bounds__(512, 1)
fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
              const __grid_constant__ CUtensorMap tm_dqacc, const uint8_t* __restrict__ folds,
              const BwdShape sh, const int num_units, unsigned* __restrict__ sched,
              const float c, const float scale, int* err) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    static_assert(sizeof(BwdBars) <= 512, "barrier block");
    BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::OFF_BAR);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    constexpr int kUidReaders = 14;  // warps 1, 3, 4-11, 12-15 (one arrival per warp)
    if (tid == 0) {
        ptx::mbar_init(ptx::smem_addr(&bars->kv_full), 1);
        ptx::mbar_init(ptx::smem_addr(&bars->kv_empty), 2);   // both MMA-issuing warps
        ptx::mbar_init(ptx::smem_addr(&bars->dkv_full), 1);
        ptx::mbar_init(ptx::smem_addr(&bars->dkv_free), 128); // the epilogue warps' threads
        for (int s = 0; s < C::NQS; ++s) {
            ptx::mbar_init(ptx::smem_addr(&bars->q_full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&bars->q_empty[s]), 1);
        }
        ptx::mbar_init(ptx::smem_addr(&bars->s_full), 1);
        ptx::mbar_init(ptx::smem_addr(&bars->s_free), 256);
        ptx::mbar_init(ptx::smem_addr(&bars->p_ready), 256);
        ptx::mbar_init(ptx::smem_addr(&bars->mma_done), 1);
        for (int b = 0; b < C::NDS; ++b) ptx::mbar_init(ptx::smem_addr(&bars->ds_free[b]), 1);
        ptx::mbar_init(ptx::smem_addr(&bars->dq_full), 1);
        ptx::mbar_init(ptx::smem_addr(&bars->dq_free), 128);
        ptx::mbar_init(ptx::smem_addr(&bars->final_bar), 2);
        for (int i = 0; i < 4; ++i) {
            ptx::mbar_init(ptx::smem_addr(&bars->uid_full[i]), 1);
            ptx::mbar_init(ptx::smem_addr(&bars->uid_empty[i]), kUidReaders);
        }
        bars->abort_flag = 0;
        ptx::fence_barrier_init();
        ptx::tma_prefetch_desc(&tm_q);
        ptx::tma_prefetch_desc(&tm_k);
        ptx::tma_prefetch_desc(&tm_v);
        ptx::tma_prefetch_desc(&tm_do);
        ptx::tma_prefetch_desc(&tm_dk);
        ptx::tma_prefetch_desc(&tm_dv);
        ptx::tma_prefetch_desc(&tm_dqacc);
    }
    if (warp == 2) {
        ptx::tmem_alloc(ptx::smem_addr(&bars->tmem_base), 512);
        ptx::tmem_relinquish();
    }
    if (warp >= 4 && warp < 8) {
        // Ones tile [128 keys x 16], no-swizzle K-major: key r has 1 at k = 0, 1, 2 (the fold
        // records' three parts) and 0 elsewhere.
        const int r = tid - 128;
        uint8_t* row = smem + C::OFF_ONES + (uint32_t)(r / 8) * 256u + (uint32_t)(r % 8) * 16u;
        const uint32_t one = 0x3F80u;  // bf16 1.0
        *reinterpret_cast<uint4*>(row) = make_uint4(one | (one << 16), one, 0u, 0u);
        *reinterpret_cast<uint4*>(row + 128) = make_uint4(0u, 0u, 0u, 0u);
        ptx::fence_proxy_async_smem();
    }
    // The prologue above overlaps the preprocess kernel's last blocks (programmatic dependent
    // launch); the fold records, the zeroed dQ accumulator and the unit counter it writes are
    // read only after this wait. The dQ conversion may launch during this kernel's tail.
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tbase = __shfl_sync(0xffffffffu, bars->tmem_base, 0);
    volatile int* abort_flag = &bars->abort_flag;
    // Units are handed out dynamically: a CTA's first unit is its block index, each later one
    // the next from a launch-wide counter (taken by the producer when it starts the unit), so
    // CTAs that drew cheap units (causal tiles far from the diagonal) simply take more. The
    // producer publishes each unit id in a four-slot ring; every other role reads it.
    volatile int* uid_ring = bars->uid;
    // (warp-wide) the unit id of this CTA's ul-th unit, -1 past the end; ok = false on abort
    auto fetch_unit = [&](int ul, bool& ok) -> int {
        const int slot = ul & 3;
        ok = warp_wait(ptx::smem_addr(&bars->uid_full[slot]), (uint32_t)(ul >> 2) & 1u, abort_flag,
                       err, kDevTimeoutLoad);
        if (!ok) return -1;
        const int u = uid_ring[slot];
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&bars->uid_empty[slot]));
        return u;
    };

    const uint32_t s_k = ptx::smem_addr(smem + C::OFF_K);
    const uint32_t s_v = ptx::smem_addr(smem + C::OFF_V);
    const uint32_t s_st = ptx::smem_addr(smem + C::OFF_ST);
    const uint32_t s_ds = ptx::smem_addr(smem + C::OFF_DS);

    if (warp == 0) {
        // ================================ TMA producer ================================
        if (lane == 0) {
            const uint64_t pol_keep = ptx::l2_policy_evict_last();
            const uint32_t b_kv = ptx::smem_addr(&bars->kv_full);
            int g = 0;   // steps issued over all units
            int ul = 0;  // units started
            bool ok = true;
            for (;; ++ul) {
                // take and publish this CTA's next unit
                const int slot = ul & 3;
                if (ul >= 4 && !wait_phase(ptx::smem_addr(&bars->uid_empty[slot]),
                                           (uint32_t)((ul >> 2) - 1) & 1u, abort_flag, err,
                                           kDevTimeoutConsumer))
                    break;
                int u = (int)blockIdx.x;
                if (ul > 0) {
                    const unsigned t = atomicAdd(sched, 1u) + (unsigned)gridDim.x;
                    u = (t < (unsigned)num_units) ? (int)t : -1;
                }
                uid_ring[slot] = u;
                ptx::mbar_arrive(ptx::smem_addr(&bars->uid_full[slot]));
                if (u < 0) break;
                const BwdUnit w = bwd_unit<D, CAUSAL, WINDOW>(u, sh);
                // K/V of the previous unit stay until every MMA reading them has completed.
                if (ul > 0 && !wait_phase(ptx::smem_addr(&bars->kv_empty), (uint32_t)(ul - 1) & 1u,
                                          abort_flag, err, kDevTimeoutMma))
                    break;
                ptx::mbar_arrive_expect_tx(b_kv, 2 * C::KTILE);
                for (int ch = 0; ch < D / 64; ++ch) {
                    ptx::tma_load_3d(s_k + ch * C::KCHUNK, &tm_k, b_kv, ch * 64, w.key0, w.bh_kv);
                    ptx::tma_load_3d(s_v + ch * C::KCHUNK, &tm_v, b_kv, ch * 64, w.key0, w.bh_kv);
                }
                StepCursor cur(w);
                for (int si = 0; si < w.nsteps; ++si, ++g, cur.next(w)) {
                    const int st = g % C::NQS;
                    const uint32_t ph = (uint32_t)(g / C::NQS) & 1u;
                    if (!wait_phase(ptx::smem_addr(&bars->q_empty[st]), ph ^ 1u, abort_flag, err,
                                    kDevTimeoutConsumer)) {
                        ok = false;
                        break;
                    }
                    const int q0 = cur.qi * C::BMQ;
                    const int bhq = cur.bhq;
                    const uint32_t b_q = ptx::smem_addr(&bars->q_full[st]);
                    const uint32_t base = s_st + st * C::STAGE_BYTES;
                    ptx::mbar_arrive_expect_tx(b_q, 2 * C::QTILE + 2 * C::FOLD_BYTES);
                    for (int ch = 0; ch < D / 64; ++ch) {
                        ptx::tma_load_3d_hint(base + ch * C::QCHUNK, &tm_q, b_q, ch * 64, q0, bhq, pol_keep);
                        ptx::tma_load_3d_hint(base + C::QTILE + ch * C::QCHUNK, &tm_do, b_q, ch * 64, q0,
                                              bhq, pol_keep);
                    }
                    const uint8_t* lf = folds + ((size_t)bhq * (size_t)sh.Npad + (size_t)q0) * 16u;
                    const uint8_t* df = lf + (size_t)sh.BHq * sh.Npad * 16u;
                    ptx::bulk_load(base + 2 * C::QTILE, lf, C::FOLD_BYTES, b_q);
                    ptx::bulk_load(base + 2 * C::QTILE + C::FOLD_BYTES, df, C::FOLD_BYTES, b_q);
                }
                if (!ok) {
                    ++ul;  // this unit's K/V load was issued
                    break;
                }
            }
            // Every copy issued must have landed before the CTA exits: the last K/V load and
            // the last ring stages.
            if (ul > 0) drain_wait(b_kv, (uint32_t)(ul - 1) & 1u);
            for (int gi = max(0, g - C::NQS); gi < g; ++gi)
                drain_wait(ptx::smem_addr(&bars->q_full[gi % C::NQS]), (uint32_t)(gi / C::NQS) & 1u);
        }
    } else if (warp == 1 || warp == 3) {
        // ================================ MMA issuers =================================
        {  // whole warp; one elected lane issues
            constexpr uint32_t idesc_s = ptx::idesc_bf16(128, C::BMQ, false, false);  // S^T, dP^T
            constexpr uint32_t idesc_kv = ptx::idesc_bf16(128, D, false, true);       // dV, dK
            // dQ: d=128 -> dQ^T = K^T dS^T (M=d, N=BMQ); d=64 -> dQ = dS K (M=BMQ, N=d)
            constexpr uint32_t idesc_q = (D == 128) ? ptx::idesc_bf16(128, C::BMQ, true, true)
                                                    : ptx::idesc_bf16(128, D, true, true);
            // Descriptors built once, stepped by constant offsets per MMA (see the forward).
            const uint64_t k_kmaj = ptx::sdesc_sw128(s_k, 16, 1024);
            const uint64_t v_kmaj = ptx::sdesc_sw128(s_v, 16, 1024);
            const uint64_t k_mn = ptx::sdesc_sw128(s_k, C::KCHUNK, 1024);
            const uint64_t st_kmaj = ptx::sdesc_sw128(s_st, 16, 1024);
            const uint64_t st_mn = ptx::sdesc_sw128(s_st, C::QCHUNK, 1024);
            const uint64_t ds_kmaj = ptx::sdesc_sw128(s_ds, 16, 1024);
            const uint64_t ds_mn = ptx::sdesc_sw128(s_ds, C::DSREG, 1024);
            // fold MMAs: A = ones tile, B = a stage's fold records (both no-swizzle K-major)
            const uint64_t ones_d = ptx::sdesc_noswz(ptx::smem_addr(smem + C::OFF_ONES), 128, 256);
            // A fold record is one 16-byte core-matrix row (k = 0..7); LBO = 0 makes the second K
            // half read the same bytes, which the ones tile's zero second half cancels.
            const uint64_t fold_d = ptx::sdesc_noswz(s_st + 2 * C::QTILE, 0, 128);
            auto issue_s_dp = [&](int si) {
                const uint32_t st_off = (uint32_t)(si % C::NQS) * C::STAGE_BYTES;
                const uint64_t qd = ptx::sdesc_add(st_kmaj, st_off);
                const uint64_t dod = ptx::sdesc_add(st_kmaj, st_off + C::QTILE);
                if (ptx::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * C::KCHUNK + (kk & 3) * 32;
                    const uint32_t qoff = (kk >> 2) * C::QCHUNK + (kk & 3) * 32;
                    ptx::mma_ss(tbase + C::S_COL, ptx::sdesc_add(k_kmaj, koff), ptx::sdesc_add(qd, qoff),
                                idesc_s, kk > 0);
                }
                // S'^T = S^T + (-LSE/scale) per query column
                ptx::mma_ss(tbase + C::S_COL, ones_d, ptx::sdesc_add(fold_d, st_off), idesc_s, 1u);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * C::KCHUNK + (kk & 3) * 32;
                    const uint32_t qoff = (kk >> 2) * C::QCHUNK + (kk & 3) * 32;
                    ptx::mma_ss(tbase + C::DP_COL, ptx::sdesc_add(v_kmaj, koff), ptx::sdesc_add(dod, qoff),
                                idesc_s, kk > 0);
                }
                // dP'^T = dP^T + (-D) per query column
                ptx::mma_ss(tbase + C::DP_COL, ones_d,
                            ptx::sdesc_add(fold_d, st_off + C::FOLD_BYTES), idesc_s, 1u);
                ptx::mma_commit(ptx::smem_addr(&bars->s_full));
                }
                __syncwarp();
            };
            auto commit = [&](uint64_t* bar) {
                if (ptx::elect_one()) ptx::mma_commit(ptx::smem_addr(bar));
                __syncwarp();
            };
            // Two issuing warps (see the forward): warp 1 issues S^T/dP^T, warp 3 issues
            // dV/dK/dQ, so one warp's MMAs run while the other waits for operands. Both count
            // steps (g) and units (ul) over the CTA's whole walk.
            bool ok = true;
            int g = 0;
            int ul = 0;
            for (;; ++ul) {
                const int u = fetch_unit(ul, ok);
                if (!ok || u < 0) break;
                const BwdUnit w = bwd_unit<D, CAUSAL, WINDOW>(u, sh);
                ok = warp_wait(ptx::smem_addr(&bars->kv_full), (uint32_t)ul & 1u, abort_flag, err,
                               kDevTimeoutLoad);
                if (!ok) break;
                if (warp == 1) {
                    for (int si = 0; si < w.nsteps; ++si, ++g) {
                        // S'^T/dP'^T of step g once its Q/dO stage has landed and the compute warps
                        // have read step g - 1's.
                        const int st = g % C::NQS;
                        ok = warp_wait(ptx::smem_addr(&bars->q_full[st]), (uint32_t)(g / C::NQS) & 1u,
                                       abort_flag, err, kDevTimeoutLoad);
                        if (ok && g > 0)
                            ok = warp_wait(ptx::smem_addr(&bars->s_free), (uint32_t)(g - 1) & 1u,
                                           abort_flag, err, kDevTimeoutSoftmax);
                        if (!ok) break;
                        ptx::tc_fence_after();
                        issue_s_dp(g);
                    }
                } else {
                    // This unit's first dV/dK overwrite TMEM the previous unit's epilogue must
                    // have read. Waited for every unit, with or without steps, so dkv_full and
                    // dkv_free strictly alternate.
                    if (ul > 0)
                        ok = warp_wait(ptx::smem_addr(&bars->dkv_free), (uint32_t)(ul - 1) & 1u,
                                       abort_flag, err, kDevTimeoutSoftmax);
                    for (int si = 0; ok && si < w.nsteps; ++si, ++g) {
                        const int st = g % C::NQS;
                        ok = warp_wait(ptx::smem_addr(&bars->p_ready), (uint32_t)g & 1u, abort_flag, err,
                                       kDevTimeoutSoftmax);
                        if (!ok) break;
                        ptx::tc_fence_after();
                        // dV += P^T dO (A = P^T in TMEM) and dK += dS^T Q (A = dS^T, K-major in smem).
                        const uint32_t st_off = (uint32_t)st * C::STAGE_BYTES;
                        const uint32_t ds_off = (uint32_t)(g % C::NDS) * C::DS_BYTES;
                        const uint64_t do_mn = ptx::sdesc_add(st_mn, st_off + C::QTILE);
                        const uint64_t q_mn = ptx::sdesc_add(st_mn, st_off);
                        const uint64_t dsk = ptx::sdesc_add(ds_kmaj, ds_off);
                        if constexpr (D == 128) {
                            // dV (then P^T is free), the dQ partial (the drain starts on it),
                            // then dK: measured 1014 -> 1033 TFLOP/s on B4 H16 N4096 causal against
                            // dV, dK, dQ (no change at d=64, which keeps that order).
                            if (ptx::elect_one()) {
#pragma unroll
                                for (int kk = 0; kk < C::BMQ / 16; ++kk)
                                    ptx::mma_ts(tbase + C::DV_COL, tbase + C::PT_COL + kk * 8,
                                                ptx::sdesc_add(do_mn, kk * 2048), idesc_kv,
                                                (si > 0 || kk > 0) ? 1u : 0u);
                                ptx::mma_commit(ptx::smem_addr(&bars->mma_done));
                            }
                            __syncwarp();
                            if (g > 0) {
                                ok = warp_wait(ptx::smem_addr(&bars->dq_free), (uint32_t)(g - 1) & 1u,
                                               abort_flag, err, kDevTimeoutSoftmax);
                                if (!ok) break;
                                ptx::tc_fence_after();
                            }
                            const uint64_t dsm = ptx::sdesc_add(ds_mn, ds_off);
                            if (ptx::elect_one()) {
#pragma unroll
                                for (int kk = 0; kk < C::KT / 16; ++kk) {
                                    if (D == 128) {
                                        // dQ^T = K^T dS^T: A = K MN-major [d x keys], B = dS MN-major [q x keys]
                                        ptx::mma_ss(tbase + C::DQ_COL, ptx::sdesc_add(k_mn, kk * 2048),
                                                    ptx::sdesc_add(dsm, kk * 2048), idesc_q, kk > 0);
                                    } else {
                                        // dQ = dS K: A = dS MN-major [q x keys], B = K MN-major [d x keys]
                                        ptx::mma_ss(tbase + C::DQ_COL, ptx::sdesc_add(dsm, kk * 2048),
                                                    ptx::sdesc_add(k_mn, kk * 2048), idesc_q, kk > 0);
                                    }
                                }
                                ptx::mma_commit(ptx::smem_addr(&bars->dq_full));
#pragma unroll
                                for (int kk = 0; kk < C::BMQ / 16; ++kk)
                                    ptx::mma_ss(tbase + C::DK_COL,
                                                ptx::sdesc_add(dsk, (kk >> 2) * C::DSREG + (kk & 3) * 32),
                                                ptx::sdesc_add(q_mn, kk * 2048), idesc_kv,
                                                (si > 0 || kk > 0) ? 1u : 0u);
                                ptx::mma_commit(ptx::smem_addr(&bars->q_empty[st]));
                                if (si + 1 == w.nsteps) ptx::mma_commit(ptx::smem_addr(&bars->dkv_full));
                                ptx::mma_commit(ptx::smem_addr(&bars->ds_free[g % C::NDS]));
                            }
                        } else {
                            if (ptx::elect_one()) {
#pragma unroll
                                for (int kk = 0; kk < C::BMQ / 16; ++kk)
                                    ptx::mma_ts(tbase + C::DV_COL, tbase + C::PT_COL + kk * 8,
                                                ptx::sdesc_add(do_mn, kk * 2048), idesc_kv,
                                                (si > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                                for (int kk = 0; kk < C::BMQ / 16; ++kk)
                                    ptx::mma_ss(tbase + C::DK_COL,
                                                ptx::sdesc_add(dsk, (kk >> 2) * C::DSREG + (kk & 3) * 32),
                                                ptx::sdesc_add(q_mn, kk * 2048), idesc_kv,
                                                (si > 0 || kk > 0) ? 1u : 0u);
                                ptx::mma_commit(ptx::smem_addr(&bars->mma_done));
                                ptx::mma_commit(ptx::smem_addr(&bars->q_empty[st]));
                                if (si + 1 == w.nsteps) ptx::mma_commit(ptx::smem_addr(&bars->dkv_full));
                            }
                            __syncwarp();
                            if (g > 0) {
                                ok = warp_wait(ptx::smem_addr(&bars->dq_free), (uint32_t)(g - 1) & 1u,
                                               abort_flag, err, kDevTimeoutSoftmax);
                                if (!ok) break;
                                ptx::tc_fence_after();
                            }
                            const uint64_t dsm = ptx::sdesc_add(ds_mn, ds_off);
                            if (ptx::elect_one()) {
#pragma unroll
                                for (int kk = 0; kk < C::KT / 16; ++kk) {
                                    if (D == 128) {
                                        // dQ^T = K^T dS^T: A = K MN-major [d x keys], B = dS MN-major [q x keys]
                                        ptx::mma_ss(tbase + C::DQ_COL, ptx::sdesc_add(k_mn, kk * 2048),
                                                    ptx::sdesc_add(dsm, kk * 2048), idesc_q, kk > 0);
                                    } else {
                                        // dQ = dS K: A = dS MN-major [q x keys], B = K MN-major [d x keys]
                                        ptx::mma_ss(tbase + C::DQ_COL, ptx::sdesc_add(dsm, kk * 2048),
                                                    ptx::sdesc_add(k_mn, kk * 2048), idesc_q, kk > 0);
                                    }
                                }
                                ptx::mma_commit(ptx::smem_addr(&bars->dq_full));
                                ptx::mma_commit(ptx::smem_addr(&bars->ds_free[g % C::NDS]));
                            }
                        }
                        __syncwarp();
                    }
                    // a unit without steps still completes its dV/dK phase (zeros are stored)
                    if (ok && w.nsteps == 0) commit(&bars->dkv_full);
                }
                if (!ok) break;
                // this warp's MMAs reading K/V of the unit are issued: the producer may reload
                // them once they complete
                commit(&bars->kv_empty);
            }
            commit(&bars->final_bar);
            drain_wait(ptx::smem_addr(&bars->final_bar), 0);
        }
    } else if (warp >= 4 && warp < 12) {
        // ============ compute warpgroups: P^T and dS^T, one thread per key row ============
        // Two warpgroups split each step's query columns (half h takes 32-column chunks
        // [h*NCH/2, (h+1)*NCH/2)), so every SMSP runs two compute warps.
        const int h = (warp - 4) >> 2;
        const int wq = warp & 3;
        const int k = wq * 32 + lane;  // key row within the tile
        // (causal) queries at positions key .. key + window see this key; no window: all after it
        const uint32_t vspan = WINDOW ? (uint32_t)sh.window : 0x7fffffffu;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t t_s = tbase + lane_off + C::S_COL;
        const uint32_t t_dp = tbase + lane_off + C::DP_COL;
        const uint32_t t_pt = tbase + lane_off + C::PT_COL;
        constexpr int NCH = C::BMQ / 32;
        constexpr int NCH_H = NCH / 2;
        bool ok = true;
        int g = 0;
        for (int ul = 0;; ++ul) {
            const int u = fetch_unit(ul, ok);
            if (!ok || u < 0) break;
            const BwdUnit w = bwd_unit<D, CAUSAL, WINDOW>(u, sh);
            const int key0 = w.key0;
            const int key = key0 + k;
            StepCursor cur(w);
            for (int si = 0; si < w.nsteps; ++si, ++g, cur.next(w)) {
                const int q0 = cur.qi * C::BMQ;
                // S'^T and dP'^T already carry the row statistics (fold MMAs): nothing else to read.
                ok = __all_sync(0xffffffffu, wait_phase(ptx::smem_addr(&bars->s_full), (uint32_t)g & 1u,
                                                        abort_flag, err, kDevTimeoutMma));
                if (!ok) break;
                ptx::tc_fence_after();
                uint8_t* dsbuf = smem + C::OFF_DS + (g % C::NDS) * C::DS_BYTES;
                // key visible to query q iff (!causal || key <= p) && (no window || key >= p - window),
                // p = offset + q; elementwise masking only where the step crosses either edge.
                const int p0 = sh.offset + q0;
                const bool need_mask = CAUSAL && ((p0 < key0 + C::KT - 1) ||
                                                  (WINDOW && p0 + C::BMQ - 1 - sh.window > key0));
                if constexpr (NCH_H == 1) {
                    // P^T (to TMEM) and dS (to shared memory) of one 32-query chunk cc
                    auto compute_chunk = [&](int cc, const uint32_t (&sv)[32], const uint32_t (&dpv)[32],
                                             uint32_t (&pk)[16], uint32_t (&dk)[16]) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            const int qi = 32 * cc + j;
                            // x = c * S' = c * S - LSE * log2(e)
                            float x0, x1, x2, x3;
                            ptx::fmul2(x0, x1, __uint_as_float(sv[j]), __uint_as_float(sv[j + 1]), c, c);
                            ptx::fmul2(x2, x3, __uint_as_float(sv[j + 2]), __uint_as_float(sv[j + 3]), c, c);
                            float pe0 = ptx::ex2_approx(x0), pe1 = ptx::ex2_approx(x1);
                            float pe2 = ptx::ex2_approx(x2), pe3 = ptx::ex2_approx(x3);
                            if (need_mask) {
                                // visible iff key <= p <= key + window, i.e. p - key in [0, vspan]
                                const uint32_t dp = (uint32_t)(p0 + qi - key);
                                if (dp > vspan) pe0 = 0.f;
                                if (dp + 1u > vspan) pe1 = 0.f;
                                if (dp + 2u > vspan) pe2 = 0.f;
                                if (dp + 3u > vspan) pe3 = 0.f;
                            }
                            // dS = P (dP - D) = P dP'
                            float d0, d1, d2, d3;
                            ptx::fmul2(d0, d1, pe0, pe1, __uint_as_float(dpv[j]), __uint_as_float(dpv[j + 1]));
                            ptx::fmul2(d2, d3, pe2, pe3, __uint_as_float(dpv[j + 2]), __uint_as_float(dpv[j + 3]));
                            pk[j / 2] = ptx::pack_bf16x2(pe0, pe1);
                            pk[j / 2 + 1] = ptx::pack_bf16x2(pe2, pe3);
                            dk[j / 2] = ptx::pack_bf16x2(d0, d1);
                            dk[j / 2 + 1] = ptx::pack_bf16x2(d2, d3);
                        }
                    };
                    auto store_chunk = [&](int cc, const uint32_t (&pk)[16], const uint32_t (&dk)[16]) {
                        ptx::tmem_st16(t_pt + 16 * cc, pk);
                        // dS row k (queries contiguous) into the 128B-swizzled dS tile.
                        uint8_t* region = dsbuf + (cc >> 1) * C::DSREG;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const uint4 wv = make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
                            *reinterpret_cast<uint4*>(region + sw128_offset((uint32_t)k, (uint32_t)((cc & 1) * 4 + u))) = wv;
                        }
                    };
                    // The waits before the first P^T / dS store: dV of step g - 1 has read P^T, and
                    // dK and dQ of step g - NDS have read this dS buffer.
                    auto wait_buffers = [&]() {
                        if (g > 0)
                            ok = __all_sync(0xffffffffu, wait_phase(ptx::smem_addr(&bars->mma_done),
                                                                    (uint32_t)(g - 1) & 1u, abort_flag,
                                                                    err, kDevTimeoutMma));
                        if (ok && g >= C::NDS)
                            ok = __all_sync(0xffffffffu, wait_phase(ptx::smem_addr(&bars->ds_free[g % C::NDS]),
                                                                    (uint32_t)(g / C::NDS - 1) & 1u,
                                                                    abort_flag, err, kDevTimeoutMma));
                        ptx::tc_fence_after();
                    };
                    auto release_s = [&]() {  // this half's S^T/dP^T are in registers
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(ptx::smem_addr(&bars->s_free));
                    };
                    // Where S^T/dP^T are released decides whether the next step's S^T/dP^T MMAs run
                    // ahead of this step's dV/dK/dQ MMAs in the tensor pipe. Measured (backward
                    // TFLOP/s, GB300): d=128 (one 32-query chunk per warpgroup) releases after the
                    // chunk's exp2 phase and before the buffer waits (B4 H16 N4096 causal: 975 with the
                    // release right after the load, 1011 here, 934 after the waits); d=64 (two chunks)
                    // releases after loading its second chunk, behind the waits (B4 H16 N2048: 880;
                    // 853 with both chunks loaded before the waits, 864 after them).
                    const int cc0 = h;
                    uint32_t pk[16], dk[16];
                    {
                        uint32_t sv[32], dpv[32];
                        ptx::tmem_ld32_nowait(t_s + 32 * cc0, sv);
                        ptx::tmem_ld32_nowait(t_dp + 32 * cc0, dpv);
                        ptx::tmem_wait_ld(sv);
                        ptx::tmem_wait_ld(dpv);
                        compute_chunk(cc0, sv, dpv, pk, dk);
                    }
                    release_s();
                    wait_buffers();
                    if (!ok) break;
                    store_chunk(cc0, pk, dk);
                } else {
                    // d=64: the same steps, written as a loop over the two chunks (the compiler
                    // generates ~2 % faster code for this form than for the d=128 branch's lambdas)
#pragma unroll
                    for (int ci = 0; ci < NCH_H; ++ci) {
                        const int cc = h * NCH_H + ci;
                        uint32_t sv[32], dpv[32];
                        ptx::tmem_ld32_nowait(t_s + 32 * cc, sv);
                        ptx::tmem_ld32_nowait(t_dp + 32 * cc, dpv);
                        ptx::tmem_wait_ld(sv);
                        ptx::tmem_wait_ld(dpv);
                        if (ci == NCH_H - 1) {
                            // this half's S^T/dP^T columns are in registers: release them
                            ptx::tc_fence_before();
                            ptx::mbar_arrive(ptx::smem_addr(&bars->s_free));
                        }
                        uint32_t pk[16], dk[16];
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            const int qi = 32 * cc + j;
                            // x = c * S' = c * S - LSE * log2(e)
                            float x0, x1, x2, x3;
                            ptx::fmul2(x0, x1, __uint_as_float(sv[j]), __uint_as_float(sv[j + 1]), c, c);
                            ptx::fmul2(x2, x3, __uint_as_float(sv[j + 2]), __uint_as_float(sv[j + 3]), c, c);
                            float pe0 = ptx::ex2_approx(x0), pe1 = ptx::ex2_approx(x1);
                            float pe2 = ptx::ex2_approx(x2), pe3 = ptx::ex2_approx(x3);
                            if (need_mask) {
                                // visible iff key <= p <= key + window, i.e. p - key in [0, vspan]
                                const uint32_t dp = (uint32_t)(p0 + qi - key);
                                if (dp > vspan) pe0 = 0.f;
                                if (dp + 1u > vspan) pe1 = 0.f;
                                if (dp + 2u > vspan) pe2 = 0.f;
                                if (dp + 3u > vspan) pe3 = 0.f;
                            }
                            // dS = P (dP - D) = P dP'
                            float d0, d1, d2, d3;
                            ptx::fmul2(d0, d1, pe0, pe1, __uint_as_float(dpv[j]), __uint_as_float(dpv[j + 1]));
                            ptx::fmul2(d2, d3, pe2, pe3, __uint_as_float(dpv[j + 2]), __uint_as_float(dpv[j + 3]));
                            pk[j / 2] = ptx::pack_bf16x2(pe0, pe1);
                            pk[j / 2 + 1] = ptx::pack_bf16x2(pe2, pe3);
                            dk[j / 2] = ptx::pack_bf16x2(d0, d1);
                            dk[j / 2 + 1] = ptx::pack_bf16x2(d2, d3);
                        }
                        if (ci == 0) {
                            if (g > 0) {
                                // dV of step g - 1 must have read P^T before it is overwritten.
                                ok = __all_sync(0xffffffffu, wait_phase(ptx::smem_addr(&bars->mma_done),
                                                                        (uint32_t)(g - 1) & 1u, abort_flag,
                                                                        err, kDevTimeoutMma));
                                if (!ok) break;
                            }
                            if (g >= C::NDS) {
                                // dK and dQ of step g - NDS must have read this dS buffer.
                                ok = __all_sync(0xffffffffu, wait_phase(ptx::smem_addr(&bars->ds_free[g % C::NDS]),
                                                                        (uint32_t)(g / C::NDS - 1) & 1u,
                                                                        abort_flag, err, kDevTimeoutMma));
                                if (!ok) break;
                            }
                            ptx::tc_fence_after();
                        }
                        ptx::tmem_st16(t_pt + 16 * cc, pk);
                        // dS row k (queries contiguous) into the 128B-swizzled dS tile.
                        uint8_t* region = dsbuf + (cc >> 1) * C::DSREG;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const uint4 wv = make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
                            *reinterpret_cast<uint4*>(region + sw128_offset((uint32_t)k, (uint32_t)((cc & 1) * 4 + u))) = wv;
                        }
                    }
                }
                if (!ok) break;
                ptx::tmem_wait_st();
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before();
                ptx::mbar_arrive(ptx::smem_addr(&bars->p_ready));
            }
        }
    } else if (warp >= 12) {
        // ======== dQ drain warpgroup, and each unit's dV / dK epilogue ========
        const int wq = warp & 3;
        const int r = wq * 32 + lane;  // TMEM lane: d index (d=128 dQ) or query / key row
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        uint8_t* dqs = smem + C::OFF_DQS;
        bool ok = true;
        bool staged = false;  // a bulk copy issued from the staging tile may still be reading it
        auto staging_free = [&]() {
            if (staged) {
                if (r == 0) ptx::bulk_wait_read_all();
                ptx::named_bar_sync(2, 128);
            }
            staged = true;
        };
        int g = 0;
        for (int ul = 0;; ++ul) {
            const int u = fetch_unit(ul, ok);
            if (!ok || u < 0) break;
            const BwdUnit w = bwd_unit<D, CAUSAL, WINDOW>(u, sh);
            StepCursor cur(w);
            for (int si = 0; si < w.nsteps; ++si, ++g, cur.next(w)) {
                const int q0 = cur.qi * C::BMQ;
                const int bhq = cur.bhq;
                ok = __all_sync(0xffffffffu, wait_phase(ptx::smem_addr(&bars->dq_full), (uint32_t)g & 1u,
                                                        abort_flag, err, kDevTimeoutMma));
                if (!ok) break;
                ptx::tc_fence_after();
                uint32_t a[32], b[32];
                ptx::tmem_ld32_nowait(tbase + lane_off + C::DQ_COL, a);
                ptx::tmem_ld32_nowait(tbase + lane_off + C::DQ_COL + 32, b);
                ptx::tmem_wait_ld(a);
                ptx::tmem_wait_ld(b);
                ptx::tc_fence_before();
                ptx::mbar_arrive(ptx::smem_addr(&bars->dq_free));
                staging_free();
                if (D == 128) {
                    // lane r = head-dim column e; a/b hold query rows 0-31 / 32-63 of the step.
                    // The accumulator is kept transposed ([e][query], see the dQ conversion), so
                    // each thread's values are one contiguous row: box bx holds queries
                    // [32 bx, 32 bx + 32) of all 128 e rows, 128 B per row, written with
                    // 16-byte stores (a row per thread instead of one element per row).
#pragma unroll
                    for (int uu = 0; uu < 8; ++uu) {
                        *reinterpret_cast<uint4*>(dqs + sw128_offset((uint32_t)r, (uint32_t)uu)) =
                            make_uint4(a[4 * uu], a[4 * uu + 1], a[4 * uu + 2], a[4 * uu + 3]);
                        *reinterpret_cast<uint4*>(dqs + C::DQBOX_T + sw128_offset((uint32_t)r, (uint32_t)uu)) =
                            make_uint4(b[4 * uu], b[4 * uu + 1], b[4 * uu + 2], b[4 * uu + 3]);
                    }
                    ptx::fence_proxy_async_smem();
                    ptx::named_bar_sync(2, 128);
                    if (r == 0) {
                        for (int bx = 0; bx < 2; ++bx)
                            ptx::tma_reduce_add_3d(&tm_dqacc, ptx::smem_addr(dqs + bx * C::DQBOX_T),
                                                   q0 + 32 * bx, 0, bhq);
                        ptx::bulk_commit();
                    }
                } else {
                    // lane r = query row; a/b hold head-dim columns 0-31 / 32-63, one fp32 box
                    // each, staged one after the other through the single box of staging.
#pragma unroll
                    for (int uu = 0; uu < 8; ++uu)
                        *reinterpret_cast<uint4*>(dqs + sw128_offset((uint32_t)r, (uint32_t)uu)) =
                            make_uint4(a[4 * uu], a[4 * uu + 1], a[4 * uu + 2], a[4 * uu + 3]);
                    ptx::fence_proxy_async_smem();
                    ptx::named_bar_sync(2, 128);
                    if (r == 0) {
                        ptx::tma_reduce_add_3d(&tm_dqacc, ptx::smem_addr(dqs), 0, q0, bhq);
                        ptx::bulk_commit();
                    }
                    staging_free();
#pragma unroll
                    for (int uu = 0; uu < 8; ++uu)
                        *reinterpret_cast<uint4*>(dqs + sw128_offset((uint32_t)r, (uint32_t)uu)) =
                            make_uint4(b[4 * uu], b[4 * uu + 1], b[4 * uu + 2], b[4 * uu + 3]);
                    ptx::fence_proxy_async_smem();
                    ptx::named_bar_sync(2, 128);
                    if (r == 0) {
                        ptx::tma_reduce_add_3d(&tm_dqacc, ptx::smem_addr(dqs), 32, q0, bhq);
                        ptx::bulk_commit();
                    }
                }
            }
            if (!ok) break;
            // ---- epilogue of the unit: dV, then dK * scale -> bf16 -> staging -> TMA store ----
            // (runs while the next unit's first steps proceed; its first dV/dK MMA waits for
            // dkv_free)
            ok = __all_sync(0xffffffffu, wait_phase(ptx::smem_addr(&bars->dkv_full), (uint32_t)ul & 1u,
                                                    abort_flag, err, kDevTimeoutMma));
            if (!ok) break;
            ptx::tc_fence_after();
#pragma unroll 1
            for (int pass = 0; pass < 2; ++pass) {
                const uint32_t col = pass ? C::DK_COL : C::DV_COL;
                const float mul = pass ? scale : 1.f;
                staging_free();
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t v[32];
                    if (w.nsteps > 0) {
                        ptx::tmem_ld32(tbase + lane_off + col + 32 * cc, v);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0u;  // no query sees these keys
                    }
                    uint8_t* chunk = dqs + (cc >> 1) * C::KCHUNK;
#pragma unroll
                    for (int uu = 0; uu < 4; ++uu) {
                        uint4 wv;
                        wv.x = ptx::pack_bf16x2(__uint_as_float(v[8 * uu + 0]) * mul, __uint_as_float(v[8 * uu + 1]) * mul);
                        wv.y = ptx::pack_bf16x2(__uint_as_float(v[8 * uu + 2]) * mul, __uint_as_float(v[8 * uu + 3]) * mul);
                        wv.z = ptx::pack_bf16x2(__uint_as_float(v[8 * uu + 4]) * mul, __uint_as_float(v[8 * uu + 5]) * mul);
                        wv.w = ptx::pack_bf16x2(__uint_as_float(v[8 * uu + 6]) * mul, __uint_as_float(v[8 * uu + 7]) * mul);
                        *reinterpret_cast<uint4*>(chunk + sw128_offset((uint32_t)r, (uint32_t)((cc & 1) * 4 + uu))) = wv;
                    }
                }
                if (pass == 1) {
                    // dV and dK are in registers / staging: the next unit may overwrite TMEM
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(ptx::smem_addr(&bars->dkv_free));
                }
                ptx::fence_proxy_async_smem();
                ptx::named_bar_sync(2, 128);
                if (r == 0) {
                    for (int ch = 0; ch < D / 64; ++ch)
                        ptx::tma_store_3d(pass ? &tm_dk : &tm_dv, ptx::smem_addr(dqs + ch * C::KCHUNK),
                                          ch * 64, w.key0, w.bh_kv);
                    ptx::bulk_commit();
                }
            }
        }
        if (r == 0) ptx::bulk_wait_all();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tbase, 512);
    }
}

// L2 budget for one chunk of the causal unit order: the chunk's Q, dO and fp32 dQ accumulator
// rows, which its units re-read and re-add while they sweep their query steps. Measured on
// B4 H16 N4096 d128 causal (GB300, main kernel): budgeting Q and dO alone at 128 MB put all 64
// heads in one chunk, a 256 MB working set, and the kernel moved 2.97 GB of DRAM per launch
// (4.4x the algorithmic 0.67 GB); this budget gives three equal chunks of 21-22 heads and
// 0.77 GB, at 1.5 % more kernel time (more units of one head run at once, and their
// reduce-adds meet on the same accumulator rows).
constexpr long long kChunkL2Bytes = 96LL << 20;

template <int D, bool CAUSAL, bool WINDOW>
cudaError_t launch_bwd_t(const BwdLaunch& a, cudaStream_t stream) {
    static_assert(CAUSAL || !WINDOW, "a window hangs off the causal diagonal");
    using C = BwdCfg<D>;
    // 1. preprocess (query heads)
    {
        const long long rows = (long long)a.BHq * a.Npad;
        const long long rpb = 256 / (D / 8);
        const long long blocks = (rows + rpb - 1) / rpb;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        cudaError_t e = launch_dependent(
            fa_bwd_pre_kernel<D>, dim3((unsigned)blocks), dim3(256), 0, stream,
            static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dout), a.lse,
            static_cast<uint8_t*>(a.folds), a.dq_acc, a.sched, a.Tq, a.Npad, a.BHq, 1.0f / a.scale);
        if (e != cudaSuccess) return e;
    }
    // 2. main (persistent; a work unit is one KV head and 128-key tile)
    {
        auto kern = fa_bwd_kernel<D, CAUSAL, WINDOW>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        BwdShape sh;
        sh.Tq = a.Tq;
        sh.Tk = a.Tk;
        sh.Npad = a.Npad;
        sh.Hq = a.Hq;
        sh.Hkv = a.Hkv;
        sh.group = a.Hq / a.Hkv;
        sh.offset = a.Tk - a.Tq;
        sh.window = a.window;
        sh.BHq = a.BHq;
        sh.BHkv = a.BHkv;
        sh.nkb = (a.Tk + C::KT - 1) / C::KT;
        const long long units = (long long)sh.nkb * a.BHkv;
        if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        // Causal: as many KV heads per chunk as keep the chunk's Q and dO (bf16) and dQ
        // accumulator (fp32) rows -- all query heads of each KV head -- within kChunkL2Bytes,
        // with the heads spread evenly over the chunks (a small last chunk would run few heads
        // on many SMs, all adding into the same accumulator rows).
        sh.kv_chunk = 1;
        if (CAUSAL) {
            const long long per_head = (long long)sh.group * a.Tq * D * (2 * 2 + 4);
            sh.kv_chunk = (int)std::max(1LL, std::min<long long>(a.BHkv, kChunkL2Bytes / std::max(1LL, per_head)));
            int nchunks = (a.BHkv + sh.kv_chunk - 1) / sh.kv_chunk;
            // A chunk starts with its costliest units; if a chunk holds less work per SM than
            // its costliest unit, the last chunk's long units outlast everything else. So there
            // are at most (steps of the launch) / (SMs * steps of the costliest unit) chunks.
            const int nq_total = (a.Tq + C::BMQ - 1) / C::BMQ;
            long long steps_per_kv = 0, max_unit = 0;
            for (int kb = 0; kb < sh.nkb; ++kb) {
                const int key0 = kb * C::KT;
                const int i0 = std::max(0, key0 - sh.offset) / C::BMQ;
                int i1 = nq_total - 1;
                if (WINDOW) {
                    const int reach = key0 + C::KT - 1 + sh.window - sh.offset;
                    i1 = (reach < 0) ? -1 : std::min(i1, reach / C::BMQ);
                }
                const long long n = (long long)std::max(0, i1 - i0 + 1) * sh.group;
                steps_per_kv += n;
                max_unit = std::max(max_unit, n);
            }
            const long long cap = (steps_per_kv * a.BHkv) /
                                  std::max(1LL, (long long)std::max(1, a.num_sms) * max_unit);
            nchunks = (int)std::max(1LL, std::min<long long>(nchunks, cap));
            sh.kv_chunk = (a.BHkv + nchunks - 1) / nchunks;
        }
        // Persistent grid: one CTA per SM walking units (the shared memory admits one CTA).
        const int grid = (int)std::min<long long>(units, (long long)std::max(1, a.num_sms));
        e = launch_dependent(kern, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM_BYTES, stream,
                             a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.tm_dk, a.tm_dv, a.tm_dqacc,
                             static_cast<const uint8_t*>(a.folds), sh, (int)units, a.sched, a.c,
                             a.scale, a.err);
        if (e != cudaSuccess) return e;
    }
    // 3. dQ convert (query heads)
    if constexpr (D == 128) {
        const long long tiles = ((long long)a.Tq + 63) / 64;
        const long long blocks = tiles * a.BHq;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        return launch_dependent(fa_bwd_dqt_kernel, dim3((unsigned)blocks), dim3(256), 0, stream,
                                static_cast<const float*>(a.dq_acc),
                                static_cast<__nv_bfloat16*>(a.dq), a.Tq, a.Npad, (int)tiles, a.scale);
    } else {
        const long long total8 = (long long)a.BHq * a.Tq * (D / 8);
        const long long blocks = (total8 + 255) / 256;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        return launch_dependent(fa_bwd_dq_kernel<D>, dim3((unsigned)blocks), dim3(256), 0, stream,
                                static_cast<const float*>(a.dq_acc),
                                static_cast<__nv_bfloat16*>(a.dq), a.Tq, a.Npad, a.BHq, a.scale);
    }
}

}  // namespace

cudaError_t launch_backward(const BwdLaunch& a, bool causal, cudaStream_t stream) {
    const bool window = a.window >= 0;
    if (window && !causal) return cudaErrorInvalidValue;
    if (a.d == 64) {
        if (!causal) return launch_bwd_t<64, false, false>(a, stream);
        return window ? launch_bwd_t<64, true, true>(a, stream) : launch_bwd_t<64, true, false>(a, stream);
    }
    if (a.d == 128) {
        if (!causal) return launch_bwd_t<128, false, false>(a, stream);
        return window ? launch_bwd_t<128, true, true>(a, stream) : launch_bwd_t<128, true, false>(a, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace fa
