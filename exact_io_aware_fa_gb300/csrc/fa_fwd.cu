// fa_fwd.cu -- exact attention forward for sm_103a: O = softmax(scale * Q K^T) V and the
// per-row log-sum-exp, computed tile by tile with the online-softmax recurrence so that
// the N x N score and probability matrices never leave the SM.
//
// Method ("15. FlashAttention", inference.shantanugoel.com, sections "Online softmax:
// normalize as you go" and "The algorithm in plain PyTorch"; "FlashAttention: from
// IO-Aware Attention to GPU work partitioning", blog.euler0525.cn, sections
// "FlashAttention-2" and "Tile Size 与 Causal Attention"):
//   per query row keep m (running max), l (running sum of exp(s - m)) and an
//   unnormalised accumulator a; for each key tile m_new = max(m, rowmax(s)),
//   alpha = exp(m - m_new), p = exp(s - m_new), l = alpha l + sum p, a = alpha a + p V;
//   at the end O = a / l and LSE = m + ln l. Tiles wholly above the causal diagonal are
//   skipped; only the diagonal tile and the ragged last tile are masked elementwise.
//
// Grouped KV heads and the query offset (query row i at key position Tk - Tq + i) follow the
// same page's "Details worth noticing"; the optional sliding window keeps keys at positions
// >= position - window (its "Stretch exercises", item 3); the split-KV variant writes per-chunk
// partials merged by the rule of its section "Decode is different: flash-decoding".
//
// GB300 mapping: a persistent grid of one CTA per SM; a CTA walks work units (one unit = 256
// query rows of one query head = two 128-row Q tiles; in the split variant, one key chunk of
// them) so that the next unit's loads and first score MMAs overlap the current unit's
// epilogue. Roles:
//   warp 0      TMA producer: Q tiles once per unit, then K_j / V_j into separate mbarrier rings
//   warp 1      MMA issuer for S_t = Q_t K_j^T (tcgen05.mma, fp32 in TMEM); at d=128 also for
//               O_t += P_t V_j, issued just before the tile's next S (P is written over S)
//   warp 3      MMA issuer for O_t += P_t V_j at d=64 (A = P from TMEM)
//   warp 2      TMEM allocation / release
//   warps 4-7   softmax for Q tile 0, warps 8-11 softmax for Q tile 1: one thread per row,
//               the whole row of S read from TMEM into registers (no cross-thread reduction),
//               exp2 with log2(e) folded into the scale, P written back to TMEM as bf16, O
//               rescaled in TMEM when some row of the warp raises its max, and the epilogue
//               (O / l -> bf16 -> swizzled smem -> TMA store; LSE -> global; or, split, the
//               fp32 partial O and LSE).
// TMEM (512 columns): d=64: S_0, S_1 [0,256), O_0, O_1 [256,384), P_0, P_1 [384,512);
// d=128: S_0, S_1 [0,256), O_0, O_1 [256,512), P written over S.
// Kernel variants (template arguments): CAUSAL, WINDOW, SPLIT as above; SORTED, the causal
// unit order (heaviest first, snake-dealt, over L2-sized chunks of heads; else a head's blocks
// in heavy/light pairs); PACKED, a KV head's query heads packed into one block of rows (short
// query blocks with grouped heads). Non-causal launches whose last round would be at most half
// full run it as single-tile half units.
#include <algorithm>

#include <cuda_bf16.h>

#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {
namespace {

constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct FwdCfg {
    static constexpr int BM = 128;        // rows per Q tile (one TMEM lane per row)
    static constexpr int BN = 128;        // keys per KV tile
    static constexpr int ROWS = 2 * BM;   // rows per CTA
    static constexpr int DCH = D / 64;    // 64-column (128-byte) chunks per row
    static constexpr int NS = (D == 64) ? 3 : 2;  // K and V ring depth
    static constexpr uint32_t TILE_BYTES = 128u * D * 2u;  // one 128-row bf16 tile
    static constexpr uint32_t CHUNK_BYTES = 128u * 128u;   // one 128-row x 64-col chunk
    // Q buffers: two at d=64 (the next unit's Q loads while this unit finishes), one at d=128
    // (the next Q waits for the epilogue, which stages O in the Q buffer, to release it).
    static constexpr int NQB = (D == 64) ? 2 : 1;
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + NQB * 2 * TILE_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + NS * TILE_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_V + NS * TILE_BYTES;
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + 512 + 1024;  // + alignment slack
    static constexpr int THREADS = 384;
    static constexpr uint32_t TMEM_COLS = 512;
    // d = 64: S_0, S_1 [0,256), O_0, O_1 [256,384), P_0, P_1 [384,512) -- P has its own
    //         columns, so S_t(j+1) can be computed while the softmax still works on tile j.
    // d = 128: S_0, S_1 [0,256), O_0, O_1 [256,512), P_t written over the S_t columns.
    static constexpr bool P_SEPARATE = (D == 64);
    __host__ __device__ static constexpr uint32_t s_col(int t) { return (uint32_t)(t * 128); }
    __host__ __device__ static constexpr uint32_t o_col(int t) { return 256u + (uint32_t)(t * D); }
    __host__ __device__ static constexpr uint32_t p_col(int t) {
        return P_SEPARATE ? 384u + (uint32_t)(t * 64) : (uint32_t)(t * 128);
    }
};

// Reference max of the online softmax (log2 domain of the scaled scores), kRefLag:
// the reference moves only when the row max exceeds it by more than 8, so after the first key
// tile of a unit O is almost never rescaled (p <= 2^8 stays far from fp32 overflow). (Moving it
// whenever the max grows, so that the largest weight is exactly 1, rescaled O on many more
// steps: 2-3 % slower at d = 128, more at d = 64.)
// The largest weight p_M = exp2(c s_M - m_ref) is then not 1, and its bf16 rounding would carry
// into O in peaked rows; the epilogue divides O by l + (bf16(p_M) - p_M), the sum with that
// weight taken as the PV product used it, which cancels the dominant weight's error (to first
// order the output error becomes w_M (1 - w_M) eps_M (v_M - v_rest), eps_M its relative rounding).
constexpr float kRefLag = 8.0f;

struct FwdBars {
    uint64_t q_full[2], q_free[2];
    uint64_t o_free[2];
    uint64_t k_full[3], k_empty[3];
    uint64_t v_full[3], v_empty[3];
    uint64_t s_full[2], s_free[2], p_full[2], o_done[2];
    uint64_t mma_final;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Wait that ignores the abort flag (used only to drain copies already in flight).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
}

// Problem shape: query heads read KV head bh_q / group; query row i sits at key position
// offset + i (offset = Tk - Tq, so the last query lines up with the last key); with a window,
// keys before position - window are not visible.
struct FwdShape {
    int Tq, Tk, Hq, Hkv, group, offset, window, nqb;
    // Query rows per head for positions: row r of a head's block sits at key position
    // offset + r % tq_pos. Equal to Tq, except with the query heads of a KV head packed into
    // one block of group * Tq rows (short query blocks), where Tq counts those rows.
    int tq_pos;
    int nsplit;  // key-range splits per unit (flash-decoding); 1 = whole range, final output
    int BHq;     // B * Hq (partial-result indexing)
    // Units numbered from full_units on are half units (non-causal, unsplit launches): the
    // 256-row block full_units + (h >> 1) cut into its two Q tiles, h & 1 selecting one. They
    // fill a last round that would otherwise leave most SMs idle.
    int full_units;
    // Causal, sorted order: query heads per chunk (chosen so that a chunk's K/V stays in L2);
    // inside a chunk units go heaviest block first, head by head (with splits: the key chunks
    // of a block are consecutive units).
    int q_chunk;
};

// One work unit: (query head bh_q, 256-row block qb) and, per Q tile t, its range of key
// tiles [jb_t, je_t) (empty when the tile lies past Tq).
struct FwdUnit {
    int bh_q, bh_kv, qb, split;
    int row0;  // first query row of Q tile 0
    int jb0, je0, jb1, je1;
    int jb_all, je_all;
    // No key tile for either Q tile (an empty key chunk, or a half unit past Tq): such a unit
    // takes no part in the Q-buffer protocol (no load, no q_full / q_free phase), and every
    // role counts Q-buffer uses over the other units only.
    __device__ __forceinline__ bool empty() const { return je_all <= jb_all; }
    __device__ __forceinline__ int jb(int t) const { return t ? jb1 : jb0; }
    __device__ __forceinline__ int je(int t) const { return t ? je1 : je0; }
};

// The k-th unit of CTA `cta` (of G), or -1 past the end.
// Non-causal: plain round robin over units numbered head by head (all cost the same).
// Causal, SORTED: units are numbered heaviest first (see fwd_unit) and
// dealt in snake order -- round k goes to CTAs 0 .. G-1 when k is even and G-1 .. 0 when odd --
// so every CTA's running sum of cost stays close to the others' and the launch ends on the
// lightest units. Causal otherwise: a head's blocks are ordered heaviest, lightest, second
// heaviest, second lightest, ... and each CTA takes consecutive pairs (with cost linear in the
// block index every pair costs the same, and a round works on a few neighbouring heads).
template <bool CAUSAL, bool SORTED>
__device__ __forceinline__ int fwd_unit_index(int cta, int k, int G, int U) {
    long long u;
    if (!CAUSAL)
        u = cta + (long long)k * G;
    else if (SORTED)
        u = (long long)k * G + ((k & 1) ? (G - 1 - cta) : cta);
    else
        u = 2LL * (cta + (long long)(k >> 1) * G) + (k & 1);
    return u < U ? (int)u : -1;
}

// Positions (within a head) of rows r0 .. r1 of a block whose rows hold tq positions per head:
// their smallest and largest, taken over all positions when the rows wrap into the next
// packed head.
__device__ __forceinline__ void tile_positions(int r0, int r1, int tq, int& lo, int& hi) {
    lo = r0 % tq;
    hi = r1 % tq;
    if (r1 - r0 >= tq || hi < lo) {
        lo = 0;
        hi = tq - 1;
    }
}

// PACKED: query heads packed into blocks of group * Tq rows (positions wrap every tq_pos rows).
template <int D, bool CAUSAL, bool WINDOW, bool SPLIT, bool SORTED, bool PACKED>
__device__ __forceinline__ FwdUnit fwd_unit(int u, const FwdShape& sh) {
    using C = FwdCfg<D>;
    FwdUnit w;
    w.split = 0;
    int half = -1;  // a half unit's Q tile (0 or 1); -1 for a full unit
    if (!CAUSAL && !SPLIT && u >= sh.full_units) {
        const int h = u - sh.full_units;
        u = sh.full_units + (h >> 1);
        half = h & 1;
    }
    if (SPLIT) {
        w.split = u % sh.nsplit;  // the splits of one query block are consecutive units
        u /= sh.nsplit;
    }
    if (CAUSAL && SORTED) {
        // chunk of q_chunk query heads (the last may be smaller); inside it, rank-major: all
        // heads' heaviest block (the last one), then all heads' next, ...
        const uint32_t per_chunk = (uint32_t)sh.q_chunk * (uint32_t)sh.nqb;
        const uint32_t chunk = (uint32_t)u / per_chunk;
        const uint32_t r = (uint32_t)u - chunk * per_chunk;
        const uint32_t h0 = chunk * (uint32_t)sh.q_chunk;
        const uint32_t hc = min((uint32_t)sh.q_chunk, (uint32_t)sh.BHq - h0);
        w.bh_q = (int)(h0 + r % hc);
        w.qb = sh.nqb - 1 - (int)(r / hc);
    } else {
        w.bh_q = u / sh.nqb;
        const int i = u % sh.nqb;
        if (CAUSAL) {
            const int q = (i & 1) ? sh.nqb - 1 - (i >> 1) : (i >> 1);  // rank by cost, 0 = heaviest
            w.qb = sh.nqb - 1 - q;
        } else {
            w.qb = i;
        }
    }
    w.bh_kv = (w.bh_q / sh.Hq) * sh.Hkv + (w.bh_q % sh.Hq) / sh.group;
    const int nk = (sh.Tk + C::BN - 1) / C::BN;
    // key tiles [jb, je) of the Q tile starting at row r0 (empty past Tq)
    auto range = [&](int r0, int& jb, int& je) {
        if (r0 >= sh.Tq) {
            jb = je = 0;
            return;
        }
        int q0 = r0, q1 = min(r0 + C::BM, sh.Tq) - 1;  // smallest and largest row position
        if (PACKED) tile_positions(r0, q1, sh.tq_pos, q0, q1);
        const int p0 = sh.offset + q0;
        const int p1 = sh.offset + q1;
        je = CAUSAL ? min(nk, p1 / C::BN + 1) : nk;
        jb = WINDOW ? max(0, p0 - sh.window) / C::BN : 0;
        if (jb >= je) jb = je = 0;  // (cannot happen for valid shapes)
        if (SPLIT && je > jb) {
            // this split's chunk of the range (empty when the range is short)
            const int c = (je - jb + sh.nsplit - 1) / sh.nsplit;
            const int b0 = jb + w.split * c;
            jb = min(je, b0);
            je = min(je, b0 + c);
        }
    };
    w.row0 = w.qb * C::ROWS + (half > 0 ? C::BM : 0);
    range(w.row0, w.jb0, w.je0);
    if (half >= 0)
        w.jb1 = w.je1 = 0;  // a half unit is its one Q tile, run as tile 0
    else
        range(w.row0 + C::BM, w.jb1, w.je1);
    if (!SPLIT) {
        // tile 0 always has keys without splits
        w.jb_all = w.jb0;
        w.je_all = max(w.je0, w.je1);
        if (w.je1 > w.jb1) w.jb_all = min(w.jb_all, w.jb1);
    } else {
        // a split chunk may be empty for either tile
        const bool e0 = w.je0 > w.jb0, e1 = w.je1 > w.jb1;
        w.jb_all = e0 ? (e1 ? min(w.jb0, w.jb1) : w.jb0) : (e1 ? w.jb1 : 0);
        w.je_all = e0 ? (e1 ? max(w.je0, w.je1) : w.je0) : (e1 ? w.je1 : 0);
    }
    return w;
}

// WINDOW (causal only): keys before position - window are not visible. SPLIT: every unit is
// one key chunk of a query block and writes a partial result for the merge kernel.
template <int D, bool CAUSAL, bool WINDOW, bool SPLIT, bool SORTED, bool PACKED>
__global__ void __launch_bounds__(384, 1)
fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
              const FwdShape sh, const int num_units, const float c, float* __restrict__ lse_out,
              float* __restrict__ part_o, float* __restrict__ part_lse, int* err) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    FwdBars* bars = reinterpret_cast<FwdBars*>(smem + C::OFF_BAR);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int G = gridDim.x;

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_addr(&bars->q_full[b]), 1);
            ptx::mbar_init(ptx::smem_addr(&bars->q_free[b]), 2);  // one arrive per Q tile
        }
        for (int s = 0; s < C::NS; ++s) {
            ptx::mbar_init(ptx::smem_addr(&bars->k_full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&bars->k_empty[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&bars->v_full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&bars->v_empty[s]), 1);
        }
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(ptx::smem_addr(&bars->s_full[t]), 1);
            ptx::mbar_init(ptx::smem_addr(&bars->s_free[t]), C::BM);
            ptx::mbar_init(ptx::smem_addr(&bars->p_full[t]), C::BM);
            ptx::mbar_init(ptx::smem_addr(&bars->o_done[t]), 1);
            ptx::mbar_init(ptx::smem_addr(&bars->o_free[t]), C::BM);
        }
        ptx::mbar_init(ptx::smem_addr(&bars->mma_final), 2);
        bars->abort_flag = 0;
        ptx::fence_barrier_init();
        ptx::tma_prefetch_desc(&tm_q);
        ptx::tma_prefetch_desc(&tm_k);
        ptx::tma_prefetch_desc(&tm_v);
        ptx::tma_prefetch_desc(&tm_o);
    }
    if (warp == 2) {
        ptx::tmem_alloc(ptx::smem_addr(&bars->tmem_base), C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    // The next kernel in the stream (the split merge, or a backward's preprocess) may start
    // launching now; it waits for this kernel's completion before using its results.
    ptx::griddep_launch_dependents();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tbase = __shfl_sync(0xffffffffu, bars->tmem_base, 0);
    volatile int* abort_flag = &bars->abort_flag;

    const uint32_t s_q = ptx::smem_addr(smem + C::OFF_Q);
    const uint32_t s_k = ptx::smem_addr(smem + C::OFF_K);
    const uint32_t s_v = ptx::smem_addr(smem + C::OFF_V);

    if (warp == 0) {
        // ================================ TMA producer ================================
        if (lane == 0) {
            const uint64_t pol_kv = ptx::l2_policy_evict_last();
            const uint64_t pol_q = ptx::l2_policy_evict_first();
            int kv = 0;   // K/V tiles loaded so far (ring position)
            int ul = 0;   // units started by this CTA
            int qn = 0;   // non-empty units started (Q-buffer uses)
            int last_q_use[2] = {-1, -1};
            bool ok = true;
            for (int u; ok && (u = fwd_unit_index<CAUSAL, SORTED>(blockIdx.x, ul, G, num_units)) >= 0; ++ul) {
                const FwdUnit w = fwd_unit<D, CAUSAL, WINDOW, SPLIT, SORTED, PACKED>(u, sh);
                if (w.empty()) continue;
                const int b = qn % C::NQB;
                const int use = qn / C::NQB;  // earlier uses of Q buffer b
                ++qn;
                if (use > 0) {
                    // the epilogues of the unit NQB uses back staged O in this buffer and stored it
                    ok = wait_phase(ptx::smem_addr(&bars->q_free[b]), (uint32_t)(use - 1) & 1u,
                                    abort_flag, err, kDevTimeoutSoftmax);
                    if (!ok) break;
                }
                const uint32_t bq = ptx::smem_addr(&bars->q_full[b]);
                const int ntl = 1 + (w.je1 > w.jb1);
                ptx::mbar_arrive_expect_tx(bq, ntl * C::TILE_BYTES);
                for (int t = 0; t < ntl; ++t)
                    for (int ch = 0; ch < C::DCH; ++ch)
                        ptx::tma_load_3d_hint(s_q + (b * 2 + t) * C::TILE_BYTES + ch * C::CHUNK_BYTES,
                                              &tm_q, bq, ch * 64, w.row0 + t * C::BM, w.bh_q,
                                              pol_q);
                last_q_use[b] = use;
                for (int j = w.jb_all; j < w.je_all; ++j, ++kv) {
                    const int s = kv % C::NS;
                    const uint32_t ph = (uint32_t)(kv / C::NS) & 1u;
                    const uint32_t bkf = ptx::smem_addr(&bars->k_full[s]);
                    const uint32_t bvf = ptx::smem_addr(&bars->v_full[s]);
                    ok = wait_phase(ptx::smem_addr(&bars->k_empty[s]), ph ^ 1u, abort_flag, err,
                                    kDevTimeoutConsumer);
                    if (!ok) break;
                    ptx::mbar_arrive_expect_tx(bkf, C::TILE_BYTES);
                    for (int ch = 0; ch < C::DCH; ++ch)
                        ptx::tma_load_3d_hint(s_k + s * C::TILE_BYTES + ch * C::CHUNK_BYTES, &tm_k,
                                              bkf, ch * 64, j * C::BN, w.bh_kv, pol_kv);
                    ok = wait_phase(ptx::smem_addr(&bars->v_empty[s]), ph ^ 1u, abort_flag, err,
                                    kDevTimeoutConsumer);
                    if (!ok) {
                        drain_wait(bkf, ph);
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(bvf, C::TILE_BYTES);
                    for (int ch = 0; ch < C::DCH; ++ch)
                        ptx::tma_load_3d_hint(s_v + s * C::TILE_BYTES + ch * C::CHUNK_BYTES, &tm_v,
                                              bvf, ch * 64, j * C::BN, w.bh_kv, pol_kv);
                }
            }
            // Drain: every copy issued must have landed before the CTA can exit.
            for (int b = 0; b < 2; ++b)
                if (last_q_use[b] >= 0)
                    drain_wait(ptx::smem_addr(&bars->q_full[b]), (uint32_t)last_q_use[b] & 1u);
            for (int x = max(0, kv - C::NS); x < kv; ++x) {
                drain_wait(ptx::smem_addr(&bars->k_full[x % C::NS]), (uint32_t)(x / C::NS) & 1u);
                drain_wait(ptx::smem_addr(&bars->v_full[x % C::NS]), (uint32_t)(x / C::NS) & 1u);
            }
        }
    } else if (warp == 1 || warp == 3) {
        // ================================ MMA issuers =================================
        // d = 64 (P in its own columns): two issuing warps, warp 1 for the S MMAs and warp 3
        // for the PV MMAs. A thread that issues MMAs stalls until the tensor pipe has (almost)
        // drained them, so with one issuer every barrier wait left the pipe empty; with two,
        // one warp's MMAs run while the other waits for its next operands. d = 128 (P over S):
        // one issuing warp, below. The whole warp runs the loop and one elected lane issues,
        // which keeps descriptors and TMEM addresses in uniform registers.
        constexpr uint32_t idesc_s = ptx::idesc_bf16(128, C::BN, false, false);
        constexpr uint32_t idesc_o = ptx::idesc_bf16(128, D, false, true);
        const uint64_t dq0 = ptx::sdesc_sw128(s_q, 16, 1024);
        const uint64_t dk0 = ptx::sdesc_sw128(s_k, 16, 1024);
        const uint64_t dv0 = ptx::sdesc_sw128(s_v, C::CHUNK_BYTES, 1024);
        auto commit = [&](uint64_t* bar) {
            if (ptx::elect_one()) ptx::mma_commit(ptx::smem_addr(bar));
            __syncwarp();
        };
        int it[2] = {0, 0};  // score tiles (S) or products (PV) issued so far, per Q tile
        int uo[2] = {0, 0};  // units in which each Q tile ran (PV issuer: o_free phases)
        int kv = 0;
        int ul = 0;
        int qn = 0;  // non-empty units (Q-buffer uses)
        bool ok = true;
        if (!C::P_SEPARATE) {
            // P over S (d = 128): warp 1 issues both products of a tile back to back,
            // O_t += P_t(j-1) V_(j-1), then S_t(j) = Q_t K_j^T. The MMAs of one thread run in
            // issue order, so S_t(j) overwrites P_t(j-1) only after the PV MMA has read it and
            // needs no completion wait in between: the tensor pipe gets PV_0, S_0, PV_1, S_1,
            // ... with no barrier round trip between a tile's PV and its next S. (A commit
            // tracks every earlier MMA of the thread, so S_t(j) complete also means PV_t(j-1)
            // complete.) Warp 3 issues nothing.
            if (warp == 1) {
                for (int u; ok && (u = fwd_unit_index<CAUSAL, SORTED>(blockIdx.x, ul, G, num_units)) >= 0; ++ul) {
                    const FwdUnit w = fwd_unit<D, CAUSAL, WINDOW, SPLIT, SORTED, PACKED>(u, sh);
                    if (w.empty()) continue;
                    const int b = qn % C::NQB;
                    const uint32_t qph = (uint32_t)(qn / C::NQB) & 1u;
                    ++qn;
                    ok = warp_wait(ptx::smem_addr(&bars->q_full[b]), qph, abort_flag, err,
                                   kDevTimeoutLoad);
                    // iteration j: the PVs of key tile j-1, then the S MMAs of key tile j
                    for (int j = w.jb_all; ok && j <= w.je_all; ++j) {
                        const bool has_k = j < w.je_all;
                        const bool has_v = j > w.jb_all;
                        const int xk = kv + (j - w.jb_all);  // ring position of key tile j
                        const int sk = xk % C::NS, sv = (xk - 1 + C::NS) % C::NS;
                        if (has_v) {
                            ok = warp_wait(ptx::smem_addr(&bars->v_full[sv]),
                                           (uint32_t)((xk - 1) / C::NS) & 1u, abort_flag, err,
                                           kDevTimeoutLoad);
                            if (!ok) break;
                        }
                        bool k_ready = false;
                        for (int t = 0; ok && t < 2; ++t) {
                            if (has_v && j - 1 >= w.jb(t) && j - 1 < w.je(t)) {
                                if (j - 1 == w.jb(t) && uo[t] > 0) {
                                    // O_t is about to be overwritten: the previous unit's
                                    // epilogue must have read it.
                                    ok = warp_wait(ptx::smem_addr(&bars->o_free[t]),
                                                   (uint32_t)(uo[t] - 1) & 1u, abort_flag, err,
                                                   kDevTimeoutSoftmax);
                                    if (!ok) break;
                                }
                                ok = warp_wait(ptx::smem_addr(&bars->p_full[t]), (uint32_t)it[t] & 1u,
                                               abort_flag, err, kDevTimeoutSoftmax);
                                if (!ok) break;
                                ptx::tc_fence_after();
                                const uint32_t d_tmem = tbase + C::o_col(t);
                                const uint32_t p_tmem = tbase + C::p_col(t);
                                const uint64_t vd = ptx::sdesc_add(dv0, (uint32_t)sv * C::TILE_BYTES);
                                if (ptx::elect_one()) {
#pragma unroll
                                    for (int kk = 0; kk < C::BN / 16; ++kk)
                                        ptx::mma_ts(d_tmem, p_tmem + kk * 8, ptx::sdesc_add(vd, kk * 2048),
                                                    idesc_o, (j - 1 > w.jb(t) || kk > 0) ? 1u : 0u);
                                    ptx::mma_commit(ptx::smem_addr(&bars->o_done[t]));
                                }
                                __syncwarp();
                                ++it[t];
                            }
                            if (has_k && j >= w.jb(t) && j < w.je(t)) {
                                if (!k_ready) {
                                    ok = warp_wait(ptx::smem_addr(&bars->k_full[sk]),
                                                   (uint32_t)(xk / C::NS) & 1u, abort_flag, err,
                                                   kDevTimeoutLoad);
                                    if (!ok) break;
                                    k_ready = true;
                                }
                                ptx::tc_fence_after();
                                const uint32_t d_tmem = tbase + C::s_col(t);
                                const uint64_t qd = ptx::sdesc_add(dq0, (uint32_t)(b * 2 + t) * C::TILE_BYTES);
                                const uint64_t kd = ptx::sdesc_add(dk0, (uint32_t)sk * C::TILE_BYTES);
                                if (ptx::elect_one()) {
#pragma unroll
                                    for (int kk = 0; kk < D / 16; ++kk) {
                                        const uint32_t off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
                                        ptx::mma_ss(d_tmem, ptx::sdesc_add(qd, off), ptx::sdesc_add(kd, off),
                                                    idesc_s, kk > 0);
                                    }
                                    ptx::mma_commit(ptx::smem_addr(&bars->s_full[t]));
                                }
                                __syncwarp();
                            }
                        }
                        if (!ok) break;
                        if (has_k && !k_ready) {
                            // (every key tile of the unit belongs to a Q tile; kept for the ring)
                            ok = warp_wait(ptx::smem_addr(&bars->k_full[sk]), (uint32_t)(xk / C::NS) & 1u,
                                           abort_flag, err, kDevTimeoutLoad);
                            if (!ok) break;
                        }
                        if (has_v) commit(&bars->v_empty[sv]);
                        if (has_k) commit(&bars->k_empty[sk]);
                    }
                    kv += w.je_all - w.jb_all;
                    for (int t = 0; t < 2; ++t) uo[t] += (w.je(t) > w.jb(t));
                }
            }
        } else
        for (int u; ok && (u = fwd_unit_index<CAUSAL, SORTED>(blockIdx.x, ul, G, num_units)) >= 0; ++ul) {
            const FwdUnit w = fwd_unit<D, CAUSAL, WINDOW, SPLIT, SORTED, PACKED>(u, sh);
            if (w.empty()) continue;
            const int b = qn % C::NQB;
            const uint32_t qph = (uint32_t)(qn / C::NQB) & 1u;
            ++qn;
            if (warp == 1) {
                ok = warp_wait(ptx::smem_addr(&bars->q_full[b]), qph, abort_flag, err,
                               kDevTimeoutLoad);
                for (int j = w.jb_all; ok && j < w.je_all; ++j, ++kv) {
                    const int s = kv % C::NS;
                    ok = warp_wait(ptx::smem_addr(&bars->k_full[s]), (uint32_t)(kv / C::NS) & 1u,
                                   abort_flag, err, kDevTimeoutLoad);
                    for (int t = 0; ok && t < 2; ++t) {
                        if (j < w.jb(t) || j >= w.je(t)) continue;
                        if (it[t] > 0) {
                            // S_t may be overwritten once the softmax has read S_t (P in its own
                            // columns) or once O_t += P_t V has consumed P_t (P over S).
                            const uint32_t rel = C::P_SEPARATE ? ptx::smem_addr(&bars->s_free[t])
                                                               : ptx::smem_addr(&bars->o_done[t]);
                            ok = warp_wait(rel, (uint32_t)(it[t] - 1) & 1u, abort_flag, err,
                                           kDevTimeoutSoftmax);
                            if (!ok) break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t d_tmem = tbase + C::s_col(t);
                        const uint64_t qd = ptx::sdesc_add(dq0, (uint32_t)(b * 2 + t) * C::TILE_BYTES);
                        const uint64_t kd = ptx::sdesc_add(dk0, (uint32_t)s * C::TILE_BYTES);
                        if (ptx::elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint32_t off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
                                ptx::mma_ss(d_tmem, ptx::sdesc_add(qd, off), ptx::sdesc_add(kd, off),
                                            idesc_s, kk > 0);
                            }
                            ptx::mma_commit(ptx::smem_addr(&bars->s_full[t]));
                        }
                        __syncwarp();
                        ++it[t];
                    }
                    if (ok) commit(&bars->k_empty[s]);
                }
            } else {
                for (int j = w.jb_all; ok && j < w.je_all; ++j, ++kv) {
                    const int s = kv % C::NS;
                    ok = warp_wait(ptx::smem_addr(&bars->v_full[s]), (uint32_t)(kv / C::NS) & 1u,
                                   abort_flag, err, kDevTimeoutLoad);
                    for (int t = 0; ok && t < 2; ++t) {
                        if (j < w.jb(t) || j >= w.je(t)) continue;
                        if (j == w.jb(t) && uo[t] > 0) {
                            // O_t is about to be overwritten: the previous unit's epilogue must
                            // have read it (o_free completes once per unit in which tile t ran).
                            ok = warp_wait(ptx::smem_addr(&bars->o_free[t]),
                                           (uint32_t)(uo[t] - 1) & 1u, abort_flag, err,
                                           kDevTimeoutSoftmax);
                            if (!ok) break;
                        }
                        ok = warp_wait(ptx::smem_addr(&bars->p_full[t]), (uint32_t)it[t] & 1u,
                                       abort_flag, err, kDevTimeoutSoftmax);
                        if (!ok) break;
                        ptx::tc_fence_after();
                        const uint32_t d_tmem = tbase + C::o_col(t);
                        const uint32_t p_tmem = tbase + C::p_col(t);
                        const uint64_t vd = ptx::sdesc_add(dv0, (uint32_t)s * C::TILE_BYTES);
                        if (ptx::elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < C::BN / 16; ++kk)
                                ptx::mma_ts(d_tmem, p_tmem + kk * 8, ptx::sdesc_add(vd, kk * 2048),
                                            idesc_o, (j > w.jb(t) || kk > 0) ? 1u : 0u);
                            ptx::mma_commit(ptx::smem_addr(&bars->o_done[t]));
                        }
                        __syncwarp();
                        ++it[t];
                    }
                    if (ok) commit(&bars->v_empty[s]);
                }
                for (int t = 0; t < 2; ++t) uo[t] += (w.je(t) > w.jb(t));
            }
        }
        // Every MMA this warp issued (and every commit arrive) must be done before TMEM and
        // the barriers are released (mma_final expects one arrive per issuing warp).
        commit(&bars->mma_final);
        drain_wait(ptx::smem_addr(&bars->mma_final), 0);
    } else if (warp >= 4) {
        // ============================ softmax + epilogue ==============================
        const int t = (warp - 4) >> 2;  // Q tile of this warpgroup
        const int wq = warp & 3;        // TMEM lane quarter
        const int r = wq * 32 + lane;   // row within the tile
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t t_s = tbase + lane_off + C::s_col(t);
        const uint32_t t_p = tbase + lane_off + C::p_col(t);
        const uint32_t t_o = tbase + lane_off + C::o_col(t);
        // Q buffer whose staged output is still being read by its TMA store (thread r == 0
        // only; -1: none). The buffer is released to the producer once the read is done.
        int rel_pending = -1;
        auto release_staging = [&]() {
            if (rel_pending >= 0) {
                ptx::bulk_wait_read_all();
                ptx::mbar_arrive(ptx::smem_addr(&bars->q_free[rel_pending]));
                rel_pending = -1;
            }
        };
        const uint32_t b_s_full = ptx::smem_addr(&bars->s_full[t]);
        const uint32_t b_s_free = ptx::smem_addr(&bars->s_free[t]);
        const uint32_t b_p_full = ptx::smem_addr(&bars->p_full[t]);
        const uint32_t b_o_done = ptx::smem_addr(&bars->o_done[t]);
        int it = 0;  // score tiles of this Q tile processed so far (all units)
        int ul = 0;
        int qn = 0;  // non-empty units (Q-buffer uses)
        bool ok = true;
        for (int u; ok && (u = fwd_unit_index<CAUSAL, SORTED>(blockIdx.x, ul, G, num_units)) >= 0; ++ul) {
            const FwdUnit w = fwd_unit<D, CAUSAL, WINDOW, SPLIT, SORTED, PACKED>(u, sh);
            const int jb = w.jb(t), je = w.je(t);
            const int n = je - jb;
            const bool unit_empty = w.empty();
            const int b = qn % C::NQB;
            const uint32_t qph = (uint32_t)(qn / C::NQB) & 1u;
            qn += unit_empty ? 0 : 1;
            const int row0 = w.row0 + t * C::BM;
            const int row = row0 + r;
            const int pos = sh.offset + (PACKED ? row % sh.tq_pos : row);  // this row's key position
            int tp0 = row0, tp1 = min(row0 + C::BM, sh.Tq) - 1;  // the tile's extreme positions
            if (PACKED) tile_positions(row0, tp1, sh.tq_pos, tp0, tp1);
            const int pos_first = sh.offset + tp0;
            const int pos_last = sh.offset + tp1;
            // Keys [vis_lo, vis_hi] are visible to this row.
            const int vis_lo = WINDOW ? max(0, pos - sh.window) : 0;
            const int vis_hi = CAUSAL ? min(pos, sh.Tk - 1) : sh.Tk - 1;
            // A warp whose rows all lie past Tq skips the per-step arithmetic (its P rows feed only
            // O rows that are never stored) but keeps every barrier step with the others.
            const bool live = !SPLIT || (row0 + wq * 32) < sh.Tq;
            // partial-result row of this thread (split mode): [split][B*Hq][Tq]
            const size_t prow = ((size_t)w.split * sh.BHq + w.bh_q) * (size_t)sh.Tq + row;
            if (n == 0) {
                // No key tile of this Q tile in this unit (rows past Tq, or an empty split
                // chunk). A unit empty for both tiles has no Q-buffer use. Otherwise release
                // this tile's share of the buffer: first wait for this use's Q load, so that
                // the arrival counts towards this use and cannot complete an earlier use's
                // phase ahead of the other tile's epilogue (an mbarrier counts arrivals, not
                // arrivers).
                if (SPLIT && row < sh.Tq) part_lse[prow] = -INFINITY;  // merge skips it
                if (unit_empty) continue;
                ok = __all_sync(0xffffffffu, wait_phase(ptx::smem_addr(&bars->q_full[b]), qph,
                                                        abort_flag, err, kDevTimeoutLoad));
                if (!ok) break;
                if (r == 0) {
                    release_staging();
                    ptx::mbar_arrive(ptx::smem_addr(&bars->q_free[b]));
                }
                continue;
            }
            // Online softmax: m_ref (scaled log2 domain) moves when the row max exceeds it by
            // more than the threshold (kRefLag); when it moves, both l and the accumulator are rescaled by
            // alpha = exp2(m_old - m_new). O is rescaled only when some row of the warp moved.
            float m_ref = -INFINITY;  // reference (scaled log2 domain)
            float m_raw = -INFINITY;  // lagging reference: largest visible raw score of the row
            float l = 0.f;            // running sum of exp2(c*s - m_ref)
            if (!live) {
                // rows all past Tq: only the barrier steps (see above)
                for (int j = jb; j < je; ++j, ++it) {
                    ok = __all_sync(0xffffffffu, wait_phase(b_s_full, (uint32_t)it & 1u, abort_flag,
                                                            err, kDevTimeoutMma));
                    if (!ok) break;
                    ptx::tc_fence_after();
                    if (C::P_SEPARATE) {
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(b_s_free);
                    }
                    if (j > jb) {
                        ok = __all_sync(0xffffffffu, wait_phase(b_o_done, (uint32_t)(it - 1) & 1u,
                                                                abort_flag, err, kDevTimeoutMma));
                        if (!ok) break;
                    }
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(b_p_full);
                }
            } else
            for (int j = jb; j < je; ++j, ++it) {
                ok = __all_sync(0xffffffffu, wait_phase(b_s_full, (uint32_t)it & 1u, abort_flag, err,
                                                        kDevTimeoutMma));
                if (!ok) break;
                ptx::tc_fence_after();
                float s[C::BN];
                {
                    uint32_t u0[32], u1[32], u2[32], u3[32];
                    ptx::tmem_ld32_nowait(t_s + 0, u0);
                    ptx::tmem_ld32_nowait(t_s + 32, u1);
                    ptx::tmem_ld32_nowait(t_s + 64, u2);
                    ptx::tmem_ld32_nowait(t_s + 96, u3);
                    ptx::tmem_wait_ld(u0);
                    ptx::tmem_wait_ld(u1);
                    ptx::tmem_wait_ld(u2);
                    ptx::tmem_wait_ld(u3);
                    if (C::P_SEPARATE) {
                        // S_t is in registers: the next S_t may be computed into its columns
                        // while this step's softmax runs.
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(b_s_free);
                    }
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        s[k] = __uint_as_float(u0[k]);
                        s[32 + k] = __uint_as_float(u1[k]);
                        s[64 + k] = __uint_as_float(u2[k]);
                        s[96 + k] = __uint_as_float(u3[k]);
                    }
                }
                const int key0 = j * C::BN;
                // Elementwise masking only on tiles that cross the causal diagonal, the window's
                // left edge or the end of the keys.
                const bool need_mask = (key0 + C::BN > sh.Tk) ||
                                       (CAUSAL && key0 + C::BN - 1 > pos_first) ||
                                       (WINDOW && key0 < pos_last - sh.window);
                if (need_mask) {
                    const int klo = vis_lo - key0;
                    const uint32_t span = (uint32_t)(vis_hi - vis_lo);
#pragma unroll
                    for (int k = 0; k < C::BN; ++k)
                        if ((uint32_t)(k - klo) > span) s[k] = -INFINITY;
                }
                // Row max: four independent chains of three-input max.
                float a0 = s[0], a1 = s[1], a2 = s[2], a3 = s[3];
#pragma unroll
                for (int k = 4; k < C::BN - 4; k += 8) {
                    a0 = ptx::fmax3(a0, s[k + 0], s[k + 1]);
                    a1 = ptx::fmax3(a1, s[k + 2], s[k + 3]);
                    a2 = ptx::fmax3(a2, s[k + 4], s[k + 5]);
                    a3 = ptx::fmax3(a3, s[k + 6], s[k + 7]);
                }
                a0 = ptx::fmax3(a0, s[C::BN - 4], s[C::BN - 3]);
                a1 = ptx::fmax3(a1, s[C::BN - 2], s[C::BN - 1]);
                const float mx = ptx::fmax3(a0, a1, fmaxf(a2, a3));
                const float mc = mx * c;
                const bool upd = mc > m_ref + kRefLag;  // false when the tile is fully masked
                // the warp's rare-rescale decision, taken here rather than after the exponentials:
                // the vote at that point cost 3-7 % of d=64 forward time (B4 H16 N2048: 899 -> 924
                // TFLOP/s, B2 H16 N8192: 1094 -> 1170) by constraining the exp loop's schedule
                const bool warp_upd = __any_sync(0xffffffffu, upd);
                m_raw = fmaxf(m_raw, mx);
                float alpha = 1.f;
                if (upd) {
                    alpha = ptx::ex2_approx(m_ref - mc);  // 0 on the first visible tile
                    m_ref = mc;
                }
                const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;  // safe reference
                if (j > jb) {
                    // P_t's columns are free and O_t stable once O_t += P_t(j-1) V is complete
                    // (issued at the end of the previous step, so normally done by now): P is
                    // then written to TMEM piece by piece while the exponentials are computed.
                    ok = __all_sync(0xffffffffu, wait_phase(b_o_done, (uint32_t)(it - 1) & 1u,
                                                            abort_flag, err, kDevTimeoutMma));
                    if (!ok) break;
                    ptx::tc_fence_after();
                }
                // p = exp2(c*s - m_ref) (packed FMA, then ex2), row sum over eight partials.
                float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f, r4 = 0.f, r5 = 0.f, r6 = 0.f, r7 = 0.f;
                uint32_t pk[C::BN / 2];
#pragma unroll
                for (int k = 0; k < C::BN; k += 8) {
                    ptx::ffma2(s[k + 0], s[k + 1], s[k + 0], s[k + 1], c, c, neg_m, neg_m);
                    ptx::ffma2(s[k + 2], s[k + 3], s[k + 2], s[k + 3], c, c, neg_m, neg_m);
                    ptx::ffma2(s[k + 4], s[k + 5], s[k + 4], s[k + 5], c, c, neg_m, neg_m);
                    ptx::ffma2(s[k + 6], s[k + 7], s[k + 6], s[k + 7], c, c, neg_m, neg_m);
#pragma unroll
                    for (int i = 0; i < 8; ++i) s[k + i] = ptx::ex2_approx(s[k + i]);
                    ptx::fadd2(r0, r1, r0, r1, s[k + 0], s[k + 1]);
                    ptx::fadd2(r2, r3, r2, r3, s[k + 2], s[k + 3]);
                    ptx::fadd2(r4, r5, r4, r5, s[k + 4], s[k + 5]);
                    ptx::fadd2(r6, r7, r6, r7, s[k + 6], s[k + 7]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) pk[k / 2 + i] = ptx::pack_bf16x2(s[k + 2 * i], s[k + 2 * i + 1]);
                    if ((k & 31) == 24) {
                        // 32 keys done: their 16 packed columns of P go to TMEM now
                        uint32_t chunk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) chunk[i] = pk[k / 2 - 12 + i];
                        ptx::tmem_st16(t_p + (k / 2 - 12), chunk);
                    }
                }
                l = l * alpha + (((r0 + r1) + (r2 + r3)) + ((r4 + r5) + (r6 + r7)));
                // rare: some row of the warp moved its reference, so O_t is rescaled
                if (j > jb && warp_upd) {
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[32];
                        ptx::tmem_ld32(t_o + cc * 32, o);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            float x0, x1;
                            ptx::fmul2(x0, x1, __uint_as_float(o[i]), __uint_as_float(o[i + 1]), alpha, alpha);
                            o[i] = __float_as_uint(x0);
                            o[i + 1] = __float_as_uint(x1);
                        }
                        ptx::tmem_st32(t_o + cc * 32, o);
                    }
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(b_p_full);
                if (j == jb) release_staging();
            }
            if (!ok) break;
            // Lagging reference: normalise O by the sum of the weights as the PV product used
            // them, l with the dominant weight p_M replaced by its bf16 value (see kRefLag).
            float l_o = l;
            if (m_ref != -INFINITY) {
                const float p_m = ptx::ex2_approx(fmaf(m_raw, c, -m_ref));
                l_o = l + (__bfloat162float(__float2bfloat16_rn(p_m)) - p_m);
            }
            // ---- epilogue: O = a / l as bf16 into this tile's part of the Q buffer, TMA store ----
            ok = __all_sync(0xffffffffu, wait_phase(b_o_done, (uint32_t)(it - 1) & 1u, abort_flag,
                                                    err, kDevTimeoutMma));
            if (!ok) break;
            ptx::tc_fence_after();
            uint32_t o_all[D];  // (loaded by every warp: a branch here costs registers)
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                ptx::tmem_ld32(t_o + cc * 32, o);
#pragma unroll
                for (int i = 0; i < 32; ++i) o_all[cc * 32 + i] = o[i];
            }
            // O_t is in registers: the next unit's first O_t += P V may overwrite it.
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_addr(&bars->o_free[t]));
            if (SPLIT) {
                // Partial result of this key chunk ("15. FlashAttention", section "Decode is
                // different: flash-decoding"): the normalised O_s = a_s / l_s in fp32 and
                // LSE_s = m_s + ln l_s, merged later by weights exp(LSE_s - LSE). A row that
                // sees no key of the chunk gets LSE_s = -inf (the merge skips it).
                if (live && row < sh.Tq) {
                    const bool any = l > 0.f;
                    const float inv_l = any ? 1.f / l_o : 0.f;
                    float4* dst = reinterpret_cast<float4*>(part_o + prow * D);
#pragma unroll
                    for (int e = 0; e < D; e += 4)
                        dst[e / 4] = make_float4(__uint_as_float(o_all[e]) * inv_l,
                                                 __uint_as_float(o_all[e + 1]) * inv_l,
                                                 __uint_as_float(o_all[e + 2]) * inv_l,
                                                 __uint_as_float(o_all[e + 3]) * inv_l);
                    part_lse[prow] = any ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
                }
                // no staging: this tile's share of the Q buffer is free once its MMAs are done
                if (r == 0) ptx::mbar_arrive(ptx::smem_addr(&bars->q_free[b]));
                continue;
            }
            const float inv_l = 1.f / l_o;
            uint8_t* stage = smem + C::OFF_Q + (b * 2 + t) * C::TILE_BYTES;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint8_t* chunk = stage + (cc >> 1) * C::CHUNK_BYTES;
#pragma unroll
                for (int uu = 0; uu < 4; ++uu) {
                    const uint32_t* o = o_all + cc * 32 + 8 * uu;
                    uint4 wv;
                    wv.x = ptx::pack_bf16x2(__uint_as_float(o[0]) * inv_l, __uint_as_float(o[1]) * inv_l);
                    wv.y = ptx::pack_bf16x2(__uint_as_float(o[2]) * inv_l, __uint_as_float(o[3]) * inv_l);
                    wv.z = ptx::pack_bf16x2(__uint_as_float(o[4]) * inv_l, __uint_as_float(o[5]) * inv_l);
                    wv.w = ptx::pack_bf16x2(__uint_as_float(o[6]) * inv_l, __uint_as_float(o[7]) * inv_l);
                    *reinterpret_cast<uint4*>(chunk + sw128_offset((uint32_t)r, (uint32_t)((cc & 1) * 4 + uu))) = wv;
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::named_bar_sync(1 + t, C::BM);
            if (row < sh.Tq) lse_out[(size_t)w.bh_q * sh.Tq + row] = (m_ref + __log2f(l)) * kLn2;
            if (r == 0) {
                for (int ch = 0; ch < C::DCH; ++ch)
                    ptx::tma_store_3d(&tm_o, ptx::smem_addr(stage + ch * C::CHUNK_BYTES), ch * 64,
                                      row0, w.bh_q);
                ptx::bulk_commit();
                // The staging area (this tile's half of Q buffer b) may be reloaded once the
                // store has read it. With two Q buffers the next unit's Q is already in the
                // other one, so the release waits until after this tile's next step (or its
                // next unit without keys, or the end) and the store's read is not waited for
                // here; with one Q buffer the next unit's Q load needs the release now.
                rel_pending = b;
                if (C::NQB < 2) release_staging();
            }
        }
        release_staging();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tbase, C::TMEM_COLS);
    }
}

// ----------------------------------------------------------------------------------------
// Merge of the split partials ("15. FlashAttention", section "Decode is different:
// flash-decoding"): with normalised partials O_s and LSE_s = m_s + ln l_s the page's rule
// m = max m_s, l = sum e^(m_s - m) l_s, a = sum e^(m_s - m) a_s, O = a / l becomes
// LSE = M + ln sum_s e^(LSE_s - M) and O = sum_s e^(LSE_s - LSE) O_s (M = max_s LSE_s).
// One warp per query row; each lane owns D/32 columns. Splits with LSE_s = -inf saw no key
// (their partial O is not written). Lane s % 32 loads LSE_s (nsplit <= 64, two per lane), so the
// max and the weights need no chain of dependent loads, and the partial rows of all splits are
// loaded independently of one another (a loop that read LSE_s before each row's partial took
// ~11 us for 16 splits of 32 rows).
// ----------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256)
fa_fwd_merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                    __nv_bfloat16* __restrict__ o, float* __restrict__ lse, long long rows,
                    int nsplit) {
    constexpr int E = D / 32;
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    ptx::griddep_wait();  // the partials of the attention kernel (this one may launch early)
    if (row >= rows) return;
    const float ls0 = lane < nsplit ? part_lse[(size_t)lane * rows + row] : -INFINITY;
    const float ls1 = lane + 32 < nsplit ? part_lse[(size_t)(lane + 32) * rows + row] : -INFINITY;
    float mx = fmaxf(ls0, ls1);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float sum = 0.f;
    if (mx != -INFINITY) {
        const float w0 = (ls0 == -INFINITY) ? 0.f : expf(ls0 - mx);
        const float w1 = (ls1 == -INFINITY) ? 0.f : expf(ls1 - mx);
        sum = w0 + w1;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
#pragma unroll 4
        for (int sp = 0; sp < nsplit; ++sp) {
            const float wgt = __shfl_sync(0xffffffffu, sp < 32 ? w0 : w1, sp & 31);
            const float* src = part_o + ((size_t)sp * rows + row) * D + lane * E;
            float x[E];
            if constexpr (E == 4) {
                const float4 t4 = *reinterpret_cast<const float4*>(src);
                x[0] = t4.x;
                x[1] = t4.y;
                x[2] = t4.z;
                x[3] = t4.w;
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) x[e] = src[e];
            }
            // a split without keys contributes nothing (its row of partials is not written)
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = fmaf(wgt, wgt != 0.f ? x[e] : 0.f, acc[e]);
        }
    }
    const float inv = (sum > 0.f) ? 1.f / sum : 0.f;
    __nv_bfloat16* dst = o + (size_t)row * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2)
        *reinterpret_cast<uint32_t*>(dst + e) = ptx::pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
    if (lane == 0) lse[row] = (sum > 0.f) ? mx + logf(sum) : -INFINITY;
}

// Causal sorted order: L2 budget for the K/V of one chunk, and the largest launch (in units
// per SM) that uses it without a window. Measured: up to 16 units per SM the sorted order wins
// by 10-90 % (the pairs order leaves SMs idle in its last round); at 27 and 54 units per SM
// (B1 H64 N16384, B8 H32 N8192, d=128) it is even or up to 2 % slower (L2 reuse).
constexpr long long kFwdChunkL2Bytes = 128LL << 20;
constexpr long long kSortedMaxRounds = 16;

template <int D, bool CAUSAL, bool WINDOW, bool SPLIT, bool SORTED, bool PACKED>
cudaError_t run_fwd_kernel(const FwdLaunch& a, const FwdShape& sh, int units, cudaStream_t stream) {
    using C = FwdCfg<D>;
    auto kern = fa_fwd_kernel<D, CAUSAL, WINDOW, SPLIT, SORTED, PACKED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int grid = std::min(units, std::max(1, a.num_sms));
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o, sh, units,
                                                      a.c, a.lse, a.part_o, a.part_lse, a.err);
    return cudaGetLastError();
}

template <int D, bool CAUSAL, bool WINDOW, bool SPLIT>
cudaError_t launch_fwd_t(const FwdLaunch& a, cudaStream_t stream) {
    static_assert(CAUSAL || !WINDOW, "a window hangs off the causal diagonal");
    using C = FwdCfg<D>;
    cudaError_t e = cudaSuccess;
    FwdShape sh;
    sh.Tq = a.Tq;
    sh.Tk = a.Tk;
    sh.Hq = a.Hq;
    sh.Hkv = a.Hkv;
    sh.group = a.Hq / a.Hkv;
    sh.tq_pos = a.tq_pos;
    sh.offset = a.Tk - a.tq_pos;
    sh.window = a.window;
    sh.nqb = (a.Tq + C::ROWS - 1) / C::ROWS;
    sh.nsplit = SPLIT ? a.nsplit : 1;
    sh.BHq = a.BHq;
    long long units = (long long)sh.nqb * a.BHq * sh.nsplit;
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // Persistent grid: one CTA per SM (the shared-memory footprint admits no more), each
    // walking its units in the order fwd_unit_index gives.
    const long long sms = std::max(1, a.num_sms);
    sh.full_units = (int)units;
    sh.q_chunk = 1;
    const bool packed = a.tq_pos != a.Tq;  // query heads packed (short blocks): few units
    const bool sorted = CAUSAL && (packed || SPLIT || WINDOW || units <= kSortedMaxRounds * sms);
    if (sorted) {
        // Sorted order: few rounds (the tail of the pairs order costs up to a round), a window
        // (block costs are not linear in the block index, so pairs are unequal) or key splits
        // (a block's equal chunks must go to different SMs).
        // K and V bytes a query head reads (its KV head's, shared by the group):
        const long long per_head = std::max(1LL, 2LL * a.Tk * D * 2 / std::max(1, sh.group));
        sh.q_chunk = (int)std::max(1LL, std::min<long long>(a.BHq, kFwdChunkL2Bytes / per_head));
    }
    if (!CAUSAL && !SPLIT) {
        // Equal units: a last round at most half full runs as half units (one Q tile each)
        // on twice as many SMs; a one-tile unit takes ~81 % of a two-tile unit's time.
        const long long rem = units % sms;
        if (units > sms && rem > 0 && 2 * rem <= sms) {
            sh.full_units = (int)(units - rem);
            units += rem;
        }
    }
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // Kernel variants: non-causal launches use the round robin; windowed, split and packed
    // causal launches always use the sorted order; plain causal launches use either. Packing
    // is a variant of its own (its row positions cost the other kernels 2-4 % at run time).
    if (packed)
        e = run_fwd_kernel<D, CAUSAL, WINDOW, SPLIT, CAUSAL, true>(a, sh, (int)units, stream);
    else if constexpr (!CAUSAL)
        e = run_fwd_kernel<D, CAUSAL, WINDOW, SPLIT, false, false>(a, sh, (int)units, stream);
    else if constexpr (WINDOW || SPLIT)
        e = run_fwd_kernel<D, CAUSAL, WINDOW, SPLIT, true, false>(a, sh, (int)units, stream);
    else
        e = sorted ? run_fwd_kernel<D, CAUSAL, WINDOW, SPLIT, true, false>(a, sh, (int)units, stream)
                   : run_fwd_kernel<D, CAUSAL, WINDOW, SPLIT, false, false>(a, sh, (int)units, stream);
    if (e != cudaSuccess || !SPLIT) return e;
    const long long rows = (long long)a.BHq * a.Tq;
    const long long blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return launch_dependent(fa_fwd_merge_kernel<D>, dim3((unsigned)blocks), dim3(256), 0, stream,
                            static_cast<const float*>(a.part_o), static_cast<const float*>(a.part_lse),
                            static_cast<__nv_bfloat16*>(a.o), a.lse, rows, sh.nsplit);
}

}  // namespace

template <int D>
cudaError_t launch_fwd_mask(const FwdLaunch& a, bool causal, bool window, bool split,
                            cudaStream_t stream) {
    if (split) {
        if (!causal) return launch_fwd_t<D, false, false, true>(a, stream);
        return window ? launch_fwd_t<D, true, true, true>(a, stream)
                      : launch_fwd_t<D, true, false, true>(a, stream);
    }
    if (!causal) return launch_fwd_t<D, false, false, false>(a, stream);
    return window ? launch_fwd_t<D, true, true, false>(a, stream)
                  : launch_fwd_t<D, true, false, false>(a, stream);
}

// The build compiles this file once per head dimension (FA_FWD_D = 64, 128) so the two sets of
// kernel variants compile in parallel; without the macro one object carries both.
#if !defined(FA_FWD_D) || FA_FWD_D == 64
cudaError_t launch_forward_d64(const FwdLaunch& a, bool causal, cudaStream_t stream) {
    if (a.window >= 0 && !causal) return cudaErrorInvalidValue;
    return launch_fwd_mask<64>(a, causal, a.window >= 0, a.nsplit > 1, stream);
}
#endif
#if !defined(FA_FWD_D) || FA_FWD_D == 128
cudaError_t launch_forward_d128(const FwdLaunch& a, bool causal, cudaStream_t stream) {
    if (a.window >= 0 && !causal) return cudaErrorInvalidValue;
    return launch_fwd_mask<128>(a, causal, a.window >= 0, a.nsplit > 1, stream);
}
#endif

}  // namespace fa
