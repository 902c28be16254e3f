// fa_naive.cu -- the row softmax of naive (materialised) attention, the comparison point the
// IO-aware method is measured against ("15. FlashAttention", inference.shantanugoel.com,
// sections "The score matrix is the problem" and "Stretch exercises" item 1; "FlashAttention
// V1", infra.bea.ai, the standard-attention baseline): the full score matrix S = Q K^T is
// written to HBM by one GEMM, this kernel reads it back, applies the scale and the causal mask,
// and writes P = softmax(S) (bf16, as the page's reference casts p to V's dtype) and the row
// log-sum-exp, and a second GEMM reads P back for O = P V. Not part of the IO-aware path.
#include <cuda_bf16.h>
#include <stdint.h>

#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {
namespace {

// One warp per row of S (fp32, raw dot products), for rows too long to hold in registers (and
// rows over 1024 keys whose N is not a multiple of 4).
// Safe softmax: m = max over visible scaled
// scores, l = sum exp(s - m), P = exp(s - m) / l, LSE = m + ln l ("FlashAttention: from
// IO-Aware Attention to GPU work partitioning", blog.euler0525.cn, section "Online Softmax",
// the definitions of m, l and p). m and l come from one online pass over the row (each lane
// keeps a running (m, l) and rescales l when its maximum grows; the lanes' pairs are merged the
// same way), so S is read twice: once for (m, l), once to write P. Masked entries get P = 0.
__global__ void __launch_bounds__(256)
fa_naive_softmax_kernel(const float* __restrict__ s, __nv_bfloat16* __restrict__ p,
                        float* __restrict__ lse, long long rows, int N, int causal, float scale) {
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int i = (int)(row % N);              // query index within its head
    const int nvis = causal ? i + 1 : N;       // keys 0 .. nvis - 1 are visible
    const float* sr = s + row * (long long)N;
    __nv_bfloat16* pr = p + row * (long long)N;
    float m = -INFINITY, l = 0.f;
    for (int j = lane; j < nvis; j += 32) {
        const float x = sr[j] * scale;
        if (x > m) {
            l = l * expf(m - x) + 1.f;        // expf(-inf) = 0 on a lane's first key
            m = x;
        } else {
            l += expf(x - m);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, off);
        const float lo = __shfl_xor_sync(0xffffffffu, l, off);
        const float mn = fmaxf(m, mo);
        // a lane that saw no key has (m, l) = (-inf, 0) and contributes nothing
        l = (m == -INFINITY ? 0.f : l * expf(m - mn)) + (mo == -INFINITY ? 0.f : lo * expf(mo - mn));
        m = mn;
    }
    const float inv = 1.f / l;
    for (int j = lane; j < N; j += 32)
        pr[j] = __float2bfloat16_rn(j < nvis ? expf(sr[j] * scale - m) * inv : 0.f);
    if (lane == 0) lse[row] = m + logf(l);
}

// Rows of at most 32 * CPL (<= 1024) scores: one warp per row, the row read once into registers
// (CPL per lane), so S is read once and P written once. VEC = 4 (N a multiple of 4): lane l holds columns
// 4 (l + 32 t) .. + 3, read as one 16-byte load and written as one 8-byte store of four bf16;
// VEC = 1: columns l + 32 t.
template <int CPL, int VEC>
__global__ void __launch_bounds__(128)
fa_naive_softmax_reg_kernel(const float* __restrict__ s, __nv_bfloat16* __restrict__ p,
                            float* __restrict__ lse, long long rows, int N, int causal,
                            float scale) {
    constexpr int NV = CPL / VEC;  // vectors per lane
    const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int i = (int)(row % N);
    const int nvis = causal ? i + 1 : N;
    const float* sr = s + row * (long long)N;
    __nv_bfloat16* pr = p + row * (long long)N;
    float x[CPL];
#pragma unroll
    for (int t = 0; t < NV; ++t) {
        const int j0 = (lane + 32 * t) * VEC;
        if (VEC == 4) {
            float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j0 < nvis) f = *reinterpret_cast<const float4*>(sr + j0);
            x[4 * t] = f.x;
            x[4 * t + 1] = f.y;
            x[4 * t + 2] = f.z;
            x[4 * t + 3] = f.w;
        } else {
            x[t] = (j0 < nvis) ? sr[j0] : 0.f;
        }
    }
    float m = -INFINITY;
#pragma unroll
    for (int t = 0; t < NV; ++t)
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const int j = (lane + 32 * t) * VEC + v;
            x[VEC * t + v] = (j < nvis) ? x[VEC * t + v] * scale : -INFINITY;
            m = fmaxf(m, x[VEC * t + v]);
        }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float l = 0.f;
#pragma unroll
    for (int t = 0; t < NV; ++t)
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const int j = (lane + 32 * t) * VEC + v;
            x[VEC * t + v] = (j < nvis) ? expf(x[VEC * t + v] - m) : 0.f;
            l += x[VEC * t + v];
        }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    const float inv = 1.f / l;
#pragma unroll
    for (int t = 0; t < NV; ++t) {
        const int j0 = (lane + 32 * t) * VEC;
        if (j0 >= N) continue;
        if (VEC == 4) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(x[4 * t] * inv, x[4 * t + 1] * inv);
            __nv_bfloat162 hi = __floats2bfloat162_rn(x[4 * t + 2] * inv, x[4 * t + 3] * inv);
            uint2 w;
            w.x = *reinterpret_cast<uint32_t*>(&lo);
            w.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(pr + j0) = w;
        } else {
            pr[j0] = __float2bfloat16_rn(x[t] * inv);
        }
    }
    if (lane == 0) lse[row] = m + logf(l);
}

// Rows of 1024 < N <= 1024 * VPT keys with N a multiple of 4: one 256-thread block per row,
// each thread holding VPT float4 of it (columns 4 (t + 256 v) .. + 3), block-wide max and sum
// through shared memory; S is read once and P written once.
template <int VPT>
__global__ void __launch_bounds__(256)
fa_naive_softmax_block_kernel(const float* __restrict__ s, __nv_bfloat16* __restrict__ p,
                              float* __restrict__ lse, int N, int causal, float scale) {
    __shared__ float red[8];
    const long long row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int i = (int)(row % N);
    const int nvis = causal ? i + 1 : N;
    const float* sr = s + row * (long long)N;
    __nv_bfloat16* pr = p + row * (long long)N;
    float x[4 * VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int j0 = 4 * (tid + 256 * v);
        float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j0 < N) f = *reinterpret_cast<const float4*>(sr + j0);
        x[4 * v] = f.x;
        x[4 * v + 1] = f.y;
        x[4 * v + 2] = f.z;
        x[4 * v + 3] = f.w;
    }
    float m = -INFINITY;
#pragma unroll
    for (int e = 0; e < 4 * VPT; ++e) {
        const int j = 4 * (tid + 256 * (e / 4)) + (e % 4);
        x[e] = (j < nvis) ? x[e] * scale : -INFINITY;
        m = fmaxf(m, x[e]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
    __syncthreads();  // every thread has read red before it is reused for the sums
    float l = 0.f;
#pragma unroll
    for (int e = 0; e < 4 * VPT; ++e) {
        x[e] = (x[e] == -INFINITY) ? 0.f : expf(x[e] - m);
        l += x[e];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    if (lane == 0) red[warp] = l;
    __syncthreads();
    l = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) l += red[w];
    const float inv = 1.f / l;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int j0 = 4 * (tid + 256 * v);
        if (j0 >= N) continue;
        __nv_bfloat162 lo = __floats2bfloat162_rn(x[4 * v] * inv, x[4 * v + 1] * inv);
        __nv_bfloat162 hi = __floats2bfloat162_rn(x[4 * v + 2] * inv, x[4 * v + 3] * inv);
        uint2 w2;
        w2.x = *reinterpret_cast<uint32_t*>(&lo);
        w2.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(pr + j0) = w2;
    }
    if (tid == 0) lse[row] = m + logf(l);
}

}  // namespace
}  // namespace fa

namespace fa {
cudaError_t launch_naive_softmax(const float* s, void* p, float* lse, long long rows, int N,
                                 int causal, float scale, cudaStream_t stream) {
    __nv_bfloat16* pb = static_cast<__nv_bfloat16*>(p);
    // N % 4 == 0 keeps every row 16-byte aligned in S (fp32) and 8-byte aligned in P (bf16)
    if (N % 4 == 0 && N > 1024 && N <= 8192) {
        if (rows > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        const unsigned g = (unsigned)rows;
        if (N <= 2048) fa_naive_softmax_block_kernel<2><<<g, 256, 0, stream>>>(s, pb, lse, N, causal, scale);
        else if (N <= 4096) fa_naive_softmax_block_kernel<4><<<g, 256, 0, stream>>>(s, pb, lse, N, causal, scale);
        else fa_naive_softmax_block_kernel<8><<<g, 256, 0, stream>>>(s, pb, lse, N, causal, scale);
        return cudaGetLastError();
    }
    if (N > 4096 || (N % 4 != 0 && N > 1024)) {
        const long long blocks = (rows + 7) / 8;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        fa_naive_softmax_kernel<<<(unsigned)blocks, 256, 0, stream>>>(s, pb, lse, rows, N, causal, scale);
        return cudaGetLastError();
    }
    const long long blocks = (rows + 3) / 4;  // four rows (warps) per block
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const unsigned g = (unsigned)blocks;
    if (N % 4 == 0) {
        if (N <= 256) fa_naive_softmax_reg_kernel<8, 4><<<g, 128, 0, stream>>>(s, pb, lse, rows, N, causal, scale);
        else fa_naive_softmax_reg_kernel<32, 4><<<g, 128, 0, stream>>>(s, pb, lse, rows, N, causal, scale);
    } else {
        if (N <= 256) fa_naive_softmax_reg_kernel<8, 1><<<g, 128, 0, stream>>>(s, pb, lse, rows, N, causal, scale);
        else fa_naive_softmax_reg_kernel<32, 1><<<g, 128, 0, stream>>>(s, pb, lse, rows, N, causal, scale);
    }
    return cudaGetLastError();
}
}  // namespace fa
