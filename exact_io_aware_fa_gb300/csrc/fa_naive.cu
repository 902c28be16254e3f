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

// One warp per row of S (fp32, raw dot products). Safe softmax: m = max over visible scaled
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

}  // namespace
}  // namespace fa

namespace fa {
cudaError_t launch_naive_softmax(const float* s, void* p, float* lse, long long rows, int N,
                                 int causal, float scale, cudaStream_t stream) {
    const long long blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    fa_naive_softmax_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        s, static_cast<__nv_bfloat16*>(p), lse, rows, N, causal, scale);
    return cudaGetLastError();
}
}  // namespace fa
