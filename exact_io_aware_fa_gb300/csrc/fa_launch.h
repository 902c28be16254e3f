// fa_launch.h -- internal interface between the C ABI (fa_api.cu) and the kernel
// translation units. Not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

struct FwdLaunch {
    CUtensorMap tm_q, tm_k, tm_v, tm_o;  // 3-D maps over [B*H, N, d] bf16, box {64, 128, 1}
    int N;                               // sequence length
    int BH;                              // B * H
    float c;                             // scale * log2(e)
    float* lse;                          // [B*H, N] fp32
    int* err;                            // device error word
    int num_sms;                         // SMs of the device (persistent grid size)
};

// Forward: O and LSE. d in {64, 128}.
cudaError_t launch_forward(const FwdLaunch& a, int d, bool causal, cudaStream_t stream);

struct BwdLaunch {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;  // loads, box {64, rows, 1}
    CUtensorMap tm_dk, tm_dv;             // stores, box {64, 128, 1}
    CUtensorMap tm_dqacc;                 // fp32 [B*H, Npad, d] accumulator, box {32, rows, 1}
    const void* o;                        // bf16 [B*H, N, d]
    const void* dout;                     // bf16 [B*H, N, d]
    const float* lse;                     // fp32 [B*H, N]
    void* dq;                             // bf16 [B*H, N, d]
    float* stats;                         // workspace: [B*H, Npad] (LSE*log2e) then [B*H, Npad] (D)
    float* dq_acc;                        // workspace: fp32 [B*H, Npad, d]
    int N, Npad, BH, d;
    float scale;
    float c;                              // scale * log2(e)
    int* err;
};

cudaError_t launch_backward(const BwdLaunch& a, bool causal, cudaStream_t stream);

}  // namespace fa
