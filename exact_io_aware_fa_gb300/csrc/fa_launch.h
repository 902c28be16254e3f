// fa_launch.h -- internal interface between the C ABI (fa_api.cu) and the kernel
// translation units. Not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

struct FwdLaunch {
    CUtensorMap tm_q, tm_o;              // 3-D maps over [B*Hq, Tq, d] bf16, box {64, 128, 1}
                                         // (packed: [B*Hkv, group*Tq, d], Hq = Hkv, Tq rows)
    CUtensorMap tm_k, tm_v;              // 3-D maps over [B*Hkv, Tk, d] bf16, box {64, 128, 1}
    int Tq, Tk;                          // query rows per head block, key sequence length
    int tq_pos;                          // query positions per head (Tq unless heads are packed)
    int Hq, Hkv;                         // query heads, KV heads (Hq % Hkv == 0)
    int BHq;                             // B * Hq
    int window;                          // -1: none; else keys >= position - window (causal)
    float c;                             // scale * log2(e)
    float* lse;                          // [B*Hq, Tq] fp32
    int* err;                            // device error word
    int num_sms;                         // SMs of the device (persistent grid size)
    int nsplit;                          // key-range splits (1: none)
    void* o;                             // bf16 [B*Hq, Tq, d] (written by the split merge)
    float* part_o;                       // nsplit > 1: fp32 [nsplit, B*Hq, Tq, d] partial O
    float* part_lse;                     // nsplit > 1: fp32 [nsplit, B*Hq, Tq] partial LSE
};

// Forward: O and LSE. d in {64, 128}.
cudaError_t launch_forward_d64(const FwdLaunch& a, bool causal, cudaStream_t stream);
cudaError_t launch_forward_d128(const FwdLaunch& a, bool causal, cudaStream_t stream);
inline cudaError_t launch_forward(const FwdLaunch& a, int d, bool causal, cudaStream_t stream) {
    if (d == 64) return launch_forward_d64(a, causal, stream);
    if (d == 128) return launch_forward_d128(a, causal, stream);
    return cudaErrorInvalidValue;
}

struct BwdLaunch {
    CUtensorMap tm_q, tm_do;              // [B*Hq, Tq, d] loads, box {64, query rows, 1}
    CUtensorMap tm_k, tm_v;               // [B*Hkv, Tk, d] loads, box {64, 128, 1}
    CUtensorMap tm_dk, tm_dv;             // [B*Hkv, Tk, d] stores, box {64, 128, 1}
    CUtensorMap tm_dqacc;                 // fp32 dQ accumulator: d = 64 [B*Hq, Npad, d], box {32, rows, 1};
                                          // d = 128 transposed [B*Hq, d, Npad], box {32, 128, 1}
    const void* o;                        // bf16 [B*Hq, Tq, d]
    const void* dout;                     // bf16 [B*Hq, Tq, d]
    const float* lse;                     // fp32 [B*Hq, Tq]
    void* dq;                             // bf16 [B*Hq, Tq, d]
    void* folds;                          // workspace: per query row, 16-byte records of
                                          // -LSE/scale then of -D ([B*Hq, Npad] each)
    float* dq_acc;                        // workspace: fp32 B*Hq*Npad*d (layout: tm_dqacc)
    unsigned* sched;                      // workspace: the main kernel's unit counter
    int Tq, Tk, Npad, Hq, Hkv, BHq, BHkv, d, window;
    float scale;
    float c;                              // scale * log2(e)
    int* err;
    int num_sms;                          // SMs of the device (CTA order choice)
};

cudaError_t launch_backward(const BwdLaunch& a, bool causal, cudaStream_t stream);

// Naive (materialised) attention's row softmax over a stored score matrix (comparison only).
cudaError_t launch_naive_softmax(const float* s, void* p, float* lse, long long rows, int N,
                                 int causal, float scale, cudaStream_t stream);

}  // namespace fa
