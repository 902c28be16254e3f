"""Naive (materialised) attention on the GPU: the comparison point of the IO-aware method.

"15. FlashAttention" (inference.shantanugoel.com), sections "The score matrix is the problem"
and "Stretch exercises" item 1, and "FlashAttention V1" (infra.bea.ai) measure FlashAttention
against standard attention that writes the N x N score and probability matrices to HBM. This
module builds that baseline from library GEMMs and this library's row-softmax kernel:

  1. S = Q K^T in fp32 (torch batched GEMM; the bf16 inputs are exact in TF32, so the tensor
     core's TF32 products are exact and the sum is accumulated in fp32), stored [B*H, N, N];
  2. P = softmax(scale S) row by row and LSE (``fa_naive_softmax``, C ABI), P stored in bf16;
  3. O = P V (torch batched bf16 GEMM, fp32 accumulate).

It is used only to compare speed, DRAM traffic and peak memory with the fused kernels; it is
not part of the IO-aware path and nothing on that path calls it.
"""
from __future__ import annotations

import math

from . import api


def forward(q, k, v, causal: bool = False, scale: float | None = None):
    """O (bf16, [B,H,N,d]) and LSE (fp32, [B,H,N]) of materialised attention."""
    import torch
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("expected q, k, v of equal shape [B,H,N,d]")
    if q.dtype != torch.bfloat16 or not q.is_cuda:
        raise ValueError("expected bf16 CUDA tensors")
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        s = torch.matmul(q.reshape(B * H, N, d).float(), k.reshape(B * H, N, d).float().transpose(1, 2))
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    p = torch.empty((B * H, N, N), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    st = api.library().fa_naive_softmax(s.data_ptr(), p.data_ptr(), lse.data_ptr(), B * H * N, N,
                                        int(bool(causal)), scale,
                                        torch.cuda.current_stream(q.device).cuda_stream)
    api._check(st, "fa_naive_softmax")
    o = torch.matmul(p, v.reshape(B * H, N, d)).reshape(B, H, N, d)
    return o, lse
