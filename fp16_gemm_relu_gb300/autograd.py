"""relu(A·B) as a differentiable torch operation whose forward and backward both run in the
library's kernels (the practitioner page, section 3.3, wraps a hand-written kernel in
torch.autograd.Function and pairs it with hand-written backward kernels).

Forward:  C = fp16(relu(A·B))                         tg_gemm_relu_f16
Backward: dZ = C > 0 ? dC : +0                        tg_relu_backward_f16
          dA = dZ·B^T  (fp32 accumulate, fp16 out)    tg_gemm_f16_t(trans_b = 1)
          dB = A^T·dZ                                  tg_gemm_f16_t(trans_a = 1)
"""

from __future__ import annotations

import torch

from . import binding


def _ld(t: torch.Tensor) -> int:
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError("expected a row-major 2-D tensor")
    return t.stride(0) if t.shape[0] > 1 else max(t.shape[1], 1)


def relu_backward(dC: torch.Tensor, C: torch.Tensor) -> torch.Tensor:
    M, N = C.shape
    dZ = torch.empty_like(C)
    s = torch.cuda.current_stream(C.device).cuda_stream
    st = binding.tg_relu_backward_f16(dC.data_ptr(), C.data_ptr(), dZ.data_ptr(), M, N,
                                      _ld(dC), _ld(C), _ld(dZ), s)
    if st != binding.TG_OK:
        raise binding.TgError(st, "tg_relu_backward_f16")
    return dZ


def gemm_t(A: torch.Tensor, B: torch.Tensor, trans_a: int, trans_b: int) -> torch.Tensor:
    """op(A)·op(B) in fp16 with fp32 accumulation (op = transpose when trans_* is 1)."""
    M = A.shape[1] if trans_a else A.shape[0]
    K = A.shape[0] if trans_a else A.shape[1]
    N = B.shape[0] if trans_b else B.shape[1]
    C = torch.empty((M, N), dtype=torch.float16, device=A.device)
    s = torch.cuda.current_stream(A.device).cuda_stream
    st = binding.tg_gemm_f16_t(trans_a, trans_b, A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N,
                               K, _ld(A), _ld(B), _ld(C), binding.TG_ACT_NONE, 0, 0, 0, None, s)
    if st != binding.TG_OK:
        raise binding.TgError(st, "tg_gemm_f16_t")
    return C


class ReluMatmul(torch.autograd.Function):
    @staticmethod
    def forward(ctx, A, B):
        C = binding.gemm_relu(A, B)
        ctx.save_for_backward(A, B, C)
        return C

    @staticmethod
    def backward(ctx, dC):
        A, B, C = ctx.saved_tensors
        dC = dC.to(torch.float16).contiguous()
        dZ = relu_backward(dC, C)
        dA = gemm_t(dZ, B, 0, 1) if ctx.needs_input_grad[0] else None
        dB = gemm_t(A, dZ, 1, 0) if ctx.needs_input_grad[1] else None
        return dA, dB


def relu_matmul(A: torch.Tensor, B: torch.Tensor) -> torch.Tensor:
    """Differentiable C = relu(A·B) for CUDA fp16 tensors."""
    return ReluMatmul.apply(A, B)
