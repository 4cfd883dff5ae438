"""GB300-native C = relu(A·B): fp16 A (M,K) and B (K,N) row-major, float32 accumulation in
tensor memory, fp16 C.  The computation is the matmul_relu example of the TileLang
paper-reading page (section 2).

The work runs in hand-written sm_103a kernels behind a C ABI (``include/tg_gemm_relu.h``);
this package is a thin binding over that library.  There is no CPU fallback: every entry point
raises if the compiled library is missing.
"""

from .binding import (  # noqa: F401
    TG_EPILOGUE_NONE,
    TG_EPILOGUE_RELU,
    TgError,
    gemm_relu,
    gemm_relu_host,
    library_path,
    load_library,
    plan,
    tg_gemm_relu_f16,
    tg_gemm_relu_f16_ex,
    tg_gemm_relu_f16_host,
    tg_last_cuda_error,
    tg_release_workspace,
    tg_status_string,
)
