"""GB300 (sm_103a) FlashAttention-2 backward: preprocess D = rowsum(dO * O),
then dQ, dK, dV from a tcgen05 tensor-core kernel.

The compute lives in the C-ABI library ``_build/libfa.so`` (include/fa.h);
this package is the thin Python binding over it (argument marshalling only,
via ctypes), a torch.autograd.Function over the forward and backward
(``autograd``) and the seeded input generators (``inputs``).  Functions take
torch CUDA tensors; every step of the path runs in the library's kernels.
If the library is missing or cannot be loaded the calls raise: there is no
fallback.
"""
from .binding import (  # noqa: F401
    FA_BF16,
    FA_F16,
    FA_F32,
    FaError,
    fa_bwd,
    fa_bwd_host,
    fa_bwd_noalloc,
    fa_bwd_preprocess,
    fa_bwd_workspace_bytes,
    fa_check_device,
    fa_fwd,
    fa_last_error,
    fa_profile,
    fa_profile_read,
    fa_selftest_timeout,
    fa_shutdown,
    fa_version,
    library_path,
    load_library,
)
from .autograd import FlashAttentionFunction, flash_attention  # noqa: F401
