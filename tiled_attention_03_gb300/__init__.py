"""GB300 (sm_103a) FlashAttention forward and backward: C-ABI library libfa.so + Python binding."""

from .binding import (FA_DTYPE_BF16, FA_DTYPE_FP16, FA_ERR_CUDA, FA_ERR_INVALID_ARG,  # noqa: F401
                      FA_ERR_TIMEOUT, FA_ERR_UNSUPPORTED, FA_MASK_CAUSAL, FA_MASK_NONE,
                      FA_MASK_WINDOW, FA_OK, FaError, fa_forward, fa_forward_gqa, fa_launch_count,
                      fa_set_wait_budget_ns, fa_status_string, fa_sync_status, fa_test_arm_fault, forward,
                      load_library, load_library_at)
from .binding import FA_DEBUG_BOUNDS_FLAG, FA_DEBUG_SERIALIZE_FLAG, FA_ERR_BOUNDS  # noqa: F401
from .binding import (FA_SPLITKV_STATIC_SCRATCH_BYTES, fa_forward_splitkv,  # noqa: F401
                      fa_forward_splitkv_static, fa_splitkv_default_splits,
                      fa_splitkv_workspace_bytes)
from .binding import backward, fa_backward, fa_backward_workspace_bytes  # noqa: F401
from .binding import fa_forward_varlen  # noqa: F401
from .binding import fa_forward_host, fa_forward_host_workspace_bytes  # noqa: F401
from .binding import fa_backward_varlen, fa_backward_varlen_workspace_bytes  # noqa: F401
