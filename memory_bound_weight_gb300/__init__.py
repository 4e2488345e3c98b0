"""GB300 (sm_103a) weight-streaming GEMV library: y = W.x and Y = X.W^T with
BF16, INT4 group-64, AWQ-style INT4 group-128 and symmetric per-channel INT8
weights.

The compute path is libmbw.so (C ABI in include/mbw.h); this package is its
binding. Submodules ``inputs`` and ``workloads`` (synthetic data and byte
accounting) import without loading the CUDA library.
"""
_EXPORTS = (
    "gemv_bf16", "gemv_int4_g64", "gemv_int4_awq_g128", "gemm_skinny_bf16", "gemv_int8_pc", "quantize_int8_pc",
    "gemv_fused", "gemv_fused_awq_g128", "MbwFusion", "FUSE_NORM", "FUSE_GLU", "FUSE_RESIDUAL", "repack_int4", "REPACKED",
    "dequant_int4_g64", "dequant_int4_awq_g128", "autotune", "plan_describe", "plan_candidates", "plan_select", "plan_index", "workspace_bytes",
    "launch_count", "check_device_error", "selftest_wait_expiry", "inject_launch_failures", "output_fp32", "MbwError",
    "OP_GEMV_BF16", "OP_GEMV_INT4_G64", "OP_GEMV_INT4_AWQ_G128", "OP_GEMM_SKINNY_BF16",
    "OP_GEMV_INT8_PC",
)


_PLAN_FILES = ("save_plans", "load_plans")


def __getattr__(name):
    if name in _EXPORTS:
        from . import _binding

        return getattr(_binding, name)
    if name in _PLAN_FILES:
        from . import plans

        return getattr(plans, name)
    raise AttributeError(name)
