"""Host-side checks of the Python binding (no GPU needed): tensors must sit on
one device, the current CUDA one (a kernel handed another device's memory
would fault), shapes of scales and zero points are checked before any call
reaches the library, and host tensors are refused."""
import pytest

torch = pytest.importorskip("torch")

import memory_bound_weight_gb300 as mbw  # noqa: E402
from memory_bound_weight_gb300 import _binding as B  # noqa: E402


class OnDevice:
    """Stands in for a tensor: only its device is looked at."""

    def __init__(self, dev):
        self.device = torch.device(dev)


def test_common_device():
    assert B._common_device(torch.zeros(2), None, torch.zeros(3)) == torch.device("cpu")
    with pytest.raises(ValueError, match="one device"):
        B._common_device(torch.zeros(2), torch.empty(2, device="meta"))


def test_tensors_must_be_on_the_current_cuda_device(monkeypatch):
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    assert B._on_current_device(OnDevice("cuda:0"), None, OnDevice("cuda:0")) == torch.device("cuda", 0)
    with pytest.raises(ValueError, match="current CUDA device is cuda:0"):
        B._on_current_device(OnDevice("cuda:1"), OnDevice("cuda:1"))
    with pytest.raises(ValueError, match="one device"):
        B._on_current_device(OnDevice("cuda:0"), OnDevice("cuda:1"))


def test_shape_check():
    B._need_shape(torch.zeros(2, 3), "scales", (2, 3))
    with pytest.raises(ValueError, match=r"scales must have shape \(2, 4\), got \(2, 3\)"):
        B._need_shape(torch.zeros(2, 3), "scales", (2, 4))


def test_host_tensors_are_refused():
    W = torch.zeros(4, 8, dtype=torch.bfloat16)
    x = torch.zeros(8, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        mbw.gemv_bf16(W, x)
    with pytest.raises(ValueError, match="CUDA tensor"):
        mbw.gemm_skinny_bf16(x.view(1, 8), W)


class RecordingLib:
    """Stands in for libmbw.so: records each call's name and argument count."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append((name, len(args)))
            return 0

        return fn


@pytest.fixture
def host_marshalling(monkeypatch):
    """Every public call runs its whole argument marshalling on host tensors:
    only the CUDA-tensor test and the stream lookup are bypassed, the library
    is the recorder, and the device check sees the host as the current device."""
    rec = RecordingLib()
    real_need = B._need

    def need(t, name, dtype, ndim):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != dtype or t.dim() != ndim or not t.is_contiguous():
            real_need(t, name, dtype, ndim)  # raises the real message

    monkeypatch.setattr(B, "_need", need)
    monkeypatch.setattr(B, "lib", lambda: rec)
    monkeypatch.setattr(B, "_stream_ptr", lambda device: 0)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: None)  # a host tensor's device index
    return rec


def test_every_call_marshals_valid_arguments(host_marshalling):
    u8, f16, bf, i8, f32 = torch.uint8, torch.float16, torch.bfloat16, torch.int8, torch.float32
    N, K, M = 6, 256, 3
    W = torch.zeros(N, K, dtype=bf)
    x = torch.zeros(K, dtype=bf)
    X = torch.zeros(M, K, dtype=bf)
    q4 = torch.zeros(N, K // 2, dtype=u8)
    s64 = torch.zeros(N, K // 64, dtype=f16)
    s128 = torch.zeros(N, K // 128, dtype=f16)
    z128 = torch.zeros(N, 1, dtype=u8)
    q8 = torch.zeros(N, K, dtype=i8)
    s8 = torch.zeros(N, dtype=f32)
    assert mbw.gemv_bf16(W, x).shape == (N,)
    assert mbw.gemv_int4_g64(q4, s64, x).shape == (N,)
    assert mbw.gemv_int4_awq_g128(q4, s128, z128, X).shape == (M, N)
    assert mbw.gemv_int4_awq_g128(q4, s128, z128, x, repacked=True).shape == (N,)
    assert mbw.repack_int4(q4).shape == q4.shape
    assert mbw.gemm_skinny_bf16(X, W).shape == (M, N)
    assert mbw.gemv_int8_pc(q8, s8, X).shape == (M, N)
    assert mbw.gemv_fused(mbw.OP_GEMV_BF16, W, None, x, norm_weight=x, residual=torch.zeros(N, dtype=bf),
                          up_weights=W).shape == (N,)
    assert mbw.gemv_fused(mbw.OP_GEMV_INT4_G64, q4, s64, x, up_weights=q4, up_scales=s64).shape == (N,)
    assert mbw.gemv_fused(mbw.OP_GEMV_INT8_PC, q8, s8, X, residual=torch.zeros(M, N, dtype=bf)).shape == (M, N)
    assert mbw.gemv_fused_awq_g128(q4, s128, z128, x, norm_weight=x, up_weights=q4, up_scales=s128,
                                   up_zeros=z128, residual=torch.zeros(N, dtype=bf)).shape == (N,)
    assert mbw.gemv_fused_awq_g128(q4, s128, z128, X, repacked=True).shape == (M, N)
    assert mbw.quantize_int8_pc(W)[0].shape == (N, K)
    assert mbw.dequant_int4_g64(q4, s64).shape == (N, K)
    assert mbw.dequant_int4_awq_g128(q4, s128, z128).shape == (N, K)
    names = [c[0] for c in host_marshalling.calls]
    assert names == ["gemv_bf16", "gemv_int4_g64", "gemv_int4_awq_g128", "gemv_int4_awq_g128_repacked",
                     "mbw_repack_int4", "gemm_skinny_bf16", "gemv_int8_pc", "gemv_fused", "gemv_fused",
                     "gemv_fused", "gemv_fused_awq_g128", "gemv_fused_awq_g128", "mbw_quantize_int8_pc",
                     "mbw_dequant_int4_g64", "mbw_dequant_int4_awq_g128"]
    for name, nargs in host_marshalling.calls:
        assert nargs == len(B.SIGNATURES[name][0]), name


def test_bad_scale_and_zero_shapes_never_reach_the_library(host_marshalling):
    N, K = 6, 256
    q4 = torch.zeros(N, K // 2, dtype=torch.uint8)
    x = torch.zeros(K, dtype=torch.bfloat16)
    s64 = torch.zeros(N, K // 64, dtype=torch.float16)
    with pytest.raises(ValueError, match="scales"):
        mbw.gemv_fused(mbw.OP_GEMV_INT4_G64, q4, s64[:, :2].contiguous(), x)
    with pytest.raises(ValueError, match="up_scales"):
        mbw.gemv_fused(mbw.OP_GEMV_INT4_G64, q4, s64, x, up_weights=q4, up_scales=s64[:3].contiguous())
    with pytest.raises(ValueError, match="scales"):
        mbw.gemv_fused(mbw.OP_GEMV_INT8_PC, torch.zeros(N, K, dtype=torch.int8),
                       torch.zeros(N + 1, dtype=torch.float32), x)
    with pytest.raises(ValueError, match="scales"):
        mbw.dequant_int4_g64(q4, torch.zeros(N, 1, dtype=torch.float16))
    with pytest.raises(ValueError, match="zeros"):
        mbw.dequant_int4_awq_g128(q4, torch.zeros(N, 2, dtype=torch.float16), torch.zeros(N, 2, dtype=torch.uint8))
    s128 = torch.zeros(N, K // 128, dtype=torch.float16)
    z128 = torch.zeros(N, 1, dtype=torch.uint8)
    with pytest.raises(ValueError, match="up_zeros"):
        mbw.gemv_fused_awq_g128(q4, s128, z128, x, up_weights=q4, up_scales=s128, up_zeros=z128[:2].contiguous())
    with pytest.raises(ValueError, match="zeros"):
        mbw.gemv_fused_awq_g128(q4, s128, torch.zeros(N, 3, dtype=torch.uint8), x)
    with pytest.raises(ValueError, match="one device"):
        mbw.gemv_bf16(torch.zeros(N, K, dtype=torch.bfloat16), torch.zeros(K, dtype=torch.bfloat16, device="meta"))
    assert host_marshalling.calls == []
