"""Helpers for the GPU parity tests: move seeded host inputs to the device and
compare kernel outputs with the fp64 oracle under the stated tolerance
|y - y_ref| <= 2e-3 * sum_k |w_ik x_k| + 1e-5 (fp32 accumulation, bf16 output)."""
import numpy as np

REL_TOL = 2e-3
ABS_TOL = 1e-5


def dev_bf16(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def dev_f16(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.float16).cuda()


def dev_u8(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def host_bits16(t):
    import torch

    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def host_f64(t):
    import torch

    return t.float().cpu().numpy().astype(np.float64)


def assert_parity(y_dev, Y_ref, Y_abs, what=""):
    y = host_f64(y_dev).reshape(Y_ref.shape)
    err = np.abs(y - Y_ref)
    bound = REL_TOL * Y_abs + ABS_TOL
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outputs out of tolerance; first {idx.tolist()}: "
                             f"got {y[tuple(idx[0])]!r} want {Y_ref[tuple(idx[0])]!r} bound {bound[tuple(idx[0])]!r}")
    return float((err / bound).max()) if err.size else 0.0
