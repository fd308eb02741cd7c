"""Helpers shared by the tests: device upload and the parity tolerance."""
import numpy as np

# Parity bar for bf16 outputs against the fp64 oracle.
MAX_ERR_OVER_RMS = 2e-2
MEAN_REL_ERR = 5e-3


def build_lib():
    from bit_quantized_expert_moe_gb300 import build
    return build.build()


def x_to_dev(x_bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(device).view(torch.bfloat16)


def f32_to_dev(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def i32_to_dev(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def bf16_to_f64(t):
    """torch bf16 tensor (any device) -> float64 numpy, exact."""
    import torch
    u = t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def err_stats(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return {
        "max_err_over_rms": float(err.max() / rms) if rms > 0 else float(err.max()),
        "mean_rel_err": float(err.mean() / np.abs(ref).mean()) if np.abs(ref).mean() > 0 else float(err.mean()),
        "rms_ref": rms,
    }


def assert_close(got, ref, what=""):
    s = err_stats(got, ref)
    assert s["max_err_over_rms"] <= MAX_ERR_OVER_RMS and s["mean_rel_err"] <= MEAN_REL_ERR, (what, s)
    return s
