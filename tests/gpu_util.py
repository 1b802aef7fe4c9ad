"""Helpers shared by the GPU tests: moving generator outputs to the device and
comparing attention outputs with the oracle."""
import numpy as np
import torch

from paged_kv_cache_store_gb300.workloads import bf16_bits_to_f32

# Attention tolerance against the float64 oracle (bf16 outputs).
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def host_bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def host_f64(t):
    return bf16_bits_to_f32(host_bits(t)).astype(np.float64)


def assert_close(got_f64, want_f64, what=""):
    assert got_f64.shape == want_f64.shape, (got_f64.shape, want_f64.shape)
    assert np.all(np.isfinite(got_f64)), f"{what}: non-finite output"
    err = np.abs(got_f64 - want_f64)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max-abs {mx:.3g} mean-abs {mean:.3g}"
    return mx, mean
