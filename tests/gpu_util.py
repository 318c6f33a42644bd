"""Helpers shared by the GPU parity tests: moving the shared seeded inputs to the
device, and the error measures with the tolerances the tests apply.

Tolerances (the bar every GPU parity test uses):
  * fp32 layers: normwise relative error max|g - r| / max|r| <= 1e-5;
  * bf16 layers (fp32 accumulation, compared with fp64 on the same
    bf16-rounded inputs): max |g - r| <= 2e-2 and ||g - r||_F / ||r||_F <= 5e-3.
Reported beside them (not a bound): the elementwise relative error
max_i |g_i - r_i| / max(|r_i|, 1e-3 rms(r)) -- elementwise relative error is
ill-posed where an output is near zero, so the denominator has a floor of a
thousandth of the outputs' root mean square.
"""
import numpy as np

F32_NORMWISE = 1e-5
BF16_MAX_ABS = 2e-2
BF16_REL_FRO = 5e-3


def to_device(a, dtype_name):
    import torch
    from transformer_head_scaled_02_gb300 import workloads as wl
    if a is None:
        return None
    if dtype_name == "bf16":
        return torch.from_numpy(wl.bf16_bits(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def to_host(t):
    return t.float().cpu().numpy().astype(np.float64)


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.abs(got - ref)
    if not d.size:
        return {"max_abs": 0.0, "rel_fro": 0.0, "normwise": 0.0, "elem_rel_floored": 0.0}
    floor = max(1e-3 * float(np.sqrt(np.mean(ref * ref))), 1e-300)
    return {
        "max_abs": float(d.max()),
        "rel_fro": float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)),
        "normwise": float(d.max() / max(np.abs(ref).max(), 1e-300)),
        "elem_rel_floored": float((d / np.maximum(np.abs(ref), floor)).max()),
    }


def assert_close(got, ref, dtype_name, what=""):
    e = errors(got, ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    if dtype_name == "f32":
        assert e["normwise"] <= F32_NORMWISE, f"{what}: {e}"
    else:
        assert e["max_abs"] <= BF16_MAX_ABS and e["rel_fro"] <= BF16_REL_FRO, f"{what}: {e}"
    return e


def torch_dtype(dtype_name):
    import torch
    return torch.bfloat16 if dtype_name == "bf16" else torch.float32
