"""Helpers for the GPU parity tests: moving seeded inputs to the device and
the tolerance checks.

Tolerances: BF16 outputs max |err| <= 2e-2 * RMS(o_oracle); FP32 states and
snapshots max |err| <= 1e-3 * RMS(S_oracle); index handling bit-exact.
"""
import numpy as np
import torch

from linear_attention_serving_gated_gb300 import kda
from oracle import kda_oracle as ko

O_TOL = 2e-2
S_TOL = 1e-3


def dev_bf16(x):
    """int16 BF16 bit array -> device bfloat16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int16)).cuda().view(torch.bfloat16)


def dev_in(x):
    """16-bit token array -> device tensor: int16 BF16 bits as bfloat16,
    float16 as float16."""
    x = np.ascontiguousarray(x)
    t = torch.from_numpy(x).cuda()
    return t.view(torch.bfloat16) if x.dtype == np.int16 else t


def dev(x, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host_f64(t):
    """Device tensor -> float64 numpy (bf16 widened exactly)."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def rms(x):
    return float(np.sqrt(np.mean(np.square(x)))) if x.size else 0.0


def assert_o_close(o_gpu, o_ref, what="o"):
    """max|o - o_ref| <= 2e-2 RMS(o_ref), on top of the BF16 output's own
    round-to-nearest: element i may also differ by 2^-8 |o_ref_i|, an upper
    bound of half a BF16 ulp at o_ref_i (the exact value is not representable
    in the output format, and the largest outputs here are ~12x the RMS)."""
    got = host_f64(o_gpu) if isinstance(o_gpu, torch.Tensor) else o_gpu
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    if not o_ref.size:
        return 0.0
    r = rms(o_ref)
    excess = np.abs(got - o_ref) - 2.0 ** -8 * np.abs(o_ref)
    worst = float(np.max(excess))
    assert worst <= O_TOL * r, (f"{what}: max(|err| - 2^-8|ref|) {worst:.3e} > {O_TOL * r:.3e} "
                                f"(2e-2 x RMS); raw max|err| {float(np.max(np.abs(got - o_ref))):.3e}")
    return max(worst, 0.0) / max(r, 1e-300)


def assert_s_close(s_gpu, s_ref, what="state"):
    got = host_f64(s_gpu) if isinstance(s_gpu, torch.Tensor) else s_gpu
    err = float(np.max(np.abs(got - s_ref))) if s_ref.size else 0.0
    bound = S_TOL * rms(s_ref)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    assert err <= bound, f"{what}: max|err| {err:.3e} > {bound:.3e} (1e-3 x RMS)"
    return err / max(rms(s_ref), 1e-300)


def gates(d, lower_bound=-5.0, beta_is_raw=True, use_qk_l2norm=True, scale=None, H=None, K=128, HV=None,
          given_decay=False):
    """Matching oracle and device gate descriptions from seeded inputs.  HV
    value heads (default: the gate parameters' head count), H q/k heads
    (default HV).  given_decay: no A_log / dt_bias, the gate input is the
    log-decay itself."""
    HV = HV if HV is not None else d["A_log"].shape[0]
    H = H if H is not None else HV
    scale = scale if scale is not None else K ** -0.5
    A_log, dt_bias = (None, None) if given_decay else (d["A_log"], d["dt_bias"])
    og = ko.Gate(H, K, K, HV=HV, A_log=A_log, dt_bias=dt_bias, lower_bound=lower_bound,
                 beta_is_raw=beta_is_raw, use_qk_l2norm=use_qk_l2norm, scale=scale)
    gg = kda.Gate(A_log=None if given_decay else dev(A_log), dt_bias=None if given_decay else dev(dt_bias),
                  lower_bound=lower_bound, beta_is_raw=beta_is_raw, use_qk_l2norm=use_qk_l2norm,
                  scale=scale)
    return og, gg
