"""Shared pieces of the GPU parity tests: the bars and the comparison helpers.

Bars: forward max|out - out_oracle| <= 1e-2
and max|lse - lse_oracle| <= 2e-3; backward max|dX - dX_oracle| <=
2e-2 * max(max|dX_oracle|, 1e-3) per tensor, X in {Q, K, V}.
"""
import numpy as np
import torch

OUT_TOL, LSE_TOL, GRAD_REL, GRAD_FLOOR = 1e-2, 2e-3, 2e-2, 1e-3


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def run_gpu(fa, q, k, v, do, causal, scale, backward=True):
    dev = torch.device("cuda", 0)
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    out, lse = fa.attention_forward(qd, kd, vd, causal, scale)
    res = {"out": out, "lse": lse}
    if backward:
        dod = do.to(dev)
        res["dq"], res["dk"], res["dv"] = fa.attention_backward(qd, kd, vd, out, dod, lse,
                                                                causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == 0
    return {name: f64(t) for name, t in res.items()}


def check_fwd(got, out_ref, lse_ref):
    e_out = np.abs(got["out"] - out_ref).max()
    e_lse = np.abs(got["lse"] - lse_ref).max()
    assert np.isfinite(got["out"]).all() and np.isfinite(got["lse"]).all()
    assert e_out <= OUT_TOL, f"out max-abs {e_out:.3e}"
    assert e_lse <= LSE_TOL, f"lse max-abs {e_lse:.3e}"


def check_grad(name, got, ref):
    assert np.isfinite(got).all(), name
    bound = GRAD_REL * max(np.abs(ref).max(), GRAD_FLOOR)
    err = np.abs(got - ref).max()
    assert err <= bound, f"{name} max-abs {err:.3e} > {bound:.3e}"
