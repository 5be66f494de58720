"""Shared helpers for the tests: moving generated inputs to the GPU, running
the library through its Python binding, and error measures."""
import numpy as np

# Tolerances, per output tensor, as max|got - ref| / max|ref| against the
# fp64 oracle fed exactly the GPU's inputs (bf16-rounded where the I/O dtype
# is bf16): fp32 forward 1e-4, fp32 gradients 1e-3, bf16 everything 2e-2.
TOL = {("f32", "fwd"): 1e-4, ("f32", "bwd"): 1e-3, ("bf16", "fwd"): 2e-2, ("bf16", "bwd"): 2e-2}


def rel_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    scale = float(np.max(np.abs(ref)))
    diff = float(np.max(np.abs(got - ref)))
    return diff / scale if scale > 0 else diff


def to_dev(inp, device="cuda"):
    import torch
    io = torch.bfloat16 if inp.io == "bf16" else torch.float32

    def t(a, dtype):
        if a is None:
            return None
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device=device, dtype=dtype)

    return {
        "x": t(inp.x, io), "z": t(inp.z, io), "Bm": t(inp.Bm, io), "Cm": t(inp.Cm, io), "dy": t(inp.dy, io),
        "dt": t(inp.dt, torch.float32), "A": t(inp.A, torch.float32), "Dskip": t(inp.Dskip, torch.float32),
        "dt_bias": t(inp.dt_bias, torch.float32), "h0": t(inp.h0, torch.float32),
        "dh_last": t(inp.dh_last, torch.float32),
    }


def to_np(t):
    import torch
    if t is None:
        return None
    return t.detach().to(torch.float32).cpu().numpy()


def run_fwd(ssm, dv, inp, **kw):
    return ssm.scan_fwd(dv["x"], dv["dt"], dv["A"], dv["Bm"], dv["Cm"], dv["z"], dv["Dskip"], dv["dt_bias"],
                        dv["h0"], bool(inp.delta_softplus), return_last_state=True, **kw)


def run_bwd(ssm, dv, inp, ckpt, **kw):
    return ssm.scan_bwd(dv["x"], dv["dt"], dv["A"], dv["Bm"], dv["Cm"], dv["dy"], ckpt, dv["z"], dv["Dskip"],
                        dv["dt_bias"], dv["h0"], dv["dh_last"], bool(inp.delta_softplus), return_dh0=True, **kw)


GRAD_KEYS = [("dx", "dx"), ("dz", "dz"), ("d_dt", "ddt"), ("dA", "dA"), ("dD", "dD"),
             ("d_dt_bias", "ddt_bias"), ("dB", "dB"), ("dC", "dC"), ("dh0", "dh0")]
