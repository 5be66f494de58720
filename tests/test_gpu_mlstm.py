"""The mLSTM stabilized chunkwise forward on the tensor cores
(Evil-Inference-Code, README_FIX_RUST.md, "mLSTM Equivalence Fixes (Rust vs
Python)") against the fp64 oracle fed exactly the GPU's bf16 operands,
through the C ABI's Python binding.

Tolerances: h is bf16 and the products are formed from bf16 operands with
fp32 accumulation (alpha*scale*q, gamma*k, P and the state's copy are
rounded to bf16 before they enter a product: 2^-9 relative each), so the
bf16 bound of the other kernels applies: max|got - ref| / max|ref| <= 2e-2
for h and C. n is updated in fp32 from the exact bf16 keys (1e-3), m is a
sum of fp32 log-gates (1e-3 absolute). The measured errors are printed
with -s.
"""
import numpy as np
import pytest

import gen
from _util import rel_err
from oracle import mlstm_oracle as M

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL, TOL_N, TOL_M = 2e-2, 1e-3, 1e-3


@pytest.fixture(scope="module")
def ssm():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import selective_state_space_07_gb300 as m
    m.build()
    return m


def dev(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device="cuda", dtype=dtype)


def run(ssm, x, with_state=True, norm=False, ws=None):
    bf = torch.bfloat16
    st = (dev(x.C0), dev(x.n0), dev(x.m0)) if with_state else None
    h, so = ssm.mlstm_fwd(dev(x.q, bf), dev(x.k, bf), dev(x.v, bf), dev(x.igate), dev(x.fgate), st, x.scale,
                          norm_weight=dev(x.norm_weight) if norm else None, workspace=ws)
    torch.cuda.synchronize()
    return h.float().cpu().numpy(), tuple(t.cpu().numpy() for t in so)


def oracle_run(x, with_state=True, norm=False):
    st = (x.C0, x.n0, x.m0) if with_state else (None, None, None)
    h, C, n, m = M.chunkwise(x.q, x.k, x.v, x.igate, x.fgate, *st, scale=x.scale, chunk=64)
    if norm:
        h = M.head_layer_norm(h, x.norm_weight, 1e-5)
    return h, (C, n, m)


def check(got, ref, tag):
    (h, (C, n, m)), (rh, (rC, rn, rm)) = got, ref
    eh, eC, en, em = rel_err(h, rh), rel_err(C, rC), rel_err(n, rn), float(np.max(np.abs(m - rm)))
    print(f"mlstm {tag}: h {eh:.2e} C {eC:.2e} n {en:.2e} m {em:.2e}")
    assert eh < TOL and eC < TOL and en < TOL_N and em < TOL_M


@pytest.mark.parametrize("B,H,T,seed,with_state,norm", [
    (1, 2, 200, 11, True, False),    # three whole chunks and an 8-token tail
    (2, 3, 64, 3, True, True),       # exactly one chunk, with the head-wise norm
    (1, 1, 1, 5, True, False),       # a single token
    (1, 2, 63, 7, False, False),     # one ragged chunk from a zero state (m = 0)
    (2, 1, 130, 9, True, True),      # two chunks and a 2-token tail
    (3, 5, 97, 13, True, False),     # 15 (batch, head) pairs
    (2, 100, 70, 17, True, False),   # 200 (batch, head) pairs: more CTAs than SMs
])
def test_matches_the_oracle(ssm, B, H, T, seed, with_state, norm):
    x = gen.make_mlstm_inputs(B, H, T, 128, 128, seed=seed, with_state=with_state)
    ws = ssm.Workspace(1, 1, 8, "cuda")
    got = run(ssm, x, with_state, norm, ws)
    check(got, oracle_run(x, with_state, norm), f"B={B} H={H} T={T} norm={norm}")
    assert ssm.poll_status(ws) == 0


def test_matches_the_recurrent_step(ssm):
    # the per-token stabilized step is an independent evaluation of the same cell
    x = gen.make_mlstm_inputs(1, 2, 150, 128, 128, seed=21)
    h, (C, n, m) = run(ssm, x)
    rh, rC, rn, rm = M.recurrent(x.q, x.k, x.v, x.igate, x.fgate, x.C0, x.n0, x.m0, scale=x.scale)
    assert rel_err(h, rh) < TOL and rel_err(C, rC) < TOL and rel_err(n, rn) < TOL_N
    assert float(np.max(np.abs(m - rm))) < TOL_M


def test_large_input_gates_stay_finite(ssm):
    # exp(60) is beyond fp32's range: only the stabilized evaluation is finite
    x = gen.make_mlstm_inputs(1, 2, 150, 128, 128, seed=22, igate_mean=60.0)
    ws = ssm.Workspace(1, 1, 8, "cuda")
    got = run(ssm, x, True, False, ws)
    assert ssm.poll_status(ws) == 0
    assert np.isfinite(got[0]).all() and all(np.isfinite(a).all() for a in got[1])
    check(got, oracle_run(x), "igate ~ N(60, 1)")


def test_split_run_chains_through_the_state(ssm):
    # two calls (128 + 72 tokens) with the state passed on equal one call
    x = gen.make_mlstm_inputs(1, 2, 200, 128, 128, seed=23)
    bf = torch.bfloat16
    t = {"q": dev(x.q, bf), "k": dev(x.k, bf), "v": dev(x.v, bf)}
    ig, fg = dev(x.igate), dev(x.fgate)
    s0 = (dev(x.C0), dev(x.n0), dev(x.m0))
    h, s = ssm.mlstm_fwd(t["q"], t["k"], t["v"], ig, fg, s0, x.scale)
    cut = 128
    p4 = lambda a, lo, hi: a[:, :, lo:hi].contiguous()  # noqa: E731
    ha, sa = ssm.mlstm_fwd(*(p4(t[n], 0, cut) for n in ("q", "k", "v")), p4(ig, 0, cut), p4(fg, 0, cut), s0, x.scale)
    hb, sb = ssm.mlstm_fwd(*(p4(t[n], cut, 200) for n in ("q", "k", "v")), p4(ig, cut, 200), p4(fg, cut, 200), sa,
                           x.scale)
    torch.cuda.synchronize()
    # chunk boundaries coincide (128 = 2 x 64): the same operations in the same order
    assert torch.equal(torch.cat([ha, hb], dim=2), h)
    assert all(torch.equal(a, b) for a, b in zip(sb, s))


def test_empty_sequence_passes_the_state_through(ssm):
    x = gen.make_mlstm_inputs(2, 2, 0, 128, 128, seed=1)
    bf = torch.bfloat16
    s0 = (dev(x.C0), dev(x.n0), dev(x.m0))
    e = torch.empty(2, 2, 0, 128, device="cuda", dtype=bf)
    g = torch.empty(2, 2, 0, device="cuda")
    h, s = ssm.mlstm_fwd(e, e, e, g, g, s0, x.scale)
    _, z = ssm.mlstm_fwd(e, e, e, g, g, None, x.scale)
    torch.cuda.synchronize()
    assert h.shape == (2, 2, 0, 128)
    assert all(torch.equal(a, b) for a, b in zip(s, s0)) and not any(a.any() for a in z)


def test_bounded_wait_expiry_is_reported_and_the_context_stays_usable(ssm):
    # the test hook leaves chunk 1's q copy unissued and bounds the waits by
    # 1 ms: every CTA's wait runs out, it waits for the copies it did issue
    # and stops; the status word says so, and the next call is normal
    x = gen.make_mlstm_inputs(1, 2, 200, 128, 128, seed=31)
    ws = ssm.Workspace(1, 1, 8, "cuda")
    h0, s0 = run(ssm, x, True, False, ws)
    assert ssm.poll_status(ws) == 0
    ssm.mlstm_arm_wait_fault(1, 1_000_000)
    run(ssm, x, True, False, ws)
    assert ssm.poll_status(ws) == -6
    assert ssm.poll_status(ws) == 0  # polling clears the word
    h1, s1 = run(ssm, x, True, False, ws)  # the hook was one-shot
    assert ssm.poll_status(ws) == 0
    assert np.array_equal(h1, h0) and all(np.array_equal(a, b) for a, b in zip(s1, s0))


def test_non_finite_gates_are_reported(ssm):
    x = gen.make_mlstm_inputs(1, 1, 64, 128, 128, seed=2)
    x.igate[0, 0, 10] = np.nan
    ws = ssm.Workspace(1, 1, 8, "cuda")
    run(ssm, x, True, False, ws)
    assert ssm.poll_status(ws) == -7
    y = gen.make_mlstm_inputs(1, 1, 64, 128, 128, seed=2)
    run(ssm, y, True, False, ws)
    assert ssm.poll_status(ws) == 0


def test_outputs_stay_inside_their_buffers(ssm):
    x = gen.make_mlstm_inputs(1, 3, 77, 128, 128, seed=29)
    bf, f32 = torch.bfloat16, torch.float32
    gb = 4096 // 2
    n = 3 * 77 * 128
    buf = torch.full((gb + n + gb,), float("nan"), dtype=bf, device="cuda")
    h = buf[gb:gb + n].view(1, 3, 77, 128)
    sg = 4096 // 4
    sizes = (3 * 128 * 128, 3 * 128, 3)
    sbufs = [torch.full((sg + z + sg,), float("nan"), dtype=f32, device="cuda") for z in sizes]
    so = tuple(b[sg:sg + z].view(shp) for b, z, shp in zip(sbufs, sizes, ((1, 3, 128, 128), (1, 3, 128), (1, 3))))
    ssm.mlstm_fwd(dev(x.q, bf), dev(x.k, bf), dev(x.v, bf), dev(x.igate), dev(x.fgate),
                  (dev(x.C0), dev(x.n0), dev(x.m0)), x.scale, norm_weight=dev(x.norm_weight), h=h, state_out=so)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:gb].float()).all() and torch.isnan(buf[gb + n:].float()).all()
    for b, z in zip(sbufs, sizes):
        assert torch.isnan(b[:sg]).all() and torch.isnan(b[sg + z:]).all()
    assert not torch.isnan(h.float()).any() and not any(torch.isnan(t).any() for t in so)


def test_full_size_sampled_heads(ssm):
    # the 8 x 16 heads x 2048 tokens workload (K = V = 128) in the launch the
    # bench times; the oracle checks two (batch, head) pairs
    B, H, T, K, V, seed = gen.MLSTM_WORKLOADS["mlstm-8x16x2048"]
    x = gen.make_mlstm_inputs(B, H, T, K, V, seed=seed)
    ws = ssm.Workspace(1, 1, 8, "cuda")
    h, (C, n, m) = run(ssm, x, True, False, ws)
    assert ssm.poll_status(ws) == 0
    for b, hh in ((0, 0), (B - 1, H - 1)):
        sl = lambda a: a[b:b + 1, hh:hh + 1]  # noqa: E731
        rh, rC, rn, rm = M.chunkwise(sl(x.q), sl(x.k), sl(x.v), sl(x.igate), sl(x.fgate), sl(x.C0), sl(x.n0),
                                     sl(x.m0), scale=x.scale, chunk=64)
        check((sl(h), (sl(C), sl(n), sl(m))), (rh, (rC, rn, rm)), f"full size (b={b}, h={hh})")


def test_forward_is_deterministic(ssm):
    # no atomics and a fixed order of every reduction: repeated calls agree bit for bit
    x = gen.make_mlstm_inputs(2, 3, 150, 128, 128, seed=37)
    h1, s1 = run(ssm, x, True, True)
    h2, s2 = run(ssm, x, True, True)
    assert np.array_equal(h1, h2) and all(np.array_equal(a, b) for a, b in zip(s1, s2))


def test_without_final_state(ssm):
    # want_state=False passes no state buffers (the NULL branch of the C ABI); h is unchanged
    x = gen.make_mlstm_inputs(1, 2, 90, 128, 128, seed=41)
    bf = torch.bfloat16
    st = (dev(x.C0), dev(x.n0), dev(x.m0))
    h1, s1 = ssm.mlstm_fwd(dev(x.q, bf), dev(x.k, bf), dev(x.v, bf), dev(x.igate), dev(x.fgate), st, x.scale)
    h2, s2 = ssm.mlstm_fwd(dev(x.q, bf), dev(x.k, bf), dev(x.v, bf), dev(x.igate), dev(x.fgate), st, x.scale,
                           want_state=False)
    torch.cuda.synchronize()
    assert s2 is None and s1 is not None
    assert torch.equal(h1, h2)


def test_binding_rejects_bad_tensors(ssm):
    x = gen.make_mlstm_inputs(1, 1, 16, 128, 128, seed=43)
    bf = torch.bfloat16
    q, k, v, ig, fg = dev(x.q, bf), dev(x.k, bf), dev(x.v, bf), dev(x.igate), dev(x.fgate)
    with pytest.raises(TypeError):
        ssm.mlstm_fwd(q, k, v, ig.to(bf), fg)                       # gates must be fp32
    with pytest.raises(TypeError):
        ssm.mlstm_fwd(q.float(), k, v, ig, fg)                      # q must be bf16
    with pytest.raises(ValueError):
        ssm.mlstm_fwd(q, k[:, :, :8], v, ig, fg)                    # shape
    with pytest.raises(ValueError):
        ssm.mlstm_fwd(q, k, v, ig, fg, (dev(x.C0),))                # state must be (C, n, m)
    small = [a[..., :64].contiguous() for a in (q, k, v)]
    with pytest.raises(ssm.SsmError):
        ssm.mlstm_fwd(*small, ig, fg)                               # K = V = 64: unsupported by the kernel


# ---------------------------------------------------------------- the recurrent step (one token)
# fp32 throughout (no bf16 operands): h carries only its own bf16 rounding, so 1e-2; the state 1e-4.
TOL_STEP_H, TOL_STEP_S = 1e-2, 1e-4


def step_run(ssm, x, norm=False):
    """Steps through x's tokens one at a time from x's initial state; returns h [B,H,T,V] and the state."""
    bf = torch.bfloat16
    st = (dev(x.C0), dev(x.n0), dev(x.m0))
    q, k, v, ig, fg = dev(x.q, bf), dev(x.k, bf), dev(x.v, bf), dev(x.igate), dev(x.fgate)
    w = dev(x.norm_weight) if norm else None
    hs = [ssm.mlstm_step(q[:, :, t].contiguous(), k[:, :, t].contiguous(), v[:, :, t].contiguous(),
                         ig[:, :, t].contiguous(), fg[:, :, t].contiguous(), st, x.scale, norm_weight=w)
          for t in range(x.T)]
    torch.cuda.synchronize()
    return torch.stack(hs, dim=2).float().cpu().numpy(), tuple(t.cpu().numpy() for t in st)


@pytest.mark.parametrize("norm,igate_mean", [(False, 0.0), (True, 0.0), (False, 60.0)])
def test_step_matches_the_recurrent_oracle(ssm, norm, igate_mean):
    x = gen.make_mlstm_inputs(2, 3, 20, 128, 128, seed=51, igate_mean=igate_mean)
    h, (C, n, m) = step_run(ssm, x, norm)
    rh, rC, rn, rm = M.recurrent(x.q, x.k, x.v, x.igate, x.fgate, x.C0, x.n0, x.m0, scale=x.scale)
    if norm:
        rh = M.head_layer_norm(rh, x.norm_weight, 1e-5)
    eh, eC, en = rel_err(h, rh), rel_err(C, rC), rel_err(n, rn)
    print(f"mlstm step norm={norm} igate~N({igate_mean},1): h {eh:.2e} C {eC:.2e} n {en:.2e}")
    assert eh < TOL_STEP_H and eC < TOL_STEP_S and en < TOL_STEP_S
    assert float(np.max(np.abs(m - rm))) < TOL_STEP_S


def test_step_continues_the_chunkwise_forward(ssm):
    # decoding after a prompt: the chunkwise kernel's final state, then one step, equals the oracle over T + 1
    x = gen.make_mlstm_inputs(2, 2, 131, 128, 128, seed=53)
    bf = torch.bfloat16
    T = 130
    q, k, v, ig, fg = dev(x.q, bf), dev(x.k, bf), dev(x.v, bf), dev(x.igate), dev(x.fgate)
    _, st = ssm.mlstm_fwd(q[:, :, :T].contiguous(), k[:, :, :T].contiguous(), v[:, :, :T].contiguous(),
                          ig[:, :, :T].contiguous(), fg[:, :, :T].contiguous(), (dev(x.C0), dev(x.n0), dev(x.m0)),
                          x.scale)
    h = ssm.mlstm_step(q[:, :, T].contiguous(), k[:, :, T].contiguous(), v[:, :, T].contiguous(),
                       ig[:, :, T].contiguous(), fg[:, :, T].contiguous(), st, x.scale)
    torch.cuda.synchronize()
    rh, rC, rn, rm = M.recurrent(x.q, x.k, x.v, x.igate, x.fgate, x.C0, x.n0, x.m0, scale=x.scale)
    assert rel_err(h.float().cpu().numpy(), rh[:, :, T]) < TOL
    assert rel_err(st[0].cpu().numpy(), rC) < TOL and rel_err(st[1].cpu().numpy(), rn) < TOL_N
    assert float(np.max(np.abs(st[2].cpu().numpy() - rm))) < TOL_M


def test_step_from_a_zero_state_and_non_finite_gates(ssm):
    x = gen.make_mlstm_inputs(1, 2, 3, 128, 128, seed=55, with_state=False)
    h, (C, n, m) = step_run(ssm, x)
    rh, rC, _, _ = M.recurrent(x.q, x.k, x.v, x.igate, x.fgate, scale=x.scale)
    assert rel_err(h, rh) < TOL_STEP_H and rel_err(C, rC) < TOL_STEP_S
    bf = torch.bfloat16
    ws = ssm.Workspace(1, 1, 8, "cuda")
    st = (dev(x.C0), dev(x.n0), dev(x.m0))
    ig = dev(x.igate[:, :, 0]).contiguous()
    ig[0, 1] = float("nan")
    ssm.mlstm_step(dev(x.q[:, :, 0], bf), dev(x.k[:, :, 0], bf), dev(x.v[:, :, 0], bf), ig,
                   dev(x.fgate[:, :, 0]).contiguous(), st, x.scale, workspace=ws)
    assert ssm.poll_status(ws) == -7
