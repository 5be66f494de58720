"""The Gated DeltaNet-2 chunkwise forward on the tensor cores (docs.rs,
burn-gdn2 0.1.4, src/forward.rs, chunk_wy_forward) against the fp64 oracle
fed exactly the GPU's bf16 operands, through the C ABI's Python binding.

Tolerance: the output is bf16 and every product is formed from bf16
operands with fp32 accumulation (the decay factors, the triangular inverse,
the right-hand side Z = w*v - b*k*exp(G) S, v_new and the state's copy are
rounded to bf16 before they enter a product: 2^-9 relative each), so the
error bound of the bf16 scan outputs applies: max|got - ref| / max|ref| <=
2e-2, output and final state. The measured errors are printed with -s; they
sit between 2e-3 and 9e-3.
"""
import numpy as np
import pytest

import gen
from _util import rel_err
from oracle import gdn2_oracle as G

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module")
def ssm():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import selective_state_space_07_gb300 as m
    m.build()
    return m


def dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device="cuda", dtype=dtype)


def run(ssm, x, with_state=True, ws=None):
    bf, f32 = torch.bfloat16, torch.float32
    out, st = ssm.gdn2_fwd(dev(x.q, bf), dev(x.k, bf), dev(x.v, bf), dev(x.g, f32), dev(x.b, bf), dev(x.w, bf),
                           dev(x.state, f32) if with_state else None, x.scale, workspace=ws)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), st.cpu().numpy()


def oracle_run(x, with_state=True, chunk=64):
    s0 = x.state if with_state else np.zeros_like(x.state)
    return G.chunk_wy_forward(x.q, x.k, x.v, x.g, x.b, x.w, s0, x.scale, chunk=chunk)


@pytest.mark.parametrize("B,H,T,seed,with_state", [
    (1, 2, 200, 11, True),    # three whole chunks and a ragged 8-token tail
    (2, 3, 64, 3, True),      # exactly one chunk
    (1, 1, 1, 5, True),       # a single token
    (1, 2, 63, 7, False),     # one ragged chunk from a zero state
    (2, 1, 130, 9, True),     # two chunks and a 2-token tail
    (3, 5, 97, 13, True),     # 15 (batch, head) pairs
    (2, 100, 70, 17, True),   # 200 (batch, head) pairs: more CTAs than SMs (one CTA per SM)
])
def test_matches_the_oracle(ssm, B, H, T, seed, with_state):
    x = gen.make_gdn2_inputs(B, H, T, 128, 128, seed=seed, with_state=with_state)
    ws = ssm.Workspace(1, 1, 8, "cuda")
    out, st = run(ssm, x, with_state, ws)
    ref_o, ref_s = oracle_run(x, with_state)
    eo, es = rel_err(out, ref_o), rel_err(st, ref_s)
    print(f"gdn2 B={B} H={H} T={T}: out {eo:.2e} state {es:.2e}")
    assert eo < TOL and es < TOL
    assert ssm.poll_status(ws) == 0


def test_key_uniform_gates_match_the_per_token_form(ssm):
    # with one gate per token the chunked method is exact: the GPU's chunks of
    # 64 must agree with the per-token recurrence, an independent evaluation
    x = gen.make_gdn2_inputs(1, 2, 150, 128, 128, seed=21, key_uniform_gates=True)
    out, st = run(ssm, x)
    ref_o, ref_s = G.recurrent(x.q, x.k, x.v, x.g, x.b, x.w, x.state, x.scale)
    assert rel_err(out, ref_o) < TOL and rel_err(st, ref_s) < TOL


def test_split_run_chains_through_the_state(ssm):
    # two calls (128 + 72 tokens) with the state passed on equal one call
    x = gen.make_gdn2_inputs(1, 2, 200, 128, 128, seed=23)
    bf, f32 = torch.bfloat16, torch.float32
    t = {n: dev(getattr(x, n), bf) for n in ("q", "k", "v", "b", "w")}
    t["g"] = dev(x.g, f32)
    s0 = dev(x.state, f32)
    o, s = ssm.gdn2_fwd(t["q"], t["k"], t["v"], t["g"], t["b"], t["w"], s0, x.scale)
    cut = 128
    part = lambda a, lo, hi: a[:, :, lo:hi].contiguous()  # noqa: E731
    oa, sa = ssm.gdn2_fwd(*(part(t[n], 0, cut) for n in ("q", "k", "v", "g", "b", "w")), s0, x.scale)
    ob, sb = ssm.gdn2_fwd(*(part(t[n], cut, 200) for n in ("q", "k", "v", "g", "b", "w")), sa, x.scale)
    torch.cuda.synchronize()
    # chunk boundaries coincide (128 = 2 x 64): the same operations in the same order
    assert torch.equal(torch.cat([oa, ob], dim=2), o)
    assert torch.equal(sb, s)


def test_empty_sequence_passes_the_state_through(ssm):
    x = gen.make_gdn2_inputs(2, 2, 0, 128, 128, seed=1)
    bf, f32 = torch.bfloat16, torch.float32
    s0 = dev(x.state, f32)
    e = torch.empty(2, 2, 0, 128, device="cuda")
    o, s = ssm.gdn2_fwd(e.to(bf), e.to(bf), e.to(bf), e, e.to(bf), e.to(bf), s0, x.scale)
    _, z = ssm.gdn2_fwd(e.to(bf), e.to(bf), e.to(bf), e, e.to(bf), e.to(bf), None, x.scale)
    torch.cuda.synchronize()
    assert o.shape == (2, 2, 0, 128)
    assert torch.equal(s, s0) and not z.any()


def test_bounded_wait_expiry_is_reported_and_the_context_stays_usable(ssm):
    # the test hook leaves chunk 1's q, k, b copies unissued and bounds the
    # waits by 1 ms: every CTA's wait runs out, it waits for the copies it did
    # issue and stops; the status word says so, and the next call is normal
    x = gen.make_gdn2_inputs(1, 2, 200, 128, 128, seed=31)
    ws = ssm.Workspace(1, 1, 8, "cuda")
    out0, st0 = run(ssm, x, True, ws)
    assert ssm.poll_status(ws) == 0
    ssm.gdn2_arm_wait_fault(1, 1_000_000)
    run(ssm, x, True, ws)
    assert ssm.poll_status(ws) == -6
    assert ssm.poll_status(ws) == 0  # polling clears the word
    out1, st1 = run(ssm, x, True, ws)  # the hook was one-shot
    assert ssm.poll_status(ws) == 0
    assert np.array_equal(out1, out0) and np.array_equal(st1, st0)


def test_out_of_range_gates_are_reported_as_non_finite(ssm):
    # a half-chunk log-gate sum below -80 overflows the decay factors: the
    # header's limit; the status word must latch it (no fault, no hang)
    x = gen.make_gdn2_inputs(1, 1, 64, 128, 128, seed=2)
    x.g[:] = -4.0
    ws = ssm.Workspace(1, 1, 8, "cuda")
    run(ssm, x, True, ws)
    assert ssm.poll_status(ws) == -7
    y = gen.make_gdn2_inputs(1, 1, 64, 128, 128, seed=2)
    run(ssm, y, True, ws)
    assert ssm.poll_status(ws) == 0


def test_output_stays_inside_its_buffer(ssm):
    x = gen.make_gdn2_inputs(1, 3, 77, 128, 128, seed=29)
    bf, f32 = torch.bfloat16, torch.float32
    gb = 4096 // 2
    n = 3 * 77 * 128
    buf = torch.full((gb + n + gb,), float("nan"), dtype=bf, device="cuda")
    out = buf[gb:gb + n].view(1, 3, 77, 128)
    sgb = 4096 // 4
    sbuf = torch.full((sgb + 3 * 128 * 128 + sgb,), float("nan"), dtype=f32, device="cuda")
    st = sbuf[sgb:sgb + 3 * 128 * 128].view(1, 3, 128, 128)
    ssm.gdn2_fwd(dev(x.q, bf), dev(x.k, bf), dev(x.v, bf), dev(x.g, f32), dev(x.b, bf), dev(x.w, bf),
                 dev(x.state, f32), x.scale, out=out, state_out=st)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:gb].float()).all() and torch.isnan(buf[gb + n:].float()).all()
    assert torch.isnan(sbuf[:sgb]).all() and torch.isnan(sbuf[sgb + 3 * 128 * 128:]).all()
    assert not torch.isnan(out.float()).any() and not torch.isnan(st).any()


def test_full_size_sampled_heads(ssm):
    # the 1.3B-like workload (8 x 16 heads x 2048 tokens, K = V = 128) in the
    # launch the bench times; the oracle checks two (batch, head) pairs
    B, H, T, K, V, seed = gen.GDN2_WORKLOADS["gdn2-1.3b-like"]
    x = gen.make_gdn2_inputs(B, H, T, K, V, seed=seed)
    ws = ssm.Workspace(1, 1, 8, "cuda")
    out, st = run(ssm, x, True, ws)
    assert ssm.poll_status(ws) == 0
    for b, h in ((0, 0), (B - 1, H - 1)):
        sl = lambda a: a[b:b + 1, h:h + 1]  # noqa: E731
        ro, rs = G.chunk_wy_forward(sl(x.q), sl(x.k), sl(x.v), sl(x.g), sl(x.b), sl(x.w), sl(x.state), x.scale,
                                    chunk=64)
        eo, es = rel_err(sl(out), ro), rel_err(sl(st), rs)
        print(f"gdn2 full size (b={b}, h={h}): out {eo:.2e} state {es:.2e}")
        assert eo < TOL and es < TOL


def test_forward_is_deterministic(ssm):
    # no atomics and a fixed order of every reduction: repeated calls agree bit for bit
    x = gen.make_gdn2_inputs(2, 3, 150, 128, 128, seed=37)
    o1, s1 = run(ssm, x)
    o2, s2 = run(ssm, x)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_without_initial_or_final_state(ssm):
    # state=None is a zero initial state; want_state=False skips the final one
    x = gen.make_gdn2_inputs(1, 2, 90, 128, 128, seed=41, with_state=False)
    bf, f32 = torch.bfloat16, torch.float32
    o, s = ssm.gdn2_fwd(dev(x.q, bf), dev(x.k, bf), dev(x.v, bf), dev(x.g, f32), dev(x.b, bf), dev(x.w, bf),
                        None, x.scale, want_state=False)
    torch.cuda.synchronize()
    assert s is None
    ref_o, _ = oracle_run(x, with_state=False)
    assert rel_err(o.float().cpu().numpy(), ref_o) < TOL


def test_binding_rejects_bad_tensors(ssm):
    x = gen.make_gdn2_inputs(1, 1, 16, 128, 128, seed=43)
    bf, f32 = torch.bfloat16, torch.float32
    t = {n: dev(getattr(x, n), bf) for n in ("q", "k", "v", "b", "w")}
    g = dev(x.g, f32)
    args = lambda **kw: [kw.get(n, t.get(n, g)) for n in ("q", "k", "v", "g", "b", "w")]  # noqa: E731
    with pytest.raises(TypeError):
        ssm.gdn2_fwd(*args(g=g.to(bf)))                      # g must be fp32
    with pytest.raises(TypeError):
        ssm.gdn2_fwd(*args(q=t["q"].float()))                # q must be bf16
    with pytest.raises(ValueError):
        ssm.gdn2_fwd(*args(k=t["k"][:, :, :8]))              # shape
    with pytest.raises(ValueError):
        ssm.gdn2_fwd(*args(v=t["v"].transpose(2, 3).contiguous().transpose(2, 3)))  # not contiguous
    small = [a[..., :64].contiguous() for a in args()]
    with pytest.raises(ssm.SsmError):
        ssm.gdn2_fwd(*small)                                 # K = V = 64: unsupported by the kernel


# ---------------------------------------------------------------- the per-token form (one token per call)
# fp32 throughout: the output carries its own bf16 rounding (1e-2), the state 1e-4.
TOL_STEP_O, TOL_STEP_S = 1e-2, 1e-4


def step_run(ssm, x, state=None):
    bf, f32 = torch.bfloat16, torch.float32
    st = dev(x.state, f32) if state is None else state
    t = {n: dev(getattr(x, n), bf) for n in ("q", "k", "v", "b", "w")}
    g = dev(x.g, f32)
    col = lambda a, i: a[:, :, i].contiguous()  # noqa: E731
    outs = [ssm.gdn2_step(col(t["q"], i), col(t["k"], i), col(t["v"], i), col(g, i), col(t["b"], i), col(t["w"], i),
                          st, x.scale) for i in range(x.T)]
    torch.cuda.synchronize()
    return torch.stack(outs, dim=2).float().cpu().numpy(), st.cpu().numpy()


def test_step_matches_the_per_token_oracle(ssm):
    x = gen.make_gdn2_inputs(2, 3, 24, 128, 128, seed=61)
    o, s = step_run(ssm, x)
    ro, rs = G.recurrent(x.q, x.k, x.v, x.g, x.b, x.w, x.state, x.scale)
    eo, es = rel_err(o, ro), rel_err(s, rs)
    print(f"gdn2 step: out {eo:.2e} state {es:.2e}")
    assert eo < TOL_STEP_O and es < TOL_STEP_S


def test_chunked_forward_against_the_per_token_form_on_the_gpu(ssm):
    # the page's check of the chunked forward against the fused recurrent one, both evaluated here: with
    # one gate per token the two agree (to the chunked products' bf16 rounding); then decoding one more
    # token from the chunked call's final state continues the same sequence
    x = gen.make_gdn2_inputs(1, 2, 151, 128, 128, seed=63, key_uniform_gates=True)
    T = 150
    bf, f32 = torch.bfloat16, torch.float32
    t = {n: dev(getattr(x, n), bf) for n in ("q", "k", "v", "b", "w")}
    g = dev(x.g, f32)
    cut = lambda a: a[:, :, :T].contiguous()  # noqa: E731
    oc, sc = ssm.gdn2_fwd(*(cut(t[n]) for n in ("q", "k", "v")), cut(g), cut(t["b"]), cut(t["w"]), dev(x.state, f32),
                          x.scale)
    xs = gen.make_gdn2_inputs(1, 2, 151, 128, 128, seed=63, key_uniform_gates=True)
    for n in ("q", "k", "v", "g", "b", "w"):
        setattr(xs, n, getattr(xs, n)[:, :, :T])
    xs.T = T
    os_, ss = step_run(ssm, xs)
    oc = oc.float().cpu().numpy()
    print(f"gdn2 chunked vs per-token (GPU): out {rel_err(oc, os_):.2e} state {rel_err(sc.cpu().numpy(), ss):.2e}")
    assert rel_err(oc, os_) < TOL and rel_err(sc.cpu().numpy(), ss) < TOL
    col = lambda a: a[:, :, T].contiguous()  # noqa: E731
    o1 = ssm.gdn2_step(*(col(t[n]) for n in ("q", "k", "v")), col(g), col(t["b"]), col(t["w"]), sc, x.scale)
    torch.cuda.synchronize()
    ro, rs = G.recurrent(x.q, x.k, x.v, x.g, x.b, x.w, x.state, x.scale)
    assert rel_err(o1.float().cpu().numpy(), ro[:, :, T]) < TOL and rel_err(sc.cpu().numpy(), rs) < TOL
