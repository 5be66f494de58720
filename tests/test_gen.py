"""The seeded generator: published SplitMix64 outputs, Box-Muller moments,
bf16 rounding and the workload recipes."""
import math

import numpy as np
import pytest

import gen


def test_splitmix64_published_seed0_outputs():
    # Reference SplitMix64 (Vigna), state 0: the first three outputs.
    got = [int(v) for v in gen.splitmix64(0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_splitmix64_slices_are_consistent():
    full = gen.splitmix64(12345, 1000)
    part = gen.splitmix64(12345, 100, start=437)
    assert np.array_equal(full[437:537], part)


def test_box_muller_first_pair_by_hand():
    s = 99
    u = gen.uniform53(s, 2)
    r = math.sqrt(-2.0 * math.log1p(-float(u[0])))
    th = 2.0 * math.pi * float(u[1])
    z = gen.normal_f32(s, 2)
    assert z[0] == np.float32(r * math.cos(th))
    assert z[1] == np.float32(r * math.sin(th))


def test_normal_moments():
    z = gen.normal_f32(7, 1 << 20, 0.0, 1.0).astype(np.float64)
    assert abs(z.mean()) < 5e-3
    assert abs(z.std() - 1.0) < 5e-3
    assert abs(np.mean(z ** 4) - 3.0) < 0.05
    w = gen.normal_f32(8, 1 << 18, -4.6, 0.5).astype(np.float64)
    assert abs(w.mean() + 4.6) < 5e-3 and abs(w.std() - 0.5) < 5e-3


def test_chunked_normals_match_single_draw():
    a = gen.normal_f32(3, 10_001)
    old = gen._CHUNK
    try:
        gen._CHUNK = 97
        b = gen.normal_f32(3, 10_001)
    finally:
        gen._CHUNK = old
    assert np.array_equal(a, b)


def test_round_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    x = gen.normal_f32(5, 100_000) * np.float32(37.0)
    # exact ties: 1 + 2^-8 sits halfway between two bf16 neighbours
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130], np.float32)
    x = np.concatenate([x, ties])
    ours = gen.round_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours, ref)


def test_workload_recipes():
    assert [w.name for w in gen.WORKLOADS.values()] == gen.WORKLOAD_ORDER
    w = gen.WORKLOADS["mamba1.4b-bf16"]
    assert (w.B, w.L, w.D, w.N, w.io, w.seed) == (4, 4096, 4096, 16, "bf16", 3)
    inp = gen.workload_inputs("s6-tiny-active-f32")
    assert inp.x.shape == (1, 64, 16) and inp.Bm.shape == (1, 64, 16)
    assert np.array_equal(inp.A[3], -np.arange(1, 17, dtype=np.float32))
    # softplus(dt_bias) = 0.69 for the active block
    b = float(inp.dt_bias[0])
    assert abs(math.log1p(math.exp(b)) - 0.69) < 1e-6
    small = gen.workload_inputs("s6-small-f32")
    assert abs(math.log1p(math.exp(float(small.dt_bias[0]))) - 0.01) < 1e-8
    bf = gen.make_inputs(1, 8, 8, 16, io="bf16", seed=2)
    assert np.array_equal(bf.x, gen.round_bf16(bf.x))
    assert not np.array_equal(bf.dt, gen.round_bf16(bf.dt))  # dt stays fp32


def test_determinism():
    a = gen.make_inputs(2, 9, 5, 4, seed=11, with_h0=True, with_dh_last=True)
    b = gen.make_inputs(2, 9, 5, 4, seed=11, with_h0=True, with_dh_last=True)
    for k in ("x", "dt", "z", "Bm", "Cm", "dy", "h0", "dh_last"):
        assert np.array_equal(getattr(a, k), getattr(b, k))
    c = gen.make_inputs(2, 9, 5, 4, seed=12)
    assert not np.array_equal(a.x, c.x)
