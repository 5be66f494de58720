"""The library's FMA-pipe 2^x (C ABI ssm_exp2_fma: a Cody-Waite split by the
1.5 * 2^23 shift, 2^f on [-0.5, 0.5] by the degree-6 polynomial through the
Chebyshev nodes that csrc/exp2_poly.py fits, n added to the exponent field)
against 2^x evaluated in float64 on the same float32 inputs: the header's
bound (relative error below 2^-23 for -125.5 <= x <= 127), exact powers of
two at the integers, 0 below -125.5."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import selective_state_space_07_gb300 as m
    m.build()
    return m


def run(ssm, x):
    y = ssm.exp2_fma(torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda())
    torch.cuda.synchronize()
    return y.cpu().numpy()


def test_relative_error_bound(ssm):
    rng = np.random.default_rng(5)
    grid = np.linspace(-125.5, 127.0, 1 << 22).astype(np.float32)
    small = rng.uniform(-1.0, 1.0, 1 << 20).astype(np.float32)  # the decays' usual range
    halves = (np.arange(-125, 127) + 0.5).astype(np.float32)    # f = +-0.5, the interval's ends
    near = np.concatenate([np.nextafter(halves, np.float32(-1e9)), np.nextafter(halves, np.float32(1e9))])
    x = np.concatenate([grid, small, halves, near])
    x = x[(x >= -125.5) & (x <= 127.0)]
    y = run(ssm, x).astype(np.float64)
    rel = np.abs(y / np.exp2(x.astype(np.float64)) - 1.0)
    print(f"exp2_fma: max relative error {rel.max():.3e} over {x.size} points")
    assert rel.max() < 2.0 ** -23


def test_integers_are_exact_powers_of_two(ssm):
    n = np.arange(-125, 128).astype(np.float32)
    assert np.array_equal(run(ssm, n), np.exp2(n.astype(np.float64)).astype(np.float32))


def test_arguments_below_the_normal_range_flush_to_zero(ssm):
    x = np.array([-125.6, -126.0, -126.5, -127.0, -130.0, -1e30, -np.inf], np.float32)
    assert not run(ssm, x).any()
