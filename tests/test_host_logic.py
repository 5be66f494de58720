"""Host-side launch logic, without a GPU: the L-group choices the C ABI
makes for the benchmark shapes (each the optimum of a measured sweep on
GB300) and the helpers' edge cases."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def choices(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    cuda_inc = "/usr/local/cuda/include"
    exe = str(tmp_path_factory.mktemp("hostlogic") / "host_groups")
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", cuda_inc, os.path.join(HERE, "host_groups.cpp"), "-o", exe],
                   check=True, capture_output=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split("\n")
    fwd = [int(l.split()[1]) for l in out if l.startswith("fwd")]
    bwd = [int(l.split()[1]) for l in out if l.startswith("bwd")]
    return fwd, bwd


def test_forward_groups(choices):
    fwd, _ = choices
    # 4x4096x4096 (256 CTAs of 64 channels): one group; 8x2048x1536 (192 CTAs): 2;
    # 1x65536x2048 (32 CTAs): fill the 456 resident slots once -> 14; capped by gmax
    assert fwd[:4] == [1, 2, 14, 4]
    assert fwd[4] == 1 and fwd[5] >= 1               # degenerate grids still get a group
    assert fwd[6] == 1 and fwd[7] == 2               # the 1.5-CTAs-per-SM threshold (456 slots / 227 = 2)


def test_backward_groups(choices):
    _, bwd = choices
    # 4x4096x4096 (128 CTAs of 128 channels, 2 per SM): 7 groups = 2.95 waves;
    # 8x2048x1536 (96 CTAs): 3; 1x65536x2048 (16 CTAs): 19
    assert bwd[:3] == [7, 3, 19]
    assert bwd[3] == 1                               # the cap wins
    assert bwd[4] == 1                               # a grid of many waves needs no groups


def test_kernel_source_hash_ignores_comments_and_layout_only():
    # the stored ncu counters are keyed by this hash: documentation edits
    # keep them, any change to the code (literals included) drops them
    import bench
    strip = bench.strip_c_comments
    code = 'int f(int a) { return a + 1; }\nconst char* s = "x // y";'
    assert strip(code) == strip("// lead\n" + code.replace("{ ", "{\n    /* note */ ") + "  // tail\n")
    assert strip(code) != strip(code.replace("a + 1", "a + 2"))
    assert "// y" in strip(code)  # inside a string literal: kept
    assert strip("char c = '\\''; // q") == "char c = '\\'';"
    for call in bench.CALL_SOURCES:
        assert len(bench.kernel_source_hash(call)) == 16
