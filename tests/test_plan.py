"""CPU tests of the kernel choice and launch plan (wo_gemm_plan, the static
counterpart of acext 1.2.1's getChosenConfig).  Pure host code: with no GPU
visible the library plans for 152 SMs, GB300's count.  The GPU parity tests
pick their small shapes to cover every tile configuration; these tests keep
that true."""
import json
import os
import subprocess
import sys

import pytest

import weight_only_quantized_fpa_gb300 as wo
from weight_only_quantized_fpa_gb300 import build as wo_build

SMS = 152
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def lib():
    wo_build.build()
    return wo.load_library()


@pytest.mark.parametrize("m,n,k,bits,group,tile,splits", [
    (250, 12736, 512, 4, 64, (256, 128), 1),
    (300, 19520, 512, 8, -1, (128, 256), 1),
    (300, 15296, 512, 8, -1, (256, 256), 1),
    (260, 19584, 512, 4, 64, (128, 256), 1),
    (300, 15296, 512, 4, 64, (256, 256), 1),
    (200, 320, 6144, 8, -1, (128, 256), 2),
    (130, 448, 12288, 4, 64, (128, 256), 4),
    (200, 384, 3584, 8, -1, (128, 128), 2),
    (130, 320, 4096, 4, 64, (128, 128), 2),
    (4096, 4096, 4096, 8, -1, (256, 256), 1),
    (512, 13312, 2048, 4, 64, (256, 256), 1),
])
def test_tensor_core_tile_configurations(m, n, k, bits, group, tile, splits):
    p = wo.gemm_plan(m, n, k, bits, group, wo.WO_F16 if bits == 8 else wo.WO_BF16)
    assert p["kernel"] == "tensor_core"
    assert (p["tile_m"], p["tile_n"]) == tile
    assert p["k_splits"] == splits
    units = -(-m // tile[0]) * -(-n // tile[1]) * splits
    assert p["ctas"] == min(units, SMS)
    if splits > 1:  # a split plan gives every CTA exactly one unit
        assert units <= SMS
    assert p["workspace_bytes"] == wo.wo_workspace_size(m, n, k, group, bits)


@pytest.mark.parametrize("bits,group", [(8, -1), (4, 64), (4, 128), (4, -1)])
def test_kernel_choice_by_m(bits, group):
    # 8-bit weights take the swap-AB tensor-core kernel at 17..64 rows
    n, k = 512, 2048
    mid = "tensor_core_swap_ab" if bits == 8 else "stream"
    for m, kern in [(1, "stream"), (16, "stream"), (17, mid),
                    (64, mid), (65, "tensor_core"), (256, "tensor_core")]:
        assert wo.gemm_plan(m, n, k, bits, group)["kernel"] == kern, (m, bits, group)


@pytest.mark.parametrize("n,k,group,persistent", [
    (131072, 2048, 64, True),   # the cluster kernel would need 512 CTAs: more than one wave
    (131072, 2048, -1, True),
    (81920, 2048, 64, True),    # 320 cluster CTAs: just over one wave
    (65536, 2048, 64, False),   # 256 cluster CTAs: one wave
    (1024, 13312, 64, False),   # long k, few channels: 64 cluster CTAs still win
    (2048, 13312, 128, False),
    (320, 16384, 64, False),
    (13312, 2048, 64, False),   # 208 CTAs in one wave
    (2048, 2048, 64, False),    # 2 MB of weights: the cluster kernel's shorter critical path
    (3072, 2048, -1, False)])
def test_4bit_decode_kernel_choice(n, k, group, persistent):
    # 4-bit decode sizes take the persistent kernel where the cluster-split
    # one would need more than one resident wave; 8-bit decode always stays
    # on the latter, and so does m = 17
    for m in (1, 16):
        want = "stream_persistent" if persistent else "stream"
        assert wo.gemm_plan(m, n, k, 4, group)["kernel"] == want, (m, n, k)
        assert wo.gemm_plan(m, n, k, 8, -1)["kernel"] == "stream"
    assert wo.gemm_plan(17, n, k, 4, group)["kernel"] == "stream"


@pytest.mark.parametrize("m,n,k,bits,group", [(24, 4608, 3584, 4, 64), (32, 3584, 18944, 4, 64),
                                              (24, 37888, 3584, 4, -1), (20, 2048, 13312, 4, 64),
                                              (64, 131072, 2048, 4, 64), (48, 3584 + 64, 3584, 8, -1)])
def test_stream_plans_fill_one_resident_wave(m, n, k, bits, group):
    p = wo.gemm_plan(m, n, k, bits, group, wo.WO_F16)
    assert p["kernel"] == "stream" and p["tile_m"] == m
    assert p["tile_n"] in (128, 256) and n % 16 == 0
    assert 1 <= p["k_splits"] <= 8                    # portable cluster size
    assert p["ctas"] == -(-n // p["tile_n"]) * p["k_splits"]
    if p["k_splits"] > 1:                             # splits only up to two CTAs per SM
        assert p["ctas"] <= 2 * SMS
    assert p["stages"] >= 1 and p["workspace_bytes"] == 256


PERSISTENT_SHAPES = [(1, 1024, 13312, 4, 64), (4, 1024, 18944, 4, 64), (16, 131072, 2048, 4, 128),
                     (1, 131072, 2048, 4, 64), (9, 256, 16384, 4, 128), (3, 320, 16384, 4, -1),
                     (2, 64, 65536, 4, 64)]


@pytest.fixture(scope="module")
def persistent_plans(lib):
    # the persistent kernel's plans, also for shapes the automatic choice
    # gives the cluster kernel: WO_DECODE_KERNEL (read once per process)
    # forces it, in a child process
    code = ("import json, sys\n"
            "import weight_only_quantized_fpa_gb300 as wo\n"
            "wo.load_library()\n"
            "print(json.dumps([wo.gemm_plan(m, n, k, b, g, wo.WO_BF16) for m, n, k, b, g in json.loads(sys.argv[1])]))\n")
    r = subprocess.run([sys.executable, "-c", code, json.dumps(PERSISTENT_SHAPES)], cwd=ROOT,
                       env=dict(os.environ, WO_DECODE_KERNEL="persistent"), capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return dict(zip(PERSISTENT_SHAPES, json.loads(r.stdout.strip().splitlines()[-1])))


@pytest.mark.parametrize("m,n,k,bits,group", PERSISTENT_SHAPES)
def test_persistent_plans_split_the_weights_evenly(persistent_plans, m, n, k, bits, group):
    # decode sizes: strips of 256 channels by stages of 128 codes, the
    # strip-major units divided evenly over two CTAs per SM (fewer when there
    # are fewer units); pieces of a strip that several CTAs share sum through
    # the workspace after the header and counter area
    p = persistent_plans[(m, n, k, bits, group)]
    assert p["kernel"] == "stream_persistent" and p["tile_m"] == m and p["tile_n"] == 256
    units = -(-n // 256) * -(-k // 128)
    assert p["ctas"] == min(units, 2 * SMS)
    q = units // p["ctas"]
    nst = -(-k // 128)
    assert 1 <= p["k_splits"] <= nst
    assert p["k_splits"] >= min(nst, -(-nst // max(q, 1)))  # room for every piece
    assert p["stages"] >= 3
    mt = 1 if m <= 8 else 2
    partial = -(-n // 256) * p["k_splits"] * 256 * (8 * mt) * 4
    assert p["workspace_bytes"] == 256 + 65536 + -(-partial // 256) * 256


def test_grouped_4bit_decode_with_unaligned_row_of_groups_uses_the_cluster_kernel():
    # scale boxes of 8 groups need k / group to be a multiple of 8
    p = wo.gemm_plan(1, 256, 320, 4, 64)
    assert p["kernel"] == "stream"


@pytest.mark.parametrize("m,n,k", [(1, 4608, 3584), (4, 3584, 18944), (16, 37888, 3584)])
def test_8bit_decode_uses_the_cluster_kernel(m, n, k):
    assert wo.gemm_plan(m, n, k, 8, -1, wo.WO_F16)["kernel"] == "stream"


@pytest.mark.parametrize("m,n,k", [(24, 4608, 3584), (32, 3584, 3584), (48, 37888, 3584),
                                   (64, 3584, 18944), (17, 384, 2048), (40, 128 * SMS, 1024),
                                   (40, 128 * SMS + 128, 1024)])
def test_swap_ab_plans(m, n, k):
    # 8-bit weights at 17..64 rows: blocks of 128 output channels, k split so
    # that the (block, split) items fill the SMs one item each, each split at
    # least 4 k blocks unless there is one, at most 8; the splits' fp32 sums
    # in the workspace after the header and counter area.  With more blocks
    # than SMs the m >= 65 tensor-core kernel takes the shape.
    p = wo.gemm_plan(m, n, k, 8, -1, wo.WO_F16)
    nb, nkb = n // 128, k // 64
    if nb > SMS:
        assert p["kernel"] == "tensor_core"
        return
    assert p["kernel"] == "tensor_core_swap_ab" and p["tile_m"] == m and p["tile_n"] == 128
    sp = p["k_splits"]
    assert 1 <= sp <= 8
    assert sp == 1 or nkb // sp >= 4 or -(-nkb // sp) >= 4
    assert p["ctas"] == nb * sp and nb * sp <= SMS
    want = max(min(SMS // nb, max(nkb // 4, 1), 8), 1)
    kps = -(-nkb // want)
    assert sp == -(-nkb // kps)
    partial = nb * sp * 128 * 64 * 4 if sp > 1 else 0
    assert p["workspace_bytes"] == 256 + 65536 + -(-partial // 256) * 256


def test_plan_argument_rules():
    assert wo.gemm_plan(0, 256, 512, 8)["ctas"] == 0
    with pytest.raises(wo.WoError):
        wo.gemm_plan(4, 100, 512, 8)
    with pytest.raises(wo.WoError):
        wo.gemm_plan(4, 256, 512, 8, 64)        # 8-bit is per channel
    assert wo.load_library().wo_gemm_plan(4, 256, 512, -1, 8, 0, None) == 1
