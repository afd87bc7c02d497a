"""CPU tests of the C ABI: the library builds, loads, exports every symbol
include/wo.h declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

import weight_only_quantized_fpa_gb300 as wo
from weight_only_quantized_fpa_gb300 import build as wo_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wo.h")


@pytest.fixture(scope="module")
def lib():
    wo_build.build()
    return wo.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"WO_API\s+[\w\s\*]*?\b(wo_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["wo_pack", "wo_unpack", "wo_packed_bytes", "wo_workspace_size", "wo_gemm",
              "wo_moe_workspace_size", "wo_moe_ffn", "wo_status_string", "wo_check_workspace",
              "wo_selftest_wait_timeout", "wo_embed", "wo_act_order_perm",
              "wo_pack_act_order", "wo_act_order_workspace_size", "wo_gemm_act_order"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_is_built_for_sm_103a():
    # the object files carry the arch in the fatbin; check the build flags instead
    assert "arch=compute_103a,code=sm_103a" in " ".join(wo_build.ARCH)


def test_status_strings(lib):
    assert wo.wo_status_string(0) == "WO_OK"
    assert wo.wo_status_string(5) == "WO_ERR_TIMEOUT"
    assert wo.wo_status_string(99) == "WO_ERR_UNKNOWN"


@pytest.mark.parametrize("n,k,bits,expect", [
    (256, 512, 4, 256 * 256), (4608, 3584, 8, 4608 * 3584), (64, 64, 8, 4096),
    (100, 512, 8, 0), (256, 500, 4, 0), (256, 512, 3, 0), (0, 512, 8, 0), (256, 0, 8, 0)])
def test_packed_bytes(lib, n, k, bits, expect):
    assert wo.wo_packed_bytes(n, k, bits) == expect


def _gemm_status(lib, m=4, n=256, k=512, group=64, bits=4, act=1, A=4096, B=8192, s=64,
                 z=None, bias=None, C=16384, ws=None, ws_bytes=0):
    return lib.wo_gemm(A, B, s, z, bias, C, m, n, k, group, bits, act, ws, ws_bytes, None)


def test_gemm_rejects_bad_shapes_before_launch(lib):
    assert _gemm_status(lib, n=100) == 1
    assert _gemm_status(lib, k=500) == 1
    assert _gemm_status(lib, k=0) == 1
    assert _gemm_status(lib, m=-1) == 1
    assert _gemm_status(lib, bits=3) == 1
    assert _gemm_status(lib, group=100) == 1   # does not divide k
    assert _gemm_status(lib, act=2) == 1


def test_gemm_unsupported_combinations(lib):
    assert _gemm_status(lib, bits=8, group=64) == 2       # 8-bit is per channel
    assert _gemm_status(lib, bits=8, group=-1, z=64) == 2  # 8-bit has no zeros
    assert _gemm_status(lib, bits=4, group=32) == 2       # groups are multiples of 64


def test_gemm_empty_is_noop(lib):
    assert _gemm_status(lib, m=0, A=None, B=None, s=None, C=None) == 0


def test_gemm_rejects_null_and_misaligned(lib):
    assert _gemm_status(lib, A=None) == 1
    assert _gemm_status(lib, C=None) == 1
    assert _gemm_status(lib, A=4096 + 8) == 1
    assert _gemm_status(lib, s=65) == 1


def test_gemm_rejects_small_workspace(lib):
    m, n, k = 256, 256, 1024   # the tensor-core kernel needs a workspace
    need = wo.wo_workspace_size(m, n, k, -1, 8)
    assert need > 0
    assert _gemm_status(lib, m=m, n=n, k=k, group=-1, bits=8, act=0, ws=None) == 3
    assert _gemm_status(lib, m=m, n=n, k=k, group=-1, bits=8, act=0, ws=1 << 20,
                        ws_bytes=need - 1) == 3


def test_workspace_size_invalid_is_zero(lib):
    assert wo.wo_workspace_size(1, 100, 512, -1, 8) == 0
    assert wo.wo_workspace_size(0, 256, 512, -1, 8) == 0


def test_pack_rejects_bad_arguments(lib):
    # every call below fails validation, so nothing is launched on these
    # placeholder addresses
    assert lib.wo_pack(None, 1 << 20, 256, 512, 4, None) == 1
    assert lib.wo_pack(4096, 1 << 20, 100, 512, 4, None) == 1
    assert lib.wo_pack(4096 + 4, 1 << 20, 256, 512, 4, None) == 1
    # overlapping source and destination
    assert lib.wo_pack(1 << 20, (1 << 20) + 4096, 256, 512, 8, None) == 1


def test_library_load_fails_loudly_when_missing(monkeypatch, tmp_path):
    monkeypatch.setattr(wo_build, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(wo, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        wo.load_library()


def test_noalloc_entry_validates_before_any_cuda_call(lib):
    # invalid shape, unsupported combination, and a problem larger than the
    # built-in scratch: all rejected before the scratch is touched
    f = lib.wo_gemm_tc_noalloc
    assert f(4096, 8192, 64, None, None, 16384, 512, 100, 2048, 64, 4, 1, None) == 1
    assert f(4096, 8192, 64, 64, None, 16384, 512, 256, 2048, -1, 8, 0, None) == 2
    assert f(4096, 8192, 64, None, None, 16384, 4096, 256, 4096, 64, 4, 1, None) == 3
    assert f(4096, 8192, 64, None, None, 16384, 0, 256, 2048, 64, 4, 1, None) == 0


def test_selftest_rejects_bad_arguments_without_launching(lib):
    # argument errors come back before any launch (nothing runs on the CPU machine)
    import ctypes
    buf = ctypes.create_string_buffer(1024)
    addr = (ctypes.addressof(buf) + 255) // 256 * 256
    f = lib.wo_selftest_wait_timeout
    f.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint, ctypes.c_void_p]
    f.restype = ctypes.c_int
    assert f(None, 256, 1000, None) == 1          # no workspace
    assert f(addr, 128, 1000, None) == 1          # too small for the header
    assert f(addr + 8, 256, 1000, None) == 1      # not 256-byte aligned
    assert f(addr, 256, 0, None) == 1             # limit out of range
    assert f(addr, 256, 2000000, None) == 1


@pytest.mark.parametrize("kw,expect", [
    (dict(), 0),                                   # T == 0: nothing to do
    (dict(T=4, bits=3), 1),                        # bad bits
    (dict(T=4, vocab=100), 1),                     # vocab % 64
    (dict(T=4, hidden=96), 1),                     # hidden % 64
    (dict(T=4, bits=8, group=64), 2),              # 8-bit tables are per channel
    (dict(T=4, bits=8, group=-1, zeros=64), 2),    # 8-bit tables have no zeros
    (dict(T=4, ids=4098), 1),                      # ids not 4-byte aligned
    (dict(T=4, B=4104), 1),                        # packed table not 16-byte aligned
    (dict(T=4, out=16392), 1),                     # output not 16-byte aligned
    (dict(T=4, act=7), 1),                         # bad activation dtype
    (dict(T=-1), 1),
])
def test_embed_rejects_bad_arguments_before_launch(lib, kw, expect):
    a = dict(ids=4096, T=0, B=8192, s=64, zeros=None, out=16384, vocab=256, hidden=512, group=64,
             bits=4, act=1)
    a.update(kw)
    st = lib.wo_embed(a["ids"], a["T"], a["B"], a["s"], a["zeros"], a["out"], a["vocab"],
                      a["hidden"], a["group"], a["bits"], a["act"], None)
    assert st == expect


# ---------------------------------------------------------- act-order -------
# wo_act_order_perm is host code, so it is tested here in full.

def _perm(g_idx, k, group):
    import numpy as np
    out = np.full(k, -7, dtype=np.int32)
    gi = np.ascontiguousarray(g_idx, dtype=np.int32)   # kept alive across the call
    st = wo.load_library().wo_act_order_perm(gi.ctypes.data, k, group, out.ctypes.data)
    return st, out


@pytest.mark.parametrize("k,group,seed", [(128, 64, 0), (4096, 128, 1), (3584, 64, 2),
                                          (512, 512, 3), (512, -1, 4)])
def test_act_order_perm_is_the_stable_group_sort(lib, k, group, seed):
    import numpy as np
    from weight_only_quantized_fpa_gb300 import inputs
    g = group if group != -1 else k
    gi = inputs.act_order_g_idx(inputs.rng_for(11, seed, inputs.T_GIDX), k, g)
    st, perm = _perm(gi, k, group)
    assert st == 0
    assert np.array_equal(perm, np.argsort(gi, kind="stable"))
    # every run of g positions holds one group, channels ascending
    assert np.array_equal(gi[perm], np.arange(k) // g)
    assert np.array_equal(np.sort(perm), np.arange(k))


def test_act_order_perm_in_order_index_is_identity(lib):
    import numpy as np
    k = 1024
    st, perm = _perm(np.arange(k) // 128, k, 128)
    assert st == 0 and np.array_equal(perm, np.arange(k))


def test_act_order_perm_rejects_bad_indices(lib):
    import numpy as np
    k = 256
    gi = (np.arange(k) // 64).astype(np.int32)
    bad = gi.copy(); bad[3] = 4          # group 4 does not exist (k / 64 = 4 groups)
    assert _perm(bad, k, 64)[0] == 1
    bad = gi.copy(); bad[3] = -1
    assert _perm(bad, k, 64)[0] == 1
    bad = gi.copy(); bad[0] = 1          # group 0 short, group 1 long
    assert _perm(bad, k, 64)[0] == 2
    assert _perm(gi, k, 100)[0] == 1     # group does not divide k
    assert _perm(gi, 0, 64)[0] == 1
    assert lib.wo_act_order_perm(None, k, 64, 4096) == 1


def test_act_order_perm_binding_checks_host_arrays(lib):
    import numpy as np
    with pytest.raises(ValueError):
        wo.wo_act_order_perm(np.zeros(10, np.int32), 64, 64, np.empty(64, np.int32))
    with pytest.raises(ValueError):
        wo.wo_act_order_perm(np.zeros(64, np.int32), 64, 64, np.empty(64, np.int64))


def _ao_status(lib, m=4, n=256, k=512, group=64, bits=4, act=1, A=4096, B=8192, perm=1 << 16,
               s=64, z=None, bias=None, C=16384, ws=None, ws_bytes=0):
    return lib.wo_gemm_act_order(A, B, perm, s, z, bias, C, m, n, k, group, bits, act, ws,
                                 ws_bytes, None)


def test_act_order_gemm_rejects_bad_arguments_before_launch(lib):
    need = wo.wo_act_order_workspace_size(4, 256, 512, 64, 4)
    plain = wo.wo_workspace_size(4, 256, 512, 64, 4)
    assert need >= max(plain, 256 + 65536) + 4 * 512 * 2   # never inside the counter area
    assert _ao_status(lib, n=100) == 1
    assert _ao_status(lib, group=32) == 2
    assert _ao_status(lib, perm=None, ws=1 << 20, ws_bytes=need) == 1
    assert _ao_status(lib, perm=(1 << 16) + 4, ws=1 << 20, ws_bytes=need) == 1   # 16-byte rule
    # the plain GEMM's workspace is not enough: the gathered A lives after it
    assert _ao_status(lib, ws=1 << 20, ws_bytes=plain) == 3
    assert _ao_status(lib, ws=(1 << 20) + 16, ws_bytes=need) == 3
    assert _ao_status(lib, m=0, A=None, B=None, s=None, C=None, perm=None) == 0
    assert wo.wo_act_order_workspace_size(0, 256, 512, 64, 4) == 0
    assert wo.wo_act_order_workspace_size(4, 100, 512, 64, 4) == 0


def test_pack_act_order_rejects_bad_arguments(lib):
    assert lib.wo_pack_act_order(4096, 1 << 20, None, 256, 512, 4, None) == 1
    assert lib.wo_pack_act_order(4096, 1 << 20, (1 << 16) + 2, 256, 512, 4, None) == 1
    assert lib.wo_pack_act_order(4096, 1 << 20, 1 << 16, 100, 512, 4, None) == 1
    assert lib.wo_pack_act_order(1 << 20, (1 << 20) + 4096, 1 << 16, 256, 512, 8, None) == 1


def test_act_order_binding_checks_perm_tensor():
    # the torch-level helpers refuse a permutation the C layer would read
    # from the wrong place or with the wrong width, before any CUDA call
    import numpy as np
    import torch
    k = 256
    good = torch.arange(k, dtype=torch.int32)
    wo._check_perm(good, k, torch.device("cpu"))
    with pytest.raises(TypeError):
        wo._check_perm(np.arange(k, dtype=np.int32), k, "cpu")
    with pytest.raises(ValueError):
        wo._check_perm(good.to(torch.int64), k, "cpu")
    with pytest.raises(ValueError):
        wo._check_perm(good[:128], k, "cpu")
    with pytest.raises(ValueError):
        wo._check_perm(torch.arange(2 * k, dtype=torch.int32)[::2], k, "cpu")
    with pytest.raises(ValueError):   # a perm on another device than the operands
        wo._check_perm(good, k, torch.device("meta"))


@pytest.mark.parametrize("m,n,k,group", [(1, 256, 1024, 64), (16, 4096, 4096, 128),
                                         (64, 192, 512, 64), (65, 256, 512, 128),
                                         (200, 320, 6144, -1), (512, 131072, 2048, 128),
                                         (130, 320, 4096, 128)])
def test_act_order_workspace_keeps_gathered_A_clear_of_shared_area(lib, m, n, k, group):
    # layout: the GEMM's own workspace (at least the header and the split-K
    # counters, 256 + 65536 bytes, shared by every call), then m*k*2 bytes
    # of gathered activations
    def up(x):
        return (x + 255) // 256 * 256
    need = wo.wo_act_order_workspace_size(m, n, k, group, 4)
    plain = wo.wo_workspace_size(m, n, k, group, 4)
    assert need == up(max(plain, 256 + 65536)) + up(m * k * 2)


def _moe_status(lib, T=16, H=4096, I=1408, E=64, topk=2, act=1, A=1 << 20, logits=1 << 21,
                fc1=1 << 22, s1=1 << 23, fc2=1 << 24, s2=1 << 25, out=1 << 26, ws=None,
                ws_bytes=0):
    return lib.wo_moe_ffn(A, logits, fc1, s1, fc2, s2, out, T, H, I, E, topk, 0, act, ws,
                          ws_bytes, None)


def test_moe_rejects_bad_arguments_before_launch(lib):
    # every call fails validation, so the placeholder addresses are never used
    need = wo.wo_moe_workspace_size(16, 4096, 1408, 64, 2)
    assert need > 0
    assert _moe_status(lib, T=-1) == 1
    assert _moe_status(lib, H=4000) == 1          # hidden % 64
    assert _moe_status(lib, I=1400) == 1          # inter % 64
    assert _moe_status(lib, E=0) == 1
    assert _moe_status(lib, topk=3, E=2) == 1     # topk > experts
    assert _moe_status(lib, topk=9, E=64) == 1    # topk > 8
    assert _moe_status(lib, act=2) == 1
    assert _moe_status(lib, A=None, ws=1 << 27, ws_bytes=need) == 1
    assert _moe_status(lib, logits=(1 << 21) + 2, ws=1 << 27, ws_bytes=need) == 1
    assert _moe_status(lib, out=(1 << 26) + 8, ws=1 << 27, ws_bytes=need) == 1
    assert _moe_status(lib) == 3                  # no workspace
    assert _moe_status(lib, ws=1 << 27, ws_bytes=need - 1) == 3
    assert _moe_status(lib, ws=(1 << 27) + 128, ws_bytes=need) == 3
    assert _moe_status(lib, T=0, A=None) == 0     # no tokens: a no-op


def test_moe_workspace_size_invalid_is_zero(lib):
    assert wo.wo_moe_workspace_size(0, 4096, 1408, 64, 2) == 0
    assert wo.wo_moe_workspace_size(16, 4096, 1408, 2, 3) == 0
    assert wo.wo_moe_workspace_size(1024, 4096, 1408, 64, 2) > \
        wo.wo_moe_workspace_size(16, 4096, 1408, 64, 2)


def test_debug_bounds_entry_in_a_normal_build(lib):
    # a library built without the index checks says so, touching no GPU
    assert wo.wo_status_string(6) == "WO_ERR_BOUNDS"
    assert wo.wo_debug_bounds() == (2, 0)  # WO_ERR_UNSUPPORTED
    lib.wo_debug_bounds.argtypes = [ctypes.c_void_p]
    assert lib.wo_debug_bounds(None) == 2  # site may be NULL
    lib.wo_debug_bounds.argtypes = [ctypes.POINTER(ctypes.c_uint)]


def test_index_checked_build_compiles_and_is_selected_by_the_environment(monkeypatch):
    # the -DWO_DEBUG_BOUNDS=1 library builds beside the normal one, exports the
    # same entry points, and WO_DEBUG_BOUNDS=1 selects it at load time
    path = wo_build.build(debug_bounds=True)
    assert path == wo_build.LIB_DEBUG_BOUNDS and os.path.exists(path)
    assert path != wo_build.LIB
    dbg = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(dbg, name), name
    monkeypatch.setenv("WO_DEBUG_BOUNDS", "1")
    assert wo.library_path() == wo_build.LIB_DEBUG_BOUNDS
    monkeypatch.delenv("WO_DEBUG_BOUNDS")
    assert wo.library_path() == wo_build.LIB
