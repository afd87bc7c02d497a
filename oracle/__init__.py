"""CPU oracle for the weight-only quantized fpA.intB GEMM and the grouped MoE FFN.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg use it; the library never imports it.  It shares no
code with the CUDA path.  The arithmetic lives in ``wo_oracle.c`` (plain C,
fp64 contraction, fp32 dequantisation); this module only compiles it with
gcc, loads it with ctypes and marshals numpy arrays.

Functions and the page passages they follow:

* ``unpack_codes`` / ``pack_nibbles`` -- vLLM-Omni ``cpu_int4.py`` module
  docstring (byte j = w[2j] | w[2j+1] << 4) and ``pack_nibbles`` /
  ``unpack_nibbles``.
* ``dequant`` -- ``cpu_int4.py`` docstring (w = (q - 8) * scale + zero, scale
  and zero per group of K) and acext User Guide 1.3.1 / 1.3.3 (per-channel
  int8 scale; group-wise int4 scale and zero).
* ``gemm`` -- acext User Guide 1.2.1 (fpA_intB runner ``gemm`` with scales,
  zero points, biases and group_size).
* ``dequant_gidx`` / ``gemm_gidx`` -- the same with a GPTQ act-order group
  index (``desc_act`` / ``has_g_idx`` in "[Misc][Kernel]: Add GPTQAllSpark
  Quantization", the case its kernel leaves out): input channel c takes the
  scale and zero of group ``g_idx[c]``; nothing is permuted.
* ``embed`` -- vLLM-Omni ``cpu_int4.py`` ``CPUInt4EmbeddingMethod.embedding``
  (rows of the token ids, dequantised in fp32, cast to the activation dtype).
* ``moe_route`` / ``moe_ffn`` -- acext User Guide 1.2.3 (MoE runner: gating
  output, top-k, fc1, activation, fc2, routing-weighted combine).
* ``to_half_bits`` / ``to_bf16_bits`` / ``decode`` -- IEEE binary16 and
  bfloat16 definitions (round to nearest, ties to even).

Every function is pinned by the CPU pin tests (hand-derived packing bytes,
brute force, closed forms, library special cases, the quantiser invariant);
none is marked "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wo_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F16 = 0
BF16 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no SIMD intrinsics, no FP contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-std=c11", "-D_GNU_SOURCE", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32 = ctypes.c_int
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_double_to_half.argtypes = [ctypes.c_double]
        lib.oracle_double_to_half.restype = ctypes.c_uint16
        lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_double_to_bf16.restype = ctypes.c_uint16
        lib.oracle_round.argtypes = [P, ctypes.c_size_t, i32, P]
        lib.oracle_round.restype = None
        lib.oracle_decode.argtypes = [P, ctypes.c_size_t, i32, P]
        lib.oracle_decode.restype = None
        lib.oracle_unpack_codes.argtypes = [P, i32, i32, i32, P]
        lib.oracle_unpack_codes.restype = i32
        lib.oracle_pack_nibbles.argtypes = [P, i32, i32, P]
        lib.oracle_pack_nibbles.restype = i32
        lib.oracle_dequant.argtypes = [P, P, P, i32, i32, i32, i32, i32, P]
        lib.oracle_dequant.restype = i32
        lib.oracle_gemm.argtypes = [P, i32, P, P, P, P, i32, i32, i32, i32, i32, i32, P]
        lib.oracle_gemm.restype = i32
        lib.oracle_dequant_gidx.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P]
        lib.oracle_dequant_gidx.restype = i32
        lib.oracle_gemm_gidx.argtypes = [P, i32, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                         P]
        lib.oracle_gemm_gidx.restype = i32
        lib.oracle_moe_route.argtypes = [P, i32, i32, i32, i32, P, P]
        lib.oracle_moe_route.restype = i32
        lib.oracle_moe_ffn.argtypes = [P, i32, P, P, P, P, P, i32, i32, i32, i32, i32,
                                       i32, P, i32, i32, P]
        lib.oracle_moe_ffn.restype = i32
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a, name):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"{name} must hold 16-bit float bit patterns as uint16")
    return a


def _u8(a, name):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError(f"{name} must be uint8")
    return a


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments")


def default_threads() -> int:
    return os.cpu_count() or 1


# -- number formats --------------------------------------------------------

def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    """fp16 (dtype 0) or bf16 (dtype 1) bit patterns -> float64."""
    b = _u16(bits, "bits")
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_decode(_ptr(b), b.size, dtype, _ptr(out))
    return out


def round_to(x: np.ndarray, dtype: int) -> np.ndarray:
    """float64 -> fp16 / bf16 bit patterns, round to nearest even."""
    xd = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(xd.shape, dtype=np.uint16)
    _load().oracle_round(_ptr(xd), xd.size, dtype, _ptr(out))
    return out


def to_half_bits(x: float) -> int:
    return int(_load().oracle_double_to_half(float(x)))


def to_bf16_bits(x: float) -> int:
    return int(_load().oracle_double_to_bf16(float(x)))


def half_value(bits: int) -> float:
    return float(_load().oracle_half_to_double(int(bits)))


def bf16_value(bits: int) -> float:
    return float(_load().oracle_bf16_to_double(int(bits)))


# -- codes -----------------------------------------------------------------

def unpack_codes(B: np.ndarray, n: int, k: int, bits: int) -> np.ndarray:
    """Row-major stored codes -> int32 [n, k]."""
    Bc = _u8(B, "B")
    q = np.empty((n, k), dtype=np.int32)
    _check(_load().oracle_unpack_codes(_ptr(Bc), n, k, bits, _ptr(q)), "unpack_codes")
    return q


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """int codes [n, k] in 0..15 -> uint8 [n, k/2], low nibble = even k."""
    qc = np.ascontiguousarray(q, dtype=np.int32)
    n, k = qc.shape
    B = np.empty((n, k // 2), dtype=np.uint8)
    _check(_load().oracle_pack_nibbles(_ptr(qc), n, k, _ptr(B)), "pack_nibbles")
    return B


def dequant(B, scales, zeros, n, k, group_size, bits, sz_dtype) -> np.ndarray:
    """fp32 [n, k] dequantised weights."""
    Bc = _u8(B, "B")
    s = _u16(scales, "scales")
    z = None if zeros is None else _u16(zeros, "zeros")
    w = np.empty((n, k), dtype=np.float32)
    _check(_load().oracle_dequant(_ptr(Bc), _ptr(s), _ptr(z), n, k, group_size, bits,
                                  sz_dtype, _ptr(w)), "dequant")
    return w


def gemm(A, act_dtype, B, scales, zeros, bias, m, n, k, group_size, bits,
         nthreads: int | None = None) -> np.ndarray:
    """fp64 C [m, n] = A . dequant(B)^T + bias (A, scales, zeros, bias as bits)."""
    Ac = _u16(A, "A")
    Bc = _u8(B, "B")
    s = _u16(scales, "scales")
    z = None if zeros is None else _u16(zeros, "zeros")
    b = None if bias is None else _u16(bias, "bias")
    C = np.empty((m, n), dtype=np.float64)
    nt = default_threads() if nthreads is None else nthreads
    _check(_load().oracle_gemm(_ptr(Ac), act_dtype, _ptr(Bc), _ptr(s), _ptr(z), _ptr(b),
                               m, n, k, group_size, bits, nt, _ptr(C)), "gemm")
    return C


def _gidx(g_idx, k) -> np.ndarray:
    g = np.ascontiguousarray(g_idx, dtype=np.int32).reshape(-1)
    if g.size != k:
        raise ValueError("g_idx must have k entries")
    return g


def dequant_gidx(B, scales, zeros, g_idx, n, k, group_size, bits, sz_dtype) -> np.ndarray:
    """fp32 [n, k] dequantised weights, channel c scaled by group g_idx[c]."""
    Bc = _u8(B, "B")
    s = _u16(scales, "scales")
    z = None if zeros is None else _u16(zeros, "zeros")
    g = _gidx(g_idx, k)
    w = np.empty((n, k), dtype=np.float32)
    _check(_load().oracle_dequant_gidx(_ptr(Bc), _ptr(s), _ptr(z), _ptr(g), n, k, group_size,
                                       bits, sz_dtype, _ptr(w)), "dequant_gidx")
    return w


def gemm_gidx(A, act_dtype, B, scales, zeros, g_idx, bias, m, n, k, group_size, bits,
              nthreads: int | None = None) -> np.ndarray:
    """fp64 C [m, n] of an act-order checkpoint: input channel c takes the
    scale and zero of group g_idx[c]; A, B and C in the original order."""
    Ac = _u16(A, "A")
    Bc = _u8(B, "B")
    s = _u16(scales, "scales")
    z = None if zeros is None else _u16(zeros, "zeros")
    g = _gidx(g_idx, k)
    b = None if bias is None else _u16(bias, "bias")
    C = np.empty((m, n), dtype=np.float64)
    nt = default_threads() if nthreads is None else nthreads
    _check(_load().oracle_gemm_gidx(_ptr(Ac), act_dtype, _ptr(Bc), _ptr(s), _ptr(z), _ptr(g),
                                    _ptr(b), m, n, k, group_size, bits, nt, _ptr(C)),
           "gemm_gidx")
    return C


def embed(ids, B, scales, zeros, vocab, hidden, group_size, bits, act_dtype) -> np.ndarray:
    """Embedding rows: act_dtype bit patterns [T, hidden], row t = the fp32
    dequantised weight row ids[t] rounded once (a zero row for an id outside
    [0, vocab))."""
    idx = np.asarray(ids, dtype=np.int64).reshape(-1)
    ok = (idx >= 0) & (idx < vocab)
    sel = idx[ok]
    G = 1 if group_size in (-1, hidden) else hidden // group_size
    # the selected rows' codes, scales and zeros, dequantised as a table of their own
    Bs = np.asarray(B).reshape(vocab, -1)[sel]
    ss = np.asarray(scales).reshape(vocab, G)[sel]
    zs = None if zeros is None else np.asarray(zeros).reshape(vocab, G)[sel]
    rows = np.zeros((idx.size, hidden), dtype=np.float64)
    if sel.size:
        rows[ok] = dequant(Bs, ss, zs, sel.size, hidden, group_size, bits, act_dtype)
    return round_to(rows, act_dtype)


# -- MoE -------------------------------------------------------------------

def moe_route(logits: np.ndarray, topk: int, renormalize: bool = False):
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    ids = np.empty((T, topk), dtype=np.int32)
    w = np.empty((T, topk), dtype=np.float64)
    _check(_load().oracle_moe_route(_ptr(lg), T, E, topk, int(bool(renormalize)),
                                    _ptr(ids), _ptr(w)), "moe_route")
    return ids, w


def moe_ffn(A, act_dtype, logits, fc1, fc1_scales, fc2, fc2_scales, T, H, I, E, topk,
            renormalize=False, tokens=None, nthreads: int | None = None) -> np.ndarray:
    """fp64 [len(tokens) or T, H] MoE FFN output for the listed tokens."""
    Ac = _u16(A, "A")
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    f1 = _u8(fc1, "fc1")
    f2 = _u8(fc2, "fc2")
    s1 = _u16(fc1_scales, "fc1_scales")
    s2 = _u16(fc2_scales, "fc2_scales")
    tk = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    S = T if tk is None else tk.size
    out = np.empty((S, H), dtype=np.float64)
    nt = default_threads() if nthreads is None else nthreads
    _check(_load().oracle_moe_ffn(_ptr(Ac), act_dtype, _ptr(lg), _ptr(f1), _ptr(s1),
                                  _ptr(f2), _ptr(s2), T, H, I, E, topk,
                                  int(bool(renormalize)), _ptr(tk),
                                  0 if tk is None else tk.size, nt, _ptr(out)), "moe_ffn")
    return out
