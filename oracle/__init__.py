"""CPU oracle for the 2-bit MoE layer: ctypes wrappers around ``oracle.c``.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs may use it; the library
and its Python binding never import it.

Everything here marshals numpy arrays; the arithmetic lives in ``oracle.c``.
``oracle.c`` is built twice: single-threaded, and with OpenMP (``parallel=True``
in the calls below), which runs independent blocks and tokens on all host
threads and gives bitwise identical results.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_moe_w2.so")
_LIB_OMP_PATH = os.path.join(_HERE, "liboracle_moe_w2_omp.so")
_lock = threading.Lock()
_libs = {}

BAD_EXPERT_ID = 1
BAD_SCALE = 2
BAD_NVFP4 = 4

_CFLAGS = ["-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False, parallel: bool | None = None) -> str:
    """Compile the oracle with gcc (plain C, no architecture flags): the
    single-threaded library, and the OpenMP one (``parallel`` None builds both
    and returns the single-threaded path)."""
    todo = [(False, _LIB_PATH), (True, _LIB_OMP_PATH)] if parallel is None else \
        [(parallel, _LIB_OMP_PATH if parallel else _LIB_PATH)]
    for omp, path in todo:
        if force or not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
            tmp = path + f".tmp{os.getpid()}"
            subprocess.run(["gcc", *_CFLAGS, *(["-fopenmp"] if omp else []), "-o", tmp, _SRC, "-lm"], check=True)
            os.replace(tmp, path)
    return todo[-1][1] if parallel is not None else _LIB_PATH


def threads(parallel: bool = True) -> int:
    """Host threads the oracle's loops use (1 for the single-threaded build)."""
    return int(lib(parallel).oracle_threads())


def lib(parallel: bool = False):
    with _lock:
        if parallel not in _libs:
            L = ctypes.CDLL(build(parallel=parallel))
            vp, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
            L.oracle_version.restype = ctypes.c_int
            L.oracle_threads.restype = ctypes.c_int
            L.oracle_e2m1_value.argtypes = [ctypes.c_uint]
            L.oracle_e2m1_value.restype = ctypes.c_double
            L.oracle_e4m3_value.argtypes = [ctypes.c_uint]
            L.oracle_e4m3_value.restype = ctypes.c_double
            L.oracle_code_value.argtypes = [ctypes.c_uint]
            L.oracle_code_value.restype = ctypes.c_double
            L.oracle_bf16_from_double.argtypes = [ctypes.c_double]
            L.oracle_bf16_from_double.restype = ctypes.c_uint16
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = ctypes.c_double
            L.oracle_requant.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp]
            L.oracle_requant.restype = u32
            L.oracle_requant_blocks.argtypes = [vp, vp, vp, i64, i64, vp, i64, vp, vp]
            L.oracle_requant_blocks.restype = u32
            L.oracle_requant_ex.argtypes = [vp, vp, vp, i64, i64, i64, u32, vp, vp]
            L.oracle_requant_ex.restype = u32
            L.oracle_requant_mxfp4.argtypes = [vp, vp, i64, i64, i64, u32, vp, vp]
            L.oracle_requant_mxfp4.restype = u32
            L.oracle_requant_fp8.argtypes = [vp, vp, i64, i64, i64, vp, vp]
            L.oracle_requant_fp8.restype = u32
            L.oracle_permute.argtypes = [vp, i64, i32, i32, vp, vp, vp]
            L.oracle_permute.restype = u32
            L.oracle_forward_tokens.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                vp, i64, vp, vp]
            L.oracle_forward_tokens.restype = u32
            L.oracle_forward_tokens_w4.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                   vp, i64, vp, vp]
            L.oracle_forward_tokens_w4.restype = u32
            L.oracle_forward_tokens_cached.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32,
                                                       vp, i64, vp, vp, vp]
            L.oracle_forward_tokens_cached.restype = u32
            _libs[parallel] = L
    return _libs[parallel]


def _p(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.c_void_p)


def e2m1_value(nib: int) -> float:
    return lib().oracle_e2m1_value(nib)


def e4m3_value(b: int) -> float:
    return lib().oracle_e4m3_value(b)


def code_value(c: int) -> float:
    return lib().oracle_code_value(c)


def bf16_from_double(v: float) -> int:
    return lib().oracle_bf16_from_double(v)


def bf16_to_double(h: int) -> float:
    return lib().oracle_bf16_to_double(h)


BALANCE_ZERO_SIGNS = 1   # option bit of the FP4 loaders: exact zeros take alternating signs


def requant(e2m1: np.ndarray, e4m3: np.ndarray, scale_2: np.ndarray, parallel: bool = False, options: int = 0):
    """e2m1 uint8 [n][rows][K/2], e4m3 uint8 [n][rows][K/16], scale_2 float32 [n]."""
    n, rows, half_k = e2m1.shape
    K = half_k * 2
    e2m1 = np.ascontiguousarray(e2m1)
    e4m3 = np.ascontiguousarray(e4m3)
    s2 = np.ascontiguousarray(scale_2, dtype=np.float32)
    codes = np.empty((n, rows, K // 4), np.uint8)
    scales = np.empty((n, rows, K // 32), np.uint8)
    st = lib(parallel).oracle_requant_ex(_p(e2m1), _p(e4m3), _p(s2), n, rows, K, options, _p(codes), _p(scales))
    return codes, scales, int(st)


def requant_mxfp4(e2m1: np.ndarray, scales: np.ndarray, parallel: bool = False, options: int = 0):
    """MXFP4: e2m1 uint8 [n][rows][K/2], UE8M0 scale bytes uint8 [n][rows][K/32]."""
    n, rows, half_k = e2m1.shape
    K = half_k * 2
    e2m1 = np.ascontiguousarray(e2m1)
    sc = np.ascontiguousarray(scales, dtype=np.uint8)
    assert sc.shape == (n, rows, K // 32)
    codes = np.empty((n, rows, K // 4), np.uint8)
    ue8m0 = np.empty((n, rows, K // 32), np.uint8)
    st = lib(parallel).oracle_requant_mxfp4(_p(e2m1), _p(sc), n, rows, K, options, _p(codes), _p(ue8m0))
    return codes, ue8m0, int(st)


def requant_blocks(e2m1: np.ndarray, e4m3: np.ndarray, scale_2: np.ndarray, block_ids, parallel: bool = False):
    """Selected blocks (flat index over n*rows*K/32) -> codes [nb][8], scales [nb]."""
    n, rows, half_k = e2m1.shape
    K = half_k * 2
    ids = np.ascontiguousarray(block_ids, dtype=np.int64)
    codes = np.empty((len(ids), 8), np.uint8)
    scales = np.empty(len(ids), np.uint8)
    s2 = np.ascontiguousarray(scale_2, dtype=np.float32)
    st = lib(parallel).oracle_requant_blocks(_p(np.ascontiguousarray(e2m1)), _p(np.ascontiguousarray(e4m3)),
                                     _p(s2), rows, K, _p(ids), len(ids), _p(codes), _p(scales))
    return codes, scales, int(st)


def requant_fp8(w8: np.ndarray, scales: np.ndarray, parallel: bool = False):
    """w8 uint8 (e4m3fn bytes) [n][rows][K], scales float32 [n][ceil(rows/128)][ceil(K/128)]."""
    n, rows, K = w8.shape
    w8 = np.ascontiguousarray(w8)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    assert sc.shape == (n, (rows + 127) // 128, (K + 127) // 128)
    codes = np.empty((n, rows, K // 4), np.uint8)
    ue8m0 = np.empty((n, rows, K // 32), np.uint8)
    st = lib(parallel).oracle_requant_fp8(_p(w8), _p(sc), n, rows, K, _p(codes), _p(ue8m0))
    return codes, ue8m0, int(st)


def permute(ids: np.ndarray, E: int):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    P = T * k
    sorted_pairs = np.empty(P, np.int32)
    inv = np.empty(P, np.int32)
    offsets = np.empty(E + 1, np.int32)
    st = lib().oracle_permute(_p(ids), T, k, E, _p(sorted_pairs), _p(inv), _p(offsets))
    return sorted_pairs, inv, offsets, int(st)


def forward_tokens(x: np.ndarray, ids: np.ndarray, weights: np.ndarray, planes: dict,
                   tokens=None, want_h: bool = False, parallel: bool = False):
    """y (bf16 bits) for the listed tokens; x uint16 [T][H], ids int32 [T][k], weights f32 [T][k]."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    weights = np.ascontiguousarray(weights, dtype=np.float32)
    T, H = x.shape
    k = ids.shape[1]
    E, two_i, _ = planes["w13_codes"].shape
    I = two_i // 2
    tok = np.arange(T, dtype=np.int64) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
    y = np.empty((len(tok), H), np.uint16)
    h = np.empty((len(tok), k, I), np.uint16) if want_h else None
    st = lib(parallel).oracle_forward_tokens(
        _p(x), _p(ids), _p(weights),
        _p(planes["w13_codes"]), _p(planes["w13_scales"]), _p(planes["w2_codes"]), _p(planes["w2_scales"]),
        E, H, I, k, _p(tok), len(tok), _p(y), _p(h) if want_h else None)
    return (y, h, int(st)) if want_h else (y, int(st))


def forward_tokens_cached(x: np.ndarray, ids: np.ndarray, weights: np.ndarray, planes: dict, slot_of: np.ndarray,
                          tokens=None, want_h: bool = False, parallel: bool = False):
    """The forward behind an expert cache: planes hold the resident slots, slot_of int32 [n_route]
    maps routed ids to slots (negative: not resident).  -> (y, [h,] status, misses)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    weights = np.ascontiguousarray(weights, dtype=np.float32)
    slot_of = np.ascontiguousarray(slot_of, dtype=np.int32)
    T, H = x.shape
    k = ids.shape[1]
    E, two_i, _ = planes["w13_codes"].shape
    I = two_i // 2
    tok = np.arange(T, dtype=np.int64) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
    y = np.empty((len(tok), H), np.uint16)
    h = np.empty((len(tok), k, I), np.uint16) if want_h else None
    misses = np.zeros(1, np.int64)
    st = lib(parallel).oracle_forward_tokens_cached(
        _p(x), _p(ids), _p(weights), _p(slot_of), len(slot_of),
        _p(planes["w13_codes"]), _p(planes["w13_scales"]), _p(planes["w2_codes"]), _p(planes["w2_scales"]),
        E, H, I, k, _p(tok), len(tok), _p(y), _p(h) if want_h else None, _p(misses))
    return (y, h, int(st), int(misses[0])) if want_h else (y, int(st), int(misses[0]))


def forward_tokens_w4(x: np.ndarray, ids: np.ndarray, weights: np.ndarray, planes: dict,
                      tokens=None, want_h: bool = False, parallel: bool = False):
    """The FP4 layer: planes of NVFP4 experts (w13_e2m1 [E][2I][H/2], w13_e4m3 [E][2I][H/16],
    w13_scale_2 f32 [E][2] (gate, up), w2_e2m1 [E][H][I/2], w2_e4m3 [E][H][I/16], w2_scale_2 f32 [E])."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    weights = np.ascontiguousarray(weights, dtype=np.float32)
    T, H = x.shape
    k = ids.shape[1]
    E, two_i, _ = planes["w13_e2m1"].shape
    I = two_i // 2
    pl = {n: np.ascontiguousarray(planes[n]) for n in ("w13_e2m1", "w13_e4m3", "w2_e2m1", "w2_e4m3")}
    s13 = np.ascontiguousarray(planes["w13_scale_2"], dtype=np.float32).reshape(E, 2)
    s2 = np.ascontiguousarray(planes["w2_scale_2"], dtype=np.float32).reshape(E)
    tok = np.arange(T, dtype=np.int64) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
    y = np.empty((len(tok), H), np.uint16)
    h = np.empty((len(tok), k, I), np.uint16) if want_h else None
    st = lib(parallel).oracle_forward_tokens_w4(
        _p(x), _p(ids), _p(weights), _p(pl["w13_e2m1"]), _p(pl["w13_e4m3"]), _p(s13),
        _p(pl["w2_e2m1"]), _p(pl["w2_e4m3"]), _p(s2), E, H, I, k, _p(tok), len(tok), _p(y),
        _p(h) if want_h else None)
    return (y, h, int(st)) if want_h else (y, int(st))


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Reinterpret bf16 bit patterns as float values (exact)."""
    return (np.asarray(a, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
