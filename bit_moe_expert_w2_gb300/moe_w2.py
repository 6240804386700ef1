"""Python binding of libmoe_w2 (ctypes).  Argument marshalling only.

Every step of the layer runs in the CUDA library: this module checks tensor
shapes and dtypes, allocates outputs and workspace with torch when the caller
did not, passes raw device pointers and the current CUDA stream, and turns a
non-zero status into an exception.  There is no fallback: if the library is
missing or the device is not sm_103, the call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_lib = None

OK = 0
DEV_BAD_EXPERT_ID = 1
DEV_BAD_SCALE = 2
DEV_BAD_NVFP4 = 4
DEV_PIPELINE_TIMEOUT = 0x80000000   # as a uint32; reads back as a negative int32 from a torch int32 tensor
REQUANT_BALANCE_ZERO_SIGNS = 1       # option bit of requant (moe_w2_requant_ex) and requant_mxfp4
DECODE_MAX_TOKENS = 64
PATH_NONE, PATH_DECODE_MMA, PATH_DECODE_BLOCK_SCALED, PATH_PREFILL, PATH_DECODE_STREAM = 0, 1, 2, 3, 4   # moe_w2_forward_path
NOALLOC_WORKSPACE_BYTES = 8 << 20   # MOE_W2_NOALLOC_WORKSPACE_BYTES


class MoeW2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} (status {status})")
        self.status = status


class Planes(ctypes.Structure):
    _fields_ = [("w13_codes", ctypes.c_void_p), ("w13_scales", ctypes.c_void_p),
                ("w2_codes", ctypes.c_void_p), ("w2_scales", ctypes.c_void_p),
                ("num_experts", ctypes.c_int32), ("hidden", ctypes.c_int32), ("inter", ctypes.c_int32)]


class W4Planes(ctypes.Structure):
    """moe_w4_planes: the FP4 layer's NVFP4 experts."""
    _fields_ = [("w13_e2m1", ctypes.c_void_p), ("w13_e4m3", ctypes.c_void_p), ("w13_scale_2", ctypes.c_void_p),
                ("w2_e2m1", ctypes.c_void_p), ("w2_e4m3", ctypes.c_void_p), ("w2_scale_2", ctypes.c_void_p),
                ("num_experts", ctypes.c_int32), ("hidden", ctypes.c_int32), ("inter", ctypes.c_int32)]


def forward_path(T: int, top_k: int, E: int, H: int, I: int) -> int:
    """moe_w2_forward_path: which kernels moe_w2_forward runs for these sizes (PATH_*)."""
    return int(load().moe_w2_forward_path(T, top_k, E, H, I))


def decode_kernel(T: int, top_k: int, H: int, I: int) -> str:
    """Name of the kernel that runs the layer of a decode step (T <= DECODE_MAX_TOKENS)."""
    path = forward_path(T, top_k, 1, H, I)
    names = {PATH_DECODE_MMA: "decode_mma_kernel", PATH_DECODE_BLOCK_SCALED: "decode_layer_kernel",
             PATH_DECODE_STREAM: "decode_stream_kernel"}
    if path not in names:
        raise ValueError(f"T={T} top_k={top_k} H={H} I={I} is not a decode step")
    return names[path]


def set_decode_stream(enable: bool) -> None:
    """moe_w2_set_decode_stream: run decode steps of at most 16 pairs on the
    stream-K kernel (True, the default) or on the mma.sync kernel (False)."""
    load().moe_w2_set_decode_stream(1 if enable else 0)


class decode_stream:
    """Context manager: the stream-K kernel for the smallest decode steps inside
    the block, the previous choice restored after it."""

    def __init__(self, enable: bool = True):
        self.enable = enable

    def __enter__(self):
        self.prev = forward_path(1, 1, 1, 512, 512) == PATH_DECODE_STREAM
        set_decode_stream(self.enable)
        return self

    def __exit__(self, *exc):
        set_decode_stream(self.prev)
        return False


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libmoe_w2.so (building it first if it is missing and nvcc is present)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build()")
        _build.build()
    L = ctypes.CDLL(path)
    vp, i32, i64, u32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t
    L.moe_w2_version.restype = ctypes.c_int
    L.moe_w2_status_string.argtypes = [ctypes.c_int]
    L.moe_w2_status_string.restype = ctypes.c_char_p
    L.moe_w2_forward_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.moe_w2_forward_workspace_size.restype = sz
    L.moe_w2_forward_path.argtypes = [i32, i32, i32, i32, i32]
    L.moe_w2_forward_path.restype = ctypes.c_int
    L.moe_w2_permute.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp]
    L.moe_w2_permute.restype = ctypes.c_int
    L.moe_w2_forward.argtypes = [vp, vp, vp, ctypes.POINTER(Planes), i32, i32, vp, vp, sz, vp, vp]
    L.moe_w2_forward.restype = ctypes.c_int
    L.moe_w2_forward_noalloc.argtypes = [vp, vp, vp, ctypes.POINTER(Planes), i32, i32, vp, vp, vp]
    L.moe_w2_forward_noalloc.restype = ctypes.c_int
    L.moe_w4_forward_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.moe_w4_forward_workspace_size.restype = sz
    L.moe_w4_forward.argtypes = [vp, vp, vp, ctypes.POINTER(W4Planes), i32, i32, vp, vp, sz, vp, vp]
    L.moe_w4_forward.restype = ctypes.c_int
    L.moe_w4_forward_traced.argtypes = [vp, vp, vp, ctypes.POINTER(W4Planes), i32, i32, vp, vp, sz, vp, vp, vp]
    L.moe_w4_forward_traced.restype = ctypes.c_int
    L.moe_w2_forward_cached_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.moe_w2_forward_cached_workspace_size.restype = sz
    L.moe_w2_forward_cached.argtypes = [vp, vp, vp, ctypes.POINTER(Planes), vp, i32, i32, i32, vp, vp, sz, vp, vp, vp]
    L.moe_w2_forward_cached.restype = ctypes.c_int
    L.moe_w2_requant.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, vp, vp]
    L.moe_w2_requant.restype = ctypes.c_int
    L.moe_w2_requant_ex.argtypes = [vp, vp, vp, i64, i64, i64, u32, vp, vp, vp, vp]
    L.moe_w2_requant_ex.restype = ctypes.c_int
    L.moe_w2_requant_mxfp4.argtypes = [vp, vp, i64, i64, i64, u32, vp, vp, vp, vp]
    L.moe_w2_requant_mxfp4.restype = ctypes.c_int
    L.moe_w2_requant_fp8.argtypes = [vp, vp, i64, i64, i64, vp, vp, vp, vp]
    L.moe_w2_requant_fp8.restype = ctypes.c_int
    L.moe_w2_debug_force_pipeline_timeout.argtypes = [i32]
    L.moe_w2_debug_force_pipeline_timeout.restype = ctypes.c_int
    L.moe_w2_set_decode_stream.argtypes = [i32]
    L.moe_w2_set_decode_stream.restype = ctypes.c_int
    _lib = L
    return L


def status_string(status: int) -> str:
    return load().moe_w2_status_string(int(status)).decode()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_cuda(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def make_planes(planes: dict) -> Planes:
    """Planes struct from the four uint8 CUDA tensors w13_codes [E][2I][H/4], w13_scales [E][2I][H/32],
    w2_codes [E][H][I/4], w2_scales [E][H][I/32]."""
    for k in ("w13_codes", "w13_scales", "w2_codes", "w2_scales"):
        _check_cuda(planes[k], k, torch.uint8)
    E, two_i, h4 = planes["w13_codes"].shape
    return Planes(planes["w13_codes"].data_ptr(), planes["w13_scales"].data_ptr(),
                  planes["w2_codes"].data_ptr(), planes["w2_scales"].data_ptr(), E, h4 * 4, two_i // 2)


def workspace_size(T: int, top_k: int, E: int, H: int, I: int) -> int:
    return int(load().moe_w2_forward_workspace_size(T, top_k, E, H, I))


def forward(x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor, planes, y=None,
            workspace=None, status=None, stream=None) -> torch.Tensor:
    """y = MoE layer(x) through moe_w2_forward.  x bf16 [T][H], ids int32 [T][k], weights f32 [T][k]."""
    L = load()
    _check_cuda(x, "x", torch.bfloat16)
    _check_cuda(topk_ids, "topk_ids", torch.int32)
    _check_cuda(topk_weights, "topk_weights", torch.float32)
    p = planes if isinstance(planes, Planes) else make_planes(planes)
    T, H = x.shape
    k = topk_ids.shape[1]
    if y is None:
        y = torch.empty_like(x)
    need = workspace_size(T, k, p.num_experts, p.hidden, p.inter)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    st = L.moe_w2_forward(_ptr(x), _ptr(topk_ids), _ptr(topk_weights), ctypes.byref(p), T, k, _ptr(y),
                          _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream))
    if st != OK:
        raise MoeW2Error(st, "moe_w2_forward")
    return y


def make_w4_planes(planes: dict) -> W4Planes:
    """W4Planes from the CUDA tensors w13_e2m1 u8 [E][2I][H/2], w13_e4m3 u8 [E][2I][H/16],
    w13_scale_2 f32 [E][2], w2_e2m1 u8 [E][H][I/2], w2_e4m3 u8 [E][H][I/16], w2_scale_2 f32 [E]."""
    for k in ("w13_e2m1", "w13_e4m3", "w2_e2m1", "w2_e4m3"):
        _check_cuda(planes[k], k, torch.uint8)
    for k in ("w13_scale_2", "w2_scale_2"):
        _check_cuda(planes[k], k, torch.float32)
    E, two_i, h2 = planes["w13_e2m1"].shape
    return W4Planes(planes["w13_e2m1"].data_ptr(), planes["w13_e4m3"].data_ptr(), planes["w13_scale_2"].data_ptr(),
                    planes["w2_e2m1"].data_ptr(), planes["w2_e4m3"].data_ptr(), planes["w2_scale_2"].data_ptr(),
                    E, h2 * 2, two_i // 2)


def w4_workspace_size(T: int, top_k: int, E: int, H: int, I: int) -> int:
    return int(load().moe_w4_forward_workspace_size(T, top_k, E, H, I))


def forward_w4(x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor, planes, y=None,
               workspace=None, status=None, stream=None) -> torch.Tensor:
    """y = the FP4 layer(x) through moe_w4_forward (NVFP4 experts, see make_w4_planes)."""
    L = load()
    _check_cuda(x, "x", torch.bfloat16)
    _check_cuda(topk_ids, "topk_ids", torch.int32)
    _check_cuda(topk_weights, "topk_weights", torch.float32)
    p = planes if isinstance(planes, W4Planes) else make_w4_planes(planes)
    T, H = x.shape
    k = topk_ids.shape[1]
    if y is None:
        y = torch.empty_like(x)
    need = w4_workspace_size(T, k, p.num_experts, p.hidden, p.inter)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    st = L.moe_w4_forward(_ptr(x), _ptr(topk_ids), _ptr(topk_weights), ctypes.byref(p), T, k, _ptr(y),
                          _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream))
    if st != OK:
        raise MoeW2Error(st, "moe_w4_forward")
    return y


def cached_workspace_size(T: int, top_k: int, num_slots: int, H: int, I: int) -> int:
    return int(load().moe_w2_forward_cached_workspace_size(T, top_k, num_slots, H, I))


def forward_cached(x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor, planes,
                   slot_of_expert: torch.Tensor, misses=None, y=None, workspace=None, status=None,
                   stream=None) -> torch.Tensor:
    """moe_w2_forward_cached: the forward with planes of resident slots and a residency table
    (int32 [num_routed], slot or negative); misses (device uint32 [1], optional) counts the
    pairs whose expert is not resident."""
    L = load()
    _check_cuda(x, "x", torch.bfloat16)
    _check_cuda(topk_ids, "topk_ids", torch.int32)
    _check_cuda(topk_weights, "topk_weights", torch.float32)
    _check_cuda(slot_of_expert, "slot_of_expert", torch.int32)
    if misses is not None:
        _check_cuda(misses, "misses")
    p = planes if isinstance(planes, Planes) else make_planes(planes)
    T, H = x.shape
    k = topk_ids.shape[1]
    if y is None:
        y = torch.empty_like(x)
    need = cached_workspace_size(T, k, p.num_experts, p.hidden, p.inter)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    st = L.moe_w2_forward_cached(_ptr(x), _ptr(topk_ids), _ptr(topk_weights), ctypes.byref(p), _ptr(slot_of_expert),
                                 slot_of_expert.numel(), T, k, _ptr(y), _ptr(workspace), workspace.numel(),
                                 _ptr(misses), _ptr(status), _stream(stream))
    if st != OK:
        raise MoeW2Error(st, "moe_w2_forward_cached")
    return y


def forward_noalloc(x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor, planes, y=None,
                    status=None, stream=None) -> torch.Tensor:
    """moe_w2_forward_noalloc: the forward with its scratch in the library's own device array
    (for callers that cannot allocate device memory).  Pass y to allocate nothing here either."""
    L = load()
    _check_cuda(x, "x", torch.bfloat16)
    _check_cuda(topk_ids, "topk_ids", torch.int32)
    _check_cuda(topk_weights, "topk_weights", torch.float32)
    p = planes if isinstance(planes, Planes) else make_planes(planes)
    T, H = x.shape
    k = topk_ids.shape[1]
    if y is None:
        y = torch.empty_like(x)
    st = L.moe_w2_forward_noalloc(_ptr(x), _ptr(topk_ids), _ptr(topk_weights), ctypes.byref(p), T, k, _ptr(y),
                                  _ptr(status), _stream(stream))
    if st != OK:
        raise MoeW2Error(st, "moe_w2_forward_noalloc")
    return y


def permute(topk_ids: torch.Tensor, E: int, status=None, stream=None):
    """(sorted_pairs, inv_pairs, expert_offsets) through moe_w2_permute."""
    L = load()
    _check_cuda(topk_ids, "topk_ids", torch.int32)
    T, k = topk_ids.shape
    dev = topk_ids.device
    sorted_pairs = torch.empty(T * k, dtype=torch.int32, device=dev)
    inv = torch.empty(T * k, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    st = L.moe_w2_permute(_ptr(topk_ids), T, k, E, _ptr(sorted_pairs), _ptr(inv), _ptr(offsets), _ptr(status),
                          _stream(stream))
    if st != OK:
        raise MoeW2Error(st, "moe_w2_permute")
    return sorted_pairs, inv, offsets


def requant(e2m1: torch.Tensor, e4m3: torch.Tensor, scale_2: torch.Tensor, codes=None, ue8m0=None,
            status=None, stream=None, options: int = 0):
    """NVFP4 [n][rows][K/2] + [n][rows][K/16] + [n] -> (codes [n][rows][K/4], ue8m0 [n][rows][K/32]).
    options: REQUANT_BALANCE_ZERO_SIGNS or 0 (moe_w2_requant_ex)."""
    L = load()
    _check_cuda(e2m1, "e2m1", torch.uint8)
    _check_cuda(e4m3, "e4m3", torch.uint8)
    _check_cuda(scale_2, "scale_2", torch.float32)
    n, rows, half_k = e2m1.shape
    K = half_k * 2
    if codes is None:
        codes = torch.empty((n, rows, K // 4), dtype=torch.uint8, device=e2m1.device)
    if ue8m0 is None:
        ue8m0 = torch.empty((n, rows, K // 32), dtype=torch.uint8, device=e2m1.device)
    st = L.moe_w2_requant_ex(_ptr(e2m1), _ptr(e4m3), _ptr(scale_2), n, rows, K, options, _ptr(codes), _ptr(ue8m0),
                             _ptr(status), _stream(stream))
    if st != OK:
        raise MoeW2Error(st, "moe_w2_requant_ex")
    return codes, ue8m0


def requant_mxfp4(e2m1: torch.Tensor, scales: torch.Tensor, codes=None, ue8m0=None, status=None, stream=None,
                  options: int = 0):
    """MXFP4: e2m1 [n][rows][K/2] + UE8M0 bytes [n][rows][K/32] -> (codes [n][rows][K/4], ue8m0 [n][rows][K/32])."""
    L = load()
    _check_cuda(e2m1, "e2m1", torch.uint8)
    _check_cuda(scales, "scales", torch.uint8)
    n, rows, half_k = e2m1.shape
    K = half_k * 2
    if tuple(scales.shape) != (n, rows, K // 32):
        raise ValueError(f"scales must be [{n}][{rows}][{K // 32}], got {tuple(scales.shape)}")
    if codes is None:
        codes = torch.empty((n, rows, K // 4), dtype=torch.uint8, device=e2m1.device)
    if ue8m0 is None:
        ue8m0 = torch.empty((n, rows, K // 32), dtype=torch.uint8, device=e2m1.device)
    st = L.moe_w2_requant_mxfp4(_ptr(e2m1), _ptr(scales), n, rows, K, options, _ptr(codes), _ptr(ue8m0),
                                _ptr(status), _stream(stream))
    if st != OK:
        raise MoeW2Error(st, "moe_w2_requant_mxfp4")
    return codes, ue8m0


def requant_fp8(w8: torch.Tensor, scales: torch.Tensor, codes=None, ue8m0=None, status=None, stream=None):
    """FP8 block-128: e4m3 bytes [n][rows][K] + f32 [n][ceil(rows/128)][ceil(K/128)]
    -> (codes [n][rows][K/4], ue8m0 [n][rows][K/32])."""
    L = load()
    _check_cuda(w8, "w8", torch.uint8)
    _check_cuda(scales, "scales", torch.float32)
    n, rows, K = w8.shape
    if tuple(scales.shape) != (n, (rows + 127) // 128, (K + 127) // 128):
        raise ValueError(f"scales must be [{n}][{(rows + 127) // 128}][{(K + 127) // 128}], got {tuple(scales.shape)}")
    if codes is None:
        codes = torch.empty((n, rows, K // 4), dtype=torch.uint8, device=w8.device)
    if ue8m0 is None:
        ue8m0 = torch.empty((n, rows, K // 32), dtype=torch.uint8, device=w8.device)
    st = L.moe_w2_requant_fp8(_ptr(w8), _ptr(scales), n, rows, K, _ptr(codes), _ptr(ue8m0), _ptr(status),
                              _stream(stream))
    if st != OK:
        raise MoeW2Error(st, "moe_w2_requant_fp8")
    return codes, ue8m0
