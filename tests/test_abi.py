"""The C ABI library builds, loads and exports every entry point declared in
include/moe_w2.h; host-side argument checks answer without a GPU (CPU only)."""
import ctypes
import os
import re

from bit_moe_expert_w2_gb300 import moe_w2

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "moe_w2.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_w2_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    L = moe_w2.load()
    names = _declared()
    assert {"moe_w2_forward", "moe_w2_permute", "moe_w2_requant", "moe_w2_forward_workspace_size"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version():
    L = moe_w2.load()
    assert L.moe_w2_version() >= 1
    for s in range(6):
        assert moe_w2.status_string(s)


def test_workspace_size_rules():
    assert moe_w2.workspace_size(1, 8, 256, 6144, 2048) > 0
    assert moe_w2.workspace_size(8192, 8, 256, 4096, 2048) > 8192 * 8 * 4096 * 4   # fp32 staging
    assert moe_w2.workspace_size(4, 2, 8, 500, 256) == 0      # H not a multiple of 256
    assert moe_w2.workspace_size(4, 17, 8, 512, 256) == 0     # top_k > 16
    assert moe_w2.workspace_size(4, 2, 2000, 512, 256) == 0   # E > 1024
    assert moe_w2.workspace_size(-1, 2, 8, 512, 256) == 0


def test_host_validation_without_device():
    L = moe_w2.load()
    p = moe_w2.Planes(0, 0, 0, 0, 8, 512, 256)
    # null planes pointer, bad top_k, bad shape: rejected on the host
    assert L.moe_w2_forward(None, None, None, None, 1, 2, None, None, 0, None, None) == 1
    assert L.moe_w2_forward(None, None, None, ctypes.byref(p), 1, 0, None, None, 0, None, None) == 1
    bad = moe_w2.Planes(0, 0, 0, 0, 8, 500, 256)
    assert L.moe_w2_forward(None, None, None, ctypes.byref(bad), 1, 2, None, None, 0, None, None) == 2
    # T = 0 is a no-op
    assert L.moe_w2_forward(None, None, None, ctypes.byref(p), 0, 2, None, None, 0, None, None) == 0
    # requant: K not a multiple of 32, and the empty call
    assert L.moe_w2_requant(None, None, None, 1, 1, 48, None, None, None, None) == 2
    assert L.moe_w2_requant(None, None, None, 0, 4, 64, None, None, None, None) == 0
    # permute: top_k out of range
    assert L.moe_w2_permute(None, 4, 0, 8, None, None, None, None, None) == 1


def test_alignment_and_workspace_checks_answer_before_any_device_access():
    """Fake device addresses are never dereferenced: alignment and workspace size
    are checked on the host first (status 1 = invalid argument, 3 = workspace)."""
    L = moe_w2.load()
    A = 0x10000000            # 256-byte aligned stand-in addresses
    p = moe_w2.Planes(A, A + 0x1000, A + 0x2000, A + 0x3000, 8, 512, 256)
    need = moe_w2.workspace_size(2, 2, 8, 512, 256)
    ok = dict(x=A, ids=A, w=A, y=A + 0x100000, ws=A + 0x200000)

    def fwd(planes=p, nbytes=need, **kw):
        a = {**ok, **kw}
        return L.moe_w2_forward(a["x"], a["ids"], a["w"], ctypes.byref(planes), 2, 2, a["y"], a["ws"], nbytes,
                                None, None)

    assert fwd(ws=A + 0x200080) == 1                   # workspace not 256-byte aligned
    assert fwd(x=A + 8) == 1                           # x not 16-byte aligned
    assert fwd(y=A + 0x100004) == 1                    # y not 16-byte aligned
    assert fwd(planes=moe_w2.Planes(A, A + 0x1008, A + 0x2000, A + 0x3000, 8, 512, 256)) == 1   # scales
    assert fwd(planes=moe_w2.Planes(A, A + 0x1000, A + 0x2000, 0, 8, 512, 256)) == 1           # null plane
    assert fwd(nbytes=need - 1) == 3                   # workspace one byte short
    # requant: misaligned e2m1, e4m3 and codes pointers
    assert L.moe_w2_requant(A + 8, A, A, 1, 4, 64, A, A, None, None) == 1
    assert L.moe_w2_requant(A, A + 1, A, 1, 4, 64, A, A, None, None) == 1
    assert L.moe_w2_requant(A, A, A, 1, 4, 64, A + 4, A, None, None) == 1
    # permute: more pairs than the library takes
    assert L.moe_w2_permute(A, 1 << 20, 16, 8, A, A, A, None, None) == 2


def test_forward_path_names_the_kernels_a_call_runs():
    P = moe_w2
    assert P.forward_path(1, 8, 256, 6144, 2048) == P.PATH_DECODE_STREAM          # 8 pairs
    assert P.forward_path(2, 8, 256, 6144, 2048) == P.PATH_DECODE_STREAM          # 16 pairs
    assert P.forward_path(3, 8, 256, 6144, 2048) == P.PATH_DECODE_BLOCK_SCALED    # 24 pairs
    assert P.forward_path(32, 8, 256, 6144, 2048) == P.PATH_DECODE_BLOCK_SCALED
    assert P.forward_path(64, 8, 256, 6144, 2048) == P.PATH_DECODE_BLOCK_SCALED
    assert P.forward_path(65, 8, 256, 6144, 2048) == P.PATH_PREFILL
    assert P.forward_path(8192, 8, 256, 4096, 2048) == P.PATH_PREFILL
    assert P.forward_path(32, 8, 8, 768, 512) == P.PATH_DECODE_MMA                # H not a multiple of 512
    assert P.forward_path(32, 8, 8, 512, 256) == P.PATH_DECODE_MMA                # I not a multiple of 512
    assert P.forward_path(1, 8, 8, 512, 256) == P.PATH_DECODE_MMA
    assert P.forward_path(0, 8, 256, 6144, 2048) == P.PATH_NONE
    assert P.forward_path(4, 2, 8, 500, 256) == P.PATH_NONE                       # invalid H
    assert P.decode_kernel(1, 8, 6144, 2048) == "decode_stream_kernel"
    assert P.decode_kernel(32, 8, 6144, 2048) == "decode_layer_kernel"
    # the stream-K kernel takes steps of at most 16 pairs with H and I multiples
    # of 512 (up to 7168); the rest of the small steps the mma.sync kernel
    assert P.forward_path(3, 8, 256, 6144, 2048) == P.PATH_DECODE_BLOCK_SCALED
    assert P.forward_path(1, 8, 8, 7680, 2048) == P.PATH_DECODE_MMA
    assert P.decode_kernel(1, 8, 6144, 1792) == "decode_mma_kernel"
    with P.decode_stream(False):
        # deselected: the mma.sync kernel takes them
        assert P.forward_path(1, 8, 256, 6144, 2048) == P.PATH_DECODE_MMA
        assert P.forward_path(2, 8, 256, 6144, 2048) == P.PATH_DECODE_MMA
        assert P.decode_kernel(1, 8, 6144, 2048) == "decode_mma_kernel"
        assert P.workspace_size(1, 8, 256, 6144, 2048) > 0
    assert P.forward_path(1, 8, 256, 6144, 2048) == P.PATH_DECODE_STREAM


def test_cached_forward_host_checks():
    """moe_w2_forward_cached: table length and pointer checks, and a workspace
    that covers the per-pair slot ids (checked before any device access)."""
    L = moe_w2.load()
    A = 0x10000000
    p = moe_w2.Planes(A, A + 0x1000, A + 0x2000, A + 0x3000, 8, 512, 256)
    need = moe_w2.cached_workspace_size(2, 2, 8, 512, 256)
    assert need >= moe_w2.workspace_size(2, 2, 8, 512, 256) + 4 * 4
    assert moe_w2.cached_workspace_size(4, 2, 8, 500, 256) == 0

    def fwd(table=A + 0x400000, n_route=300, nbytes=need, T=2):
        return L.moe_w2_forward_cached(A, A, A, ctypes.byref(p), table, n_route, T, 2, A + 0x100000, A + 0x200000,
                                       nbytes, None, None, None)

    assert fwd(n_route=0) == 1                          # empty table
    assert fwd(n_route=(1 << 20) + 1) == 1              # longer than the library takes
    assert fwd(table=None) == 1                         # no table
    assert fwd(nbytes=need - 1) == 3                    # no room for the slot ids
    assert fwd(table=None, T=0) == 0                    # T = 0 is a no-op


def test_fp4_loader_options_host_checks():
    L = moe_w2.load()
    A = 0x10000000
    # reserved option bits are refused before any device access
    assert L.moe_w2_requant_ex(A, A, A, 1, 4, 64, 2, A, A, None, None) == 1
    assert L.moe_w2_requant_mxfp4(A, A, 1, 4, 64, 0x80, A, A, None, None) == 1
    # MXFP4: K not a multiple of 32, misaligned e2m1 and codes, the empty call
    assert L.moe_w2_requant_mxfp4(A, A, 1, 4, 48, 0, A, A, None, None) == 2
    assert L.moe_w2_requant_mxfp4(A + 8, A, 1, 4, 64, 0, A, A, None, None) == 1
    assert L.moe_w2_requant_mxfp4(A, A, 1, 4, 64, 0, A + 4, A, None, None) == 1
    assert L.moe_w2_requant_mxfp4(None, None, 0, 4, 64, 1, None, None, None, None) == 0


def test_w4_forward_host_checks():
    """moe_w4_forward: the same host checks as moe_w2_forward, plus its scale_2 arrays."""
    L = moe_w2.load()
    A = 0x10000000
    need = moe_w2.w4_workspace_size(2, 2, 8, 512, 256)
    assert need > 0 and moe_w2.w4_workspace_size(2, 2, 8, 500, 256) == 0
    ok = moe_w2.W4Planes(A, A + 0x1000, A + 0x2000, A + 0x3000, A + 0x4000, A + 0x5000, 8, 512, 256)

    def fwd(p=ok, nbytes=need, T=2):
        return L.moe_w4_forward(A, A, A, ctypes.byref(p), T, 2, A + 0x100000, A + 0x200000, nbytes, None, None)

    assert L.moe_w4_forward(A, A, A, None, 2, 2, A, A, need, None, None) == 1
    assert fwd(p=moe_w2.W4Planes(A, A + 0x1000, 0, A + 0x3000, A + 0x4000, A + 0x5000, 8, 512, 256)) == 1   # no scale_2
    assert fwd(p=moe_w2.W4Planes(A, A + 0x1000, A + 0x2002, A + 0x3000, A + 0x4000, A + 0x5000, 8, 512, 256)) == 1
    assert fwd(p=moe_w2.W4Planes(A, A + 0x1008, A + 0x2000, A + 0x3000, A + 0x4000, A + 0x5000, 8, 512, 256)) == 1
    assert fwd(p=moe_w2.W4Planes(A, A, A, A, A, A, 8, 500, 256)) == 2
    assert fwd(nbytes=need - 1) == 3
    assert fwd(T=0) == 0
