"""C ABI checks that need no GPU: the library builds, loads and exports every
declared symbol; host-only entry points (planners, shape checks, workspace
sizes) behave as documented.  No device compute is called here."""
import ctypes
import os
import re

import numpy as np
import pytest

import seeded_inputs as si
from oracle import packing as op

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def va():
    from packed_sequence_varlen_gb300 import build as b
    b.build()
    import packed_sequence_varlen_gb300 as pkg
    pkg._lib.load()
    return pkg


def header_functions():
    text = open(os.path.join(ROOT, "include", "varlen_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(varlen_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(va):
    lib = va._lib.load()
    declared = header_functions()
    assert len(declared) >= 14
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(va._lib.EXPORTS) == declared
    assert b"sm_103a" in lib.varlen_version()


def test_library_is_built_for_sm103a_only(va):
    from packed_sequence_varlen_gb300 import build as b
    assert b.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


@pytest.mark.parametrize("name", ["sft8k", "gqa16k", "tiny4k"])
def test_host_planners_match_oracle(va, name):
    lengths = si.raw_lengths(name).tolist()
    cap = si.WORKLOADS[name].capacity
    assert va.pack_next_fit(lengths, cap) == op.next_fit(lengths, cap)
    assert va.pack_best_fit_decreasing(lengths, cap) == op.best_fit_decreasing(lengths, cap)


def test_host_planner_random_and_errors(va):
    rng = np.random.default_rng(7)
    for _ in range(200):
        n = int(rng.integers(0, 80))
        cap = int(rng.integers(8, 200))
        lengths = rng.integers(1, cap + 1, size=n).tolist()
        assert va.pack_next_fit(lengths, cap) == op.next_fit(lengths, cap)
        assert va.pack_best_fit_decreasing(lengths, cap) == op.best_fit_decreasing(lengths, cap)
    assert va.pack_next_fit([3, 2, 4], 6) == [[0, 1], [2]]     # course capacity-6 example
    with pytest.raises(va.VarlenError) as e:
        va.pack_next_fit([7], 6)
    assert e.value.status == 7
    with pytest.raises(va.VarlenError) as e:
        va.pack_best_fit_decreasing([0, 3], 6)
    assert e.value.status == 1
    # any flat integer sequence; nothing is converted silently
    assert va.pack_next_fit(np.array([3, 2, 4], dtype=np.int64), 6) == [[0, 1], [2]]
    assert va.pack_best_fit_decreasing((3, 2, 4), 6) == op.best_fit_decreasing([3, 2, 4], 6)
    assert va.pack_next_fit([], 6) == []
    for bad, err in (([3.5, 2], TypeError), ([[1, 2]], TypeError), ([2 ** 40], ValueError)):
        with pytest.raises(err):
            va.pack_next_fit(bad, 6)


def test_tile_sizes_and_workspace(va):
    for kind in (0, 1, 2):
        for d in (64, 128):
            BM, BN = va.tile_sizes(kind, d)
            assert BM > 0 and BN > 0
            assert (BM % BN == 0) if kind != 1 else (BN % BM == 0)
    n0 = va.workspace_size(8192, 10, 32, 32, 128, 2048, False)
    n1 = va.workspace_size(8192, 10, 32, 32, 128, 2048, True)
    assert n0 >= 256 and n1 >= 256 + 32 * 8192 * 4
    with pytest.raises(va.VarlenError) as e:
        va.workspace_size(8192, 10, 32, 32, 96, 2048, False)
    assert e.value.status == 2                                   # d = 96 unsupported
    with pytest.raises(va.VarlenError) as e:
        va.workspace_size(8192, 10, 30, 8, 128, 2048, False)
    assert e.value.status == 2                                   # Hq % Hkv != 0


def test_host_side_argument_errors(va):
    """Entry points reject bad arguments on the host, before touching a device."""
    lib = va._lib.load()
    s = va._lib.VaShape()
    lib.varlen_shape_contiguous(ctypes.byref(s), 16, 1, 2, 2, 64, 16)
    p = ctypes.c_void_p(16)
    # null q
    st = lib.varlen_attn_fwd(None, p, p, p, ctypes.byref(s), 0.125, 1, p, p, p, 1 << 20, None)
    assert st == 1 and b"null" in lib.varlen_last_error()
    # misaligned pointer
    bad = ctypes.c_void_p(18)
    st = lib.varlen_attn_fwd(bad, p, p, p, ctypes.byref(s), 0.125, 1, p, p, p, 1 << 20, None)
    assert st == 1 and b"aligned" in lib.varlen_last_error()
    # workspace too small
    st = lib.varlen_attn_fwd(p, p, p, p, ctypes.byref(s), 0.125, 1, p, p, p, 16, None)
    assert st == 3
    # bad scale
    st = lib.varlen_attn_fwd(p, p, p, p, ctypes.byref(s), float("nan"), 1, p, p, p, 1 << 20, None)
    assert st == 1
    # stride not a multiple of 8
    s2 = va._lib.VaShape()
    lib.varlen_shape_contiguous(ctypes.byref(s2), 16, 1, 2, 2, 64, 16)
    s2.q_row_stride = 130
    st = lib.varlen_attn_bwd(p, p, p, p, p, p, p, ctypes.byref(s2), 0.125, 1, p, p, p, p, 1 << 24, None)
    assert st == 1
    # max_seqlen beyond T
    s3 = va._lib.VaShape()
    lib.varlen_shape_contiguous(ctypes.byref(s3), 16, 1, 2, 2, 64, 17)
    assert lib.varlen_attn_workspace_size(ctypes.byref(s3), 0) == 0


def test_loss_entry_points_reject_bad_arguments(va):
    """The packed-loss entry points check their arguments on the host."""
    lib = va._lib.load()
    p = ctypes.c_void_p(16)
    assert lib.varlen_token_ce_workspace_size(1000) == 256 + 4096  # header + 4 bytes a row, 256-aligned
    assert lib.varlen_token_ce_workspace_size(-1) == 0
    ws = lib.varlen_token_ce_workspace_size(8)
    assert lib.varlen_loss_targets(None, p, 1, 8, -100, p, None) == 1
    assert lib.varlen_loss_targets(p, p, 0, 8, -100, p, None) == 1
    # null logits, bad dtype, stride below V, misaligned or small workspace
    assert lib.varlen_token_ce(None, 1, 64, p, 8, 64, -100, p, p, None, 0, p, ws, None) == 1
    assert lib.varlen_token_ce(p, 2, 64, p, 8, 64, -100, p, p, None, 0, p, ws, None) == 1
    assert lib.varlen_token_ce(p, 1, 63, p, 8, 64, -100, p, p, None, 0, p, ws, None) == 1
    assert lib.varlen_token_ce(p, 1, 64, p, 8, 64, -100, p, p, p, 32, p, ws, None) == 1
    assert lib.varlen_token_ce(p, 1, 64, p, 8, 64, -100, p, p, None, 0, ctypes.c_void_p(24), ws, None) == 1
    assert lib.varlen_token_ce(p, 1, 64, p, 8, 64, -100, p, p, None, 0, p, ws - 16, None) == 3


def test_bridge_entry_points_reject_bad_arguments(va):
    """The padded-batch bridge checks its arguments on the host."""
    lib = va._lib.load()
    p = ctypes.c_void_p(16)
    assert lib.varlen_unpad_index(None, 2, 8, p, p, p, p, p, p, None) == 1
    assert lib.varlen_unpad_index(p, 0, 8, p, p, p, p, p, p, None) == 1
    assert lib.varlen_unpad_index(p, 65536, 65536, p, p, p, p, p, p, None) == 1  # Bp * S >= 2^31
    assert lib.varlen_gather_rows(p, 64, p, 4, 24, p, 64, None) == 1     # row not a multiple of 16
    assert lib.varlen_gather_rows(p, 16, p, 4, 32, p, 64, None) == 1     # stride below the row
    assert lib.varlen_gather_rows(ctypes.c_void_p(8), 64, p, 4, 32, p, 64, None) == 1  # misaligned
    assert lib.varlen_gather_rows(p, 64, p, -1, 32, p, 64, None) == 1


def test_noalloc_size_limit_is_the_forward_workspace(va):
    """The allocation-free forward takes a shape exactly when the ordinary forward's workspace
    fits its 1 MiB static array; past that it returns VA_ERR_WORKSPACE before any CUDA call."""
    lib = va._lib.load()
    T, H, d = 65536, 8, 64

    def size(B):
        s = va._lib.VaShape()
        lib.varlen_shape_contiguous(ctypes.byref(s), T, B, H, H, d, 1)
        return s, lib.varlen_attn_workspace_size(ctypes.byref(s), 0)

    # the documented formula: 256 + align256(16 (T/256 + B) H) + align256(4 B)
    a256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for B in (1, 100, 7000, 7693, 7694):
        assert size(B)[1] == 256 + a256(16 * (T // 256 + B) * H) + a256(4 * B)
    inside = max(B for B in range(7000, 8000) if size(B)[1] <= 1 << 20)
    s, n = size(inside + 1)
    assert n > 1 << 20
    p = ctypes.c_void_p(256)
    assert lib.varlen_attn_fwd_noalloc(p, p, p, p, ctypes.byref(s), 0.1, 1, p, p, None) == 3
    assert b"1048576" in lib.varlen_last_error()
    assert lib.varlen_noalloc_read_status(None, None) == 1
