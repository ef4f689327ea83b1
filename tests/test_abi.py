"""The C ABI on the host (no GPU needed): the library builds, loads, exports
every function include/attn.h declares, and rejects bad arguments with the
documented status codes before touching CUDA."""
import ctypes
import os
import re

import pytest

from attention_forward_sm_gb300 import binding as attn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    from attention_forward_sm_gb300 import _build
    _build.build()
    return attn.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(attn.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(attn.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_status_strings(lib):
    for code, name in attn.ATTN_STATUS.items():
        assert attn.attn_status_string(code).startswith(name)
    assert "unknown" in attn.attn_status_string(-100)


def test_workspace_bytes(lib):
    assert attn.attn_decode_workspace_bytes(8, 32, 128, 32) == 8 * 32 * 32 * 129 * 4
    assert attn.attn_decode_workspace_bytes(0, 32, 128, 32) == 0


ALIGNED = 0x10000  # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("args,status", [
    ((0, ALIGNED, ALIGNED, ALIGNED, ALIGNED, 1, 2, 2, 8, 8, 64, 0, 0.1), -1),
    ((ALIGNED,) * 5 + (1, 3, 2, 8, 8, 64, 0, 0.1), -3),          # Hq % Hkv
    ((ALIGNED,) * 5 + (1, 2, 2, 8, 8, 96, 0, 0.1), -3),          # D
    ((ALIGNED,) * 5 + (0, 2, 2, 8, 8, 64, 0, 0.1), -3),          # B
    ((ALIGNED,) * 5 + (1, 2, 2, 0, 8, 64, 0, 0.1), -3),          # Nq
    ((ALIGNED,) * 5 + (1, 2, 2, 8, 8, 64, 0, -0.5), -3),         # negative scale
    ((ALIGNED,) * 5 + (1, 2, 2, 8, 8, 64, 0, float("inf")), -3),  # non-finite scale
    ((ALIGNED + 8,) + (ALIGNED,) * 4 + (1, 2, 2, 8, 8, 64, 0, 0.1), -2),
])
def test_fwd_validation(lib, args, status):
    assert lib.attn_fwd(*args, None) == status


@pytest.mark.parametrize("q_offset,causal,status", [
    (-1, 1, -3),                 # negative offset
    (-1, 0, -3),                 # rejected without the causal mask too
    (2**31 - 8 - 1024, 1, -3),   # offset + rows would overflow the kernel's int rows
])
def test_fwd_rows_validation(lib, q_offset, causal, status):
    args = (ALIGNED,) * 5 + (1, 2, 2, 8, 8, 64, causal, q_offset, 0.1)
    assert lib.attn_fwd_rows(*args, None) == status
    bad_ptr = (0,) + (ALIGNED,) * 4 + (1, 2, 2, 8, 8, 64, causal, 0, 0.1)
    assert lib.attn_fwd_rows(*bad_ptr, None) == -1


@pytest.mark.parametrize("fn", ["attn_decode_splitkv", "attn_decode_splitkv_noalloc"])
@pytest.mark.parametrize("args,status", [
    ((ALIGNED, 0, ALIGNED, ALIGNED, ALIGNED, 1, 4, 2, 16, 128, 4), -1),
    ((ALIGNED,) * 5 + (1, 4, 2, 16, 128, 17), -3),   # nsplit > Nk
    ((ALIGNED,) * 5 + (1, 4, 2, 16, 128, 0), -3),    # nsplit < 1
    ((ALIGNED,) * 5 + (1, 4, 3, 16, 128, 4), -3),    # Hq % Hkv
    ((ALIGNED,) * 5 + (1, 4, 2, 16, 80, 4), -3),     # D
    ((ALIGNED,) * 4 + (ALIGNED + 4,) + (1, 4, 2, 16, 128, 4), -2),
])
def test_decode_validation(lib, fn, args, status):
    assert getattr(lib, fn)(*args, None) == status


def test_noalloc_scratch_limit(lib):
    # 64*64*64*(128+1)*4 bytes > 8 MiB
    assert lib.attn_decode_splitkv_noalloc(*(ALIGNED,) * 5, 64, 64, 8, 64, 128, 64, None) == -9


def test_selftest_limit_validation(lib):
    assert lib.attn_selftest_wait_timeout(0, None) == -3
    assert lib.attn_selftest_wait_timeout(2000000, None) == -3


def test_states_and_combine_validation(lib):
    A = ALIGNED
    assert lib.attn_decode_splitkv_states(A, A, A, 0, A, 1, 4, 2, 16, 128, 4, None) == -1
    assert lib.attn_decode_splitkv_states(A, A, A, A, A, 1, 4, 2, 16, 128, 17, None) == -3
    assert lib.attn_combine_states(A, A, A, A, 0, 4, 128, None) == -3
    assert lib.attn_combine_states(A, A, A, A, 4, 0, 128, None) == -3
    assert lib.attn_combine_states(A, A, A, A, 4, 4, 96, None) == -3
    assert lib.attn_combine_states(A + 4, A, A, A, 4, 4, 128, None) == -2


def test_decode_graph_validation(lib):
    A = ALIGNED
    h = ctypes.c_void_p()
    # out == NULL
    assert lib.attn_decode_graph_create(A, A, A, A, A, 1, 4, 2, 16, 128, 4, None) == -1
    # NULL tensor, bad shapes, nsplit > Nk, misaligned: rejected before any CUDA call
    assert lib.attn_decode_graph_create(A, A, A, 0, A, 1, 4, 2, 16, 128, 4, ctypes.byref(h)) == -1
    assert lib.attn_decode_graph_create(A, A, A, A, A, 1, 4, 3, 16, 128, 4, ctypes.byref(h)) == -3
    assert lib.attn_decode_graph_create(A, A, A, A, A, 1, 4, 2, 16, 96, 4, ctypes.byref(h)) == -3
    assert lib.attn_decode_graph_create(A, A, A, A, A, 1, 4, 2, 16, 128, 17, ctypes.byref(h)) == -3
    assert lib.attn_decode_graph_create(A + 8, A, A, A, A, 1, 4, 2, 16, 128, 4,
                                        ctypes.byref(h)) == -2
    assert h.value is None  # nothing handed out on failure
    assert lib.attn_decode_graph_launch(None, None) == -1
    assert lib.attn_decode_graph_destroy(None) == 0


def test_fwd_fp8_validation(lib):
    A = ALIGNED
    args = (1, 2, 1, 128, 256, 128, 0)
    assert lib.attn_fwd_fp8(0, A, A, A, A, *args, 0.1, 1.0, 1.0, 1.0, None) == -1
    assert lib.attn_fwd_fp8(A, A, A, A, A, 1, 2, 1, 128, 250, 128, 0, 0.1, 1.0, 1.0, 1.0,
                            None) == -3  # Nk % 16
    assert lib.attn_fwd_fp8(A, A, A, A, A, 1, 2, 1, 128, 256, 64, 0, 0.1, 1.0, 1.0, 1.0,
                            None) == -3  # D
    assert lib.attn_fwd_fp8(A, A, A, A, A, *args, 0.1, float("nan"), 1.0, 1.0, None) == -3
    assert lib.attn_fwd_fp8(A, A, A, A, A, *args, 0.1, 1.0, 1.0, -2.0, None) == -3
    assert lib.attn_fwd_fp8(A, A, A + 4, A, A, *args, 0.1, 1.0, 1.0, 1.0, None) == -2


def test_fwd_host_validation(lib):
    A = ALIGNED
    assert lib.attn_fwd_host(0, A, A, A, A, 1, 2, 2, 8, 8, 64, 0, 0.1, None) == -1
    assert lib.attn_fwd_host(A, A, A, A, A, 1, 3, 2, 8, 8, 64, 0, 0.1, None) == -3
    assert lib.attn_fwd_host(A, A, A, A, A, 1, 2, 2, 8, 8, 96, 0, 0.1, None) == -3
    assert lib.attn_fwd_host(A, A, A, A, A, 1, 2, 2, 8, 8, 64, 0, -1.0, None) == -3


def test_fwd_host_workspace_plan(lib):
    # B8 Hq=Hkv=32 N8192 D128: 32 q-tile pairs per head -> 19 heads fill four
    # waves of 152 CTAs -> two blocks of 16 heads; a slot holds q, k, v, o of
    # 16 heads and their lse
    per_head = 8192 * 128 * 2
    slot = 4 * 16 * per_head + 16 * 8192 * 4
    assert attn.attn_fwd_host_workspace_bytes(8, 32, 32, 8192, 8192, 128) == 2 * slot
    assert attn.attn_fwd_host_workspace_bytes(0, 32, 32, 8192, 8192, 128) == 0


def test_tensor_helpers_reject_bad_inputs():
    """forward / decode check dtype, device, contiguity and matching sizes
    before any library call (the raw C-ABI names take pointers and cannot)."""
    import torch
    from attention_forward_sm_gb300 import binding as attn
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        attn.forward(q, q, q)
    with pytest.raises(TypeError, match="bfloat16"):
        attn.forward(q.float(), q, q)
    with pytest.raises(ValueError, match="dimensions"):
        attn.forward(q[0], q, q)
    q1 = torch.zeros(1, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        attn.decode(q1, q, q, nsplit=2)
    with pytest.raises(TypeError, match="torch tensor"):
        attn.decode(q1, 0, q, nsplit=2)
