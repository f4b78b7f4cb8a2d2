"""The C-ABI library on a machine without a GPU: it loads, exports every entry point the
header declares, and validates arguments before touching CUDA."""
import ctypes
import math
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine",
                 "moe_layer_forward", "moe_workspace_size", "moe_pack_weights"):
        assert must in names


@pytest.fixture(scope="module")
def moe():
    import expert_token_dispatch_gemm_b300 as m
    return m


def test_library_exports_every_declared_symbol(moe):
    lib = ctypes.CDLL(moe.binding._LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", moe.binding._LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (moe_\w+)$", out, flags=re.M))
    assert set(declared_functions()) <= exported


def test_library_is_built_for_sm103a_only(moe):
    out = subprocess.run(["cuobjdump", "--list-elf", moe.binding._LIB_PATH],
                         capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    arches = set(re.findall(r"sm_(\d+a?)", out.stdout))
    assert arches == {"103a"}, arches


def cfg(moe, **kw):
    base = dict(N=64, H=64, I=32, E=8, top_k=2, ep_size=4)
    base.update(kw)
    return moe.config(**base)


def status_of(moe, c):
    n = ctypes.c_size_t(0)
    return moe.lib.moe_workspace_size(ctypes.byref(c), ctypes.byref(n)), n.value


@pytest.mark.parametrize("kw,status", [
    (dict(), 0),
    (dict(N=0), 0),
    (dict(E=6, ep_size=4), 1),       # ep_size must divide E
    (dict(H=60), 1),                 # hidden multiple of 8
    (dict(I=12), 1),
    (dict(top_k=9), 1),              # k <= E
    (dict(top_k=0), 1),
    (dict(N=-1), 1),
    (dict(E=512, ep_size=8), 2),     # beyond the kernels' limit
    (dict(E=64, top_k=33, ep_size=8), 2),
    (dict(capacity_factor=float("nan")), 1),
    (dict(capacity_factor=1.25), 0),
    (dict(mode="mask_sum"), 0),
    (dict(dtype="fp32"), 0),
    (dict(group_limit=-1), 1),
    (dict(group_limit=1), 0),                      # 1 partition of 2 experts holds k = 2
    (dict(group_limit=1, ep_size=8), 1),           # 1 partition of 1 expert < k = 2
    (dict(group_limit=4), 0),                      # >= ep_size: no limit
    (dict(E=128, ep_size=16, group_limit=9), 2),   # beyond the supported group limit
    (dict(E=128, ep_size=128, group_limit=2), 2),  # beyond the supported partition count
    (dict(capacity_priority="slot"), 0),
])
def test_config_validation(moe, kw, status):
    c = cfg(moe, **kw)
    st, n = status_of(moe, c)
    assert st == status, moe.lib.moe_last_error()
    if st == 0:
        assert n > 0
    else:
        assert moe.lib.moe_last_error().decode()


def test_workspace_size_grows_with_tokens_not_with_mode(moe):
    _, a = status_of(moe, cfg(moe, N=64))
    _, b = status_of(moe, cfg(moe, N=640))
    _, c = status_of(moe, cfg(moe, N=640, mode="mask_sum"))
    assert a < b
    # the send buffer, h and out_slots alone need pairs * (2H + Ipad) * 2 bytes
    pairs = 640 * 2
    assert b >= pairs * (2 * 64 + 128) * 2
    # mask-and-sum keeps each partition's partial in registers: no extra buffer
    assert c == b


def test_packed_size(moe):
    n = ctypes.c_size_t(0)
    c = cfg(moe, I=200)
    assert moe.lib.moe_packed_gate_up_size(ctypes.byref(c), ctypes.byref(n)) == 0
    assert n.value == 8 * 2 * 256 * 64 * 2   # Ipad = 256


FAKE = ctypes.c_void_p(1 << 20)   # aligned, never dereferenced: validation fails first


def test_forward_rejects_missing_or_small_workspace(moe):
    c = cfg(moe)
    P = FAKE
    st = moe.lib.moe_layer_forward(ctypes.byref(c), P, P, None, P, P, P, None, None, 0, None)
    assert st == moe.binding.MOE_ERR_WORKSPACE
    st = moe.lib.moe_layer_forward(ctypes.byref(c), P, P, None, P, P, P, None, P, 100, None)
    assert st == moe.binding.MOE_ERR_WORKSPACE
    assert "needed" in moe.lib.moe_last_error().decode()


def test_forward_rejects_misaligned_or_null_pointers(moe):
    c = cfg(moe)
    _, n = status_of(moe, c)
    P = FAKE
    bad = ctypes.c_void_p((1 << 20) + 8)
    st = moe.lib.moe_layer_forward(ctypes.byref(c), bad, P, None, P, P, P, None, P, n, None)
    assert st == moe.binding.MOE_ERR_INVALID_ARG
    assert "x must be 16-byte aligned" in moe.lib.moe_last_error().decode()
    st = moe.lib.moe_layer_forward(ctypes.byref(c), None, P, None, P, P, P, None, P, n, None)
    assert st == moe.binding.MOE_ERR_INVALID_ARG
    cb = cfg(moe, has_bias=True)
    st = moe.lib.moe_layer_forward(ctypes.byref(cb), P, P, None, P, P, P, None, P, n, None)
    assert st == moe.binding.MOE_ERR_INVALID_ARG
    assert "b_router" in moe.lib.moe_last_error().decode()
    st = moe.lib.moe_route(None, P, P, None, P, P, None)
    assert st == moe.binding.MOE_ERR_INVALID_ARG


def test_expert_range_validation(moe):
    c = cfg(moe)
    _, n = status_of(moe, c)
    P = FAKE
    for b, e in ((0, 0), (-1, 4), (4, 9), (5, 3)):
        st = moe.lib.moe_expert_ffn(ctypes.byref(c), P, P, b, e, P, P, P, P, P, P, n, None)
        assert st == moe.binding.MOE_ERR_INVALID_ARG


def test_empty_batch_is_a_no_op(moe):
    c = cfg(moe, N=0)
    _, n = status_of(moe, c)
    # no diagnostics requested: nothing is enqueued, so no CUDA call is needed
    st = moe.lib.moe_layer_forward(ctypes.byref(c), None, None, None, None, None, None, None,
                                   FAKE, n, None)
    assert st == 0
    assert moe.lib.moe_route(ctypes.byref(c), None, None, None, None, None, None) == 0


def test_status_strings(moe):
    for s in range(6):
        assert moe.lib.moe_status_string(s).decode().startswith("MOE_")


def test_misaligned_selection_bias_is_rejected_before_any_access(moe):
    c = cfg(moe)
    c.selection_bias = 0x1002     # never dereferenced: validation comes first
    st, _ = status_of(moe, c)
    assert st == 1 and b"selection_bias" in moe.lib.moe_last_error()


def test_unknown_capacity_priority_is_rejected(moe):
    c = cfg(moe)
    c.capacity_priority = 2
    st, _ = status_of(moe, c)
    assert st == 1 and b"capacity_priority" in moe.lib.moe_last_error()
    with pytest.raises(ValueError):
        moe.config(N=8, H=64, I=32, E=8, top_k=2, ep_size=4, capacity_priority="expert")


def test_slot_priority_workspace_holds_its_histograms(moe):
    # k slots x ceil(N / 64k) spans of histograms instead of ceil(N / 64) segments
    _, tok = status_of(moe, cfg(moe, N=4096, E=64, top_k=8, ep_size=8))
    _, slot = status_of(moe, cfg(moe, N=4096, E=64, top_k=8, ep_size=8, capacity_priority="slot"))
    assert slot >= tok


@pytest.mark.parametrize("N,tp", [(0, 1), (0, 3), (1, 2), (1, 4), (7, 3), (8, 2), (5, 8),
                                  (100, 3), (32768, 7)])
def test_tp_slice_matches_the_oracle_rule(moe, N, tp):
    import oracle
    got = [moe.moe_tp_slice(N, tp, r) for r in range(tp)]
    assert got == oracle.tp_slices(N, tp)


@pytest.mark.parametrize("args", [(-1, 2, 0), (4, 0, 0), (4, 2, 2), (4, 2, -1)])
def test_tp_slice_rejects_bad_arguments(moe, args):
    with pytest.raises(moe.MoeError):
        moe.moe_tp_slice(*args)


def test_balance_stats_and_tp_reduce_validate_before_any_access(moe):
    c = cfg(moe)
    ws = ctypes.c_void_p(1 << 20)
    st = moe.lib.moe_balance_stats(ctypes.byref(c), FAKE, None, FAKE, FAKE, ws, 1 << 30, None)
    assert st == 1 and b"routed_counts" in moe.lib.moe_last_error()
    st = moe.lib.moe_balance_stats(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, ws, 16, None)
    assert st == 3                                           # workspace too small
    st = moe.lib.moe_tp_reduce(ctypes.byref(c), 0, FAKE, FAKE, None)
    assert st == 1
    st = moe.lib.moe_tp_reduce(ctypes.byref(c), 2, ctypes.c_void_p((1 << 20) + 4), FAKE, None)
    assert st == 1 and b"aligned" in moe.lib.moe_last_error()


def test_training_grows_the_workspace(moe):
    for dtype in ("bf16", "fp32"):
        c = cfg(moe, dtype=dtype)
        _, base = status_of(moe, c)
        c.training = 1
        st, grown = status_of(moe, c)
        assert st == 0 and grown > base
    c = cfg(moe)
    c.training = 3
    assert status_of(moe, c)[0] == 1


def test_bf16_training_workspace_holds_the_transposed_operands(moe):
    """A bf16 training workspace also holds x^T [H, T] and (w a)^T [Ipad, T], the
    weight-gradient GEMMs' K-major operands (T = N*k rounded up to 64, plus 64 E: every
    expert's rows in whole 64-row blocks), on top of what the fp32 backward needs."""
    N, H, I, E, k = 64, 64, 32, 8, 2
    Ipad = 128
    T = (N * k + 63) // 64 * 64 + 64 * E
    sizes = {}
    for dtype, es in (("bf16", 2), ("fp32", 4)):
        c = cfg(moe, dtype=dtype)
        _, base = status_of(moe, c)
        c.training = 1
        _, grown = status_of(moe, c)
        sizes[dtype] = (grown - base) / es   # elements
    assert sizes["bf16"] - sizes["fp32"] >= (H + Ipad) * T


def test_backward_needs_a_training_config(moe):
    c = cfg(moe)
    st = moe.lib.moe_layer_backward(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                                    FAKE, FAKE, FAKE, FAKE, 1 << 40, None)
    assert st == 1 and b"training" in moe.lib.moe_last_error()
