"""The C ABI library loads, exports every entry point declared in include/moe.h, and its
host-side validation rejects bad arguments before touching the GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

from sparse_mixture_experts_56_b300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_native.LIB_PATH):
        from sparse_mixture_experts_56_b300 import build
        build.build()
    return _native.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_router_topk", "moe_permute", "moe_grouped_swiglu", "moe_combine",
                     "moe_layer_forward", "moe_workspace_size", "moe_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _native.SIGNATURES, f"{name} has no ctypes signature"


def header_constants():
    """NAME = value pairs of the enums in include/moe.h."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(MOE_[A-Z0-9_]+)\s*=\s*(\d+)", src)}


def test_binding_constants_match_the_header():
    """The Python binding's copies of the header's enum values (dtypes, GEMM forms, status
    codes) are the header's."""
    consts = header_constants()
    for name in ("MOE_F32", "MOE_BF16", "MOE_TC_FORM_AUTO", "MOE_TC_FORM_SINGLE",
                 "MOE_TC_FORM_PAIR", "MOE_TC_FORM_SWAP"):
        assert getattr(_native, name) == consts[name], name
    for code, name in _native.STATUS_NAMES.items():
        assert consts[name] == code, name
    assert sorted(v for k, v in consts.items() if k.startswith("MOE_ERR") or k == "MOE_OK") == \
        sorted(_native.STATUS_NAMES)


def test_tc_form_selection_is_validated(lib):
    """Every declared GEMM form is accepted and anything else rejected (no launch happens);
    the default is restored afterwards."""
    try:
        for form in (_native.MOE_TC_FORM_SINGLE, _native.MOE_TC_FORM_PAIR, _native.MOE_TC_FORM_SWAP,
                     _native.MOE_TC_FORM_AUTO):
            assert lib.moe_set_tc_form(form) == OK
        for bad in (-1, 4, 99):
            assert lib.moe_set_tc_form(bad) == INVALID
    finally:
        lib.moe_set_tc_form(_native.MOE_TC_FORM_AUTO)


def test_status_strings(lib):
    for code, name in _native.STATUS_NAMES.items():
        assert lib.moe_status_string(code).decode() == name
    assert lib.moe_status_string(99).decode() == "MOE_ERR_UNKNOWN"
    assert lib.moe_version() >= 100


def test_workspace_size(lib):
    ws = lib.moe_workspace_size
    assert ws(0, 4096, 14336, 8, 2, 1) > 0
    small = ws(32, 4096, 14336, 8, 2, 1)
    big = ws(16384, 4096, 14336, 8, 2, 1)
    assert 0 < small < big
    # x_perm + h + y_perm dominate: A*(2d + f)*2 bytes
    A = 16384 * 2
    assert big >= A * (2 * 4096 + 14336) * 2
    assert ws(64, 128, 256, 8, 2, 0) >= 128 * (2 * 128 + 256) * 4
    for bad in [(-1, 8, 8, 8, 2, 1), (8, 0, 8, 8, 2, 1), (8, 8, 0, 8, 2, 1), (8, 8, 8, 0, 1, 1),
                (8, 8, 8, 33, 2, 1), (8, 8, 8, 8, 9, 1), (8, 8, 8, 8, 0, 1), (8, 8, 8, 8, 2, 7),
                (2 ** 30, 8, 8, 8, 2, 1)]:
        assert ws(*bad) == 0, bad


def test_host_validation_rejects_before_launch(lib):
    nul = None
    fake = ctypes.c_void_p(4096)           # never dereferenced: validation fails first
    # bad dtype / sizes
    assert lib.moe_router_topk(fake, fake, nul, 4, 8, 8, 2, 5, fake, fake, nul, nul) == INVALID
    assert lib.moe_router_topk(fake, fake, nul, 4, 8, 8, 9, 1, fake, fake, nul, nul) == INVALID
    assert lib.moe_router_topk(nul, fake, nul, 4, 8, 8, 2, 1, fake, fake, nul, nul) == INVALID
    assert lib.moe_router_topk(ctypes.c_void_p(4098), fake, nul, 4, 8, 8, 2, 1, fake, fake, nul,
                               nul) == INVALID                        # misaligned x
    # nothing to do for T == 0
    assert lib.moe_router_topk(nul, nul, nul, 0, 8, 8, 2, 1, nul, nul, nul, nul) == OK
    assert lib.moe_grouped_swiglu(nul, nul, nul, nul, nul, nul, 0, 64, 64, 8, 2, 1, nul, nul, 0,
                                  nul) == OK
    assert lib.moe_combine(nul, nul, nul, nul, 0, 64, 2, 1, nul, nul) == OK
    # permute: missing outputs, then a workspace that is too small
    assert lib.moe_permute(fake, 4, 2, 8, nul, fake, fake, fake, 1 << 20, nul) == INVALID
    assert lib.moe_permute(fake, 4, 2, 8, fake, fake, fake, nul, 0, nul) == WORKSPACE
    assert lib.moe_permute(fake, 4, 2, 8, fake, fake, fake, fake, 16, nul) == WORKSPACE
    # grouped: undersized workspace
    need = lib.moe_workspace_size(4, 64, 64, 8, 2, 1)
    assert lib.moe_grouped_swiglu(fake, fake, fake, fake, fake, fake, 4, 64, 64, 8, 2, 1, fake,
                                  fake, 256, nul) == WORKSPACE
    assert lib.moe_layer_forward(fake, fake, nul, fake, fake, fake, nul, 4, 64, 64, 8, 2, 1, fake,
                                 nul, nul, fake, need - 1, nul) == WORKSPACE
    assert lib.moe_layer_forward(fake, fake, nul, nul, fake, fake, nul, 4, 64, 64, 8, 2, 1, fake,
                                 nul, nul, fake, need, nul) == INVALID
    # rmsnorm: aliasing and negative eps
    assert lib.moe_rmsnorm(fake, 4, 64, 1e-5, 1, fake, nul) == INVALID
    assert lib.moe_rmsnorm(fake, 4, 64, -1.0, 1, ctypes.c_void_p(8192), nul) == INVALID
    # routing statistics: bad sizes, missing outputs, misaligned counters, then T == 0 is
    # still a launch (it zeroes the outputs), so only the rejections are checked here
    assert lib.moe_routing_stats(fake, 4, 2, 8, -1, fake, fake, nul) == INVALID
    assert lib.moe_routing_stats(fake, 4, 9, 8, 0, fake, fake, nul) == INVALID
    assert lib.moe_routing_stats(fake, 4, 2, 8, 0, nul, fake, nul) == INVALID
    assert lib.moe_routing_stats(nul, 4, 2, 8, 0, fake, fake, nul) == INVALID
    assert lib.moe_routing_stats(fake, 4, 2, 8, 0, ctypes.c_void_p(4100), fake, nul) == INVALID
    # backward: sizes for both dtypes; bad dtype, workspace and missing pointers rejected
    assert lib.moe_backward_workspace_size(64, 128, 256, 8, 2, 7) == 0
    assert lib.moe_backward_workspace_size(64, 128, 256, 8, 2, 0) > \
        lib.moe_backward_workspace_size(64, 128, 256, 8, 2, 1) > \
        lib.moe_workspace_size(64, 128, 256, 8, 2, 1) // 2
    assert lib.moe_layer_backward(fake, fake, nul, fake, fake, fake, fake, 4, 64, 64, 8, 2, 5,
                                  fake, fake, nul, fake, fake, fake, fake, 1 << 30, nul) == INVALID
    assert lib.moe_layer_backward(fake, fake, nul, fake, fake, fake, fake, 4, 64, 64, 8, 2, 1,
                                  fake, fake, nul, fake, fake, fake, fake, 16, nul) == WORKSPACE
    assert lib.moe_layer_backward(fake, fake, nul, fake, fake, fake, nul, 4, 64, 64, 8, 2, 1,
                                  fake, fake, nul, fake, fake, fake, fake, 1 << 30, nul) == INVALID
    # training pair: tensor-core shapes only; the saved buffer is checked before launch
    assert lib.moe_train_saved_size(64, 128, 256, 8, 2, 0) == 0
    assert lib.moe_train_saved_size(64, 96, 256, 8, 2, 1) == 0
    assert lib.moe_train_saved_size(64, 128, 256, 8, 2, 1) >= 2 * 2 * 256 * (128 + 8 * 127)
    assert lib.moe_layer_forward_train(fake, fake, nul, fake, fake, fake, nul, 4, 64, 64, 8, 2, 0,
                                       fake, fake, 1 << 30, fake, 1 << 30, nul) == UNSUPPORTED
    assert lib.moe_layer_forward_train(fake, fake, nul, fake, fake, fake, nul, 4, 64, 64, 8, 2, 1,
                                       fake, fake, 16, fake, 1 << 30, nul) == WORKSPACE
    assert lib.moe_layer_backward_saved(fake, fake, fake, fake, fake, fake, 4, 64, 64, 8, 2, 1,
                                        fake, 16, fake, fake, nul, fake, fake, fake, fake,
                                        1 << 30, nul) == WORKSPACE
    # attention: head dimension 128 in bf16 only; grouping and workspace checked first
    assert lib.moe_attention_gqa(fake, fake, fake, 8, 0, 8, 3, 128, 1, fake, fake, 256, nul) == INVALID
    assert lib.moe_attention_gqa(fake, fake, fake, 8, 0, 8, 2, 64, 1, fake, fake, 256, nul) == UNSUPPORTED
    assert lib.moe_attention_gqa(fake, fake, fake, 8, 0, 8, 2, 128, 0, fake, fake, 256, nul) == UNSUPPORTED
    assert lib.moe_attention_gqa(fake, fake, fake, 8, 0, 8, 2, 128, 1, fake, fake, 16, nul) == WORKSPACE
    assert lib.moe_attention_gqa(nul, fake, fake, 8, 0, 8, 2, 128, 1, fake, fake, 256, nul) == INVALID
    # expert-parallel regrouping and the row gather: sizes and pointers before launch
    assert lib.moe_ep_regroup(fake, 0, 4, 10, fake, fake, fake, nul) == INVALID
    assert lib.moe_ep_regroup(fake, 2, 33, 10, fake, fake, fake, nul) == INVALID
    assert lib.moe_ep_regroup(fake, 2, 4, -1, fake, fake, fake, nul) == INVALID
    assert lib.moe_ep_regroup(fake, 2, 4, 10, fake, nul, fake, nul) == INVALID
    assert lib.moe_ep_regroup(nul, 2, 4, 0, fake, nul, nul, nul) == INVALID
    assert lib.moe_gather_rows(fake, 4, fake, -1, 1, 16, fake, nul) == INVALID
    assert lib.moe_gather_rows(fake, 4, fake, 8, 0, 16, fake, nul) == INVALID
    assert lib.moe_gather_rows(fake, 4, fake, 8, 1, 0, fake, nul) == INVALID
    assert lib.moe_gather_rows(nul, 4, fake, 8, 1, 16, fake, nul) == INVALID
    assert lib.moe_gather_rows(nul, 0, nul, 0, 1, 16, nul, nul) == OK
    # decoder layer: bf16 tensor-core shapes only, grouping of heads, workspace
    dws = lib.moe_decoder_workspace_size
    assert dws(64, 512, 256, 8, 2, 4, 2) > lib.moe_workspace_size(64, 512, 256, 8, 2, 1)
    assert dws(64, 512, 256, 8, 2, 4, 3) == 0 and dws(64, 512, 256, 8, 9, 4, 2) == 0
    args = [fake] * 6 + [nul] + [fake] * 3
    assert lib.moe_decoder_layer_forward(*args, 64, 512, 256, 8, 2, 4, 3, 0, 1e-5, 1, fake, nul,
                                         fake, 1 << 30, nul) == INVALID
    assert lib.moe_decoder_layer_forward(*args, 64, 512, 256, 8, 2, 4, 2, 0, -1.0, 1, fake, nul,
                                         fake, 1 << 30, nul) == INVALID
    assert lib.moe_decoder_layer_forward(*args, 64, 512, 256, 8, 2, 4, 2, 0, 1e-5, 0, fake, nul,
                                         fake, 1 << 30, nul) == UNSUPPORTED
    assert lib.moe_decoder_layer_forward(*args, 64, 500, 256, 8, 2, 4, 2, 0, 1e-5, 1, fake, nul,
                                         fake, 1 << 30, nul) == UNSUPPORTED
    assert lib.moe_decoder_layer_forward(*args, 64, 512, 256, 8, 2, 4, 2, 0, 1e-5, 1, fake, nul,
                                         fake, 256, nul) == WORKSPACE
    assert lib.moe_decoder_layer_forward(*args, 0, 512, 256, 8, 2, 4, 2, 0, 1e-5, 1, fake, nul,
                                         fake, 0, nul) == OK
    assert lib.moe_check_device_error(nul, 0, nul) == WORKSPACE
    lib.moe_set_wait_limit_ns(0)


def test_python_binding_names_match_the_abi():
    import sparse_mixture_experts_56_b300 as moe
    for name in declared_functions():
        if name in ("moe_status_string",):
            continue
        assert hasattr(moe, name), name
