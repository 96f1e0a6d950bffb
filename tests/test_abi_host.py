"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, and its host-side argument checks answer before any device work."""
import ctypes
import os
import re

import pytest

from situ_glu_activation_gb300 import _native

BAD, ALIAS, WS = 1, 3, 8
from situ_glu_activation_gb300.build import INCLUDE

HEADER = os.path.join(INCLUDE, "situ.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(situ_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for must in ["situ_glu_act", "situ_ffn_forward", "situ_moe_grouped_forward",
                 "situ_moe_build_index", "situ_device_status"]:
        assert must in names


def test_every_declared_symbol_is_exported(situ_lib):
    names = declared_functions()
    assert set(names) == set(_native.SIGNATURES), "binding and header disagree"
    for n in names:
        assert hasattr(situ_lib, n), f"libsitu.so does not export {n}"


def test_version_and_status_strings(situ_lib):
    assert situ_lib.situ_abi_version() == 2
    for code, name in _native.STATUS_NAMES.items():
        assert situ_lib.situ_status_string(code).decode() == name
    assert situ_lib.situ_status_string(99).decode() == "SITU_ERR_UNKNOWN"


def test_workspace_sizes(situ_lib):
    # bf16: h, then one int32 h-ready count per 128-row tile (rounded to 256 B)
    assert situ_lib.situ_ffn_workspace_size(16384, 2048, 3072, 0) == 16384 * 3072 * 2 + 512
    assert situ_lib.situ_ffn_workspace_size(300, 8, 8, 0) == 4864 + 256
    assert situ_lib.situ_ffn_workspace_size(3, 8, 5, 1) == 256  # fp32 h, rounded to 256 B
    assert situ_lib.situ_ffn_workspace_size(0, 8, 8, 0) == 0
    R, E, M, I = 1000, 7, 64, 96
    expect = 3 * 256 + ((R * M * 2 + 255) // 256) * 256 + ((R * I * 2 + 255) // 256) * 256
    assert situ_lib.situ_moe_workspace_size(R, E, M, I, 0) == expect
    assert situ_lib.situ_moe_workspace_size(R, E, M, I, 1) == 0  # grouped path is bf16 only
    assert situ_lib.situ_moe_index_workspace_size(1024, 10) == 256
    assert situ_lib.situ_moe_index_workspace_size(1025, 10) == 256


@pytest.mark.parametrize("beta,lbeta", [(0.0, 25.0), (4.0, -1.0), (float("nan"), 25.0),
                                        (4.0, -float("inf")), (2.0e6, 25.0), (4.0, 1e10)])
def test_caps_must_be_positive(situ_lib, beta, lbeta):
    # Rejected before any pointer is touched (the problem page: both caps positive;
    # finite caps up to 2^20, +inf = uncapped).
    assert situ_lib.situ_glu_act(16, 32, 4, 8, beta, lbeta, 0, None) == BAD
    assert situ_lib.situ_ffn_forward(16, 16, 16, 16, 16, 0, 4, 8, 8, beta, lbeta, 0, None) == BAD


@pytest.mark.parametrize("beta,lbeta", [(4.0, float("inf")), (float("inf"), 25.0),
                                        (float("inf"), float("inf")), (1048576.0, 1.0)])
def test_infinite_cap_means_uncapped(situ_lib, beta, lbeta):
    # Accepted caps: the call proceeds to the pointer checks (here: overlap).
    assert situ_lib.situ_glu_act(4096, 4096 + 64, 4, 8, beta, lbeta, 0, None) == ALIAS


def test_python_caps_follow_the_activation_module():
    from situ_glu_activation_gb300.api import caps
    inf = float("inf")
    assert caps(4.0, 25.0) == (4.0, 25.0)
    assert caps(None, 25.0) == (1.0, 25.0) and caps(0, 25.0) == (1.0, 25.0)  # beta or 1.0
    assert caps(4.0, None) == (4.0, inf)                                       # no up cap
    assert caps(inf, inf) == (inf, inf)


def test_argument_checks(situ_lib):
    f = situ_lib.situ_glu_act
    assert f(None, None, 0, 8, 4.0, 25.0, 0, None) == 0          # zero rows: no-op
    assert f(None, None, 4, 8, 4.0, 25.0, 0, None) == BAD        # null pointers
    assert f(4096, 8192, 4, 0, 4.0, 25.0, 0, None) == BAD        # I < 1
    assert f(4096, 8192, 4, 8, 4.0, 25.0, 7, None) == BAD        # bad dtype
    # out overlapping gate_up: [4096, 4096 + 4*16*2) vs out at 4096 + 64
    assert f(4096, 4096 + 64, 4, 8, 4.0, 25.0, 0, None) == ALIAS
    g = situ_lib.situ_ffn_forward
    # workspace too small / misaligned
    assert g(1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20, 10, 4, 8, 8, 4.0, 25.0, 0, None) == WS
    assert g(1 << 20, 2 << 20, 3 << 20, 4 << 20, (5 << 20) + 16, 1 << 20, 4, 8, 8, 4.0, 25.0, 0,
             None) == WS
    # y overlapping x
    assert g(1 << 20, 2 << 20, 3 << 20, (1 << 20) + 32, 5 << 20, 1 << 20, 4, 8, 8, 4.0, 25.0, 0,
             None) == ALIAS
    m = situ_lib.situ_moe_grouped_forward
    assert m(0, 0, 0, 0, 0, 0, 0, 0, 4, 2, 3, 8, 8, 4.0, 25.0, 1, None) == 6  # fp32: unsupported
    assert m(0, 0, 0, 0, 0, 0, 0, 0, 0, 2, 3, 8, 8, 4.0, 25.0, 0, None) == 0  # no tokens
    b = situ_lib.situ_moe_build_index
    assert b(0, 0, 0, 0, 0, 10, 0, None) == BAD   # E = 0
    assert b(1 << 20, 2 << 20, 3 << 20, 0, 0, 10, 4, None) == WS


def test_training_and_mx_argument_checks(situ_lib):
    UNSUP = 6
    # grouped training: fp32 unsupported, no routes -> no-op / zeroing path needs weights
    f = situ_lib.situ_moe_grouped_forward_train
    assert f(0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 4, 2, 3, 8, 8, 4.0, 25.0, 1, None) == UNSUP
    assert f(0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 2, 3, 8, 8, 4.0, 25.0, 0, None) == 0
    b = situ_lib.situ_moe_grouped_backward
    assert b(0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 4, 2, 3, 8, 8, 0.0, 25.0, 0, None) == BAD
    assert b(0, 0, 0, 0, 0, 0, 0, 0, 0, None, None, 0, 0, 0, 2, 3, 8, 8, 4.0, 25.0, 0, None) == BAD
    # MX quantizers: K must be a multiple of 128; bad kind / format rejected
    q = situ_lib.situ_mx_quantize_act
    assert q(1 << 20, 2 << 20, 3 << 20, 4, 136, None) == UNSUP
    assert q(None, None, None, 0, 128, None) == 0
    assert q(None, 2 << 20, 3 << 20, 4, 128, None) == BAD
    w = situ_lib.situ_mx_quantize_weights
    assert w(1 << 20, 2 << 20, 3 << 20, 1, 256, 384, 2, 0, None) == BAD      # bad kind
    assert w(1 << 20, 2 << 20, 3 << 20, 1, 256, 384, 0, 7, None) == BAD      # bad format
    assert w(1 << 20, 2 << 20, 3 << 20, 1, 200, 384, 0, 0, None) == UNSUP   # M % 128
    assert situ_lib.situ_mx_act_scales_size(300, 256) == 3 * 2 * 512
    assert situ_lib.situ_mx_weight_scales_size(1, 2048, 3072, 0) == 32 * 16 * 1024
    assert situ_lib.situ_mx_weight_scales_size(2, 2048, 3072, 1) == 2 * 11 * 24 * 1024
    assert situ_lib.situ_mx_weight_scales_size(1, 200, 3072, 0) == 0
    ffn = situ_lib.situ_ffn_forward_mxfp8
    args = [1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20, 0, 6 << 20, 7 << 20, 16, 4, 256, 384,
            4.0, 25.0, None]
    assert ffn(*args) == WS                                  # workspace too small
    bad_fmt = list(args)
    bad_fmt[5] = 3
    assert ffn(*bad_fmt) == BAD
    assert situ_lib.situ_ffn_mxfp8_workspace_size(4, 256, 384) > 0
    assert situ_lib.situ_ffn_mxfp8_workspace_size(4, 250, 384) == 0
    # fused combine: needs weights and an output
    c = situ_lib.situ_moe_grouped_forward_combined
    assert c(1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20, None, 6 << 20, 7 << 20, 16, 4, 2, 3,
             256, 384, 4.0, 25.0, 0, None) == BAD
    assert situ_lib.situ_moe_combined_workspace_size(4, 2, 3, 256, 384, 0) == \
        situ_lib.situ_moe_workspace_size(8, 3, 256, 384, 0) + 4 * 256 * 4


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not found"):
        _native.lib(str(tmp_path / "libsitu.so"))


def test_ffn_single_launch_switch(situ_lib):
    """The process-wide switch for the one-launch dense forward: on by default,
    returns the previous setting; no dense call has run on this thread yet."""
    assert situ_lib.situ_ffn_last_path() == 0
    assert situ_lib.situ_ffn_set_single_launch(0) == 1
    assert situ_lib.situ_ffn_set_single_launch(7) == 0
    assert situ_lib.situ_ffn_set_single_launch(1) == 1


def test_kgrouped_two_cta_switch(situ_lib):
    """The process-wide switch for the two-CTA weight gradients of the grouped backward:
    on by default, returns the previous setting."""
    assert situ_lib.situ_moe_set_kgrouped_two_cta(0) == 1
    assert situ_lib.situ_moe_set_kgrouped_two_cta(3) == 0
    assert situ_lib.situ_moe_set_kgrouped_two_cta(1) == 1


def test_moe_backward_workspace_holds_the_expert_maps(situ_lib):
    """The grouped backward's workspace: four per-expert prefix arrays, two 128-byte
    tensor maps per expert for each of the two weight-gradient GEMMs, the [R, M] rows
    buffer and d(g, u) [R, 2I], each rounded up to 256 bytes."""
    up = lambda n: (n + 255) // 256 * 256
    for R, E, M, I in [(1000, 7, 64, 96), (131072, 64, 2048, 3072), (5, 898, 8, 8)]:
        expect = 4 * up((E + 1) * 4) + 2 * up(E * 256) + up(R * M * 2) + up(R * 2 * I * 2)
        assert situ_lib.situ_moe_backward_workspace_size(R, E, M, I, 0) == expect
    assert situ_lib.situ_moe_backward_workspace_size(10, 0, 8, 8, 0) == 0


def test_group_maps_selftest_argument_checks(situ_lib):
    """situ_selftest_group_maps refuses offsets that are not non-decreasing within
    [0, rows], bad group counts and widths, before any device work."""
    def call(offsets, rows=64, cols=64, groups=None):
        off = (ctypes.c_int32 * len(offsets))(*offsets)
        g = len(offsets) - 1 if groups is None else groups
        flags = (ctypes.c_int32 * max(2 * g, 2))()
        return situ_lib.situ_selftest_group_maps(off, g, rows, cols, flags, None)
    assert call([0, 5, 3]) == BAD            # decreasing
    assert call([-1, 5]) == BAD              # negative start
    assert call([0, 65], rows=64) == BAD     # past the rows
    assert call([0, 5], cols=60) == BAD      # width not a multiple of 8
    assert call([0, 5], cols=0) == BAD
    assert call([0, 5], rows=0) == BAD
    assert call([0, 5], groups=0) == BAD
    assert situ_lib.situ_selftest_group_maps(None, 1, 64, 64, None, None) == BAD


def test_size_limits(situ_lib):
    """The largest sizes: row counts and weight-row counts index the tensor maps and the
    kernels' tile arithmetic as int32, so the calls refuse 2^31 and more before touching
    any pointer (no GPU needed), and take 2^31 - 1 past that check."""
    UNSUP = 6
    g = situ_lib.situ_ffn_forward
    p = [1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20, 64]
    assert g(*p, 1 << 31, 8, 8, 4.0, 25.0, 0, None) == UNSUP          # R
    assert g(*p, 8, 8, 1 << 30, 4.0, 25.0, 0, None) == UNSUP          # 2I
    assert g(*p, 8, 1 << 31, 8, 4.0, 25.0, 0, None) == UNSUP          # M
    assert g(*p, (1 << 31) - 1, 8, 8, 4.0, 25.0, 0, None) == WS       # past the limit check
    m = situ_lib.situ_moe_grouped_forward
    q = [1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20, 6 << 20, 7 << 20, 64]
    assert m(*q, 1 << 28, 8, 4, 8, 8, 4.0, 25.0, 0, None) == UNSUP     # T * k_eff = 2^31
    assert m(*q, 4, 2, 65536, 8, 16384, 4.0, 25.0, 0, None) == UNSUP  # E * 2I = 2^31
    assert m(*q, 4, 2, 65536, 32768, 8, 4.0, 25.0, 0, None) == UNSUP  # E * M = 2^31
    assert m(*q, 4, 2, 65537, 8, 8, 4.0, 25.0, 0, None) == BAD        # more than 65536 experts


def test_wait_limit_setting(situ_lib):
    """The GEMMs' wait bound is a process-wide setting: 10 s by default, 0 restores it,
    and each call returns the previous bound."""
    default = 10 * 1000 * 1000 * 1000
    first = situ_lib.situ_set_wait_limit_ns(5000)
    try:
        assert first == default
        assert situ_lib.situ_set_wait_limit_ns(0) == 5000
        assert situ_lib.situ_set_wait_limit_ns(0) == default
    finally:
        situ_lib.situ_set_wait_limit_ns(first)
