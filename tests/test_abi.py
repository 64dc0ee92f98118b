"""The C-ABI library builds, loads, and exports every function include/m2rnn.h declares.

These run without a GPU: only calls that return before touching the device are
made (status strings, version, variant table, and argument checks that reject a
call before anything is enqueued).
"""
import ctypes
import os
import re

import pytest

import __graft_entry__
from matrix_state_nonlinear_gb300 import m2rnn as binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "m2rnn.h")


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(m2rnn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("m2rnn_forward_f32", "m2rnn_forward_bf16", "m2rnn_stream_status",
                 "m2rnn_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names, "no declarations parsed"
    for name in names:
        assert hasattr(lib, name), f"{name} declared in m2rnn.h but not exported"
        assert name in binding.SYMBOLS, f"{name} has no binding"


def test_status_strings_and_version(lib):
    assert binding.status_string(0) == "ok"
    assert "invalid" in binding.status_string(1)
    assert "timed out" in binding.status_string(4)
    assert binding.version() >= 100
    assert binding.variant_name(0) == "auto"
    assert binding.variant_name(999) is None


def test_variant_support_table(lib):
    assert binding.variant_supports(1, 1, 8, 1, 128, 128)
    assert binding.variant_supports(2, 1, 8, 1, 64, 64)
    assert not binding.variant_supports(2, 1, 8, 1, 128, 64)   # pipelined: K <= 64
    assert not binding.variant_supports(2, 1, 8, 1, 64, 128)   # pipelined: V <= 64
    assert not binding.variant_supports(0, 1, 8, 1, 64, 64)    # 0 is "auto", not a kernel
    assert binding.variant_supports(3, 1, 8, 1, 128, 128)      # tcgen05: K = V = 128 only
    assert not binding.variant_supports(3, 1, 8, 1, 64, 128)
    assert binding.pick_variant(16, 8192, 32, 128, 128) == 7    # 512 pairs > 2 per SM: balanced
    assert binding.pick_variant(8, 8192, 38, 128, 128) == 3     # 304 pairs: one wave
    assert binding.pick_variant(8, 8192, 39, 128, 128) == 7
    assert binding.variant_supports(7, 1, 8, 1, 128, 128)
    assert not binding.variant_supports(7, 1, 8, 1, 64, 128)
    assert binding.variant_name(7) == "tcgen05_k128_v128_balanced"
    assert binding.variant_supports(4, 1, 8, 1, 64, 128)       # 4-CTA cluster: K = 64, V = 128
    assert not binding.variant_supports(4, 1, 8, 1, 64, 64)
    assert binding.variant_supports(8, 1, 8, 1, 64, 128)       # 8-CTA cluster: K = 64, V = 128
    assert not binding.variant_supports(8, 1, 8, 1, 128, 128)
    assert binding.variant_supports(9, 1, 8, 1, 64, 128)       # two 4-CTA clusters per pair
    assert binding.variant_name(9) == "mma_sync_rows8_cluster4x2_k64_v128"
    assert binding.pick_variant(1, 65536, 15, 64, 128) == 8    # 15 clusters of 8 resident at once
    assert binding.pick_variant(1, 65536, 16, 64, 128) == 9    # the 16th cluster of 8 would wait
    assert binding.pick_variant(8, 8192, 16, 64, 128) == 4     # 128 pairs: four SMs per pair
    assert binding.variant_name(2) is not None


def test_pick_variant_host_logic(lib):
    assert binding.pick_variant(8, 16384, 16, 64, 64) == 5   # eight-row warps + helper warps
    assert binding.pick_variant(4, 2048, 8, 64, 64) == 6     # 32 pairs: two-block clusters
    assert binding.pick_variant(4, 2048, 19, 64, 64) == 6    # 76 pairs fill half of 152 SMs
    assert binding.pick_variant(4, 2048, 20, 64, 64) == 5    # 80 pairs: one block per pair
    assert binding.variant_supports(6, 1, 8, 1, 64, 48)
    assert not binding.variant_supports(6, 1, 8, 1, 32, 64)  # K = 32: one warp per SP already
    assert binding.pick_variant(8, 16384, 16, 32, 32) == 5
    assert binding.pick_variant(8, 16384, 16, 48, 64) == 2   # K = 48: the pipelined kernel
    assert binding.pick_variant(8, 16384, 16, 64, 96) == 1   # V = 96: the row-warp kernel
    assert binding.pick_variant(1, 64, 2, 8, 8) == 0       # V = 8: not a multiple of 16
    assert binding.pick_variant(1, 64, 2, 64, 40) == 0     # V = 40: not a multiple of 16
    assert binding.pick_variant(1, 64, 2, 129, 64) == 0    # K > 128
    assert binding.pick_variant(1, 64, 2, 64, 144) == 0    # V > 128


# Every 1 <= K <= 128 and every V that is a multiple of 16 up to 128 has a bf16 kernel
# (ragged K on the row-warp kernel with zero padding rows).
@pytest.mark.parametrize("K", [1, 8, 17, 24, 40, 64, 100, 127, 128])
@pytest.mark.parametrize("V", [16, 32, 48, 64, 80, 96, 112, 128])
def test_every_contract_shape_has_a_variant(lib, K, V):
    v = binding.pick_variant(2, 100, 3, K, V)
    assert v > 0, (K, V)
    assert binding.variant_supports(v, 2, 100, 3, K, V)
    assert binding.variant_supports(1, 2, 100, 3, K, V)   # the row-warp kernel takes them all


NULL = None


def call_f32(lib, ptrs, dims):
    return lib.m2rnn_forward_f32(*ptrs, *dims, None)


def call_bf16(lib, ptrs, dims, variant=0):
    return lib.m2rnn_forward_bf16_variant(*ptrs, *dims, variant, None)


def fake_ptrs(n=11, base=1 << 20):
    # distinct, 256-byte aligned, never dereferenced (rejected before any launch)
    return [base + 256 * i for i in range(n)]


@pytest.mark.parametrize("which", range(8))
def test_null_required_pointer_is_invalid_arg(lib, which):
    p = fake_ptrs()
    p[which] = None                          # q k v a alpha beta W w_r
    assert call_f32(lib, p, (1, 4, 1, 8, 8)) == binding.ERR_INVALID_ARG
    assert call_bf16(lib, p, (1, 4, 1, 16, 16)) == binding.ERR_INVALID_ARG


@pytest.mark.parametrize("dims", [(0, 4, 1, 8, 8), (1, -1, 1, 8, 8), (1, 4, 0, 8, 8),
                                  (1, 4, 1, 0, 8), (1, 4, 1, 8, 0)])
def test_bad_sizes_are_invalid_arg(lib, dims):
    assert call_f32(lib, fake_ptrs(), dims) == binding.ERR_INVALID_ARG


def test_null_y_with_steps_is_invalid_arg(lib):
    p = fake_ptrs()
    p[9] = None
    assert call_f32(lib, p, (1, 4, 1, 8, 8)) == binding.ERR_INVALID_ARG


@pytest.mark.parametrize("dims", [(1, 4, 1, 129, 8), (1, 4, 1, 8, 129)])
def test_f32_too_large_is_unsupported(lib, dims):
    assert call_f32(lib, fake_ptrs(), dims) == binding.ERR_UNSUPPORTED


@pytest.mark.parametrize("dims", [(1, 4, 1, 129, 16), (1, 4, 1, 16, 40), (1, 4, 1, 16, 8),
                                  (1, 4, 1, 144, 64), (1, 4, 1, 64, 256), (1, 4, 1, 24, 136)])
def test_bf16_unsupported_shapes(lib, dims):
    assert call_bf16(lib, fake_ptrs(), dims) == binding.ERR_UNSUPPORTED


def test_bf16_misaligned_is_invalid_arg(lib):
    p = fake_ptrs()
    p[0] += 8                                 # q not 16-byte aligned
    assert call_bf16(lib, p, (1, 4, 1, 16, 16)) == binding.ERR_INVALID_ARG


def test_unknown_variant_is_invalid_arg(lib):
    assert call_bf16(lib, fake_ptrs(), (1, 4, 1, 16, 16), variant=77) == binding.ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(lib):
    import torch
    from matrix_state_nonlinear_gb300.inputs import WORKLOADS, make_inputs
    inp = make_inputs(WORKLOADS["tiny_f32_b1_t64_n2_k8_v8"], "cpu")
    with pytest.raises(ValueError):
        binding.m2rnn_forward(inp)


# ---------------------------------------------------------------- training entry points
def call_bwd(lib, ptrs, dims, ws_bytes, bf16=False, variant=0):
    # ptrs: 21 pointers (inputs, Hs, dy, dH_T, gradients), dims: (B, T, N, Nqk, K, V)
    ws = (1 << 30) if ws_bytes else None
    if bf16:
        return lib.m2rnn_backward_bf16(*ptrs, *dims, variant, ws, ws_bytes, None)
    return lib.m2rnn_backward_f32(*ptrs, *dims, ws, ws_bytes, None)


def test_workspace_bytes_formula(lib):
    # per pair: K V + V V + V + 2 floats, padded to 4; plus 2 B T N K floats when q, k shared
    def pair(K, V):
        return (K * V + V * V + V + 2 + 3) // 4 * 4
    assert binding.backward_workspace_bytes(2, 5, 3, 3, 8, 8) == 4 * 6 * pair(8, 8)
    assert binding.backward_workspace_bytes(2, 5, 3, 1, 8, 16) == 4 * (6 * pair(8, 16) + 2 * 2 * 5 * 3 * 8)
    assert binding.backward_workspace_bytes(1, 5, 1, 1, 8, 8) == 4 * pair(8, 8)   # N = 1: nothing to sum
    assert binding.backward_workspace_bytes(1, 5, 2, 3, 8, 8) == 0                # bad Nqk
    assert binding.backward_workspace_bytes(1, 5, 1, 1, 129, 8) == 0


def test_backward_argument_checks(lib):
    dims = (1, 4, 2, 2, 8, 8)
    need = binding.backward_workspace_bytes(*dims)
    p = fake_ptrs(21)
    assert call_bwd(lib, p, dims, need - 4) == binding.ERR_INVALID_ARG          # workspace too small
    assert call_bwd(lib, p, (1, 4, 2, 2, 8, 129), 1 << 30) == binding.ERR_UNSUPPORTED
    assert call_bwd(lib, p, (1, 4, 2, 3, 8, 8), need) == binding.ERR_INVALID_ARG   # Nqk not 1 or N
    for which in (0, 4, 6, 9, 10, 12, 16, 18):   # q, alpha, W, Hs, dy, dq, dalpha, dW
        pp = list(p)
        pp[which] = None
        assert call_bwd(lib, pp, dims, need) == binding.ERR_INVALID_ARG, which
    assert call_bwd(lib, p, dims, need, bf16=True, variant=9) == binding.ERR_INVALID_ARG


def test_forward_train_argument_checks(lib):
    p = fake_ptrs(12)
    p[11] = None                                   # Hs missing with T > 0
    assert lib.m2rnn_forward_train_f32(*p, 1, 4, 1, 1, 8, 8, None) == binding.ERR_INVALID_ARG
    p = fake_ptrs(12)
    assert lib.m2rnn_forward_train_bf16(*p, 1, 4, 1, 1, 129, 64, None) == binding.ERR_UNSUPPORTED
    assert lib.m2rnn_forward_train_bf16(*p, 1, 4, 1, 1, 64, 40, None) == binding.ERR_UNSUPPORTED


def test_decode_argument_checks(lib):
    p = fake_ptrs(11)
    pp = list(p)
    pp[9] = None                                   # H_out
    assert lib.m2rnn_decode_step_bf16(*pp, 2, 3, 3, 64, 64, None) == binding.ERR_INVALID_ARG
    assert lib.m2rnn_decode_step_bf16(*p, 2, 3, 3, 129, 64, None) == binding.ERR_UNSUPPORTED
    assert lib.m2rnn_decode_step_bf16(*p, 2, 3, 3, 64, 40, None) == binding.ERR_UNSUPPORTED
    assert lib.m2rnn_decode_step_bf16(*p, 2, 3, 3, 144, 128, None) == binding.ERR_UNSUPPORTED
    assert lib.m2rnn_decode_step_bf16(*p, 2, 3, 2, 64, 64, None) == binding.ERR_INVALID_ARG
    v = lib.m2rnn_decode_step_bf16_variant
    assert v(*p, 2, 3, 3, 64, 64, 3, None) == binding.ERR_INVALID_ARG      # unknown kernel
    assert v(*p, 2, 3, 3, 64, 40, 1, None) == binding.ERR_UNSUPPORTED


def test_block_argument_checks(lib):
    p = fake_ptrs(4)
    assert lib.m2rnn_conv_silu_bf16(*p, 2, 5, 12, None) == binding.ERR_UNSUPPORTED      # C % 8
    assert lib.m2rnn_conv_silu_bf16(None, p[1], None, p[3], 2, 5, 16, None) == binding.ERR_INVALID_ARG
    assert lib.m2rnn_conv_silu_bf16(*p, 2, 0, 16, None) == binding.OK                  # T = 0: nothing
    q = fake_ptrs(4)
    assert lib.m2rnn_gate_rmsnorm_bf16(q[0], q[1], q[2], 1e-6, q[3], 4, 12, None) == binding.ERR_UNSUPPORTED
    assert lib.m2rnn_gate_rmsnorm_bf16(q[0], q[1], q[2], -1.0, q[3], 4, 16, None) == binding.ERR_INVALID_ARG
    assert lib.m2rnn_gate_rmsnorm_bf16(q[0], None, q[2], 1e-6, q[3], 4, 16, None) == binding.ERR_INVALID_ARG


def test_fused_prologue_argument_checks(lib):
    p = fake_ptrs(17)
    dims = (2, 8, 3, 3, 64, 64)   # B, T, N, Nqk, K, V
    taps = p[3:9]
    rest = p[9:]
    assert lib.m2rnn_forward_conv_bf16(*p[:3], *taps, *rest, 2, 8, 3, 3, 128, 128, None) \
        == binding.ERR_UNSUPPORTED                                   # not an eight-row shape
    no_tap = list(taps)
    no_tap[0] = None
    assert lib.m2rnn_forward_conv_bf16(*p[:3], *no_tap, *rest, *dims, None) \
        == binding.ERR_INVALID_ARG                                   # null q taps
    assert lib.m2rnn_forward_conv_bf16(*p[:3], *taps, *rest, 2, 8, 3, 2, 64, 64, None) \
        == binding.ERR_INVALID_ARG                                   # Nqk neither 1 nor N
    bad = list(taps)
    bad[2] = bad[2] + 4
    assert lib.m2rnn_forward_conv_bf16(*p[:3], *bad, *rest, *dims, None) \
        == binding.ERR_INVALID_ARG                                   # taps not 16-byte aligned
