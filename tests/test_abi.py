"""libgdn builds, loads and exports every entry point include/gdn.h declares (CPU only).

Only host-side paths run here: size queries, status strings and argument
validation that returns before any CUDA call. No kernel is launched.
"""
import ctypes

import pytest

from gated_deltanet_linear_conv1d_gb300 import build as gdn_build
from gated_deltanet_linear_conv1d_gb300 import synth


@pytest.fixture(scope="module")
def b():
    gdn_build.build()
    from gated_deltanet_linear_conv1d_gb300 import binding
    return binding


def test_every_declared_symbol_is_exported(b):
    names = b.header_symbols()
    assert {"gdn_conv_update", "gdn_decode_step", "gdn_chunk_prefill", "gdn_spec_verify",
            "gdn_gated_rmsnorm", "gdn_spec_commit"} <= set(names)
    lib = ctypes.CDLL(b.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), name


def test_size_queries_match_the_page(b):
    d = b.make_dims(synth.FULL_HEADS, 512)
    assert b.gdn_state_bytes(d) == 48 * 128 * 128 * 4 == 3 * 2**20  # "3 MiB per sequence per layer"
    assert b.gdn_conv_hist_bytes(d) == 10240 * 3 * 2
    r = b.make_dims(synth.RANK_HEADS, 8)
    assert b.gdn_state_bytes(r) == 12 * 128 * 128 * 4
    assert b.gdn_conv_hist_bytes(r) == 2560 * 3 * 2
    assert b.gdn_state_bytes(b.GdnDims(0, 0, 0, 0, 0, 0)) == 0


def test_prefill_workspace_holds_the_schedule_and_the_tickets(b):
    d = b.make_dims(synth.FULL_HEADS, 512)
    # schedule (N int32, 256-byte rounded) + tickets (N x 16 key heads int32, 256-byte rounded)
    assert b.gdn_prefill_workspace_bytes(d, 64, 71068) == 256 + 4096
    assert b.gdn_prefill_workspace_bytes(d, 65, 100) == 512 + 4352
    assert b.gdn_prefill_workspace_bytes(d, 1000, 1000) == 4096 + 64000
    assert b.gdn_prefill_workspace_bytes(d, 0, 0) == 0
    assert b.gdn_prefill_workspace_bytes(b.GdnDims(0, 0, 0, 0, 0, 0), 64, 64) == 0


def test_status_strings(b):
    for s in range(6):
        assert b._lib.gdn_status_string(s).decode().startswith("GDN_")


def _decode_call(b, dims, eps=1e-6, num_seqs=1, ptr=1):
    # Non-NULL dummy pointers: validation must reject before touching them.
    p = ctypes.c_void_p(ptr) if ptr else None
    return b._lib.gdn_decode_step(ctypes.byref(dims), p, p, p, p, p, p, p, p, p, eps, p, p, num_seqs, None, None)


@pytest.mark.parametrize("geom,expect", [
    (synth.Dims(16, 48, 64, 128, 4), 2),   # dk != 128
    (synth.Dims(16, 48, 128, 128, 3), 2),  # 3 taps
    (synth.Dims(16, 40, 128, 128, 4), 2),  # Hv not a multiple of Hk
    (synth.Dims(2, 48, 128, 128, 4), 2),   # group 24 > 8
    (synth.Dims(0, 48, 128, 128, 4), 1),
])
def test_geometry_is_rejected_before_launch(b, geom, expect):
    assert _decode_call(b, b.make_dims(geom, 4)) == expect


def test_arguments_are_rejected_before_launch(b):
    d = b.make_dims(synth.FULL_HEADS, 4)
    assert _decode_call(b, d, ptr=0) == b.GDN_ERR_INVALID_ARG  # NULL pointers
    assert _decode_call(b, d, eps=float("nan")) == b.GDN_ERR_INVALID_ARG
    assert _decode_call(b, d, eps=-1.0) == b.GDN_ERR_INVALID_ARG
    assert _decode_call(b, d, num_seqs=-1) == b.GDN_ERR_INVALID_ARG
    assert _decode_call(b, d, ptr=2) == b.GDN_ERR_INVALID_ARG  # state not 16-byte aligned
    assert _decode_call(b, d, num_seqs=0) == b.GDN_OK  # empty batch: nothing to launch
    p = ctypes.c_void_p(16)
    lib = b._lib
    assert lib.gdn_spec_verify(ctypes.byref(d), *([p] * 10), 1e-6, p, p, 4, 9, None, None) == 1  # 9 positions
    assert lib.gdn_spec_commit(ctypes.byref(d), p, p, p, p, p, 4, 4, 7, None, None) == 1  # bad mode
    assert lib.gdn_gated_rmsnorm(p, p, p, 1e-6, p, 4, 4, 6, None) == 2  # D not a multiple of 4
    assert lib.gdn_gated_rmsnorm(p, p, p, 1e-6, p, 0, 4, 128, None) == 0  # no rows
    assert lib.gdn_chunk_prefill(ctypes.byref(d), *([p] * 11), 1e-6, p, p, 0, 5, None, 0, None, None) == 1
    assert lib.gdn_conv_update(ctypes.byref(d), p, p, p, p, p, None, 0, 0, p, None, None) == 0
    host = ctypes.c_int32(0)
    assert lib.gdn_read_device_error(None, ctypes.byref(host), 0, None) == 1


def test_in_proj_rejects_bad_arguments_on_the_host(b):
    """Shape and pointer checks of gdn_in_proj happen before any launch (no GPU needed)."""
    lib = b._lib
    D = b.make_dims(synth.FULL_HEADS, 1)
    P = ctypes.c_void_p
    fake = P(256)  # never dereferenced: every call below is rejected or returns before a launch
    # hidden size not a multiple of 8
    assert lib.gdn_in_proj(ctypes.byref(D), fake, 5121, fake, fake, None, fake, fake, None, 4,
                           None, None) == b.GDN_ERR_UNSUPPORTED
    # w_ab without ab
    assert lib.gdn_in_proj(ctypes.byref(D), fake, 5120, fake, fake, fake, fake, fake, None, 4,
                           None, None) == b.GDN_ERR_INVALID_ARG
    # no tokens: nothing to do
    assert lib.gdn_in_proj(ctypes.byref(D), None, 5120, None, None, None, None, None, None, 0,
                           None, None) == b.GDN_OK


def test_rmsnorm_rejects_bad_arguments_on_the_host(b):
    lib = b._lib
    p, odd = ctypes.c_void_p(256), ctypes.c_void_p(264)  # never dereferenced
    assert lib.gdn_rmsnorm(p, None, p, 1e-6, p, 4, 5124, None) == b.GDN_ERR_UNSUPPORTED  # not a multiple of 8
    assert lib.gdn_rmsnorm(p, None, p, 1e-6, p, 4, 8200, None) == b.GDN_ERR_UNSUPPORTED  # above 8192
    assert lib.gdn_rmsnorm(p, None, p, float("nan"), p, 4, 5120, None) == b.GDN_ERR_INVALID_ARG
    assert lib.gdn_rmsnorm(p, odd, p, 1e-6, p, 4, 5120, None) == b.GDN_ERR_INVALID_ARG  # residual not 16 B aligned
    assert lib.gdn_rmsnorm(None, None, p, 1e-6, p, 4, 5120, None) == b.GDN_ERR_INVALID_ARG
    assert lib.gdn_rmsnorm(None, None, None, 1e-6, None, 0, 5120, None) == b.GDN_OK


def test_fp8_entry_points_reject_bad_arguments_on_the_host(b):
    lib = b._lib
    p, odd = ctypes.c_void_p(256), ctypes.c_void_p(264)  # never dereferenced
    assert lib.gdn_fp8_quant_act(p, p, p, 4, 200, None) == b.GDN_ERR_UNSUPPORTED   # K not a multiple of 128
    assert lib.gdn_fp8_quant_act(p, odd, p, 4, 256, None) == b.GDN_ERR_INVALID_ARG  # misaligned codes
    assert lib.gdn_fp8_quant_act(None, None, None, 0, 256, None) == b.GDN_OK       # no tokens
    assert lib.gdn_fp8_quant_weight(p, p, p, 16, 100, None) == b.GDN_ERR_UNSUPPORTED
    assert lib.gdn_fp8_quant_weight(p, p, None, 16, 128, None) == b.GDN_ERR_INVALID_ARG
    assert lib.gdn_fp8_linear(p, p, p, p, None, p, 4, 128, 24, None, 0, None, None) == b.GDN_ERR_UNSUPPORTED  # N % 16
    assert lib.gdn_fp8_linear(p, p, p, p, None, p, 4, 130, 32, None, 0, None, None) == b.GDN_ERR_UNSUPPORTED  # K % 128
    assert lib.gdn_fp8_linear(p, p, p, p, odd, p, 4, 128, 32, None, 0, None, None) == b.GDN_ERR_INVALID_ARG
    assert lib.gdn_fp8_linear(None, None, None, None, None, None, 0, 128, 32, None, 0, None, None) == b.GDN_OK
    assert lib.gdn_fp8_linear_workspace_bytes(256, 100, 5120) == 0  # K not a multiple of 128


def test_noalloc_prefill_limits_are_checked_on_the_host(b):
    """The allocation-free prefill refuses, before any CUDA call, request counts beyond its fixed
    schedule (65,535) and (request, key head) pairs beyond its fixed ticket array (2^20)."""
    lib = b._lib
    p = ctypes.c_void_p(256)  # never dereferenced
    for geom, n in ((synth.RANK_HEADS, 65536), (synth.Dims(32, 32, 128, 128, 4), 40000),
                    (synth.Dims(16, 16, 128, 128, 4), 65536 + 1)):
        D = b.make_dims(geom, 4)
        assert lib.gdn_chunk_prefill_noalloc(ctypes.byref(D), p, p, p, p, p, p, None, p, p, p, p, 1e-6, None, p,
                                             n, 100, None, None) == b.GDN_ERR_INVALID_ARG, (geom, n)


def test_spec_verify_rejects_misaligned_inputs_on_the_host(b):
    """gdn_spec_verify streams qkv0, the conv history and z with 16-byte copies: a buffer off
    that alignment is refused before any launch."""
    lib = b._lib
    d = b.make_dims(synth.RANK_HEADS, 8)
    a, odd = ctypes.c_void_p(256), ctypes.c_void_p(258)  # never dereferenced
    args = [a] * 10  # qkv0, conv_w, conv_hist, state, slot_idx, spec_slot_idx, alpha, beta, z, gamma
    for i in (0, 2, 8):  # qkv0, conv_hist, z
        bad = list(args)
        bad[i] = odd
        assert lib.gdn_spec_verify(ctypes.byref(d), *bad, 1e-6, None, a, 2, 4, None, None) == b.GDN_ERR_INVALID_ARG
