"""ctypes binding of libgdn (include/gdn.h) for PyTorch tensors.

Argument marshalling only: every function checks dtypes, devices, shapes and
contiguity, then passes raw device pointers and the current CUDA stream to the
C entry point of the same name. All compute runs in libgdn's CUDA kernels;
there is no fallback. Importing this module raises if libgdn.so has not been
built (``python -m gated_deltanet_linear_conv1d_gb300.build``).

bf16 tensors are torch.bfloat16; fp32 tensors torch.float32; index tensors
torch.int32; has_init torch.uint8 (or bool).
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA, GDN_ERR_DEVICE_CHECK, GDN_ERR_TIMEOUT = range(6)
GDN_DEVERR_SLOT, GDN_DEVERR_OFFSETS, GDN_DEVERR_TIMEOUT, GDN_DEVERR_ACCEPTED = 1, 2, 4, 8
GDN_COMMIT_COPY, GDN_COMMIT_REPOINT = 0, 1


class GdnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_lib.gdn_status_string(status).decode()} (status {status})")


class GdnDims(ctypes.Structure):
    _fields_ = [("num_k_heads", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("head_k_dim", ctypes.c_int32), ("head_v_dim", ctypes.c_int32),
                ("conv_kernel", ctypes.c_int32), ("num_slots", ctypes.c_int32)]

    @property
    def channels(self) -> int:
        return 2 * self.num_k_heads * self.head_k_dim + self.num_v_heads * self.head_v_dim


def make_dims(geom, num_slots: int) -> GdnDims:
    """gdn_dims from any object with num_k_heads, num_v_heads, head_k_dim, head_v_dim, conv_kernel."""
    return GdnDims(geom.num_k_heads, geom.num_v_heads, geom.head_k_dim, geom.head_v_dim,
                   geom.conv_kernel, int(num_slots))


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libgdn.so is not built ({LIB_PATH}); run "
                          "`python -m gated_deltanet_linear_conv1d_gb300.build` on a machine with nvcc")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    i32, f32, sz = ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    D = ctypes.POINTER(GdnDims)
    sigs = {
        "gdn_conv_update": [D, P, P, P, P, P, P, i32, i32, P, P, P],
        "gdn_decode_step": [D, P, P, P, P, P, P, P, P, P, f32, P, P, i32, P, P],
        "gdn_chunk_prefill": [D, P, P, P, P, P, P, P, P, P, P, P, f32, P, P, i32, i32, P, sz, P, P],
        "gdn_chunk_prefill_noalloc": [D, P, P, P, P, P, P, P, P, P, P, P, f32, P, P, i32, i32, P, P],
        "gdn_chunk_prefill_align": [D, P, P, P, P, P, P, P, P, P, P, P, f32, P, P, i32, i32, P, i32, P, i32, P, sz,
                                    P, P],
        "gdn_spec_verify": [D, P, P, P, P, P, P, P, P, P, P, f32, P, P, i32, i32, P, P],
        "gdn_spec_commit": [D, P, P, P, P, P, i32, i32, i32, P, P],
        "gdn_gated_rmsnorm": [P, P, P, f32, P, i32, i32, i32, P],
        "gdn_out_proj": [P, P, P, P, i32, i32, i32, P, P],
        "gdn_in_proj": [D, P, i32, P, P, P, P, P, P, i32, P, P],
        "gdn_rmsnorm": [P, P, P, f32, P, i32, i32, P],
        "gdn_fp8_quant_act": [P, P, P, i32, i32, P],
        "gdn_fp8_quant_weight": [P, P, P, i32, i32, P],
        "gdn_fp8_linear": [P, P, P, P, P, P, i32, i32, i32, P, sz, P, P],
        "gdn_read_device_error": [P, ctypes.POINTER(i32), i32, P],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    for name in ("gdn_state_bytes", "gdn_conv_hist_bytes"):
        getattr(lib, name).argtypes = [D]
        getattr(lib, name).restype = sz
    lib.gdn_prefill_workspace_bytes.argtypes = [D, i32, i32]
    lib.gdn_prefill_workspace_bytes.restype = sz
    lib.gdn_fp8_linear_workspace_bytes.argtypes = [i32, i32, i32]
    lib.gdn_fp8_linear_workspace_bytes.restype = sz
    lib.gdn_status_string.argtypes = [ctypes.c_int]
    lib.gdn_status_string.restype = ctypes.c_char_p
    return lib


_lib = _load()


def header_symbols() -> list[str]:
    """Names of the functions include/gdn.h declares."""
    hdr = os.path.join(os.path.dirname(_PKG), "include", "gdn.h")
    text = open(hdr).read()
    return sorted(set(re.findall(r"^\s*(?:gdn_status|size_t|const char \*)\s*(gdn_\w+)\(", text, re.M)))


# ---------------------------------------------------------------- marshalling helpers

def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t, name: str, dtype, shape=None, optional: bool = False):
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libgdn has no CPU path)")
    dts = dtype if isinstance(dtype, tuple) else (dtype,)
    if t.dtype not in dts:
        raise TypeError(f"{name} must have dtype {dts}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _scratch(nbytes: int, device, stream) -> torch.Tensor:
    """Device scratch for one call. Freed when the caller drops it; recorded on the call's
    stream, so the caching allocator does not hand it out again before that stream's work
    (the launch that uses it) has finished."""
    t = torch.empty(nbytes, dtype=torch.uint8, device=device)
    if isinstance(stream, torch.cuda.Stream):
        t.record_stream(stream)
    return t


def _check(status: int, what: str):
    if status != GDN_OK:
        raise GdnError(status, what)


def _common(dims: GdnDims, conv_w, conv_hist, state, gamma):
    CH, K, Rs = dims.channels, dims.conv_kernel, dims.num_slots
    _need(conv_w, "conv_w", torch.float32, (CH, K))
    _need(conv_hist, "conv_hist", torch.bfloat16, (Rs, CH, K - 1))
    if state is not None:
        _need(state, "state", torch.float32, (Rs, dims.num_v_heads, dims.head_v_dim, dims.head_k_dim))
    _need(gamma, "gamma", torch.float32, (dims.head_v_dim,), optional=True)


# ---------------------------------------------------------------- entry points

def gdn_conv_update(dims, x, conv_w, conv_hist, query_start_loc, slot_idx, y, has_init=None,
                    dev_err=None, stream=None):
    N = slot_idx.shape[0]
    T = x.shape[0]
    _common(dims, conv_w, conv_hist, None, None)
    _need(x, "x", torch.bfloat16, (T, dims.channels))
    _need(y, "y", torch.bfloat16, (T, dims.channels))
    _need(query_start_loc, "query_start_loc", torch.int32, (N + 1,))
    _need(slot_idx, "slot_idx", torch.int32, (N,))
    _need(has_init, "has_init", (torch.uint8, torch.bool), (N,), optional=True)
    _need(dev_err, "dev_err", torch.int32, (1,), optional=True)
    _check(_lib.gdn_conv_update(ctypes.byref(dims), _ptr(x), _ptr(conv_w), _ptr(conv_hist),
                                _ptr(query_start_loc), _ptr(slot_idx), _ptr(has_init), N, T, _ptr(y),
                                _ptr(dev_err), _stream(stream)), "gdn_conv_update")


def gdn_decode_step(dims, qkv0, conv_w, conv_hist, state, slot_idx, alpha, beta, z, gamma, eps,
                    o=None, ogate=None, dev_err=None, stream=None):
    N = slot_idx.shape[0]
    Hv, dv = dims.num_v_heads, dims.head_v_dim
    _common(dims, conv_w, conv_hist, state, gamma)
    _need(qkv0, "qkv0", torch.bfloat16, (N, dims.channels))
    _need(slot_idx, "slot_idx", torch.int32, (N,))
    _need(alpha, "alpha", torch.float32, (N, Hv))
    _need(beta, "beta", torch.float32, (N, Hv))
    _need(z, "z", torch.bfloat16, (N, Hv, dv), optional=ogate is None)
    _need(o, "o", torch.bfloat16, (N, Hv, dv), optional=True)
    _need(ogate, "ogate", torch.bfloat16, (N, Hv * dv), optional=True)
    _need(dev_err, "dev_err", torch.int32, (1,), optional=True)
    _check(_lib.gdn_decode_step(ctypes.byref(dims), _ptr(qkv0), _ptr(conv_w), _ptr(conv_hist), _ptr(state),
                                _ptr(slot_idx), _ptr(alpha), _ptr(beta), _ptr(z), _ptr(gamma), float(eps),
                                _ptr(o), _ptr(ogate), N, _ptr(dev_err), _stream(stream)), "gdn_decode_step")


def gdn_prefill_workspace_bytes(dims, num_seqs: int, num_tokens: int) -> int:
    return int(_lib.gdn_prefill_workspace_bytes(ctypes.byref(dims), int(num_seqs), int(num_tokens)))


def gdn_chunk_prefill(dims, qkv0, conv_w, conv_hist, state, query_start_loc, slot_idx, alpha, beta, z, gamma,
                      eps, o=None, ogate=None, has_init=None, workspace=None, dev_err=None, stream=None):
    N = slot_idx.shape[0]
    T = qkv0.shape[0]
    Hv, dv = dims.num_v_heads, dims.head_v_dim
    _common(dims, conv_w, conv_hist, state, gamma)
    _need(qkv0, "qkv0", torch.bfloat16, (T, dims.channels))
    _need(query_start_loc, "query_start_loc", torch.int32, (N + 1,))
    _need(slot_idx, "slot_idx", torch.int32, (N,))
    _need(has_init, "has_init", (torch.uint8, torch.bool), (N,), optional=True)
    _need(alpha, "alpha", torch.float32, (T, Hv))
    _need(beta, "beta", torch.float32, (T, Hv))
    _need(z, "z", torch.bfloat16, (T, Hv, dv), optional=ogate is None)
    _need(o, "o", torch.bfloat16, (T, Hv, dv), optional=True)
    _need(ogate, "ogate", torch.bfloat16, (T, Hv * dv), optional=True)
    _need(dev_err, "dev_err", torch.int32, (1,), optional=True)
    need = gdn_prefill_workspace_bytes(dims, N, T)
    if need and workspace is None:
        workspace = _scratch(need, qkv0.device, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.gdn_chunk_prefill(ctypes.byref(dims), _ptr(qkv0), _ptr(conv_w), _ptr(conv_hist), _ptr(state),
                                  _ptr(query_start_loc), _ptr(slot_idx), _ptr(has_init), _ptr(alpha),
                                  _ptr(beta), _ptr(z), _ptr(gamma), float(eps), _ptr(o), _ptr(ogate), N, T,
                                  _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream)),
           "gdn_chunk_prefill")


def gdn_chunk_prefill_align(dims, qkv0, conv_w, conv_hist, state, query_start_loc, slot_idx, alpha, beta, z,
                            gamma, eps, block_tokens, snap_slot=None, prefix_len=None, o=None, ogate=None,
                            has_init=None, workspace=None, dev_err=None, stream=None):
    N = slot_idx.shape[0]
    T = qkv0.shape[0]
    Hv, dv = dims.num_v_heads, dims.head_v_dim
    _common(dims, conv_w, conv_hist, state, gamma)
    _need(qkv0, "qkv0", torch.bfloat16, (T, dims.channels))
    _need(query_start_loc, "query_start_loc", torch.int32, (N + 1,))
    _need(slot_idx, "slot_idx", torch.int32, (N,))
    _need(has_init, "has_init", (torch.uint8, torch.bool), (N,), optional=True)
    _need(alpha, "alpha", torch.float32, (T, Hv))
    _need(beta, "beta", torch.float32, (T, Hv))
    _need(z, "z", torch.bfloat16, (T, Hv, dv), optional=ogate is None)
    _need(o, "o", torch.bfloat16, (T, Hv, dv), optional=True)
    _need(ogate, "ogate", torch.bfloat16, (T, Hv * dv), optional=True)
    _need(prefix_len, "prefix_len", torch.int32, (N,), optional=True)
    max_snaps = 0 if snap_slot is None else snap_slot.shape[1]
    _need(snap_slot, "snap_slot", torch.int32, (N, max_snaps), optional=True)
    _need(dev_err, "dev_err", torch.int32, (1,), optional=True)
    need = gdn_prefill_workspace_bytes(dims, N, T)
    if need and workspace is None:
        workspace = _scratch(need, qkv0.device, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.gdn_chunk_prefill_align(ctypes.byref(dims), _ptr(qkv0), _ptr(conv_w), _ptr(conv_hist), _ptr(state),
                                        _ptr(query_start_loc), _ptr(slot_idx), _ptr(has_init), _ptr(alpha),
                                        _ptr(beta), _ptr(z), _ptr(gamma), float(eps), _ptr(o), _ptr(ogate), N, T,
                                        _ptr(prefix_len), int(block_tokens), _ptr(snap_slot), max_snaps,
                                        _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream)),
           "gdn_chunk_prefill_align")


def gdn_chunk_prefill_noalloc(dims, qkv0, conv_w, conv_hist, state, query_start_loc, slot_idx, alpha, beta, z,
                              gamma, eps, o=None, ogate=None, has_init=None, dev_err=None, stream=None):
    N = slot_idx.shape[0]
    T = qkv0.shape[0]
    Hv, dv = dims.num_v_heads, dims.head_v_dim
    _common(dims, conv_w, conv_hist, state, gamma)
    _need(qkv0, "qkv0", torch.bfloat16, (T, dims.channels))
    _need(query_start_loc, "query_start_loc", torch.int32, (N + 1,))
    _need(slot_idx, "slot_idx", torch.int32, (N,))
    _need(has_init, "has_init", (torch.uint8, torch.bool), (N,), optional=True)
    _need(alpha, "alpha", torch.float32, (T, Hv))
    _need(beta, "beta", torch.float32, (T, Hv))
    _need(z, "z", torch.bfloat16, (T, Hv, dv), optional=ogate is None)
    _need(o, "o", torch.bfloat16, (T, Hv, dv), optional=True)
    _need(ogate, "ogate", torch.bfloat16, (T, Hv * dv), optional=True)
    _need(dev_err, "dev_err", torch.int32, (1,), optional=True)
    _check(_lib.gdn_chunk_prefill_noalloc(ctypes.byref(dims), _ptr(qkv0), _ptr(conv_w), _ptr(conv_hist),
                                          _ptr(state), _ptr(query_start_loc), _ptr(slot_idx), _ptr(has_init),
                                          _ptr(alpha), _ptr(beta), _ptr(z), _ptr(gamma), float(eps), _ptr(o),
                                          _ptr(ogate), N, T, _ptr(dev_err), _stream(stream)),
           "gdn_chunk_prefill_noalloc")


def gdn_out_proj(ogate, w, out, residual=None, dev_err=None, stream=None):
    """out[T][N] = ogate[T][K] w[N][K]^T (+ residual[T][N]); residual may be out itself."""
    T, K = ogate.shape
    N = w.shape[0]
    _need(ogate, "ogate", torch.bfloat16, (T, K))
    _need(w, "w", torch.bfloat16, (N, K))
    _need(out, "out", torch.bfloat16, (T, N))
    _need(residual, "residual", torch.bfloat16, (T, N), optional=True)
    _need(dev_err, "dev_err", torch.int32, (1,), optional=True)
    _check(_lib.gdn_out_proj(_ptr(ogate), _ptr(w), _ptr(residual), _ptr(out), T, K, N, _ptr(dev_err),
                             _stream(stream)), "gdn_out_proj")


def gdn_rmsnorm(x, gamma, eps, out, residual=None, stream=None):
    """out = RMSNorm(x) * gamma, or with residual: residual <- bf16(x + residual), out = RMSNorm(residual) * gamma."""
    T, Dh = x.shape
    _need(x, "x", torch.bfloat16, (T, Dh))
    _need(gamma, "gamma", torch.float32, (Dh,))
    _need(out, "out", torch.bfloat16, (T, Dh))
    _need(residual, "residual", torch.bfloat16, (T, Dh), optional=True)
    _check(_lib.gdn_rmsnorm(_ptr(x), _ptr(residual), _ptr(gamma), float(eps), _ptr(out), T, Dh, _stream(stream)),
           "gdn_rmsnorm")


def gdn_fp8_quant_act(x, x8, x_scale, stream=None):
    """x [T, K] bf16 -> x8 [T, K] e4m3 (uint8 storage) and x_scale [T, K/128] fp32."""
    T, K = x.shape
    _need(x, "x", torch.bfloat16, (T, K))
    _need(x8, "x8", torch.uint8, (T, K))
    _need(x_scale, "x_scale", torch.float32, (T, K // 128))
    _check(_lib.gdn_fp8_quant_act(_ptr(x), _ptr(x8), _ptr(x_scale), T, K, _stream(stream)), "gdn_fp8_quant_act")


def gdn_fp8_quant_weight(w, w8, w_scale, stream=None):
    """w [N, K] bf16 -> w8 [N, K] e4m3 (uint8 storage) and w_scale [ceil(N/128), K/128] fp32."""
    N, K = w.shape
    _need(w, "w", torch.bfloat16, (N, K))
    _need(w8, "w8", torch.uint8, (N, K))
    _need(w_scale, "w_scale", torch.float32, ((N + 127) // 128, K // 128))
    _check(_lib.gdn_fp8_quant_weight(_ptr(w), _ptr(w8), _ptr(w_scale), N, K, _stream(stream)),
           "gdn_fp8_quant_weight")


def gdn_fp8_linear_workspace_bytes(num_tokens: int, k: int, n: int) -> int:
    return int(_lib.gdn_fp8_linear_workspace_bytes(int(num_tokens), int(k), int(n)))


def gdn_fp8_linear(x8, x_scale, w8, w_scale, out, residual=None, workspace=None, dev_err=None, stream=None):
    """out [T, N] = dequant(x8) dequant(w8)^T (+ residual), block-scaled FP8 operands, bf16 out.
    workspace: zero-filled before its first use (each call resets its tickets)."""
    T, K = x8.shape
    N = w8.shape[0]
    _need(x8, "x8", torch.uint8, (T, K))
    _need(w8, "w8", torch.uint8, (N, K))
    _need(x_scale, "x_scale", torch.float32, (T, K // 128))
    _need(w_scale, "w_scale", torch.float32, ((N + 127) // 128, K // 128))
    _need(out, "out", torch.bfloat16, (T, N))
    _need(residual, "residual", torch.bfloat16, (T, N), optional=True)
    _need(dev_err, "dev_err", torch.int32, (1,), optional=True)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.gdn_fp8_linear(_ptr(x8), _ptr(x_scale), _ptr(w8), _ptr(w_scale), _ptr(residual), _ptr(out), T, K, N,
                               _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream)), "gdn_fp8_linear")


def gdn_in_proj(dims, hidden, w_qkv, w_z, qkv0, z, w_ab=None, ab=None, dev_err=None, stream=None):
    """QKV0 = hidden W_qkv^T, Z = hidden W_z^T and, when given, [a | b] = hidden W_ab^T (fp32), in one
    launch."""
    T, Dh = hidden.shape
    _need(hidden, "hidden", torch.bfloat16, (T, Dh))
    _need(w_qkv, "w_qkv", torch.bfloat16, (dims.channels, Dh))
    _need(w_z, "w_z", torch.bfloat16, (dims.num_v_heads * dims.head_v_dim, Dh))
    _need(qkv0, "qkv0", torch.bfloat16, (T, dims.channels))
    _need(z, "z", torch.bfloat16, (T, dims.num_v_heads * dims.head_v_dim))
    _need(w_ab, "w_ab", torch.bfloat16, (2 * dims.num_v_heads, Dh), optional=True)
    _need(ab, "ab", torch.float32, (T, 2 * dims.num_v_heads), optional=True)
    _need(dev_err, "dev_err", torch.int32, (1,), optional=True)
    _check(_lib.gdn_in_proj(ctypes.byref(dims), _ptr(hidden), Dh, _ptr(w_qkv), _ptr(w_z), _ptr(w_ab), _ptr(qkv0),
                            _ptr(z), _ptr(ab), T, _ptr(dev_err), _stream(stream)), "gdn_in_proj")


def gdn_spec_verify(dims, qkv0, conv_w, conv_hist, state, slot_idx, spec_slot_idx, alpha, beta, z, gamma, eps,
                    o=None, ogate=None, dev_err=None, stream=None):
    N, P = spec_slot_idx.shape
    Hv, dv = dims.num_v_heads, dims.head_v_dim
    _common(dims, conv_w, conv_hist, state, gamma)
    _need(qkv0, "qkv0", torch.bfloat16, (N * P, dims.channels))
    _need(slot_idx, "slot_idx", torch.int32, (N,))
    _need(spec_slot_idx, "spec_slot_idx", torch.int32, (N, P))
    _need(alpha, "alpha", torch.float32, (N * P, Hv))
    _need(beta, "beta", torch.float32, (N * P, Hv))
    _need(z, "z", torch.bfloat16, (N * P, Hv, dv), optional=ogate is None)
    _need(o, "o", torch.bfloat16, (N * P, Hv, dv), optional=True)
    _need(ogate, "ogate", torch.bfloat16, (N * P, Hv * dv), optional=True)
    _need(dev_err, "dev_err", torch.int32, (1,), optional=True)
    _check(_lib.gdn_spec_verify(ctypes.byref(dims), _ptr(qkv0), _ptr(conv_w), _ptr(conv_hist), _ptr(state),
                                _ptr(slot_idx), _ptr(spec_slot_idx), _ptr(alpha), _ptr(beta), _ptr(z),
                                _ptr(gamma), float(eps), _ptr(o), _ptr(ogate), N, P, _ptr(dev_err),
                                _stream(stream)), "gdn_spec_verify")


def gdn_spec_commit(dims, accepted, spec_slot_idx, slot_idx, state=None, conv_hist=None,
                    mode: int = GDN_COMMIT_COPY, dev_err=None, stream=None):
    N, P = spec_slot_idx.shape
    _need(accepted, "accepted", torch.int32, (N,))
    _need(spec_slot_idx, "spec_slot_idx", torch.int32, (N, P))
    _need(slot_idx, "slot_idx", torch.int32, (N,))
    if mode == GDN_COMMIT_COPY:
        _need(state, "state", torch.float32,
              (dims.num_slots, dims.num_v_heads, dims.head_v_dim, dims.head_k_dim))
        _need(conv_hist, "conv_hist", torch.bfloat16, (dims.num_slots, dims.channels, dims.conv_kernel - 1))
    _need(dev_err, "dev_err", torch.int32, (1,), optional=True)
    _check(_lib.gdn_spec_commit(ctypes.byref(dims), _ptr(accepted), _ptr(spec_slot_idx), _ptr(slot_idx),
                                _ptr(state), _ptr(conv_hist), N, P, int(mode), _ptr(dev_err), _stream(stream)),
           "gdn_spec_commit")


def gdn_gated_rmsnorm(o, z, gamma, eps, out, stream=None):
    T, H, D = o.shape
    _need(o, "o", torch.bfloat16, (T, H, D))
    _need(z, "z", torch.bfloat16, (T, H, D))
    _need(gamma, "gamma", torch.float32, (D,))
    _need(out, "out", torch.bfloat16, (T, H * D))
    _check(_lib.gdn_gated_rmsnorm(_ptr(o), _ptr(z), _ptr(gamma), float(eps), _ptr(out), T, H, D,
                                  _stream(stream)), "gdn_gated_rmsnorm")


def gdn_state_bytes(dims) -> int:
    return int(_lib.gdn_state_bytes(ctypes.byref(dims)))


def gdn_conv_hist_bytes(dims) -> int:
    return int(_lib.gdn_conv_hist_bytes(ctypes.byref(dims)))


def gdn_read_device_error(dev_err: torch.Tensor, reset: bool = True, stream=None) -> int:
    """Synchronises the stream and returns the device error word (GDN_DEVERR_* bits)."""
    _need(dev_err, "dev_err", torch.int32, (1,))
    host = ctypes.c_int32(0)
    st = _lib.gdn_read_device_error(_ptr(dev_err), ctypes.byref(host), int(bool(reset)), _stream(stream))
    if st not in (GDN_OK, GDN_ERR_DEVICE_CHECK, GDN_ERR_TIMEOUT):
        raise GdnError(st, "gdn_read_device_error")
    return int(host.value)
