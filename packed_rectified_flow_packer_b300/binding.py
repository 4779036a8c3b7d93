"""Thin ctypes binding of libmageflow.so.  Argument marshalling only: every step of the path
runs in the library's kernels.  Function names are the C entry points' names.

Device memory is whatever the caller passes: torch tensors (their data_ptr() is used), raw
integer addresses, or None for NULL.  Streams default to torch's current CUDA stream.
A non-OK status raises MageflowError.  Importing this module fails loudly when the library has
not been built (python packed_rectified_flow_packer_b300/build.py).
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

__all__ = ["MageflowError", "mf_sample", "mf_plan_info", "mf_dims", "mf_temb_weights", "mf_stream_weights", "mf_block_weights", "temb_struct", "block_struct", "Plan", "samples_struct", "mf_pack", "mf_pack_status", "mf_plan_upload", "mf_block_workspace_bytes", "mf_block_workspace_layout", "mf_block_forward", "mf_block_forward_ex", "BLOCK_LN_ROW_GROUPS", "BLOCK_LN_STATS_FUSED", "BLOCK_COND_GIVEN", "mf_block_train_workspace_bytes", "mf_block_forward_train", "mf_block_backward_workspace_bytes", "mf_block_backward", "grads_struct", "mf_stream_grads", "mf_block_grads", "GRAD_FIELDS", "mf_block_fp8_workspace_bytes", "mf_block_forward_fp8", "block_struct_fp8", "mf_stream_weights_fp8", "mf_block_weights_fp8", "mf_embed", "mf_final_workspace_bytes", "mf_final", "mf_final_ex", "mf_interpolate", "mf_cfg_combine", "mf_euler_step", "mf_flow_loss_workspace_bytes", "mf_flow_loss", "mf_flow_loss_noalloc", "NOALLOC_MAX_IMG_ROWS", "mf_nft_loss", "mf_attention", "mf_attention_lse", "mf_attention_backward_workspace_bytes", "mf_attention_backward", "mf_gemm", "mf_quantize_fp8_rows", "mf_gemm_fp8", "mf_check", "mf_selftest_timeout", "mf_status_str", "mf_version", "mf_trace_entry", "mf_trace_enable", "mf_trace_kinds", "mf_trace_read", "mf_launch_count", "KERNEL_KINDS", "LIB_PATH", "STATUS", "STATUS_CODE", "EXPORTED", "PLAN_ARRAYS", "STREAM_FIELDS", "lib"]

# MAGEFLOW_LIB=checked selects the bounds-checked build (same ABI; see mf_check)
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "libmageflow_checked.so" if os.environ.get("MAGEFLOW_LIB") == "checked"
                        else "libmageflow.so")

STATUS = {0: "MF_OK", 1: "MF_ERR_INVALID_ARG", 2: "MF_ERR_SAMPLE_TOO_LONG", 3: "MF_ERR_BUDGET",
          4: "MF_ERR_ALIGNMENT", 5: "MF_ERR_CUDA", 6: "MF_ERR_DEVICE_TIMEOUT",
          7: "MF_ERR_UNSUPPORTED", 8: "MF_ERR_NOT_UPLOADED", 9: "MF_ERR_WORKSPACE",
          10: "MF_ERR_DEVICE_BOUNDS"}
STATUS_CODE = {v: k for k, v in STATUS.items()}


class MageflowError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        self.name = STATUS.get(status, f"status {status}")
        super().__init__(f"{call} failed: {self.name}")


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python packed_rectified_flow_packer_b300/build.py`")
lib = C.CDLL(LIB_PATH)


# ------------------------------------------------------------------ structs (mageflow.h)
class mf_sample(C.Structure):
    _fields_ = [("txt_len", C.c_int32), ("frames", C.c_int32), ("lat_h", C.c_int32),
                ("lat_w", C.c_int32), ("t", C.c_float), ("cfg_role", C.c_int32),
                ("cfg_pair", C.c_int32)]


class mf_plan_info(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("n_seq", "n_tok", "n_txt", "n_img", "n_items", "budget",
                                          "uploaded", "reserved")]


class mf_dims(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("hidden", "heads", "channels", "mlp_ratio", "freq_dim")]


class mf_temb_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("w_t1", "b_t1", "w_t2", "b_t2")]


STREAM_FIELDS = ("w_mod", "b_mod", "w_qkv", "b_qkv", "w_o", "b_o", "w_1", "b_1", "w_2", "b_2")
STREAM_OPTIONAL = ("w_qnorm", "w_knorm")   # QK-RMSNorm scales; NULL when absent


class mf_stream_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in STREAM_FIELDS + STREAM_OPTIONAL]


class mf_block_weights(C.Structure):
    _fields_ = [("temb", mf_temb_weights), ("txt", mf_stream_weights), ("img", mf_stream_weights)]


STREAM_FP8_FIELDS = ("q_qkv", "s_qkv", "q_o", "s_o", "q_1", "s_1", "q_2", "s_2")


class mf_stream_weights_fp8(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in STREAM_FP8_FIELDS]


class mf_block_weights_fp8(C.Structure):
    _fields_ = [("txt", mf_stream_weights_fp8), ("img", mf_stream_weights_fp8)]


GRAD_FIELDS = STREAM_FIELDS   # mf_stream_grads: one f32 array per weight, same names


class mf_stream_grads(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in GRAD_FIELDS]


class mf_block_grads(C.Structure):
    _fields_ = [("txt", mf_stream_grads), ("img", mf_stream_grads)]


class mf_trace_entry(C.Structure):
    _fields_ = [("launches", C.c_int64), ("ms", C.c_double), ("flops", C.c_double),
                ("bytes", C.c_double)]


KERNEL_KINDS = ("cond", "ln", "gemm_qkv", "attn", "gemm_oproj", "gemm_up", "gemm_down", "gemm_embed",
                "gemm_final", "gemm_plain", "latent", "loss", "fp8", "attn_bwd", "block_bwd",
                "gemm_dgrad", "gemm_wgrad")

_P = C.c_void_p
_S = C.c_int   # mf_status
_sigs = {
    "mf_status_str": (C.c_char_p, [C.c_int]),
    "mf_version": (C.c_int32, []),
    "mf_pack": (_S, [C.POINTER(mf_sample), C.c_int32, C.c_int32, C.POINTER(_P)]),
    "mf_plan_upload": (_S, [_P, _P]),
    "mf_plan_free": (None, [_P]),
    "mf_plan_get_info": (_S, [_P, C.POINTER(mf_plan_info)]),
    "mf_plan_array": (_S, [_P, C.c_int32, C.POINTER(C.POINTER(C.c_int32)), C.POINTER(C.c_int64)]),
    "mf_block_workspace_bytes": (C.c_size_t, [_P, C.POINTER(mf_dims)]),
    "mf_block_workspace_layout": (_S, [_P, C.POINTER(mf_dims), C.POINTER(C.c_size_t), C.c_int32]),
    "mf_block_forward": (_S, [_P, C.POINTER(mf_dims), C.POINTER(mf_block_weights), _P, _P, _P, _P,
                              C.c_size_t, _P]),
    "mf_block_forward_ex": (_S, [_P, C.POINTER(mf_dims), C.POINTER(mf_block_weights), _P, _P, _P, _P,
                                 C.c_size_t, C.c_int32, _P]),
    "mf_block_train_workspace_bytes": (C.c_size_t, [_P, C.POINTER(mf_dims)]),
    "mf_block_forward_train": (_S, [_P, C.POINTER(mf_dims), C.POINTER(mf_block_weights), _P, _P, _P, _P,
                                    C.c_size_t, _P]),
    "mf_block_backward_workspace_bytes": (C.c_size_t, [_P, C.POINTER(mf_dims)]),
    "mf_block_backward": (_S, [_P, C.POINTER(mf_dims), C.POINTER(mf_block_weights), _P, C.c_size_t, _P, _P,
                               C.POINTER(mf_block_grads), _P, _P, C.c_size_t, _P]),
    "mf_embed": (_S, [_P, C.POINTER(mf_dims), _P, _P, _P, _P, _P]),
    "mf_final_workspace_bytes": (C.c_size_t, [_P, C.POINTER(mf_dims)]),
    "mf_final": (_S, [_P, C.POINTER(mf_dims), C.POINTER(mf_temb_weights), _P, _P, _P, _P, _P, _P,
                      _P, _P, C.c_size_t, _P]),
    "mf_final_ex": (_S, [_P, C.POINTER(mf_dims), C.POINTER(mf_temb_weights), _P, _P, _P, _P, _P, _P,
                         _P, _P, C.c_size_t, _P, _P]),
    "mf_interpolate": (_S, [_P, C.c_int32, _P, _P, _P, _P, _P, _P]),
    "mf_cfg_combine": (_S, [_P, C.c_int32, C.c_float, _P, _P, _P]),
    "mf_euler_step": (_S, [_P, C.c_int32, C.c_float, _P, _P, _P, _P]),
    "mf_flow_loss_workspace_bytes": (C.c_size_t, [_P]),
    "mf_flow_loss": (_S, [_P, C.c_int32, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "mf_flow_loss_noalloc": (_S, [_P, C.c_int32, _P, _P, _P, _P, _P, _P, _P]),
    "mf_nft_loss": (_S, [_P, C.c_int32, _P, _P, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "mf_attention": (_S, [_P, C.c_int32, C.c_int32, _P, _P, _P, _P, _P]),
    "mf_attention_lse": (_S, [_P, C.c_int32, C.c_int32, _P, _P, _P, _P, _P, _P]),
    "mf_attention_backward_workspace_bytes": (C.c_size_t, [_P, C.c_int32, C.c_int32]),
    "mf_attention_backward": (_S, [_P, C.c_int32, C.c_int32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                   C.c_size_t, _P]),
    "mf_gemm": (_S, [C.c_int32, C.c_int32, C.c_int32, _P, _P, _P, _P, C.c_int32, _P]),
    "mf_quantize_fp8_rows": (_S, [C.c_int32, C.c_int32, _P, _P, _P, _P]),
    "mf_gemm_fp8": (_S, [C.c_int32, C.c_int32, C.c_int32, _P, _P, _P, _P, _P, _P, _P]),
    "mf_block_fp8_workspace_bytes": (C.c_size_t, [_P, _P]),
    "mf_block_forward_fp8": (_S, [_P, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "mf_check": (_S, [_P]),
    "mf_selftest_timeout": (_S, [C.c_int32, _P]),
    "mf_trace_enable": (_S, [C.c_int32]),
    "mf_trace_kinds": (_S, [C.c_uint32]),
    "mf_trace_read": (_S, [C.POINTER(mf_trace_entry), C.c_int32]),
    "mf_launch_count": (C.c_int64, []),
}
for _name, (_res, _args) in _sigs.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_sigs)


# ------------------------------------------------------------------ marshalling helpers
def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _ok(status: int, call: str):
    if status != 0:
        raise MageflowError(status, call)


def _dims(d) -> mf_dims:
    if isinstance(d, mf_dims):
        return d
    return mf_dims(d.hidden, d.heads, d.channels, d.mlp_ratio, d.freq_dim)


def temb_struct(w) -> mf_temb_weights:
    return mf_temb_weights(*[_ptr(w[k]) for k in ("w_t1", "b_t1", "w_t2", "b_t2")])


def block_struct(temb, txt, img) -> mf_block_weights:
    """temb, txt, img: dicts name -> device tensor (bf16)."""
    def stream(d):
        return mf_stream_weights(*[_ptr(d[k]) for k in STREAM_FIELDS],
                                 *[_ptr(d.get(k)) for k in STREAM_OPTIONAL])
    return mf_block_weights(temb_struct(temb), stream(txt), stream(img))


# ------------------------------------------------------------------ plan
PLAN_ARRAYS = ("order", "cu_seqlens", "cu_txt", "cu_img", "pos", "txt_seq", "txt_joint", "img_seq",
               "img_joint", "img_pair", "img_target", "seq_role", "items")


class Plan:
    """Owns an mf_plan*."""

    def __init__(self, handle):
        self.handle = handle

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h:
            lib.mf_plan_free(h)

    @property
    def _as_parameter_(self):
        return self.handle

    def info(self) -> mf_plan_info:
        i = mf_plan_info()
        _ok(lib.mf_plan_get_info(self.handle, C.byref(i)), "mf_plan_get_info")
        return i

    def array(self, name: str) -> np.ndarray:
        which = PLAN_ARRAYS.index(name)
        data = C.POINTER(C.c_int32)()
        n = C.c_int64()
        _ok(lib.mf_plan_array(self.handle, which, C.byref(data), C.byref(n)), "mf_plan_array")
        if n.value == 0:
            return np.zeros(0, np.int32)
        return np.ctypeslib.as_array(data, shape=(n.value,)).copy()

    @property
    def n_seq(self): return self.info().n_seq

    @property
    def n_tok(self): return self.info().n_tok

    @property
    def n_txt(self): return self.info().n_txt

    @property
    def n_img(self): return self.info().n_img


def samples_struct(samples):
    arr = (mf_sample * max(1, len(samples)))()
    for i, s in enumerate(samples):
        g = (lambda k: s[k]) if isinstance(s, dict) else (lambda k: getattr(s, k))
        arr[i] = mf_sample(int(g("txt_len")), int(g("frames")), int(g("lat_h")), int(g("lat_w")),
                           float(g("t")), int(g("cfg_role")), int(g("cfg_pair")))
    return arr


def mf_pack(samples, budget: int) -> Plan:
    arr = samples_struct(samples)
    h = C.c_void_p()
    _ok(lib.mf_pack(arr, len(samples), int(budget), C.byref(h)), "mf_pack")
    return Plan(h.value)


def mf_pack_status(samples, budget: int) -> int:
    """Status code of mf_pack without raising (for error-path tests)."""
    arr = samples_struct(samples)
    h = C.c_void_p()
    st = lib.mf_pack(arr, len(samples), int(budget), C.byref(h))
    if st == 0:
        lib.mf_plan_free(h.value)
    return st


def mf_plan_upload(plan: Plan, stream=None):
    _ok(lib.mf_plan_upload(plan.handle, _stream(stream)), "mf_plan_upload")


# ------------------------------------------------------------------ block, embed, final
def mf_block_workspace_bytes(plan: Plan, dims) -> int:
    return lib.mf_block_workspace_bytes(plan.handle, C.byref(_dims(dims)))


def mf_block_workspace_layout(plan: Plan, dims):
    off = (C.c_size_t * 9)()
    _ok(lib.mf_block_workspace_layout(plan.handle, C.byref(_dims(dims)), off, 9),
        "mf_block_workspace_layout")
    return list(off)


def mf_block_forward(plan: Plan, dims, weights: mf_block_weights, t, x_txt, x_img, ws, ws_bytes=None,
                     stream=None):
    nbytes = ws_bytes if ws_bytes is not None else (ws.numel() * ws.element_size() if ws is not None else 0)
    _ok(lib.mf_block_forward(plan.handle, C.byref(_dims(dims)), C.byref(weights), _ptr(t), _ptr(x_txt),
                             _ptr(x_img), _ptr(ws), nbytes, _stream(stream)), "mf_block_forward")


# LN + modulate variants of mf_block_forward_ex (the header's MF_BLOCK_LN_*)
BLOCK_LN_ROW_GROUPS = 1
BLOCK_LN_STATS_FUSED = 2
BLOCK_COND_GIVEN = 4


def mf_block_forward_ex(plan: Plan, dims, weights: mf_block_weights, t, x_txt, x_img, ws, flags, ws_bytes=None,
                        stream=None):
    nbytes = ws_bytes if ws_bytes is not None else (ws.numel() * ws.element_size() if ws is not None else 0)
    _ok(lib.mf_block_forward_ex(plan.handle, C.byref(_dims(dims)), C.byref(weights), _ptr(t), _ptr(x_txt),
                                _ptr(x_img), _ptr(ws), nbytes, int(flags), _stream(stream)), "mf_block_forward_ex")


def mf_block_train_workspace_bytes(plan: Plan, dims) -> int:
    return lib.mf_block_train_workspace_bytes(plan.handle, C.byref(_dims(dims)))


def mf_block_forward_train(plan: Plan, dims, weights: mf_block_weights, t, x_txt, x_img, ws, ws_bytes=None,
                           stream=None):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _ok(lib.mf_block_forward_train(plan.handle, C.byref(_dims(dims)), C.byref(weights), _ptr(t), _ptr(x_txt),
                                   _ptr(x_img), _ptr(ws), nbytes, _stream(stream)), "mf_block_forward_train")


def grads_struct(txt, img) -> mf_block_grads:
    """txt, img: dicts weight name -> f32 device tensor of that weight's shape."""
    return mf_block_grads(mf_stream_grads(*[_ptr(txt[k]) for k in GRAD_FIELDS]),
                          mf_stream_grads(*[_ptr(img[k]) for k in GRAD_FIELDS]))


def mf_block_backward_workspace_bytes(plan: Plan, dims) -> int:
    return lib.mf_block_backward_workspace_bytes(plan.handle, C.byref(_dims(dims)))


def mf_block_backward(plan: Plan, dims, weights: mf_block_weights, train_ws, dx_txt, dx_img,
                      grads: mf_block_grads, dc, ws, ws_bytes=None, train_ws_bytes=None, stream=None):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    tbytes = train_ws_bytes if train_ws_bytes is not None else train_ws.numel() * train_ws.element_size()
    _ok(lib.mf_block_backward(plan.handle, C.byref(_dims(dims)), C.byref(weights), _ptr(train_ws), tbytes,
                              _ptr(dx_txt), _ptr(dx_img), C.byref(grads), _ptr(dc), _ptr(ws), nbytes,
                              _stream(stream)), "mf_block_backward")


def block_struct_fp8(txt8, img8) -> mf_block_weights_fp8:
    """txt8, img8: dicts q_* (uint8 codes) / s_* (f32 scales) -> device tensors."""
    return mf_block_weights_fp8(mf_stream_weights_fp8(*[_ptr(txt8[k]) for k in STREAM_FP8_FIELDS]),
                                mf_stream_weights_fp8(*[_ptr(img8[k]) for k in STREAM_FP8_FIELDS]))


def mf_block_fp8_workspace_bytes(plan: Plan, dims) -> int:
    return lib.mf_block_fp8_workspace_bytes(plan.handle, C.byref(_dims(dims)))


def mf_block_forward_fp8(plan: Plan, dims, weights: mf_block_weights, weights8: mf_block_weights_fp8, t,
                         x_txt, x_img, ws, ws_bytes=None, stream=None):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _ok(lib.mf_block_forward_fp8(plan.handle, C.byref(_dims(dims)), C.byref(weights), C.byref(weights8), _ptr(t),
                                 _ptr(x_txt), _ptr(x_img), _ptr(ws), nbytes, _stream(stream)),
        "mf_block_forward_fp8")


def mf_embed(plan: Plan, dims, w_in, b_in, zt, x_img, stream=None):
    _ok(lib.mf_embed(plan.handle, C.byref(_dims(dims)), _ptr(w_in), _ptr(b_in), _ptr(zt), _ptr(x_img),
                     _stream(stream)), "mf_embed")


def mf_final_workspace_bytes(plan: Plan, dims) -> int:
    return lib.mf_final_workspace_bytes(plan.handle, C.byref(_dims(dims)))


def mf_final(plan: Plan, dims, temb: mf_temb_weights, w_fmod, b_fmod, w_out, b_out, t, x_img, v, ws,
             ws_bytes=None, stream=None):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _ok(lib.mf_final(plan.handle, C.byref(_dims(dims)), C.byref(temb), _ptr(w_fmod), _ptr(b_fmod),
                     _ptr(w_out), _ptr(b_out), _ptr(t), _ptr(x_img), _ptr(v), _ptr(ws), nbytes,
                     _stream(stream)), "mf_final")


def mf_final_ex(plan: Plan, dims, temb: mf_temb_weights, w_fmod, b_fmod, w_out, b_out, t, x_img, v, ws, c,
                ws_bytes=None, stream=None):
    """mf_final with the timestep condition c (device f32 [S][H], or an address) given."""
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _ok(lib.mf_final_ex(plan.handle, C.byref(_dims(dims)), C.byref(temb), _ptr(w_fmod), _ptr(b_fmod),
                        _ptr(w_out), _ptr(b_out), _ptr(t), _ptr(x_img), _ptr(v), _ptr(ws), nbytes, _ptr(c),
                        _stream(stream)), "mf_final_ex")


# ------------------------------------------------------------------ rectified-flow epilogues
def mf_interpolate(plan: Plan, channels: int, t, z, eps, zt=None, zt_bf16=None, stream=None):
    _ok(lib.mf_interpolate(plan.handle, channels, _ptr(t), _ptr(z), _ptr(eps), _ptr(zt), _ptr(zt_bf16),
                           _stream(stream)), "mf_interpolate")


def mf_cfg_combine(plan: Plan, channels: int, w: float, v, v_out, stream=None):
    _ok(lib.mf_cfg_combine(plan.handle, channels, float(w), _ptr(v), _ptr(v_out), _stream(stream)),
        "mf_cfg_combine")


def mf_euler_step(plan: Plan, channels: int, dt: float, v, z, z_bf16=None, stream=None):
    _ok(lib.mf_euler_step(plan.handle, channels, float(dt), _ptr(v), _ptr(z), _ptr(z_bf16),
                          _stream(stream)), "mf_euler_step")


def mf_flow_loss_workspace_bytes(plan: Plan) -> int:
    return lib.mf_flow_loss_workspace_bytes(plan.handle)


def mf_flow_loss(plan: Plan, channels: int, z, eps, v, loss_sum, count, mean, ws, ws_bytes=None,
                 stream=None):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _ok(lib.mf_flow_loss(plan.handle, channels, _ptr(z), _ptr(eps), _ptr(v), _ptr(loss_sum),
                         _ptr(count), _ptr(mean), _ptr(ws), nbytes, _stream(stream)), "mf_flow_loss")


def mf_nft_loss(plan: Plan, channels: int, z, eps, v_pos, v_neg, reward, loss_sum, count, mean, ws,
                ws_bytes=None, stream=None):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _ok(lib.mf_nft_loss(plan.handle, channels, _ptr(z), _ptr(eps), _ptr(v_pos), _ptr(v_neg), _ptr(reward),
                        _ptr(loss_sum), _ptr(count), _ptr(mean), _ptr(ws), nbytes, _stream(stream)),
        "mf_nft_loss")


NOALLOC_MAX_IMG_ROWS = 65536   # MF_NOALLOC_MAX_IMG_ROWS


def mf_flow_loss_noalloc(plan: Plan, channels: int, z, eps, v, loss_sum, count, mean, stream=None):
    """mf_flow_loss with the library's own fixed scratch (no workspace, no allocation)."""
    _ok(lib.mf_flow_loss_noalloc(plan.handle, channels, _ptr(z), _ptr(eps), _ptr(v), _ptr(loss_sum),
                                 _ptr(count), _ptr(mean), _stream(stream)), "mf_flow_loss_noalloc")


# ------------------------------------------------------------------ building blocks, status
def mf_attention(plan: Plan, heads: int, head_dim: int, q, k, v, o, stream=None):
    _ok(lib.mf_attention(plan.handle, heads, head_dim, _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                         _stream(stream)), "mf_attention")


def mf_attention_lse(plan: Plan, heads: int, head_dim: int, q, k, v, o, lse, stream=None):
    _ok(lib.mf_attention_lse(plan.handle, heads, head_dim, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                             _stream(stream)), "mf_attention_lse")


def mf_attention_backward_workspace_bytes(plan: Plan, heads: int, head_dim: int) -> int:
    return lib.mf_attention_backward_workspace_bytes(plan.handle, heads, head_dim)


def mf_attention_backward(plan: Plan, heads: int, head_dim: int, q, k, v, o, lse, do, dq, dk, dv, ws,
                          ws_bytes=None, stream=None):
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _ok(lib.mf_attention_backward(plan.handle, heads, head_dim, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                  _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), nbytes, _stream(stream)),
        "mf_attention_backward")


def mf_quantize_fp8_rows(x, q, scale, stream=None):
    """x bf16 [M][K] -> q uint8 E4M3 codes [M][K], scale f32 [M]."""
    M, K = x.shape
    _ok(lib.mf_quantize_fp8_rows(M, K, _ptr(x), _ptr(q), _ptr(scale), _stream(stream)), "mf_quantize_fp8_rows")


def mf_gemm_fp8(a, a_scale, b, b_scale, c, bias=None, stream=None):
    """c bf16 [M][N] = (a b^T) * a_scale[:, None] * b_scale[None, :] + bias, a / b uint8 E4M3 codes."""
    M, K = a.shape
    N = b.shape[0]
    _ok(lib.mf_gemm_fp8(M, N, K, _ptr(a), _ptr(a_scale), _ptr(b), _ptr(b_scale), _ptr(bias), _ptr(c),
                        _stream(stream)), "mf_gemm_fp8")


def mf_gemm(a, b, c, bias=None, out_f32=False, stream=None):
    M, K = a.shape
    N = b.shape[0]
    _ok(lib.mf_gemm(M, N, K, _ptr(a), _ptr(b), _ptr(bias), _ptr(c), 1 if out_f32 else 0,
                    _stream(stream)), "mf_gemm")


def mf_check(stream=None):
    _ok(lib.mf_check(_stream(stream)), "mf_check")


def mf_selftest_timeout(limit_us: int, stream=None) -> int:
    return lib.mf_selftest_timeout(int(limit_us), _stream(stream))


def mf_status_str(s: int) -> str:
    return lib.mf_status_str(s).decode()


def mf_version() -> int:
    return lib.mf_version()


# ------------------------------------------------------------------ tracing
def mf_trace_enable(on: bool = True):
    _ok(lib.mf_trace_enable(1 if on else 0), "mf_trace_enable")


def mf_trace_kinds(kinds=None):
    """Restrict tracing to the given kind names (KERNEL_KINDS); None traces every kind."""
    mask = 0xFFFFFFFF if kinds is None else sum(1 << KERNEL_KINDS.index(k) for k in kinds)
    _ok(lib.mf_trace_kinds(mask), "mf_trace_kinds")


def mf_trace_read() -> dict:
    """{kind: {"launches", "ms", "flops", "bytes"}} since tracing was enabled (then cleared)."""
    arr = (mf_trace_entry * len(KERNEL_KINDS))()
    _ok(lib.mf_trace_read(arr, len(KERNEL_KINDS)), "mf_trace_read")
    return {k: {"launches": e.launches, "ms": e.ms, "flops": e.flops, "bytes": e.bytes}
            for k, e in zip(KERNEL_KINDS, arr)}


def mf_launch_count() -> int:
    return lib.mf_launch_count()
