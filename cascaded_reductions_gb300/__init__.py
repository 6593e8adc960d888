"""cascaded_reductions_gb300 -- Python binding of librf.so.

Argument marshalling only: every step of every cascade runs in the library's
CUDA kernels.  Each ``rf_*`` function here has the name and meaning of the C
entry point declared in ``include/rf.h``; it takes torch CUDA tensors, checks
their dtype, shape and contiguity, and passes raw device pointers and the
current stream.  A status other than RF_OK raises :class:`RFError`.

The convenience wrappers (``attn_decode``, ``softmax_topk``,
``absmax_quant_fp8_gemm``, ``attn_prefill``) only allocate the output tensors
with torch and call the entry points.

There is no fallback: importing this package fails if librf.so has not been
built (``cascaded_reductions_gb300._build.build()``).  The environment
variable ``RF_LIBRARY`` names another build of the same library to load
instead, e.g. the bounds-checked debug variant that
``cascaded_reductions_gb300._build.build_checked()`` makes.
"""

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("RF_LIBRARY") or os.path.join(_HERE, "librf.so")

(RF_OK, RF_ERR_INVALID_ARG, RF_ERR_UNSUPPORTED, RF_ERR_MISALIGNED, RF_ERR_CUDA, RF_ERR_TIMEOUT,
 RF_ERR_BOUNDS) = range(7)
RF_F32, RF_BF16 = 0, 1
RF_FUSE_NONE, RF_FUSE_THREAD, RF_FUSE_WARP, RF_FUSE_BLOCK = range(4)

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float

_SIGNATURES = {
    "rf_status_string": (ctypes.c_char_p, [_I]),
    "rf_version": (_I, []),
    "rf_attn_decode_split": (_I, [_P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P, _P, _P]),
    "rf_state_merge": (_I, [_P, _P, _P, _I, _I, _I, _P, _I, _P, _P]),
    "rf_attn_prefill": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, _P]),
    "rf_softmax_topk": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "rf_absmax_quant_fp8_gemm": (_I, [_P, _I, _I, _P, _P, _I, _P, _P, _P, _P]),
    "rf_absmax_quant_e4m3": (_I, [_P, _I, _I, _P, _P, _P]),
    "rf_fp8_gemm_scaled": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "rf_device_error": (_I, [ctypes.POINTER(_I), _P]),
    "rf_attn_decode_noalloc": (_I, [_P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _I, _P, _P]),
    "rf_row_softmax": (_I, [_P, _I, _I, _P, _I, _P, _P]),
    "rf_row_variance": (_I, [_P, _I, _I, _P, _P, _I, _P]),
    "rf_moment_of_inertia": (_I, [_P, _P, _I, _I, _P, _P, _I, _P]),
    "rf_layer_norm": (_I, [_P, _P, _P, _I, _I, _F, _P, _I, _P, _P]),
    "rf_attn_decode_split_twopass": (_I, [_P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P, _P, _P]),
    "rf_incremental_quant_fp8_gemm": (_I, [_P, _I, _I, _P, _P, _I, _P, _P, _P]),
    "rf_mla_decode_split": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P]),
    "rf_selftest_wait_timeout": (_I, [_P, _P]),
    "rf_rms_norm": (_I, [_P, _P, _I, _I, _F, _P, _I, _P, _P]),
    "rf_attn_decode_fused": (_I, [_P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P, _P, _P, _P, _I, _P, _P]),
    "rf_bounds_checked": (_I, []),
    "rf_selftest_bounds": (_I, [_P]),
    "rf_stream_read": (_I, [_P, ctypes.c_size_t, _P, _P]),
}


def load_library(path=LIB_PATH):
    """Open librf.so and declare every entry point's C signature."""
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is not built; run cascaded_reductions_gb300._build.build() "
            "(nvcc for sm_103a).  There is no CPU fallback.")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = load_library()


class RFError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {_lib.rf_status_string(status).decode()}")


def _check(status, where):
    if status != RF_OK:
        raise RFError(status, where)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need(t, dtype, name, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _dtype_code(dt):
    if dt == torch.float32:
        return RF_F32
    if dt == torch.bfloat16:
        return RF_BF16
    raise ValueError(f"unsupported dtype {dt}")


def version():
    return _lib.rf_version()


# ------------------------------------------------------------ entry points --

def rf_attn_decode_split(q, k, v, S, scale, seg_m, seg_l, seg_acc, stream=None):
    """q [R, D], k/v [R, L, D] (fp32 D=64 or bf16 D=128) -> seg_m/seg_l [R, S], seg_acc [R, S, D]."""
    R, L, D = k.shape
    _need(q, k.dtype, "q", (R, D))
    _need(k, k.dtype, "k")
    _need(v, k.dtype, "v", (R, L, D))
    _need(seg_m, torch.float32, "seg_m", (R, S))
    _need(seg_l, torch.float32, "seg_l", (R, S))
    _need(seg_acc, torch.float32, "seg_acc", (R, S, D))
    _check(_lib.rf_attn_decode_split(_ptr(q), _ptr(k), _ptr(v), R, L, D, S, float(scale),
                                     _dtype_code(k.dtype), _ptr(seg_m), _ptr(seg_l), _ptr(seg_acc),
                                     _stream(stream)), "rf_attn_decode_split")


def rf_attn_decode_fused(q, k, v, S, scale, seg_m, seg_l, seg_acc, counters, out, lse=None,
                         stream=None):
    """Split-KV decode with the merge done by each row's last CTA, in one launch.
    counters: int32 [R] CUDA tensor, zero before the first call (calls leave it zero)."""
    R, L, D = k.shape
    dt = _dtype_code(q.dtype)
    _need(q, q.dtype, "q", (R, D))
    _need(k, q.dtype, "k", (R, L, D))
    _need(v, q.dtype, "v", (R, L, D))
    _need(seg_m, torch.float32, "seg_m", (R, S))
    _need(seg_l, torch.float32, "seg_l", (R, S))
    _need(seg_acc, torch.float32, "seg_acc", (R, S, D))
    _need(counters, torch.int32, "counters", (R,))
    _need(out, out.dtype, "out", (R, D))
    if lse is not None:
        _need(lse, torch.float32, "lse", (R,))
    _check(_lib.rf_attn_decode_fused(_ptr(q), _ptr(k), _ptr(v), R, L, D, S, float(scale), dt,
                                     _ptr(seg_m), _ptr(seg_l), _ptr(seg_acc), _ptr(counters),
                                     _ptr(out), _dtype_code(out.dtype), _ptr(lse), _stream(stream)),
           "rf_attn_decode_fused")


def rf_attn_decode_split_twopass(q, k, v, S, scale, seg_m, seg_l, seg_acc, stream=None):
    """Non-incremental split-KV decode: same arguments and outputs as
    rf_attn_decode_split; segments of at most 16384 keys."""
    R, L, D = k.shape
    _need(q, k.dtype, "q", (R, D))
    _need(k, k.dtype, "k")
    _need(v, k.dtype, "v", (R, L, D))
    _need(seg_m, torch.float32, "seg_m", (R, S))
    _need(seg_l, torch.float32, "seg_l", (R, S))
    _need(seg_acc, torch.float32, "seg_acc", (R, S, D))
    _check(_lib.rf_attn_decode_split_twopass(_ptr(q), _ptr(k), _ptr(v), R, L, D, S, float(scale),
                                             _dtype_code(k.dtype), _ptr(seg_m), _ptr(seg_l),
                                             _ptr(seg_acc), _stream(stream)),
           "rf_attn_decode_split_twopass")


def rf_mla_decode_split(q, c, S, scale, seg_m, seg_l, seg_acc, stream=None):
    """q [B, H, 576], c [B, L, 576] bf16 (shared latent cache) -> seg_m/seg_l [B, H, S],
    seg_acc [B, H, S, 512] fp32."""
    B, H, Dk = q.shape
    L = c.shape[1]
    Dv = seg_acc.shape[-1]
    _need(q, torch.bfloat16, "q")
    _need(c, torch.bfloat16, "c", (B, L, Dk))
    _need(seg_m, torch.float32, "seg_m", (B, H, S))
    _need(seg_l, torch.float32, "seg_l", (B, H, S))
    _need(seg_acc, torch.float32, "seg_acc", (B, H, S, Dv))
    _check(_lib.rf_mla_decode_split(_ptr(q), _ptr(c), B, H, L, Dk, Dv, S, float(scale),
                                    _ptr(seg_m), _ptr(seg_l), _ptr(seg_acc), _stream(stream)),
           "rf_mla_decode_split")


def rf_state_merge(seg_m, seg_l, seg_acc, out, lse=None, stream=None):
    """seg_* [R, S(, D)] fp32 -> out [R, D] (fp32 or bf16), lse [R] fp32 (optional)."""
    R, S, D = seg_acc.shape
    _need(seg_m, torch.float32, "seg_m", (R, S))
    _need(seg_l, torch.float32, "seg_l", (R, S))
    _need(seg_acc, torch.float32, "seg_acc")
    _need(out, out.dtype, "out", (R, D))
    if lse is not None:
        _need(lse, torch.float32, "lse", (R,))
    _check(_lib.rf_state_merge(_ptr(seg_m), _ptr(seg_l), _ptr(seg_acc), R, S, D, _ptr(out),
                               _dtype_code(out.dtype), _ptr(lse), _stream(stream)),
           "rf_state_merge")


def rf_attn_prefill(q, k, v, causal, scale, out, lse=None, stream=None):
    """q/k/v/out [B, H, N, D] bf16; lse [B, H, N] fp32 (optional)."""
    B, H, N, D = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _need(t, torch.bfloat16, name, (B, H, N, D))
    if lse is not None:
        _need(lse, torch.float32, "lse", (B, H, N))
    _check(_lib.rf_attn_prefill(_ptr(q), _ptr(k), _ptr(v), B, H, N, D, int(bool(causal)),
                                float(scale), _ptr(out), _ptr(lse), _stream(stream)),
           "rf_attn_prefill")


def rf_softmax_topk(logits, k, renormalize, idx, w, stream=None):
    """logits [T, E] fp32 -> idx [T, k] int32, w [T, k] fp32."""
    T, E = logits.shape
    _need(logits, torch.float32, "logits")
    _need(idx, torch.int32, "idx", (T, k))
    _need(w, torch.float32, "w", (T, k))
    _check(_lib.rf_softmax_topk(_ptr(logits), T, E, k, int(bool(renormalize)), _ptr(idx), _ptr(w),
                                _stream(stream)), "rf_softmax_topk")


def rf_absmax_quant_e4m3(x, xq, sx, stream=None):
    """x [M, K] bf16 -> xq [M, K] uint8 (e4m3 codes), sx [M] fp32."""
    M, K = x.shape
    _need(x, torch.bfloat16, "x")
    _need(xq, torch.uint8, "xq", (M, K))
    _need(sx, torch.float32, "sx", (M,))
    _check(_lib.rf_absmax_quant_e4m3(_ptr(x), M, K, _ptr(xq), _ptr(sx), _stream(stream)),
           "rf_absmax_quant_e4m3")


def rf_fp8_gemm_scaled(xq, sx, wq, sw, y, stream=None):
    """xq [M, K], wq [N, K] uint8 e4m3; sx [M], sw [N] fp32 -> y [M, N] bf16."""
    M, K = xq.shape
    N = wq.shape[0]
    _need(xq, torch.uint8, "xq")
    _need(wq, torch.uint8, "wq", (N, K))
    _need(sx, torch.float32, "sx", (M,))
    _need(sw, torch.float32, "sw", (N,))
    _need(y, torch.bfloat16, "y", (M, N))
    _check(_lib.rf_fp8_gemm_scaled(_ptr(xq), _ptr(sx), _ptr(wq), _ptr(sw), M, N, K, _ptr(y),
                                   _stream(stream)), "rf_fp8_gemm_scaled")


def rf_absmax_quant_fp8_gemm(x, wq, sw, xq, sx, y, stream=None):
    """x [M, K] bf16, wq [N, K] uint8, sw [N] -> xq [M, K] uint8, sx [M], y [M, N] bf16."""
    M, K = x.shape
    N = wq.shape[0]
    _need(x, torch.bfloat16, "x")
    _need(wq, torch.uint8, "wq", (N, K))
    _need(sw, torch.float32, "sw", (N,))
    _need(xq, torch.uint8, "xq", (M, K))
    _need(sx, torch.float32, "sx", (M,))
    _need(y, torch.bfloat16, "y", (M, N))
    _check(_lib.rf_absmax_quant_fp8_gemm(_ptr(x), M, K, _ptr(wq), _ptr(sw), N, _ptr(xq), _ptr(sx),
                                         _ptr(y), _stream(stream)), "rf_absmax_quant_fp8_gemm")


def rf_attn_decode_noalloc(q, k, v, S, scale, out, lse=None, stream=None):
    """Decode split + merge with the segment states in the library's fixed
    16 MiB device array: for callers that cannot allocate device memory.

    q [R, D], k/v [R, L, D] (fp32 D=64 or bf16 D=128); out [R, D] fp32 or
    bf16; lse [R] fp32 (optional).  Calls that may overlap on the GPU share the
    array and race; the first call on a device must precede stream capture."""
    R, L, D = k.shape
    _need(q, k.dtype, "q", (R, D))
    _need(k, k.dtype, "k")
    _need(v, k.dtype, "v", (R, L, D))
    _need(out, out.dtype, "out", (R, D))
    if lse is not None:
        _need(lse, torch.float32, "lse", (R,))
    _check(_lib.rf_attn_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), R, L, D, S, float(scale),
                                       _dtype_code(k.dtype), _ptr(out), _dtype_code(out.dtype),
                                       _ptr(lse), _stream(stream)), "rf_attn_decode_noalloc")


def rf_row_softmax(x, y, level, work=None, stream=None):
    """x, y [R, n] fp32; work [2R] fp32 for RF_FUSE_NONE."""
    R, n = x.shape
    _need(x, torch.float32, "x")
    _need(y, torch.float32, "y", (R, n))
    if work is not None:
        _need(work, torch.float32, "work", (2 * R,))
    _check(_lib.rf_row_softmax(_ptr(x), R, n, _ptr(y), int(level), _ptr(work), _stream(stream)),
           "rf_row_softmax")


def rf_row_variance(x, mean, var, level, stream=None):
    """x [R, n] fp32 -> mean [R], var [R] (population variance)."""
    R, n = x.shape
    _need(x, torch.float32, "x")
    _need(mean, torch.float32, "mean", (R,))
    _need(var, torch.float32, "var", (R,))
    _check(_lib.rf_row_variance(_ptr(x), R, n, _ptr(mean), _ptr(var), int(level),
                                _stream(stream)), "rf_row_variance")


def rf_moment_of_inertia(mass, pos, center, inertia, level, stream=None):
    """mass [R, n], pos [R, 3, n] fp32 -> center [R, 3], inertia [R]."""
    R, n = mass.shape
    _need(mass, torch.float32, "mass")
    _need(pos, torch.float32, "pos", (R, 3, n))
    _need(center, torch.float32, "center", (R, 3))
    _need(inertia, torch.float32, "inertia", (R,))
    _check(_lib.rf_moment_of_inertia(_ptr(mass), _ptr(pos), R, n, _ptr(center), _ptr(inertia),
                                     int(level), _stream(stream)), "rf_moment_of_inertia")


def rf_layer_norm(x, gamma, beta, eps, y, level, work=None, stream=None):
    """x, y [R, n] fp32; gamma, beta [n]; work [2R] fp32 for RF_FUSE_NONE."""
    R, n = x.shape
    _need(x, torch.float32, "x")
    _need(gamma, torch.float32, "gamma", (n,))
    _need(beta, torch.float32, "beta", (n,))
    _need(y, torch.float32, "y", (R, n))
    if work is not None:
        _need(work, torch.float32, "work", (2 * R,))
    _check(_lib.rf_layer_norm(_ptr(x), _ptr(gamma), _ptr(beta), R, n, float(eps), _ptr(y),
                              int(level), _ptr(work), _stream(stream)), "rf_layer_norm")


def rf_rms_norm(x, gamma, eps, y, level, work=None, stream=None):
    """x, y [R, n] fp32; gamma [n]; level RF_FUSE_NONE needs work [R] fp32."""
    R, n = x.shape
    _need(x, torch.float32, "x")
    _need(gamma, torch.float32, "gamma", (n,))
    _need(y, torch.float32, "y", (R, n))
    if work is not None:
        _need(work, torch.float32, "work", (R,))
    _check(_lib.rf_rms_norm(_ptr(x), _ptr(gamma), R, n, float(eps), _ptr(y), int(level), _ptr(work),
                            _stream(stream)), "rf_rms_norm")


def rf_incremental_quant_fp8_gemm(x, wq, sw, y, sx_final=None, stream=None):
    """x [M, K] bf16, wq [N, K] uint8 e4m3, sw [N] -> y [M, N] bf16, sx_final [M] (optional)."""
    M, K = x.shape
    N = wq.shape[0]
    _need(x, torch.bfloat16, "x")
    _need(wq, torch.uint8, "wq", (N, K))
    _need(sw, torch.float32, "sw", (N,))
    _need(y, torch.bfloat16, "y", (M, N))
    if sx_final is not None:
        _need(sx_final, torch.float32, "sx_final", (M,))
    _check(_lib.rf_incremental_quant_fp8_gemm(_ptr(x), M, K, _ptr(wq), _ptr(sw), N, _ptr(y),
                                              _ptr(sx_final), _stream(stream)),
           "rf_incremental_quant_fp8_gemm")


def rf_stream_read(x, out_xor, stream=None):
    """XOR every 32-bit word of the CUDA tensor ``x`` into ``out_xor`` (one
    int32 element, device memory) with one streaming read of ``x``."""
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")
    _need(out_xor, torch.int32, "out_xor", (1,))
    _check(_lib.rf_stream_read(_ptr(x), x.numel() * x.element_size(), _ptr(out_xor),
                               _stream(stream)), "rf_stream_read")


def rf_selftest_wait_timeout(waited_ms, stream=None):
    """waited_ms: int32 CUDA tensor of one element; the timeout shows up in rf_device_error()."""
    _need(waited_ms, torch.int32, "waited_ms", (1,))
    _check(_lib.rf_selftest_wait_timeout(_ptr(waited_ms), _stream(stream)), "rf_selftest_wait_timeout")


def rf_selftest_bounds(stream=None):
    """One refused index through the bounds check (bounds-checked build only);
    RF_ERR_BOUNDS then shows up in rf_device_error()."""
    _check(_lib.rf_selftest_bounds(_stream(stream)), "rf_selftest_bounds")


def rf_bounds_checked():
    """True if the loaded library checks every kernel's global indices."""
    return bool(_lib.rf_bounds_checked())


def rf_device_error(stream=None):
    """Synchronise and return (and clear) the on-device status words: bounded
    waits, and in the bounds-checked build the index checks."""
    st = _I(0)
    _check(_lib.rf_device_error(ctypes.byref(st), _stream(stream)), "rf_device_error")
    return st.value


# ----------------------------------------------------- convenience wrappers --

def attn_decode(q, k, v, S, scale, out_dtype=None, return_states=False, stream=None):
    """Split-KV decode: rf_attn_decode_split then rf_state_merge.

    q [R, D], k/v [R, L, D]; returns out [R, D] (and lse, and the segment states
    if ``return_states``)."""
    R, L, D = k.shape
    dev = k.device
    seg_m = torch.empty(R, S, device=dev, dtype=torch.float32)
    seg_l = torch.empty(R, S, device=dev, dtype=torch.float32)
    seg_acc = torch.empty(R, S, D, device=dev, dtype=torch.float32)
    out = torch.empty(R, D, device=dev, dtype=out_dtype or k.dtype)
    lse = torch.empty(R, device=dev, dtype=torch.float32)
    rf_attn_decode_split(q, k, v, S, scale, seg_m, seg_l, seg_acc, stream)
    rf_state_merge(seg_m, seg_l, seg_acc, out, lse, stream)
    if return_states:
        return out, lse, (seg_m, seg_l, seg_acc)
    return out, lse


def mla_decode(q, c, S, scale, dv=512, return_states=False, stream=None):
    """MLA split decode: rf_mla_decode_split then rf_state_merge.

    q [B, H, 576], c [B, L, 576] bf16; returns out [B, H, dv] bf16 and lse [B, H]
    (and the segment states if ``return_states``)."""
    B, H, _ = q.shape
    dev = q.device
    seg_m = torch.empty(B, H, S, device=dev, dtype=torch.float32)
    seg_l = torch.empty(B, H, S, device=dev, dtype=torch.float32)
    seg_acc = torch.empty(B, H, S, dv, device=dev, dtype=torch.float32)
    out = torch.empty(B, H, dv, device=dev, dtype=torch.bfloat16)
    lse = torch.empty(B, H, device=dev, dtype=torch.float32)
    rf_mla_decode_split(q, c, S, scale, seg_m, seg_l, seg_acc, stream)
    rf_state_merge(seg_m.view(B * H, S), seg_l.view(B * H, S), seg_acc.view(B * H, S, dv),
                   out.view(B * H, dv), lse.view(B * H), stream)
    if return_states:
        return out, lse, (seg_m, seg_l, seg_acc)
    return out, lse


def softmax_topk(logits, k, renormalize=True, stream=None):
    T = logits.shape[0]
    idx = torch.empty(T, k, device=logits.device, dtype=torch.int32)
    w = torch.empty(T, k, device=logits.device, dtype=torch.float32)
    rf_softmax_topk(logits, k, renormalize, idx, w, stream)
    return idx, w


def absmax_quant_fp8_gemm(x, wq, sw, stream=None):
    M, K = x.shape
    N = wq.shape[0]
    xq = torch.empty(M, K, device=x.device, dtype=torch.uint8)
    sx = torch.empty(M, device=x.device, dtype=torch.float32)
    y = torch.empty(M, N, device=x.device, dtype=torch.bfloat16)
    rf_absmax_quant_fp8_gemm(x, wq, sw, xq, sx, y, stream)
    return xq, sx, y


def attn_prefill(q, k, v, causal=True, scale=None, stream=None):
    B, H, N, D = q.shape
    if scale is None:
        scale = D ** -0.5
    out = torch.empty_like(q)
    lse = torch.empty(B, H, N, device=q.device, dtype=torch.float32)
    rf_attn_prefill(q, k, v, causal, scale, out, lse, stream)
    return out, lse
