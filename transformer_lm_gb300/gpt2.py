"""Thin ctypes binding of libgpt2.so: the same names as the C ABI in include/gpt2.h.

Argument marshalling only -- every step of the training step and of the fused
operator runs in the library's CUDA kernels. Host arrays are numpy arrays;
device arguments are raw pointers (ints) or objects with ``data_ptr()``
(e.g. torch CUDA tensors). If the library has not been built, the first call
raises immediately: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgpt2.so")

GPT2_FP32 = 0
GPT2_BF16 = 1
GPT2_FP16 = 2

ERRORS = {0: "OK", -1: "CONFIG", -2: "STATE", -3: "SHAPE", -4: "TOKEN", -5: "ALIGN", -6: "CUDA",
          -7: "NOMEM", -8: "ARG", -9: "DEVICE_TIMEOUT"}

ACT = dict(encoded=0, ln1=1, qkv=2, atty=4, residual2=5, ln2=6, fch=7, fch_gelu=8, residual3=9,
           lnf=10, logits=11, probs=12, lse=18)

EPI = dict(store=0, gelu=1, resid=2, gelu_bwd=3, accum=4)

FAMILIES = ["gemm", "attn_fwd", "attn_bwd", "ln_fwd", "ln_bwd", "classifier", "adamw", "encoder",
            "other"]


class GPT2Error(RuntimeError):
    def __init__(self, name: str, code: int, msg: str):
        super().__init__(f"{name} -> {ERRORS.get(code, code)} ({code}): {msg}")
        self.code = code


_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_ll = ctypes.c_longlong
_f = ctypes.c_float
_sz = ctypes.c_size_t
_fp = ctypes.POINTER(ctypes.c_float)
_ip = ctypes.POINTER(ctypes.c_int)

_SIGS = {
    "gpt2_init": (_i, [_i, _i, _i, _i, _i, _i, ctypes.c_ulonglong]),
    "gpt2_init_ex": (_i, [_i, _i, _i, _i, _i, _i, ctypes.c_ulonglong, _i, _i]),
    "gpt2_set_stream": (_i, [_vp]),
    "gpt2_forward": (_f, [_ip, _ip, _i, _i]),
    "gpt2_forward_device": (_i, [_vp, _vp, _i, _i, _vp]),
    "gpt2_zero_grad": (_i, []),
    "gpt2_set_grad_accum": (_i, [_i]),
    "gpt2_get_grad_accum": (_i, []),
    "gpt2_backward": (_i, []),
    "gpt2_adamw": (_i, [_f, _f, _f, _f, _f, _i]),
    "gpt2_set_master_weights": (_i, [_i]),
    "gpt2_sync": (_i, []),
    "gpt2_set_wait_limit": (_i, [ctypes.c_ulonglong]),
    "gpt2_num_params": (_sz, []),
    "gpt2_param_sizes": (_i, [ctypes.POINTER(_sz)]),
    "gpt2_get_params": (_i, [_fp]),
    "gpt2_set_params": (_i, [_fp]),
    "gpt2_get_grads": (_i, [_fp]),
    "gpt2_set_grads": (_i, [_fp]),
    "gpt2_get_master": (_i, [_fp]),
    "gpt2_get_losses": (_i, [_fp]),
    "gpt2_get_activation": (_i, [_i, _i, _fp, ctypes.POINTER(_sz)]),
    "gpt2_free": (_i, []),
    "gpt2_sample": (_i, [_i, _fp, _ip]),
    "gpt2_set_loss_scaling": (_i, [_f, _i]),
    "gpt2_get_loss_scale": (_i, [_fp, ctypes.POINTER(_ll)]),
    "gpt2_generate": (_i, [_ip, _i, _i, _i, _i, ctypes.POINTER(ctypes.c_ulonglong)]),
    "gpt2_last_error": (ctypes.c_char_p, []),
    "gpt2_last_status": (_i, []),
    "gpt2_timing_begin": (_i, [_i]),
    "gpt2_timing_end": (_i, []),
    "gpt2_timing_get": (_i, [_i, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_ll),
                             ctypes.POINTER(ctypes.c_double)]),
    "fused_linear_bias_gelu_softmax": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _vp]),
    "fused_linear_bias_gelu_softmax_noalloc": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _vp]),
    "gpt2_gemm": (_i, [_i, _i, _i, _vp, _ll, _i, _vp, _ll, _i, _vp, _ll, _vp, _vp, _ll, _vp, _i, _i,
                       _i, _vp, _sz, _vp]),
    "gpt2_attention_forward": (_i, [_i, _i, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "gpt2_attention_backward": (_i, [_i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "gpt2_device_status": (_i, []),
    "gpt2_train_step": (_i, [_vp, _vp, _i, _i, _f, _f, _f, _f, _f, _i, _vp]),
    "gpt2_train_step_host": (_i, [_ip, _ip, _i, _i, _f, _f, _f, _f, _f, _i, _fp]),
    "gpt2_layernorm_forward": (_i, [_i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _vp]),
    "gpt2_layernorm_backward_scratch_floats": (_sz, [_i]),
    "gpt2_layernorm_backward": (_i, [_i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _vp,
                                     _vp]),
    "gpt2_launch_count": (_ll, []),
}


def lib():
    """Load libgpt2.so (built by transformer_lm_gb300.build); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run __graft_entry__.build() first "
                               "(there is no non-CUDA fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def gpt2_last_error() -> str:
    return lib().gpt2_last_error().decode()


def gpt2_last_status() -> int:
    return int(lib().gpt2_last_status())


def _check(name: str, rc: int) -> None:
    if rc != 0:
        raise GPT2Error(name, rc, gpt2_last_error())


def ptr(x) -> int | None:
    """Device pointer of an int, None, or an object with data_ptr()."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _ints(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32).reshape(-1)


def _as_ip(a):
    return None if a is None else a.ctypes.data_as(_ip)


def gpt2_init(L, C, NH, V, Vp, maxT, seed=1337) -> None:
    _check("gpt2_init", lib().gpt2_init(L, C, NH, V, Vp, maxT, seed))


def gpt2_init_ex(L, C, NH, V, Vp, maxT, seed, precision, tensor_cores) -> None:
    _check("gpt2_init_ex", lib().gpt2_init_ex(L, C, NH, V, Vp, maxT, seed, precision, tensor_cores))


def gpt2_set_stream(stream) -> None:
    _check("gpt2_set_stream", lib().gpt2_set_stream(stream))


def gpt2_forward(tokens, targets, B, T) -> float:
    tok = _ints(tokens)
    tgt = None if targets is None else _ints(targets)
    loss = lib().gpt2_forward(_as_ip(tok), _as_ip(tgt), B, T)
    if np.isnan(loss):
        raise GPT2Error("gpt2_forward", gpt2_last_status(), gpt2_last_error())
    return float(loss)


def gpt2_forward_device(d_tokens, d_targets, B, T, d_mean_loss=None) -> None:
    _check("gpt2_forward_device",
           lib().gpt2_forward_device(ptr(d_tokens), ptr(d_targets), B, T, ptr(d_mean_loss)))


def gpt2_zero_grad() -> None:
    _check("gpt2_zero_grad", lib().gpt2_zero_grad())


def gpt2_set_grad_accum(k) -> None:
    _check("gpt2_set_grad_accum", lib().gpt2_set_grad_accum(k))


def gpt2_get_grad_accum() -> int:
    k = int(lib().gpt2_get_grad_accum())
    if k < 1:
        raise GPT2Error("gpt2_get_grad_accum", k, gpt2_last_error())
    return k


def gpt2_backward() -> None:
    _check("gpt2_backward", lib().gpt2_backward())


def gpt2_adamw(lr, beta1, beta2, eps, weight_decay, step) -> None:
    _check("gpt2_adamw", lib().gpt2_adamw(lr, beta1, beta2, eps, weight_decay, step))


def gpt2_set_master_weights(enabled: bool) -> None:
    _check("gpt2_set_master_weights", lib().gpt2_set_master_weights(int(bool(enabled))))


def gpt2_train_step(d_tokens, d_targets, B, T, lr, beta1, beta2, eps, weight_decay, step,
                    d_mean_loss=None) -> None:
    """Forward, zero_grad, backward and AdamW on device buffers (CUDA-graph replays)."""
    _check("gpt2_train_step", lib().gpt2_train_step(ptr(d_tokens), ptr(d_targets), B, T, lr, beta1,
                                                    beta2, eps, weight_decay, step,
                                                    ptr(d_mean_loss)))


def gpt2_train_step_host(tokens, targets, B, T, lr, beta1, beta2, eps, weight_decay,
                         step) -> np.ndarray:
    """The whole step on host ids (k*B*T each, k = the accumulation count);
    returns the k micro-step mean losses."""
    tok, tgt = _ints(tokens), _ints(targets)
    k = gpt2_get_grad_accum()
    if tok.size != k * B * T or tgt.size != k * B * T:
        raise ValueError(f"expected {k}*{B}*{T} token and target ids, got {tok.size}, {tgt.size}")
    out = np.empty(k, dtype=np.float32)
    _check("gpt2_train_step_host",
           lib().gpt2_train_step_host(_as_ip(tok), _as_ip(tgt), B, T, lr, beta1, beta2, eps,
                                      weight_decay, step, out.ctypes.data_as(_fp)))
    return out


def gpt2_set_wait_limit(ns: int) -> None:
    _check("gpt2_set_wait_limit", lib().gpt2_set_wait_limit(int(ns)))


def gpt2_sync() -> None:
    _check("gpt2_sync", lib().gpt2_sync())


def gpt2_num_params() -> int:
    return int(lib().gpt2_num_params())


def gpt2_param_sizes() -> list[int]:
    out = (_sz * 16)()
    _check("gpt2_param_sizes", lib().gpt2_param_sizes(out))
    return [int(x) for x in out]


def _host_f32(n):
    return np.empty(n, dtype=np.float32)


def gpt2_get_params() -> np.ndarray:
    out = _host_f32(gpt2_num_params())
    _check("gpt2_get_params", lib().gpt2_get_params(out.ctypes.data_as(_fp)))
    return out


def gpt2_set_params(params) -> None:
    a = np.ascontiguousarray(params, dtype=np.float32).reshape(-1)
    if a.size != gpt2_num_params():
        raise ValueError(f"expected {gpt2_num_params()} parameters, got {a.size}")
    _check("gpt2_set_params", lib().gpt2_set_params(a.ctypes.data_as(_fp)))


def gpt2_get_grads() -> np.ndarray:
    out = _host_f32(gpt2_num_params())
    _check("gpt2_get_grads", lib().gpt2_get_grads(out.ctypes.data_as(_fp)))
    return out


def gpt2_set_grads(grads) -> None:
    a = np.ascontiguousarray(grads, dtype=np.float32).reshape(-1)
    if a.size != gpt2_num_params():
        raise ValueError(f"expected {gpt2_num_params()} gradients, got {a.size}")
    _check("gpt2_set_grads", lib().gpt2_set_grads(a.ctypes.data_as(_fp)))


def gpt2_get_master() -> np.ndarray:
    out = _host_f32(gpt2_num_params())
    _check("gpt2_get_master", lib().gpt2_get_master(out.ctypes.data_as(_fp)))
    return out


def gpt2_get_losses(n: int) -> np.ndarray:
    out = _host_f32(n)
    _check("gpt2_get_losses", lib().gpt2_get_losses(out.ctypes.data_as(_fp)))
    return out


def gpt2_get_activation(name: str, layer: int = 0) -> np.ndarray:
    which = ACT[name]
    n = _sz(0)
    _check("gpt2_get_activation", lib().gpt2_get_activation(which, layer, None, ctypes.byref(n)))
    out = _host_f32(n.value)
    _check("gpt2_get_activation",
           lib().gpt2_get_activation(which, layer, out.ctypes.data_as(_fp), None))
    return out


def gpt2_sample(t: int, coins) -> np.ndarray:
    c = np.ascontiguousarray(coins, dtype=np.float32).reshape(-1)
    out = np.empty(c.size, dtype=np.int32)
    _check("gpt2_sample", lib().gpt2_sample(t, c.ctypes.data_as(_fp), out.ctypes.data_as(_ip)))
    return out


def gpt2_generate(tokens, B, T, t_begin, t_end, rng_state: int):
    """Returns (tokens (B, T) int32, advanced rng_state)."""
    tok = np.array(tokens, dtype=np.int32).reshape(-1).copy()
    st = ctypes.c_ulonglong(rng_state)
    _check("gpt2_generate", lib().gpt2_generate(tok.ctypes.data_as(_ip), B, T, t_begin, t_end,
                                                ctypes.byref(st)))
    return tok.reshape(B, T), int(st.value)


def gpt2_set_loss_scaling(init_scale: float, growth_interval: int) -> None:
    _check("gpt2_set_loss_scaling", lib().gpt2_set_loss_scaling(init_scale, growth_interval))


def gpt2_get_loss_scale():
    """(current loss scale, updates skipped so far)."""
    sc = ctypes.c_float()
    sk = _ll()
    _check("gpt2_get_loss_scale", lib().gpt2_get_loss_scale(ctypes.byref(sc), ctypes.byref(sk)))
    return float(sc.value), int(sk.value)


def gpt2_free() -> None:
    _check("gpt2_free", lib().gpt2_free())


def gpt2_timing_begin(max_launches: int) -> None:
    _check("gpt2_timing_begin", lib().gpt2_timing_begin(max_launches))


def gpt2_timing_end() -> None:
    _check("gpt2_timing_end", lib().gpt2_timing_end())


def gpt2_timing_get(family: int | str):
    f = FAMILIES.index(family) if isinstance(family, str) else family
    ms = ctypes.c_double()
    n = _ll()
    work = ctypes.c_double()
    _check("gpt2_timing_get", lib().gpt2_timing_get(f, ctypes.byref(ms), ctypes.byref(n),
                                                    ctypes.byref(work)))
    return ms.value, n.value, work.value


def fused_linear_bias_gelu_softmax(x, W, b, out, M, K, N, stream=None) -> None:
    _check("fused_linear_bias_gelu_softmax",
           lib().fused_linear_bias_gelu_softmax(ptr(x), ptr(W), ptr(b), ptr(out), M, K, N, stream))


def fused_linear_bias_gelu_softmax_noalloc(x, W, b, out, M, K, N, stream=None) -> None:
    _check("fused_linear_bias_gelu_softmax_noalloc",
           lib().fused_linear_bias_gelu_softmax_noalloc(ptr(x), ptr(W), ptr(b), ptr(out), M, K, N,
                                                        stream))


def gpt2_gemm(dtype, tensor_cores, epilogue, A, lda, a_kmajor, B, ldb, b_kmajor, D, ldd, bias=None,
              aux=None, ldaux=0, D2=None, M=0, N=0, K=0, ws=None, ws_floats=0,
              stream=None) -> None:
    epi = EPI[epilogue] if isinstance(epilogue, str) else epilogue
    _check("gpt2_gemm", lib().gpt2_gemm(dtype, tensor_cores, epi, ptr(A), lda, int(a_kmajor), ptr(B),
                                        ldb, int(b_kmajor), ptr(D), ldd, ptr(bias), ptr(aux), ldaux,
                                        ptr(D2), M, N, K, ptr(ws), ws_floats if ws is not None else 0,
                                        stream))


def gpt2_attention_forward(dtype, tensor_cores, qkv, out, lse, B, T, C, NH, stream=None) -> None:
    _check("gpt2_attention_forward",
           lib().gpt2_attention_forward(dtype, tensor_cores, ptr(qkv), ptr(out), ptr(lse), B, T, C,
                                        NH, stream))


def gpt2_attention_backward(dtype, tensor_cores, dout, qkv, out, lse, dqkv, scratch_D, B, T, C, NH,
                            stream=None) -> None:
    _check("gpt2_attention_backward",
           lib().gpt2_attention_backward(dtype, tensor_cores, ptr(dout), ptr(qkv), ptr(out),
                                         ptr(lse), ptr(dqkv), ptr(scratch_D), B, T, C, NH, stream))


def gpt2_layernorm_forward(dtype, out, mean, rstd, inp, w, b, N, C, stream=None) -> None:
    _check("gpt2_layernorm_forward",
           lib().gpt2_layernorm_forward(dtype, ptr(out), ptr(mean), ptr(rstd), ptr(inp), ptr(w),
                                        ptr(b), N, C, stream))


def gpt2_layernorm_backward_scratch_floats(C) -> int:
    return int(lib().gpt2_layernorm_backward_scratch_floats(C))


def gpt2_layernorm_backward(dtype, dinp, dw, db, dout, inp, w, mean, rstd, N, C, accumulate,
                            scratch, stream=None) -> None:
    _check("gpt2_layernorm_backward",
           lib().gpt2_layernorm_backward(dtype, ptr(dinp), ptr(dw), ptr(db), ptr(dout), ptr(inp),
                                         ptr(w), ptr(mean), ptr(rstd), N, C, int(accumulate),
                                         ptr(scratch), stream))


def gpt2_launch_count() -> int:
    return int(lib().gpt2_launch_count())


def gpt2_device_status() -> None:
    _check("gpt2_device_status", lib().gpt2_device_status())
