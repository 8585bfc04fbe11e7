"""CPU oracle for the GPT-2 training step and the fused Linear+GELU+softmax op.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``. The GPU product path never imports it.

The arithmetic lives in ``gpt2_oracle.c`` (plain C, double precision); this
module only compiles it and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gpt2_oracle.c")
_HDR = os.path.join(_HERE, "gpt2_oracle.h")
_LIB = os.path.join(_HERE, "libgpt2_oracle.so")
_lock = threading.Lock()
_lib = None

NUM_PARAM_TENSORS = 16
PARAM_NAMES = ["wte", "wpe", "ln1w", "ln1b", "qkvw", "qkvb", "attprojw", "attprojb",
               "ln2w", "ln2b", "fcw", "fcb", "fcprojw", "fcprojb", "lnfw", "lnfb"]

ACT = dict(encoded=0, ln1=1, qkv=2, att=3, atty=4, residual2=5, ln2=6, fch=7, fch_gelu=8,
           residual3=9, lnf=10, logits=11, probs=12, losses=13, dlogits=14, ln1_mean=15,
           ln1_rstd=16)


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library beside its source."""
    with _lock:
        newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
        if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
            return _LIB
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-D_GNU_SOURCE", "-ffp-contract=off", "-fPIC", "-shared",
               "-fopenmp",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int), ("C", ctypes.c_int), ("NH", ctypes.c_int),
                ("V", ctypes.c_int), ("Vp", ctypes.c_int), ("maxT", ctypes.c_int)]


_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def lib():
    global _lib
    if _lib is None:
        path = build()
        L = ctypes.CDLL(path)
        L.oracle_param_sizes.restype = ctypes.c_size_t
        L.oracle_param_sizes.argtypes = [ctypes.POINTER(_Cfg), ctypes.POINTER(ctypes.c_size_t)]
        L.oracle_create.restype = ctypes.c_void_p
        L.oracle_create.argtypes = [ctypes.POINTER(_Cfg), ctypes.c_int, ctypes.c_int]
        L.oracle_destroy.argtypes = [ctypes.c_void_p]
        L.oracle_forward.restype = ctypes.c_double
        L.oracle_forward.argtypes = [ctypes.c_void_p, _dp, _ip, _ip, ctypes.c_int]
        L.oracle_backward.restype = ctypes.c_int
        L.oracle_backward.argtypes = [ctypes.c_void_p, _dp, _dp]
        L.oracle_get_act.restype = ctypes.c_size_t
        L.oracle_get_act.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, _dp]
        L.oracle_adamw.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_size_t, ctypes.c_double,
                                   ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                   ctypes.c_double, ctypes.c_int]
        L.oracle_fused_linear_bias_gelu_softmax.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int,
                                                            ctypes.c_int, ctypes.c_int]
        L.oracle_encoder_forward.argtypes = [_dp, _ip, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int]
        L.oracle_layernorm_forward.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int,
                                               ctypes.c_int]
        L.oracle_layernorm_backward.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                                                ctypes.c_int, ctypes.c_int]
        L.oracle_matmul_forward.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int]
        L.oracle_matmul_backward.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int]
        L.oracle_gelu_forward.argtypes = [_dp, _dp, ctypes.c_size_t]
        L.oracle_gelu_backward.argtypes = [_dp, _dp, _dp, ctypes.c_size_t]
        L.oracle_attention_forward.argtypes = [_dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int]
        L.oracle_attention_backward.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int]
        L.oracle_num_threads.restype = ctypes.c_int
        _u64p = ctypes.POINTER(ctypes.c_ulonglong)
        L.oracle_random_u32.restype = ctypes.c_uint
        L.oracle_random_u32.argtypes = [_u64p]
        L.oracle_random_f32.restype = ctypes.c_float
        L.oracle_random_f32.argtypes = [_u64p]
        L.oracle_squirrel_noise5.restype = ctypes.c_uint
        L.oracle_squirrel_noise5.argtypes = [ctypes.c_uint, ctypes.c_uint]
        L.oracle_noise_2d.restype = ctypes.c_uint
        L.oracle_noise_2d.argtypes = [ctypes.c_uint, ctypes.c_uint, ctypes.c_uint]
        L.oracle_bf16_rne.restype = ctypes.c_ushort
        L.oracle_bf16_rne.argtypes = [ctypes.c_float]
        L.oracle_stochastic_round_bf16.restype = ctypes.c_ushort
        L.oracle_stochastic_round_bf16.argtypes = [ctypes.c_float, ctypes.c_uint]
        _usp = ctypes.POINTER(ctypes.c_ushort)
        _fp = ctypes.POINTER(ctypes.c_float)
        L.oracle_adamw_bf16_sr.argtypes = [_usp, _usp, _fp, _fp, ctypes.c_size_t, ctypes.c_float,
                                           ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                           ctypes.c_float, ctypes.c_int, ctypes.c_uint]
        L.oracle_sample_softmax.restype = ctypes.c_int
        L.oracle_sample_softmax.argtypes = [_dp, ctypes.c_int, ctypes.c_double]
        _lib = L
    return _lib


def _d(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(_dp)


def _i(a: np.ndarray):
    assert a.dtype == np.int32 and a.flags.c_contiguous
    return a.ctypes.data_as(_ip)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def param_sizes(L, C, NH, V, Vp, maxT):
    cfg = _Cfg(L, C, NH, V, Vp, maxT)
    out = (ctypes.c_size_t * NUM_PARAM_TENSORS)()
    total = lib().oracle_param_sizes(ctypes.byref(cfg), out)
    return [int(x) for x in out], int(total)


class Model:
    """One (B, T) batch shape of the oracle model; params/grads are flat float64."""

    def __init__(self, L, C, NH, V, Vp, maxT, B, T):
        self.cfg = _Cfg(L, C, NH, V, Vp, maxT)
        self.dims = dict(L=L, C=C, NH=NH, V=V, Vp=Vp, maxT=maxT)
        self.B, self.T = B, T
        self._h = lib().oracle_create(ctypes.byref(self.cfg), B, T)
        if not self._h:
            raise ValueError("oracle_create failed (bad shape or out of memory)")
        self.sizes, self.num_params = param_sizes(L, C, NH, V, Vp, maxT)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib().oracle_destroy(h)
            self._h = None

    def forward(self, params, tokens, targets=None, grad_accum_k=1) -> float:
        self._params = _f64(params)
        tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(-1)
        tgt = None if targets is None else np.ascontiguousarray(targets, dtype=np.int32).reshape(-1)
        return float(lib().oracle_forward(self._h, _d(self._params), _i(tok),
                                          None if tgt is None else _i(tgt), int(grad_accum_k)))

    def backward(self, grads: np.ndarray) -> None:
        """Accumulates into ``grads`` (float64, flat) in place."""
        assert grads.dtype == np.float64 and grads.size == self.num_params
        rc = lib().oracle_backward(self._h, _d(self._params), _d(grads))
        if rc != 0:
            raise RuntimeError("oracle backward without targets")

    def act(self, name: str, layer: int = 0) -> np.ndarray:
        B, T, d = self.B, self.T, self.dims
        C, NH, Vp, L = d["C"], d["NH"], d["Vp"], d["L"]
        n = {"encoded": B * T * C, "ln1": B * T * C, "qkv": B * T * 3 * C,
             "att": B * NH * T * T, "atty": B * T * C, "residual2": B * T * C,
             "ln2": B * T * C, "fch": B * T * 4 * C, "fch_gelu": B * T * 4 * C,
             "residual3": B * T * C, "lnf": B * T * C, "logits": B * T * Vp,
             "probs": B * T * Vp, "losses": B * T, "dlogits": B * T * Vp,
             "ln1_mean": B * T, "ln1_rstd": B * T}[name]
        out = np.empty(n, dtype=np.float64)
        got = lib().oracle_get_act(self._h, ACT[name], int(layer), _d(out))
        assert got == n
        return out

    def split(self, flat: np.ndarray) -> dict:
        out, off = {}, 0
        for name, s in zip(PARAM_NAMES, self.sizes):
            out[name] = flat[off:off + s]
            off += s
        return out


def adamw(params, grads, m, v, lr, beta1, beta2, eps, wd, t):
    """In-place AdamW on float64 arrays."""
    n = params.size
    lib().oracle_adamw(_d(params), _d(_f64(grads)), _d(m), _d(v), n, lr, beta1, beta2, eps, wd,
                       int(t))


class Rng:
    """The page's xorshift* generator on a 64-bit state."""

    def __init__(self, state: int):
        self.state = ctypes.c_ulonglong(state)

    def u32(self) -> int:
        return int(lib().oracle_random_u32(ctypes.byref(self.state)))

    def f32(self) -> float:
        return float(lib().oracle_random_f32(ctypes.byref(self.state)))


def squirrel_noise5(position: int, seed: int) -> int:
    return int(lib().oracle_squirrel_noise5(position & 0xFFFFFFFF, seed & 0xFFFFFFFF))


def noise_2d(x: int, y: int, seed: int) -> int:
    return int(lib().oracle_noise_2d(x & 0xFFFFFFFF, y & 0xFFFFFFFF, seed & 0xFFFFFFFF))


def bf16_rne(x: float) -> int:
    return int(lib().oracle_bf16_rne(x))


def stochastic_round_bf16(x: float, random: int) -> int:
    return int(lib().oracle_stochastic_round_bf16(x, random & 0xFFFFFFFF))


def adamw_bf16_sr(params_bits, grads_bits, m, v, lr, beta1, beta2, eps, wd, t, seed):
    """In place: uint16 bf16 bit patterns of params, float32 m and v."""
    assert params_bits.dtype == np.uint16 and params_bits.flags.c_contiguous
    g = np.ascontiguousarray(grads_bits, dtype=np.uint16)
    assert m.dtype == np.float32 and v.dtype == np.float32
    _usp = ctypes.POINTER(ctypes.c_ushort)
    _fp = ctypes.POINTER(ctypes.c_float)
    lib().oracle_adamw_bf16_sr(params_bits.ctypes.data_as(_usp), g.ctypes.data_as(_usp),
                               m.ctypes.data_as(_fp), v.ctypes.data_as(_fp), params_bits.size,
                               lr, beta1, beta2, eps, wd, int(t), seed & 0xFFFFFFFF)


def sample_softmax(logits, coin: float) -> int:
    lg = _f64(logits).reshape(-1)
    return int(lib().oracle_sample_softmax(_d(lg), lg.size, float(coin)))


def layernorm_forward(x, w, b):
    x = _f64(x)
    N, C = x.shape
    out = np.empty_like(x)
    mean = np.empty(N)
    rstd = np.empty(N)
    lib().oracle_layernorm_forward(_d(out), _d(mean), _d(rstd), _d(x), _d(_f64(w)), _d(_f64(b)),
                                   N, C)
    return out, mean, rstd


def layernorm_backward(dinp, dw, db, dout, x, w, mean, rstd):
    N, C = x.shape
    lib().oracle_layernorm_backward(_d(dinp), _d(dw), _d(db), _d(_f64(dout)), _d(_f64(x)),
                                    _d(_f64(w)), _d(_f64(mean)), _d(_f64(rstd)), N, C)


def matmul_forward(x, w, bias=None):
    x = _f64(x)
    w = _f64(w)
    N, Cin = x.shape
    Cout = w.shape[0]
    out = np.empty((N, Cout))
    lib().oracle_matmul_forward(_d(out), _d(x), _d(w), None if bias is None else _d(_f64(bias)),
                                N, Cin, Cout)
    return out


def matmul_backward(dout, x, w, dw, dbias=None):
    x = _f64(x)
    w = _f64(w)
    N, Cin = x.shape
    Cout = w.shape[0]
    dinp = np.empty((N, Cin))
    lib().oracle_matmul_backward(_d(dinp), _d(dw), None if dbias is None else _d(dbias),
                                 _d(_f64(dout)), _d(x), _d(w), N, Cin, Cout)
    return dinp


def gelu_forward(x):
    x = _f64(x)
    out = np.empty_like(x)
    lib().oracle_gelu_forward(_d(out), _d(x), x.size)
    return out


def gelu_backward(x, dout):
    x = _f64(x)
    out = np.empty_like(x)
    lib().oracle_gelu_backward(_d(out), _d(x), _d(_f64(dout)), x.size)
    return out


def encoder_forward(tokens, wte, wpe, B, T, C):
    out = np.empty((B * T * C,))
    tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(-1)
    lib().oracle_encoder_forward(_d(out), _i(tok), _d(_f64(wte)), _d(_f64(wpe)), B, T, C)
    return out


def attention_forward(qkv, B, T, C, NH):
    qkv = _f64(qkv)
    out = np.empty((B * T * C,))
    att = np.empty((B * NH * T * T,))
    lib().oracle_attention_forward(_d(out), _d(att), _d(qkv), B, T, C, NH)
    return out, att


def attention_backward(dout, qkv, att, B, T, C, NH):
    dqkv = np.empty((B * T * 3 * C,))
    lib().oracle_attention_backward(_d(dqkv), _d(_f64(dout)), _d(_f64(qkv)), _d(_f64(att)),
                                    B, T, C, NH)
    return dqkv


def fused_linear_bias_gelu_softmax(x, W, b):
    x = _f64(x)
    W = _f64(W)
    M, K = x.shape
    N = W.shape[0]
    y = np.empty((M, N))
    lib().oracle_fused_linear_bias_gelu_softmax(_d(x), _d(W), _d(_f64(b)), _d(y), M, K, N)
    return y
