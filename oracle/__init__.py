"""fp64 CPU oracle for Kimi Delta Attention (KDA).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` import this package.  The product
path (``linear_attention_layer_gb300`` and its CUDA library) never imports it,
and it imports nothing from there.

The arithmetic lives in ``kda_oracle.c`` (plain C, double precision): the
per-token recurrence of the state update and read-out defined on
mhpq.cn/news/56770, section "KDA 到底在算什么", with the lower-bounded gate of
blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构", section "下界衰减".
This module compiles it with gcc, widens the caller's arrays to float64
exactly and calls it.

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, hand-derived fixtures and an independent dense-matrix formulation.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")

#: The library's fixed L2-normalisation epsilon; the oracle default matches.
DEFAULT_EPS = 1e-6

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``_build/libkda_oracle.so`` (gcc -O2)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.kda_oracle_recurrent.restype = ctypes.c_int
            lib.kda_oracle_recurrent.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.POINTER(ctypes.c_int64), dp, dp, dp, dp, dp, dp, dp, dp,
                ctypes.c_int, ctypes.c_double, ctypes.c_int, dp]
            lib.kda_oracle_backward.restype = ctypes.c_int
            lib.kda_oracle_backward.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.POINTER(ctypes.c_int64)] + [dp] * 15 + [ctypes.c_double, ctypes.c_int]
            lib.kda_oracle_log_decay.restype = ctypes.c_double
            lib.kda_oracle_log_decay.argtypes = [ctypes.c_double]
            lib.kda_oracle_l2norm.restype = None
            lib.kda_oracle_l2norm.argtypes = [dp, dp, ctypes.c_int, ctypes.c_double]
            lib.kda_oracle_available_cpus.restype = ctypes.c_int
            lib.kda_oracle_available_cpus.argtypes = []
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Widen a numpy array or torch tensor to a C-contiguous float64 array."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widening bf16/fp32 -> fp64 is exact
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def available_cpus() -> int:
    return int(_load().kda_oracle_available_cpus())


def log_decay(z) -> np.ndarray:
    """g = -5 * sigmoid(z), elementwise, via the C oracle (fp64)."""
    lib = _load()
    z = _f64(z)
    return np.vectorize(lib.kda_oracle_log_decay, otypes=[np.float64])(z)


def l2norm(x, eps: float = DEFAULT_EPS) -> np.ndarray:
    """Row-wise x / sqrt(sum x^2 + eps) over the last axis, via the C oracle."""
    lib = _load()
    x = _f64(x)
    flat = x.reshape(-1, x.shape[-1])
    out = np.empty_like(flat)
    for i in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[i])
        o = np.empty_like(row)
        lib.kda_oracle_l2norm(_ptr(row), _ptr(o), row.shape[0], eps)
        out[i] = o
    return out.reshape(x.shape)


def recurrent(q, k, v, z, beta, cu_seqlens, initial_state=None, *,
              raw_log_decay: bool = False, eps: float = DEFAULT_EPS,
              threads: int = 0, with_final_state: bool = True, a_log=None):
    """Per-token KDA recurrence over a packed variable-length batch.

    q, k: [T_tot, H, dk]; v: [T_tot, H, dv]; z: [T_tot, H, dk] gate logits
    (or raw log-decay g when ``raw_log_decay``); beta: [T_tot, H];
    cu_seqlens: [N + 1] int; initial_state: [N, H, dk, dv] or None (zeros);
    a_log: [H] per-head gate log-scale A (g = -5 sigmoid(e^A z)) or None (A = 0).

    Returns ``(out [T_tot, H, dv], final_state [N, H, dk, dv] or None,
    threads_used)``, all float64.
    """
    lib = _load()
    q, k, v, z, beta = (_f64(a) for a in (q, k, v, z, beta))
    s0 = _f64(initial_state)
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
        dtype=np.int64))
    T, H, dk = q.shape
    dv = v.shape[-1]
    N = cu.shape[0] - 1
    assert k.shape == (T, H, dk) and z.shape == (T, H, dk)
    assert v.shape == (T, H, dv) and beta.shape == (T, H)
    assert cu[0] == 0 and cu[-1] == T
    if s0 is not None:
        assert s0.shape == (N, H, dk, dv)
    al = _f64(a_log)
    if al is not None:
        assert al.shape == (H,)
    out = np.zeros((T, H, dv), dtype=np.float64)
    fin = np.zeros((N, H, dk, dv), dtype=np.float64) if with_final_state else None
    used = lib.kda_oracle_recurrent(
        N, H, dk, dv, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(s0),
        _ptr(out), _ptr(fin), 1 if raw_log_decay else 0, float(eps), int(threads), _ptr(al))
    if used < 0:
        raise ValueError("kda_oracle_recurrent rejected its arguments")
    return out, fin, used


def backward(q, k, v, z, beta, cu_seqlens, initial_state, d_out, d_final=None, *,
             a_log=None, eps: float = DEFAULT_EPS, threads: int = 0):
    """Reverse mode of ``recurrent``: given dL/d out [T_tot, H, dv] and dL/d
    final_state [N, H, dk, dv] (or None = 0), the gradients
    ``(dq, dk, dv, dz, dbeta, d_initial_state)`` in float64 (dz with respect
    to the gate logits z; d_initial_state also when no initial state was given).
    """
    lib = _load()
    q, k, v, z, beta, do = (_f64(a) for a in (q, k, v, z, beta, d_out))
    s0, dfin, al = _f64(initial_state), _f64(d_final), _f64(a_log)
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
        dtype=np.int64))
    T, H, dk = q.shape
    dv = v.shape[-1]
    N = cu.shape[0] - 1
    assert do.shape == (T, H, dv)
    outs = [np.zeros((T, H, dk)), np.zeros((T, H, dk)), np.zeros((T, H, dv)),
            np.zeros((T, H, dk)), np.zeros((T, H)), np.zeros((N, H, dk, dv))]
    used = lib.kda_oracle_backward(
        N, H, dk, dv, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(s0), _ptr(al), _ptr(do),
        _ptr(dfin), *[_ptr(o) for o in outs], float(eps), int(threads))
    if used < 0:
        raise ValueError("kda_oracle_backward rejected its arguments")
    return tuple(outs)


def decode_step(q, k, v, z, beta, state, *, eps: float = DEFAULT_EPS,
                threads: int = 0, raw_log_decay: bool = False, a_log=None):
    """One recurrent step for a batch of live requests.

    q, k: [N, H, dk]; v: [N, H, dv]; z: [N, H, dk]; beta: [N, H];
    state: [N, H, dk, dv].  Each request is a sequence of length one, so this
    is ``recurrent`` with cu_seqlens = 0, 1, ..., N.  Returns
    ``(out [N, H, dv], new_state [N, H, dk, dv])`` in float64.
    """
    N = int(q.shape[0])
    cu = np.arange(N + 1, dtype=np.int64)
    out, fin, _ = recurrent(q, k, v, z, beta, cu, state, eps=eps,
                            threads=threads, raw_log_decay=raw_log_decay, a_log=a_log)
    return out, fin


# The Q/K preprocessing convolution + Swish (pure numpy, fp64).
from .short_conv import short_conv, swish  # noqa: E402,F401


def affine_summary(q, k, v, z, beta, cu_seqlens, *, a_log=None, eps: float = DEFAULT_EPS,
                   threads: int = 0):
    """The affine map a sequence applies to its entering state.

    The state update is affine in S (mhpq.cn/news/56770, "KDA 到底在算什么"), so
    the state after a sequence is S_out = M S_in + S~ with M [dk, dk] the
    product of the per-token transitions (I - b k k^T) Diag(alpha) and S~
    [dk, dv] the state reached from S_in = 0.  Here both come straight from
    the recurrence: S~ is the final state from zeros, M the final state from
    the identity with every v set to zero (blog.higcp.com "猜想：K3 可能是最适合
    TPU 的 MoE 架构", section "第二层": each device summarises its segment by
    such an affine map before the all-gather).

    Returns ``(M [N, H, dk, dk], S~ [N, H, dk, dv])`` in float64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, dk = q.shape
    cu = np.asarray(cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
                    dtype=np.int64)
    N = cu.shape[0] - 1
    _, s_tilde, _ = recurrent(q, k, v, z, beta, cu, None, eps=eps, threads=threads,
                              a_log=a_log)
    eye = np.broadcast_to(np.eye(dk), (N, H, dk, dk)).copy()
    _, m, _ = recurrent(q, k, np.zeros((T, H, dk)), z, beta, cu, eye, eps=eps,
                        threads=threads, a_log=a_log)
    return m, s_tilde


def state_scan(transitions, offsets, initial_state=None, count=None):
    """Apply the first ``count`` affine maps in order to the initial state:
    S <- M_i S + S~_i for i = 0 .. count-1 (blog.higcp.com "猜想：K3 可能是最适合
    TPU 的 MoE 架构", section "第二层": the prefix scan that gives each device
    the state entering its segment).  transitions [R, N, H, dk, dk], offsets
    [R, N, H, dk, dv], initial_state [N, H, dk, dv] or None (zeros).
    Returns float64 [N, H, dk, dv]."""
    m, s = _f64(transitions), _f64(offsets)
    count = m.shape[0] if count is None else int(count)
    state = np.zeros(s.shape[1:]) if initial_state is None else _f64(initial_state).copy()
    for i in range(count):
        state = np.matmul(m[i], state) + s[i]
    return state
from .output_norm import rms_norm  # noqa: E402,F401
