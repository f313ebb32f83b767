"""Python binding of libkda (Kimi Delta Attention on GB300).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``_lib/libkda.so``, reached through its C ABI (``include/kda.h``)
with ctypes.  PyTorch supplies device memory and streams.  There is no CPU
fallback: if the library is missing or a call fails, these functions raise.

Entry points (same names as the C ABI, without the ``kda_`` prefix):
    chunk_fwd      -- chunked prefill over a packed variable-length batch
    recurrent_fwd  -- token-by-token prefill (the GPU reference path)
    decode_step    -- one token for each live request, state updated in place
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["chunk_fwd", "chunk_fwd_noalloc", "recurrent_fwd", "decode_step",
           "chunk_fwd_workspace_size", "NOALLOC_SCRATCH_BYTES",
           "get_device_error", "status_string", "KDAError", "load", "LIB_PATH",
           "checkpoint_offsets", "decode_window", "decode_replay", "decode_replay_window",
           "recurrent_bwd", "recurrent_bwd_workspace_size", "short_conv", "chunk_fwd_host",
           "chunk_fwd_host_workspace_size", "chunk_fwd_summary",
           "chunk_fwd_summary_workspace_size", "state_scan", "decode_step_fused",
           "decode_replay_window_fused", "chunk_fwd_fused", "chunk_bwd",
           "chunk_bwd_workspace_size", "EXPORTED_SYMBOLS"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libkda.so")

KDA_OK = 0
KDA_F32, KDA_BF16 = 0, 1
_STATUS = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARGUMENT", 2: "KDA_ERR_UNSUPPORTED",
           3: "KDA_ERR_CUDA", 4: "KDA_ERR_TIMEOUT", 5: "KDA_ERR_DEVICE_CHECK"}

#: Every function include/kda.h declares.
EXPORTED_SYMBOLS = ("kda_chunk_fwd", "kda_chunk_fwd_workspace_size", "kda_recurrent_fwd",
                    "kda_decode_step", "kda_decode_window", "kda_decode_replay",
                    "kda_decode_replay_window", "kda_status_string", "kda_get_device_error",
                    "kda_chunk_fwd_noalloc", "kda_testing_inject_wait_timeout",
                    "kda_recurrent_bwd", "kda_recurrent_bwd_workspace_size", "kda_short_conv",
                    "kda_chunk_fwd_host", "kda_chunk_fwd_host_workspace_size",
                    "kda_chunk_fwd_summary", "kda_chunk_fwd_summary_workspace_size",
                    "kda_state_scan", "kda_decode_step_fused",
                    "kda_decode_replay_window_fused", "kda_chunk_fwd_fused", "kda_chunk_bwd",
                    "kda_chunk_bwd_workspace_size")

#: Size of the library's own scratch array used by chunk_fwd_noalloc
#: (KDA_NOALLOC_SCRATCH_BYTES in include/kda.h).
NOALLOC_SCRATCH_BYTES = 32 << 20


class KDAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where} failed: {_STATUS.get(status, status)}")


class KdaDesc(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("io_dtype", ctypes.c_int32), ("cu_seqlens_host", ctypes.POINTER(ctypes.c_int32)),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("a_log", ctypes.c_void_p), ("checkpoints", ctypes.c_void_p),
                ("checkpoint_offsets", ctypes.c_void_p), ("checkpoint_every", ctypes.c_int32),
                ("gate_per_head", ctypes.c_int32)]


class KdaFusion(ctypes.Structure):
    _fields_ = [("conv_width", ctypes.c_int32), ("conv_weight_q", ctypes.c_void_p),
                ("conv_weight_k", ctypes.c_void_p), ("conv_state_q", ctypes.c_void_p),
                ("conv_state_k", ctypes.c_void_p), ("out_norm_weight", ctypes.c_void_p),
                ("out_norm_eps", ctypes.c_float)]


_lib = None
_lock = threading.Lock()


def load() -> ctypes.CDLL:
    """Load libkda.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libkda.so not found at {LIB_PATH}; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        vp, dp = ctypes.c_void_p, ctypes.POINTER(KdaDesc)
        for name in ("kda_chunk_fwd", "kda_recurrent_fwd", "kda_chunk_fwd_noalloc"):
            f = getattr(lib, name)
            f.restype = ctypes.c_int
            f.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.kda_decode_step.restype = ctypes.c_int
        lib.kda_decode_step.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.kda_chunk_fwd_workspace_size.restype = ctypes.c_int
        lib.kda_chunk_fwd_workspace_size.argtypes = [dp, ctypes.POINTER(ctypes.c_size_t)]
        for f in (lib.kda_recurrent_bwd, lib.kda_chunk_bwd):
            f.restype = ctypes.c_int
            f.argtypes = [dp] + [vp] * 16
        lib.kda_chunk_fwd_host.restype = ctypes.c_int
        lib.kda_chunk_fwd_host.argtypes = [dp, ctypes.c_int32] + [vp] * 10
        lib.kda_chunk_fwd_host_workspace_size.restype = ctypes.c_int
        lib.kda_chunk_fwd_host_workspace_size.argtypes = [dp, ctypes.POINTER(ctypes.c_size_t)]
        lib.kda_short_conv.restype = ctypes.c_int
        lib.kda_short_conv.argtypes = [dp, ctypes.c_int32] + [vp] * 7
        for f in (lib.kda_recurrent_bwd_workspace_size, lib.kda_chunk_bwd_workspace_size):
            f.restype = ctypes.c_int
            f.argtypes = [dp, ctypes.POINTER(ctypes.c_size_t)]
        lib.kda_chunk_fwd_summary.restype = ctypes.c_int
        lib.kda_chunk_fwd_summary.argtypes = [dp] + [vp] * 9
        lib.kda_chunk_fwd_summary_workspace_size.restype = ctypes.c_int
        lib.kda_chunk_fwd_summary_workspace_size.argtypes = [dp, ctypes.POINTER(ctypes.c_size_t)]
        lib.kda_state_scan.restype = ctypes.c_int
        lib.kda_state_scan.argtypes = [dp, ctypes.c_int32] + [vp] * 5
        fp = ctypes.POINTER(KdaFusion)
        lib.kda_decode_step_fused.restype = ctypes.c_int
        lib.kda_decode_step_fused.argtypes = [dp, fp] + [vp] * 8
        lib.kda_chunk_fwd_fused.restype = ctypes.c_int
        lib.kda_chunk_fwd_fused.argtypes = [dp, fp] + [vp] * 10
        lib.kda_decode_replay_window_fused.restype = ctypes.c_int
        lib.kda_decode_replay_window_fused.argtypes = (
            [dp, fp, ctypes.c_int32] + [vp] * 6 + [ctypes.c_int32] + [vp] * 8)
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_testing_inject_wait_timeout.restype = None
        lib.kda_testing_inject_wait_timeout.argtypes = [ctypes.c_int]
        lib.kda_get_device_error.restype = ctypes.c_int
        lib.kda_get_device_error.argtypes = [vp]
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_tensor(name, t, dtype, shape, device):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.device != device or not t.is_cuda:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_host(name, t, dtype, shape):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a host (CPU) tensor, got {t.device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _io_code(dtype):
    if dtype == torch.float32:
        return KDA_F32
    if dtype == torch.bfloat16:
        return KDA_BF16
    raise ValueError(f"q/k/v must be float32 or bfloat16, got {dtype}")


def make_desc(num_seqs, total_tokens, num_heads, dk, dv, io_dtype, cu_seqlens_host=None,
              workspace=None, a_log=None):
    """Build the C descriptor.  Returns (desc, keepalive) -- keep both alive
    for the duration of the call.  a_log: optional device fp32 [H] tensor, the
    per-head gate log-scale (g = -5 sigmoid(e^{A_h} z))."""
    d = KdaDesc()
    d.num_seqs, d.total_tokens, d.num_heads = int(num_seqs), int(total_tokens), int(num_heads)
    d.dk, d.dv, d.io_dtype = int(dk), int(dv), int(io_dtype)
    keep = None
    if cu_seqlens_host is not None:
        keep = (ctypes.c_int32 * len(cu_seqlens_host))(*[int(x) for x in cu_seqlens_host])
        d.cu_seqlens_host = ctypes.cast(keep, ctypes.POINTER(ctypes.c_int32))
    if workspace is not None:
        d.workspace = ctypes.c_void_p(workspace.data_ptr())
        d.workspace_bytes = workspace.numel() * workspace.element_size()
    if a_log is not None:
        d.a_log = ctypes.c_void_p(a_log.data_ptr())
    return d, keep


def checkpoint_offsets(cu_seqlens_host, every):
    """Exclusive prefix sums of floor(len_n / every) over the sequences: where
    each sequence's state checkpoints start (and, last, how many there are)."""
    cu = [int(x) for x in cu_seqlens_host]
    offs = [0]
    for n in range(len(cu) - 1):
        offs.append(offs[-1] + (cu[n + 1] - cu[n]) // every)
    return offs


def _prefill(name, q, k, v, z, beta, cu_seqlens, initial_state, out, final_state,
             output_final_state, cu_seqlens_host, workspace, stream, a_log=None,
             checkpoint_every=0, checkpoints=None, fusion=None):
    lib = load()
    if q.dim() != 3:
        raise ValueError("q must be [T_tot, H, dk]")
    T, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    dev = q.device
    _check_tensor("q", q, q.dtype, (T, H, dk), dev)
    _check_tensor("k", k, q.dtype, (T, H, dk), dev)
    _check_tensor("v", v, q.dtype, (T, H, dv), dev)
    per_head = z.dim() == 2  # [T, H]: one gate per head (scalar alpha)
    _check_tensor("z", z, torch.float32, (T, H) if per_head else (T, H, dk), dev)
    _check_tensor("beta", beta, torch.float32, (T, H), dev)
    _check_tensor("cu_seqlens", cu_seqlens, torch.int32, (N + 1,), dev)
    if initial_state is not None:
        _check_tensor("initial_state", initial_state, torch.float32, (N, H, dk, dv), dev)
    if a_log is not None:
        _check_tensor("a_log", a_log, torch.float32, (H,), dev)
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    _check_tensor("out", out, q.dtype, (T, H, dv), dev)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    if final_state is not None:
        _check_tensor("final_state", final_state, torch.float32, (N, H, dk, dv), dev)
    desc, keep = make_desc(N, T, H, dk, dv, _io_code(q.dtype), cu_seqlens_host, workspace, a_log)
    desc.gate_per_head = 1 if per_head else 0
    offs_dev = None
    if checkpoint_every:
        if cu_seqlens_host is None:
            raise ValueError("checkpoint_every needs cu_seqlens_host (to place the checkpoints)")
        offs = checkpoint_offsets(cu_seqlens_host, checkpoint_every)
        if checkpoints is None:
            checkpoints = torch.empty((offs[-1], H, dk, dv), dtype=torch.float32, device=dev)
        _check_tensor("checkpoints", checkpoints, torch.float32, (offs[-1], H, dk, dv), dev)
        offs_dev = torch.tensor(offs, dtype=torch.int32, device=dev)
        desc.checkpoint_every = int(checkpoint_every)
        desc.checkpoints = ctypes.c_void_p(checkpoints.data_ptr()) if offs[-1] else \
            ctypes.c_void_p(offs_dev.data_ptr())  # any valid pointer when there are none
        desc.checkpoint_offsets = ctypes.c_void_p(offs_dev.data_ptr())
    pre = (ctypes.byref(desc),) if fusion is None else (ctypes.byref(desc), ctypes.byref(fusion))
    with torch.cuda.device(dev):
        st = getattr(lib, name)(*pre, _ptr(q), _ptr(k), _ptr(v), _ptr(z),
                                _ptr(beta), _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
                                _ptr(final_state), _stream_handle(stream))
    del keep
    if st != KDA_OK:
        raise KDAError(st, name)
    if checkpoint_every:
        return out, final_state, checkpoints
    return out, final_state


def chunk_fwd(q, k, v, z, beta, cu_seqlens, initial_state=None, *, out=None, final_state=None,
              output_final_state=True, cu_seqlens_host=None, workspace=None, stream=None,
              a_log=None, checkpoint_every=0, checkpoints=None):
    """Chunked KDA prefill (``kda_chunk_fwd``).  Returns (out, final_state), or
    (out, final_state, checkpoints) when ``checkpoint_every`` > 0.
    ``z``: [T, H, dk] gate logits (one per key channel), or [T, H] for one gate
    per head (the scalar-alpha, Gated DeltaNet case).
    ``a_log``: optional fp32 [H] per-head gate log-scale A (g = -5 sigmoid(e^A z)).
    ``checkpoint_every``: a multiple of 64; the state after every that many
    tokens of each sequence, [sum_n floor(len_n / E), H, dk, dv] fp32 in
    sequence order (``checkpoint_offsets`` gives where each sequence starts).

    ``workspace``: a device tensor of scratch (at least
    ``chunk_fwd_workspace_size`` bytes, 256-byte aligned) that lets long
    sequences be split across SMs, ``"auto"`` to allocate it here with torch,
    or None (no split).  Results agree either way within the tolerances."""
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be a tensor, 'auto' or None")
        workspace = None
        if cu_seqlens_host is not None:
            nbytes = chunk_fwd_workspace_size(len(cu_seqlens_host) - 1, q.shape[0], q.shape[1],
                                              q.shape[2], v.shape[-1], q.dtype, cu_seqlens_host)
            if nbytes:
                workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    return _prefill("kda_chunk_fwd", q, k, v, z, beta, cu_seqlens, initial_state, out,
                    final_state, output_final_state, cu_seqlens_host, workspace, stream, a_log,
                    checkpoint_every, checkpoints)


def chunk_fwd_fused(q, k, v, z, beta, cu_seqlens, initial_state=None, *, conv_weight_q,
                    conv_weight_k, conv_state_q=None, conv_state_k=None, out=None,
                    final_state=None, output_final_state=True, cu_seqlens_host=None,
                    workspace=None, stream=None, a_log=None, checkpoint_every=0,
                    checkpoints=None):
    """``kda_chunk_fwd_fused``: the chunked prefill over RAW q, k, with the short
    convolution + Swish (conv_weight_* [H, dk, W]) fused into the kernel.
    conv_state_* [N, H, dk, W-1] (required for W > 1) are read as each
    sequence's inputs before its start and overwritten with its last W-1 raw
    inputs.  Other arguments and the return value as ``chunk_fwd``."""
    T, H, dk = q.shape
    N = cu_seqlens.numel() - 1
    f = _fusion(H, dk, v.shape[-1], N, q.device, conv_weight_q, conv_weight_k, conv_state_q,
                conv_state_k, None, 0.0)
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be a tensor, 'auto' or None")
        workspace = None
        if cu_seqlens_host is not None:
            nbytes = chunk_fwd_workspace_size(N, T, H, dk, v.shape[-1], q.dtype, cu_seqlens_host)
            if nbytes:
                workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    return _prefill("kda_chunk_fwd_fused", q, k, v, z, beta, cu_seqlens, initial_state, out,
                    final_state, output_final_state, cu_seqlens_host, workspace, stream, a_log,
                    checkpoint_every, checkpoints, fusion=f)


def recurrent_fwd(q, k, v, z, beta, cu_seqlens, initial_state=None, *, out=None,
                  final_state=None, output_final_state=True, cu_seqlens_host=None, stream=None,
                  a_log=None, checkpoint_every=0, checkpoints=None):
    """Token-by-token KDA prefill (``kda_recurrent_fwd``).  Returns (out, final_state)
    (and the checkpoints, as ``chunk_fwd``).  ``initial_state``, ``final_state``
    and ``checkpoints`` must start on a 16-byte boundary (the library refuses
    them otherwise: KDA_ERR_INVALID_ARGUMENT)."""
    return _prefill("kda_recurrent_fwd", q, k, v, z, beta, cu_seqlens, initial_state, out,
                    final_state, output_final_state, cu_seqlens_host, None, stream, a_log,
                    checkpoint_every, checkpoints)


def chunk_fwd_noalloc(q, k, v, z, beta, cu_seqlens, initial_state=None, *, out=None,
                      final_state=None, output_final_state=True, cu_seqlens_host=None,
                      stream=None, a_log=None, checkpoint_every=0, checkpoints=None):
    """``kda_chunk_fwd_noalloc``: the chunked prefill for callers that cannot
    allocate device memory; its scratch for splitting long sequences is an
    array inside the library (NOALLOC_SCRATCH_BYTES).  Pass ``out`` and
    ``final_state`` to keep this wrapper from allocating them with torch.
    Returns (out, final_state)."""
    return _prefill("kda_chunk_fwd_noalloc", q, k, v, z, beta, cu_seqlens, initial_state, out,
                    final_state, output_final_state, cu_seqlens_host, None, stream, a_log,
                    checkpoint_every, checkpoints)


def chunk_fwd_workspace_size(num_seqs, total_tokens, num_heads, dk, dv, dtype, cu_seqlens_host):
    """Bytes of device scratch that let ``chunk_fwd`` split long sequences."""
    desc, keep = make_desc(num_seqs, total_tokens, num_heads, dk, dv, _io_code(dtype),
                           cu_seqlens_host)
    n = ctypes.c_size_t(0)
    st = load().kda_chunk_fwd_workspace_size(ctypes.byref(desc), ctypes.byref(n))
    del keep
    if st != KDA_OK:
        raise KDAError(st, "kda_chunk_fwd_workspace_size")
    return int(n.value)


def chunk_fwd_host_workspace_size(num_seqs, total_tokens, num_heads, dk, dv, dtype,
                                  gate_per_head=False):
    """Bytes of device staging area ``chunk_fwd_host`` needs."""
    desc, keep = make_desc(num_seqs, total_tokens, num_heads, dk, dv, _io_code(dtype))
    desc.gate_per_head = 1 if gate_per_head else 0
    n = ctypes.c_size_t(0)
    st = load().kda_chunk_fwd_host_workspace_size(ctypes.byref(desc), ctypes.byref(n))
    if st != KDA_OK:
        raise KDAError(st, "kda_chunk_fwd_host_workspace_size")
    return int(n.value)


def chunk_fwd_host(q, k, v, z, beta, cu_seqlens_host, initial_state=None, *, out=None,
                   final_state=None, output_final_state=True, workspace=None, groups=8,
                   device=None, stream=None, a_log=None):
    """``kda_chunk_fwd_host``: the chunked prefill over HOST tensors (pinned for
    the copies to overlap the kernels).  q, k, v, z, beta, initial_state and the
    returned out / final_state live in host memory; ``workspace`` is a device
    uint8 tensor of ``chunk_fwd_host_workspace_size`` bytes (allocated here when
    None).  Returns (out, final_state) once they are written (the call
    synchronises the stream)."""
    lib = load()
    T, H, dk = q.shape
    dv = v.shape[-1]
    cu = [int(c) for c in cu_seqlens_host]
    N = len(cu) - 1
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    per_head = z.dim() == 2
    _check_host("q", q, q.dtype, (T, H, dk))
    _check_host("k", k, q.dtype, (T, H, dk))
    _check_host("v", v, q.dtype, (T, H, dv))
    _check_host("z", z, torch.float32, (T, H) if per_head else (T, H, dk))
    _check_host("beta", beta, torch.float32, (T, H))
    if initial_state is not None:
        _check_host("initial_state", initial_state, torch.float32, (N, H, dk, dv))
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype).pin_memory()
    _check_host("out", out, q.dtype, (T, H, dv))
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32).pin_memory()
    if final_state is not None:
        _check_host("final_state", final_state, torch.float32, (N, H, dk, dv))
    if a_log is not None:
        _check_tensor("a_log", a_log, torch.float32, (H,), dev)
    if workspace is None:
        nbytes = chunk_fwd_host_workspace_size(N, T, H, dk, dv, q.dtype, per_head)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    desc, keep = make_desc(N, T, H, dk, dv, _io_code(q.dtype), None, workspace, a_log)
    desc.gate_per_head = 1 if per_head else 0
    cu_arr = (ctypes.c_int32 * len(cu))(*cu)
    with torch.cuda.device(dev):
        st = lib.kda_chunk_fwd_host(ctypes.byref(desc), int(groups), _ptr(q), _ptr(k), _ptr(v),
                                    _ptr(z), _ptr(beta), _ptr(initial_state), cu_arr, _ptr(out),
                                    _ptr(final_state), _stream_handle(stream))
        if st == KDA_OK:
            (stream or torch.cuda.current_stream()).synchronize()
    del keep
    if st != KDA_OK:
        raise KDAError(st, "kda_chunk_fwd_host")
    return out, final_state


def short_conv(x, weight, cu_seqlens, conv_state=None, *, out=None, final_state=None,
               output_final_state=True, stream=None):
    """The Q/K preprocessing (``kda_short_conv``): depthwise causal convolution
    of width W = weight.shape[-1] (1..4) over each sequence, then Swish.
    x [T, H, D] (bf16 or fp32), weight [H, D, W] fp32, conv_state [N, H, D,
    W - 1] fp32 or None (zeros).  Returns (y, final conv state or None);
    ``final_state`` may be ``conv_state`` itself (updated in place)."""
    lib = load()
    T, H, D = x.shape
    W = weight.shape[-1]
    N = cu_seqlens.numel() - 1
    dev = x.device
    _check_tensor("x", x, x.dtype, (T, H, D), dev)
    _check_tensor("weight", weight, torch.float32, (H, D, W), dev)
    _check_tensor("cu_seqlens", cu_seqlens, torch.int32, (N + 1,), dev)
    if conv_state is not None:
        _check_tensor("conv_state", conv_state, torch.float32, (N, H, D, W - 1), dev)
    if out is None:
        out = torch.empty_like(x)
    _check_tensor("out", out, x.dtype, (T, H, D), dev)
    if final_state is None and output_final_state and W > 1:
        final_state = torch.empty((N, H, D, W - 1), dtype=torch.float32, device=dev)
    if final_state is not None:
        _check_tensor("final_state", final_state, torch.float32, (N, H, D, W - 1), dev)
    desc, keep = make_desc(N, T, H, D, D, _io_code(x.dtype))
    with torch.cuda.device(dev):
        st = lib.kda_short_conv(ctypes.byref(desc), int(W), _ptr(x), _ptr(weight),
                                _ptr(conv_state), _ptr(cu_seqlens), _ptr(out),
                                _ptr(final_state), _stream_handle(stream))
    del keep
    if st != KDA_OK:
        raise KDAError(st, "kda_short_conv")
    return out, final_state


def _bwd_workspace_size(fn, num_heads, dtype, cu_seqlens_host, dk, dv):
    N = len(cu_seqlens_host) - 1
    desc, keep = make_desc(N, int(cu_seqlens_host[-1]), num_heads, dk, dv, _io_code(dtype),
                           cu_seqlens_host)
    n = ctypes.c_size_t(0)
    st = getattr(load(), fn)(ctypes.byref(desc), ctypes.byref(n))
    del keep
    if st != KDA_OK:
        raise KDAError(st, fn)
    return int(n.value)


def recurrent_bwd_workspace_size(num_heads, dtype, cu_seqlens_host, dk=128, dv=128):
    """Bytes of device workspace ``recurrent_bwd`` needs."""
    return _bwd_workspace_size("kda_recurrent_bwd_workspace_size", num_heads, dtype,
                               cu_seqlens_host, dk, dv)


def chunk_bwd_workspace_size(num_heads, dtype, cu_seqlens_host, dk=128, dv=128):
    """Bytes of device workspace ``chunk_bwd`` needs."""
    return _bwd_workspace_size("kda_chunk_bwd_workspace_size", num_heads, dtype,
                               cu_seqlens_host, dk, dv)


def _bwd(fn, ws_size, q, k, v, z, beta, cu_seqlens, initial_state, d_out, d_final,
         cu_seqlens_host, a_log, workspace, grads, stream):
    lib = load()
    T, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    dev = q.device
    _check_tensor("q", q, q.dtype, (T, H, dk), dev)
    _check_tensor("k", k, q.dtype, (T, H, dk), dev)
    _check_tensor("v", v, q.dtype, (T, H, dv), dev)
    per_head = z.dim() == 2
    zshape = (T, H) if per_head else (T, H, dk)
    _check_tensor("z", z, torch.float32, zshape, dev)
    _check_tensor("beta", beta, torch.float32, (T, H), dev)
    _check_tensor("cu_seqlens", cu_seqlens, torch.int32, (N + 1,), dev)
    _check_tensor("d_out", d_out, q.dtype, (T, H, dv), dev)
    if initial_state is not None:
        _check_tensor("initial_state", initial_state, torch.float32, (N, H, dk, dv), dev)
    if d_final is not None:
        _check_tensor("d_final", d_final, torch.float32, (N, H, dk, dv), dev)
    if a_log is not None:
        _check_tensor("a_log", a_log, torch.float32, (H,), dev)
    if grads is None:
        f32 = dict(dtype=torch.float32, device=dev)
        grads = (torch.empty((T, H, dk), **f32), torch.empty((T, H, dk), **f32),
                 torch.empty((T, H, dv), **f32), torch.empty(zshape, **f32),
                 torch.empty((T, H), **f32), torch.empty((N, H, dk, dv), **f32))
    shapes = ((T, H, dk), (T, H, dk), (T, H, dv), zshape, (T, H), (N, H, dk, dv))
    for name, g, shp in zip(("dq", "dk", "dv", "dz", "dbeta", "d_initial"), grads, shapes):
        _check_tensor(name, g, torch.float32, shp, dev)
    if workspace is None:
        nbytes = ws_size(H, q.dtype, cu_seqlens_host, dk, dv)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    desc, keep = make_desc(N, T, H, dk, dv, _io_code(q.dtype), cu_seqlens_host, workspace, a_log)
    desc.gate_per_head = 1 if per_head else 0
    with torch.cuda.device(dev):
        st = getattr(lib, fn)(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(z),
                              _ptr(beta), _ptr(initial_state), _ptr(cu_seqlens), _ptr(d_out),
                              _ptr(d_final), *[_ptr(g) for g in grads], _stream_handle(stream))
    del keep
    if st != KDA_OK:
        raise KDAError(st, fn)
    return grads


def recurrent_bwd(q, k, v, z, beta, cu_seqlens, initial_state, d_out, d_final=None, *,
                  cu_seqlens_host, a_log=None, workspace=None, grads=None, stream=None):
    """Reverse mode of the prefill (``kda_recurrent_bwd``): given dL/d out and
    dL/d final_state (None: zeros), returns (dq, dk, dv, dz, dbeta,
    d_initial_state), fp32, for the inputs of the forward call (same q, k, v,
    z, beta, cu_seqlens, initial_state and a_log; any supported dk, dv).  ``z`` [T, H]
    (one gate per head) gives dz [T, H].  ``cu_seqlens_host`` is required; ``workspace`` (a device
    tensor of ``recurrent_bwd_workspace_size`` bytes) is allocated here when
    None; ``grads`` may give the six output tensors to fill."""
    return _bwd("kda_recurrent_bwd", recurrent_bwd_workspace_size, q, k, v, z, beta, cu_seqlens,
                initial_state, d_out, d_final, cu_seqlens_host, a_log, workspace, grads, stream)


def chunk_bwd(q, k, v, z, beta, cu_seqlens, initial_state, d_out, d_final=None, *,
              cu_seqlens_host, a_log=None, workspace=None, grads=None, stream=None):
    """The same gradients as ``recurrent_bwd`` from the chunked form on the
    tensor cores (``kda_chunk_bwd``; tf32 products, fp32 states): arguments and
    results as for ``recurrent_bwd``, workspace ``chunk_bwd_workspace_size``."""
    return _bwd("kda_chunk_bwd", chunk_bwd_workspace_size, q, k, v, z, beta, cu_seqlens,
                initial_state, d_out, d_final, cu_seqlens_host, a_log, workspace, grads, stream)


def decode_step(q, k, v, z, beta, state, *, out=None, stream=None, a_log=None):
    """One decode step (``kda_decode_step``); ``state`` is updated in place.
    q, k: [N, H, dk]; v: [N, H, dv]; z: [N, H, dk] fp32; beta: [N, H] fp32;
    state: [N, H, dk, dv] fp32; a_log: optional [H] fp32 gate log-scale.
    Returns out [N, H, dv]."""
    lib = load()
    N, H, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    _check_tensor("q", q, q.dtype, (N, H, dk), dev)
    _check_tensor("k", k, q.dtype, (N, H, dk), dev)
    _check_tensor("v", v, q.dtype, (N, H, dv), dev)
    per_head = z.dim() == 2  # [N, H]: one gate per head
    _check_tensor("z", z, torch.float32, (N, H) if per_head else (N, H, dk), dev)
    _check_tensor("beta", beta, torch.float32, (N, H), dev)
    _check_tensor("state", state, torch.float32, (N, H, dk, dv), dev)
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=dev)
    _check_tensor("out", out, q.dtype, (N, H, dv), dev)
    if a_log is not None:
        _check_tensor("a_log", a_log, torch.float32, (H,), dev)
    desc, _ = make_desc(N, N, H, dk, dv, _io_code(q.dtype), a_log=a_log)
    desc.gate_per_head = 1 if per_head else 0
    with torch.cuda.device(dev):
        st = lib.kda_decode_step(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(z),
                                 _ptr(beta), _ptr(state), _ptr(out), _stream_handle(stream))
    if st != KDA_OK:
        raise KDAError(st, "kda_decode_step")
    return out


def _window_args(q, k, v, z, beta, state):
    """Shapes of a speculative-decoding window: q, k [B, W, H, dk]; v [B, W, H, dv];
    z [B, W, H, dk] fp32; beta [B, W, H] fp32; state [B, H, dk, dv] fp32."""
    B, W, H, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    _check_tensor("q", q, q.dtype, (B, W, H, dk), dev)
    _check_tensor("k", k, q.dtype, (B, W, H, dk), dev)
    _check_tensor("v", v, q.dtype, (B, W, H, dv), dev)
    per_head = z.dim() == 3  # [B, W, H]: one gate per head
    _check_tensor("z", z, torch.float32, (B, W, H) if per_head else (B, W, H, dk), dev)
    _check_tensor("beta", beta, torch.float32, (B, W, H), dev)
    _check_tensor("state", state, torch.float32, (B, H, dk, dv), dev)
    return B, W, H, dk, dv, dev, per_head


def decode_window(q, k, v, z, beta, state, *, out=None, stream=None, a_log=None):
    """``kda_decode_window``: outputs [B, W, H, dv] of W draft tokens per request
    from the committed ``state`` (not changed); draft i sees drafts 0..i."""
    lib = load()
    B, W, H, dk, dv, dev, per_head = _window_args(q, k, v, z, beta, state)
    if out is None:
        out = torch.empty((B, W, H, dv), dtype=q.dtype, device=dev)
    _check_tensor("out", out, q.dtype, (B, W, H, dv), dev)
    if a_log is not None:
        _check_tensor("a_log", a_log, torch.float32, (H,), dev)
    desc, _ = make_desc(B, B * W, H, dk, dv, _io_code(q.dtype), a_log=a_log)
    desc.gate_per_head = 1 if per_head else 0
    with torch.cuda.device(dev):
        st = lib.kda_decode_window(ctypes.byref(desc), ctypes.c_int32(W), _ptr(q), _ptr(k),
                                   _ptr(v), _ptr(z), _ptr(beta), _ptr(state), _ptr(out),
                                   _stream_handle(stream))
    if st != KDA_OK:
        raise KDAError(st, "kda_decode_window")
    return out


def decode_replay(q, k, v, z, beta, accept_len, state, *, stream=None, a_log=None):
    """``kda_decode_replay``: apply the first accept_len[b] drafts of the cached
    window to each request's ``state`` (in place).  accept_len: int32 [B] on
    the device."""
    lib = load()
    B, W, H, dk, dv, dev, per_head = _window_args(q, k, v, z, beta, state)
    _check_tensor("accept_len", accept_len, torch.int32, (B,), dev)
    if a_log is not None:
        _check_tensor("a_log", a_log, torch.float32, (H,), dev)
    desc, _ = make_desc(B, B * W, H, dk, dv, _io_code(q.dtype), a_log=a_log)
    desc.gate_per_head = 1 if per_head else 0
    with torch.cuda.device(dev):
        st = lib.kda_decode_replay(ctypes.byref(desc), ctypes.c_int32(W), _ptr(q), _ptr(k),
                                   _ptr(v), _ptr(z), _ptr(beta), _ptr(accept_len), _ptr(state),
                                   _stream_handle(stream))
    if st != KDA_OK:
        raise KDAError(st, "kda_decode_replay")
    return state


def decode_replay_window(prev, accept_len, q, k, v, z, beta, state, *, out=None, stream=None,
                         a_log=None):
    """``kda_decode_replay_window``: replay the first accept_len[b] drafts of the
    previous window ``prev`` = (q, k, v, z, beta) into ``state`` (in place),
    then return the outputs [B, W, H, dv] of the new window from it."""
    lib = load()
    B, W, H, dk, dv, dev, per_head = _window_args(q, k, v, z, beta, state)
    pq, pk, pv, pz, pb = prev
    Bp, Wp, Hp, dkp, dvp, _, per_head_p = _window_args(pq, pk, pv, pz, pb, state)
    if (Bp, Hp, dkp, dvp, per_head_p) != (B, H, dk, dv, per_head) or pq.dtype != q.dtype:
        raise ValueError("the previous window must match the new one but for its length")
    _check_tensor("accept_len", accept_len, torch.int32, (B,), dev)
    if out is None:
        out = torch.empty((B, W, H, dv), dtype=q.dtype, device=dev)
    _check_tensor("out", out, q.dtype, (B, W, H, dv), dev)
    if a_log is not None:
        _check_tensor("a_log", a_log, torch.float32, (H,), dev)
    desc, _ = make_desc(B, B * W, H, dk, dv, _io_code(q.dtype), a_log=a_log)
    desc.gate_per_head = 1 if per_head else 0
    with torch.cuda.device(dev):
        st = lib.kda_decode_replay_window(
            ctypes.byref(desc), ctypes.c_int32(Wp), _ptr(pq), _ptr(pk), _ptr(pv), _ptr(pz),
            _ptr(pb), _ptr(accept_len), ctypes.c_int32(W), _ptr(q), _ptr(k), _ptr(v), _ptr(z),
            _ptr(beta), _ptr(state), _ptr(out), _stream_handle(stream))
    if st != KDA_OK:
        raise KDAError(st, "kda_decode_replay_window")
    return out


def _fusion(H, dk, dv, B, dev, conv_weight_q, conv_weight_k, conv_state_q, conv_state_k,
            out_norm_weight, out_norm_eps):
    """The kda_fusion_t of the fused decode calls (None when nothing is fused)."""
    f = KdaFusion()
    if conv_weight_q is not None or conv_weight_k is not None:
        W = conv_weight_q.shape[-1]
        _check_tensor("conv_weight_q", conv_weight_q, torch.float32, (H, dk, W), dev)
        _check_tensor("conv_weight_k", conv_weight_k, torch.float32, (H, dk, W), dev)
        f.conv_width = W
        f.conv_weight_q = ctypes.c_void_p(conv_weight_q.data_ptr())
        f.conv_weight_k = ctypes.c_void_p(conv_weight_k.data_ptr())
        if W > 1:
            _check_tensor("conv_state_q", conv_state_q, torch.float32, (B, H, dk, W - 1), dev)
            _check_tensor("conv_state_k", conv_state_k, torch.float32, (B, H, dk, W - 1), dev)
            f.conv_state_q = ctypes.c_void_p(conv_state_q.data_ptr())
            f.conv_state_k = ctypes.c_void_p(conv_state_k.data_ptr())
    if out_norm_weight is not None:
        _check_tensor("out_norm_weight", out_norm_weight, torch.float32, (H, dv), dev)
        f.out_norm_weight = ctypes.c_void_p(out_norm_weight.data_ptr())
        f.out_norm_eps = float(out_norm_eps)
    return f


def decode_step_fused(q, k, v, z, beta, state, *, conv_weight_q=None, conv_weight_k=None,
                      conv_state_q=None, conv_state_k=None, out_norm_weight=None,
                      out_norm_eps=1e-6, out=None, stream=None, a_log=None):
    """``kda_decode_step_fused``: one decode step with raw q, k through the short
    convolution + Swish (conv_weight_* [H, dk, W], conv_state_* [N, H, dk, W-1],
    advanced in place) and the outputs through the per-head RMS norm
    (out_norm_weight [H, dv]).  Returns out [N, H, dv]; ``state`` is updated."""
    lib = load()
    N, H, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    _check_tensor("q", q, q.dtype, (N, H, dk), dev)
    _check_tensor("k", k, q.dtype, (N, H, dk), dev)
    _check_tensor("v", v, q.dtype, (N, H, dv), dev)
    per_head = z.dim() == 2
    _check_tensor("z", z, torch.float32, (N, H) if per_head else (N, H, dk), dev)
    _check_tensor("beta", beta, torch.float32, (N, H), dev)
    _check_tensor("state", state, torch.float32, (N, H, dk, dv), dev)
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=dev)
    _check_tensor("out", out, q.dtype, (N, H, dv), dev)
    if a_log is not None:
        _check_tensor("a_log", a_log, torch.float32, (H,), dev)
    f = _fusion(H, dk, dv, N, dev, conv_weight_q, conv_weight_k, conv_state_q, conv_state_k,
                out_norm_weight, out_norm_eps)
    desc, _ = make_desc(N, N, H, dk, dv, _io_code(q.dtype), a_log=a_log)
    desc.gate_per_head = 1 if per_head else 0
    with torch.cuda.device(dev):
        st = lib.kda_decode_step_fused(ctypes.byref(desc), ctypes.byref(f), _ptr(q), _ptr(k),
                                       _ptr(v), _ptr(z), _ptr(beta), _ptr(state), _ptr(out),
                                       _stream_handle(stream))
    if st != KDA_OK:
        raise KDAError(st, "kda_decode_step_fused")
    return out


def decode_replay_window_fused(prev, accept_len, window, state, *, conv_weight_q=None,
                               conv_weight_k=None, conv_state_q=None, conv_state_k=None,
                               out_norm_weight=None, out_norm_eps=1e-6, out=None, stream=None,
                               a_log=None):
    """``kda_decode_replay_window_fused``: replay the first accept_len[b] raw
    drafts of ``prev`` = (q, k, v, z, beta) [B, Wp, H, .] into ``state`` and the
    convolution states (in place), then the outputs [B, W, H, dv] of ``window``
    = (q, k, v, z, beta) [B, W, H, .] through the output norm.  ``prev`` or
    ``window`` may be None (no replay / no outputs; returns None then).
    ``state`` and ``out_norm_weight`` must start on a 16-byte boundary (the
    library refuses them otherwise: KDA_ERR_INVALID_ARGUMENT)."""
    lib = load()
    ref = window if window is not None else prev
    if ref is None:
        raise ValueError("prev and window cannot both be None")
    B, Wr, H, dk, dv, dev, per_head = _window_args(*ref, state)
    W = 0
    if window is not None:
        W = Wr
    Wp = 0
    if prev is not None:
        Bp, Wp, Hp, dkp, dvp, _, per_head_p = _window_args(*prev, state)
        if (Bp, Hp, dkp, dvp, per_head_p) != (B, H, dk, dv, per_head) or \
                prev[0].dtype != ref[0].dtype:
            raise ValueError("the previous window must match the new one but for its length")
        _check_tensor("accept_len", accept_len, torch.int32, (B,), dev)
    if window is not None:
        if out is None:
            out = torch.empty((B, W, H, dv), dtype=ref[0].dtype, device=dev)
        _check_tensor("out", out, ref[0].dtype, (B, W, H, dv), dev)
    if a_log is not None:
        _check_tensor("a_log", a_log, torch.float32, (H,), dev)
    f = _fusion(H, dk, dv, B, dev, conv_weight_q, conv_weight_k, conv_state_q, conv_state_k,
                out_norm_weight, out_norm_eps)
    desc, _ = make_desc(B, B * W, H, dk, dv, _io_code(ref[0].dtype), a_log=a_log)
    desc.gate_per_head = 1 if per_head else 0
    pq = prev if prev is not None else (None,) * 5
    wq = window if window is not None else (None,) * 5
    with torch.cuda.device(dev):
        st = lib.kda_decode_replay_window_fused(
            ctypes.byref(desc), ctypes.byref(f), ctypes.c_int32(Wp), *[_ptr(x) for x in pq],
            _ptr(accept_len) if prev is not None else None, ctypes.c_int32(W),
            *[_ptr(x) for x in wq], _ptr(state), _ptr(out) if window is not None else None,
            _stream_handle(stream))
    if st != KDA_OK:
        raise KDAError(st, "kda_decode_replay_window_fused")
    return out if window is not None else None


def get_device_error(stream=None) -> int:
    """Synchronise and read/clear the device error word (a kda_status_t)."""
    lib = load()
    return int(lib.kda_get_device_error(_stream_handle(stream)))


def testing_inject_wait_timeout(launches: int = 1) -> None:
    """Make the next `launches` tensor-core prefill launches of this thread hit
    an expired device wait (``kda_testing_inject_wait_timeout``)."""
    load().kda_testing_inject_wait_timeout(int(launches))


def chunk_fwd_summary_workspace_size(num_seqs, total_tokens, num_heads, dk, dv, dtype,
                                     cu_seqlens_host):
    """Bytes of device scratch that let ``chunk_fwd_summary`` split long
    sequences across SMs (0: no split would be planned)."""
    desc, keep = make_desc(num_seqs, total_tokens, num_heads, dk, dv, _io_code(dtype),
                           cu_seqlens_host)
    n = ctypes.c_size_t(0)
    st = load().kda_chunk_fwd_summary_workspace_size(ctypes.byref(desc), ctypes.byref(n))
    del keep
    if st != KDA_OK:
        raise KDAError(st, "kda_chunk_fwd_summary_workspace_size")
    return int(n.value)


def chunk_fwd_summary(q, k, v, z, beta, cu_seqlens, cu_seqlens_host, *, transition=None,
                      offset_state=None, workspace="auto", stream=None, a_log=None):
    """``kda_chunk_fwd_summary``: the affine map each sequence applies to its
    entering state, S_out = transition @ S_in + offset_state.  Returns
    (transition [N, H, dk, dk], offset_state [N, H, dk, dv]), fp32.
    ``workspace``: device scratch of ``chunk_fwd_summary_workspace_size`` bytes
    that lets long sequences split across SMs, "auto" (allocated here with
    torch) or None."""
    lib = load()
    T, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    dev = q.device
    _check_tensor("q", q, q.dtype, (T, H, dk), dev)
    _check_tensor("k", k, q.dtype, (T, H, dk), dev)
    _check_tensor("v", v, q.dtype, (T, H, dv), dev)
    per_head = z.dim() == 2
    _check_tensor("z", z, torch.float32, (T, H) if per_head else (T, H, dk), dev)
    _check_tensor("beta", beta, torch.float32, (T, H), dev)
    _check_tensor("cu_seqlens", cu_seqlens, torch.int32, (N + 1,), dev)
    if a_log is not None:
        _check_tensor("a_log", a_log, torch.float32, (H,), dev)
    if transition is None:
        transition = torch.empty((N, H, dk, dk), dtype=torch.float32, device=dev)
    if offset_state is None:
        offset_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    _check_tensor("transition", transition, torch.float32, (N, H, dk, dk), dev)
    _check_tensor("offset_state", offset_state, torch.float32, (N, H, dk, dv), dev)
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be a tensor, 'auto' or None")
        nbytes = chunk_fwd_summary_workspace_size(N, T, H, dk, dv, q.dtype, cu_seqlens_host)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None
    desc, keep = make_desc(N, T, H, dk, dv, _io_code(q.dtype), cu_seqlens_host, workspace, a_log)
    desc.gate_per_head = 1 if per_head else 0
    with torch.cuda.device(dev):
        st = lib.kda_chunk_fwd_summary(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(z),
                                       _ptr(beta), _ptr(cu_seqlens), _ptr(transition),
                                       _ptr(offset_state), _stream_handle(stream))
    del keep
    if st != KDA_OK:
        raise KDAError(st, "kda_chunk_fwd_summary")
    return transition, offset_state


def state_scan(transitions, offsets, initial_state=None, *, count=None, out=None, stream=None):
    """``kda_state_scan``: S <- transitions[i] @ S + offsets[i] for
    i = 0 .. count-1 (default: all), from ``initial_state`` (zeros if None).
    transitions [R, N, H, dk, dk], offsets [R, N, H, dk, dv] fp32 on the
    device.  Returns the state [N, H, dk, dv] (``out`` may be initial_state)."""
    lib = load()
    R, N, H, dk, dv = offsets.shape
    dev = offsets.device
    count = R if count is None else int(count)
    if not 0 <= count <= R:
        raise ValueError(f"count must be in 0..{R}")
    _check_tensor("transitions", transitions, torch.float32, (R, N, H, dk, dk), dev)
    _check_tensor("offsets", offsets, torch.float32, (R, N, H, dk, dv), dev)
    if initial_state is not None:
        _check_tensor("initial_state", initial_state, torch.float32, (N, H, dk, dv), dev)
    if out is None:
        out = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    _check_tensor("out", out, torch.float32, (N, H, dk, dv), dev)
    desc, keep = make_desc(N, 0, H, dk, dv, KDA_F32)
    with torch.cuda.device(dev):
        st = lib.kda_state_scan(ctypes.byref(desc), count, _ptr(transitions), _ptr(offsets),
                                _ptr(initial_state), _ptr(out), _stream_handle(stream))
    del keep
    if st != KDA_OK:
        raise KDAError(st, "kda_state_scan")
    return out
