"""ctypes binding to libringattn.so -- argument marshalling only.

Every step of the computation runs in the library's CUDA kernels.  PyTorch is
used for device allocation and the current stream; no function here computes
attention values.  If the library is missing the first call raises
``RuntimeError`` (there is no fallback).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libringattn.so")
_CHECKED_PATH = os.path.join(_HERE, "libringattn_checked.so")
_lib = None
_lock = threading.Lock()
_loaded = {}        # path -> CDLL

RA_OK, RA_ERR_ARG, RA_ERR_UNSUPPORTED, RA_ERR_CUDA, RA_ERR_TIMEOUT = range(5)
RA_F32, RA_BF16, RA_F32_BF16 = 0, 1, 2
RA_CONTIGUOUS, RA_STRIPED = 0, 1
_LAYOUT = {"contiguous": RA_CONTIGUOUS, "striped": RA_STRIPED}
_DTYPE = {torch.float32: RA_F32, torch.bfloat16: RA_BF16}

# exported symbol -> (restype, argtypes)
_i64, _vp, _fp, _int, _sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "ra_fwd": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _int, _int, _int, _vp, _fp, _vp]),
    "ra_fwd_step": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _int, _int, _int, _vp, _fp,
                           _vp]),
    "ra_fwd_step_fold": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _int, _int, _int, _fp,
                                _fp, _vp]),
    "ra_merge": (_int, [_vp, _fp, _vp, _fp, _i64, _i64, _int, _vp]),
    "ra_bwd_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64, _i64]),
    "ra_bwd": (_int, [_vp, _vp, _vp, _vp, _fp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                      _int, _int, _int, _vp, _sz, _vp]),
    "ra_bwd_step": (_int, [_vp, _vp, _vp, _vp, _fp, _vp, _fp, _fp, _fp, _i64, _i64, _i64, _i64, _i64, _i64, _i64,
                           _int, _int, _int, _vp, _sz, _vp]),
    "ra_bwd_noalloc": (_int, [_vp, _vp, _vp, _vp, _fp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                              _int, _int, _int, _vp]),
    "ra_decode_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64, _i64]),
    "ra_decode": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _int, _vp, _fp, _vp, _sz, _vp]),
    "ra_ffn_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64]),
    "ra_ffn": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _int, _vp, _sz, _vp]),
    "ra_set_timing_buffer": (_int, [_vp, _sz]),
    "ra_check_device_status": (_int, [_vp]),
    "ra_set_kernel_timing": (_int, [_int]),
    "ra_set_wait_test": (_int, [_int]),
    "ra_set_fwd_kernel": (_int, [_int]),
    "ra_kernel_times": (_int, [_vp, _int, ctypes.POINTER(ctypes.c_int)]),
    "ra_read_checks": (_int, [_vp, _vp]),
    "ra_last_error": (ctypes.c_char_p, []),
    "ra_version": (ctypes.c_char_p, []),
}


class RingAttnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"ringattn status {code}: {msg}")
        self.code = code


def _load(path: str):
    if path not in _loaded:
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m ring_attention_fwd_gb300.build` "
                "(there is no non-CUDA fallback)")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _loaded[path] = L
    return _loaded[path]


def lib():
    """The library every call goes through: libringattn.so unless
    ``use_checked_build(True)`` selected the bounds-checked build.  Loaded on
    first use; raises RuntimeError if it was not built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            _lib = _load(_LIB_PATH)
    return _lib


def use_checked_build(enable: bool = True):
    """Route every later call through libringattn_checked.so (every global
    index and TMA box checked against its extent, kernel events counted; see
    ``read_checks``) or, with False, back through libringattn.so.  The two
    libraries keep separate device state: buffers are plain device memory and
    work with either."""
    global _lib
    with _lock:
        _lib = _load(_CHECKED_PATH if enable else _LIB_PATH)


class CheckReport(ctypes.Structure):
    _fields_ = [("events", ctypes.c_uint64 * 8), ("violations", ctypes.c_uint32), ("first_site", ctypes.c_uint32),
                ("first_index", ctypes.c_int64), ("first_extent", ctypes.c_int64)]


CHECK_EVENTS = ("fwd_rescale_rows", "fwd_rescale_passes", "tma_boxes_checked", "accesses_checked")


def read_checks(stream=None) -> dict:
    """Synchronise and return (then clear) the checked build's record:
    event counts, and the number and first site of out-of-bounds accesses.
    Raises RingAttnError(RA_ERR_UNSUPPORTED) on the default build."""
    r = CheckReport()
    _check(lib().ra_read_checks(ctypes.addressof(r), _stream_ptr(stream)))
    out = {name: int(r.events[k]) for k, name in enumerate(CHECK_EVENTS)}
    out.update(violations=int(r.violations), first_site=hex(r.first_site), first_index=int(r.first_index),
               first_extent=int(r.first_extent))
    return out


def _check(rc: int):
    if rc != RA_OK:
        raise RingAttnError(rc, lib().ra_last_error().decode())


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype=None, shape=None, device=None):
    """Check what the C ABI cannot: the kernels take sizes from q alone, so a
    tensor of another shape, dtype or device would be read or written out of
    its bounds."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


def _need_4d(q: torch.Tensor, name: str = "q"):
    _need(q, name)
    if q.dim() != 4:
        raise ValueError(f"{name} must be [B, H, S, D], got shape {tuple(q.shape)}")
    if q.dtype not in _DTYPE:
        raise ValueError("dtype must be bfloat16 or float32")
    return q.shape


def fwd(q, k, v, n_blocks: int, causal: bool = True, layout: str = "contiguous", *,
        o=None, lse=None, stream=None):
    """Ring-order blockwise attention forward.  q, k, v: [B, H, S, D] CUDA
    tensors (bf16 or f32) in storage order.  Returns (o, lse)."""
    B, H, S, D = _need_4d(q)
    for name, t in (("k", k), ("v", v)):
        _need(t, name, q.dtype, q.shape, q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    _need(o, "o", q.dtype, q.shape, q.device)
    _need(lse, "lse", torch.float32, (B, H, S), q.device)
    _check(lib().ra_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, H, S, D, int(n_blocks),
                        int(bool(causal)), _LAYOUT[layout], _DTYPE[q.dtype], o.data_ptr(), lse.data_ptr(),
                        _stream_ptr(stream)))
    return o, lse


def fwd_step(q_i, k_j, v_j, n_blocks: int, i: int, j: int, causal: bool = True, layout: str = "contiguous", *,
             o=None, lse=None, stream=None):
    """One ring step of host i: its query block q_i [B, H, c, D] against KV
    block j (k_j, v_j of the same shape).  Returns the partial (o, lse) over
    block j's keys; chain the steps with merge()."""
    B, H, c, D = _need_4d(q_i, "q_i")
    for name, t in (("k_j", k_j), ("v_j", v_j)):
        _need(t, name, q_i.dtype, q_i.shape, q_i.device)
    if o is None:
        o = torch.empty_like(q_i)
    if lse is None:
        lse = torch.empty((B, H, c), dtype=torch.float32, device=q_i.device)
    _need(o, "o", q_i.dtype, q_i.shape, q_i.device)
    _need(lse, "lse", torch.float32, (B, H, c), q_i.device)
    _check(lib().ra_fwd_step(q_i.data_ptr(), k_j.data_ptr(), v_j.data_ptr(), B, H, c, D, int(n_blocks), int(i),
                             int(j), int(bool(causal)), _LAYOUT[layout], _DTYPE[q_i.dtype], o.data_ptr(),
                             lse.data_ptr(), _stream_ptr(stream)))
    return o, lse


def fwd_step_fold(q_i, k_j, v_j, n_blocks: int, i: int, j: int, causal: bool = True, layout: str = "contiguous",
                  *, o_acc, lse_acc, stream=None):
    """One ring step of host i folded into its running state: the partial of
    query block q_i [B, H, c, 128] (bf16) over KV block j is LogSumExp-merged
    in place into o_acc [B, H, c, 128] and lse_acc [B, H, c] (float32).
    Start a host's state with lse_acc = -inf.  Returns (o_acc, lse_acc)."""
    B, H, c, D = _need_4d(q_i, "q_i")
    for name, t in (("k_j", k_j), ("v_j", v_j)):
        _need(t, name, q_i.dtype, q_i.shape, q_i.device)
    _need(o_acc, "o_acc", torch.float32, q_i.shape, q_i.device)
    _need(lse_acc, "lse_acc", torch.float32, (B, H, c), q_i.device)
    _check(lib().ra_fwd_step_fold(q_i.data_ptr(), k_j.data_ptr(), v_j.data_ptr(), B, H, c, D, int(n_blocks), int(i),
                                  int(j), int(bool(causal)), _LAYOUT[layout], _DTYPE[q_i.dtype], o_acc.data_ptr(),
                                  lse_acc.data_ptr(), _stream_ptr(stream)))
    return o_acc, lse_acc


def merge(o_a, lse_a, o_b, lse_b, *, stream=None):
    """In-place LogSumExp merge of (o_b, lse_b) into (o_a, lse_a).  o_a and
    o_b are both float32 or both bf16, or o_a float32 and o_b bf16 (a float32
    running state folding bf16 partials)."""
    _need(o_a, "o_a")
    if o_a.dtype not in _DTYPE or o_a.dim() < 1:
        raise ValueError("o_a must be a bfloat16 or float32 tensor [..., D]")
    mixed = o_a.dtype == torch.float32 and o_b.dtype == torch.bfloat16
    _need(o_b, "o_b", o_b.dtype if mixed else o_a.dtype, o_a.shape, o_a.device)
    _need(lse_a, "lse_a", torch.float32, o_a.shape[:-1], o_a.device)
    _need(lse_b, "lse_b", torch.float32, o_a.shape[:-1], o_a.device)
    D = o_a.shape[-1]
    rows = o_a.numel() // D if D else 0
    if lse_a.numel() != rows or lse_b.numel() != rows or o_b.numel() != o_a.numel():
        raise ValueError("shape mismatch")
    _check(lib().ra_merge(o_a.data_ptr(), lse_a.data_ptr(), o_b.data_ptr(), lse_b.data_ptr(), rows, D,
                          RA_F32_BF16 if mixed else _DTYPE[o_a.dtype], _stream_ptr(stream)))
    return o_a, lse_a


def bwd_workspace_bytes(B, H, S, D, N) -> int:
    return int(lib().ra_bwd_workspace_bytes(B, H, S, D, N))


def _bwd_args(q, k, v, o, lse, do, qname="q"):
    """Shape, dtype and device checks shared by the backward entry points."""
    B, H, S, D = _need_4d(q, qname)
    for name, t in (("k", k), ("v", v), ("o", o), ("do", do)):
        _need(t, name, q.dtype, q.shape, q.device)
    _need(lse, "lse", torch.float32, (B, H, S), q.device)
    return B, H, S, D


def bwd(q, k, v, o, lse, do, n_blocks: int, causal: bool = True, layout: str = "contiguous", *,
        dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward from the saved (o, lse).  Returns (dq, dk, dv)."""
    B, H, S, D = _bwd_args(q, k, v, o, lse, do)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _need(t, name, q.dtype, q.shape, q.device)
    need = bwd_workspace_bytes(B, H, S, D, int(n_blocks))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", device=q.device)
    _check(lib().ra_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, S, D, int(n_blocks),
                        int(bool(causal)), _LAYOUT[layout], _DTYPE[q.dtype], workspace.data_ptr(),
                        workspace.numel() * workspace.element_size(), _stream_ptr(stream)))
    return dq, dk, dv


def bwd_step(q_i, k_j, v_j, o_i, lse_i, do_i, dq_i, dk_j, dv_j, n_blocks: int, i: int, j: int,
             causal: bool = True, layout: str = "contiguous", *, workspace=None, stream=None):
    """One ring round of the backward: add the contributions of query block i
    against KV block j into the float32 accumulators dq_i, dk_j, dv_j (in
    place).  q_i, o_i, do_i, k_j, v_j: [B, H, c, D] bf16; lse_i: block i's
    final [B, H, c] LSE.  Returns (dq_i, dk_j, dv_j)."""
    B, H, c, D = _bwd_args(q_i, k_j, v_j, o_i, lse_i, do_i, "q_i")
    for name, t in (("dq_i", dq_i), ("dk_j", dk_j), ("dv_j", dv_j)):
        _need(t, name, torch.float32, q_i.shape, q_i.device)
    if workspace is None:
        workspace = torch.empty(bwd_workspace_bytes(B, H, c, D, 1), dtype=torch.uint8, device=q_i.device)
    _need(workspace, "workspace", device=q_i.device)
    _check(lib().ra_bwd_step(q_i.data_ptr(), k_j.data_ptr(), v_j.data_ptr(), o_i.data_ptr(), lse_i.data_ptr(),
                             do_i.data_ptr(), dq_i.data_ptr(), dk_j.data_ptr(), dv_j.data_ptr(), B, H, c, D,
                             int(n_blocks), int(i), int(j), int(bool(causal)), _LAYOUT[layout], _DTYPE[q_i.dtype],
                             workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                             _stream_ptr(stream)))
    return dq_i, dk_j, dv_j


def bwd_noalloc(q, k, v, o, lse, do, n_blocks: int, causal: bool = True, layout: str = "contiguous", *,
                dq=None, dk=None, dv=None, stream=None):
    """Backward without a workspace argument, for callers that cannot allocate
    device memory: the library uses its own fixed 48 MiB device array (larger
    problems raise RingAttnError).  The output tensors may be passed in, so a
    caller that cannot allocate can reuse its own buffers.  Concurrent calls on
    one device race on that array.  Returns (dq, dk, dv)."""
    B, H, S, D = _bwd_args(q, k, v, o, lse, do)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _need(t, name, q.dtype, q.shape, q.device)
    _check(lib().ra_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, S, D,
                                int(n_blocks), int(bool(causal)), _LAYOUT[layout], _DTYPE[q.dtype],
                                _stream_ptr(stream)))
    return dq, dk, dv


def decode_workspace_bytes(B, H, S, D, N) -> int:
    return int(lib().ra_decode_workspace_bytes(B, H, S, D, N))


def decode(q, k, v, n_blocks: int = 1, *, o=None, lse=None, workspace=None, stream=None):
    """Ring decode: one new query token per (b, h) against its KV cache.

    q: [B, H, D]; k, v: [B, H, S, D] (bf16 CUDA tensors).  The cache is cut
    into ``n_blocks`` ring blocks of ceil(S / n_blocks) rows whose partial
    states are LogSumExp-merged.  With n_blocks = 1 on one block's segment it
    is the per-host ring step (chain the results with merge()).
    Returns (o [B, H, D], lse [B, H] float32)."""
    _need(q, "q")
    _need(k, "k", q.dtype, device=q.device)
    _need(v, "v", q.dtype, device=q.device)
    if q.dtype not in _DTYPE:
        raise ValueError("dtype must be bfloat16 or float32")
    B, H, S, D = k.shape
    if tuple(q.shape) != (B, H, D) or tuple(v.shape) != (B, H, S, D):
        raise ValueError("q must be [B, H, D] and v the shape of k")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    _need(o, "o", q.dtype, (B, H, D), q.device)
    _need(lse, "lse", torch.float32, (B, H), q.device)
    if workspace is None:
        need = decode_workspace_bytes(B, H, S, D, int(n_blocks))
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check(lib().ra_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, H, S, D, int(n_blocks), _DTYPE[q.dtype],
                           o.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
                           workspace.numel() * workspace.element_size(), _stream_ptr(stream)))
    return o, lse


def ffn_workspace_bytes(T, h, f, block_rows) -> int:
    return int(lib().ra_ffn_workspace_bytes(T, h, f, block_rows))


def ffn(x, w1, w3, w2, block_rows: int, *, y=None, workspace=None, stream=None):
    """Blockwise gated feedforward Y = (silu(X W1^T) * (X W3^T)) W2^T.

    x: [T, h]; w1, w3: [f, h]; w2: [h, f] (bf16 CUDA tensors).  Rows are
    processed ``block_rows`` at a time.  Returns y [T, h]."""
    for name, t in (("x", x), ("w1", w1), ("w3", w3), ("w2", w2)):
        _need(t, name, x.dtype, device=x.device)
    if x.dtype not in _DTYPE:
        raise ValueError("dtype must be bfloat16 or float32")
    T, h = x.shape
    f = w1.shape[0]
    if tuple(w1.shape) != (f, h) or tuple(w3.shape) != (f, h) or tuple(w2.shape) != (h, f):
        raise ValueError("w1, w3 must be [f, h] and w2 [h, f]")
    y = torch.empty_like(x) if y is None else y
    _need(y, "y", x.dtype, x.shape, x.device)
    if workspace is None:
        workspace = torch.empty(max(1, ffn_workspace_bytes(T, h, f, int(block_rows))), dtype=torch.uint8,
                                device=x.device)
    _check(lib().ra_ffn(x.data_ptr(), w1.data_ptr(), w3.data_ptr(), w2.data_ptr(), y.data_ptr(), T, h, f,
                        int(block_rows), _DTYPE[x.dtype], workspace.data_ptr(),
                        workspace.numel() * workspace.element_size(), _stream_ptr(stream)))
    return y


FWD_KERNELS = {"single": 0, "pair": 1}


def set_fwd_kernel(kind: str):
    """Which kernel later bf16 forward calls launch: "single" (the default,
    one CTA per SM) or "pair" (2-CTA clusters whose MMAs span an SM pair).
    The two kernels give bit-identical results."""
    if kind not in FWD_KERNELS:
        raise ValueError(f"set_fwd_kernel: kind must be one of {sorted(FWD_KERNELS)}, got {kind!r}")
    _check(lib().ra_set_fwd_kernel(FWD_KERNELS[kind]))


def set_timing_buffer(buf):
    """Enable per-(virtual host, ring step) timing into a uint64/int64 CUDA
    tensor of >= N*N entries (caller zeroes it); None disables."""
    if buf is None:
        _check(lib().ra_set_timing_buffer(None, 0))
    else:
        _need(buf, "timing buffer")
        _check(lib().ra_set_timing_buffer(buf.data_ptr(), buf.numel()))


class KernelTime(ctypes.Structure):
    _fields_ = [("call", ctypes.c_int), ("kernel", ctypes.c_int), ("ms", ctypes.c_float),
                ("sm_mhz", ctypes.c_float)]


KERNEL_NAMES = {(0, 0): "fwd", (0, 1): "fwd_pair", (1, 0): "bwd_prep", (1, 1): "bwd_dkv", (1, 2): "bwd_dq", (2, 0): "decode_split",
                (2, 1): "decode_combine"}


def set_kernel_timing(enable: bool):
    """Record CUDA events around every later kernel of fwd/bwd/decode calls
    (see kernel_times)."""
    _check(lib().ra_set_kernel_timing(int(bool(enable))))


def kernel_times(capacity: int = 4096, with_clock: bool = False):
    """Per-kernel durations of the calls timed since the last read: a list of
    (name, ms), oldest first, or (name, ms, sm_mhz) with `with_clock` (the SM
    clock a tensor-core kernel ran at, -1 for the others).  Waits for the
    recorded events."""
    buf = (KernelTime * capacity)()
    n = ctypes.c_int(0)
    _check(lib().ra_kernel_times(ctypes.addressof(buf), capacity, ctypes.byref(n)))
    recs = [buf[k] for k in range(n.value)]
    if with_clock:
        return [(_kernel_name(r.call, r.kernel), r.ms, r.sm_mhz) for r in recs]
    return [(_kernel_name(r.call, r.kernel), r.ms) for r in recs]


def _kernel_name(call: int, kernel: int) -> str:
    if call == 3:                                   # feedforward: up/down per block
        return "ffn_down" if kernel % 2 else "ffn_up"
    return KERNEL_NAMES.get((call, kernel), f"{call}.{kernel}")


def check_device_status(stream=None):
    """Synchronise and raise RingAttnError(RA_ERR_TIMEOUT) if a kernel gave up
    a bounded wait since the last check."""
    _check(lib().ra_check_device_status(_stream_ptr(stream)))


def version() -> str:
    return lib().ra_version().decode()
