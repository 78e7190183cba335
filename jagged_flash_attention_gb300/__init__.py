"""GB300 (sm_103a) jagged flash attention: a thin Python binding of libjfa.so.

The binding only marshals arguments (pointers, sizes, the current CUDA
stream) into the C ABI of include/jfa.h; every step of the computation runs
in the library's CUDA kernels.  PyTorch supplies device memory and streams.
There is no fallback: if the library is missing, calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os

from .build import LIB_PATH

__all__ = ["JfaError", "lib", "jfa_fwd", "jfa_bwd", "jfa_fwd_bq", "jfa_bwd_bq", "jfa_fwd_ex",
           "jfa_bwd_ex", "jfa_block_select", "jfa_fwd_sparse", "jfa_block_select_ex",
           "jfa_fwd_sparse_ex", "block_select", "forward_sparse",
           "jfa_fwd_bq_noalloc", "jfa_worklist", "jfa_sync_and_check", "forward", "backward",
           "STATUS"]

STATUS = {0: "JFA_OK", 1: "JFA_ERR_INVALID_ARG", 2: "JFA_ERR_UNSUPPORTED", 3: "JFA_ERR_CUDA",
          4: "JFA_ERR_TIMEOUT", 5: "JFA_ERR_WORKSPACE"}

_LIB = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float


class JfaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libjfa.so (built by jagged_flash_attention_gb300.build)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run jagged_flash_attention_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        fwd = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P]
        bwd = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P]
        L.jfa_fwd.argtypes = fwd
        L.jfa_bwd.argtypes = bwd
        L.jfa_fwd_bq.argtypes = fwd[:8] + [_I] + fwd[8:]
        L.jfa_bwd_bq.argtypes = bwd[:8] + [_I] + bwd[8:]
        # _ex: H_kv after H; window_left, window_right after causal
        L.jfa_fwd_ex.argtypes = fwd[:6] + [_I] * 8 + fwd[10:]
        L.jfa_bwd_ex.argtypes = bwd[:6] + [_I] * 8 + bwd[10:]
        for f in (L.jfa_fwd, L.jfa_bwd, L.jfa_fwd_bq, L.jfa_bwd_bq, L.jfa_fwd_ex, L.jfa_bwd_ex):
            f.restype = _I
        L.jfa_sync_and_check.argtypes = [_P]
        L.jfa_sync_and_check.restype = _I
        L.jfa_last_error.restype = ctypes.c_char_p
        L.jfa_launch_count.restype = ctypes.c_longlong
        L.jfa_launch_count.argtypes = []
        L.jfa_profile_enable.argtypes = [_I]
        L.jfa_profile_enable.restype = _I
        L.jfa_profile_read.argtypes = [_P, _P, _I]
        L.jfa_profile_read.restype = _I
        L.jfa_profile_select.argtypes = [ctypes.c_uint]
        L.jfa_profile_select.restype = _I
        L.jfa_version.restype = ctypes.c_char_p
        _LIB = L
    return _LIB


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int):
    if status != 0:
        raise JfaError(status, lib().jfa_last_error().decode())


def jfa_fwd(q, k, v, offsets, B, H, D, max_len, broadcast_q, causal, scale, out, lse, stream=None):
    _check(lib().jfa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(offsets), B, H, D, max_len,
                         int(broadcast_q), int(causal), float(scale), _ptr(out), _ptr(lse),
                         _stream(stream)))


def jfa_bwd(q, k, v, offsets, B, H, D, max_len, broadcast_q, causal, scale, out, lse, dout,
            dq, dk, dv, stream=None):
    _check(lib().jfa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(offsets), B, H, D, max_len,
                         int(broadcast_q), int(causal), float(scale), _ptr(out), _ptr(lse),
                         _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)))


def jfa_fwd_bq(q, k, v, offsets, B, H, D, max_len, q_len, broadcast_q, causal, scale, out, lse,
               stream=None):
    _check(lib().jfa_fwd_bq(_ptr(q), _ptr(k), _ptr(v), _ptr(offsets), B, H, D, max_len, q_len,
                            int(broadcast_q), int(causal), float(scale), _ptr(out), _ptr(lse),
                            _stream(stream)))


def jfa_bwd_bq(q, k, v, offsets, B, H, D, max_len, q_len, broadcast_q, causal, scale, out, lse,
               dout, dq, dk, dv, stream=None):
    _check(lib().jfa_bwd_bq(_ptr(q), _ptr(k), _ptr(v), _ptr(offsets), B, H, D, max_len, q_len,
                            int(broadcast_q), int(causal), float(scale), _ptr(out), _ptr(lse),
                            _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)))


def jfa_fwd_ex(q, k, v, offsets, B, H, H_kv, D, max_len, q_len, broadcast_q, causal,
               window_left, window_right, scale, out, lse, stream=None):
    _check(lib().jfa_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(offsets), B, H, H_kv, D, max_len,
                            q_len, int(broadcast_q), int(causal), int(window_left),
                            int(window_right), float(scale), _ptr(out), _ptr(lse),
                            _stream(stream)))


def jfa_bwd_ex(q, k, v, offsets, B, H, H_kv, D, max_len, q_len, broadcast_q, causal,
               window_left, window_right, scale, out, lse, dout, dq, dk, dv, stream=None):
    _check(lib().jfa_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(offsets), B, H, H_kv, D, max_len,
                            q_len, int(broadcast_q), int(causal), int(window_left),
                            int(window_right), float(scale), _ptr(out), _ptr(lse), _ptr(dout),
                            _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)))


def jfa_block_select(q, k, offsets, B, H, H_kv, D, max_len, q_len, broadcast_q, permille,
                     blocks, counts, stream=None):
    fn = lib().jfa_block_select
    if fn.argtypes is None:
        fn.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P]
        fn.restype = _I
    _check(fn(_ptr(q), _ptr(k), _ptr(offsets), B, H, H_kv, D, max_len, q_len, int(broadcast_q),
              int(permille), _ptr(blocks), _ptr(counts), _stream(stream)))


def jfa_fwd_sparse(q, k, v, offsets, B, H, H_kv, D, max_len, q_len, broadcast_q, scale, blocks,
                   counts, out, lse, stream=None):
    fn = lib().jfa_fwd_sparse
    if fn.argtypes is None:
        fn.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P]
        fn.restype = _I
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(offsets), B, H, H_kv, D, max_len, q_len,
              int(broadcast_q), float(scale), _ptr(blocks), _ptr(counts), _ptr(out), _ptr(lse),
              _stream(stream)))


def jfa_block_select_ex(q, k, offsets, B, H, H_kv, D, max_len, q_len, broadcast_q, causal,
                        window_left, window_right, permille, blocks, counts, stream=None):
    fn = lib().jfa_block_select_ex
    if fn.argtypes is None:
        fn.argtypes = [_P, _P, _P] + [_I] * 11 + [_P, _P, _P]
        fn.restype = _I
    _check(fn(_ptr(q), _ptr(k), _ptr(offsets), B, H, H_kv, D, max_len, q_len, int(broadcast_q),
              int(causal), int(window_left), int(window_right), int(permille), _ptr(blocks),
              _ptr(counts), _stream(stream)))


def jfa_fwd_sparse_ex(q, k, v, offsets, B, H, H_kv, D, max_len, q_len, broadcast_q, causal,
                      window_left, window_right, scale, blocks, counts, out, lse, stream=None):
    fn = lib().jfa_fwd_sparse_ex
    if fn.argtypes is None:
        fn.argtypes = [_P, _P, _P, _P] + [_I] * 10 + [_F, _P, _P, _P, _P, _P]
        fn.restype = _I
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(offsets), B, H, H_kv, D, max_len, q_len,
              int(broadcast_q), int(causal), int(window_left), int(window_right), float(scale),
              _ptr(blocks), _ptr(counts), _ptr(out), _ptr(lse), _stream(stream)))


def jfa_fwd_bq_noalloc(q, k, v, offsets, B, H, D, max_len, q_len, broadcast_q, causal, scale,
                       out, lse, stream=None):
    """Allocation-free forward (see include/jfa.h): for callers that must not
    allocate device memory during the call.  The caller passes every buffer;
    the library's scratch is a fixed 1 MiB device array."""
    L = lib()
    fn = L.jfa_fwd_bq_noalloc
    if fn.argtypes is None:
        fn.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P]
        fn.restype = _I
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(offsets), B, H, D, max_len, q_len,
              int(broadcast_q), int(causal), float(scale), _ptr(out), _ptr(lse), _stream(stream)))


def jfa_worklist(offsets, B, H, max_len, q_len, broadcast_q, causal, which, items, capacity,
                 count, stream=None):
    """Builds work list `which` (0 forward, 1 dK/dV pass, 2 self-attention dQ
    pass, 3 broadcast dQ-pass chunks) into the device int32 buffer `items`
    (4 ints per entry, `capacity` entries) and `count` (device int32[2])."""
    L = lib()
    fn = L.jfa_worklist
    if fn.argtypes is None:
        fn.argtypes = [_P, _I, _I, _I, _I, _I, _I, _I, _P, _I, _P, _P]
        fn.restype = _I
    _check(fn(_ptr(offsets), B, H, max_len, q_len, int(broadcast_q), int(causal), which,
              _ptr(items), capacity, _ptr(count), _stream(stream)))


def jfa_sync_and_check(stream=None):
    _check(lib().jfa_sync_and_check(_stream(stream)))


KERNEL_KINDS = ("sched", "fwd", "prep", "bwd_kv", "bwd_q", "bwd_qb", "finalize", "fill",
                "bwd_bs", "fwd_combine", "sparse_pool", "sparse_select", "bwd_kv_pair",
                "sparse_check")


def launch_count() -> int:
    """Kernels this library has enqueued in this process."""
    return int(lib().jfa_launch_count())


def profile_enable(on: bool):
    _check(lib().jfa_profile_enable(1 if on else 0))


def profile_select(kinds=None):
    """Kernel kinds profiling brackets with events (names of KERNEL_KINDS;
    None: every kind)."""
    mask = 0xFFFFFFFF if kinds is None else sum(1 << KERNEL_KINDS.index(k) for k in kinds)
    _check(lib().jfa_profile_select(mask))


def profile_read():
    """{kind: (total device ms, launches)} since the last read (synchronises)."""
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_longlong * n)()
    _check(lib().jfa_profile_read(ctypes.addressof(ms), ctypes.addressof(cnt), n))
    return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNEL_KINDS)}


def _shapes(q, k, offsets, broadcast_q):
    """(B, H query heads, H_kv K/V heads, D, dense Q length or 0)."""
    T, Hkv, D = k.shape
    B = offsets.numel() - 1
    return B, q.shape[1], Hkv, D, (q.shape[0] if broadcast_q else 0)


def _window(window):
    wl, wr = (-1, -1) if window is None else window
    return (-1 if wl is None else int(wl)), (-1 if wr is None else int(wr))


def forward(q, k, v, offsets, max_len, causal=False, broadcast_q=False, scale=None, out=None,
            lse=None, stream=None, window=None):
    """Allocate out / lse with torch and call the C ABI.  Tensors are CUDA
    tensors in the layouts of include/jfa.h; offsets is int32 [B+1].  k and
    v may carry fewer heads than q (GQA); window = (left, right) bounds the
    keys of query i to [i - left, i + right] (None: unbounded side)."""
    import torch
    B, H, Hkv, D, Lq = _shapes(q, k, offsets, broadcast_q)
    wl, wr = _window(window)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    if out is None:
        out = torch.empty((B, Lq, H, D) if broadcast_q else tuple(q.shape), dtype=q.dtype,
                          device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Lq) if broadcast_q else (H, k.shape[0]), dtype=torch.float32,
                          device=q.device)
    if Hkv != H or (wl, wr) != (-1, -1):
        jfa_fwd_ex(q, k, v, offsets, B, H, Hkv, D, max_len, Lq, int(broadcast_q), causal, wl, wr,
                   scale, out, lse, stream)
    elif broadcast_q:
        jfa_fwd_bq(q, k, v, offsets, B, H, D, max_len, Lq, 1, causal, scale, out, lse, stream)
    else:
        jfa_fwd(q, k, v, offsets, B, H, D, max_len, 0, causal, scale, out, lse, stream)
    return out, lse


def backward(q, k, v, offsets, max_len, out, lse, dout, causal=False, broadcast_q=False,
             scale=None, dq=None, dk=None, dv=None, stream=None, window=None):
    """Allocate dq / dk / dv with torch and call the C ABI (arguments as for
    forward)."""
    import torch
    B, H, Hkv, D, Lq = _shapes(q, k, offsets, broadcast_q)
    wl, wr = _window(window)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if Hkv != H or (wl, wr) != (-1, -1):
        jfa_bwd_ex(q, k, v, offsets, B, H, Hkv, D, max_len, Lq, int(broadcast_q), causal, wl, wr,
                   scale, out, lse, dout, dq, dk, dv, stream)
    elif broadcast_q:
        jfa_bwd_bq(q, k, v, offsets, B, H, D, max_len, Lq, 1, causal, scale, out, lse, dout,
                   dq, dk, dv, stream)
    else:
        jfa_bwd(q, k, v, offsets, B, H, D, max_len, 0, causal, scale, out, lse, dout, dq, dk, dv,
                stream)
    return dq, dk, dv


def block_select(q, k, offsets, max_len, permille, blocks=None, counts=None, stream=None,
                 broadcast_q=False, causal=False, window=None):
    """Top-k K blocks per (sequence, query head, 256-row Q block) (see
    jfa_block_select in include/jfa.h); returns int32 (blocks [B, H, nqb,
    kcap], counts [B, H, nqb]).  causal / window restrict the candidates to
    the blocks inside each Q block's band (jfa_block_select_ex)."""
    import torch
    B, H, Hkv, D, Lq = _shapes(q, k, offsets, broadcast_q)
    nqb, kcap = -(-(Lq if broadcast_q else max_len) // 256), -(-max_len // 128)
    if blocks is None:
        blocks = torch.empty((B, H, nqb, kcap), dtype=torch.int32, device=q.device)
    if counts is None:
        counts = torch.empty((B, H, nqb), dtype=torch.int32, device=q.device)
    wl, wr = _window(window)
    if causal or (wl, wr) != (-1, -1):
        jfa_block_select_ex(q, k, offsets, B, H, Hkv, D, max_len, Lq, int(broadcast_q), causal,
                            wl, wr, permille, blocks, counts, stream)
    else:
        jfa_block_select(q, k, offsets, B, H, Hkv, D, max_len, Lq, int(broadcast_q), permille,
                         blocks, counts, stream)
    return blocks, counts


def forward_sparse(q, k, v, offsets, max_len, blocks, counts, scale=None, out=None, lse=None,
                   stream=None, broadcast_q=False, causal=False, window=None):
    """Attention over the listed K blocks of each Q block (jfa_fwd_sparse;
    with causal / window, over the admissible keys of those blocks:
    jfa_fwd_sparse_ex)."""
    import torch
    B, H, Hkv, D, Lq = _shapes(q, k, offsets, broadcast_q)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    if out is None:
        out = torch.empty((B, Lq, H, D) if broadcast_q else tuple(q.shape), dtype=q.dtype,
                          device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Lq) if broadcast_q else (H, k.shape[0]), dtype=torch.float32,
                          device=q.device)
    wl, wr = _window(window)
    if causal or (wl, wr) != (-1, -1):
        jfa_fwd_sparse_ex(q, k, v, offsets, B, H, Hkv, D, max_len, Lq, int(broadcast_q), causal,
                          wl, wr, scale, blocks, counts, out, lse, stream)
    else:
        jfa_fwd_sparse(q, k, v, offsets, B, H, Hkv, D, max_len, Lq, int(broadcast_q), scale,
                       blocks, counts, out, lse, stream)
    return out, lse
