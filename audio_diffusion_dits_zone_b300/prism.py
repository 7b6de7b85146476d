"""Thin ctypes binding of libprism.so (include/prism.h), with the C names.

Argument marshalling only: torch tensors are passed as device pointers, their
token row stride is read from the tensor's stride, and the stream is torch's
current CUDA stream.  Every step of the path runs in the library's kernels; if
the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

PRISM_OK, PRISM_EINVAL, PRISM_EUNSUPPORTED, PRISM_ECUDA, PRISM_ETIMEOUT, PRISM_EINDEX = range(6)
PRISM_F32, PRISM_BF16 = 0, 1
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libprism.so")
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "prism.h")

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.POINTER(ctypes.c_size_t)
_SIGS = {
    "prism_zone_shapes": [_P, _I32, _I64, _I32, _P, _I32, _I32, _I32, _I32, _I32, _I32, _P, _I32, _P, _P, _P, _SZ, _P],
    "prism_zone_shapes_noalloc": [_P, _I32, _I64, _I32, _P, _I32, _I32, _I32, _I32, _I32, _I32, _P, _I32, _P, _P,
                                  _P],
    "prism_zone_partials": [_P, _I32, _I64, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _SZ, _P],
    "prism_zone_shapes_from_partials": [_P, _I32, _I32, _P, _I32, _I32, _I32, _I32, _I32, _I32, _P, _I32, _P, _P, _P,
                                        _SZ, _P],
    "prism_pool_score": [_P, _P, _P, _I32, _I64, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _I64, _P, _P, _P, _P],
    "prism_select": [_P, _I32, _I32, ctypes.c_double, ctypes.c_double, _P, _P, _P],
    "prism_score_select": [_P, _P, _I32, _I32, _I32, ctypes.c_double, ctypes.c_double, _P, _P, _P],
    "prism_bsa_fwd": [_P, _P, _P, _I32, _I64, _I32, _I32, _I32, _I32, _P, _P, _I32, _P, _P, _P, _P, _SZ, _P],
    "prism_bsa_bwd": [_P, _P, _P, _P, _P, _P, _I32, _I64, _I32, _I32, _I32, _I32, _P, _P, _I32, _P, _P, _P, _P, _P,
                      _SZ, _P],
    "prism_pool_score_chunked": [_P, _P, _P, _I32, _I64, _I32, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _I64, _P, _P,
                                 _P, _P],
    "prism_zone_chunked_size": [_I32, _I32, _I32, _I32, _I32, _I32, _I32, ctypes.POINTER(ctypes.c_int32),
                                ctypes.POINTER(ctypes.c_int64)],
    "prism_zone_perm_chunked": [_P, _I32, _I32, _I32, _I32, _I32, _I32, _P, _I32, _I32, _P, _P, _P, _SZ, _P],
    "prism_a2v_norm": [_P, _P, _P, _I32, _I64, _I64, _I32, _I32, _I32, _I32, _P, _P, _P, _SZ, _P],
    "prism_attn_mse": [_P, _P, _I32, _I64, _I32, _I32, _I32, _P, _P, _SZ, _P],
    "prism_status_check": [_P, ctypes.POINTER(ctypes.c_uint32)],
    "prism_last_error": [],
    "prism_launch_count": [],
    "prism_build_info": [],
    "prism_selftest_umma": [_P, _P, _P, _P, _I32, _P],
    "prism_selftest_wait_timeout": [_I64, _P, _P],
    "prism_set_launch_hook": [_P, _P],
}
LAUNCH_HOOK = ctypes.CFUNCTYPE(None, ctypes.c_char_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p)
_lib = None


class PrismError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"libprism status {code}: {msg}")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m audio_diffusion_dits_zone_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_char_p if name in ("prism_last_error", "prism_build_info") else ctypes.c_int
            if name == "prism_launch_count":
                f.restype = ctypes.c_uint64
            if name == "prism_set_launch_hook":
                f.argtypes = [LAUNCH_HOOK, ctypes.c_void_p]
                f.restype = None
        _lib = L
    return _lib


def header_functions() -> list:
    """Names of the functions include/prism.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(prism_\w+)\s*\(", text, re.M)))


def _check(rc):
    if rc != PRISM_OK:
        raise PrismError(rc, lib().prism_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype(t):
    if t.dtype == torch.bfloat16:
        return PRISM_BF16
    if t.dtype == torch.float32:
        return PRISM_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ld(t):
    """Token row stride (elements) of a [N, Hh, d] view with contiguous heads."""
    assert t.dim() == 3 and t.stride(2) == 1 and (t.shape[1] == 1 or t.stride(1) == t.shape[2]), \
        "need a [N, Hh, d] view, d contiguous"
    return t.stride(0)


def launch_count() -> int:
    """Kernels the library has enqueued so far."""
    return int(lib().prism_launch_count())


def prism_set_launch_hook(fn):
    """Install a Python observer fn(kernel_name: str, stream_ptr: int, phase: int) called
    right before (0) and after (1) each kernel launch; None removes it.  Returns the
    ctypes callback object, which must be kept alive while installed."""
    if fn is None:
        lib().prism_set_launch_hook(LAUNCH_HOOK(), None)
        return None
    cb = LAUNCH_HOOK(lambda name, stream, phase, user: fn(name.decode(), stream or 0, phase))
    lib().prism_set_launch_hook(cb, None)
    return cb


class KernelTimer:
    """CUDA events recorded on the launching stream around every library kernel."""

    def __init__(self):
        self.records = []
        self._cb = None

    def _on_launch(self, name, stream, phase):
        ev = torch.cuda.Event(enable_timing=True)
        ev.record(torch.cuda.ExternalStream(stream) if stream else torch.cuda.current_stream())
        self.records.append((name, phase, ev))

    def __enter__(self):
        self._cb = prism_set_launch_hook(self._on_launch)
        return self

    def __exit__(self, *exc):
        prism_set_launch_hook(None)
        self._cb = None

    def durations(self) -> dict:
        """kernel name -> list of launch durations (ms); call after synchronising."""
        out, open_ = {}, {}
        for name, phase, ev in self.records:
            if phase == 0:
                open_[name] = ev
            elif name in open_:
                out.setdefault(name, []).append(open_.pop(name).elapsed_time(ev))
        return out


def build_info() -> str:
    return lib().prism_build_info().decode()


def status_check(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    w = ctypes.c_uint32(0)
    rc = lib().prism_status_check(_stream(stream), ctypes.byref(w))
    if rc not in (PRISM_OK, PRISM_ETIMEOUT, PRISM_EINDEX):
        _check(rc)
    return w.value


def _ws(query, ws, device):
    n = ctypes.c_size_t(0)
    _check(query(None, ctypes.byref(n)))
    if ws is None or ws.numel() < n.value:
        ws = torch.empty(n.value, dtype=torch.uint8, device=device)
    return ws, ctypes.c_size_t(ws.numel())


# ------------------------------------------------------------------- step 1
def prism_zone_shapes(feat, C, a2v, grid, zone, shapes, zone_shape, perm, ws=None, stream=None):
    """Zone shapes and block-order permutation (see include/prism.h).  feat: [N, ld]."""
    assert feat.dim() == 2 and feat.stride(1) == 1
    T, H, W = grid
    sh = (ctypes.c_int32 * (3 * len(shapes)))(*[int(e) for s in shapes for e in s])
    st = _stream(stream)

    def call(wsp, nbytes):
        return lib().prism_zone_shapes(_ptr(feat), _dtype(feat), feat.stride(0), C, _ptr(a2v), T, H, W, *zone, sh,
                                       len(shapes), _ptr(zone_shape), _ptr(perm), wsp, nbytes, st)

    ws, nbytes = _ws(call, ws, feat.device)
    _check(call(_ptr(ws), ctypes.byref(nbytes)))
    return ws


def prism_zone_shapes_noalloc(feat, C, a2v, grid, zone, shapes, zone_shape, perm, stream=None):
    """Zone shapes and permutation with no workspace: the library's built-in scratch is used.

    For callers that cannot provide device memory; calls on one device must not
    overlap on the GPU (they share the scratch)."""
    assert feat.dim() == 2 and feat.stride(1) == 1
    T, H, W = grid
    sh = (ctypes.c_int32 * (3 * len(shapes)))(*[int(e) for s in shapes for e in s])
    _check(lib().prism_zone_shapes_noalloc(_ptr(feat), _dtype(feat), feat.stride(0), C, _ptr(a2v), T, H, W, *zone,
                                           sh, len(shapes), _ptr(zone_shape), _ptr(perm), _stream(stream)))


def prism_zone_partials(feat, C, grid, zone, partials, ws=None, stream=None):
    """Per-zone, per-axis partial sums [Z, 3] of feat's first C channels (one rank's share
    of the zone statistics).  feat: [N, ld].  Returns the workspace tensor it used."""
    assert feat.dim() == 2 and feat.stride(1) == 1
    T, H, W = grid
    st = _stream(stream)

    def call(wsp, nbytes):
        return lib().prism_zone_partials(_ptr(feat), _dtype(feat), feat.stride(0), C, T, H, W, *zone,
                                         _ptr(partials), wsp, nbytes, st)

    ws, nbytes = _ws(call, ws, feat.device)
    _check(call(_ptr(ws), ctypes.byref(nbytes)))
    return ws


def prism_zone_shapes_from_partials(partials, C_total, a2v, grid, zone, shapes, zone_shape, perm, ws=None,
                                    stream=None):
    """Zone shapes and permutation from gathered partial sums [n_parts, Z, 3] (summed in
    part order) of C_total channels.  Returns the workspace tensor it used."""
    assert partials.dim() == 3 and partials.is_contiguous() and partials.shape[2] == 3
    T, H, W = grid
    sh = (ctypes.c_int32 * (3 * len(shapes)))(*[int(e) for s in shapes for e in s])
    st = _stream(stream)

    def call(wsp, nbytes):
        return lib().prism_zone_shapes_from_partials(_ptr(partials), partials.shape[0], C_total, _ptr(a2v), T, H, W,
                                                     *zone, sh, len(shapes), _ptr(zone_shape), _ptr(perm), wsp,
                                                     nbytes, st)

    ws, nbytes = _ws(call, ws, partials.device)
    _check(call(_ptr(ws), ctypes.byref(nbytes)))
    return ws


def prism_zone_chunked_size(grid, zone, B):
    """(nb, np): blocks and padded length of the zone-chunked block order (host only)."""
    nb, np_ = ctypes.c_int32(0), ctypes.c_int64(0)
    _check(lib().prism_zone_chunked_size(*grid, *zone, B, ctypes.byref(nb), ctypes.byref(np_)))
    return nb.value, np_.value


def prism_zone_perm_chunked(zone_shape, grid, zone, shapes, B, perm_padded, blen, ws=None, stream=None):
    """Padded zone-chunked block order (-1 at padding) and block lengths from zone shapes."""
    sh = (ctypes.c_int32 * (3 * len(shapes)))(*[int(e) for s in shapes for e in s])
    st = _stream(stream)

    def call(wsp, nbytes):
        return lib().prism_zone_perm_chunked(_ptr(zone_shape), *grid, *zone, sh, len(shapes), B, _ptr(perm_padded),
                                             _ptr(blen), wsp, nbytes, st)

    ws, nbytes = _ws(call, ws, zone_shape.device)
    _check(call(_ptr(ws), ctypes.byref(nbytes)))
    return ws


def prism_pool_score_chunked(q, k, v, perm_padded, B, q_blk=None, k_blk=None, v_blk=None, qbar=None, kbar=None,
                             scores=None, stream=None):
    """prism_pool_score over the padded zone-chunked block order; q, k, v: [n_src, Hh, d]."""
    n_src, Hh, d = q.shape
    np_ = perm_padded.numel()
    ldb = _ld(q_blk) if q_blk is not None else (_ld(k_blk) if k_blk is not None else
                                                (_ld(v_blk) if v_blk is not None else 0))
    _check(lib().prism_pool_score_chunked(_ptr(q), _ptr(k), _ptr(v), _dtype(q), _ld(q), n_src, _ptr(perm_padded),
                                          np_, Hh, d, B, _ptr(q_blk), _ptr(k_blk), _ptr(v_blk), ldb, _ptr(qbar),
                                          _ptr(kbar), _ptr(scores), _stream(stream)))


# ------------------------------------------------------------------- step 2
def prism_pool_score(q, k, v, perm, B, q_blk=None, k_blk=None, v_blk=None, qbar=None, kbar=None, scores=None,
                     stream=None):
    """Block-order copies, block means and block scores.  q, k, v: [N, Hh, d] views."""
    N, Hh, d = q.shape
    ldb = _ld(q_blk) if q_blk is not None else (_ld(k_blk) if k_blk is not None else
                                                (_ld(v_blk) if v_blk is not None else 0))
    _check(lib().prism_pool_score(_ptr(q), _ptr(k), _ptr(v), _dtype(q), _ld(q), _ptr(perm), N, Hh, d, B,
                                  _ptr(q_blk), _ptr(k_blk), _ptr(v_blk), ldb, _ptr(qbar), _ptr(kbar), _ptr(scores),
                                  _stream(stream)))


# ------------------------------------------------------------------- step 3
def prism_select(scores, sparsity, cdf_tau, counts, idx, stream=None):
    """Hybrid block selection.  scores: [Hh, nb, nb] fp32."""
    Hh, nb, _ = scores.shape
    _check(lib().prism_select(_ptr(scores), Hh, nb, float(sparsity), float(cdf_tau), _ptr(counts), _ptr(idx),
                              _stream(stream)))


def prism_score_select(qbar, kbar, sparsity, cdf_tau, counts, idx, stream=None):
    """Block scores and hybrid selection in one call (no score matrix).  qbar, kbar:
    [Hh, nb, d] fp32."""
    Hh, nb, d = qbar.shape
    assert kbar.shape == qbar.shape and qbar.is_contiguous() and kbar.is_contiguous()
    _check(lib().prism_score_select(_ptr(qbar), _ptr(kbar), Hh, nb, d, float(sparsity), float(cdf_tau), _ptr(counts),
                                    _ptr(idx), _stream(stream)))


# ------------------------------------------------------------------- step 4
def prism_bsa_fwd(q_blk, k_blk, v_blk, B, counts, idx, o_blk, lse, ws=None, stream=None, blen=None):
    """Block-sparse attention forward.  blen: per-block token counts of zone-chunked
    blocks (padded block order), or None.  Returns the workspace tensor it used."""
    N, Hh, d = q_blk.shape
    nb = -(-N // B)
    st = _stream(stream)

    def call(wsp, nbytes):
        return lib().prism_bsa_fwd(_ptr(q_blk), _ptr(k_blk), _ptr(v_blk), _dtype(q_blk), _ld(q_blk), N, Hh, d, B,
                                   _ptr(counts), _ptr(idx), nb, _ptr(blen), _ptr(o_blk), _ptr(lse), wsp, nbytes, st)

    ws, nbytes = _ws(call, ws, q_blk.device)
    _check(call(_ptr(ws), ctypes.byref(nbytes)))
    return ws


# --------------------------------------------------------------- A2V field
def prism_a2v_norm(qv, ka, va, a2v, o=None, ws=None, stream=None):
    """Audio-to-video cross-attention and its per-token feature norm (a2v [N] fp32).
    qv [N, Hh, d], ka / va [M, Hh, d] bf16; o ([N, Hh, d] or None) receives the
    attention output.  Returns the workspace tensor it used."""
    N, Hh, d = qv.shape
    M = ka.shape[0]
    assert _ld(ka) == _ld(va), "ka and va share one row stride"
    st = _stream(stream)

    def call(wsp, nbytes):
        return lib().prism_a2v_norm(_ptr(qv), _ptr(ka), _ptr(va), _dtype(qv), _ld(qv), _ld(ka), N, M, Hh, d,
                                    _ptr(o), _ptr(a2v), wsp, nbytes, st)

    ws, nbytes = _ws(call, ws, qv.device)
    _check(call(_ptr(ws), ctypes.byref(nbytes)))
    return ws


# ------------------------------------------------------------------- step 5
def prism_bsa_bwd(q_blk, k_blk, v_blk, o_blk, do_blk, lse, B, counts, idx, dq, dk, dv, ws=None, stream=None,
                  blen=None):
    """Block-sparse attention backward (blen as prism_bsa_fwd).  Returns the workspace
    tensor it used."""
    N, Hh, d = q_blk.shape
    nb = -(-N // B)
    st = _stream(stream)

    def call(wsp, nbytes):
        return lib().prism_bsa_bwd(_ptr(q_blk), _ptr(k_blk), _ptr(v_blk), _ptr(o_blk), _ptr(do_blk), _ptr(lse),
                                   _dtype(q_blk), _ld(q_blk), N, Hh, d, B, _ptr(counts), _ptr(idx), nb, _ptr(blen),
                                   _ptr(dq), _ptr(dk), _ptr(dv), wsp, nbytes, st)

    ws, nbytes = _ws(call, ws, q_blk.device)
    _check(call(_ptr(ws), ctypes.byref(nbytes)))
    return ws


# -------------------------------------------------- attention broadcast
def prism_attn_mse(a, b, mse, ws=None, stream=None):
    """Per-head mean squared difference of two [N, Hh, d] tensors into mse [Hh] fp32.
    Returns the workspace tensor it used."""
    assert a.shape == b.shape and a.dtype == b.dtype and _ld(a) == _ld(b)
    N, Hh, d = a.shape
    st = _stream(stream)

    def call(wsp, nbytes):
        return lib().prism_attn_mse(_ptr(a), _ptr(b), _dtype(a), _ld(a), N, Hh, d, _ptr(mse), wsp, nbytes, st)

    ws, nbytes = _ws(call, ws, a.device)
    _check(call(_ptr(ws), ctypes.byref(nbytes)))
    return ws


def prism_selftest_umma(a, b, out_s, out_o, variant=0, stream=None):
    _check(lib().prism_selftest_umma(_ptr(a), _ptr(b), _ptr(out_s), _ptr(out_o), variant, _stream(stream)))


def prism_selftest_wait_timeout(limit_ns, marker, stream=None):
    """Run the bounded-wait failure check (see include/prism.h); marker: int32 device tensor."""
    _check(lib().prism_selftest_wait_timeout(int(limit_ns), _ptr(marker), _stream(stream)))
