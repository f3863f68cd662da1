"""ctypes wrapper around ``oracle.c`` (test infrastructure; see package docstring)."""
from __future__ import annotations

import contextlib
import ctypes
import hashlib
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
KINDS = {"clip": 0, "siglip": 1, "rows": 2}

_lib = None


def _so_path() -> str:
    with open(_SRC, "rb") as f:
        h = hashlib.sha1(f.read()).hexdigest()[:12]
    return os.path.join(_BUILD, f"liboracle_{os.uname().machine}_{h}.so")


def build() -> str:
    """Compile oracle.c (if needed) and return the shared-object path."""
    so = _so_path()
    if not os.path.exists(so):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = so + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, so)
    return so


def _bind(path):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.orc_fwd_bwd.argtypes = [ctypes.c_int, P, P, i64, i64, ctypes.c_int, P, ctypes.c_int,
                                ctypes.c_double, ctypes.c_double, P, P, P, P, P, P]
    lib.orc_fwd_bwd_f64.argtypes = lib.orc_fwd_bwd.argtypes
    lib.orc_row_stats.argtypes = [ctypes.c_int, P, P, i64, i64, ctypes.c_int, P, ctypes.c_int,
                                  ctypes.c_double, ctypes.c_double, P, i64, P, P]
    lib.orc_grad_rows.argtypes = [ctypes.c_int, ctypes.c_int, P, P, i64, i64, ctypes.c_int, P,
                                  ctypes.c_int, ctypes.c_double, ctypes.c_double, P, P, P, P,
                                  i64, P]
    lib.orc_scale_grads.argtypes = [ctypes.c_int, P, P, i64, i64, ctypes.c_int, P, ctypes.c_int,
                                    ctypes.c_double, ctypes.c_double, P, P, P]
    lib.orc_scale_grads_f64.argtypes = lib.orc_scale_grads.argtypes
    # SigLIP with a label matrix: the same arguments without the kind, the labels after the weights
    lib.orc_fwd_bwd_labels.argtypes = [P, P, i64, i64, ctypes.c_int, P, ctypes.c_int, ctypes.c_double,
                                       ctypes.c_double, P, P, P, P, P, P, P]
    lib.orc_fwd_bwd_labels_f64.argtypes = lib.orc_fwd_bwd_labels.argtypes
    lib.orc_scale_grads_labels.argtypes = [P, P, i64, i64, ctypes.c_int, P, ctypes.c_int, ctypes.c_double,
                                           ctypes.c_double, P, P, P, P]
    lib.orc_scale_grads_labels_f64.argtypes = lib.orc_scale_grads_labels.argtypes
    lib.orc_oneset.argtypes = [P, i64, ctypes.c_int, P, ctypes.c_int, ctypes.c_double, ctypes.c_double, P, P, P, P,
                               P, P, P]
    lib.orc_oneset_f64.argtypes = lib.orc_oneset.argtypes
    for f in (lib.orc_fwd_bwd, lib.orc_fwd_bwd_f64, lib.orc_row_stats, lib.orc_grad_rows, lib.orc_scale_grads,
              lib.orc_scale_grads_f64, lib.orc_fwd_bwd_labels, lib.orc_fwd_bwd_labels_f64,
              lib.orc_scale_grads_labels, lib.orc_scale_grads_labels_f64, lib.orc_oneset, lib.orc_oneset_f64):
        f.restype = ctypes.c_int
    return lib


@contextlib.contextmanager
def use_library(path):
    """Temporarily route every call to another build of oracle.c (planted-mistake tests)."""
    global _lib
    saved = _load()
    _lib = _bind(path)
    try:
        yield
    finally:
        _lib = saved


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(build())
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _bits(x):
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("embeddings must be bf16 bit patterns (uint16)")
    return x


def _prefix_array(prefixes):
    return np.ascontiguousarray(np.asarray(prefixes, dtype=np.int32))


def label_matrix(labels, Na, Nb):
    """Dense Na x Nb uint8 label matrix (1 = positive pair) from a boolean matrix or from
    CSR positive lists ``(offsets, ids)`` (row i's positives are ids[offsets[i]:offsets[i+1]])."""
    if isinstance(labels, tuple):
        offsets, ids = (np.asarray(x, np.int64) for x in labels)
        if offsets.shape != (Na + 1,) or offsets[0] != 0 or np.any(np.diff(offsets) < 0):
            raise ValueError("bad CSR offsets")
        if ids.size != offsets[-1] or (ids.size and (ids.min() < 0 or ids.max() >= Nb)):
            raise ValueError("bad CSR ids")
        Z = np.zeros((Na, Nb), np.uint8)
        rows = np.repeat(np.arange(Na), np.diff(offsets))
        Z[rows, ids] = 1
        return Z
    Z = np.ascontiguousarray(np.asarray(labels) != 0, dtype=np.uint8)
    if Z.shape != (Na, Nb):
        raise ValueError("label matrix must be Na x Nb")
    return Z


def fwd_bwd(kind, A, B, prefixes, scale, bias=0.0, weights=None, grads=True, labels=None):
    """Full float64 forward and backward.

    A and B are bf16 bit patterns (uint16), or float64 arrays (used by the
    finite-difference pins, which need continuous inputs).  ``labels`` (SigLIP only): the
    positive pairs, as for ``label_matrix``; by default the diagonal cells (i, i), i < Na.
    Returns dict(loss=[n], dA=(Na,D), dB=(Nb,D), row_terms=(n,Na), col_terms=(n,Nb)).
    """
    A, B = np.ascontiguousarray(A), np.ascontiguousarray(B)
    f64 = A.dtype == np.float64 and B.dtype == np.float64
    if not f64:
        A, B = _bits(A), _bits(B)
    if labels is not None:
        if kind != "siglip":
            raise ValueError("label matrices are defined for SigLIP only")
        Z = label_matrix(labels, A.shape[0], B.shape[0])
        lab = _load().orc_fwd_bwd_labels_f64 if f64 else _load().orc_fwd_bwd_labels
        fn = lambda _k, *a: lab(*a[:10], _ptr(Z), *a[10:])  # noqa: E731
    else:
        fn = _load().orc_fwd_bwd_f64 if f64 else _load().orc_fwd_bwd
    Na, D = A.shape
    Nb = B.shape[0]
    pre = _prefix_array(prefixes)
    n = pre.size
    w = None if weights is None else np.ascontiguousarray(np.asarray(weights, np.float64))
    loss = np.zeros(n)
    dA = np.zeros((Na, D)) if grads else None
    dB = np.zeros((Nb, D)) if grads else None
    rt = np.zeros((n, Na))
    ct = np.zeros((n, Nb))
    rc = fn(KINDS[kind], _ptr(A), _ptr(B), Na, Nb, D, _ptr(pre), n, float(scale), float(bias), _ptr(w),
            _ptr(loss), _ptr(dA), _ptr(dB), _ptr(rt), _ptr(ct))
    if rc:
        raise ValueError(f"oracle fwd_bwd failed ({rc})")
    return dict(loss=loss, dA=dA, dB=dB, row_terms=rt, col_terms=ct)


def row_stats(kind, X, Y, prefixes, scale, bias, rows):
    """Per selected row of X against all of Y: (lse[r, k], pos[r, k]); see oracle.c."""
    X, Y = _bits(X), _bits(Y)
    pre = _prefix_array(prefixes)
    rows = np.ascontiguousarray(np.asarray(rows, np.int64))
    lse = np.zeros((rows.size, pre.size))
    pos = np.zeros((rows.size, pre.size))
    rc = _load().orc_row_stats(KINDS[kind], _ptr(X), _ptr(Y), X.shape[0], Y.shape[0], X.shape[1],
                               _ptr(pre), pre.size, float(scale), float(bias), _ptr(rows), rows.size,
                               _ptr(lse), _ptr(pos))
    if rc:
        raise ValueError(f"oracle row_stats failed ({rc})")
    return lse, pos


def softmax_normalisers(kind, X, Y, prefixes, scale, row_chunk=None):
    """Every row's softmax log-normaliser at every prefix, for large batches: (lse, pos) with
    lse[k, i] = log sum_j exp(scale cos^k_ij) over all rows j of Y and pos[k, i] = scale cos^k_ii
    (0 for i >= len(Y)).  These are the log-sum-exp terms of the InfoNCE losses (blog
    "Scaling-Up Contrastive Learning over NVLink Multicast", section "One Set or Two": each
    row of cosines becomes a softmax over the batch); ``grad_rows`` takes them as lse_x /
    lse_y, and CLIP's column normalisers are this function with X and Y exchanged.

    The same definition as ``row_stats`` (bf16 widened exactly to float64; each prefix
    normalised on its own, inverse norm 1/max(|x[:p]|, 1e-30)), with one float64 library
    matmul per prefix and row chunk as the dot-product step, in torch CPU ops (all host
    cores) so that a batch of 65536 x 65536 takes minutes rather than the C loops' hour.
    CLIP and ROWS only (SigLIP has no normaliser)."""
    import torch

    if kind not in ("clip", "rows"):
        raise ValueError("softmax normalisers exist for clip and rows only")
    X, Y = _bits(X), _bits(Y)
    pre = [int(p) for p in prefixes]
    Xd = torch.from_numpy(_widen(X))
    Yd = torch.from_numpy(_widen(Y))
    Nx, Ny = Xd.shape[0], Yd.shape[0]
    if row_chunk is None:
        row_chunk = max(64, min(Nx, (1 << 27) // Ny))  # about 1 GiB of float64 scores per chunk
    lse = np.zeros((len(pre), Nx))
    pos = np.zeros((len(pre), Nx))
    for k, p in enumerate(pre):
        xn = Xd[:, :p] / Xd[:, :p].norm(dim=1, keepdim=True).clamp_min(1e-30)
        yn = Yd[:, :p] / Yd[:, :p].norm(dim=1, keepdim=True).clamp_min(1e-30)
        for r0 in range(0, Nx, row_chunk):
            s = xn[r0:r0 + row_chunk] @ yn.T
            s.mul_(float(scale))
            m = min(r0 + s.shape[0], Ny) - r0
            if m > 0:
                idx = torch.arange(m)
                pos[k, r0:r0 + m] = s[idx, r0 + idx].numpy()
            # log-sum-exp with the shift |scale| (|cos| <= 1 bounds every logit by it, and
            # e^(-2 |scale|) is far inside float64's range for every accepted scale)
            sh = abs(float(scale))
            lse[k, r0:r0 + s.shape[0]] = (s.sub_(sh).exp_().sum(dim=1).log_() + sh).numpy()
    return lse, pos


def _widen(bits):
    """bf16 bit patterns -> float64, exactly."""
    return (np.ascontiguousarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def row_terms_sampled(kind, X, Y, prefixes, scale, bias, rows):
    """Per-row loss terms (shape (n, len(rows))), computed one row at a time."""
    lse, pos = row_stats(kind, X, Y, prefixes, scale, bias, rows)
    return (lse - pos).T if kind != "siglip" else lse.T


def grad_rows(kind, x_is_a, X, Y, prefixes, scale, bias, rows, lse_x=None, lse_y=None, weights=None):
    """Gradient rows of sum_k w_k L_k for selected rows of X; see oracle.c."""
    X, Y = _bits(X), _bits(Y)
    pre = _prefix_array(prefixes)
    rows = np.ascontiguousarray(np.asarray(rows, np.int64))
    w = None if weights is None else np.ascontiguousarray(np.asarray(weights, np.float64))
    lx = None if lse_x is None else np.ascontiguousarray(np.asarray(lse_x, np.float64))
    ly = None if lse_y is None else np.ascontiguousarray(np.asarray(lse_y, np.float64))
    out = np.zeros((rows.size, X.shape[1]))
    rc = _load().orc_grad_rows(KINDS[kind], int(bool(x_is_a)), _ptr(X), _ptr(Y), X.shape[0], Y.shape[0],
                               X.shape[1], _ptr(pre), pre.size, float(scale), float(bias), _ptr(w),
                               _ptr(lx), _ptr(ly), _ptr(rows), rows.size, _ptr(out))
    if rc:
        raise ValueError(f"oracle grad_rows failed ({rc})")
    return out


def scale_grads(kind, A, B, prefixes, scale, bias=0.0, weights=None, labels=None):
    """(dL/dscale, dL/dbias) of sum_k w_k L_k, from the loss definitions; see oracle.c.

    A and B are bf16 bit patterns (uint16) or float64 arrays; ``labels`` as in fwd_bwd."""
    A, B = np.ascontiguousarray(A), np.ascontiguousarray(B)
    f64 = A.dtype == np.float64 and B.dtype == np.float64
    if not f64:
        A, B = _bits(A), _bits(B)
    if labels is not None:
        if kind != "siglip":
            raise ValueError("label matrices are defined for SigLIP only")
        Z = label_matrix(labels, A.shape[0], B.shape[0])
        lab = _load().orc_scale_grads_labels_f64 if f64 else _load().orc_scale_grads_labels
        fn = lambda _k, *a: lab(*a[:10], _ptr(Z), *a[10:])  # noqa: E731
    else:
        fn = _load().orc_scale_grads_f64 if f64 else _load().orc_scale_grads
    pre = _prefix_array(prefixes)
    w = None if weights is None else np.ascontiguousarray(np.asarray(weights, np.float64))
    ds = np.zeros(1)
    db = np.zeros(1)
    rc = fn(KINDS[kind], _ptr(A), _ptr(B), A.shape[0], B.shape[0], A.shape[1], _ptr(pre), pre.size, float(scale),
            float(bias), _ptr(w), _ptr(ds), _ptr(db))
    if rc:
        raise ValueError(f"oracle scale_grads failed ({rc})")
    return float(ds[0]), float(db[0])


def oneset(X, prefixes, t, b, labels, weights=None, grads=True):
    """One-set SigLIP of the set X against itself (see oracle.c): dict(loss=[n], dX=(N, D),
    row_terms=(n, N), dscale, dbias).  X: bf16 bit patterns or float64; labels as for
    ``label_matrix`` (symmetric; the diagonal is ignored)."""
    X = np.ascontiguousarray(X)
    f64 = X.dtype == np.float64
    if not f64:
        X = _bits(X)
    N, D = X.shape
    Z = label_matrix(labels, N, N)
    pre = _prefix_array(prefixes)
    n = pre.size
    w = None if weights is None else np.ascontiguousarray(np.asarray(weights, np.float64))
    loss = np.zeros(n)
    dX = np.zeros((N, D)) if grads else None
    rt = np.zeros((n, N))
    ds = np.zeros(1)
    db = np.zeros(1)
    fn = _load().orc_oneset_f64 if f64 else _load().orc_oneset
    rc = fn(_ptr(X), N, D, _ptr(pre), n, float(t), float(b), _ptr(w), _ptr(Z), _ptr(loss), _ptr(dX), _ptr(rt),
            _ptr(ds), _ptr(db))
    if rc:
        raise ValueError(f"oracle oneset failed ({rc})")
    return dict(loss=loss, dX=dX, row_terms=rt, dscale=float(ds[0]), dbias=float(db[0]))
