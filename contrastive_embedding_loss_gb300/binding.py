"""Thin Python binding of ``include/uf_contrastive.h`` (argument marshalling only).

The functions named like the C entry points take plain integers (device pointers,
sizes, a stream handle) and return the C status.  ``contrastive_fwd_bwd`` is the
torch-facing convenience: it allocates the outputs and the workspace with torch (device
memory only) and makes one C call on the current stream.  Every step of the loss runs in
the library's CUDA kernels; there is no fallback: if the library is missing, or a call
fails, this module raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

KINDS = {"clip": 0, "siglip": 1, "rows": 2}
STATUS_NAMES = {0: "ok", 1: "invalid-argument", 2: "unsupported", 3: "workspace-too-small", 4: "cuda-error",
                5: "device-timeout"}
UF_OK = 0
UF_DEVICE_TIMEOUT = 5


class UfError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, 'unknown')} ({status})")
        self.status = status


_lib = None


def library_path() -> str:
    return _build.lib_path()


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the shared library (built by ``__graft_entry__.build()``); raise if it is absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or library_path()
    if not os.path.exists(p):
        raise ImportError(f"the uf_contrastive CUDA library is not built ({p} is missing); "
                          "run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(p)
    P, I64, I32, F32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.uf_status_name.argtypes = [I32]
    lib.uf_status_name.restype = ctypes.c_char_p
    lib.uf_contrastive_version.argtypes = []
    lib.uf_contrastive_version.restype = I32
    lib.uf_contrastive_init.argtypes = [I32]
    lib.uf_contrastive_init.restype = I32
    lib.uf_contrastive_workspace_size.argtypes = [I64, I64, I32, P, I32, I32, I32]
    lib.uf_contrastive_workspace_size.restype = SZ
    lib.uf_contrastive_workspace_min.argtypes = [I64, I64, I32, P, I32, I32, I32]
    lib.uf_contrastive_workspace_min.restype = SZ
    lib.uf_contrastive_fwd_bwd.argtypes = [P, P, I64, I64, I32, P, I32, I32, F32, F32, P, P, P, P, P, P, P, SZ,
                                           P, P]
    lib.uf_contrastive_fwd_bwd.restype = I32
    lib.uf_contrastive_fwd_bwd_ex.argtypes = [P, P, I64, I64, I32, P, I32, I32, F32, F32, P, P, P, P, P, P, P, P, P,
                                              P, P, P, P, SZ, P, P]
    lib.uf_contrastive_fwd_bwd_ex.restype = I32
    lib.uf_contrastive_oneset_fwd_bwd.argtypes = [P, I64, I32, P, I32, F32, F32, P, P, P, P, P, P, P, P, P, P, P, SZ,
                                                  P, P]
    lib.uf_contrastive_oneset_fwd_bwd.restype = I32
    lib.uf_contrastive_selftest_wait.argtypes = [P, I32, P]
    lib.uf_contrastive_selftest_wait.restype = I32
    lib.uf_contrastive_profile.argtypes = [I32]
    lib.uf_contrastive_profile.restype = I32
    lib.uf_contrastive_profile_read.argtypes = [I32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(I64),
                                                ctypes.POINTER(I64)]
    lib.uf_contrastive_profile_read.restype = I32
    lib.uf_contrastive_profile_name.argtypes = [I32]
    lib.uf_contrastive_profile_name.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def _int_array(values, ctype=ctypes.c_int):
    arr = (ctype * len(values))(*values)
    return arr


# ---- the C entry points, same names ------------------------------------------------

def uf_status_name(status: int) -> str:
    return load().uf_status_name(int(status)).decode()


def uf_contrastive_version() -> int:
    return int(load().uf_contrastive_version())


def uf_contrastive_init(device: int) -> int:
    return int(load().uf_contrastive_init(int(device)))


def uf_contrastive_workspace_size(Na, Nb, D, prefixes, kind, want_grads) -> int:
    pre = _int_array(list(prefixes))
    return int(load().uf_contrastive_workspace_size(int(Na), int(Nb), int(D), pre, len(prefixes), int(kind),
                                                    int(bool(want_grads))))


def uf_contrastive_workspace_min(Na, Nb, D, prefixes, kind, want_grads) -> int:
    pre = _int_array(list(prefixes))
    return int(load().uf_contrastive_workspace_min(int(Na), int(Nb), int(D), pre, len(prefixes), int(kind),
                                                   int(bool(want_grads))))


def uf_contrastive_fwd_bwd(A, B, Na, Nb, D, prefixes, kind, logit_scale, bias, prefix_weights, loss_per_prefix,
                           row_terms, col_terms, dA, dB, workspace, workspace_bytes, device_status, stream) -> int:
    """Raw call: every pointer argument is an int device address (or 0 / None for NULL)."""
    pre = _int_array(list(prefixes))
    w = None if prefix_weights is None else (ctypes.c_float * len(prefix_weights))(*prefix_weights)
    return int(load().uf_contrastive_fwd_bwd(A, B, int(Na), int(Nb), int(D), pre, len(prefixes), int(kind),
                                             float(logit_scale), float(bias), w, loss_per_prefix, row_terms,
                                             col_terms, dA, dB, workspace, int(workspace_bytes), device_status,
                                             stream))


def uf_contrastive_fwd_bwd_ex(A, B, Na, Nb, D, prefixes, kind, logit_scale, bias, logit_scale_dev, bias_dev,
                              pos_offsets, pos_ids, prefix_weights, loss_per_prefix, row_terms, col_terms, dA, dB,
                              d_logit_scale, d_bias, workspace, workspace_bytes, device_status, stream) -> int:
    """Raw call with the scalars optionally on the device (``*_dev``), SigLIP positives as
    device CSR lists (``pos_offsets`` int64, ``pos_ids`` int32) and the scalars' gradients
    (``d_logit_scale``, ``d_bias``): device addresses or None."""
    pre = _int_array(list(prefixes))
    w = None if prefix_weights is None else (ctypes.c_float * len(prefix_weights))(*prefix_weights)
    return int(load().uf_contrastive_fwd_bwd_ex(A, B, int(Na), int(Nb), int(D), pre, len(prefixes), int(kind),
                                                float(logit_scale), float(bias), logit_scale_dev, bias_dev,
                                                pos_offsets, pos_ids, w, loss_per_prefix, row_terms, col_terms, dA,
                                                dB, d_logit_scale, d_bias, workspace, int(workspace_bytes),
                                                device_status, stream))


def uf_contrastive_oneset_fwd_bwd(X, N, D, prefixes, logit_scale, bias, logit_scale_dev, bias_dev, pos_offsets,
                                  pos_ids, prefix_weights, loss_per_prefix, row_terms, dX, d_logit_scale, d_bias,
                                  workspace, workspace_bytes, device_status, stream) -> int:
    """Raw call of the one-set loss: every pointer argument is an int device address or None."""
    pre = _int_array(list(prefixes))
    w = None if prefix_weights is None else (ctypes.c_float * len(prefix_weights))(*prefix_weights)
    return int(load().uf_contrastive_oneset_fwd_bwd(X, int(N), int(D), pre, len(prefixes), float(logit_scale),
                                                    float(bias), logit_scale_dev, bias_dev, pos_offsets, pos_ids, w,
                                                    loss_per_prefix, row_terms, dX, d_logit_scale, d_bias, workspace,
                                                    int(workspace_bytes), device_status, stream))


def uf_contrastive_selftest_wait(device_status, limit_ms, stream) -> int:
    """Raw call: one kernel whose bounded wait runs out stores UF_DEVICE_TIMEOUT at the int
    device address device_status (a check of the kernels' failure path)."""
    return int(load().uf_contrastive_selftest_wait(device_status, int(limit_ms), stream))


KERNEL_GROUPS = ("prep", "transpose", "fwd_tile", "stats", "bwd_tile", "norm_bwd", "gemm")


def uf_contrastive_profile(enable: bool) -> int:
    return int(load().uf_contrastive_profile(int(bool(enable))))


def uf_contrastive_profile_name(group: int) -> str:
    return load().uf_contrastive_profile_name(int(group)).decode()


def uf_contrastive_profile_read(group: int):
    """(total_ms, timed_pairs, launches) of one kernel group since profiling was enabled."""
    ms, pairs, launches = ctypes.c_double(), ctypes.c_int64(), ctypes.c_int64()
    st = int(load().uf_contrastive_profile_read(int(group), ctypes.byref(ms), ctypes.byref(pairs),
                                                ctypes.byref(launches)))
    if st != UF_OK:
        raise UfError(st, "uf_contrastive_profile_read")
    return ms.value, pairs.value, launches.value


# ---- torch convenience ------------------------------------------------------------

_EMPTY_IDS = {}


def _empty_ids(dev):
    """A valid device address for an ids array with no entries (a labelled batch without positives)."""
    import torch

    if dev not in _EMPTY_IDS:
        _EMPTY_IDS[dev] = torch.zeros(1, dtype=torch.int32, device=dev)
    return _EMPTY_IDS[dev].data_ptr()

def _check_buffers(dev, workspace, device_status):
    """The caller's scratch and status word: a contiguous uint8 workspace and an int32 status
    tensor, both on the inputs' device."""
    import torch

    if workspace is not None and (workspace.dtype != torch.uint8 or workspace.device != dev
                                  or not workspace.is_contiguous()):
        raise TypeError("workspace must be a contiguous uint8 tensor on the inputs' device")
    if device_status is not None and (device_status.dtype != torch.int32 or device_status.device != dev
                                      or device_status.numel() < 1):
        raise TypeError("device_status must be an int32 tensor (one element) on the inputs' device")


def _check_labels(offs, n_rows):
    if offs.dim() != 1 or offs.numel() != n_rows + 1:
        raise ValueError(f"label offsets must hold rows + 1 = {n_rows + 1} entries, not {offs.numel()}")


def contrastive_fwd_bwd(A, B, kind="clip", prefixes=(64, 128, 256, 512, 1024), logit_scale=1 / 0.07, bias=0.0,
                        prefix_weights=None, grads=True, terms=False, workspace=None, device_status=None,
                        stream=None, scale_grads=False, labels=None):
    """Run the loss on bf16 CUDA tensors A (Na x D) and B (Nb x D).

    Returns a dict with ``loss`` (n_prefix fp32), ``dA``/``dB`` (fp32, when grads) and
    ``row_terms``/``col_terms`` (when terms), and with ``scale_grads`` the one-element
    fp32 tensors ``d_logit_scale`` and ``d_bias`` (the weighted loss's derivatives in
    the logit scale and the SigLIP bias; needs grads).  ``logit_scale`` and ``bias`` may
    be floats or one-element fp32 CUDA tensors; a tensor is read by the kernels when they
    run (graph capture of a learned scale).  ``labels`` (SigLIP): the positive pairs as CSR
    lists ``(offsets, ids)`` (int64 [Na + 1] and int32 CUDA tensors, or host arrays, which
    are copied to the device) in place of the diagonal.  ``workspace`` may be a preallocated uint8
    CUDA tensor of at least ``uf_contrastive_workspace_min`` bytes (its size sets how many
    rows of backward weights the library keeps at once); by default one of the
    recommended ``uf_contrastive_workspace_size`` bytes is allocated.
    """
    import torch

    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be 2-D (rows x D)")
    if A.shape[1] != B.shape[1]:
        raise ValueError(f"A and B must have the same width D ({A.shape[1]} vs {B.shape[1]})")
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16 or not A.is_cuda or not B.is_cuda:
        raise TypeError("A and B must be bf16 CUDA tensors")
    if A.device != B.device:
        raise ValueError("A and B must be on the same device")
    _check_buffers(A.device, workspace, device_status)
    A = A.contiguous()
    B = B.contiguous()
    Na, D = A.shape
    Nb = B.shape[0]
    k = KINDS[kind] if isinstance(kind, str) else int(kind)
    dev = A.device
    n = len(prefixes)
    need = uf_contrastive_workspace_size(Na, Nb, D, prefixes, k, grads)
    if need == 0:
        raise UfError(1, "uf_contrastive_workspace_size")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    out = {"loss": torch.empty(n, dtype=torch.float32, device=dev)}
    if grads:
        out["dA"] = torch.empty((Na, D), dtype=torch.float32, device=dev)
        out["dB"] = torch.empty((Nb, D), dtype=torch.float32, device=dev)
    if terms:
        out["row_terms"] = torch.empty((n, Na), dtype=torch.float32, device=dev)
        out["col_terms"] = torch.empty((n, Nb), dtype=torch.float32, device=dev)
    if scale_grads:
        out["d_logit_scale"] = torch.empty(1, dtype=torch.float32, device=dev)
        out["d_bias"] = torch.empty(1, dtype=torch.float32, device=dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731

    def scalar(v):  # (host value, device pointer)
        if isinstance(v, torch.Tensor):
            if v.dtype != torch.float32 or v.device != dev or v.numel() != 1:
                raise TypeError("a device logit scale / bias must be a one-element fp32 tensor on A's device")
            return 0.0, v.data_ptr()
        return float(v), None

    ls_host, ls_dev = scalar(logit_scale)
    b_host, b_dev = scalar(bias)
    offs = ids = None
    if labels is not None:
        offs, ids = labels
        offs = torch.as_tensor(offs, dtype=torch.int64, device=dev).contiguous()
        ids = torch.as_tensor(ids, dtype=torch.int32, device=dev).contiguous()
        _check_labels(offs, Na)
    with torch.cuda.device(dev):
        st = uf_contrastive_fwd_bwd_ex(A.data_ptr(), B.data_ptr(), Na, Nb, D, prefixes, k, ls_host, b_host, ls_dev,
                                       b_dev, ptr(offs), ptr(ids) if ids is not None and ids.numel() else
                                       (None if ids is None else _empty_ids(dev)), prefix_weights, out["loss"].data_ptr(), ptr(out.get("row_terms")),
                                       ptr(out.get("col_terms")), ptr(out.get("dA")), ptr(out.get("dB")),
                                       ptr(out.get("d_logit_scale")), ptr(out.get("d_bias")), workspace.data_ptr(),
                                       workspace.numel(), ptr(device_status), s.cuda_stream)
    if st != UF_OK:
        raise UfError(st, "uf_contrastive_fwd_bwd")
    return out


def oneset_fwd_bwd(X, labels, prefixes=(64, 128, 256, 512, 1024), logit_scale=10.0, bias=-10.0,
                   prefix_weights=None, grads=True, terms=False, workspace=None, device_status=None, stream=None,
                   scale_grads=False):
    """One-set SigLIP of the bf16 CUDA tensor X (N x D) against itself.  ``labels``: the
    symmetric positive pairs as CSR lists ``(offsets, ids)`` (device tensors or host arrays).
    Returns a dict with ``loss``, ``dX`` (when grads), ``row_terms`` (when terms) and, with
    ``scale_grads``, ``d_logit_scale`` / ``d_bias``.  Scalars may be one-element fp32 CUDA
    tensors, as in ``contrastive_fwd_bwd``."""
    import torch

    if X.dim() != 2:
        raise ValueError("X must be 2-D (rows x D)")
    if X.dtype != torch.bfloat16 or not X.is_cuda:
        raise TypeError("X must be a bf16 CUDA tensor")
    _check_buffers(X.device, workspace, device_status)
    X = X.contiguous()
    N, D = X.shape
    dev = X.device
    n = len(prefixes)
    k = KINDS["siglip"]
    if workspace is None:
        need = uf_contrastive_workspace_size(N, N, D, prefixes, k, grads)
        if need == 0:
            raise UfError(1, "uf_contrastive_workspace_size")
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    out = {"loss": torch.empty(n, dtype=torch.float32, device=dev)}
    if grads:
        out["dX"] = torch.empty((N, D), dtype=torch.float32, device=dev)
    if terms:
        out["row_terms"] = torch.empty((n, N), dtype=torch.float32, device=dev)
    if scale_grads:
        out["d_logit_scale"] = torch.empty(1, dtype=torch.float32, device=dev)
        out["d_bias"] = torch.empty(1, dtype=torch.float32, device=dev)
    offs, ids = labels
    offs = torch.as_tensor(offs, dtype=torch.int64, device=dev).contiguous()
    ids = torch.as_tensor(ids, dtype=torch.int32, device=dev).contiguous()
    _check_labels(offs, N)
    ids_ptr = ids.data_ptr() if ids.numel() else _empty_ids(dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731

    def scalar(v):
        if isinstance(v, torch.Tensor):
            if v.dtype != torch.float32 or v.device != dev or v.numel() != 1:
                raise TypeError("a device logit scale / bias must be a one-element fp32 tensor on X's device")
            return 0.0, v.data_ptr()
        return float(v), None

    ls_host, ls_dev = scalar(logit_scale)
    b_host, b_dev = scalar(bias)
    with torch.cuda.device(dev):
        st = uf_contrastive_oneset_fwd_bwd(X.data_ptr(), N, D, prefixes, ls_host, b_host, ls_dev, b_dev,
                                           offs.data_ptr(), ids_ptr, prefix_weights, out["loss"].data_ptr(),
                                           ptr(out.get("row_terms")), ptr(out.get("dX")),
                                           ptr(out.get("d_logit_scale")), ptr(out.get("d_bias")),
                                           workspace.data_ptr(), workspace.numel(), ptr(device_status),
                                           s.cuda_stream)
    if st != UF_OK:
        raise UfError(st, "uf_contrastive_oneset_fwd_bwd")
    return out


# ---- the entry point for callers that cannot allocate device memory -----------------

UF_STATIC_WORKSPACE_BYTES = 96 << 20


def uf_contrastive_fwd_bwd_static(A, B, Na, Nb, D, prefixes, kind, logit_scale, bias, prefix_weights,
                                  loss_per_prefix, row_terms, col_terms, dA, dB, device_status, stream) -> int:
    """Raw call of the library-owned-scratch variant: like ``uf_contrastive_fwd_bwd`` but
    without a workspace.  For callers that must not allocate device memory; calls whose GPU
    work overlaps share one scratch array and race.  Pointers are int device addresses."""
    lib = load()
    if not getattr(lib, "_static_bound", False):
        P, I64, I32, F32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        lib.uf_contrastive_fwd_bwd_static.argtypes = [P, P, I64, I64, I32, P, I32, I32, F32, F32, P, P, P, P, P, P,
                                                      P, P]
        lib.uf_contrastive_fwd_bwd_static.restype = I32
        lib._static_bound = True
    pre = _int_array(list(prefixes))
    w = None if prefix_weights is None else (ctypes.c_float * len(prefix_weights))(*prefix_weights)
    return int(lib.uf_contrastive_fwd_bwd_static(A, B, int(Na), int(Nb), int(D), pre, len(prefixes), int(kind),
                                                 float(logit_scale), float(bias), w, loss_per_prefix, row_terms,
                                                 col_terms, dA, dB, device_status, stream))
