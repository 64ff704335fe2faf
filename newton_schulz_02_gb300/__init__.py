"""Python binding of the GB300 batched Muon step (libmuon_gb300.so).

Argument marshalling only: every step of the Muon update runs in the CUDA
library behind the C ABI of ``include/muon.h``; PyTorch supplies device
memory and streams.  The functions keep the C names.  There is no CPU
fallback: a call raises if the library is not built or no GPU is present.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_int64, c_size_t, c_uint32, c_uint64, c_void_p
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libmuon_gb300.so")

# status codes (muon_status_t)
MUON_OK = 0
MUON_ERR_INVALID_ARG = 1
MUON_ERR_MISALIGNED = 2
MUON_ERR_UNSUPPORTED = 3
MUON_ERR_WORKSPACE_TOO_SMALL = 4
MUON_ERR_CUDA = 5
MUON_ERR_TIMEOUT = 6
# device status bits
MUON_FLAG_NONFINITE = 0x1
MUON_FLAG_TIMEOUT = 0x2
MUON_FLAG_MISALIGNED = 0x4
# enums
MUON_BF16, MUON_F32 = 0, 1
MUON_NESTEROV_SGD, MUON_NESTEROV_EMA = 0, 1
MUON_SCALE_SPECTRAL, MUON_SCALE_UNIT_RMS_NORM, MUON_SCALE_NONE = 0, 1, 2
MUON_NS_BF16, MUON_NS_TF32, MUON_NS_BF16X3 = 0, 1, 2

_DT = {torch.bfloat16: MUON_BF16, torch.float32: MUON_F32}
_SCALE = {"spectral": MUON_SCALE_SPECTRAL, "unit_rms_norm": MUON_SCALE_UNIT_RMS_NORM,
          "none": MUON_SCALE_NONE}
_STYLE = {"sgd": MUON_NESTEROV_SGD, "ema": MUON_NESTEROV_EMA}


class muon_ns_stage_t(ctypes.Structure):
    _fields_ = [("steps", c_int), ("a", c_float), ("b", c_float), ("c", c_float)]


class muon_ns_schedule_t(ctypes.Structure):
    _fields_ = [("stages", POINTER(muon_ns_stage_t)), ("n_stages", c_int), ("normalize", c_int),
                ("prec", c_int), ("merge_groups", c_int)]


class muon_view_t(ctypes.Structure):
    _fields_ = [("rows", c_int), ("cols", c_int), ("row_stride", c_int64),
                ("batch_stride", c_int64), ("fan_out_axis", c_int)]


class muon_group_t(ctypes.Structure):
    _fields_ = [("batch", c_int), ("view", muon_view_t), ("w_dtype", c_int), ("g_dtype", c_int),
                ("w_ptrs", c_void_p), ("g_ptrs", c_void_p), ("m_ptrs", c_void_p),
                ("wd_mask", c_void_p)]


class muon_hparams_t(ctypes.Structure):
    _fields_ = [("mu", c_float), ("nesterov", c_int), ("style", c_int), ("t", c_int64),
                ("scale_mode", c_int), ("gamma", c_float), ("lr", c_float),
                ("weight_decay", c_float)]


class muon_tensor_desc_t(ctypes.Structure):
    _fields_ = [("rows", c_int), ("cols", c_int), ("row_stride", c_int64), ("w_dtype", c_int),
                ("g_dtype", c_int), ("fan_out_axis", c_int)]


class muon_kernel_stats_t(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", c_uint64), ("total_ms", ctypes.c_double),
                ("alg_flops", ctypes.c_double), ("alg_bytes", ctypes.c_double)]


class muon_adamw_group_t(ctypes.Structure):
    _fields_ = [("count", c_int), ("numel", c_int64), ("w_dtype", c_int), ("g_dtype", c_int),
                ("w_ptrs", c_void_p), ("g_ptrs", c_void_p), ("m_ptrs", c_void_p),
                ("v_ptrs", c_void_p), ("wd_mask", c_void_p)]


class muon_adamw_hparams_t(ctypes.Structure):
    _fields_ = [("lr", c_float), ("beta1", c_float), ("beta2", c_float), ("eps", c_float),
                ("weight_decay", c_float), ("t", c_int64)]


# C prototypes: name -> (restype, argtypes)
PROTOTYPES = {
    "muon_ns_hybrid_schedule": (c_int, [POINTER(muon_ns_schedule_t)]),
    "muon_group_by_shape": (c_int, [POINTER(muon_tensor_desc_t), c_int, c_int, POINTER(c_int),
                                    POINTER(c_int)]),
    "muon_step_workspace_size": (c_int, [POINTER(muon_group_t), c_int,
                                         POINTER(muon_ns_schedule_t), POINTER(c_size_t)]),
    "muon_step_batched": (c_int, [POINTER(muon_group_t), c_int, POINTER(muon_hparams_t),
                                  POINTER(muon_ns_schedule_t), c_void_p, c_size_t, c_void_p]),
    "newton_schulz_workspace_size": (c_int, [POINTER(muon_view_t), c_int,
                                             POINTER(muon_ns_schedule_t), POINTER(c_size_t)]),
    "newton_schulz_batched": (c_int, [c_void_p, c_int, POINTER(muon_view_t), c_int, c_void_p,
                                      c_int, POINTER(muon_ns_schedule_t), c_void_p, c_size_t,
                                      c_void_p]),
    "newton_schulz_batched_noalloc": (c_int, [c_void_p, c_int, POINTER(muon_view_t), c_int,
                                              c_void_p, c_int, POINTER(muon_ns_schedule_t),
                                              c_void_p, c_void_p]),
    "muon_get_status": (c_int, [c_void_p, c_void_p, POINTER(c_uint32)]),
    "muon_set_wait_timeout_ns": (c_int, [c_uint64]),
    "muon_check_wait_timeout": (c_int, [c_void_p, c_size_t, c_uint64, c_void_p]),
    "muon_occupy_sms": (c_int, [c_int, c_size_t, c_uint64, c_void_p]),
    "muon_profile_enable": (c_int, [c_int]),
    "muon_profile_reset": (c_int, []),
    "muon_profile_query": (c_int, [POINTER(muon_kernel_stats_t), c_int, POINTER(c_int)]),
    "muon_status_string": (c_char_p, [c_int]),
    "muon_adamw_step": (c_int, [POINTER(muon_adamw_group_t), c_int, POINTER(muon_adamw_hparams_t),
                                c_void_p, c_void_p]),
}

_lib = None


class MuonError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)}")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmuon_gb300.so (raises if it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built; run `python -m newton_schulz_02_gb300.build` "
                               "(or __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        for name, (res, args) in PROTOTYPES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(code: int) -> str:
    try:
        return load_library().muon_status_string(int(code)).decode()
    except RuntimeError:
        return f"status {code}"


def _check(code: int, where: str) -> None:
    if code != MUON_OK:
        raise MuonError(code, where)


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ---------------------------------------------------------------------------
# schedules and hyperparameters
# ---------------------------------------------------------------------------
class Schedule:
    """Owns a muon_ns_schedule_t and its stage array."""

    def __init__(self, stages: Sequence, normalize: bool = True, prec: int = MUON_NS_BF16,
                 merge_groups: bool = False):
        arr = (muon_ns_stage_t * max(1, len(stages)))()
        for i, (steps, (a, b, c)) in enumerate(stages):
            arr[i] = muon_ns_stage_t(int(steps), float(a), float(b), float(c))
        self._arr = arr
        self.c = muon_ns_schedule_t(ctypes.cast(arr, POINTER(muon_ns_stage_t)), len(stages),
                                    int(bool(normalize)), int(prec), int(bool(merge_groups)))

    @property
    def ref(self):
        return ctypes.byref(self.c)


def muon_ns_hybrid_schedule() -> muon_ns_schedule_t:
    s = muon_ns_schedule_t()
    _check(load_library().muon_ns_hybrid_schedule(ctypes.byref(s)), "muon_ns_hybrid_schedule")
    return s


def hparams(mu=0.95, nesterov=True, style="sgd", t=1, scale_mode="spectral", gamma=0.18,
            lr=2.7e-4, weight_decay=0.1) -> muon_hparams_t:
    return muon_hparams_t(float(mu), int(bool(nesterov)), _STYLE[style], int(t),
                          _SCALE[scale_mode], float(gamma), float(lr), float(weight_decay))


def _sched_ref(schedule):
    if schedule is None:
        return None
    if isinstance(schedule, Schedule):
        return schedule.ref
    return ctypes.byref(schedule)


# ---------------------------------------------------------------------------
# groups
# ---------------------------------------------------------------------------
class Group:
    """One batched group: same-shape matrices given as lists of 2-D tensors (or
    views), a stacked 3-D tensor, or the heads of a split_head weight.  Holds
    the device arrays of device pointers the C ABI takes."""

    def __init__(self, W: Sequence[torch.Tensor], G: Sequence[torch.Tensor],
                 M: Sequence[torch.Tensor], wd_mask: Optional[Sequence[bool]] = None,
                 fan_out_axis: int = 0):
        if not (len(W) == len(G) == len(M) and len(W) > 0):
            raise ValueError("W, G, M must be equally long and non-empty")
        r, c = W[0].shape
        rs = W[0].stride(0)
        for t in list(W) + list(G) + list(M):
            if t.dim() != 2 or tuple(t.shape) != (r, c) or t.stride(1) != 1 or t.stride(0) != rs:
                raise ValueError("all matrices of a group need one shape and one row stride")
        dev = W[0].device
        self.tensors = (list(W), list(G), list(M))
        self.ptrs = torch.tensor([[t.data_ptr() for t in W], [t.data_ptr() for t in G],
                                  [t.data_ptr() for t in M]], dtype=torch.int64, device=dev)
        self.mask = None
        if wd_mask is not None:
            self.mask = torch.tensor([1 if m else 0 for m in wd_mask], dtype=torch.uint8, device=dev)
        stride = self.ptrs.stride(0) * 8
        base = self.ptrs.data_ptr()
        self.c = muon_group_t(len(W), muon_view_t(r, c, rs, 0, fan_out_axis), _DT[W[0].dtype],
                              _DT[G[0].dtype], base, base + stride, base + 2 * stride,
                              self.mask.data_ptr() if self.mask is not None else None)

    @classmethod
    def stacked(cls, W: torch.Tensor, G: torch.Tensor, M: torch.Tensor, wd_mask=None,
                fan_out_axis: int = 0) -> "Group":
        return cls(list(W.unbind(0)), list(G.unbind(0)), list(M.unbind(0)), wd_mask, fan_out_axis)

    @classmethod
    def split_head(cls, W: torch.Tensor, G: torch.Tensor, M: torch.Tensor, n_heads: int,
                   head_dim: int, wd_mask=None) -> "Group":
        """[embed, heads*head_dim] weight -> `heads` sub-matrices embed x head_dim
        (heads form the batch; fan_out = head_dim, on the column axis)."""
        sl = [slice(h * head_dim, (h + 1) * head_dim) for h in range(n_heads)]
        return cls([W[:, s] for s in sl], [G[:, s] for s in sl], [M[:, s] for s in sl],
                   wd_mask, fan_out_axis=1)


def split_rows(W: torch.Tensor, G: torch.Tensor, M: torch.Tensor, parts: int,
               wd_mask=None) -> Group:
    """A fused weight stacked along rows (e.g. an FC1 [gate; up] weight,
    [parts*rows, cols]) as `parts` sub-matrices rows x cols orthogonalised
    separately (split_linear_fc1; each part keeps fan_out = its rows)."""
    if W.shape[0] % parts != 0:
        raise ValueError("rows must split into equal parts")
    r = W.shape[0] // parts
    sl = [slice(k * r, (k + 1) * r) for k in range(parts)]
    return Group([W[s] for s in sl], [G[s] for s in sl], [M[s] for s in sl], wd_mask, fan_out_axis=0)


Group.split_rows = staticmethod(split_rows)


def _group_array(groups: Sequence[Group]):
    arr = (muon_group_t * len(groups))(*[g.c for g in groups])
    return arr


def muon_group_by_shape(descs: Sequence[tuple], max_batch: int = 0):
    """descs: (rows, cols, row_stride, w_dtype, g_dtype, fan_out_axis) per tensor."""
    n = len(descs)
    arr = (muon_tensor_desc_t * max(1, n))(*[muon_tensor_desc_t(*map(int, d)) for d in descs])
    out = (c_int * max(1, n))()
    ng = c_int(0)
    _check(load_library().muon_group_by_shape(arr, n, int(max_batch), out, ctypes.byref(ng)),
           "muon_group_by_shape")
    return [out[i] for i in range(n)], ng.value


def muon_step_workspace_size(groups: Sequence[Group], schedule=None) -> int:
    arr = _group_array(groups)
    nb = c_size_t(0)
    _check(load_library().muon_step_workspace_size(arr, len(groups), _sched_ref(schedule),
                                                   ctypes.byref(nb)), "muon_step_workspace_size")
    return nb.value


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A caller-owned workspace buffer (256-byte aligned by the caching allocator)."""
    ws = torch.empty(max(256, nbytes), dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


def muon_step_batched(groups: Sequence[Group], hp: muon_hparams_t, ws: torch.Tensor,
                      schedule=None, stream=None) -> None:
    arr = _group_array(groups)
    _check(load_library().muon_step_batched(arr, len(groups), ctypes.byref(hp),
                                            _sched_ref(schedule), ws.data_ptr(), ws.numel(),
                                            _stream(stream)), "muon_step_batched")


def newton_schulz_workspace_size(rows: int, cols: int, batch: int, schedule=None) -> int:
    v = muon_view_t(rows, cols, cols, rows * cols, 0)
    nb = c_size_t(0)
    _check(load_library().newton_schulz_workspace_size(ctypes.byref(v), batch,
                                                       _sched_ref(schedule), ctypes.byref(nb)),
           "newton_schulz_workspace_size")
    return nb.value


def newton_schulz_batched(x: torch.Tensor, out: torch.Tensor, ws: torch.Tensor, schedule=None,
                          stream=None, view: Optional[muon_view_t] = None, batch: int = None) -> None:
    """O' of each matrix of x ([batch, rows, cols] or [rows, cols], unit column
    stride) into the dense tensor out of the same shape."""
    if view is None:
        x3 = x if x.dim() == 3 else x.unsqueeze(0)
        if x3.stride(2) != 1:
            raise ValueError("x needs unit column stride")
        batch = x3.shape[0]
        view = muon_view_t(x3.shape[1], x3.shape[2], x3.stride(1), x3.stride(0), 0)
    if not out.is_contiguous():
        raise ValueError("out must be contiguous")
    _check(load_library().newton_schulz_batched(x.data_ptr(), _DT[x.dtype], ctypes.byref(view),
                                                int(batch), out.data_ptr(), _DT[out.dtype],
                                                _sched_ref(schedule), ws.data_ptr(), ws.numel(),
                                                _stream(stream)), "newton_schulz_batched")


def newton_schulz_batched_noalloc(x: torch.Tensor, out: torch.Tensor, schedule=None,
                                  device_flags: Optional[torch.Tensor] = None,
                                  stream=None) -> int:
    """newton_schulz_batched on the library's own static scratch (no
    workspace argument, no device allocation).  For callers that cannot
    allocate device memory themselves; see include/muon.h.  Returns the C
    status code instead of raising, so callers can see a too-large request
    (MUON_ERR_WORKSPACE_TOO_SMALL)."""
    x3 = x if x.dim() == 3 else x.unsqueeze(0)
    if x3.stride(2) != 1 or not out.is_contiguous():
        raise ValueError("x needs unit column stride and out must be contiguous")
    view = muon_view_t(x3.shape[1], x3.shape[2], x3.stride(1), x3.stride(0), 0)
    flags_ptr = None
    if device_flags is not None:
        # one 4-byte word on the device x lives on: the call ends with a
        # device-to-device copy of its status word into it
        if not (device_flags.is_cuda and device_flags.device == x.device
                and device_flags.element_size() == 4 and device_flags.numel() >= 1):
            raise ValueError("device_flags must be a non-empty 4-byte tensor on x's device")
        flags_ptr = device_flags.data_ptr()
    return load_library().newton_schulz_batched_noalloc(
        x.data_ptr(), _DT[x.dtype], ctypes.byref(view), x3.shape[0], out.data_ptr(),
        _DT[out.dtype], _sched_ref(schedule), flags_ptr, _stream(stream))


def muon_get_status(ws: torch.Tensor, stream=None) -> tuple[int, int]:
    """(status code, device flags) after synchronising the stream."""
    flags = c_uint32(0)
    code = load_library().muon_get_status(ws.data_ptr(), _stream(stream), ctypes.byref(flags))
    return code, flags.value


def muon_set_wait_timeout_ns(ns: int) -> None:
    _check(load_library().muon_set_wait_timeout_ns(int(ns)), "muon_set_wait_timeout_ns")


def muon_check_wait_timeout(ws: torch.Tensor, timeout_ns: int, stream=None) -> None:
    _check(load_library().muon_check_wait_timeout(ws.data_ptr(), ws.numel(), int(timeout_ns),
                                                  _stream(stream)), "muon_check_wait_timeout")


def muon_occupy_sms(blocks: int, smem_bytes: int, ns: int, stream=None) -> None:
    """Hold `blocks` SMs (one block of `smem_bytes` shared memory each) for
    `ns` nanoseconds on `stream`; see include/muon.h."""
    _check(load_library().muon_occupy_sms(int(blocks), int(smem_bytes), int(ns), _stream(stream)),
           "muon_occupy_sms")


def muon_profile_enable(on: bool) -> None:
    _check(load_library().muon_profile_enable(int(bool(on))), "muon_profile_enable")


def muon_profile_reset() -> None:
    _check(load_library().muon_profile_reset(), "muon_profile_reset")


def muon_profile_query() -> dict:
    """{kernel kind: dict(launches, total_ms, alg_flops, alg_bytes)} since the last reset."""
    arr = (muon_kernel_stats_t * 16)()
    n = c_int(0)
    _check(load_library().muon_profile_query(arr, 16, ctypes.byref(n)), "muon_profile_query")
    return {arr[i].name.decode(): dict(launches=arr[i].launches, total_ms=arr[i].total_ms,
                                       alg_flops=arr[i].alg_flops, alg_bytes=arr[i].alg_bytes)
            for i in range(min(n.value, 16))}


# ---------------------------------------------------------------------------
# AdamW partition
# ---------------------------------------------------------------------------
class AdamWGroup:
    """Tensors of one element count and dtype pair (any shapes, contiguous):
    the device arrays of device pointers muon_adamw_step takes."""

    def __init__(self, W: Sequence[torch.Tensor], G: Sequence[torch.Tensor],
                 m: Sequence[torch.Tensor], v: Sequence[torch.Tensor],
                 wd_mask: Optional[Sequence[bool]] = None):
        if not (len(W) == len(G) == len(m) == len(v) and len(W) > 0):
            raise ValueError("W, G, m, v must be equally long and non-empty")
        n = W[0].numel()
        for t in list(W) + list(G) + list(m) + list(v):
            if t.numel() != n or not t.is_contiguous():
                raise ValueError("all tensors of a group need one element count and to be contiguous")
        for t in list(m) + list(v):
            if t.dtype != torch.float32:
                raise ValueError("moments are fp32")
        dev = W[0].device
        self.tensors = (list(W), list(G), list(m), list(v))
        self.ptrs = torch.tensor([[t.data_ptr() for t in x] for x in self.tensors],
                                 dtype=torch.int64, device=dev)
        self.mask = None
        if wd_mask is not None:
            self.mask = torch.tensor([1 if k else 0 for k in wd_mask], dtype=torch.uint8, device=dev)
        stride = self.ptrs.stride(0) * 8
        base = self.ptrs.data_ptr()
        self.c = muon_adamw_group_t(len(W), n, _DT[W[0].dtype], _DT[G[0].dtype], base,
                                    base + stride, base + 2 * stride, base + 3 * stride,
                                    self.mask.data_ptr() if self.mask is not None else None)


def adamw_groups(W, G, m, v, wd_mask=None) -> list:
    """Group parallel lists of tensors by (element count, W dtype, G dtype), in
    order of first appearance."""
    keys, members = [], {}
    for i, w in enumerate(W):
        k = (w.numel(), w.dtype, G[i].dtype)
        if k not in members:
            keys.append(k)
            members[k] = []
        members[k].append(i)
    out = []
    for k in keys:
        idx = members[k]
        out.append(AdamWGroup([W[i] for i in idx], [G[i] for i in idx], [m[i] for i in idx],
                              [v[i] for i in idx],
                              None if wd_mask is None else [wd_mask[i] for i in idx]))
    return out


def adamw_hparams(lr=2.7e-4, beta1=0.9, beta2=0.95, eps=1e-20, weight_decay=0.1,
                  t=1) -> muon_adamw_hparams_t:
    return muon_adamw_hparams_t(float(lr), float(beta1), float(beta2), float(eps),
                                float(weight_decay), int(t))


def muon_adamw_step(groups: Sequence[AdamWGroup], hp: muon_adamw_hparams_t,
                    flags: Optional[torch.Tensor] = None, stream=None) -> None:
    """flags: optional int32 device tensor of one element (MUON_FLAG_* are ORed in)."""
    arr = (muon_adamw_group_t * max(1, len(groups)))(*[g.c for g in groups])
    _check(load_library().muon_adamw_step(arr, len(groups), ctypes.byref(hp),
                                          flags.data_ptr() if flags is not None else None,
                                          _stream(stream)), "muon_adamw_step")
