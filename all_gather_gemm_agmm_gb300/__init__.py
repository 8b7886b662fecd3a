"""GB300 (sm_103a) fused all-gather matmul: a thin Python binding of libagmm.so.

    O = concat(X_0, ..., X_{P-1}) @ (Y if not rhs_transpose else Y.T)

Every step of the computation runs in the CUDA kernels of ``libagmm.so``
(``include/agmm.h``); this module only marshals arguments through ctypes.
PyTorch supplies device memory and streams.  There is no CPU fallback: if the
library is missing or the device is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, List, Optional, Sequence

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libagmm.so")

# Status codes of agmm.h.
AGMM_OK = 0
AGMM_ERR_INVALID_ARG = 1
AGMM_ERR_UNSUPPORTED = 2
AGMM_ERR_ALIGNMENT = 3
AGMM_ERR_CUDA = 4
AGMM_ERR_TIMEOUT = 5
AGMM_ERR_NOMEM = 6
AGMM_BF16 = 0
AGMM_BF16_F32OUT = 1
AGMM_F16 = 2
AGMM_F16_F32OUT = 3

# Every symbol agmm.h declares.
EXPORTED_SYMBOLS = [
    "agmm_plan", "agmm_destroy", "agmm_workspace_bytes", "agmm_run", "agmm_run_unfused",
    "agmm_run_host", "agmm_query_status", "agmm_plan_info", "agmm_ring_chunks",
    "agmm_status_string", "agmm_last_error", "agmm_version", "agmm_trace_bytes", "agmm_set_trace",
    "agmm_run_unfused_noalloc", "agmm_run_gather", "agmm_plan_preview", "agmm_plan_config",
]

# agmm_tile_config_t: 0 leaves a field to the planner (the tuned table, else
# its rules); on/off fields take AGMM_CFG_OFF / AGMM_CFG_ON.
AGMM_CFG_AUTO = 0
AGMM_CFG_OFF = 1
AGMM_CFG_ON = 2
CONFIG_FIELDS = ("path", "chunks", "box_rows", "tile_n", "cluster_m", "cta_pair", "stages", "group_m",
                 "stream_k", "row_groups", "splits", "dsmem_reduce", "tuned_table")
_ON_OFF = ("cta_pair", "stream_k", "dsmem_reduce", "tuned_table")
_NAMED = {"path": {"rows": 1, "swap": 2}, "chunks": {"half": 1, "whole": 2}}


class AgmmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int), ("box_rows", ctypes.c_int), ("whole_shards", ctypes.c_int), ("chunks", ctypes.c_int),
        ("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int), ("tile_k", ctypes.c_int),
        ("stages", ctypes.c_int), ("splits", ctypes.c_int), ("num_tiles", ctypes.c_int),
        ("num_ctas", ctypes.c_int), ("group_m", ctypes.c_int), ("num_sms", ctypes.c_int),
        ("smem_bytes", ctypes.c_size_t), ("row_groups", ctypes.c_int), ("cluster_m", ctypes.c_int),
        ("cta_pair", ctypes.c_int), ("stream_k_tiles", ctypes.c_int), ("dsmem_reduce", ctypes.c_int),
        ("config_source", ctypes.c_int), ("k_blocks_per_stage", ctypes.c_int),
    ]


class TileConfig(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int) for f in CONFIG_FIELDS]


def tile_config(config: Optional[Dict[str, object]]) -> Optional[TileConfig]:
    """A TileConfig from a dict of agmm_tile_config_t fields (None: no config).

    ``path`` takes "rows" / "swap" (or 1 / 2), ``chunks`` "half" / "whole" (or
    1 / 2); on/off fields (cta_pair, stream_k, dsmem_reduce, tuned_table) take
    booleans; the rest are integers.  Missing or None fields stay 0, the
    planner's choice."""
    if config is None:
        return None
    unknown = set(config) - set(CONFIG_FIELDS)
    if unknown:
        raise ValueError(f"unknown tile config fields: {sorted(unknown)}")
    tc = TileConfig()
    for f, v in config.items():
        if v is None:
            continue
        if f in _ON_OFF and isinstance(v, bool):
            v = AGMM_CFG_ON if v else AGMM_CFG_OFF
        elif f in _NAMED and isinstance(v, str):
            v = _NAMED[f][v]
        setattr(tc, f, int(v))
    return tc


def config_dict(tc: TileConfig) -> Dict[str, object]:
    """The set fields of a TileConfig, in tile_config's notation."""
    out: Dict[str, object] = {}
    for f in CONFIG_FIELDS:
        v = getattr(tc, f)
        if v == 0:
            continue
        if f in _ON_OFF:
            out[f] = v == AGMM_CFG_ON
        elif f in _NAMED:
            out[f] = {b: a for a, b in _NAMED[f].items()}.get(v, v)
        else:
            out[f] = v
    return out


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libagmm.so (built by ``__graft_entry__.build()``) and declare its ABI."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    vp, i64, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.agmm_plan.argtypes = [c_int, i64, i64, i64, c_int, c_int, ctypes.POINTER(vp)]
    lib.agmm_plan.restype = c_int
    lib.agmm_destroy.argtypes = [vp]
    lib.agmm_destroy.restype = None
    lib.agmm_workspace_bytes.argtypes = [vp, c_int]
    lib.agmm_workspace_bytes.restype = ctypes.c_size_t
    lib.agmm_run.argtypes = [vp, ctypes.POINTER(vp), vp, vp, c_int, vp, vp]
    lib.agmm_run.restype = c_int
    lib.agmm_run_unfused.argtypes = [vp, ctypes.POINTER(vp), vp, vp, c_int, vp, vp]
    lib.agmm_run_unfused.restype = c_int
    lib.agmm_run_gather.argtypes = [vp, ctypes.POINTER(vp), vp, vp, vp, c_int, vp, vp]
    lib.agmm_run_gather.restype = c_int
    lib.agmm_plan_preview.argtypes = [c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, c_int, c_int,
                                      ctypes.POINTER(TileConfig), c_int, ctypes.POINTER(PlanInfo)]
    lib.agmm_plan_config.argtypes = [c_int, i64, i64, i64, c_int, c_int, ctypes.POINTER(TileConfig),
                                     ctypes.POINTER(vp)]
    lib.agmm_plan_config.restype = c_int
    lib.agmm_plan_preview.restype = c_int
    lib.agmm_run_host.argtypes = [vp, ctypes.POINTER(vp), vp, vp, ctypes.POINTER(vp), vp, vp, c_int, vp, vp]
    lib.agmm_run_host.restype = c_int
    lib.agmm_query_status.argtypes = [vp, vp, vp]
    lib.agmm_query_status.restype = c_int
    lib.agmm_plan_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
    lib.agmm_plan_info.restype = c_int
    lib.agmm_ring_chunks.argtypes = [c_int, i64, c_int, c_int, c_int, ctypes.POINTER(ctypes.c_int32),
                                     ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_int32),
                                     i64, ctypes.POINTER(i64)]
    lib.agmm_ring_chunks.restype = c_int
    lib.agmm_status_string.argtypes = [c_int]
    lib.agmm_status_string.restype = ctypes.c_char_p
    lib.agmm_last_error.argtypes = []
    lib.agmm_last_error.restype = ctypes.c_char_p
    lib.agmm_version.argtypes = []
    lib.agmm_version.restype = c_int
    lib.agmm_run_unfused_noalloc.argtypes = [vp, ctypes.POINTER(vp), vp, vp, c_int, vp]
    lib.agmm_run_unfused_noalloc.restype = c_int
    lib.agmm_trace_bytes.argtypes = [vp]
    lib.agmm_trace_bytes.restype = ctypes.c_size_t
    lib.agmm_set_trace.argtypes = [vp, vp, ctypes.c_size_t]
    lib.agmm_set_trace.restype = c_int
    if path == LIB_PATH:
        _lib = lib
    return lib


def _status_name(status: int) -> str:
    names = {0: "AGMM_OK", 1: "AGMM_ERR_INVALID_ARG", 2: "AGMM_ERR_UNSUPPORTED", 3: "AGMM_ERR_ALIGNMENT",
             4: "AGMM_ERR_CUDA", 5: "AGMM_ERR_TIMEOUT", 6: "AGMM_ERR_NOMEM"}
    return names.get(status, f"AGMM_STATUS_{status}")


def _check(status: int) -> None:
    if status != AGMM_OK:
        raise AgmmError(status, load_library().agmm_last_error().decode())


def _ptr_array(ptrs: Sequence[int]):
    return (ctypes.c_void_p * len(ptrs))(*[ctypes.c_void_p(int(p)) for p in ptrs])


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def ring_chunks(P: int, m_per_device: int, my_id: int, box_rows: int, whole_shards: bool = False
                ) -> Dict[str, List[int]]:
    """The ring-ordered row chunks (host logic of agmm_ring_chunks)."""
    lib = load_library()
    n = ctypes.c_int64(0)
    w = int(bool(whole_shards))
    _check(lib.agmm_ring_chunks(P, m_per_device, my_id, box_rows, w, None, None, None, None, 0, ctypes.byref(n)))
    cnt = n.value
    shard = (ctypes.c_int32 * cnt)()
    src = (ctypes.c_int64 * cnt)()
    out = (ctypes.c_int64 * cnt)()
    valid = (ctypes.c_int32 * cnt)()
    _check(lib.agmm_ring_chunks(P, m_per_device, my_id, box_rows, w, shard, src, out, valid, cnt, ctypes.byref(n)))
    return {"shard": list(shard), "src_row": list(src), "out_row": list(out), "valid": list(valid)}


def plan_preview(P: int, m_per_device: int, k: int, n: int, rhs_transpose: bool = False, num_sms: int = 152,
                 out_f32: bool = False, f16: bool = False,
                 config: Optional[Dict[str, object]] = None) -> Dict[str, int]:
    """The tile choice for a device with ``num_sms`` SMs, computed on the host
    without CUDA (see agmm_plan_preview in agmm.h); ``config`` as for Plan."""
    lib = load_library()
    if f16:
        dtype = AGMM_F16_F32OUT if out_f32 else AGMM_F16
    else:
        dtype = AGMM_BF16_F32OUT if out_f32 else AGMM_BF16
    inf = PlanInfo()
    tc = tile_config(config)
    _check(lib.agmm_plan_preview(int(P), int(m_per_device), int(k), int(n), dtype, int(bool(rhs_transpose)),
                                 ctypes.byref(tc) if tc is not None else None, int(num_sms), ctypes.byref(inf)))
    return {f: getattr(inf, f) for f, _ in PlanInfo._fields_}


class Plan:
    """A planned problem: P shards of [m_per_device, k] times Y ([k, n] or [n, k]).

    ``config`` (a dict, see tile_config) fixes tile choices; fields it leaves
    out come from the tuned table for this exact shape, else the planner's
    rules."""

    def __init__(self, P: int, m_per_device: int, k: int, n: int, rhs_transpose: bool = False,
                 out_f32: bool = False, f16: bool = False, config: Optional[Dict[str, object]] = None):
        self._lib = load_library()
        self.P, self.m_per_device, self.k, self.n = int(P), int(m_per_device), int(k), int(n)
        self.rhs_transpose = bool(rhs_transpose)
        self.out_f32 = bool(out_f32)
        self.f16 = bool(f16)
        if self.f16:
            dtype = AGMM_F16_F32OUT if out_f32 else AGMM_F16
        else:
            dtype = AGMM_BF16_F32OUT if out_f32 else AGMM_BF16
        h = ctypes.c_void_p()
        tc = tile_config(config)
        _check(self._lib.agmm_plan_config(self.P, self.m_per_device, self.k, self.n, dtype,
                                          int(self.rhs_transpose), ctypes.byref(tc) if tc is not None else None,
                                          ctypes.byref(h)))
        self._h = h

    @property
    def M(self) -> int:
        return self.P * self.m_per_device

    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.agmm_destroy(self._h)
            self._h = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass

    def info(self) -> Dict[str, int]:
        inf = PlanInfo()
        _check(self._lib.agmm_plan_info(self._h, ctypes.byref(inf)))
        return {f: getattr(inf, f) for f, _ in PlanInfo._fields_}

    def enable_trace(self, device=None):
        """Allocate and attach a device trace buffer; returns it ([CTAs, 16] int64)."""
        import torch

        nbytes = int(self._lib.agmm_trace_bytes(self._h))
        buf = torch.zeros((nbytes // 128, 16), dtype=torch.int64, device=device or "cuda")
        _check(self._lib.agmm_set_trace(self._h, buf.data_ptr(), nbytes))
        self._trace = buf
        return buf

    def disable_trace(self) -> None:
        _check(self._lib.agmm_set_trace(self._h, None, 0))
        self._trace = None

    def workspace_bytes(self, unfused: bool = False) -> int:
        return int(self._lib.agmm_workspace_bytes(self._h, int(bool(unfused))))

    def new_workspace(self, unfused: bool = False, device=None):
        """A zero-filled workspace.  It is zeroed on the current stream: launches
        on another stream must first wait for it (the kernels rely on its
        counters starting at zero)."""
        import torch

        return torch.zeros(self.workspace_bytes(unfused), dtype=torch.uint8, device=device or "cuda")

    def run(self, xs, y, o, my_id: int, workspace, stream=None) -> None:
        """Fused path.  xs: P device tensors; y, o, workspace: device tensors."""
        _check(self._lib.agmm_run(self._h, _ptr_array([x.data_ptr() for x in xs]), y.data_ptr(), o.data_ptr(),
                                  int(my_id), workspace.data_ptr(), _stream_handle(stream)))

    def run_ptrs(self, x_ptrs: Sequence[int], y_ptr: int, o_ptr: int, my_id: int, ws_ptr: int,
                 stream_handle: Optional[int]) -> None:
        _check(self._lib.agmm_run(self._h, _ptr_array(x_ptrs), y_ptr, o_ptr, int(my_id), ws_ptr, stream_handle))

    def run_gather(self, xs, y, o, xcat, my_id: int, workspace, stream=None) -> None:
        """Fused path that also writes concat(xs) into xcat ([P*m, k], input dtype)."""
        _check(self._lib.agmm_run_gather(self._h, _ptr_array([x.data_ptr() for x in xs]), y.data_ptr(),
                                         o.data_ptr(), xcat.data_ptr(), int(my_id), workspace.data_ptr(),
                                         _stream_handle(stream)))

    def run_unfused(self, xs, y, o, my_id: int, workspace, stream=None) -> None:
        """Gather into the workspace, then the same GEMM on the gathered buffer."""
        _check(self._lib.agmm_run_unfused(self._h, _ptr_array([x.data_ptr() for x in xs]), y.data_ptr(),
                                          o.data_ptr(), int(my_id), workspace.data_ptr(), _stream_handle(stream)))

    def run_host(self, xs_host, y_host, o_host, xs_dev, y_dev, o_dev, my_id: int, workspace, stream=None) -> None:
        """Upload host inputs, run the fused path, download O (asynchronous)."""
        _check(self._lib.agmm_run_host(self._h, _ptr_array([x.data_ptr() for x in xs_host]), y_host.data_ptr(),
                                       o_host.data_ptr(), _ptr_array([x.data_ptr() for x in xs_dev]),
                                       y_dev.data_ptr(), o_dev.data_ptr(), int(my_id), workspace.data_ptr(),
                                       _stream_handle(stream)))

    def query_status(self, workspace, stream=None) -> int:
        """Synchronize and return (and clear) the device status; raises on error."""
        st = self._lib.agmm_query_status(self._h, workspace.data_ptr(), _stream_handle(stream))
        _check(st)
        return st


def _check_operands(xs, y, rhs_transpose: bool):
    import torch

    if len(xs) < 1:
        raise ValueError("need at least one shard")
    m, k = xs[0].shape
    if xs[0].dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("inputs must be bfloat16 or float16")
    for x in xs:
        if x.dtype != xs[0].dtype or y.dtype != xs[0].dtype:
            raise ValueError("shards and y must share one dtype")
        if x.shape != (m, k) or not x.is_contiguous() or not x.is_cuda:
            raise ValueError("shards must be contiguous CUDA tensors of one shape")
    if y.dim() != 2 or not y.is_contiguous() or not y.is_cuda:
        raise ValueError("y must be a contiguous 2-D CUDA tensor")
    n, ky = (y.shape if rhs_transpose else (y.shape[1], y.shape[0]))
    if ky != k:
        raise ValueError(f"contracting dimension mismatch: shards have k={k}, y gives {ky}")
    return m, k, n


_plan_cache: Dict[tuple, Plan] = {}


def all_gather_matmul(xs, y, my_id: int = 0, rhs_transpose: bool = False, out=None, unfused: bool = False,
                      out_f32: bool = False, workspace=None, stream=None, return_gathered: bool = False):
    """all-gather(xs, axis=0) @ y on one GPU; returns O [P*m, n] in the input
    dtype (bf16 or fp16) or float32.  With return_gathered it returns
    (O, concat(xs)): the fused kernel stores the gathered rows as it loads them."""
    import torch

    m, k, n = _check_operands(xs, y, rhs_transpose)
    f16 = xs[0].dtype == torch.float16
    key = (len(xs), m, k, n, bool(rhs_transpose), bool(out_f32), f16, torch.cuda.current_device())
    plan = _plan_cache.get(key)
    if plan is None:
        plan = Plan(len(xs), m, k, n, rhs_transpose, out_f32, f16)
        _plan_cache[key] = plan
    if out is None:
        out = torch.empty((plan.M, n), dtype=torch.float32 if out_f32 else xs[0].dtype, device=y.device)
    if workspace is None:
        workspace = plan.new_workspace(unfused, device=y.device)
    if return_gathered:
        if unfused:
            raise ValueError("return_gathered uses the fused path")
        xcat = torch.empty((plan.M, k), dtype=xs[0].dtype, device=y.device)
        plan.run_gather(xs, y, out, xcat, my_id, workspace, stream)
        return out, xcat
    (plan.run_unfused if unfused else plan.run)(xs, y, out, my_id, workspace, stream)
    return out
